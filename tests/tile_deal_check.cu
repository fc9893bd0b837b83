// Host check of TileDeal (common.cuh): the tile ranges the attention kernel,
// its combine and the planner share.  For every deal the planner can make
// (balanced; balanced with a per-query start cost; query-aligned) it checks
// that the ranges cover [0, total) in order, that cta_of(g) is the CTA whose
// range holds tile g, that balanced ranges differ by at most one tile, and
// that no range is empty where the planner relies on it.  Deals near 2^31
// units are checked at their range ends.  Prints "cases N bad B".
#include <cstdint>
#include <cstdio>

#include "common.cuh"
using namespace csa;

static long bad = 0, cases = 0;

static void check(const TileDeal& d, bool exhaustive) {
    cases++;
    if (d.begin(0) != 0 || d.begin(d.grid) != d.total) {
        bad++;
        return;
    }
    for (int c = 0; c < d.grid; c++) {
        const int64_t b0 = d.begin(c), b1 = d.begin(c + 1);
        if (b1 <= b0) {
            bad++;
            continue;
        }
        if (exhaustive) {
            for (int64_t g = b0; g < b1; g++)
                if (d.cta_of(g) != c) bad++;
        } else if (d.cta_of(b0) != c || d.cta_of(b1 - 1) != c) {
            bad++;
        }
    }
}

int main() {
    for (int Q = 1; Q <= 70; Q++)
        for (int T = 1; T <= 40; T += (T < 12 ? 1 : 7))
            for (int grid = 1; grid <= 160; grid += (grid < 20 ? 1 : 13)) {
                const int64_t total = (int64_t)Q * T;
                if (grid > total) continue;
                for (int qc = 0; qc <= 5; qc++) {
                    // the planner adds the cost only where every share holds a tile
                    if (qc && (int64_t)Q * (T + qc) / grid < qc + 1) continue;
                    const TileDeal d{total, T, grid, 0, 0, qc};
                    check(d, true);
                    if (qc == 0)
                        for (int c = 0; c < grid; c++) {
                            const int64_t n = d.begin(c + 1) - d.begin(c);
                            if (n != total / grid && n != total / grid + 1) bad++;
                        }
                }
                if (Q <= grid && T >= 2) {  // query-aligned, as planned
                    const int qcta = grid / Q < T ? grid / Q : T;
                    const int qrem = qcta < T ? grid - Q * qcta : 0;
                    check(TileDeal{total, T, Q * qcta + qrem, qcta, qrem, 0}, true);
                }
            }
    const int64_t Ts[] = {18, 130, 2050};
    const int grids[] = {148, 147, 1000};
    for (int64_t T : Ts)
        for (int grid : grids)
            for (int qc = 0; qc <= 5; qc += 5) {
                const int64_t Q = ((1LL << 31) - 1) / (T + qc);
                check(TileDeal{Q * T, T, grid, 0, 0, qc}, false);
            }
    printf("cases %ld bad %ld\n", cases, bad);
    return bad != 0;
}
