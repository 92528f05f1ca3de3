// Host-side planner of the pass kernels: the lags between sweeps, the group
// kernel's plan (sweeps per CTA, buffer size, run-ahead, write-back mode) and
// the flag kernel's block size.  Everything here fixes how a pass kernel is
// launched; the C-ABI layer (bb_api.cu) only checks arguments and sequences
// the passes.
#include <algorithm>
#include <vector>

#include "bb_internal.h"

namespace bb {

// Half-step lag of the persistent scheduler: half-step h of sweep r waits for
// sweep r-1 to have completed h + lagh half-steps.  Two half-steps (one full
// cycle) keep the windows disjoint while b - t >= 3; b - t == 2 brings sweep
// r-2's next row block into reach and needs three; the last pass
// (b - t == 1) needs four, the paper's three-cycle rule at half-step grain.
int pass_lag_half(int b, int t) {
    int bp = b - t;
    return bp >= 3 ? 2 : (bp == 2 ? 3 : 4);
}

// Cycle lag of the per-cycle scheduler: the paper's separation condition
// R + n*BW > R + 1 + BW + TW holds for n = 2 when BW > 1 + TW, else n = 3.
int pass_lag_cycle(int b, int t) { return (b > t + 1) ? 2 : 3; }

int group_footprint(const PassArgs& P, int g, int ahead, ChaseKind kind) {
    // Replays the group kernel's buffer bookkeeping for the group at sweep 0:
    // the loader copies in tick u's columns once the storer has written back
    // what ticks < u - ahead alone touch, so the buffer holds the columns from
    // the first one a tick >= tau touches up to the last one ticks
    // <= tau + ahead touch.
    const int ng = (int)std::min<long long>(g, P.nsweeps);
    if (ng <= 0) return 0;
    const int L = P.lagh;
    const bool sym = kind == ChaseKind::kSym;
    const int U = sym ? 1 : 2;  // units per step
    auto steps = [&](long long r) -> long long {
        long long last = P.n - 2 - r - P.bp;
        return last < 0 ? 0 : last / P.b + 1;
    };
    // the columns unit h of sweep r touches (BidiagChase / SymChase)
    auto maxcol = [&](long long r, long long h) -> long long {
        const long long k = h / U;
        const long long c = r + P.bp + k * P.b;
        const long long ce = std::min(c + P.t, P.n - 1);
        return (!sym && (h & 1)) ? std::min(ce + P.b, P.n - 1) : ce;
    };
    auto mincol = [&](long long r, long long h) -> long long {
        if (sym) return h == 0 ? r : r + P.bp + (h - 1) * P.b;
        return r + P.bp + (h >> 1) * P.b;
    };
    long long tend = 0;
    for (int jj = 0; jj < ng; ++jj) tend = std::max(tend, (long long)L * jj + U * steps(jj));
    std::vector<long long> xrun(tend), amin(tend);
    long long x = -1;
    for (long long tau = 0; tau < tend; ++tau) {
        long long a = P.n;
        for (int jj = 0; jj < ng; ++jj) {
            const long long h = tau - (long long)L * jj;
            if (h >= 0 && h < U * steps(jj)) x = std::max(x, maxcol(jj, h));
            if (h < U * steps(jj)) a = std::min(a, mincol(jj, std::max(h, 0LL)));
        }
        xrun[tau] = x;
        amin[tau] = a;
    }
    long long fp = 0, amax = -1;
    for (long long tau = 0; tau < tend; ++tau) {
        amax = std::max(amax, amin[tau]);  // the kernel's A never moves back
        const long long u = std::min(tau + ahead, tend - 1);
        fp = std::max(fp, xrun[u] - amax + 1);
    }
    return (int)fp;
}

bool plan_group(const PassArgs& P, int wmax, size_t elem, int requested, GroupArgs* out, ChaseKind kind,
                size_t selem) {
    const size_t budget = 220 * 1024;
    const int nvec = chase_vecs(kind);
    if (selem == 0) selem = elem;
    GroupArgs best{};
    const int gcap = group_max_warps(wmax, elem);
    const int gmax = requested > 0 ? std::min(requested, gcap) : gcap;
    for (int g = 1; g <= gmax; ++g) {
        GroupArgs ga;
        ga.g = g;
        ga.ngroups = (int)((P.nsweeps + g - 1) / g);
        // rows top .. top + lds - 1 hold the pass's rows (ku-b-t .. ku+t of
        // the upper band; ku .. ku+b+t of the lower, symmetric band), both
        // ends rounded out to 16 bytes (the extra rows are ones the pass
        // leaves alone: copied in and written back unchanged)
        const int q = (int)(16 / selem);
        const int lo = (kind == ChaseKind::kSym) ? P.ku : P.ku - P.b - P.t;
        const int hi = (kind == ChaseKind::kSym) ? P.ku + P.b + P.t : P.ku + P.t;
        ga.top = lo / q * q;
        ga.lds = (hi + 1 - ga.top + q - 1) / q * q;
        ga.ahead = kGroupAhead;
        // wide columns go back with bulk copies (one instruction a column);
        // narrow ones with plain copies, which spare the compute warps a
        // proxy fence every tick
        ga.bulk_store = ((size_t)ga.lds * selem >= 256) ? 1 : 0;
        ga.nslot = std::max(1, group_footprint(P, g, ga.ahead, kind));
        if (group_smem_bytes(ga, wmax, elem, nvec, selem) > budget) break;
        best = ga;
        if (requested > 0 && g == requested) break;
    }
    if (best.g == 0) return false;
    if (requested > 0 && best.g != requested) return false;
    // With g fixed, let the loader run further ahead (a larger buffer) while
    // shared memory allows: the loader then issues its copies earlier and
    // waits less for the storer to free slots.
    for (int a = best.ahead + 1; a <= kMaxStages - 2; ++a) {
        GroupArgs ga = best;
        ga.ahead = a;
        ga.nslot = std::max(1, group_footprint(P, ga.g, a, kind));
        if (group_smem_bytes(ga, wmax, elem, nvec, selem) > budget) break;
        best = ga;
    }
    *out = best;
    return true;
}

// Threads per block of the flag and per-cycle kernels (capped by the
// kernel's register budget when launched).  Measured on the n = 16384 and
// n = 32768 workloads' passes: from b = 96 the most threads the kernel allows
// is fastest; below, one thread per row of the (b + t + 1)-row block with at
// least four warps.
int auto_tpb(int b, int t) {
    if (b >= 96) return 1024;
    const int tpb = ((b + t + 31) / 32) * 32;
    return std::min(1024, std::max(128, tpb));
}
}  // namespace bb
