// Host check of the tensor-core sweeps' persistent schedules (dense and under the causal and band pair
// masks of the torchpairwise guide's Score Expressions): every tile that holds a kept pair is visited
// exactly once, by the CTA ranges in order; every row block gets at least one tile; the order of the row
// blocks (sched_rb, sched_pos) is a permutation; the partial slots (position + CTA) are distinct and below
// RB + G; the CTAs a merge reads are exactly those whose ranges met the row block. The device-side table
// lookups (tile_start, pos_of_tile, SchedCursor) are restated here over a host prefix table; the interval
// of each row block (live_tiles), the order, the tile count (sched_total) and the CTA ranges
// (range_start, cta_of_tile) are the header's own, as are the triangle's numbering and cursor (sym_start,
// SymCursor).
#include <cstdio>
#include <cstdlib>
#include <set>
#include <vector>

#include "../../lazy_score_matrix_gb300/csrc/tp_tc.cuh"

using namespace tp::tc;

static int fails = 0;
#define CHECK(c, ...)                                    \
    do {                                                 \
        if (!(c)) {                                      \
            if (fails < 20) std::printf(__VA_ARGS__);    \
            ++fails;                                     \
        }                                                \
    } while (0)

static bool kept(int pm, long long band, int col, long long r, long long q) {
    // r: a row point of the sweep, q: a streamed point; the score's (query i, key j) pair
    const long long i = col ? q : r, j = col ? r : q;
    if (pm == kPairsCausal) return j <= i;
    if (pm == kPairsBand) return (i > j ? i - j : j - i) <= band;
    return true;
}

static void run(int pm, int col, long long band, long long R, long long C, int BM, int BN, int grid) {
    const Sched s = make_sched(pm, col, band, R, C, BM, BN, nullptr);
    std::vector<long long> pfx(s.RB + 1, 0);
    std::set<long long> order;
    for (long long v = 0; v < s.RB; ++v) {
        const long long rb = sched_rb(s, v);
        CHECK(rb >= 0 && rb < s.RB && sched_pos(s, rb) == v && order.insert(rb).second, "order at %lld\n", v);
        pfx[v + 1] = pfx[v] + sched_tiles(s, rb);
    }
    const long long T = sched_total(s);
    CHECK(T == pfx[s.RB], "total %lld != prefix %lld\n", T, pfx[s.RB]);
    const int G = (int)(T < grid ? T : grid);
    auto start = [&](long long v) { return pm ? pfx[v] : v * s.CT; };
    auto pos_of = [&](long long t) {
        long long v = 0;
        while (v + 1 <= s.RB && start(v + 1) <= t) ++v;
        return v;
    };
    std::set<std::pair<long long, int>> seen;
    std::set<long long> slots;
    std::vector<std::set<int>> touched(s.RB);
    for (int c = 0; c < G; ++c) {
        const long long tb = range_start(T, G, c), te = range_start(T, G, c + 1);
        CHECK(te > tb, "empty range of CTA %d\n", c);
        long long v = pos_of(tb), rb = sched_rb(s, v);
        int c0, c1;
        live_tiles(s, rb, c0, c1);
        int ct = c0 + (int)(tb - start(v));
        for (long long t = tb; t < te; ++t) {
            CHECK(v < s.RB && ct >= c0 && ct < c1 && ct < s.CT, "tile %lld out of its row block\n", t);
            CHECK(seen.insert({rb, ct}).second, "tile (%lld, %d) visited twice\n", rb, ct);
            touched[rb].insert(c);
            if (++ct == c1) {
                ++v;
                if (v < s.RB) rb = sched_rb(s, v), live_tiles(s, rb, ct, c1), c0 = ct;
            }
        }
    }
    CHECK((long long)seen.size() == T, "%zu tiles visited of %lld\n", seen.size(), T);
    for (long long rb = 0; rb < s.RB; ++rb) {
        CHECK(!touched[rb].empty(), "row block %lld has no tile\n", rb);
        const long long v = sched_pos(s, rb);
        for (int c : touched[rb]) CHECK(slots.insert(v + c).second && v + c < s.RB + G, "slot %lld\n", v + c);
        const int lo = cta_of_tile(T, G, start(v)), hi = cta_of_tile(T, G, start(v + 1) - 1);
        CHECK((int)touched[rb].size() == hi - lo + 1 && *touched[rb].begin() == lo && *touched[rb].rbegin() == hi,
              "merge CTAs of row block %lld\n", rb);
        // every tile with a kept pair is in the schedule
        for (int ct = 0; ct < s.CT; ++ct) {
            bool any = false;
            for (long long r = rb * BM; r < R && r < (rb + 1) * BM && !any; ++r)
                for (long long q = (long long)ct * BN; q < C && q < (long long)(ct + 1) * BN && !any; ++q)
                    any = kept(pm, band, col, r, q);
            if (any) CHECK(seen.count({rb, ct}), "kept tile (%lld, %d) skipped (pm %d col %d R %lld C %lld)\n", rb, ct,
                           pm, col, R, C);
        }
    }
}

// The triangle of the X = Y log-sum-exp forward: every tile (I, J >= I) visited once by the CTA ranges in
// order (SymCursor); the row partial slots (I + CTA) distinct and below RB + G; the CTAs the merge reads for
// row block R (cta_of_tile of R's first and last tile) exactly those that swept R's row tiles; every
// off-diagonal tile (I, R) at sym_start(I) + R - I.
static void run_tri(long long N, int grid) {
    const int RB = (int)((N + 127) / 128);
    const long long T = (long long)RB * (RB + 1) / 2;
    const int G = (int)(T < grid ? T : grid);
    std::set<std::pair<int, int>> seen;
    std::set<long long> slots;
    std::vector<std::set<int>> rows(RB);
    std::vector<std::vector<long long>> cols(RB);
    for (int c = 0; c < G; ++c) {
        const long long tb = range_start(T, G, c), te = range_start(T, G, c + 1);
        CHECK(te > tb, "empty triangle range of CTA %d\n", c);
        SymCursor cur(tb, RB);
        for (long long t = tb; t < te; ++t, cur.next()) {
            CHECK(cur.I >= 0 && cur.I <= cur.J && cur.J < RB && sym_start(cur.I, RB) + cur.J - cur.I == t,
                  "triangle tile %lld at (%d, %d)\n", t, cur.I, cur.J);
            CHECK(seen.insert({cur.I, cur.J}).second, "triangle tile (%d, %d) twice\n", cur.I, cur.J);
            rows[cur.I].insert(c);
            if (cur.J != cur.I) cols[cur.J].push_back(t);
        }
    }
    CHECK((long long)seen.size() == T, "%zu triangle tiles of %lld\n", seen.size(), T);
    for (int R = 0; R < RB; ++R) {
        for (int c : rows[R]) CHECK(slots.insert(R + c).second && R + c < RB + G, "triangle slot %d\n", R + c);
        const long long t0 = sym_start(R, RB);
        const int lo = cta_of_tile(T, G, t0), hi = cta_of_tile(T, G, t0 + (RB - R) - 1);
        CHECK((int)rows[R].size() == hi - lo + 1 && *rows[R].begin() == lo && *rows[R].rbegin() == hi,
              "triangle merge CTAs of row block %d\n", R);
        CHECK((int)cols[R].size() == R, "row block %d has %zu column tiles\n", R, cols[R].size());
        for (int I = 0; I < R && I < (int)cols[R].size(); ++I)
            CHECK(cols[R][I] == sym_start(I, RB) + R - I, "column tile (%d, %d)\n", I, R);
    }
}

int main() {
    const long long sizes[] = {1, 5, 64, 127, 128, 129, 300, 517, 1000, 2049};
    const long long bands[] = {0, 1, 17, 63, 64, 200, 5000};
    int cases = 0;
    for (int BN : {64, 128})
        for (int grid : {3, 152})
            for (long long R : sizes)
                for (long long C : sizes)
                    for (int col = 0; col < 2; ++col) {
                        run(0, col, 0, R, C, 128, BN, grid);
                        run(kPairsCausal, col, 0, R, C, 128, BN, grid);
                        for (long long b : bands) run(kPairsBand, col, b, R, C, 128, BN, grid);
                        cases += 9;
                    }
    int tri = 0;
    for (int grid : {1, 3, 7, 152})
        for (long long N = 1; N <= 96 * 128; N += (N < 1100 ? 37 : 1021)) {
            run_tri(N, grid);
            ++tri;
        }
    std::printf("%d schedules, %d triangles, %d failures\n", cases, tri, fails);
    return fails ? 1 : 0;
}
