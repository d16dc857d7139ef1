// Host-only check of the split-KV work schedule (schedule.cuh), compiled with
// nvcc and run on the CPU by tests/test_schedule_cpu.py.  It walks every work
// item exactly as the decode kernels do (TileCursor from item_begin(w) to
// item_begin(w+1), flushing at unit ends and item ends) and checks:
//   * every tile of every unit is visited exactly once, in order;
//   * partial slots are unique across the grid and lie in [0, 2W);
//   * the pieces recorded for each unit match num_pieces / piece_slot, the
//     functions the merging CTA uses to find them;
//   * a unit is written directly exactly when it lies inside one item;
//   * with a unit start cost c > 0, item_begin is the first tile whose cost
//     position reaches the item's cut, found by brute force.
#include <cstdio>
#include <cstdlib>
#include <map>
#include <random>
#include <set>
#include <vector>

#include "../decode_attention_kv_softmax_b300/csrc/schedule.cuh"

using namespace kvdec;

static int fails = 0;
#define CHECK(c, ...)                          \
    do {                                       \
        if (!(c)) {                            \
            if (fails < 20) {                  \
                printf("FAIL %s: ", #c);       \
                printf(__VA_ARGS__);           \
                printf("\n");                  \
            }                                  \
            ++fails;                           \
        }                                      \
    } while (0)

static void run_case(const std::vector<int>& lens, int upb, int grid, int min_tiles, int c = 0) {
    const int B = (int)lens.size();
    std::vector<int> cum(B + 1, 0);
    for (int b = 0; b < B; ++b) cum[b + 1] = cum[b] + (lens[b] + 63) / 64;
    TileSchedule S;
    S.cum = cum.data();
    S.B = B;
    S.upb = upb;
    S.T = (long long)cum[B] * upb;
    S.W = effective_items(S.T, grid, min_tiles);
    S.c = c;
    CHECK(S.W >= 1 && S.W <= grid, "W=%d grid=%d", S.W, grid);
    // item boundaries against a brute-force walk of the cost axis
    if (S.T > 0) {
        std::vector<long long> cost;   // cost position of every tile, in order
        for (int b = 0; b < B; ++b)
            for (int j = 0; j < upb; ++j)
                for (int lt = 0; lt < S.ntiles(b); ++lt)
                    cost.push_back((long long)cost.size() + (long long)c * ((long long)b * upb + j + 1));
        const long long C = S.T + (long long)c * B * upb;
        for (int w = 0; w <= S.W; ++w) {
            const long long cut = C * w / S.W;
            long long want = S.T;
            for (long long t = 0; t < S.T; ++t)
                if (cost[t] >= cut) {
                    want = t;
                    break;
                }
            CHECK(S.item_begin(w) == want, "c=%d item_begin(%d)=%lld want %lld", c, w, S.item_begin(w), want);
        }
    }
    // expected global order
    std::vector<std::tuple<int, int, int>> order;
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < upb; ++j)
            for (int lt = 0; lt < S.ntiles(b); ++lt) order.emplace_back(b, j, lt);
    CHECK((long long)order.size() == S.T, "T mismatch");
    std::map<std::pair<int, int>, std::set<int>> slots_of_unit;
    std::set<int> used_slots;
    std::map<std::pair<int, int>, int> direct;
    long long visited = 0;
    for (int w = 0; w < S.W; ++w) {
        const long long t0 = S.T ? S.item_begin(w) : 0, t1 = S.T ? S.item_begin(w + 1) : 0;
        if (t0 >= t1) continue;
        TileCursor cur;
        cur.start(S, t0);
        bool seg_start = true, item_first = true, unit_first = true;
        for (long long t = t0; t < t1; ++t) {
            if (seg_start) {
                seg_start = false;
                item_first = (t == t0);
                unit_first = (cur.lt == 0);
            }
            auto e = order[t];
            CHECK(std::get<0>(e) == cur.b && std::get<1>(e) == cur.j && std::get<2>(e) == cur.lt,
                  "tile %lld: cursor (%d,%d,%d)", t, cur.b, cur.j, cur.lt);
            CHECK(S.item_of(t) == w, "item_of(%lld)=%d w=%d", t, S.item_of(t), w);
            ++visited;
            const bool seg_end = (cur.lt == cur.nt - 1) || (t == t1 - 1);
            if (seg_end) {
                const bool complete = unit_first && (cur.lt == cur.nt - 1);
                auto key = std::make_pair(cur.b, cur.j);
                if (complete) {
                    direct[key]++;
                    CHECK(S.num_pieces(cur.b, cur.j) == 1, "complete unit with pieces");
                } else {
                    const int slot = 2 * w + (item_first ? 0 : 1);
                    CHECK(slot >= 0 && slot < 2 * S.W, "slot range");
                    CHECK(used_slots.insert(slot).second, "slot %d reused", slot);
                    slots_of_unit[key].insert(slot);
                }
                seg_start = true;
            }
            cur.advance(S);
        }
    }
    CHECK(visited == S.T, "visited %lld of %lld", visited, S.T);
    for (int b = 0; b < B; ++b) {
        if (S.ntiles(b) == 0) continue;
        for (int j = 0; j < upb; ++j) {
            auto key = std::make_pair(b, j);
            const int np = S.num_pieces(b, j);
            if (np == 1) {
                CHECK(direct[key] == 1 && slots_of_unit[key].empty(), "unit (%d,%d) direct", b, j);
                continue;
            }
            std::set<int> want;
            for (int s = 0; s < np; ++s) want.insert(S.piece_slot(b, j, s));
            int w0, kind0;
            S.first_piece(b, j, w0, kind0);
            for (int s = 0; s < np; ++s)
                CHECK(S.piece_slot(b, j, s) == 2 * (w0 + s) + (s == 0 ? kind0 : 0),
                      "unit (%d,%d) first_piece progression", b, j);
            CHECK(want == slots_of_unit[key], "unit (%d,%d) slots", b, j);
            CHECK((int)want.size() == np, "unit (%d,%d) piece count", b, j);
        }
    }
}

int main() {
    std::mt19937 rng(12345);
    int cases = 0;
    // hand-picked edges
    run_case({1}, 1, 1, 1);
    run_case({0, 0, 5}, 2, 7, 1);
    run_case({64, 65, 128, 129}, 3, 5, 1);
    run_case({4096}, 8, 296, 8);
    run_case({0}, 4, 3, 8);
    run_case({64, 0, 0, 4096, 1}, 1, 74, 4, 5);
    run_case({3000, 100, 0, 70000}, 2, 37, 1, 8);
    {
        // hundreds of empty sequences and one long one: items without tiles
        std::vector<int> sparse(300, 0);
        sparse[250] = 5000;
        sparse[17] = 5;
        run_case(sparse, 1, 74, 4, 4);
        run_case(sparse, 1, 4, 4, 4);
    }
    cases += 9;
    for (int it = 0; it < 3000; ++it) {
        const int B = 1 + rng() % 40;
        std::vector<int> lens(B);
        const int maxlen = (it % 3 == 0) ? 300 : (it % 3 == 1 ? 5000 : 70000);
        for (auto& l : lens) l = (rng() % 7 == 0) ? 0 : (int)(rng() % (maxlen + 1));
        const int upb = 1 + rng() % 9;
        const int grid = 1 + rng() % 400;
        const int min_tiles = 1 + rng() % 10;
        const int c = (it % 2 == 0) ? 0 : (int)(rng() % 9);
        run_case(lens, upb, grid, min_tiles, c);
        ++cases;
    }
    if (fails) {
        printf("%d failures over %d cases\n", fails, cases);
        return 1;
    }
    printf("OK %d cases\n", cases);
    return 0;
}
