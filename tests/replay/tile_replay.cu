// Host replay of the warp-tile kernels' plans and index arithmetic (test infrastructure).
//
// It includes the library source itself and runs its host planner (plan_tile) for a described
// GB300, without a GPU or driver. For every plan it then walks, on the CPU, the partitions and
// shared-memory indexes that the kernels form, and checks that:
//   * the shared-memory regions are ordered, aligned and inside the launch's allocation;
//   * every item (or stream-K job) belongs to exactly one unit, every TMA box of a row to
//     exactly one K slice, and every output to exactly one reducing thread;
//   * each lane's codes, scales and staged-x reads stay inside its ring slot and slice, and the
//     codes of one 8-lane phase hit eight different 16-byte bank groups (no conflicts);
//   * the bulk-copy x staging has aligned copies and an aligned, private mbarrier per slice,
//     and its in-place transpose of 16-byte chunks lands on the tensor-core order;
//   * fused gate/up items hold whole gate/up tile pairs and write every output row once;
//   * the stream-K combine stores every job exactly once with all of its boxes;
//   * the MoE group building places every valid slot in exactly one group of its expert;
//   * the same holds for a seeded random sweep of dense, gate/up and FFN-block shapes.
// Prints "... fails N" and exits non-zero when any check fails.

#include "../../nvfp4_weight_only_gemv_gb300/csrc/nvfp4_gemv.cu"

#include <algorithm>
#include <array>
#include <vector>

using namespace nvfp4;

static int fails = 0;
#define CHECK(c, ...)                                  \
    do {                                               \
        if (!(c)) {                                    \
            if (fails < 30) {                          \
                printf("FAIL %s: ", #c);               \
                printf(__VA_ARGS__);                   \
                printf("\n");                          \
            }                                          \
            ++fails;                                   \
        }                                              \
    } while (0)

static const int kSms = 152, kOptin = 232448, kPerSm = 233472;

static int perm(int nc, int g) { return nc == 2 ? tile_row_perm<2>(g) : tile_row_perm<1>(g); }

// The bulk-copy staging of `slices` K slices of `rows` x rows, kn_max elements at most each.
static void check_bulk(const TileParams& p, int slices, int rows, int kn_max, int k0_step) {
    for (int sl = 0; sl < slices; ++sl) {
        const uint32_t gmax_b = p.misc_off + 8 * 32 + sl * 128;  // the slice's 32 scratch words
        const uint32_t bar_b = gmax_b + 24 * 4;                  // words 24, 25: its mbarrier
        CHECK(bar_b % 8 == 0 && bar_b + 8 <= gmax_b + 128 && bar_b + 8 <= p.bar_off, "slice mbarrier %u", bar_b);
        const uint32_t xs = p.x_off + sl * rows * p.sstride;
        for (int m = 0; m < rows; ++m) {
            CHECK((xs + m * p.sstride) % 16 == 0, "bulk destination alignment");
            CHECK(m * p.sstride + kn_max * 2 <= rows * p.sstride, "bulk destination range");
        }
        CHECK((k0_step * 2) % 16 == 0 && (kn_max * 2) % 16 == 0, "bulk source alignment and size");
        CHECK(rows * kn_max * 2 < (1 << 20), "mbarrier transaction count");
    }
    // the in-place conversion: one trip count per warp whatever the lane or the x values (the
    // loop's only inputs are the warp's number, the slice's warps and the block count), and the
    // blocks its half-warps take cover the slice exactly once
    for (int gw = 1; gw <= 8; gw *= 2) {
        for (int nblk = 0; nblk <= 16 * 96; nblk += (nblk < 64 ? 1 : 37)) {
            std::vector<int> seen(nblk, 0);
            for (int gi = 0; gi < gw; ++gi) {
                const int trips = bulk_convert_trips(gi, gw, nblk);
                for (int lane = 0; lane < 32; ++lane) {
                    const int half = lane >> 4;
                    int own = 0;
                    for (int it = 0; it < trips; ++it) {
                        const int b = gi * 2 + it * gw * 2 + half;
                        if (b < nblk && (lane & 15) == 0) ++seen[b];
                        own += b < nblk;
                    }
                    CHECK(own <= trips, "trip count %d gw %d nblk %d", trips, gw, nblk);
                }
                // the last trip still has work for the warp: no trip is wasted on every lane
                CHECK(trips == 0 || gi * 2 + (trips - 1) * gw * 2 < nblk, "trips gi %d gw %d nblk %d", gi, gw, nblk);
            }
            for (int b = 0; b < nblk; ++b) CHECK(seen[b] == 1, "block %d of %d converted %d times (gw %d)", b, nblk, seen[b], gw);
        }
    }
    // raw chunk 4t + q holds elements 32t + 8q .. + 7; the staged order puts them at chunk 4q + t
    for (int pos = 0; pos < 16; ++pos) {
        const int t = pos >> 2, q = pos & 3;
        for (int e = 0; e < 8; ++e) {
            const int k = 32 * t + 8 * q + e;
            CHECK(2 * k == pos * 16 + 2 * e, "raw position");
            CHECK(mma_x_off(k) == (q * 4 + t) * 16 + 2 * e, "staged position");
        }
    }
}

// A per-item plan (gemv_tile_kernel): layout, partitions, lane indexes, bank conflicts.
static void check_walk(const TilePlan& tp, int M, int K, int groups);

static void check_items(const TilePlan& tp, int M, int K, int groups) {
    const TileParams& p = tp.p;
    const int ksplit = 1 << p.ksplit_log2, S = 1 << p.s_log2;
    const uint32_t kWBox = tp.nc * 2048, kSBox = tp.nc * 256;
    CHECK(tp.smem <= (uint32_t)kOptin, "smem %u", tp.smem);
    CHECK(p.ring_s == p.ring_w + 8u * p.stages * kWBox, "ring_s");
    CHECK(p.x_off >= p.ring_s + 8u * p.stages * kSBox && p.x_off % 128 == 0, "x_off");
    CHECK(p.red_off >= p.x_off + (uint32_t)(ksplit * M) * p.sstride, "red_off");
    CHECK(p.cpart_off >= p.red_off + (ksplit > 1 ? 8192u : 0u), "cpart_off");
    CHECK(p.misc_off >= p.cpart_off + (S > 1 ? 8192u : 0u), "misc_off");
    CHECK(p.bar_off >= p.misc_off + 256 + 8 * 128 && p.bar_off % 8 == 0, "bar_off");
    CHECK(p.bar_off + 8 * 4 * 8 + 1024 <= tp.smem, "total");
    check_walk(tp, M, K, groups);
}

// The partition and index checks of a per-item plan, whatever its shared-memory layout.
static void check_walk(const TilePlan& tp, int M, int K, int groups) {
    const TileParams& p = tp.p;
    const int ksplit = 1 << p.ksplit_log2, S = 1 << p.s_log2;
    const uint32_t kWBox = tp.nc * 2048, kSBox = tp.nc * 256;
    CHECK(p.sstride % 128 == 64, "sstride");
    CHECK(p.stages >= 2 && p.stages <= 4, "stages");
    CHECK(p.nbox * tp.nc * 256 == K, "nbox");
    CHECK(S * ksplit <= p.nbox && p.tpi * ksplit == 8, "ksplit");
    CHECK(tp.grid_x % S == 0 && tp.grid_y == 1 && tp.grid_x / S <= 2 * kSms, "grid");
    {
        const int nbs = (p.nbox + S - 1) / S, nbmax = (nbs + ksplit - 1) / ksplit;
        check_bulk(p, ksplit, M, nbmax * tp.nc * 256, tp.nc * 256);
    }
    // items: a balanced contiguous block per unit, walked without divisions
    const int items = groups * p.ipg, units = tp.grid_x / S;
    CHECK(p.ipg * p.tpi >= p.tiles && p.items_q * units + p.items_r == items && p.items_r < units, "items");
    std::vector<int> seen(items, 0);
    for (int u = 0; u < units; ++u) {
        const int ib = u * p.items_q + std::min(u, p.items_r), ie = ib + p.items_q + (u < p.items_r ? 1 : 0);
        CHECK(ib >= 0 && ie <= items && (ib < ie || items < units), "unit range");  // (fused FFN: idle units)
        for (int i = ib; i < ie; ++i) seen[i]++;
        int grp = ib / p.ipg, t = ib - grp * p.ipg;
        for (int it = ib; it < ie; ++it) {
            CHECK(grp == it / p.ipg && t == it % p.ipg && grp < groups, "item walk");
            if (++t == p.ipg) {
                t = 0;
                ++grp;
            }
        }
    }
    for (int i = 0; i < items; ++i) CHECK(seen[i] == 1, "item %d seen %d", i, seen[i]);
    // every box of a row once over ranks x slices; every output once over ranks
    std::vector<int> box(p.nbox, 0);
    const int outs = p.tpi * 16 * M;
    std::vector<int> oseen(outs, 0);
    for (int rank = 0; rank < S; ++rank) {
        const int c_lo = (rank * p.nbox) >> p.s_log2, c_n = (((rank + 1) * p.nbox) >> p.s_log2) - c_lo;
        const int o_lo = (rank * outs) >> p.s_log2, o_hi = ((rank + 1) * outs) >> p.s_log2;
        for (int i = o_lo; i < o_hi; ++i) oseen[i]++;
        for (int warp = 0; warp < 8; ++warp) {
            const int kslice = warp & (ksplit - 1), tin = warp >> p.ksplit_log2;
            const int b_lo = c_lo + ((kslice * c_n) >> p.ksplit_log2);
            const int b_hi = c_lo + (((kslice + 1) * c_n) >> p.ksplit_log2);
            const int nb = b_hi - b_lo;
            if (tin == 0)
                for (int bb = b_lo; bb < b_hi; ++bb) box[bb]++;
            CHECK(nb >= 1 && (uint32_t)nb * tp.nc * 512 + 64 <= p.sstride, "slice %d boxes %d", kslice, nb);
            const int kn = nb * tp.nc * 256;
            for (int c = 0; c < kn / 8; ++c) CHECK(mma_x_off(c * 8) + 16 <= kn * 2, "staged x write");
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, t = lane & 3;
                const int ra = perm(tp.nc, g), rb = ra + 8;
                CHECK(tin * 128 + rb * 8 + 2 * t + 1 < 1024, "partial-sum index");
                for (int b = 0; b < nb; ++b)
                    for (int c = 0; c < tp.nc; ++c)
                        for (int h = 0; h < 2; ++h) {
                            const int la = ra * tp.nc + c, lb = rb * tp.nc + c, u = h * 4 + t;
                            CHECK(la * 128 + ((u ^ (la & 7)) << 4) + 16 <= (int)kWBox, "codes read a");
                            CHECK(lb * 128 + ((u ^ (lb & 7)) << 4) + 16 <= (int)kWBox, "codes read b");
                            CHECK(lb * 16 + h * 8 + 2 * t + 2 <= (int)kSBox, "scales read");
                            CHECK((b * tp.nc * 2 + c * 2 + h) * 256 + 256 <= kn * 2, "staged x read");
                        }
            }
        }
    }
    for (int i = 0; i < p.nbox; ++i) CHECK(box[i] == 1, "box %d covered %d times", i, box[i]);
    for (int i = 0; i < outs; ++i) CHECK(oseen[i] == 1, "output %d", i);
    // codes of one 8-lane phase: eight different 16-byte groups of a 128-byte line
    for (int c = 0; c < tp.nc; ++c)
        for (int h = 0; h < 2; ++h)
            for (int ph = 0; ph < 4; ++ph) {
                int used[8] = {0};
                for (int l = ph * 8; l < ph * 8 + 8; ++l) {
                    const int g = l >> 2, t = l & 3;
                    const int la = perm(tp.nc, g) * tp.nc + c, u = h * 4 + t;
                    used[((la * 128 + ((u ^ (la & 7)) << 4)) % 128) / 16]++;
                }
                for (int i = 0; i < 8; ++i) CHECK(used[i] == 1, "bank conflict");
            }
}

// Fused gate/up: gate tile j and up tile j form tiles 2j, 2j + 1 of one item.
static void check_swiglu(const TilePlan& tp, int M, int N, bool separate_layout = true) {
    const TileParams& p = tp.p;
    const int ksplit = 1 << p.ksplit_log2, S = 1 << p.s_log2;
    const int rt = (N + 15) / 16;
    CHECK(p.tiles == 2 * rt, "tiles %d", p.tiles);
    CHECK(p.tpi % 2 == 0, "tiles per item %d", p.tpi);
    if (separate_layout) {
        CHECK(p.misc_off >= p.cpart_off + 8192u, "partial sums allocated");
        CHECK(p.cpart_off >= p.red_off + (ksplit > 1 ? 8192u : 0u), "partial sums after the reduction buffer");
    }
    const int units = tp.grid_x / S;
    std::vector<int> rows(N, 0);
    for (int u = 0; u < units; ++u) {
        const int ib = u * p.items_q + std::min(u, p.items_r), ie = ib + p.items_q + (u < p.items_r ? 1 : 0);
        for (int t = ib; t < ie; ++t) {
            for (int tin = 0; tin < p.tpi; ++tin) {  // warp tin loads tile t * tpi + tin
                const int L = t * p.tpi + tin;
                if (L >= p.tiles) continue;
                CHECK((L & 1) == (tin & 1), "gate/up parity");
                CHECK((L >> 1) * 16 < rt * 16, "row0");
            }
            const int pair_outs = (p.tpi / 2) * 16 * M;
            for (int rank = 0; rank < S; ++rank) {
                int o_lo = 0, o_hi = pair_outs;
                if (S > 1) {
                    o_lo = (rank * pair_outs) >> p.s_log2;
                    o_hi = ((rank + 1) * pair_outs) >> p.s_log2;
                }
                for (int i = o_lo; i < o_hi; ++i) {
                    const int pi = i / (16 * M), rem = i - pi * 16 * M, r = rem / M, m = rem - r * M;
                    const int jt = t * (p.tpi / 2) + pi, row = jt * 16 + r;
                    CHECK((2 * pi + 1) * 128 + r * 8 + m < 1024, "partial-sum read");
                    if (2 * jt < p.tiles && row < N && m == 0) rows[row]++;
                }
            }
        }
    }
    for (int n = 0; n < N; ++n) CHECK(rows[n] == 1, "row %d written %d times", n, rows[n]);
}

// The stream-K kernel's box walk and combine: every job stored once, with all of its boxes.
// Group-aligned plans (items_r != 0) also keep every CTA inside one of the ng groups.
static void check_sk(const TilePlan& tp, int jobs_total, int ng) {
    const TileParams& p = tp.p;
    const int nbox = p.nbox, G = tp.grid_x;
    CHECK(tp.smem <= (uint32_t)kOptin && p.bar_off + 256 + 1024 <= tp.smem, "stream-K smem");
    CHECK(p.x_off >= p.ring_s + 8u * p.stages * tp.nc * 256, "stream-K x_off");
    CHECK(p.misc_off >= p.x_off + (uint32_t)p.M * p.sstride, "stream-K misc_off");
    CHECK(1024u <= (uint32_t)p.stages * tp.nc * 2048u, "partial records fit a drained ring");
    check_bulk(p, 1, p.M, p.nbox * tp.nc * 256, 256);
    std::vector<int> stored(jobs_total, 0), boxes(jobs_total, 0);
    for (int cta = 0; cta < G; ++cta) {
        const int q = jobs_total / G, r = jobs_total % G;
        int j0 = cta * q + std::min(cta, r), j1 = j0 + q + (cta < r ? 1 : 0);
        if (p.items_r) {  // the kernel's group-aligned ranges
            CHECK(G >= ng, "a CTA per group");
            const int g = static_cast<int>((static_cast<long long>(cta) + 1) * ng - 1) / G;
            const int lo = static_cast<int>(static_cast<long long>(G) * g / ng);
            const int c = static_cast<int>(static_cast<long long>(G) * (g + 1) / ng) - lo;
            const int i = cta - lo;
            CHECK(c >= 1 && i >= 0 && i < c, "group share");
            j0 = g * p.tiles + static_cast<int>(static_cast<long long>(p.tiles) * i / c);
            j1 = g * p.tiles + static_cast<int>(static_cast<long long>(p.tiles) * (i + 1) / c);
            CHECK(j0 >= g * p.tiles && j1 <= (g + 1) * p.tiles, "CTA inside its group");
            CHECK(p.M >= 1 && p.M <= 8, "aligned row bound");
        }
        const int total = (j1 - j0) * nbox;
        int bsv[8], bev[8], rjob[8][2], rcnt[8][2];  // records: [warp][first/last] -> (job, boxes)
        for (int w = 0; w < 8; ++w) {
            bsv[w] = (w * total) >> 3;
            bev[w] = ((w + 1) * total) >> 3;
            rjob[w][0] = rjob[w][1] = -1;
            rcnt[w][0] = rcnt[w][1] = 0;
        }
        for (int w = 0; w < 8; ++w) {
            const int bs = bsv[w], be = bev[w];
            if (bs >= be) continue;
            int job = j0 + bs / nbox, kb = bs % nbox, cnt = 0;
            const int first = job;
            bool whole = kb == 0;
            for (int b = bs; b < be; ++b) {
                ++cnt;
                if (kb == nbox - 1 || b == be - 1) {
                    if (whole && kb == nbox - 1) {
                        stored[job]++;
                        boxes[job] += cnt;
                        CHECK(cnt == nbox, "whole job box count");
                    } else {
                        const int sl = job == first ? 0 : 1;
                        CHECK(rjob[w][sl] == -1, "record slot reused");
                        rjob[w][sl] = job;
                        rcnt[w][sl] = cnt;
                    }
                    cnt = 0;
                    kb = 0;
                    whole = true;
                    ++job;
                } else {
                    ++kb;
                }
            }
        }
        for (int w = 0; w < 8; ++w) {  // the warp holding a cut job's first box adds the records
            const int bs = bsv[w], be = bev[w];
            if (bs >= be) continue;
            const int jf = j0 + bs / nbox, jl = j0 + (be - 1) / nbox;
            for (int sl = 0; sl < 2; ++sl) {
                const int j = sl == 0 ? jf : jl;
                if (sl == 1 && jl == jf) break;
                const int jb = (j - j0) * nbox, je = jb + nbox;
                if (jb < bs || je <= be) continue;  // starts in an earlier warp, or whole here
                CHECK(rjob[w][sl] == j, "finishing warp's record");
                int sum = rcnt[w][sl];
                for (int v = w + 1; v < 8; ++v) {
                    if (bsv[v] >= je) break;
                    if (bev[v] > bsv[v]) {
                        CHECK(rjob[v][0] == j, "following warp's record: job %d vs %d", rjob[v][0], j);
                        sum += rcnt[v][0];
                    }
                }
                stored[j]++;
                boxes[j] += sum;
            }
        }
    }
    for (int j = 0; j < jobs_total; ++j)
        CHECK(stored[j] == 1 && boxes[j] == nbox, "job %d stored %d times, %d boxes", j, stored[j], boxes[j]);
}

// tile_moe_groups on the host: every valid slot in exactly one group of its expert, slot order.
static void check_moe_groups(int slots, int E, int top_k, bool per_slot, unsigned seed) {
    std::vector<int> ids(slots);
    unsigned st = seed;
    for (int s = 0; s < slots; ++s) {  // some ids out of range on purpose
        st = st * 1103515245u + 12345u;
        ids[s] = static_cast<int>((st >> 8) % static_cast<unsigned>(E + 2)) - 1;
    }
    int expert[32], count[32], slot[32][8], xrow[32][8], rank[32];
    bool valid[32];
    uint32_t same[32], leaders = 0;
    for (int l = 0; l < 32; ++l) valid[l] = l < slots && ids[l] >= 0 && ids[l] < E;
    for (int l = 0; l < 32; ++l) {  // __match_any_sync over the lanes' keys
        same[l] = 0;
        for (int u = 0; u < 32; ++u) {
            const int a = valid[l] ? ids[l] : -1 - l, b = valid[u] ? ids[u] : -1 - u;
            if (a == b) same[l] |= 1u << u;
        }
    }
    for (int l = 0; l < 32; ++l) {
        rank[l] = __builtin_popcount(same[l] & ((1u << l) - 1u));
        if (valid[l] && (rank[l] & 7) == 0) leaders |= 1u << l;
    }
    for (int l = 0; l < 32; ++l) {
        if (!valid[l]) continue;
        uint32_t rest = same[l];
        for (int i = 0; i < (rank[l] & ~7); ++i) rest &= rest - 1u;
        const int lead = __builtin_ffs(rest) - 1;
        const int g = __builtin_popcount(leaders & ((1u << lead) - 1u)), j = rank[l] & 7;
        CHECK(g >= 0 && g < 32 && j < 8, "group index %d %d", g, j);
        slot[g][j] = l;
        xrow[g][j] = per_slot ? l : l / top_k;
        if (j == 0) {
            expert[g] = ids[l];
            count[g] = std::min(8, __builtin_popcount(same[l]) - rank[l]);
        }
    }
    const int ngroups = __builtin_popcount(leaders);
    std::vector<int> seen(slots, 0);
    for (int g = 0; g < ngroups; ++g) {
        CHECK(count[g] >= 1 && count[g] <= 8, "group size");
        for (int j = 0; j < count[g]; ++j) {
            const int s = slot[g][j];
            CHECK(s >= 0 && s < slots && ids[s] == expert[g], "member");
            seen[s]++;
            if (j) CHECK(slot[g][j] > slot[g][j - 1], "slot order");
            CHECK(xrow[g][j] >= 0 && xrow[g][j] < 32, "x row");
        }
    }
    for (int s = 0; s < slots; ++s) CHECK(seen[s] == ((ids[s] >= 0 && ids[s] < E) ? 1 : 0), "slot %d seen %d", s, seen[s]);
}

// tile_moe_groups_big and tile_moe_window on the host, step for step: leaders are experts' first
// slots, groups of up to 8 slots numbered by an exclusive scan over the leaders; every valid slot
// lands in exactly one window entry when the CTA ranges walk all groups in windows.
static void check_moe_groups_big(int slots, int E, int top_k, bool per_slot, unsigned seed) {
    std::vector<int> ids(slots), cnt(slots), ngr(slots);
    unsigned r = seed;
    for (int s = 0; s < slots; ++s) {
        r = r * 1103515245u + 12345u;
        const int hot = (r >> 8) % 4 == 0;  // a quarter of the slots go to three hot experts
        ids[s] = hot ? (int)((r >> 4) % 3) : (int)((r >> 12) % (E + 2)) - 1;  // some invalid (-1, E)
    }
    std::vector<int> sid(slots);
    for (int s = 0; s < slots; ++s) sid[s] = (ids[s] >= 0 && ids[s] < E) ? ids[s] : -1;
    for (int t = 0; t < slots; ++t) {
        bool leader = sid[t] >= 0;
        for (int u = 0; u < t && leader; ++u) leader = sid[u] != sid[t];
        int c = 0;
        if (leader)
            for (int u = t; u < slots; ++u) c += sid[u] == sid[t];
        cnt[t] = c;
        ngr[t] = (c + 7) / 8;
    }
    int run = 0;
    for (int t = 0; t < slots; ++t) {
        const int v = ngr[t];
        ngr[t] = run;
        run += v;
    }
    const int ngroups = run;
    std::vector<int> seen(slots, 0);
    for (int g_lo = 0; g_lo < ngroups; g_lo += kMoeWindow) {
        const int g_hi = std::min(ngroups - 1, g_lo + kMoeWindow - 1);
        int count[kMoeWindow] = {}, expert[kMoeWindow], slot[kMoeWindow][8];
        for (int t = 0; t < slots; ++t) {
            const int c = cnt[t];
            if (c == 0) continue;
            const int gf = ngr[t], gl = gf + (c + 7) / 8 - 1;
            if (gl < g_lo || gf > g_hi) continue;
            int i = 0;
            for (int u = t; u < slots && i < c; ++u) {
                if (sid[u] != sid[t]) continue;
                const int g = gf + (i >> 3), j = i & 7;
                if (g >= g_lo && g <= g_hi) {
                    slot[g - g_lo][j] = u;
                    if (j == 0) {
                        expert[g - g_lo] = sid[t];
                        count[g - g_lo] = std::min(8, c - i);
                    }
                }
                ++i;
            }
        }
        std::vector<int> rows;
        for (int lg = 0; lg <= g_hi - g_lo; ++lg) {
            CHECK(count[lg] >= 1 && count[lg] <= 8, "big group size %d", count[lg]);
            for (int j = 0; j < count[lg]; ++j) {
                const int u = slot[lg][j];
                CHECK(u >= 0 && u < slots && sid[u] == expert[lg], "big member");
                if (j) CHECK(slot[lg][j] > slot[lg][j - 1], "big slot order");
                seen[u]++;
                rows.push_back(per_slot ? u : u / top_k);
            }
        }
        std::sort(rows.begin(), rows.end());
        rows.erase(std::unique(rows.begin(), rows.end()), rows.end());
        CHECK(rows.size() <= 32, "window rows %zu", rows.size());
    }
    for (int s = 0; s < slots; ++s) CHECK(seen[s] == (sid[s] >= 0 ? 1 : 0), "big slot %d seen %d", s, seen[s]);
}

// The fused FFN launch: both phases share the ring; A's x slices and pair buffer and B's h
// slices share the x region; each phase's indexes pass the per-item checks; A's round-robin and
// B's reversed round-robin item deals cover every item exactly once; the readiness counts add up
// (every A item counts into the B slice holding its h rows, and each slice expects exactly the
// items it gets); and the issue order (A's boxes, then B's, skipping tiles past the end) is
// exactly the order in which the phases consume them.
static void check_ffn(const FfnPlan& fp, int M, int H, int I) {
    const TileParams& A = fp.p.a;
    const TileParams& B = fp.p.b;
    const int nc = fp.nc, st = A.stages;
    const int ka = 1 << A.ksplit_log2, kb = 1 << B.ksplit_log2;
    CHECK(fp.grid == 2 * kSms, "grid %d", fp.grid);
    CHECK(A.s_log2 == 0 && B.s_log2 == 0 && A.stages == B.stages, "one ring, no clusters");
    for (uint32_t TileParams::*f : {&TileParams::ring_w, &TileParams::ring_s, &TileParams::x_off, &TileParams::red_off,
                                    &TileParams::cpart_off, &TileParams::misc_off, &TileParams::bar_off})
        CHECK(A.*f == B.*f, "shared layout");
    CHECK(A.ring_s == A.ring_w + 8u * st * nc * 2048 && A.x_off == A.ring_s + 8u * st * nc * 256, "rings");
    CHECK(A.x_off % 128 == 0 && A.cpart_off % 128 == 0, "x region alignment");
    CHECK(A.cpart_off >= A.x_off + (uint32_t)(ka * M) * A.sstride, "A's x slices before its pair buffer");
    CHECK(A.red_off >= A.cpart_off + 8192u, "pair buffer inside the x region");
    CHECK(A.red_off >= A.x_off + (uint32_t)(kb * M) * B.sstride, "B's h slices inside the x region");
    CHECK(A.misc_off >= A.red_off + ((ka > 1 || kb > 1) ? 8192u : 0u), "reduction buffer");
    CHECK(A.bar_off >= A.misc_off + 256 + 8 * 128 && A.bar_off % 8 == 0, "bar_off");
    CHECK(A.bar_off + 8 * 4 * 8 + 1024 <= fp.smem && fp.smem <= (uint32_t)(kPerSm / 2 - 1024), "two CTAs per SM");
    CHECK(A.M == M && B.M == M && A.K == H && A.N == I && B.K == I && B.N == H && A.swiglu == 1, "shapes");
    CHECK(kb <= kFfnSlices && 32 * (1 + kFfnSlices) * 4 <= kFfnSyncBytes, "counters inside the workspace header");
    TilePlan ta{}, tb{};
    ta.p = A; ta.nc = nc; ta.grid_x = fp.grid; ta.grid_y = 1; ta.smem = fp.smem;
    tb.p = B; tb.nc = nc; tb.grid_x = fp.grid; tb.grid_y = 1; tb.smem = fp.smem;
    check_walk(ta, M, H, 1);
    check_swiglu(ta, M, I, false);
    check_walk(tb, M, I, 1);
    const int units = fp.grid;
    // the deals: every item of each phase on exactly one CTA
    for (int ph = 0; ph < 2; ++ph) {
        const TileParams& q = ph ? B : A;
        const int items = q.items_q * units + q.items_r;
        std::vector<int> seen(items, 0);
        for (int u = 0; u < units; ++u) {
            const FfnGeo g = ffn_geo(q, 0, u, units, ph == 1);
            for (int j = 0; j < g.count; ++j) {
                const int it = g.first + j * g.stride;
                CHECK(it >= 0 && it < items, "phase %d item %d", ph, it);
                if (it >= 0 && it < items) seen[it]++;
            }
        }
        for (int i = 0; i < items; ++i) CHECK(seen[i] == 1, "phase %d item %d dealt %d times", ph, i, seen[i]);
    }
    // readiness counts: A items per B slice, as counted and as expected
    {
        const int items_a = A.items_q * units + A.items_r;
        std::vector<int> got(kb, 0);
        for (int it = 0; it < items_a; ++it) {
            if (!(2 * it * (A.tpi >> 1) < A.tiles)) continue;
            const int r0 = it * ffn_item_rows(A);
            const int s = ffn_slice_of(B, r0, nc);
            CHECK(s >= 0 && s < kb && ffn_slice_lo(B, s, nc) <= r0 && r0 < ffn_slice_lo(B, s + 1, nc), "slice of row %d", r0);
            CHECK(r0 + ffn_item_rows(A) <= ffn_slice_lo(B, s + 1, nc) || r0 + ffn_item_rows(A) > I,
                  "item %d straddles slices", it);
            if (s >= 0 && s < kb) got[s]++;
        }
        for (int s = 0; s < kb; ++s) CHECK(got[s] == ffn_slice_items(A, B, s, nc), "slice %d counts %d, expects %d", s,
                                           got[s], ffn_slice_items(A, B, s, nc));
        for (int w = 0; w < 8; ++w) {
            const FfnGeo g = ffn_geo(B, w, 0, units, true);
            CHECK(ffn_slice_lo(B, g.kslice, nc) == g.b_lo * nc * 256 &&
                  ffn_slice_lo(B, g.kslice + 1, nc) == (g.b_lo + g.nb) * nc * 256, "warp %d slice bounds", w);
        }
    }
    // issue order against consumption order, per CTA and warp
    for (int unit = 0; unit < units; unit += (unit < 8 || unit > units - 8) ? 1 : 13) {
        for (int warp = 0; warp < 8; ++warp) {
            const FfnGeo ga = ffn_geo(A, warp, unit, units, false), gb = ffn_geo(B, warp, unit, units, true);
            std::vector<std::array<int, 3>> cons, iss;
            for (int ph = 0; ph < 2; ++ph) {
                const TileParams& q = ph ? B : A;
                const FfnGeo& g = ph ? gb : ga;
                for (int j = 0; j < g.count; ++j) {
                    const int tile = (g.first + j * g.stride) * q.tpi + g.tin;
                    if (tile < q.tiles)
                        for (int b = 0; b < g.nb; ++b) cons.push_back({ph, tile, g.b_lo + b});
                }
            }
            int iph = 0, jj = 0, box = 0;
            for (int guard = 0; guard < 1000000; ++guard) {
                bool done = false;
                for (;;) {
                    if (iph == 2) { done = true; break; }
                    const bool pa = iph == 0;
                    const FfnGeo& g = pa ? ga : gb;
                    const int tpi = pa ? A.tpi : B.tpi, tiles = pa ? A.tiles : B.tiles;
                    while (jj < g.count && (box >= g.nb || (g.first + jj * g.stride) * tpi + g.tin >= tiles)) {
                        ++jj;
                        box = 0;
                    }
                    if (jj < g.count) break;
                    iph = pa ? 1 : 2;
                    jj = 0;
                    box = 0;
                }
                if (done) break;
                const TileParams& q = iph ? B : A;
                const FfnGeo& g = iph ? gb : ga;
                iss.push_back({iph, (g.first + jj * g.stride) * q.tpi + g.tin, g.b_lo + box});
                ++box;
            }
            CHECK(iss == cons, "unit %d warp %d: %zu boxes issued, %zu consumed", unit, warp, iss.size(), cons.size());
        }
    }
}

int main() {
    DeviceInfo d;
    d.sm_count = kSms;
    d.smem_optin = kOptin;
    d.smem_per_sm = kPerSm;
    d.init = true;
    const uint8_t* fake = reinterpret_cast<const uint8_t*>(static_cast<uintptr_t>(4096));
    const uint8_t* w[2] = {fake, fake};
    const int shapes[][2] = {{256, 512},   {4096, 4096}, {1024, 4096}, {12288, 4096}, {4096, 12288},
                             {151936, 4096}, {3072, 4096}, {4096, 1536}, {1000, 1024}, {37, 2560},
                             {300, 512},   {1, 256},     {5, 256},     {513, 768},   {50, 256},
                             {2000, 2048}, {64, 256},    {300, 12288}, {4096, 768}};
    int n_items = 0, n_sw = 0, n_moe = 0, n_aligned = 0;
    for (const auto& s : shapes)
        for (int M = 1; M <= 8; ++M) {
            for (int groups = 1; groups <= 2; ++groups) {
                TilePlan tp{};
                CHECK(plan_tile(tp, M, s[0], s[1], groups, d, w, w, fake, false, 0, 0, false, false), "no plan");
                if (tp.sk) continue;
                check_items(tp, M, s[1], groups);
                ++n_items;
            }
            TilePlan tp{};
            CHECK(plan_tile(tp, M, s[0], s[1], 2, d, w, w, fake, false, 0, 0, true, false), "no fused plan");
            CHECK(!tp.sk, "fused plan in stream-K form");
            check_items(tp, M, s[1], 1);
            check_swiglu(tp, M, s[0]);
            ++n_sw;
        }
    for (unsigned seed = 1; seed < 2000; ++seed)
        for (int slots : {1, 5, 8, 17, 32})
            for (int E : {1, 3, 40, 288}) check_moe_groups(slots, E, 8, seed & 1, seed * 31 + slots + E);
    // MoE plans: {N, K, x rows}; the group tables follow the barriers
    for (const auto& mm : std::vector<std::array<int, 3>>{{3072, 4096, 4}, {4096, 1536, 32}, {200, 1024, 15},
                                                          {512, 1024, 12}, {64, 256, 32}}) {
        TilePlan tp{};
        if (!plan_tile(tp, 8, mm[0], mm[1], 30, d, w, w, fake, true, mm[2], 32, false, false)) {
            CHECK(false, "no MoE plan for %d x %d", mm[0], mm[1]);
            continue;
        }
        ++n_moe;
        if (tp.p.items_r && tp.sk) ++n_aligned;
        if (tp.sk) {
            for (int ng = 1; ng <= 32; ++ng) check_sk(tp, ng * tp.p.tiles, ng);
        } else {
            check_items(tp, tp.p.M, mm[1], 30);
        }
        // the staged x rows of any unit fit the planned capacity for 1..32 groups
        for (int ng = 1; ng <= 32 && !tp.sk; ++ng) {
            const int units = tp.grid_x, items = ng * tp.p.ipg, q = items / units, r = items % units;
            for (int u = 0; u < units; ++u) {
                const int ib = u * q + std::min(u, r), ie = ib + q + (u < r ? 1 : 0);
                if (ib >= ie) continue;
                const int span = (ie - 1) / tp.p.ipg - ib / tp.p.ipg + 1;
                CHECK(std::min(mm[2], 8 * span) <= tp.p.M, "x rows ng=%d unit=%d", ng, u);
            }
        }
        CHECK(tp.p.moe_off % 16 == 0 && tp.p.moe_off >= tp.p.bar_off + 8 * 4 * 8, "group tables offset");
        CHECK(tp.p.moe_off + sizeof(TileMoe) + 1024 <= tp.smem, "group tables inside the allocation");
    }
    // more than 32 slots: the stream-K form, scratch room in the x region, windows of groups
    int n_big = 0;
    for (unsigned seed = 1; seed < 400; ++seed)
        for (int slots : {33, 40, 64, 128, 200, 256})
            for (int E : {3, 40, 288}) check_moe_groups_big(slots, E, 8, seed & 1, seed * 131 + slots + E);
    for (const auto& mm : std::vector<std::array<int, 2>>{{3072, 4096}, {4096, 1536}, {200, 1024}, {64, 256}}) {
        for (int slots : {40, 64, 128, 256}) {
            for (int per_slot = 0; per_slot < 2; ++per_slot) {
                TilePlan tp{};
                const int xrows = per_slot ? slots : slots / 8;
                if (!plan_tile(tp, 8, mm[0], mm[1], expected_groups(288, slots / 8, 8), d, w, w, fake, true, xrows,
                               slots, false, false)) {
                    CHECK(false, "no MoE plan for %d x %d, %d slots", mm[0], mm[1], slots);
                    continue;
                }
                ++n_big;
                CHECK(tp.sk, "more than 32 slots take the stream-K form");
                CHECK(tp.p.misc_off - tp.p.x_off >= kMoeScratchInts * 4u, "group-building scratch in the x region");
                CHECK(tp.p.M <= 8 && tp.p.M >= 1, "x rows staged");
                for (int ng = 1; ng <= slots; ng += (ng < 16 ? 1 : 7)) {
                    check_sk(tp, ng * tp.p.tiles, ng);
                    const int jobs = ng * tp.p.tiles, G = tp.grid_x;
                    for (int cta = 0; cta < G && !tp.p.items_r; ++cta) {
                        const int q = jobs / G, r = jobs % G;
                        const int j0 = cta * q + std::min(cta, r), j1 = j0 + q + (cta < r ? 1 : 0);
                        if (j0 < j1) CHECK((j1 - 1) / tp.p.tiles - j0 / tp.p.tiles + 1 <= kMoeWindow, "window span");
                    }
                }
            }
        }
    }
    // a seeded random sweep of shapes: N up to 40000, K a multiple of 256 up to 16384, M 1..8
    int n_rand = 0;
    uint32_t rs = 12345u;
    auto rnd = [&](uint32_t n) {
        rs = rs * 1664525u + 1013904223u;
        return (rs >> 8) % n;
    };
    for (int it = 0; it < 240; ++it) {
        const int N = 1 + static_cast<int>(rnd(40000)), K = 256 * (1 + static_cast<int>(rnd(64))),
                  M = 1 + static_cast<int>(rnd(8));
        const int groups = 1 + static_cast<int>(rnd(2));
        TilePlan tp{};
        if (plan_tile(tp, M, N, K, groups, d, w, w, fake, false, 0, 0, false, false) && !tp.sk) {
            check_items(tp, M, K, groups);
            ++n_rand;
        }
        TilePlan ts{};
        if (plan_tile(ts, M, N, K, 2, d, w, w, fake, false, 0, 0, true, false)) {
            check_items(ts, M, K, 1);
            check_swiglu(ts, M, N);
            ++n_rand;
        }
    }
    // the FFN block in one launch: {H, I}
    int n_ffn = 0;
    std::vector<std::array<int, 2>> ffn_shapes{{4096, 12288}, {4096, 1536}, {1024, 512}, {256, 256},
                                               {2048, 768}, {4096, 4096}, {768, 3072}, {4096, 768}};
    for (int it = 0; it < 40; ++it)
        ffn_shapes.push_back({256 * (1 + static_cast<int>(rnd(16))), 256 * (1 + static_cast<int>(rnd(24)))});
    for (const auto& f : ffn_shapes)
        for (int M = 1; M <= 8; ++M) {
            FfnPlan fp{};
            if (!plan_ffn(fp, M, f[0], f[1], d)) continue;
            check_ffn(fp, M, f[0], f[1]);
            ++n_ffn;
        }
    printf("per-item plans %d, fused gate/up plans %d, MoE plans %d, group-aligned %d, large MoE plans %d, "
           "FFN plans %d, random plans %d, fails %d\n",
           n_items, n_sw, n_moe, n_aligned, n_big, n_ffn, n_rand, fails);
    return fails != 0;
}
