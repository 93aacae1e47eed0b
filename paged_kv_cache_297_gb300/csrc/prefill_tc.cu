// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Same operation as the mma.sync kernel in prefill.cu: query j of a chunk of n
// tokens of a sequence with L cached tokens attends causally to tokens
// 0 .. L-n+j (caffein.top, "Chunked Prefill"), K/V gathered through the block
// table.  Used for bf16 caches with head_dim 128.
//
// Work unit: one CTA per (tile of 128 packed query rows, kv head, sequence);
// row r of the tile is query position R / G, head kvh*G + R % G
// (R = tile*128 + r), so the G heads of a kv head share every K/V tile.
// Key tiles are 128 keys (8 cache blocks):
//   S(t)  = Q K(t)^T : tcgen05.mma M=128, N=128, K=d; A = Q, B = K (smem)
//   O    += P(t) V(t): tcgen05.mma M=128, N=d, K=128; A = P (TMEM),
//                      B = V (smem, MN-major); accumulators in TMEM.
// A tcgen05.mma costs roughly the same to issue whatever its N, so tiles are
// as wide as tensor memory allows.
// Warp roles (one CTA per SM, 12 warps):
//   * two softmax teams of 4 warps: team 0 takes key tiles 0, 2, 4, ..., team 1
//     tiles 1, 3, 5, ...  Thread r of a team owns query row r (TMEM lane r).
//     It reads its 128 scores from TMEM 64 at a time, twice (once for the row
//     maximum, once for the powers, so only 64 stay in registers), masks them,
//     computes p = 2^(s * scale * log2 e - m) (one paired multiply-add per two
//     elements, ex2.approx on the special-function unit) and stores P as bf16 pairs
//     over the first 64 columns of the same S buffer, handing each half (64
//     keys) to the MMA warp as soon as it is stored.  Each team has its own
//     S/P buffer, O accumulator and running (m, l); the two partial results
//     are merged by log-sum-exp at the end.  The teams run independently, so
//     one team's softmax overlaps the other team's MMAs.
//   * one MMA-issuing thread (lane 0 of warp 8) for both teams, tiles in
//     order: PV(t) (half by half as P(t) is stored) and then S(t+2) into
//     the same buffer.  tcgen05.mma operations issued by one thread execute
//     in order, so S(t+2) cannot overwrite P(t) before PV(t) has read it,
//     and a team that sees S(t) complete also knows its previous PV is
//     done.  The pipe then runs PV(t), S(t+2), PV(t+1), S(t+3), ...: each
//     team's next S completes a unit before the other team's, so the teams'
//     softmax phases stay apart.  One thread also waits on every ring phase
//     in order: with a stage's consecutive tiles going to different
//     waiters, a parity wait could not tell "phase k done" from "phase k-1
//     still running".  (Two issuing threads, one per team, measured the
//     same once their waits were ordered.)
//   * two loader warps, one for K and one for V, that gather tiles through
//     the block table: a tile of whole blocks with 2-D TMA boxes (one
//     16-row x 64-column box per block and half; the cache is viewed as
//     [num_blocks * num_kv_heads * 16 rows][128] with 128-byte swizzle, which
//     writes exactly the layout the MMAs read); the last tile, which may end
//     inside a block, with zero-filling 16-byte cp.async instead, because rows
//     past the context may hold anything (even NaN) and P = 0 times NaN would
//     still poison O.  K and V use 3-stage rings, refilled when the S (for
//     K) or PV (for V) that read a stage has finished: a tile's load then
//     starts about three tiles before its MMA, more than an HBM round trip.
// The running max of a row is only moved when a tile maximum exceeds it by
// more than 8 (log2 units), so P <= 256 and O is rarely rescaled; numerator
// and denominator share the same reference, so the result is exact.
//
// TMEM columns (all 512): S/P of team t at 128t, O of team t at 256 + 128t.
// Shared memory, all in the 128-byte-swizzled canonical layout (8-row atoms
// of 8 x 128 bytes, 16-byte chunk c of row r at chunk c ^ (r % 8)):
//   Q : two 64-column halves of 128 rows                       (32 KB)
//   K : three stages x two 64-column halves of 128 rows        (96 KB)
//   V : three stages x two 64-column halves of 128 rows        (96 KB)
// Every wait on an mbarrier is bounded.  A thread whose wait expires records
// the failure and carries on without waiting (its results are garbage), so
// every arrival is still made; the CTA then records PKV_STATUS_INTERNAL,
// drains its copies, frees its TMEM and returns.
#include <math.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <string.h>

#include "common.cuh"
#include "prefill_common.cuh"
#include "tcgen05.cuh"

namespace {

using pkv::kBlock;
using pkv::PrefillParams;

constexpr int D = 128;
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kTeamThreads = 128;
constexpr int kMmaWarp = 8;  // warp 8: MMA issue (warp 9 only takes part in the TMEM allocation)
constexpr int kKLoadWarp = 10, kVLoadWarp = 11;
constexpr int kThreads = 12 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;  // S/P of team t at 128t, O of team t at kOCol + 128t
constexpr int kKStages = 3, kVStages = 3;

constexpr int kHalf = 128 * 128;             // 16 KB: 128 rows x 64 bf16
constexpr int kTile = 2 * kHalf;             // 32 KB: 128 rows x 128 bf16
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;                     // 32768
constexpr int kOffV = kOffK + kKStages * kTile;          // 131072
constexpr int kOffBar = kOffV + kVStages * kTile;        // 229376
// barriers: per team s, o (4); per team and half of P (4); K full/empty; V
// full/empty; go (2); item queue full/empty (4); MMA drain (1); Q buffer
// free (1)
constexpr int kNumBars = 8 + 2 * kKStages + 2 * kVStages + 2 + 4 + 1 + 1;
constexpr int kItemReaders = 1 + 1 + 8;  // item queue readers: V loader, MMA lane, softmax warps
constexpr int kOffSlots = (kOffBar + kNumBars * 8 + 15) & ~15;  // TMEM address (16 B), two item slots (int4)
static_assert(kOffSlots % 16 == 0, "item slots are 16-byte vectors");
constexpr int kOffRed = kOffSlots + 16 + 2 * 16;
constexpr int kSmemBytes = kOffRed + 2 * 2 * BM * 4;     // [team][m, l][row]
static_assert(kSmemBytes <= 232448, "more shared memory than a CTA may have");
constexpr unsigned kWaitIters = 1u << 24;

constexpr uint32_t kIdescS = pkv::tc::idesc_bf16_f32(BM, BN, false, false);
constexpr uint32_t kIdescPV = pkv::tc::idesc_bf16_f32(BM, D, false, true);

__device__ __forceinline__ int sw128(int r, int c16) {
    return (r >> 3) * 1024 + (r & 7) * 128 + ((c16 ^ (r & 7)) << 4);
}

// The next work item for this CTA: items below gridDim.x are each CTA's
// first; later ones are handed out in order by one fetch-and-add on a
// counter in the workspace, which the launch clears on the stream first.
__device__ __forceinline__ int next_item(const PrefillParams &p) {
    const unsigned long long k = atomicAdd(p.item_counter, 1ull);
    return k < (unsigned long long)p.num_items ? (int)gridDim.x + (int)k : 0x7fffffff;
}

// Item (sequence, q tile, kv head) as published in the shared-memory queue:
// (item, q0, n, L); every role derives the rest.
struct ItemInfo {
    int item, s, kvh, tile, q0, n, L, nkt, kv_end, mask_from;
    bool stop, skip, bad_len, bad_qlen;
};

__device__ __forceinline__ ItemInfo item_info(const PrefillParams &p, int4 v) {
    ItemInfo it;
    it.item = v.x;
    it.q0 = v.y;
    it.n = v.z;
    it.L = v.w;
    it.stop = v.x >= p.num_items;
    // later sequences first, later q tiles (more keys) first within a sequence
    const int per_seq = p.num_kv_heads * p.tiles_per_seq;
    const int zi = it.stop ? 0 : v.x / per_seq;
    const int rem = it.stop ? 0 : v.x - zi * per_seq;
    it.s = p.num_seqs - 1 - zi;
    it.tile = p.tiles_per_seq - 1 - rem / p.num_kv_heads;
    it.kvh = rem - (rem / p.num_kv_heads) * p.num_kv_heads;
    it.bad_len = !it.stop && (it.L < 0 || it.L > p.len_cap);
    it.bad_qlen = !it.stop && !it.bad_len && !p.prefix_len &&
                  (it.q0 < 0 || it.n < 0 || it.n > it.L || it.n > p.max_q_len || it.q0 + it.n > p.total_q);
    it.skip = it.stop || it.bad_len || it.bad_qlen || it.tile * BM >= it.n * p.group;
    if (it.skip) {
        it.nkt = it.kv_end = it.mask_from = 0;
    } else if (p.prefix_len) {  // every query sees the whole shared prefix, nothing after it
        it.kv_end = it.mask_from = p.prefix_len;
        it.nkt = (p.prefix_len + BN - 1) / BN;
    } else {
        const int prior = it.L - it.n;
        const int j_last = min(it.n - 1, (it.tile * BM + BM - 1) / p.group);
        it.kv_end = prior + j_last + 1;
        it.nkt = (it.kv_end + BN - 1) / BN;
        it.mask_from = prior + (it.tile * BM) / p.group + 1;  // keys below this need no causal mask
    }
    return it;
}

template <typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_q) {
    extern __shared__ __align__(1024) unsigned char smem[];
    // a dependent launch (the decode partitions beside the shared-prefix
    // mode) may start as soon as every CTA of this one has
    pkv::allow_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.group;
    const uint32_t sbase = pkv::smem_u32(smem);
    if (sbase & 1023u) {  // the swizzled layouts need 1024-byte alignment
        if (tid == 0) pkv::flag(p.status, PKV_STATUS_INTERNAL);
        return;
    }

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *bar_s = bars;           // [team] S(t) computed (and the team's PV(t-2) done)
    uint64_t *bar_o = bars + 2;       // [team] PV(t) done
    uint64_t *bar_pfull = bars + 4;   // [team][half] P(t) of keys 64h .. 64h+63 stored (128 arrivals)
    uint64_t *bar_kfull = bars + 8;   // [stage] K tile landed
    uint64_t *bar_kempty = bar_kfull + kKStages;   // [stage] the S reading it is done
    uint64_t *bar_vfull = bar_kempty + kKStages;   // [stage] V tile landed
    uint64_t *bar_vempty = bar_vfull + kVStages;   // [stage] the PV reading it is done
    uint64_t *bar_go = bar_vempty + kVStages;      // [k & 1] Q of the k-th item with work landed (256 arrivals)
    uint64_t *bar_item_full = bar_go + 2;          // [slot] item published
    uint64_t *bar_item_empty = bar_item_full + 2;  // [slot] every role has read it
    uint64_t *bar_done = bar_item_empty + 2;       // all MMAs finished
    uint64_t *bar_qfree = bar_done + 1;            // every S of the k-th item with work finished (2 arrivals)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffSlots);
    int4 *item_slots = reinterpret_cast<int4 *>(smem + kOffSlots + 16);
    float *red = reinterpret_cast<float *>(smem + kOffRed);  // [team][m, l][row]

    if (tid == 0) {
        for (int t = 0; t < 2; t++) {
            pkv::tc::mbar_init(bar_s + t, 1);
            pkv::tc::mbar_init(bar_o + t, 1);
            pkv::tc::mbar_init(bar_pfull + 2 * t, kTeamThreads);
            pkv::tc::mbar_init(bar_pfull + 2 * t + 1, kTeamThreads);
            pkv::tc::mbar_init(bar_item_full + t, 1);
            pkv::tc::mbar_init(bar_item_empty + t, kItemReaders);
        }
        pkv::tc::mbar_init(bar_done, 1);
        pkv::tc::mbar_init(bar_qfree, 2);
        for (int st = 0; st < kKStages; st++) {
            pkv::tc::mbar_init(bar_kfull + st, 1);
            pkv::tc::mbar_init(bar_kempty + st, 1);
        }
        for (int st = 0; st < kVStages; st++) {
            pkv::tc::mbar_init(bar_vfull + st, 1);
            pkv::tc::mbar_init(bar_vempty + st, 1);
        }
        // Q lands by TMA (one arrival with its bytes) or by the softmax threads' copies
        pkv::tc::mbar_init(bar_go, p.q_tma ? 1 : 2 * kTeamThreads);
        pkv::tc::mbar_init(bar_go + 1, p.q_tma ? 1 : 2 * kTeamThreads);
        pkv::tc::fence_mbar_init();
    }
    __syncthreads();  // barriers initialised: the loaders can start right away

    // TMEM for every warp but the loaders (which never touch it); they meet on
    // named barrier 5 so that the loaders need not wait for the allocation
    uint32_t tmem = 0;
    if (warp < kKLoadWarp) {
        if (warp == 0) {
            pkv::tc::tmem_alloc(tmem_slot, kTmemCols);
            pkv::tc::tmem_relinquish();
        }
        pkv::tc::fence_before_sync();
        asm volatile("bar.sync 5, %0;\n" ::"r"(kKLoadWarp * 32) : "memory");
        pkv::tc::fence_after_sync();
        tmem = *tmem_slot;
    }

    bool failed = false;
    auto wait = [&](uint64_t *bar, unsigned parity) {
        if (!failed && !pkv::tc::mbar_wait(bar, parity, kWaitIters)) failed = true;
    };
    // Take item i from the queue (every role reads every item): lane 0 waits,
    // the warp reads, lane 0 reports the slot read.
    auto take_item = [&](int i) {
        if (lane == 0) wait(bar_item_full + (i & 1), (unsigned)((i >> 1) & 1));
        __syncwarp();
        const int4 v = item_slots[i & 1];
        __syncwarp();
        if (lane == 0) pkv::tc::mbar_arrive(bar_item_empty + (i & 1));
        return item_info(p, v);
    };
    // Q of the k-th item with work: barrier k & 1, phase k >> 1
    auto wait_go = [&](int k) { wait(bar_go + (k & 1), (unsigned)((k >> 1) & 1)); };

    // Running counts that carry the barrier phases from one item to the next:
    // key tiles (K/V rings), tiles of each team (S, P, O barriers) and items
    // with work (the Q barrier).  Every role walks the same items, so every
    // role's counts agree.
    int kt_base = 0, team_base0 = 0, team_base1 = 0, go_count = 0;
    auto advance = [&](const ItemInfo &it) {
        kt_base += it.nkt;
        team_base0 += (it.nkt + 1) / 2;
        team_base1 += it.nkt / 2;
        go_count += it.skip ? 0 : 1;
    };

    if (warp == kKLoadWarp || warp == kVLoadWarp) {
        // ---------------- loaders; the K loader also runs the item queue
        const bool is_k = warp == kKLoadWarp;
        const int nst = is_k ? kKStages : kVStages;
        uint64_t *full = is_k ? bar_kfull : bar_vfull;
        uint64_t *empty = is_k ? bar_kempty : bar_vempty;
        const void *tmap = is_k ? static_cast<const void *>(&tmap_k) : static_cast<const void *>(&tmap_v);
        const unsigned char *cache = static_cast<const unsigned char *>(is_k ? p.k_cache : p.v_cache);
        const int box_rows = p.num_blocks * p.num_kv_heads * kBlock;  // rows of the 2-D view
        int item = blockIdx.x;  // the CTA's first item; later ones come from the counter
        for (int i = 0;; i++) {
            ItemInfo it;
            if (is_k) {
                int4 v = make_int4(item, 0, 0, 0);
                if (lane == 0) {
                    if (i >= 2) wait(bar_item_empty + (i & 1), (unsigned)(((i >> 1) - 1) & 1));
                    if (item < p.num_items && p.prefix_len) {
                        v.y = 0;                // the decode queries, one "position" per sequence
                        v.z = p.max_q_len;
                        v.w = p.prefix_len;
                    } else if (item < p.num_items) {
                        const int s = p.num_seqs - 1 - item / (p.num_kv_heads * p.tiles_per_seq);
                        v.y = p.cu_q_lens[s];
                        v.z = p.cu_q_lens[s + 1] - v.y;
                        v.w = p.context_lens[s];
                    }
                    item_slots[i & 1] = v;
                    pkv::tc::mbar_arrive(bar_item_full + (i & 1));  // release: the slot is visible to the waiters
                }
                v.x = __shfl_sync(0xffffffffu, v.x, 0);
                v.y = __shfl_sync(0xffffffffu, v.y, 0);
                v.z = __shfl_sync(0xffffffffu, v.z, 0);
                v.w = __shfl_sync(0xffffffffu, v.w, 0);
                it = item_info(p, v);
                if (lane == 0 && it.tile == 0 && it.kvh == 0) {
                    if (it.bad_len) pkv::flag(p.status, PKV_STATUS_BAD_LENGTH);
                    if (it.bad_qlen) pkv::flag(p.status, PKV_STATUS_BAD_QLEN);
                }
            } else {
                it = take_item(i);
            }
            if (it.stop) break;
            if (is_k && p.q_tma && !it.skip) {
                // This item's q tile, as soon as the previous one's S MMAs are
                // done with the buffer: it lands while that item finishes.  Row
                // r = j * G + h of the tile is query q0 + tile*128/G + j, head
                // kvh*G + h: one 3-D box {64 columns, G heads, 128/G queries}
                // per half.  Rows past the chunk read other queries or zeros
                // and are masked.
                if (go_count > 0) wait(bar_qfree, (unsigned)((go_count - 1) & 1));
                if (lane == 0) {
                    uint64_t *go = bar_go + (go_count & 1);
                    pkv::tc::mbar_arrive_expect_tx(go, kTile);
                    const int z = it.q0 + it.tile * (BM / G);
#pragma unroll
                    for (int h = 0; h < 2; h++)
                        pkv::tc::tma_load_3d(smem + kOffQ + h * kHalf, &tmap_q, h * 64, it.kvh * G, z, go);
                }
            }
            const int32_t *table = p.block_tables + (size_t)(it.skip ? 0 : it.s) * p.max_blocks;
            for (int t = 0; t < it.nkt; t++) {
                const int g = kt_base + t;  // ring position across items
                const int st = g % nst;
                if (g >= nst) wait(empty + st, (unsigned)((g / nst - 1) & 1));
                unsigned char *dst = smem + (is_k ? kOffK : kOffV) + st * kTile;
                // Keys [t*128, t*128 + 128) sit in 8 blocks, each loaded with two
                // 16-row x 64-column TMA boxes.  Blocks past the keys are not
                // loaded: K rows there are masked out of S whatever they hold, V
                // rows are zeroed in place (P = 0 times a NaN would poison O).
                // A V block that the keys end inside is copied with zero fill.
                const int tile_keys = min(BN, it.kv_end - t * BN);
                const int nbk = (tile_keys + kBlock - 1) / kBlock;
                const int cpq = (!is_k && (tile_keys % kBlock)) ? tile_keys / kBlock : -1;
                const int ntma = cpq >= 0 ? nbk - 1 : nbk;  // blocks 0 .. ntma-1 by TMA
                int my_id = 0;
                if (lane < nbk) my_id = table[t * 8 + lane];
                int y = box_rows;
                if (lane < ntma) {
                    if (my_id >= 0 && my_id < p.num_blocks)
                        y = (my_id * p.num_kv_heads + it.kvh) * kBlock;
                    else
                        pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                }
                int ys[8];
#pragma unroll
                for (int q = 0; q < 8; q++) ys[q] = __shfl_sync(0xffffffffu, y, q);
                const bool extra = cpq >= 0 || (!is_k && nbk < 8);
                if (extra) {
                    // generic-proxy part of the V tile: the partial block's live
                    // rows by zero-filling copies, every other row past the keys
                    // zeroed with stores
                    const int phys = cpq >= 0 ? __shfl_sync(0xffffffffu, my_id, cpq) : 0;
                    const bool ok = phys >= 0 && phys < p.num_blocks;
                    if (cpq >= 0 && !ok && lane == 0) pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                    for (int e = lane + 256 * ntma; e < 16 * 128; e += 32) {
                        const int r = e >> 4, c = e & 15;
                        unsigned char *d = dst + (c >> 3) * kHalf + sw128(r, c & 7);
                        if (r < tile_keys) {
                            const int rb = r % kBlock;
                            const size_t go = ok ? ((((size_t)phys * p.num_kv_heads + it.kvh) * kBlock + rb) * D) * 2 + c * 16 : 0;
                            pkv::cp_async16(d, cache + go, ok ? 16 : 0);
                        } else {
                            *reinterpret_cast<uint4 *>(d) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    pkv::cp_async_commit();
                    pkv::cp_async_wait<0>();
                    pkv::tc::fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    pkv::tc::mbar_arrive_expect_tx(full + st, (uint32_t)(ntma * 2 * 2048));
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        if (q >= ntma) break;
#pragma unroll
                        for (int h = 0; h < 2; h++)
                            pkv::tc::tma_load_2d(dst + h * kHalf + q * 2048, tmap, h * 64, ys[q], full + st);
                    }
                }
            }
            advance(it);
            if (is_k) {  // the next item, fetched while the consumers work on this one
                if (lane == 0) item = next_item(p);
                item = __shfl_sync(0xffffffffu, item, 0);
            }
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // ---------------- MMA issue: lane 0 of warp 8 issues every tile of both
        // teams; warp 9 has no role after the TMEM allocation
        if (warp == kMmaWarp && lane == 0) {
            int nkt_cur = 0;  // key tiles of the item being issued
            auto issue_s = [&](int t) {  // S(t) = Q K(t)^T into the S/P buffer of team t & 1 (K(t) landed)
                const uint32_t qa = sbase + kOffQ;
                const uint32_t kb = sbase + kOffK + ((kt_base + t) % kKStages) * kTile;
#pragma unroll
                for (int ks = 0; ks < D / 16; ks++) {
                    const uint64_t a = pkv::tc::smem_desc_sw128(qa + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024);
                    const uint64_t b = pkv::tc::smem_desc_sw128(kb + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024);
                    pkv::tc::mma_ss(tmem + (t & 1) * BN, a, b, kIdescS, ks > 0 ? 1u : 0u);
                }
                pkv::tc::mma_commit(bar_kempty + ((kt_base + t) % kKStages));
                pkv::tc::mma_commit(bar_s + (t & 1));
                // the item's last two S are the last reads of Q: the Q barrier
                // expects two arrivals per item
                if (t + 2 >= nkt_cur) pkv::tc::mma_commit(bar_qfree);
            };
            // O(team t & 1) (+)= P(t) V(t) over keys 64h .. 64h+63 (V(t) landed,
            // that half of P(t) stored)
            auto issue_pv_half = [&](int t, int h) {
                const uint32_t vb = sbase + kOffV + ((kt_base + t) % kVStages) * kTile;
#pragma unroll
                for (int kq = 4 * h; kq < 4 * h + 4; kq++) {  // 16 keys = 8 TMEM columns of P
                    // V is MN-major: next 64-column half at +16 KB (LBO), next 8 keys at +1 KB (SBO)
                    const uint64_t b = pkv::tc::smem_desc_sw128(vb + kq * 2048, kHalf, 1024);
                    pkv::tc::mma_ts(tmem + kOCol + (t & 1) * D, tmem + (t & 1) * BN + kq * 8, b, kIdescPV,
                                    (t < 2 && kq == 0) ? 0u : 1u);
                }
                if (h == 1) {
                    pkv::tc::mma_commit(bar_vempty + ((kt_base + t) % kVStages));
                    pkv::tc::mma_commit(bar_o + (t & 1));
                }
            };
            auto wait_k = [&](int t) {
                const int g = kt_base + t;
                wait(bar_kfull + g % kKStages, (unsigned)((g / kKStages) & 1));
            };
            auto wait_v = [&](int t) {
                const int g = kt_base + t;
                wait(bar_vfull + g % kVStages, (unsigned)((g / kVStages) & 1));
            };
            for (int i = 0;; i++) {
                // Take item i alone (the other lanes idle).  The slot is
                // reported read only after this item's Q barrier has been
                // waited for: the queue then cannot run two items ahead of
                // this lane, so neither Q barrier can complete a phase that
                // this lane has not yet waited for.
                wait(bar_item_full + (i & 1), (unsigned)((i >> 1) & 1));
                const ItemInfo it = item_info(p, item_slots[i & 1]);
                if (!it.stop && !it.skip) wait_go(go_count);
                pkv::tc::mbar_arrive(bar_item_empty + (i & 1));
                if (it.stop) break;
                if (!it.skip) {
                    const int nkt = it.nkt;
                    nkt_cur = nkt;
                    if (nkt == 1) pkv::tc::mbar_arrive(bar_qfree);  // one S reads this Q
                    for (int t = 0; t < nkt && t < 2; t++) {
                        wait_k(t);
                        pkv::tc::fence_after_sync();
                        issue_s(t);
                    }
                    // One issuing thread, tiles in order: the tensor pipe runs PV(t),
                    // S(t+2), PV(t+1), S(t+3), ...  Each team's next S is queued right
                    // behind its own PV, a whole unit before the other team's, which
                    // keeps the two teams' softmax phases apart.  PV(t) goes half by
                    // half as P(t) is stored (the first half runs while the team
                    // computes the second); S(t+2) follows once K(t+2) has landed.
                    for (int t = 0; t < nkt; t++) {
                        const int tb = (t & 1) ? team_base1 : team_base0;  // the team's tiles before this item
                        wait_v(t);
                        for (int h = 0; h < 2; h++) {
                            wait(bar_pfull + 2 * (t & 1) + h, (unsigned)((tb + (t >> 1)) & 1));
                            pkv::tc::fence_after_sync();
                            issue_pv_half(t, h);
                        }
                        if (t + 2 < nkt) {
                            wait_k(t + 2);
                            pkv::tc::fence_after_sync();
                            issue_s(t + 2);
                        }
                    }
                }
                advance(it);
            }
            // every MMA has finished before TMEM is released
            pkv::tc::mma_commit(bar_done);
            if (!pkv::tc::mbar_wait(bar_done, 0, kWaitIters)) failed = true;
        }
        __syncwarp();
    } else {
        // ---------------- softmax teams
        const int team = warp >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_col = (uint32_t)team * BN, o_col = kOCol + (uint32_t)team * D;
        const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
        for (int i = 0;; i++) {
            const ItemInfo it = take_item(i);
            if (it.stop) break;
            if (it.skip) {
                advance(it);
                continue;
            }
            const int nkt = it.nkt;
            // Without TMA, the Q tile: 128 rows x 16 chunks, 8 copies per
            // softmax thread.  The previous item's S MMAs are all complete:
            // this thread has been through that item's epilogue, which
            // follows both teams' last PV.
#pragma unroll
            for (int u = 0; u < 8 && !p.q_tma; u++) {
                const int e = tid + 2 * kTeamThreads * u;
                const int r = e >> 4, c = e & 15;
                const int R = it.tile * BM + r;
                const int jr = R / G;
                const bool ok = jr < it.n;
                const __nv_bfloat16 *src =
                    ok ? qg + ((size_t)(it.q0 + jr) * p.num_q_heads + it.kvh * G + (R - jr * G)) * D + c * 8 : qg;
                pkv::cp_async16(smem + kOffQ + (c >> 3) * kHalf + sw128(r, c & 7), src, ok ? 16 : 0);
            }
            if (!p.q_tma) {
                pkv::cp_async_commit();
                pkv::cp_async_wait<0>();
                pkv::tc::fence_proxy_async_smem();
                pkv::tc::mbar_arrive(bar_go + (go_count & 1));
            }

            const int R = it.tile * BM + row;
            const int jrow = R / G;
            const bool row_ok = jrow < it.n;
            // last visible key: causal within the chunk, or the whole shared prefix
            const int pos = !row_ok ? -1 : p.prefix_len ? p.prefix_len - 1 : it.L - it.n + jrow;
            float m_used = -INFINITY, lsum = 0.f;
            const int tb = team ? team_base1 : team_base0;  // this team's tiles before this item

            for (int t = team; t < nkt; t += 2) {
                // S(t) done; the team's PV(t-2), issued before it, is done too
                wait(bar_s + team, (unsigned)((tb + (t >> 1)) & 1));
                pkv::tc::fence_after_sync();
                const bool full_tile = t * BN + BN <= it.mask_from;
                const int lim0 = pos - t * BN;  // keys i <= lim0 of this tile are visible
                // The row's scores are read from TMEM twice, 64 at a time (for the
                // maximum, then for the powers), so that only 64 stay live and the
                // rest of the register file is free to overlap the exponentials.
                // Unmasked, the first read's own reduction gives the maximum.
                const bool masked = !full_tile || !row_ok;
                float mraw = -INFINITY;
    #pragma unroll
                for (int h = 0; h < 2; h++) {
                    float sv[64], hmax;
                    pkv::tc::tmem_ld64_max(t_lane + s_col + h * 64, sv, hmax);
                    if (masked) {
    #pragma unroll
                        for (int i = 0; i < 64; i++) sv[i] = h * 64 + i <= lim0 ? sv[i] : -INFINITY;
                        float mx[16];
    #pragma unroll
                        for (int i = 0; i < 16; i++)
                            mx[i] = fmaxf(fmaxf(sv[i], sv[i + 16]), fmaxf(sv[i + 32], sv[i + 48]));
    #pragma unroll
                        for (int i = 0; i < 8; i++) mx[i] = fmaxf(mx[i], mx[i + 8]);
    #pragma unroll
                        for (int i = 0; i < 4; i++) mx[i] = fmaxf(mx[i], mx[i + 4]);
                        hmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                    }
                    mraw = fmaxf(mraw, hmax);
                }
                if (!row_ok) mraw = -INFINITY;
                const float mt = mraw * p.scale_log2;  // scale > 0 commutes with max; -inf stays
                const bool need = mt > m_used + 8.f;
                float alpha = 1.f;
                if (need) {
                    alpha = pkv::tc::ex2(m_used - mt);  // 0 when nothing was seen yet
                    lsum *= alpha;
                    m_used = mt;
                }
                if (t >= 2 && __any_sync(0xffffffffu, need)) {
    #pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        float o[32];
                        pkv::tc::tmem_ld32(t_lane + o_col + c, o);
    #pragma unroll
                        for (int i = 0; i < 32; i++) o[i] *= alpha;
                        pkv::tc::tmem_st32(t_lane + o_col + c, o);
                    }
                }
                // P = 2^(s * scale - m) as bf16 pairs over the first 64 columns;
                // the scaling and the row sum run on paired fp32 instructions
                const float nbase = m_used == -INFINITY ? 0.f : -m_used;
                const uint64_t sc2 = pkv::tc::f2(p.scale_log2, p.scale_log2), nb2 = pkv::tc::f2(nbase, nbase);
                uint64_t acc2[2] = {pkv::tc::f2(0.f, 0.f), pkv::tc::f2(0.f, 0.f)};
    #pragma unroll
                for (int c = 0; c < BN; c += 64) {
                    float sv[64];
                    pkv::tc::tmem_ld64(t_lane + s_col + c, sv);
                    if (masked) {
    #pragma unroll
                        for (int i = 0; i < 64; i++) sv[i] = c + i <= lim0 ? sv[i] : -INFINITY;
                    }
                    float pk[32];
    #pragma unroll
                    for (int i = 0; i < 32; i++) {
                        float x0, x1;
                        pkv::tc::unf2(pkv::tc::ffma2(pkv::tc::f2(sv[2 * i], sv[2 * i + 1]), sc2, nb2), x0, x1);
                        // all on the special-function unit: the fewest instructions
                        // leave the most issue slots to the MMA-issuing thread
                        const float e0 = pkv::tc::ex2(x0), e1 = pkv::tc::ex2(x1);
                        acc2[i & 1] = pkv::tc::fadd2(acc2[i & 1], pkv::tc::f2(e0, e1));
                        pk[i] = __uint_as_float(pkv::pack_bf16(e0, e1));
                    }
                    // keys c .. c+63 -> P columns c/2 .. c/2+31, handed to the MMA lane
                    pkv::tc::tmem_st32(t_lane + s_col + c / 2, pk);
                    pkv::tc::fence_before_sync();
                    pkv::tc::mbar_arrive(bar_pfull + 2 * team + c / 64);
                }
                {
                    float a0, a1, b0, b1;
                    pkv::tc::unf2(acc2[0], a0, a1);
                    pkv::tc::unf2(acc2[1], b0, b1);
                    lsum += (a0 + a1) + (b0 + b1);
                }
            }

            // merge the two teams: exchange (m, l) with the partner thread of the same row
            const int my_tiles = nkt > team ? (nkt - team + 1) / 2 : 0;
            if (my_tiles > 0) {
                wait(bar_o + team, (unsigned)((tb + my_tiles - 1) & 1));
                pkv::tc::fence_after_sync();
            }
            red[(team * 2 + 0) * BM + row] = m_used;
            red[(team * 2 + 1) * BM + row] = lsum;
            // The fences order this thread's later reads of both teams' O
            // after the completion its partner observed; without them the
            // first tcgen05.ld waited microseconds.
            pkv::tc::fence_before_sync();
            asm volatile("bar.sync %0, 64;\n" ::"r"(1 + quarter) : "memory");
            pkv::tc::fence_after_sync();
            const float m0 = red[0 * BM + row], l0 = red[1 * BM + row];
            const float m1 = red[2 * BM + row], l1 = red[3 * BM + row];
            const float M = fmaxf(m0, m1);
            const float f0 = M == -INFINITY ? 0.f : pkv::tc::ex2(m0 - M);
            const float f1 = (M == -INFINITY || nkt < 2) ? 0.f : pkv::tc::ex2(m1 - M);
            const float ltot = l0 * f0 + l1 * f1;
            const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
            const float g0 = f0 * inv, g1 = f1 * inv;
            // Output: each thread writes its half row (team 0 columns 0..63,
            // team 1 columns 64..127) straight from registers, 16 bytes at a
            // time; shared memory stays free for the next item's tiles.
            OutT *orow = static_cast<OutT *>(p.out) +
                         ((size_t)(it.q0 + (row_ok ? jrow : 0)) * p.num_q_heads + it.kvh * G + (R - jrow * G)) * D;
#pragma unroll 1
            for (int c = 0; c < D / 2; c += 32) {
                float a[32], b[32];
                const uint32_t col = (uint32_t)(team * (D / 2) + c);
                pkv::tc::tmem_ld32(t_lane + kOCol + col, a);
                if (nkt >= 2) {
                    pkv::tc::tmem_ld32(t_lane + kOCol + D + col, b);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e++) b[e] = 0.f;
                }
                if (row_ok && !failed && p.prefix_len) {
                    // shared-prefix mode: the unnormalised state (M, L, O)
                    // goes to partial slot 0 of the decode row (s = jrow)
                    const size_t prow = ((size_t)jrow * p.num_q_heads + it.kvh * G + (R - jrow * G)) * p.part_stride;
                    float4 *po = reinterpret_cast<float4 *>(p.part_o + prow * D + col);
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        po[k] = make_float4(a[4 * k] * f0 + b[4 * k] * f1, a[4 * k + 1] * f0 + b[4 * k + 1] * f1,
                                            a[4 * k + 2] * f0 + b[4 * k + 2] * f1, a[4 * k + 3] * f0 + b[4 * k + 3] * f1);
                    if (team == 0 && c == 0) *reinterpret_cast<float2 *>(p.part_ml + prow * 2) = make_float2(M, ltot);
                } else if (row_ok && !failed) {
                    alignas(16) OutT v[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) pkv::store2(v + e, a[e] * g0 + b[e] * g1, a[e + 1] * g0 + b[e + 1] * g1);
                    if (p.out_v8) {
                        // 32 bytes per store: each fills whole sectors of the row
                        constexpr int kVec = 32 * (int)sizeof(OutT) / 32;
#pragma unroll
                        for (int k = 0; k < kVec; k++)
                            pkv::tc::st_global_32B(orow + col + k * (32 / (int)sizeof(OutT)),
                                                   reinterpret_cast<const uint4 *>(v) + 2 * k);
                    } else {
                        constexpr int kVec = 32 * (int)sizeof(OutT) / 16;
#pragma unroll
                        for (int k = 0; k < kVec; k++)
                            reinterpret_cast<uint4 *>(orow + col)[k] = reinterpret_cast<const uint4 *>(v)[k];
                    }
                }
            }
            // the O reads are done before the next item's first PV may overwrite
            pkv::tc::fence_before_sync();
            advance(it);
        }
    }

    pkv::cp_async_wait<0>();
    pkv::tc::fence_before_sync();
    if (__syncthreads_or(failed) && tid == 0) pkv::flag(p.status, PKV_STATUS_INTERNAL);
    if (warp == 0) {
        pkv::tc::fence_after_sync();
        pkv::tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

namespace pkv {

bool prefill_tc_supported(int dtype, int head_dim) { return dtype == PKV_BF16 && head_dim == D; }

}  // namespace pkv

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// 2-D view of one cache: [num_blocks * num_kv_heads * 16 rows][128 columns]
// bf16, boxes of 16 rows x 64 columns, 128-byte swizzle, zero fill.
int make_cache_map(CUtensorMap *map, const void *cache, int num_blocks, int num_kv_heads) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    if (!g_encode) return pkv::fail(PKV_ERR_CUDA, "prefill: cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)num_blocks * num_kv_heads * kBlock};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBlock};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(cache), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return pkv::fail(PKV_ERR_CUDA, "prefill: cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

// 3-D view of the queries [total_q][Hq][128] bf16: boxes of {64 columns, G
// heads, 128/G queries}, the 128 packed rows of one q tile, 128-byte swizzle.
int make_q_map(CUtensorMap *map, const void *q, int num_q_heads, int total_q, int group) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)num_q_heads * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(BM / group)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return pkv::fail(PKV_ERR_CUDA, "prefill: cuTensorMapEncodeTiled (q) failed (%d)", (int)r);
    return PKV_OK;
}

}  // namespace

namespace pkv {

int launch_prefill_tc(const PrefillParams &p, int num_seqs, int out_dtype, cudaStream_t st) {
    if ((long long)p.num_blocks * p.num_kv_heads * kBlock > 0x7fffffffLL)
        return fail(PKV_ERR_INVALID, "prefill: cache too large for 32-bit row coordinates");
    CUtensorMap tk, tv;
    int rc = make_cache_map(&tk, p.k_cache, p.num_blocks, p.num_kv_heads);
    if (rc) return rc;
    rc = make_cache_map(&tv, p.v_cache, p.num_blocks, p.num_kv_heads);
    if (rc) return rc;
    // q tiles by TMA when a tile is whole queries (G divides 128)
    CUtensorMap tq;
    memset(&tq, 0, sizeof(tq));
    const bool q_tma = p.group <= BM && BM % p.group == 0 && p.total_q > 0;
    if (q_tma) {
        rc = make_q_map(&tq, p.q, p.num_q_heads, p.total_q, p.group);
        if (rc) return rc;
    }
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const int which = out_dtype == PKV_F32 ? 0 : 1;
    if (dev >= 0 && dev < 64 && !attr_set[which][dev]) {
        cudaError_t e = which == 0
                            ? cudaFuncSetAttribute(prefill_tc_kernel<float>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)
                            : cudaFuncSetAttribute(prefill_tc_kernel<__nv_bfloat16>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return check_launch("prefill_tc: set shared memory size");
        attr_set[which][dev] = true;
    }
    PrefillParams pp = p;
    pp.q_tma = q_tma ? 1 : 0;
    pp.out_v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0 ? 1 : 0;
    pp.num_seqs = num_seqs;
    pp.tiles_per_seq = (p.max_q_len * p.group + BM - 1) / BM;
    const long long items = (long long)num_seqs * p.num_kv_heads * pp.tiles_per_seq;
    if (items > 0x7fff0000LL) return fail(PKV_ERR_INVALID, "prefill: too many q tiles");
    pp.num_items = (int)items;
    cudaError_t me = cudaMemsetAsync(pp.item_counter, 0, sizeof(unsigned long long), st);
    if (me != cudaSuccess) return fail(PKV_ERR_CUDA, "prefill: clear item counter: %s", cudaGetErrorString(me));
    static int sms[64] = {0};
    int nsm = 148;
    if (dev >= 0 && dev < 64) {
        if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (sms[dev] > 0) nsm = sms[dev];
    }
    // one persistent CTA per SM (its shared memory allows no second)
    const unsigned grid = (unsigned)(pp.num_items < nsm ? pp.num_items : nsm);
    if (which == 0)
        prefill_tc_kernel<float><<<grid, kThreads, kSmemBytes, st>>>(pp, tk, tv, tq);
    else
        prefill_tc_kernel<__nv_bfloat16><<<grid, kThreads, kSmemBytes, st>>>(pp, tk, tv, tq);
    return check_launch("prefill_tc");
}

}  // namespace pkv
