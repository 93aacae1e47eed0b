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
// Warp roles (one CTA per SM, 11 warps):
//   * two softmax teams of 4 warps: team 0 takes key tiles 0, 2, 4, ..., team 1
//     tiles 1, 3, 5, ...  Thread r of a team owns query row r (TMEM lane r).
//     It reads its 128 scores with one tcgen05.ld, masks them, finds the row
//     maximum, computes p = 2^(s * scale * log2 e - m) (one multiply-add per
//     element; a quarter of the powers on the FMA pipe with a polynomial, the
//     rest with ex2.approx on the special-function unit) and stores P as bf16
//     pairs over the first 64 columns of the same S buffer.  Each team has its own S/P buffer, O accumulator and
//     running (m, l); the two partial results are merged by log-sum-exp at
//     the end.  The teams run independently, so one team's softmax overlaps
//     the other team's MMAs.
//   * one MMA warp whose first lane issues, per tile t, PV(t) as soon as P(t)
//     is stored and then S(t+2) into the same team's buffer.  tcgen05.mma
//     operations issued by one thread execute in order, so S(t+2) cannot
//     overwrite P(t) before PV(t) has read it, and a team that sees S(t)
//     complete also knows its previous PV is done.
//   * two loader warps, one for K and one for V, that gather tiles through
//     the block table: a tile of whole blocks with 2-D TMA boxes (one
//     16-row x 64-column box per block and half; the cache is viewed as
//     [num_blocks * num_kv_heads * 16 rows][128] with 128-byte swizzle, which
//     writes exactly the layout the MMAs read); the last tile, which may end
//     inside a block, with zero-filling 16-byte cp.async instead, because rows
//     past the context may hold anything (even NaN) and P = 0 times NaN would
//     still poison O.  K uses a 2-stage ring refilled when the S that read a
//     stage has finished, V a 3-stage ring refilled when the PV has (K(t) is
//     needed two tiles before V(t), so both get about the same lead).
// The running max of a row is only moved when a tile maximum exceeds it by
// more than 8 (log2 units), so P <= 256 and O is rarely rescaled; numerator
// and denominator share the same reference, so the result is exact.
//
// TMEM columns (all 512): S/P of team t at 128t, O of team t at 256 + 128t.
// Shared memory, all in the 128-byte-swizzled canonical layout (8-row atoms
// of 8 x 128 bytes, 16-byte chunk c of row r at chunk c ^ (r % 8)):
//   Q : two 64-column halves of 128 rows                       (32 KB)
//   K : two stages x two 64-column halves of 128 rows          (64 KB)
//   V : three stages x two 64-column halves of 128 rows        (96 KB)
// Every wait on an mbarrier is bounded.  A thread whose wait expires records
// the failure and carries on without waiting (its results are garbage), so
// every arrival is still made; the CTA then records PKV_STATUS_INTERNAL,
// drains its copies, frees its TMEM and returns.
#include <math.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

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
constexpr int kMmaWarp = 8, kKLoadWarp = 9, kVLoadWarp = 10;
constexpr int kThreads = 11 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;  // S/P of team t at 128t, O of team t at kOCol + 128t
constexpr int kKStages = 2, kVStages = 3;

constexpr int kHalf = 128 * 128;             // 16 KB: 128 rows x 64 bf16
constexpr int kTile = 2 * kHalf;             // 32 KB: 128 rows x 128 bf16
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;                     // 32768
constexpr int kOffV = kOffK + kKStages * kTile;          // 98304
constexpr int kOffBar = kOffV + kVStages * kTile;        // 196608
// barriers: per team s, o, pfull (6); K full/empty (6); V full/empty (4); go (1)
constexpr int kNumBars = 6 + 2 * kKStages + 2 * kVStages + 1;
constexpr int kOffRed = kOffBar + kNumBars * 8 + 8;      // + TMEM address slot
constexpr int kSmemBytes = kOffRed + 2 * 2 * BM * 4;     // [team][m, l][row]
constexpr unsigned kWaitIters = 1u << 24;

constexpr uint32_t kIdescS = pkv::tc::idesc_bf16_f32(BM, BN, false, false);
constexpr uint32_t kIdescPV = pkv::tc::idesc_bf16_f32(BM, D, false, true);

__device__ __forceinline__ int sw128(int r, int c16) {
    return (r >> 3) * 1024 + (r & 7) * 128 + ((c16 ^ (r & 7)) << 4);
}

template <typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, kvh = blockIdx.y;
    const int s = gridDim.z - 1 - blockIdx.z;  // later (typically longer) sequences first
    const int G = p.group;

    const int q0 = p.cu_q_lens[s];
    const int n = p.cu_q_lens[s + 1] - q0;
    const int L = p.context_lens[s];
    if (L < 0 || L > p.len_cap) {
        if (tile == 0 && kvh == 0 && tid == 0) pkv::flag(p.status, PKV_STATUS_BAD_LENGTH);
        return;
    }
    if (q0 < 0 || n < 0 || n > L || n > p.max_q_len || q0 + n > p.total_q) {
        if (tile == 0 && kvh == 0 && tid == 0) pkv::flag(p.status, PKV_STATUS_BAD_QLEN);
        return;
    }
    if (tile * BM >= n * G) return;
    const uint32_t sbase = pkv::smem_u32(smem);
    if (sbase & 1023u) {  // the swizzled layouts need 1024-byte alignment
        if (tid == 0) pkv::flag(p.status, PKV_STATUS_INTERNAL);
        return;
    }
    const int prior = L - n;
    const int j_last = min(n - 1, (tile * BM + BM - 1) / G);
    const int kv_end = prior + j_last + 1;
    const int nkt = (kv_end + BN - 1) / BN;
    const int j_first = (tile * BM) / G;
    const int mask_from = prior + j_first + 1;  // keys below this need no causal mask

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *bar_s = bars;           // [team] S(t) computed (and the team's PV(t-2) done)
    uint64_t *bar_o = bars + 2;       // [team] PV(t) done
    uint64_t *bar_pfull = bars + 4;   // [team] P(t) stored (128 arrivals)
    uint64_t *bar_kfull = bars + 6;   // [stage] K tile landed
    uint64_t *bar_kempty = bar_kfull + kKStages;   // [stage] the S reading it is done
    uint64_t *bar_vfull = bar_kempty + kKStages;   // [stage] V tile landed
    uint64_t *bar_vempty = bar_vfull + kVStages;   // [stage] the PV reading it is done
    uint64_t *bar_go = bar_vempty + kVStages;      // Q landed (256 arrivals)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    float *red = reinterpret_cast<float *>(smem + kOffRed);  // [team][m, l][row]

    if (tid == 0) {
        for (int t = 0; t < 2; t++) {
            pkv::tc::mbar_init(bar_s + t, 1);
            pkv::tc::mbar_init(bar_o + t, 1);
            pkv::tc::mbar_init(bar_pfull + t, kTeamThreads);
        }
        for (int st = 0; st < kKStages; st++) {
            pkv::tc::mbar_init(bar_kfull + st, 1);
            pkv::tc::mbar_init(bar_kempty + st, 1);
        }
        for (int st = 0; st < kVStages; st++) {
            pkv::tc::mbar_init(bar_vfull + st, 1);
            pkv::tc::mbar_init(bar_vempty + st, 1);
        }
        pkv::tc::mbar_init(bar_go, 2 * kTeamThreads);
        pkv::tc::fence_mbar_init();
    }
    __syncthreads();  // barriers initialised: the loaders can start right away

    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
    const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;

    if (warp < 8) {
        // Q tile: 128 rows x 16 chunks, 8 copies per softmax thread
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int i = tid + 2 * kTeamThreads * u;
            const int r = i >> 4, c = i & 15;
            const int R = tile * BM + r;
            const int jr = R / G;
            const bool ok = jr < n;
            const __nv_bfloat16 *src =
                ok ? qg + ((size_t)(q0 + jr) * p.num_q_heads + kvh * G + (R - jr * G)) * D + c * 8 : qg;
            pkv::cp_async16(smem + kOffQ + (c >> 3) * kHalf + sw128(r, c & 7), src, ok ? 16 : 0);
        }
        pkv::cp_async_commit();
    }

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

    if (warp == kKLoadWarp || warp == kVLoadWarp) {
        // ---------------- loaders: K tile t -> K stage t % 3, V tile t -> V stage t % 2
        const bool is_k = warp == kKLoadWarp;
        const int nst = is_k ? kKStages : kVStages;
        uint64_t *full = is_k ? bar_kfull : bar_vfull;
        uint64_t *empty = is_k ? bar_kempty : bar_vempty;
        const void *tmap = is_k ? static_cast<const void *>(&tmap_k) : static_cast<const void *>(&tmap_v);
        const unsigned char *cache = static_cast<const unsigned char *>(is_k ? p.k_cache : p.v_cache);
        const int box_rows = p.num_blocks * p.num_kv_heads * kBlock;  // rows of the 2-D view
        for (int t = 0; t < nkt; t++) {
            const int st = t % nst;
            if (t >= nst) wait(empty + st, (unsigned)((t / nst - 1) & 1));
            unsigned char *dst = smem + (is_k ? kOffK : kOffV) + st * kTile;
            // physical ids of the 8 blocks holding keys [t*128, t*128 + 128)
            int my_id = 0;
            if (lane < 8 && t * BN + lane * kBlock < kv_end) my_id = table[t * 8 + lane];
            if ((t + 1) * BN <= kv_end) {
                // eight whole blocks: TMA
                int y = box_rows;  // out of range: the box reads as zeros
                if (lane < 8) {
                    if (my_id >= 0 && my_id < p.num_blocks)
                        y = (my_id * p.num_kv_heads + kvh) * kBlock;
                    else
                        pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                }
                int ys[8];
#pragma unroll
                for (int q = 0; q < 8; q++) ys[q] = __shfl_sync(0xffffffffu, y, q);
                if (lane == 0) {
                    pkv::tc::mbar_arrive_expect_tx(full + st, kTile);
#pragma unroll
                    for (int q = 0; q < 8; q++) {
#pragma unroll
                        for (int h = 0; h < 2; h++)
                            pkv::tc::tma_load_2d(dst + h * kHalf + q * 2048, tmap, h * 64, ys[q], full + st);
                    }
                }
            } else {
                // the last tile may end inside a block: zero-filling copies
#pragma unroll 4
                for (int u = 0; u < 64; u++) {
                    const int i = lane + 32 * u;
                    const int r = i >> 4, c = i & 15;  // r >> 4 == u >> 3
                    const int key = t * BN + r;
                    const int phys = __shfl_sync(0xffffffffu, my_id, u >> 3);
                    int nb = 0;
                    size_t go = 0;
                    if (key < kv_end) {
                        if (phys >= 0 && phys < p.num_blocks) {
                            nb = 16;
                            go = ((((size_t)phys * p.num_kv_heads + kvh) * kBlock + (key % kBlock)) * D) * 2 + c * 16;
                        } else if (c == 0 && (key % kBlock) == 0) {
                            pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                        }
                    }
                    pkv::cp_async16(dst + (c >> 3) * kHalf + sw128(r, c & 7), cache + go, nb);
                }
                pkv::cp_async_commit();
                pkv::cp_async_wait<0>();
                pkv::tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) pkv::tc::mbar_arrive(full + st);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (one lane)
        if (lane == 0) {
            auto issue_s = [&](int t) {  // S(t) = Q K(t)^T into the S/P buffer of team t & 1 (K(t) landed)
                const uint32_t qa = sbase + kOffQ;
                const uint32_t kb = sbase + kOffK + (t % kKStages) * kTile;
#pragma unroll
                for (int ks = 0; ks < D / 16; ks++) {
                    const uint64_t a = pkv::tc::smem_desc_sw128(qa + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024);
                    const uint64_t b = pkv::tc::smem_desc_sw128(kb + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024);
                    pkv::tc::mma_ss(tmem + (t & 1) * BN, a, b, kIdescS, ks > 0 ? 1u : 0u);
                }
                pkv::tc::mma_commit(bar_kempty + (t % kKStages));
                pkv::tc::mma_commit(bar_s + (t & 1));
            };
            auto issue_pv = [&](int t) {  // O(team t & 1) (+)= P(t) V(t) (V(t) landed, P(t) stored)
                const uint32_t vb = sbase + kOffV + (t % kVStages) * kTile;
#pragma unroll
                for (int kq = 0; kq < BN / 16; kq++) {  // 16 keys = 8 TMEM columns of P
                    // V is MN-major: next 64-column half at +16 KB (LBO), next 8 keys at +1 KB (SBO)
                    const uint64_t b = pkv::tc::smem_desc_sw128(vb + kq * 2048, kHalf, 1024);
                    pkv::tc::mma_ts(tmem + kOCol + (t & 1) * D, tmem + (t & 1) * BN + kq * 8, b, kIdescPV,
                                    (t < 2 && kq == 0) ? 0u : 1u);
                }
                pkv::tc::mma_commit(bar_vempty + (t % kVStages));
                pkv::tc::mma_commit(bar_o + (t & 1));
            };
            auto wait_k = [&](int t) { wait(bar_kfull + (t % kKStages), (unsigned)((t / kKStages) & 1)); };
            auto wait_v = [&](int t) { wait(bar_vfull + (t % kVStages), (unsigned)((t / kVStages) & 1)); };
            wait(bar_go, 0);
            wait_k(0);
            pkv::tc::fence_after_sync();
            issue_s(0);
            if (nkt > 1) {
                wait_k(1);
                pkv::tc::fence_after_sync();
                issue_s(1);
            }
            for (int t = 0; t < nkt; t++) {
                // operand tiles first, while the team is still computing P(t):
                // each wait costs some hundreds of cycles even when already satisfied
                wait_v(t);
                if (t + 2 < nkt) wait_k(t + 2);
                wait(bar_pfull + (t & 1), (unsigned)((t >> 1) & 1));  // P(t) stored
                pkv::tc::fence_after_sync();
                issue_pv(t);
                if (t + 2 < nkt) issue_s(t + 2);
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax teams
        const int team = warp >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_col = (uint32_t)team * BN, o_col = kOCol + (uint32_t)team * D;
        const int R = tile * BM + row;
        const int jrow = R / G;
        const bool row_ok = jrow < n;
        const int pos = row_ok ? prior + jrow : -1;
        float m_used = -INFINITY, lsum = 0.f;

        pkv::cp_async_wait<0>();  // this thread's Q copies
        pkv::tc::fence_proxy_async_smem();
        pkv::tc::mbar_arrive(bar_go);

        for (int t = team; t < nkt; t += 2) {
            // S(t) done; the team's PV(t-2), issued before it, is done too
            wait(bar_s + team, (unsigned)((t >> 1) & 1));
            pkv::tc::fence_after_sync();
            const bool full_tile = t * BN + BN <= mask_from;
            const int lim0 = pos - t * BN;  // keys i <= lim0 of this tile are visible

            // all 128 raw scores of this row, masked
            float sv[128];
            pkv::tc::tmem_ld128(t_lane + s_col, sv);
            if (!full_tile || !row_ok) {
#pragma unroll
                for (int i = 0; i < 128; i++) sv[i] = i <= lim0 ? sv[i] : -INFINITY;
            }
            float mx[16];
#pragma unroll
            for (int i = 0; i < 16; i++)
                mx[i] = fmaxf(fmaxf(fmaxf(sv[i], sv[i + 16]), fmaxf(sv[i + 32], sv[i + 48])),
                              fmaxf(fmaxf(sv[i + 64], sv[i + 80]), fmaxf(sv[i + 96], sv[i + 112])));
#pragma unroll
            for (int i = 0; i < 8; i++) mx[i] = fmaxf(mx[i], mx[i + 8]);
#pragma unroll
            for (int i = 0; i < 4; i++) mx[i] = fmaxf(mx[i], mx[i + 4]);
            float mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
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
            // P = 2^(s * scale - m) as bf16 pairs over the first 64 columns
            const float nbase = m_used == -INFINITY ? 0.f : -m_used;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < BN; c += 64) {
                float pk[32];
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    const float x0 = fmaf(sv[c + 2 * i], p.scale_log2, nbase);
                    const float x1 = fmaf(sv[c + 2 * i + 1], p.scale_log2, nbase);
                    // one pair in four on the FMA pipe, the rest on the special-function unit
                    const float e0 = (i & 3) == 3 ? pkv::tc::exp2_poly(x0) : pkv::tc::ex2(x0);
                    const float e1 = (i & 3) == 3 ? pkv::tc::exp2_poly(x1) : pkv::tc::ex2(x1);
                    ls[(2 * i) & 3] += e0;
                    ls[(2 * i + 1) & 3] += e1;
                    pk[i] = __uint_as_float(pkv::pack_bf16(e0, e1));
                }
                // keys c .. c+63 -> P columns c/2 .. c/2+31
                pkv::tc::tmem_st32(t_lane + s_col + c / 2, pk);
            }
            lsum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            pkv::tc::fence_before_sync();
            pkv::tc::mbar_arrive(bar_pfull + team);
        }

        // merge the two teams: exchange (m, l) with the partner thread of the same row
        const int my_tiles = nkt > team ? (nkt - team + 1) / 2 : 0;
        if (my_tiles > 0) {
            const int last = team + 2 * (my_tiles - 1);
            wait(bar_o + team, (unsigned)((last >> 1) & 1));
            pkv::tc::fence_after_sync();
        }
        red[(team * 2 + 0) * BM + row] = m_used;
        red[(team * 2 + 1) * BM + row] = lsum;
        asm volatile("bar.sync %0, 64;\n" ::"r"(1 + quarter) : "memory");
        const float m0 = red[0 * BM + row], l0 = red[1 * BM + row];
        const float m1 = red[2 * BM + row], l1 = red[3 * BM + row];
        const float M = fmaxf(m0, m1);
        const float f0 = M == -INFINITY ? 0.f : pkv::tc::ex2(m0 - M);
        const float f1 = (M == -INFINITY || nkt < 2) ? 0.f : pkv::tc::ex2(m1 - M);
        const float ltot = l0 * f0 + l1 * f1;
        const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
        const float g0 = f0 * inv, g1 = f1 * inv;
        // Output: each thread puts its half row (team 0 columns 0..63, team 1
        // columns 64..127) into shared memory, and the 256 softmax threads
        // then write whole rows with coalesced 16-byte stores.  The staging
        // area is the Q and K region: every S has completed by now (the last
        // one was issued before either team's last PV), whereas the other
        // team's last PV may still be reading V.
        constexpr int kRowBytes = D * (int)sizeof(OutT);
        constexpr int kStride = kRowBytes + 16;  // padded rows
        static_assert(BM * kStride <= kOffV, "output staging must not reach the V ring");
        unsigned char *stage = smem + kOffQ;
#pragma unroll 1
        for (int c = 0; c < D / 2; c += 32) {
            float a[32], b[32];
            const uint32_t col = (uint32_t)(team * (D / 2) + c);
            pkv::tc::tmem_ld32(t_lane + kOCol + col, a);
            if (nkt >= 2) {
                pkv::tc::tmem_ld32(t_lane + kOCol + D + col, b);
            } else {
#pragma unroll
                for (int i = 0; i < 32; i++) b[i] = 0.f;
            }
            OutT *srow = reinterpret_cast<OutT *>(stage + row * kStride) + col;
#pragma unroll
            for (int i = 0; i < 32; i += 2) pkv::store2(srow + i, a[i] * g0 + b[i] * g1, a[i + 1] * g0 + b[i + 1] * g1);
        }
        asm volatile("bar.sync 6, %0;\n" ::"r"(2 * kTeamThreads) : "memory");
        constexpr int kChunks = kRowBytes / 16;  // 16-byte chunks per row
        for (int i = tid; i < BM * kChunks; i += 2 * kTeamThreads) {
            const int r = i / kChunks, ch = i - r * kChunks;
            const int Rr = tile * BM + r;
            const int jr = Rr / G;
            if (jr < n && !failed) {
                unsigned char *dst = reinterpret_cast<unsigned char *>(static_cast<OutT *>(p.out)) +
                                     ((size_t)(q0 + jr) * p.num_q_heads + kvh * G + (Rr - jr * G)) * kRowBytes +
                                     ch * 16;
                *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(stage + r * kStride + ch * 16);
            }
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
    const int tiles = (p.max_q_len * p.group + BM - 1) / BM;
    dim3 grid((unsigned)tiles, (unsigned)p.num_kv_heads, (unsigned)num_seqs);
    if (which == 0)
        prefill_tc_kernel<float><<<grid, kThreads, kSmemBytes, st>>>(p, tk, tv);
    else
        prefill_tc_kernel<__nv_bfloat16><<<grid, kThreads, kSmemBytes, st>>>(p, tk, tv);
    return check_launch("prefill_tc");
}

}  // namespace pkv
