// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Same operation as the mma.sync kernel in prefill.cu: query j of a chunk of n
// tokens of a sequence with L cached tokens attends causally to tokens
// 0 .. L-n+j (caffein.top, "Chunked Prefill"), K/V gathered through the block
// table.  Used for bf16 caches with head_dim 128.
//
// Work unit: one CTA of 9 warps per (tile of 128 packed query rows, kv head,
// sequence): 8 softmax warps and one warp whose first lane issues the MMAs.  Row r of the tile is query position R / G, head kvh*G + R % G
// (R = tile*128 + r), so the G heads of a kv head share every K/V tile.
//   S  = Q K^T   : tcgen05.mma M=128, N=64 keys, K=d, A = Q (smem), B = K (smem)
//   O += P V     : tcgen05.mma M=128, N=d, K=64 keys, A = P (smem), B = V (smem,
//                  MN-major), accumulated in TMEM across key tiles.
// TMEM columns: two S buffers at [0, 64) and [64, 128), O at [128, 256).
// Warps w and w+4 share TMEM lane quarter w (query rows 32w .. 32w+31) and
// split each row's 64 scores into two halves of 32: each thread reads its half
// with tcgen05.ld, applies the causal mask, exchanges its half-row maximum
// with its partner through shared memory, and runs the online softmax in
// registers (scale and max-subtraction fused into one multiply-add, exp2 on
// the special-function unit), writing its half of the row of P (bf16) to
// shared memory for the PV MMA.  O's 128 columns are split the same way.
// Software pipeline, one CTA per SM: when all 256 softmax threads have
// arrived on the P barrier of tile kt (P written, tile kt+2 landed), the MMA
// lane issues PV(kt) and S(kt+2), so the tensor core computes them while the
// softmax warps work on tile kt+1, whose S was issued one tile earlier.  No
// CTA-wide barrier is used inside the loop.  K/V tiles are fetched four tiles ahead into a 5-stage ring, and
// the block ids they need are read one further tile ahead.
// The running max is only moved when a row's tile maximum exceeds it by more
// than 8 (log2 units), so P <= 256 and O is rarely rescaled; the final O / l
// uses the same reference for numerator and denominator, so this is exact.
//
// Shared memory (all operands in the 128-byte-swizzled canonical layout:
// 8-row atoms of 8 x 128 bytes, 16-byte chunk c of row r stored at chunk
// c ^ (r % 8)):
//   Q   : two 64-column halves of 128 rows                         (32 KB)
//   K,V : five stages x (K, V) x two 64-column halves of 64 rows    (160 KB)
//   P   : two buffers of 128 rows x 64 keys                         (32 KB)
// K/V tiles are filled with 16-byte cp.async copies (zero-filled past the
// needed keys).
// Every wait on an mbarrier is bounded.  A thread whose wait expires records
// the failure and carries on without waiting (its results are garbage), so
// every arrival and pair barrier is still reached; the CTA then records
// PKV_STATUS_INTERNAL, drains its copies, frees its TMEM and returns.
#include <math.h>

#include "common.cuh"
#include "prefill_common.cuh"
#include "tcgen05.cuh"

namespace {

using pkv::kBlock;
using pkv::PrefillParams;

constexpr int D = 128;
constexpr int BM = 128;
constexpr int BN = 64;
constexpr int kSoftmaxThreads = 256;
constexpr int kThreads = kSoftmaxThreads + 32;  // + the MMA-issue warp
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kOCol = 128;  // S buffers at columns 0 and 64
constexpr int kStages = 5;

constexpr int kQHalf = BM * 128;            // 16 KB: 128 rows x 64 bf16
constexpr int kKVHalf = BN * 128;           // 8 KB: 64 rows x 64 bf16
constexpr int kTileBytes = 2 * kKVHalf;     // one K or V tile (both halves)
constexpr int kStageBytes = 2 * kTileBytes; // K + V
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + 2 * kQHalf;              // 32768
constexpr int kPBytes = BM * BN * 2;                    // 16384
constexpr int kOffP = kOffKV + kStages * kStageBytes;   // 196608
constexpr int kOffBar = kOffP + 2 * kPBytes;            // 229376
constexpr int kOffRed = kOffBar + 64;                   // [2][2][128] floats
constexpr int kSmemBytes = kOffRed + 2 * 2 * BM * 4;
constexpr unsigned kWaitIters = 1u << 24;

constexpr uint32_t kIdescS = pkv::tc::idesc_bf16_f32(BM, BN, false, false);
constexpr uint32_t kIdescPV = pkv::tc::idesc_bf16_f32(BM, D, false, true);

__device__ __forceinline__ int sw128(int r, int c16) {
    return (r >> 3) * 1024 + (r & 7) * 128 + ((c16 ^ (r & 7)) << 4);
}

template <typename OutT>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const PrefillParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;  // TMEM lane quarter, score-column half
    const int row = quarter * 32 + lane;             // this thread's query row in the tile
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

    uint64_t *bar_s = reinterpret_cast<uint64_t *>(smem + kOffBar);  // S(kt) done, per S buffer
    uint64_t *bar_o = bar_s + 2;   // PV(kt) done
    uint64_t *bar_p = bar_s + 3;   // P(kt) written and tile kt+2 landed, per P buffer
    uint64_t *bar_go = bar_s + 5;  // Q, tiles 0 and 1 landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_s + 6);
    // [parity][half][row]: half-row maxima exchanged between partner warps.
    // Alternating by tile parity, a slot is rewritten only after the next pair
    // barrier, by which time the partner has read it.
    float *xmax = reinterpret_cast<float *>(smem + kOffRed);

    if (warp == 0) {
        pkv::tc::tmem_alloc(tmem_slot, kTmemCols);
        pkv::tc::tmem_relinquish();
    }
    if (tid == 0) {
        pkv::tc::mbar_init(bar_s, 1);
        pkv::tc::mbar_init(bar_s + 1, 1);
        pkv::tc::mbar_init(bar_o, 1);
        pkv::tc::mbar_init(bar_p, kSoftmaxThreads);
        pkv::tc::mbar_init(bar_p + 1, kSoftmaxThreads);
        pkv::tc::mbar_init(bar_go, kSoftmaxThreads);
        pkv::tc::fence_mbar_init();
    }

    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
    const unsigned char *kc = static_cast<const unsigned char *>(p.k_cache);
    const unsigned char *vc = static_cast<const unsigned char *>(p.v_cache);
    const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;

    // physical ids of the 4 blocks holding keys [kt*64, kt*64 + 64)
    auto tile_ids = [&](int kt, int (&ids)[4]) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int t = kt * BN + q * kBlock;
            ids[q] = t < kv_end ? table[t / kBlock] : 0;
        }
    };
    auto load_kv = [&](int kt, const int (&ids)[4]) {
        unsigned char *kd = smem + kOffKV + (kt % kStages) * kStageBytes;
        unsigned char *vd = kd + kTileBytes;
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int i = tid + kSoftmaxThreads * u;
            const int r = i >> 4, c = i & 15;  // r >> 4 == u
            const int t = kt * BN + r;
            int nb = 0;
            size_t go = 0;
            if (t < kv_end) {
                const int phys = ids[u];
                if (phys >= 0 && phys < p.num_blocks) {
                    nb = 16;
                    go = ((((size_t)phys * p.num_kv_heads + kvh) * kBlock + (t % kBlock)) * D) * 2 + c * 16;
                } else if (c == 0 && (t % kBlock) == 0) {
                    pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                }
            }
            const int off = (c >> 3) * kKVHalf + sw128(r, c & 7);
            pkv::cp_async16(kd + off, kc + go, nb);
            pkv::cp_async16(vd + off, vc + go, nb);
        }
    };

    int ids_next[4];
    if (warp < 8) {
        // Q tile: 128 rows x 16 chunks, 8 copies per thread
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int i = tid + kSoftmaxThreads * u;
            const int r = i >> 4, c = i & 15;
            const int R = tile * BM + r;
            const int jr = R / G;
            const bool ok = jr < n;
            const __nv_bfloat16 *src =
                ok ? qg + ((size_t)(q0 + jr) * p.num_q_heads + kvh * G + (R - jr * G)) * D + c * 8 : qg;
            pkv::cp_async16(smem + kOffQ + (c >> 3) * kQHalf + sw128(r, c & 7), src, ok ? 16 : 0);
        }

        int ids[4];
        tile_ids(0, ids);
        load_kv(0, ids);  // same copy group as Q
        pkv::cp_async_commit();
#pragma unroll
        for (int t = 1; t < kStages - 1; t++) {
            tile_ids(t, ids);
            if (t < nkt) load_kv(t, ids);
            pkv::cp_async_commit();
        }
        tile_ids(kStages - 1, ids_next);
    }

    pkv::tc::fence_before_sync();
    __syncthreads();
    pkv::tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);

    // S(kt) = Q K(kt)^T into S buffer kt & 1
    auto issue_s = [&](int kt) {
        const uint32_t qa = sbase + kOffQ;
        const uint32_t kb = sbase + kOffKV + (kt % kStages) * kStageBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ks++) {
            const uint64_t a = pkv::tc::smem_desc_sw128(qa + (ks >> 2) * kQHalf + (ks & 3) * 32, 16, 1024);
            const uint64_t b = pkv::tc::smem_desc_sw128(kb + (ks >> 2) * kKVHalf + (ks & 3) * 32, 16, 1024);
            pkv::tc::mma_ss(tmem + (kt & 1) * BN, a, b, kIdescS, ks > 0 ? 1u : 0u);
        }
        pkv::tc::mma_commit(bar_s + (kt & 1));
    };
    // O (+)= P(kt) V(kt)
    auto issue_pv = [&](int kt) {
        const uint32_t pa = sbase + kOffP + (kt & 1) * kPBytes;
        const uint32_t vb = sbase + kOffKV + (kt % kStages) * kStageBytes + kTileBytes;
#pragma unroll
        for (int kq = 0; kq < BN / 16; kq++) {
            const uint64_t a = pkv::tc::smem_desc_sw128(pa + kq * 32, 16, 1024);
            // V is MN-major: next 64-column half at +8 KB (LBO), next 8 keys at +1 KB (SBO)
            const uint64_t b = pkv::tc::smem_desc_sw128(vb + kq * 2048, kKVHalf, 1024);
            pkv::tc::mma_ss(tmem + kOCol, a, b, kIdescPV, (kt == 0 && kq == 0) ? 0u : 1u);
        }
        pkv::tc::mma_commit(bar_o);
    };

    // this thread's query row (softmax warps)
    const int R = tile * BM + row;
    const int jrow = R / G;
    const bool row_ok = jrow < n;
    const int pos = row_ok ? prior + jrow : -1;
    bool failed = false;
    auto wait = [&](uint64_t *bar, unsigned parity) {
        if (!failed && !pkv::tc::mbar_wait(bar, parity, kWaitIters)) failed = true;
    };
    auto pair_sync = [&]() {  // warps w and w+4 (same rows) meet on named barrier 1 + w
        asm volatile("bar.sync %0, 64;\n" ::"r"(1 + quarter) : "memory");
    };

    if (warp == 8) {
        // ---------------- MMA issue (one lane)
        if (lane == 0) {
            wait(bar_go, 0);
            pkv::tc::fence_after_sync();
            issue_s(0);
            if (nkt > 1) issue_s(1);
            for (int kt = 0; kt < nkt; kt++) {
                wait(bar_p + (kt & 1), (unsigned)((kt >> 1) & 1));
                pkv::tc::fence_after_sync();
                issue_pv(kt);
                if (kt + 2 < nkt) issue_s(kt + 2);
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps
        float m_used = -INFINITY, lsum = 0.f;
        pkv::cp_async_wait<kStages - 3>();  // Q, tile 0 and tile 1 have landed
        pkv::tc::fence_proxy_async_smem();
        pkv::tc::mbar_arrive(bar_go);

        for (int kt = 0; kt < nkt; kt++) {
            // S(kt) done; it was issued after PV(kt-2), so that one is done too
            wait(bar_s + (kt & 1), (unsigned)((kt >> 1) & 1));
            pkv::tc::fence_after_sync();

            // this thread's 32 raw scores (keys t0 + i)
            float sv[32];
            pkv::tc::tmem_ld32(t_lane + (kt & 1) * BN + half * 32, sv);
            const int t0 = kt * BN + half * 32;
            if (kt * BN + BN <= mask_from) {
                if (!row_ok) {
#pragma unroll
                    for (int i = 0; i < 32; i++) sv[i] = -INFINITY;
                }
            } else {
                const int lim = pos - t0;  // keys i <= lim are visible
#pragma unroll
                for (int i = 0; i < 32; i++) sv[i] = i <= lim ? sv[i] : -INFINITY;
            }
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; i++)
                mx[i] = fmaxf(fmaxf(sv[i], sv[i + 8]), fmaxf(sv[i + 16], sv[i + 24]));
#pragma unroll
            for (int i = 0; i < 4; i++) mx[i] = fmaxf(mx[i], mx[i + 4]);
            float mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            float *xm = xmax + (kt & 1) * 2 * BM;
            xm[half * BM + row] = mraw;
            pair_sync();
            mraw = fmaxf(mraw, xm[(half ^ 1) * BM + row]);
            const float mt = mraw * p.scale_log2;  // scale > 0 commutes with max; -inf stays
            const bool need = mt > m_used + 8.f;
            float alpha = 1.f;
            if (need) {
                alpha = pkv::tc::ex2(m_used - mt);  // 0 when nothing was seen yet
                lsum *= alpha;
                m_used = mt;
            }
            if (kt > 0 && __any_sync(0xffffffffu, need)) {
                // rescaling O needs PV(kt-1) to have finished
                wait(bar_o, (unsigned)((kt - 1) & 1));
                pkv::tc::fence_after_sync();
#pragma unroll 1
                for (int c = 0; c < D / 2; c += 32) {
                    float o[32];
                    pkv::tc::tmem_ld32(t_lane + kOCol + half * (D / 2) + c, o);
#pragma unroll
                    for (int i = 0; i < 32; i++) o[i] *= alpha;
                    pkv::tc::tmem_st32(t_lane + kOCol + half * (D / 2) + c, o);
                }
            }
            const float nbase = m_used == -INFINITY ? 0.f : -m_used;
            unsigned char *prow = smem + kOffP + (kt & 1) * kPBytes;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 4; c++) {
                float e[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    e[i] = pkv::tc::ex2(fmaf(sv[c * 8 + i], p.scale_log2, nbase));
                    ls[i & 3] += e[i];
                }
                uint4 pk;
                pk.x = pkv::pack_bf16(e[0], e[1]);
                pk.y = pkv::pack_bf16(e[2], e[3]);
                pk.z = pkv::pack_bf16(e[4], e[5]);
                pk.w = pkv::pack_bf16(e[6], e[7]);
                *reinterpret_cast<uint4 *>(prow + sw128(row, half * 4 + c)) = pk;
            }
            lsum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // PV(kt-1) done frees stage (kt-1) % kStages: fetch tile kt+kStages-1 into it
            if (kt > 0) wait(bar_o, (unsigned)((kt - 1) & 1));
            if (kt + kStages - 1 < nkt) load_kv(kt + kStages - 1, ids_next);
            pkv::cp_async_commit();
            tile_ids(kt + kStages, ids_next);
            pkv::cp_async_wait<kStages - 3>();  // every tile up to kt+2 has landed
            pkv::tc::fence_proxy_async_smem();
            pkv::tc::fence_before_sync();
            pkv::tc::mbar_arrive(bar_p + (kt & 1));
        }

        wait(bar_o, (unsigned)((nkt - 1) & 1));
        pkv::tc::fence_after_sync();
        float *xl = xmax + (nkt & 1) * 2 * BM;
        xl[half * BM + row] = lsum;
        pair_sync();
        const float ltot = lsum + xl[(half ^ 1) * BM + row];
        const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
        OutT *orow = static_cast<OutT *>(p.out) +
                     ((size_t)(q0 + jrow) * p.num_q_heads + kvh * G + (R - jrow * G)) * D + half * (D / 2);
#pragma unroll 1
        for (int c = 0; c < D / 2; c += 32) {
            float o[32];
            pkv::tc::tmem_ld32(t_lane + kOCol + half * (D / 2) + c, o);
            if (row_ok && !failed) {
#pragma unroll
                for (int i = 0; i < 32; i += 2) pkv::store2(orow + c + i, o[i] * inv, o[i + 1] * inv);
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

int launch_prefill_tc(const PrefillParams &p, int num_seqs, int out_dtype, cudaStream_t st) {
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
        prefill_tc_kernel<float><<<grid, kThreads, kSmemBytes, st>>>(p);
    else
        prefill_tc_kernel<__nv_bfloat16><<<grid, kThreads, kSmemBytes, st>>>(p);
    return check_launch("prefill_tc");
}

}  // namespace pkv
