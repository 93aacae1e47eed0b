// Paged-attention decode with split-K partitions and a log-sum-exp reduce.
//
// Work unit: one CTA per (kv head [x q-head chunk], sequence, partition of
// `partition` tokens).  The G = Hq / Hkv query heads that share a kv head
// share every K/V byte fetched (GQA, chengxuchu #47 section 2.3): for G <= 8
// (and for fp8 caches) the block's 16 tokens are the M side of each
// tensor-core product and the G query rows its N side (decode_bf16t_kernel,
// decode_fp8_kernel); for larger groups the query rows are the M = 16 side
// (decode_bf16_kernel).  The partition's 16-token
// blocks are split between the CTA's 4 warps; each warp streams its blocks
// through a private ring of shared-memory stages filled by 16-byte cp.async
// copies, looked up through the block table (section 5.2), and keeps its own
// online-softmax state (running max m, sum l, unnormalised O).  The 4 warp
// states are merged in shared memory; a sequence that fits one partition gets
// its final output here, otherwise (m, l, O) go to the workspace and a second
// launch merges the partitions:
//   M = max_p m_p,  L = sum_p l_p 2^(m_p - M),  out = sum_p 2^(m_p - M) O_p / L.
// Logits are kept in base-2 units (scale * log2 e folded into one multiply).
#include <math.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "prefill_common.cuh"

namespace {

using pkv::kBlock;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;   // per-warp ring depth, in blocks
constexpr int kRows = 16;    // q heads per tile (mma M)

struct DecodeParams {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    void *out;
    float *part_o;   // [S][Hq][max_parts][D]
    float *part_ml;  // [S][Hq][max_parts][2]
    int max_blocks;
    int num_q_heads;
    int num_kv_heads;
    int group;       // Hq / Hkv
    int head_chunks; // ceil(group / 16)
    int num_blocks;
    int len_cap;     // min(max_blocks * 16, max_context_len)
    int partition;
    int max_parts;
    float scale_log2;
    unsigned *status;
    // fused append: token L-1 of sequence s (k_new/v_new [S][Hkv][D]) is
    // written into the cache by the CTA(s) of the last partition, or nullptr
    const void *k_new;
    const void *v_new;
    // shared prefix: tokens [0, prefix_len) of every sequence are handled
    // elsewhere (their merged state is partial slot 0); the partitions here
    // cover [prefix_len, L) and write slots 1, 2, ...  0 = no prefix.
    int prefix_len;
    // The launch before this one is the shared-prefix kernel, whose results
    // this kernel does not read: do not wait for it at the start (run beside
    // it). The grid's last CTA waits for it before exiting, so this grid
    // completes after it, and the merge launch, which waits for this grid,
    // also sees the prefix kernel's partials.
    int overlap_prev;
    // 1: each warp of a thread block streams the whole partition for its own
    // (kv head, head chunk), four per block; 0: the four warps split one
    // (kv head, chunk)'s partition and merge (set by the host, see
    // use_head_warps)
    int head_warps;
    // fp8 E4M3 caches: per kv head scales (stored = value / scale), else null
    const float *k_scale;
    const float *v_scale;
};


// Partitions of the tokens this launch covers for a sequence of L tokens.
__device__ __forceinline__ int own_parts(const DecodeParams &p, int L) {
    if (p.prefix_len == 0) return L > 0 ? (L + p.partition - 1) / p.partition : 1;
    const int suf = L - p.prefix_len;
    return suf > 0 ? (suf + p.partition - 1) / p.partition : 0;
}

// Write the new token of sequence s, kv head kvh, at logical position L-1.
// Called by the threads [first, first + count) that own the partition holding
// L-1, followed by a barrier over them before the partition is read.
template <typename T>
__device__ __forceinline__ void append_new_token(const DecodeParams &p, const int32_t *table, int s, int kvh,
                                                 int L, int D, int first, int count) {
    const int t = L - 1;
    const int phys = table[t / kBlock];
    if (phys < 0 || phys >= p.num_blocks) return;  // reported by the gather
    const int chunks = D * (int)sizeof(T) / 16;
    const size_t dst = (((size_t)phys * p.num_kv_heads + kvh) * kBlock + (t % kBlock)) * chunks;
    const size_t src = ((size_t)s * p.num_kv_heads + kvh) * chunks;
    for (int i = first; i < 2 * chunks; i += count) {
        const bool is_v = i >= chunks;
        const int c = is_v ? i - chunks : i;
        const uint4 *from = static_cast<const uint4 *>(is_v ? p.v_new : p.k_new) + src + c;
        uint4 *to = static_cast<uint4 *>(const_cast<void *>(is_v ? p.v_cache : p.k_cache)) + dst + c;
        *to = *from;
    }
}

// fp8 caches: quantise and write the new token's K and V rows (bf16, d =
// 128) of sequence s, kv head kvh at logical position L-1, exactly as
// pkv_kv_append_fp8 does (code = E4M3(x / scale): IEEE division, nearest
// even, saturated at 448).  16 chunks of 16 values (8 for K, 8 for V), taken
// by the threads [first, first + count); a barrier over them follows before
// the row is read.
__device__ __forceinline__ void append_new_token_fp8(const DecodeParams &p, const int32_t *table, int s, int kvh,
                                                     int L, int first, int count) {
    const int t = L - 1;
    const int phys = table[t / kBlock];
    if (phys < 0 || phys >= p.num_blocks) return;  // reported by the gather
    const size_t row = ((size_t)phys * p.num_kv_heads + kvh) * kBlock + (t % kBlock);  // 128-byte rows
    const size_t src = ((size_t)s * p.num_kv_heads + kvh) * 128;
    for (int i = first; i < 16; i += count) {
        const bool is_v = i >= 8;
        const int c = i & 7;
        const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(is_v ? p.v_new : p.k_new) + src + 16 * c;
        const float sc = is_v ? p.v_scale[kvh] : p.k_scale[kvh];
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const float a0 = __fdiv_rn(__bfloat162float(x[4 * q]), sc), a1 = __fdiv_rn(__bfloat162float(x[4 * q + 1]), sc);
            const float a2 = __fdiv_rn(__bfloat162float(x[4 * q + 2]), sc), a3 = __fdiv_rn(__bfloat162float(x[4 * q + 3]), sc);
            w[q] = (uint32_t)pkv::f32x2_to_e4m3x2(a0, a1) | ((uint32_t)pkv::f32x2_to_e4m3x2(a2, a3) << 16);
        }
        uint4 *dst = static_cast<uint4 *>(const_cast<void *>(is_v ? p.v_cache : p.k_cache)) + row * 8 + c;
        *dst = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__device__ __forceinline__ int clamp_len(int L, int cap, unsigned *status, bool report) {
    if (L < 0 || L > cap) {
        if (report) pkv::flag(status, PKV_STATUS_BAD_LENGTH);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// ----------------------------------------------------------------------------
// bf16 tensor-core decode, query rows on the M side (groups above 8 heads, in
// chunks of 16)
// ----------------------------------------------------------------------------

template <int D>
struct DecodeSmem {
    static constexpr int kRing = kStages;                  // ring depth in blocks
    static constexpr int kRowBytes = D * 2;                // one cached row
    static constexpr int kTile = kBlock * kRowBytes;      // one block of one kv head
    static constexpr int kStage = 2 * kTile;               // K + V
    static constexpr int kWarp = kRing * kStage;
    static constexpr int kStaging = kWarps * kWarp;
    static constexpr int kMergeStride = D + 8;             // floats per merged row
    static constexpr int kMergeWarp = kRows * kMergeStride + 2 * kRows;
    static constexpr int kMerge = kWarps * kMergeWarp * 4;
    static constexpr int kBytes = kStaging > kMerge ? kStaging : kMerge;
};

template <int D, typename OutT, bool kHeadWarps>
__global__ void __launch_bounds__(kThreads, 2) decode_bf16_kernel(const DecodeParams p) {
    using Sm = DecodeSmem<D>;
    constexpr int CH = Sm::kRowBytes / 16;    // 16-byte chunks per cached row
    constexpr int PER_LANE = kBlock * CH / 32;
    constexpr int KSTEPS = D / 16;
    constexpr int NT = D / 8;                 // n-tiles of the output

    extern __shared__ __align__(128) unsigned char smem[];
    pkv::allow_dependents();
    if (!p.overlap_prev) pkv::grid_dependency_wait();  // the appended tokens of the previous launch
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gid = lane >> 2, tig = lane & 3;
    // the (kv head, head chunk) unit of this warp
    const int unit = kHeadWarps ? blockIdx.x * kWarps + warp : blockIdx.x;
    const bool idle = kHeadWarps && unit >= p.num_kv_heads * p.head_chunks;
    const int kvh = unit / p.head_chunks, chunk = unit - kvh * p.head_chunks;
    const int s = blockIdx.y, part = blockIdx.z;
    const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;
    const int blk_begin = (p.prefix_len + part * p.partition) / kBlock;
    // The warp's blocks: a head warp takes every block of the partition; a
    // split warp every fourth, starting at its own index.  The positions do
    // not depend on the length, so the first 32 block ids are fetched now,
    // alongside the length rather than after it, with one coalesced load;
    // issuing a copy then never waits on a dependent block-table read.
    const int bstride = kHeadWarps ? 1 : kWarps;
    const int bfirst = blk_begin + (kHeadWarps ? 0 : warp);
    int my_id = 0;
    if (!idle && bfirst + bstride * lane < p.max_blocks) my_id = table[bfirst + bstride * lane];

    const int L = clamp_len(p.context_lens[s], p.len_cap, p.status,
                            part == 0 && blockIdx.x == 0 && threadIdx.x == 0);
    if (p.prefix_len && L <= p.prefix_len && part == 0 && blockIdx.x == 0 && threadIdx.x == 0)
        pkv::flag(p.status, PKV_STATUS_BAD_LENGTH);  // no private token after the shared prefix
    const int nparts = own_parts(p, L);
    const bool tail_wait = p.overlap_prev && blockIdx.x == gridDim.x - 1 &&
                           blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1;
    if (part >= nparts || idle) {
        if (tail_wait) pkv::grid_dependency_wait();
        return;
    }
    const int slot0 = p.prefix_len ? 1 : 0;  // partial slot 0 holds the shared prefix
    const int nslots = slot0 + nparts;

    const int h0 = kvh * p.group + chunk * kRows;
    const int rows = min(kRows, p.group - chunk * kRows);
    const int t_begin = p.prefix_len + part * p.partition;
    const int t_end = min(L, t_begin + p.partition);
    const int nblk = (t_end + kBlock - 1) / kBlock - blk_begin;
    const int n = kHeadWarps ? nblk : max(0, (nblk - warp + kWarps - 1) / kWarps);

    const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
    const unsigned char *kc = static_cast<const unsigned char *>(p.k_cache);
    const unsigned char *vc = static_cast<const unsigned char *>(p.v_cache);

    // query rows of this tile as mma A fragments (rows >= `rows` are zero)
    uint32_t qa[KSTEPS][4];
    {
        const bool va = gid < rows, vb = gid + 8 < rows;
        const __nv_bfloat16 *qa_row = qb + ((size_t)s * p.num_q_heads + h0 + gid) * D;
        const __nv_bfloat16 *qb_row = qa_row + 8 * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; kk++) {
            const int col = kk * 16 + tig * 2;
            qa[kk][0] = va ? *reinterpret_cast<const uint32_t *>(qa_row + col) : 0u;
            qa[kk][1] = vb ? *reinterpret_cast<const uint32_t *>(qb_row + col) : 0u;
            qa[kk][2] = va ? *reinterpret_cast<const uint32_t *>(qa_row + col + 8) : 0u;
            qa[kk][3] = vb ? *reinterpret_cast<const uint32_t *>(qb_row + col + 8) : 0u;
        }
    }
    const float sl2 = p.scale_log2;  // softmax scale in base-2 units

    if (p.k_new && part == nparts - 1 && L > 0) {
        // the new row is read below through L2 by other threads
        if (kHeadWarps) {
            // (warps of other chunks of the same kv head write the same bytes)
            append_new_token<__nv_bfloat16>(p, table, s, kvh, L, D, lane, 32);
            __syncwarp();
        } else {
            append_new_token<__nv_bfloat16>(p, table, s, kvh, L, D, threadIdx.x, kThreads);
            __syncthreads();
        }
    }

    unsigned char *ring = smem + warp * Sm::kWarp;

    auto block_id = [&](int li) -> int {
        return li < 32 ? __shfl_sync(0xffffffffu, my_id, li) : table[bfirst + bstride * li];
    };
    // rows of the warp's li-th block that hold tokens of this partition (-1 for a bad id)
    auto block_rows = [&](int li, int &phys) -> int {
        phys = block_id(li);
        if (phys < 0 || phys >= p.num_blocks) return -1;
        return min(kBlock, t_end - (bfirst + bstride * li) * kBlock);
    };

    auto issue = [&](int li, int st) {
        int phys;
        int valid = block_rows(li, phys);
        if (valid < 0) {
            if (lane == 0) pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
            valid = 0;
            phys = 0;
        }
        const size_t base = ((size_t)phys * p.num_kv_heads + kvh) * kBlock * Sm::kRowBytes;
        const unsigned char *kg = kc + base;
        const unsigned char *vg = vc + base;
        unsigned char *ks = ring + st * Sm::kStage;
        unsigned char *vs = ks + Sm::kTile;
#pragma unroll
        for (int j = 0; j < PER_LANE; j++) {
            const int i = lane + 32 * j;
            const int r = i / CH, c = i - (i / CH) * CH;
            const int nb = r < valid ? 16 : 0;
            const int go = r * Sm::kRowBytes + c * 16;
            pkv::cp_async16(ks + pkv::swz(r, c, Sm::kRowBytes), kg + (nb ? go : 0), nb);
            pkv::cp_async16(vs + pkv::swz(r, c, Sm::kRowBytes), vg + (nb ? go : 0), nb);
        }
    };

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

#pragma unroll
    for (int st = 0; st < Sm::kRing - 1; st++) {
        if (st < n) issue(st, st);
        pkv::cp_async_commit();
    }

    for (int i = 0; i < n; i++) {
        {
            const int nx = i + Sm::kRing - 1;
            if (nx < n) issue(nx, nx % Sm::kRing);
            pkv::cp_async_commit();
        }
        pkv::cp_async_wait<Sm::kRing - 1>();
        __syncwarp();

        const int st = i % Sm::kRing;
        const unsigned char *ks = ring + st * Sm::kStage;
        const unsigned char *vs = ks + Sm::kTile;

        int phys;
        int valid = block_rows(i, phys);
        if (valid < 0) valid = 0;

        // S = q . K^T for the block's 16 tokens (two n-tiles of 8 tokens)
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        {
#pragma unroll
            for (int kk = 0; kk < KSTEPS; kk++) {
                uint32_t b0, b1, b2, b3;
                const int tok = ((lane >> 4) << 3) + (lane & 7);
                const int ch = kk * 2 + ((lane >> 3) & 1);
                pkv::ldsm_x4(b0, b1, b2, b3, ks + pkv::swz(tok, ch, D * 2));
                pkv::mma_bf16(s0, qa[kk], b0, b1);
                pkv::mma_bf16(s1, qa[kk], b2, b3);
            }
        }
        // scale to base-2 units and mask rows past the context
        const int t0 = tig * 2;
        float x[8] = {s0[0], s0[1], s1[0], s1[1], s0[2], s0[3], s1[2], s1[3]};
        const int tk[4] = {t0, t0 + 1, t0 + 8, t0 + 9};
#pragma unroll
        for (int e = 0; e < 8; e++) {
            x[e] = tk[e & 3] < valid ? x[e] * sl2 : -INFINITY;
        }
        float mxA = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        float mxB = fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7]));
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
        // The running maximum moves only when a row's scores exceed it by
        // more than 2^8 (base-2 units), so the state (m, l, O) is rescaled
        // rarely; P = 2^(x - m) then stays at most 256, which fp16 and the
        // bf16 hi/lo split of P hold without loss of relative precision,
        // and the result O / l does not depend on which m is used.
        if (__any_sync(0xffffffffu, mxA > mA + 8.f || mxB > mB + 8.f)) {
            const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
            const float alA = pkv::fast_exp2(mA - (nA == -INFINITY ? 0.f : nA));
            const float alB = pkv::fast_exp2(mB - (nB == -INFINITY ? 0.f : nB));
            mA = nA;
            mB = nB;
            lA *= alA;
            lB *= alB;
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                o[nt][0] *= alA;
                o[nt][1] *= alA;
                o[nt][2] *= alB;
                o[nt][3] *= alB;
            }
        }
        const float baseA = mA == -INFINITY ? 0.f : mA;
        const float baseB = mB == -INFINITY ? 0.f : mB;
        float pr[8];
#pragma unroll
        for (int e = 0; e < 4; e++) pr[e] = pkv::fast_exp2(x[e] - baseA);
#pragma unroll
        for (int e = 4; e < 8; e++) pr[e] = pkv::fast_exp2(x[e] - baseB);
        lA += (pr[0] + pr[1] + pr[2] + pr[3]);
        lB += (pr[4] + pr[5] + pr[6] + pr[7]);
        {
            // P as two bf16 A fragments, hi + lo, so P keeps ~16 significant bits
            float hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; e++) pkv::split_bf16(pr[e], hi[e], lo[e]);
            const uint32_t ph[4] = {pkv::pack_bf16(hi[0], hi[1]), pkv::pack_bf16(hi[4], hi[5]),
                                    pkv::pack_bf16(hi[2], hi[3]), pkv::pack_bf16(hi[6], hi[7])};
            const uint32_t pl[4] = {pkv::pack_bf16(lo[0], lo[1]), pkv::pack_bf16(lo[4], lo[5]),
                                    pkv::pack_bf16(lo[2], lo[3]), pkv::pack_bf16(lo[6], lo[7])};
            // O += P . V
#pragma unroll
            for (int nn = 0; nn < D / 16; nn++) {
                uint32_t v0, v1, v2, v3;
                const int j = lane >> 3;
                const int tok = ((j & 1) << 3) + (lane & 7);
                const int ch = nn * 2 + (j >> 1);
                pkv::ldsm_x4_t(v0, v1, v2, v3, vs + pkv::swz(tok, ch, D * 2));
                pkv::mma_bf16(o[2 * nn], ph, v0, v1);
                pkv::mma_bf16(o[2 * nn], pl, v0, v1);
                pkv::mma_bf16(o[2 * nn + 1], ph, v2, v3);
                pkv::mma_bf16(o[2 * nn + 1], pl, v2, v3);
            }
        }
        __syncwarp();
    }

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);

    pkv::cp_async_wait<0>();
    // The accumulator as pairs of adjacent output columns: slot k holds, for
    // row gid (hi = 0) or gid + 8 (hi = 1), the values of columns col and
    // col + 1.
    auto out_pair = [&](int k, int hi, float &x0, float &x1) -> int {
        x0 = o[k][2 * hi];
        x1 = o[k][2 * hi + 1];
        return k * 8 + tig * 2;
    };
    if (kHeadWarps) {
        // the warp holds its rows' whole state for this partition
        const size_t orow = (size_t)s * p.num_q_heads + h0 + gid;
        const bool okA = gid < rows, okB = gid + 8 < rows;
        if (nslots == 1) {
            OutT *oa = static_cast<OutT *>(p.out) + orow * D;
            OutT *ob = oa + 8 * D;
            const float ia = lA > 0.f ? 1.f / lA : 0.f, ib = lB > 0.f ? 1.f / lB : 0.f;
#pragma unroll
            for (int k = 0; k < NT; k++) {
                float x0, x1, y0, y1;
                const int col = out_pair(k, 0, x0, x1);
                out_pair(k, 1, y0, y1);
                if (okA) pkv::store2(oa + col, x0 * ia, x1 * ia);
                if (okB) pkv::store2(ob + col, y0 * ib, y1 * ib);
            }
        } else {
            const size_t pa = orow * p.max_parts + slot0 + part, pb = pa + 8 * (size_t)p.max_parts;
#pragma unroll
            for (int k = 0; k < NT; k++) {
                float x0, x1, y0, y1;
                const int col = out_pair(k, 0, x0, x1);
                out_pair(k, 1, y0, y1);
                if (okA) *reinterpret_cast<float2 *>(p.part_o + pa * D + col) = make_float2(x0, x1);
                if (okB) *reinterpret_cast<float2 *>(p.part_o + pb * D + col) = make_float2(y0, y1);
            }
            if (tig == 0 && okA) *reinterpret_cast<float2 *>(p.part_ml + pa * 2) = make_float2(mA, lA);
            if (tig == 0 && okB) *reinterpret_cast<float2 *>(p.part_ml + pb * 2) = make_float2(mB, lB);
        }
        if (tail_wait) pkv::grid_dependency_wait();
        return;
    }
    __syncthreads();  // every warp is done with its ring; reuse it for the merge

    float *mw = reinterpret_cast<float *>(smem) + warp * Sm::kMergeWarp;
    float *mm = mw + kRows * Sm::kMergeStride;
    float *ll = mm + kRows;
    if (tig == 0) {
        mm[gid] = mA;
        mm[gid + 8] = mB;
        ll[gid] = lA;
        ll[gid + 8] = lB;
    }
#pragma unroll
    for (int k = 0; k < NT; k++) {
        float x0, x1, y0, y1;
        const int col = out_pair(k, 0, x0, x1);
        out_pair(k, 1, y0, y1);
        *reinterpret_cast<float2 *>(mw + gid * Sm::kMergeStride + col) = make_float2(x0, x1);
        *reinterpret_cast<float2 *>(mw + (gid + 8) * Sm::kMergeStride + col) = make_float2(y0, y1);
    }
    __syncthreads();

    const float *base = reinterpret_cast<const float *>(smem);
    for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
        const int r = idx / D, c = idx - (idx / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; w++) M = fmaxf(M, base[w * Sm::kMergeWarp + kRows * Sm::kMergeStride + r]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; w++) {
                const float *bw = base + w * Sm::kMergeWarp;
                const float f = pkv::fast_exp2(bw[kRows * Sm::kMergeStride + r] - M);
                lsum += bw[kRows * Sm::kMergeStride + kRows + r] * f;
                acc += bw[r * Sm::kMergeStride + c] * f;
            }
        }
        const size_t orow = (size_t)s * p.num_q_heads + h0 + r;
        if (nslots == 1) {
            pkv::store1(static_cast<OutT *>(p.out) + orow * D + c, lsum > 0.f ? acc / lsum : 0.f);
        } else {
            const size_t prow = orow * p.max_parts + slot0 + part;
            p.part_o[prow * D + c] = acc;
            if (c == 0) {
                p.part_ml[prow * 2] = M;
                p.part_ml[prow * 2 + 1] = lsum;
            }
        }
    }
    if (tail_wait) pkv::grid_dependency_wait();
}

// ----------------------------------------------------------------------------
// bf16 decode with the products transposed (query groups of at most 8)
// ----------------------------------------------------------------------------
// S^T = K q^T and O^T = V^T P^T, as in the fp8 kernel below: the block's 16
// tokens are the M side of each m16n8k16 product and the unit's (at most 8)
// query rows its N side, which halves the products and the exponentials per
// block against the layout with the queries on the M side when a kv head
// has 4 or 8 query heads.  K reaches the A fragments by ldmatrix, V^T by
// ldmatrix.trans; q^T is read from global memory as B fragments once; P^T
// goes from the score accumulator to B fragments by one 8x8 transpose in
// registers per 8 tokens, as two bf16 halves (hi + lo, about 16 significant
// bits, as in the bf16 kernel above).  The state of the rows leaves through
// shared memory, so every row is written out (or merged) contiguously.
constexpr int kRows8 = 8;  // query rows of one unit of the transposed kernels

template <int D>
struct DecodeTSmem {
    static constexpr int kRing = kStages;
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTile = kBlock * kRowBytes;
    static constexpr int kStage = 2 * kTile;
    static constexpr int kWarp = kRing * kStage;
    static constexpr int kStaging = kWarps * kWarp;
    static constexpr int kStride = D + 4;                  // floats per staged row
    static constexpr int kStateWarp = 8 * kStride + 16;    // O rows, then m[8], l[8]
    static constexpr int kState = kWarps * kStateWarp * 4;
    static constexpr int kBytes = kStaging > kState ? kStaging : kState;
};

__device__ __forceinline__ uint32_t transpose8x8_b16(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
    return d;
}

template <int D, typename OutT, bool kHeadWarps>
__global__ void __launch_bounds__(kThreads, 2) decode_bf16t_kernel(const DecodeParams p) {
    using Sm = DecodeTSmem<D>;
    constexpr int CH = Sm::kRowBytes / 16;    // 16-byte chunks per cached row
    constexpr int PER_LANE = kBlock * CH / 32;
    constexpr int KSTEPS = D / 16, MT = D / 16;

    extern __shared__ __align__(128) unsigned char smem[];
    pkv::allow_dependents();
    if (!p.overlap_prev) pkv::grid_dependency_wait();  // the appended tokens of the previous launch
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gid = lane >> 2, tig = lane & 3;
    const int unit = kHeadWarps ? blockIdx.x * kWarps + warp : blockIdx.x;
    const bool idle = kHeadWarps && unit >= p.num_kv_heads * p.head_chunks;
    const int kvh = unit / p.head_chunks, chunk = unit - kvh * p.head_chunks;
    const int s = blockIdx.y, part = blockIdx.z;
    const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;
    const int blk_begin = (p.prefix_len + part * p.partition) / kBlock;
    const int bstride = kHeadWarps ? 1 : kWarps;
    const int bfirst = blk_begin + (kHeadWarps ? 0 : warp);
    int my_id = 0;
    if (!idle && bfirst + bstride * lane < p.max_blocks) my_id = table[bfirst + bstride * lane];

    const int L = clamp_len(p.context_lens[s], p.len_cap, p.status,
                            part == 0 && blockIdx.x == 0 && threadIdx.x == 0);
    if (p.prefix_len && L <= p.prefix_len && part == 0 && blockIdx.x == 0 && threadIdx.x == 0)
        pkv::flag(p.status, PKV_STATUS_BAD_LENGTH);  // no private token after the shared prefix
    const int nparts = own_parts(p, L);
    const bool tail_wait = p.overlap_prev && blockIdx.x == gridDim.x - 1 &&
                           blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1;
    if (part >= nparts || idle) {
        if (tail_wait) pkv::grid_dependency_wait();
        return;
    }
    const int slot0 = p.prefix_len ? 1 : 0;  // partial slot 0 holds the shared prefix
    const int nslots = slot0 + nparts;

    const int h0 = kvh * p.group + chunk * kRows8;
    const int rows = min(kRows8, p.group - chunk * kRows8);
    const int t_begin = p.prefix_len + part * p.partition;
    const int t_end = min(L, t_begin + p.partition);
    const int nblk = (t_end + kBlock - 1) / kBlock - blk_begin;
    const int n = kHeadWarps ? nblk : max(0, (nblk - warp + kWarps - 1) / kWarps);
    const unsigned char *kc = static_cast<const unsigned char *>(p.k_cache);
    const unsigned char *vc = static_cast<const unsigned char *>(p.v_cache);

    // q^T as B fragments: query row gid of the unit (zero past `rows`),
    // d = 16 kk + 2 tig + {0, 1} and + 8
    uint32_t qb[KSTEPS][2];
    {
        const bool ok = gid < rows;
        const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(p.q) +
                                    ((size_t)s * p.num_q_heads + h0 + (ok ? gid : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; kk++) {
            qb[kk][0] = ok ? *reinterpret_cast<const uint32_t *>(qrow + 16 * kk + 2 * tig) : 0u;
            qb[kk][1] = ok ? *reinterpret_cast<const uint32_t *>(qrow + 16 * kk + 2 * tig + 8) : 0u;
        }
    }
    const float sl2 = p.scale_log2;

    if (p.k_new && part == nparts - 1 && L > 0) {
        // the new row is read below through L2 by other threads
        if (kHeadWarps) {
            append_new_token<__nv_bfloat16>(p, table, s, kvh, L, D, lane, 32);
            __syncwarp();
        } else {
            append_new_token<__nv_bfloat16>(p, table, s, kvh, L, D, threadIdx.x, kThreads);
            __syncthreads();
        }
    }

    unsigned char *ring = smem + warp * Sm::kWarp;
    auto block_id = [&](int li) -> int {
        return li < 32 ? __shfl_sync(0xffffffffu, my_id, li) : table[bfirst + bstride * li];
    };
    auto block_rows = [&](int li, int &phys) -> int {
        phys = block_id(li);
        if (phys < 0 || phys >= p.num_blocks) return -1;
        return min(kBlock, t_end - (bfirst + bstride * li) * kBlock);
    };
    auto issue = [&](int li, int st) {
        int phys;
        int valid = block_rows(li, phys);
        if (valid < 0) {
            if (lane == 0) pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
            valid = 0;
            phys = 0;
        }
        const size_t base = ((size_t)phys * p.num_kv_heads + kvh) * Sm::kTile;
        unsigned char *ks = ring + st * Sm::kStage;
#pragma unroll
        for (int j = 0; j < PER_LANE; j++) {
            const int i = lane + 32 * j;
            const int r = i / CH, c = i - (i / CH) * CH;
            const int nb = r < valid ? 16 : 0;
            const int go = nb ? r * Sm::kRowBytes + c * 16 : 0;
            pkv::cp_async16(ks + pkv::swz(r, c, Sm::kRowBytes), kc + base + go, nb);
            pkv::cp_async16(ks + Sm::kTile + pkv::swz(r, c, Sm::kRowBytes), vc + base + go, nb);
        }
    };

    float o[MT][4];
#pragma unroll
    for (int i = 0; i < MT; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // running max and this thread's part of the sum, query rows 2 tig, 2 tig + 1
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

#pragma unroll
    for (int st = 0; st < Sm::kRing - 1; st++) {
        if (st < n) issue(st, st);
        pkv::cp_async_commit();
    }
    // ldmatrix row addresses: K as A (matrix j = lane / 8: tokens 8 (j & 1) ..,
    // column chunk 2 kk + j / 2), V as A of V^T (tokens 8 (j / 2) .., column
    // chunk 2 mt + (j & 1))
    const int ktok = ((lane >> 3) & 1) * 8 + (lane & 7), kch = lane >> 4;
    const int vtok = (lane >> 4) * 8 + (lane & 7), vch = (lane >> 3) & 1;
    for (int i = 0; i < n; i++) {
        {
            const int nx = i + Sm::kRing - 1;
            if (nx < n) issue(nx, nx % Sm::kRing);
            pkv::cp_async_commit();
        }
        pkv::cp_async_wait<Sm::kRing - 1>();
        __syncwarp();
        const unsigned char *ks = ring + (i % Sm::kRing) * Sm::kStage;
        const unsigned char *vs = ks + Sm::kTile;
        int phys;
        int valid = block_rows(i, phys);
        if (valid < 0) valid = 0;

        // S^T: c[0], c[1] token gid, rows 2 tig, 2 tig + 1; c[2], c[3] token gid + 8
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < KSTEPS; kk++) {
            uint32_t a[4];
            pkv::ldsm_x4(a[0], a[1], a[2], a[3], ks + pkv::swz(ktok, 2 * kk + kch, Sm::kRowBytes));
            pkv::mma_bf16(c, a, qb[kk][0], qb[kk][1]);
        }
        const float x0 = gid < valid ? c[0] * sl2 : -INFINITY;
        const float x1 = gid < valid ? c[1] * sl2 : -INFINITY;
        const float x2 = gid + 8 < valid ? c[2] * sl2 : -INFINITY;
        const float x3 = gid + 8 < valid ? c[3] * sl2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // the running maximum moves only when a row's scores pass it by more
        // than 2^8; P <= 256 then, and O, l are rescaled rarely
        if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float al0 = pkv::fast_exp2(m0 - (n0 == -INFINITY ? 0.f : n0));
            const float al1 = pkv::fast_exp2(m1 - (n1 == -INFINITY ? 0.f : n1));
            m0 = n0;
            m1 = n1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int mt = 0; mt < MT; mt++) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
        }
        const float base0 = m0 == -INFINITY ? 0.f : m0, base1 = m1 == -INFINITY ? 0.f : m1;
        const float p0 = pkv::fast_exp2(x0 - base0), p1 = pkv::fast_exp2(x1 - base1);
        const float p2 = pkv::fast_exp2(x2 - base0), p3 = pkv::fast_exp2(x3 - base1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // P^T as B fragments (hi and lo halves): {P[row gid][token 2 tig],
        // [2 tig + 1]} and the same 8 tokens later
        float h0f, h1f, h2f, h3f, q0, q1, q2, q3;
        pkv::split_bf16(p0, h0f, q0);
        pkv::split_bf16(p1, h1f, q1);
        pkv::split_bf16(p2, h2f, q2);
        pkv::split_bf16(p3, h3f, q3);
        const uint32_t ph0 = transpose8x8_b16(pkv::pack_bf16(h0f, h1f));
        const uint32_t ph1 = transpose8x8_b16(pkv::pack_bf16(h2f, h3f));
        const uint32_t pl0 = transpose8x8_b16(pkv::pack_bf16(q0, q1));
        const uint32_t pl1 = transpose8x8_b16(pkv::pack_bf16(q2, q3));

        // O^T += V^T P^T: m-tile mt is d = 16 mt .. 16 mt + 15
#pragma unroll
        for (int mt = 0; mt < MT; mt++) {
            uint32_t a[4];
            pkv::ldsm_x4_t(a[0], a[1], a[2], a[3], vs + pkv::swz(vtok, 2 * mt + vch, Sm::kRowBytes));
            pkv::mma_bf16(o[mt], a, ph0, ph1);
            pkv::mma_bf16(o[mt], a, pl0, pl1);
        }
        __syncwarp();
    }
    pkv::cp_async_wait<0>();
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }

    // stage the warp's state in shared memory: O rows [8][D] (o[mt][2h + e]
    // is row 2 tig + e, column 16 mt + gid + 8 h), then m[8], l[8]
    if (!kHeadWarps) __syncthreads();  // every warp is done with its ring
    float *sw = reinterpret_cast<float *>(kHeadWarps ? ring : smem) + (kHeadWarps ? 0 : warp * Sm::kStateWarp);
    __syncwarp();
#pragma unroll
    for (int mt = 0; mt < MT; mt++)
#pragma unroll
        for (int h = 0; h < 2; h++)
#pragma unroll
            for (int e = 0; e < 2; e++) sw[(2 * tig + e) * Sm::kStride + 16 * mt + gid + 8 * h] = o[mt][2 * h + e];
    if (gid == 0) {
        sw[8 * Sm::kStride + 2 * tig] = m0;
        sw[8 * Sm::kStride + 2 * tig + 1] = m1;
        sw[8 * Sm::kStride + 8 + 2 * tig] = l0;
        sw[8 * Sm::kStride + 8 + 2 * tig + 1] = l1;
    }

    if (kHeadWarps) {
        __syncwarp();
        // lane: 4 consecutive columns of a row per pass
        for (int idx = lane; idx < rows * (D / 4); idx += 32) {
            const int r = idx / (D / 4), c = (idx - r * (D / 4)) * 4;
            const float4 v = *reinterpret_cast<const float4 *>(sw + r * Sm::kStride + c);
            const float m = sw[8 * Sm::kStride + r], l = sw[8 * Sm::kStride + 8 + r];
            const size_t orow = (size_t)s * p.num_q_heads + h0 + r;
            if (nslots == 1) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                OutT *op = static_cast<OutT *>(p.out) + orow * D + c;
                pkv::store2(op, v.x * inv, v.y * inv);
                pkv::store2(op + 2, v.z * inv, v.w * inv);
            } else {
                const size_t prow = orow * p.max_parts + slot0 + part;
                *reinterpret_cast<float4 *>(p.part_o + prow * D + c) = v;
                if (c == 0) *reinterpret_cast<float2 *>(p.part_ml + prow * 2) = make_float2(m, l);
            }
        }
        if (tail_wait) pkv::grid_dependency_wait();
        return;
    }

    __syncthreads();
    const float *base = reinterpret_cast<const float *>(smem);
    for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
        const int r = idx / D, col = idx - (idx / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; w++) M = fmaxf(M, base[w * Sm::kStateWarp + 8 * Sm::kStride + r]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; w++) {
                const float *bw = base + w * Sm::kStateWarp;
                const float f = pkv::fast_exp2(bw[8 * Sm::kStride + r] - M);
                lsum += bw[8 * Sm::kStride + 8 + r] * f;
                acc += bw[r * Sm::kStride + col] * f;
            }
        }
        const size_t orow = (size_t)s * p.num_q_heads + h0 + r;
        if (nslots == 1) {
            pkv::store1(static_cast<OutT *>(p.out) + orow * D + col, lsum > 0.f ? acc / lsum : 0.f);
        } else {
            const size_t prow = orow * p.max_parts + slot0 + part;
            p.part_o[prow * D + col] = acc;
            if (col == 0) {
                p.part_ml[prow * 2] = M;
                p.part_ml[prow * 2 + 1] = lsum;
            }
        }
    }
    if (tail_wait) pkv::grid_dependency_wait();
}

// ----------------------------------------------------------------------------
// fp8 decode with the operands swapped
// ----------------------------------------------------------------------------
// The scores are computed transposed, S^T = K q^T, and the output as
// O^T = V^T P^T: the 16 tokens of a block are the M side of each
// m16n8k16 product and the unit's (at most) 8 query rows its N side.  With
// 4 or 8 query heads per kv head this wastes at most half of each product
// (the layout with queries on the M side wastes 12 of 16 rows for 4), so a
// block takes half the tensor-core products, half the exponentials and half
// the accumulator registers, and four thread blocks (16 warps) fit per SM.
// The codes still reach the fragments as whole 4-byte words, widened to
// fp16 in registers:
//  - S^T: in k-step kk, fragment columns {2 tig, 2 tig + 1} take
//    d = 32 tig + 4 kk + {0, 1} and {2 tig + 8, 2 tig + 9} take + {2, 3}
//    (the query is read in the same order), so thread (gid, tig) reads the
//    32-byte run [32 tig, 32 tig + 32) of tokens gid and gid + 8;
//  - O^T: accumulator row (mt, gid + 8 h) of m-tile mt is d = 16 gid +
//    2 mt + h, so the thread reads the 16 bytes [16 gid, 16 gid + 16) of
//    tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9 and ends holding 16
//    consecutive output columns of query rows 2 tig and 2 tig + 1;
//  - P^T reaches the B fragments through one 8x8 transpose (movmatrix) per
//    8 tokens of the score accumulator.

struct Fp8Smem {
    static constexpr int kRing = 3;                        // blocks per warp ring
    static constexpr int kRowBytes = 128;                  // one cached row (d = 128 codes)
    static constexpr int kTile = kBlock * kRowBytes;       // one block of one kv head
    static constexpr int kStage = 2 * kTile;               // K + V
    static constexpr int kWarp = kRing * kStage;
    static constexpr int kStaging = kWarps * kWarp;
    static constexpr int kMergeStride = 128 + 4;           // floats per merged row
    static constexpr int kMergeWarp = kRows8 * kMergeStride + 2 * kRows8;
    static constexpr int kMerge = kWarps * kMergeWarp * 4;
    static constexpr int kBytes = kStaging > kMerge ? kStaging : kMerge;
};

template <typename OutT, bool kHeadWarps>
__global__ void __launch_bounds__(kThreads, 4) decode_fp8_kernel(const DecodeParams p) {
    using Sm = Fp8Smem;
    constexpr int D = 128, KSTEPS = 8, MT = 8;
    constexpr int PER_LANE = kBlock * (Sm::kRowBytes / 16) / 32;

    extern __shared__ __align__(128) unsigned char smem[];
    pkv::allow_dependents();
    pkv::grid_dependency_wait();  // the rows the previous launch appended
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gid = lane >> 2, tig = lane & 3;
    const int unit = kHeadWarps ? blockIdx.x * kWarps + warp : blockIdx.x;
    const bool idle = kHeadWarps && unit >= p.num_kv_heads * p.head_chunks;
    const int kvh = unit / p.head_chunks, chunk = unit - kvh * p.head_chunks;
    const int s = blockIdx.y, part = blockIdx.z;
    const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;
    const int blk_begin = part * p.partition / kBlock;
    // the warp's blocks (a head warp: all of the partition; a split warp:
    // every fourth); the first 32 block ids come with one coalesced load
    const int bstride = kHeadWarps ? 1 : kWarps;
    const int bfirst = blk_begin + (kHeadWarps ? 0 : warp);
    int my_id = 0;
    if (!idle && bfirst + bstride * lane < p.max_blocks) my_id = table[bfirst + bstride * lane];

    const int L = clamp_len(p.context_lens[s], p.len_cap, p.status,
                            part == 0 && blockIdx.x == 0 && threadIdx.x == 0);
    const int nparts = own_parts(p, L);
    if (part >= nparts || idle) return;

    const int h0 = kvh * p.group + chunk * kRows8;
    const int rows = min(kRows8, p.group - chunk * kRows8);
    const int t_end = min(L, (part + 1) * p.partition);
    const int nblk = (t_end + kBlock - 1) / kBlock - blk_begin;
    const int n = kHeadWarps ? nblk : max(0, (nblk - warp + kWarps - 1) / kWarps);
    const unsigned char *kc = static_cast<const unsigned char *>(p.k_cache);
    const unsigned char *vc = static_cast<const unsigned char *>(p.v_cache);

    // q^T as B fragments (query row gid of the unit, zero past `rows`), d
    // in the order the K codes are read
    uint32_t qb[KSTEPS][2];
    {
        const bool ok = gid < rows;
        const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(p.q) +
                                    ((size_t)s * p.num_q_heads + h0 + (ok ? gid : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; kk++) {
            const uint2 r = ok ? *reinterpret_cast<const uint2 *>(qrow + 32 * tig + 4 * kk) : make_uint2(0u, 0u);
            const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&r.x);
            const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&r.y);
            qb[kk][0] = pkv::pack_f16(__low2float(lo), __high2float(lo));
            qb[kk][1] = pkv::pack_f16(__low2float(hi), __high2float(hi));
        }
    }
    // base-2 softmax scale times the kv head's K scale; the V scale
    const float sl2 = p.scale_log2 * p.k_scale[kvh];
    const float vsc = p.v_scale[kvh];

    if (p.k_new && part == nparts - 1 && L > 0) {
        // the new row is read below through L2 by other threads
        if (kHeadWarps) {
            // (warps of other chunks of the same kv head write the same bytes)
            append_new_token_fp8(p, table, s, kvh, L, lane, 32);
            __syncwarp();
        } else {
            append_new_token_fp8(p, table, s, kvh, L, threadIdx.x, kThreads);
            __syncthreads();
        }
    }

    unsigned char *ring = smem + warp * Sm::kWarp;
    auto block_id = [&](int li) -> int {
        return li < 32 ? __shfl_sync(0xffffffffu, my_id, li) : table[bfirst + bstride * li];
    };
    // rows of the warp's li-th block that hold tokens of this partition (-1 for a bad id)
    auto block_rows = [&](int li, int &phys) -> int {
        phys = block_id(li);
        if (phys < 0 || phys >= p.num_blocks) return -1;
        return min(kBlock, t_end - (bfirst + bstride * li) * kBlock);
    };
    // copies of the li-th block into stage st, rows past the keys zeroed
    auto issue = [&](int li, int st) {
        int phys;
        int valid = block_rows(li, phys);
        if (valid < 0) {
            if (lane == 0) pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
            valid = 0;
            phys = 0;
        }
        const size_t base = ((size_t)phys * p.num_kv_heads + kvh) * Sm::kTile;
        unsigned char *ks = ring + st * Sm::kStage;
#pragma unroll
        for (int j = 0; j < PER_LANE; j++) {
            const int i = lane + 32 * j;
            const int r = i >> 3, c = i & 7;
            const int nb = r < valid ? 16 : 0;
            const int go = nb ? r * Sm::kRowBytes + c * 16 : 0;
            pkv::cp_async16(ks + pkv::swz(r, c, Sm::kRowBytes), kc + base + go, nb);
            pkv::cp_async16(ks + Sm::kTile + pkv::swz(r, c, Sm::kRowBytes), vc + base + go, nb);
        }
    };

    float o[MT][4];
#pragma unroll
    for (int i = 0; i < MT; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // running max and (this thread's part of the) sum of query rows 2 tig, 2 tig + 1
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

#pragma unroll
    for (int st = 0; st < Sm::kRing - 1; st++) {
        if (st < n) issue(st, st);
        pkv::cp_async_commit();
    }
    for (int i = 0; i < n; i++) {
        {
            const int nx = i + Sm::kRing - 1;
            if (nx < n) issue(nx, nx % Sm::kRing);
            pkv::cp_async_commit();
        }
        pkv::cp_async_wait<Sm::kRing - 1>();
        __syncwarp();
        const unsigned char *ks = ring + (i % Sm::kRing) * Sm::kStage;
        const unsigned char *vs = ks + Sm::kTile;
        int phys;
        int valid = block_rows(i, phys);
        if (valid < 0) valid = 0;

        // S^T for the block: tokens gid and gid + 8 (codes d = 32 tig ..)
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint4 a0 = *reinterpret_cast<const uint4 *>(ks + pkv::swz(gid, 2 * tig, Sm::kRowBytes));
            const uint4 a1 = *reinterpret_cast<const uint4 *>(ks + pkv::swz(gid, 2 * tig + 1, Sm::kRowBytes));
            const uint4 b0 = *reinterpret_cast<const uint4 *>(ks + pkv::swz(gid + 8, 2 * tig, Sm::kRowBytes));
            const uint4 b1 = *reinterpret_cast<const uint4 *>(ks + pkv::swz(gid + 8, 2 * tig + 1, Sm::kRowBytes));
            const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int kk = 0; kk < KSTEPS; kk++) {
                const uint32_t af[4] = {pkv::e4m3x2_to_f16x2((uint16_t)(wa[kk] & 0xffffu)),
                                        pkv::e4m3x2_to_f16x2((uint16_t)(wb[kk] & 0xffffu)),
                                        pkv::e4m3x2_to_f16x2((uint16_t)(wa[kk] >> 16)),
                                        pkv::e4m3x2_to_f16x2((uint16_t)(wb[kk] >> 16))};
                pkv::mma_f16(c, af, qb[kk][0], qb[kk][1]);
            }
        }
        // base-2 units, tokens past the keys masked; c[0], c[1]: token gid,
        // rows 2 tig, 2 tig + 1; c[2], c[3]: token gid + 8
        const float x0 = gid < valid ? c[0] * sl2 : -INFINITY;
        const float x1 = gid < valid ? c[1] * sl2 : -INFINITY;
        const float x2 = gid + 8 < valid ? c[2] * sl2 : -INFINITY;
        const float x3 = gid + 8 < valid ? c[3] * sl2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // the running maximum moves only when a row's scores pass it by more
        // than 2^8, so P <= 256 (exact enough in fp16) and O, l are rescaled rarely
        if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float al0 = pkv::fast_exp2(m0 - (n0 == -INFINITY ? 0.f : n0));
            const float al1 = pkv::fast_exp2(m1 - (n1 == -INFINITY ? 0.f : n1));
            m0 = n0;
            m1 = n1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int mt = 0; mt < MT; mt++) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
        }
        const float base0 = m0 == -INFINITY ? 0.f : m0, base1 = m1 == -INFINITY ? 0.f : m1;
        const float p0 = pkv::fast_exp2(x0 - base0), p1 = pkv::fast_exp2(x1 - base1);
        const float p2 = pkv::fast_exp2(x2 - base0), p3 = pkv::fast_exp2(x3 - base1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // P^T as B fragments: {P[row gid][token 2 tig], [2 tig + 1]} and + 8
        const uint32_t pb0 = transpose8x8_b16(pkv::pack_f16(p0, p1));
        const uint32_t pb1 = transpose8x8_b16(pkv::pack_f16(p2, p3));

        // O^T += V^T P^T: tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9, codes
        // d = 16 gid .. 16 gid + 15
        const int t0 = 2 * tig;
        const uint4 v0 = *reinterpret_cast<const uint4 *>(vs + pkv::swz(t0, gid, Sm::kRowBytes));
        const uint4 v1 = *reinterpret_cast<const uint4 *>(vs + pkv::swz(t0 + 1, gid, Sm::kRowBytes));
        const uint4 v2 = *reinterpret_cast<const uint4 *>(vs + pkv::swz(t0 + 8, gid, Sm::kRowBytes));
        const uint4 v3 = *reinterpret_cast<const uint4 *>(vs + pkv::swz(t0 + 9, gid, Sm::kRowBytes));
        const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
        const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w}, w3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
        for (int mt = 0; mt < MT; mt++) {
            // bytes 2 mt, 2 mt + 1 of each row: (token, token + 1) code pairs
            const unsigned sel = (mt & 1) ? 0x7362u : 0x5140u;
            const uint32_t lo = __byte_perm(w0[mt >> 1], w1[mt >> 1], sel);
            const uint32_t hi = __byte_perm(w2[mt >> 1], w3[mt >> 1], sel);
            const uint32_t af[4] = {pkv::e4m3x2_to_f16x2((uint16_t)(lo & 0xffffu)),
                                    pkv::e4m3x2_to_f16x2((uint16_t)(lo >> 16)),
                                    pkv::e4m3x2_to_f16x2((uint16_t)(hi & 0xffffu)),
                                    pkv::e4m3x2_to_f16x2((uint16_t)(hi >> 16))};
            pkv::mma_f16(o[mt], af, pb0, pb1);
        }
        __syncwarp();
    }
    pkv::cp_async_wait<0>();

    // the row sums over all 32 lanes' tokens
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const int nslots = nparts;
    // this thread's values of query row 2 tig + e, columns 16 gid + j
    auto val = [&](int j, int e) -> float { return o[j >> 1][2 * (j & 1) + e]; };

    if (kHeadWarps) {
#pragma unroll
        for (int e = 0; e < 2; e++) {
            const int r = 2 * tig + e;
            if (r >= rows) continue;
            const float m = e ? m1 : m0, l = e ? l1 : l0;
            const size_t orow = (size_t)s * p.num_q_heads + h0 + r;
            if (nslots == 1) {
                OutT *op = static_cast<OutT *>(p.out) + orow * D + 16 * gid;
                const float inv = l > 0.f ? vsc / l : 0.f;
#pragma unroll
                for (int j = 0; j < 16; j += 2) pkv::store2(op + j, val(j, e) * inv, val(j + 1, e) * inv);
            } else {
                const size_t prow = orow * p.max_parts + part;
                float *po = p.part_o + prow * D + 16 * gid;
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4 *>(po + j) =
                        make_float4(val(j, e) * vsc, val(j + 1, e) * vsc, val(j + 2, e) * vsc, val(j + 3, e) * vsc);
                if (gid == 0) *reinterpret_cast<float2 *>(p.part_ml + prow * 2) = make_float2(m, l);
            }
        }
        return;
    }

    __syncthreads();  // every warp is done with its ring; reuse it for the merge
    float *mw = reinterpret_cast<float *>(smem) + warp * Sm::kMergeWarp;
    float *mm = mw + kRows8 * Sm::kMergeStride;
    float *ll = mm + kRows8;
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int r = 2 * tig + e;
        if (gid == 0) {
            mm[r] = e ? m1 : m0;
            ll[r] = e ? l1 : l0;
        }
#pragma unroll
        for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4 *>(mw + r * Sm::kMergeStride + 16 * gid + j) =
                make_float4(val(j, e), val(j + 1, e), val(j + 2, e), val(j + 3, e));
    }
    __syncthreads();

    const float *base = reinterpret_cast<const float *>(smem);
    for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
        const int r = idx / D, col = idx - (idx / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; w++) M = fmaxf(M, base[w * Sm::kMergeWarp + kRows8 * Sm::kMergeStride + r]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; w++) {
                const float *bw = base + w * Sm::kMergeWarp;
                const float f = pkv::fast_exp2(bw[kRows8 * Sm::kMergeStride + r] - M);
                lsum += bw[kRows8 * Sm::kMergeStride + kRows8 + r] * f;
                acc += bw[r * Sm::kMergeStride + col] * f;
            }
        }
        const size_t orow = (size_t)s * p.num_q_heads + h0 + r;
        if (nslots == 1) {
            pkv::store1(static_cast<OutT *>(p.out) + orow * D + col, lsum > 0.f ? acc * vsc / lsum : 0.f);
        } else {
            const size_t prow = orow * p.max_parts + part;
            p.part_o[prow * D + col] = acc * vsc;
            if (col == 0) {
                p.part_ml[prow * 2] = M;
                p.part_ml[prow * 2 + 1] = lsum;
            }
        }
    }
}

// ----------------------------------------------------------------------------
// CUDA-core decode for fp32 caches (and any head group): one CTA per
// (q head, sequence, partition), one token per thread per pass of 128 tokens,
// two-pass softmax within the pass and online rescaling across passes.
// ----------------------------------------------------------------------------

template <typename T>
__device__ __forceinline__ float ld_elem(const T *p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float *p) { return *p; }

__device__ __forceinline__ float block_reduce(float v, float *red, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, off);
        v = is_max ? fmaxf(v, u) : v + u;
    }
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; w++) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

// Attention of one query row over tokens [t_begin, t_end) of one sequence.
// Returns (m, l) and leaves this thread's output column (tid < D) in `acc`.
template <typename T>
__device__ void rows_cuda_core(const T *qrow, const T *kc, const T *vc, const int32_t *table,
                               int t_begin, int t_end, int num_blocks, int num_kv_heads, int kvh,
                               int D, float scale_log2, unsigned *status, float *sq, float *sp,
                               int *sb, float *red, float &m, float &l, float &acc) {
    const int tid = threadIdx.x;
    for (int c = tid; c < D; c += kThreads) sq[c] = ld_elem(qrow + c);
    m = -INFINITY;
    l = 0.f;
    acc = 0.f;
    __syncthreads();
    for (int t0 = t_begin; t0 < t_end; t0 += kThreads) {
        const int t = t0 + tid;
        float x = -INFINITY;
        int phys = -1;
        if (t < t_end) {
            phys = table[t / kBlock];
            if (phys < 0 || phys >= num_blocks) {
                pkv::flag(status, PKV_STATUS_BAD_BLOCK);
                phys = -1;
            } else {
                const T *kr = kc + (((size_t)phys * num_kv_heads + kvh) * kBlock + t % kBlock) * D;
                float dot = 0.f;
                for (int c = 0; c < D; c++) dot = fmaf(sq[c], ld_elem(kr + c), dot);
                x = dot * scale_log2;
            }
        }
        const float cmax = block_reduce(x, red, true);
        const float mn = fmaxf(m, cmax);
        const float base = mn == -INFINITY ? 0.f : mn;
        const float alpha = pkv::fast_exp2(m - base);
        const float pt = pkv::fast_exp2(x - base);
        sp[tid] = pt;
        sb[tid] = phys;
        const float psum = block_reduce(pt, red, false);  // also orders sp/sb writes
        l = l * alpha + psum;
        m = mn;
        acc *= alpha;
        const int cnt = min(kThreads, t_end - t0);
        if (tid < D) {
            for (int i = 0; i < cnt; i++) {
                if (sb[i] < 0) continue;
                const int t2 = t0 + i;
                const T *vr = vc + (((size_t)sb[i] * num_kv_heads + kvh) * kBlock + t2 % kBlock) * D;
                acc = fmaf(sp[i], ld_elem(vr + tid), acc);
            }
        }
        __syncthreads();
    }
}

template <typename T, typename OutT>
__global__ void __launch_bounds__(kThreads) decode_cuda_core_kernel(const DecodeParams p, int D) {
    __shared__ float sq[128];
    __shared__ float sp[kThreads];
    __shared__ int sb[kThreads];
    __shared__ float red[kWarps];
    const int h = blockIdx.x, s = blockIdx.y, part = blockIdx.z;
    const int L = clamp_len(p.context_lens[s], p.len_cap, p.status,
                            part == 0 && h == 0 && threadIdx.x == 0);
    const int nparts = own_parts(p, L);
    if (part >= nparts) return;
    const int slot0 = p.prefix_len ? 1 : 0;
    const int nslots = slot0 + nparts;
    const int kvh = h / p.group;
    if (p.k_new && part == nparts - 1 && L > 0) {
        // every q head of the group writes the same bytes for its kv head
        append_new_token<T>(p, p.block_tables + (size_t)s * p.max_blocks, s, kvh, L, D, threadIdx.x, blockDim.x);
        __syncthreads();
    }
    const T *qrow = static_cast<const T *>(p.q) + ((size_t)s * p.num_q_heads + h) * D;
    float m, l, acc;
    rows_cuda_core<T>(qrow, static_cast<const T *>(p.k_cache), static_cast<const T *>(p.v_cache),
                      p.block_tables + (size_t)s * p.max_blocks, p.prefix_len + part * p.partition,
                      min(L, p.prefix_len + (part + 1) * p.partition), p.num_blocks, p.num_kv_heads, kvh, D,
                      p.scale_log2, p.status, sq, sp, sb, red, m, l, acc);
    const int c = threadIdx.x;
    if (c >= D) return;
    const size_t orow = (size_t)s * p.num_q_heads + h;
    if (nslots == 1) {
        pkv::store1(static_cast<OutT *>(p.out) + orow * D + c, l > 0.f ? acc / l : 0.f);
    } else {
        const size_t prow = orow * p.max_parts + slot0 + part;
        p.part_o[prow * D + c] = acc;
        if (c == 0) {
            p.part_ml[prow * 2] = m;
            p.part_ml[prow * 2 + 1] = l;
        }
    }
}

// ----------------------------------------------------------------------------
// log-sum-exp merge of the partitions of each (sequence, q head)
// ----------------------------------------------------------------------------

// One warp per (sequence, q head); each lane owns D/32 output columns.
// Rows of at most kEager partitions (the common case) issue every load at
// once: the slots' addresses do not depend on the length, so the length, the
// first kEager slots' (m, l) and this lane's columns of their O rows travel
// in one round trip, and the slots past the row's count are dropped
// afterwards.  Longer rows compute the weights 2^(m_p - M) lane-parallel,
// broadcast them by shuffles and keep four partitions' loads in flight.
template <int D, typename OutT>
__global__ void __launch_bounds__(128) decode_reduce_kernel(const DecodeParams p, int rows) {
    constexpr int VEC = D / 32;
    constexpr int kEager = 4;
    using VecT = typename std::conditional<VEC == 4, float4, float2>::type;
    pkv::grid_dependency_wait();  // the partials of the partition launch
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int s = row / p.num_q_heads;
    const size_t prow = (size_t)row * p.max_parts;
    const float *ml = p.part_ml + prow * 2;
    const float *po = p.part_o + prow * D + lane * VEC;

    const int Lraw = p.context_lens[s];
    const int eager = min(kEager, p.max_parts);  // slots inside this row's workspace
    float2 mle[kEager];
    float xe[kEager][VEC];
#pragma unroll
    for (int u = 0; u < kEager; u++) {
        if (u < eager) {
            mle[u] = *reinterpret_cast<const float2 *>(ml + 2 * u);
            const VecT w = *reinterpret_cast<const VecT *>(po + (size_t)u * D);
            const float *wf = reinterpret_cast<const float *>(&w);
#pragma unroll
            for (int v = 0; v < VEC; v++) xe[u][v] = wf[v];
        }
    }
    const int L = clamp_len(Lraw, p.len_cap, p.status, false);
    const int nparts = (p.prefix_len ? 1 : 0) + own_parts(p, L);  // partial slots of this row
    if (nparts <= 1) return;

    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; v++) acc[v] = 0.f;
    float lsum = 0.f;
    if (nparts <= kEager) {
        float M = -INFINITY;
#pragma unroll
        for (int u = 0; u < kEager; u++)
            if (u < nparts) M = fmaxf(M, mle[u].x);
        if (M != -INFINITY) {
#pragma unroll
            for (int u = 0; u < kEager; u++) {
                if (u < nparts) {
                    const float w = pkv::fast_exp2(mle[u].x - M);
                    lsum += mle[u].y * w;
#pragma unroll
                    for (int v = 0; v < VEC; v++) acc[v] = fmaf(w, xe[u][v], acc[v]);
                }
            }
        }
    } else {
        float M = -INFINITY;
        for (int q = lane; q < nparts; q += 32) M = fmaxf(M, ml[2 * q]);
#pragma unroll
        for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        if (M != -INFINITY) {
            for (int q0 = 0; q0 < nparts; q0 += 32) {
                const int cnt = min(32, nparts - q0);
                float w = 0.f;
                if (lane < cnt) {
                    w = pkv::fast_exp2(ml[2 * (q0 + lane)] - M);
                    lsum += ml[2 * (q0 + lane) + 1] * w;
                }
                int j = 0;
                for (; j + 4 <= cnt; j += 4) {
                    float x[4][VEC];
#pragma unroll
                    for (int u = 0; u < 4; u++) {
#pragma unroll
                        for (int v = 0; v < VEC; v++) x[u][v] = po[(size_t)(q0 + j + u) * D + v];
                    }
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const float wj = __shfl_sync(0xffffffffu, w, j + u);
#pragma unroll
                        for (int v = 0; v < VEC; v++) acc[v] = fmaf(wj, x[u][v], acc[v]);
                    }
                }
                for (; j < cnt; j++) {
                    const float wj = __shfl_sync(0xffffffffu, w, j);
#pragma unroll
                    for (int v = 0; v < VEC; v++) acc[v] = fmaf(wj, po[(size_t)(q0 + j) * D + v], acc[v]);
                }
            }
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    OutT *o = static_cast<OutT *>(p.out) + (size_t)row * D + lane * VEC;
#pragma unroll
    for (int v = 0; v < VEC; v += 2) pkv::store2(o + v, acc[v] * inv, acc[v + 1] * inv);
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t workspace_for(int num_seqs, int num_q_heads, int head_dim, int max_parts) {
    if (max_parts <= 1) return 0;
    const size_t rows = (size_t)num_seqs * num_q_heads * max_parts;
    return align256(rows * head_dim * sizeof(float)) + align256(rows * 2 * sizeof(float));
}

int resolve_partition(int partition_size, int *out) {
    if (partition_size == 0) partition_size = PKV_DEFAULT_PARTITION;
    if (partition_size < kBlock || partition_size % kBlock != 0)
        return pkv::fail(PKV_ERR_INVALID, "partition_size must be a positive multiple of 16 (got %d)",
                         partition_size);
    *out = partition_size;
    return PKV_OK;
}

// partition_size 0: the largest of 3072, 2048, 1536, 1024 tokens that still
// leaves an estimated 4 work units per SM, else 512.  The host knows only the
// largest context, so a sequence is assumed to hold half of it.  Larger
// partitions amortise each thread block's start-up and cut the split-K
// partials; enough units keep every SM streaming.
// SM count of the current device (148 when there is none to ask)
// (cached per device; host threads that race here store the same count)
int device_sms() {
    static std::atomic<int> sm_count[64];
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        int n = sm_count[dev].load(std::memory_order_relaxed);
        if (n <= 0 && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
            sm_count[dev].store(n, std::memory_order_relaxed);
        if (n > 0) sms = n;
    }
    cudaGetLastError();
    return sms;
}

int adaptive_partition(int num_seqs, int num_kv_heads, int max_context_len) {
    const long long target = 4LL * device_sms();
    const int candidates[] = {3072, 2048, 1536, 1024};
    for (int c : candidates) {
        const long long per_seq = max(1, (max_context_len + 2 * c - 1) / (2 * c));
        if ((long long)num_seqs * num_kv_heads * per_seq >= target) return c;
    }
    return PKV_DEFAULT_PARTITION;
}

// The fp8 kernel's choice: when the (sequence, unit) pairs fill between two
// and four of its thread blocks per SM and no context exceeds
// kFp8UnsplitTokens, a sequence is not split at all: one resident wave
// covers the batch, and the partials and the merge launch cost more than the
// uneven lengths do.  (Longer contexts make a thread block's work, and the
// spread between the longest and the rest, large against the merge.)
// Otherwise as adaptive_partition.
constexpr int kFp8UnsplitTokens = 8192;

int fp8_partition(int num_seqs, int units_per_seq, int num_kv_heads, int max_context_len) {
    const long long units = (long long)num_seqs * units_per_seq, sms = device_sms();
    if (units >= 2 * sms && units <= 4 * sms && max_context_len > 0 && max_context_len <= kFp8UnsplitTokens)
        return (max_context_len + kBlock - 1) / kBlock * kBlock;
    return adaptive_partition(num_seqs, num_kv_heads, max_context_len);
}

// Head warps when a partition spans at most this many tokens (split four
// ways it would give each warp at most 8 blocks, too few to amortise the
// block's start: length, block ids, first copies, merge), provided the
// launch still has two thread blocks per SM: a head-warp block covers four
// (kv head, chunk) units, so it cuts the block count fourfold.
constexpr int kHeadWarpTokens = 512;

// own_max: the most tokens one launch covers for a sequence (the context
// minus any shared prefix); units: kv heads x head chunks.
bool use_head_warps(int num_seqs, int units, int own_max, int partition) {
    if ((own_max < partition ? own_max : partition) > kHeadWarpTokens) return false;
    const long long parts = own_max > 0 ? (own_max + partition - 1) / partition : 1;
    return (long long)num_seqs * ((units + kWarps - 1) / kWarps) * parts >= 2LL * device_sms();
}

template <int D, typename OutT, bool kHeadWarps>
int launch_bf16_variant(const DecodeParams &p, int num_seqs, cudaStream_t st) {
    constexpr int bytes = DecodeSmem<D>::kBytes;
    // set once per device (setting it twice from racing host threads is harmless)
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        // two thread blocks per SM: the largest shared-memory carve-out
        if (cudaFuncSetAttribute(decode_bf16_kernel<D, OutT, kHeadWarps>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
            cudaFuncSetAttribute(decode_bf16_kernel<D, OutT, kHeadWarps>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return pkv::check_launch("decode: set shared memory size");
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int units = p.num_kv_heads * p.head_chunks;
    // (with a shared prefix, partial slot 0 comes from another kernel)
    dim3 grid((unsigned)(kHeadWarps ? (units + kWarps - 1) / kWarps : units), (unsigned)num_seqs,
              (unsigned)(p.max_parts - (p.prefix_len ? 1 : 0)));
    cudaError_t e =
        pkv::launch_dependent(decode_bf16_kernel<D, OutT, kHeadWarps>, grid, dim3(kThreads), bytes, st, p);
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "decode_bf16: %s", cudaGetErrorString(e));
    return pkv::check_launch("decode_bf16");
}

template <int D, typename OutT, bool kHeadWarps>
int launch_bf16t_variant(const DecodeParams &p, int num_seqs, cudaStream_t st) {
    constexpr int bytes = DecodeTSmem<D>::kBytes;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(decode_bf16t_kernel<D, OutT, kHeadWarps>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
            cudaFuncSetAttribute(decode_bf16t_kernel<D, OutT, kHeadWarps>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return pkv::check_launch("decode: set shared memory size");
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int units = p.num_kv_heads * p.head_chunks;
    // (with a shared prefix, partial slot 0 comes from another kernel)
    dim3 grid((unsigned)(kHeadWarps ? (units + kWarps - 1) / kWarps : units), (unsigned)num_seqs,
              (unsigned)(p.max_parts - (p.prefix_len ? 1 : 0)));
    cudaError_t e =
        pkv::launch_dependent(decode_bf16t_kernel<D, OutT, kHeadWarps>, grid, dim3(kThreads), bytes, st, p);
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "decode_bf16t: %s", cudaGetErrorString(e));
    return pkv::check_launch("decode_bf16t");
}

// Query groups of at most 8 heads per kv head (one unit of 8 rows) take the
// transposed kernel, larger groups the one with the queries on the M side.
template <int D, typename OutT>
int launch_bf16(const DecodeParams &p, int num_seqs, cudaStream_t st) {
    if (p.group <= kRows8)
        return p.head_warps ? launch_bf16t_variant<D, OutT, true>(p, num_seqs, st)
                            : launch_bf16t_variant<D, OutT, false>(p, num_seqs, st);
    return p.head_warps ? launch_bf16_variant<D, OutT, true>(p, num_seqs, st)
                        : launch_bf16_variant<D, OutT, false>(p, num_seqs, st);
}

template <typename OutT, bool kHeadWarps>
int launch_fp8_variant(const DecodeParams &p, int num_seqs, cudaStream_t st) {
    constexpr int bytes = Fp8Smem::kBytes;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        // four thread blocks per SM: the largest shared-memory carve-out
        if (cudaFuncSetAttribute(decode_fp8_kernel<OutT, kHeadWarps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 bytes) != cudaSuccess ||
            cudaFuncSetAttribute(decode_fp8_kernel<OutT, kHeadWarps>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return pkv::check_launch("decode_fp8: set shared memory size");
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int units = p.num_kv_heads * p.head_chunks;
    dim3 grid((unsigned)(kHeadWarps ? (units + kWarps - 1) / kWarps : units), (unsigned)num_seqs,
              (unsigned)p.max_parts);
    cudaError_t e = pkv::launch_dependent(decode_fp8_kernel<OutT, kHeadWarps>, grid, dim3(kThreads), bytes, st, p);
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "decode_fp8: %s", cudaGetErrorString(e));
    return pkv::check_launch("decode_fp8");
}

template <typename T, typename OutT>
int launch_core(const DecodeParams &p, int num_seqs, int D, cudaStream_t st) {
    dim3 grid((unsigned)p.num_q_heads, (unsigned)num_seqs, (unsigned)p.max_parts);
    decode_cuda_core_kernel<T, OutT><<<grid, kThreads, 0, st>>>(p, D);
    return pkv::check_launch("decode_cuda_core");
}

template <typename OutT>
int launch_decode(const DecodeParams &p, int num_seqs, int D, int dtype, cudaStream_t st) {
    int rc;
    if (dtype == PKV_BF16) {
        rc = D == 128 ? launch_bf16<128, OutT>(p, num_seqs, st) : launch_bf16<64, OutT>(p, num_seqs, st);
    } else if (dtype == PKV_FP8_E4M3) {
        rc = p.head_warps ? launch_fp8_variant<OutT, true>(p, num_seqs, st)
                          : launch_fp8_variant<OutT, false>(p, num_seqs, st);
    } else {
        rc = launch_core<float, OutT>(p, num_seqs, D, st);
    }
    if (rc || p.max_parts <= 1) return rc;
    const int rows = num_seqs * p.num_q_heads;
    const unsigned blocks = (unsigned)((rows + 3) / 4);
    cudaError_t e = D == 128 ? pkv::launch_dependent(decode_reduce_kernel<128, OutT>, dim3(blocks), dim3(128), 0,
                                                     st, p, rows)
                             : pkv::launch_dependent(decode_reduce_kernel<64, OutT>, dim3(blocks), dim3(128), 0,
                                                     st, p, rows);
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "decode_reduce: %s", cudaGetErrorString(e));
    return pkv::check_launch("decode_reduce");
}

}  // namespace

extern "C" int pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                          int max_context_len, int partition_size, size_t *bytes) {
    int part;
    int rc = resolve_partition(partition_size, &part);
    if (rc) return rc;
    if (!bytes || num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0 ||
        (head_dim != 64 && head_dim != 128))
        return pkv::fail(PKV_ERR_INVALID, "decode_workspace_bytes: bad argument");
    const int max_parts = max_context_len > 0 ? (max_context_len + part - 1) / part : 1;
    *bytes = workspace_for(num_seqs, num_q_heads, head_dim, max_parts);
    return PKV_OK;
}

extern "C" int pkv_decode_partition_size(int num_seqs, int num_kv_heads, int max_context_len,
                                         int partition_size, int *out) {
    int part;
    int rc = resolve_partition(partition_size, &part);
    if (rc) return rc;
    if (!out || num_seqs < 0 || num_kv_heads <= 0 || max_context_len < 0)
        return pkv::fail(PKV_ERR_INVALID, "decode_partition_size: bad argument");
    *out = partition_size == 0 ? adaptive_partition(num_seqs, num_kv_heads, max_context_len) : part;
    return PKV_OK;
}

extern "C" int pkv_decode_partition_size_fp8(int num_seqs, int num_q_heads, int num_kv_heads, int max_context_len,
                                             int partition_size, int *out) {
    int part;
    int rc = resolve_partition(partition_size, &part);
    if (rc) return rc;
    if (!out || num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        max_context_len < 0)
        return pkv::fail(PKV_ERR_INVALID, "decode_partition_size_fp8: bad argument");
    const int units = num_kv_heads * ((num_q_heads / num_kv_heads + kRows8 - 1) / kRows8);
    *out = partition_size == 0 ? fp8_partition(num_seqs, units, num_kv_heads, max_context_len) : part;
    return PKV_OK;
}

namespace {

int decode_impl(const void *q, const void *k_new, const void *v_new, const void *k_cache, const void *v_cache,
                const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                int max_context_len, int partition_size, float scale, void *out, int dtype, int out_dtype,
                void *workspace, size_t workspace_bytes, void *stream, const float *k_scale = nullptr,
                const float *v_scale = nullptr) {
    int part;
    int rc = resolve_partition(partition_size, &part);
    if (rc) return rc;
    if (block_size != kBlock) return pkv::fail(PKV_ERR_INVALID, "block_size must be 16 (got %d)", block_size);
    if (head_dim != 64 && head_dim != 128)
        return pkv::fail(PKV_ERR_INVALID, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (dtype != PKV_F32 && dtype != PKV_BF16 && dtype != PKV_FP8_E4M3)
        return pkv::fail(PKV_ERR_INVALID, "bad dtype %d", dtype);
    if (dtype == PKV_FP8_E4M3) {  // bf16 queries over an fp8 cache
        if (head_dim != 128) return pkv::fail(PKV_ERR_INVALID, "fp8 decode: head_dim must be 128");
        if (!k_scale || !v_scale) return pkv::fail(PKV_ERR_INVALID, "fp8 decode: null scales");
        // (the fused append of pkv_decode_step_fp8 takes bf16 rows)
    }
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "bad out_dtype %d", out_dtype);
    if (num_seqs < 0 || num_blocks < 0 || max_blocks_per_seq < 0 || max_context_len < 0)
        return pkv::fail(PKV_ERR_INVALID, "decode: negative size");
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return pkv::fail(PKV_ERR_INVALID, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                         num_q_heads, num_kv_heads);
    if (!(scale == scale)) return pkv::fail(PKV_ERR_INVALID, "decode: scale is NaN");
    if (num_seqs == 0) return PKV_OK;
    if (num_seqs > 65535) return pkv::fail(PKV_ERR_INVALID, "decode: at most 65535 sequences per call");
    if (partition_size == 0)
        part = dtype == PKV_FP8_E4M3
                   ? fp8_partition(num_seqs, num_kv_heads * ((num_q_heads / num_kv_heads + kRows8 - 1) / kRows8),
                                   num_kv_heads, max_context_len)
                   : adaptive_partition(num_seqs, num_kv_heads, max_context_len);
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return pkv::fail(PKV_ERR_INVALID, "decode: null pointer");
    if (!pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache) || !pkv::aligned16(out))
        return pkv::fail(PKV_ERR_INVALID, "decode: q, caches and out must be 16-byte aligned");

    DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    p.max_blocks = max_blocks_per_seq;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_q_heads / num_kv_heads;
    // query rows per unit: 16 for the bf16 kernel, 8 for the fp8 one
    const int unit_rows = dtype == PKV_FP8_E4M3 ? kRows8 : kRows;
    p.head_chunks = (p.group + unit_rows - 1) / unit_rows;
    p.num_blocks = num_blocks;
    const long long cap = (long long)max_blocks_per_seq * kBlock;
    p.len_cap = (int)(cap < max_context_len ? cap : max_context_len);
    p.partition = part;
    p.max_parts = p.len_cap > 0 ? (p.len_cap + part - 1) / part : 1;
    if (p.max_parts > 65535) return pkv::fail(PKV_ERR_INVALID, "decode: too many partitions");
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = pkv::status_ptr();
    p.k_new = k_new;
    p.v_new = v_new;
    p.head_warps = use_head_warps(num_seqs, num_kv_heads * p.head_chunks, p.len_cap, part);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    if ((k_new || v_new) && (!k_new || !v_new || !pkv::aligned16(k_new) || !pkv::aligned16(v_new)))
        return pkv::fail(PKV_ERR_INVALID, "decode_step: k_new and v_new must both be 16-byte aligned device pointers");

    const size_t need = workspace_for(num_seqs, num_q_heads, head_dim, p.max_parts);
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return pkv::fail(PKV_ERR_INVALID, "decode: workspace of %zu bytes needed, %zu given", need,
                             workspace_bytes);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return pkv::fail(PKV_ERR_INVALID, "decode: workspace must be 256-byte aligned");
        const size_t rows = (size_t)num_seqs * num_q_heads * p.max_parts;
        p.part_o = static_cast<float *>(workspace);
        p.part_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                              align256(rows * head_dim * sizeof(float)));
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return out_dtype == PKV_F32 ? launch_decode<float>(p, num_seqs, head_dim, dtype, st)
                                : launch_decode<__nv_bfloat16>(p, num_seqs, head_dim, dtype, st);
}

}  // namespace

extern "C" int pkv_paged_attention_decode(const void *q, const void *k_cache, const void *v_cache,
                                          const int32_t *block_tables, int max_blocks_per_seq,
                                          const int32_t *context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, int max_context_len,
                                          int partition_size, float scale, void *out, int dtype,
                                          int out_dtype, void *workspace, size_t workspace_bytes,
                                          void *stream) {
    return decode_impl(q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len,
                       partition_size, scale, out, dtype, out_dtype, workspace, workspace_bytes, stream);
}

extern "C" int pkv_paged_attention_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                              const float *k_scale, const float *v_scale,
                                              const int32_t *block_tables, int max_blocks_per_seq,
                                              const int32_t *context_lens, int num_seqs, int num_q_heads,
                                              int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                              int max_context_len, int partition_size, float scale, void *out,
                                              int out_dtype, void *workspace, size_t workspace_bytes,
                                              void *stream) {
    return decode_impl(q, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len,
                       partition_size, scale, out, PKV_FP8_E4M3, out_dtype, workspace, workspace_bytes, stream,
                       k_scale, v_scale);
}

extern "C" int pkv_decode_step_fp8(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                   void *v_cache, const float *k_scale, const float *v_scale,
                                   const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                   int num_blocks, int max_context_len, int partition_size, float scale, void *out,
                                   int out_dtype, void *workspace, size_t workspace_bytes, void *stream) {
    if (num_seqs > 0 && (!k_new || !v_new))
        return pkv::fail(PKV_ERR_INVALID, "decode_step_fp8: null k_new or v_new");
    return decode_impl(q, k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, partition_size,
                       scale, out, PKV_FP8_E4M3, out_dtype, workspace, workspace_bytes, stream, k_scale, v_scale);
}

extern "C" int pkv_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache,
                               void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               int max_context_len, int partition_size, float scale, void *out,
                               int dtype, int out_dtype, void *workspace, size_t workspace_bytes,
                               void *stream) {
    if (num_seqs > 0 && (!k_new || !v_new))
        return pkv::fail(PKV_ERR_INVALID, "decode_step: null k_new or v_new");
    return decode_impl(q, k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len,
                       partition_size, scale, out, dtype, out_dtype, workspace, workspace_bytes, stream);
}

// ----------------------------------------------------------------------------
// decode over a prefix shared by the whole batch (cascade)
// ----------------------------------------------------------------------------

namespace {

constexpr size_t kCounterBytes = 256;  // the prefix kernel's work-item counter

int shared_prefix_parts(int len_cap, int prefix_len, int partition) {
    const int suf = len_cap - prefix_len;
    return 1 + (suf > 0 ? (suf + partition - 1) / partition : 0);
}

}  // namespace

extern "C" int pkv_decode_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                                        int max_context_len, int prefix_len, int partition_size,
                                                        size_t *bytes) {
    int part;
    int rc = resolve_partition(partition_size, &part);
    if (rc) return rc;
    if (!bytes || num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0 || head_dim != 128 || prefix_len <= 0 ||
        prefix_len % kBlock != 0 || prefix_len > max_context_len)
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix_workspace_bytes: bad argument");
    // partition_size 0 may choose any adaptive size; 512 needs the most slots
    *bytes = workspace_for(num_seqs, num_q_heads, head_dim, shared_prefix_parts(max_context_len, prefix_len, part)) +
             kCounterBytes;
    return PKV_OK;
}

extern "C" int pkv_paged_attention_decode_shared_prefix(
    const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int num_blocks, int max_context_len, int prefix_len, int partition_size,
    float scale, void *out, int dtype, int out_dtype, void *workspace, size_t workspace_bytes, void *stream) {
    int part;
    int rc = resolve_partition(partition_size, &part);
    if (rc) return rc;
    if (block_size != kBlock) return pkv::fail(PKV_ERR_INVALID, "block_size must be 16 (got %d)", block_size);
    if (dtype != PKV_BF16 || head_dim != 128)
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: bf16 caches with head_dim 128 only");
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "bad out_dtype %d", out_dtype);
    if (num_seqs < 0 || num_blocks < 0 || max_blocks_per_seq < 0 || max_context_len < 0)
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: negative size");
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        num_q_heads / num_kv_heads > kRows)
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: num_q_heads must be 1..16 times num_kv_heads");
    if (!(scale == scale)) return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: scale is NaN");
    const long long cap = (long long)max_blocks_per_seq * kBlock;
    const int len_cap = (int)(cap < max_context_len ? cap : max_context_len);
    if (prefix_len <= 0 || prefix_len % kBlock != 0 || prefix_len >= len_cap)
        return pkv::fail(PKV_ERR_INVALID,
                         "decode_shared_prefix: prefix_len (%d) must be a positive multiple of 16 below the "
                         "context bound (%d)", prefix_len, len_cap);
    if (num_seqs == 0) return PKV_OK;
    if (num_seqs > 65535) return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: at most 65535 sequences per call");
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: null pointer");
    if (!pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache) || !pkv::aligned16(out))
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: q, caches and out must be 16-byte aligned");
    if ((k_new || v_new) && (!k_new || !v_new || !pkv::aligned16(k_new) || !pkv::aligned16(v_new)))
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: k_new and v_new must both be 16-byte aligned");
    if (partition_size == 0) part = adaptive_partition(num_seqs, num_kv_heads, len_cap - prefix_len);
    const int max_parts = shared_prefix_parts(len_cap, prefix_len, part);
    if (max_parts > 65535) return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: too many partitions");
    const size_t rows = (size_t)num_seqs * num_q_heads * max_parts;
    const size_t part_bytes = workspace_for(num_seqs, num_q_heads, head_dim, max_parts);
    if (!workspace || workspace_bytes < part_bytes + kCounterBytes)
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: workspace of %zu bytes needed, %zu given",
                         part_bytes + kCounterBytes, workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return pkv::fail(PKV_ERR_INVALID, "decode_shared_prefix: workspace must be 256-byte aligned");
    char *ws = static_cast<char *>(workspace);
    float *part_o = reinterpret_cast<float *>(ws);
    float *part_ml = reinterpret_cast<float *>(ws + align256(rows * head_dim * sizeof(float)));
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // 1. the shared prefix, once for every query of the batch: a dense tile
    //    on the tensor cores (partial slot 0 of every row)
    pkv::PrefillParams pp{};
    pp.q = q;
    pp.k_cache = k_cache;
    pp.v_cache = v_cache;
    pp.block_tables = block_tables;  // row 0 holds the prefix blocks
    pp.out = out;
    pp.max_blocks = max_blocks_per_seq;
    pp.num_q_heads = num_q_heads;
    pp.num_kv_heads = num_kv_heads;
    pp.group = num_q_heads / num_kv_heads;
    pp.num_blocks = num_blocks;
    pp.len_cap = len_cap;
    pp.max_q_len = num_seqs;
    pp.total_q = num_seqs;
    pp.scale_log2 = scale * 1.4426950408889634f;
    pp.status = pkv::status_ptr();
    pp.item_counter = reinterpret_cast<unsigned long long *>(ws + part_bytes);
    pp.prefix_len = prefix_len;
    pp.part_o = part_o;
    pp.part_ml = part_ml;
    pp.part_stride = max_parts;
    rc = pkv::launch_prefill_tc(pp, 1, out_dtype, st);
    if (rc) return rc;

    // 2. each sequence's own tokens after the prefix (slots 1, 2, ...), with
    //    the optional fused append, then 3. the log-sum-exp merge of all slots
    DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    p.max_blocks = max_blocks_per_seq;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_q_heads / num_kv_heads;
    p.head_chunks = (p.group + kRows - 1) / kRows;
    p.num_blocks = num_blocks;
    p.len_cap = len_cap;
    p.partition = part;
    p.max_parts = max_parts;
    p.scale_log2 = pp.scale_log2;
    p.status = pp.status;
    p.k_new = k_new;
    p.v_new = v_new;
    p.prefix_len = prefix_len;
    p.overlap_prev = 1;  // the partitions run beside the prefix kernel
    p.head_warps = use_head_warps(num_seqs, num_kv_heads * p.head_chunks, len_cap - prefix_len, part);
    p.part_o = part_o;
    p.part_ml = part_ml;
    return out_dtype == PKV_F32 ? launch_decode<float>(p, num_seqs, head_dim, dtype, st)
                                : launch_decode<__nv_bfloat16>(p, num_seqs, head_dim, dtype, st);
}
