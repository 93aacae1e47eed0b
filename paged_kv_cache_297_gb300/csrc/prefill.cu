// Chunked-prefill attention over the paged cache.
//
// A chunk of n query tokens of a sequence whose cache holds L tokens (the
// chunk included) sits at positions L-n .. L-1; query j attends causally to
// tokens 0 .. L-n+j (caffein.top, "Chunked Prefill").
//
// Work unit: one CTA per (tile of 64 packed query rows, kv head, sequence).
// Row r of a tile is query position j = R / G and head kvh * G + R % G with
// R = tile * 64 + r, so the G heads sharing a kv head share every K/V tile
// (GQA).  K/V tiles of 64 tokens (4 blocks) are gathered through the block
// table into swizzled shared memory by 16-byte cp.async copies, double
// buffered; each warp owns 16 rows and runs S = Q K^T, the online softmax and
// O += P V on the tensor cores.
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "prefill_common.cuh"

namespace {

// x rounded to the nearest bf16 (ties to even), as a float.
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

using pkv::kBlock;
using pkv::PrefillParams;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileQ = 64;   // packed query rows per CTA
constexpr int kTileK = 64;   // keys per stage
constexpr int kStages = 2;


template <int D>
struct PrefillSmem {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTile = kTileK * kRowBytes;
    static constexpr int kStage = 2 * kTile;
    static constexpr int kBytes = kStages * kStage;
};

template <int D, typename OutT>
__global__ void __launch_bounds__(kThreads) prefill_bf16_kernel(const PrefillParams p) {
    using Sm = PrefillSmem<D>;
    constexpr int CH = D / 8;
    constexpr int PER_THREAD = kTileK * CH / kThreads;
    constexpr int KSTEPS = D / 16;
    constexpr int NT = D / 8;
    constexpr int ST = kTileK / 8;  // score n-tiles per key tile

    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gid = lane >> 2, tig = lane & 3;
    const int tile = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
    const int G = p.group;

    const int q0 = p.cu_q_lens[s];
    const int n = p.cu_q_lens[s + 1] - q0;
    int L = p.context_lens[s];
    if (L < 0 || L > p.len_cap) {
        if (tile == 0 && kvh == 0 && threadIdx.x == 0) pkv::flag(p.status, PKV_STATUS_BAD_LENGTH);
        return;
    }
    if (q0 < 0 || n < 0 || n > L || n > p.max_q_len || q0 + n > p.total_q) {
        if (tile == 0 && kvh == 0 && threadIdx.x == 0) pkv::flag(p.status, PKV_STATUS_BAD_QLEN);
        return;
    }
    if (tile * kTileQ >= n * G) return;
    const int prior = L - n;
    const int j_last = min(n - 1, (tile * kTileQ + kTileQ - 1) / G);
    const int kv_end = prior + j_last + 1;  // keys this CTA needs
    const int nkt = (kv_end + kTileK - 1) / kTileK;

    // this thread's two rows
    const int RA = tile * kTileQ + warp * 16 + gid, RB = RA + 8;
    const int jA = RA / G, jB = RB / G;
    const bool vA = jA < n, vB = jB < n;
    const int posA = vA ? prior + jA : -1, posB = vB ? prior + jB : -1;
    const int warp_R_last = tile * kTileQ + warp * 16 + 15;
    const int warp_pos_max = prior + min(n - 1, warp_R_last / G);
    const bool warp_live = (tile * kTileQ + warp * 16) / G < n;

    const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *kc = static_cast<const __nv_bfloat16 *>(p.k_cache);
    const __nv_bfloat16 *vc = static_cast<const __nv_bfloat16 *>(p.v_cache);
    const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;

    uint32_t qa[KSTEPS][4];
    {
        const __nv_bfloat16 *ra = qb + ((size_t)(q0 + jA) * p.num_q_heads + kvh * G + RA % G) * D;
        const __nv_bfloat16 *rb = qb + ((size_t)(q0 + jB) * p.num_q_heads + kvh * G + RB % G) * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; kk++) {
            const int col = kk * 16 + tig * 2;
            qa[kk][0] = vA ? *reinterpret_cast<const uint32_t *>(ra + col) : 0u;
            qa[kk][1] = vB ? *reinterpret_cast<const uint32_t *>(rb + col) : 0u;
            qa[kk][2] = vA ? *reinterpret_cast<const uint32_t *>(ra + col + 8) : 0u;
            qa[kk][3] = vB ? *reinterpret_cast<const uint32_t *>(rb + col + 8) : 0u;
        }
    }

    auto issue = [&](int kt, int st) {
        unsigned char *ks = smem + st * Sm::kStage;
        unsigned char *vs = ks + Sm::kTile;
#pragma unroll
        for (int j = 0; j < PER_THREAD; j++) {
            const int i = threadIdx.x + kThreads * j;
            const int r = i / CH, c = i - (i / CH) * CH;
            const int t = kt * kTileK + r;
            int nb = 0;
            size_t go = 0;
            if (t < kv_end) {
                const int phys = table[t / kBlock];
                if (phys >= 0 && phys < p.num_blocks) {
                    nb = 16;
                    go = ((((size_t)phys * p.num_kv_heads + kvh) * kBlock + (t % kBlock)) * D) * 2 + c * 16;
                } else if (c == 0 && (t % kBlock) == 0) {
                    pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                }
            }
            pkv::cp_async16(ks + pkv::swz(r, c, Sm::kRowBytes), reinterpret_cast<const unsigned char *>(kc) + go, nb);
            pkv::cp_async16(vs + pkv::swz(r, c, Sm::kRowBytes), reinterpret_cast<const unsigned char *>(vc) + go, nb);
        }
    };

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    issue(0, 0);
    pkv::cp_async_commit();
    for (int kt = 0; kt < nkt; kt++) {
        if (kt + 1 < nkt) issue(kt + 1, (kt + 1) % kStages);
        pkv::cp_async_commit();
        pkv::cp_async_wait<1>();
        __syncthreads();

        if (warp_live && kt * kTileK <= warp_pos_max) {
            const unsigned char *ks = smem + (kt % kStages) * Sm::kStage;
            const unsigned char *vs = ks + Sm::kTile;
            float sc[ST][4];
#pragma unroll
            for (int i = 0; i < ST; i++) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; kk++) {
#pragma unroll
                for (int np = 0; np < ST / 2; np++) {
                    uint32_t b0, b1, b2, b3;
                    const int tok = np * 16 + ((lane >> 4) << 3) + (lane & 7);
                    const int ch = kk * 2 + ((lane >> 3) & 1);
                    pkv::ldsm_x4(b0, b1, b2, b3, ks + pkv::swz(tok, ch, Sm::kRowBytes));
                    pkv::mma_bf16(sc[2 * np], qa[kk], b0, b1);
                    pkv::mma_bf16(sc[2 * np + 1], qa[kk], b2, b3);
                }
            }
            float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < ST; nt++) {
                const int t = kt * kTileK + nt * 8 + tig * 2;
                sc[nt][0] = t <= posA ? sc[nt][0] * p.scale_log2 : -INFINITY;
                sc[nt][1] = t + 1 <= posA ? sc[nt][1] * p.scale_log2 : -INFINITY;
                sc[nt][2] = t <= posB ? sc[nt][2] * p.scale_log2 : -INFINITY;
                sc[nt][3] = t + 1 <= posB ? sc[nt][3] * p.scale_log2 : -INFINITY;
                mxA = fmaxf(mxA, fmaxf(sc[nt][0], sc[nt][1]));
                mxB = fmaxf(mxB, fmaxf(sc[nt][2], sc[nt][3]));
            }
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
            const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
            const float baseA = nA == -INFINITY ? 0.f : nA;
            const float baseB = nB == -INFINITY ? 0.f : nB;
            const float alA = pkv::fast_exp2(mA - baseA), alB = pkv::fast_exp2(mB - baseB);
            mA = nA;
            mB = nB;
            float sumA = 0.f, sumB = 0.f;
#pragma unroll
            for (int nt = 0; nt < ST; nt++) {
                // P rounded to bf16 here, as the PV product takes it, so that
                // the row sum adds the same values (numerator and denominator
                // share the rounding)
                sc[nt][0] = round_bf16(pkv::fast_exp2(sc[nt][0] - baseA));
                sc[nt][1] = round_bf16(pkv::fast_exp2(sc[nt][1] - baseA));
                sc[nt][2] = round_bf16(pkv::fast_exp2(sc[nt][2] - baseB));
                sc[nt][3] = round_bf16(pkv::fast_exp2(sc[nt][3] - baseB));
                sumA += sc[nt][0] + sc[nt][1];
                sumB += sc[nt][2] + sc[nt][3];
            }
            lA = lA * alA + sumA;
            lB = lB * alB + sumB;
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                o[nt][0] *= alA;
                o[nt][1] *= alA;
                o[nt][2] *= alB;
                o[nt][3] *= alB;
            }
#pragma unroll
            for (int kq = 0; kq < kTileK / 16; kq++) {
                const uint32_t pa[4] = {pkv::pack_bf16(sc[2 * kq][0], sc[2 * kq][1]),
                                        pkv::pack_bf16(sc[2 * kq][2], sc[2 * kq][3]),
                                        pkv::pack_bf16(sc[2 * kq + 1][0], sc[2 * kq + 1][1]),
                                        pkv::pack_bf16(sc[2 * kq + 1][2], sc[2 * kq + 1][3])};
#pragma unroll
                for (int nn = 0; nn < D / 16; nn++) {
                    uint32_t v0, v1, v2, v3;
                    const int jm = lane >> 3;
                    const int tok = kq * 16 + ((jm & 1) << 3) + (lane & 7);
                    const int ch = nn * 2 + (jm >> 1);
                    pkv::ldsm_x4_t(v0, v1, v2, v3, vs + pkv::swz(tok, ch, Sm::kRowBytes));
                    pkv::mma_bf16(o[2 * nn], pa, v0, v1);
                    pkv::mma_bf16(o[2 * nn + 1], pa, v2, v3);
                }
            }
        }
        __syncthreads();
    }
    pkv::cp_async_wait<0>();

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    OutT *out = static_cast<OutT *>(p.out);
    const float iA = lA > 0.f ? 1.f / lA : 0.f, iB = lB > 0.f ? 1.f / lB : 0.f;
    OutT *oa = out + ((size_t)(q0 + jA) * p.num_q_heads + kvh * G + RA % G) * D;
    OutT *ob = out + ((size_t)(q0 + jB) * p.num_q_heads + kvh * G + RB % G) * D;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        const int col = nt * 8 + tig * 2;
        if (vA) pkv::store2(oa + col, o[nt][0] * iA, o[nt][1] * iA);
        if (vB) pkv::store2(ob + col, o[nt][2] * iB, o[nt][3] * iB);
    }
}

// ----------------------------------------------------------------------------
// CUDA-core prefill (fp32 caches): one CTA per (q head, query, sequence)
// ----------------------------------------------------------------------------

template <typename T>
__device__ __forceinline__ float ld_elem(const T *p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

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

template <typename T, typename OutT>
__global__ void __launch_bounds__(kThreads) prefill_cuda_core_kernel(const PrefillParams p, int D) {
    __shared__ float sq[128];
    __shared__ float sp[kThreads];
    __shared__ int sb[kThreads];
    __shared__ float red[kWarps];
    const int h = blockIdx.x, j = blockIdx.y, s = blockIdx.z, tid = threadIdx.x;
    const int q0 = p.cu_q_lens[s];
    const int n = p.cu_q_lens[s + 1] - q0;
    const int L = p.context_lens[s];
    if (L < 0 || L > p.len_cap) {
        if (h == 0 && j == 0 && tid == 0) pkv::flag(p.status, PKV_STATUS_BAD_LENGTH);
        return;
    }
    if (q0 < 0 || n < 0 || n > L || n > p.max_q_len || q0 + n > p.total_q) {
        if (h == 0 && j == 0 && tid == 0) pkv::flag(p.status, PKV_STATUS_BAD_QLEN);
        return;
    }
    if (j >= n) return;
    const int kvh = h / p.group;
    const int t_end = L - n + j + 1;
    const T *qrow = static_cast<const T *>(p.q) + ((size_t)(q0 + j) * p.num_q_heads + h) * D;
    const T *kc = static_cast<const T *>(p.k_cache);
    const T *vc = static_cast<const T *>(p.v_cache);
    const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;
    for (int c = tid; c < D; c += kThreads) sq[c] = ld_elem(qrow + c);
    float m = -INFINITY, l = 0.f, acc = 0.f;
    __syncthreads();
    for (int t0 = 0; t0 < t_end; t0 += kThreads) {
        const int t = t0 + tid;
        float x = -INFINITY;
        int phys = -1;
        if (t < t_end) {
            phys = table[t / kBlock];
            if (phys < 0 || phys >= p.num_blocks) {
                pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                phys = -1;
            } else {
                const T *kr = kc + (((size_t)phys * p.num_kv_heads + kvh) * kBlock + t % kBlock) * D;
                float dot = 0.f;
                for (int c = 0; c < D; c++) dot = fmaf(sq[c], ld_elem(kr + c), dot);
                x = dot * p.scale_log2;
            }
        }
        const float cmax = block_reduce(x, red, true);
        const float mn = fmaxf(m, cmax);
        const float base = mn == -INFINITY ? 0.f : mn;
        const float alpha = pkv::fast_exp2(m - base);
        const float pt = pkv::fast_exp2(x - base);
        sp[tid] = pt;
        sb[tid] = phys;
        const float psum = block_reduce(pt, red, false);
        l = l * alpha + psum;
        m = mn;
        acc *= alpha;
        const int cnt = min(kThreads, t_end - t0);
        if (tid < D) {
            for (int i = 0; i < cnt; i++) {
                if (sb[i] < 0) continue;
                const int t2 = t0 + i;
                const T *vr = vc + (((size_t)sb[i] * p.num_kv_heads + kvh) * kBlock + t2 % kBlock) * D;
                acc = fmaf(sp[i], ld_elem(vr + tid), acc);
            }
        }
        __syncthreads();
    }
    if (tid < D)
        pkv::store1(static_cast<OutT *>(p.out) + ((size_t)(q0 + j) * p.num_q_heads + h) * D + tid,
                    l > 0.f ? acc / l : 0.f);
}

template <int D, typename OutT>
int launch_bf16(const PrefillParams &p, int num_seqs, cudaStream_t st) {
    constexpr int bytes = PrefillSmem<D>::kBytes;
    // set once per device (setting it twice from racing host threads is harmless)
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(prefill_bf16_kernel<D, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 bytes) != cudaSuccess)
            return pkv::check_launch("prefill: set shared memory size");
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int tiles = (p.max_q_len * p.group + kTileQ - 1) / kTileQ;
    dim3 grid((unsigned)tiles, (unsigned)p.num_kv_heads, (unsigned)num_seqs);
    prefill_bf16_kernel<D, OutT><<<grid, kThreads, bytes, st>>>(p);
    return pkv::check_launch("prefill_bf16");
}

template <typename OutT>
int launch_prefill(const PrefillParams &p, int num_seqs, int D, int dtype, cudaStream_t st) {
    if (pkv::prefill_tc_supported(dtype, D))
        return pkv::launch_prefill_tc(p, num_seqs, sizeof(OutT) == 4 ? PKV_F32 : PKV_BF16, st);
    if (dtype == PKV_BF16)
        return D == 128 ? launch_bf16<128, OutT>(p, num_seqs, st) : launch_bf16<64, OutT>(p, num_seqs, st);
    dim3 grid((unsigned)p.num_q_heads, (unsigned)p.max_q_len, (unsigned)num_seqs);
    prefill_cuda_core_kernel<float, OutT><<<grid, kThreads, 0, st>>>(p, D);
    return pkv::check_launch("prefill_cuda_core");
}

}  // namespace

extern "C" int pkv_prefill_workspace_bytes(int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                                           int head_dim, int max_q_len, int max_context_len,
                                           size_t *bytes) {
    if (!bytes || num_seqs < 0 || total_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        max_q_len < 0 || max_context_len < 0 || (head_dim != 64 && head_dim != 128))
        return pkv::fail(PKV_ERR_INVALID, "prefill_workspace_bytes: bad argument");
    // the tcgen05 path's work-item counters (32 bytes, in a 256-byte block)
    *bytes = head_dim == 128 ? 256 : 0;
    return PKV_OK;
}

extern "C" int pkv_paged_attention_prefill_chunk(const void *q, const int32_t *cu_q_lens,
                                                 const void *k_cache, const void *v_cache,
                                                 const int32_t *block_tables, int max_blocks_per_seq,
                                                 const int32_t *context_lens, int num_seqs,
                                                 int total_q, int max_q_len, int max_context_len,
                                                 int num_q_heads, int num_kv_heads, int head_dim,
                                                 int block_size, int num_blocks, float scale,
                                                 void *out, int dtype, int out_dtype, void *workspace,
                                                 size_t workspace_bytes, void *stream) {
    if (block_size != kBlock) return pkv::fail(PKV_ERR_INVALID, "block_size must be 16 (got %d)", block_size);
    if (head_dim != 64 && head_dim != 128)
        return pkv::fail(PKV_ERR_INVALID, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (dtype != PKV_F32 && dtype != PKV_BF16) return pkv::fail(PKV_ERR_INVALID, "bad dtype %d", dtype);
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "bad out_dtype %d", out_dtype);
    if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || max_context_len < 0 || num_blocks < 0 ||
        max_blocks_per_seq < 0)
        return pkv::fail(PKV_ERR_INVALID, "prefill: negative size");
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return pkv::fail(PKV_ERR_INVALID, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                         num_q_heads, num_kv_heads);
    if (dtype == PKV_BF16 && num_q_heads / num_kv_heads > kTileQ)
        return pkv::fail(PKV_ERR_INVALID, "prefill: at most %d q heads per kv head", kTileQ);
    if (!(scale == scale)) return pkv::fail(PKV_ERR_INVALID, "prefill: scale is NaN");
    if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
    if (num_seqs > 65535 || max_q_len > 65535 || num_kv_heads > 65535)
        return pkv::fail(PKV_ERR_INVALID, "prefill: at most 65535 sequences and 65535 queries per sequence");
    if (!q || !cu_q_lens || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return pkv::fail(PKV_ERR_INVALID, "prefill: null pointer");
    if (!pkv::aligned16(q) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache) || !pkv::aligned16(out))
        return pkv::fail(PKV_ERR_INVALID, "prefill: q, caches and out must be 16-byte aligned");
    PrefillParams p{};
    p.q = q;
    p.cu_q_lens = cu_q_lens;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    p.max_blocks = max_blocks_per_seq;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_q_heads / num_kv_heads;
    p.num_blocks = num_blocks;
    const long long cap = (long long)max_blocks_per_seq * kBlock;
    p.len_cap = (int)(cap < max_context_len ? cap : max_context_len);
    p.max_q_len = max_q_len;
    p.total_q = total_q;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = pkv::status_ptr();
    if (pkv::prefill_tc_supported(dtype, head_dim)) {
        if (!workspace || workspace_bytes < 16 || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
            return pkv::fail(PKV_ERR_INVALID,
                             "prefill: workspace of 16 bytes (16-byte aligned) needed, %zu given", workspace_bytes);
        p.item_counter = static_cast<unsigned long long *>(workspace);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return out_dtype == PKV_F32 ? launch_prefill<float>(p, num_seqs, head_dim, dtype, st)
                                : launch_prefill<__nv_bfloat16>(p, num_seqs, head_dim, dtype, st);
}
