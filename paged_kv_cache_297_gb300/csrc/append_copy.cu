// KV append (slot scatter) and copy-on-write block copy.
//
// Both are pure data movement: 16-byte vector loads and stores, one thread per
// 16-byte chunk, fully coalesced on both sides (a K or V row of one kv head is
// head_dim * elem bytes contiguous in the source and in the cache).
#include "common.cuh"

namespace {

using pkv::kBlock;

// One thread per (token, kv head, 16-byte chunk of the row); K and V together.
__global__ void __launch_bounds__(256) kv_append_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const int64_t *__restrict__ slots,
    int num_tokens, uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, int64_t num_slots,
    int num_kv_heads, int chunks_per_row, unsigned *status) {
    pkv::allow_dependents();
    pkv::grid_dependency_wait();
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    int64_t per_token = (int64_t)num_kv_heads * chunks_per_row;
    if (i >= (int64_t)num_tokens * per_token) return;
    int64_t tok = i / per_token;
    int64_t rem = i - tok * per_token;
    int64_t head = rem / chunks_per_row;
    int64_t c = rem - head * chunks_per_row;
    int64_t slot = slots[tok];
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        if (head == 0 && c == 0) pkv::flag(status, PKV_STATUS_BAD_SLOT);
        return;
    }
    int64_t blk = slot / kBlock, row = slot - blk * kBlock;
    int64_t dst = ((blk * num_kv_heads + head) * kBlock + row) * chunks_per_row + c;
    k_cache[dst] = k[i];
    v_cache[dst] = v[i];
}

// Append into an fp8 E4M3 cache.  One thread per (token, kv head, 16 values
// of the row): reads them (bf16 or fp32), divides each by the kv head's scale
// (IEEE division, so the code is the one of the correctly rounded quotient),
// and stores the 16 codes (round to nearest even, saturated at 448) as one
// 16-byte vector.
template <typename T>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(
    const T *__restrict__ k, const T *__restrict__ v, const int64_t *__restrict__ slots, int num_tokens,
    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, int64_t num_slots, int num_kv_heads,
    int chunks_per_row, const float *__restrict__ k_scale, const float *__restrict__ v_scale,
    unsigned *status) {
    pkv::allow_dependents();
    pkv::grid_dependency_wait();
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    int64_t per_token = (int64_t)num_kv_heads * chunks_per_row;
    if (i >= (int64_t)num_tokens * per_token) return;
    int64_t tok = i / per_token;
    int64_t rem = i - tok * per_token;
    int64_t head = rem / chunks_per_row;
    int64_t c = rem - head * chunks_per_row;
    int64_t slot = slots[tok];
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        if (head == 0 && c == 0) pkv::flag(status, PKV_STATUS_BAD_SLOT);
        return;
    }
    const float ks = k_scale[head], vs = v_scale[head];
    const T *kr = k + i * 16, *vr = v + i * 16;  // 16 values per chunk, rows contiguous
    uint32_t kw[4], vw[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const float k0 = __fdiv_rn(float(kr[4 * q]), ks), k1 = __fdiv_rn(float(kr[4 * q + 1]), ks);
        const float k2 = __fdiv_rn(float(kr[4 * q + 2]), ks), k3 = __fdiv_rn(float(kr[4 * q + 3]), ks);
        const float v0 = __fdiv_rn(float(vr[4 * q]), vs), v1 = __fdiv_rn(float(vr[4 * q + 1]), vs);
        const float v2 = __fdiv_rn(float(vr[4 * q + 2]), vs), v3 = __fdiv_rn(float(vr[4 * q + 3]), vs);
        kw[q] = (uint32_t)pkv::f32x2_to_e4m3x2(k0, k1) | ((uint32_t)pkv::f32x2_to_e4m3x2(k2, k3) << 16);
        vw[q] = (uint32_t)pkv::f32x2_to_e4m3x2(v0, v1) | ((uint32_t)pkv::f32x2_to_e4m3x2(v2, v3) << 16);
    }
    int64_t blk = slot / kBlock, row = slot - blk * kBlock;
    int64_t dst = ((blk * num_kv_heads + head) * kBlock + row) * chunks_per_row + c;
    k_cache[dst] = make_uint4(kw[0], kw[1], kw[2], kw[3]);
    v_cache[dst] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
}

// grid.x = pair, grid.y splits the block; uint4 chunks of one whole block.
__global__ void __launch_bounds__(256) copy_blocks_kernel(
    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, const int64_t *__restrict__ pairs,
    int num_blocks, int64_t chunks_per_block, unsigned *status) {
    int64_t src = pairs[2 * blockIdx.x], dst = pairs[2 * blockIdx.x + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) pkv::flag(status, PKV_STATUS_BAD_BLOCK);
        return;
    }
    const uint4 *ks = k_cache + src * chunks_per_block;
    const uint4 *vs = v_cache + src * chunks_per_block;
    uint4 *kd = k_cache + dst * chunks_per_block;
    uint4 *vd = v_cache + dst * chunks_per_block;
    for (int64_t c = blockIdx.y * (int64_t)blockDim.x + threadIdx.x; c < chunks_per_block;
         c += (int64_t)gridDim.y * blockDim.x) {
        uint4 a = ks[c];
        uint4 b = vs[c];
        kd[c] = a;
        vd[c] = b;
    }
}

int check_common(int num_kv_heads, int head_dim, int block_size, int dtype) {
    if (block_size != kBlock) return pkv::fail(PKV_ERR_INVALID, "block_size must be 16 (got %d)", block_size);
    if (head_dim != 64 && head_dim != 128)
        return pkv::fail(PKV_ERR_INVALID, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (num_kv_heads <= 0) return pkv::fail(PKV_ERR_INVALID, "num_kv_heads must be positive");
    if (dtype != PKV_F32 && dtype != PKV_BF16 && dtype != PKV_FP8_E4M3)
        return pkv::fail(PKV_ERR_INVALID, "bad dtype %d", dtype);
    return PKV_OK;
}

int elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : dtype == PKV_BF16 ? 2 : 1; }

}  // namespace

extern "C" int pkv_kv_append(const void *k, const void *v, const int64_t *slot_mapping,
                             int num_tokens, void *k_cache, void *v_cache, int num_blocks,
                             int num_kv_heads, int head_dim, int block_size, int dtype,
                             void *stream) {
    int rc = check_common(num_kv_heads, head_dim, block_size, dtype);
    if (rc) return rc;
    if (dtype == PKV_FP8_E4M3) return pkv::fail(PKV_ERR_INVALID, "kv_append: an fp8 cache takes pkv_kv_append_fp8");
    if (num_tokens < 0 || num_blocks < 0) return pkv::fail(PKV_ERR_INVALID, "negative size");
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return pkv::fail(PKV_ERR_INVALID, "kv_append: null pointer");
    if (!pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return pkv::fail(PKV_ERR_INVALID, "kv_append: tensors must be 16-byte aligned");
    int elem = dtype == PKV_F32 ? 4 : 2;
    int chunks = head_dim * elem / 16;
    int64_t total = (int64_t)num_tokens * num_kv_heads * chunks;
    int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    cudaError_t e = pkv::launch_dependent(
        kv_append_kernel, dim3((unsigned)blocks), dim3(threads), 0, static_cast<cudaStream_t>(stream),
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, num_tokens,
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), (int64_t)num_blocks * kBlock,
        num_kv_heads, chunks, pkv::status_ptr());
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "kv_append: %s", cudaGetErrorString(e));
    return pkv::check_launch("kv_append");
}

extern "C" int pkv_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs,
                               int num_pairs, int num_blocks, int num_kv_heads, int head_dim,
                               int block_size, int dtype, void *stream) {
    int rc = check_common(num_kv_heads, head_dim, block_size, dtype);
    if (rc) return rc;
    if (num_pairs < 0 || num_blocks < 0) return pkv::fail(PKV_ERR_INVALID, "negative size");
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src_dst_pairs) return pkv::fail(PKV_ERR_INVALID, "copy_blocks: null pointer");
    if (!pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return pkv::fail(PKV_ERR_INVALID, "copy_blocks: caches must be 16-byte aligned");
    int64_t chunks = (int64_t)num_kv_heads * kBlock * head_dim * elem_bytes(dtype) / 16;
    int threads = 256;
    int ysplit = (int)((chunks + threads * 4 - 1) / (threads * 4));  // ~4 chunks per thread
    if (ysplit < 1) ysplit = 1;
    dim3 grid((unsigned)num_pairs, (unsigned)ysplit);
    copy_blocks_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), src_dst_pairs, num_blocks,
        chunks, pkv::status_ptr());
    return pkv::check_launch("copy_blocks");
}

extern "C" int pkv_kv_append_fp8(const void *k, const void *v, int in_dtype, const int64_t *slot_mapping,
                                 int num_tokens, void *k_cache, void *v_cache, const float *k_scale,
                                 const float *v_scale, int num_blocks, int num_kv_heads, int head_dim,
                                 int block_size, void *stream) {
    int rc = check_common(num_kv_heads, head_dim, block_size, PKV_FP8_E4M3);
    if (rc) return rc;
    if (in_dtype != PKV_F32 && in_dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "kv_append_fp8: inputs must be fp32 or bf16 (got %d)", in_dtype);
    if (num_tokens < 0 || num_blocks < 0) return pkv::fail(PKV_ERR_INVALID, "negative size");
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
        return pkv::fail(PKV_ERR_INVALID, "kv_append_fp8: null pointer");
    if (!pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return pkv::fail(PKV_ERR_INVALID, "kv_append_fp8: tensors must be 16-byte aligned");
    const int chunks = head_dim / 16;  // 16 codes per 16-byte chunk
    int64_t total = (int64_t)num_tokens * num_kv_heads * chunks;
    int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t slots = (int64_t)num_blocks * kBlock;
    cudaError_t e =
        in_dtype == PKV_BF16
            ? pkv::launch_dependent(kv_append_fp8_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(threads), 0,
                                    st, static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v),
                                    slot_mapping, num_tokens, static_cast<uint4 *>(k_cache),
                                    static_cast<uint4 *>(v_cache), slots, num_kv_heads, chunks, k_scale, v_scale,
                                    pkv::status_ptr())
            : pkv::launch_dependent(kv_append_fp8_kernel<float>, dim3((unsigned)blocks), dim3(threads), 0, st,
                                    static_cast<const float *>(k), static_cast<const float *>(v), slot_mapping,
                                    num_tokens, static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slots,
                                    num_kv_heads, chunks, k_scale, v_scale, pkv::status_ptr());
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "kv_append_fp8: %s", cudaGetErrorString(e));
    return pkv::check_launch("kv_append_fp8");
}
