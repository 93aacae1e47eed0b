// Paged-attention decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run decode: code inside a custom memory pool or an allocator hook
// (which must not re-enter the allocator), embedders whose device memory is
// fully budgeted up front, or runtimes that forbid allocation on their
// serving path.  The ordinary entry point needs a caller-provided workspace
// for the split-K partials; this variant instead uses one fixed-size scratch
// array that lives in the library's own device image, so it allocates
// nothing and needs no workspace argument.
//
// The array below is a file-scope static __device__ array: every GPU that
// loads this library holds kNoAllocScratchBytes of device memory for it until
// the process exits.  Host code cannot use its name as a device address (on
// the host the name is only a stand-in), so the address is looked up once
// per device with cudaGetSymbolAddress and handed to the kernels.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(PKV_NO_ALLOC_SCRATCH_BYTES);

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of g_decode_scratch on the current device (looked up on the
// first call per device; later calls reuse it).  Returns an error code.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return pkv::fail(PKV_ERR_CUDA, "decode_no_alloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return pkv::fail(PKV_ERR_INVALID, "decode_no_alloc: device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();  // a later call's launch check must not see this error
            return pkv::fail(PKV_ERR_CUDA, "decode_no_alloc: cudaGetSymbolAddress: %s",
                             cudaGetErrorString(e));
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_attention_decode_no_alloc(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int num_blocks, int max_context_len,
    int partition_size, float scale, void *out, int dtype, int out_dtype, void *stream) {
    // The partition the call will use (partition_size 0: the adaptive choice),
    // so that the scratch is sized for the launch that runs, not for the
    // smallest partitions.
    int part = 0;
    int rc = pkv_decode_partition_size(num_seqs, num_kv_heads, max_context_len, partition_size, &part);
    if (rc) return rc;
    size_t need = 0;
    rc = pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len, part, &need);
    if (rc) return rc;
    if (need > kNoAllocScratchBytes)
        return pkv::fail(PKV_ERR_INVALID,
                         "decode_no_alloc: these sizes need %zu bytes of split-K scratch but the "
                         "static scratch holds %zu; use pkv_paged_attention_decode with a "
                         "caller workspace",
                         need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    if (need > 0) {
        rc = scratch_address(&scratch);
        if (rc) return rc;
    }
    // Nothing in the scratch has to start at zero: every partial the reduce
    // reads is written by the partition kernel of the same call.
    return pkv_paged_attention_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                      context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      block_size, num_blocks, max_context_len, part,
                                      scale, out, dtype, out_dtype, scratch,
                                      need > 0 ? kNoAllocScratchBytes : 0, stream);
}
