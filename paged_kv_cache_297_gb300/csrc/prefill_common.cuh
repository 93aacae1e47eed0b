// Parameters shared by the chunked-prefill kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct PrefillParams {
    const void *q;
    const int32_t *cu_q_lens;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    void *out;
    int max_blocks;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int num_blocks;
    int len_cap;
    int max_q_len;
    int total_q;
    float scale_log2;
    unsigned *status;
    // tcgen05 kernel only: persistent CTA pairs take (sequence, q tile, kv
    // head) items from a counter in the workspace: 32 bytes, 16-byte
    // aligned, {launch tag, items taken} and {launch tag, CTAs done}, kept
    // by the kernel itself (the last CTA clears both tags)
    int num_seqs;
    int tiles_per_seq;
    int num_items;
    unsigned long long *item_counter;
    unsigned long long launch_tag;
    // set by the launch: 1 when the q tiles are loaded by TMA (the group
    // divides the 128-row tile), 0 when the softmax threads copy them
    int q_tma;
    // set by the launch: 1 when the output is 32-byte aligned (32-byte stores)
    int out_v8;
    // shared-prefix mode (prefix_len > 0): the "chunk" is the batch's decode
    // queries (one position per sequence, max_q_len = sequences), every one
    // attends to keys [0, prefix_len) of block table row 0, and the result
    // is written unnormalised as partial slot 0 of each decode row:
    // part_o [rows][part_stride][D], part_ml [rows][part_stride][2]
    int prefix_len;
    float *part_o;
    float *part_ml;
    int part_stride;
    // tcgen05 kernel, set by the launch: the longest any of its waits may
    // last (nanoseconds, %globaltimer) before it gives up
    unsigned long long wait_ns;
};

// tcgen05 kernel (prefill_tc.cu): bf16 caches with head_dim 128.
bool prefill_tc_supported(int dtype, int head_dim);
int launch_prefill_tc(const PrefillParams &p, int num_seqs, int out_dtype, cudaStream_t st);
// Process-wide bound on each wait of the tcgen05 kernel (0: the default).
void set_wait_limit_ns(unsigned long long ns);

}  // namespace pkv
