// Shared device helpers for the pkv kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pkv.h"

namespace pkv {

constexpr int kBlock = 16;  // tokens per cache block

// ---------------------------------------------------------------- host side

// Device address of this device's status word (nullptr if it cannot be had).
unsigned *status_ptr();
// A 64-bit value drawn afresh for each launch that tags the work counters it
// keeps in a caller's workspace (no clearing pass is needed before it).
unsigned long long next_launch_tag();
// Record a message for pkv_last_error_string() and return `code`.
int fail(int code, const char *fmt, ...);
// Turn a pending launch error into PKV_ERR_CUDA.
int check_launch(const char *what);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch `kernel` with programmatic stream serialisation, so that its launch
// overlaps the tail of the previous kernel on the stream (see
// grid_dependency_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- device side

// Programmatic dependent launch.  A kernel launched with
// pkv::launch_dependent may start while the previous kernel on the stream is
// still running; it must call grid_dependency_wait() before reading anything
// that kernel writes (the wait returns once the previous grid has completed and
// its memory is visible; without the launch attribute it returns at once).
// allow_dependents() lets the next dependent kernel launch early.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void flag(unsigned *status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Compare-and-swap of the 16 bytes at `addr` (16-byte aligned); returns the
// previous contents through old_lo / old_hi.
__device__ __forceinline__ void cas128(unsigned long long *addr, unsigned long long cmp_lo, unsigned long long cmp_hi,
                                       unsigned long long new_lo, unsigned long long new_hi,
                                       unsigned long long &old_lo, unsigned long long &old_hi) {
    asm volatile(
        "{\n .reg .b128 d, c, n;\n mov.b128 c, {%3, %4};\n mov.b128 n, {%5, %6};\n"
        " atom.relaxed.gpu.global.cas.b128 d, [%2], c, n;\n mov.b128 {%0, %1}, d;\n}\n"
        : "=l"(old_lo), "=l"(old_hi)
        : "l"(addr), "l"(cmp_lo), "l"(cmp_hi), "l"(new_lo), "l"(new_hi)
        : "memory");
}

// A work counter in a caller's workspace that needs no clearing pass: the
// 16 bytes at `c` (16-byte aligned) hold {launch tag, count}.  The first
// caller of a launch finds another tag (an earlier launch's, a cleared 0, or
// whatever the workspace held) and installs {tag, 0} with one 16-byte
// compare-and-swap; every call then adds one to the count and returns the
// count before it.  Tags are non-zero 64-bit values drawn per launch.
__device__ __forceinline__ unsigned long long tagged_add(unsigned long long *c, unsigned long long tag) {
    unsigned long long t = *reinterpret_cast<volatile unsigned long long *>(c);
    if (t != tag) {
        unsigned long long cnt = *reinterpret_cast<volatile unsigned long long *>(c + 1);
        for (int tries = 0; tries < 64 && t != tag; tries++) {
            unsigned long long ot, oc;
            cas128(c, t, cnt, tag, 0ull, ot, oc);
            if (ot == t && oc == cnt) break;  // installed
            t = ot;
            cnt = oc;
        }
    }
    return atomicAdd(c + 1, 1ull);
}

// 16-byte global->shared copy; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                        const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                          const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}

// D += A(16x16, row) * B(16x8, col); bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulation (fragment layouts as
// for the bf16 form).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// fp16 pair in one 32-bit register (lo in the low half), round to nearest
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp8 E4M3 values (low byte first) to an fp16 pair; exact (every E4M3
// value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(v));
    return r;
}

// Two fp32 values to E4M3 codes (lo to the low byte), round to nearest even,
// magnitudes beyond 448 saturated to 448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Split x into hi + lo with both halves bf16 (hi = RNE(x), lo = RNE(x - hi)).
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - hi;
}

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// Byte offset of 16-byte chunk `c` of row `r` in a tile whose rows are
// `row_bytes` long, XOR-swizzled so that 8 consecutive rows at the same chunk
// land in 8 different bank groups (conflict-free ldmatrix).
__device__ __forceinline__ int swz(int r, int c, int row_bytes) {
    return r * row_bytes + ((c ^ (r & 7)) << 4);
}

template <typename T>
__device__ __forceinline__ void store2(T *p, float a, float b);
template <>
__device__ __forceinline__ void store2<float>(float *p, float a, float b) {
    *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}
template <>
__device__ __forceinline__ void store2<__nv_bfloat16>(__nv_bfloat16 *p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}
template <typename T>
__device__ __forceinline__ void store1(T *p, float a);
template <>
__device__ __forceinline__ void store1<float>(float *p, float a) { *p = a; }
template <>
__device__ __forceinline__ void store1<__nv_bfloat16>(__nv_bfloat16 *p, float a) {
    *p = __float2bfloat16_rn(a);
}

}  // namespace pkv
