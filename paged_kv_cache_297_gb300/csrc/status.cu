// Per-device status word, error strings and version.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <chrono>

#include "common.cuh"
#include "prefill_common.cuh"

namespace {
// One word per device that loads the library; kernels OR PKV_STATUS_* bits in.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
// Looked up once per device; host threads that race here both store the same
// address.
std::atomic<unsigned *> g_status_addr[kMaxDevices];
thread_local char g_err[512];
}  // namespace

namespace pkv {

// A fresh 64-bit tag per launch: the splitmix64 finaliser of a per-process
// starting point (the clock and an address) plus a launch count.
unsigned long long next_launch_tag() {
    static const unsigned long long salt =
        (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() ^
        (unsigned long long)reinterpret_cast<uintptr_t>(&g_status_addr);
    static std::atomic<unsigned long long> count{0};
    unsigned long long x = salt + 0x9e3779b97f4a7c15ull * (count.fetch_add(1) + 1);
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

unsigned *status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned *addr = g_status_addr[dev].load(std::memory_order_acquire);
    if (!addr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        addr = static_cast<unsigned *>(p);
        g_status_addr[dev].store(addr, std::memory_order_release);
    }
    return addr;
}

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return PKV_OK;
}

}  // namespace pkv

extern "C" int pkv_get_status(void *stream, unsigned int *flags) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned *p = pkv::status_ptr();
    if (!p) return pkv::fail(PKV_ERR_CUDA, "pkv_get_status: no device status word");
    cudaError_t e = cudaStreamSynchronize(s);
    unsigned v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return pkv::fail(PKV_ERR_CUDA, "pkv_get_status: %s", cudaGetErrorString(e));
    if (flags) *flags = v;
    return v ? PKV_ERR_OOB : PKV_OK;
}

extern "C" int pkv_set_wait_limit_ns(unsigned long long ns) {
    pkv::set_wait_limit_ns(ns);
    return PKV_OK;
}

extern "C" const char *pkv_last_error_string(void) { return g_err; }

extern "C" int pkv_version(void) { return 100; }
