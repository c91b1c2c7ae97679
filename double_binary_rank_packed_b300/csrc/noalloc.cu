// dbf_matmul_decode_noalloc: the decode-path product for callers that cannot
// hand the library any device scratch memory.
//
// Some callers have no way to allocate: code running while a CUDA graph is
// being captured (cudaMalloc is not a stream operation and cannot be
// recorded), latency-critical serving loops where cudaMalloc's implicit
// device synchronisation is not acceptable, and runtimes whose device memory
// is planned up front in a fixed arena with nothing left to lend.  For them
// this entry point keeps the decode kernels' only scratch buffer (the fp16
// intermediate V, ell*T rows of round_up(R, 64) halves) in a file-scope
// device array of fixed size.  The caller still passes x, y and the factors.
//
// The array is a static __device__ object: every GPU that loads this library
// holds its kNoAllocScratchBytes until the process exits.  In host code the
// name g_noalloc_scratch only stands for the symbol, it is not a device
// address; the address is looked up once per device with
// cudaGetSymbolAddress (on the first call made on that device) and then
// passed to the kernels.
#include <stdio.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void *g_scratch_addr[kNoAllocMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (set-up on the
// first call per device).  Returns nullptr if the lookup fails.
void *scratch_for_current_device(cudaError_t *err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*err != cudaSuccess || !p) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

}  // namespace

extern "C" int dbf_matmul_decode_noalloc(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y,
                                         int accumulate, void *stream) {
    using namespace dbfk;
    if (!f) return DBF_ERR_INVALID_ARG;
    if (f->N < 1 || f->M < 1 || f->R < 1 || f->ell < 1 || f->ell > 4) return DBF_ERR_INVALID_ARG;
    if (!f->B1 || !f->B2 || !f->alpha || !f->beta || !f->gamma) return DBF_ERR_INVALID_ARG;
    if (f->ldw1 < ceil_div(f->R, 32) || f->ldw2 < ceil_div(f->M, 32)) return DBF_ERR_INVALID_ARG;
    if (!aligned16(f->B1) || !aligned16(f->B2) || !aligned16(f->alpha) || !aligned16(f->beta) ||
        !aligned16(f->gamma))
        return DBF_ERR_ALIGNMENT;
    if (T < 0 || (accumulate != 0 && accumulate != 1)) return DBF_ERR_INVALID_ARG;
    if (T == 0) return DBF_OK;
    if (!x || !y) return DBF_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return DBF_ERR_ALIGNMENT;

    // scratch needed by the decode kernels: V [ell*T][round_up(R, 64)] fp16
    const int64_t ldv = round_up(f->R, 64);
    const double need = double(f->ell) * double(T) * double(ldv) * 2.0;
    if (need > double(kNoAllocScratchBytes)) {
        set_last_error("dbf_matmul_decode_noalloc: ell*T*round_up(R,64)*2 bytes of scratch exceed the "
                       "2 MiB static array");
        return DBF_ERR_WORKSPACE;
    }

    cudaError_t err = cudaSuccess;
    void *scratch = scratch_for_current_device(&err);
    if (!scratch) {
        set_last_error("dbf_matmul_decode_noalloc: cudaGetSymbolAddress of the static scratch failed");
        return DBF_ERR_CUDA;
    }

    // the two-stage decode kernels of dbf_matmul's decode path, with V in the static array
    int sms = 148;
    {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 148;
    }
    DecodeCall c = {};
    c.f = f;
    c.N = f->N;
    c.M = f->M;
    c.R = f->R;
    c.ell = f->ell;
    c.T = static_cast<int>(T);
    c.tokens_per_problem = static_cast<int>(T);
    c.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    c.y = reinterpret_cast<__nv_bfloat16 *>(y);
    c.accumulate = accumulate;
    c.status = nullptr;
    err = launch_decode_two_stage(c, static_cast<__half *>(scratch), static_cast<int>(ldv), sms,
                                  static_cast<cudaStream_t>(stream));
    if (err == cudaErrorNotSupported) {
        set_last_error("dbf_matmul_decode_noalloc: no decode tile plan fits this shape");
        return DBF_ERR_UNSUPPORTED;
    }
    if (err != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof(msg), "dbf_matmul_decode_noalloc: %s", cudaGetErrorString(err));
        set_last_error(msg);
        return DBF_ERR_CUDA;
    }
    return DBF_OK;
}
