// dbf_matmul_decode_noalloc: the decode-path product for callers that cannot
// hand the library any device scratch memory.
//
// Some callers have no way to allocate device memory for a call: serving
// loops that must never take cudaMalloc's implicit device synchronisation on
// the token path, runtimes whose device memory is one arena planned at
// start-up with nothing left to lend, and plug-in hosts that pass a library
// only its inputs and outputs.  For them this entry point runs the decode
// path of dbf_matmul (the same kernels, chosen the same way) with its
// workspace -- the fp16 intermediate V of the two-stage kernels, ell*T rows of
// round_up(R, 64) halves -- in a file-scope device array of fixed size.  The
// caller still passes x, y and the factors.  The papers have no counterpart:
// this is a deployment variant, not a step of the method.
//
// The array is a static __device__ object: every GPU that loads this library
// holds its kNoAllocScratchBytes until the process exits.  In host code the
// name g_noalloc_scratch only stands for the symbol, it is not a device
// address; the address is looked up once per device with
// cudaGetSymbolAddress (on the first call made on that device, with that
// device current) and then handed to the kernels as their workspace.
#include <stdio.h>

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
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kNoAllocMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*err != cudaSuccess || !p) {
            if (*err == cudaSuccess) *err = cudaErrorInvalidSymbol;
            cudaGetLastError();  // leave no error behind for the caller's next launch check
            return nullptr;
        }
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" int dbf_matmul_decode_noalloc(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y,
                                         int accumulate, void *stream) {
    // the argument checks of dbf_matmul_path, so both entry points reject the same calls with the same codes
    const int rc = dbfk::check_matmul_args(f, x, T, y, accumulate, DBF_PATH_DECODE);
    if (rc != DBF_OK || T == 0) return rc;
    const size_t need = dbf_workspace_bytes_path(f, T, DBF_PATH_DECODE);
    if (need > kNoAllocScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "dbf_matmul_decode_noalloc: %zu bytes of scratch (ell*T*round_up(R,64)*2) exceed the 2 MiB "
                 "static array",
                 need);
        dbfk::set_last_error(msg);
        return DBF_ERR_WORKSPACE;
    }
    cudaError_t err = cudaSuccess;
    void *scratch = scratch_for_current_device(&err);
    if (!scratch) {
        char msg[200];
        snprintf(msg, sizeof(msg), "dbf_matmul_decode_noalloc: cudaGetSymbolAddress of the static scratch: %s",
                 cudaGetErrorString(err));
        dbfk::set_last_error(msg);
        return DBF_ERR_CUDA;
    }
    // the decode path of dbf_matmul_path: the same argument checks, kernels and device status word
    return dbf_matmul_path(f, x, T, y, accumulate, scratch, kNoAllocScratchBytes, stream, DBF_PATH_DECODE);
}
