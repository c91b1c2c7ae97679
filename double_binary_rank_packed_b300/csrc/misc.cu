// Sign packing, unpacking, and the bounded-wait self test.
//
// Storage of the binary factors at one bit per entry (LoRDBA page, section 2,
// "Eficiencia de Almacenamiento"): bit j of word w of a row is the sign of
// column 32w + j, 1 for +1, 0 for -1, pad bits 0.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dbfk {

namespace {

// One warp per packed word: lane j reads column 32w + j and the warp ballot
// is the word (bit j = lane j's predicate).
__global__ void pack_kernel(const int8_t *__restrict__ signs, int64_t rows, int64_t cols,
                            uint32_t *__restrict__ words, int64_t ldw) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t total = rows * ldw;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); idx < total;
         idx += warps) {
        const int64_t r = idx / ldw, w = idx - r * ldw;
        const int64_t col = 32 * w + lane;
        const int8_t s = (col < cols) ? signs[r * cols + col] : int8_t(0);
        const uint32_t word = __ballot_sync(0xffffffffu, s > 0);
        if (lane == 0) words[idx] = word;
    }
}

__global__ void unpack_kernel(const uint32_t *__restrict__ words, int64_t rows, int64_t cols, int64_t ldw,
                              int8_t *__restrict__ signs) {
    const int64_t total = rows * cols;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = e / cols, c = e - r * cols;
        const uint32_t w = words[r * ldw + (c >> 5)];
        signs[e] = ((w >> (c & 31)) & 1u) ? int8_t(1) : int8_t(-1);
    }
}

// Packed bit-matrix transpose, one warp per 32 x 32 block: lane l holds word
// w of source row r0 + l; the ballot of bit k over the 32 lanes is word r0/32
// of destination row 32w + k (bit l = source row r0 + l).  Source rows past
// `rows` read as 0, so the pad bits of the destination are 0; destination
// words past ceil(rows/32) are written as 0.
__global__ void transpose_kernel(const uint32_t *__restrict__ words, int64_t rows, int64_t cols, int64_t ldw,
                                 uint32_t *__restrict__ words_t, int64_t ldw_t) {
    const int lane = threadIdx.x & 31;
    const int64_t rb = (rows + 31) / 32;  // destination words per row that hold data
    const int64_t cw = (cols + 31) / 32;  // source words per row that hold data
    const int64_t blocks = rb * cw;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); b < blocks;
         b += warps) {
        const int64_t w = b / rb, r32 = b - w * rb;  // source word column, destination word column
        const int64_t r = 32 * r32 + lane;
        const uint32_t v = (r < rows) ? words[r * ldw + w] : 0u;
        uint32_t mine = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const uint32_t bk = __ballot_sync(0xffffffffu, (v >> k) & 1u);
            if (lane == k) mine = bk;
        }
        const int64_t c = 32 * w + lane;
        if (c < cols) words_t[c * ldw_t + r32] = mine;
    }
    // destination row padding words [rb, ldw_t)
    const int64_t pad = ldw_t - rb;
    if (pad > 0) {
        const int64_t total = cols * pad;
        for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
             e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const int64_t c = e / pad;
            words_t[c * ldw_t + rb + (e - c * pad)] = 0u;
        }
    }
}

// Waits on an mbarrier that nothing ever arrives on; the bounded wait gives
// up after limit_ns and records DBF_ERR_TIMEOUT.
__global__ void selftest_wait_kernel(int *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait_bounded(&bar, 0, nullptr, limit_ns)) record_status(status, DBF_ERR_TIMEOUT);
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_pack(const int8_t *signs, int64_t rows, int64_t cols, uint32_t *words, int64_t ldw,
                        cudaStream_t stream) {
    const int64_t total = rows * ldw;
    const int64_t blocks = std::min<int64_t>((total * 32 + 255) / 256, 148 * 32);
    pack_kernel<<<static_cast<int>(std::max<int64_t>(blocks, 1)), 256, 0, stream>>>(signs, rows, cols, words, ldw);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw, int8_t *signs,
                          cudaStream_t stream) {
    const int64_t total = rows * cols;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 148 * 32);
    unpack_kernel<<<static_cast<int>(std::max<int64_t>(blocks, 1)), 256, 0, stream>>>(words, rows, cols, ldw,
                                                                                      signs);
    return cudaGetLastError();
}

cudaError_t launch_transpose(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw, uint32_t *words_t,
                             int64_t ldw_t, cudaStream_t stream) {
    const int64_t blocks = ((rows + 31) / 32) * ((cols + 31) / 32);
    const int64_t ctas = std::min<int64_t>(std::max<int64_t>((blocks + 7) / 8, (cols * (ldw_t - (rows + 31) / 32) + 255) / 256),
                                           148 * 32);
    transpose_kernel<<<static_cast<int>(std::max<int64_t>(ctas, 1)), 256, 0, stream>>>(words, rows, cols, ldw, words_t,
                                                                                      ldw_t);
    return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int *status, uint64_t limit_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace dbfk
