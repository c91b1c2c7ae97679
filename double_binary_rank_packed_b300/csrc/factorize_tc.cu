// Tensor-core GEMM of the double binary factorization (DBF page, section 2,
// "Factorización"; the ADMM P-update Y = RHS (F F^T + rho I)^-1 of each
// iteration, and T F^T): C = alpha * A B^T + beta * C with fp32 A [m x kk], B [n x kk]
// in memory, on tcgen05.mma kind::tf32 with fp32 accumulation in tensor
// memory.
//
// fp32 accuracy from tf32 products: every operand x is split into
// hi = tf32(x) and lo = tf32(x - hi), and A B^T is taken as
// A_hi B_hi^T + A_hi B_lo^T + A_lo B_hi^T (the lo * lo term is below fp32's
// resolution).  A matrix in split form holds each row as [hi | lo], each
// half kk2 = kk rounded up to 32 wide (zero past kk), so one split serves as
// either operand; the kernel runs the three products as three passes over K
// that read the (hi, hi), (hi, lo) and (lo, hi) halves, all accumulating
// into one TMEM tile.  The split forms are written by fz_split2_kernel here
// and by the dual pass of factorize.cu for the right-hand side.
//
// Tile 128 x 256 (one CTA per SM: a 4-stage TMA ring of 48 KB stages), K step
// 32 fp32 (one 128-byte swizzle row); warp 0 loads the ring with TMA, warp 1
// issues the MMAs (M 128, N 256, K 8; four per K step) and owns the tensor
// memory, warps 2..5 read the accumulator back (tcgen05.ld) and write C.
// Every wait is bounded: a timeout records DBF_ERR_TIMEOUT, lets the copies
// and MMAs in flight finish, frees the tensor memory and exits.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "factorize.h"

namespace dbfk {

namespace {

constexpr int kTcBM = 128, kTcBN = 256, kTcBK = 32, kTcStages = 4;
constexpr int kTcThreads = 192;
constexpr uint32_t kTcABytes = kTcBM * kTcBK * 4;          // 16 KB
constexpr uint32_t kTcBBytes = kTcBN * kTcBK * 4;          // 32 KB
constexpr uint32_t kTcStageBytes = kTcABytes + kTcBBytes;  // 48 KB, 1024-byte aligned
constexpr uint32_t kTcBarOffset = kTcStages * kTcStageBytes;
constexpr uint32_t kTcSmem = kTcBarOffset + 128 + 1024;    // + barriers, + alignment slack
constexpr uint32_t kTcTmemCols = 256;

// Instruction descriptor of kind::tf32: tf32 A and B (format 2), fp32 D,
// both K-major, tile M x N (same bit layout as kind::f16).
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D(tmem) (+)= A(smem descriptor) * B(smem descriptor)^T, kind::tf32, one CTA.
__device__ __forceinline__ void tc_mma_ss_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1)
    fz_tc_gemm_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap b_map, int m,
                      int n, int kk2, float alpha, float beta, float *C, int64_t ldc, int lower, int *status) {
    extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kTcBarOffset);
    uint64_t *full = bars;                   // [kTcStages] A and B tiles of the stage landed
    uint64_t *empty = bars + kTcStages;      // [kTcStages] the MMAs that read the stage are done
    uint64_t *acc_full = bars + 2 * kTcStages;
    uint64_t *drain = acc_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    constexpr uint32_t kIdesc = idesc_tf32_f32(kTcBM, kTcBN);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.y * kTcBM, col0 = blockIdx.x * kTcBN;
    if (lower && col0 >= row0 + kTcBM) return;  // the whole tile is above the diagonal
    const int kpass = kk2 / kTcBK;              // K steps of one product
    const int nk = 3 * kpass;                   // (hi, hi), (hi, lo), (lo, hi)

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&a_map);
        tma_prefetch_desc(&b_map);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTcTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        int issued = 0;
        for (int ks = 0; ks < nk; ++ks) {
            const int s = ks % kTcStages;
            const uint32_t u = ks / kTcStages;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], (u & 1) ^ 1, abort_flag))) {
                *abort_flag = 1;
                record_status(status, DBF_ERR_TIMEOUT);
                break;
            }
            if (elect_one()) {
                unsigned char *st = smem + s * kTcStageBytes;
                const int pass = ks / kpass, kin = (ks - pass * kpass) * kTcBK;
                const int xa = (pass == 2 ? kk2 : 0) + kin, xb = (pass == 1 ? kk2 : 0) + kin;
                mbar_arrive_expect_tx(&full[s], kTcStageBytes);
                tma_load_2d(st, &a_map, &full[s], xa, row0);
                tma_load_2d(st + kTcABytes, &b_map, &full[s], xb, col0);
            }
            __syncwarp();
            ++issued;
        }
        if (*abort_flag && lane == 0) {
            // let every copy still in flight land before the block can exit
            for (int ks = (issued > kTcStages ? issued - kTcStages : 0); ks < issued; ++ks)
                mbar_wait_bounded(&full[ks % kTcStages], (ks / kTcStages) & 1, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        for (int ks = 0; ks < nk; ++ks) {
            const int s = ks % kTcStages;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (ks / kTcStages) & 1, abort_flag))) {
                *abort_flag = 1;
                record_status(status, DBF_ERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + s * kTcStageBytes);
            const uint32_t b_addr = a_addr + kTcABytes;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kTcBK / 8; ++kk)  // K 8 per MMA: 32 bytes along the swizzled row
                    tc_mma_ss_tf32(tmem, desc_sw128(a_addr + kk * 32), desc_sw128(b_addr + kk * 32), kIdesc,
                                   (ks | kk) != 0);
                tc_commit(&empty[s]);
            }
            __syncwarp();
        }
        if (elect_one()) {
            if (*abort_flag) {
                tc_commit(drain);
                mbar_wait_bounded(drain, 0, nullptr);
            } else {
                tc_commit(acc_full);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue: TMEM -> C
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = row0 + 32 * q + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        if (__all_sync(0xffffffffu, mbar_wait_bounded(acc_full, 0, abort_flag))) {
            tc_fence_after();
            const bool vec = ((ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(C) & 15) == 0);
            for (int cb = 0; cb < kTcBN; cb += 16) {
                if (col0 + cb >= n) break;  // warp-uniform
                uint32_t raw[16];
                tmem_ld_32x32b_x16(tmem + lane_addr + cb, raw);
                tmem_ld_wait();
                if (row >= m) continue;
                float *crow = C + int64_t(row) * ldc + col0 + cb;
                if (vec && col0 + cb + 16 <= n) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        float4 o = make_float4(alpha * __uint_as_float(raw[4 * v]), alpha * __uint_as_float(raw[4 * v + 1]),
                                               alpha * __uint_as_float(raw[4 * v + 2]),
                                               alpha * __uint_as_float(raw[4 * v + 3]));
                        if (beta != 0.f) {
                            const float4 c = *reinterpret_cast<const float4 *>(crow + 4 * v);
                            o.x = fmaf(beta, c.x, o.x);
                            o.y = fmaf(beta, c.y, o.y);
                            o.z = fmaf(beta, c.z, o.z);
                            o.w = fmaf(beta, c.w, o.w);
                        }
                        *reinterpret_cast<float4 *>(crow + 4 * v) = o;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (col0 + cb + j >= n) break;
                        const float o = alpha * __uint_as_float(raw[j]);
                        crow[j] = (beta != 0.f) ? fmaf(beta, crow[j], o) : o;
                    }
                }
            }
        } else {
            *abort_flag = 1;
            record_status(status, DBF_ERR_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTcTmemCols);
    }
}

// X2[r] = [hi(X[r]) | lo(X[r])], each half kk2 wide, zero past kk.  Grid: x
// over column blocks of 256 (covering kk2), y over rows.
__global__ void __launch_bounds__(256) fz_split2_kernel(const float *__restrict__ X, int64_t ldx, int kk,
                                                        float *__restrict__ X2, int kk2) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= kk2) return;
    const float x = j < kk ? X[int64_t(blockIdx.y) * ldx + j] : 0.f;
    const float hi = tf32_rna(x), lo = tf32_rna(x - hi);
    float *o = X2 + int64_t(blockIdx.y) * 2 * kk2;
    o[j] = hi;
    o[kk2 + j] = lo;
}

bool encode_f32_map(CUtensorMap *map, const float *base, int rows, int cols, int64_t ld, int box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult qr;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess || !fn)
            return false;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t tc_prepare() {
    return cudaFuncSetAttribute(fz_tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kTcSmem));
}

int tc_split_half(int kk) { return (kk + kTcBK - 1) / kTcBK * kTcBK; }

cudaError_t tc_split2(const float *X, int64_t ldx, int rows, int kk, float *X2, cudaStream_t s) {
    if (rows <= 0 || kk <= 0) return cudaSuccess;
    const int kk2 = tc_split_half(kk);
    fz_split2_kernel<<<dim3((kk2 + 255) / 256, rows), 256, 0, s>>>(X, ldx, kk, X2, kk2);
    return cudaGetLastError();
}

cudaError_t tc_gemm_nt_split(int m, int n, int kk, float alpha, const float *A2, const float *B2, float beta, float *C,
                             int64_t ldc, int *status, cudaStream_t s, int lower) {
    if (m <= 0 || n <= 0) return cudaSuccess;
    const int kk2 = tc_split_half(kk);
    CUtensorMap a_map, b_map;
    if (!encode_f32_map(&a_map, A2, m, 2 * kk2, 2 * int64_t(kk2), kTcBM) ||
        !encode_f32_map(&b_map, B2, n, 2 * kk2, 2 * int64_t(kk2), kTcBN))
        return cudaErrorInvalidValue;
    const dim3 grid((n + kTcBN - 1) / kTcBN, (m + kTcBM - 1) / kTcBM);
    fz_tc_gemm_kernel<<<grid, kTcThreads, kTcSmem, s>>>(a_map, b_map, m, n, kk2, alpha, beta, C, ldc, lower, status);
    return cudaGetLastError();
}

}  // namespace dbfk
