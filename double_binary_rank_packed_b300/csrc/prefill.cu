// Prefill-regime kernels: the same product for thousands of tokens, where the
// two sign contractions are genuine dense GEMMs (DBF page, section 2,
// "Cálculo en la inferencia": ((((X . b^T) B^T) . m^T) A^T) . a^T).
//
// Layout of one projection:
//   prologue   X'[t*ell+i][k]  = fp16(gamma_i[k] * x[t][k])          (activation order)
//   gemm<1>    V [t*ell+i][r]  = fp16(beta_i[r] * sum_k B2[r][k] X'[t*ell+i][k])
//   gemm<2>    y [t][n]        = bf16(sum_i alpha_i[n] * sum_r B1[n][r] V[t*ell+i][r])
//
// GEMM design (one CTA = 128 weight rows x BN activation rows, 192 threads):
//   warp 0      TMA producer: 64-wide K slices of the activation tile
//               (128-byte swizzle) into a 6-stage shared-memory ring
//   warp 1      allocates tensor memory and issues tcgen05.mma
//   (both loops run on the whole converged warp, one elect.sync lane issuing:
//   a loop run by one lane alone left the tensor pipe near half rate)
//   warps 2..5  unpack: each thread owns one weight row (= one TMEM lane),
//               reads two packed words per K step and writes 32 columns of
//               +-1 fp16 pairs straight into tensor memory with tcgen05.st;
//               the MMA reads that as its A operand.  Afterwards the same
//               warps run the epilogue from the fp32 accumulator.
// The sign matrix never goes through shared memory, which leaves the shared
// memory bandwidth to the activation operand.  Every mbarrier wait is
// bounded; a timeout records DBF_ERR_TIMEOUT, drains in-flight copies and
// MMAs, frees tensor memory and exits.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dbfk {

namespace {

constexpr int kPfThreads = 192;
constexpr int kBK = 64;  // K elements per stage (128 bytes of fp16)

// Tile layouts.  BN <= 192 (192, or 176 and 160 for ell <= 2, which leave a
// smaller last wave): two CTAs per SM, each with 256 tensor-memory columns
// (accumulator [0, BN), a 2-stage ring of A slices from column 192) and a
// 4-stage shared-memory ring; the two CTAs interleave their MMA streams and
// hide each other's tile prologue and epilogue.  Wider tiles: one CTA per SM,
// 6-stage rings, all 512 columns.  The A ring (signs in tensor memory) and
// the activation ring (shared memory) have their own barriers.
template <int BN>
struct PfSmem {
    static constexpr bool kPair = BN <= 192;
    static constexpr int kStages = kPair ? 4 : 6;    // shared-memory ring
    static constexpr int kAStages = kPair ? 2 : 6;   // tensor-memory ring
    static constexpr uint32_t kTmemCols = kPair ? 256 : 512;
    static constexpr uint32_t kAOff = kPair ? 192 : 256;  // first A-ring column
    static constexpr int kTileBytes = BN * 128;
    static constexpr int kBarOffset = kStages * kTileBytes;
    static constexpr int kBytes = kBarOffset + 256 + 1024;  // + barriers + alignment slack
    static_assert(kAOff >= BN && kAOff + 32 * kAStages <= kTmemCols, "tensor memory layout");
    static_assert(!kPair || 3 * (kBytes + 1024) > 228 * 1024, "a third CTA must not fit next to two");
    static_assert(2 * kStages + 2 * kAStages + 2 <= 30, "barrier area");
};

__device__ __forceinline__ uint32_t tmem_lane_base(int q) { return static_cast<uint32_t>(32 * q) << 16; }

// Copy the reduction operand of one tile into shared memory, row-major with
// 128 halves per line (the tile's 128 weight rows): stage 1 the BN columns of
// H (line c = activation row col0 + c, positions row0 .. row0+127 of V's
// layout), stage 2 the BN/ELL tokens of red_src (line t = token col0/ELL + t,
// rows row0 .. row0+127).  Entries outside the matrices are 0.  e = 0..127.
template <int STAGE, int BN, int ELL>
__device__ __forceinline__ void stage_reduction_tile(const PfArgs &a, unsigned char *smem, int row0, int col0, int e) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the ring was last used by TMA and MMA
    uint4 *dst = reinterpret_cast<uint4 *>(smem);
    // 16-byte cp.async copies, all in flight at once; a source size of 0 writes zeros
    // the operand's base (16-byte aligned whenever copies are issued) stands in for empty sources
    const void *base = (STAGE == 1) ? static_cast<const void *>(a.h_in) : static_cast<const void *>(a.red_src);
    auto copy16 = [&](int v, const void *src, bool in) {
        const void *p = in ? src : base;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst + v)), "l"(p),
                     "r"(in ? 16 : 0)
                     : "memory");
    };
    if constexpr (STAGE == 1) {
        // lines = BN columns, 16 vectors of 8 halves each; ldv is a multiple of 64
        for (int v = e; v < BN * 16; v += 128) {
            const int c = v >> 4, q = v & 15;
            const int col = col0 + c, p = row0 + 8 * q;
            const bool in = col < a.C && p + 8 <= a.ldv;
            copy16(v, a.h_in + (in ? static_cast<size_t>(col) * a.ldv + p : 0), in);
        }
    } else {
        constexpr int NT = BN / ELL;
        const int T = a.C / ELL, t0 = col0 / ELL;
        const bool vec = (a.ld_src % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.red_src) & 15) == 0);
        for (int v = e; v < NT * 16; v += 128) {
            const int tl = v >> 4, q = v & 15;
            const int t = t0 + tl, n = row0 + 8 * q;
            const __nv_bfloat16 *src = a.red_src + static_cast<size_t>(t < T ? t : 0) * a.ld_src + n;
            if (vec && (t >= T || n + 8 <= a.rows)) {
                copy16(v, src, t < T);
            } else {
                // unaligned rows or the last partial vector of a row: element copies
                uint16_t h[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    h[j] = (t < T && n + j < a.rows) ? reinterpret_cast<const uint16_t *>(src)[j] : uint16_t(0);
                dst[v] = make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                                    h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
            }
        }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <int BN, int STAGE, int ELL>
__global__ void __launch_bounds__(kPfThreads, 1) pf_gemm_kernel(const __grid_constant__ CUtensorMap act_map,
                                                                 const PfArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int kStages = PfSmem<BN>::kStages, kAStages = PfSmem<BN>::kAStages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + PfSmem<BN>::kBarOffset);
    uint64_t *act_full = bars;                 // [kStages] activation slice landed
    uint64_t *empty = bars + kStages;          // [kStages] MMAs that read the slice are done
    uint64_t *a_full = bars + 2 * kStages;     // [kAStages] 128 unpack threads wrote the A slice
    uint64_t *a_empty = a_full + kAStages;     // [kAStages] MMAs that read the A slice are done
    uint64_t *acc_full = a_empty + kAStages;   // [1]
    uint64_t *drain = acc_full + 1;            // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    constexpr uint32_t kTmemCols = PfSmem<BN>::kTmemCols;
    constexpr uint32_t kAccCols = PfSmem<BN>::kAOff;  // accumulator columns [0, BN), the A ring after
    constexpr uint32_t kIdesc = idesc_f16_f32(128, BN);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // weight row blocks vary fastest across the grid: the CTAs resident at one
    // time share a few activation tiles, which stay in L2 while every row
    // block of the weights consumes them
    const int row0 = blockIdx.x * 128;  // first weight row
    const int col0 = blockIdx.y * BN;   // first activation row (token*ell + term)
    const int nk = a.nk;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&act_full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&a_full[s], 128);
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&act_map);
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        // the whole warp runs the loop; one elected lane issues each copy
        pdl_wait();  // the activations are written by the previous kernel
        int issued = 0;
        for (int ks = 0; ks < nk; ++ks) {
            const int s = ks % kStages;
            const uint32_t n = ks / kStages;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], (n & 1) ^ 1, abort_flag))) {
                *abort_flag = 1;
                record_status(a.status, DBF_ERR_TIMEOUT);
                break;
            }
            if (elect_one()) {
                mbar_arrive_expect_tx(&act_full[s], PfSmem<BN>::kTileBytes);
                tma_load_2d(smem + s * PfSmem<BN>::kTileBytes, &act_map, &act_full[s], ks * kBK, col0);
            }
            __syncwarp();
            ++issued;
        }
        if (*abort_flag && lane == 0) {
            // let every copy still in flight land before the block can exit
            for (int ks = (issued > kStages ? issued - kStages : 0); ks < issued; ++ks)
                mbar_wait_bounded(&act_full[ks % kStages], (ks / kStages) & 1, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // the whole warp runs the loop; one elected lane issues the MMAs and
        // the commits
        for (int ks = 0; ks < nk; ++ks) {
            const int s = ks % kStages, sa = ks % kAStages;
            const bool ready = mbar_wait_bounded(&act_full[s], (ks / kStages) & 1, abort_flag) &&
                               mbar_wait_bounded(&a_full[sa], (ks / kAStages) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ready)) {
                *abort_flag = 1;
                record_status(a.status, DBF_ERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t a_col = tmem + kAccCols + sa * 32;
            const uint32_t b_addr = smem_u32(smem + s * PfSmem<BN>::kTileBytes);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    tc_mma_ts(tmem, a_col + kk * 8, desc_sw128(b_addr + kk * 32), kIdesc, (ks | kk) != 0);
                tc_commit(&empty[s]);
                tc_commit(&a_empty[sa]);
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
        // ------------------------------------------------ unpack, then epilogue
        const int q = warp & 3;                // TMEM lane quarter this warp may access
        const int row = row0 + 32 * q + lane;  // weight row == TMEM lane
        const bool row_ok = row < a.rows;
        const uint32_t *wrow = a.bits + static_cast<size_t>(row_ok ? row : 0) * a.ldw;
        const uint32_t lane_addr = tmem_lane_base(q);
        uint32_t cur[8], nxt[8];
        auto load_block = [&](uint32_t (&dst)[8], int kb) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int w = kb * 8 + j;
                dst[j] = (row_ok && w < a.Kw) ? __ldg(wrow + w) : 0u;
            }
        };
        const int nkb = (nk + 3) / 4;
        load_block(cur, 0);
        bool ok = true;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            if (kb + 1 < nkb) load_block(nxt, kb + 1);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int ks = kb * 4 + u;
                if (ks >= nk || !ok) break;
                const int s = ks % kAStages;
                const uint32_t n = ks / kAStages;
                // warp-uniform decision: tcgen05.st below is a warp-collective instruction
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&a_empty[s], (n & 1) ^ 1, abort_flag))) {
                    *abort_flag = 1;
                    record_status(a.status, DBF_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                tc_fence_after();  // the MMAs that read this stage are complete
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    v[j] = sign_pair(cur[2 * u], 15 - j);
                    v[16 + j] = sign_pair(cur[2 * u + 1], 15 - j);
                }
                tmem_st_32x32b_x32(tmem + lane_addr + kAccCols + s * 32, v);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&a_full[s]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
        }

        // epilogue
        pdl_wait();  // outputs may still be read by the previous kernel
        const bool acc_ready = ok && __all_sync(0xffffffffu, mbar_wait_bounded(acc_full, 0, abort_flag));
        // backward reductions: the tile of the second operand (H for stage 1, dy or x for stage 2)
        // is staged in the ring, idle once the accumulator is complete, with one batch of
        // coalesced loads instead of a dependent load per accumulator chunk
        const __half *stile = reinterpret_cast<const __half *>(smem);
        const bool staged = (STAGE == 1) ? (a.h_in != nullptr) : (a.red_src != nullptr);
        if (staged) {
            if (acc_ready) stage_reduction_tile<STAGE, BN, ELL>(a, smem, row0, col0, threadIdx.x - 64);
            asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
        }
        if (acc_ready) {
            tc_fence_after();
            if constexpr (STAGE == 1) {
                // V[c][perm(row)] = fp16(beta_{c%ELL}[row] * acc), 0 for rows >= R
                float bsc[ELL];
#pragma unroll
                for (int i = 0; i < ELL; ++i)
                    bsc[i] = row_ok ? __half2float(a.beta[static_cast<size_t>(i) * a.rows + row]) : 0.f;
                const bool store_row = row < a.rows_store;  // whole 32-row groups agree
                const int pos = (row & ~31) + 2 * (lane & 15);
                const int own_pos = pos + (lane >> 4);      // where this lane's own row lands
                float red_part[ELL];
#pragma unroll
                for (int i = 0; i < ELL; ++i) red_part[i] = 0.f;
                constexpr int CW = 8 * ELL;  // columns per chunk (whole tokens)
                for (int cb = 0; cb < BN; cb += CW) {
                    uint32_t raw[32];
                    if constexpr (CW == 8) {
                        uint32_t (&r8)[8] = *reinterpret_cast<uint32_t(*)[8]>(raw);
                        tmem_ld_32x32b_x8(tmem + lane_addr + cb, r8);
                    } else if constexpr (CW == 16) {
                        tmem_ld_32x32b_x16(tmem + lane_addr + cb, raw);
                    } else if constexpr (CW == 24) {
                        tmem_ld_32x32b_x16(tmem + lane_addr + cb, raw);
                        uint32_t (&r8)[8] = *reinterpret_cast<uint32_t(*)[8]>(raw + 16);
                        tmem_ld_32x32b_x8(tmem + lane_addr + cb + 16, r8);
                    } else {
                        tmem_ld_32x32b_x16(tmem + lane_addr + cb, raw);
                        tmem_ld_32x32b_x16(tmem + lane_addr + cb + 16, raw + 16);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < CW; j += 2) {
                        const float v0 = bsc[j % ELL] * __uint_as_float(raw[j]);
                        const float v1 = bsc[(j + 1) % ELL] * __uint_as_float(raw[j + 1]);
                        // lanes s and s+16 hold rows that land at positions 2s and 2s+1
                        const float send = (lane < 16) ? v1 : v0;
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        const int c = col0 + cb + j + (lane < 16 ? 0 : 1);
                        const __half2 h = (lane < 16) ? __floats2half2_rn(v0, recv) : __floats2half2_rn(recv, v1);
                        if (store_row && c < a.C && in_range(pos + 1 < a.ldv, a.status))
                            *reinterpret_cast<__half2 *>(a.V + static_cast<size_t>(c) * a.ldv + pos) = h;
                        if (a.h_out) {
                            // the unscaled product, same layout
                            const float u0 = __uint_as_float(raw[j]), u1 = __uint_as_float(raw[j + 1]);
                            const float usend = (lane < 16) ? u1 : u0;
                            const float urecv = __shfl_xor_sync(0xffffffffu, usend, 16);
                            const __half2 hu =
                                (lane < 16) ? __floats2half2_rn(u0, urecv) : __floats2half2_rn(urecv, u1);
                            if (store_row && c < a.C)
                                *reinterpret_cast<__half2 *>(a.h_out + static_cast<size_t>(c) * a.ldv + pos) = hu;
                        }
                    }
                    if (a.h_in && row_ok) {
                        // dbeta: acc(t, i) * H[t*ell+i][row], summed over this tile's tokens
                        // (columns past C were staged as 0)
#pragma unroll
                        for (int j = 0; j < CW; ++j)
                            red_part[j % ELL] +=
                                __uint_as_float(raw[j]) * __half2float(stile[(cb + j) * 128 + (own_pos - row0)]);
                    }
                }
                if (a.red && row_ok) {
#pragma unroll
                    for (int i = 0; i < ELL; ++i) atomicAdd(a.red + static_cast<size_t>(i) * a.rows + row, red_part[i]);
                }
            } else {
                // y[t][row] = bf16(sum_i alpha_i[row] * acc[t*ELL+i] (+ y))
                float asc[ELL];
#pragma unroll
                for (int i = 0; i < ELL; ++i)
                    asc[i] = row_ok ? __half2float(a.alpha[static_cast<size_t>(i) * a.rows + row]) : 0.f;
                const bool paired = (a.ldy % 2 == 0) && (a.rows_store % 2 == 0);
                constexpr int CW = 8 * ELL;
                const int T = a.C / ELL;
                float red_part[ELL];
#pragma unroll
                for (int i = 0; i < ELL; ++i) red_part[i] = 0.f;
                for (int cb = 0; cb < BN; cb += CW) {
                    uint32_t raw[32];
                    if constexpr (CW == 8) {
                        uint32_t (&r8)[8] = *reinterpret_cast<uint32_t(*)[8]>(raw);
                        tmem_ld_32x32b_x8(tmem + lane_addr + cb, r8);
                    } else if constexpr (CW == 16) {
                        tmem_ld_32x32b_x16(tmem + lane_addr + cb, raw);
                    } else if constexpr (CW == 24) {
                        tmem_ld_32x32b_x16(tmem + lane_addr + cb, raw);
                        uint32_t (&r8)[8] = *reinterpret_cast<uint32_t(*)[8]>(raw + 16);
                        tmem_ld_32x32b_x8(tmem + lane_addr + cb + 16, r8);
                    } else {
                        tmem_ld_32x32b_x16(tmem + lane_addr + cb, raw);
                        tmem_ld_32x32b_x16(tmem + lane_addr + cb + 16, raw + 16);
                    }
                    tmem_ld_wait();
                    const int tb = (col0 + cb) / ELL;
                    if (a.red_src && row_ok) {
                        // dalpha / dgamma: red_src[t][row] * acc(t, i), summed over this tile's tokens
                        // (tokens past T were staged as 0)
                        const __nv_bfloat16 *st = reinterpret_cast<const __nv_bfloat16 *>(smem);
#pragma unroll
                        for (int tt = 0; tt < 8; ++tt) {
                            const float src = __bfloat162float(st[(cb / ELL + tt) * 128 + (row - row0)]);
#pragma unroll
                            for (int i = 0; i < ELL; ++i) red_part[i] += src * __uint_as_float(raw[tt * ELL + i]);
                        }
                    }
                    if (a.skip_store) continue;
                    float out[8];
#pragma unroll
                    for (int tt = 0; tt < 8; ++tt) {
                        float s = 0.f;
#pragma unroll
                        for (int i = 0; i < ELL; ++i) s += asc[i] * __uint_as_float(raw[tt * ELL + i]);
                        out[tt] = s;
                    }
                    if (paired) {
#pragma unroll
                        for (int tt = 0; tt < 8; tt += 2) {
                            // even lanes write tokens tt, odd lanes tokens tt+1, as bf16 pairs (n, n+1)
                            const bool even = (lane & 1) == 0;
                            const float send = even ? out[tt + 1] : out[tt];
                            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                            const int t = tb + tt + (even ? 0 : 1);
                            const int n = even ? row : row - 1;
                            float lo = even ? out[tt] : recv;
                            float hi = even ? recv : out[tt + 1];
                            if (t < T && n < a.rows_store && in_range(n + 1 < a.ldy, a.status)) {
                                __nv_bfloat162 *yp =
                                    reinterpret_cast<__nv_bfloat162 *>(a.y + static_cast<size_t>(t) * a.ldy + n);
                                if (a.accumulate) {
                                    const float2 old = __bfloat1622float2(*yp);
                                    lo += old.x;
                                    hi += old.y;
                                }
                                *yp = __floats2bfloat162_rn(lo, hi);
                            }
                        }
                    } else {
#pragma unroll
                        for (int tt = 0; tt < 8; ++tt) {
                            const int t = tb + tt;
                            if (t < T && row < a.rows_store && in_range(row < a.ldy, a.status)) {
                                __nv_bfloat16 *yp = a.y + static_cast<size_t>(t) * a.ldy + row;
                                float s = out[tt];
                                if (a.accumulate) s += __bfloat162float(*yp);
                                *yp = __float2bfloat16_rn(s);
                            }
                        }
                    }
                }
                if (a.red && row_ok) {
#pragma unroll
                    for (int i = 0; i < ELL; ++i) atomicAdd(a.red + static_cast<size_t>(i) * a.rows + row, red_part[i]);
                }
            }
        } else {
            *abort_flag = 1;
            record_status(a.status, DBF_ERR_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// x [T][M] bf16 -> X' [T*ell + i][ldxs] fp16 in activation order, zero past M.
// One thread per (token, 32-group g, half q): the 8 k at 32g + 8q and the 8
// at 32g + 8q + 16 become the 16 consecutive logical positions 32g + 16q ..
// (see perm32_pos), written as two 16-byte stores per term.  16-byte loads
// of x and gamma when M is a multiple of 8, element loads otherwise.
__global__ void pf_prologue_kernel(const __nv_bfloat16 *__restrict__ x, int T, int M, int ldx,
                                   const __half *__restrict__ gamma, int ell, __half *__restrict__ xs, int ldxs) {
    pdl_trigger();
    pdl_wait();
    const int groups = ldxs / 32;
    const bool vec = ((M & 7) == 0) && ((ldx & 7) == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(gamma) & 15) == 0);
    const int64_t total = static_cast<int64_t>(T) * groups * 2;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int q = static_cast<int>(e & 1);
        const int64_t tg = e >> 1;
        const int g = static_cast<int>(tg % groups);
        const int t = static_cast<int>(tg / groups);
        const int k0 = 32 * g + 8 * q;  // first physical k of the low half; the high half is k0 + 16
        const __nv_bfloat16 *xr = x + static_cast<size_t>(t) * ldx;
        float xa[8], xb[8];
        if (vec && k0 + 24 <= M) {
            const uint4 va = *reinterpret_cast<const uint4 *>(xr + k0);
            const uint4 vb = *reinterpret_cast<const uint4 *>(xr + k0 + 16);
            const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                xa[2 * j] = __uint_as_float(wa[j] << 16);
                xa[2 * j + 1] = __uint_as_float(wa[j] & 0xFFFF0000u);
                xb[2 * j] = __uint_as_float(wb[j] << 16);
                xb[2 * j + 1] = __uint_as_float(wb[j] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                xa[j] = (k0 + j < M) ? __bfloat162float(xr[k0 + j]) : 0.f;
                xb[j] = (k0 + 16 + j < M) ? __bfloat162float(xr[k0 + 16 + j]) : 0.f;
            }
        }
        for (int i = 0; i < ell; ++i) {
            const __half *gi = gamma + static_cast<size_t>(i) * M;
            float ga[8], gb[8];
            if (vec && k0 + 24 <= M) {
                const uint4 ua = *reinterpret_cast<const uint4 *>(gi + k0);
                const uint4 ub = *reinterpret_cast<const uint4 *>(gi + k0 + 16);
                const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&wa[j]));
                    const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&wb[j]));
                    ga[2 * j] = fa.x;
                    ga[2 * j + 1] = fa.y;
                    gb[2 * j] = fb.x;
                    gb[2 * j + 1] = fb.y;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    ga[j] = (k0 + j < M) ? __half2float(gi[k0 + j]) : 0.f;
                    gb[j] = (k0 + 16 + j < M) ? __half2float(gi[k0 + 16 + j]) : 0.f;
                }
            }
            uint32_t out[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __half2 h = __floats2half2_rn(ga[j] * xa[j], gb[j] * xb[j]);
                out[j] = *reinterpret_cast<const uint32_t *>(&h);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(xs + (static_cast<size_t>(t) * ell + i) * ldxs + 32 * g + 16 * q);
            dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
            dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
        }
    }
}

template <int BN, int STAGE, int ELL>
cudaError_t launch_gemm_t(const CUtensorMap &map, const PfArgs &a, cudaStream_t stream, bool pdl) {
    auto kern = pf_gemm_kernel<BN, STAGE, ELL>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmem<BN>::kBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int rows_cover = (STAGE == 1) ? a.rows_store : a.rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows_cover + 127) / 128, (a.C + BN - 1) / BN, 1);
    cfg.blockDim = dim3(kPfThreads, 1, 1);
    cfg.dynamicSmemBytes = PfSmem<BN>::kBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, map, a);
}

template <int STAGE>
cudaError_t launch_gemm_stage(const CUtensorMap &map, const PfArgs &a, int bn, cudaStream_t stream, bool pdl) {
    switch (a.ell * 1000 + bn) {
        case 1256: return launch_gemm_t<256, STAGE, 1>(map, a, stream, pdl);
        case 1240: return launch_gemm_t<240, STAGE, 1>(map, a, stream, pdl);
        case 1192: return launch_gemm_t<192, STAGE, 1>(map, a, stream, pdl);
        case 1176: return launch_gemm_t<176, STAGE, 1>(map, a, stream, pdl);
        case 1160: return launch_gemm_t<160, STAGE, 1>(map, a, stream, pdl);
        case 2256: return launch_gemm_t<256, STAGE, 2>(map, a, stream, pdl);
        case 2240: return launch_gemm_t<240, STAGE, 2>(map, a, stream, pdl);
        case 2192: return launch_gemm_t<192, STAGE, 2>(map, a, stream, pdl);
        case 2176: return launch_gemm_t<176, STAGE, 2>(map, a, stream, pdl);
        case 2160: return launch_gemm_t<160, STAGE, 2>(map, a, stream, pdl);
        case 3240: return launch_gemm_t<240, STAGE, 3>(map, a, stream, pdl);
        case 3192: return launch_gemm_t<192, STAGE, 3>(map, a, stream, pdl);
        case 4256: return launch_gemm_t<256, STAGE, 4>(map, a, stream, pdl);
        case 4224: return launch_gemm_t<224, STAGE, 4>(map, a, stream, pdl);
        case 4192: return launch_gemm_t<192, STAGE, 4>(map, a, stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Activation rows per tile of one GEMM launch.  The candidates are multiples
// of 16 (MMA N) and of 8*ell (whole tokens per epilogue chunk); the model is
// the slowest SM: whole waves of tiles times the time of a wave.  One CTA per
// SM: a K step measured max(2*BN, ~400) cycles for a 128-row tile with its A
// operand in tensor memory, plus a tile's prologue, pipeline fill and
// epilogue (~8 us, from the gap between that rate and the measured GEMMs).
// Two CTAs per SM (BN <= 192): their MMA streams keep the pipe busy at 2*BN
// cycles a step each, and the per-tile costs overlap the other CTA's MMAs.
// Equal costs keep the first candidate.  0 when no candidate keeps the grid's
// second dimension within 65535.
int prefill_pick_bn(int ell, int rows_cover, int64_t C, int nk, int num_sms) {
    static const int w12[] = {256, 240, 192, 176, 160}, w3[] = {240, 192}, w4[] = {256, 224, 192};
    const int *w = (ell == 3) ? w3 : (ell == 4 ? w4 : w12);
    const int nw = (ell == 3) ? 2 : (ell == 4 ? 3 : 5);
    const int64_t rb = (rows_cover + 127) / 128;
    const double tile_cost = 15000.0;  // cycles
    int best = 0;
    double best_cost = 1e300;
    for (int k = 0; k < nw; ++k) {
        const int64_t cb = (C + w[k] - 1) / w[k];
        if (cb > 65535) continue;
        const double tiles = double(rb * cb);
        const int sms = std::max(num_sms, 1);
        double cost;
        if (w[k] <= 192)
            cost = std::ceil(tiles / (2.0 * sms)) * (2.0 * nk * 2.0 * w[k] + 0.5 * tile_cost);
        else
            cost = std::ceil(tiles / sms) * (nk * std::max(2.0 * w[k], 400.0) + tile_cost);
        if (cost < best_cost * (1.0 - 1e-9)) {
            best_cost = cost;
            best = w[k];
        }
    }
    return best;
}

cudaError_t launch_prefill_prologue(const __nv_bfloat16 *x, int T, int M, int ldx, const __half *gamma, int ell,
                                    __half *xs, int ldxs, cudaStream_t stream, bool pdl) {
    const int64_t total = static_cast<int64_t>(T) * (ldxs / 32) * 2;
    int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 148 * 16));
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, pf_prologue_kernel, x, T, M, ldx, gamma, ell, xs, ldxs);
}

cudaError_t launch_prefill_gemm(int stage, const CUtensorMap &act_map, const PfArgs &args, int bn,
                                cudaStream_t stream, bool pdl) {
    return stage == 1 ? launch_gemm_stage<1>(act_map, args, bn, stream, pdl)
                      : launch_gemm_stage<2>(act_map, args, bn, stream, pdl);
}

// Tensor map over an fp16 activation matrix [rows][ld] (logical K extent
// cols_pad), box = 64 K elements x box_rows rows, 128-byte swizzle, zero fill
// outside the matrix.
bool encode_act_map(CUtensorMap *map, const __half *base, int rows, int cols_pad, int ld, int box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols_pad), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace dbfk
