// Host-side launchers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dbf.h"

namespace dbfk {

// ----------------------------------------------------------- decode path

// Arguments of one decode stage launch.  Stage 1 contracts x (scaled by
// gamma) with B2 and writes V = beta * u in fp16 (activation order); stage 2
// contracts V with B1 and writes y = sum_i alpha_i * w_i in bf16.
struct DecArgs {
    const uint32_t *bits;   // packed weights of this stage (B2 or B1)
    int ldw;                // words per packed row
    int rows;               // weight rows (R or N)
    int rows_cover;         // rows the launch covers (stage 1: round_up(R, 32))
    int Kw;                 // packed words per row that hold data (ceil(K/32))
    int K;                  // contraction length (M or R)
    int ell;
    int T;                  // tokens (plain mode)
    const __nv_bfloat16 *x; // stage 1 input [T][M]
    int ldx;
    const __half *gamma;    // [ell][M]
    const __half *beta;     // [ell][R]
    __half *V;              // [ell*T][ldv] fp16 intermediate
    int ldv;
    const __half *alpha;    // [ell][N]
    __nv_bfloat16 *y;       // [T][ldy]
    int ldy;
    int accumulate;
    int RB;                 // 16-row blocks per CTA (1, 2, 4 or 8)
    int KS;                 // CTAs per cluster along K
    int Wc;                 // packed words per CTA K-slice
    // multi-adapter mode
    const int32_t *seg_off;
    const int32_t *seg_ad;
    const dbf_factors *adapters;
    int n_adapters;
    int *status;
};

struct DecPlan {
    int CT;          // n8 column tiles (columns per chunk = 8*CT)
    int RB, KS, Wc;
    int grid_x;
    size_t smem;
};

DecPlan plan_decode_stage(int rows_cover, int Kw, int columns, int max_ct, int num_sms);

// One-launch decode for small R: a cluster splits stage 1 over K, shares
// the partial u through distributed shared memory, then each CTA computes
// its slice of the N output rows.
struct FusedArgs {
    const uint32_t *B1, *B2;
    int ldw1, ldw2;
    const __half *alpha, *beta, *gamma;
    int N, M, R, ell, T;
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    int accumulate;
    int KS;    // cluster size (stage-1 K split)
    int RB2;   // stage-2 row blocks (16 rows) per CTA
    int Wc1;   // stage-1 packed words per CTA
    const int32_t *seg_off;
    const int32_t *seg_ad;
    const dbf_factors *adapters;
    int n_adapters;
    int *status;
};

struct FusedPlan {
    int CT, KS, NQ, RB2, Wc1, grid_x;
    size_t smem;
};

// problems: independent calls launched together (segments); the grid is
// problems x grid_x CTAs.
FusedPlan plan_fused(int N, int M, int R, int ell, int columns, int num_sms, int problems, bool accumulate);
cudaError_t launch_decode_fused(bool segmented, const FusedPlan &plan, const FusedArgs &args, int grid_y,
                                cudaStream_t stream, bool pdl);
size_t decode_smem_bytes(int CT, int RB, int Wc);
cudaError_t launch_decode_stage(int stage, bool segmented, const DecPlan &plan, const DecArgs &args,
                                int grid_y, cudaStream_t stream, bool pdl);

// ---------------------------------------------------------- prefill path

struct PfArgs {
    const uint32_t *bits;   // packed weights (B2 for stage 1, B1 for stage 2)
    int ldw;
    int rows;               // weight rows (R or N)
    int rows_store;         // stage 1: ldv (V row length); stage 2: N
    int Kw;                 // ceil(K/32)
    int nk;                 // k-steps of 64
    int C;                  // activation rows (ell*T)
    int ell;
    const __half *beta;     // stage 1 epilogue
    __half *V;
    int ldv;
    const __half *alpha;    // stage 2 epilogue
    __nv_bfloat16 *y;
    int ldy;
    int accumulate;
    int *status;
};

cudaError_t launch_prefill_prologue(const __nv_bfloat16 *x, int T, int M, int ldx, const __half *gamma, int ell,
                                    __half *xs, int ldxs, cudaStream_t stream, bool pdl);
cudaError_t launch_prefill_gemm(int stage, const CUtensorMap &act_map, const PfArgs &args, int bn,
                                cudaStream_t stream, bool pdl);
int prefill_bn(int ell);
bool encode_act_map(CUtensorMap *map, const __half *base, int rows, int cols_pad, int ld, int box_rows);

// --------------------------------------------------------------- misc

cudaError_t launch_pack(const int8_t *signs, int64_t rows, int64_t cols, uint32_t *words, int64_t ldw,
                        cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw, int8_t *signs,
                          cudaStream_t stream);
cudaError_t launch_selftest_wait(int *status, uint64_t limit_ns, cudaStream_t stream);

// Text returned by dbf_last_cuda_error() on this thread.
void set_last_error(const char *msg);

}  // namespace dbfk
