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

// Largest R the one-launch fused decode kernel takes (it recomputes stage 1
// in every cluster; the plan also checks its shared memory).
constexpr int kFusedMaxR = 256;

// Arguments of one decode stage launch.  Stage 1 contracts x (scaled by
// gamma) with B2 and writes V = beta * u in fp16 (activation order); stage 2
// contracts V with B1 and writes y = sum_i alpha_i * w_i in bf16.
struct DecArgs {
    const uint32_t *bits;   // packed weights of this stage (B2 or B1)
    int ldw;                // words per packed row
    int rows;               // weight rows that exist (R or N)
    int rows_out;           // rows the launch writes (stage 1: round_up(R, 32); stage 2: N)
    int Kw;                 // packed words per row that hold data (ceil(K/32))
    int K;                  // contraction length (M or R)
    int ell;
    int T;                  // tokens of the call (all segments in segmented mode)
    const __nv_bfloat16 *x; // stage 1 input [T][ldx]
    int ldx;
    const __half *gamma;    // [ell][M]
    const __half *beta;     // [ell][R]
    __half *V;              // [ell*T][ldv] fp16 intermediate
    int ldv;
    const __half *alpha;    // [ell][N]
    __nv_bfloat16 *y;       // [T][ldy]
    int ldy;
    int accumulate;
    int KS;                 // CTAs per cluster along K
    int Wc;                 // packed words per CTA K-slice
    // multi-adapter mode
    const int32_t *seg_off;
    const int32_t *seg_ad;
    const dbf_factors *adapters;
    int n_adapters;
    int *status;
};

// Grouped decode launch (several problems of different shapes, one launch
// per stage): the per-problem arguments travel as the kernel parameter.
constexpr int kMaxGroup = 16;
struct DecGroupArgs {
    int G;
    int block0[kMaxGroup + 1];  // first CTA of each problem along x; block0[G] = grid size
    DecArgs p[kMaxGroup];
};

struct DecPlan {
    int CT;          // n8 column tiles (columns per chunk = 8*CT); 0 = no plan
    int RBW;         // 16-row blocks per CTA (2 or 4)
    int KS, Wc;
    int grid_x;
    size_t smem;
};

DecPlan plan_decode_stage(int rows_cover, int Kw, int columns, int max_ct, int num_sms, int ell, bool stage1);

// One-launch decode for small R: a cluster splits stage 1 over M, shares
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
    int C;     // cluster size (stage-1 split of M)
    int Wc;    // stage-1 packed words per CTA
    int RW;    // stage-2 output rows per CTA (multiple of 16)
    const int32_t *seg_off;
    const int32_t *seg_ad;
    const dbf_factors *adapters;
    int n_adapters;
    int *status;
    // routed batches: 0 = blockIdx.y is a segment and the CTA runs all of its
    // chunks; > 0 = the number of segments S (at most kChunkMapMaxS), and
    // blockIdx.y is one chunk of the batch's chunk list (every segment in
    // order, cut into chunks of the plan's tokens; slots past the list exit)
    int chunk_map_S;
};

// Routed batches of at most this many segments give every chunk its own
// cluster; each CTA finds its chunk with a scan of the segment table.
constexpr int kChunkMapMaxS = 1024;

struct FusedPlan {
    int CT, RBW, C, RW, Wc, grid_x;  // CT = 0: no plan; RBW: stage-1 16-row blocks per warp
    size_t smem;
};

// problems: independent calls launched together (segments); the grid is
// problems x grid_x CTAs.
FusedPlan plan_fused(int N, int M, int R, int ell, int columns, int num_sms, int problems, bool accumulate);
cudaError_t launch_decode_fused(bool segmented, const FusedPlan &plan, const FusedArgs &args, int grid_y,
                                cudaStream_t stream, bool pdl);
cudaError_t launch_decode_stage(int stage, bool segmented, const DecPlan &plan, const DecArgs &args,
                                int grid_y, cudaStream_t stream, bool pdl);

// One-launch decode with a reduce-scatter / all-gather cluster exchange
// (decode_rs.cu), for R <= 128 and ell in {1, 2, 4}.
struct RsArgs {
    const uint32_t *B1, *B2;
    int ldw1, ldw2;
    const __half *alpha, *beta, *gamma;
    int N, M, R, ell, T;
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    int accumulate;
    int C;    // cluster size (stage-1 split of M)
    int Wc;   // stage-1 packed words per CTA
    int RW;   // stage-2 output rows per CTA
    int IPW;  // stage-2 items (16 rows x 8 columns) per warp
    const int32_t *seg_off;
    const int32_t *seg_ad;
    const dbf_factors *adapters;
    int n_adapters;
    int *status;
};

struct RsPlan {
    int CT, RB1, NW, C, RW, IPW, WARPS, Wc, grid_x;  // CT = 0: no plan; WARPS: 8 or 16 per CTA
    size_t smem;
};

RsPlan plan_rs(int N, int M, int R, int ell, int columns, int num_sms, int problems, bool accumulate);
size_t rs_smem_bytes(int CT, int RB1, int NW, int RW, int IPW, int ell, int WARPS);
cudaError_t launch_decode_rs(bool segmented, const RsPlan &plan, const RsArgs &args, int grid_y,
                             cudaStream_t stream);

// One decode call (f set, seg_off null) or a routed batch of S segments
// (f null; seg_off, seg_ad, adapters set) for the two-stage kernels.
struct DecodeCall {
    const dbf_factors *f;        // host copy of the factors (single call)
    int N, M, R, ell;
    int T;                       // tokens in x / y
    int tokens_per_problem;      // tokens one launch problem covers (T, or about twice the mean segment)
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    int accumulate;
    const int32_t *seg_off;
    const int32_t *seg_ad;
    const dbf_factors *adapters;
    int n_adapters;
    int S;
    int *status;
};

// Both stages; V is device scratch of ell*T rows x ldv halves.  Returns
// cudaErrorNotSupported when no tile plan fits the shape.
cudaError_t launch_decode_two_stage(const DecodeCall &c, __half *V, int ldv, int num_sms, cudaStream_t stream);
// The same two stages in one cooperative launch with a grid-wide barrier
// between them; bar: two device words, zero before the first call, owned by
// one stream at a time (every completed call advances bar[0] by 1024 and
// leaves bar[1] at 0).
cudaError_t launch_decode_one_launch(const DecodeCall &c, __half *V, int ldv, unsigned int *bar, int num_sms,
                                     cudaStream_t stream);

// G independent problems (same ell and T, any N, M, R), both stages in one
// launch each; V[p] is scratch of ell*T rows x ldv[p] halves.  Returns
// cudaErrorNotSupported when no common tile plan fits.
struct DecodeGroupCall {
    int G, T, ell, accumulate;
    const dbf_factors *f[kMaxGroup];
    const __nv_bfloat16 *x[kMaxGroup];
    __nv_bfloat16 *y[kMaxGroup];
    __half *V[kMaxGroup];
    int ldv[kMaxGroup];
    int *status;
};
cudaError_t launch_decode_grouped(const DecodeGroupCall &c, int num_sms, cudaStream_t stream);

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
    // backward-pass options (all zero for the forward product).  acc(t, i)
    // is the accumulator of activation row t*ell + i before the epilogue scale.
    __half *h_out;                 // stage 1: also store fp16(acc) in V's layout
    const __half *h_in;            // stage 1: red[i][row] += sum_t acc(t, i) * H[t*ell+i][row]
    const __nv_bfloat16 *red_src;  // stage 2: red[i][row] += sum_t red_src[t][row] * acc(t, i)
    int ld_src;
    float *red;                    // [ell][rows] fp32, accumulated with atomics
    int skip_store;                // stage 2: do not write y (reduction only)
};

cudaError_t launch_prefill_prologue(const __nv_bfloat16 *x, int T, int M, int ldx, const __half *gamma, int ell,
                                    __half *xs, int ldxs, cudaStream_t stream, bool pdl);
cudaError_t launch_prefill_gemm(int stage, const CUtensorMap &act_map, const PfArgs &args, int bn,
                                cudaStream_t stream, bool pdl);
int prefill_pick_bn(int ell, int rows_cover, int64_t C, int nk, int num_sms);
bool encode_act_map(CUtensorMap *map, const __half *base, int rows, int cols_pad, int ld, int box_rows);

// --------------------------------------------------------------- misc

cudaError_t launch_pack(const int8_t *signs, int64_t rows, int64_t cols, uint32_t *words, int64_t ldw,
                        cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw, int8_t *signs,
                          cudaStream_t stream);
cudaError_t launch_transpose(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw, uint32_t *words_t,
                             int64_t ldw_t, cudaStream_t stream);
cudaError_t launch_selftest_wait(int *status, uint64_t limit_ns, cudaStream_t stream);

// Text returned by dbf_last_cuda_error() on this thread.
void set_last_error(const char *msg);

// Host-side argument checks of dbf_matmul_path (no device work): DBF_OK or
// the DBF_ERR_* code the call returns.  T = 0 passes (the call is a no-op).
int check_matmul_args(const dbf_factors *f, const uint16_t *x, int64_t T, const uint16_t *y, int accumulate,
                      int path);

}  // namespace dbfk
