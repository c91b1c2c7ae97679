// Host-side launchers of the dense double binary factorization (factorize.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dbf.h"

namespace dbfk {

// Workspace, launch count and launches of dbf_factorize.
size_t factorize_workspace_bytes(int64_t N, int64_t M, int64_t k);
int factorize_launch_count(int64_t N, int64_t M, int64_t k, const dbf_factorize_params &p);
size_t factorize_tri_smem(int64_t k);
cudaError_t prepare_factorize(int64_t k);
cudaError_t launch_factorize(const float *W, int N, int M, int k, const dbf_factorize_params &p, float *a,
                             int8_t *A, float *m_left, float *m_right, int8_t *B, float *b, void *workspace,
                             int *status, cudaStream_t s);

// Importance-weighted variant: the same steps on diag(d_out) W diag(d_in)
// (kept after the plain scratch in the workspace), scales converted in and out.
size_t factorize_weighted_workspace_bytes(int64_t N, int64_t M, int64_t k);
int factorize_weighted_launch_count(int64_t N, int64_t M, int64_t k, const dbf_factorize_params &p);
cudaError_t launch_factorize_weighted(const float *W, int N, int M, int k, const dbf_factorize_params &p,
                                      const float *d_out, const float *d_in, float *a, int8_t *A, float *m_left,
                                      float *m_right, int8_t *B, float *b, void *workspace, int *status,
                                      cudaStream_t s);

// Tensor-core GEMM of the factorization (factorize_tc.cu).  Operands in
// split form: X2 rows of 2 * tc_split_half(kk) floats, [hi | lo] of X's row
// (hi = tf32(x), lo = tf32(x - hi), each half zero past kk).
// tc_gemm_nt_split computes C = alpha * A B^T + beta * C from A2 [m rows] and
// B2 [n rows] with three tf32 products per term (fp32 accuracy) on tcgen05;
// with `lower` set, tiles wholly above the diagonal are skipped.  A timeout of
// one of its bounded waits records DBF_ERR_TIMEOUT in *status.
cudaError_t tc_prepare();  // the GEMM's shared-memory attribute, before its first launch on a device
int tc_split_half(int kk);
cudaError_t tc_split2(const float *X, int64_t ldx, int rows, int kk, float *X2, cudaStream_t s);
cudaError_t tc_gemm_nt_split(int m, int n, int kk, float alpha, const float *A2, const float *B2, float beta,
                             float *C, int64_t ldc, int *status, cudaStream_t s, int lower = 0);

}  // namespace dbfk
