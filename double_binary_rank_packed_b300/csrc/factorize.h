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

}  // namespace dbfk
