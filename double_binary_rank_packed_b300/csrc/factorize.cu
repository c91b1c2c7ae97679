// Double binary factorization of a dense matrix on the GPU.
//
// "Addition is almost all you need: Compressing large language models with
// double binary factorization", section 2: W [N x M] ~ (a . A . m^T)(B . b^T)
// with sign matrices A [N x k], B [k x M].  The factors are found by
// alternating minimisation (Algoritmo de Optimización): with one factor
// fixed, the other solves min 1/2 ||T - P F||^2 over P of the form
// diag(r) S diag(c) by ADMM whose projection is SVID (the sign of the matrix
// times a rank-1 approximation of its magnitude).  Written out:
//
//   P-update  P = (T F^T + rho (Z - U)) (F F^T + rho I)^-1
//   Z-update  Z = SVID(P + U)       (power iteration from the all-ones direction)
//   U-update  U = U + P - Z
//
// starting from Z = the factor being replaced and U = 0; rho is rho_rel times
// the mean diagonal of F F^T (rho_rel when F is zero).  The A-step has T = W
// and F = Q = diag(mR) B diag(b); the B-step is the same step on W^T with
// F = P^T, whose result is Q^T = diag(b) B^T diag(mR).
//
// Everything is fp32-accurate: this is an optimiser step that needs fp32
// products, not reduced-precision ones.  The P-update and T F^T run on the
// tensor cores with each operand split into two tf32 parts and three
// products per term (factorize_tc.cu), which keeps fp32 accuracy; F F^T and
// the inverse, whose errors the condition number amplifies, run on a
// shared-memory-tiled SIMT GEMM.
// (F F^T + rho I)^-1 is formed once per step (blocked Cholesky, triangular
// inverse, then the lower triangle of L^-T L^-1 as an NT product, mirrored,
// so it is exactly symmetric and the P-update can read it in the NT layout),
// so each ADMM iteration is one GEMM plus memory-bound passes.
// All reductions have a fixed order: results do not vary between runs.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "factorize.h"

namespace dbfk {

namespace {

constexpr int kGemmBM = 128, kGemmBN = 128, kGemmBK = 16, kGemmStages = 3;
constexpr int kGemmPitch = kGemmBM + 4;  // floats per k row of a staged tile
constexpr size_t kGemmSmem = sizeof(float) * 2 * kGemmStages * kGemmBK * kGemmPitch;  // 50,688 B
constexpr int kCholNB = 32;
constexpr int kColsThreads = 256;
constexpr int kMaxColChunks = 32;

// 4-byte asynchronous copy global -> shared; valid == false writes a zero
// (source size 0) and reads nothing.
__device__ __forceinline__ void fz_cp_async_4(float *dst, const float *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}

template <int N>
__device__ __forceinline__ void fz_cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// C = alpha * A B^T + beta * C; A [m x kk] (lda), B [n x kk] (ldb), C [m x n]
// (ldc), all row-major fp32.  C is not read when beta == 0.  A 128 x 128 tile
// per CTA, 8 x 8 outputs per thread.  Operand tiles of 16 k-steps are copied
// straight into shared memory, transposed (k-major, row pitch 132 floats so
// the copies conflict at most 2-way and the fragment reads stay 16-byte
// aligned), by 4-byte asynchronous copies three stages deep: two stages are
// in flight while one is multiplied, one barrier per stage.  Out-of-range
// rows and k are zero-filled.  lower: only the tiles that touch the lower
// triangle (col <= row) are computed; the others are left as they are (for
// products whose upper triangle nothing reads).
__global__ void __launch_bounds__(256, 2) fz_gemm_nt_kernel(int m, int n, int kk, float alpha,
                                                            const float *__restrict__ A, int64_t lda,
                                                            const float *__restrict__ B, int64_t ldb, float beta,
                                                            float *C, int64_t ldc, int lower) {
    extern __shared__ __align__(16) float fz_gemm_smem[];
    float *As = fz_gemm_smem;                                       // [stage][k][kGemmPitch]
    float *Bs = fz_gemm_smem + kGemmStages * kGemmBK * kGemmPitch;  // same
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int row0 = blockIdx.y * kGemmBM, col0 = blockIdx.x * kGemmBN;
    if (lower && col0 >= row0 + kGemmBM) return;  // the whole tile is above the diagonal
    const int lk = tid & 15, lr0 = tid >> 4;       // copies: k offset lk, rows lr0 + 16 i
    auto issue = [&](int stage, int t0) {
        float *as = As + stage * kGemmBK * kGemmPitch + lk * kGemmPitch;
        float *bs = Bs + stage * kGemmBK * kGemmPitch + lk * kGemmPitch;
        const int gt = t0 + lk;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = lr0 + 16 * i;
            const int ga = row0 + r, gb = col0 + r;
            const bool va = ga < m && gt < kk, vb = gb < n && gt < kk;
            fz_cp_async_4(as + r, va ? A + int64_t(ga) * lda + gt : A, va);
            fz_cp_async_4(bs + r, vb ? B + int64_t(gb) * ldb + gt : B, vb);
        }
    };
    // accumulators in column pairs: one paired fp32 FMA (__ffma2_rn: two fused multiply-adds,
    // each rounded to nearest as fmaf is) updates two outputs, which halves the FMA
    // instructions of a kernel whose issue slots, not its FMA pipe, were the limit
    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.f, 0.f);

    const int nsteps = (kk + kGemmBK - 1) / kGemmBK;
    issue(0, 0);
    cp_async_commit();
    if (nsteps > 1) issue(1, kGemmBK);
    cp_async_commit();
    for (int st = 0; st < nsteps; ++st) {
        fz_cp_async_wait<1>();  // this thread's copies of stage st have landed
        __syncthreads();        // everyone's have; stage (st + 2) % 3 was last read in st - 1
        if (st + 2 < nsteps) issue((st + 2) % kGemmStages, (st + 2) * kGemmBK);
        cp_async_commit();      // possibly empty: keeps one group per stage
        const float *as = As + (st % kGemmStages) * kGemmBK * kGemmPitch;
        const float *bs = Bs + (st % kGemmStages) * kGemmBK * kGemmPitch;
#pragma unroll
        for (int t = 0; t < kGemmBK; ++t) {
            const float4 a0 = *reinterpret_cast<const float4 *>(as + t * kGemmPitch + ty * 4);
            const float4 a1 = *reinterpret_cast<const float4 *>(as + t * kGemmPitch + 64 + ty * 4);
            const float4 b0 = *reinterpret_cast<const float4 *>(bs + t * kGemmPitch + tx * 4);
            const float4 b1 = *reinterpret_cast<const float4 *>(bs + t * kGemmPitch + 64 + tx * 4);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                  make_float2(b1.z, b1.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 ai = make_float2(av[i], av[i]);
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][q] = __ffma2_rn(ai, bp[q], acc[i][q]);
            }
        }
    }
    fz_cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gr = row0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        if (gr >= m) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int gc = col0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
            if (gc >= n) continue;
            float *c = C + int64_t(gr) * ldc + gc;
            const float v = alpha * ((j & 1) ? acc[i][j >> 1].y : acc[i][j >> 1].x);
            *c = (beta != 0.f) ? fmaf(beta, *c, v) : v;
        }
    }
}

// X[r][c] = X[c][r] for c > r: the upper triangle of a k x k matrix copied
// from its lower one through 32 x 32 tiles (block 32 x 8).  Tiles wholly in
// the lower triangle exit; a diagonal tile reads before it writes.
__global__ void fz_mirror_lower_kernel(float *X, int k) {
    __shared__ float tile[32][33];
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    if (c0 < r0) return;
    for (int dj = threadIdx.y; dj < 32; dj += 8) {
        const int c = c0 + dj, r = r0 + threadIdx.x;
        if (c < k && r < k) tile[dj][threadIdx.x] = X[int64_t(c) * k + r];
    }
    __syncthreads();
    for (int di = threadIdx.y; di < 32; di += 8) {
        const int r = r0 + di, c = c0 + threadIdx.x;
        if (r < k && c < k && c > r) X[int64_t(r) * k + c] = tile[threadIdx.x][di];
    }
}

// out[c][r] = in[r][c] through a 32 x 32 shared tile (block 32 x 8).
template <typename Tv>
__global__ void fz_transpose_kernel(const Tv *__restrict__ in, int rows, int cols, Tv *__restrict__ out) {
    __shared__ Tv tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int dy = threadIdx.y; dy < 32; dy += 8) {
        const int r = r0 + dy, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[dy][threadIdx.x] = in[int64_t(r) * cols + c];
    }
    __syncthreads();
    for (int dy = threadIdx.y; dy < 32; dy += 8) {
        const int c = c0 + dy, r = r0 + threadIdx.x;
        if (c < cols && r < rows) out[int64_t(c) * rows + r] = tile[threadIdx.x][dy];
    }
}

// F[j][i] = c[j] * S[i][j] * r[i] for j < k, i < p: the fixed factor in the
// orientation the GEMMs read (S is [p x k] int8).  32 x 32 tiles.
__global__ void fz_build_f_kernel(const float *__restrict__ r, const int8_t *__restrict__ S,
                                  const float *__restrict__ c, int p, int k, float *__restrict__ F) {
    __shared__ float tile[32][33];
    const int j0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    for (int di = threadIdx.y; di < 32; di += 8) {
        const int i = i0 + di, j = j0 + threadIdx.x;
        if (i < p && j < k) tile[di][threadIdx.x] = float(S[int64_t(i) * k + j]) * r[i];
    }
    __syncthreads();
    for (int dj = threadIdx.y; dj < 32; dj += 8) {
        const int j = j0 + dj, i = i0 + threadIdx.x;
        if (j < k && i < p) F[int64_t(j) * p + i] = c[j] * tile[threadIdx.x][dj];
    }
}

// Fixed-order sum over a 1024-thread block (tree in shared memory).
__device__ float block_sum_1024(float v, float *red) {
    const int tid = threadIdx.x;
    red[tid] = v;
    __syncthreads();
    for (int s = 512; s > 0; s >>= 1) {
        if (tid < s) red[tid] += red[tid + s];
        __syncthreads();
    }
    const float total = red[0];
    __syncthreads();
    return total;
}

// rho = rho_rel * mean(diag G) (rho_rel when that is 0), then G += rho I;
// rho is left in *rho_out for the later passes.  One 1024-thread block.
__global__ void __launch_bounds__(1024) fz_ridge_kernel(float *G, int k, float rho_rel, float *rho_out) {
    __shared__ float red[1024];
    float s = 0.f;
    for (int j = threadIdx.x; j < k; j += 1024) s += G[int64_t(j) * k + j];
    const float mean = block_sum_1024(s, red) / float(k);
    const float rho = mean > 0.f ? rho_rel * mean : rho_rel;
    for (int j = threadIdx.x; j < k; j += 1024) G[int64_t(j) * k + j] += rho;
    if (threadIdx.x == 0) *rho_out = rho;
}

// One step of the 32-column right-looking Cholesky, diagonal block and panel in
// one launch.  Every CTA factors the nb x nb diagonal block at (j0, j0) itself
// (warp 0: lane = row, the row held in registers, column c passed between
// lanes by shuffles; a pivot that is not positive records DBF_ERR_NUMERIC and
// continues with FLT_MIN), then solves its 128 panel rows r >= j0 + nb,
// x L_jj^T = G[r, j0:j0+nb], by forward substitution (one thread per row).
// The factored block cannot go back into G in this launch (other CTAs may
// still be reading the original), so CTA 0 parks it in slot (j0 / 32) & 1 of
// `park` and the next step's CTA 0 writes it into G, with the strict upper
// triangle zeroed; the last step (no panel) writes its own block as well.
__global__ void __launch_bounds__(128) fz_chol_step_kernel(float *G, int k, int j0, int nb, float *park,
                                                           int *status) {
    __shared__ float L[kCholNB][kCholNB + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool last = j0 + nb >= k;
    if (blockIdx.x == 0 && j0 > 0) {
        // the previous step's factored block into G
        const float *prev = park + (((j0 / kCholNB) - 1) & 1) * kCholNB * kCholNB;
        const int pj = j0 - kCholNB;
        for (int e = tid; e < kCholNB * kCholNB; e += blockDim.x) {
            const int a = e / kCholNB, b = e - a * kCholNB;
            G[int64_t(pj + a) * k + pj + b] = (b <= a) ? prev[e] : 0.f;
        }
    }
    if (warp == 0) {
        if (lane < nb)
#pragma unroll 8
            for (int a = 0; a < nb; ++a) L[a][lane] = G[int64_t(j0 + a) * k + j0 + lane];  // row a, coalesced
        __syncwarp();
        float row[kCholNB];
#pragma unroll
        for (int c = 0; c < kCholNB; ++c) row[c] = (lane < nb && c < nb) ? L[lane][c] : 0.f;
#pragma unroll
        for (int c = 0; c < kCholNB; ++c) {
            if (c < nb) {  // warp-uniform
                float d = __shfl_sync(0xffffffffu, row[c], c);
                if (!(d > 0.f)) {
                    if (lane == 0 && blockIdx.x == 0) record_status(status, DBF_ERR_NUMERIC);
                    d = FLT_MIN;
                }
                const float sd = sqrtf(d);
                if (lane == c) row[c] = sd;
                else if (lane > c) row[c] = row[c] / sd;
                const float lc = row[c];
#pragma unroll
                for (int cc = c + 1; cc < kCholNB; ++cc) {
                    const float lcc = __shfl_sync(0xffffffffu, lc, cc);  // L[cc][c]
                    if (lane >= cc) row[cc] = fmaf(-lc, lcc, row[cc]);
                }
            }
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < kCholNB; ++c) L[lane][c] = row[c];
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        if (last) {
            for (int e = tid; e < nb * nb; e += blockDim.x) {
                const int a = e / nb, b = e - a * nb;
                G[int64_t(j0 + a) * k + j0 + b] = (b <= a) ? L[a][b] : 0.f;
            }
        } else {
            float *slot = park + ((j0 / kCholNB) & 1) * kCholNB * kCholNB;
            for (int e = tid; e < kCholNB * kCholNB; e += blockDim.x) slot[e] = L[e / kCholNB][e % kCholNB];
        }
    }
    const int r = j0 + nb + blockIdx.x * blockDim.x + tid;
    if (last || r >= k) return;
    float *row = G + int64_t(r) * k + j0;
    float x[kCholNB];
#pragma unroll
    for (int c = 0; c < kCholNB; ++c) {
        if (c < nb) {
            float s = row[c];
#pragma unroll
            for (int t = 0; t < c; ++t) s -= x[t] * L[c][t];
            x[c] = s / L[c][c];
        }
    }
#pragma unroll
    for (int c = 0; c < kCholNB; ++c)
        if (c < nb) row[c] = x[c];
}

// ---------------------------------------------- triangular inverse by blocks
//
// X = L^-1 (lower) and Z = L^-T = X^T (upper) of the Cholesky factor L (the
// lower triangle of G), by recursion on the diagonal: for
// L = [[L11, 0], [L21, L22]], X = [[X11, 0], [X21, X22]] with
// X21 = -X22 L21 X11, which two NT GEMMs give from the halves' inverses:
// Tt = Z11 L21^T (= (L21 X11)^T), then X21 = -X22 Tt^T, and Z12 = X21^T.
// The leaves (kTriLeaf rows) are solved by forward substitution.  The GEMMs
// read whole blocks, so X and Z start zeroed.

constexpr int kTriLeaf = 128;

__global__ void __launch_bounds__(256) fz_zero2_kernel(float *a, float *b, int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        a[i] = 0.f;
        b[i] = 0.f;
    }
}

// One leaf block [lo, lo + nb) per CTA, one thread per column c of its
// inverse: x[i][c] = (delta_ic - sum_{t<i} L[i][t] x[t][c]) / L[i][i] for
// i >= c (0 above), the block of L and the columns of x in shared memory;
// then X's block row-major and Z's block as its transpose.
__global__ void __launch_bounds__(kTriLeaf) fz_tri_leaf_kernel(const float *__restrict__ G, int k,
                                                               float *__restrict__ X, float *__restrict__ Z) {
    extern __shared__ float tri_sm[];
    float *Ls = tri_sm;                              // [kTriLeaf][kTriLeaf + 1]
    float *xs = tri_sm + kTriLeaf * (kTriLeaf + 1);  // [kTriLeaf][kTriLeaf + 1]
    constexpr int ld = kTriLeaf + 1;
    const int lo = blockIdx.x * kTriLeaf, nb = min(kTriLeaf, k - lo), c = threadIdx.x;
    for (int e = c; e < nb * kTriLeaf; e += kTriLeaf) {
        const int i = e / kTriLeaf, t = e - i * kTriLeaf;
        Ls[i * ld + t] = (t <= i && t < nb) ? G[int64_t(lo + i) * k + lo + t] : 0.f;
    }
    __syncthreads();
    if (c < nb) {
        for (int i = 0; i < nb; ++i) {
            float v = 0.f;
            if (i >= c) {
                float s = (i == c) ? 1.f : 0.f;
                for (int t = c; t < i; ++t) s = fmaf(-Ls[i * ld + t], xs[t * ld + c], s);
                v = s / Ls[i * ld + i];
            }
            xs[i * ld + c] = v;
        }
    }
    __syncthreads();
    for (int i = 0; i < nb; ++i)
        if (c < nb) X[int64_t(lo + i) * k + lo + c] = xs[i * ld + c];  // row i of the block
    for (int r = 0; r < nb; ++r)
        if (c < nb) Z[int64_t(lo + r) * k + lo + c] = xs[c * ld + r];  // row r of Z = column r of x
}

// out[j][i] = in[i][j] for an rows x cols block with row strides ldi, ldo
// (32 x 32 tiles, block 32 x 8).
__global__ void fz_transpose_block_kernel(const float *__restrict__ in, int64_t ldi, int rows, int cols,
                                          float *__restrict__ out, int64_t ldo) {
    __shared__ float tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int dy = threadIdx.y; dy < 32; dy += 8) {
        const int r = r0 + dy, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[dy][threadIdx.x] = in[int64_t(r) * ldi + c];
    }
    __syncthreads();
    for (int dy = threadIdx.y; dy < 32; dy += 8) {
        const int c = c0 + dy, r = r0 + threadIdx.x;
        if (c < cols && r < rows) out[int64_t(c) * ldo + r] = tile[threadIdx.x][dy];
    }
}

// out[i] = sum_j |Y[i][j]| * v[j] (v == null: the constant vconst), one warp
// per row; with S_out set, also S_out[i][j] = sign(Y[i][j]) (sign(0) = +1).
__global__ void __launch_bounds__(256) fz_rows_absdot_kernel(const float *__restrict__ Y, int n, int k,
                                                             const float *__restrict__ v, float vconst,
                                                             float *__restrict__ out, int8_t *__restrict__ S_out) {
    const int warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (warp >= n) return;
    const float *y = Y + int64_t(warp) * k;
    float s = 0.f;
    for (int j = lane; j < k; j += 32) {
        const float yv = y[j];
        s += fabsf(yv) * (v ? v[j] : vconst);
        if (S_out) S_out[int64_t(warp) * k + j] = yv >= 0.f ? int8_t(1) : int8_t(-1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) out[warp] = s;
}

// part[ch][j] = sum over rows i of chunk ch of |Y[i][j]| * u[i]; one thread per column.
__global__ void __launch_bounds__(kColsThreads) fz_cols_partial_kernel(const float *__restrict__ Y, int n, int k,
                                                                       const float *__restrict__ u, int rows_per_chunk,
                                                                       float *__restrict__ part) {
    const int j = blockIdx.x * kColsThreads + threadIdx.x;
    if (j >= k) return;
    const int i0 = blockIdx.y * rows_per_chunk, i1 = min(n, i0 + rows_per_chunk);
    float s = 0.f;
    for (int i = i0; i < i1; ++i) s += fabsf(Y[int64_t(i) * k + j]) * u[i];
    part[int64_t(blockIdx.y) * k + j] = s;
}

// v[j] = sum_ch part[ch][j], then v /= ||v|| when ||v|| > 0.  One block.
__global__ void __launch_bounds__(1024) fz_cols_final_kernel(const float *__restrict__ part, int chunks, int k,
                                                             float *__restrict__ v) {
    __shared__ float red[1024];
    float ss = 0.f;
    for (int j = threadIdx.x; j < k; j += 1024) {
        float s = 0.f;
        for (int ch = 0; ch < chunks; ++ch) s += part[int64_t(ch) * k + j];
        v[j] = s;
        ss += s * s;
    }
    const float nrm = sqrtf(block_sum_1024(ss, red));
    if (nrm > 0.f)
        for (int j = threadIdx.x; j < k; j += 1024) v[j] = v[j] / nrm;
}

__global__ void fz_fill_kernel(float *v, int k, float value) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < k) v[j] = value;
}

// The dual and right-hand-side pass.  z = s * r[i] * c[j] with s the sign of
// the warm-start factor (init) or of Y = P + U held in UY (otherwise).
//   init:  UY = 0,        RHS = Cw + rho z
//   else:  UY = Y - z,    RHS = Cw + rho (z - UY)
// Grid: x over column blocks of 256, y over rows.
__global__ void __launch_bounds__(256) fz_dual_rhs_kernel(const float *__restrict__ Cw, float *UY,
                                                          float *__restrict__ RHS2, int k2,
                                                          const int8_t *__restrict__ S0, const float *__restrict__ r,
                                                          const float *__restrict__ c, const float *__restrict__ rho_p,
                                                          int k, int init) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= k2) return;
    const int i = blockIdx.y;
    float *o = RHS2 + int64_t(i) * 2 * k2;  // the right-hand side in split form [hi | lo]
    if (j >= k) {
        o[j] = 0.f;
        o[k2 + j] = 0.f;
        return;
    }
    const int64_t e = int64_t(i) * k + j;
    const float rho = *rho_p;
    const float rc = r[i] * c[j];
    float v;
    if (init) {
        const float z = float(S0[e]) * rc;
        UY[e] = 0.f;
        v = fmaf(rho, z, Cw[e]);
    } else {
        const float y = UY[e];
        const float z = y >= 0.f ? rc : -rc;
        const float un = y - z;
        UY[e] = un;
        v = fmaf(rho, z - un, Cw[e]);
    }
    const float hi = tf32_rna(v);
    o[j] = hi;
    o[k2 + j] = tf32_rna(v - hi);
}

// Importance weighting: W'[i][j] = d_out[i] * W[i][j] * d_in[j].  Grid: x over
// column blocks of 256, y over rows.
__global__ void __launch_bounds__(256) fz_weight_kernel(const float *__restrict__ W, const float *__restrict__ d_out,
                                                        const float *__restrict__ d_in, int M,
                                                        float *__restrict__ Wp) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= M) return;
    const int64_t e = int64_t(blockIdx.y) * M + j;
    Wp[e] = d_out[blockIdx.y] * W[e] * d_in[j];
}

// v[i] *= d[i] (divide == 0) or v[i] /= d[i]; a weight that is not positive
// and finite records DBF_ERR_DEVICE_ARG and leaves v[i] as it is.
__global__ void fz_scale_vec_kernel(float *v, const float *__restrict__ d, int n, int divide, int *status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float w = d[i];
    if (!(w > 0.f && w <= FLT_MAX)) {
        record_status(status, DBF_ERR_DEVICE_ARG);
        return;
    }
    v[i] = divide ? v[i] / w : v[i] * w;
}

inline unsigned cdiv(int64_t a, int64_t b) { return unsigned((a + b - 1) / b); }
inline size_t align_up(size_t v) { return (v + 255) & ~size_t(255); }

cudaError_t gemm_nt(int m, int n, int kk, float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                    float beta, float *C, int64_t ldc, cudaStream_t s, int lower = 0) {
    if (m <= 0 || n <= 0) return cudaSuccess;
    const dim3 grid(cdiv(n, kGemmBN), cdiv(m, kGemmBM));
    fz_gemm_nt_kernel<<<grid, 256, kGemmSmem, s>>>(m, n, kk, alpha, A, lda, B, ldb, beta, C, ldc, lower);
    return cudaGetLastError();
}

// Scratch of one factorization, carved from the caller's workspace.
struct FzScratch {
    float *Wt, *F, *G, *LinvT, *Ginv, *Cw, *UY, *u, *part, *rho, *Tt, *park;
    // split forms [hi | lo] of the tensor-core GEMMs' operands: W, W^T, F, the inverse and the
    // right-hand side
    float *W2, *Wt2, *F2, *Ginv2, *RHS2;
    int8_t *Bt;
};

size_t carve(void *base, int64_t N, int64_t M, int64_t k, FzScratch *s) {
    const int64_t nmax = std::max(N, M);
    size_t off = 0;
    char *b = static_cast<char *>(base);
    auto take = [&](size_t bytes) {
        char *p = b ? b + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    FzScratch t;
    t.Wt = reinterpret_cast<float *>(take(sizeof(float) * size_t(M) * N));
    t.F = reinterpret_cast<float *>(take(sizeof(float) * size_t(k) * nmax));
    t.G = reinterpret_cast<float *>(take(sizeof(float) * size_t(k) * k));
    t.LinvT = reinterpret_cast<float *>(take(sizeof(float) * size_t(k) * k));
    t.Ginv = reinterpret_cast<float *>(take(sizeof(float) * size_t(k) * k));
    t.Cw = reinterpret_cast<float *>(take(sizeof(float) * size_t(nmax) * k));
    t.UY = reinterpret_cast<float *>(take(sizeof(float) * size_t(nmax) * k));
    const size_t k2 = 2 * size_t(tc_split_half(int(k))), n2 = 2 * size_t(tc_split_half(int(nmax)));
    t.W2 = reinterpret_cast<float *>(take(sizeof(float) * size_t(N) * 2 * tc_split_half(int(M))));
    t.Wt2 = reinterpret_cast<float *>(take(sizeof(float) * size_t(M) * 2 * tc_split_half(int(N))));
    t.F2 = reinterpret_cast<float *>(take(sizeof(float) * size_t(k) * n2));
    t.Ginv2 = reinterpret_cast<float *>(take(sizeof(float) * size_t(k) * k2));
    t.RHS2 = reinterpret_cast<float *>(take(sizeof(float) * size_t(nmax) * k2));
    t.u = reinterpret_cast<float *>(take(sizeof(float) * size_t(nmax)));
    t.part = reinterpret_cast<float *>(take(sizeof(float) * size_t(kMaxColChunks) * k));
    t.rho = reinterpret_cast<float *>(take(sizeof(float) * 4));
    t.Tt = reinterpret_cast<float *>(take(sizeof(float) * size_t(k) * k));  // blocked inverse scratch
    t.park = reinterpret_cast<float *>(take(sizeof(float) * 2 * kCholNB * kCholNB));  // Cholesky blocks
    t.Bt = reinterpret_cast<int8_t *>(take(size_t(M) * k));
    if (s) *s = t;
    return off;
}

int chol_steps(int k) { return (k + kCholNB - 1) / kCholNB; }

int tri_leaves(int k) { return (k + kTriLeaf - 1) / kTriLeaf; }
size_t tri_leaf_smem() { return sizeof(float) * 2 * kTriLeaf * (kTriLeaf + 1); }

// Merge leaves [l0, l1) of the blocked inverse (both halves first).
cudaError_t tri_merge(const float *G, int k, float *X, float *Z, float *Tt, int l0, int l1, cudaStream_t s) {
    if (l1 - l0 <= 1) return cudaSuccess;
    const int lm = l0 + (l1 - l0 + 1) / 2;
    cudaError_t e;
    if ((e = tri_merge(G, k, X, Z, Tt, l0, lm, s)) != cudaSuccess) return e;
    if ((e = tri_merge(G, k, X, Z, Tt, lm, l1, s)) != cudaSuccess) return e;
    const int lo = l0 * kTriLeaf, mid = lm * kTriLeaf, hi = std::min(k, l1 * kTriLeaf);
    const int s1 = mid - lo, s2 = hi - mid;
    // Tt = Z11 L21^T  [s1 x s2]
    if ((e = gemm_nt(s1, s2, s1, 1.f, Z + int64_t(lo) * k + lo, k, G + int64_t(mid) * k + lo, k, 0.f, Tt, s2, s)) !=
        cudaSuccess)
        return e;
    // X21 = -X22 Tt^T  [s2 x s1]
    if ((e = gemm_nt(s2, s1, s2, -1.f, X + int64_t(mid) * k + mid, k, Tt, s2, 0.f, X + int64_t(mid) * k + lo, k,
                     s)) != cudaSuccess)
        return e;
    // Z12 = X21^T
    fz_transpose_block_kernel<<<dim3(cdiv(s1, 32), cdiv(s2, 32)), dim3(32, 8), 0, s>>>(
        X + int64_t(mid) * k + lo, k, s2, s1, Z + int64_t(lo) * k + mid, k);
    return cudaGetLastError();
}

// X = L^-1, Z = L^-T of the lower triangle L of G [k x k].
cudaError_t tri_inverse(const float *G, int k, float *X, float *Z, float *Tt, cudaStream_t s) {
    const int64_t kk = int64_t(k) * k;
    fz_zero2_kernel<<<unsigned(std::min<int64_t>((kk + 255) / 256, 4736)), 256, 0, s>>>(X, Z, kk);
    fz_tri_leaf_kernel<<<tri_leaves(k), kTriLeaf, tri_leaf_smem(), s>>>(G, k, X, Z);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return tri_merge(G, k, X, Z, Tt, 0, tri_leaves(k), s);
}

// Launches of one ADMM step (a half of an alternating round).
int step_launches(int k, int inner, int power_iters) {
    if (inner <= 0) return 0;
    const int chol = 2 * chol_steps(k) - 1;  // diagonal + panel, then the trailing update (none after the last)
    const int svid = (power_iters > 0 ? 3 * power_iters : 1) + 1;
    // F and its split form, F F^T, ridge; Cholesky; the blocked L^-1 (zero fill, leaves, two GEMMs
    // and a transpose per merge); inverse, its mirror and its split form, T F^T, first dual pass;
    // per iteration the P-update GEMM, the SVID passes and (but the last) a dual pass
    const int tri = 2 + 3 * (tri_leaves(k) - 1);
    return 4 + chol + tri + 5 + inner * (1 + svid) + (inner - 1);
}

// SVID of Y [n x k]: c (= v) by power iteration, then r = |Y| c; S_out optional.
cudaError_t svid(const float *Y, int n, int k, int power_iters, const FzScratch &w, float *r, float *c,
                 int8_t *S_out, cudaStream_t s) {
    const float v0 = float(1.0 / sqrt(double(k)));
    const int rows_per_chunk = std::max<int>(32, int((int64_t(n) + kMaxColChunks - 1) / kMaxColChunks));
    const int chunks = int((int64_t(n) + rows_per_chunk - 1) / rows_per_chunk);
    const unsigned row_blocks = cdiv(n, 8);
    if (power_iters <= 0) {
        fz_fill_kernel<<<cdiv(k, 256), 256, 0, s>>>(c, k, v0);
    }
    for (int q = 0; q < power_iters; ++q) {
        fz_rows_absdot_kernel<<<row_blocks, 256, 0, s>>>(Y, n, k, q == 0 ? nullptr : c, v0, w.u, nullptr);
        fz_cols_partial_kernel<<<dim3(cdiv(k, kColsThreads), chunks), kColsThreads, 0, s>>>(Y, n, k, w.u,
                                                                                           rows_per_chunk, w.part);
        fz_cols_final_kernel<<<1, 1024, 0, s>>>(w.part, chunks, k, c);
    }
    fz_rows_absdot_kernel<<<row_blocks, 256, 0, s>>>(Y, n, k, c, v0, r, S_out);
    return cudaGetLastError();
}

// One alternating step: the left factor (r, S [n x k], c) of T [n x p] ~ P F
// with F built from the other side's factor (r2 [p], S2 [p x k], c2 [k]).
// T2 is T in the split form of the tensor-core GEMM.
cudaError_t admm_step(const float *T2, int n, int p, int k, const float *r2, const int8_t *S2, const float *c2,
                      float *r, int8_t *S, float *c, const dbf_factorize_params &prm, const FzScratch &w,
                      int *status, cudaStream_t s) {
    if (prm.inner <= 0) return cudaSuccess;
    cudaError_t e;
    fz_build_f_kernel<<<dim3(cdiv(k, 32), cdiv(p, 32)), dim3(32, 8), 0, s>>>(r2, S2, c2, p, k, w.F);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = tc_split2(w.F, p, k, p, w.F2, s)) != cudaSuccess) return e;
    // F F^T: the Cholesky steps read only its lower triangle (and the diagonal).  On the SIMT
    // GEMM, as the inverse product below: an error in F F^T reaches the inverse multiplied by its
    // condition number (up to k / rho_rel + 1), and the three-product tensor-core sum moved
    // enough sign decisions downstream to fail the oracle's agreement bands (98.9% of B's signs
    // after two weighted rounds at 300 x 260, k = 130, against 99%)
    if ((e = gemm_nt(k, k, p, 1.f, w.F, p, w.F, p, 0.f, w.G, k, s, 1)) != cudaSuccess) return e;
    fz_ridge_kernel<<<1, 1024, 0, s>>>(w.G, k, prm.rho_rel, w.rho);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    for (int j0 = 0; j0 < k; j0 += kCholNB) {
        const int nb = std::min(kCholNB, k - j0);
        const int j1 = j0 + nb;
        fz_chol_step_kernel<<<j1 < k ? cdiv(k - j1, 128) : 1, 128, 0, s>>>(w.G, k, j0, nb, w.park, status);
        if (j1 < k) {
            if ((e = gemm_nt(k - j1, k - j1, nb, -1.f, w.G + int64_t(j1) * k + j0, k, w.G + int64_t(j1) * k + j0, k,
                             1.f, w.G + int64_t(j1) * k + j1, k, s, 1)) != cudaSuccess)
                return e;
        }
    }
    // L^-1 (in Ginv until the product below overwrites it) and L^-T by blocks
    if ((e = tri_inverse(w.G, k, w.Ginv, w.LinvT, w.Tt, s)) != cudaSuccess) return e;
    // L^-T (L^-T)^T: the lower triangle, then the upper one copied from it
    if ((e = gemm_nt(k, k, k, 1.f, w.LinvT, k, w.LinvT, k, 0.f, w.Ginv, k, s, 1)) != cudaSuccess) return e;
    fz_mirror_lower_kernel<<<dim3(cdiv(k, 32), cdiv(k, 32)), dim3(32, 8), 0, s>>>(w.Ginv, k);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = tc_split2(w.Ginv, k, k, k, w.Ginv2, s)) != cudaSuccess) return e;
    if ((e = tc_gemm_nt_split(n, k, p, 1.f, T2, w.F2, 0.f, w.Cw, k, status, s)) != cudaSuccess) return e;
    const int k2 = tc_split_half(k);
    const dim3 ew(cdiv(k2, 256), n);
    fz_dual_rhs_kernel<<<ew, 256, 0, s>>>(w.Cw, w.UY, w.RHS2, k2, S, r, c, w.rho, k, 1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    for (int it = 0; it < prm.inner; ++it) {
        const bool last = it == prm.inner - 1;
        // UY += RHS (F F^T + rho I)^-1 on the tensor cores (three tf32 products per term)
        if ((e = tc_gemm_nt_split(n, k, k, 1.f, w.RHS2, w.Ginv2, 1.f, w.UY, k, status, s)) != cudaSuccess) return e;
        if ((e = svid(w.UY, n, k, prm.power_iters, w, r, c, last ? S : nullptr, s)) != cudaSuccess) return e;
        if (!last) {
            fz_dual_rhs_kernel<<<ew, 256, 0, s>>>(w.Cw, w.UY, w.RHS2, k2, nullptr, r, c, w.rho, k, 0);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace

size_t factorize_workspace_bytes(int64_t N, int64_t M, int64_t k) { return carve(nullptr, N, M, k, nullptr); }

int factorize_launch_count(int64_t N, int64_t M, int64_t k, const dbf_factorize_params &p) {
    (void)N;
    (void)M;
    if (p.outer <= 0 || p.inner <= 0) return 0;
    // transposes of W and B in, the split forms of W and W^T, the rounds, the transpose of B out
    return 4 + p.outer * 2 * step_launches(int(k), p.inner, p.power_iters) + 1;
}

size_t factorize_tri_smem(int64_t k) {
    (void)k;
    return tri_leaf_smem();
}

cudaError_t prepare_factorize(int64_t k) {
    cudaError_t e = cudaFuncSetAttribute(fz_gemm_nt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kGemmSmem));
    if (e != cudaSuccess) return e;
    if ((e = tc_prepare()) != cudaSuccess) return e;
    return cudaFuncSetAttribute(fz_tri_leaf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(factorize_tri_smem(k)));
}

size_t factorize_weighted_workspace_bytes(int64_t N, int64_t M, int64_t k) {
    return carve(nullptr, N, M, k, nullptr) + align_up(sizeof(float) * size_t(N) * M);
}

int factorize_weighted_launch_count(int64_t N, int64_t M, int64_t k, const dbf_factorize_params &p) {
    const int base = factorize_launch_count(N, M, k, p);
    return base > 0 ? base + 5 : 0;  // W', the scales in, the factorization, the scales out
}

cudaError_t launch_factorize_weighted(const float *W, int N, int M, int k, const dbf_factorize_params &p,
                                      const float *d_out, const float *d_in, float *a, int8_t *A, float *m_left,
                                      float *m_right, int8_t *B, float *b, void *workspace, int *status,
                                      cudaStream_t s) {
    // The weighted problem is the plain one for W' = diag(d_out) W diag(d_in)
    // in the variables d_out . a and b . d_in; W' lives after the scratch.
    float *Wp = reinterpret_cast<float *>(static_cast<char *>(workspace) + carve(nullptr, N, M, k, nullptr));
    fz_weight_kernel<<<dim3(cdiv(M, 256), N), 256, 0, s>>>(W, d_out, d_in, M, Wp);
    fz_scale_vec_kernel<<<cdiv(N, 256), 256, 0, s>>>(a, d_out, N, 0, status);
    fz_scale_vec_kernel<<<cdiv(M, 256), 256, 0, s>>>(b, d_in, M, 0, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const cudaError_t ef = launch_factorize(Wp, N, M, k, p, a, A, m_left, m_right, B, b, workspace, status, s);
    // divide the weights out again, also after a failed launch inside (a launch error that leaves
    // the context usable still lets these run); the first error is the one returned
    fz_scale_vec_kernel<<<cdiv(N, 256), 256, 0, s>>>(a, d_out, N, 1, status);
    fz_scale_vec_kernel<<<cdiv(M, 256), 256, 0, s>>>(b, d_in, M, 1, status);
    const cudaError_t ed = cudaGetLastError();
    return ef != cudaSuccess ? ef : ed;
}

cudaError_t launch_factorize(const float *W, int N, int M, int k, const dbf_factorize_params &p, float *a,
                             int8_t *A, float *m_left, float *m_right, int8_t *B, float *b, void *workspace,
                             int *status, cudaStream_t s) {
    FzScratch w;
    carve(workspace, N, M, k, &w);
    cudaError_t e;
    fz_transpose_kernel<float><<<dim3(cdiv(M, 32), cdiv(N, 32)), dim3(32, 8), 0, s>>>(W, N, M, w.Wt);
    fz_transpose_kernel<int8_t><<<dim3(cdiv(M, 32), cdiv(k, 32)), dim3(32, 8), 0, s>>>(B, k, M, w.Bt);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = tc_split2(W, M, N, M, w.W2, s)) != cudaSuccess) return e;
    if ((e = tc_split2(w.Wt, N, M, N, w.Wt2, s)) != cudaSuccess) return e;
    for (int o = 0; o < p.outer; ++o) {
        // A-step: W ~ P Q with Q^T = diag(b) B^T diag(mR) fixed.
        if ((e = admm_step(w.W2, N, M, k, b, w.Bt, m_right, a, A, m_left, p, w, status, s)) != cudaSuccess)
            return e;
        // B-step: W^T ~ Q^T P^T with P = diag(a) A diag(mL) fixed.
        if ((e = admm_step(w.Wt2, M, N, k, a, A, m_left, b, w.Bt, m_right, p, w, status, s)) != cudaSuccess)
            return e;
    }
    fz_transpose_kernel<int8_t><<<dim3(cdiv(k, 32), cdiv(M, 32)), dim3(32, 8), 0, s>>>(w.Bt, M, k, B);
    return cudaGetLastError();
}

}  // namespace dbfk
