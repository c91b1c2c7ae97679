// Decode-regime kernels: y = sum_i alpha_i . B1 (beta_i . (B2 (gamma_i . x)))
// for a handful of tokens (LoRDBA page, section 2, "Núcleo de Inferencia":
// two sign-accumulate matrix products with per-channel scaling between
// them; DBF page, section 2, "Cálculo en la inferencia": the order
// gamma -> B2 -> beta -> B1 -> alpha).
//
// The sign contraction runs on the tensor cores with mma.sync m16n8k16:
// packed sign words are unpacked in registers straight into the A fragment
// (one shift + one LOP3 per fp16 pair, see sign_pair), the activations (the
// ell*T columns) are the B operand, loaded with ldmatrix from shared memory in
// the permuted K order sign_pair expects.  A CUDA-core add/subtract needs
// about T+2 instructions per sign bit; this costs about one per bit for any
// T <= 64 columns.
//
// Two kernel shapes:
//   dec_fused_kernel  (R small, the adapter case): one launch per call.  A
//       thread-block cluster splits stage 1 over K; every CTA pushes its
//       partial u into every CTA of the cluster (distributed shared memory),
//       each sums the partials in rank order, forms the fp16 v = beta*u
//       locally, and runs stage 2 for its own slice of the N output rows.
//       Every cluster recomputes stage 1 (R*M bits, small next to the call
//       when R is small); no intermediate goes through global memory.
//   dec_stage_kernel  (any R): one launch per stage; stage 1 writes V (fp16)
//       to the workspace, stage 2 reads it.  CTAs own 16*RB weight rows and
//       a K-slice; KS CTAs of a cluster split K and reduce through DSMEM.
// Both prefetch every input that no earlier kernel writes (packed signs and
// scales) with cp.async before griddepcontrol.wait, so that after the
// dependency resolves a call waits for one more memory latency (x or V).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dbfk {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__host__ __device__ inline int ldws_for(int W) {
    // row stride of packed words in shared memory: the 8 rows read by one LDS
    // fall into 8 distinct banks; strides >= 4 stay 16-byte multiples
    if (W < 4) return (W == 2) ? 3 : W;
    int s = (W + 3) & ~3;
    if ((s & 7) == 0) s += 4;
    return s;
}

__host__ __device__ inline int lda_for(int W) { return 32 * W + 8; }  // halves; +16 B kills ldmatrix conflicts

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// Copy nrows rows of row_bytes each from global to shared memory with
// cp.async; the chunk size (16, 4 or 2 bytes) is the largest that every
// address and stride allows.  2-byte chunks use plain loads and stores.
__device__ __forceinline__ void copy_rows_async(void *dst, int dst_stride, const void *src, size_t src_stride,
                                                int nrows, int row_bytes, int tid, int nthr) {
    if (nrows <= 0 || row_bytes <= 0) return;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    const uintptr_t all = d | s | static_cast<uintptr_t>(dst_stride) | static_cast<uintptr_t>(src_stride) |
                          static_cast<uintptr_t>(row_bytes);
    if ((all & 15) == 0) {
        const int q = row_bytes >> 4;
        for (int e = tid; e < nrows * q; e += nthr) {
            const int r = e / q, c = e - r * q;
            cp_async_16(static_cast<char *>(dst) + r * dst_stride + 16 * c,
                        static_cast<const char *>(src) + r * src_stride + 16 * c);
        }
    } else if ((all & 3) == 0) {
        const int q = row_bytes >> 2;
        for (int e = tid; e < nrows * q; e += nthr) {
            const int r = e / q, c = e - r * q;
            cp_async_4(static_cast<char *>(dst) + r * dst_stride + 4 * c,
                       static_cast<const char *>(src) + r * src_stride + 4 * c);
        }
    } else {
        const int q = row_bytes >> 1;
        for (int e = tid; e < nrows * q; e += nthr) {
            const int r = e / q, c = e - r * q;
            *reinterpret_cast<uint16_t *>(static_cast<char *>(dst) + r * dst_stride + 2 * c) =
                *reinterpret_cast<const uint16_t *>(static_cast<const char *>(src) + r * src_stride + 2 * c);
        }
    }
}

// Zero nrows x row_bytes (row_bytes a multiple of 4) of shared memory.
__device__ __forceinline__ void zero_rows(void *dst, int dst_stride, int nrows, int row_bytes, int tid, int nthr) {
    const int q = row_bytes >> 2;
    for (int e = tid; e < nrows * q; e += nthr) {
        const int r = e / q, c = e - r * q;
        *reinterpret_cast<uint32_t *>(static_cast<char *>(dst) + r * dst_stride + 4 * c) = 0u;
    }
}

// One warp: 16 weight rows (rowA points at the lane's row g) x words
// [wb, we) x CT column tiles of 8 activation rows.
template <int CT>
__device__ __forceinline__ void mma_rows(const uint32_t *__restrict__ rowA, int ldws, uint32_t act_base, int lda_s,
                                         int wb, int we, float (&acc)[CT][4], int lane) {
    const int c = lane & 3;
    const uint32_t sh0 = 15 - c, sh1 = 11 - c, sh2 = 7 - c, sh3 = 3 - c;
    const uint32_t *rowB = rowA + 8 * ldws;
#pragma unroll 2
    for (int j = wb; j < we; ++j) {
        const uint32_t wa = rowA[j], wv = rowB[j];
        const uint32_t a00 = sign_pair(wa, sh0), a01 = sign_pair(wv, sh0);
        const uint32_t a02 = sign_pair(wa, sh1), a03 = sign_pair(wv, sh1);
        const uint32_t a10 = sign_pair(wa, sh2), a11 = sign_pair(wv, sh2);
        const uint32_t a12 = sign_pair(wa, sh3), a13 = sign_pair(wv, sh3);
#pragma unroll
        for (int ct = 0; ct < CT; ++ct) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(act_base + static_cast<uint32_t>((ct * 8 * lda_s + 32 * j) * 2), b0, b1, b2, b3);
            mma_16816(acc[ct], a00, a01, a02, a03, b0, b1);
            mma_16816(acc[ct], a10, a11, a12, a13, b2, b3);
        }
    }
}

// Accumulator fragments (16 rows x 8*CT columns) -> shared-memory tile.
template <int CT>
__device__ __forceinline__ void store_tile(float *tile, int ld, const float (&acc)[CT][4], int lane) {
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int ct = 0; ct < CT; ++ct) {
        const int col = ct * 8 + 2 * c;
        *reinterpret_cast<float2 *>(tile + g * ld + col) = make_float2(acc[ct][0], acc[ct][1]);
        *reinterpret_cast<float2 *>(tile + (g + 8) * ld + col) = make_float2(acc[ct][2], acc[ct][3]);
    }
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// x rows of a token chunk -> activation rows t*ell+i in logical K order:
// act[t*ell+i][32g + 2s + e] = fp16(gamma_i[k] * x[t][k]), k = 32g + s + 16e
// (g, k local to this CTA's K slice).  gam_s holds gamma for the slice in
// physical order, zero past kvalid.  One piece = 8 consecutive k and the 8 k
// sixteen further on, which become 16 consecutive logical positions; x is
// read straight from global memory (16-byte loads when vec).
__device__ __forceinline__ void load_x_act(__half *act, int lda, const __nv_bfloat16 *x, size_t ldx, int ntok,
                                           const __half *gam_s, int ldg, int ell, int Wslice, int kvalid, bool vec,
                                           int tid, int nthr) {
    const int npieces = ntok * Wslice * 2;
    for (int p = tid; p < npieces; p += nthr) {
        const int q = p & 1;
        const int gt = p >> 1;
        const int t = gt / Wslice;
        const int g = gt - t * Wslice;
        const int kl = 32 * g + 8 * q;  // local physical k of the first element
        const __nv_bfloat16 *xr = x + size_t(t) * ldx;
        float xa[8], xb[8];
        if (vec && kl + 24 <= kvalid) {
            const uint4 va = *reinterpret_cast<const uint4 *>(xr + kl);
            const uint4 vb = *reinterpret_cast<const uint4 *>(xr + kl + 16);
            xa[0] = bf16lo(va.x); xa[1] = bf16hi(va.x); xa[2] = bf16lo(va.y); xa[3] = bf16hi(va.y);
            xa[4] = bf16lo(va.z); xa[5] = bf16hi(va.z); xa[6] = bf16lo(va.w); xa[7] = bf16hi(va.w);
            xb[0] = bf16lo(vb.x); xb[1] = bf16hi(vb.x); xb[2] = bf16lo(vb.y); xb[3] = bf16hi(vb.y);
            xb[4] = bf16lo(vb.z); xb[5] = bf16hi(vb.z); xb[6] = bf16lo(vb.w); xb[7] = bf16hi(vb.w);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                xa[j] = (kl + j < kvalid) ? __bfloat162float(xr[kl + j]) : 0.f;
                xb[j] = (kl + 16 + j < kvalid) ? __bfloat162float(xr[kl + 16 + j]) : 0.f;
            }
        }
        for (int i = 0; i < ell; ++i) {
            const __half *gi = gam_s + i * ldg + kl;
            uint32_t out[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __half2 h = __floats2half2_rn(__half2float(gi[j]) * xa[j], __half2float(gi[16 + j]) * xb[j]);
                out[j] = *reinterpret_cast<const uint32_t *>(&h);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(act + (t * ell + i) * lda + 32 * g + 16 * q);
            dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
            dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
        }
    }
}

// gamma of a K slice -> shared memory (physical order), zero past kvalid.
__device__ __forceinline__ void load_gamma(__half *gam_s, int ldg, const __half *gamma, int K, int k0, int ell,
                                           int kvalid, int klen, int tid, int nthr) {
    if (kvalid > 0) copy_rows_async(gam_s, ldg * 2, gamma + k0, size_t(K) * 2, ell, kvalid * 2, tid, nthr);
    const int tail = klen - kvalid;
    if (tail > 0) {
        for (int e = tid; e < ell * tail; e += nthr) {
            const int i = e / tail;
            gam_s[i * ldg + kvalid + (e - i * tail)] = __float2half_rn(0.f);
        }
    }
}

// ============================================================ two-stage kernel

struct StageSmem {
    size_t act, gam, bits, sc, yst, red, total;
};

__host__ __device__ inline StageSmem stage_smem(int CPAD, int RB, int Wc, int ell, bool stage1, bool acc) {
    StageSmem L;
    size_t o = 0;
    L.act = o;
    o += align16(size_t(CPAD) * lda_for(Wc) * 2);
    L.gam = o;
    if (stage1) o += align16(size_t(ell) * 32 * Wc * 2);
    L.bits = o;
    o += align16(size_t(16) * RB * ldws_for(Wc) * 4);
    L.sc = o;
    o += align16(size_t(ell) * 16 * RB * 2);
    L.yst = o;
    if (!stage1 && acc) o += align16(size_t(CPAD) * 16 * RB * 2);
    L.red = o;
    o += size_t(kWarps) * 16 * (CPAD + 4) * 4;
    L.total = o;
    return L;
}

template <int CT, int STAGE, bool SEG>
__global__ void __launch_bounds__(kThreads) dec_stage_kernel(const DecArgs a) {
    constexpr int CPAD = 8 * CT;
    constexpr int RED_LD = CPAD + 4;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int KS = a.KS, RB = a.RB, Wc = a.Wc;
    const int kc = (KS > 1) ? static_cast<int>(cluster_ctarank()) : 0;
    const int row0 = (blockIdx.x / KS) * RB * 16;
    const int ell = a.ell;
    const int rows_cta = 16 * RB;

    // ---- which factors and which tokens
    const uint32_t *bits = a.bits;
    int ldw = a.ldw;
    const __half *scale_in = (STAGE == 1) ? a.gamma : nullptr;
    const __half *scale_out = (STAGE == 1) ? a.beta : a.alpha;
    int t0 = 0, Tseg = a.T;
    if constexpr (SEG) {
        pdl_wait();
        const int s = blockIdx.y;
        const int o0 = a.seg_off[s], o1 = a.seg_off[s + 1], ad = a.seg_ad[s];
        if (o0 < 0 || o1 < o0 || o1 > a.T || ad < 0 || ad >= a.n_adapters) {
            if (tid == 0 && kc == 0) record_status(a.status, DBF_ERR_DEVICE_ARG);
            return;  // uniform over the cluster: every CTA of it reads the same entry
        }
        t0 = o0;
        Tseg = o1 - o0;
        const dbf_factors f = a.adapters[ad];
        if (STAGE == 1) {
            bits = f.B2;
            ldw = f.ldw2;
            scale_in = reinterpret_cast<const __half *>(f.gamma);
            scale_out = reinterpret_cast<const __half *>(f.beta);
        } else {
            bits = f.B1;
            ldw = f.ldw1;
            scale_out = reinterpret_cast<const __half *>(f.alpha);
        }
        if (Tseg == 0) return;
    }

    const StageSmem L = stage_smem(CPAD, RB, Wc, ell, STAGE == 1, a.accumulate != 0);
    const int w0 = kc * Wc;
    const int Wslice = max(0, min(Wc, a.Kw - w0));
    const int lda_s = lda_for(Wc);
    const int ldws = ldws_for(Wc);
    const int kvalid = max(0, min(32 * Wslice, a.K - 32 * w0));  // valid elements of this K slice
    const int nr = max(0, min(rows_cta, a.rows - row0));          // weight rows that exist
    __half *act_s = reinterpret_cast<__half *>(smem + L.act);
    __half *gam_s = reinterpret_cast<__half *>(smem + L.gam);
    uint32_t *bits_s = reinterpret_cast<uint32_t *>(smem + L.bits);
    __half *sc_s = reinterpret_cast<__half *>(smem + L.sc);
    __nv_bfloat16 *yst = reinterpret_cast<__nv_bfloat16 *>(smem + L.yst);
    float *red_s = reinterpret_cast<float *>(smem + L.red);

    // ---- 1. inputs no earlier kernel writes: packed signs and scales
    copy_rows_async(bits_s, ldws * 4, bits + size_t(row0) * ldw + w0, size_t(ldw) * 4, nr, Wslice * 4, tid,
                    kThreads);
    zero_rows(bits_s + nr * ldws, ldws * 4, rows_cta - nr, Wslice * 4, tid, kThreads);
    // output-side scale of this CTA's rows: beta (stage 1) or alpha (stage 2)
    copy_rows_async(sc_s, rows_cta * 2, scale_out + row0, size_t(a.rows) * 2, ell, nr * 2, tid, kThreads);
    if (STAGE == 1) load_gamma(gam_s, 32 * Wc, scale_in, a.K, 32 * w0, ell, kvalid, 32 * Wslice, tid, kThreads);
    cp_async_commit();
    pdl_trigger();
    if constexpr (!SEG) pdl_wait();

    const int tpc = CPAD / ell;  // whole tokens per column chunk
    const int nchunks = (Tseg + tpc - 1) / tpc;
    const bool xvec = ((a.ldx & 7) == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0);
    const uint32_t act_base =
        smem_u32(act_s) + static_cast<uint32_t>(((lane & 7) * lda_s + 8 * (lane >> 3)) * 2);

    for (int chunk = 0; chunk < nchunks; ++chunk) {
        const int tc0 = chunk * tpc;
        const int ntok = min(tpc, Tseg - tc0);
        const int ncol = ntok * ell;

        // ---- 2. activations (written by the previous kernel) -> shared memory
        if constexpr (STAGE == 2) {
            copy_rows_async(act_s, lda_s * 2, a.V + size_t(t0 + tc0) * ell * a.ldv + 32 * w0, size_t(a.ldv) * 2,
                            ncol, Wslice * 64, tid, kThreads);
            if (a.accumulate)
                copy_rows_async(yst, rows_cta * 2, a.y + size_t(t0 + tc0) * a.ldy + row0, size_t(a.ldy) * 2, ntok,
                                nr * 2, tid, kThreads);
        }
        cp_async_commit();
        zero_rows(act_s + ncol * lda_s, lda_s * 2, CPAD - ncol, Wslice * 64, tid, kThreads);
        cp_async_wait_all();
        __syncthreads();  // gamma in place (stage 1), V / y staged (stage 2)
        if constexpr (STAGE == 1) {
            load_x_act(act_s, lda_s, a.x + size_t(t0 + tc0) * a.ldx + 32 * w0, size_t(a.ldx), ntok, gam_s, 32 * Wc,
                       ell, Wslice, kvalid, xvec, tid, kThreads);
            __syncthreads();
        }

        // ---- 3. tensor-core sign contraction
        const int KP = kWarps / RB;
        const int rb = warp % RB, kp = warp / RB;
        const int Wp = (Wslice + KP - 1) / KP;
        const int wb = min(Wslice, kp * Wp), we = min(Wslice, wb + Wp);
        float acc[CT][4];
#pragma unroll
        for (int ct = 0; ct < CT; ++ct) acc[ct][0] = acc[ct][1] = acc[ct][2] = acc[ct][3] = 0.f;
        mma_rows<CT>(bits_s + (rb * 16 + (lane >> 2)) * ldws, ldws, act_base, lda_s, wb, we, acc, lane);

        // ---- 4. per-warp partials -> shared memory, then fixed-order sum over K parts
        store_tile<CT>(red_s + warp * 16 * RED_LD, RED_LD, acc, lane);
        __syncthreads();
        if (KP > 1) {
            for (int e = tid; e < RB * 16 * RED_LD; e += kThreads) {
                const int r = e / (16 * RED_LD), off = e - r * 16 * RED_LD;
                float s = red_s[r * 16 * RED_LD + off];
                for (int p = 1; p < KP; ++p) s += red_s[(p * RB + r) * 16 * RED_LD + off];
                red_s[r * 16 * RED_LD + off] = s;
            }
            __syncthreads();
        }

        // ---- 5. cluster reduction (fixed order of ranks) and epilogue
        if (KS > 1) cluster_sync_all();
        const int per = (rows_cta + KS - 1) / KS;
        const int rbeg = kc * per, rend = min(rows_cta, rbeg + per);
        const int nrr = max(0, rend - rbeg);
        const uint32_t red_addr = smem_u32(red_s);

        auto reduced = [&](int rl, int col) -> float {
            const int off = rl * RED_LD + col;
            if (KS == 1) return red_s[off];
            float s = 0.f;
            for (int q = 0; q < KS; ++q) s += ld_dsmem_f32(mapa_shared(red_addr + 4u * off, q));
            return s;
        };

        if constexpr (STAGE == 1) {
            // V[(t0+tc0)*ell + col][perm(r)] = fp16(beta_i[r] * u), zero for r >= R
            const size_t vrow0 = size_t(t0 + tc0) * ell;
            for (int e = tid; e < ncol * nrr; e += kThreads) {
                const int col = e / nrr, rl = rbeg + (e - col * nrr);
                const int r = row0 + rl;
                if (r >= a.rows_cover) continue;
                const float u = reduced(rl, col);
                const int i = col % ell;
                const float v = (r < a.rows) ? __half2float(sc_s[i * rows_cta + rl]) * u : 0.f;
                a.V[(vrow0 + col) * a.ldv + perm32_pos(r)] = __float2half_rn(v);
            }
        } else {
            // y[t][n] = bf16(sum_i alpha_i[n] * w[t*ell+i] (+ y))
            for (int e = tid; e < ntok * nrr; e += kThreads) {
                const int t = e / nrr, rl = rbeg + (e - t * nrr);
                const int n = row0 + rl;
                if (n >= a.rows) continue;
                float s = 0.f;
                for (int i = 0; i < ell; ++i) s += __half2float(sc_s[i * rows_cta + rl]) * reduced(rl, t * ell + i);
                if (a.accumulate) s += __bfloat162float(yst[t * rows_cta + rl]);
                a.y[size_t(t0 + tc0 + t) * a.ldy + n] = __float2bfloat16_rn(s);
            }
        }
        if (KS > 1) cluster_sync_all();  // peers may still read our partials
        __syncthreads();                 // act_s / red_s are reused by the next chunk
    }
}

// ============================================================== fused kernel

constexpr int kFusedThreads = 512;
constexpr int kFusedWarps = kFusedThreads / 32;

struct FusedSmem {
    size_t act1, gam, b2, red1, slots, act2, beta, b1, alp, yst, tile, total;
};

__host__ __device__ inline int fused_kp1(int RB1) { return RB1 >= kFusedWarps ? 1 : kFusedWarps / RB1; }

__host__ __device__ inline FusedSmem fused_smem(int CPAD, int Wc1, int R1, int Kw2, int RW, int ell, int KS,
                                                bool acc) {
    FusedSmem L;
    const int RB1 = R1 / 16;
    const int KP1 = fused_kp1(RB1);
    size_t o = 0;
    L.act1 = o;
    o += align16(size_t(CPAD) * lda_for(Wc1) * 2);
    L.gam = o;
    o += align16(size_t(ell) * 32 * Wc1 * 2);
    L.b2 = o;
    o += align16(size_t(R1) * ldws_for(Wc1) * 4);
    L.red1 = o;
    o += align16(size_t(RB1) * KP1 * 16 * (CPAD + 4) * 4);
    L.slots = o;
    o += align16(size_t(KS) * R1 * CPAD * 4);
    L.act2 = o;
    o += align16(size_t(CPAD) * lda_for(Kw2) * 2);
    L.beta = o;
    o += align16(size_t(ell) * R1 * 2);
    L.b1 = o;
    o += align16(size_t(RW) * ldws_for(Kw2) * 4);
    L.alp = o;
    o += align16(size_t(ell) * RW * 2);
    L.yst = o;
    if (acc) o += align16(size_t(CPAD) * RW * 2);
    L.tile = o;
    o += size_t(kFusedWarps) * 16 * (CPAD + 4) * 4;
    L.total = o;
    return L;
}

template <int CT, bool SEG>
__global__ void __launch_bounds__(kFusedThreads) dec_fused_kernel(const FusedArgs a) {
    constexpr int CPAD = 8 * CT;
    constexpr int RED_LD = CPAD + 4;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int KS = a.KS;
    const int kc = (KS > 1) ? static_cast<int>(cluster_ctarank()) : 0;
    const int ell = a.ell;
    const int N = a.N, M = a.M, R = a.R;
    const int R1 = (R + 31) & ~31;  // stage-1 rows covered (activation positions up to round_up(R, 32))
    const int Kw1 = (M + 31) / 32, Kw2 = R1 / 32;
    const int Wc1 = a.Wc1;
    const int RW = 16 * a.RB2;
    const int row_base = blockIdx.x * RW;  // first stage-2 output row of this CTA

    const uint32_t *B1 = a.B1, *B2 = a.B2;
    int ldw1 = a.ldw1, ldw2 = a.ldw2;
    const __half *alpha = a.alpha, *beta = a.beta, *gamma = a.gamma;
    int t0 = 0, Tseg = a.T;
    if constexpr (SEG) {
        pdl_wait();
        const int s = blockIdx.y;
        const int o0 = a.seg_off[s], o1 = a.seg_off[s + 1], ad = a.seg_ad[s];
        if (o0 < 0 || o1 < o0 || o1 > a.T || ad < 0 || ad >= a.n_adapters) {
            if (tid == 0 && blockIdx.x == 0) record_status(a.status, DBF_ERR_DEVICE_ARG);
            return;  // uniform over the cluster
        }
        t0 = o0;
        Tseg = o1 - o0;
        const dbf_factors f = a.adapters[ad];
        B1 = f.B1;
        B2 = f.B2;
        ldw1 = f.ldw1;
        ldw2 = f.ldw2;
        alpha = reinterpret_cast<const __half *>(f.alpha);
        beta = reinterpret_cast<const __half *>(f.beta);
        gamma = reinterpret_cast<const __half *>(f.gamma);
        if (Tseg == 0) return;
    }

    const FusedSmem L = fused_smem(CPAD, Wc1, R1, Kw2, RW, ell, KS, a.accumulate != 0);
    __half *act1 = reinterpret_cast<__half *>(smem + L.act1);
    __half *gam_s = reinterpret_cast<__half *>(smem + L.gam);
    uint32_t *b2_s = reinterpret_cast<uint32_t *>(smem + L.b2);
    float *red1 = reinterpret_cast<float *>(smem + L.red1);
    float *slots = reinterpret_cast<float *>(smem + L.slots);
    __half *act2 = reinterpret_cast<__half *>(smem + L.act2);
    __half *beta_s = reinterpret_cast<__half *>(smem + L.beta);
    uint32_t *b1_s = reinterpret_cast<uint32_t *>(smem + L.b1);
    __half *alp_s = reinterpret_cast<__half *>(smem + L.alp);
    __nv_bfloat16 *yst = reinterpret_cast<__nv_bfloat16 *>(smem + L.yst);
    float *tiles = reinterpret_cast<float *>(smem + L.tile);

    const int lda1 = lda_for(Wc1), lda2 = lda_for(Kw2);
    const int ldb2 = ldws_for(Wc1), ldb1 = ldws_for(Kw2);
    const int w0 = kc * Wc1;
    const int Wslice = max(0, min(Wc1, Kw1 - w0));
    const int kvalid = max(0, min(32 * Wslice, M - 32 * w0));
    const int nrows2 = max(0, min(RW, N - row_base));

    // ---- 1. inputs no earlier kernel writes: signs and scales
    copy_rows_async(b2_s, ldb2 * 4, B2 + w0, size_t(ldw2) * 4, R, Wslice * 4, tid, kFusedThreads);
    zero_rows(b2_s + R * ldb2, ldb2 * 4, R1 - R, Wslice * 4, tid, kFusedThreads);
    load_gamma(gam_s, 32 * Wc1, gamma, M, 32 * w0, ell, kvalid, 32 * Wslice, tid, kFusedThreads);
    copy_rows_async(beta_s, R1 * 2, beta, size_t(R) * 2, ell, R * 2, tid, kFusedThreads);
    copy_rows_async(b1_s, ldb1 * 4, B1 + size_t(row_base) * ldw1, size_t(ldw1) * 4, nrows2, Kw2 * 4, tid,
                    kFusedThreads);
    zero_rows(b1_s + nrows2 * ldb1, ldb1 * 4, RW - nrows2, Kw2 * 4, tid, kFusedThreads);
    copy_rows_async(alp_s, RW * 2, alpha + row_base, size_t(N) * 2, ell, nrows2 * 2, tid, kFusedThreads);
    cp_async_commit();
    if (KS > 1) cluster_arrive_relaxed();  // matched by the wait before the first push
    pdl_trigger();
    if constexpr (!SEG) pdl_wait();

    const int tpc = CPAD / ell;
    const int nchunks = (Tseg + tpc - 1) / tpc;
    const int RB1 = R1 / 16;
    const int KP1 = fused_kp1(RB1);
    const int items1 = RB1 * KP1;
    const bool xvec = ((M & 7) == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0);
    const uint32_t act1_base = smem_u32(act1) + static_cast<uint32_t>(((lane & 7) * lda1 + 8 * (lane >> 3)) * 2);
    const uint32_t act2_base = smem_u32(act2) + static_cast<uint32_t>(((lane & 7) * lda2 + 8 * (lane >> 3)) * 2);
    const uint32_t slots_addr = smem_u32(slots);

    for (int chunk = 0; chunk < nchunks; ++chunk) {
        const int tc0 = chunk * tpc;
        const int ntok = min(tpc, Tseg - tc0);
        const int ncol = ntok * ell;
        if (chunk > 0 && KS > 1) cluster_sync_all();  // peers finished reading the previous chunk's slots

        // ---- 2. activations (and the old y of this CTA's rows)
        if (a.accumulate)
            copy_rows_async(yst, RW * 2, a.y + size_t(t0 + tc0) * N + row_base, size_t(N) * 2, ntok, nrows2 * 2,
                            tid, kFusedThreads);
        cp_async_commit();
        zero_rows(act1 + ncol * lda1, lda1 * 2, CPAD - ncol, Wslice * 64, tid, kFusedThreads);
        cp_async_wait_all();  // gamma must be in place for the conversion
        __syncthreads();
        load_x_act(act1, lda1, a.x + size_t(t0 + tc0) * M + 32 * w0, size_t(M), ntok, gam_s, 32 * Wc1, ell, Wslice,
                   kvalid, xvec, tid, kFusedThreads);
        __syncthreads();

        // ---- 3. stage 1 on this CTA's K slice: items (row block, K part)
        for (int it = warp; it < items1; it += kFusedWarps) {
            const int rb = it % RB1, kp = it / RB1;
            const int Wp = (Wslice + KP1 - 1) / KP1;
            const int wb = min(Wslice, kp * Wp), we = min(Wslice, wb + Wp);
            float acc[CT][4];
#pragma unroll
            for (int ct = 0; ct < CT; ++ct) acc[ct][0] = acc[ct][1] = acc[ct][2] = acc[ct][3] = 0.f;
            mma_rows<CT>(b2_s + (rb * 16 + (lane >> 2)) * ldb2, ldb2, act1_base, lda1, wb, we, acc, lane);
            store_tile<CT>(red1 + it * 16 * RED_LD, RED_LD, acc, lane);
        }
        __syncthreads();

        // ---- 4. sum the K parts (fixed order) and push this CTA's partial u
        //         into slot kc of every CTA of the cluster
        if (chunk == 0 && KS > 1) cluster_wait();  // every CTA of the cluster has started
        {
            constexpr int C4 = CPAD / 4;
            for (int e = tid; e < R1 * C4; e += kFusedThreads) {
                const int r = e / C4, c4 = e - r * C4;
                const int rb = r >> 4, r16 = r & 15;
                float4 s = *reinterpret_cast<const float4 *>(red1 + (rb * 16 + r16) * RED_LD + 4 * c4);
                for (int p = 1; p < KP1; ++p) {
                    const float4 o =
                        *reinterpret_cast<const float4 *>(red1 + ((p * RB1 + rb) * 16 + r16) * RED_LD + 4 * c4);
                    s.x += o.x;
                    s.y += o.y;
                    s.z += o.z;
                    s.w += o.w;
                }
                if (KS == 1) {
                    *reinterpret_cast<float4 *>(slots + (r * CPAD + 4 * c4)) = s;
                } else {
                    const uint32_t off = 4u * static_cast<uint32_t>((kc * R1 + r) * CPAD + 4 * c4);
                    for (int q = 0; q < KS; ++q)
                        asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         mapa_shared(slots_addr + off, q)),
                                     "f"(s.x), "f"(s.y), "f"(s.z), "f"(s.w)
                                     : "memory");
                }
            }
        }
        if (KS > 1)
            cluster_sync_all();  // every slot of every CTA is filled
        else
            __syncthreads();

        // ---- 5. u = sum over ranks (fixed order), v = beta * u as fp16 in activation order
        {
            constexpr int C4 = CPAD / 4;
            for (int e = tid; e < R1 * C4; e += kFusedThreads) {
                const int r = e / C4, c4 = e - r * C4;
                float4 u = *reinterpret_cast<const float4 *>(slots + (r * CPAD + 4 * c4));
                for (int q = 1; q < KS; ++q) {
                    const float4 o = *reinterpret_cast<const float4 *>(slots + ((q * R1 + r) * CPAD + 4 * c4));
                    u.x += o.x;
                    u.y += o.y;
                    u.z += o.z;
                    u.w += o.w;
                }
                const float uu[4] = {u.x, u.y, u.z, u.w};
                const int pos = perm32_pos(r);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int col = 4 * c4 + j;
                    const int i = col % ell;
                    const float v = (r < R && col < ncol) ? __half2float(beta_s[i * R1 + r]) * uu[j] : 0.f;
                    act2[col * lda2 + pos] = __float2half_rn(v);
                }
            }
        }
        __syncthreads();

        // ---- 6. stage 2 on this CTA's output rows, epilogue per warp
        float *tile = tiles + warp * 16 * RED_LD;
        for (int rb2 = warp; rb2 * 16 < nrows2; rb2 += kFusedWarps) {
            float acc[CT][4];
#pragma unroll
            for (int ct = 0; ct < CT; ++ct) acc[ct][0] = acc[ct][1] = acc[ct][2] = acc[ct][3] = 0.f;
            mma_rows<CT>(b1_s + (rb2 * 16 + (lane >> 2)) * ldb1, ldb1, act2_base, lda2, 0, Kw2, acc, lane);
            store_tile<CT>(tile, RED_LD, acc, lane);
            __syncwarp();
            for (int e = lane; e < ntok * 16; e += 32) {
                const int t = e >> 4, r16 = e & 15;
                const int rl = rb2 * 16 + r16;
                if (rl >= nrows2) continue;
                float s = 0.f;
                for (int i = 0; i < ell; ++i) s += __half2float(alp_s[i * RW + rl]) * tile[r16 * RED_LD + t * ell + i];
                if (a.accumulate) s += __bfloat162float(yst[t * RW + rl]);
                a.y[size_t(t0 + tc0 + t) * N + row_base + rl] = __float2bfloat16_rn(s);
            }
            __syncwarp();
        }
        __syncthreads();  // act1 / act2 / red1 are reused by the next chunk
    }
}

// ================================================================ launchers

template <typename Kern, typename Args>
cudaError_t launch_ex(Kern kern, int &configured_smem, int grid_x, int grid_y, int threads, size_t smem, int KS,
                      const Args &args, cudaStream_t stream, bool pdl) {
    if (smem > 48 * 1024 && static_cast<int>(smem) > configured_smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured_smem = static_cast<int>(smem);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, grid_y, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (KS > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = KS;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

template <int CT, int STAGE, bool SEG>
cudaError_t launch_stage_one(const DecPlan &plan, const DecArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    static int configured = 0;
    return launch_ex(dec_stage_kernel<CT, STAGE, SEG>, configured, plan.grid_x, grid_y, kThreads, plan.smem, plan.KS,
                     args, stream, pdl);
}

template <int STAGE, bool SEG>
cudaError_t launch_stage_ct(const DecPlan &plan, const DecArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    switch (plan.CT) {
        case 1: return launch_stage_one<1, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 2: return launch_stage_one<2, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 4: return launch_stage_one<4, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 8: return launch_stage_one<8, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

template <int CT, bool SEG>
cudaError_t launch_fused_one(const FusedPlan &plan, const FusedArgs &args, int grid_y, cudaStream_t stream,
                             bool pdl) {
    static int configured = 0;
    return launch_ex(dec_fused_kernel<CT, SEG>, configured, plan.grid_x, grid_y, kFusedThreads, plan.smem, plan.KS,
                     args, stream, pdl);
}

template <bool SEG>
cudaError_t launch_fused_ct(const FusedPlan &plan, const FusedArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    switch (plan.CT) {
        case 1: return launch_fused_one<1, SEG>(plan, args, grid_y, stream, pdl);
        case 2: return launch_fused_one<2, SEG>(plan, args, grid_y, stream, pdl);
        case 4: return launch_fused_one<4, SEG>(plan, args, grid_y, stream, pdl);
        case 8: return launch_fused_one<8, SEG>(plan, args, grid_y, stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

int ct_for(int columns, int max_ct) {
    int ct = 1;
    while (ct * 8 < columns && ct < max_ct) ct *= 2;
    return ct;
}

}  // namespace

size_t decode_smem_bytes(int CT, int RB, int Wc) {
    // upper bound over both stages, any ell <= 4, with or without accumulate
    size_t m = 0;
    for (int ell = 1; ell <= 4; ++ell)
        m = std::max(m, std::max(stage_smem(8 * CT, RB, Wc, ell, true, true).total,
                                 stage_smem(8 * CT, RB, Wc, ell, false, true).total));
    return m;
}

// Choose rows per CTA (RB), cluster split of K (KS) and column tiles (CT)
// for one stage.  The cost model counts, per SM, the unpack work (one
// instruction per sign bit, 128 lanes per clock), the activation fill, and
// a fixed per-CTA cost.
DecPlan plan_decode_stage(int rows_cover, int Kw, int columns, int max_ct, int num_sms) {
    DecPlan best = {};
    const int ct = ct_for(columns, max_ct);
    const int nb = (rows_cover + 15) / 16;
    const size_t smem_cap = 200 * 1024;
    double best_cost = 1e300;
    for (int KS = 1; KS <= 8; KS *= 2) {
        if (KS > Kw) break;
        const int Wc = (Kw + KS - 1) / KS;
        for (int RB = 1; RB <= 8; RB *= 2) {
            if (RB > 1 && (RB / 2) * 16 >= rows_cover) break;
            const size_t smem = decode_smem_bytes(ct, RB, Wc);
            if (smem > smem_cap) continue;
            const int groups = (nb + RB - 1) / RB;
            const int ctas = groups * KS;
            int occ = static_cast<int>(std::min<size_t>(size_t(228 * 1024) / (smem + 1024), 8));
            if (occ < 1) occ = 1;
            const double per_sm = double(ctas) / num_sms;
            const double waves = std::ceil(per_sm / occ);
            const double unpack = 4.0 * RB * Wc;                 // clocks of sign unpack per CTA
            const double fill = double(ct * 8) * Wc * 0.75;      // activation fill per CTA
            const double fixed = 900.0 + (KS > 1 ? 500.0 : 0.0);  // launch, syncs, epilogue
            const double cost = std::ceil(per_sm) * (unpack + fill) + waves * fixed;
            if (cost < best_cost) {
                best_cost = cost;
                best.CT = ct;
                best.RB = RB;
                best.KS = KS;
                best.Wc = Wc;
                best.grid_x = ctas;
                best.smem = smem;
            }
        }
    }
    return best;
}

// Fused plan: cluster size KS (stage-1 K split), clusters per problem NQ and
// stage-2 row blocks per CTA RB2.  One 512-thread CTA fits an SM, so the
// grid of problems x NQ x KS CTAs runs in ceil(total / num_sms) waves; the
// cost is waves x the clocks of one CTA (stage-1 and stage-2 unpack, the
// activation fill, the bytes it streams at ~24 B/clk, the cluster exchange).
FusedPlan plan_fused(int N, int M, int R, int ell, int columns, int num_sms, int problems, bool accumulate) {
    FusedPlan best = {};
    const int ct = ct_for(columns, 8);
    const int R1 = (R + 31) & ~31;
    const int Kw1 = (M + 31) / 32, Kw2 = R1 / 32;
    const size_t smem_cap = 200 * 1024;
    double best_cost = 1e300;
    if (problems < 1) problems = 1;
    for (int KS = 1; KS <= 8; KS *= 2) {
        if (KS > Kw1) break;
        const int Wc1 = (Kw1 + KS - 1) / KS;
        for (int NQ = 1; NQ * KS <= std::max(num_sms, KS); NQ *= 2) {
            const int ctas = NQ * KS;
            const int RB2 = std::max(1, (N + 16 * ctas - 1) / (16 * ctas));
            const int RW = 16 * RB2;
            const size_t smem = fused_smem(8 * ct, Wc1, R1, Kw2, RW, ell, KS, accumulate).total;
            if (smem > smem_cap) continue;
            const double s1 = 4.0 * (R1 / 16) * Wc1 + double(ct * 8) * Wc1 * 0.75;
            const double s2 = 4.0 * RB2 * Kw2 + 2.0 * RB2 * ct * 8;
            const double bytes = double(R1) * Wc1 * 4 + double(RW) * Kw2 * 4 + 2.0 * ell * (32.0 * Wc1 + RW);
            const double mem = bytes / 24.0;
            const double xch = KS > 1 ? 600.0 + double(R1) * ct * 8 / 64.0 : 0.0;
            const double waves = std::ceil(double(problems) * ctas / num_sms);
            const double cost = waves * (s1 + s2 + mem + xch + 2000.0);
            if (cost < best_cost) {
                best_cost = cost;
                best.CT = ct;
                best.KS = KS;
                best.NQ = NQ;
                best.RB2 = RB2;
                best.Wc1 = Wc1;
                best.grid_x = ctas;
                best.smem = smem;
            }
        }
    }
    return best;
}

cudaError_t launch_decode_stage(int stage, bool segmented, const DecPlan &plan, const DecArgs &args, int grid_y,
                                cudaStream_t stream, bool pdl) {
    if (stage == 1)
        return segmented ? launch_stage_ct<1, true>(plan, args, grid_y, stream, pdl)
                         : launch_stage_ct<1, false>(plan, args, grid_y, stream, pdl);
    return segmented ? launch_stage_ct<2, true>(plan, args, grid_y, stream, pdl)
                     : launch_stage_ct<2, false>(plan, args, grid_y, stream, pdl);
}

cudaError_t launch_decode_fused(bool segmented, const FusedPlan &plan, const FusedArgs &args, int grid_y,
                                cudaStream_t stream, bool pdl) {
    return segmented ? launch_fused_ct<true>(plan, args, grid_y, stream, pdl)
                     : launch_fused_ct<false>(plan, args, grid_y, stream, pdl);
}

}  // namespace dbfk
