// Decode-regime kernels: y = sum_i alpha_i . B1 (beta_i . (B2 (gamma_i . x)))
// for a handful of tokens (LoRDBA page, section 2, "Núcleo de Inferencia":
// two sign-accumulate matrix products with per-channel scaling between
// them; DBF page, section 2, "Cálculo en la inferencia": the order
// gamma -> B2 -> beta -> B1 -> alpha).
//
// One launch per stage.  Each CTA owns 16*RB weight rows and one K-slice of
// Wc packed words; KS CTAs of a thread-block cluster split K and reduce their
// partial sums through distributed shared memory in a fixed order.
//
// The sign contraction runs on the tensor cores with mma.sync m16n8k16:
// packed sign words are unpacked in registers straight into the A fragment
// (one shift + one LOP3 per fp16 pair, see sign_pair), the activations (the
// ell*T columns) are the B operand, loaded with ldmatrix from shared memory in
// the permuted K order sign_pair expects.  A CUDA-core add/subtract needs
// about T+2 instructions per sign bit; this costs about one per bit for any
// T <= 64 columns.
//
// Stage 1 converts x to fp16 activations on the fly (gamma_i * x, exact in
// fp32, rounded once) and writes V = beta_i * u as fp16 in activation order;
// stage 2 reads V, contracts with B1 and writes y = bf16(sum_i alpha_i w_i).
//
// Both stages prefetch their packed signs with cp.async before
// griddepcontrol.wait, so with programmatic dependent launch the sign stream
// of a call overlaps the tail of the previous kernel.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dbfk {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__host__ __device__ inline int ldws_for(int Wc) {
    // smallest stride >= Wc with stride = 4 (mod 8): 16-byte rows and the 8
    // rows read by one LDS fall into 8 distinct banks
    int s = (Wc + 3) & ~3;
    if ((s & 7) == 0) s += 4;
    return s;
}

__host__ __device__ inline int lda_for(int Wc) { return 32 * Wc + 8; }  // halves; +16 B kills ldmatrix conflicts

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// One warp: 16 weight rows x words [wb, we) x CT column tiles.
template <int CT>
__device__ __forceinline__ void mma_rows(const uint32_t *__restrict__ bits_s, int ldws, uint32_t act_base,
                                         int lda_s, int rb, int wb, int we, float (&acc)[CT][4], int lane) {
    const int g = lane >> 2, c = lane & 3;
    const uint32_t sh0 = 15 - c, sh1 = 11 - c, sh2 = 7 - c, sh3 = 3 - c;
    const uint32_t *rowA = bits_s + (rb * 16 + g) * ldws;
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

    // ---- which factors and which tokens
    const uint32_t *bits = a.bits;
    int ldw = a.ldw;
    const __half *scale_in = (STAGE == 1) ? a.gamma : nullptr;     // gamma (stage 1)
    const __half *scale_out = (STAGE == 1) ? a.beta : a.alpha;     // beta or alpha
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

    // ---- shared memory carve-up
    const int w0 = kc * Wc;
    const int Wslice = max(0, min(Wc, a.Kw - w0));
    const int lda_s = lda_for(Wc);
    const int ldws = ldws_for(Wc);
    __half *act_s = reinterpret_cast<__half *>(smem);
    uint32_t *bits_s = reinterpret_cast<uint32_t *>(smem + align16(size_t(CPAD) * lda_s * 2));
    float *red_s = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(bits_s) +
                                             align16(size_t(16) * RB * ldws * 4));

    // ---- 1. packed signs of this CTA -> shared memory (asynchronous)
    {
        const int nrows = 16 * RB;
        const bool vec = ((ldw & 3) == 0) && ((w0 & 3) == 0) && ((Wslice & 3) == 0) &&
                         ((reinterpret_cast<uintptr_t>(bits) & 15) == 0);
        if (vec) {
            const int q = Wslice >> 2;
            for (int e = tid; e < nrows * q; e += kThreads) {
                const int r = e / q, j = (e - r * q) * 4;
                const int gr = row0 + r;
                if (gr < a.rows)
                    cp_async_16(bits_s + r * ldws + j, bits + size_t(gr) * ldw + w0 + j);
                else
                    *reinterpret_cast<uint4 *>(bits_s + r * ldws + j) = make_uint4(0, 0, 0, 0);
            }
        } else {
            for (int e = tid; e < nrows * Wslice; e += kThreads) {
                const int r = e / Wslice, j = e - r * Wslice;
                const int gr = row0 + r;
                if (gr < a.rows)
                    cp_async_4(bits_s + r * ldws + j, bits + size_t(gr) * ldw + w0 + j);
                else
                    bits_s[r * ldws + j] = 0u;
            }
        }
        cp_async_commit();
    }
    pdl_trigger();
    if constexpr (!SEG) pdl_wait();

    const int tpc = CPAD / ell;           // whole tokens per column chunk
    const int nchunks = (Tseg + tpc - 1) / tpc;
    const uint32_t act_base =
        smem_u32(act_s) + static_cast<uint32_t>(((lane & 7) * lda_s + 8 * (lane >> 3)) * 2);

    for (int chunk = 0; chunk < nchunks; ++chunk) {
        const int tc0 = chunk * tpc;
        const int ntok = min(tpc, Tseg - tc0);
        const int ncol = ntok * ell;

        // ---- 2. activations of this chunk -> shared memory (logical K order)
        if constexpr (STAGE == 1) {
            // act[t*ell+i][32j + 2s + e] = fp16(gamma_i[k] * x[t][k]),  k = 32(w0+j) + s + 16e
            const int per_t = Wslice * 16;
            for (int e = tid; e < ntok * per_t; e += kThreads) {
                const int t = e / per_t, rem = e - t * per_t;
                const int j = rem >> 4, s = rem & 15;
                const int k = 32 * (w0 + j) + s;
                const __nv_bfloat16 *xr = a.x + size_t(t0 + tc0 + t) * a.ldx;
                const float xlo = (k < a.K) ? __bfloat162float(xr[k]) : 0.f;
                const float xhi = (k + 16 < a.K) ? __bfloat162float(xr[k + 16]) : 0.f;
                for (int i = 0; i < ell; ++i) {
                    const __half *gi = scale_in + size_t(i) * a.K;
                    const float glo = (k < a.K) ? __half2float(gi[k]) : 0.f;
                    const float ghi = (k + 16 < a.K) ? __half2float(gi[k + 16]) : 0.f;
                    const __half2 v = __floats2half2_rn(glo * xlo, ghi * xhi);
                    *reinterpret_cast<__half2 *>(act_s + (t * ell + i) * lda_s + 32 * j + 2 * s) = v;
                }
            }
        } else {
            // act rows = V rows of this chunk, copied as they are (already in logical order)
            const int q = Wslice * 4;  // 16-byte pieces per row
            const size_t vrow0 = size_t(t0 + tc0) * ell;
            for (int e = tid; e < ncol * q; e += kThreads) {
                const int c = e / q, p = e - c * q;
                cp_async_16(act_s + c * lda_s + 8 * p, a.V + (vrow0 + c) * a.ldv + 32 * w0 + 8 * p);
            }
            cp_async_commit();
        }
        // zero the column rows past this chunk's tokens
        {
            const int q = Wslice * 4;
            for (int e = tid; e < (CPAD - ncol) * q; e += kThreads) {
                const int c = ncol + e / q, p = e % q;
                *reinterpret_cast<uint4 *>(act_s + c * lda_s + 8 * p) = make_uint4(0, 0, 0, 0);
            }
        }
        cp_async_wait_all();
        __syncthreads();

        // ---- 3. tensor-core sign contraction
        const int KP = kWarps / RB;
        const int rb = warp % RB, kp = warp / RB;
        const int Wp = (Wslice + KP - 1) / KP;
        const int wb = min(Wslice, kp * Wp), we = min(Wslice, wb + Wp);
        float acc[CT][4];
#pragma unroll
        for (int ct = 0; ct < CT; ++ct) acc[ct][0] = acc[ct][1] = acc[ct][2] = acc[ct][3] = 0.f;
        mma_rows<CT>(bits_s, ldws, act_base, lda_s, rb, wb, we, acc, lane);

        // ---- 4. per-warp partials -> shared memory, then fixed-order sum over K parts
        {
            const int g = lane >> 2, c = lane & 3;
            float *mine = red_s + warp * 16 * RED_LD;
#pragma unroll
            for (int ct = 0; ct < CT; ++ct) {
                const int col = ct * 8 + 2 * c;
                mine[g * RED_LD + col] = acc[ct][0];
                mine[g * RED_LD + col + 1] = acc[ct][1];
                mine[(g + 8) * RED_LD + col] = acc[ct][2];
                mine[(g + 8) * RED_LD + col + 1] = acc[ct][3];
            }
        }
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
        const int rows_cta = 16 * RB;
        const int per = (rows_cta + KS - 1) / KS;
        const int rbeg = kc * per, rend = min(rows_cta, rbeg + per);
        const int nr = max(0, rend - rbeg);
        const uint32_t red_addr = smem_u32(red_s);

        auto reduced = [&](int rl, int col) -> float {
            const int off = ((rl >> 4) * 16 + (rl & 15)) * RED_LD + col;
            if (KS == 1) return red_s[off];
            float s = 0.f;
            for (int q = 0; q < KS; ++q) s += ld_dsmem_f32(mapa_shared(red_addr + 4u * off, q));
            return s;
        };

        if constexpr (STAGE == 1) {
            // V[(t0+tc0)*ell + col][perm(r)] = fp16(beta_i[r] * u), zero for r >= R
            const size_t vrow0 = size_t(t0 + tc0) * ell;
            for (int e = tid; e < ncol * nr; e += kThreads) {
                const int col = e / nr, rl = rbeg + (e - col * nr);
                const int r = row0 + rl;
                if (r >= a.rows_cover) continue;
                const float u = reduced(rl, col);
                const int i = col % ell;
                const float v = (r < a.rows) ? __half2float(scale_out[size_t(i) * a.rows + r]) * u : 0.f;
                a.V[(vrow0 + col) * a.ldv + perm32_pos(r)] = __float2half_rn(v);
            }
        } else {
            // y[t][n] = bf16(sum_i alpha_i[n] * w[t*ell+i] (+ y))
            for (int e = tid; e < ntok * nr; e += kThreads) {
                const int t = e / nr, rl = rbeg + (e - t * nr);
                const int n = row0 + rl;
                if (n >= a.rows) continue;
                float s = 0.f;
                for (int i = 0; i < ell; ++i)
                    s += __half2float(scale_out[size_t(i) * a.rows + n]) * reduced(rl, t * ell + i);
                __nv_bfloat16 *yp = a.y + size_t(t0 + tc0 + t) * a.ldy + n;
                if (a.accumulate) s += __bfloat162float(*yp);
                *yp = __float2bfloat16_rn(s);
            }
        }
        if (KS > 1) cluster_sync_all();  // peers may still read our partials
        __syncthreads();                 // act_s / red_s are reused by the next chunk
    }
}

template <int CT, int STAGE, bool SEG>
cudaError_t launch_one(const DecPlan &plan, const DecArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    auto kern = dec_stage_kernel<CT, STAGE, SEG>;
    static int configured_smem = 0;
    if (plan.smem > 48 * 1024 && static_cast<int>(plan.smem) > configured_smem) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(plan.smem));
        if (e != cudaSuccess) return e;
        configured_smem = static_cast<int>(plan.smem);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid_x, grid_y, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (plan.KS > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = plan.KS;
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

template <int STAGE, bool SEG>
cudaError_t launch_ct(const DecPlan &plan, const DecArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    switch (plan.CT) {
        case 1: return launch_one<1, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 2: return launch_one<2, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 4: return launch_one<4, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 8: return launch_one<8, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t decode_smem_bytes(int CT, int RB, int Wc) {
    const int CPAD = 8 * CT;
    return align16(size_t(CPAD) * lda_for(Wc) * 2) + align16(size_t(16) * RB * ldws_for(Wc) * 4) +
           size_t(kWarps) * 16 * (CPAD + 4) * 4;
}

// Choose rows per CTA (RB), cluster split of K (KS) and column tiles (CT).
// The cost model counts, per SM, the unpack work (one instruction per sign
// bit, 128 lanes per clock), the activation fill, and a fixed per-CTA cost.
DecPlan plan_decode_stage(int rows_cover, int Kw, int columns, int max_ct, int num_sms) {
    DecPlan best = {};
    int ct = 1;
    while (ct * 8 < columns && ct < max_ct) ct *= 2;
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

cudaError_t launch_decode_stage(int stage, bool segmented, const DecPlan &plan, const DecArgs &args, int grid_y,
                                cudaStream_t stream, bool pdl) {
    if (stage == 1)
        return segmented ? launch_ct<1, true>(plan, args, grid_y, stream, pdl)
                         : launch_ct<1, false>(plan, args, grid_y, stream, pdl);
    return segmented ? launch_ct<2, true>(plan, args, grid_y, stream, pdl)
                     : launch_ct<2, false>(plan, args, grid_y, stream, pdl);
}

}  // namespace dbfk
