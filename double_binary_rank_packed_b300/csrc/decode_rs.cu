// One-launch decode with a reduce-scatter / all-gather exchange inside a
// thread-block cluster, for adapter-sized middle dimensions (R <= 128):
// y = sum_i alpha_i . B1 (beta_i . (B2 (gamma_i . x))) for a handful of
// tokens (LoRDBA page, section 2, "Núcleo de Inferencia": two sign-accumulate
// products with per-channel scaling between them; DBF page, section 2,
// "Cálculo en la inferencia": the order gamma -> B2 -> beta -> B1 -> alpha).
//
// Measured on B300 in a chain of dependent launches (CUDA graph, programmatic
// dependent launch): a launch that only reads x and writes y costs about
// 1.4 us, of which ~0.7 us is the hand-over from the previous launch; every
// dependent round trip inside the kernel adds to that.  The kernel is built
// to keep that chain short:
//   * before griddepcontrol.wait (overlapping the previous launch) each CTA
//     unpacks its sign words into mma.sync A fragments in shared memory,
//     stages the scales, and prefetches its slice of x (and of y when
//     accumulating) into L2 -- a prefetch returns no data to the SM, so it is
//     safe on memory the previous kernel may still be writing;
//   * it triggers its dependents at its first instruction;
//   * stage 1 is split over M across the C CTAs of a cluster (C <= 16); each
//     warp contracts its packed words of B2 with the activations on the
//     tensor cores, the 8 warp partials are summed in shared memory, and
//     every row of the partial u goes straight to the CTA that owns it with
//     st.async (reduce-scatter, completion counted on the owner's mbarrier);
//   * each owner sums the C partials of its rows in rank order, forms
//     v = fp16(beta * u) and writes it into every CTA of the cluster, again
//     with st.async (all-gather);
//   * stage 2 reads v from shared memory and writes y from the fragments.
// Two mbarrier waits replace the cluster barriers of an all-to-all exchange;
// the exchange moves R*cols fp32 values out of each CTA instead of C times
// that.  Every cluster recomputes stage 1 (R*M sign bits, small next to the
// call when R is small).  Token chunks of 8*CT columns run one after another
// with double-buffered exchange areas.
#include <algorithm>

#include "common.cuh"
#include "decode_frag.cuh"
#include "kernels.h"

namespace dbfk {

namespace {

// Partials of stage 1 are kept per group of 8 warps along K (kKGroups); with 16
// warps per CTA the two halves of the warps split the row blocks of u.
constexpr int kKGroups = 8;

__host__ __device__ inline size_t rs_align16(size_t v) { return (v + 15) & ~size_t(15); }

// Row of u stored at perm8 position p (inverse of perm8_pos inside a group of 8).
__host__ __device__ inline int perm8_row(int p) { return (p & ~7) | ((p >> 1) & 3) | ((p & 1) << 2); }

struct RsSmem {
    size_t part, rs, vs, fa, fb, alp, bet, bars, total;
};

// R2 = round_up(R, 32) rows of u, CPAD = 8*CT columns per chunk, NW words of
// B2 per K group, WARPS warps per CTA, IPW stage-2 items per warp.
__host__ __device__ inline RsSmem rs_smem(int CPAD, int R2, int NW, int RW, int IPW, int ell, int WARPS) {
    RsSmem L;
    size_t o = 0;
    L.part = o;  // [8 K groups][R2][CPAD] fp32 stage-1 partials
    o += size_t(kKGroups) * R2 * CPAD * 4;
    L.rs = o;  // [2 buffers][C][R2/C][CPAD] fp32 partials received as owner
    o += size_t(2) * R2 * CPAD * 4;
    L.vs = o;  // [2 buffers][CPAD][R2 + 8] fp16 v in perm8 order
    o += rs_align16(size_t(2) * CPAD * (R2 + 8) * 2);
    L.fa = o;  // [K group][NW][R2/16][8][32] stage-1 A fragments (each warp owns its row blocks)
    o += size_t(kKGroups) * NW * (R2 / 16) * 8 * 32 * 4;
    L.fb = o;  // [warp][IPW][R2/32][8][32] stage-2 A fragments
    o += size_t(WARPS) * IPW * (R2 / 32) * 8 * 32 * 4;
    L.alp = o;  // [ell][RW] fp16
    o += rs_align16(size_t(ell) * RW * 2);
    L.bet = o;  // [ell][R2] fp16, zero past R
    o += rs_align16(size_t(ell) * R2 * 2);
    L.bars = o;  // [2 buffers][reduce-scatter, all-gather]
    o += 4 * 8;
    L.total = o;
    return L;
}

__device__ __forceinline__ void wait_or_flag(uint64_t *bar, uint32_t parity, int *status) {
    if (!mbar_wait_bounded(bar, parity, nullptr)) record_status(status, DBF_ERR_TIMEOUT);
}

template <int CT, int RB1, int NW, bool SEG, int WARPS>
__global__ void __launch_bounds__(32 * WARPS, WARPS == 8 ? 2 : 1) dec_rs_kernel(const RsArgs a) {
    constexpr int CPAD = 8 * CT, C4 = CPAD / 4, R2 = 16 * RB1, LDV = R2 + 8, KW2 = R2 / 32;
    constexpr int kRsThreads = 32 * WARPS, kRsWarps = WARPS;
    constexpr int RH = WARPS / kKGroups;  // row-block halves of stage 1
    constexpr int RBH = RB1 / RH;         // row blocks of u per warp
    static_assert(RB1 % RH == 0, "row blocks split evenly over the warp halves");
    extern __shared__ __align__(128) unsigned char smem[];
    // the next call's CTAs may start their own preparation at once
    pdl_trigger();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, c = lane & 3;
    const int C = a.C, RW = a.RW, IPW = a.IPW;
    const int ROWN = R2 / C;  // perm8 positions of u each CTA owns
    const int rank = static_cast<int>(cluster_ctarank());
    const int ell = a.ell, N = a.N, M = a.M, R = a.R;
    const RsSmem L = rs_smem(CPAD, R2, NW, RW, IPW, ell, WARPS);
    float *part = reinterpret_cast<float *>(smem + L.part);
    float *rsb = reinterpret_cast<float *>(smem + L.rs);
    __half *vsb = reinterpret_cast<__half *>(smem + L.vs);
    uint32_t *fa_s = reinterpret_cast<uint32_t *>(smem + L.fa);
    uint32_t *fb_s = reinterpret_cast<uint32_t *>(smem + L.fb);
    __half *alp_s = reinterpret_cast<__half *>(smem + L.alp);
    __half *bet_s = reinterpret_cast<__half *>(smem + L.bet);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);

    // ---- exchange barriers: each phase expects the bytes of one chunk
    const uint32_t rs_bytes = uint32_t(R2) * CPAD * 4, ag_bytes = uint32_t(R2) * CPAD * 2;
    if (tid == 0) {
        for (int k = 0; k < 4; ++k) mbar_init(&bars[k], 1);
        mbar_arrive_expect_tx(&bars[0], rs_bytes);
        mbar_arrive_expect_tx(&bars[1], ag_bytes);
        mbar_arrive_expect_tx(&bars[2], rs_bytes);
        mbar_arrive_expect_tx(&bars[3], ag_bytes);
        fence_mbar_init();
    }
    if (C > 1) {
        cluster_arrive_relaxed();  // every CTA of the cluster has initialised its barriers
        cluster_wait();
    } else {
        __syncthreads();
    }

    const uint32_t *B1 = a.B1, *B2 = a.B2;
    int ldw1 = a.ldw1, ldw2 = a.ldw2;
    const __half *alpha = a.alpha, *beta = a.beta, *gamma = a.gamma;
    int t0 = 0, Tseg = a.T;
    if constexpr (SEG) {
        pdl_wait();  // the routing table may come from the previous kernel
        const int s = blockIdx.y;
        const int o0 = a.seg_off[s], o1 = a.seg_off[s + 1], ad = a.seg_ad[s];
        if (o0 < 0 || o1 < o0 || o1 > a.T || ad < 0 || ad >= a.n_adapters) {
            if (tid == 0 && blockIdx.x == 0) record_status(a.status, DBF_ERR_DEVICE_ARG);
            return;  // uniform over the cluster: every CTA of it reads the same entry
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

    // ---- stage-1 geometry: this CTA's packed words [w0, w0 + Wslice), this warp's [wb, we)
    const int Kw1 = (M + 31) >> 5;
    const int w0 = rank * a.Wc;
    const int Wslice = max(0, min(a.Wc, Kw1 - w0));
    const int kg = warp % kKGroups, rh = warp / kKGroups;  // K group, row-block half
    const int wb = min(Wslice, kg * NW), we = min(Wslice, wb + NW);
    int ctok[CT], cterm[CT];
#pragma unroll
    for (int ct = 0; ct < CT; ++ct) {
        const int col = 8 * ct + g;
        ctok[ct] = col / ell;
        cterm[ct] = col - ctok[ct] * ell;
    }

    // ---- inputs no earlier kernel writes: sign fragments, scales
    uint4 gv[NW][CT];
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const int wl = wb + w;
        const bool wok = wl < we;
#pragma unroll
        for (int rbl = 0; rbl < RBH; ++rbl) {
            const int rb = rh * RBH + rbl;
            const int r0 = 16 * rb + g;
            const bool wrd = wok && in_range(w0 + wl < ldw2, a.status);
            const uint32_t lo = (wrd && r0 < R) ? __ldg(B2 + size_t(r0) * ldw2 + w0 + wl) : 0u;
            const uint32_t hi = (wrd && r0 + 8 < R) ? __ldg(B2 + size_t(r0 + 8) * ldw2 + w0 + wl) : 0u;
            uint32_t pa[4], pv[4];
            sign_pairs8(lo, c, pa);
            sign_pairs8(hi, c, pv);
            uint32_t *fp = fa_s + ((kg * NW + w) * RB1 + rb) * 256 + lane;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                fp[32 * j] = (r0 < R) ? pa[j] : 0u;  // rows past R contribute nothing
                fp[32 * (4 + j)] = (r0 + 8 < R) ? pv[j] : 0u;
            }
        }
#pragma unroll
        for (int ct = 0; ct < CT; ++ct) {
            const int k0 = 32 * (w0 + wl) + 8 * c;
            const __half *gr = gamma + size_t(cterm[ct]) * M;
            if (wok && k0 + 8 <= M && ((reinterpret_cast<uintptr_t>(gr + k0) & 15) == 0)) {
                gv[w][ct] = *reinterpret_cast<const uint4 *>(gr + k0);
            } else {
                uint16_t hv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    hv[j] = (wok && k0 + j < M) ? reinterpret_cast<const uint16_t *>(gr)[k0 + j] : uint16_t(0);
                gv[w][ct] = make_uint4(hv[0] | (uint32_t(hv[1]) << 16), hv[2] | (uint32_t(hv[3]) << 16),
                                       hv[4] | (uint32_t(hv[5]) << 16), hv[6] | (uint32_t(hv[7]) << 16));
            }
        }
    }
    const int RB2 = RW / 16;
    const int row_base = blockIdx.x * RW;
    const int nrows2 = max(0, min(RW, N - row_base));
    for (int i = 0; i < IPW; ++i) {
        const int it = warp + kRsWarps * i;
        if (it >= RB2 * CT) break;
        const int n0 = row_base + 16 * (it % RB2) + g;
#pragma unroll
        for (int w = 0; w < KW2; ++w) {
            const bool wrd = in_range(w < ldw1, a.status);
            const uint32_t lo = (wrd && n0 < N) ? __ldg(B1 + size_t(n0) * ldw1 + w) : 0u;
            const uint32_t hi = (wrd && n0 + 8 < N) ? __ldg(B1 + size_t(n0 + 8) * ldw1 + w) : 0u;
            uint32_t pa[4], pv[4];
            sign_pairs8(lo, c, pa);
            sign_pairs8(hi, c, pv);
            uint32_t *fp = fb_s + ((warp * IPW + i) * KW2 + w) * 256 + lane;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                fp[32 * j] = pa[j];
                fp[32 * (4 + j)] = pv[j];
            }
        }
    }
    for (int e = tid; e < ell * RW; e += kRsThreads) {
        const int i = e / RW, nl = e - i * RW;
        alp_s[e] = (nl < nrows2) ? alpha[size_t(i) * N + row_base + nl] : __float2half_rn(0.f);
    }
    for (int e = tid; e < ell * R2; e += kRsThreads) {
        const int i = e / R2, r = e - i * R2;
        bet_s[e] = (r < R) ? beta[size_t(i) * R + r] : __float2half_rn(0.f);
    }
    // owner role: item (pair, dg) sums two consecutive positions of one column
    // and writes them to the CTAs dg, dg + DG, ... of the cluster
    const int P = CPAD * (ROWN / 2);
    const int DG = max(1, min(C, kRsThreads / P));
    if constexpr (!SEG) {
        // x (and y when accumulating) of every chunk into L2 ahead of the wait
        const int lines = (Wslice * 64 + 127) / 128;
        for (int e = tid; e < Tseg * lines; e += kRsThreads) {
            const int t = e / lines, l = e - t * lines;
            if (32 * w0 + 64 * l < M) prefetch_l2(a.x + size_t(t) * M + 32 * w0 + 64 * l);
        }
        if (a.accumulate) {
            const int ylines = (nrows2 * 2 + 127) / 128;
            for (int e = tid; e < Tseg * ylines; e += kRsThreads) {
                const int t = e / ylines, l = e - t * ylines;
                prefetch_l2(a.y + size_t(t) * N + row_base + 64 * l);
            }
        }
        pdl_wait();  // x and y may be written / read by the previous kernel
    }

    const int tpc = CPAD / ell;  // whole tokens per chunk
    const int nchunks = (Tseg + tpc - 1) / tpc;
    const bool xvec = ((M & 7) == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0);
    for (int ch = 0; ch < nchunks; ++ch) {
        const int buf = ch & 1;
        const uint32_t ph = (ch >> 1) & 1;
        const int tc0 = ch * tpc;
        const int ntok = min(tpc, Tseg - tc0);
        const int ncol = ntok * ell;
        float *rs = rsb + buf * R2 * CPAD;
        __half *vs = vsb + buf * CPAD * LDV;
        uint64_t *bar_rs = &bars[2 * buf], *bar_ag = &bars[2 * buf + 1];
        if (ch > 0) __syncthreads();  // the previous chunk's reads of part and of its buffers are done
        if (ch >= 2 && tid == 0) {
            // next phase of this buffer's barriers (the previous one completed in chunk ch - 2)
            mbar_arrive_expect_tx(bar_rs, rs_bytes);
            mbar_arrive_expect_tx(bar_ag, ag_bytes);
        }

        // ---- stage 1 on this warp's words
        uint4 xr[NW][CT];
#pragma unroll
        for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int ct = 0; ct < CT; ++ct) {
                const int col = 8 * ct + g;
                if (wb + w < we && col < ncol && in_range(t0 + tc0 + ctok[ct] < a.T, a.status))
                    xr[w][ct] = load_x8(a.x + size_t(t0 + tc0 + ctok[ct]) * M, 32 * (w0 + wb + w) + 8 * c, M, xvec);
                else
                    xr[w][ct] = make_uint4(0u, 0u, 0u, 0u);
            }
        float acc[RBH][CT][4];
#pragma unroll
        for (int rbl = 0; rbl < RBH; ++rbl) zero_acc<CT>(acc[rbl]);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (wb + w >= we) break;
            uint32_t bx[CT][4];
#pragma unroll
            for (int ct = 0; ct < CT; ++ct) x_pairs(xr[w][ct], gv[w][ct], bx[ct]);
#pragma unroll
            for (int rbl = 0; rbl < RBH; ++rbl) {
                const uint32_t *fp = fa_s + ((kg * NW + w) * RB1 + rh * RBH + rbl) * 256 + lane;
                // fragment registers j = 0..3: row g, k pairs; 4..7: row g + 8
#pragma unroll
                for (int kh = 0; kh < 2; ++kh)
#pragma unroll
                    for (int ct = 0; ct < CT; ++ct)
                        mma_16816_nv(acc[rbl][ct], fp[32 * (2 * kh)], fp[32 * (4 + 2 * kh)], fp[32 * (2 * kh + 1)],
                                     fp[32 * (5 + 2 * kh)], bx[ct][2 * kh], bx[ct][2 * kh + 1]);
            }
        }
#pragma unroll
        for (int rbl = 0; rbl < RBH; ++rbl)
            put_frag<CT>(smem_u32(part) + 4u * static_cast<uint32_t>((kg * R2 + 16 * (rh * RBH + rbl)) * CPAD), CPAD,
                         acc[rbl], lane, false, 0);
        __syncthreads();

        // ---- reduce-scatter: the 8 K-group parts in order, each row to its owner
        for (int e = tid; e < R2 * C4; e += kRsThreads) {
            const int r = e / C4, q4 = e - r * C4;
            float4 u = *reinterpret_cast<const float4 *>(part + r * CPAD + 4 * q4);
#pragma unroll
            for (int wq = 1; wq < kKGroups; ++wq)
                add4(u, *reinterpret_cast<const float4 *>(part + (wq * R2 + r) * CPAD + 4 * q4));
            const int pos = perm8_pos(r);
            const int owner = pos / ROWN, lp = pos - owner * ROWN;
            if (!in_range(owner < C && rank * ROWN + lp < R2, a.status)) continue;
            st_async_v4(mapa_shared(smem_u32(rs + (rank * ROWN + lp) * CPAD + 4 * q4), static_cast<uint32_t>(owner)),
                        u, mapa_shared(smem_u32(bar_rs), static_cast<uint32_t>(owner)));
        }

        // ---- owner: u = sum of the C partials in rank order, v = fp16(beta u), all-gather
        if (tid < P * DG) {  // thread 0 is always one of these
            wait_or_flag(bar_rs, ph, a.status);
            const uint32_t bar_off = smem_u32(bar_ag);
            for (int e = tid; e < P * DG; e += kRsThreads) {
                const int pr = e % P, dg = e / P;
                const int ocol = pr / (ROWN / 2), owd = pr - ocol * (ROWN / 2);
                const int p0 = rank * ROWN + 2 * owd;
                float u0 = 0.f, u1 = 0.f;
                for (int q = 0; q < C; ++q) {
                    u0 += rs[(q * ROWN + 2 * owd) * CPAD + ocol];
                    u1 += rs[(q * ROWN + 2 * owd + 1) * CPAD + ocol];
                }
                const int term = ocol % ell;
                const float b0 = __half2float(bet_s[term * R2 + perm8_row(p0)]);
                const float b1 = __half2float(bet_s[term * R2 + perm8_row(p0 + 1)]);
                const __half2 h = __floats2half2_rn(b0 * u0, b1 * u1);
                const uint32_t word = *reinterpret_cast<const uint32_t *>(&h);
                const uint32_t off = smem_u32(vs + ocol * LDV + p0);
                if (!in_range(p0 + 1 < R2 && ocol < CPAD, a.status)) continue;
                for (int dq = dg; dq < C; dq += DG)
                    st_async_b32(mapa_shared(off, static_cast<uint32_t>(dq)), word,
                                 mapa_shared(bar_off, static_cast<uint32_t>(dq)));
            }
        }

        // ---- stage 2 per (row block, column tile); y straight from the fragment
        for (int i = 0; i < IPW; ++i) {
            const int it = warp + kRsWarps * i;
            if (it >= RB2 * CT) break;
            if (i == 0) wait_or_flag(bar_ag, ph, a.status);
            const int rb2 = it % RB2, ct2 = it / RB2;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < KW2; ++w) {
                const uint4 bv = *reinterpret_cast<const uint4 *>(vs + (8 * ct2 + g) * LDV + 32 * w + 8 * c);
                const uint32_t *fp = fb_s + ((warp * IPW + i) * KW2 + w) * 256 + lane;
                mma_16816_nv(d, fp[0], fp[128], fp[32], fp[160], bv.x, bv.y);
                mma_16816_nv(d, fp[64], fp[192], fp[96], fp[224], bv.z, bv.w);
            }
            // rows n0 (d[0], d[1]) and n0 + 8 (d[2], d[3]); columns 8ct2 + 2c, 8ct2 + 2c + 1
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int nl = 16 * rb2 + g + 8 * hh;
                const bool row_ok = nl < nrows2;
                const int n = row_base + nl;
                const float d0 = d[2 * hh], d1 = d[2 * hh + 1];
                __nv_bfloat16 *ycol = a.y + size_t(t0 + tc0) * N + n;
                // (debug build) every token row written is a row of y
                auto y_ok = [&](int t) { return in_range(t0 + tc0 + t < a.T && n < N, a.status); };
                if (ell == 1) {
                    const float al = row_ok ? __half2float(alp_s[nl]) : 0.f;
#pragma unroll
                    for (int e2 = 0; e2 < 2; ++e2) {
                        const int t = 8 * ct2 + 2 * c + e2;
                        if (row_ok && t < ntok && y_ok(t)) {
                            float o = al * (e2 ? d1 : d0);
                            if (a.accumulate) o += __bfloat162float(ycol[size_t(t) * N]);
                            ycol[size_t(t) * N] = __float2bfloat16_rn(o);
                        }
                    }
                } else if (ell == 2) {
                    const int t = 4 * ct2 + c;
                    if (row_ok && t < ntok && y_ok(t)) {
                        float o = __half2float(alp_s[nl]) * d0 + __half2float(alp_s[RW + nl]) * d1;
                        if (a.accumulate) o += __bfloat162float(ycol[size_t(t) * N]);
                        ycol[size_t(t) * N] = __float2bfloat16_rn(o);
                    }
                } else {  // ell == 4: terms 0, 1 in lanes with c even, 2, 3 in lanes with c odd
                    const int i0 = 2 * (c & 1);
                    float o = row_ok ? __half2float(alp_s[i0 * RW + nl]) * d0 +
                                           __half2float(alp_s[(i0 + 1) * RW + nl]) * d1
                                     : 0.f;
                    o += __shfl_xor_sync(0xffffffffu, o, 1);
                    const int t = 2 * ct2 + (c >> 1);
                    if ((c & 1) == 0 && row_ok && t < ntok && y_ok(t)) {
                        if (a.accumulate) o += __bfloat162float(ycol[size_t(t) * N]);
                        ycol[size_t(t) * N] = __float2bfloat16_rn(o);
                    }
                }
            }
        }
    }
    // Every byte a peer sends to this CTA has arrived once the waits above
    // returned (warp 0 always has a stage-2 item, and thread 0 is an owner
    // thread), so no peer can write into this CTA's shared memory after it exits.
}

template <int CT, int RB1, int NW, bool SEG, int WARPS>
cudaError_t launch_rs_one(const RsPlan &plan, const RsArgs &args, int grid_y, cudaStream_t stream) {
    static int configured_smem = 0;
    auto kern = dec_rs_kernel<CT, RB1, NW, SEG, WARPS>;
    if (plan.smem > 48 * 1024 && static_cast<int>(plan.smem) > configured_smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(plan.smem));
        if (e != cudaSuccess) return e;
        configured_smem = static_cast<int>(plan.smem);
    }
    if (plan.C > 8) {
        static bool nonportable = false;
        if (!nonportable) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            nonportable = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid_x, grid_y, 1);
    cfg.blockDim = dim3(32 * WARPS, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    // always a cluster launch (of one CTA when C = 1): the exchange addresses
    // shared memory through the cluster window
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = plan.C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

// 8 warps per CTA: 16 (the two halves splitting the row blocks of u) measured
// slower on B300 at every tile shape tried (adapter N=M=4096, R=64, T=16: 4.21 us
// at best against 3.89)
template <int CT, int RB1, bool SEG>
cudaError_t launch_rs_nw(const RsPlan &plan, const RsArgs &args, int grid_y, cudaStream_t stream) {
    if (plan.WARPS != 8) return cudaErrorInvalidValue;
    return plan.NW == 1 ? launch_rs_one<CT, RB1, 1, SEG, 8>(plan, args, grid_y, stream)
                        : launch_rs_one<CT, RB1, 2, SEG, 8>(plan, args, grid_y, stream);
}

// (CT, RB1) pairs with RB1 * CT <= 8 (the stage-1 accumulators stay in registers)
template <bool SEG>
cudaError_t launch_rs_shape(const RsPlan &plan, const RsArgs &args, int grid_y, cudaStream_t stream) {
    switch (plan.RB1 * 16 + plan.CT) {
        case 2 * 16 + 1: return launch_rs_nw<1, 2, SEG>(plan, args, grid_y, stream);
        case 2 * 16 + 2: return launch_rs_nw<2, 2, SEG>(plan, args, grid_y, stream);
        case 2 * 16 + 4: return launch_rs_nw<4, 2, SEG>(plan, args, grid_y, stream);
        case 4 * 16 + 1: return launch_rs_nw<1, 4, SEG>(plan, args, grid_y, stream);
        case 4 * 16 + 2: return launch_rs_nw<2, 4, SEG>(plan, args, grid_y, stream);
        case 6 * 16 + 1: return launch_rs_nw<1, 6, SEG>(plan, args, grid_y, stream);
        case 8 * 16 + 1: return launch_rs_nw<1, 8, SEG>(plan, args, grid_y, stream);
        default: return cudaErrorInvalidValue;
    }
}

int next_pow2(int v) {
    int p = 1;
    while (p < v) p *= 2;
    return p;
}

}  // namespace

// Plan of the reduce-scatter kernel, or CT = 0 when it does not apply (ell = 3,
// R > 128, M > 8192, a partial sum that does not fit the registers).
//   C: the smallest power of two that leaves each warp at most NW packed
//      words of B2 (NW = 1 up to M = 4096, else 2), at most 16.
//   RW: stage-2 rows per CTA; a single call aims at about 64 CTAs (measured
//      on B300 at N = M = 4096: 64 CTAs 3.4 us, 128 CTAs 3.7 us per call),
//      a routed batch at the fewest CTAs per segment.
RsPlan plan_rs(int N, int M, int R, int ell, int columns, int num_sms, int problems, bool accumulate) {
    (void)num_sms;
    (void)accumulate;
    RsPlan best = {};
    if (ell < 1 || ell > 4 || ell == 3 || R < 1 || N < 1 || M < 1) return best;
    const int R2 = (R + 31) & ~31;
    const int RB1 = R2 / 16;
    if (RB1 > 8) return best;
    int CT = 1;
    while (CT * 8 < columns && CT < 8) CT *= 2;
    while (RB1 * CT > 8 && CT > 1) CT /= 2;
    if (RB1 * CT > 8) return best;
    const int CPAD = 8 * CT;
    if (CPAD / ell < 1) return best;
    const int Kw1 = (M + 31) / 32;
    int NW = 1, C = next_pow2((Kw1 + 7) / 8);
    if (C > 16) {
        NW = 2;
        C = next_pow2((Kw1 + 15) / 16);
    }
    if (C > 16) return best;
    if (R2 / C < 2) return best;  // every CTA owns at least one pair of positions of u
    const int Wc = (Kw1 + C - 1) / C;
    double best_cost = 1e300;
    for (int RW = 32; RW <= 128; RW *= 2) {
        const int WARPS = 8;
        const int items = (RW / 16) * CT;
        const int IPW = (items + WARPS - 1) / WARPS;
        if (IPW > 2) continue;
        const int used = (N + RW - 1) / RW;
        const int grid = ((used + C - 1) / C) * C;
        const size_t smem = rs_smem(CPAD, R2, NW, RW, IPW, ell, WARPS).total;
        if (smem > 200 * 1024) continue;
        const double ctas = double(grid) * problems;
        // one column tile: half the CTAs (measured at T = 1: 32 CTAs 3.00 us, 64 CTAs 3.12 us)
        const double aim = CT == 1 ? 32.0 : 64.0;
        const double cost = problems > 1 ? ctas : std::abs(ctas - aim) + (ctas < aim ? 0.5 * RW : 0.0);
        if (cost < best_cost) {
            best_cost = cost;
            best.CT = CT;
            best.RB1 = RB1;
            best.NW = NW;
            best.C = C;
            best.RW = RW;
            best.IPW = IPW;
            best.WARPS = WARPS;
            best.Wc = Wc;
            best.grid_x = grid;
            best.smem = smem;
        }
    }
    return best;
}

size_t rs_smem_bytes(int CT, int RB1, int NW, int RW, int IPW, int ell, int WARPS) {
    return rs_smem(8 * CT, 16 * RB1, NW, RW, IPW, ell, WARPS).total;
}

cudaError_t launch_decode_rs(bool segmented, const RsPlan &plan, const RsArgs &args, int grid_y,
                             cudaStream_t stream) {
    if (plan.CT == 0) return cudaErrorInvalidValue;
    return segmented ? launch_rs_shape<true>(plan, args, grid_y, stream)
                     : launch_rs_shape<false>(plan, args, grid_y, stream);
}

}  // namespace dbfk
