// Decode-regime kernels: y = sum_i alpha_i . B1 (beta_i . (B2 (gamma_i . x)))
// for a handful of tokens (LoRDBA page, section 2, "Núcleo de Inferencia":
// two sign-accumulate matrix products with per-channel scaling between
// them; DBF page, section 2, "Cálculo en la inferencia": the order
// gamma -> B2 -> beta -> B1 -> alpha).
//
// At decode sizes a call moves a few hundred KB to a few MB, which HBM
// delivers in well under a microsecond; what a call costs is its chain of
// dependent latencies.  The kernels are laid out for that:
//   * every input no earlier kernel writes (packed signs, scales) is
//     prefetched with cp.async before griddepcontrol.wait, so it overlaps the
//     previous kernel under programmatic dependent launch;
//   * after the wait a CTA issues all its activation loads at once, and every
//     later phase is spread over all threads (one or two iterations each);
//   * partial sums go from the CTA that made them into the shared memory of
//     the CTA that needs them (st.async inside a thread-block cluster), and
//     their arrival is counted on that CTA's mbarrier: no cluster barrier on
//     the exchange path (the fused kernel's reduce-scatter mode for 32 or more
//     columns keeps its two).
//
// The sign contraction runs on mma.sync m16n8k16 (fp16 in, fp32 accumulate):
// packed sign words are unpacked in registers straight into the A fragment
// (one shift + one LOP3 per fp16 pair, see sign_pair); the activation columns
// (token t, term i -> column t*ell + i) are the B operand, loaded from global
// memory straight into registers in the permuted K order sign_pair expects
// (see decode_frag.cuh).
//
// Two kernel shapes:
//   dec_fused_kernel  (R <= 256; the adapters the reduce-scatter kernel of
//       decode_rs.cu does not take, and routed batches): one launch per call.
//       The CTAs of a cluster split stage 1 over M; every CTA pushes its
//       partial u into every CTA of the cluster, each sums them in rank order,
//       forms the fp16 v = beta*u itself and runs stage 2 for its own slice of
//       the N output rows.  Every cluster recomputes stage 1 (R*M bits, small
//       next to the call when R is small); no intermediate goes through HBM.
//       A routed batch gives every chunk of every segment its own cluster.
//   dec_stage_kernel  (any R): one launch per stage.  Stage 1 writes V (fp16)
//       to the workspace, stage 2 reads it.  A CTA owns 16*RB weight rows and a
//       K slice; the KS CTAs of a cluster split K and push their partials to
//       the CTA that finishes each row.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "decode_frag.cuh"
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

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// The prologue helpers below are kept out of line: each call site inlined
// (an integer division and a loop apiece) made the decode kernels' code larger
// than the SM's instruction cache, and their warps then stalled on
// instruction fetch.

// Copy nrows rows of row_bytes each from global to shared memory with
// cp.async; the chunk size (16, 4 or 2 bytes) is the largest that every
// address and stride allows.  2-byte chunks use plain loads and stores.
__device__ __noinline__ void copy_rows_async(void *dst, int dst_stride, const void *src, size_t src_stride,
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

// As copy_rows_async, for data an earlier kernel may have written (x, V, the
// old y): 16-byte cp.async.cg (through L2 only) when aligned, else plain
// coherent loads and stores.
__device__ __noinline__ void copy_rows_dep(void *dst, int dst_stride, const void *src, size_t src_stride,
                                           int nrows, int row_bytes, int tid, int nthr) {
    if (nrows <= 0 || row_bytes <= 0) return;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    const uintptr_t all = d | s | static_cast<uintptr_t>(dst_stride) | static_cast<uintptr_t>(src_stride) |
                          static_cast<uintptr_t>(row_bytes);
    if ((all & 15) == 0) {
        copy_rows_async(dst, dst_stride, src, src_stride, nrows, row_bytes, tid, nthr);
        return;
    }
    const int q = row_bytes >> 1;
    for (int e = tid; e < nrows * q; e += nthr) {
        const int r = e / q, c = e - r * q;
        *reinterpret_cast<uint16_t *>(static_cast<char *>(dst) + r * dst_stride + 2 * c) =
            *reinterpret_cast<const uint16_t *>(static_cast<const char *>(src) + r * src_stride + 2 * c);
    }
}

// Zero nrows x row_bytes (row_bytes a multiple of 4) of shared memory.
__device__ __noinline__ void zero_rows(void *dst, int dst_stride, int nrows, int row_bytes, int tid, int nthr) {
    const int q = row_bytes >> 2;
    for (int e = tid; e < nrows * q; e += nthr) {
        const int r = e / q, c = e - r * q;
        *reinterpret_cast<uint32_t *>(static_cast<char *>(dst) + r * dst_stride + 4 * c) = 0u;
    }
}

// Zero the tail [from, len) of each of nrows fp16 rows of length len.
__device__ __noinline__ void zero_half_tails(__half *base, int nrows, int len, int from, int tid, int nthr) {
    const int w = len - from;
    if (w <= 0) return;
    for (int e = tid; e < nrows * w; e += nthr) {
        const int i = e / w;
        base[i * len + from + (e - i * w)] = __float2half_rn(0.f);
    }
}

// Words a warp streams per batch: every activation load of a batch is in
// flight before the first conversion.
template <int CT>
__host__ __device__ constexpr int words_per_batch() {
    return CT >= 4 ? 1 : (CT >= 2 ? 2 : 4);
}

// Stage-2 tile (RW rows x columns, fp32) -> y[t][n] = bf16(sum_i alpha_i[n]
// w[t*ell+i][n] (+ y_in)), pairs of adjacent n per thread.
__device__ __forceinline__ void epilogue_tile(const float *tile, int ldt, const __half *alp, int lda_al, int ell,
                                              int ntok, int nrows, int row_base, __nv_bfloat16 *y, size_t ldy,
                                              const __nv_bfloat16 *yst, int ldyst, bool accumulate, bool pairs_ok,
                                              int tid) {
    const int np = (nrows + 1) >> 1;  // row pairs
    for (int e = tid; e < ntok * np; e += kThreads) {
        const int t = e / np, p = e - t * np;
        const int n = 2 * p;
        float s0 = 0.f, s1 = 0.f;
        for (int i = 0; i < ell; ++i) {
            s0 += __half2float(alp[i * lda_al + n]) * tile[n * ldt + t * ell + i];
            s1 += __half2float(alp[i * lda_al + n + 1]) * tile[(n + 1) * ldt + t * ell + i];
        }
        if (accumulate) {
            s0 += __bfloat162float(yst[t * ldyst + n]);
            if (n + 1 < nrows) s1 += __bfloat162float(yst[t * ldyst + n + 1]);
        }
        __nv_bfloat16 *yp = y + size_t(t) * ldy + row_base + n;
        if (pairs_ok && n + 1 < nrows) {
            *reinterpret_cast<__nv_bfloat162 *>(yp) = __floats2bfloat162_rn(s0, s1);
        } else {
            yp[0] = __float2bfloat16_rn(s0);
            if (n + 1 < nrows) yp[1] = __float2bfloat16_rn(s1);
        }
    }
}

// ============================================================ fused kernel

struct FusedSmem {
    size_t gam, b2, beta, b1, alp, red, slots, vs, yst, tile, bar, total;
};

__host__ __device__ inline int fused_g1(int R, int RBW) { return ((R + 15) / 16 + RBW - 1) / RBW; }

// Exchange of the fused kernel.  All-to-all: every CTA pushes its whole
// partial u into every CTA of the cluster, one barrier.  Reduce-scatter +
// broadcast: every row of the partial goes to the CTA that owns it, the owner
// finishes v for its rows and broadcasts it, two barriers.  Measured on B300
// the second barrier costs more than the all-to-all traffic it saves until a
// chunk has 32 or more columns; the scatter also needs every CTA to own a
// whole number of 8-row groups of v.
__host__ __device__ inline bool fused_scatter(int C, int R, int CPAD) {
    const int R2 = (R + 31) & ~31;
    return CPAD >= 32 && C > 1 && R2 % (8 * C) == 0;
}
__host__ __device__ inline int fused_kp(int G1) { return G1 >= kWarps ? 1 : kWarps / G1; }

__host__ __device__ inline FusedSmem fused_smem(int CPAD, int RBW, int Wc, int R, int RW, int ell, int C, bool acc) {
    const int G1 = fused_g1(R, RBW), R1 = 16 * RBW * G1, R2 = (R + 31) & ~31, Kw2 = R2 / 32;
    const int KP = fused_kp(G1);
    FusedSmem L;
    size_t o = 0;
    L.gam = o;
    o += align16(size_t(ell) * 32 * Wc * 2);
    L.b2 = o;
    o += align16(size_t(R1) * ldws_for(Wc) * 4);
    L.beta = o;
    o += align16(size_t(ell) * R2 * 2);
    L.b1 = o;
    o += align16(size_t(RW) * ldws_for(Kw2) * 4);
    L.alp = o;
    o += align16(size_t(ell) * RW * 2);
    L.red = o;
    o += align16(size_t(KP) * R1 * CPAD * 4);
    L.slots = o;  // all-to-all: slot q = partial u of rank q; scatter: [C][R2/C][CPAD] of the owned rows
    o += align16(fused_scatter(C, R, CPAD) ? size_t(C) * (R2 / C) * CPAD * 4 : size_t(C) * R1 * CPAD * 4);
    L.vs = o;
    o += align16(size_t(CPAD) * (R2 + 8) * 2);
    L.yst = o;
    if (acc) o += align16(size_t(CPAD) * RW * 2);
    L.tile = o;
    if (ell == 3) o += size_t(RW) * (CPAD + 4) * 4;
    L.bar = align16(o);  // all-to-all exchange: the mbarrier counting the bytes of every CTA's partial
    o = L.bar + 16;
    L.total = o;
    return L;
}

// Chunk list of a routed batch: segment s (tokens [off[s], off[s+1])) is cut
// into ceil(len / tpc) chunks of tpc tokens, segments in order.  Finds chunk
// q: its segment s, the segment's first token o0, the chunk's first token jt
// inside the segment and its token count jn, and the segment's adapter ad,
// all read in one pass over the table.  Returns false (the same in every
// thread) when q is past the end of the list.  An empty segment and an
// invalid entry (negative length, offsets outside [0, T]; reported with
// o0 = -1) count as one chunk, so that a cluster checks every entry, as in
// the one-segment-per-cluster mode.  Uses 8 ints of shared memory before any
// other use of it; all threads of the CTA take part.
constexpr int kAdTableSmemMax = 8192;  // adapter tables up to this size go to shared memory
static_assert(sizeof(dbf_factors) % 16 == 0, "the adapter table is copied in 16-byte pieces");

__device__ __forceinline__ bool fused_find_chunk(const int32_t *off, const int32_t *seg_ad, int S, int T, int tpc, int q,
                                                 int &s, int &o0, int &jt, int &jn, int &ad, int *sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kPer = (kChunkMapMaxS + kThreads - 1) / kThreads;  // segments per thread
    int lo[kPer], hi[kPer], sa[kPer], cnt[kPer];
    int mine = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = tid * kPer + k;
        lo[k] = i < S ? off[i] : 0;
        hi[k] = i < S ? off[i + 1] : 0;
        sa[k] = i < S ? seg_ad[i] : 0;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = tid * kPer + k;
        const bool ok = !(lo[k] < 0 || hi[k] < lo[k] || hi[k] > T);
        cnt[k] = i >= S ? 0 : (ok ? max(1, (hi[k] - lo[k] + tpc - 1) / tpc) : 1);
        mine += cnt[k];
    }
    // exclusive prefix of the per-thread totals across the CTA (thread order = segment order)
    int incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) sm[warp] = incl;
    __syncthreads();
    int before = incl - mine;
    for (int w = 0; w < warp; ++w) before += sm[w];
    int total = 0;
    for (int w = 0; w < kWarps; ++w) total += sm[w];
    __syncthreads();  // sm is reused below
    if (q >= total) return false;
    if (q >= before && q < before + mine) {
        int acc = before;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            if (q >= acc && q < acc + cnt[k]) {
                const int i = tid * kPer + k;
                const int j = q - acc;
                const bool ok = !(lo[k] < 0 || hi[k] < lo[k] || hi[k] > T);
                sm[0] = i;
                sm[1] = ok ? lo[k] : -1;
                sm[2] = ok ? j * tpc : 0;
                sm[3] = ok ? min(tpc, hi[k] - lo[k] - j * tpc) : 0;
                sm[4] = sa[k];
            }
            acc += cnt[k];
        }
    }
    __syncthreads();
    s = sm[0];
    o0 = sm[1];
    jt = sm[2];
    jn = sm[3];
    ad = sm[4];
    __syncthreads();  // the caller reuses sm
    return true;
}

// What the stage-2 epilogue of the fused kernel needs besides the item.
struct FusedEpi {
    __nv_bfloat16 *y;  // row (t0 + tc0) of y, column row_base: y of the chunk's first token
    const __half *alp_s;
    const __nv_bfloat16 *yst;
    int *status;
    uint32_t tile_addr;
    int N, RW, ell, nrows2, ntok, ldt, acc;
    int tok_left, rows_left;  // (debug build) token rows of y from the chunk's first, rows from row_base
};

// One stage-2 item (rows 16*rb2 .. +15 of the CTA's slice, column tile ct;
// accumulator fragment q0..q3) -> y[t][n] = bf16(sum_i alpha_i[n] q (+ y)),
// or into the fp32 tile for ell = 3.  Inlined: a routed batch runs four
// items side by side, and the epilogues of the four overlap only inline
// (out of line, the routed batch measured 17.4 -> 22.5 us).
__device__ __forceinline__ void fused_epilogue_item(const FusedEpi &e, float q0, float q1, float q2, float q3, int rb2,
                                                 int ct) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int n0 = 16 * rb2 + g;
    if (e.ell == 3) {
        float dd[1][4] = {{q0, q1, q2, q3}};
        put_frag<1>(e.tile_addr + 4u * static_cast<uint32_t>(16 * rb2 * e.ldt + 8 * ct), e.ldt, dd, lane, false, 0);
        return;
    }
    // rows n0 (q0, q1) and n0 + 8 (q2, q3); columns 8ct + 2c, 8ct + 2c + 1
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int nl = n0 + 8 * hh;
        const float d0 = hh ? q2 : q0, d1 = hh ? q3 : q1;
        const bool row_ok = nl < e.nrows2;
        __nv_bfloat16 *yrow = e.y + nl;
        // (debug build) every token row written is a row of y
        auto y_ok = [&](int t) { return in_range(t < e.tok_left && nl < e.rows_left, e.status); };
        if (e.ell == 1) {
            const float al = row_ok ? __half2float(e.alp_s[nl]) : 0.f;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int t = 8 * ct + 2 * c + k;
                if (row_ok && t < e.ntok && y_ok(t)) {
                    float o = al * (k ? d1 : d0);
                    if (e.acc) o += __bfloat162float(e.yst[t * e.RW + nl]);
                    yrow[size_t(t) * e.N] = __float2bfloat16_rn(o);
                }
            }
        } else if (e.ell == 2) {
            const int t = 4 * ct + c;
            if (row_ok && t < e.ntok && y_ok(t)) {
                float o = __half2float(e.alp_s[nl]) * d0 + __half2float(e.alp_s[e.RW + nl]) * d1;
                if (e.acc) o += __bfloat162float(e.yst[t * e.RW + nl]);
                yrow[size_t(t) * e.N] = __float2bfloat16_rn(o);
            }
        } else {  // ell == 4: terms 0,1 in lane c even, 2,3 in lane c odd
            const int i0 = 2 * (c & 1);
            float o = row_ok ? __half2float(e.alp_s[i0 * e.RW + nl]) * d0 +
                                   __half2float(e.alp_s[(i0 + 1) * e.RW + nl]) * d1
                             : 0.f;
            o += __shfl_xor_sync(0xffffffffu, o, 1);
            const int t = 2 * ct + (c >> 1);
            if ((c & 1) == 0 && row_ok && t < e.ntok && y_ok(t)) {
                if (e.acc) o += __bfloat162float(e.yst[t * e.RW + nl]);
                yrow[size_t(t) * e.N] = __float2bfloat16_rn(o);
            }
        }
    }
}

template <int CT, int RBW, bool SEG>
__global__ void __launch_bounds__(kThreads, 2) dec_fused_kernel(const FusedArgs a) {
    constexpr int CPAD = 8 * CT;
    constexpr int C4 = CPAD / 4;
    constexpr int NWB = words_per_batch<CT>();
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, c = lane & 3;
    const int C = a.C;
    const int rank = (C > 1) ? static_cast<int>(cluster_ctarank()) : 0;
    const int ell = a.ell;
    const int N = a.N, M = a.M, R = a.R;

    const uint32_t *B1 = a.B1, *B2 = a.B2;
    int ldw1 = a.ldw1, ldw2 = a.ldw2;
    const __half *alpha = a.alpha, *beta = a.beta, *gamma = a.gamma;
    const int G1 = fused_g1(R, RBW);
    const int R1 = 16 * RBW * G1, R2 = (R + 31) & ~31;
    const int Kw1 = (M + 31) >> 5, Kw2 = R2 >> 5;
    const int KP = fused_kp(G1);
    const int Wc = a.Wc, RW = a.RW;
    const bool acc_mode = a.accumulate != 0;
    const FusedSmem L = fused_smem(CPAD, RBW, Wc, R, RW, ell, C, acc_mode);
    const int w0 = rank * Wc;
    const int Wslice = max(0, min(Wc, Kw1 - w0));

    int t0 = 0, Tseg = a.T;
    if constexpr (SEG) {
        // The adapter table is factor memory (no earlier kernel writes it): in chunk-list
        // mode a small table goes to shared memory (the stage-1 reduction area, unused
        // until stage 1) while the previous kernel finishes, which takes a dependent
        // memory round trip off the path behind the wait.
        const size_t table_bytes = size_t(a.n_adapters) * sizeof(dbf_factors);
        const bool table_s = a.chunk_map_S > 0 && table_bytes <= kAdTableSmemMax &&
                             table_bytes <= size_t(KP) * R1 * CPAD * 4 &&
                             (reinterpret_cast<uintptr_t>(a.adapters) & 15) == 0;
        const dbf_factors *tab = reinterpret_cast<const dbf_factors *>(smem + L.red);
        if (table_s) {
            for (int e = tid; e < static_cast<int>(table_bytes / 16); e += kThreads)
                cp_async_16(smem + L.red + 16 * e, reinterpret_cast<const char *>(a.adapters) + 16 * e);
            cp_async_commit();
        }
        pdl_wait();  // the routing table may come from the previous kernel
        int s = blockIdx.y, o0, ad;
        if (a.chunk_map_S > 0) {
            // every segment in order contributes ceil(len / tpc) chunks; find chunk
            // blockIdx.y (uniform over the cluster: all its CTAs scan the same table)
            const int tpc = CPAD / ell;
            int jt, jn;
            if (table_s) cp_async_wait_all();  // made visible by the barriers of the scan
            if (!fused_find_chunk(a.seg_off, a.seg_ad, a.chunk_map_S, a.T, tpc, static_cast<int>(blockIdx.y), s, o0,
                                  jt, jn, ad, reinterpret_cast<int *>(smem)))
                return;  // a slot past the end of the chunk list
            if (o0 < 0 || jn < 0 || ad < 0 || ad >= a.n_adapters) {
                // reported once per segment: by the cluster of its first chunk
                if (tid == 0 && blockIdx.x == 0 && jt == 0) record_status(a.status, DBF_ERR_DEVICE_ARG);
                return;  // uniform over the cluster: every CTA of it reads the same entry
            }
            t0 = o0 + jt;
            Tseg = jn;
            // this CTA's activation slice into L2 while the factors are looked up and fetched
            if (Tseg > 0) {
                const int lines = (Wslice * 64 + 127) / 128;
                for (int e = tid; e < Tseg * lines; e += kThreads) {
                    const int t = e / lines, l = e - t * lines;
                    prefetch_l2(a.x + size_t(t0 + t) * M + 32 * w0 + 64 * l);
                }
            }
        } else {
            o0 = a.seg_off[s];
            const int o1 = a.seg_off[s + 1];
            ad = a.seg_ad[s];
            if (o0 < 0 || o1 < o0 || o1 > a.T || ad < 0 || ad >= a.n_adapters) {
                if (tid == 0 && blockIdx.x == 0) record_status(a.status, DBF_ERR_DEVICE_ARG);
                return;  // uniform over the cluster: every CTA of it reads the same entry
            }
            t0 = o0;
            Tseg = o1 - o0;
        }
        const dbf_factors f = table_s ? tab[ad] : a.adapters[ad];
        B1 = f.B1;
        B2 = f.B2;
        ldw1 = f.ldw1;
        ldw2 = f.ldw2;
        alpha = reinterpret_cast<const __half *>(f.alpha);
        beta = reinterpret_cast<const __half *>(f.beta);
        gamma = reinterpret_cast<const __half *>(f.gamma);
        if (Tseg == 0) return;
        if (table_s) __syncthreads();  // every thread holds its copy of the entry before the area is reused
    }

    __half *gam_s = reinterpret_cast<__half *>(smem + L.gam);
    uint32_t *b2_s = reinterpret_cast<uint32_t *>(smem + L.b2);
    __half *beta_s = reinterpret_cast<__half *>(smem + L.beta);
    uint32_t *b1_s = reinterpret_cast<uint32_t *>(smem + L.b1);
    __half *alp_s = reinterpret_cast<__half *>(smem + L.alp);
    float *red = reinterpret_cast<float *>(smem + L.red);
    float *slots = reinterpret_cast<float *>(smem + L.slots);
    __half *vs = reinterpret_cast<__half *>(smem + L.vs);
    __nv_bfloat16 *yst = reinterpret_cast<__nv_bfloat16 *>(smem + L.yst);
    float *tile = reinterpret_cast<float *>(smem + L.tile);

    const int ldb2 = ldws_for(Wc), ldb1 = ldws_for(Kw2);
    const int ldv = R2 + 8, ldt = CPAD + 4;
    const int kvalid = max(0, min(32 * Wslice, M - 32 * w0));
    const int row_base = blockIdx.x * RW;  // first stage-2 output row of this CTA
    const int nrows2 = max(0, min(RW, N - row_base));

    // ---- 1. inputs no earlier kernel writes: signs and scales
    copy_rows_async(b2_s, ldb2 * 4, B2 + w0, size_t(ldw2) * 4, R, Wslice * 4, tid, kThreads);
    zero_rows(b2_s + R * ldb2, ldb2 * 4, R1 - R, Wslice * 4, tid, kThreads);
    if (kvalid > 0) copy_rows_async(gam_s, 64 * Wc, gamma + 32 * w0, size_t(M) * 2, ell, kvalid * 2, tid, kThreads);
    zero_half_tails(gam_s, ell, 32 * Wc, kvalid, tid, kThreads);
    copy_rows_async(beta_s, R2 * 2, beta, size_t(R) * 2, ell, R * 2, tid, kThreads);
    zero_half_tails(beta_s, ell, R2, R, tid, kThreads);
    copy_rows_async(b1_s, ldb1 * 4, B1 + size_t(row_base) * ldw1, size_t(ldw1) * 4, nrows2, Kw2 * 4, tid, kThreads);
    zero_rows(b1_s + nrows2 * ldb1, ldb1 * 4, RW - nrows2, Kw2 * 4, tid, kThreads);
    copy_rows_async(alp_s, RW * 2, alpha + row_base, size_t(N) * 2, ell, nrows2 * 2, tid, kThreads);
    cp_async_commit();
    // all-to-all exchange: every CTA of the cluster (this one included) sends its partial u
    // of a chunk with st.async, counted on this CTA's mbarrier (one phase per chunk)
    const bool scatter = CPAD >= 32 && fused_scatter(C, R, CPAD);  // (compiled for 32+ columns only)
    uint64_t *xbar = reinterpret_cast<uint64_t *>(smem + L.bar);
    const uint32_t a2a_bytes = uint32_t(C) * R1 * CPAD * 4;
    if (C > 1 && !scatter && tid == 0) {
        mbar_init(xbar, 1);
        mbar_arrive_expect_tx(xbar, a2a_bytes);
        fence_mbar_init();
    }
    if (C > 1) cluster_arrive_relaxed();  // matched by the wait before the first push
    pdl_trigger();
    if constexpr (!SEG) pdl_wait();

    // this warp's stage-1 item: row group gr, K part kp, words [wb, we) of the slice
    const bool has1 = warp < G1 * KP;
    const int gr = warp % G1, kp = warp / G1;
    const int Wp = (Wslice + KP - 1) / KP;
    const int wb = min(Wslice, kp * Wp), we = has1 ? min(Wslice, wb + Wp) : wb;
    // the lane's activation column in each column tile: token, term
    int ctok[CT], cterm[CT];
#pragma unroll
    for (int ct = 0; ct < CT; ++ct) {
        const int col = 8 * ct + g;
        ctok[ct] = col / ell;
        cterm[ct] = col - ctok[ct] * ell;
    }
    // the thread's columns in the reduction phases (the stride is a multiple of C4)
    const int c4 = tid % C4;
    int term4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) term4[j] = (4 * c4 + j) % ell;

    const int tpc = CPAD / ell;  // whole tokens per column chunk
    const int nchunks = (Tseg + tpc - 1) / tpc;
    const bool xvec = ((M & 7) == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0);
    const bool pairs_ok = ((N & 1) == 0);
    const uint32_t red_addr = smem_u32(red), slots_addr = smem_u32(slots), tile_addr = smem_u32(tile);
    const uint32_t vs_addr = smem_u32(vs);
    const int RB2 = RW / 16;
    const int RO = R2 / C;  // rows of v each CTA of the cluster finishes (scatter mode)

    for (int chunk = 0; chunk < nchunks; ++chunk) {
        const int tc0 = chunk * tpc;
        const int ntok = min(tpc, Tseg - tc0);
        const int ncol = ntok * ell;
        const int ctu = (ncol + 7) >> 3;  // column tiles that hold a column of this chunk
        if (chunk > 0 && C > 1) {
            // re-armed before the barrier: no peer sends this chunk's partial until it has passed it
            if (!scatter && tid == 0) mbar_arrive_expect_tx(xbar, a2a_bytes);
            cluster_sync_all();  // peers finished reading the previous chunk's slots
        }
        const __nv_bfloat16 *xc = a.x + size_t(t0 + tc0) * M;

        // ---- 2. old y by cp.async; the first batch of x straight into registers
        if (acc_mode)
            copy_rows_dep(yst, RW * 2, a.y + size_t(t0 + tc0) * N + row_base, size_t(N) * 2, ntok, nrows2 * 2,
                          tid, kThreads);
        cp_async_commit();
        uint4 xr[NWB][CT];
        auto load_batch = [&](int wbat) {
#pragma unroll
            for (int w = 0; w < NWB; ++w)
#pragma unroll
                for (int ct = 0; ct < CT; ++ct) {
                    const int col = 8 * ct + g;
                    if (wbat + w < we && col < ncol)
                        xr[w][ct] = load_x8(xc + size_t(ctok[ct]) * M, 32 * (w0 + wbat + w) + 8 * c, M, xvec);
                    else
                        xr[w][ct] = make_uint4(0u, 0u, 0u, 0u);
                }
        };
        load_batch(wb);
        cp_async_wait_all();
        __syncthreads();  // signs, scales and the old y are in shared memory
        if (chunk == 0 && C > 1) cluster_wait();  // every CTA of the cluster has started

        // ---- 3. stage 1 on this warp's words: x pairs from registers, signs from shared memory
        if (has1) {
            float acc[RBW][CT][4];
#pragma unroll
            for (int rb = 0; rb < RBW; ++rb) zero_acc<CT>(acc[rb]);
            for (int wbat = wb; wbat < we; wbat += NWB) {
                if (wbat != wb) load_batch(wbat);
#pragma unroll
                for (int w = 0; w < NWB; ++w) {
                    const int wl = wbat + w;
                    if (wl >= we) break;
                    uint32_t bx[CT][4];
#pragma unroll
                    for (int ct = 0; ct < CT; ++ct) {
                        if (ct >= ctu) break;
                        const uint4 gv = *reinterpret_cast<const uint4 *>(gam_s + cterm[ct] * 32 * Wc + 32 * wl + 8 * c);
                        x_pairs(xr[w][ct], gv, bx[ct]);
                    }
#pragma unroll
                    for (int rb = 0; rb < RBW; ++rb) {
                        const int r0 = 16 * (gr * RBW + rb) + g;
                        uint32_t pa[4], pv[4];
                        sign_pairs8(b2_s[r0 * ldb2 + wl], c, pa);
                        sign_pairs8(b2_s[(r0 + 8) * ldb2 + wl], c, pv);
#pragma unroll
                        for (int ct = 0; ct < CT; ++ct)
                            if (ct < ctu) mma_word8(acc[rb][ct], pa, pv, bx[ct]);
                    }
                }
            }
#pragma unroll
            for (int rb = 0; rb < RBW; ++rb)
                put_frag<CT>(red_addr + 4u * static_cast<uint32_t>((kp * R1 + 16 * (gr * RBW + rb)) * CPAD), CPAD,
                             acc[rb], lane, false, 0);
        }
        __syncthreads();

        if (scatter) {
            // ---- 4. sum the K parts; each row of the partial u goes to the CTA
            //         that owns it (slot `rank` of owner r / RO)
            const int rows_x = min(R1, R2);  // rows of u stage 2 reads (owner ranks < C)
            for (int e = tid; e < rows_x * C4; e += kThreads) {
                const int r = e / C4;
                float4 u = *reinterpret_cast<const float4 *>(red + r * CPAD + 4 * c4);
                for (int q = 1; q < KP; ++q)
                    add4(u, *reinterpret_cast<const float4 *>(red + (q * R1 + r) * CPAD + 4 * c4));
                const int owner = r / RO, rl = r - owner * RO;
                asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(mapa_shared(
                                 slots_addr + 4u * static_cast<uint32_t>((rank * RO + rl) * CPAD + 4 * c4),
                                 static_cast<uint32_t>(owner))),
                             "f"(u.x), "f"(u.y), "f"(u.z), "f"(u.w)
                             : "memory");
            }
            cluster_sync_all();  // every owner holds the partials of its rows

            // ---- 5. owner: u of its RO rows = sum over ranks (rank order), v =
            //         beta * u (fp16) staged in perm8 order, then broadcast in
            //         16-byte pieces into v of every CTA of the cluster
            __half *stage = reinterpret_cast<__half *>(red);  // [CPAD][RO], free after step 4
            for (int e = tid; e < CPAD * RO; e += kThreads) {
                const int col = e / RO, rl = e - col * RO;
                const int r = rank * RO + rl;
                float u = 0.f;
                if (r < R1)
                    for (int q = 0; q < C; ++q) u += slots[(q * RO + rl) * CPAD + col];
                const float v = __half2float(beta_s[(col % ell) * R2 + r]) * u;
                stage[col * RO + (perm8_pos(r) - rank * RO)] = __float2half_rn(v);
            }
            __syncthreads();
            const int pieces = CPAD * (RO / 8);
            for (int e = tid; e < pieces * C; e += kThreads) {
                const int q = e / pieces, pc = e - q * pieces;
                const int col = pc / (RO / 8), k8 = pc - col * (RO / 8);
                const uint4 val = *reinterpret_cast<const uint4 *>(stage + col * RO + 8 * k8);
                const uint32_t dst = vs_addr + 2u * static_cast<uint32_t>(col * ldv + rank * RO + 8 * k8);
                asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 mapa_shared(dst, static_cast<uint32_t>(q))),
                             "r"(val.x), "r"(val.y), "r"(val.z), "r"(val.w)
                             : "memory");
            }
            cluster_sync_all();  // v of every CTA is complete
        } else {
            // ---- 4. sum the K parts, push the CTA's partial u into slot `rank` of every CTA
            for (int e = tid; e < R1 * C4; e += kThreads) {
                const int r = e / C4;
                float4 u = *reinterpret_cast<const float4 *>(red + r * CPAD + 4 * c4);
                for (int q = 1; q < KP; ++q)
                    add4(u, *reinterpret_cast<const float4 *>(red + (q * R1 + r) * CPAD + 4 * c4));
                const uint32_t off = slots_addr + 4u * static_cast<uint32_t>((rank * R1 + r) * CPAD + 4 * c4);
                if (C > 1) {
                    for (int q = 0; q < C; ++q)
                        st_async_v4(mapa_shared(off, static_cast<uint32_t>(q)), u,
                                    mapa_shared(smem_u32(xbar), static_cast<uint32_t>(q)));
                } else {
                    *reinterpret_cast<float4 *>(slots + r * CPAD + 4 * c4) = u;
                }
            }
            if (C > 1) {
                // every slot of this CTA is filled once the chunk's bytes have all arrived
                if (!mbar_wait_bounded(xbar, static_cast<uint32_t>(chunk & 1), nullptr))
                    record_status(a.status, DBF_ERR_TIMEOUT);
            } else {
                __syncthreads();
            }

            // ---- 5. u = sum of the slots in rank order, v = beta * u (fp16, perm8 order)
            for (int e = tid; e < R2 * C4; e += kThreads) {
                const int r = e / C4;
                float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < R1)
                    for (int q = 0; q < C; ++q)
                        add4(u, *reinterpret_cast<const float4 *>(slots + (q * R1 + r) * CPAD + 4 * c4));
                const float uu[4] = {u.x, u.y, u.z, u.w};
                const int pos = perm8_pos(r);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    vs[(4 * c4 + j) * ldv + pos] = __float2half_rn(__half2float(beta_s[term4[j] * R2 + r]) * uu[j]);
            }
            __syncthreads();
        }

        // ---- 6. stage 2 per (row block, column tile); y straight from the fragment.
        //         Routed batches give a warp many items (a CTA covers up to 1024
        //         rows); there a warp runs kIB of them side by side, so their
        //         independent chains of loads, MMAs and epilogue overlap.
        constexpr int kIB = 4;
        FusedEpi epi;
        epi.y = a.y + size_t(t0 + tc0) * N + row_base;
        epi.alp_s = alp_s;
        epi.yst = yst;
        epi.status = a.status;
        epi.tile_addr = tile_addr;
        epi.N = N;
        epi.RW = RW;
        epi.ell = ell;
        epi.nrows2 = nrows2;
        epi.ntok = ntok;
        epi.ldt = ldt;
        epi.acc = acc_mode;
        epi.tok_left = a.T - (t0 + tc0);
        epi.rows_left = N - row_base;
        auto epilogue_item = [&](const float (&d)[4], int rb2, int ct) {
            fused_epilogue_item(epi, d[0], d[1], d[2], d[3], rb2, ct);
        };
        // items of the column tiles that hold columns (a routed segment is often
        // shorter than the chunk); a single adapter gives a warp few items: one
        // at a time there, as a batch only adds work
        const int items = RB2 * ctu;
        if constexpr (!SEG) {
            for (int it = warp; it < items; it += kWarps) {
                const int rb2 = it % RB2, ct = it / RB2;
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                const int n0 = 16 * rb2 + g;
                for (int w = 0; w < Kw2; ++w) {
                    const uint4 bv = *reinterpret_cast<const uint4 *>(vs + (8 * ct + g) * ldv + 32 * w + 8 * c);
                    const uint32_t bb[4] = {bv.x, bv.y, bv.z, bv.w};
                    uint32_t pa[4], pv[4];
                    sign_pairs8(b1_s[n0 * ldb1 + w], c, pa);
                    sign_pairs8(b1_s[(n0 + 8) * ldb1 + w], c, pv);
                    mma_word8(d, pa, pv, bb);
                }
                epilogue_item(d, rb2, ct);
            }
        }
        if constexpr (SEG) {
        for (int it0 = warp; it0 < items; it0 += kWarps * kIB) {
            float d[kIB][4];
            int rbv[kIB], ctv[kIB];
#pragma unroll
            for (int b = 0; b < kIB; ++b) {
                const int it = it0 + b * kWarps;  // warp-uniform
                rbv[b] = it % RB2;
                ctv[b] = it / RB2;
#pragma unroll
                for (int j = 0; j < 4; ++j) d[b][j] = 0.f;
            }
            for (int w = 0; w < Kw2; ++w) {
#pragma unroll
                for (int b = 0; b < kIB; ++b) {
                    if (it0 + b * kWarps >= items) break;
                    const int n0 = 16 * rbv[b] + g;
                    const uint4 bv = *reinterpret_cast<const uint4 *>(vs + (8 * ctv[b] + g) * ldv + 32 * w + 8 * c);
                    const uint32_t bb[4] = {bv.x, bv.y, bv.z, bv.w};
                    uint32_t pa[4], pv[4];
                    sign_pairs8(b1_s[n0 * ldb1 + w], c, pa);
                    sign_pairs8(b1_s[(n0 + 8) * ldb1 + w], c, pv);
                    mma_word8(d[b], pa, pv, bb);
                }
            }
#pragma unroll
            for (int b = 0; b < kIB; ++b) {
                if (it0 + b * kWarps >= items) break;
                epilogue_item(d[b], rbv[b], ctv[b]);
            }
        }
        }
        if (ell == 3) {
            __syncthreads();
            epilogue_tile(tile, ldt, alp_s, RW, ell, ntok, nrows2, row_base, a.y + size_t(t0 + tc0) * N, size_t(N), yst,
                          RW, acc_mode, pairs_ok, tid);
        }
        __syncthreads();  // vs / red / slots / yst / tile are reused by the next chunk
    }
}

// ============================================================== stage kernel
//
// One stage of the two-stage decode.  A CTA owns 16*RBW weight rows
// [row0, row0 + 16*RBW) and one K slice (the KS CTAs of a cluster split the
// packed words); its 8 warps split the slice again.  Warp partials are summed
// in shared memory; with KS > 1 each CTA then pushes the rows owned by rank q
// (16*RBW/KS consecutive rows) into slot `rank` of CTA q, which sums the KS
// slots and writes the outputs of its rows.

struct StageSmem {
    size_t gam, bits, sc, yst, red, slots, total;
};

__host__ __device__ inline StageSmem stage_smem(int CPAD, int RBW, int KS, int Wc, int ell, bool stage1, bool acc) {
    const int RWS = 16 * RBW;
    StageSmem L;
    size_t o = 0;
    L.gam = o;
    if (stage1) o += align16(size_t(ell) * 32 * Wc * 2);
    L.bits = o;
    o += align16(size_t(RWS) * ldws_for(Wc) * 4);
    L.sc = o;
    o += align16(size_t(ell) * RWS * 2);
    L.yst = o;
    if (!stage1 && acc) o += align16(size_t(CPAD) * RWS * 2);
    L.red = o;
    o += align16(size_t(kWarps) * RWS * CPAD * 4);
    L.slots = o;  // KS > 1: [2 buffers][KS][RWS/KS][CPAD] partials of the owned rows, then 2 mbarriers
    if (KS > 1) o += align16(size_t(2) * RWS * CPAD * 4) + 16;
    L.total = o;
    return L;
}

// bx: this CTA's index along the rows of its problem (blockIdx.x, or the
// offset inside its problem's range in a grouped launch); smem_off: where this
// stage's shared-memory layout starts in the dynamic shared memory (a 128-byte
// multiple; nonzero only when one launch runs both stages).  PART 0 runs the
// whole stage; when one launch runs both stages, PART 1 only starts the
// asynchronous copies of the signs and scales (no wait) and PART 2 runs the
// rest without them, after the CTA's own cp.async groups have completed.
template <int CT, int RBW, int STAGE, bool SEG, int PART = 0>
__device__ __forceinline__ void dec_stage_body(const DecArgs &a, const int bx, const uint32_t smem_off = 0) {
    static_assert(PART == 0 || !SEG, "split stages are not segmented");
    constexpr int CPAD = 8 * CT;
    constexpr int C4 = CPAD / 4;
    constexpr int RWS = 16 * RBW;
    constexpr int NWB = words_per_batch<CT>();
    extern __shared__ __align__(128) unsigned char smem_dyn[];
    unsigned char *const smem = smem_dyn + smem_off;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, c = lane & 3;
    const int KS = a.KS, Wc = a.Wc;
    const int rank = (KS > 1) ? static_cast<int>(cluster_ctarank()) : 0;
    const int row0 = (bx / KS) * RWS;
    const int ell = a.ell;

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
            if (tid == 0 && bx == 0) record_status(a.status, DBF_ERR_DEVICE_ARG);
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

    const StageSmem L = stage_smem(CPAD, RBW, KS, Wc, ell, STAGE == 1, a.accumulate != 0);
    const int w0 = rank * Wc;
    const int Wslice = max(0, min(Wc, a.Kw - w0));
    const int kvalid = max(0, min(32 * Wslice, a.K - 32 * w0));
    const int ldws = ldws_for(Wc);
    const int nr = max(0, min(RWS, a.rows - row0));  // weight rows that exist
    const int ROWN = RWS / KS;                       // rows each CTA of the cluster finishes
    __half *gam_s = reinterpret_cast<__half *>(smem + L.gam);
    uint32_t *bits_s = reinterpret_cast<uint32_t *>(smem + L.bits);
    __half *sc_s = reinterpret_cast<__half *>(smem + L.sc);
    __nv_bfloat16 *yst = reinterpret_cast<__nv_bfloat16 *>(smem + L.yst);
    float *red = reinterpret_cast<float *>(smem + L.red);
    float *slots = reinterpret_cast<float *>(smem + L.slots);

    // ---- 1. inputs no earlier kernel writes: packed signs and scales
    if constexpr (PART != 2) {
        copy_rows_async(bits_s, ldws * 4, bits + size_t(row0) * ldw + w0, size_t(ldw) * 4, nr, Wslice * 4, tid,
                        kThreads);
        zero_rows(bits_s + nr * ldws, ldws * 4, RWS - nr, Wslice * 4, tid, kThreads);
        copy_rows_async(sc_s, RWS * 2, scale_out + row0, size_t(a.rows) * 2, ell, nr * 2, tid, kThreads);
        zero_half_tails(sc_s, ell, RWS, nr, tid, kThreads);
        if (STAGE == 1) {
            if (kvalid > 0)
                copy_rows_async(gam_s, 64 * Wc, scale_in + 32 * w0, size_t(a.K) * 2, ell, kvalid * 2, tid, kThreads);
            zero_half_tails(gam_s, ell, 32 * Wc, kvalid, tid, kThreads);
        }
        cp_async_commit();
    }
    if constexpr (PART == 1) return;
    // KS > 1: the partial of every owned row arrives from each CTA of the cluster with st.async;
    // one mbarrier per buffer counts the bytes of one chunk
    uint64_t *xbar = reinterpret_cast<uint64_t *>(smem + L.slots + align16(size_t(2) * RWS * CPAD * 4));
    const uint32_t chunk_bytes = uint32_t(RWS) * CPAD * 4;
    if (KS > 1) {
        if (tid == 0) {
            mbar_init(&xbar[0], 1);
            mbar_init(&xbar[1], 1);
            mbar_arrive_expect_tx(&xbar[0], chunk_bytes);
            mbar_arrive_expect_tx(&xbar[1], chunk_bytes);
            fence_mbar_init();
        }
        cluster_arrive_relaxed();  // matched by the wait before the first send
    }
    pdl_trigger();
    if constexpr (!SEG) pdl_wait();

    // this warp's words of the slice
    const int Wp = (Wslice + kWarps - 1) / kWarps;
    const int wb = min(Wslice, warp * Wp), we = min(Wslice, wb + Wp);
    int ctok[CT], cterm[CT];
#pragma unroll
    for (int ct = 0; ct < CT; ++ct) {
        const int col = 8 * ct + g;
        ctok[ct] = col / ell;
        cterm[ct] = col - ctok[ct] * ell;
    }
    const int tpc = CPAD / ell;  // whole tokens per column chunk
    const int nchunks = (Tseg + tpc - 1) / tpc;
    const bool xvec = ((a.ldx & 7) == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0);
    const uint32_t red_addr = smem_u32(red);
    const int c4 = tid % C4;
    const int nsl = (KS > 1) ? KS : kWarps;      // partial slices summed in the epilogue, in order
    const int prows = (KS > 1) ? ROWN : RWS;     // rows per slice
    const int rown0 = (KS > 1) ? rank * ROWN : 0;
    const bool pairs_ok = ((a.ldy & 1) == 0);

    for (int chunk = 0; chunk < nchunks; ++chunk) {
        const int tc0 = chunk * tpc;
        const int ntok = min(tpc, Tseg - tc0);
        const int ncol = ntok * ell;
        const int buf = chunk & 1;
        const uint32_t ph = (chunk >> 1) & 1;
        // KS > 1: the owned rows' partials of this chunk, [KS][ROWN][CPAD]; else the warp partials
        const float *part = (KS > 1) ? slots + size_t(buf) * RWS * CPAD : red;
        if (chunk > 0 && KS > 1) {
            // the previous chunk's epilogue is done with `red` and its buffer; a peer writes into this
            // chunk's buffer only after it received this CTA's partial of the chunk before
            __syncthreads();
            if (chunk >= 2 && tid == 0) mbar_arrive_expect_tx(&xbar[buf], chunk_bytes);
        }

        // ---- 2. the first batch of activations straight into registers
        if (STAGE == 2 && a.accumulate)
            copy_rows_dep(yst, RWS * 2, a.y + size_t(t0 + tc0) * a.ldy + row0, size_t(a.ldy) * 2, ntok, nr * 2, tid,
                          kThreads);
        cp_async_commit();
        uint4 xr[NWB][CT];
        auto load_batch = [&](int wbat) {
#pragma unroll
            for (int w = 0; w < NWB; ++w)
#pragma unroll
                for (int ct = 0; ct < CT; ++ct) {
                    const int col = 8 * ct + g;
                    if (wbat + w < we && col < ncol) {
                        if constexpr (STAGE == 1) {
                            xr[w][ct] = load_x8(a.x + size_t(t0 + tc0 + ctok[ct]) * a.ldx,
                                                32 * (w0 + wbat + w) + 8 * c, a.K, xvec);
                        } else {
                            xr[w][ct] = *reinterpret_cast<const uint4 *>(
                                a.V + (size_t(t0 + tc0) * ell + col) * a.ldv + 32 * (w0 + wbat + w) + 8 * c);
                        }
                    } else {
                        xr[w][ct] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
        };
        load_batch(wb);
        cp_async_wait_all();
        __syncthreads();  // signs and scales are in shared memory

        // ---- 3. tensor-core sign contraction over this warp's words
        {
            float acc[RBW][CT][4];
#pragma unroll
            for (int rb = 0; rb < RBW; ++rb) zero_acc<CT>(acc[rb]);
            if (we - wb == NWB) {
                // exactly one batch of words: straight-line code, so the scheduler sees every
                // shared-memory load, unpack and MMA of the warp at once (measured on the 1.5-bit
                // layer: the stage-1 contraction 1.54 -> 1.22 us per CTA)
                uint32_t bxs[NWB][CT][4];
#pragma unroll
                for (int w = 0; w < NWB; ++w)
#pragma unroll
                    for (int ct = 0; ct < CT; ++ct) {
                        if constexpr (STAGE == 1) {
                            const uint4 gv =
                                *reinterpret_cast<const uint4 *>(gam_s + cterm[ct] * 32 * Wc + 32 * (wb + w) + 8 * c);
                            x_pairs(xr[w][ct], gv, bxs[w][ct]);
                        } else {
                            bxs[w][ct][0] = xr[w][ct].x;
                            bxs[w][ct][1] = xr[w][ct].y;
                            bxs[w][ct][2] = xr[w][ct].z;
                            bxs[w][ct][3] = xr[w][ct].w;
                        }
                    }
#pragma unroll
                for (int w = 0; w < NWB; ++w)
#pragma unroll
                    for (int rb = 0; rb < RBW; ++rb) {
                        const int r0 = 16 * rb + g;
                        uint32_t pa[4], pv[4];
                        sign_pairs8(bits_s[r0 * ldws + wb + w], c, pa);
                        sign_pairs8(bits_s[(r0 + 8) * ldws + wb + w], c, pv);
#pragma unroll
                        for (int ct = 0; ct < CT; ++ct) mma_word8(acc[rb][ct], pa, pv, bxs[w][ct]);
                    }
            } else {
                for (int wbat = wb; wbat < we; wbat += NWB) {
                    if (wbat != wb) load_batch(wbat);
#pragma unroll
                    for (int w = 0; w < NWB; ++w) {
                        const int wl = wbat + w;
                        if (wl >= we) break;
                        uint32_t bx[CT][4];
#pragma unroll
                        for (int ct = 0; ct < CT; ++ct) {
                            if constexpr (STAGE == 1) {
                                const uint4 gv =
                                    *reinterpret_cast<const uint4 *>(gam_s + cterm[ct] * 32 * Wc + 32 * wl + 8 * c);
                                x_pairs(xr[w][ct], gv, bx[ct]);
                            } else {
                                bx[ct][0] = xr[w][ct].x;
                                bx[ct][1] = xr[w][ct].y;
                                bx[ct][2] = xr[w][ct].z;
                                bx[ct][3] = xr[w][ct].w;
                            }
                        }
#pragma unroll
                        for (int rb = 0; rb < RBW; ++rb) {
                            const int r0 = 16 * rb + g;
                            uint32_t pa[4], pv[4];
                            sign_pairs8(bits_s[r0 * ldws + wl], c, pa);
                            sign_pairs8(bits_s[(r0 + 8) * ldws + wl], c, pv);
#pragma unroll
                            for (int ct = 0; ct < CT; ++ct) mma_word8(acc[rb][ct], pa, pv, bx[ct]);
                        }
                    }
                }
            }
#pragma unroll
            for (int rb = 0; rb < RBW; ++rb)
                put_frag<CT>(red_addr + 4u * static_cast<uint32_t>((warp * RWS + 16 * rb) * CPAD), CPAD, acc[rb], lane,
                             false, 0);
        }
        __syncthreads();

        // ---- 4. cluster: sum the warp partials (in warp order) and send each row to the CTA
        //         of the cluster that finishes it (st.async, counted on its mbarrier)
        if (KS > 1) {
            if (chunk == 0) cluster_wait();  // every CTA of the cluster has initialised its barriers
            for (int e = tid; e < RWS * C4; e += kThreads) {
                const int r = e / C4;
                float4 u = *reinterpret_cast<const float4 *>(red + r * CPAD + 4 * c4);
                for (int q = 1; q < kWarps; ++q)
                    add4(u, *reinterpret_cast<const float4 *>(red + (q * RWS + r) * CPAD + 4 * c4));
                const int owner = r / ROWN, rl = r - owner * ROWN;
                if (!in_range(owner < KS, a.status)) continue;
                const float *dst = slots + size_t(buf) * RWS * CPAD + (size_t(rank) * ROWN + rl) * CPAD + 4 * c4;
                st_async_v4(mapa_shared(smem_u32(dst), static_cast<uint32_t>(owner)), u,
                            mapa_shared(smem_u32(&xbar[buf]), static_cast<uint32_t>(owner)));
            }
            if (!mbar_wait_bounded(&xbar[buf], ph, nullptr)) record_status(a.status, DBF_ERR_TIMEOUT);
        }

        // ---- 5. epilogue of this CTA's rows [rown0, rown0 + prows)
        if constexpr (STAGE == 1) {
            // V[(t0+tc0)*ell + col][perm8(r)]: pairs (r, r+4) of each 8-row group
            const size_t vrow0 = size_t(t0 + tc0) * ell;
            const int npairs = prows / 2;
            for (int e = tid; e < ncol * npairs; e += kThreads) {
                const int col = e / npairs, p = e - col * npairs;
                const int rl = 8 * (p >> 2) + (p & 3);  // row inside the owned range, first of the pair
                const int r = row0 + rown0 + rl;
                if (r >= a.rows_out) continue;
                float u0 = 0.f, u1 = 0.f;
                for (int q = 0; q < nsl; ++q) {
                    const float *b = part + size_t(q) * prows * CPAD;
                    u0 += b[rl * CPAD + col];
                    u1 += b[(rl + 4) * CPAD + col];
                }
                const int i = col % ell;
                const float v0 = __half2float(sc_s[i * RWS + rown0 + rl]) * u0;
                const float v1 = __half2float(sc_s[i * RWS + rown0 + rl + 4]) * u1;
                if (!in_range(vrow0 + col < size_t(a.T) * ell && (r & ~7) + 2 * (r & 3) + 1 < a.ldv, a.status))
                    continue;
                *reinterpret_cast<__half2 *>(a.V + (vrow0 + col) * a.ldv + (r & ~7) + 2 * (r & 3)) =
                    __floats2half2_rn(v0, v1);
            }
        } else {
            // y[t][n], n pairs (n, n+1)
            const int npairs = prows / 2;
            for (int e = tid; e < ntok * npairs; e += kThreads) {
                const int t = e / npairs, p = e - t * npairs;
                const int rl = 2 * p;
                const int n = row0 + rown0 + rl;
                if (n >= a.rows) continue;
                float s0 = 0.f, s1 = 0.f;
                for (int q = 0; q < nsl; ++q) {
                    const float *b = part + size_t(q) * prows * CPAD;
                    for (int i = 0; i < ell; ++i) {
                        s0 += __half2float(sc_s[i * RWS + rown0 + rl]) * b[rl * CPAD + t * ell + i];
                        s1 += __half2float(sc_s[i * RWS + rown0 + rl + 1]) * b[(rl + 1) * CPAD + t * ell + i];
                    }
                }
                const bool two = n + 1 < a.rows;
                if (a.accumulate) {
                    s0 += __bfloat162float(yst[t * RWS + rown0 + rl]);
                    if (two) s1 += __bfloat162float(yst[t * RWS + rown0 + rl + 1]);
                }
                if (!in_range(t0 + tc0 + t < a.T && n + (two ? 1 : 0) < a.ldy, a.status)) continue;
                __nv_bfloat16 *yp = a.y + size_t(t0 + tc0 + t) * a.ldy + n;
                if (pairs_ok && two) {
                    *reinterpret_cast<__nv_bfloat162 *>(yp) = __floats2bfloat162_rn(s0, s1);
                } else {
                    yp[0] = __float2bfloat16_rn(s0);
                    if (two) yp[1] = __float2bfloat16_rn(s1);
                }
            }
        }
        __syncthreads();  // red / slots / yst are reused by the next chunk
    }
    // Every byte a peer sends to this CTA has arrived once its waits above returned, so no
    // peer writes into this CTA's shared memory after it exits.
}

template <int CT, int RBW, int STAGE, bool SEG>
__global__ void __launch_bounds__(kThreads, 2) dec_stage_kernel(const DecArgs a) {
    dec_stage_body<CT, RBW, STAGE, SEG>(a, static_cast<int>(blockIdx.x));
}

// Grouped launch: G independent problems of any shape (same ell and T) in one
// launch.  Problem p owns CTAs [block0[p], block0[p+1]) along x, a multiple of
// the cluster size, and runs exactly as its own launch would.
template <int CT, int RBW, int STAGE>
__global__ void __launch_bounds__(kThreads, 2) dec_stage_group_kernel(const __grid_constant__ DecGroupArgs g) {
    const int b = static_cast<int>(blockIdx.x);
    int p = 0;
    while (p + 1 < g.G && b >= g.block0[p + 1]) ++p;
    dec_stage_body<CT, RBW, STAGE, false>(g.p[p], b - g.block0[p]);
}

// One-launch form of the two stages (the comparison arm of the two-launch
// path): CTAs [0, grid1) run stage 1 and write V, every CTA meets at a
// grid-wide barrier, then CTAs [0, grid2) run stage 2 from V.  The launch's
// cluster is the larger of the two stages' K splits and the other split is
// either the same or 1 (a stage with KS = 1 uses no cluster feature), so a
// cluster is wholly inside or wholly outside a stage's range; stage 2's
// shared memory starts at smem2 so that no mbarrier is re-initialised in
// place.  The launch is cooperative (every CTA resident), the barrier wait is
// bounded.
struct PairArgs {
    DecArgs a1, a2;
    int grid1, grid2;
    uint32_t smem2;
    unsigned int *bar;  // [0] arrival counter (a multiple of kPairQuantum between calls), [1] reserved, 0
};

// Each launch advances the arrival counter by exactly this much, whatever its grid (<= this).
constexpr unsigned int kPairQuantum = 1024;

// Grid-wide barrier over nblocks <= kPairQuantum CTAs with one atomic per CTA
// and no reset: CTA 0 adds kPairQuantum - (nblocks - 1), every other CTA 1,
// so the launch moves the counter from base to base + kPairQuantum and every
// CTA's pre-add value lies in [base, base + kPairQuantum).  Thread 0 of each
// CTA fences (the __syncthreads before makes the CTA's writes cumulative),
// adds, and polls the counter with acquire loads until it reaches the next
// multiple of kPairQuantum, for at most kWaitLimitNs.  Returns false in every
// thread of a CTA whose wait ran out (DBF_ERR_TIMEOUT recorded; the counter is
// then off its multiple and must be zeroed before the next call).
__device__ __noinline__ bool grid_barrier_bounded(unsigned int *bar, unsigned int nblocks, int *status) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const unsigned int inc = (blockIdx.x == 0) ? kPairQuantum - (nblocks - 1u) : 1u;
        __threadfence();
        const unsigned int old = atomicAdd(bar, inc);
        const unsigned int target = (old & ~(kPairQuantum - 1u)) + kPairQuantum;
        const uint64_t t0 = global_ns();
        for (;;) {
            unsigned int now;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(now) : "l"(bar) : "memory");
            if (static_cast<int>(now - target) >= 0) break;
            if (global_ns() - t0 > kWaitLimitNs) {
                record_status(status, DBF_ERR_TIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(100);  // spaces the polls of up to 1024 CTAs on one word
        }
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

// True in every CTA of the cluster when `ok` holds in all of them.  Stage 2
// pushes partials into the other CTAs of its cluster, so after a barrier wait
// that ran out somewhere, either the whole cluster runs stage 2 or none of it
// does: no CTA exits while a peer may still write into its shared memory.
// `bad` is this CTA's flag, cleared and published to the cluster (a cluster
// barrier) at the start of the kernel; a CTA whose wait ran out sets it in
// every CTA of the cluster, and one more cluster barrier makes the sets
// visible before each CTA reads its own.
__device__ __noinline__ bool cluster_all_ok(bool ok, uint32_t *bad) {
    if (cluster_nctarank() == 1) return ok;
    if (threadIdx.x == 0 && !ok) {
        const uint32_t n = cluster_nctarank();
        for (uint32_t r = 0; r < n; ++r)
            asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(mapa_shared(smem_u32(bad), r)), "r"(1u)
                         : "memory");
    }
    cluster_sync_all();
    return *reinterpret_cast<volatile uint32_t *>(bad) == 0u;
}

template <int CT, int RBW1, int RBW>
__global__ void __launch_bounds__(kThreads, 2) dec_stage_pair_kernel(const __grid_constant__ PairArgs p) {
    const int bx = static_cast<int>(blockIdx.x);
    __shared__ uint32_t bad;  // a CTA of the cluster gave up at the grid barrier
    if (threadIdx.x == 0) bad = 0u;
    if (cluster_nctarank() > 1)
        cluster_sync_all();  // every CTA's flag is clear before any peer may set it
    // this CTA's stage-2 signs and scales into its stage-2 shared memory while stage 1 runs
    // (factor memory: no earlier kernel writes it); stage 1's cp.async wait covers these too
    if (bx < p.grid2) dec_stage_body<CT, RBW, 2, false, 1>(p.a2, bx, p.smem2);
    if (bx < p.grid1) dec_stage_body<CT, RBW1, 1, false>(p.a1, bx, 0);
    // CTAs past grid1 have not waited yet: the previous kernel (possibly the previous call on this
    // barrier, still counting its arrivals) must be complete before any CTA arrives
    pdl_wait();
    const bool passed = grid_barrier_bounded(p.bar, gridDim.x, p.a1.status);
    if (!cluster_all_ok(passed, &bad)) {
        cp_async_wait_all();  // this CTA's own stage-2 copies land before it exits
        return;
    }
    if (bx < p.grid2) {
        cp_async_wait_all();  // CTAs that ran no stage 1
        dec_stage_body<CT, RBW, 2, false, 2>(p.a2, bx, p.smem2);
    }
}

// ================================================================ launchers

template <typename Kern, typename Args>
cudaError_t launch_ex(Kern kern, int &configured_smem, int grid_x, int grid_y, size_t smem, int cluster,
                      const Args &args, cudaStream_t stream, bool pdl) {
    if (smem > 48 * 1024 && static_cast<int>(smem) > configured_smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured_smem = static_cast<int>(smem);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, grid_y, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster;
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

template <int CT, int RBW, int STAGE, bool SEG>
cudaError_t launch_stage_one(const DecPlan &plan, const DecArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    static int configured = 0;
    return launch_ex(dec_stage_kernel<CT, RBW, STAGE, SEG>, configured, plan.grid_x, grid_y, plan.smem, plan.KS, args,
                     stream, pdl);
}

template <int CT, int STAGE, bool SEG>
cudaError_t launch_stage_rbw(const DecPlan &plan, const DecArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    switch (plan.RBW) {
        case 2: return launch_stage_one<CT, 2, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 4: return launch_stage_one<CT, 4, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

template <int STAGE, bool SEG>
cudaError_t launch_stage_ct(const DecPlan &plan, const DecArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    switch (plan.CT) {
        case 1: return launch_stage_rbw<1, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 2: return launch_stage_rbw<2, STAGE, SEG>(plan, args, grid_y, stream, pdl);
        case 4: return plan.RBW == 2 ? launch_stage_one<4, 2, STAGE, SEG>(plan, args, grid_y, stream, pdl)
                                     : cudaErrorInvalidValue;
        case 8: return plan.RBW == 2 ? launch_stage_one<8, 2, STAGE, SEG>(plan, args, grid_y, stream, pdl)
                                     : cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

template <int CT, int RBW, int STAGE>
cudaError_t launch_group_one(const DecPlan &plan, const DecGroupArgs &g, cudaStream_t stream, bool pdl) {
    static int configured = 0;
    return launch_ex(dec_stage_group_kernel<CT, RBW, STAGE>, configured, plan.grid_x, 1, plan.smem, plan.KS, g,
                     stream, pdl);
}

template <int STAGE>
cudaError_t launch_group_stage(const DecPlan &plan, const DecGroupArgs &g, cudaStream_t stream, bool pdl) {
    switch (plan.CT) {
        case 1: return plan.RBW == 2 ? launch_group_one<1, 2, STAGE>(plan, g, stream, pdl)
                                     : launch_group_one<1, 4, STAGE>(plan, g, stream, pdl);
        case 2: return plan.RBW == 2 ? launch_group_one<2, 2, STAGE>(plan, g, stream, pdl)
                                     : launch_group_one<2, 4, STAGE>(plan, g, stream, pdl);
        case 4: return plan.RBW == 2 ? launch_group_one<4, 2, STAGE>(plan, g, stream, pdl) : cudaErrorInvalidValue;
        case 8: return plan.RBW == 2 ? launch_group_one<8, 2, STAGE>(plan, g, stream, pdl) : cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

template <int CT, int RBW, bool SEG>
cudaError_t launch_fused_one(const FusedPlan &plan, const FusedArgs &args, int grid_y, cudaStream_t stream,
                             bool pdl) {
    static int configured = 0;
    return launch_ex(dec_fused_kernel<CT, RBW, SEG>, configured, plan.grid_x, grid_y, plan.smem, plan.C, args, stream,
                     pdl);
}

template <int CT, bool SEG>
cudaError_t launch_fused_rbw(const FusedPlan &plan, const FusedArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    switch (plan.RBW) {
        case 1: return launch_fused_one<CT, 1, SEG>(plan, args, grid_y, stream, pdl);
        case 2: return launch_fused_one<CT, 2, SEG>(plan, args, grid_y, stream, pdl);
        case 4: return launch_fused_one<CT, 4, SEG>(plan, args, grid_y, stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

template <bool SEG>
cudaError_t launch_fused_ct(const FusedPlan &plan, const FusedArgs &args, int grid_y, cudaStream_t stream, bool pdl) {
    switch (plan.CT) {
        case 1: return launch_fused_rbw<1, SEG>(plan, args, grid_y, stream, pdl);
        case 2: return launch_fused_rbw<2, SEG>(plan, args, grid_y, stream, pdl);
        case 4:
            if (plan.RBW == 1) return launch_fused_one<4, 1, SEG>(plan, args, grid_y, stream, pdl);
            if (plan.RBW == 2) return launch_fused_one<4, 2, SEG>(plan, args, grid_y, stream, pdl);
            return cudaErrorInvalidValue;
        case 8: return plan.RBW == 1 ? launch_fused_one<8, 1, SEG>(plan, args, grid_y, stream, pdl)
                                     : cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

int ct_for(int columns, int max_ct) {
    int ct = 1;
    while (ct * 8 < columns && ct < max_ct) ct *= 2;
    return ct;
}

constexpr size_t kSmemCap = 200 * 1024;

// CTAs per SM: shared memory, and the registers of __launch_bounds__(kThreads, 2)
int occupancy_for(size_t smem) {
    int occ = static_cast<int>(std::min<size_t>(size_t(228 * 1024) / (smem + 1024), 2));
    return occ < 1 ? 1 : occ;
}

}  // namespace

// Stage plan: 16*RBW rows per CTA, cluster split of K (KS), column tiles CT.
// Latency model (clocks) of the slowest SM: per wave a fixed cost (launch,
// the activation round trip, barriers) plus the words each warp streams;
// a cluster exchange costs a barrier and the pushes.
DecPlan plan_decode_stage(int rows_cover, int Kw, int columns, int max_ct, int num_sms, int ell, bool stage1) {
    DecPlan best = {};
    const int ct = ct_for(columns, max_ct);
    const int cpad = 8 * ct;
    double best_cost = 1e300;
    for (int RBW = 2; RBW <= 4; RBW *= 2) {
        if (ct >= 4 && RBW > 2) break;  // accumulators of RBW x CT fragments stay in registers
        for (int KS = 1; KS <= 8; KS *= 2) {
            if (KS > 1 && (KS > Kw || 16 * RBW / KS < 8)) break;
            const int Wc = (Kw + KS - 1) / KS;
            const size_t smem = stage_smem(cpad, RBW, KS, Wc, ell, stage1, true).total;
            if (smem > kSmemCap) continue;
            const int groups = (rows_cover + 16 * RBW - 1) / (16 * RBW);
            const int ctas = groups * KS;
            const int occ = occupancy_for(smem);
            const double waves = std::ceil(double(ctas) / (double(num_sms) * occ));
            const double per_sm = std::ceil(double(ctas) / num_sms);
            const int Wp = (Wc + kWarps - 1) / kWarps;
            const int nwb = ct >= 4 ? 1 : (ct >= 2 ? 2 : 4);
            const double batches = std::ceil(double(Wp) / nwb);
            const double warp_work = Wp * (60.0 * ct + 30.0 * RBW + 12.0 * RBW * ct);
            const double epi = double(16 * RBW / KS) * cpad * 8.0 / kThreads * 20.0;
            const double cost = waves * 1500.0 + per_sm * (warp_work + epi) + (batches - 1.0) * 700.0 +
                                (KS > 1 ? 900.0 : 0.0);
            if (cost < best_cost) {
                best_cost = cost;
                best.CT = ct;
                best.RBW = RBW;
                best.KS = KS;
                best.Wc = Wc;
                best.grid_x = ctas;
                best.smem = smem;
            }
        }
    }
    return best;
}

// Fused plan: cluster size C (stage-1 split of M), stage-2 rows per CTA RW.
// Same latency model: waves, the stage-1 words per warp, the stage-2 items
// per warp, the cluster exchange.
FusedPlan plan_fused(int N, int M, int R, int ell, int columns, int num_sms, int problems, bool accumulate) {
    FusedPlan best = {};
    if (R > kFusedMaxR) return best;
    const int ct = ct_for(columns, 8);
    const int cpad = 8 * ct;
    const int RB1 = (R + 15) / 16;
    int RBW = RB1 >= 4 ? 4 : (RB1 >= 2 ? 2 : 1);
    if (ct >= 4 && RBW > 2) RBW = 2;  // accumulators of RBW x CT fragments stay in registers
    if (ct >= 8) RBW = 1;
    const int G1 = fused_g1(R, RBW), KP = fused_kp(G1);
    const int R2 = (R + 31) & ~31, Kw1 = (M + 31) / 32, Kw2 = R2 / 32;
    if (problems < 1) problems = 1;
    double best_cost = 1e300;
    for (int C = 1; C <= 8; C *= 2) {
        if (C > 1 && C > Kw1) break;
        const int Wc = (Kw1 + C - 1) / C;
        const int Wp = (Wc + KP - 1) / KP;
        for (int RW = 16; RW <= 1024; RW *= 2) {
            const int used = (N + RW - 1) / RW;          // CTAs that own output rows
            const int grid = ((used + C - 1) / C) * C;   // whole clusters
            const size_t smem = fused_smem(cpad, RBW, Wc, R, RW, ell, C, accumulate).total;
            if (smem > kSmemCap) continue;
            const int occ = occupancy_for(smem);
            const double waves = std::ceil(double(problems) * grid / (double(num_sms) * occ));
            const double per_sm = std::ceil(double(problems) * grid / num_sms);
            const int nwb = ct >= 4 ? 1 : (ct >= 2 ? 2 : 4);
            const double s1 = Wp * (60.0 * ct + 30.0 * RBW + 12.0 * RBW * ct) + std::ceil(double(Wp) / nwb - 1.0) * 700.0;
            const double s2 = std::ceil(double(RW / 16) * ct / kWarps) * Kw2 * 40.0;
            const double red = double(16 * RBW * G1) * cpad / kThreads * (KP + 2.0 * C) * 8.0;
            // measured on B300: every CTA costs about 400 clocks of launch and
            // prologue on its SM, so fewer, fatter CTAs win until stage 2 dominates
            const double cost = waves * (1500.0 + (C > 1 ? 900.0 : 0.0)) + per_sm * (s1 + s2 + red) +
                                400.0 * double(problems) * grid / num_sms;
            if (cost < best_cost) {
                best_cost = cost;
                best.CT = ct;
                best.RBW = RBW;
                best.C = C;
                best.RW = RW;
                best.Wc = Wc;
                best.grid_x = grid;
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

// Both decode stages of one call (or of a routed batch when seg_off is set):
// stage 1 writes V = beta * (B2 (gamma * x)) to `V` (fp16, [ell*T][ldv]),
// stage 2 reads it.
// The plans and arguments of the two stages of one decode call.
static cudaError_t plan_two_stage(const DecodeCall &c, __half *V, int ldv, int num_sms, DecPlan &p1, DecArgs &a1,
                                  DecPlan &p2, DecArgs &a2) {
    const int ell = c.ell;
    const int64_t cols = std::min<int64_t>(int64_t(ell) * c.tokens_per_problem, 64);
    const int problems = std::max(1, c.S);
    const int sms_per_problem = std::max(1, num_sms / problems);
    DecArgs a = {};
    a.ell = ell;
    a.T = c.T;
    a.x = c.x;
    a.ldx = c.M;
    a.V = V;
    a.ldv = ldv;
    a.y = c.y;
    a.ldy = c.N;
    a.accumulate = c.accumulate;
    a.seg_off = c.seg_off;
    a.seg_ad = c.seg_ad;
    a.adapters = c.adapters;
    a.n_adapters = c.n_adapters;
    a.status = c.status;
    const bool seg = c.seg_off != nullptr;

    a1 = a;
    if (!seg) {
        a1.bits = c.f->B2;
        a1.ldw = c.f->ldw2;
        a1.gamma = reinterpret_cast<const __half *>(c.f->gamma);
        a1.beta = reinterpret_cast<const __half *>(c.f->beta);
    }
    a1.rows = c.R;
    a1.rows_out = (c.R + 31) & ~31;
    a1.K = c.M;
    a1.Kw = (c.M + 31) / 32;
    p1 = plan_decode_stage(a1.rows_out, a1.Kw, static_cast<int>(cols), 8, sms_per_problem, ell, true);
    a1.KS = p1.KS;
    a1.Wc = p1.Wc;

    a2 = a;
    if (!seg) {
        a2.bits = c.f->B1;
        a2.ldw = c.f->ldw1;
        a2.alpha = reinterpret_cast<const __half *>(c.f->alpha);
    }
    a2.rows = c.N;
    a2.rows_out = c.N;
    a2.K = c.R;
    a2.Kw = (c.R + 31) / 32;
    p2 = plan_decode_stage(c.N, a2.Kw, static_cast<int>(cols), p1.CT, sms_per_problem, ell, false);
    p2.CT = p1.CT;  // both stages use the same column chunking
    if (p2.smem == 0 || p1.smem == 0) return cudaErrorNotSupported;
    if (p2.CT >= 8 && p2.RBW > 2) return cudaErrorNotSupported;
    p2.smem = stage_smem(8 * p2.CT, p2.RBW, p2.KS, p2.Wc, ell, false, c.accumulate != 0).total;
    a2.KS = p2.KS;
    a2.Wc = p2.Wc;
    return cudaSuccess;
}

cudaError_t launch_decode_two_stage(const DecodeCall &c, __half *V, int ldv, int num_sms, cudaStream_t stream) {
    DecPlan p1, p2;
    DecArgs a1, a2;
    cudaError_t e = plan_two_stage(c, V, ldv, num_sms, p1, a1, p2, a2);
    if (e != cudaSuccess) return e;
    const bool seg = c.seg_off != nullptr;
    const int problems = std::max(1, c.S);
    e = launch_decode_stage(1, seg, p1, a1, problems, stream, true);
    if (e != cudaSuccess) return e;
    return launch_decode_stage(2, seg, p2, a2, problems, stream, true);
}

template <int CT, int RBW1, int RBW2>
static cudaError_t launch_pair_one(const PairArgs &pa, int grid, int cluster, size_t smem, cudaStream_t stream) {
    static int configured = 0;
    auto kern = dec_stage_pair_kernel<CT, RBW1, RBW2>;
    if (smem > 48 * 1024 && static_cast<int>(smem) > configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = static_cast<int>(smem);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    int na = 0;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    // every CTA must be resident at once: check before launching, then ask for a cooperative launch
    int active = 0;
    if (cluster > 1) {
        cudaError_t e = cudaOccupancyMaxActiveClusters(&active, kern, &cfg);
        if (e != cudaSuccess) return e;
        active *= cluster;
    } else {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&active, kern, kThreads, smem);
        if (e != cudaSuccess) return e;
        active *= sms;
    }
    if (active < grid) return cudaErrorCooperativeLaunchTooLarge;
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, pa);
}

cudaError_t launch_decode_one_launch(const DecodeCall &c, __half *V, int ldv, unsigned int *bar, int num_sms,
                                     cudaStream_t stream) {
    if (c.seg_off != nullptr || bar == nullptr) return cudaErrorInvalidValue;
    DecPlan p1, p2;
    PairArgs pa = {};
    cudaError_t e = plan_two_stage(c, V, ldv, num_sms, p1, pa.a1, p2, pa.a2);
    if (e != cudaSuccess) return e;
    const int cluster = std::max(p1.KS, p2.KS);
    if (std::min(p1.KS, p2.KS) != 1 && p1.KS != p2.KS) return cudaErrorNotSupported;
    pa.grid1 = p1.grid_x;
    pa.grid2 = p2.grid_x;
    pa.smem2 = static_cast<uint32_t>((p1.smem + 127) & ~size_t(127));
    pa.bar = bar;
    const int grid = (std::max(pa.grid1, pa.grid2) + cluster - 1) / cluster * cluster;
    const size_t smem = pa.smem2 + p2.smem;
    if (smem > size_t(227) * 1024 || grid > static_cast<int>(kPairQuantum)) return cudaErrorNotSupported;
    switch (p1.CT * 100 + p1.RBW * 10 + p2.RBW) {
        case 122: return launch_pair_one<1, 2, 2>(pa, grid, cluster, smem, stream);
        case 124: return launch_pair_one<1, 2, 4>(pa, grid, cluster, smem, stream);
        case 142: return launch_pair_one<1, 4, 2>(pa, grid, cluster, smem, stream);
        case 144: return launch_pair_one<1, 4, 4>(pa, grid, cluster, smem, stream);
        case 222: return launch_pair_one<2, 2, 2>(pa, grid, cluster, smem, stream);
        case 224: return launch_pair_one<2, 2, 4>(pa, grid, cluster, smem, stream);
        case 242: return launch_pair_one<2, 4, 2>(pa, grid, cluster, smem, stream);
        case 244: return launch_pair_one<2, 4, 4>(pa, grid, cluster, smem, stream);
        case 422: return launch_pair_one<4, 2, 2>(pa, grid, cluster, smem, stream);
        case 822: return launch_pair_one<8, 2, 2>(pa, grid, cluster, smem, stream);
        default: return cudaErrorNotSupported;
    }
}

// Plan of a grouped stage: one CT, RBW and KS for every problem of the launch
// (the cluster size is a launch property), each problem with its own K slice
// width; the same latency model as a single problem, with the work of all
// problems spread over the SMs and the slowest CTA as a floor.
DecPlan plan_group_stage(const int *rows_cover, const int *Kw, int G, int columns, int max_ct, int num_sms, int ell,
                         bool stage1, bool accumulate) {
    DecPlan best = {};
    const int ct = ct_for(columns, max_ct);
    const int cpad = 8 * ct;
    int min_kw = Kw[0];
    for (int p = 1; p < G; ++p) min_kw = std::min(min_kw, Kw[p]);
    double best_cost = 1e300;
    for (int RBW = 2; RBW <= 4; RBW *= 2) {
        if (ct >= 4 && RBW > 2) break;
        for (int KS = 1; KS <= 8; KS *= 2) {
            if (KS > 1 && (KS > min_kw || 16 * RBW / KS < 8)) break;
            size_t smem = 0;
            int64_t ctas = 0;
            double work = 0.0, max_work = 0.0;
            const int nwb = ct >= 4 ? 1 : (ct >= 2 ? 2 : 4);
            const double epi = double(16 * RBW / KS) * cpad * 8.0 / kThreads * 20.0;
            for (int p = 0; p < G; ++p) {
                const int Wc = (Kw[p] + KS - 1) / KS;
                smem = std::max(smem, stage_smem(cpad, RBW, KS, Wc, ell, stage1, accumulate).total);
                const int groups = (rows_cover[p] + 16 * RBW - 1) / (16 * RBW);
                const int Wp = (Wc + kWarps - 1) / kWarps;
                const double w = Wp * (60.0 * ct + 30.0 * RBW + 12.0 * RBW * ct) +
                                 (std::ceil(double(Wp) / nwb) - 1.0) * 700.0 + epi;
                ctas += int64_t(groups) * KS;
                work += double(groups) * KS * w;
                max_work = std::max(max_work, w);
            }
            if (smem > kSmemCap || ctas > (int64_t(1) << 30)) continue;
            const int occ = occupancy_for(smem);
            const double waves = std::ceil(double(ctas) / (double(num_sms) * occ));
            const double cost = waves * 1500.0 + std::max(work / num_sms, max_work) + (KS > 1 ? 900.0 : 0.0);
            if (cost < best_cost) {
                best_cost = cost;
                best.CT = ct;
                best.RBW = RBW;
                best.KS = KS;
                best.Wc = 0;  // per problem
                best.grid_x = static_cast<int>(ctas);
                best.smem = smem;
            }
        }
    }
    return best;
}

// Both decode stages of a group of independent problems, one launch per stage.
cudaError_t launch_decode_grouped(const DecodeGroupCall &c, int num_sms, cudaStream_t stream) {
    const int G = c.G, ell = c.ell;
    if (G < 1 || G > kMaxGroup) return cudaErrorInvalidValue;
    const int cols = static_cast<int>(std::min<int64_t>(int64_t(ell) * c.T, 64));
    int rows1[kMaxGroup], kw1[kMaxGroup], rows2[kMaxGroup], kw2[kMaxGroup];
    for (int p = 0; p < G; ++p) {
        const dbf_factors *f = c.f[p];
        rows1[p] = (f->R + 31) & ~31;
        kw1[p] = (f->M + 31) / 32;
        rows2[p] = f->N;
        kw2[p] = (f->R + 31) / 32;
    }
    const DecPlan p1 = plan_group_stage(rows1, kw1, G, cols, 8, num_sms, ell, true, true);
    if (p1.smem == 0) return cudaErrorNotSupported;
    DecPlan p2 = plan_group_stage(rows2, kw2, G, cols, p1.CT, num_sms, ell, false, c.accumulate != 0);
    if (p2.smem == 0 || p2.CT != p1.CT) return cudaErrorNotSupported;

    DecGroupArgs g1 = {}, g2 = {};
    g1.G = g2.G = G;
    int b1 = 0, b2 = 0;
    for (int p = 0; p < G; ++p) {
        const dbf_factors *f = c.f[p];
        DecArgs a = {};
        a.ell = ell;
        a.T = c.T;
        a.x = c.x[p];
        a.ldx = f->M;
        a.V = c.V[p];
        a.ldv = c.ldv[p];
        a.y = c.y[p];
        a.ldy = f->N;
        a.accumulate = c.accumulate;
        a.status = c.status;

        DecArgs a1 = a;
        a1.bits = f->B2;
        a1.ldw = f->ldw2;
        a1.gamma = reinterpret_cast<const __half *>(f->gamma);
        a1.beta = reinterpret_cast<const __half *>(f->beta);
        a1.rows = f->R;
        a1.rows_out = rows1[p];
        a1.K = f->M;
        a1.Kw = kw1[p];
        a1.KS = p1.KS;
        a1.Wc = (kw1[p] + p1.KS - 1) / p1.KS;
        g1.p[p] = a1;
        g1.block0[p] = b1;
        b1 += ((rows1[p] + 16 * p1.RBW - 1) / (16 * p1.RBW)) * p1.KS;

        DecArgs a2 = a;
        a2.bits = f->B1;
        a2.ldw = f->ldw1;
        a2.alpha = reinterpret_cast<const __half *>(f->alpha);
        a2.rows = f->N;
        a2.rows_out = f->N;
        a2.K = f->R;
        a2.Kw = kw2[p];
        a2.KS = p2.KS;
        a2.Wc = (kw2[p] + p2.KS - 1) / p2.KS;
        g2.p[p] = a2;
        g2.block0[p] = b2;
        b2 += ((rows2[p] + 16 * p2.RBW - 1) / (16 * p2.RBW)) * p2.KS;
    }
    g1.block0[G] = b1;
    g2.block0[G] = b2;
    if (b1 != p1.grid_x || b2 != p2.grid_x) return cudaErrorInvalidValue;
    cudaError_t e = launch_group_stage<1>(p1, g1, stream, true);
    if (e != cudaSuccess) return e;
    return launch_group_stage<2>(p2, g2, stream, true);
}

}  // namespace dbfk
