// C ABI of the packed double-binary matmul library: argument checks,
// workspace sizing, kernel-path choice and launches.  No call allocates
// device memory; all scratch lives in the caller's workspace.
#include <stdio.h>
#include <string.h>

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "factorize.h"

namespace {

// Device status word, one per device the library runs on.
__device__ int g_dbf_status;

constexpr int kMaxDevices = 64;
constexpr int kDecodeMaxTokens = 16;
constexpr size_t kAlign = 256;

thread_local char g_last_error[256] = "";

int cuda_fail(cudaError_t e, const char *where) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
    cudaGetLastError();  // a failed call leaves no error behind for the next launch check to pick up
    return DBF_ERR_CUDA;
}

int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

int *status_ptr() {
    static int *ptrs[kMaxDevices] = {nullptr};
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dbf_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int *>(p);
    }
    return ptrs[dev];
}

int num_sms() {
    static int sms[kMaxDevices] = {0};
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 148;
    if (!sms[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        sms[dev] = v > 0 ? v : 148;
    }
    return sms[dev];
}

// Streams and events of the pipelined host-io call, created once per device.
constexpr int kPipeSlots = 4;
struct HostioPipe {
    cudaStream_t in = nullptr, cmp = nullptr, out = nullptr;
    cudaEvent_t fork = nullptr, join[3] = {nullptr, nullptr, nullptr};
    cudaEvent_t h2d[kPipeSlots] = {}, done[kPipeSlots] = {}, d2h[kPipeSlots] = {};
};
std::mutex g_pipe_mu;

HostioPipe *hostio_pipe(cudaError_t *err) {
    static HostioPipe pipes[kMaxDevices];
    static bool ready[kMaxDevices] = {false};
    const int dev = current_device();
    *err = cudaSuccess;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    HostioPipe &p = pipes[dev];
    if (!ready[dev]) {
        cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.cmp, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
        cudaEvent_t *all[] = {&p.fork, &p.join[0], &p.join[1], &p.join[2]};
        for (cudaEvent_t *ev : all)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        for (int k = 0; k < kPipeSlots && e == cudaSuccess; ++k) {
            e = cudaEventCreateWithFlags(&p.h2d[k], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.done[k], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.d2h[k], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) {
            *err = e;
            return nullptr;
        }
        ready[dev] = true;
    }
    return &p;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

// V row length in halves: round_up(R, 64) keeps every row 128-byte aligned
// and covers the K extent of both paths.
inline int64_t v_ld(int64_t R) { return round_up(R, 64); }
inline int64_t xs_ld(int64_t M) { return round_up(M, 64); }

int check_dims(int64_t N, int64_t M, int64_t R, int64_t ell) {
    if (N < 1 || M < 1 || R < 1) return DBF_ERR_INVALID_ARG;
    if (ell < 1 || ell > 4) return DBF_ERR_INVALID_ARG;
    if (N > (1 << 24) || M > (1 << 24) || R > (1 << 20)) return DBF_ERR_UNSUPPORTED;
    return DBF_OK;
}

int check_factors(const dbf_factors *f) {
    if (!f) return DBF_ERR_INVALID_ARG;
    int rc = check_dims(f->N, f->M, f->R, f->ell);
    if (rc) return rc;
    if (!f->B1 || !f->B2 || !f->alpha || !f->beta || !f->gamma) return DBF_ERR_INVALID_ARG;
    if (f->ldw1 < ceil_div(f->R, 32) || f->ldw2 < ceil_div(f->M, 32)) return DBF_ERR_INVALID_ARG;
    if (!aligned16(f->B1) || !aligned16(f->B2) || !aligned16(f->alpha) || !aligned16(f->beta) ||
        !aligned16(f->gamma))
        return DBF_ERR_ALIGNMENT;
    return DBF_OK;
}

int resolve_path(int path, int64_t T) {
    if (path == DBF_PATH_AUTO) return T <= kDecodeMaxTokens ? DBF_PATH_DECODE : DBF_PATH_PREFILL;
    return path;
}

size_t ws_decode(int64_t N, int64_t M, int64_t R, int64_t ell, int64_t T) {
    (void)N;
    (void)M;
    return align_up(size_t(ell * T) * v_ld(R) * 2);
}

size_t ws_prefill(int64_t N, int64_t M, int64_t R, int64_t ell, int64_t T) {
    (void)N;
    return align_up(size_t(ell * T) * xs_ld(M) * 2) + align_up(size_t(ell * T) * v_ld(R) * 2);
}

size_t ws_for(const dbf_factors *f, int64_t T, int path) {
    path = resolve_path(path, T);
    if (path == DBF_PATH_DECODE) return ws_decode(f->N, f->M, f->R, f->ell, T);
    return ws_prefill(f->N, f->M, f->R, f->ell, T);
}

dbfk::FusedArgs fused_args(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y, int accumulate,
                           const dbfk::FusedPlan &p) {
    dbfk::FusedArgs a = {};
    a.B1 = f->B1;
    a.B2 = f->B2;
    a.ldw1 = f->ldw1;
    a.ldw2 = f->ldw2;
    a.alpha = reinterpret_cast<const __half *>(f->alpha);
    a.beta = reinterpret_cast<const __half *>(f->beta);
    a.gamma = reinterpret_cast<const __half *>(f->gamma);
    a.N = f->N;
    a.M = f->M;
    a.R = f->R;
    a.ell = f->ell;
    a.T = static_cast<int>(T);
    a.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    a.y = reinterpret_cast<__nv_bfloat16 *>(y);
    a.accumulate = accumulate;
    a.C = p.C;
    a.RW = p.RW;
    a.Wc = p.Wc;
    a.status = status_ptr();
    return a;
}

// Columns (token x term) one decode launch covers per chunk.
int64_t decode_columns(int64_t ell, int64_t tokens) { return std::min<int64_t>(ell * tokens, 64); }

// Tokens one segment's share of a routed batch is planned for: about twice
// the mean segment length.
int64_t segment_tokens(int64_t T, int64_t S) {
    const int64_t mean_tok = ceil_div(T, std::max<int64_t>(S, 1));
    return std::min<int64_t>(T, std::max<int64_t>(2 * mean_tok, 4));
}

dbfk::FusedPlan fused_plan_for(int N, int M, int R, int ell, int64_t tokens, int problems, bool accumulate) {
    if (R > dbfk::kFusedMaxR) return dbfk::FusedPlan{};
    return dbfk::plan_fused(N, M, R, ell, static_cast<int>(decode_columns(ell, tokens)), num_sms(), problems,
                            accumulate);
}

dbfk::RsPlan rs_plan_for(int N, int M, int R, int ell, int64_t tokens, int problems, bool accumulate) {
    return dbfk::plan_rs(N, M, R, ell, static_cast<int>(decode_columns(ell, tokens)), num_sms(), problems,
                         accumulate);
}

dbfk::RsArgs rs_args(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y, int accumulate,
                     const dbfk::RsPlan &p) {
    dbfk::RsArgs a = {};
    a.B1 = f->B1;
    a.B2 = f->B2;
    a.ldw1 = f->ldw1;
    a.ldw2 = f->ldw2;
    a.alpha = reinterpret_cast<const __half *>(f->alpha);
    a.beta = reinterpret_cast<const __half *>(f->beta);
    a.gamma = reinterpret_cast<const __half *>(f->gamma);
    a.N = f->N;
    a.M = f->M;
    a.R = f->R;
    a.ell = f->ell;
    a.T = static_cast<int>(T);
    a.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    a.y = reinterpret_cast<__nv_bfloat16 *>(y);
    a.accumulate = accumulate;
    a.C = p.C;
    a.Wc = p.Wc;
    a.RW = p.RW;
    a.IPW = p.IPW;
    a.status = status_ptr();
    return a;
}

int map_launch_error(cudaError_t e, const char *where) {
    if (e == cudaErrorNotSupported) {
        snprintf(g_last_error, sizeof(g_last_error), "%s: no decode tile plan fits this shape", where);
        return DBF_ERR_UNSUPPORTED;
    }
    return cuda_fail(e, where);
}

// decode path: one launch when R is small (the reduce-scatter kernel, else the
// all-to-all fused kernel), else the two stages (x -> V, V -> y) through the
// workspace
int run_decode(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y, int accumulate, void *ws,
               cudaStream_t stream) {
    using namespace dbfk;
    const RsPlan rp = rs_plan_for(f->N, f->M, f->R, f->ell, T, 1, accumulate != 0);
    if (rp.CT != 0) {
        cudaError_t e = launch_decode_rs(false, rp, rs_args(f, x, T, y, accumulate, rp), 1, stream);
        return e == cudaSuccess ? DBF_OK : cuda_fail(e, "decode");
    }
    const FusedPlan fp = fused_plan_for(f->N, f->M, f->R, f->ell, T, 1, accumulate != 0);
    if (fp.CT != 0) {
        cudaError_t e = launch_decode_fused(false, fp, fused_args(f, x, T, y, accumulate, fp), 1, stream, true);
        return e == cudaSuccess ? DBF_OK : cuda_fail(e, "fused decode");
    }
    DecodeCall c = {};
    c.f = f;
    c.N = f->N;
    c.M = f->M;
    c.R = f->R;
    c.ell = f->ell;
    c.T = static_cast<int>(T);
    c.tokens_per_problem = static_cast<int>(T);
    c.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    c.y = reinterpret_cast<__nv_bfloat16 *>(y);
    c.accumulate = accumulate;
    c.status = status_ptr();
    cudaError_t e = launch_decode_two_stage(c, static_cast<__half *>(ws), static_cast<int>(v_ld(f->R)), num_sms(),
                                            stream);
    return e == cudaSuccess ? DBF_OK : map_launch_error(e, "decode");
}

int run_prefill(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y, int accumulate, void *ws,
                cudaStream_t stream) {
    using namespace dbfk;
    const int ell = f->ell;
    const int64_t C = ell * T;
    const int ldxs = static_cast<int>(xs_ld(f->M));
    const int ldv = static_cast<int>(v_ld(f->R));
    __half *xs = static_cast<__half *>(ws);
    __half *V = reinterpret_cast<__half *>(static_cast<char *>(ws) + align_up(size_t(C) * ldxs * 2));
    // tile widths per GEMM; activation tiles are the second grid dimension (at most 65535 of them)
    const int bn1 = prefill_pick_bn(ell, ldv, C, static_cast<int>(ceil_div(f->M, 64)), num_sms());
    const int bn2 = prefill_pick_bn(ell, f->N, C, static_cast<int>(ceil_div(f->R, 64)), num_sms());
    if (bn1 == 0 || bn2 == 0) return DBF_ERR_UNSUPPORTED;

    cudaError_t e = launch_prefill_prologue(reinterpret_cast<const __nv_bfloat16 *>(x), static_cast<int>(T), f->M,
                                            f->M, reinterpret_cast<const __half *>(f->gamma), ell, xs, ldxs, stream,
                                            true);
    if (e != cudaSuccess) return cuda_fail(e, "prefill prologue");

    CUtensorMap map1, map2;
    if (!encode_act_map(&map1, xs, static_cast<int>(C), ldxs, ldxs, bn1) ||
        !encode_act_map(&map2, V, static_cast<int>(C), ldv, ldv, bn2)) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed");
        return DBF_ERR_CUDA;
    }
    PfArgs a = {};
    a.ell = ell;
    a.C = static_cast<int>(C);
    a.V = V;
    a.ldv = ldv;
    a.beta = reinterpret_cast<const __half *>(f->beta);
    a.alpha = reinterpret_cast<const __half *>(f->alpha);
    a.y = reinterpret_cast<__nv_bfloat16 *>(y);
    a.ldy = f->N;
    a.accumulate = accumulate;
    a.status = status_ptr();

    PfArgs a1 = a;
    a1.bits = f->B2;
    a1.ldw = f->ldw2;
    a1.rows = f->R;
    a1.rows_store = ldv;
    a1.Kw = static_cast<int>(ceil_div(f->M, 32));
    a1.nk = static_cast<int>(ceil_div(f->M, 64));
    e = launch_prefill_gemm(1, map1, a1, bn1, stream, true);
    if (e != cudaSuccess) return cuda_fail(e, "prefill gemm 1");

    PfArgs a2 = a;
    a2.bits = f->B1;
    a2.ldw = f->ldw1;
    a2.rows = f->N;
    a2.rows_store = f->N;
    a2.Kw = static_cast<int>(ceil_div(f->R, 32));
    a2.nk = static_cast<int>(ceil_div(f->R, 64));
    e = launch_prefill_gemm(2, map2, a2, bn2, stream, true);
    if (e != cudaSuccess) return cuda_fail(e, "prefill gemm 2");
    return DBF_OK;
}

// workspace of the backward call: X' (max(M, N) columns), V (reused as V'), H
size_t ws_backward(int64_t N, int64_t M, int64_t R, int64_t ell, int64_t T) {
    const int64_t C = ell * T;
    return align_up(size_t(C) * xs_ld(std::max(M, N)) * 2) + 2 * align_up(size_t(C) * v_ld(R) * 2);
}

// Backward of y = sum_i alpha_i . B1 (beta_i . B2 (gamma_i . x)) for the output
// gradient dy, on the prefill GEMMs (six launches):
//   prologue   X'  = fp16(gamma_i . x)
//   gemm<1>    V   = fp16(beta_i . B2 X'),  H = fp16(B2 X')
//   gemm<2>    dalpha_i[n] = sum_t dy[t][n] (B1 V)[t, i][n]          (no y)
//   prologue   DY' = fp16(alpha_i . dy)
//   gemm<1>    V'  = fp16(beta_i . B1^T DY'),  dbeta_i[r] = sum_t (B1^T DY')[t, i][r] H[t, i][r]
//   gemm<2>    dx  = bf16(sum_i gamma_i . B2^T V'),  dgamma_i[k] = sum_t x[t][k] (B2^T V')[t, i][k]
int run_backward(const dbf_factors *f, const dbf_factors *ft, const uint16_t *x, const uint16_t *dy, int64_t T,
                 uint16_t *dx, float *dalpha, float *dbeta, float *dgamma, void *ws, cudaStream_t stream) {
    using namespace dbfk;
    const int ell = f->ell;
    const int64_t C = ell * T;
    const int N = f->N, M = f->M, R = f->R;
    const int ldv = static_cast<int>(v_ld(R));
    const int ldm = static_cast<int>(xs_ld(M)), ldn = static_cast<int>(xs_ld(N));
    char *base = static_cast<char *>(ws);
    __half *xs = reinterpret_cast<__half *>(base);
    __half *V = reinterpret_cast<__half *>(base + align_up(size_t(C) * xs_ld(std::max(M, N)) * 2));
    __half *H = reinterpret_cast<__half *>(reinterpret_cast<char *>(V) + align_up(size_t(C) * ldv * 2));
    // tile widths of the four GEMMs: rows R, N, R and M
    const int nkM = static_cast<int>(ceil_div(M, 64)), nkN = static_cast<int>(ceil_div(N, 64));
    const int nkR = static_cast<int>(ceil_div(R, 64));
    const int bn1 = prefill_pick_bn(ell, ldv, C, nkM, num_sms()), bn2 = prefill_pick_bn(ell, N, C, nkR, num_sms());
    const int bn3 = prefill_pick_bn(ell, ldv, C, nkN, num_sms()), bn4 = prefill_pick_bn(ell, M, C, nkR, num_sms());
    if (bn1 == 0 || bn2 == 0 || bn3 == 0 || bn4 == 0) return DBF_ERR_UNSUPPORTED;
    const auto *xb = reinterpret_cast<const __nv_bfloat16 *>(x);
    const auto *dyb = reinterpret_cast<const __nv_bfloat16 *>(dy);
    const auto *alpha = reinterpret_cast<const __half *>(f->alpha);
    const auto *beta = reinterpret_cast<const __half *>(f->beta);
    const auto *gamma = reinterpret_cast<const __half *>(f->gamma);

    cudaError_t e = cudaMemsetAsync(dalpha, 0, sizeof(float) * size_t(ell) * N, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, sizeof(float) * size_t(ell) * R, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dgamma, 0, sizeof(float) * size_t(ell) * M, stream);
    if (e != cudaSuccess) return cuda_fail(e, "backward: zero the scale gradients");

    PfArgs a = {};
    a.ell = ell;
    a.C = static_cast<int>(C);
    a.V = V;
    a.ldv = ldv;
    a.status = status_ptr();

    // ---- forward recompute: X', V and H, then dalpha
    // no programmatic overlap with the memsets above
    e = launch_prefill_prologue(xb, static_cast<int>(T), M, M, gamma, ell, xs, ldm, stream, false);
    if (e != cudaSuccess) return cuda_fail(e, "backward prologue x");
    CUtensorMap map;
    if (!encode_act_map(&map, xs, static_cast<int>(C), ldm, ldm, bn1)) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed");
        return DBF_ERR_CUDA;
    }
    PfArgs s1 = a;
    s1.bits = f->B2;
    s1.ldw = f->ldw2;
    s1.rows = R;
    s1.rows_store = ldv;
    s1.Kw = static_cast<int>(ceil_div(M, 32));
    s1.nk = static_cast<int>(ceil_div(M, 64));
    s1.beta = beta;
    s1.h_out = H;
    e = launch_prefill_gemm(1, map, s1, bn1, stream, true);
    if (e != cudaSuccess) return cuda_fail(e, "backward gemm: x -> V, H");

    if (!encode_act_map(&map, V, static_cast<int>(C), ldv, ldv, bn2)) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed");
        return DBF_ERR_CUDA;
    }
    PfArgs s2 = a;
    s2.bits = f->B1;
    s2.ldw = f->ldw1;
    s2.rows = N;
    s2.rows_store = N;
    s2.Kw = static_cast<int>(ceil_div(R, 32));
    s2.nk = static_cast<int>(ceil_div(R, 64));
    s2.alpha = alpha;
    s2.ldy = N;
    s2.skip_store = 1;
    s2.red_src = dyb;
    s2.ld_src = N;
    s2.red = dalpha;
    e = launch_prefill_gemm(2, map, s2, bn2, stream, true);
    if (e != cudaSuccess) return cuda_fail(e, "backward gemm: dalpha");

    // ---- through the transposed factors: V' and dbeta, then dx and dgamma
    e = launch_prefill_prologue(dyb, static_cast<int>(T), N, N, alpha, ell, xs, ldn, stream, true);
    if (e != cudaSuccess) return cuda_fail(e, "backward prologue dy");
    if (!encode_act_map(&map, xs, static_cast<int>(C), ldn, ldn, bn3)) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed");
        return DBF_ERR_CUDA;
    }
    PfArgs t1 = a;
    t1.bits = ft->B2;  // B1^T [R x N]
    t1.ldw = ft->ldw2;
    t1.rows = R;
    t1.rows_store = ldv;
    t1.Kw = static_cast<int>(ceil_div(N, 32));
    t1.nk = static_cast<int>(ceil_div(N, 64));
    t1.beta = beta;
    t1.h_in = H;
    t1.red = dbeta;
    e = launch_prefill_gemm(1, map, t1, bn3, stream, true);
    if (e != cudaSuccess) return cuda_fail(e, "backward gemm: dbeta");

    if (!encode_act_map(&map, V, static_cast<int>(C), ldv, ldv, bn4)) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed");
        return DBF_ERR_CUDA;
    }
    PfArgs t2 = a;
    t2.bits = ft->B1;  // B2^T [M x R]
    t2.ldw = ft->ldw1;
    t2.rows = M;
    t2.rows_store = M;
    t2.Kw = static_cast<int>(ceil_div(R, 32));
    t2.nk = static_cast<int>(ceil_div(R, 64));
    t2.alpha = gamma;
    t2.y = reinterpret_cast<__nv_bfloat16 *>(dx);
    t2.ldy = M;
    t2.skip_store = dx ? 0 : 1;
    t2.red_src = xb;
    t2.ld_src = M;
    t2.red = dgamma;
    e = launch_prefill_gemm(2, map, t2, bn4, stream, true);
    if (e != cudaSuccess) return cuda_fail(e, "backward gemm: dx, dgamma");
    return DBF_OK;
}

}  // namespace

namespace dbfk {
void set_last_error(const char *msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

int check_matmul_args(const dbf_factors *f, const uint16_t *x, int64_t T, const uint16_t *y, int accumulate,
                      int path) {
    const int rc = check_factors(f);
    if (rc) return rc;
    if (T < 0 || (accumulate != 0 && accumulate != 1)) return DBF_ERR_INVALID_ARG;
    if (path < DBF_PATH_AUTO || path > DBF_PATH_PREFILL) return DBF_ERR_INVALID_ARG;
    if (T == 0) return DBF_OK;
    if (T > (int64_t(1) << 26)) return DBF_ERR_UNSUPPORTED;
    if (!x || !y) return DBF_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return DBF_ERR_ALIGNMENT;
    return DBF_OK;
}
}  // namespace dbfk

extern "C" {

const char *dbf_status_string(int code) {
    switch (code) {
        case DBF_OK: return "ok";
        case DBF_ERR_INVALID_ARG: return "invalid argument";
        case DBF_ERR_ALIGNMENT: return "pointer not aligned as required";
        case DBF_ERR_UNSUPPORTED: return "shape not supported";
        case DBF_ERR_WORKSPACE: return "workspace missing or too small";
        case DBF_ERR_CUDA: return "CUDA error";
        case DBF_ERR_TIMEOUT: return "device wait timed out";
        case DBF_ERR_DEVICE_ARG: return "device-side argument out of range";
        case DBF_ERR_NUMERIC: return "non-positive pivot in the factorization's Cholesky step";
        case DBF_ERR_BOUNDS: return "index out of range in a kernel (debug build): the access was skipped";
        default: return "unknown status";
    }
}

const char *dbf_last_cuda_error(void) { return g_last_error; }

int dbf_decode_max_tokens(void) { return kDecodeMaxTokens; }

int dbf_pack(const int8_t *signs, int64_t rows, int64_t cols, uint32_t *words, int64_t ldw, void *stream) {
    if (rows < 0 || cols < 0) return DBF_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return DBF_OK;
    if (!signs || !words) return DBF_ERR_INVALID_ARG;
    if (ldw < ceil_div(cols, 32)) return DBF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(words) & 3) != 0) return DBF_ERR_ALIGNMENT;
    cudaError_t e = dbfk::launch_pack(signs, rows, cols, words, ldw, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DBF_OK : cuda_fail(e, "dbf_pack");
}

int dbf_unpack(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw, int8_t *signs, void *stream) {
    if (rows < 0 || cols < 0) return DBF_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return DBF_OK;
    if (!signs || !words) return DBF_ERR_INVALID_ARG;
    if (ldw < ceil_div(cols, 32)) return DBF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(words) & 3) != 0) return DBF_ERR_ALIGNMENT;
    cudaError_t e = dbfk::launch_unpack(words, rows, cols, ldw, signs, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DBF_OK : cuda_fail(e, "dbf_unpack");
}

int dbf_transpose_packed(const uint32_t *words, int64_t rows, int64_t cols, int64_t ldw, uint32_t *words_t,
                         int64_t ldw_t, void *stream) {
    if (rows < 0 || cols < 0) return DBF_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return DBF_OK;
    if (!words || !words_t) return DBF_ERR_INVALID_ARG;
    if (ldw < ceil_div(cols, 32) || ldw_t < ceil_div(rows, 32)) return DBF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(words) & 3) != 0 || (reinterpret_cast<uintptr_t>(words_t) & 3) != 0)
        return DBF_ERR_ALIGNMENT;
    cudaError_t e = dbfk::launch_transpose(words, rows, cols, ldw, words_t, ldw_t, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DBF_OK : cuda_fail(e, "dbf_transpose_packed");
}

int dbf_factors_transposed(const dbf_factors *f, const uint32_t *B2T, int32_t ldw_b2t, const uint32_t *B1T,
                           int32_t ldw_b1t, dbf_factors *out) {
    const int rc = check_factors(f);
    if (rc) return rc;
    if (!out || !B2T || !B1T) return DBF_ERR_INVALID_ARG;
    if (ldw_b2t < ceil_div(f->R, 32) || ldw_b1t < ceil_div(f->N, 32)) return DBF_ERR_INVALID_ARG;
    if (!aligned16(B2T) || !aligned16(B1T)) return DBF_ERR_ALIGNMENT;
    dbf_factors t = {};
    t.N = f->M;
    t.M = f->N;
    t.R = f->R;
    t.ell = f->ell;
    t.B1 = B2T;
    t.ldw1 = ldw_b2t;
    t.B2 = B1T;
    t.ldw2 = ldw_b1t;
    t.alpha = f->gamma;
    t.beta = f->beta;
    t.gamma = f->alpha;
    *out = t;
    return DBF_OK;
}

size_t dbf_workspace_bytes_path(const dbf_factors *f, int64_t T, int path) {
    if (check_factors(f) != DBF_OK || T < 0) return 0;
    if (path < DBF_PATH_AUTO || path > DBF_PATH_PREFILL) return 0;
    return ws_for(f, T, path);
}

size_t dbf_workspace_bytes(const dbf_factors *f, int64_t T) {
    return dbf_workspace_bytes_path(f, T, DBF_PATH_AUTO);
}

int dbf_matmul_path(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y, int accumulate, void *workspace,
                    size_t ws_bytes, void *stream, int path) {
    const int rc = dbfk::check_matmul_args(f, x, T, y, accumulate, path);
    if (rc != DBF_OK || T == 0) return rc;
    path = resolve_path(path, T);
    const size_t need = ws_for(f, T, path);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    if (!status_ptr()) return cuda_fail(cudaGetLastError(), "status word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (path == DBF_PATH_DECODE) return run_decode(f, x, T, y, accumulate, workspace, s);
    return run_prefill(f, x, T, y, accumulate, workspace, s);
}

int dbf_matmul(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y, int accumulate, void *workspace,
               size_t ws_bytes, void *stream) {
    return dbf_matmul_path(f, x, T, y, accumulate, workspace, ws_bytes, stream, DBF_PATH_AUTO);
}

int dbf_selftest_decode_one_launch(const dbf_factors *f, const uint16_t *x, int64_t T, uint16_t *y, int accumulate,
                                   void *workspace, size_t ws_bytes, uint32_t *barrier, void *stream) {
    const int rc = dbfk::check_matmul_args(f, x, T, y, accumulate, DBF_PATH_DECODE);
    if (rc != DBF_OK || T == 0) return rc;
    if (T > kDecodeMaxTokens || !barrier || (reinterpret_cast<uintptr_t>(barrier) & 7) != 0)
        return DBF_ERR_INVALID_ARG;
    const size_t need = ws_for(f, T, DBF_PATH_DECODE);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    if (!status_ptr()) return cuda_fail(cudaGetLastError(), "status word");
    dbfk::DecodeCall c = {};
    c.f = f;
    c.N = f->N;
    c.M = f->M;
    c.R = f->R;
    c.ell = f->ell;
    c.T = static_cast<int>(T);
    c.tokens_per_problem = static_cast<int>(T);
    c.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    c.y = reinterpret_cast<__nv_bfloat16 *>(y);
    c.accumulate = accumulate;
    c.status = status_ptr();
    const cudaError_t e =
        dbfk::launch_decode_one_launch(c, static_cast<__half *>(workspace), static_cast<int>(v_ld(f->R)), barrier,
                                       num_sms(), static_cast<cudaStream_t>(stream));
    if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorNotSupported) {
        snprintf(g_last_error, sizeof(g_last_error), "one-launch decode: %s",
                 e == cudaErrorNotSupported ? "the two stages' plans split K over different cluster sizes, or "
                                                                 "need more shared memory than a CTA has"
                                            : "the grid does not fit on the GPU at once");
        return DBF_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? DBF_OK : cuda_fail(e, "one-launch decode");
}

}  // extern "C"

namespace {

// grouped call: validation shared by the workspace query and the call
int check_group(const dbf_factors *fs, int32_t G) {
    if (!fs || G < 1) return DBF_ERR_INVALID_ARG;
    if (G > dbfk::kMaxGroup) return DBF_ERR_UNSUPPORTED;
    for (int p = 0; p < G; ++p) {
        const int rc = check_factors(&fs[p]);
        if (rc) return rc;
        if (fs[p].ell != fs[0].ell) return DBF_ERR_INVALID_ARG;
    }
    return DBF_OK;
}

size_t ws_grouped(const dbf_factors *fs, int G, int64_t T) {
    size_t need = 0;
    for (int p = 0; p < G; ++p) {
        const dbf_factors &f = fs[p];
        if (T <= kDecodeMaxTokens)
            need += ws_decode(f.N, f.M, f.R, f.ell, T);  // each problem its own V
        else
            need = std::max(need, ws_prefill(f.N, f.M, f.R, f.ell, T));  // problems run one after another
    }
    return need;
}

}  // namespace

extern "C" {

size_t dbf_grouped_workspace_bytes(const dbf_factors *fs, int32_t G, int64_t T) {
    if (check_group(fs, G) != DBF_OK || T < 0) return 0;
    return ws_grouped(fs, G, T);
}

int dbf_grouped_launch_count(const dbf_factors *fs, int32_t G, int64_t T) {
    if (check_group(fs, G) != DBF_OK || T < 0) return -1;
    if (T == 0) return 0;
    return T <= kDecodeMaxTokens ? 2 : 3 * G;
}

int dbf_matmul_grouped(const dbf_factors *fs, int32_t G, const uint16_t *const *xs, uint16_t *const *ys, int64_t T,
                       int accumulate, void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_group(fs, G);
    if (rc) return rc;
    if (T < 0 || (accumulate != 0 && accumulate != 1)) return DBF_ERR_INVALID_ARG;
    if (T == 0) return DBF_OK;
    if (T > (int64_t(1) << 26)) return DBF_ERR_UNSUPPORTED;
    if (!xs || !ys) return DBF_ERR_INVALID_ARG;
    for (int p = 0; p < G; ++p) {
        if (!xs[p] || !ys[p]) return DBF_ERR_INVALID_ARG;
        if (!aligned16(xs[p]) || !aligned16(ys[p])) return DBF_ERR_ALIGNMENT;
    }
    const size_t need = ws_grouped(fs, G, T);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    if (!status_ptr()) return cuda_fail(cudaGetLastError(), "status word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > kDecodeMaxTokens) {
        // large batches: each problem is a full set of GEMMs, launch cost is negligible
        for (int p = 0; p < G; ++p) {
            rc = run_prefill(&fs[p], xs[p], T, ys[p], accumulate, workspace, s);
            if (rc) return rc;
        }
        return DBF_OK;
    }
    dbfk::DecodeGroupCall c = {};
    c.G = G;
    c.T = static_cast<int>(T);
    c.ell = fs[0].ell;
    c.accumulate = accumulate;
    c.status = status_ptr();
    char *base = static_cast<char *>(workspace);
    for (int p = 0; p < G; ++p) {
        c.f[p] = &fs[p];
        c.x[p] = reinterpret_cast<const __nv_bfloat16 *>(xs[p]);
        c.y[p] = reinterpret_cast<__nv_bfloat16 *>(ys[p]);
        c.V[p] = reinterpret_cast<__half *>(base);
        c.ldv[p] = static_cast<int>(v_ld(fs[p].R));
        base += ws_decode(fs[p].N, fs[p].M, fs[p].R, fs[p].ell, T);
    }
    const cudaError_t e = dbfk::launch_decode_grouped(c, num_sms(), s);
    return e == cudaSuccess ? DBF_OK : map_launch_error(e, "grouped decode");
}

size_t dbf_backward_workspace_bytes(const dbf_factors *f, int64_t T) {
    if (check_factors(f) != DBF_OK || T < 0) return 0;
    return ws_backward(f->N, f->M, f->R, f->ell, T);
}

int dbf_backward(const dbf_factors *f, const dbf_factors *ft, const uint16_t *x, const uint16_t *dy, int64_t T,
                 uint16_t *dx, float *dalpha, float *dbeta, float *dgamma, void *workspace, size_t ws_bytes,
                 void *stream) {
    int rc = check_factors(f);
    if (rc) return rc;
    rc = check_factors(ft);
    if (rc) return rc;
    if (ft->N != f->M || ft->M != f->N || ft->R != f->R || ft->ell != f->ell) return DBF_ERR_INVALID_ARG;
    if (T < 0 || !dalpha || !dbeta || !dgamma) return DBF_ERR_INVALID_ARG;
    if (T > (int64_t(1) << 26)) return DBF_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !dy)) return DBF_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (dy && !aligned16(dy)) || (dx && !aligned16(dx)) || !aligned16(dalpha) ||
        !aligned16(dbeta) || !aligned16(dgamma))
        return DBF_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(dalpha, 0, sizeof(float) * size_t(f->ell) * f->N, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, sizeof(float) * size_t(f->ell) * f->R, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dgamma, 0, sizeof(float) * size_t(f->ell) * f->M, s);
        return e == cudaSuccess ? DBF_OK : cuda_fail(e, "backward: zero the scale gradients");
    }
    const size_t need = ws_backward(f->N, f->M, f->R, f->ell, T);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    if (!status_ptr()) return cuda_fail(cudaGetLastError(), "status word");
    return run_backward(f, ft, x, dy, T, dx, dalpha, dbeta, dgamma, workspace, s);
}

size_t dbf_hostio_workspace_bytes(const dbf_factors *f, int64_t T) {
    if (check_factors(f) != DBF_OK || T < 0) return 0;
    return align_up(size_t(T) * f->M * 2) + align_up(size_t(T) * f->N * 2) + ws_for(f, T, DBF_PATH_AUTO);
}

int dbf_matmul_hostio(const dbf_factors *f, const uint16_t *x_host, int64_t T, uint16_t *y_host, int accumulate,
                      void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_factors(f);
    if (rc) return rc;
    if (T < 0 || (accumulate != 0 && accumulate != 1)) return DBF_ERR_INVALID_ARG;
    if (T == 0) return DBF_OK;
    if (!x_host || !y_host) return DBF_ERR_INVALID_ARG;
    const size_t need = dbf_hostio_workspace_bytes(f, T);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(workspace);
    uint16_t *xd = reinterpret_cast<uint16_t *>(base);
    uint16_t *yd = reinterpret_cast<uint16_t *>(base + align_up(size_t(T) * f->M * 2));
    char *inner = base + align_up(size_t(T) * f->M * 2) + align_up(size_t(T) * f->N * 2);
    const size_t inner_bytes = ws_bytes - size_t(inner - base);
    cudaError_t e = cudaMemcpyAsync(xd, x_host, size_t(T) * f->M * 2, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "hostio x copy");
    if (accumulate) {
        e = cudaMemcpyAsync(yd, y_host, size_t(T) * f->N * 2, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "hostio y copy");
    }
    rc = dbf_matmul(f, xd, T, yd, accumulate, inner, inner_bytes, stream);
    if (rc) return rc;
    e = cudaMemcpyAsync(y_host, yd, size_t(T) * f->N * 2, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "hostio y readback");
    return DBF_OK;
}

}  // extern "C"

namespace {

// Calls whose host buffers are contiguous share one copy each way, up to this
// many (with the four slots: 16 per copy and 3 slots gave 3.86 M tokens/s end to
// end on the 4096 x 4096, R = 64, T = 16 adapter, 32 and 4 slots 3.99 M).
constexpr int kPipeChunk = 32;

// [start, end) of the allocation that holds host pointer p, as the driver
// knows it (page-locked memory under unified addressing); false for memory
// the driver does not know (pageable), whose calls are then copied one by one.
bool host_allocation(const void *p, uintptr_t *start, uintptr_t *end) {
    static PFN_cuPointerGetAttribute_v4000 get = nullptr;
    static bool looked = false;
    if (!looked) {
        looked = true;
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &fn, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get = reinterpret_cast<PFN_cuPointerGetAttribute_v4000>(fn);
    }
    if (!get) return false;
    CUdeviceptr base = 0;
    size_t size = 0;
    const CUdeviceptr dp = static_cast<CUdeviceptr>(reinterpret_cast<uintptr_t>(p));
    if (get(&base, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, dp) != CUDA_SUCCESS ||
        get(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, dp) != CUDA_SUCCESS || size == 0) {
        cudaGetLastError();
        return false;
    }
    *start = static_cast<uintptr_t>(base);
    *end = static_cast<uintptr_t>(base) + size;
    return *start <= reinterpret_cast<uintptr_t>(p) && reinterpret_cast<uintptr_t>(p) < *end;
}

struct BatchSizes {
    size_t x, y, inner, slot;  // per call maxima (aligned) and one slot
};

// Slot layout: x of up to kPipeChunk calls back to back, then their y, then
// one inner workspace (the calls of a chunk run one after another on one
// stream, so they share it, as consecutive dbf_matmul calls do).
int batch_sizes(const dbf_factors *fs, int32_t L, int64_t T, BatchSizes *b) {
    *b = {};
    for (int l = 0; l < L; ++l) {
        const int rc = check_factors(&fs[l]);
        if (rc) return rc;
        b->x = std::max(b->x, size_t(T) * fs[l].M * 2);
        b->y = std::max(b->y, size_t(T) * fs[l].N * 2);
        b->inner = std::max(b->inner, align_up(ws_for(&fs[l], T, DBF_PATH_AUTO)));
    }
    const size_t chunk = size_t(std::min(L, kPipeChunk));
    b->slot = align_up(chunk * b->x) + align_up(chunk * b->y) + b->inner;
    return DBF_OK;
}

}  // namespace

extern "C" {

size_t dbf_hostio_batch_workspace_bytes(const dbf_factors *fs, int32_t L, int64_t T) {
    if (!fs || L < 1 || T < 0) return 0;
    BatchSizes b;
    if (batch_sizes(fs, L, T, &b) != DBF_OK) return 0;
    return kPipeSlots * b.slot;
}

int dbf_matmul_hostio_batch(const dbf_factors *fs, int32_t L, const uint16_t *const *x_host, uint16_t *const *y_host,
                            int64_t T, int accumulate, void *workspace, size_t ws_bytes, void *stream) {
    if (!fs || L < 0 || T < 0 || (accumulate != 0 && accumulate != 1)) return DBF_ERR_INVALID_ARG;
    if (L == 0 || T == 0) return DBF_OK;
    if (!x_host || !y_host) return DBF_ERR_INVALID_ARG;
    BatchSizes b;
    int rc = batch_sizes(fs, L, T, &b);
    if (rc) return rc;
    for (int l = 0; l < L; ++l)
        if (!x_host[l] || !y_host[l]) return DBF_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < kPipeSlots * b.slot) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    cudaError_t e;
    HostioPipe *p = hostio_pipe(&e);
    if (!p) return cuda_fail(e, "hostio pipeline streams");
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    // fork: the three pipeline streams start after the work already on the caller's stream
    e = cudaEventRecord(p->fork, user);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->in, p->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->cmp, p->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->out, p->fork, 0);
    if (e != cudaSuccess) rc = cuda_fail(e, "hostio pipeline fork");  // still joined below
    char *ws = static_cast<char *>(workspace);
    const size_t chunk_cap = size_t(std::min(L, kPipeChunk));
    // Chunk sizes ramp up (4, 8, 16, ... calls) so that the first kernels start after a short
    // copy-in, and down over the last 2 * kPipeChunk calls (half of what is left, at least 4) so
    // that the last read-back is short.
    auto cap_for = [&](int c, int l0) {
        size_t cap = std::min(chunk_cap, size_t(4) << std::min(c, 20));
        const int left = L - l0;
        if (left <= 2 * kPipeChunk) cap = std::min(cap, size_t(std::max(4, left / 2)));
        return std::max<size_t>(1, cap);
    };
    int l0 = 0;
    for (int c = 0; l0 < L && rc == DBF_OK; ++c) {
        // the chunk: calls l0 .. l1-1 whose host x (and y) follow one another in memory, with
        // byte sizes that keep every device copy 16-byte aligned
        auto xbytes = [&](int l) { return size_t(T) * fs[l].M * 2; };
        auto ybytes = [&](int l) { return size_t(T) * fs[l].N * 2; };
        // (both ends of a merged copy inside one allocation)
        int l1 = l0 + 1;
        uintptr_t xa = 0, xe = 0, ya = 0, ye = 0;
        const size_t cap = cap_for(c, l0);
        if (cap > 1 && host_allocation(x_host[l0], &xa, &xe) && host_allocation(y_host[l0], &ya, &ye)) {
            while (l1 < L && size_t(l1 - l0) < cap && xbytes(l1 - 1) % 16 == 0 && ybytes(l1 - 1) % 16 == 0) {
                const uintptr_t xp = reinterpret_cast<uintptr_t>(x_host[l1]);
                const uintptr_t yp = reinterpret_cast<uintptr_t>(y_host[l1]);
                if (xp != reinterpret_cast<uintptr_t>(x_host[l1 - 1]) + xbytes(l1 - 1) ||
                    yp != reinterpret_cast<uintptr_t>(y_host[l1 - 1]) + ybytes(l1 - 1) || xp + xbytes(l1) > xe ||
                    yp + ybytes(l1) > ye)
                    break;
                ++l1;
            }
        }
        size_t xs = 0, ys = 0;
        for (int l = l0; l < l1; ++l) {
            xs += xbytes(l);
            ys += ybytes(l);
        }
        const int k = c % kPipeSlots;
        char *base = ws + size_t(k) * b.slot;
        char *xd = base;
        char *yd = base + align_up(chunk_cap * b.x);
        char *inner = yd + align_up(chunk_cap * b.y);
        // copy-in: the slot is free once its previous read-back has finished
        if (c >= kPipeSlots && (e = cudaStreamWaitEvent(p->in, p->d2h[k], 0)) != cudaSuccess) {
            rc = cuda_fail(e, "hostio pipeline: wait for a free slot");
            break;
        }
        if ((e = cudaMemcpyAsync(xd, x_host[l0], xs, cudaMemcpyHostToDevice, p->in)) != cudaSuccess) {
            rc = cuda_fail(e, "hostio pipeline: copy x in");
            break;
        }
        if (accumulate && (e = cudaMemcpyAsync(yd, y_host[l0], ys, cudaMemcpyHostToDevice, p->in)) != cudaSuccess) {
            rc = cuda_fail(e, "hostio pipeline: copy y in");
            break;
        }
        if ((e = cudaEventRecord(p->h2d[k], p->in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(p->cmp, p->h2d[k], 0)) != cudaSuccess) {
            rc = cuda_fail(e, "hostio pipeline: hand the slot to the compute stream");
            break;
        }
        size_t xo = 0, yo = 0;
        for (int l = l0; l < l1 && rc == DBF_OK; ++l) {
            rc = dbf_matmul(&fs[l], reinterpret_cast<const uint16_t *>(xd + xo), T,
                            reinterpret_cast<uint16_t *>(yd + yo), accumulate, inner, b.inner, p->cmp);
            xo += xbytes(l);
            yo += ybytes(l);
        }
        if (rc) break;
        e = cudaEventRecord(p->done[k], p->cmp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(p->out, p->done[k], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(y_host[l0], yd, ys, cudaMemcpyDeviceToHost, p->out);
        if (e == cudaSuccess) e = cudaEventRecord(p->d2h[k], p->out);
        if (e != cudaSuccess) {
            rc = cuda_fail(e, "hostio pipeline read-back");
            break;
        }
        l0 = l1;
    }
    // join, also after an error: the caller's stream continues after all three pipeline streams
    // (work already queued there stays ordered before the caller's next work, and a CUDA graph
    // capture never sees a fork without its join)
    cudaStream_t ss[3] = {p->in, p->cmp, p->out};
    cudaError_t ej = cudaSuccess;
    for (int j = 0; j < 3 && ej == cudaSuccess; ++j) {
        ej = cudaEventRecord(p->join[j], ss[j]);
        if (ej == cudaSuccess) ej = cudaStreamWaitEvent(user, p->join[j], 0);
    }
    if (rc) return rc;
    return ej == cudaSuccess ? DBF_OK : cuda_fail(ej, "hostio pipeline join");
}

size_t dbf_segmented_workspace_bytes(int32_t N, int32_t M, int32_t R, int32_t ell, int64_t T, int32_t S) {
    (void)S;
    if (check_dims(N, M, R, ell) != DBF_OK || T < 0) return 0;
    return ws_decode(N, M, R, ell, T);
}

int dbf_matmul_segmented(const dbf_factors *d_adapters, int32_t n_adapters, int32_t N, int32_t M, int32_t R,
                         int32_t ell, const uint16_t *x, int64_t T, uint16_t *y, const int32_t *d_seg_offsets,
                         const int32_t *d_seg_adapter, int32_t S, int accumulate, void *workspace, size_t ws_bytes,
                         void *stream) {
    using namespace dbfk;
    int rc = check_dims(N, M, R, ell);
    if (rc) return rc;
    if (T < 0 || S < 0 || n_adapters < 0 || (accumulate != 0 && accumulate != 1)) return DBF_ERR_INVALID_ARG;
    if (T == 0 || S == 0) return DBF_OK;
    if (S > 65535 || T > (int64_t(1) << 26)) return DBF_ERR_UNSUPPORTED;
    if (!d_adapters || n_adapters < 1 || !x || !y || !d_seg_offsets || !d_seg_adapter) return DBF_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || !aligned16(d_adapters)) return DBF_ERR_ALIGNMENT;
    const size_t need = dbf_segmented_workspace_bytes(N, M, R, ell, T, S);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    if (!status_ptr()) return cuda_fail(cudaGetLastError(), "status word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int64_t tok = segment_tokens(T, S);
    dbf_factors shape = {};
    shape.N = N;
    shape.M = M;
    shape.R = R;
    shape.ell = ell;
    // routed batches: the reduce-scatter kernel is planned per segment and
    // measured slower there (70.6 against 22.6 us per 256-token batch of 64
    // adapters), so only a batch of one segment takes it
    const RsPlan rp = S == 1 ? rs_plan_for(N, M, R, ell, tok, S, accumulate != 0) : RsPlan{};
    if (rp.CT != 0) {
        RsArgs ra = rs_args(&shape, x, T, y, accumulate, rp);
        ra.seg_off = d_seg_offsets;
        ra.seg_ad = d_seg_adapter;
        ra.adapters = d_adapters;
        ra.n_adapters = n_adapters;
        cudaError_t e = launch_decode_rs(true, rp, ra, S, s);
        return e == cudaSuccess ? DBF_OK : cuda_fail(e, "segmented decode");
    }
    FusedPlan p = fused_plan_for(N, M, R, ell, tok, S, accumulate != 0);
    if (p.CT != 0) {
        FusedArgs fa = fused_args(&shape, x, T, y, accumulate, p);
        fa.seg_off = d_seg_offsets;
        fa.seg_ad = d_seg_adapter;
        fa.adapters = d_adapters;
        fa.n_adapters = n_adapters;
        // up to kChunkMapMaxS segments: one cluster per chunk of the plan's tokens, so that a
        // segment longer than one chunk spreads over several clusters instead of running its
        // chunks one after another.  Segment s gives max(1, ceil(len_s / tpc)) chunks, at most
        // S + (T - 1) / tpc in all; the slots past the actual list exit at once.
        int grid_y = S;
        const int64_t tpc = 8 * int64_t(p.CT) / ell;
        const int64_t slots = int64_t(S) + (T - 1) / tpc;
        if (S <= kChunkMapMaxS && slots <= 65535) {
            fa.chunk_map_S = S;
            grid_y = static_cast<int>(slots);
        }
        cudaError_t e = launch_decode_fused(true, p, fa, grid_y, s, true);
        return e == cudaSuccess ? DBF_OK : cuda_fail(e, "segmented fused decode");
    }
    DecodeCall c = {};
    c.N = N;
    c.M = M;
    c.R = R;
    c.ell = ell;
    c.T = static_cast<int>(T);
    c.tokens_per_problem = static_cast<int>(tok);
    c.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    c.y = reinterpret_cast<__nv_bfloat16 *>(y);
    c.accumulate = accumulate;
    c.seg_off = d_seg_offsets;
    c.seg_ad = d_seg_adapter;
    c.adapters = d_adapters;
    c.n_adapters = n_adapters;
    c.S = S;
    c.status = status_ptr();
    cudaError_t e = launch_decode_two_stage(c, static_cast<__half *>(workspace), static_cast<int>(v_ld(R)), num_sms(),
                                            s);
    return e == cudaSuccess ? DBF_OK : map_launch_error(e, "segmented decode");
}

int dbf_launch_count(const dbf_factors *f, int64_t T, int path) {
    if (check_factors(f) != DBF_OK || T <= 0) return 0;
    if (path < DBF_PATH_AUTO || path > DBF_PATH_PREFILL) return 0;
    path = resolve_path(path, T);
    if (path == DBF_PATH_PREFILL) return 3;
    if (rs_plan_for(f->N, f->M, f->R, f->ell, T, 1, false).CT != 0) return 1;
    return fused_plan_for(f->N, f->M, f->R, f->ell, T, 1, false).CT != 0 ? 1 : 2;
}

int dbf_segmented_launch_count(int32_t N, int32_t M, int32_t R, int32_t ell, int64_t T, int32_t S) {
    if (check_dims(N, M, R, ell) != DBF_OK || T <= 0 || S <= 0) return 0;
    if (S == 1 && rs_plan_for(N, M, R, ell, segment_tokens(T, S), S, false).CT != 0) return 1;
    return fused_plan_for(N, M, R, ell, segment_tokens(T, S), S, false).CT != 0 ? 1 : 2;
}

static int check_factorize_args(int64_t N, int64_t M, int64_t k, const dbf_factorize_params *p) {
    if (!p || N < 1 || M < 1 || k < 1) return DBF_ERR_INVALID_ARG;
    if (p->outer < 0 || p->inner < 0 || p->power_iters < 0 || !(p->rho_rel > 0.f)) return DBF_ERR_INVALID_ARG;
    if (N > 65535 || M > 65535 || k > 16384) return DBF_ERR_UNSUPPORTED;
    return DBF_OK;
}

size_t dbf_factorize_workspace_bytes(int64_t N, int64_t M, int64_t k) {
    if (N < 1 || M < 1 || k < 1 || N > 65535 || M > 65535 || k > 16384) return 0;
    return dbfk::factorize_workspace_bytes(N, M, k);
}

int dbf_factorize_launch_count(int64_t N, int64_t M, int64_t k, const dbf_factorize_params *p) {
    if (check_factorize_args(N, M, k, p) != DBF_OK) return -1;
    return dbfk::factorize_launch_count(N, M, k, *p);
}

int dbf_factorize(const float *W, int64_t N, int64_t M, int64_t k, const dbf_factorize_params *p, float *a,
                  int8_t *A, float *m_left, float *m_right, int8_t *B, float *b, void *workspace, size_t ws_bytes,
                  void *stream) {
    int rc = check_factorize_args(N, M, k, p);
    if (rc) return rc;
    if (!W || !a || !A || !m_left || !m_right || !B || !b) return DBF_ERR_INVALID_ARG;
    const size_t need = dbfk::factorize_workspace_bytes(N, M, k);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    const uintptr_t f4 = reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(a) |
                         reinterpret_cast<uintptr_t>(m_left) | reinterpret_cast<uintptr_t>(m_right) |
                         reinterpret_cast<uintptr_t>(b);
    if (f4 & 3) return DBF_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return cuda_fail(cudaGetLastError(), "status word");
    cudaError_t e = dbfk::prepare_factorize(k);
    if (e != cudaSuccess) return cuda_fail(e, "factorize: shared memory attribute");
    if (p->outer == 0 || p->inner == 0) return DBF_OK;
    e = dbfk::launch_factorize(W, int(N), int(M), int(k), *p, a, A, m_left, m_right, B, b, workspace, st,
                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DBF_OK : cuda_fail(e, "factorize");
}

size_t dbf_factorize_weighted_workspace_bytes(int64_t N, int64_t M, int64_t k) {
    if (N < 1 || M < 1 || k < 1 || N > 65535 || M > 65535 || k > 16384) return 0;
    return dbfk::factorize_weighted_workspace_bytes(N, M, k);
}

int dbf_factorize_weighted_launch_count(int64_t N, int64_t M, int64_t k, const dbf_factorize_params *p) {
    if (check_factorize_args(N, M, k, p) != DBF_OK) return -1;
    return dbfk::factorize_weighted_launch_count(N, M, k, *p);
}

int dbf_factorize_weighted(const float *W, int64_t N, int64_t M, int64_t k, const dbf_factorize_params *p,
                           const float *d_out, const float *d_in, float *a, int8_t *A, float *m_left,
                           float *m_right, int8_t *B, float *b, void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_factorize_args(N, M, k, p);
    if (rc) return rc;
    if (!W || !d_out || !d_in || !a || !A || !m_left || !m_right || !B || !b) return DBF_ERR_INVALID_ARG;
    const size_t need = dbfk::factorize_weighted_workspace_bytes(N, M, k);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DBF_ERR_ALIGNMENT;
    const uintptr_t f4 = reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(d_out) |
                         reinterpret_cast<uintptr_t>(d_in) | reinterpret_cast<uintptr_t>(a) |
                         reinterpret_cast<uintptr_t>(m_left) | reinterpret_cast<uintptr_t>(m_right) |
                         reinterpret_cast<uintptr_t>(b);
    if (f4 & 3) return DBF_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return cuda_fail(cudaGetLastError(), "status word");
    cudaError_t e = dbfk::prepare_factorize(k);
    if (e != cudaSuccess) return cuda_fail(e, "factorize: shared memory attribute");
    if (p->outer == 0 || p->inner == 0) return DBF_OK;
    e = dbfk::launch_factorize_weighted(W, int(N), int(M), int(k), *p, d_out, d_in, a, A, m_left, m_right, B, b,
                                        workspace, st, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DBF_OK : cuda_fail(e, "factorize (weighted)");
}

int dbf_check_status(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dbf_check_status sync");
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_dbf_status, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "dbf_check_status read");
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dbf_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "dbf_check_status clear");
    return v;
}

int dbf_selftest_bounded_wait(int64_t limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 2000000) return DBF_ERR_INVALID_ARG;
    int *st = status_ptr();
    if (!st) return cuda_fail(cudaGetLastError(), "status word");
    cudaError_t e = dbfk::launch_selftest_wait(st, static_cast<uint64_t>(limit_us) * 1000ull,
                                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DBF_OK : cuda_fail(e, "dbf_selftest_bounded_wait");
}

size_t dbf_selftest_split_gemm_workspace_bytes(int32_t m, int32_t n, int32_t kk) {
    if (m < 1 || n < 1 || kk < 1 || m > 65535 || n > 65535 || kk > 65535) return 0;
    const size_t half = static_cast<size_t>(dbfk::tc_split_half(kk));
    const size_t a = (sizeof(float) * size_t(m) * 2 * half + 255) & ~size_t(255);
    return a + sizeof(float) * size_t(n) * 2 * half;
}

int dbf_selftest_split_gemm(int32_t m, int32_t n, int32_t kk, float alpha, const float *A, int64_t lda,
                            const float *B, int64_t ldb, float beta, float *C, int64_t ldc, int lower,
                            void *workspace, size_t ws_bytes, void *stream) {
    if (m < 1 || n < 1 || kk < 1 || !A || !B || !C || (lower != 0 && lower != 1)) return DBF_ERR_INVALID_ARG;
    if (m > 65535 || n > 65535 || kk > 65535) return DBF_ERR_UNSUPPORTED;
    if (lda < kk || ldb < kk || ldc < n) return DBF_ERR_INVALID_ARG;
    const size_t need = dbf_selftest_split_gemm_workspace_bytes(m, n, kk);
    if (!workspace || ws_bytes < need) return DBF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return DBF_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return cuda_fail(cudaGetLastError(), "status word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = dbfk::tc_prepare();
    const size_t half = static_cast<size_t>(dbfk::tc_split_half(kk));
    float *A2 = static_cast<float *>(workspace);
    float *B2 = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                          ((sizeof(float) * size_t(m) * 2 * half + 255) & ~size_t(255)));
    if (e == cudaSuccess) e = dbfk::tc_split2(A, lda, m, kk, A2, s);
    if (e == cudaSuccess) e = dbfk::tc_split2(B, ldb, n, kk, B2, s);
    if (e == cudaSuccess) e = dbfk::tc_gemm_nt_split(m, n, kk, alpha, A2, B2, beta, C, ldc, st, s, lower);
    return e == cudaSuccess ? DBF_OK : cuda_fail(e, "dbf_selftest_split_gemm");
}

}  // extern "C"
