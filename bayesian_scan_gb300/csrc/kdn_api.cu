// kdn_api.cu -- the C ABI declared in include/kdn.h: host-side argument
// validation, dispatch to the kernels, status strings and the device error
// word.  Every error detectable on the host is returned before any launch.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "kdn.h"
#include "kdn_internal.h"

namespace kdn {

namespace {
constexpr long long kDefaultWaitNs = 2000000000LL;   // 2 s of GPU time
std::atomic<long long> g_wait_ns{kDefaultWaitNs};
std::atomic<long long> g_stall_tile{-1};
int g_sm_count[64] = {};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool head_dim_ok(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }
}  // namespace

cudaError_t diag_take_device_error_bf16(int* status);
cudaError_t diag_take_device_error_f32(int* status);

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

kdn_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return KDN_OK;
    cudaGetLastError();   // clear this thread's (non-sticky) last-error state
    if (e == cudaErrorMemoryAllocation) return KDN_ERR_ALLOC;
    return KDN_ERR_CUDA;
}

}  // namespace kdn

using namespace kdn;

extern "C" {

kdn_status kdn_diag_scan_fwd(const void* q, const void* k, const void* v, const void* beta,
                             const void* d, const float* A, float I_prior, const float* I0,
                             const float* mu0, float* out, float* final_state, int B, int H, int T,
                             int dk, int dv, kdn_dtype in_dtype, void* stream) {
    if (B < 1 || H < 1 || T < 0) return KDN_ERR_INVALID_ARG;
    // with no tokens the per-token tensors (and A) are never read
    if (T > 0 && (!q || !k || !v || !beta || !d || !A || !out)) return KDN_ERR_INVALID_ARG;
    if (in_dtype != KDN_F32 && in_dtype != KDN_BF16) return KDN_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    const long long dmax = dk > dv ? dk : dv;
    if (BH > (1LL << 40) || BH * (T > 0 ? T : 1) > (1LL << 62) / dmax) return KDN_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, beta, out, I0, mu0, final_state};
    for (const void* p : ptrs16)
        if (p && !aligned(p, 16)) return KDN_ERR_INVALID_ARG;
    if ((A && !aligned(A, 4)) || (d && !aligned(d, in_dtype == KDN_BF16 ? 2 : 4)))
        return KDN_ERR_INVALID_ARG;

    DiagArgs a{q, k, v, beta, d, A, I_prior, I0, mu0, out, final_state, B, H, T, dk, dv, in_dtype};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long wait_ns = g_wait_ns.load();
    return in_dtype == KDN_BF16 ? diag_launch_bf16(a, st, wait_ns) : diag_launch_f32(a, st, wait_ns);
}

kdn_status kdn_diag_mobius_scan_fwd(const void* q, const void* k, const void* v, const void* beta,
                                    const void* d, const float* A, float I_prior, const float* I0,
                                    const float* mu0, float* out, float* final_state, const float* ma,
                                    const float* mb, const float* mc, const float* md,
                                    const float* lambda0, float* lambda_out, int B, int H, int T,
                                    int dk, int dv, kdn_dtype in_dtype, void* stream) {
    if (B < 1 || H < 1 || T < 0) return KDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !beta || !d || !A || !out || !ma || !mb || !mc || !md ||
                  !lambda0 || !lambda_out))
        return KDN_ERR_INVALID_ARG;
    if (in_dtype != KDN_F32 && in_dtype != KDN_BF16) return KDN_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    const long long dmax = dk > dv ? dk : dv;
    if (BH > (1LL << 40) || BH * (T > 0 ? T : 1) > (1LL << 62) / dmax) return KDN_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, beta, out, I0, mu0, final_state};
    for (const void* p : ptrs16)
        if (p && !aligned(p, 16)) return KDN_ERR_INVALID_ARG;
    const void* ptrs4[] = {A, ma, mb, mc, md, lambda0, lambda_out};
    for (const void* p : ptrs4)
        if (p && !aligned(p, 4)) return KDN_ERR_INVALID_ARG;
    if (d && !aligned(d, in_dtype == KDN_BF16 ? 2 : 4)) return KDN_ERR_INVALID_ARG;

    DiagArgs a{q, k, v, beta, d, A, I_prior, I0, mu0, out, final_state, B, H, T, dk, dv, in_dtype};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long wait_ns = g_wait_ns.load();
    // the lambda walkers stream whole 16-byte rows; other layouts take the
    // Moebius scan as its own launch after the scan
    const bool fused = T % 4 == 0 && aligned(ma, 16) && aligned(mb, 16) && aligned(mc, 16) &&
                       aligned(md, 16) && aligned(lambda_out, 16);
    if (fused) {
        a.ma = ma; a.mb = mb; a.mc = mc; a.md = md; a.lam0 = lambda0; a.lam_out = lambda_out;
    }
    const kdn_status s =
        in_dtype == KDN_BF16 ? diag_launch_bf16(a, st, wait_ns) : diag_launch_f32(a, st, wait_ns);
    if (s != KDN_OK || fused) return s;
    return mobius_launch(ma, mb, mc, md, lambda0, lambda_out, BH, T, st, wait_ns, -1);
}

kdn_status kdn_lin_scan_fwd(const void* q, const void* k, const void* v, const void* beta,
                            const void* d, const float* A, float I_prior, const float* mu0,
                            float* out, float* final_mu, int B, int H, int T, int dk, int dv,
                            kdn_dtype in_dtype, void* stream) {
    if (B < 1 || H < 1 || T < 0) return KDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !beta || !d || !A || !out)) return KDN_ERR_INVALID_ARG;
    if (in_dtype != KDN_F32 && in_dtype != KDN_BF16) return KDN_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    const long long dmax = dk > dv ? dk : dv;
    if (BH > (1LL << 40) || BH * (T > 0 ? T : 1) > (1LL << 62) / dmax) return KDN_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, beta, out, mu0, final_mu};
    for (const void* p : ptrs16)
        if (p && !aligned(p, 16)) return KDN_ERR_INVALID_ARG;
    if ((A && !aligned(A, 4)) || (d && !aligned(d, in_dtype == KDN_BF16 ? 2 : 4)))
        return KDN_ERR_INVALID_ARG;
    DiagArgs a{q, k, v, beta, d, A, I_prior, nullptr, mu0, out, final_mu, B, H, T, dk, dv, in_dtype};
    a.lin = true;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long wait_ns = g_wait_ns.load();
    return in_dtype == KDN_BF16 ? diag_launch_bf16(a, st, wait_ns) : diag_launch_f32(a, st, wait_ns);
}

kdn_status kdn_diag_scan_bwd(const void* q, const void* k, const void* v, const void* beta,
                             const void* d, const float* A, float I_prior, const float* I0,
                             const float* mu0, const float* grad_out, const float* grad_final_state,
                             float* grad_q, float* grad_k, float* grad_v, float* grad_beta,
                             float* grad_d, float* grad_A, float* grad_init_state, int B, int H,
                             int T, int dk, int dv, kdn_dtype in_dtype, void* workspace,
                             long long workspace_bytes, void* stream) {
    if (B < 1 || H < 1 || T < 0) return KDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !beta || !d || !A || !grad_out || !grad_q || !grad_k ||
                  !grad_v || !grad_beta || !grad_d))
        return KDN_ERR_INVALID_ARG;
    if (in_dtype != KDN_F32 && in_dtype != KDN_BF16) return KDN_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    const long long dmax = dk > dv ? dk : dv;
    if (BH > (1LL << 40) || BH * (T > 0 ? T : 1) > (1LL << 62) / (dmax * dmax)) return KDN_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, beta, grad_out, I0, mu0, grad_final_state, grad_q, grad_k,
                            grad_v, grad_beta, grad_init_state};
    for (const void* p : ptrs16)
        if (p && !aligned(p, 16)) return KDN_ERR_INVALID_ARG;
    const void* ptrs4[] = {A, grad_d, grad_A};
    for (const void* p : ptrs4)
        if (p && !aligned(p, 4)) return KDN_ERR_INVALID_ARG;
    if (d && !aligned(d, in_dtype == KDN_BF16 ? 2 : 4)) return KDN_ERR_INVALID_ARG;
    if (workspace && (!aligned(workspace, 256) ||
                      workspace_bytes < diag_bwd_workspace_bytes(B, H, T, dk, dv)))
        return KDN_ERR_INVALID_ARG;
    if (T == 0 && !grad_init_state && !grad_A) return KDN_OK;
    DiagBwdArgs a{q, k, v, beta, d, A, I_prior, I0, mu0, grad_out, grad_final_state, grad_q,
                  grad_k, grad_v, grad_beta, grad_d, grad_A, grad_init_state, B, H, T, dk, dv,
                  in_dtype, workspace};
    return diag_bwd_launch(a, static_cast<cudaStream_t>(stream));
}

kdn_status kdn_diag_scan_bwd_workspace(int B, int H, int T, int dk, int dv,
                                       long long* workspace_bytes) {
    if (B < 1 || H < 1 || T < 0 || !workspace_bytes) return KDN_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    const long long dmax = dk > dv ? dk : dv;
    if (BH > (1LL << 40) || BH * (T > 0 ? T : 1) > (1LL << 62) / (dmax * dmax)) return KDN_ERR_INVALID_ARG;
    *workspace_bytes = diag_bwd_workspace_bytes(B, H, T, dk, dv);
    return KDN_OK;
}

kdn_status kdn_diag_step(const void* q, const void* k, const void* v, const void* beta, const void* d,
                         const float* A, float I_prior, float* state, float* out, int B, int H, int dk,
                         int dv, kdn_dtype in_dtype, void* stream) {
    if (B < 1 || H < 1) return KDN_ERR_INVALID_ARG;
    if (!q || !k || !v || !beta || !d || !A || !state || !out) return KDN_ERR_INVALID_ARG;
    if (in_dtype != KDN_F32 && in_dtype != KDN_BF16) return KDN_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    if (BH > (1LL << 40)) return KDN_ERR_INVALID_ARG;
    const size_t es = in_dtype == KDN_BF16 ? 2 : 4;
    const void* ins[] = {q, k, v, beta, d};
    for (const void* p : ins)
        if (!aligned(p, es)) return KDN_ERR_INVALID_ARG;
    if (!aligned(A, 4) || !aligned(out, 4) || !aligned(state, 16)) return KDN_ERR_INVALID_ARG;
    return diag_step_launch(q, k, v, beta, d, A, I_prior, state, out, B, H, dk, dv, in_dtype,
                            static_cast<cudaStream_t>(stream));
}

kdn_status kdn_diag_scan_fwd_host(const void* q, const void* k, const void* v, const void* beta,
                                  const void* d, const float* A, float I_prior, const float* I0,
                                  const float* mu0, float* out, float* final_state, int B, int H,
                                  int T, int dk, int dv, kdn_dtype in_dtype, void* stream) {
    if (B < 1 || H < 1 || T < 0) return KDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !beta || !d || !A || !out)) return KDN_ERR_INVALID_ARG;
    if (in_dtype != KDN_F32 && in_dtype != KDN_BF16) return KDN_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDN_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * H;
    const long long dmax = dk > dv ? dk : dv;
    if (BH > (1LL << 40) || BH * (T > 0 ? T : 1) > (1LL << 62) / dmax) return KDN_ERR_INVALID_ARG;
    const void* ins[] = {q, k, v, beta, d};
    for (const void* p : ins)
        if (p && !aligned(p, in_dtype == KDN_BF16 ? 2 : 4)) return KDN_ERR_INVALID_ARG;
    const void* f32s[] = {A, I0, mu0, out, final_state};
    for (const void* p : f32s)
        if (p && !aligned(p, 4)) return KDN_ERR_INVALID_ARG;
    DiagArgs a{q, k, v, beta, d, A, I_prior, I0, mu0, out, final_state, B, H, T, dk, dv, in_dtype};
    return diag_host(a, static_cast<cudaStream_t>(stream), g_wait_ns.load());
}

kdn_status kdn_mobius_scan_host(const float* a, const float* b, const float* c, const float* d,
                                const float* lambda0, float* out, long long N, long long T,
                                void* stream) {
    if (N < 0 || T < 0) return KDN_ERR_INVALID_ARG;
    if (N > 0 && T > 0 && N > (1LL << 62) / T) return KDN_ERR_INVALID_ARG;
    if (N == 0 || T == 0) return KDN_OK;
    if (!a || !b || !c || !d || !lambda0 || !out) return KDN_ERR_INVALID_ARG;
    const void* ptrs[] = {a, b, c, d, lambda0, out};
    for (const void* p : ptrs)
        if (!aligned(p, 4)) return KDN_ERR_INVALID_ARG;
    return mobius_host(a, b, c, d, lambda0, out, N, T, static_cast<cudaStream_t>(stream),
                       g_wait_ns.load());
}

kdn_status kdn_mobius_scan(const float* a, const float* b, const float* c, const float* d,
                           const float* lambda0, float* out, long long N, long long T,
                           void* stream) {
    if (N < 0 || T < 0) return KDN_ERR_INVALID_ARG;
    if (N > 0 && T > 0 && N > (1LL << 62) / T) return KDN_ERR_INVALID_ARG;
    if (N == 0 || T == 0) return KDN_OK;
    if (!a || !b || !c || !d || !lambda0 || !out) return KDN_ERR_INVALID_ARG;
    const void* ptrs[] = {a, b, c, d, lambda0, out};
    for (const void* p : ptrs)
        if (!aligned(p, 4)) return KDN_ERR_INVALID_ARG;
    return mobius_launch(a, b, c, d, lambda0, out, N, T, static_cast<cudaStream_t>(stream),
                         g_wait_ns.load(), g_stall_tile.load());
}

kdn_status kdn_diag_scan_plan(int B, int H, int T, int dk, int dv, kdn_dtype in_dtype,
                              int* parts, int* kernels, long long* scratch_bytes) {
    if (B < 1 || H < 1 || T < 0) return KDN_ERR_INVALID_ARG;
    if (in_dtype != KDN_F32 && in_dtype != KDN_BF16) return KDN_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDN_ERR_UNSUPPORTED;
    DiagArgs a{};
    a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.dtype = in_dtype;
    int p = 0, k = 0;
    size_t sb = 0;
    const kdn_status s = in_dtype == KDN_BF16 ? diag_plan_bf16(a, &p, &k, &sb) : diag_plan_f32(a, &p, &k, &sb);
    if (s != KDN_OK) return s;
    if (parts) *parts = p;
    if (kernels) *kernels = k;
    if (scratch_bytes) *scratch_bytes = static_cast<long long>(sb);
    return KDN_OK;
}

kdn_status kdn_mobius_scan_plan(long long N, long long T, int* kernels, long long* scratch_bytes) {
    if (N < 0 || T < 0) return KDN_ERR_INVALID_ARG;
    if (N > 0 && T > 0 && N > (1LL << 62) / T) return KDN_ERR_INVALID_ARG;
    int k = 0;
    size_t sb = 0;
    mobius_plan(N, T, &k, &sb);
    if (kernels) *kernels = k;
    if (scratch_bytes) *scratch_bytes = static_cast<long long>(sb);
    return KDN_OK;
}

kdn_status kdn_mobius_scan_noalloc(const float* a, const float* b, const float* c,
                                   const float* d, const float* lambda0, float* out, long long N,
                                   long long T, void* stream) {
    if (N < 0 || T < 0) return KDN_ERR_INVALID_ARG;
    if (N > 0 && T > 0 && N > (1LL << 62) / T) return KDN_ERR_INVALID_ARG;
    if (N == 0 || T == 0) return KDN_OK;
    if (!a || !b || !c || !d || !lambda0 || !out) return KDN_ERR_INVALID_ARG;
    const void* ptrs[] = {a, b, c, d, lambda0, out};
    for (const void* p : ptrs)
        if (!aligned(p, 4)) return KDN_ERR_INVALID_ARG;
    return mobius_launch_noalloc(a, b, c, d, lambda0, out, N, T, static_cast<cudaStream_t>(stream),
                                 g_wait_ns.load());
}

const char* kdn_status_string(kdn_status s) {
    switch (s) {
        case KDN_OK: return "KDN_OK";
        case KDN_ERR_INVALID_ARG: return "KDN_ERR_INVALID_ARG: invalid argument";
        case KDN_ERR_UNSUPPORTED: return "KDN_ERR_UNSUPPORTED: unsupported head dimension or dtype";
        case KDN_ERR_CUDA: return "KDN_ERR_CUDA: CUDA runtime error";
        case KDN_ERR_TIMEOUT: return "KDN_ERR_TIMEOUT: a bounded device-side wait ran out";
        case KDN_ERR_ALLOC: return "KDN_ERR_ALLOC: scratch allocation failed";
    }
    return "unknown kdn_status";
}

kdn_status kdn_get_device_error(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    int s1 = 0, s2 = 0, s3 = 0;
    if ((e = diag_take_device_error_bf16(&s1)) != cudaSuccess) return from_cuda(e);
    if ((e = diag_take_device_error_f32(&s2)) != cudaSuccess) return from_cuda(e);
    if ((e = mobius_take_device_error(&s3)) != cudaSuccess) return from_cuda(e);
    if (s1) return static_cast<kdn_status>(s1);
    if (s2) return static_cast<kdn_status>(s2);
    return static_cast<kdn_status>(s3);
}

void kdn_set_wait_limit_ns(long long ns) { g_wait_ns.store(ns > 0 ? ns : kDefaultWaitNs); }

void kdn_debug_stall_mobius_tile(long long tile) { g_stall_tile.store(tile); }

const char* kdn_version(void) { return "kdn 0.1.0 sm_103a"; }

}  // extern "C"
