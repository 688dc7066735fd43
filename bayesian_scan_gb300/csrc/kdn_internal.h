// kdn_internal.h -- declarations shared by the library's translation units
// (not part of the public ABI).
#pragma once
#include <cuda_runtime.h>

#include "kdn.h"

namespace kdn {

// Arguments of one diagonal-scan call after host-side validation.
struct DiagArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* beta;
    const void* d;
    const float* A;
    float I_prior;
    const float* I0;
    const float* mu0;
    float* out;
    float* final_state;
    int B, H, T, dk, dv;
    kdn_dtype dtype;
    // tokens between the rows of consecutive heads in `out` and in `d` (0: T,
    // i.e. [B,H,T,...]); lets a call use a token range of longer tensors
    long long out_ld = 0;
    long long d_ld = 0;
    // the non-metaplastic limit: importance held at I_prior (I0 unused,
    // final_state is mu_T alone, [B,H,dv,dk])
    bool lin = false;
    // per-head Moebius lambda computed in the same launch as the scan (lam_out
    // non-null): coefficients [B*H, T] fp32 with 16-byte aligned rows (T % 4
    // == 0), lam0 [B*H], lam_out [B*H, T]
    const float* ma = nullptr;
    const float* mb = nullptr;
    const float* mc = nullptr;
    const float* md = nullptr;
    const float* lam0 = nullptr;
    float* lam_out = nullptr;
};

// Per-dtype launchers (diag_bf16.cu / diag_f32.cu).
kdn_status diag_launch_bf16(const DiagArgs& a, cudaStream_t stream, long long wait_ns);
kdn_status diag_launch_f32(const DiagArgs& a, cudaStream_t stream, long long wait_ns);

// Launch plans (no launch): token parts, kernels launched, scratch bytes.
kdn_status diag_plan_bf16(const DiagArgs& a, int* parts, int* kernels, size_t* scratch);
kdn_status diag_plan_f32(const DiagArgs& a, int* parts, int* kernels, size_t* scratch);
void mobius_plan(long long N, long long T, int* kernels, size_t* scratch);

// Moebius scan launcher (mobius_scan.cu).
kdn_status mobius_launch(const float* a, const float* b, const float* c, const float* d,
                         const float* lambda0, float* out, long long N, long long T,
                         cudaStream_t stream, long long wait_ns, long long stall_tile);

// Allocation-free Moebius scan: look-back scratch in a fixed device array.
kdn_status mobius_launch_noalloc(const float* a, const float* b, const float* c, const float* d,
                                 const float* lambda0, float* out, long long N, long long T,
                                 cudaStream_t stream, long long wait_ns);
long long mobius_noalloc_max_tiles();

// One-token step of the diagonal update on a device-resident state
// (diag_step.cu); arguments validated.
kdn_status diag_step_launch(const void* q, const void* k, const void* v, const void* beta,
                            const void* d, const float* A, float I_prior, float* state, float* out,
                            int B, int H, int dk, int dv, kdn_dtype dtype, cudaStream_t stream);

// Arguments of one backward call after host-side validation (diag_bwd.cu).
struct DiagBwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* beta;
    const void* d;
    const float* A;
    float I_prior;
    const float* I0;
    const float* mu0;
    const float* grad_out;
    const float* grad_final_state;
    float* grad_q;
    float* grad_k;
    float* grad_v;
    float* grad_beta;
    float* grad_d;
    float* grad_A;
    float* grad_init_state;
    int B, H, T, dk, dv;
    kdn_dtype dtype;
    void* workspace;   // caller's scratch of diag_bwd_workspace_bytes, or null
};
kdn_status diag_bwd_launch(const DiagBwdArgs& a, cudaStream_t stream);
long long diag_bwd_workspace_bytes(int B, int H, int T, int dk, int dv);

// Host-buffer pipelines (kdn_host.cu): arguments validated, every pointer a
// host pointer; synchronous.
kdn_status diag_host(const DiagArgs& a, cudaStream_t stream, long long wait_ns);
kdn_status mobius_host(const float* a, const float* b, const float* c, const float* d,
                       const float* lambda0, float* out, long long N, long long T,
                       cudaStream_t stream, long long wait_ns);

// Each translation unit that launches kernels with bounded waits owns one
// device error word; these read-and-clear it on the current device.
cudaError_t diag_take_device_error(int* status);
cudaError_t mobius_take_device_error(int* status);

// Number of SMs of the current device (cached per device).
int sm_count();

// Maps a CUDA error to a status (KDN_OK on cudaSuccess, KDN_ERR_ALLOC on
// memory allocation errors, KDN_ERR_CUDA otherwise).
kdn_status from_cuda(cudaError_t e);

}  // namespace kdn
