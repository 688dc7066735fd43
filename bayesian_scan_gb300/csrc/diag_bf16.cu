// diag_bf16.cu -- diagonal-scan kernels for bf16 inputs (instantiations of
// diag_impl.cuh).
#include "diag_impl.cuh"

namespace kdn {

kdn_status diag_launch_bf16(const DiagArgs& a, cudaStream_t stream, long long wait_ns) {
    return diag::launch_any<__nv_bfloat16>(a, stream, wait_ns);
}

kdn_status diag_plan_bf16(const DiagArgs& a, int* parts, int* kernels, size_t* scratch) {
    diag::Plan pl;
    const kdn_status s = diag::plan_any<__nv_bfloat16>(a, &pl);
    if (s == KDN_OK) {
        *parts = pl.P;
        *kernels = pl.kernels;
        *scratch = pl.scratch;
    }
    return s;
}

cudaError_t diag_take_device_error_bf16(int* status) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, diag::g_diag_error, sizeof(int));
    if (e == cudaSuccess && v != 0) e = cudaMemcpyToSymbol(diag::g_diag_error, &zero, sizeof(int));
    *status = v;
    return e;
}

}  // namespace kdn
