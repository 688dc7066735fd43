// diag_step.cu -- one token of the diagonal metaplastic update for a batch of
// heads whose (mu, I) state lives in device memory (batched decoding): the
// same equations as the scan ("Learning to Remember, Learn, and Forget in
// Attention-Based Models", Metodologia 1-2; readout as in "Kalman Linear
// Attention (KLA)", Metodologia 1), for T = 1, with the state read and
// overwritten in place:
//     alpha = exp(-A d)
//     I'  = alpha I + (1 - alpha) I_prior + beta_i k_j^2
//     mu' = (alpha I mu + beta_i v_i k_j) / I'        (= alpha (I/I') mu + beta v k / I')
//     o_i = sum_j mu'_ij q_j
// Every state element is read once (mu, I: 8 bytes) and written once: the
// step is bound by HBM bandwidth (16 bytes and ~10 FLOP per element), so the
// division is a correctly rounded one.
//
// Layout: a warp owns one or more whole state rows (d_k / 4 lanes per row);
// a lane owns 4 consecutive columns, loaded and stored as 16-byte vectors;
// the row sums of the readout are warp-shuffle reductions over the lanes of
// a row.  One row group per warp, grid-stride over all rows of all heads.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kdn.h"
#include "kdn_internal.h"

namespace kdn {
namespace {

constexpr float STEP_LOG2E = 1.4426950408889634f;
constexpr int STEP_THREADS = 256;

template <typename TIn>
__device__ __forceinline__ float in_f32(const TIn* p, long long i);
template <>
__device__ __forceinline__ float in_f32<float>(const float* p, long long i) { return __ldg(p + i); }
template <>
__device__ __forceinline__ float in_f32<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
    return __bfloat162float(p[i]);
}

// DK columns per row, 4 per lane: LPR = DK / 4 lanes per row (4..32), RPW =
// 32 / LPR rows per warp; UNR row groups per warp and iteration, whose state
// loads are all issued before any arithmetic (more bytes in flight per warp).
constexpr int STEP_UNR = 2;

template <int DK, typename TIn>
__global__ void __launch_bounds__(STEP_THREADS, 4)
diag_step_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                 const TIn* __restrict__ beta, const TIn* __restrict__ d, const float* __restrict__ A,
                 float I_prior, float* __restrict__ state, float* __restrict__ out, long long BH,
                 int H, int dv) {
    constexpr int LPR = DK / 4, RPW = 32 / LPR;
    const long long S = static_cast<long long>(dv) * DK;
    float* mu_s = state;
    float* I_s = state + BH * S;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, col = (lane % LPR) * 4;
    const long long rows = BH * dv;
    const long long warps = static_cast<long long>(gridDim.x) * (STEP_THREADS / 32);
    const long long w0 = static_cast<long long>(blockIdx.x) * (STEP_THREADS / 32) + (threadIdx.x >> 5);
    for (long long rg = w0 * RPW * STEP_UNR; rg < rows; rg += warps * RPW * STEP_UNR) {
        long long row[STEP_UNR], e[STEP_UNR];
        bool valid[STEP_UNR];
        float4 m4[STEP_UNR], i4[STEP_UNR];
#pragma unroll
        for (int u = 0; u < STEP_UNR; ++u) {
            row[u] = rg + u * RPW + sub;                      // global state row (head, i)
            valid[u] = row[u] < rows;
            const long long bh = valid[u] ? row[u] / dv : 0;
            e[u] = bh * S + (row[u] - bh * dv) * DK + col;
            if (valid[u]) {
                m4[u] = __ldcs(reinterpret_cast<const float4*>(mu_s + e[u]));
                i4[u] = __ldcs(reinterpret_cast<const float4*>(I_s + e[u]));
            }
        }
#pragma unroll
        for (int u = 0; u < STEP_UNR; ++u) {
            float part = 0.f;
            const long long bh = valid[u] ? row[u] / dv : 0;
            const int i = valid[u] ? static_cast<int>(row[u] - bh * dv) : 0;
            if (valid[u]) {
                const float alpha = exp2f(-A[bh % H] * in_f32(d, bh) * STEP_LOG2E);
                const float b = in_f32(beta, bh * dv + i), bv = b * in_f32(v, bh * dv + i);
                const float mu[4] = {m4[u].x, m4[u].y, m4[u].z, m4[u].w};
                const float Iv[4] = {i4[u].x, i4[u].y, i4[u].z, i4[u].w};
                float mo[4], io[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float kj = in_f32(k, bh * DK + col + c), qj = in_f32(q, bh * DK + col + c);
                    const float In = alpha * Iv[c] + (1.f - alpha) * I_prior + b * (kj * kj);
                    mo[c] = (alpha * Iv[c] * mu[c] + bv * kj) / In;
                    io[c] = In;
                    part += mo[c] * qj;
                }
                __stcs(reinterpret_cast<float4*>(mu_s + e[u]), make_float4(mo[0], mo[1], mo[2], mo[3]));
                __stcs(reinterpret_cast<float4*>(I_s + e[u]), make_float4(io[0], io[1], io[2], io[3]));
            }
            // row sum over the LPR lanes of the row (an aligned group of the warp)
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if (valid[u] && lane % LPR == 0) out[bh * dv + i] = part;
        }
    }
}

template <int DK, typename TIn>
cudaError_t launch_step(const void* q, const void* k, const void* v, const void* beta, const void* d,
                        const float* A, float I_prior, float* state, float* out, long long BH, int H,
                        int dv, cudaStream_t st) {
    constexpr int RPW = 32 / (DK / 4);
    const long long rows = BH * dv;
    const long long warps_needed = (rows + RPW * STEP_UNR - 1) / (RPW * STEP_UNR);
    long long blocks = (warps_needed + (STEP_THREADS / 32) - 1) / (STEP_THREADS / 32);
    const long long cap = static_cast<long long>(sm_count()) * 16;   // grid-stride beyond this
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    diag_step_kernel<DK, TIn><<<static_cast<unsigned>(blocks), STEP_THREADS, 0, st>>>(
        static_cast<const TIn*>(q), static_cast<const TIn*>(k), static_cast<const TIn*>(v),
        static_cast<const TIn*>(beta), static_cast<const TIn*>(d), A, I_prior, state, out, BH, H, dv);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t dispatch_step(int dk, const void* q, const void* k, const void* v, const void* beta,
                          const void* d, const float* A, float I_prior, float* state, float* out,
                          long long BH, int H, int dv, cudaStream_t st) {
    switch (dk) {
        case 16: return launch_step<16, TIn>(q, k, v, beta, d, A, I_prior, state, out, BH, H, dv, st);
        case 32: return launch_step<32, TIn>(q, k, v, beta, d, A, I_prior, state, out, BH, H, dv, st);
        case 64: return launch_step<64, TIn>(q, k, v, beta, d, A, I_prior, state, out, BH, H, dv, st);
        default: return launch_step<128, TIn>(q, k, v, beta, d, A, I_prior, state, out, BH, H, dv, st);
    }
}

}  // namespace

kdn_status diag_step_launch(const void* q, const void* k, const void* v, const void* beta,
                            const void* d, const float* A, float I_prior, float* state, float* out,
                            int B, int H, int dk, int dv, kdn_dtype dtype, cudaStream_t st) {
    const long long BH = static_cast<long long>(B) * H;
    const cudaError_t e =
        dtype == KDN_BF16
            ? dispatch_step<__nv_bfloat16>(dk, q, k, v, beta, d, A, I_prior, state, out, BH, H, dv, st)
            : dispatch_step<float>(dk, q, k, v, beta, d, A, I_prior, state, out, BH, H, dv, st);
    return from_cuda(e);
}

}  // namespace kdn
