// diag_bwd.cu -- backward pass of the diagonal metaplastic scan (the pages'
// kernels exist "for efficient GPU training": "Learning to Remember, Learn,
// and Forget in Attention-Based Models", Contributi Chiave; the forward
// update is that page's Metodologia 2, the readout "Kalman Linear Attention
// (KLA)", Metodologia 1).
//
// What is computed.  For the scalar L = sum dout.o + sum dmu_T.mu_T +
// sum dI_T.I_T of one forward call, the gradients with respect to q, k, v,
// beta, d, A and the initial state (mu_0, I_0).  In the information form
// (J = I - I_prior, eta = I mu) the forward state is two linear recurrences,
//     J_t = alpha_t J_{t-1} + beta_i k_j^2,   eta_t = alpha_t eta_{t-1} + beta_i v_i k_j,
// read out through mu_t = eta_t / (J_t + I_prior), o_t[i] = sum_j mu_t[i][j] q_j.
// Their adjoints GJ, GE (total derivatives of L with respect to J_t, eta_t)
// run backwards in time, per state element:
//     r = 1 / (J_t + I_prior),  mu = eta_t r,  a = dout_i q_j r
//     GE_t = alpha_{t+1} GE_{t+1} + a
//     GJ_t = alpha_{t+1} GJ_{t+1} - a mu
// (at t = T the carried terms are the final-state gradients dmu_T r and
// dI_T - dmu_T mu r).  Token t's input gradients are sums over the state:
//     dq_j    = sum_i dout_i mu_ij
//     dk_j    = 2 k_j sum_i GJ_ij beta_i + sum_i GE_ij beta_i v_i
//     dbeta_i = sum_j GJ_ij k_j^2 + v_i sum_j GE_ij k_j,   dv_i = beta_i sum_j GE_ij k_j
//     dL/dalpha_t = sum_ij (GJ_t J_{t-1} + GE_t eta_{t-1})
// (taken with the previous token's state, so that no difference of large
// numbers appears when alpha_t is tiny), and
//     dd_t = -A alpha_t dL/dalpha_t,   dA = -sum_t d_t alpha_t dL/dalpha_t,
// and after the first token the adjoints alpha_1 (GJ, GE) give
//     dI_0 = GJ + GE mu_0,   dmu_0 = GE I_0.
//
// How.  The adjoint sweep needs every forward state in reverse order.  A CTA
// owns all d_v rows of a head and a block of CWB (<= 32) key columns: 16
// elements (4 rows x 4 columns) per thread, so all column sums of a token
// (dq, dk) finish inside the CTA and the row sums leave it as CWB-column
// partials.  The CTA first runs the forward update over the whole sequence,
// storing its tile's state every C = 8 tokens (a checkpoint) in device
// memory; it then walks the chunks backwards: load the chunk's checkpoint,
// re-run the chunk's C forward steps keeping each token's state in tensor
// memory (TMEM: 512 columns x 128 lanes = 8 tokens x 32 words per thread,
// written with tcgen05.st, read back with tcgen05.ld), and take the C adjoint
// steps from the last token down.  Inputs, checkpoints and dout of the next
// chunk are brought into shared memory by cp.async while the current chunk
// computes.  Column sums go through warp shuffles (a halving transpose-
// reduction), row sums and the alpha sums through shared memory once per
// chunk.  The alpha sum of token t+1 is formed in the step of token t (whose
// state is token t+1's previous state), before the adjoints move on.  A
// second kernel adds the column blocks' partials and forms dbeta, dv, dd, and
// a third sums dA over the batch and the tokens (deterministic order).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kdn.h"
#include "kdn_device.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace bwd {
namespace {

constexpr int C = 8;             // tokens per chunk (TMEM history depth)
constexpr int MAX_THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MIN_SMEM = 120 * 1024;   // keeps one CTA per SM (the CTA owns all of TMEM)
constexpr unsigned FULL = 0xffffffffu;

struct Args {
    const void* q;
    const void* k;
    const void* v;
    const void* beta;
    const void* d;
    const float* A;
    float Ip;
    const float* I0;
    const float* mu0;
    const float* dout;
    const float* dfinal;   // [2,BH,dv,dk] (dmu_T, dI_T) or null
    float* gq;
    float* gk;
    float* dinit;          // [2,BH,dv,dk] (dmu_0, dI_0) or null
    float* ckpt;           // [BH*NCB][nC][32*NT]
    float* prow;           // [NCB][BH*T][2*dv]
    float* pD;             // [NCB][BH*T]  partial dL/dalpha_t
    long long BH;
    int H, T, dk, dv, cwb, ncb, nt, nC;
};

// Shared-memory carve-up of one CTA (byte offsets, all 16-byte aligned).
struct Layout {
    int s_k, s_kk, s_q, s_b, s_bv, s_al;           // converted chunk inputs (fp32)
    int raw[2];                                     // raw chunk buffers (cp.async targets)
    int r_k, r_q, r_b, r_v, r_do, r_ck;             // offsets inside a raw buffer
    int s_row, s_dq, s_dk, s_D, holder;
    int total;
};

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline Layout make_layout(int dv, int cwb, int nt, int es) {
    Layout L{};
    int o = 0;
    L.s_k = o;  o += align16(C * cwb * 4);
    L.s_kk = o; o += align16(C * cwb * 4);
    L.s_q = o;  o += align16(C * cwb * 4);
    L.s_b = o;  o += align16(C * dv * 4);
    L.s_bv = o; o += align16(C * dv * 4);
    L.s_al = o; o += align16(C * 4);
    int r = 0;
    L.r_k = r;  r += align16(C * cwb * es);
    L.r_q = r;  r += align16(C * cwb * es);
    L.r_b = r;  r += align16(C * dv * es);
    L.r_v = r;  r += align16(C * dv * es);
    L.r_do = r; r += align16(C * dv * 4);
    L.r_ck = r; r += align16(32 * nt * 4);
    L.raw[0] = o; o += r;
    L.raw[1] = o; o += r;
    L.s_row = o; o += align16(C * 2 * (cwb / 4) * dv * 4);
    L.s_dq = o;  o += align16(C * cwb * 4);
    L.s_dk = o;  o += align16(C * cwb * 4);
    L.s_D = o;   o += align16(C * (MAX_THREADS / 32) * 4);
    L.holder = o; o += 16;
    L.total = o < MIN_SMEM ? MIN_SMEM : o;
    return L;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <typename TIn>
__device__ __forceinline__ float to_f(TIn x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename TIn>
__device__ __forceinline__ float load_in(const TIn* p) { return to_f<TIn>(*p); }

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// TMEM store / load of 32 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float v[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
        "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
        "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
        "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Issue the cp.async copies of chunk c (tokens [c*C, c*C + n)) into raw
// buffer `rb`: the CTA's k (and q) column block, beta, v (and dout) rows and,
// in the backward sweep, the chunk's checkpoint.
template <typename TIn>
__device__ void issue_chunk(const Args& p, unsigned char* rb, const Layout& L, long long bh, int cb,
                            int c, int n, bool bwd, int tid) {
    const int es = sizeof(TIn);
    const long long tok0 = bh * p.T + static_cast<long long>(c) * C;
    // column-block slices: n rows of cwb*es bytes
    const int kp = p.cwb * es / 16;                      // 16-byte pieces per token row
    const char* kg = static_cast<const char*>(p.k) + (tok0 * p.dk + cb * p.cwb) * es;
    const char* qg = static_cast<const char*>(p.q) + (tok0 * p.dk + cb * p.cwb) * es;
    for (int i = tid; i < n * kp; i += p.nt) {
        const int s = i / kp, w = i % kp;
        cp_async16(rb + L.r_k + s * p.cwb * es + w * 16, kg + static_cast<long long>(s) * p.dk * es + w * 16);
        if (bwd)
            cp_async16(rb + L.r_q + s * p.cwb * es + w * 16, qg + static_cast<long long>(s) * p.dk * es + w * 16);
    }
    // rows: n * dv contiguous elements
    const int rp = n * p.dv * es / 16;
    const char* bg = static_cast<const char*>(p.beta) + tok0 * p.dv * es;
    const char* vg = static_cast<const char*>(p.v) + tok0 * p.dv * es;
    for (int i = tid; i < rp; i += p.nt) {
        cp_async16(rb + L.r_b + i * 16, bg + i * 16);
        cp_async16(rb + L.r_v + i * 16, vg + i * 16);
    }
    if (bwd) {
        const int op = n * p.dv * 4 / 16;
        const char* og = reinterpret_cast<const char*>(p.dout + tok0 * p.dv);
        for (int i = tid; i < op; i += p.nt) cp_async16(rb + L.r_do + i * 16, og + i * 16);
        const char* cg = reinterpret_cast<const char*>(
            p.ckpt + ((bh * p.ncb + cb) * p.nC + c) * 32LL * p.nt);
        for (int i = tid; i < 32 * p.nt / 4; i += p.nt) cp_async16(rb + L.r_ck + i * 16, cg + i * 16);
    }
    cp_async_commit();
}

// Converts the raw chunk inputs to fp32 (k, k^2, q, beta, beta v, alpha).
template <typename TIn>
__device__ void convert_chunk(const Args& p, unsigned char* sm, const unsigned char* rb,
                              const Layout& L, int n, bool bwd, float alpha, int tid) {
    const TIn* rk = reinterpret_cast<const TIn*>(rb + L.r_k);
    const TIn* rq = reinterpret_cast<const TIn*>(rb + L.r_q);
    const TIn* rbt = reinterpret_cast<const TIn*>(rb + L.r_b);
    const TIn* rv = reinterpret_cast<const TIn*>(rb + L.r_v);
    float* sk = reinterpret_cast<float*>(sm + L.s_k);
    float* skk = reinterpret_cast<float*>(sm + L.s_kk);
    float* sq = reinterpret_cast<float*>(sm + L.s_q);
    float* sb = reinterpret_cast<float*>(sm + L.s_b);
    float* sbv = reinterpret_cast<float*>(sm + L.s_bv);
    for (int i = tid; i < n * p.cwb; i += p.nt) {
        const float kv = to_f<TIn>(rk[i]);
        sk[i] = kv;
        skk[i] = kv * kv;
        if (bwd) sq[i] = to_f<TIn>(rq[i]);
    }
    for (int i = tid; i < n * p.dv; i += p.nt) {
        const float b = to_f<TIn>(rbt[i]);
        sb[i] = b;
        sbv[i] = b * to_f<TIn>(rv[i]);
    }
    if (tid < n) reinterpret_cast<float*>(sm + L.s_al)[tid] = alpha;
}

// alpha of token t of head bh (t < T), from d and A.
template <typename TIn>
__device__ __forceinline__ float alpha_of(const Args& p, long long bh, long long t) {
    const float dd = load_in<TIn>(static_cast<const TIn*>(p.d) + bh * p.T + t);
    return expf(-p.A[bh % p.H] * dd);
}

// Sum over the NR lanes sharing a column quad of 12 values (3 per column:
// dq, dk-from-J, dk-from-eta partials).  Two halving levels leave each lane
// 3 values that are then summed over the remaining levels; afterwards a lane
// holds the totals of column g = 2 [rq & NR/2] + [rq & NR/4].
__device__ __forceinline__ void column_reduce(float v[12], int NR, int rq) {
    int o = NR >> 1;
    bool up = (rq & o) != 0;
#pragma unroll
    for (int m = 0; m < 6; ++m) {
        const float send = up ? v[m] : v[m + 6];
        const float keep = up ? v[m + 6] : v[m];
        v[m] = keep + __shfl_xor_sync(FULL, send, o);
    }
    o >>= 1;
    up = (rq & o) != 0;
#pragma unroll
    for (int m = 0; m < 3; ++m) {
        const float send = up ? v[m] : v[m + 3];
        const float keep = up ? v[m + 3] : v[m];
        v[m] = keep + __shfl_xor_sync(FULL, send, o);
    }
    for (o >>= 1; o > 0; o >>= 1) {
#pragma unroll
        for (int m = 0; m < 3; ++m) v[m] += __shfl_xor_sync(FULL, v[m], o);
    }
}

template <typename TIn>
__global__ void __launch_bounds__(MAX_THREADS, 1) diag_bwd_kernel(const Args p) {
    extern __shared__ __align__(128) unsigned char sm[];
    const int es = sizeof(TIn);
    const Layout L = make_layout(p.dv, p.cwb, p.nt, es);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long bh = blockIdx.x / p.ncb;
    const int cb = blockIdx.x % p.ncb;
    const int NR = p.dv / 4, NCQ = p.cwb / 4;
    const bool valid = tid < NR * NCQ;
    const int rq = valid ? tid % NR : 0, cq = valid ? tid / NR : 0;
    const int row0 = 4 * rq, col0 = 4 * cq;                    // inside the tile
    const long long S = static_cast<long long>(p.dv) * p.dk;
    const float Ip = p.Ip;
    uint32_t* holder = reinterpret_cast<uint32_t*>(sm + L.holder);

    if (warp == 0) tmem_alloc(holder, TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = *holder;
    const uint32_t tlane = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                           static_cast<uint32_t>((warp >> 2) * 256);

    // ---- initial state of the tile: J = I_0 - I_prior, E = I_0 mu_0 -------
    float2 J[4][2], E[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const long long off = bh * S + static_cast<long long>(row0 + r) * p.dk + cb * p.cwb + col0;
        float4 i4 = make_float4(Ip, Ip, Ip, Ip), m4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid && p.I0) i4 = *reinterpret_cast<const float4*>(p.I0 + off);
        if (valid && p.mu0) m4 = *reinterpret_cast<const float4*>(p.mu0 + off);
        J[r][0] = make_float2(i4.x - Ip, i4.y - Ip);
        J[r][1] = make_float2(i4.z - Ip, i4.w - Ip);
        E[r][0] = make_float2(i4.x * m4.x, i4.y * m4.y);
        E[r][1] = make_float2(i4.z * m4.z, i4.w * m4.w);
    }

    auto raw = [&](int i) { return sm + (i ? L.raw[1] : L.raw[0]); };
    const float* sk = reinterpret_cast<const float*>(sm + L.s_k);
    const float* skk = reinterpret_cast<const float*>(sm + L.s_kk);
    const float* sq = reinterpret_cast<const float*>(sm + L.s_q);
    const float* sb = reinterpret_cast<const float*>(sm + L.s_b);
    const float* sbv = reinterpret_cast<const float*>(sm + L.s_bv);
    const float* sal = reinterpret_cast<const float*>(sm + L.s_al);
    float* ckpt_cta = p.ckpt + (bh * p.ncb + cb) * static_cast<long long>(p.nC) * 32 * p.nt;
    const int nC = p.nC;
    auto ntok = [&](int c) { return min(C, p.T - c * C); };

    // ---- forward sweep: checkpoints every C tokens -------------------------
    float dreg = 1.f;   // alpha of token (chunk start + tid), prefetched
    if (nC > 0) {
        issue_chunk<TIn>(p, raw(0), L, bh, cb, 0, ntok(0), false, tid);
        if (tid < ntok(0)) dreg = alpha_of<TIn>(p, bh, tid);
    }
    for (int c = 0; c < nC; ++c) {
        const int n = ntok(c);
        // checkpoint: the tile's state before chunk c
        {
            float* dst = ckpt_cta + static_cast<long long>(c) * 32 * p.nt;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                reinterpret_cast<float4*>(dst)[(2 * r) * p.nt + tid] =
                    make_float4(J[r][0].x, J[r][0].y, J[r][1].x, J[r][1].y);
                reinterpret_cast<float4*>(dst)[(2 * r + 1) * p.nt + tid] =
                    make_float4(E[r][0].x, E[r][0].y, E[r][1].x, E[r][1].y);
            }
        }
        cp_async_wait_all();
        __syncthreads();   // chunk c landed; chunk c-1's compute finished
        convert_chunk<TIn>(p, sm, raw(c & 1), L, n, false, dreg, tid);
        if (c + 1 < nC) {
            issue_chunk<TIn>(p, raw((c + 1) & 1), L, bh, cb, c + 1, ntok(c + 1), false, tid);
            if (tid < ntok(c + 1)) dreg = alpha_of<TIn>(p, bh, static_cast<long long>(c + 1) * C + tid);
        }
        __syncthreads();
        for (int s = 0; s < n; ++s) {
            const float2 al = f2(sal[s]);
            const float4 b4 = *reinterpret_cast<const float4*>(sb + s * p.dv + row0);
            const float4 v4 = *reinterpret_cast<const float4*>(sbv + s * p.dv + row0);
            const float4 k4 = *reinterpret_cast<const float4*>(sk + s * p.cwb + col0);
            const float4 kk4 = *reinterpret_cast<const float4*>(skk + s * p.cwb + col0);
            const float bet[4] = {b4.x, b4.y, b4.z, b4.w}, bvv[4] = {v4.x, v4.y, v4.z, v4.w};
            const float2 kf[2] = {make_float2(k4.x, k4.y), make_float2(k4.z, k4.w)};
            const float2 kq[2] = {make_float2(kk4.x, kk4.y), make_float2(kk4.z, kk4.w)};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    J[r][c2] = __ffma2_rn(al, J[r][c2], __fmul2_rn(f2(bet[r]), kq[c2]));
                    E[r][c2] = __ffma2_rn(al, E[r][c2], __fmul2_rn(f2(bvv[r]), kf[c2]));
                }
        }
    }
    // checkpoints written by other threads are read back through cp.async
    __threadfence();
    __syncthreads();

    // ---- adjoints at t = T from the final-state gradients ------------------
    float2 GJ[4][2], GE[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const long long off = bh * S + static_cast<long long>(row0 + r) * p.dk + cb * p.cwb + col0;
        float4 dm = make_float4(0.f, 0.f, 0.f, 0.f), di = dm;
        if (valid && p.dfinal) {
            dm = *reinterpret_cast<const float4*>(p.dfinal + off);
            di = *reinterpret_cast<const float4*>(p.dfinal + p.BH * S + off);
        }
        const float dmv[4] = {dm.x, dm.y, dm.z, dm.w}, div[4] = {di.x, di.y, di.z, di.w};
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            const float2 den = __fadd2_rn(J[r][c2], f2(Ip));
            const float2 rr = make_float2(1.f / den.x, 1.f / den.y);
            const float2 mu = __fmul2_rn(E[r][c2], rr);
            const float2 dmu = make_float2(dmv[2 * c2], dmv[2 * c2 + 1]);
            const float2 a = __fmul2_rn(dmu, rr);
            GE[r][c2] = a;
            GJ[r][c2] = make_float2(div[2 * c2] - a.x * mu.x, div[2 * c2 + 1] - a.y * mu.y);
        }
    }

    // ---- backward sweep over the chunks, last first ------------------------
    float* s_row = reinterpret_cast<float*>(sm + L.s_row);
    float* s_dq = reinterpret_cast<float*>(sm + L.s_dq);
    float* s_dk = reinterpret_cast<float*>(sm + L.s_dk);
    float* s_D = reinterpret_cast<float*>(sm + L.s_D);
    const int nwarps = p.nt / 32;
    const int o1 = NR >> 1, o2 = NR >> 2;
    const int g = 2 * ((rq & o1) ? 1 : 0) + ((rq & o2) ? 1 : 0);
    const bool col_writer = valid && (rq & (o2 - 1)) == 0;
    float alpha_next = 1.f;   // alpha of the token after the one being processed
    if (nC > 0) {
        const int c = nC - 1;
        issue_chunk<TIn>(p, raw(c & 1), L, bh, cb, c, ntok(c), true, tid);
        if (tid < ntok(c)) dreg = alpha_of<TIn>(p, bh, static_cast<long long>(c) * C + tid);
    }
    for (int c = nC - 1; c >= 0; --c) {
        const int n = ntok(c);
        const long long t0 = static_cast<long long>(c) * C;
        cp_async_wait_all();
        __syncthreads();   // chunk c landed; the previous chunk's epilogue finished
        unsigned char* rb = raw(c & 1);
        convert_chunk<TIn>(p, sm, rb, L, n, true, dreg, tid);
        if (c > 0) {
            issue_chunk<TIn>(p, raw((c - 1) & 1), L, bh, cb, c - 1, C, true, tid);
            if (tid < C) dreg = alpha_of<TIn>(p, bh, t0 - C + tid);
        }
        // the chunk's checkpoint
        {
            const float4* src = reinterpret_cast<const float4*>(rb + L.r_ck);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float4 a = src[(2 * r) * p.nt + tid], b = src[(2 * r + 1) * p.nt + tid];
                J[r][0] = make_float2(a.x, a.y);
                J[r][1] = make_float2(a.z, a.w);
                E[r][0] = make_float2(b.x, b.y);
                E[r][1] = make_float2(b.z, b.w);
            }
        }
        __syncthreads();   // converted inputs visible
        // forward again through the chunk; token s's state goes to TMEM slot s
        for (int s = 0; s < n; ++s) {
            const float2 al = f2(sal[s]);
            const float4 b4 = *reinterpret_cast<const float4*>(sb + s * p.dv + row0);
            const float4 v4 = *reinterpret_cast<const float4*>(sbv + s * p.dv + row0);
            const float4 k4 = *reinterpret_cast<const float4*>(sk + s * p.cwb + col0);
            const float4 kk4 = *reinterpret_cast<const float4*>(skk + s * p.cwb + col0);
            const float bet[4] = {b4.x, b4.y, b4.z, b4.w}, bvv[4] = {v4.x, v4.y, v4.z, v4.w};
            const float2 kf[2] = {make_float2(k4.x, k4.y), make_float2(k4.z, k4.w)};
            const float2 kq[2] = {make_float2(kk4.x, kk4.y), make_float2(kk4.z, kk4.w)};
            float st[32];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    J[r][c2] = __ffma2_rn(al, J[r][c2], __fmul2_rn(f2(bet[r]), kq[c2]));
                    E[r][c2] = __ffma2_rn(al, E[r][c2], __fmul2_rn(f2(bvv[r]), kf[c2]));
                    st[4 * r + 2 * c2] = J[r][c2].x;
                    st[4 * r + 2 * c2 + 1] = J[r][c2].y;
                    st[16 + 4 * r + 2 * c2] = E[r][c2].x;
                    st[16 + 4 * r + 2 * c2 + 1] = E[r][c2].y;
                }
            tmem_st32(tlane + static_cast<uint32_t>(s * 32), st);
        }
        tmem_wait_st();
        const float* sdo = reinterpret_cast<const float*>(rb + L.r_do);
        for (int s = n - 1; s >= 0; --s) {
            float st[32];
            tmem_ld32(tlane + static_cast<uint32_t>(s * 32), st);
            const float2 ap = f2(alpha_next);
            const float4 b4 = *reinterpret_cast<const float4*>(sb + s * p.dv + row0);
            const float4 v4 = *reinterpret_cast<const float4*>(sbv + s * p.dv + row0);
            const float4 o4 = *reinterpret_cast<const float4*>(sdo + s * p.dv + row0);
            const float4 k4 = *reinterpret_cast<const float4*>(sk + s * p.cwb + col0);
            const float4 kk4 = *reinterpret_cast<const float4*>(skk + s * p.cwb + col0);
            const float4 q4 = *reinterpret_cast<const float4*>(sq + s * p.cwb + col0);
            const float bet[4] = {b4.x, b4.y, b4.z, b4.w}, bvv[4] = {v4.x, v4.y, v4.z, v4.w};
            const float dov[4] = {o4.x, o4.y, o4.z, o4.w};
            const float2 kf[2] = {make_float2(k4.x, k4.y), make_float2(k4.z, k4.w)};
            const float2 kq[2] = {make_float2(kk4.x, kk4.y), make_float2(kk4.z, kk4.w)};
            const float2 qf[2] = {make_float2(q4.x, q4.y), make_float2(q4.z, q4.w)};
            float2 cdq[2], cck[2], cce[2], rsb[4], rse[4], dacc = make_float2(0.f, 0.f);
            // dL/dalpha of token t+1: its adjoints (not yet moved) against this
            // token's state, the previous state of token t+1
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) cdq[c2] = cck[c2] = cce[c2] = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                rsb[r] = rse[r] = make_float2(0.f, 0.f);
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const float2 Jt = make_float2(st[4 * r + 2 * c2], st[4 * r + 2 * c2 + 1]);
                    const float2 Et = make_float2(st[16 + 4 * r + 2 * c2], st[16 + 4 * r + 2 * c2 + 1]);
                    const float2 den = __fadd2_rn(Jt, f2(Ip));
                    const float2 rr = make_float2(rcp_approx(den.x), rcp_approx(den.y));
                    const float2 mu = __fmul2_rn(Et, rr);
                    const float2 a = __fmul2_rn(__fmul2_rn(f2(dov[r]), qf[c2]), rr);
                    dacc = __ffma2_rn(GJ[r][c2], Jt, dacc);
                    dacc = __ffma2_rn(GE[r][c2], Et, dacc);
                    GE[r][c2] = __ffma2_rn(ap, GE[r][c2], a);
                    const float2 am = __fmul2_rn(a, mu);
                    GJ[r][c2] = __ffma2_rn(ap, GJ[r][c2], make_float2(-am.x, -am.y));
                    cdq[c2] = __ffma2_rn(f2(dov[r]), mu, cdq[c2]);
                    rsb[r] = __ffma2_rn(GJ[r][c2], kq[c2], rsb[r]);
                    rse[r] = __ffma2_rn(GE[r][c2], kf[c2], rse[r]);
                    cck[c2] = __ffma2_rn(f2(bet[r]), GJ[r][c2], cck[c2]);
                    cce[c2] = __ffma2_rn(f2(bvv[r]), GE[r][c2], cce[c2]);
                }
            }
            alpha_next = sal[s];
            // column sums over the d_v rows: lanes sharing the column quad
            float cv[12];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                cv[3 * (2 * c2)] = cdq[c2].x;
                cv[3 * (2 * c2) + 1] = cck[c2].x;
                cv[3 * (2 * c2) + 2] = cce[c2].x;
                cv[3 * (2 * c2 + 1)] = cdq[c2].y;
                cv[3 * (2 * c2 + 1) + 1] = cck[c2].y;
                cv[3 * (2 * c2 + 1) + 2] = cce[c2].y;
            }
            column_reduce(cv, NR, rq);
            if (col_writer) {
                const int j = col0 + g;
                s_dq[s * p.cwb + j] = cv[0];
                s_dk[s * p.cwb + j] = 2.f * sk[s * p.cwb + j] * cv[1] + cv[2];
            }
            // row partials over this thread's 4 columns
            if (valid) {
                float* rowp = s_row + static_cast<long long>(s) * 2 * NCQ * p.dv;
                *reinterpret_cast<float4*>(rowp + cq * p.dv + row0) =
                    make_float4(rsb[0].x + rsb[0].y, rsb[1].x + rsb[1].y, rsb[2].x + rsb[2].y,
                                rsb[3].x + rsb[3].y);
                *reinterpret_cast<float4*>(rowp + (NCQ + cq) * p.dv + row0) =
                    make_float4(rse[0].x + rse[0].y, rse[1].x + rse[1].y, rse[2].x + rse[2].y,
                                rse[3].x + rse[3].y);
            }
            float dsum = valid ? dacc.x + dacc.y : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(FULL, dsum, o);
            if (lane == 0) s_D[s * (MAX_THREADS / 32) + warp] = dsum;
        }
        __syncthreads();   // the chunk's partials are complete
        // ---- epilogue of the chunk: row partials, D partials, dq, dk -------
        {
            const long long tokbase = bh * p.T + t0;
            float* prow = p.prow + (static_cast<long long>(cb) * p.BH * p.T + tokbase) * 2 * p.dv;
            for (int i = tid; i < n * 2 * p.dv; i += p.nt) {
                const int s = i / (2 * p.dv), rem = i % (2 * p.dv), qi = rem / p.dv, row = rem % p.dv;
                const float* src = s_row + static_cast<long long>(s) * 2 * NCQ * p.dv + qi * NCQ * p.dv + row;
                float acc = 0.f;
                for (int x = 0; x < NCQ; ++x) acc += src[x * p.dv];
                prow[i] = acc;
            }
            // slot s holds token t0 + s + 1 (none after the last token)
            if (tid < n && t0 + tid + 1 < p.T) {
                float acc = 0.f;
                for (int w = 0; w < nwarps; ++w) acc += s_D[tid * (MAX_THREADS / 32) + w];
                p.pD[static_cast<long long>(cb) * p.BH * p.T + tokbase + tid + 1] = acc;
            }
            for (int i = tid; i < n * p.cwb; i += p.nt) {
                const int s = i / p.cwb, j = i % p.cwb;
                const long long o = (tokbase + s) * p.dk + cb * p.cwb + j;
                p.gq[o] = s_dq[i];
                p.gk[o] = s_dk[i];
            }
        }
    }

    // ---- token 0's alpha sum and the gradients of the initial state --------
    __syncthreads();   // the last epilogue has read s_D
    {
        const float2 a0 = f2(alpha_next);   // alpha of token 0 (1 when T = 0)
        float dsum = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const long long off = bh * S + static_cast<long long>(row0 + r) * p.dk + cb * p.cwb + col0;
            float4 i4 = make_float4(Ip, Ip, Ip, Ip), m4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (valid && p.I0) i4 = *reinterpret_cast<const float4*>(p.I0 + off);
            if (valid && p.mu0) m4 = *reinterpret_cast<const float4*>(p.mu0 + off);
            // J_0 = I_0 - I_prior, eta_0 = I_0 mu_0
            dsum += GJ[r][0].x * (i4.x - Ip) + GJ[r][0].y * (i4.y - Ip) + GJ[r][1].x * (i4.z - Ip) +
                    GJ[r][1].y * (i4.w - Ip);
            dsum += GE[r][0].x * (i4.x * m4.x) + GE[r][0].y * (i4.y * m4.y) +
                    GE[r][1].x * (i4.z * m4.z) + GE[r][1].y * (i4.w * m4.w);
            if (p.dinit && valid) {
                const float2 gj0 = __fmul2_rn(a0, GJ[r][0]), gj1 = __fmul2_rn(a0, GJ[r][1]);
                const float2 ge0 = __fmul2_rn(a0, GE[r][0]), ge1 = __fmul2_rn(a0, GE[r][1]);
                *reinterpret_cast<float4*>(p.dinit + off) =
                    make_float4(ge0.x * i4.x, ge0.y * i4.y, ge1.x * i4.z, ge1.y * i4.w);
                *reinterpret_cast<float4*>(p.dinit + p.BH * S + off) =
                    make_float4(gj0.x + ge0.x * m4.x, gj0.y + ge0.y * m4.y, gj1.x + ge1.x * m4.z,
                                gj1.y + ge1.y * m4.w);
            }
        }
        if (!valid) dsum = 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(FULL, dsum, o);
        if (lane == 0) s_D[warp] = dsum;
        __syncthreads();
        if (tid == 0 && p.T > 0) {
            float acc = 0.f;
            for (int w = 0; w < nwarps; ++w) acc += s_D[w];
            p.pD[static_cast<long long>(cb) * p.BH * p.T + bh * p.T] = acc;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, TMEM_COLS);
}

// Per (head, token): adds the column blocks' partials and forms dbeta, dv,
// dd = -A alpha dL/dalpha and the token's dA term -d alpha dL/dalpha.  One
// warp per token.
template <typename TIn>
__global__ void __launch_bounds__(256) diag_bwd_finalize_kernel(
    const TIn* __restrict__ v, const TIn* __restrict__ beta, const TIn* __restrict__ d,
    const float* __restrict__ A, const float* __restrict__ prow, const float* __restrict__ pD,
    float* __restrict__ dv_out, float* __restrict__ dbeta, float* __restrict__ dd,
    float* __restrict__ eA, long long BHT, int T, int H, int dv, int ncb) {
    const long long tok = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= BHT) return;
    for (int i = lane; i < dv; i += 32) {
        float sb = 0.f, se = 0.f;
        for (int cb = 0; cb < ncb; ++cb) {
            const float* pr = prow + (static_cast<long long>(cb) * BHT + tok) * 2 * dv;
            sb += pr[i];
            se += pr[dv + i];
        }
        const float b = to_f<TIn>(beta[tok * dv + i]), vv = to_f<TIn>(v[tok * dv + i]);
        dbeta[tok * dv + i] = sb + vv * se;
        dv_out[tok * dv + i] = b * se;
    }
    if (lane == 0) {
        float g_alpha = 0.f;
        for (int cb = 0; cb < ncb; ++cb) g_alpha += pD[static_cast<long long>(cb) * BHT + tok];
        const long long bh = tok / T;
        const float Ah = A[bh % H], dt = to_f<TIn>(d[tok]);
        const float alpha = expf(-Ah * dt);
        dd[tok] = -Ah * alpha * g_alpha;
        eA[tok] = -dt * alpha * g_alpha;
    }
}

// dA_h = sum over b and t of the terms of head h; one CTA per head.
__global__ void __launch_bounds__(256) diag_bwd_dA_kernel(const float* __restrict__ eA,
                                                          float* __restrict__ dA, int B, int H,
                                                          int T) {
    __shared__ float red[256];
    const int h = blockIdx.x;
    float acc = 0.f;
    for (int b = 0; b < B; ++b) {
        const float* e = eA + (static_cast<long long>(b) * H + h) * T;
        for (int t = threadIdx.x; t < T; t += 256) acc += e[t];
    }
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) dA[h] = red[0];
}

template <typename TIn>
kdn_status launch(const DiagBwdArgs& a, cudaStream_t st) {
    const long long BH = static_cast<long long>(a.B) * a.H;
    const int cwb = a.dk < 32 ? a.dk : 32;
    const int ncb = a.dk / cwb;
    const int nta = (a.dv / 4) * (cwb / 4);
    const int nt = nta < 32 ? 32 : nta;
    const int nC = (a.T + C - 1) / C;
    const Layout L = make_layout(a.dv, cwb, nt, static_cast<int>(sizeof(TIn)));
    const size_t ck_bytes = static_cast<size_t>(BH) * ncb * nC * 32 * nt * 4;
    const size_t row_bytes = static_cast<size_t>(ncb) * BH * a.T * 2 * a.dv * 4;
    const size_t pd_bytes = static_cast<size_t>(ncb) * BH * a.T * 4;
    const size_t ea_bytes = static_cast<size_t>(BH) * a.T * 4;
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t total = up(ck_bytes) + up(row_bytes) + up(pd_bytes) + up(ea_bytes);
    void* scratch = nullptr;
    cudaError_t e = cudaSuccess;
    if (total > 0) {
        e = cudaMallocAsync(&scratch, total, st);
        if (e != cudaSuccess) return from_cuda(e);
    }
    unsigned char* base = static_cast<unsigned char*>(scratch);
    Args p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.beta = a.beta; p.d = a.d; p.A = a.A; p.Ip = a.I_prior;
    p.I0 = a.I0; p.mu0 = a.mu0; p.dout = a.grad_out; p.dfinal = a.grad_final_state;
    p.gq = a.grad_q; p.gk = a.grad_k; p.dinit = a.grad_init_state;
    p.ckpt = reinterpret_cast<float*>(base);
    p.prow = reinterpret_cast<float*>(base + up(ck_bytes));
    p.pD = reinterpret_cast<float*>(base + up(ck_bytes) + up(row_bytes));
    float* eA = reinterpret_cast<float*>(base + up(ck_bytes) + up(row_bytes) + up(pd_bytes));
    p.BH = BH; p.H = a.H; p.T = a.T; p.dk = a.dk; p.dv = a.dv; p.cwb = cwb; p.ncb = ncb; p.nt = nt;
    p.nC = nC;
    e = cudaFuncSetAttribute(diag_bwd_kernel<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (e == cudaSuccess) {
        diag_bwd_kernel<TIn><<<static_cast<unsigned>(BH * ncb), nt, L.total, st>>>(p);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && a.T > 0) {
        const long long BHT = BH * a.T;
        diag_bwd_finalize_kernel<TIn><<<static_cast<unsigned>((BHT + 7) / 8), 256, 0, st>>>(
            static_cast<const TIn*>(a.v), static_cast<const TIn*>(a.beta), static_cast<const TIn*>(a.d),
            a.A, p.prow, p.pD, a.grad_v, a.grad_beta, a.grad_d, eA, BHT, a.T, a.H, a.dv, ncb);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && a.grad_A) {
        if (a.T > 0) {
            diag_bwd_dA_kernel<<<a.H, 256, 0, st>>>(eA, a.grad_A, a.B, a.H, a.T);
            e = cudaGetLastError();
        } else {
            e = cudaMemsetAsync(a.grad_A, 0, sizeof(float) * a.H, st);
        }
    }
    if (scratch) {
        const cudaError_t ef = cudaFreeAsync(scratch, st);
        if (e == cudaSuccess) e = ef;
    }
    return from_cuda(e);
}

}  // namespace
}  // namespace bwd

kdn_status diag_bwd_launch(const DiagBwdArgs& a, cudaStream_t st) {
    return a.dtype == KDN_BF16 ? bwd::launch<__nv_bfloat16>(a, st) : bwd::launch<float>(a, st);
}

}  // namespace kdn
