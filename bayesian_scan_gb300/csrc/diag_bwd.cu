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
// owns all d_v rows of a head and a block of CWB (<= 32) key columns: 4
// rows x CPT columns per thread (CPT = 4 for 32-column blocks, 2 for
// 16-column blocks, which then have as many threads as 32-column ones), so
// all column sums of a token (dq, dk) finish inside the CTA and the row sums
// leave it as CWB-column partials.  The CTA first runs the forward update over the whole sequence,
// storing its tile's state every C = 8 tokens (a checkpoint) in device
// memory; it then walks the chunks backwards: load the chunk's checkpoint,
// re-run the chunk's C forward steps keeping each token's state in tensor
// memory (TMEM: 8 tokens x 8 CPT words per thread in its warp's lane
// quarter, written with tcgen05.st, read back with tcgen05.ld), and take the C adjoint
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
#include <mutex>

#include "kdn.h"
#include "kdn_device.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace bwd {
namespace {

constexpr int C = 8;             // tokens per chunk (TMEM history depth)
// Tensor memory and CTAs per SM: a thread's history takes 8 tokens x 8 CPT
// columns of its warp's lane quarter (256 for CPT = 4, 128 for CPT = 2),
// doubled for CTAs of 8 warps (two per quarter).  The shared-memory floors
// keep the CTA count per SM within what tensor memory holds (a CTA past it
// would wait in tcgen05.alloc holding its SM slot).
constexpr int MIN_SMEM_ALONE = 120 * 1024;   // one CTA per SM
constexpr int MIN_SMEM_PAIR = 80 * 1024;     // at most two CTAs per SM
constexpr int MIN_SMEM_QUAD = 48 * 1024;     // at most four CTAs per SM
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
    // per launch (heads bh0 .. bh0 + nbh - 1), indexed by the launch's own heads:
    float* ckpt;           // [nbh*NCB][nC][SW*NT]
    float* prow;           // [NCB][nbh*T][2*dv]
    float* pD;             // [NCB][nbh*T]  partial dL/dalpha_t
    long long BH;          // all heads of the call
    long long bh0, nbh;    // this launch's heads
    int H, T, dk, ncb, nC;
};

__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

// Tile of one CTA: all DV rows x CWB key columns; a thread owns 4 rows x
// CPT columns (NR row quads x NCQ column groups; lanes run over the row
// quads): CPT = 4 for 32-column blocks, 2 for 16-column blocks, whose CTAs
// then have as many warps as the 32-column ones (the few-head calls that
// take 16-column blocks had one warp per scheduler with 4 columns a thread).
template <typename TIn, int DV, int CWB>
struct Tile {
    static constexpr int ES = sizeof(TIn);
    static constexpr int CPT = CWB == 32 ? 4 : 2;
    static constexpr int NR = DV / 4, NCQ = CWB / CPT, NTA = NR * NCQ;
    static constexpr int SW = 8 * CPT;           // state words of a thread per token (J, eta)
    static constexpr int NT = NTA < 32 ? 32 : NTA, NW = NT / 32;
    static_assert(NT <= 256, "at most 8 warps (two per TMEM lane quarter)");
    // shared memory (byte offsets)
    static constexpr int s_k = 0;
    static constexpr int s_kk = s_k + align16(C * CWB * 4);
    static constexpr int s_q = s_kk + align16(C * CWB * 4);
    static constexpr int s_b = s_q + align16(C * CWB * 4);
    static constexpr int s_bv = s_b + align16(C * DV * 4);
    static constexpr int s_al = s_bv + align16(C * DV * 4);
    static constexpr int r_k = 0;                                 // inside a raw buffer
    static constexpr int r_q = r_k + align16(C * CWB * ES);
    static constexpr int r_b = r_q + align16(C * CWB * ES);
    static constexpr int r_v = r_b + align16(C * DV * ES);
    static constexpr int r_do = r_v + align16(C * DV * ES);
    static constexpr int r_ck = r_do + align16(C * DV * 4);
    static constexpr int RAW = r_ck + align16(SW * NT * 4);
    static constexpr int raw0 = s_al + align16(C * 4);
    static constexpr int raw1 = raw0 + RAW;
    static constexpr int s_row = raw1 + RAW;
    static constexpr int s_dq = s_row + align16(C * 2 * NCQ * DV * 4);
    static constexpr int s_dk = s_dq + align16(C * CWB * 4);
    static constexpr int s_D = s_dk + align16(C * CWB * 4);
    static constexpr int holder = s_D + align16(C * NW * 4);
    static constexpr int used = holder + 16;
    // TMEM: C tokens x SW columns of history per thread, in its warp's lane
    // quarter; two warps share a quarter when there are more than four
    static constexpr uint32_t HIST_COLS = C * SW;
    static constexpr uint32_t TMEM_COLS = HIST_COLS * (NT > 128 ? 2 : 1);
    static constexpr int MIN_SMEM = TMEM_COLS == 512 ? MIN_SMEM_ALONE
                                    : TMEM_COLS == 256 ? MIN_SMEM_PAIR : MIN_SMEM_QUAD;
    static constexpr int SMEM = used < MIN_SMEM ? MIN_SMEM : used;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    // The forward sweep stages F1 tokens at a time (several checkpoint
    // intervals per barrier pair): raw k, beta, v in a raw buffer, converted
    // k, k^2, beta, beta v, alpha in the row-partial area (free until the
    // backward sweep).  F1 is the longest of 32, 16, 8 that fits both.
    static constexpr int f1_raw(int f) { return align16(f * CWB * ES) + 2 * align16(f * DV * ES); }
    static constexpr int f1_cvt(int f) { return 2 * align16(f * CWB * 4) + 2 * align16(f * DV * 4) + align16(f * 4); }
    static constexpr int s_row_bytes = align16(C * 2 * NCQ * DV * 4);
    static constexpr int F1 = (f1_raw(32) <= RAW && f1_cvt(32) <= s_row_bytes) ? 32
                              : (f1_raw(16) <= RAW && f1_cvt(16) <= s_row_bytes) ? 16 : C;
    static constexpr int f1_k = 0, f1_b = align16(F1 * CWB * ES), f1_v = f1_b + align16(F1 * DV * ES);
    static constexpr int g_k = (F1 == C) ? s_k : s_row;
    static constexpr int g_kk = (F1 == C) ? s_kk : g_k + align16(F1 * CWB * 4);
    static constexpr int g_b = (F1 == C) ? s_b : g_kk + align16(F1 * CWB * 4);
    static constexpr int g_bv = (F1 == C) ? s_bv : g_b + align16(F1 * DV * 4);
    static constexpr int g_al = (F1 == C) ? s_al : g_bv + align16(F1 * DV * 4);
    static_assert(F1 % C == 0, "a stage holds whole checkpoint intervals");
};

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

// 4 consecutive inputs (16-byte aligned for fp32, 8-byte for bf16) as fp32
template <typename TIn>
__device__ __forceinline__ float4 load4(const TIn* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// CPT consecutive fp32 columns (16- or 8-byte aligned) as CPT / 2 pairs
template <int CPT>
__device__ __forceinline__ void ld_cols(const float* p, float2 (&o)[CPT / 2]) {
    if constexpr (CPT == 4) {
        const float4 a = *reinterpret_cast<const float4*>(p);
        o[0] = make_float2(a.x, a.y);
        o[1] = make_float2(a.z, a.w);
    } else {
        o[0] = *reinterpret_cast<const float2*>(p);
    }
}
template <int CPT>
__device__ __forceinline__ void st_cols(float* p, const float2 (&v)[CPT / 2]) {
    if constexpr (CPT == 4)
        *reinterpret_cast<float4*>(p) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
    else
        *reinterpret_cast<float2*>(p) = v[0];
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Issue the cp.async copies of chunk c (tokens [c*C, c*C + n)) into raw
// buffer `rb`: the CTA's k (and q) column block, beta, v (and dout) rows and,
// in the backward sweep, the chunk's checkpoint.
template <typename TIn, int DV, int CWB>
__device__ __forceinline__ void issue_chunk(const Args& p, unsigned char* rb, long long bh, int cb,
                                            int c, int n, bool bwd, int tid) {
    using Tl = Tile<TIn, DV, CWB>;
    constexpr int ES = Tl::ES, NT = Tl::NT;
    constexpr int KP = CWB * ES / 16;                      // 16-byte pieces per token row
    const long long tok0 = bh * p.T + static_cast<long long>(c) * C;
    const char* kg = static_cast<const char*>(p.k) + (tok0 * p.dk + cb * CWB) * ES;
    const char* qg = static_cast<const char*>(p.q) + (tok0 * p.dk + cb * CWB) * ES;
    for (int i = tid; i < n * KP; i += NT) {
        const int s = i / KP, w = i % KP;
        cp_async16(rb + Tl::r_k + i * 16, kg + static_cast<long long>(s) * p.dk * ES + w * 16);
        if (bwd) cp_async16(rb + Tl::r_q + i * 16, qg + static_cast<long long>(s) * p.dk * ES + w * 16);
    }
    const int rp = n * (DV * ES / 16);
    const char* bg = static_cast<const char*>(p.beta) + tok0 * DV * ES;
    const char* vg = static_cast<const char*>(p.v) + tok0 * DV * ES;
    for (int i = tid; i < rp; i += NT) {
        cp_async16(rb + Tl::r_b + i * 16, bg + i * 16);
        cp_async16(rb + Tl::r_v + i * 16, vg + i * 16);
    }
    if (bwd) {
        const int op = n * (DV / 4);
        const char* og = reinterpret_cast<const char*>(p.dout + tok0 * DV);
        for (int i = tid; i < op; i += NT) cp_async16(rb + Tl::r_do + i * 16, og + i * 16);
        const char* cg = reinterpret_cast<const char*>(
            p.ckpt + (((bh - p.bh0) * p.ncb + cb) * p.nC + c) * static_cast<long long>(Tl::SW) * NT);
#pragma unroll
        for (int m = 0; m < Tl::SW / 4; ++m)
            cp_async16(rb + Tl::r_ck + (m * NT + tid) * 16, cg + (m * NT + tid) * 16);
    }
    cp_async_commit();
}

// Converts the raw chunk inputs to fp32 (k, k^2, q, beta, beta v, alpha).
template <typename TIn, int DV, int CWB>
__device__ __forceinline__ void convert_chunk(unsigned char* sm, const unsigned char* rb, int n,
                                              bool bwd, TIn d_raw, float A_h, int tid) {
    using Tl = Tile<TIn, DV, CWB>;
    constexpr int NT = Tl::NT;
    const TIn* rk = reinterpret_cast<const TIn*>(rb + Tl::r_k);
    const TIn* rq = reinterpret_cast<const TIn*>(rb + Tl::r_q);
    const TIn* rbt = reinterpret_cast<const TIn*>(rb + Tl::r_b);
    const TIn* rv = reinterpret_cast<const TIn*>(rb + Tl::r_v);
    float* sk = reinterpret_cast<float*>(sm + Tl::s_k);
    float* skk = reinterpret_cast<float*>(sm + Tl::s_kk);
    float* sq = reinterpret_cast<float*>(sm + Tl::s_q);
    float* sb = reinterpret_cast<float*>(sm + Tl::s_b);
    float* sbv = reinterpret_cast<float*>(sm + Tl::s_bv);
    for (int i = tid; i < n * CWB; i += NT) {
        const float kv = to_f<TIn>(rk[i]);
        sk[i] = kv;
        skk[i] = kv * kv;
        if (bwd) sq[i] = to_f<TIn>(rq[i]);
    }
    for (int i = tid; i < n * DV; i += NT) {
        const float b = to_f<TIn>(rbt[i]);
        sb[i] = b;
        sbv[i] = b * to_f<TIn>(rv[i]);
    }
    if (tid < n) reinterpret_cast<float*>(sm + Tl::s_al)[tid] = expf(-A_h * to_f<TIn>(d_raw));
}

// d of token t of head bh (t < T), raw: converted when the chunk is (the
// load stays in flight across a chunk's compute)
template <typename TIn>
__device__ __forceinline__ TIn d_of(const Args& p, long long bh, long long t) {
    return static_cast<const TIn*>(p.d)[bh * p.T + t];
}

// Sum over the NR lanes sharing a column group of 3 CPT values (3 per
// column: dq, dk-from-J, dk-from-eta partials).  Halving levels (two for 4
// columns, one for 2) leave each lane 3 values that are then summed over the
// remaining levels; afterwards a lane holds the totals of column
// g = 2 [rq & NR/2] + [rq & NR/4] (4 columns) or g = [rq & NR/2] (2).
template <int NR, int CPT>
__device__ __forceinline__ void column_reduce(float v[3 * CPT], int rq) {
    constexpr int o1 = NR / 2, o2 = NR / 4;
    const bool up1 = (rq & o1) != 0;
#pragma unroll
    for (int m = 0; m < 3 * CPT / 2; ++m) {
        const float send = up1 ? v[m] : v[m + 3 * CPT / 2];
        const float keep = up1 ? v[m + 3 * CPT / 2] : v[m];
        v[m] = keep + __shfl_xor_sync(FULL, send, o1);
    }
    constexpr int orest = CPT == 4 ? o2 : o1;   // the level after the halving ones
    if constexpr (CPT == 4) {
        const bool up2 = (rq & o2) != 0;
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            const float send = up2 ? v[m] : v[m + 3];
            const float keep = up2 ? v[m + 3] : v[m];
            v[m] = keep + __shfl_xor_sync(FULL, send, o2);
        }
    }
#pragma unroll
    for (int o = orest / 2; o > 0; o /= 2)
#pragma unroll
        for (int m = 0; m < 3; ++m) v[m] += __shfl_xor_sync(FULL, v[m], o);
}

// Per-token inputs of one thread: its 4 rows and CPT columns.
template <int CPT>
struct TokIn {
    float bet[4], bvv[4], dov[4];
    float2 kf[CPT / 2], kq[CPT / 2], qf[CPT / 2];
};

// One adjoint step (token t, state st = (J_t, eta_t) as stored in TMEM): the
// alpha sum of token t+1 with the adjoints as they come in, then the
// adjoints of token t, then token t's partial sums.
template <int CPT>
__device__ __forceinline__ void adjoint_step(const float st[8 * CPT], const TokIn<CPT>& in, float alpha_next,
                                             float Ip, float2 (&GJ)[4][CPT / 2], float2 (&GE)[4][CPT / 2],
                                             float cv[3 * CPT], float rsum[8], float& dsum) {
    constexpr int P = CPT / 2;
    const float2 ap = f2(alpha_next), ipp = f2(Ip);
    float2 cdq[P], cck[P], cce[P], dacc[2];
    dacc[0] = dacc[1] = make_float2(0.f, 0.f);
#pragma unroll
    for (int c2 = 0; c2 < P; ++c2) cdq[c2] = cck[c2] = cce[c2] = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        float2 rsb = make_float2(0.f, 0.f), rse = rsb;
        const float2 dov = f2(in.dov[r]), bet = f2(in.bet[r]), bvv = f2(in.bvv[r]);
#pragma unroll
        for (int c2 = 0; c2 < P; ++c2) {
            const float2 Jt = make_float2(st[CPT * r + 2 * c2], st[CPT * r + 2 * c2 + 1]);
            const float2 Et = make_float2(st[4 * CPT + CPT * r + 2 * c2], st[4 * CPT + CPT * r + 2 * c2 + 1]);
            const float2 den = __fadd2_rn(Jt, ipp);
            const float2 rr = make_float2(rcp_approx(den.x), rcp_approx(den.y));
            const float2 mu = __fmul2_rn(Et, rr);
            const float2 a = __fmul2_rn(__fmul2_rn(dov, in.qf[c2]), rr);
            dacc[c2 & 1] = __ffma2_rn(GJ[r][c2], Jt, dacc[c2 & 1]);
            dacc[c2 & 1] = __ffma2_rn(GE[r][c2], Et, dacc[c2 & 1]);
            GE[r][c2] = __ffma2_rn(ap, GE[r][c2], a);
            const float2 am = __fmul2_rn(a, mu);
            GJ[r][c2] = __ffma2_rn(ap, GJ[r][c2], make_float2(-am.x, -am.y));
            cdq[c2] = __ffma2_rn(dov, mu, cdq[c2]);
            rsb = __ffma2_rn(GJ[r][c2], in.kq[c2], rsb);
            rse = __ffma2_rn(GE[r][c2], in.kf[c2], rse);
            cck[c2] = __ffma2_rn(bet, GJ[r][c2], cck[c2]);
            cce[c2] = __ffma2_rn(bvv, GE[r][c2], cce[c2]);
        }
        rsum[r] = rsb.x + rsb.y;
        rsum[4 + r] = rse.x + rse.y;
    }
#pragma unroll
    for (int c2 = 0; c2 < P; ++c2) {
        cv[3 * (2 * c2)] = cdq[c2].x;
        cv[3 * (2 * c2) + 1] = cck[c2].x;
        cv[3 * (2 * c2) + 2] = cce[c2].x;
        cv[3 * (2 * c2 + 1)] = cdq[c2].y;
        cv[3 * (2 * c2 + 1) + 1] = cck[c2].y;
        cv[3 * (2 * c2 + 1) + 2] = cce[c2].y;
    }
    const float2 ds = __fadd2_rn(dacc[0], dacc[1]);
    dsum = ds.x + ds.y;
}

template <typename TIn, int DV, int CWB>
__global__ void __launch_bounds__(Tile<TIn, DV, CWB>::NT, 1) diag_bwd_kernel(const Args p) {
    using Tl = Tile<TIn, DV, CWB>;
    constexpr int NR = Tl::NR, NCQ = Tl::NCQ, NT = Tl::NT, NW = Tl::NW, CPT = Tl::CPT, P2 = CPT / 2;
    constexpr int SW = Tl::SW;
    extern __shared__ __align__(128) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long lbh = blockIdx.x / p.ncb;   // head within this launch
    const long long bh = p.bh0 + lbh;
    const int cb = blockIdx.x % p.ncb;
    const bool valid = tid < Tl::NTA;
    const int rq = valid ? tid % NR : 0, cq = valid ? tid / NR : 0;
    const int row0 = 4 * rq, col0 = CPT * cq;                  // inside the tile
    const long long S = static_cast<long long>(DV) * p.dk;
    const float Ip = p.Ip;
    uint32_t* holder = reinterpret_cast<uint32_t*>(sm + Tl::holder);

    if (warp == 0) tmem_alloc(holder, Tl::TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = *holder;
    const uint32_t tlane = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                           static_cast<uint32_t>(warp >> 2) * Tl::HIST_COLS;

    // ---- initial state of the tile: J = I_0 - I_prior, E = I_0 mu_0 -------
    float2 J[4][P2], E[4][P2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const long long off = bh * S + static_cast<long long>(row0 + r) * p.dk + cb * CWB + col0;
        float2 i2[P2], m2[P2];
#pragma unroll
        for (int c2 = 0; c2 < P2; ++c2) {
            i2[c2] = f2(Ip);
            m2[c2] = f2(0.f);
        }
        if (valid && p.I0) ld_cols<CPT>(p.I0 + off, i2);
        if (valid && p.mu0) ld_cols<CPT>(p.mu0 + off, m2);
#pragma unroll
        for (int c2 = 0; c2 < P2; ++c2) {
            J[r][c2] = make_float2(i2[c2].x - Ip, i2[c2].y - Ip);
            E[r][c2] = make_float2(i2[c2].x * m2[c2].x, i2[c2].y * m2[c2].y);
        }
    }
    // the state as SW / 4 float4 (J rows, then eta rows) and back: the
    // layout of a checkpoint
    auto state_f4 = [&](int m) {
        const float2 (&X)[4][P2] = m < SW / 8 ? J : E;
        const int r = ((m % (SW / 8)) * 4) / CPT;   // first row of the float4
        if constexpr (CPT == 4)
            return make_float4(X[r][0].x, X[r][0].y, X[r][1].x, X[r][1].y);
        else
            return make_float4(X[r][0].x, X[r][0].y, X[r + 1][0].x, X[r + 1][0].y);
    };
    auto set_state_f4 = [&](int m, float4 a) {
        float2 (&X)[4][P2] = m < SW / 8 ? J : E;
        const int r = ((m % (SW / 8)) * 4) / CPT;
        if constexpr (CPT == 4) {
            X[r][0] = make_float2(a.x, a.y);
            X[r][1] = make_float2(a.z, a.w);
        } else {
            X[r][0] = make_float2(a.x, a.y);
            X[r + 1][0] = make_float2(a.z, a.w);
        }
    };

    auto raw = [&](int i) { return sm + (i ? Tl::raw1 : Tl::raw0); };
    const float* sk = reinterpret_cast<const float*>(sm + Tl::s_k);
    const float* skk = reinterpret_cast<const float*>(sm + Tl::s_kk);
    const float* sq = reinterpret_cast<const float*>(sm + Tl::s_q);
    const float* sb = reinterpret_cast<const float*>(sm + Tl::s_b);
    const float* sbv = reinterpret_cast<const float*>(sm + Tl::s_bv);
    const float* sal = reinterpret_cast<const float*>(sm + Tl::s_al);
    float* ckpt_cta = p.ckpt + (lbh * p.ncb + cb) * static_cast<long long>(p.nC) * SW * NT;
    const int nC = p.nC;
    auto ntok = [&](int c) { return min(C, p.T - c * C); };
    // one forward step of the tile on token s of the converted chunk
    auto forward_step = [&](int s) {
        const float2 al = f2(sal[s]);
        const float4 b4 = *reinterpret_cast<const float4*>(sb + s * DV + row0);
        const float4 v4 = *reinterpret_cast<const float4*>(sbv + s * DV + row0);
        const float bet[4] = {b4.x, b4.y, b4.z, b4.w}, bvv[4] = {v4.x, v4.y, v4.z, v4.w};
        float2 kf[P2], kq[P2];
        ld_cols<CPT>(sk + s * CWB + col0, kf);
        ld_cols<CPT>(skk + s * CWB + col0, kq);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c2 = 0; c2 < P2; ++c2) {
                J[r][c2] = __ffma2_rn(al, J[r][c2], __fmul2_rn(f2(bet[r]), kq[c2]));
                E[r][c2] = __ffma2_rn(al, E[r][c2], __fmul2_rn(f2(bvv[r]), kf[c2]));
            }
    };

    // ---- forward sweep: checkpoints every C tokens, staged F1 tokens at a time
    constexpr int F1 = Tl::F1;
    const float A_h = p.A[bh % p.H];
    TIn dreg{};   // d of token (stage start + tid), prefetched
    const int nS = (p.T + F1 - 1) / F1;
    auto f1n = [&](int g) { return min(F1, p.T - g * F1); };
    auto issue_stage = [&](int g, unsigned char* rb) {   // k column block, beta, v rows of stage g
        constexpr int ES = Tl::ES, KP = CWB * ES / 16;
        const int n = f1n(g);
        const long long tok0 = bh * p.T + static_cast<long long>(g) * F1;
        const char* kg = static_cast<const char*>(p.k) + (tok0 * p.dk + cb * CWB) * ES;
        for (int i = tid; i < n * KP; i += NT) {
            const int ss = i / KP, w = i % KP;
            cp_async16(rb + Tl::f1_k + i * 16, kg + static_cast<long long>(ss) * p.dk * ES + w * 16);
        }
        const int rp = n * (DV * ES / 16);
        const char* bg = static_cast<const char*>(p.beta) + tok0 * DV * ES;
        const char* vg = static_cast<const char*>(p.v) + tok0 * DV * ES;
        for (int i = tid; i < rp; i += NT) {
            cp_async16(rb + Tl::f1_b + i * 16, bg + i * 16);
            cp_async16(rb + Tl::f1_v + i * 16, vg + i * 16);
        }
        cp_async_commit();
    };
    const float* gk = reinterpret_cast<const float*>(sm + Tl::g_k);
    const float* gkk = reinterpret_cast<const float*>(sm + Tl::g_kk);
    const float* gb = reinterpret_cast<const float*>(sm + Tl::g_b);
    const float* gbv = reinterpret_cast<const float*>(sm + Tl::g_bv);
    const float* gal = reinterpret_cast<const float*>(sm + Tl::g_al);
    if (nS > 0) {
        issue_stage(0, raw(0));
        if (tid < f1n(0)) dreg = d_of<TIn>(p, bh, tid);
    }
    for (int g = 0; g < nS; ++g) {
        const int n = f1n(g);
        cp_async_wait_all();
        __syncthreads();   // stage g landed; stage g-1's compute finished
        {   // convert: k -> k, k^2; beta, v -> beta, beta v; d -> alpha
            const unsigned char* rb = raw(g & 1);
            const TIn* rk = reinterpret_cast<const TIn*>(rb + Tl::f1_k);
            const TIn* rbt = reinterpret_cast<const TIn*>(rb + Tl::f1_b);
            const TIn* rv = reinterpret_cast<const TIn*>(rb + Tl::f1_v);
            float* wk = reinterpret_cast<float*>(sm + Tl::g_k);
            float* wkk = reinterpret_cast<float*>(sm + Tl::g_kk);
            float* wb = reinterpret_cast<float*>(sm + Tl::g_b);
            float* wbv = reinterpret_cast<float*>(sm + Tl::g_bv);
            for (int i = tid; i < n * CWB; i += NT) {
                const float kv = to_f<TIn>(rk[i]);
                wk[i] = kv;
                wkk[i] = kv * kv;
            }
            for (int i = tid; i < n * DV; i += NT) {
                const float b = to_f<TIn>(rbt[i]);
                wb[i] = b;
                wbv[i] = b * to_f<TIn>(rv[i]);
            }
            if (tid < n) reinterpret_cast<float*>(sm + Tl::g_al)[tid] = expf(-A_h * to_f<TIn>(dreg));
        }
        if (g + 1 < nS) {
            issue_stage(g + 1, raw((g + 1) & 1));
            if (tid < f1n(g + 1)) dreg = d_of<TIn>(p, bh, static_cast<long long>(g + 1) * F1 + tid);
        }
        __syncthreads();
#pragma unroll 1
        for (int s = 0; s < n; ++s) {
            if ((s & (C - 1)) == 0) {   // checkpoint: the tile's state before chunk (g F1 + s) / C
                const int c = (g * F1 + s) / C;
                float4* dst = reinterpret_cast<float4*>(ckpt_cta + static_cast<long long>(c) * SW * NT);
#pragma unroll
                for (int m = 0; m < SW / 4; ++m) dst[m * NT + tid] = state_f4(m);
            }
            const float2 al = f2(gal[s]);
            const float4 b4 = *reinterpret_cast<const float4*>(gb + s * DV + row0);
            const float4 v4 = *reinterpret_cast<const float4*>(gbv + s * DV + row0);
            const float bet[4] = {b4.x, b4.y, b4.z, b4.w}, bvv[4] = {v4.x, v4.y, v4.z, v4.w};
            float2 kf[P2], kq[P2];
            ld_cols<CPT>(gk + s * CWB + col0, kf);
            ld_cols<CPT>(gkk + s * CWB + col0, kq);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c2 = 0; c2 < P2; ++c2) {
                    J[r][c2] = __ffma2_rn(al, J[r][c2], __fmul2_rn(f2(bet[r]), kq[c2]));
                    E[r][c2] = __ffma2_rn(al, E[r][c2], __fmul2_rn(f2(bvv[r]), kf[c2]));
                }
        }
    }
    cp_async_wait_all();
    // checkpoints written by other threads are read back through cp.async
    __threadfence();
    __syncthreads();

    // ---- adjoints at t = T from the final-state gradients ------------------
    float2 GJ[4][P2], GE[4][P2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const long long off = bh * S + static_cast<long long>(row0 + r) * p.dk + cb * CWB + col0;
        float2 dm[P2], di[P2];
#pragma unroll
        for (int c2 = 0; c2 < P2; ++c2) dm[c2] = di[c2] = f2(0.f);
        if (valid && p.dfinal) {
            ld_cols<CPT>(p.dfinal + off, dm);
            ld_cols<CPT>(p.dfinal + p.BH * S + off, di);
        }
#pragma unroll
        for (int c2 = 0; c2 < P2; ++c2) {
            const float2 den = __fadd2_rn(J[r][c2], f2(Ip));
            const float2 rr = make_float2(1.f / den.x, 1.f / den.y);
            const float2 mu = __fmul2_rn(E[r][c2], rr);
            const float2 a = __fmul2_rn(dm[c2], rr);
            GE[r][c2] = a;
            GJ[r][c2] = make_float2(di[c2].x - a.x * mu.x, di[c2].y - a.y * mu.y);
        }
    }

    // ---- backward sweep over the chunks, last first ------------------------
    float* s_row = reinterpret_cast<float*>(sm + Tl::s_row);
    float* s_dq = reinterpret_cast<float*>(sm + Tl::s_dq);
    float* s_dk = reinterpret_cast<float*>(sm + Tl::s_dk);
    float* s_D = reinterpret_cast<float*>(sm + Tl::s_D);
    // after column_reduce a lane holds the totals of column g of its group;
    // one lane per column writes them
    constexpr int o1 = NR / 2, o2 = NR / 4;
    const int g = CPT == 4 ? 2 * ((rq & o1) ? 1 : 0) + ((rq & o2) ? 1 : 0) : ((rq & o1) ? 1 : 0);
    const bool col_writer = valid && (rq & ((CPT == 4 ? o2 : o1) - 1)) == 0;
    float alpha_next = 1.f;   // alpha of the token after the one being processed
    if (nC > 0) {
        const int c = nC - 1;
        issue_chunk<TIn, DV, CWB>(p, raw(c & 1), bh, cb, c, ntok(c), true, tid);
        if (tid < ntok(c)) dreg = d_of<TIn>(p, bh, static_cast<long long>(c) * C + tid);
    }
    for (int c = nC - 1; c >= 0; --c) {
        const int n = ntok(c);
        const long long t0 = static_cast<long long>(c) * C;
        cp_async_wait_all();
        __syncthreads();   // chunk c landed; the previous chunk's epilogue finished
        unsigned char* rb = raw(c & 1);
        convert_chunk<TIn, DV, CWB>(sm, rb, n, true, dreg, A_h, tid);
        if (c > 0) {
            issue_chunk<TIn, DV, CWB>(p, raw((c - 1) & 1), bh, cb, c - 1, C, true, tid);
            if (tid < C) dreg = d_of<TIn>(p, bh, t0 - C + tid);
        }
        {   // the chunk's checkpoint
            const float4* src = reinterpret_cast<const float4*>(rb + Tl::r_ck);
#pragma unroll
            for (int m = 0; m < SW / 4; ++m) set_state_f4(m, src[m * NT + tid]);
        }
        __syncthreads();   // converted inputs visible
        // forward again through the chunk; token s's state goes to TMEM slot s
        auto fwd_store = [&](int s) {
            forward_step(s);
            float st[SW];   // J rows, then eta rows
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c2 = 0; c2 < P2; ++c2) {
                    st[CPT * r + 2 * c2] = J[r][c2].x;
                    st[CPT * r + 2 * c2 + 1] = J[r][c2].y;
                    st[4 * CPT + CPT * r + 2 * c2] = E[r][c2].x;
                    st[4 * CPT + CPT * r + 2 * c2 + 1] = E[r][c2].y;
                }
            if constexpr (SW == 32)
                tmem_st32(tlane + static_cast<uint32_t>(s * SW), st);
            else
                tmem_st16(tlane + static_cast<uint32_t>(s * SW), st);
        };
#pragma unroll 2
        for (int s = 0; s < n; ++s) fwd_store(s);
        tmem_wait_st();
        const float* sdo = reinterpret_cast<const float*>(rb + Tl::r_do);
        auto load_in = [&](int s, TokIn<CPT>& in) {
            const float4 b4 = *reinterpret_cast<const float4*>(sb + s * DV + row0);
            const float4 v4 = *reinterpret_cast<const float4*>(sbv + s * DV + row0);
            const float4 o4 = *reinterpret_cast<const float4*>(sdo + s * DV + row0);
            in.bet[0] = b4.x; in.bet[1] = b4.y; in.bet[2] = b4.z; in.bet[3] = b4.w;
            in.bvv[0] = v4.x; in.bvv[1] = v4.y; in.bvv[2] = v4.z; in.bvv[3] = v4.w;
            in.dov[0] = o4.x; in.dov[1] = o4.y; in.dov[2] = o4.z; in.dov[3] = o4.w;
            ld_cols<CPT>(sk + s * CWB + col0, in.kf);
            ld_cols<CPT>(skk + s * CWB + col0, in.kq);
            ld_cols<CPT>(sq + s * CWB + col0, in.qf);
        };
        // a token's partial sums into shared memory (column sums reduced here)
        auto emit = [&](int s, float cv[3 * CPT], const float rsum[8], float dsum) {
            column_reduce<NR, CPT>(cv, rq);
            if (col_writer) {
                const int j = col0 + g;
                s_dq[s * CWB + j] = cv[0];
                s_dk[s * CWB + j] = 2.f * sk[s * CWB + j] * cv[1] + cv[2];
            }
            if (valid) {
                float* rowp = s_row + s * 2 * NCQ * DV;
                *reinterpret_cast<float4*>(rowp + cq * DV + row0) =
                    make_float4(rsum[0], rsum[1], rsum[2], rsum[3]);
                *reinterpret_cast<float4*>(rowp + (NCQ + cq) * DV + row0) =
                    make_float4(rsum[4], rsum[5], rsum[6], rsum[7]);
            }
            if (!valid) dsum = 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(FULL, dsum, o);
            if (lane == 0) s_D[s * NW + warp] = dsum;
        };
        // adjoint steps from the chunk's last token down.  Token s+1's sums are
        // reduced in the same step as token s's element arithmetic (the two are
        // independent), so the shuffle latency overlaps arithmetic.
        float cur[SW], cv[3 * CPT], rsum[8], dsum;
        auto hist_load = [&](int s) {   // token s's state from TMEM into cur
            if constexpr (SW == 32) {
                tmem_ld32_async(tlane + static_cast<uint32_t>(s * SW), cur);
                tmem_wait_ld(cur);
            } else {
                tmem_ld16_async(tlane + static_cast<uint32_t>(s * SW), cur);
                tmem_wait_ld16(cur);
            }
        };
        hist_load(n - 1);
        {
            TokIn<CPT> in;
            load_in(n - 1, in);
            adjoint_step<CPT>(cur, in, alpha_next, Ip, GJ, GE, cv, rsum, dsum);
            alpha_next = sal[n - 1];
        }
        // two tokens per iteration with the partial-sum buffers swapped (no
        // register copies between steps)
        auto step_back = [&](int s, float (&cvi)[3 * CPT], float (&rsi)[8], float& dsi,
                             float (&cvo)[3 * CPT], float (&rso)[8], float& dso) {
            hist_load(s);
            TokIn<CPT> in;
            load_in(s, in);
            adjoint_step<CPT>(cur, in, alpha_next, Ip, GJ, GE, cvo, rso, dso);
            emit(s + 1, cvi, rsi, dsi);
            alpha_next = sal[s];
        };
        float cvb[3 * CPT], rsumb[8], dsumb;
        int s = n - 2;
#pragma unroll 1
        for (; s >= 1; s -= 2) {
            step_back(s, cv, rsum, dsum, cvb, rsumb, dsumb);
            step_back(s - 1, cvb, rsumb, dsumb, cv, rsum, dsum);
        }
        if (s == 0) {
            step_back(0, cv, rsum, dsum, cvb, rsumb, dsumb);
#pragma unroll
            for (int m = 0; m < 3 * CPT; ++m) cv[m] = cvb[m];
#pragma unroll
            for (int m = 0; m < 8; ++m) rsum[m] = rsumb[m];
            dsum = dsumb;
        }
        emit(0, cv, rsum, dsum);
        __syncthreads();   // the chunk's partials are complete
        // ---- epilogue of the chunk: row partials, alpha sums, dq, dk -------
        {
            const long long tokbase = bh * p.T + t0;
            const long long ltok = lbh * p.T + t0;   // in this launch's partials
            float* prow = p.prow + (static_cast<long long>(cb) * p.nbh * p.T + ltok) * 2 * DV;
            // 4 rows per thread and item: all NCQ partials loaded, then a tree sum
            constexpr int R4 = DV / 4;
#pragma unroll 2
            for (int i = tid; i < n * 2 * R4; i += NT) {
                const int ss = i / (2 * R4), rem = i % (2 * R4), qi = rem / R4, r4 = rem % R4;
                const float4* src =
                    reinterpret_cast<const float4*>(s_row + ss * 2 * NCQ * DV + qi * NCQ * DV) + r4;
                float4 part[NCQ];
#pragma unroll
                for (int x = 0; x < NCQ; ++x) part[x] = src[x * R4];
#pragma unroll
                for (int w = 1; w < NCQ; w *= 2)
#pragma unroll
                    for (int x = 0; x + w < NCQ; x += 2 * w) {
                        part[x].x += part[x + w].x;
                        part[x].y += part[x + w].y;
                        part[x].z += part[x + w].z;
                        part[x].w += part[x + w].w;
                    }
                reinterpret_cast<float4*>(prow)[i] = part[0];
            }
            // slot s holds token t0 + s + 1 (none after the last token)
            if (tid < n && t0 + tid + 1 < p.T) {
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) acc += s_D[tid * NW + w];
                p.pD[static_cast<long long>(cb) * p.nbh * p.T + ltok + tid + 1] = acc;
            }
            for (int i = tid; i < n * CWB; i += NT) {
                const int ss = i / CWB, j = i % CWB;
                const long long o = (tokbase + ss) * p.dk + cb * CWB + j;
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
            const long long off = bh * S + static_cast<long long>(row0 + r) * p.dk + cb * CWB + col0;
            float2 i2[P2], m2[P2];
#pragma unroll
            for (int c2 = 0; c2 < P2; ++c2) {
                i2[c2] = f2(Ip);
                m2[c2] = f2(0.f);
            }
            if (valid && p.I0) ld_cols<CPT>(p.I0 + off, i2);
            if (valid && p.mu0) ld_cols<CPT>(p.mu0 + off, m2);
            // J_0 = I_0 - I_prior, eta_0 = I_0 mu_0
#pragma unroll
            for (int c2 = 0; c2 < P2; ++c2) {
                dsum += GJ[r][c2].x * (i2[c2].x - Ip) + GJ[r][c2].y * (i2[c2].y - Ip);
                dsum += GE[r][c2].x * (i2[c2].x * m2[c2].x) + GE[r][c2].y * (i2[c2].y * m2[c2].y);
            }
            if (p.dinit && valid) {
                float2 dmu[P2], dI[P2];
#pragma unroll
                for (int c2 = 0; c2 < P2; ++c2) {
                    const float2 gj = __fmul2_rn(a0, GJ[r][c2]), ge = __fmul2_rn(a0, GE[r][c2]);
                    dmu[c2] = make_float2(ge.x * i2[c2].x, ge.y * i2[c2].y);
                    dI[c2] = make_float2(gj.x + ge.x * m2[c2].x, gj.y + ge.y * m2[c2].y);
                }
                st_cols<CPT>(p.dinit + off, dmu);
                st_cols<CPT>(p.dinit + p.BH * S + off, dI);
            }
        }
        if (!valid) dsum = 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(FULL, dsum, o);
        if (lane == 0) s_D[warp] = dsum;
        __syncthreads();
        if (tid == 0 && p.T > 0) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) acc += s_D[w];
            p.pD[static_cast<long long>(cb) * p.nbh * p.T + lbh * p.T] = acc;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, Tl::TMEM_COLS);
}

// Per (head, token): adds the column blocks' partials and forms dbeta, dv,
// dd = -A alpha dL/dalpha and the token's dA term -d alpha dL/dalpha.  One
// warp per token; the launch covers the BHT tokens from tok0 on, whose
// partials (of one main-kernel launch) start at prow and pD.
template <typename TIn, int NCBM>
__global__ void __launch_bounds__(256) diag_bwd_finalize_kernel(
    const TIn* __restrict__ v, const TIn* __restrict__ beta, const TIn* __restrict__ d,
    const float* __restrict__ A, const float* __restrict__ prow, const float* __restrict__ pD,
    float* __restrict__ dv_out, float* __restrict__ dbeta, float* __restrict__ dd,
    float* __restrict__ eA, long long tok0, long long BHT, int T, int H, int dv, int ncb) {
    const long long ltok = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (ltok >= BHT) return;
    const long long tok = tok0 + ltok;
    // 4 rows per lane: every partial is one 16-byte load, all issued before
    // the sums (at most NCBM column blocks: 4, or 8 for 16-column blocks)
    for (int i4 = lane; i4 < dv / 4; i4 += 32) {
        float4 pb[NCBM], pe[NCBM];
#pragma unroll
        for (int cb = 0; cb < NCBM; ++cb) {
            if (cb < ncb) {
                const float4* pr = reinterpret_cast<const float4*>(prow + (static_cast<long long>(cb) * BHT + ltok) * 2 * dv);
                pb[cb] = pr[i4];
                pe[cb] = pr[dv / 4 + i4];
            } else {
                pb[cb] = pe[cb] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int w = 1; w < NCBM; w *= 2)
#pragma unroll
            for (int x = 0; x + w < NCBM; x += 2 * w) {
                pb[x].x += pb[x + w].x; pb[x].y += pb[x + w].y; pb[x].z += pb[x + w].z; pb[x].w += pb[x + w].w;
                pe[x].x += pe[x + w].x; pe[x].y += pe[x + w].y; pe[x].z += pe[x + w].z; pe[x].w += pe[x + w].w;
            }
        const float4 b4 = load4<TIn>(beta + tok * dv + 4 * i4), v4 = load4<TIn>(v + tok * dv + 4 * i4);
        const float4 sb = pb[0], se = pe[0];
        reinterpret_cast<float4*>(dbeta + tok * dv)[i4] =
            make_float4(sb.x + v4.x * se.x, sb.y + v4.y * se.y, sb.z + v4.z * se.z, sb.w + v4.w * se.w);
        reinterpret_cast<float4*>(dv_out + tok * dv)[i4] = make_float4(b4.x * se.x, b4.y * se.y, b4.z * se.z, b4.w * se.w);
    }
    if (lane == 0) {
        float g_alpha = 0.f;
        for (int cb = 0; cb < ncb; ++cb) g_alpha += pD[static_cast<long long>(cb) * BHT + ltok];
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

template <typename TIn, int DV, int CWB>
cudaError_t launch_main(const Args& p, long long grid, cudaStream_t st) {
    using Tl = Tile<TIn, DV, CWB>;
    cudaError_t e = cudaFuncSetAttribute(diag_bwd_kernel<TIn, DV, CWB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Tl::SMEM);
    if (e != cudaSuccess) return e;
    diag_bwd_kernel<TIn, DV, CWB><<<static_cast<unsigned>(grid), Tl::NT, Tl::SMEM, st>>>(p);
    return cudaGetLastError();
}

template <typename TIn, int CWB>
cudaError_t launch_dv(int dv, const Args& p, long long grid, cudaStream_t st) {
    switch (dv) {
        case 16: return launch_main<TIn, 16, CWB>(p, grid, st);
        case 32: return launch_main<TIn, 32, CWB>(p, grid, st);
        case 64: return launch_main<TIn, 64, CWB>(p, grid, st);
        default: return launch_main<TIn, 128, CWB>(p, grid, st);
    }
}

// Key columns per CTA: all of d_k below 32; else 32, or 16 when 32-column
// blocks would leave more than half of the SMs idle (few heads: 16-column
// blocks double the CTAs; the row partials to add up double too).
inline int bwd_cwb(long long BH, int dk) {
    if (dk < 32) return dk;
    return BH * (dk / 32) * 2 <= sm_count() ? 16 : 32;
}

// The main kernel's launches: heads [0, heads_a) with cwb_a-column blocks,
// then heads [heads_a, BH) with cwb_b.  A wave is the CTA slots of the GPU
// (one 8-warp CTA per SM, or two of up to 4 warps).  When 32-column blocks
// fill W >= 1 whole waves and leave a remainder of r CTAs with 2 r <= one
// wave, the remainder's heads take 16-column blocks instead: one partial
// wave of 16-column CTAs (each ~0.75 of a 32-column CTA's time) instead of
// one of 32-column CTAs.
struct BwdPlan {
    int cwb_a, ncb_a, cwb_b, ncb_b;
    long long heads_a, heads_b;
};

inline BwdPlan bwd_plan(long long BH, int dk, int dv) {
    BwdPlan pl{};
    pl.cwb_a = bwd_cwb(BH, dk);
    pl.ncb_a = dk / pl.cwb_a;
    pl.heads_a = BH;
    pl.cwb_b = pl.cwb_a;
    pl.ncb_b = pl.ncb_a;
    if (pl.cwb_a == 32) {
        const int nt = (dv / 4) * 8;   // threads of a 32-column CTA
        const long long S = static_cast<long long>(sm_count()) * (nt > 128 ? 1 : 2), n = BH * pl.ncb_a;
        const long long W = n / S, r = n % S;
        if (W >= 1 && r > 0 && 2 * r <= S && (W * S) % pl.ncb_a == 0) {
            pl.heads_a = W * S / pl.ncb_a;
            pl.cwb_b = 16;
            pl.ncb_b = dk / 16;
        }
    }
    pl.heads_b = BH - pl.heads_a;
    return pl;
}

// Scratch of one call: checkpoints, row partials, alpha partials (each per
// launch), dA terms.
struct Scratch {
    size_t ck_a, row_a, pd_a, ck_b, row_b, pd_b, ea, total;
};

inline size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

inline Scratch scratch_of(int B, int H, int T, int dk, int dv) {
    const long long BH = static_cast<long long>(B) * H;
    const BwdPlan pl = bwd_plan(BH, dk, dv);
    const long long nC = (static_cast<long long>(T) + C - 1) / C;
    auto ck_words = [&](int cwb) {   // checkpoint words of a CTA: 8 CPT per thread
        const int cpt = cwb == 32 ? 4 : 2, nta = (dv / 4) * (cwb / cpt);
        return static_cast<size_t>(8 * cpt) * (nta < 32 ? 32 : nta);
    };
    Scratch s{};
    s.ck_a = up256(static_cast<size_t>(pl.heads_a) * pl.ncb_a * nC * ck_words(pl.cwb_a) * 4);
    s.row_a = up256(static_cast<size_t>(pl.ncb_a) * pl.heads_a * T * 2 * dv * 4);
    s.pd_a = up256(static_cast<size_t>(pl.ncb_a) * pl.heads_a * T * 4);
    s.ck_b = up256(static_cast<size_t>(pl.heads_b) * pl.ncb_b * nC * ck_words(pl.cwb_b) * 4);
    s.row_b = up256(static_cast<size_t>(pl.ncb_b) * pl.heads_b * T * 2 * dv * 4);
    s.pd_b = up256(static_cast<size_t>(pl.ncb_b) * pl.heads_b * T * 4);
    s.ea = up256(static_cast<size_t>(BH) * T * 4);
    s.total = s.ck_a + s.row_a + s.pd_a + s.ck_b + s.row_b + s.pd_b + s.ea;
    return s;
}

// The main kernel over heads [bh0, bh0 + nbh).
template <typename TIn>
cudaError_t launch_main_range(const DiagBwdArgs& a, Args p, long long bh0, long long nbh, int cwb,
                              float* ck, float* prow, float* pD, cudaStream_t st) {
    if (nbh == 0) return cudaSuccess;
    p.bh0 = bh0;
    p.nbh = nbh;
    p.ncb = a.dk / cwb;
    p.ckpt = ck;
    p.prow = prow;
    p.pD = pD;
    const long long grid = nbh * p.ncb;
    return cwb == 16 ? launch_dv<TIn, 16>(a.dv, p, grid, st) : launch_dv<TIn, 32>(a.dv, p, grid, st);
}

// The finalize kernel over the same heads (their row and alpha partials).
template <typename TIn>
cudaError_t launch_finalize_range(const DiagBwdArgs& a, long long bh0, long long nbh, int cwb,
                                  const float* prow, const float* pD, float* eA, cudaStream_t st) {
    if (nbh == 0 || a.T <= 0) return cudaSuccess;
    const int ncb = a.dk / cwb;
    const long long BHT = nbh * a.T;
    auto fin = ncb <= 4 ? diag_bwd_finalize_kernel<TIn, 4> : diag_bwd_finalize_kernel<TIn, 8>;
    fin<<<static_cast<unsigned>((BHT + 7) / 8), 256, 0, st>>>(
        static_cast<const TIn*>(a.v), static_cast<const TIn*>(a.beta), static_cast<const TIn*>(a.d),
        a.A, prow, pD, a.grad_v, a.grad_beta, a.grad_d, eA, bh0 * a.T, BHT, a.T, a.H, a.dv, ncb);
    return cudaGetLastError();
}

// A stream of the library's own per device, on which the first launch's
// finalize (HBM-bound) runs while the second launch's main kernel (which
// leaves SMs free) computes; joined back by events.
cudaError_t side_stream(cudaStream_t* out) {
    static cudaStream_t streams[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!streams[dev]) {
        e = cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking);
        if (e != cudaSuccess) return e;
    }
    *out = streams[dev];
    return cudaSuccess;
}

template <typename TIn>
kdn_status launch(const DiagBwdArgs& a, cudaStream_t st) {
    const long long BH = static_cast<long long>(a.B) * a.H;
    const BwdPlan pl = bwd_plan(BH, a.dk, a.dv);
    const int nC = (a.T + C - 1) / C;
    const Scratch sc = scratch_of(a.B, a.H, a.T, a.dk, a.dv);
    void* scratch = a.workspace;
    cudaError_t e = cudaSuccess;
    const bool own = scratch == nullptr && sc.total > 0;
    if (own) {
        e = cudaMallocAsync(&scratch, sc.total, st);
        if (e != cudaSuccess) return from_cuda(e);
    }
    unsigned char* base = static_cast<unsigned char*>(scratch);
    auto at = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
    Args p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.beta = a.beta; p.d = a.d; p.A = a.A; p.Ip = a.I_prior;
    p.I0 = a.I0; p.mu0 = a.mu0; p.dout = a.grad_out; p.dfinal = a.grad_final_state;
    p.gq = a.grad_q; p.gk = a.grad_k; p.dinit = a.grad_init_state;
    p.BH = BH; p.H = a.H; p.T = a.T; p.dk = a.dk; p.nC = nC;
    size_t off = 0;
    float* ck_a = at(off);  off += sc.ck_a;
    float* row_a = at(off); off += sc.row_a;
    float* pd_a = at(off);  off += sc.pd_a;
    float* ck_b = at(off);  off += sc.ck_b;
    float* row_b = at(off); off += sc.row_b;
    float* pd_b = at(off);  off += sc.pd_b;
    float* eA = at(off);
    e = launch_main_range<TIn>(a, p, 0, pl.heads_a, pl.cwb_a, ck_a, row_a, pd_a, st);
    if (e == cudaSuccess && pl.heads_b == 0) {
        e = launch_finalize_range<TIn>(a, 0, pl.heads_a, pl.cwb_a, row_a, pd_a, eA, st);
    } else if (e == cudaSuccess) {
        // the first launch's finalize on the side stream, concurrent with the
        // second launch's main kernel; the caller's stream waits for it
        cudaStream_t side = nullptr;
        cudaEvent_t fork = nullptr, join = nullptr;
        e = side_stream(&side);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventRecord(fork, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side, fork, 0);
        if (e == cudaSuccess) e = launch_finalize_range<TIn>(a, 0, pl.heads_a, pl.cwb_a, row_a, pd_a, eA, side);
        const bool forked = e == cudaSuccess;   // side-stream work is enqueued from here on
        if (forked) e = cudaEventRecord(join, side);
        if (e == cudaSuccess)
            e = launch_main_range<TIn>(a, p, pl.heads_a, pl.heads_b, pl.cwb_b, ck_b, row_b, pd_b, st);
        if (e == cudaSuccess)
            e = launch_finalize_range<TIn>(a, pl.heads_a, pl.heads_b, pl.cwb_b, row_b, pd_b, eA, st);
        // join even after an error, so that no later work on the caller's
        // stream (freeing the scratch) overtakes the side stream's finalize
        if (forked) {
            const cudaError_t ej = cudaStreamWaitEvent(st, join, 0);
            if (e == cudaSuccess) e = ej;
        }
        if (fork) cudaEventDestroy(fork);
        if (join) cudaEventDestroy(join);
    }
    if (e == cudaSuccess && a.grad_A) {
        if (a.T > 0) {
            diag_bwd_dA_kernel<<<a.H, 256, 0, st>>>(eA, a.grad_A, a.B, a.H, a.T);
            e = cudaGetLastError();
        } else {
            e = cudaMemsetAsync(a.grad_A, 0, sizeof(float) * a.H, st);
        }
    }
    if (own) {
        const cudaError_t ef = cudaFreeAsync(scratch, st);
        if (e == cudaSuccess) e = ef;
    }
    return from_cuda(e);
}

}  // namespace
}  // namespace bwd

long long diag_bwd_workspace_bytes(int B, int H, int T, int dk, int dv) {
    return static_cast<long long>(bwd::scratch_of(B, H, T, dk, dv).total);
}

kdn_status diag_bwd_launch(const DiagBwdArgs& a, cudaStream_t st) {
    return a.dtype == KDN_BF16 ? bwd::launch<__nv_bfloat16>(a, st) : bwd::launch<float>(a, st);
}

}  // namespace kdn
