// diag_impl.cuh -- the diagonal metaplastic scan with readout, for sm_103a.
//
// What is computed ("Learning to Remember, Learn, and Forget in Attention-
// Based Models", Metodologia 1-2; readout as in "Kalman Linear Attention
// (KLA)", Metodologia 1), per head, per token t, per state element (i, j):
//     alpha_t = exp(-A d_t)
//     I_t  = alpha_t I_{t-1} + (1 - alpha_t) I_prior + beta_i k_j^2
//     mu_t = alpha_t (I_{t-1}/I_t) mu_{t-1} + beta_i v_i k_j / I_t
//     o_t[i] = sum_j mu_t[i][j] q_j
//
// How it is computed.  Write J = I - I_prior and eta = I mu.  The two
// updates above are then exactly
//     J_t   = alpha_t J_{t-1}   + beta_i k_j^2
//     eta_t = alpha_t eta_{t-1} + beta_i v_i k_j,      mu_t = eta_t / (I_prior + J_t)
// (the information form).  The kernel stores the state multiplied by a
// per-head working scale W_t (Jw = W J, Ew = W eta) with
//     W_t = W_{t-1} / alpha_t * 2^{-r_t},
// r_t an integer chosen so that W stays in [1, 2^48).  Per element and token
// the update then needs no multiply by alpha:
//     Jw <- f_t Jw + (W beta_i) k_j^2,  Ew <- f_t Ew + (W beta_i v_i) k_j,
// with f_t = 2^{-r_t} = 1 on all but the rare rescaling tokens (where the
// multiply is exact).  The readout divides per element:
//     mu q = sigma * q_j Ew / (sigma Jw + sigma W I_prior),  sigma = 2^-24,
// where sigma centres the scaled denominators on 1 so that products of two
// of them stay in range (the row sum is scaled back by sigma).  Pairs of
// quotients may share one reciprocal,
// n1/d1 + n2/d2 = (n1 d2 + n2 d1) / (d1 d2), which trades one MUFU op for one
// FP32 op; PAIRS of the 4 column-pair groups of a lane row are combined that
// way to balance the FMA pipe (128 lanes/clk/SM) against the MUFU pipe
// (16 rcp/clk/SM).  Element arithmetic uses packed FFMA2/FMUL2.
//
// Work decomposition.  Every state element is an independent scalar
// recurrence; only the readout reduces over j.  A CTA owns 128 consecutive
// state rows (whole heads: 128/d_v of them) for a token range and keeps them
// in registers for the whole range.  It has d_k/16 warps; a lane holds 4 rows
// x 16 columns (64 elements, 128 fp32 registers).  The readout's row sums
// over the d_k/16 lanes of a row set go through shared memory: each lane
// stores its 4 row partials every token, and every RB tokens the warp adds
// the partials of each row and writes whole 16-byte row quads (no shuffle
// latency on the token loop).  There is no producer warp (a ninth warp would
// cap registers at 168 per thread); instead:
//   * q, k, v, beta, d of each chunk of TC tokens are brought into shared
//     memory by 1-D bulk TMA copies that complete on an mbarrier; the warp
//     that finishes a chunk last refills its stage with the chunk three
//     ahead (no warp ever blocks on stage reuse);
//   * one chunk ahead of its compute, every warp converts its share of the
//     next chunk's tokens k -> (k, k^2) and q to fp32 in a bank-conflict-free
//     interleaved layout, and one warp (rotating with the chunk) runs the
//     per-head scale recursion (W_t, f_t) over the chunk's tokens; lanes then
//     read (f_t, W_t, sigma W_t I_prior) with one shared load per token; all
//     arrive on the chunk's "params ready" barrier.
// All waits are bounded by GPU time and record KDN_ERR_TIMEOUT instead of
// blocking forever.
// Long sequences with few heads are split into P token ranges (parts): an
// aggregate pass (AGG = true: updates only, zero initial state, no readout)
// gives each part's end state, a carry pass chains them, and the full pass
// runs every part from its carried start state.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "kdn_device.cuh"
#include "kdn_internal.h"
#include "mobius_device.cuh"

namespace kdn {
namespace diag {
// everything here is instantiated per translation unit (one per input dtype)
namespace {

constexpr int RT = 4;            // rows per lane
constexpr int CW = 16;           // columns per lane
constexpr int NSTAGE = 3;        // chunks in flight
constexpr int ROWS_PER_CTA = 128;
constexpr int PAIRS = 3;         // of the 4 column-pair groups of a lane row, how many share reciprocals
constexpr float SIGMA = 5.9604644775390625e-08f;   // 2^-24
constexpr float INV_SIGMA = 16777216.f;             // 2^24
constexpr float W_LIMIT = 281474976710656.0f;      // 2^48
constexpr float LOG2E = 1.4426950408889634f;
// Readout reduction through shared memory: every token each lane stores its 4
// row partials; every RB tokens the warp sums the column groups of each row
// and stores whole 16-byte row quads.
constexpr int RB = 8;

// Floats one token's row partials take in a warp's reduction buffer, laid
// out [row set][column group][4 rows]: a row set takes 4 M + 4 floats and the
// token 16 (mod 32) more than a multiple of 32, so that the 16-byte stores of
// a quarter warp and the summing reads of consecutive row sets and tokens
// fall on different banks.  m = lanes per row set (d_k / 16).
__host__ __device__ constexpr int red_rs_stride(int m) { return 4 * m + 4; }
__host__ __device__ constexpr int red_token_stride(int m) {
    return (32 / m) * red_rs_stride(m) + (16 - ((32 / m) * red_rs_stride(m)) % 32 + 32) % 32;
}

struct AggScale {
    float W;   // working scale at the end of the part (zero start, W = 1 at its start)
    int R;     // total power-of-two exponent removed by rescaling within the part
};

struct Params {
    const void* q;
    const void* k;
    const void* v;
    const void* beta;
    const void* d;
    const float* A;
    float I_prior;
    const float* I0;
    const float* mu0;
    float* out;              // [BH, out_ld, dv] (full pass) or unused (aggregate pass)
    long long out_ld;        // tokens between consecutive heads' rows of out
    long long d_ld;          // tokens between consecutive heads' rows of d
    float* final_state;      // [2,BH,dv,dk] or null
    float* agg;              // [P-1][BH][2][dv][dk] part end states / carried start states
    AggScale* agg_scale;     // [P-1][BH]
    long long BH;
    long long ctas;          // CTAs per token part (head groups)
    int P;                   // token parts of this pass
    int H, T, dv;
    int part_len;            // tokens per part (multiple of TC)
    int TC;                  // tokens per chunk
    int d_tma;               // 1: d staged by TMA (aligned), 0: plain loads
    long long wait_ns;
    // per-head Moebius lambda run by extra CTAs of the full pass (nlam of
    // them, after the ctas * P scan CTAs): [BH, T] coefficients (rows 16-byte
    // aligned, T % 4 == 0), lam0 [BH], lam_out [BH, T]; nlam = 0: none
    const float* ma;
    const float* mb;
    const float* mc;
    const float* md;
    const float* lam0;
    float* lam_out;
    int nlam;
};

template <int DK>
struct Geo {
    static constexpr int M = DK / CW;              // lanes sharing a row set
    static constexpr int RS = 32 / M;              // row sets per warp
    static constexpr int WR = RS * RT;             // rows per warp
    static constexpr int NW = ROWS_PER_CTA / WR;   // warps per CTA (= M)
    static constexpr int NTHREADS = NW * 32;
    static constexpr int PAR_FLOATS = 3 * DK + 4;  // per token: k, k^2, q, then (f, W, sigma W I_prior, 0)
};

// shared-memory layout of one chunk stage for `hpc` heads
struct Layout {
    int raw_qk, raw_vb, raw_d, par;   // bytes per head of each region
    int head, stage;                  // bytes per head, per stage
    __host__ __device__ Layout(int dk, int dv, int es, int TC, int hpc) {
        raw_qk = TC * dk * es;
        raw_vb = TC * dv * es;
        raw_d = (TC * es + 15) & ~15;
        par = TC * (3 * dk + 4) * 4;
        head = 2 * raw_qk + 2 * raw_vb + raw_d + par;
        stage = hpc * head;
    }
};

// per warp: RB tokens of row partials
__host__ __device__ constexpr int red_bytes_per_warp(int dk) { return RB * red_token_stride(dk / CW) * 4; }

__host__ __device__ inline int smem_bytes(int dk, int dv, int es, int TC) {
    const int hpc = ROWS_PER_CTA / dv;
    Layout L(dk, dv, es, TC, hpc);
    const int nw = dk / CW;   // warps per CTA
    return NSTAGE * L.stage + nw * red_bytes_per_warp(dk) + 2 * NSTAGE * 8 + NSTAGE * 4 + 2 * hpc * 4;
}

// one error word per translation unit that instantiates these kernels
__device__ int g_diag_error = 0;

template <typename TIn>
__device__ __forceinline__ float to_f32(TIn x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// four consecutive inputs -> fp32 (8-byte or 16-byte aligned shared memory)
__device__ __forceinline__ void load4(const float* p, float* o) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* o) {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    o[0] = __uint_as_float(x.x << 16);
    o[1] = __uint_as_float(x.x & 0xffff0000u);
    o[2] = __uint_as_float(x.y << 16);
    o[3] = __uint_as_float(x.y & 0xffff0000u);
}

// two consecutive inputs -> fp32
__device__ __forceinline__ float2 load2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load2(const __nv_bfloat16* p) {
    const uint32_t x = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// hardware reciprocal (MUFU), max relative error 2^-23 per the PTX ISA;
// denormal results flush to zero (the scaled denominators stay normal)
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// The per-head scale recursion for one token (see the header comment):
// returns f_t = 2^-r_t and updates (W, R).  x = A d / ln 2.
__device__ __forceinline__ float scale_step(float x, float& W, int& R) {
    float p;
    int r;
    if (fabsf(x) <= 64.f) {
        p = W * exp2f(x);                      // in [2^-64, 2^112)
        if (p >= 1.f && p < W_LIMIT) {
            r = 0;
        } else {
            r = exponent_of(p);
            p = __int_as_float(__float_as_int(p) - (r << 23));
        }
    } else if (x > 64.f) {                     // very fast forgetting (or +inf)
        const float n = fminf(floorf(x), 1.0e6f);
        p = W * exp2f(x - n);                  // x - n in [0, 1)
        const int e = exponent_of(p);
        p = __int_as_float(__float_as_int(p) - (e << 23));
        r = e + static_cast<int>(n);
        if (!(x < __int_as_float(0x7f800000))) p = 1.f;   // x = +inf: W restarts at 1
    } else if (x < -64.f) {                    // growth (alpha > 1)
        const float n = fmaxf(floorf(x), -1.0e6f);
        p = W * exp2f(x - n);
        const int e = exponent_of(p);
        p = __int_as_float(__float_as_int(p) - (e << 23));
        r = e + static_cast<int>(n);
    } else {                                   // NaN propagates
        p = x;
        r = 0;
    }
    // beyond +-4096 the factor is 0 or inf anyway; keep R in int range
    r = max(-4096, min(4096, r));
    W = p;
    R = max(-(1 << 30), min(1 << 30, R + r));
    return r == 0 ? 1.f : pow2i(-r);
}

template <int DK, typename TIn, bool AGG, bool LIN>
__global__ void __launch_bounds__(Geo<DK>::NTHREADS, (DK >= 128 ? 1 : 2))
diag_scan_kernel(const Params p) {
    using G = Geo<DK>;
    constexpr int M = G::M, NW = G::NW, PF = G::PAR_FLOATS;
    constexpr int ES = sizeof(TIn);
    extern __shared__ __align__(128) unsigned char smem[];

    const int dv = p.dv, HPC = ROWS_PER_CTA / dv, TC = p.TC;
    const Layout L(DK, dv, ES, TC, HPC);
    constexpr int RSS = red_rs_stride(M), RTS = red_token_stride(M);
    float* red_all = reinterpret_cast<float*>(smem + NSTAGE * L.stage);   // [NW][RB][RTS]
    uint64_t* full_raw = reinterpret_cast<uint64_t*>(smem + NSTAGE * L.stage + NW * red_bytes_per_warp(DK));
    uint64_t* full_par = full_raw + NSTAGE;
    int* done_cnt = reinterpret_cast<int*>(full_par + NSTAGE);
    float* w_state = reinterpret_cast<float*>(done_cnt + NSTAGE);   // [HPC] scale W per head
    int* r_state = reinterpret_cast<int*>(w_state + HPC);             // [HPC] exponent sum R
    auto region = [&](int s, int h, int off) { return smem + s * L.stage + h * L.head + off; };
    auto raw_q = [&](int s, int h) { return reinterpret_cast<TIn*>(region(s, h, 0)); };
    auto raw_k = [&](int s, int h) { return reinterpret_cast<TIn*>(region(s, h, L.raw_qk)); };
    auto raw_v = [&](int s, int h) { return reinterpret_cast<TIn*>(region(s, h, 2 * L.raw_qk)); };
    auto raw_b = [&](int s, int h) {
        return reinterpret_cast<TIn*>(region(s, h, 2 * L.raw_qk + L.raw_vb));
    };
    auto raw_d = [&](int s, int h) {
        return reinterpret_cast<TIn*>(region(s, h, 2 * L.raw_qk + 2 * L.raw_vb));
    };
    auto par = [&](int s, int h) {
        return reinterpret_cast<float*>(region(s, h, 2 * L.raw_qk + 2 * L.raw_vb + L.raw_d));
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // linear grid: part-major scan CTAs (head group fastest), then the lambda
    // walkers of the full pass
    const long long lin = blockIdx.x;
    if (lin >= p.ctas * p.P) {
        if constexpr (!AGG && !LIN) {
            const int tps = static_cast<int>((p.T + mob::Walk<G::NTHREADS>::TILE - 1) / mob::Walk<G::NTHREADS>::TILE);
            mob::mobius_walk<G::NTHREADS>(p.ma, p.mb, p.mc, p.md, p.lam0, p.lam_out, p.BH, p.T, tps,
                                          lin - p.ctas * p.P, p.nlam, p.wait_ns, smem, &g_diag_error);
        }
        return;
    }
    const int part = static_cast<int>(lin / p.ctas);
    const long long head0 = (lin - static_cast<long long>(part) * p.ctas) * HPC;
    const int nheads = static_cast<int>(min(static_cast<long long>(HPC), p.BH - head0));
    const int T = p.T;
    const int tb = min(T, part * p.part_len);
    const int te = min(T, tb + p.part_len);
    const int nchunks = (te - tb + TC - 1) / TC;
    const TIn* gq = static_cast<const TIn*>(p.q);
    const TIn* gk = static_cast<const TIn*>(p.k);
    const TIn* gv = static_cast<const TIn*>(p.v);
    const TIn* gb = static_cast<const TIn*>(p.beta);
    const TIn* gd = static_cast<const TIn*>(p.d);
    const float Ip = p.I_prior;

    // Issue the bulk copies of chunk c into its stage (one warp, all lanes).
    auto issue = [&](int c) {
        const int s = c % NSTAGE;
        const int t0 = tb + c * TC, tcn = min(TC, te - t0);
        const int dbytes = p.d_tma ? tcn * ES : 0;
        if (lane == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&full_raw[s],
                                  static_cast<uint32_t>(nheads * (tcn * ((AGG ? 1 : 2) * DK + 2 * dv) * ES +
                                                                  dbytes)));
        }
        __syncwarp();
        for (int x = lane; x < nheads * 5; x += 32) {
            const int h = x / 5, which = x - h * 5;
            const long long tok = (head0 + h) * T + t0;
            if (which == 0) {
                if (!AGG) bulk_g2s(raw_q(s, h), gq + tok * DK, tcn * DK * ES, &full_raw[s]);
            } else if (which == 1) {
                bulk_g2s(raw_k(s, h), gk + tok * DK, tcn * DK * ES, &full_raw[s]);
            } else if (which == 2) {
                bulk_g2s(raw_v(s, h), gv + tok * dv, tcn * dv * ES, &full_raw[s]);
            } else if (which == 3) {
                bulk_g2s(raw_b(s, h), gb + tok * dv, tcn * dv * ES, &full_raw[s]);
            } else if (dbytes) {
                bulk_g2s(raw_d(s, h), gd + (head0 + h) * p.d_ld + t0, dbytes, &full_raw[s]);
            }
        }
    };

    bool ok = true;
    // Prepare chunk c once its copies have landed:
    //  * every warp converts its tokens (tt = warp, warp + NW, ...): k ->
    //    (k, k^2) and q to fp32, interleaved so that the 16-column group cg of
    //    a lane is float4 number (s4 * M + cg), s4 = 0..3;
    //  * warp c % NW runs the per-head scale recursion over the chunk's tokens
    //    (sequential in t; W and R carried across chunks in shared memory) and
    //    stores (f_t, W_t, sigma W_t I_prior) behind each token's columns.
    // Callers guarantee that chunk c-1's recursion has finished (they passed
    // the full_par wait of chunk c-1, which its recursion arrives on).
    auto prepare = [&](int c) {
        const int s = c % NSTAGE;
        const int t0 = tb + c * TC, tcn = min(TC, te - t0);
        if (!mbar_wait(&full_raw[s], (c / NSTAGE) & 1, p.wait_ns)) ok = false;
        constexpr int HP = DK / 2;   // column pairs per token
        for (int tt = warp; tt < tcn; tt += NW) {
            for (int x = lane; x < nheads * HP; x += 32) {
                const int h = x / HP;
                const int j = 2 * (x - h * HP);
                const int cgj = j / CW, jj = j % CW;
                const int pos = ((jj >> 2) * M + cgj) * 4 + (jj & 3);
                float* base = par(s, h) + tt * PF;
                const float2 kv = load2(raw_k(s, h) + tt * DK + j);
                *reinterpret_cast<float2*>(base + pos) = kv;
                if (!LIN) *reinterpret_cast<float2*>(base + DK + pos) = make_float2(kv.x * kv.x, kv.y * kv.y);
                if (!AGG) *reinterpret_cast<float2*>(base + 2 * DK + pos) = load2(raw_q(s, h) + tt * DK + j);
            }
        }
        if (warp == c % NW) {
            if (!p.d_tma) {
                for (int x = lane; x < nheads * tcn; x += 32) {
                    const int h = x / tcn, tt = x - h * tcn;
                    raw_d(s, h)[tt] = gd[(head0 + h) * p.d_ld + t0 + tt];
                }
                __syncwarp();
            }
            if (lane < nheads) {
                const float Ah = p.A[(head0 + lane) % p.H];
                float W = w_state[lane];
                int R = r_state[lane];
                const TIn* rd = raw_d(s, lane);
                float* ps = par(s, lane) + 3 * DK;
                uint32_t mask = 0;   // tokens of the chunk that rescale the state
                for (int tt = 0; tt < tcn; ++tt) {
                    const float f = scale_step(Ah * to_f32<TIn>(rd[tt]) * LOG2E, W, R);
                    *reinterpret_cast<float4*>(ps + tt * PF) = make_float4(f, W, W * Ip * SIGMA, 0.f);
                    if (f != 1.f) mask |= 1u << tt;
                }
                ps[3] = __uint_as_float(mask);   // 4th scalar of the chunk's first token
                w_state[lane] = W;
                r_state[lane] = R;
            }
        }
        mbar_arrive(&full_par[s]);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full_raw[s], 1);
            mbar_init(&full_par[s], NW * 32);
            done_cnt[s] = 0;
        }
        for (int h = 0; h < HPC; ++h) {
            w_state[h] = 1.f;
            r_state[h] = 0;
        }
        mbar_init_fence();
    }
    __syncthreads();
    if (warp == 0)
        for (int c = 0; c < min(NSTAGE, nchunks); ++c) issue(c);
    if (nchunks > 0) prepare(0);

    // ------------------------------ lane state ------------------------------
    const int rs = lane / M, cg = lane % M;
    const int crow = warp * G::WR + rs * RT;      // first of my rows within the CTA
    const int hl = crow / dv, i0 = crow - hl * dv;
    const bool active = hl < nheads;
    const long long bh = head0 + hl;
    const long long S = static_cast<long long>(dv) * DK;

    float2 J[RT][CW / 2], E[RT][CW / 2];
    {
        // initial state of this part, in scaled form (W = 1 at the part start)
        const float* src_J = nullptr;
        const float* src_E = nullptr;
        if (!AGG && part > 0) {
            src_J = p.agg + (static_cast<long long>(part - 1) * p.BH + bh) * 2 * S;
            src_E = src_J + S;
        }
#pragma unroll
        for (int r = 0; r < RT; ++r) {
#pragma unroll
            for (int c2 = 0; c2 < CW / 2; ++c2) {
                float2 j2 = make_float2(0.f, 0.f), e2 = make_float2(0.f, 0.f);
                const long long off = static_cast<long long>(i0 + r) * DK + cg * CW + 2 * c2;
                if (active && !AGG) {
                    if (src_J) {
                        j2 = *reinterpret_cast<const float2*>(src_J + off);
                        e2 = *reinterpret_cast<const float2*>(src_E + off);
                    } else if (part == 0 && (p.I0 || p.mu0)) {
                        float2 i02 = make_float2(Ip, Ip);
                        if (p.I0) i02 = *reinterpret_cast<const float2*>(p.I0 + bh * S + off);
                        j2 = make_float2(i02.x - Ip, i02.y - Ip);
                        if (p.mu0) {
                            const float2 m2 = *reinterpret_cast<const float2*>(p.mu0 + bh * S + off);
                            e2 = make_float2(i02.x * m2.x, i02.y * m2.y);
                        }
                    }
                }
                J[r][c2] = j2;
                E[r][c2] = e2;
            }
        }
    }

    float W = 1.f;
    float* gout = p.out;
    float* red = red_all + warp * (RB * RTS);
    // Sum the row partials of tokens t_first .. t_first + ntok - 1 (slots
    // 0 .. ntok-1) over the M column groups and store them: a work item is one
    // token and one row set (4 consecutive rows) of this warp.
    auto flush = [&](int t_first, int ntok) {
        constexpr int QUADS = G::RS;   // row sets per warp
        __syncwarp();
        for (int g = lane; g < ntok * QUADS; g += 32) {
            const int ts = g / QUADS, qd = g - ts * QUADS;
            const float* src = red + ts * RTS + qd * RSS;
            const float4 x0 = *reinterpret_cast<const float4*>(src);
            float2 lo = make_float2(x0.x, x0.y), hi = make_float2(x0.z, x0.w);
#pragma unroll
            for (int c = 1; c < M; ++c) {
                const float4 x = *reinterpret_cast<const float4*>(src + 4 * c);
                lo = __fadd2_rn(lo, make_float2(x.x, x.y));
                hi = __fadd2_rn(hi, make_float2(x.z, x.w));
            }
            const int crow_q = warp * G::WR + RT * qd;         // CTA row of the row set
            const int hq = crow_q / dv, iq = crow_q - hq * dv;
            if (hq < nheads) {
                lo = __fmul2_rn(lo, f2(SIGMA));
                hi = __fmul2_rn(hi, f2(SIGMA));
                float* o = gout + ((head0 + hq) * p.out_ld + t_first + ts) * dv + iq;
                __stcs(reinterpret_cast<float4*>(o), make_float4(lo.x, lo.y, hi.x, hi.y));
            }
        }
        __syncwarp();
    };
    for (int c = 0; c < nchunks; ++c) {
        const int s = c % NSTAGE;
        if (!mbar_wait(&full_par[s], (c / NSTAGE) & 1, p.wait_ns)) ok = false;
        if (c + 1 < nchunks) prepare(c + 1);
        const int t0 = tb + c * TC, tcn = min(TC, te - t0);
        const TIn* rv = raw_v(s, hl) + i0;
        const TIn* rb = raw_b(s, hl) + i0;
        const float* pbase = par(s, hl);
        // Tokens run in segments between rescaling tokens, so that the token
        // loop itself has no branch; the segment breaks are the union over
        // the warp's heads (a lane whose head does not rescale multiplies by 1).
        const uint32_t mask = __reduce_or_sync(
            0xffffffffu, active ? __float_as_uint(pbase[3 * DK + 3]) : 0u);
        int tt = 0;
        while (tt < tcn) {
            if ((mask >> tt) & 1u) {                 // exact power-of-two rescale
                const float2 f22 = f2(pbase[tt * PF + 3 * DK]);
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int c2 = 0; c2 < CW / 2; ++c2) {
                        if (!LIN) J[r][c2] = __fmul2_rn(J[r][c2], f22);
                        E[r][c2] = __fmul2_rn(E[r][c2], f22);
                    }
            }
            const uint32_t later = mask >> (tt + 1);   // tt + 1 <= TC <= 16
            const int stop = later ? min(tcn, tt + __ffs(later)) : tcn;
        for (; tt < stop; ++tt) {
            const float* pt = pbase + tt * PF;
            const float4 sc = *reinterpret_cast<const float4*>(pt + 3 * DK);
            float bet[RT], val[RT];
            load4(rb + tt * dv, bet);
            load4(rv + tt * dv, val);
            W = sc.y;
            float2 SB[RT], SBV[RT];
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                const float sb = W * bet[r];
                SB[r] = f2(sb);
                SBV[r] = f2(sb * val[r]);
            }
            const float2 SP = f2(sc.z), SG = f2(SIGMA);
            float2 acc[RT];
#pragma unroll
            for (int r = 0; r < RT; ++r) acc[r] = make_float2(0.f, 0.f);
            if constexpr (LIN) {
                // importance held at I_prior: Ew <- Ew + (W beta_i v_i) k_j and
                // o_i = sum_j q_j Ew_ij / (W I_prior) (one scale per token)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float2 kf[4], qv[4];
#pragma unroll
                    for (int h4 = 0; h4 < 2; ++h4) {
                        const int f4 = ((2 * half + h4) * M + cg) * 4;
                        const float4 a = *reinterpret_cast<const float4*>(pt + f4);
                        kf[2 * h4] = make_float2(a.x, a.y);
                        kf[2 * h4 + 1] = make_float2(a.z, a.w);
                        if (!AGG) {
                            const float4 q = *reinterpret_cast<const float4*>(pt + 2 * DK + f4);
                            qv[2 * h4] = make_float2(q.x, q.y);
                            qv[2 * h4 + 1] = make_float2(q.z, q.w);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < RT; ++r)
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const int c2 = half * 4 + c4;
                            E[r][c2] = __ffma2_rn(SBV[r], kf[c4], E[r][c2]);
                            if (!AGG) acc[r] = __ffma2_rn(qv[c4], E[r][c2], acc[r]);
                        }
                }
                if (!AGG) {
                    // the flush multiplies by sigma: store sum / (sigma W I_prior)
                    const float rz = 1.f / sc.z;
#pragma unroll
                    for (int r = 0; r < RT; ++r) acc[r] = __fmul2_rn(acc[r], f2(rz));
                }
            } else {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                // this lane's 8 columns of the half: float4 numbers (2*half+h4)*M + cg
                float2 kf[4], kk[4], qv[4];
#pragma unroll
                for (int h4 = 0; h4 < 2; ++h4) {
                    const int f4 = ((2 * half + h4) * M + cg) * 4;
                    const float4 a = *reinterpret_cast<const float4*>(pt + f4);
                    const float4 b = *reinterpret_cast<const float4*>(pt + DK + f4);
                    kf[2 * h4] = make_float2(a.x, a.y);
                    kf[2 * h4 + 1] = make_float2(a.z, a.w);
                    kk[2 * h4] = make_float2(b.x, b.y);
                    kk[2 * h4 + 1] = make_float2(b.z, b.w);
                    if (!AGG) {
                        const float4 q = *reinterpret_cast<const float4*>(pt + 2 * DK + f4);
                        qv[2 * h4] = make_float2(q.x, q.y);
                        qv[2 * h4 + 1] = make_float2(q.z, q.w);
                    }
                }
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    float2 den[4], num[4];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int c2 = half * 4 + c4;
                        J[r][c2] = __ffma2_rn(SB[r], kk[c4], J[r][c2]);
                        E[r][c2] = __ffma2_rn(SBV[r], kf[c4], E[r][c2]);
                        if (!AGG) {
                            den[c4] = __ffma2_rn(J[r][c2], SG, SP);
                            num[c4] = __fmul2_rn(qv[c4], E[r][c2]);
                        }
                    }
                    if (!AGG) {
                        // column-pair groups (0,1) and (2,3) of this half; group
                        // g of every half shares reciprocals when g < PAIRS / 2
#pragma unroll
                        for (int g = 0; g < 2; ++g) {
                            const int x = 2 * g, y = 2 * g + 1;
                            if (2 * g + half < PAIRS) {
                                const float2 N = __ffma2_rn(num[x], den[y], __fmul2_rn(num[y], den[x]));
                                const float2 Dn = __fmul2_rn(den[x], den[y]);
                                acc[r] = __ffma2_rn(N, make_float2(rcp_approx(Dn.x), rcp_approx(Dn.y)), acc[r]);
                            } else {
                                acc[r] = __ffma2_rn(num[x], make_float2(rcp_approx(den[x].x), rcp_approx(den[x].y)), acc[r]);
                                acc[r] = __ffma2_rn(num[y], make_float2(rcp_approx(den[y].x), rcp_approx(den[y].y)), acc[r]);
                            }
                        }
                    }
                }
            }
            }
            if (!AGG) {
                const int slot = tt & (RB - 1);
                *reinterpret_cast<float4*>(red + slot * RTS + rs * RSS + 4 * cg) =
                    make_float4(acc[0].x + acc[0].y, acc[1].x + acc[1].y, acc[2].x + acc[2].y,
                                acc[3].x + acc[3].y);
                if (slot == RB - 1 || tt == tcn - 1) flush(t0 + tt - slot, slot + 1);
            }
        }
        }
        // the warp that finishes this chunk last refills the stage
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&done_cnt[s], 1) == NW - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            if (lane == 0) done_cnt[s] = 0;
            if (c + NSTAGE < nchunks) issue(c + NSTAGE);
        }
    }
    if (!ok) record_error(&g_diag_error, KDN_ERR_TIMEOUT);
    if (!active) return;

    if (AGG) {
        float* dJ = p.agg + (static_cast<long long>(part) * p.BH + bh) * 2 * S;
        float* dE = dJ + S;
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int c2 = 0; c2 < CW / 2; ++c2) {
                const long long off = static_cast<long long>(i0 + r) * DK + cg * CW + 2 * c2;
                *reinterpret_cast<float2*>(dJ + off) = J[r][c2];
                *reinterpret_cast<float2*>(dE + off) = E[r][c2];
            }
        // the head's scale state after the part: W of its last token, total R
        if (i0 == 0 && cg == 0) p.agg_scale[static_cast<long long>(part) * p.BH + bh] = {W, r_state[hl]};
    } else if (LIN && p.final_state && part == p.P - 1) {
        // mu_T = Ew / (W I_prior)
        float* fm = p.final_state + bh * S;
        const float rw = 1.f / (W * Ip);
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int c2 = 0; c2 < CW / 2; ++c2) {
                const long long off = static_cast<long long>(i0 + r) * DK + cg * CW + 2 * c2;
                *reinterpret_cast<float2*>(fm + off) = __fmul2_rn(E[r][c2], f2(rw));
            }
    } else if (p.final_state && part == p.P - 1) {
        // mu_T = eta / (I_prior + J) = Ew / (Jw + W I_prior);  I_T = Jw / W + I_prior
        float* fm = p.final_state + bh * S;
        float* fi = p.final_state + (p.BH + bh) * S;
        const float wI = W * Ip;
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int c2 = 0; c2 < CW / 2; ++c2) {
                const long long off = static_cast<long long>(i0 + r) * DK + cg * CW + 2 * c2;
                const float2 j2 = J[r][c2], e2 = E[r][c2];
                *reinterpret_cast<float2*>(fm + off) =
                    make_float2(e2.x / (j2.x + wI), e2.y / (j2.y + wI));
                *reinterpret_cast<float2*>(fi + off) = make_float2(j2.x / W + Ip, j2.y / W + Ip);
            }
    }
}

// Carry pass: chains the part end states.  For part p (p = 0..P-2) the end
// state from the true start state X is X * prod(alpha) + Delta with
// prod(alpha) = 2^-R / W_end and Delta = (Jw, Ew) / W_end of the aggregate
// pass.  Overwrites agg[p] with the start state of part p+1.
__global__ void diag_carry_kernel(float* agg, const AggScale* scl, const float* I0,
                                  const float* mu0, float I_prior, long long BH, long long S,
                                  int P) {
    grid_dep_signal();   // the full pass may start its prologue (it waits before reading agg)
    // four consecutive elements of one head per thread (S is a multiple of 4)
    const long long idx = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (idx >= BH * S) return;
    const long long bh = idx / S, e = idx - bh * S;
    float4 Jv = make_float4(0.f, 0.f, 0.f, 0.f), Ev = Jv;
    if (I0 || mu0) {
        const float4 i0 = I0 ? *reinterpret_cast<const float4*>(I0 + idx)
                             : make_float4(I_prior, I_prior, I_prior, I_prior);
        Jv = make_float4(i0.x - I_prior, i0.y - I_prior, i0.z - I_prior, i0.w - I_prior);
        if (mu0) {
            const float4 m = *reinterpret_cast<const float4*>(mu0 + idx);
            Ev = make_float4(i0.x * m.x, i0.y * m.y, i0.z * m.z, i0.w * m.w);
        }
    }
    auto step = [](float x, int R, float d, float W) { return (ldexpf(x, -R) + d) / W; };
#pragma unroll 4
    for (int pp = 0; pp + 1 < P; ++pp) {
        const AggScale a = scl[static_cast<long long>(pp) * BH + bh];
        float4* dJ = reinterpret_cast<float4*>(agg + (static_cast<long long>(pp) * BH + bh) * 2 * S + e);
        float4* dE = reinterpret_cast<float4*>(reinterpret_cast<float*>(dJ) + S);
        const float4 j = *dJ, h = *dE;
        Jv = make_float4(step(Jv.x, a.R, j.x, a.W), step(Jv.y, a.R, j.y, a.W), step(Jv.z, a.R, j.z, a.W),
                         step(Jv.w, a.R, j.w, a.W));
        Ev = make_float4(step(Ev.x, a.R, h.x, a.W), step(Ev.y, a.R, h.y, a.W), step(Ev.z, a.R, h.z, a.W),
                         step(Ev.w, a.R, h.w, a.W));
        *dJ = Jv;
        *dE = Ev;
    }
}


}  // namespace
}  // namespace diag
}  // namespace kdn

// the aggregate pass on the tensor cores (uses AggScale, LOG2E, g_diag_error)
#include "diag_agg_tc.cuh"
// the non-metaplastic full pass on the tensor cores (d = 128, bf16)
#include "lin_tc.cuh"
// the warp-specialised full pass of the metaplastic scan (d_k = 64, 128)
#include "diag_ws.cuh"

namespace kdn {
namespace diag {
namespace {

// ---------------------------------------------------------------------------
// host side

struct Cache {
    bool init[64] = {};
    int occ[64] = {};
};

// Opt the tensor-core aggregate kernels into their shared memory (once per
// device).
cudaError_t agg_tc_prepare() {
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) dev = 0;
    if (!done[dev]) {
        e = cudaFuncSetAttribute(diag_agg_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AggShape<16>::SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(diag_agg_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AggShape<32>::SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(diag_agg_tc_kernel<32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AggShape<32>::SMEM);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    return cudaSuccess;
}

template <int DK, typename TIn, bool AGG, bool LIN>
cudaError_t prepare(int dev, int smem, int* occ) {
    static Cache cache;
    static int smem_set[64] = {};
    auto kern = diag_scan_kernel<DK, TIn, AGG, LIN>;
    cudaError_t e = cudaSuccess;
    if (dev < 0 || dev >= 64) dev = 0;
    if (smem > smem_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        smem_set[dev] = smem;
        cache.init[dev] = false;
    }
    if (!cache.init[dev]) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Geo<DK>::NTHREADS, smem);
        if (e != cudaSuccess) return e;
        cache.occ[dev] = n > 0 ? n : 1;
        cache.init[dev] = true;
    }
    *occ = cache.occ[dev];
    return e;
}

// Whether the metaplastic full pass may take the warp-specialised kernel.
constexpr bool kWsFullPass = true;

// Whether a split call's aggregate pass runs on the tensor cores.
template <int DK, typename TIn>
constexpr bool tc_aggregates(int dv) {
    return DK == AG_D && std::is_same<TIn, __nv_bfloat16>::value && dv == AG_D;
}

// Launch plan of one call: chunk length, token parts, scratch bytes.
struct Plan {
    int TC = 16;
    int smem = 0;
    int P = 1;
    int part_len = 1;
    long long ctas = 0;      // CTAs per part of the CUDA-core kernel (aggregate pass)
    size_t scratch = 0;
    int kernels = 0;
    int occ = 1;             // resident full-pass CTAs per SM
    // full pass: the warp-specialised kernel (ws) or diag_scan_kernel
    bool ws = false;
    long long ctas_full = 0; // CTAs per part of the full pass
    int TC_full = 16;
    int smem_full = 0;
};

// Set-up of the warp-specialised full pass on the current device: opts it
// into its shared memory and checks that it was built with the launch
// register allocation its setmaxnreg split assumes (else the split could
// wait forever: the caller then keeps the CUDA-core kernel).
template <int DK, typename TIn, int TC>
cudaError_t ws_prepare(int dev, int smem, bool* usable) {
    static int smem_set[64] = {};
    static int regs_ok[64] = {};   // 0 unknown, 1 yes, 2 no
    if (dev < 0 || dev >= 64) dev = 0;
    auto kern = diag_ws_kernel<DK, TIn, TC>;
    if (regs_ok[dev] == 0) {
        cudaFuncAttributes fa;
        const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        regs_ok[dev] = fa.numRegs == WS_LAUNCH_REG ? 1 : 2;
    }
    *usable = regs_ok[dev] == 1;
    if (*usable && smem > smem_set[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        smem_set[dev] = smem;
    }
    return cudaSuccess;
}

template <int DK, typename TIn, bool LIN>
kdn_status plan_dk(const DiagArgs& a, Plan* pl) {
    constexpr int ES = sizeof(TIn);
    const int dv = a.dv;
    const int hpc = ROWS_PER_CTA / dv;
    const long long BH = static_cast<long long>(a.B) * a.H;
    pl->ctas = (BH + hpc - 1) / hpc;
    if (pl->ctas > 0x7fffffffLL) return KDN_ERR_INVALID_ARG;
    // chunk length: as long as the three stages fit the budget
    const int budget = (DK >= 128) ? 200 * 1024 : 100 * 1024;
    int TC = 16;
    while (TC > 1 && smem_bytes(DK, dv, ES, TC) > budget) TC >>= 1;
    pl->TC = TC;
    pl->smem = smem_bytes(DK, dv, ES, TC);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return from_cuda(e);
    int occ = 1, occ_agg = 1;
    e = prepare<DK, TIn, false, LIN>(dev, pl->smem, &occ);
    if (e != cudaSuccess) return from_cuda(e);
    e = prepare<DK, TIn, true, LIN>(dev, pl->smem, &occ_agg);
    if (e != cudaSuccess) return from_cuda(e);
    pl->occ = occ;
    pl->ctas_full = pl->ctas;
    pl->TC_full = TC;
    pl->smem_full = pl->smem;
    if constexpr (kWsFullPass && !LIN && (DK == 64 || DK == 128)) {
        // warp-specialised full pass: chunks of 16 tokens when they fit (never
        // longer than the aggregate pass's, so parts hold whole chunks of both)
        using WG = WsGeo<DK>;
        if (WG::ROWS % dv == 0) {
            int tcw = 16;
            while (tcw > 8 && ws_smem_bytes<DK>(dv, ES, tcw) > 227 * 1024) tcw >>= 1;
            tcw = std::min(tcw, TC);
            const int smem_ws = std::max(ws_smem_bytes<DK>(dv, ES, tcw), mob::Walk<WS_THREADS>::SMEM);
            bool usable = false;
            if (tcw >= 8 && smem_ws <= 227 * 1024) {
                e = tcw == 16 ? ws_prepare<DK, TIn, 16>(dev, smem_ws, &usable)
                              : ws_prepare<DK, TIn, 8>(dev, smem_ws, &usable);
                if (e != cudaSuccess) return from_cuda(e);
            }
            if (usable) {
                pl->ws = true;
                pl->TC_full = tcw;
                pl->smem_full = smem_ws;
                const int hpcw = WG::ROWS / dv;
                pl->ctas_full = (BH + hpcw - 1) / hpcw;
                pl->occ = occ = 1;
            }
        }
    }
    // token split: enough parts to give every CTA slot work
    const long long slots = static_cast<long long>(sm_count()) * occ;
    int P = 1;
    if (pl->ctas_full * 2 <= slots && a.T >= 8 * TC) {
        const long long want = slots / pl->ctas_full;
        const long long maxp = a.T / (4 * TC);
        P = static_cast<int>(want < maxp ? want : maxp);
        if (P < 1) P = 1;
    }
    // Fill split.  With d_k = d_v = 128 and bf16 inputs the aggregate pass
    // runs on the tensor cores and costs little, so the part count is chosen
    // by a model in full-pass token steps of one CTA: waves x part length,
    // plus for a split 23 (two extra launches), 0.07 per extra (head, part)
    // (carry and start-state traffic) and 6.6e-4 per token of an extra
    // (head, part) (the aggregate pass), fitted to GB300 timings of the
    // 750M-shaped layer and the 65536-token context.  Every count that
    // keeps parts at least 8 chunks long is weighed, the slot-filling one
    // above included; a split is taken when it saves more than 2 %.
    if (!LIN && tc_aggregates<DK, TIn>(dv) && a.T >= 32 * TC) {
        auto est = [&](int parts, int plen) {
            const long long waves = (pl->ctas_full * parts + slots - 1) / slots;
            const double extra = static_cast<double>(BH) * (parts - 1);
            return static_cast<double>(waves) * plen +
                   (parts > 1 ? 23.0 + extra * (0.07 + 6.6e-4 * plen) : 0.0);
        };
        auto plen_of = [&](int cand) { return ((a.T + cand - 1) / cand + TC - 1) / TC * TC; };
        const double one = est(1, a.T);
        double best = one;
        int bestP = 1;
        for (int cand = 2; cand <= 64; ++cand) {
            const int plen = plen_of(cand);
            if (plen < 8 * TC) break;
            const int pe = (a.T + plen - 1) / plen;
            const double e = est(pe, plen);
            if (e < best) {
                best = e;
                bestP = pe;
            }
        }
        P = best < 0.98 * one ? bestP : 1;
    }
    int part_len = a.T > 0 ? a.T : 1;
    if (P > 1) {
        part_len = ((a.T + P - 1) / P + TC - 1) / TC * TC;
        P = (a.T + part_len - 1) / part_len;
        if (P <= 1) {
            P = 1;
            part_len = a.T;
        }
    }
    pl->P = P;
    pl->part_len = part_len;
    const long long S = static_cast<long long>(dv) * DK;
    pl->scratch = P > 1 ? static_cast<size_t>(P - 1) * BH * (2 * S * sizeof(float) + sizeof(AggScale)) : 0;
    pl->kernels = P > 1 ? 3 : 1;
    return KDN_OK;
}

template <int DK, typename TIn, bool LIN>
kdn_status launch_dk(const DiagArgs& a, cudaStream_t st, long long wait_ns) {
    constexpr int ES = sizeof(TIn);
    Plan pl;
    kdn_status ps = plan_dk<DK, TIn, LIN>(a, &pl);
    if (ps != KDN_OK) return ps;
    const int dv = a.dv, TC = pl.TC, smem = pl.smem, P = pl.P;
    const long long BH = static_cast<long long>(a.B) * a.H;
    const long long ctas = pl.ctas;

    Params prm{};
    prm.q = a.q; prm.k = a.k; prm.v = a.v; prm.beta = a.beta; prm.d = a.d;
    prm.A = a.A; prm.I_prior = a.I_prior; prm.I0 = a.I0; prm.mu0 = a.mu0;
    prm.out = a.out; prm.final_state = a.final_state;
    prm.out_ld = a.out_ld > 0 ? a.out_ld : a.T;
    prm.d_ld = a.d_ld > 0 ? a.d_ld : a.T;
    prm.BH = BH; prm.H = a.H; prm.T = a.T; prm.dv = dv;
    prm.ctas = ctas; prm.P = P;
    prm.part_len = pl.part_len; prm.TC = TC; prm.wait_ns = wait_ns;
    // d chunks can be bulk-copied when every chunk starts and ends on 16 bytes
    prm.d_tma = (static_cast<long long>(a.T) * ES % 16 == 0) && (TC * ES % 16 == 0) &&
                (prm.d_ld * ES % 16 == 0) && ((reinterpret_cast<uintptr_t>(a.d) & 15u) == 0);

    void* scratch = nullptr;
    cudaError_t e = cudaSuccess;
    const long long S = static_cast<long long>(dv) * DK;
    if (P > 1) {
        const size_t state_bytes = static_cast<size_t>(P - 1) * BH * 2 * S * sizeof(float);
        e = cudaMallocAsync(&scratch, pl.scratch, st);
        if (e != cudaSuccess) return from_cuda(e);
        prm.agg = static_cast<float*>(scratch);
        prm.agg_scale = reinterpret_cast<AggScale*>(static_cast<char*>(scratch) + state_bytes);
        if (tc_aggregates<DK, TIn>(dv)) {
            e = agg_tc_prepare();
            if (e == cudaSuccess) {
                AggArgs ag{static_cast<const __nv_bfloat16*>(a.k), static_cast<const __nv_bfloat16*>(a.beta),
                           static_cast<const __nv_bfloat16*>(a.v), static_cast<const __nv_bfloat16*>(a.d),
                           a.A, prm.agg, prm.agg_scale, BH, a.H, a.T, prm.d_ld, pl.part_len, wait_ns};
                // two CTAs per SM when the grid fills them, else one wider CTA per SM
                const dim3 grid(static_cast<unsigned>(BH), P - 1);
                if constexpr (LIN) {
                    // the non-metaplastic limit needs only the eta aggregates; its
                    // parts come from the first rule of plan_dk alone, so BH * (P - 1)
                    // stays below one wave of full-pass CTAs: always one CTA per SM
                    diag_agg_tc_kernel<32, true><<<grid, AggShape<32>::THREADS, AggShape<32>::SMEM, st>>>(ag);
                } else {
                    // the two-CTA variant when it fills both slots of every SM
                    // (288 CTAs on 152 SMs: two waves of the one-CTA variant
                    // measured 280 us, one wave of the two-CTA variant 294 us)
                    if (BH * (P - 1) >= 2LL * sm_count())
                        diag_agg_tc_kernel<16><<<grid, AggShape<16>::THREADS, AggShape<16>::SMEM, st>>>(ag);
                    else
                        diag_agg_tc_kernel<32><<<grid, AggShape<32>::THREADS, AggShape<32>::SMEM, st>>>(ag);
                }
                e = cudaGetLastError();
            }
        } else {
            Params pa = prm;
            pa.P = P - 1;
            pa.ctas = ctas;
            diag_scan_kernel<DK, TIn, true, LIN>
                <<<static_cast<unsigned>(ctas * (P - 1)), Geo<DK>::NTHREADS, smem, st>>>(pa);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) {
            const long long n4 = BH * S / 4;
            diag_carry_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, st>>>(
                prm.agg, prm.agg_scale, a.I0, a.mu0, a.I_prior, BH, S, P);
            e = cudaGetLastError();
        }
    }
    bool tc_full = false;
    if constexpr (LIN && DK == lintc::LD && std::is_same<TIn, __nv_bfloat16>::value) {
        if (e == cudaSuccess && dv == lintc::LD) {
            // full pass on the tensor cores: one CTA per (head, part)
            tc_full = true;
            static bool attr[64] = {};
            int dev = 0;
            e = cudaGetDevice(&dev);
            if (e == cudaSuccess && dev >= 0 && dev < 64 && !attr[dev]) {
                e = cudaFuncSetAttribute(lintc::lin_tc_kernel<lintc::LD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, lintc::LSMEM);
                if (e == cudaSuccess) attr[dev] = true;
            }
            if (e == cudaSuccess) {
                lintc::LinArgs la{static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
                                  static_cast<const __nv_bfloat16*>(a.v), static_cast<const __nv_bfloat16*>(a.beta),
                                  static_cast<const __nv_bfloat16*>(a.d), a.A, a.I_prior, a.mu0, prm.agg,
                                  a.out, a.final_state, BH, a.H, a.T, pl.part_len, wait_ns};
                lintc::lin_tc_kernel<lintc::LD>
                    <<<dim3(static_cast<unsigned>(BH), P), lintc::LTHREADS, lintc::LSMEM, st>>>(la);
                e = cudaGetLastError();
            }
        }
    }
    if (e == cudaSuccess && !tc_full) {
        // Per-head lambda walkers: appended after the scan CTAs, so they take
        // the CTA slots that the scan's last wave leaves free (at least one
        // walker per 64 tiles of lambda work).
        int launch_smem = pl.ws ? pl.smem_full : smem;
        const long long ctas_f = pl.ws ? pl.ctas_full : ctas;
        prm.ctas = ctas_f;
        prm.TC = pl.TC_full;
        if constexpr (!LIN) {
            if (a.lam_out && a.T > 0) {
                const int walk_tile = pl.ws ? mob::Walk<WS_THREADS>::TILE : mob::Walk<Geo<DK>::NTHREADS>::TILE;
                const int walk_smem = pl.ws ? mob::Walk<WS_THREADS>::SMEM : mob::Walk<Geo<DK>::NTHREADS>::SMEM;
                const long long tps = (a.T + walk_tile - 1) / walk_tile;
                const long long slots = static_cast<long long>(sm_count()) * pl.occ;
                const long long total = ctas_f * P;
                const long long free_slots = (total + slots - 1) / slots * slots - total;
                long long nl = std::max(free_slots, (BH * tps + 63) / 64);
                nl = std::min(std::max(nl, 1LL), BH);
                prm.nlam = static_cast<int>(nl);
                prm.ma = a.ma; prm.mb = a.mb; prm.mc = a.mc; prm.md = a.md;
                prm.lam0 = a.lam0; prm.lam_out = a.lam_out;
                launch_smem = std::max(launch_smem, walk_smem);
            }
        }
        const unsigned grid = static_cast<unsigned>(ctas_f * P + prm.nlam);
        bool launched = false;
        if constexpr (!LIN && (DK == 64 || DK == 128)) {
            if (pl.ws) {
                // launch_smem == pl.smem_full: the walkers' stages fit it (plan_dk).
                // After the carry kernel (P > 1) the full pass is launched as its
                // programmatic dependent: its CTAs may start while the carry
                // finishes (the caller's inputs were complete before the
                // aggregate pass began) and wait for it only where they read
                // a carried start state.
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(grid);
                cfg.blockDim = dim3(WS_THREADS);
                cfg.dynamicSmemBytes = static_cast<size_t>(launch_smem);
                cfg.stream = st;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                attr[0].val.programmaticStreamSerializationAllowed = 1;
                cfg.attrs = attr;
                cfg.numAttrs = P > 1 ? 1 : 0;
                e = pl.TC_full == 16 ? cudaLaunchKernelEx(&cfg, diag_ws_kernel<DK, TIn, 16>, prm)
                                     : cudaLaunchKernelEx(&cfg, diag_ws_kernel<DK, TIn, 8>, prm);
                launched = true;
            }
        }
        if (!launched) {
            if (launch_smem > smem) {
                e = cudaFuncSetAttribute(diag_scan_kernel<DK, TIn, false, LIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, launch_smem);
            }
            if (e == cudaSuccess) {
                diag_scan_kernel<DK, TIn, false, LIN><<<grid, Geo<DK>::NTHREADS, launch_smem, st>>>(prm);
                e = cudaGetLastError();
            }
        }
    }
    if (scratch) {
        const cudaError_t ef = cudaFreeAsync(scratch, st);
        if (e == cudaSuccess) e = ef;
    }
    return from_cuda(e);
}

template <typename TIn>
kdn_status plan_any(const DiagArgs& a, Plan* pl) {
    switch (a.dk) {
        case 16: return plan_dk<16, TIn, false>(a, pl);
        case 32: return plan_dk<32, TIn, false>(a, pl);
        case 64: return plan_dk<64, TIn, false>(a, pl);
        case 128: return plan_dk<128, TIn, false>(a, pl);
        default: return KDN_ERR_UNSUPPORTED;
    }
}

template <typename TIn, bool LIN>
kdn_status launch_lin(const DiagArgs& a, cudaStream_t st, long long wait_ns) {
    switch (a.dk) {
        case 16: return launch_dk<16, TIn, LIN>(a, st, wait_ns);
        case 32: return launch_dk<32, TIn, LIN>(a, st, wait_ns);
        case 64: return launch_dk<64, TIn, LIN>(a, st, wait_ns);
        case 128: return launch_dk<128, TIn, LIN>(a, st, wait_ns);
        default: return KDN_ERR_UNSUPPORTED;
    }
}

template <typename TIn>
kdn_status launch_any(const DiagArgs& a, cudaStream_t st, long long wait_ns) {
    return a.lin ? launch_lin<TIn, true>(a, st, wait_ns) : launch_lin<TIn, false>(a, st, wait_ns);
}

}  // namespace
}  // namespace diag
}  // namespace kdn
