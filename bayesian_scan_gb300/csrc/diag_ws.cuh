// diag_ws.cuh -- the full pass of the diagonal metaplastic scan for d_k in
// {64, 128}, warp-specialised ("Learning to Remember, Learn, and Forget in
// Attention-Based Models", Metodologia 1-2; readout o_t = mu_t q_t).
//
// Same arithmetic and results as diag_scan_kernel (the scaled information
// form with per-head power-of-two working scale, paired reciprocals, packed
// FP32; see diag_impl.cuh).  The consumers keep J as sigma W J (sigma =
// 2^-24) rather than W J, with sigma in the row factor of the update, so
// that the denominator sigma W (J + I_prior) is one addition (sigma is a
// power of two: the same results).  When the producers form the row factors
// (d_k = 128) the consumers need W only for the final state and read it
// after the token loop.  The division of labour inside the CTA:
//
//  * 8 consumer warps own the state, 4 rows x 16 columns per lane, and do
//    nothing but the element updates and the readout partials: per token they
//    read the converted k, k^2, q, the token scalars and their rows' W beta,
//    W beta v (for d_k = 64: beta and v from the raw chunk, scaled by W
//    themselves) from shared memory, update 64 elements and store 4 row
//    partials to a reduction buffer.  After `setmaxnreg.inc` they hold 232
//    registers each.
//  * 4 producer warps (one warpgroup, 40 registers each after
//    `setmaxnreg.dec`) keep the consumers fed: they issue the 1-D bulk copies
//    of each chunk of q, k, v, beta, d, convert k -> (k, k^2) and q to fp32 in
//    the consumers' interleaved layout, run the per-head scale recursion and
//    (d_k = 128) scale each row's beta and beta v by the token's W, and sum
//    the readout partials of every 8 tokens over the lanes of a row and
//    store o with streaming 16-byte stores.  (For d_k = 128 the row scaling moved here
//    from the consumers: it took them ~16 instructions per token, and with
//    no consumer reading the raw chunk two raw stages are enough, which pays
//    for the larger converted chunk.)
//
// Pipeline (mbarriers, every wait bounded by GPU time):
//   raw_full[r]   bulk copies of a chunk landed          (tx count; r = 2 or 3)
//   par_full[2]   a chunk's converted inputs and scalars  (128 producer threads)
//   par_empty[2]  consumers finished a chunk              (256 consumer threads)
//   red_full[n]   8 tokens of row partials written        (256 consumer threads)
//   red_empty[n]  those partials summed and stored        (128 producer threads)
// The producers prepare chunk c + 2 as soon as the consumers release chunk
// c; with two raw stages they then (after a producer-only named barrier)
// refill its raw stage with the copies of chunk c + 4, with three they first
// issue the copies of chunk c + 3 into chunk c's stage.  The consumers never
// wait on them in steady state.  Row partials go to n = TC / 8 + 1 buffers
// of 8 tokens; consumers wait for a buffer at the start of a chunk, never in
// the token loop (its registers hold the state and the token's operands
// only).
//
// A CTA owns ROWS = 8 * rows-per-warp consecutive state rows (128 for
// d_k = 128, 256 for d_k = 64: whole heads, ROWS / d_v of them) for one
// token part.  Extra CTAs after the scan's (the per-head Moebius lambda)
// walk their sequences with all 384 threads.
#pragma once

namespace kdn {
namespace diag {
namespace {

constexpr int WS_CW = 8;                         // consumer warps
constexpr int WS_PW = 4;                         // producer warps (one warpgroup)
constexpr int WS_THREADS = (WS_CW + WS_PW) * 32;  // 384
constexpr int WS_CREG = 232;                     // registers per consumer thread after setmaxnreg
constexpr int WS_PREG = 40;                      // registers per producer thread after setmaxnreg
constexpr int WS_LAUNCH_REG = 168;               // per thread at launch (65536 / 384, rounded down to 8)
static_assert(WS_CW * 32 * WS_CREG + WS_PW * 32 * WS_PREG <= WS_THREADS * WS_LAUNCH_REG,
              "the register split must fit the CTA's launch allocation");
// Where each row's W beta and W beta v are formed: by the producers for
// d_k = 128 (the consumers then read no raw input and two raw stages
// suffice; measured 2.1 % faster on both d_k = 128 workloads), by the
// consumers for d_k = 64, whose producers serve 4 heads per CTA and became
// the bottleneck with the extra pass (4.8 % slower).
__host__ __device__ constexpr bool ws_row_scale_in_producers(int dk) { return dk == 128; }
// raw chunk stages: 2 when only the producers read them, else 3 (the
// consumers read beta and v of a chunk while the producers prepare the next)
__host__ __device__ constexpr int ws_raw(int dk) { return ws_row_scale_in_producers(dk) ? 2 : 3; }
constexpr int WS_PAR = 2;                        // converted chunk stages
constexpr int WS_RB = 8;                         // tokens per reduction buffer
// Column-pair groups (of 4 per lane row) whose two quotients share one
// reciprocal: 3 (measured on GB300 with the denominator one addition: all 4
// paired made the 1.3B layer's d_k = 64 call 2.477 -> 2.533 ms and the
// 65536-token call 4.079 -> 4.087 ms; 2 paired 2.48 -> 2.60 and 4.08 ->
// 4.25 ms).
template <int DK>
__host__ __device__ constexpr int ws_pairs() { return 3; }
// Reduction buffers for chunks of TC tokens: consumers wait for a buffer's
// previous flush at the start of a chunk (never inside the token loop), so
// the TC / 8 groups of a chunk need TC / 8 + 1 buffers for the flush of the
// previous chunk's last group to overlap the next chunk.
__host__ __device__ constexpr int ws_nred(int TC) { return TC / WS_RB + 1; }
// Floats per token and head of a converted chunk: k, k^2, q (d_k each, in
// the consumers' interleaving), the token's scalars (rescale factor, W,
// W I_prior sigma, rescale mask), then, when the producers scale the rows,
// per value row W beta and W beta v (d_v each).
__host__ __device__ constexpr int ws_par_floats(int dk, int dv) {
    return 3 * dk + 4 + (ws_row_scale_in_producers(dk) ? 2 * dv : 0);
}

template <int DK>
struct WsGeo {
    static constexpr int M = DK / CW;            // lanes sharing a row set
    static constexpr int RS = 32 / M;            // row sets per warp
    static constexpr int WR = RS * RT;           // rows per warp
    static constexpr int ROWS = WS_CW * WR;      // rows per CTA
    static constexpr int RSS = red_rs_stride(M);
    static constexpr int RTS = red_token_stride(M);
    static constexpr int RED_FLOATS = WS_CW * WS_RB * RTS;   // one reduction buffer
};

// Shared-memory layout of the warp-specialised kernel (bytes).
struct WsLayout {
    int raw_qk, raw_vb, raw_d, raw_head, raw_stage;
    int par_head, par_stage;
    int red_buf;
    int off_par, off_red, off_bar, total;
    __host__ __device__ WsLayout(int dk, int dv, int es, int TC, int hpc, int red_floats) {
        const int nred = ws_nred(TC);
        raw_qk = TC * dk * es;
        raw_vb = TC * dv * es;
        raw_d = (TC * es + 15) & ~15;
        raw_head = 2 * raw_qk + 2 * raw_vb + raw_d;
        raw_stage = hpc * raw_head;
        par_head = TC * ws_par_floats(dk, dv) * 4;
        par_stage = hpc * par_head;
        red_buf = red_floats * 4;
        off_par = ws_raw(dk) * raw_stage;
        off_red = off_par + WS_PAR * par_stage;
        off_bar = off_red + nred * red_buf;
        // barriers: raw_full[ws_raw], par_full[2], par_empty[2], red_full[nred],
        // red_empty[nred]; then the scale state W[hpc], R[hpc]
        total = off_bar + (ws_raw(dk) + 2 * WS_PAR + 2 * nred) * 8 + 8 * hpc;
    }
};

template <int DK>
__host__ __device__ inline int ws_smem_bytes(int dv, int es, int TC) {
    // TC: 16 or 8
    using G = WsGeo<DK>;
    return WsLayout(DK, dv, es, TC, G::ROWS / dv, G::RED_FLOATS).total;
}

template <int DK, typename TIn, int TC>
__global__ void __launch_bounds__(WS_THREADS, 1)
diag_ws_kernel(const Params p) {
    using G = WsGeo<DK>;
    constexpr int M = G::M, RSS = G::RSS, RTS = G::RTS, WR = G::WR;
    constexpr int WS_PAIRS = ws_pairs<DK>();
    constexpr int ES = sizeof(TIn);
    constexpr int NRED = ws_nred(TC), GPC = TC / WS_RB;   // reduction buffers, groups per chunk
    static_assert(TC % WS_RB == 0 && TC <= 16, "whole reduction groups per chunk; rescale masks hold 16 tokens");
    extern __shared__ __align__(128) unsigned char smem[];

    const int dv = p.dv, HPC = G::ROWS / dv;
    const int PF = ws_par_floats(DK, dv);
    constexpr bool PSCALE = ws_row_scale_in_producers(DK);
    constexpr int WS_RAW = ws_raw(DK);
    const WsLayout L(DK, dv, ES, TC, HPC, G::RED_FLOATS);
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
    uint64_t* par_full = raw_full + WS_RAW;
    uint64_t* par_empty = par_full + WS_PAR;
    uint64_t* red_full = par_empty + WS_PAR;
    uint64_t* red_empty = red_full + NRED;
    float* w_state = reinterpret_cast<float*>(red_empty + NRED);   // [HPC]
    int* r_state = reinterpret_cast<int*>(w_state + HPC);       // [HPC]
    auto rawp = [&](int s, int h, int off) { return smem + s * L.raw_stage + h * L.raw_head + off; };
    auto raw_q = [&](int s, int h) { return reinterpret_cast<TIn*>(rawp(s, h, 0)); };
    auto raw_k = [&](int s, int h) { return reinterpret_cast<TIn*>(rawp(s, h, L.raw_qk)); };
    auto raw_v = [&](int s, int h) { return reinterpret_cast<TIn*>(rawp(s, h, 2 * L.raw_qk)); };
    auto raw_b = [&](int s, int h) { return reinterpret_cast<TIn*>(rawp(s, h, 2 * L.raw_qk + L.raw_vb)); };
    auto raw_d = [&](int s, int h) { return reinterpret_cast<TIn*>(rawp(s, h, 2 * L.raw_qk + 2 * L.raw_vb)); };
    auto par = [&](int s, int h) {
        return reinterpret_cast<float*>(smem + L.off_par + s * L.par_stage + h * L.par_head);
    };
    auto red = [&](int b) { return reinterpret_cast<float*>(smem + L.off_red + b * L.red_buf); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // linear grid: part-major scan CTAs (head group fastest), then the lambda walkers
    const long long lin = blockIdx.x;
    if (lin >= p.ctas * p.P) {
        const int tps = static_cast<int>((p.T + mob::Walk<WS_THREADS>::TILE - 1) / mob::Walk<WS_THREADS>::TILE);
        mob::mobius_walk<WS_THREADS>(p.ma, p.mb, p.mc, p.md, p.lam0, p.lam_out, p.BH, p.T, tps,
                                     lin - p.ctas * p.P, p.nlam, p.wait_ns, smem, &g_diag_error);
        return;
    }
    const int part = static_cast<int>(lin / p.ctas);
    const long long head0 = (lin - static_cast<long long>(part) * p.ctas) * HPC;
    const int nheads = static_cast<int>(min(static_cast<long long>(HPC), p.BH - head0));
    const int T = p.T;
    const int tb = min(T, part * p.part_len);
    const int te = min(T, tb + p.part_len);
    const int nch = (te - tb + TC - 1) / TC;
    const float Ip = p.I_prior;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WS_RAW; ++s) mbar_init(&raw_full[s], 1);
        for (int s = 0; s < WS_PAR; ++s) {
            mbar_init(&par_full[s], WS_PW * 32);
            mbar_init(&par_empty[s], WS_CW * 32);
        }
        for (int b = 0; b < NRED; ++b) {
            mbar_init(&red_full[b], WS_CW * 32);
            mbar_init(&red_empty[b], WS_PW * 32);
        }
        for (int h = 0; h < HPC; ++h) {
            w_state[h] = 1.f;
            r_state[h] = 0;
        }
        mbar_init_fence();
    }
    __syncthreads();
    bool ok = true;

    if (warp >= WS_CW) {
        // =========================== producers ================================
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(WS_PREG));
        const int pt = threadIdx.x - WS_CW * 32;   // 0..127
        const int pw = warp - WS_CW;               // 0..3
        const TIn* gq = static_cast<const TIn*>(p.q);
        const TIn* gk = static_cast<const TIn*>(p.k);
        const TIn* gv = static_cast<const TIn*>(p.v);
        const TIn* gb = static_cast<const TIn*>(p.beta);
        const TIn* gd = static_cast<const TIn*>(p.d);

        // bulk copies of chunk c into raw stage c % 3 (one thread)
        auto issue = [&](int c) {
            const int s = c % WS_RAW;
            const int t0 = tb + c * TC, tcn = min(TC, te - t0);
            const int dbytes = p.d_tma ? tcn * ES : 0;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&raw_full[s], static_cast<uint32_t>(nheads * (tcn * (2 * DK + 2 * dv) * ES + dbytes)));
            for (int h = 0; h < nheads; ++h) {
                const long long tok = (head0 + h) * T + t0;
                bulk_g2s(raw_q(s, h), gq + tok * DK, tcn * DK * ES, &raw_full[s]);
                bulk_g2s(raw_k(s, h), gk + tok * DK, tcn * DK * ES, &raw_full[s]);
                bulk_g2s(raw_v(s, h), gv + tok * dv, tcn * dv * ES, &raw_full[s]);
                bulk_g2s(raw_b(s, h), gb + tok * dv, tcn * dv * ES, &raw_full[s]);
                if (dbytes) bulk_g2s(raw_d(s, h), gd + (head0 + h) * p.d_ld + t0, dbytes, &raw_full[s]);
            }
        };

        // convert chunk c into par stage c & 1 and run the scale recursion
        auto prepare = [&](int c) {
            const int s3 = c % WS_RAW, s2 = c & 1;
            const int t0 = tb + c * TC, tcn = min(TC, te - t0);
            if (!mbar_wait(&raw_full[s3], (c / WS_RAW) & 1, p.wait_ns)) ok = false;
            // items (head, token, float4 slot f); slot f = s4 * M + cg holds
            // columns cg * 16 + s4 * 4 .. + 3 (the consumers' interleaving)
            constexpr int F4 = DK / 4;
            for (int x = pt; x < nheads * tcn * F4; x += WS_PW * 32) {
                const int f = x % F4, ht = x / F4;
                const int tt = ht % tcn, h = ht / tcn;
                const int j = (f % M) * CW + (f / M) * 4;
                float kf[4], qf[4];
                load4(raw_k(s3, h) + tt * DK + j, kf);
                load4(raw_q(s3, h) + tt * DK + j, qf);
                float* dst = par(s2, h) + tt * PF + 4 * f;
                *reinterpret_cast<float4*>(dst) = make_float4(kf[0], kf[1], kf[2], kf[3]);
                *reinterpret_cast<float4*>(dst + DK) =
                    make_float4(kf[0] * kf[0], kf[1] * kf[1], kf[2] * kf[2], kf[3] * kf[3]);
                *reinterpret_cast<float4*>(dst + 2 * DK) = make_float4(qf[0], qf[1], qf[2], qf[3]);
            }
            if (pw == WS_PW - 1 && lane < nheads) {
                const int h = lane;
                const float Ah = p.A[(head0 + h) % p.H];
                float W = w_state[h];
                int R = r_state[h];
                const TIn* rd = raw_d(s3, h);
                const TIn* gdh = gd + (head0 + h) * p.d_ld + t0;
                float* ps = par(s2, h) + 3 * DK;
                uint32_t mask = 0;   // tokens of the chunk that rescale the state
                for (int tt = 0; tt < tcn; ++tt) {
                    const float dval = p.d_tma ? to_f32<TIn>(rd[tt]) : to_f32<TIn>(gdh[tt]);
                    const float f = scale_step(Ah * dval * LOG2E, W, R);
                    *reinterpret_cast<float4*>(ps + tt * PF) = make_float4(f, W, W * Ip * SIGMA, 0.f);
                    if (f != 1.f) mask |= 1u << tt;
                }
                ps[3] = __uint_as_float(mask);   // 4th scalar of the chunk's first token
                w_state[h] = W;
                r_state[h] = R;
            }
            if constexpr (PSCALE) {
                // the rows' scaled inputs W beta, W beta v of every token, by
                // all producers once the tokens' W are written
                asm volatile("bar.sync 1, %0;" ::"n"(WS_PW * 32) : "memory");
                const int Q = dv / 4;
                for (int x = pt; x < nheads * tcn * Q; x += WS_PW * 32) {
                    const int i4 = x % Q, ht = x / Q;
                    const int tt = ht % tcn, h = ht / tcn;
                    float* ps = par(s2, h) + tt * PF + 3 * DK;
                    const float W = ps[1];
                    float bet[4], val[4];
                    load4(raw_b(s3, h) + tt * dv + 4 * i4, bet);
                    load4(raw_v(s3, h) + tt * dv + 4 * i4, val);
                    const float4 sb = make_float4(W * bet[0], W * bet[1], W * bet[2], W * bet[3]);
                    *reinterpret_cast<float4*>(ps + 4 + 4 * i4) =
                        make_float4(sb.x * SIGMA, sb.y * SIGMA, sb.z * SIGMA, sb.w * SIGMA);
                    *reinterpret_cast<float4*>(ps + 4 + dv + 4 * i4) =
                        make_float4(sb.x * val[0], sb.y * val[1], sb.z * val[2], sb.w * val[3]);
                }
            }
            mbar_arrive(&par_full[s2]);
        };
        // prepare chunk c, then (once every producer has read its raw stage)
        // refill that stage with the copies of chunk c + WS_RAW
        auto prepare_refill = [&](int c) {
            prepare(c);
            if constexpr (PSCALE) {
                asm volatile("bar.sync 1, %0;" ::"n"(WS_PW * 32) : "memory");
                if (pt == 0 && c + WS_RAW < nch) issue(c + WS_RAW);
            }
        };

        // sum the row partials of reduction group g (tokens g*8 .. of the
        // part) over the M lanes of each row and store o
        auto flush = [&](int g) {
            const int b = g % NRED;
            if (!mbar_wait(&red_full[b], (g / NRED) & 1, p.wait_ns)) ok = false;
            const int t_first = tb + g * WS_RB;
            const int ntok = min(WS_RB, te - t_first);
            const float* rb = red(b);
            constexpr int ITEMS_PER_TOKEN = WS_CW * G::RS;   // row quads of the CTA
            for (int x = pt; x < ntok * ITEMS_PER_TOKEN; x += WS_PW * 32) {
                const int ts = x / ITEMS_PER_TOKEN, q = x - ts * ITEMS_PER_TOKEN;
                const int w = q / G::RS, rq = q - w * G::RS;
                const int crow = w * WR + rq * RT;
                const int hq = crow / dv, iq = crow - hq * dv;
                if (hq >= nheads) continue;
                const float* src = rb + (w * WS_RB + ts) * RTS + rq * RSS;
                const float4 x0 = *reinterpret_cast<const float4*>(src);
                float2 lo = make_float2(x0.x, x0.y), hi = make_float2(x0.z, x0.w);
#pragma unroll
                for (int c = 1; c < M; ++c) {
                    const float4 y = *reinterpret_cast<const float4*>(src + 4 * c);
                    lo = __fadd2_rn(lo, make_float2(y.x, y.y));
                    hi = __fadd2_rn(hi, make_float2(y.z, y.w));
                }
                lo = __fmul2_rn(lo, f2(SIGMA));
                hi = __fmul2_rn(hi, f2(SIGMA));
                float* o = p.out + ((head0 + hq) * p.out_ld + t_first + ts) * dv + iq;
                __stcs(reinterpret_cast<float4*>(o), make_float4(lo.x, lo.y, hi.x, hi.y));
            }
            mbar_arrive(&red_empty[b]);
        };

        if (pt == 0)
            for (int c = 0; c < WS_RAW && c < nch; ++c) issue(c);
        if (nch > 0) prepare_refill(0);
        if (nch > 1) prepare_refill(1);
        int g_next = 0;   // next reduction group to flush
        for (int c = 0; c < nch; ++c) {
            const int t_end = min(te, tb + (c + 1) * TC);   // tokens before t_end belong to chunks <= c
            for (; tb + g_next * WS_RB < t_end; ++g_next) flush(g_next);
            // the consumers have released chunk c: its stages can be reused
            if (!mbar_wait(&par_empty[c & 1], (c >> 1) & 1, p.wait_ns)) ok = false;
            // (consumers reading raw beta, v: chunk c's raw stage is free now)
            if (!PSCALE && pt == 0 && c + WS_RAW < nch) issue(c + WS_RAW);
            if (c + 2 < nch) prepare_refill(c + 2);
        }
    } else {
        // =========================== consumers ================================
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(WS_CREG));
        const int rs = lane / M, cg = lane % M;
        const int crow = warp * WR + rs * RT;
        const int hl = crow / dv, i0 = crow - hl * dv;
        const bool active = hl < nheads;
        const long long bh = head0 + hl;
        const long long S = static_cast<long long>(dv) * DK;

        float2 J[RT][CW / 2], E[RT][CW / 2];
        {
            const float* src_J = nullptr;
            const float* src_E = nullptr;
            if (part > 0) {
                grid_dep_wait();   // the carry kernel's start states (launched ahead of it)
                src_J = p.agg + (static_cast<long long>(part - 1) * p.BH + bh) * 2 * S;
                src_E = src_J + S;
            }
#pragma unroll
            for (int r = 0; r < RT; ++r) {
#pragma unroll
                for (int c2 = 0; c2 < CW / 2; ++c2) {
                    float2 j2 = make_float2(0.f, 0.f), e2 = make_float2(0.f, 0.f);
                    const long long off = static_cast<long long>(i0 + r) * DK + cg * CW + 2 * c2;
                    if (active) {
                        if (src_J) {
                            j2 = *reinterpret_cast<const float2*>(src_J + off);
                            e2 = *reinterpret_cast<const float2*>(src_E + off);
                        } else if (p.I0 || p.mu0) {
                            float2 i02 = make_float2(Ip, Ip);
                            if (p.I0) i02 = *reinterpret_cast<const float2*>(p.I0 + bh * S + off);
                            j2 = make_float2(i02.x - Ip, i02.y - Ip);
                            if (p.mu0) {
                                const float2 m2 = *reinterpret_cast<const float2*>(p.mu0 + bh * S + off);
                                e2 = make_float2(i02.x * m2.x, i02.y * m2.y);
                            }
                        }
                    }
                    J[r][c2] = __fmul2_rn(j2, f2(SIGMA));   // the state keeps sigma W J
                    E[r][c2] = e2;
                }
            }
        }

        float W = 1.f;
        const int hsafe = active ? hl : 0;
        for (int c = 0; c < nch; ++c) {
            const int s2 = c & 1, s3 = c % WS_RAW;
            if (!mbar_wait(&par_full[s2], (c >> 1) & 1, p.wait_ns)) ok = false;
            const int tcn = min(TC, te - (tb + c * TC));
            // the reduction buffers of this chunk's groups: their previous
            // groups (NRED earlier) must have been flushed
#pragma unroll
            for (int gg = 0; gg < GPC; ++gg) {
                const int g = c * GPC + gg;
                if (g >= NRED && gg * WS_RB < tcn &&
                    !mbar_wait(&red_empty[g % NRED], (g / NRED - 1) & 1, p.wait_ns))
                    ok = false;
            }
            float* redc = red(0) + warp * WS_RB * RTS + rs * RSS + 4 * cg;   // this lane's slot 0, buffer 0
            const TIn* rv = raw_v(s3, hsafe) + i0;
            const TIn* rbp = raw_b(s3, hsafe) + i0;
            const float* pbase = par(s2, hsafe);
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
                            J[r][c2] = __fmul2_rn(J[r][c2], f22);
                            E[r][c2] = __fmul2_rn(E[r][c2], f22);
                        }
                }
                const uint32_t later = mask >> (tt + 1);   // tt + 1 <= TC <= 16
                const int stop = later ? min(tcn, tt + __ffs(later)) : tcn;
                for (; tt < stop; ++tt) {
                    const int slot = tt & (WS_RB - 1);
                    const int b = (c * GPC + tt / WS_RB) % NRED;
                    const float* ptk = pbase + tt * PF;
                    float SPs;   // sigma W I_prior of the token
                    if constexpr (PSCALE) {
                        SPs = ptk[3 * DK + 2];
                    } else {
                        const float4 sc = *reinterpret_cast<const float4*>(ptk + 3 * DK);
                        W = sc.y;
                        SPs = sc.z;
                    }
                    static_assert(RT == 4, "one float4 of row scalars per lane");
                    float2 SB[RT], SBV[RT];
                    if constexpr (PSCALE) {
                        const float4 sb4 = *reinterpret_cast<const float4*>(ptk + 3 * DK + 4 + i0);
                        const float4 sv4 = *reinterpret_cast<const float4*>(ptk + 3 * DK + 4 + dv + i0);
                        SB[0] = f2(sb4.x); SB[1] = f2(sb4.y); SB[2] = f2(sb4.z); SB[3] = f2(sb4.w);
                        SBV[0] = f2(sv4.x); SBV[1] = f2(sv4.y); SBV[2] = f2(sv4.z); SBV[3] = f2(sv4.w);
                    } else {
                        float bet[RT], val[RT];
                        load4(rbp + tt * dv, bet);
                        load4(rv + tt * dv, val);
#pragma unroll
                        for (int r = 0; r < RT; ++r) {
                            const float sb = W * bet[r];
                            SB[r] = f2(sb * SIGMA);
                            SBV[r] = f2(sb * val[r]);
                        }
                    }
                    const float2 SP = f2(SPs);
                    float2 acc[RT];
#pragma unroll
                    for (int r = 0; r < RT; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float2 kf[4], kk[4], qv[4];
#pragma unroll
                        for (int h4 = 0; h4 < 2; ++h4) {
                            const int f4 = ((2 * half + h4) * M + cg) * 4;
                            const float4 a = *reinterpret_cast<const float4*>(ptk + f4);
                            const float4 bq = *reinterpret_cast<const float4*>(ptk + DK + f4);
                            const float4 q = *reinterpret_cast<const float4*>(ptk + 2 * DK + f4);
                            kf[2 * h4] = make_float2(a.x, a.y);
                            kf[2 * h4 + 1] = make_float2(a.z, a.w);
                            kk[2 * h4] = make_float2(bq.x, bq.y);
                            kk[2 * h4 + 1] = make_float2(bq.z, bq.w);
                            qv[2 * h4] = make_float2(q.x, q.y);
                            qv[2 * h4 + 1] = make_float2(q.z, q.w);
                        }
#pragma unroll
                        for (int r = 0; r < RT; ++r) {
                            float2 den[4], num[4];
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const int c2 = half * 4 + c4;
                                J[r][c2] = __ffma2_rn(SB[r], kk[c4], J[r][c2]);
                                E[r][c2] = __ffma2_rn(SBV[r], kf[c4], E[r][c2]);
                                den[c4] = __fadd2_rn(J[r][c2], SP);
                                num[c4] = __fmul2_rn(qv[c4], E[r][c2]);
                            }
#pragma unroll
                            for (int g = 0; g < 2; ++g) {
                                const int x = 2 * g, y = 2 * g + 1;
                                if (2 * g + half < WS_PAIRS) {
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
                    float* dst = redc + b * G::RED_FLOATS + slot * RTS;
                    *reinterpret_cast<float4*>(dst) =
                        make_float4(acc[0].x + acc[0].y, acc[1].x + acc[1].y, acc[2].x + acc[2].y,
                                    acc[3].x + acc[3].y);
                    if (slot == WS_RB - 1 || tt == tcn - 1) mbar_arrive(&red_full[b]);
                }
            }
            mbar_arrive(&par_empty[s2]);
        }

        if constexpr (PSCALE) W = w_state[hsafe];   // the part's last W (chunks all prepared)
        if (active && p.final_state && part == p.P - 1) {
            // mu_T = eta / (I_prior + J) = Ew / (Jw + W I_prior);  I_T = Jw / W + I_prior
            float* fm = p.final_state + bh * S;
            float* fi = p.final_state + (p.BH + bh) * S;
            const float wI = W * Ip;
#pragma unroll
            for (int r = 0; r < RT; ++r)
#pragma unroll
                for (int c2 = 0; c2 < CW / 2; ++c2) {
                    const long long off = static_cast<long long>(i0 + r) * DK + cg * CW + 2 * c2;
                    const float2 j2 = __fmul2_rn(J[r][c2], f2(INV_SIGMA)), e2 = E[r][c2];
                    *reinterpret_cast<float2*>(fm + off) = make_float2(e2.x / (j2.x + wI), e2.y / (j2.y + wI));
                    *reinterpret_cast<float2*>(fi + off) = make_float2(j2.x / W + Ip, j2.y / W + Ip);
                }
        }
    }
    if (!ok) record_error(&g_diag_error, KDN_ERR_TIMEOUT);
}

}  // namespace
}  // namespace diag
}  // namespace kdn
