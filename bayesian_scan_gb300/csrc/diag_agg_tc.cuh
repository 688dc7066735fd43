// diag_agg_tc.cuh -- the aggregate pass of a token-split diagonal scan on the
// tensor cores (d_k = d_v = 128, bf16 inputs).
//
// When a long sequence is split into token parts, each part p < P-1 needs
// only its end state from a zero start ("Learning to Remember, Learn, and
// Forget in Attention-Based Models", Metodologia 2, unrolled over the part):
//     Delta J[i][j]   = sum_t w_t beta_t[i] k_t[j]^2
//     Delta eta[i][j] = sum_t w_t beta_t[i] v_t[i] k_t[j],
//     w_t = prod_{s > t in the part} alpha_s = 2^-(sum_{s>t} A d_s log2 e),
// plus the part's total decay prod alpha = 2^-L.  Both sums are dense
// contractions over the part's tokens, [d_v x T_p] x [T_p x d_k]: here they
// run as tcgen05.mma (kind::f16, bf16 operands, fp32 accumulators in tensor
// memory), K = 16 or 32 tokens per chunk.
//
// Precision.  beta and k are bf16 inputs, so they are exact operands.  The
// decay weight goes with k^2 for Delta J, Delta J = sum_t beta_t[i] (w_t
// k_t[j]^2), and with beta v for Delta eta, Delta eta = sum_t (w_t beta_t[i]
// v_t[i]) k_t[j]; the fp32 factors w k^2 and w beta v are each split into
// three bf16 pieces (hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi -
// mid); both differences are exact in fp32), which carry all 24 bits of the
// fp32 value.  So each sum takes three products, accumulated in fp32, and
// every term is as accurate as the fp32 product it stands for: the carried
// states are fp32-accurate, not bf16-accurate.  The decay exponents are
// summed in fp64 (the part's suffix sums) and w_t = 2^-floor(S) *
// exp2(-frac(S)).
//
// Output: the same (J_w, eta_w) = W (Delta J, Delta eta) and (W, R) with
// 2^-R / W = 2^-L, W in [1, 2), that the CUDA-core aggregate pass leaves for
// the carry kernel.
//
// Per CTA: one (head, part); 8 KC build threads and one issuing warp.
// Chunks of the part are visited from the last to the first (so the suffix
// sums accumulate).  The weights w_t of a super-chunk of tokens are prepared
// by the build threads (8 tokens each, fp64 suffix sums across them); per
// chunk the build threads write the 7 operand tiles (128 x KC bf16 each,
// core-matrix layout) from the raw chunk (k, beta, v, brought in by 1-D bulk
// copies two chunks ahead) and arrive, one lane per warp, on the chunk's
// operand barrier; the issuing warp waits there, issues the next copies into
// the consumed raw stage and the chunk's 6 KC / 16 MMAs, and commits them to
// an mbarrier.  Operand tiles are double-buffered on that barrier, so the
// build threads never wait for the products to be issued (a build thread
// that also issued held its warp, and at the chunk barrier all others, for
// about 770 cycles a chunk).  All waits are bounded by GPU time.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kdn_device.cuh"

namespace kdn {
namespace diag {
namespace {

constexpr int AG_D = 128;                          // d_k = d_v
constexpr int AG_NTILE = 8;                        // A_beta, A_E hi/mid/lo, B_k, B_wk2 hi/mid/lo
constexpr int AG_TMEM_COLS = 256;                  // J in columns [0,128), eta in [128,256)
constexpr uint32_t AG_LBO = 128;                   // core matrices: next 8 tokens (K)

// Chunk shapes: KC tokens per chunk, 8 KC build threads (one per row pair
// and group of 8 tokens) and one more warp that issues the products and the
// copies.  KC = 32: 288 threads, one CTA per SM; KC = 16: 160 threads, two
// CTAs per SM (each holding 256 of the SM's 512 TMEM columns), for grids
// with at least two CTAs per SM.
template <int KC>
struct AggShape {
    static constexpr int BUILD = 8 * KC;
    static constexpr int THREADS = BUILD + 32;
    static constexpr int CTAS_PER_SM = KC == 16 ? 2 : 1;
    static constexpr int TILE = AG_D * KC * 2;          // one 128 x KC bf16 operand tile, bytes
    static constexpr int OPS = AG_NTILE * TILE;         // one operand buffer
    static constexpr int RAW = KC * AG_D * 2;           // one raw array (k, beta or v) of a chunk
    static constexpr uint32_t SBO = (KC / 8) * 128;     // core matrices: next 8 rows (M or N)
    static constexpr int SUP = 8 * BUILD;               // tokens per super-chunk of decay weights
    static constexpr int SMEM = 2 * OPS + 2 * 3 * RAW + SUP * 4 + 8 * 8 + 6 * 8 + 16;
};

// 2^-S for S = n + f (fp64 sum of decay exponents): exact power of two times
// exp2 of the fractional part; 0 for S beyond the float range, NaN stays NaN.
__device__ __forceinline__ float exp2_neg(double S) {
    if (!(S < 1.0e9)) return S != S ? __int_as_float(0x7fc00000) : 0.f;
    const double n = floor(S);
    const float f = static_cast<float>(S - n);                  // [0, 1)
    const int e = static_cast<int>(fmax(fmin(n, 300.0), -300.0));
    return ldexpf(exp2f(-f), -e);
}

// (x0, x1) -> bf16x2 pieces hi = rn(x), mid = rn(x - hi), lo = rn(x - hi -
// mid), low half = x0; hi + mid + lo equals x to fp32 rounding (x - hi and
// x - hi - mid are exact in fp32)
__device__ __forceinline__ void split3(float x0, float x1, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    const float r0 = x0 - __uint_as_float(hi << 16), r1 = x1 - __uint_as_float(hi & 0xffff0000u);
    const __nv_bfloat162 m = __floats2bfloat162_rn(r0, r1);
    mid = *reinterpret_cast<const uint32_t*>(&m);
    const __nv_bfloat162 l = __floats2bfloat162_rn(r0 - __uint_as_float(mid << 16),
                                                   r1 - __uint_as_float(mid & 0xffff0000u));
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Named CTA barrier `ID` (0 is __syncthreads) over `n` threads, whole warps.
template <int ID>
__device__ __forceinline__ void named_sync(int n) {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "r"(n) : "memory");
}

struct AggArgs {
    const __nv_bfloat16* k;
    const __nv_bfloat16* beta;
    const __nv_bfloat16* v;
    const __nv_bfloat16* d;
    const float* A;
    float* agg;              // [P-1][BH][2][128][128]
    AggScale* agg_scale;     // [P-1][BH]
    long long BH;
    int H, T;
    long long d_ld;          // tokens between consecutive heads' rows of d
    int part_len;
    long long wait_ns;
};

// ETA_ONLY: the non-metaplastic limit needs only Delta eta (its carry and
// full pass ignore the J half): 4 operand tiles and 3 products a K step
// instead of 8 and 6, and J written as zeros.
template <int KC, bool ETA_ONLY = false>
__global__ void __launch_bounds__(AggShape<KC>::THREADS, AggShape<KC>::CTAS_PER_SM)
diag_agg_tc_kernel(const AggArgs p) {
    using Sh = AggShape<KC>;
    constexpr int AG_KC = KC, AG_BUILD = Sh::BUILD, AG_TILE = Sh::TILE, AG_OPS = Sh::OPS,
                  AG_RAW = Sh::RAW, AG_SUP = Sh::SUP;
    constexpr uint32_t AG_SBO = Sh::SBO;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ops = smem;                                  // [2][7 tiles]
    unsigned char* raw = smem + 2 * AG_OPS;                     // [2 stages][k, beta, v]
    float* wsup = reinterpret_cast<float*>(raw + 2 * 3 * AG_RAW);   // [AG_SUP] weights of a super-chunk
    double* wtot = reinterpret_cast<double*>(wsup + AG_SUP);        // [warps] warp totals
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(wtot + 8);
    uint64_t* mma_done = raw_full + 2;
    uint64_t* ops_full = mma_done + 2;                          // a chunk's operands built (per build warp)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(ops_full + 2);
    float* s_wend = reinterpret_cast<float*>(tmem_holder + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long bh = blockIdx.x;
    const int part = blockIdx.y;
    const int T = p.T;
    const int tb = part * p.part_len;
    const int te = min(T, tb + p.part_len);
    const int nch = (te - tb + AG_KC - 1) / AG_KC;
    const long long S = static_cast<long long>(AG_D) * AG_D;
    bool ok = true;

    // raw chunk of iteration `it` (chunk nch-1-it) into stage it & 1 (thread 0)
    auto issue = [&](int it) {
        const int st = it & 1;
        const int c = nch - 1 - it;
        const int t0 = tb + c * AG_KC, n = min(AG_KC, te - t0);
        const uint32_t bytes = static_cast<uint32_t>(n * AG_D * 2);
        const long long off = (bh * T + t0) * AG_D;
        unsigned char* dst = raw + st * 3 * AG_RAW;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&raw_full[st], 3 * bytes);
        bulk_g2s(dst, p.k + off, bytes, &raw_full[st]);
        bulk_g2s(dst + AG_RAW, p.beta + off, bytes, &raw_full[st]);
        bulk_g2s(dst + 2 * AG_RAW, p.v + off, bytes, &raw_full[st]);
    };

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&mma_done[i], 1);
            mbar_init(&ops_full[i], AG_BUILD / 32);
        }
        mbar_init_fence();
        for (int it = 0; it < 2 && it < nch; ++it) issue(it);
    }
    if (warp == 0) tmem_alloc(tmem_holder, AG_TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    const float Ah = p.A[bh % p.H];
    double Z = 0.0;          // sum of the decay exponents of the tokens after the current super-chunk
    int sup0 = tb;           // first token of the current super-chunk
    const bool builder = tid < AG_BUILD;    // else the issuing warp
    const int pr = tid & 63;                // a builder's operand rows 2 pr, 2 pr + 1
    const int kg = tid >> 6;                // and its group of 8 tokens of a chunk (AG_KC / 8 groups)
    static_assert(AG_BUILD == 64 * (AG_KC / 8), "one build thread per (row pair, token group)");
    static_assert(AG_SUP == 8 * AG_BUILD, "a build thread prepares 8 weights of a super-chunk");
    constexpr uint32_t IDESC = umma_idesc_bf16_f32(AG_D, AG_D);

    for (int it = 0; it < nch; ++it) {
        const int st = it & 1, ob = it & 1;
        const int c = nch - 1 - it;
        const int t0 = tb + c * AG_KC, n = min(AG_KC, te - t0);
        if (!builder) {
            // ---- the issuing warp: once every build warp has arrived on the
            // chunk's operand barrier, the next copies into the consumed raw
            // stage and the chunk's products ----
            if (!mbar_wait(&ops_full[ob], (it >> 1) & 1, p.wait_ns)) ok = false;
            if (lane == 0) {
                if (it + 2 < nch) issue(it + 2);
                tc_fence_after_sync();
                const uint32_t base = smem_addr(ops + ob * AG_OPS);
#pragma unroll
                for (int s = 0; s < AG_KC / 16; ++s) {
                    auto desc = [&](int tile) {
                        return umma_desc_kmajor(base + tile * AG_TILE + s * 2 * 128, AG_LBO, AG_SBO);
                    };
                    const uint32_t first = (it == 0 && s == 0) ? 0u : 1u;
                    if (!ETA_ONLY) {
                        umma_bf16(tmem, desc(0), desc(5), IDESC, first);       // J += A_beta B_wk2 hi
                        umma_bf16(tmem, desc(0), desc(6), IDESC, 1u);          //    + A_beta B_wk2 mid
                        umma_bf16(tmem, desc(0), desc(7), IDESC, 1u);          //    + A_beta B_wk2 lo
                    }
                    umma_bf16(tmem + AG_D, desc(1), desc(4), IDESC, first);    // eta += A_E hi B_k
                    umma_bf16(tmem + AG_D, desc(2), desc(4), IDESC, 1u);       //      + A_E mid B_k
                    umma_bf16(tmem + AG_D, desc(3), desc(4), IDESC, 1u);       //      + A_E lo B_k
                }
                umma_commit(&mma_done[ob]);
            }
            __syncwarp();
            continue;
        }
        if (it == 0 || ((c + 1) % (AG_SUP / AG_KC)) == 0) {
            // ---- decay weights of this chunk's super-chunk: chunks
            // [SC, SC + AG_SUP / AG_KC) of the part, SC a multiple of it, so
            // super-chunks hold whole chunks.  The builders' barrier 1 below
            // orders every build that read wsup before its rewrite.
            sup0 = tb + (c / (AG_SUP / AG_KC)) * AG_SUP;
            const int s1 = min(te, sup0 + AG_SUP);
            const int u0 = sup0 + 8 * tid;
            double x[8], loc = 0.0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = u0 + u;
                x[u] = t < s1 ? static_cast<double>(Ah * __bfloat162float(p.d[bh * p.d_ld + t]) * LOG2E) : 0.0;
                loc += x[u];
            }
            // exclusive suffix sum over the threads after this one
            double suf = loc;      // inclusive suffix within the warp
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double y = __shfl_down_sync(0xffffffffu, suf, off);
                if (lane + off < 32) suf += y;
            }
            if (lane == 0) wtot[warp] = suf;
            named_sync<1>(AG_BUILD);
            double later = suf - loc;
            double all = 0.0;
#pragma unroll
            for (int w = 0; w < AG_BUILD / 32; ++w) {
                const double tw = wtot[w];
                all += tw;
                if (w > warp) later += tw;
            }
            later += Z;
#pragma unroll
            for (int u = 7; u >= 0; --u) {
                wsup[8 * tid + u] = u0 + u < s1 ? exp2_neg(later) : 0.f;
                later += x[u];
            }
            Z += all;
            named_sync<1>(AG_BUILD);   // weights ready; wtot may be reused
        }
        if (!mbar_wait(&raw_full[st], (it >> 1) & 1, p.wait_ns)) ok = false;
        // the operand buffer was last read by the MMAs of iteration it - 2
        if (it >= 2 && !mbar_wait(&mma_done[ob], ((it - 2) >> 1) & 1, p.wait_ns)) ok = false;

        // ---- build the 8 operand tiles of this chunk (rows 2pr, 2pr+1; tokens 8kg..8kg+7) ----
        {
            const unsigned char* rk = raw + st * 3 * AG_RAW;
            const unsigned char* rb = rk + AG_RAW;
            const unsigned char* rv = rb + AG_RAW;
            const float* w = wsup + (t0 - sup0);
            uint32_t t[AG_NTILE][2][4];   // [tile][row of the pair][4 x bf16x2 along the tokens]
#pragma unroll
            for (int u2 = 0; u2 < 4; ++u2) {
                float ae[2][2], wk2[2][2];
                uint32_t kbits[2][2], bbits[2][2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = kg * 8 + 2 * u2 + e;
                    const bool valid = tok < n;
                    const float wt = valid ? w[tok] : 0.f;
                    const int o4 = (tok * AG_D + 2 * pr) * 2;
                    const uint32_t bb = valid ? *reinterpret_cast<const uint32_t*>(rb + o4) : 0u;
                    const uint32_t vv = valid ? *reinterpret_cast<const uint32_t*>(rv + o4) : 0u;
                    const uint32_t kk = valid ? *reinterpret_cast<const uint32_t*>(rk + o4) : 0u;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        bbits[r][e] = r ? (bb >> 16) : (bb & 0xffffu);
                        const float bf = __uint_as_float(bbits[r][e] << 16);
                        const float vf = __uint_as_float(r ? (vv & 0xffff0000u) : (vv << 16));
                        kbits[r][e] = r ? (kk >> 16) : (kk & 0xffffu);
                        const float kf = __uint_as_float(kbits[r][e] << 16);
                        ae[r][e] = (wt * bf) * vf;
                        wk2[r][e] = wt * (kf * kf);   // k^2 is exact in fp32 (16 significant bits)
                    }
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (!ETA_ONLY) {
                        t[0][r][u2] = bbits[r][0] | (bbits[r][1] << 16);
                        split3(wk2[r][0], wk2[r][1], t[5][r][u2], t[6][r][u2], t[7][r][u2]);
                    }
                    split3(ae[r][0], ae[r][1], t[1][r][u2], t[2][r][u2], t[3][r][u2]);
                    t[4][r][u2] = kbits[r][0] | (kbits[r][1] << 16);
                }
            }
            unsigned char* o = ops + ob * AG_OPS;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int rho = 2 * pr + r;
                const int off = ((rho >> 3) * (AG_KC / 8) + kg) * 128 + (rho & 7) * 16;   // core matrix (rho/8, kg)
#pragma unroll
                for (int tile = ETA_ONLY ? 1 : 0; tile < (ETA_ONLY ? 5 : AG_NTILE); ++tile)
                    *reinterpret_cast<uint4*>(o + tile * AG_TILE + off) =
                        make_uint4(t[tile][r][0], t[tile][r][1], t[tile][r][2], t[tile][r][3]);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&ops_full[ob]);   // operands written, raw stage consumed
    }

    // ---- end state and scale of the part -------------------------------------
    if (nch > 0 && !mbar_wait(&mma_done[(nch - 1) & 1], ((nch - 1) >> 1) & 1, p.wait_ns)) ok = false;
    if (tid == 0) {
        // Z = L, the part's total decay exponent
        int R;
        float W;
        if (!(Z < 1073741824.0)) {                 // decays to 0 (or NaN): 2^-R underflows
            R = 1 << 30;
            W = 1.f;
        } else if (!(Z > -1073741824.0)) {         // growth beyond any float
            R = -(1 << 30);
            W = 1.f;
        } else {
            const double fl = floor(Z);
            R = static_cast<int>(fl);
            W = exp2f(static_cast<float>(Z - fl));
        }
        *s_wend = W;
        p.agg_scale[static_cast<long long>(part) * p.BH + bh] = {W, R};
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (builder) {
        const float W = *s_wend;
        // build warp w reads TMEM lanes 32 (w % 4) .. + 31; the warps of a
        // lane quarter share its 256 columns (J, then eta)
        constexpr int QW = AG_BUILD / 128;                   // warps per lane quarter
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const int c_begin = (warp >> 2) * (2 * AG_D / QW), c_end = c_begin + 2 * AG_D / QW;
        for (int cc = c_begin; cc < c_end; cc += 32) {
            const int half = cc / AG_D, c0 = cc - half * AG_D;   // J (0) or eta (1)
            float* dst = p.agg + (static_cast<long long>(part) * p.BH + bh) * 2 * S + half * S +
                         static_cast<long long>(row) * AG_D;
            float v[32];
            if (ETA_ONLY && half == 0) {   // J: not accumulated
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            } else {
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + half * AG_D + c0, v);
            }
            if (nch == 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(dst + c0 + j) =
                    make_float4(v[j] * W, v[j + 1] * W, v[j + 2] * W, v[j + 3] * W);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, AG_TMEM_COLS);
    if (!ok) record_error(&g_diag_error, KDN_ERR_TIMEOUT);
}

}  // namespace
}  // namespace diag
}  // namespace kdn
