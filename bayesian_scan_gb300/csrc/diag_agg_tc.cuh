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
// v_t[i]) k_t[j].  The fp32 factor w beta v is split into three bf16 pieces
// whose sum is the fp32 value exactly (split3 below), so every term of
// Delta eta, whose signed terms can cancel, is as accurate as the fp32
// product it stands for.  The factor w k^2 is split into two (split2): a
// term of Delta J then falls short by less than 2^-16 of itself, and with
// beta >= 0 (a gate in (0, 1) on the pages) every term is non-negative, so
// Delta J is within 2^-16 of its fp32 value, with no cancellation to
// amplify it: the carried states are fp32-accurate (eta) or within 2^-16
// (J), not bf16-accurate.  The decay exponents are summed in two-float form
// (about 48 significant bits from error-free fp32 additions;
// fp64 on this GPU runs at a small fraction of the fp32 rate, and fp64 sums
// took 13-15 thousand cycles per super-chunk) and w_t = 2^-floor(S) *
// exp2(-frac(S)).
//
// Output: the same (J_w, eta_w) = W (Delta J, Delta eta) and (W, R) with
// 2^-R / W = 2^-L, W in [1, 2), that the CUDA-core aggregate pass leaves for
// the carry kernel.
//
// Per CTA: one (head, part); 8 KC build threads and one issuing warp.
// Chunks of the part are visited from the last to the first (so the suffix
// sums accumulate).  The weights w_t of a super-chunk of tokens are prepared
// by the build threads (8 tokens each, two-float suffix sums across them).
// Per chunk the build threads load their part of the raw chunk (k, beta, v,
// brought in by 1-D bulk copies AG_NS chunks ahead) into registers and
// release its stage on the stage's empty barrier, then write the 7 operand
// tiles (128 x KC bf16 each, core-matrix layout) and arrive, one lane per
// warp, on the chunk's operand barrier.  The issuing warp refills each
// released stage with the copies of the chunk AG_NS later, waits for the
// operands, issues the chunk's products and commits them to an mbarrier.
// Operand tiles are double-buffered on that barrier, so the build threads
// never wait for the products to be issued (a build thread that also issued
// held its warp, and at the chunk barrier all others, for about 770 cycles a
// chunk).  The operand build, not HBM, sets the kernel's speed: a clock64
// timeline of a 32-token chunk showed ~1200 cycles of build arithmetic and
// stores, ~300 of loads and ~300 waiting for the products of two chunks
// before, against ~770 of tensor-core work.  All waits are bounded by GPU
// time.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kdn_device.cuh"

namespace kdn {
namespace diag {
namespace {

constexpr int AG_D = 128;                          // d_k = d_v
constexpr int AG_NTILE = 8;                        // A_beta, A_E hi/mid/lo, B_k, B_wk2 hi/lo, (unused)
constexpr int AG_NTILE_BUILT = 7;                  // the tiles a chunk writes
// tensor memory: 256 columns (J in [0,128), eta in [128,256)); the wide
// form takes 512 (J pieces in [0,256), eta^T pieces in [256,512))
constexpr int AG_TMEM_COLS = 256;
constexpr uint32_t AG_LBO = 128;                   // core matrices: next 8 tokens (K)
constexpr int AG_NS = 3;                           // raw chunk stages (copies in flight)

// Chunk shapes: KC tokens per chunk, 8 KC build threads (one per row pair
// and group of 8 tokens) and one more warp that issues the products and the
// copies.  KC = 32: 288 threads, one CTA per SM (208 KB of shared memory);
// KC = 16: 160 threads, two CTAs per SM (104 KB each; each CTA holds 256 of
// the SM's 512 TMEM columns), for grids with at least two CTAs per SM.
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
    // Wide products (the one-CTA shape, whose CTA may hold all 512 TMEM
    // columns): J takes A_beta x [B_wk2 hi | B_wk2 lo] as one N = 256
    // product (two accumulators, added in the epilogue), and eta is formed
    // transposed, eta^T = k x [A_E hi | A_E mid] + k x A_E lo: 3 products a
    // K step instead of 5, and less shared memory read by the tensor core;
    // the eta-only variant takes the two eta^T products.
    static constexpr bool WIDE = KC == 32;
    static constexpr int NBAR = 2 * AG_NS + 4;          // raw_full, raw_empty [AG_NS]; mma_done, ops_full [2]
    static constexpr int SMEM = 2 * OPS + AG_NS * 3 * RAW + SUP * 4 + 8 * 8 + NBAR * 8 + 16;
};

// A sum of decay exponents in two-float form, hi + lo with |lo| at most
// half an ulp of hi.  Addition takes the exact rounding error of hi + hi
// (Knuth's TwoSum: six fp32 additions, no rounding-mode or FMA tricks), adds
// the low parts to it and renormalises: about 48 significant bits.  An
// infinite or NaN sum is kept as it is (hi), as fp64 would.
struct Xs {
    float hi, lo;
};

__device__ __forceinline__ Xs xs_add(Xs a, Xs b) {
    const float s = a.hi + b.hi;
    const float bp = s - a.hi;
    const float e = ((a.hi - (s - bp)) + (b.hi - bp)) + (a.lo + b.lo);
    const float h = s + e;
    if (!(fabsf(s) <= 3.0e38f)) return {s, 0.f};
    return {h, e - (h - s)};
}

__device__ __forceinline__ Xs xs_shfl_down(Xs a, int off) {
    return {__shfl_down_sync(0xffffffffu, a.hi, off), __shfl_down_sync(0xffffffffu, a.lo, off)};
}

// S = n + f with n = floor(S) and f in [0, 1) (f rounded to fp32)
__device__ __forceinline__ void xs_floor_frac(Xs S, float& n, float& f) {
    n = floorf(S.hi);
    f = (S.hi - n) + S.lo;        // S.hi - n is exact
    if (f < 0.f) {
        f += 1.f;
        n -= 1.f;
    } else if (f >= 1.f) {
        f -= 1.f;
        n += 1.f;
    }
}

// 2^-S for a sum S of decay exponents: exact power of two times exp2 of the
// fractional part; 0 for S beyond the float range, NaN stays NaN.
__device__ __forceinline__ float exp2_neg(Xs S) {
    if (!(S.hi < 1.0e9f)) return S.hi != S.hi ? __int_as_float(0x7fc00000) : 0.f;
    float n, f;
    xs_floor_frac(S, n, f);
    const int e = static_cast<int>(fmaxf(fminf(n, 300.f), -300.f));
    return ldexpf(exp2f(-f), -e);
}

// Three bf16 pieces of each of x.x, x.y, as fp32 bit patterns with the low
// 16 bits zero: hi keeps the top 8 significant bits of x (truncation), mid
// the top 8 of the remainder x - hi, and the remainder after that has at most
// 8 significant bits, so lo holds it exactly; both differences are exact in
// fp32, so hi + mid + lo = x exactly.  Bit operations and two packed
// subtractions, no conversions.
__device__ __forceinline__ void split3(float2 x, uint32_t (&h)[2], uint32_t (&m)[2], uint32_t (&l)[2]) {
    h[0] = __float_as_uint(x.x) & 0xffff0000u;
    h[1] = __float_as_uint(x.y) & 0xffff0000u;
    const float2 r = __fadd2_rn(x, make_float2(-__uint_as_float(h[0]), -__uint_as_float(h[1])));
    m[0] = __float_as_uint(r.x) & 0xffff0000u;
    m[1] = __float_as_uint(r.y) & 0xffff0000u;
    const float2 s = __fadd2_rn(r, make_float2(-__uint_as_float(m[0]), -__uint_as_float(m[1])));
    l[0] = __float_as_uint(s.x);
    l[1] = __float_as_uint(s.y);
}

// Two bf16 pieces of each of x.x, x.y (bit patterns, low 16 bits of lo not
// cleared: packing takes the upper halves): hi keeps the top 8 significant
// bits by truncation and lo the top 8 of the exact remainder, so hi + lo
// falls short of x by less than 2^-16 |x|.
__device__ __forceinline__ void split2(float2 x, uint32_t (&h)[2], uint32_t (&l)[2]) {
    h[0] = __float_as_uint(x.x) & 0xffff0000u;
    h[1] = __float_as_uint(x.y) & 0xffff0000u;
    const float2 r = __fadd2_rn(x, make_float2(-__uint_as_float(h[0]), -__uint_as_float(h[1])));
    l[0] = __float_as_uint(r.x);
    l[1] = __float_as_uint(r.y);
}

// bf16x2 of the upper halves of a (low half) and b
__device__ __forceinline__ uint32_t pack_hi(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

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
    unsigned char* ops = smem;                                  // [2][8 tiles]
    unsigned char* raw = smem + 2 * AG_OPS;                     // [AG_NS stages][k, beta, v]
    float* wsup = reinterpret_cast<float*>(raw + AG_NS * 3 * AG_RAW);   // [AG_SUP] weights of a super-chunk
    Xs* wtot = reinterpret_cast<Xs*>(wsup + AG_SUP);            // [warps] warp totals
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(wtot + 8);  // a stage's copies landed
    uint64_t* raw_empty = raw_full + AG_NS;                     // a stage read by every build warp
    uint64_t* mma_done = raw_empty + AG_NS;
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

    // raw chunk of iteration `it` (chunk nch-1-it) into stage it % AG_NS (one thread)
    auto issue = [&](int it) {
        const int st = it % AG_NS;
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
        for (int i = 0; i < AG_NS; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], AG_BUILD / 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&mma_done[i], 1);
            mbar_init(&ops_full[i], AG_BUILD / 32);
        }
        mbar_init_fence();
        for (int it = 0; it < AG_NS && it < nch; ++it) issue(it);
    }
    constexpr bool WIDE = Sh::WIDE;
    constexpr int TMEM_COLS = WIDE ? 4 * AG_D : AG_TMEM_COLS;
    if (warp == 0) tmem_alloc(tmem_holder, TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    const float Ah = p.A[bh % p.H];
    Xs Z = {0.f, 0.f};       // sum of the decay exponents of the tokens after the current super-chunk
    int sup0 = tb;           // first token of the current super-chunk
    const bool builder = tid < AG_BUILD;    // else the issuing warp
    const int pr = tid & 63;                // a builder's operand rows 2 pr, 2 pr + 1
    // A builder keeps its two rows in the order (2 pr + flip, 2 pr + 1 -
    // flip), flip = bit 2 of pr, so that the 8 lanes of each quarter-warp
    // 16-byte store cover all 8 rows of a core matrix row group (8 distinct
    // bank groups): without it a store met 2-way bank conflicts.
    const uint32_t flip = (pr >> 2) & 1;
    const uint32_t swap_sel = flip ? 0x1032u : 0x3210u;   // swaps the bf16 halves of a word
    const int kg = tid >> 6;                // and its group of 8 tokens of a chunk (AG_KC / 8 groups)
    static_assert(AG_BUILD == 64 * (AG_KC / 8), "one build thread per (row pair, token group)");
    static_assert(AG_SUP == 8 * AG_BUILD, "a build thread prepares 8 weights of a super-chunk");
    constexpr uint32_t IDESC = umma_idesc_bf16_f32(AG_D, AG_D);
    constexpr uint32_t IDESC_WIDE = umma_idesc_bf16_f32(AG_D, 2 * AG_D);

    int st = 0;              // raw stage of iteration it (it % AG_NS)
    uint32_t rph = 0;        // its barriers' phase ((it / AG_NS) & 1)
    for (int it = 0; it < nch; ++it) {
        const int ob = it & 1;
        const int c = nch - 1 - it;
        const int t0 = tb + c * AG_KC, n = min(AG_KC, te - t0);
        if (!builder) {
            // ---- the issuing warp: refill the stage once every build warp
            // has read it, then the chunk's products once its operands are
            // built ----
            if (it + AG_NS < nch) {
                if (!mbar_wait(&raw_empty[st], rph, p.wait_ns)) ok = false;
                if (lane == 0) issue(it + AG_NS);
            }
            if (!mbar_wait(&ops_full[ob], (it >> 1) & 1, p.wait_ns)) ok = false;
            if (lane == 0) {
                tc_fence_after_sync();
                const uint32_t base = smem_addr(ops + ob * AG_OPS);
#pragma unroll
                for (int s = 0; s < AG_KC / 16; ++s) {
                    auto desc = [&](int tile) {
                        return umma_desc_kmajor(base + tile * AG_TILE + s * 2 * 128, AG_LBO, AG_SBO);
                    };
                    const uint32_t first = (it == 0 && s == 0) ? 0u : 1u;
                    if (WIDE) {
                        // tiles 5, 6 (and 1, 2) are adjacent: one 256-row operand
                        if (!ETA_ONLY)
                            umma_bf16(tmem, desc(0), desc(5), IDESC_WIDE, first);      // J: hi | lo
                        umma_bf16(tmem + 2 * AG_D, desc(4), desc(1), IDESC_WIDE, first);   // eta^T: hi | mid
                        umma_bf16(tmem + 2 * AG_D, desc(4), desc(3), IDESC, 1u);       //  + lo
                        continue;
                    }
                    if (!ETA_ONLY) {
                        umma_bf16(tmem, desc(0), desc(5), IDESC, first);       // J += A_beta B_wk2 hi
                        umma_bf16(tmem, desc(0), desc(6), IDESC, 1u);          //    + A_beta B_wk2 lo
                    }
                    umma_bf16(tmem + AG_D, desc(1), desc(4), IDESC, first);    // eta += A_E hi B_k
                    umma_bf16(tmem + AG_D, desc(2), desc(4), IDESC, 1u);       //      + A_E mid B_k
                    umma_bf16(tmem + AG_D, desc(3), desc(4), IDESC, 1u);       //      + A_E lo B_k
                }
                umma_commit(&mma_done[ob]);
            }
            __syncwarp();
            if (++st == AG_NS) { st = 0; rph ^= 1u; }
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
            const __nv_bfloat16* dp = p.d + bh * p.d_ld + u0;
            float dv8[8];
            if (u0 + 8 <= s1 && (reinterpret_cast<uintptr_t>(dp) & 15) == 0) {
                const uint4 raw8 = __ldg(reinterpret_cast<const uint4*>(dp));   // 8 tokens in one load
                const uint32_t w4[4] = {raw8.x, raw8.y, raw8.z, raw8.w};
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    dv8[u] = __uint_as_float((u & 1) ? (w4[u >> 1] & 0xffff0000u) : (w4[u >> 1] << 16));
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) dv8[u] = u0 + u < s1 ? __bfloat162float(dp[u]) : 0.f;
            }
            float x[8];
            Xs loc = {0.f, 0.f};
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                x[u] = u0 + u < s1 ? Ah * dv8[u] * LOG2E : 0.f;
                loc = xs_add(loc, {x[u], 0.f});
            }
            // inclusive suffix sum over the lanes from this one on
            Xs suf = loc;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const Xs y = xs_shfl_down(suf, off);
                if (lane + off < 32) suf = xs_add(suf, y);
            }
            Xs later = xs_shfl_down(suf, 1);       // the lanes after this one
            if (lane == 31) later = {0.f, 0.f};
            if (lane == 0) wtot[warp] = suf;     // the warp's total
            named_sync<1>(AG_BUILD);
            Xs all = {0.f, 0.f};
#pragma unroll
            for (int w = 0; w < AG_BUILD / 32; ++w) {
                const Xs tw = wtot[w];
                all = xs_add(all, tw);
                if (w > warp) later = xs_add(later, tw);
            }
            later = xs_add(later, Z);
#pragma unroll
            for (int u = 7; u >= 0; --u) {
                wsup[8 * tid + u] = u0 + u < s1 ? exp2_neg(later) : 0.f;
                later = xs_add(later, {x[u], 0.f});
            }
            Z = xs_add(Z, all);
            named_sync<1>(AG_BUILD);   // weights ready; wtot may be reused
        }
        if (!mbar_wait(&raw_full[st], rph, p.wait_ns)) ok = false;

        // ---- this thread's part of the raw chunk (rows 2pr, 2pr+1; tokens
        // 8kg..8kg+7) into registers, then the stage goes back to the copies ----
        uint32_t kk[8], bb[8], vv[8];
        float wt[8];
        {
            const unsigned char* rk = raw + st * 3 * AG_RAW;
            const unsigned char* rb = rk + AG_RAW;
            const unsigned char* rv = rb + AG_RAW;
            const float* w = wsup + (t0 - sup0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int tok = kg * 8 + u;
                const bool valid = tok < n;
                const int o4 = (tok * AG_D + 2 * pr) * 2;
                wt[u] = valid ? w[tok] : 0.f;
                bb[u] = valid ? *reinterpret_cast<const uint32_t*>(rb + o4) : 0u;
                vv[u] = valid ? *reinterpret_cast<const uint32_t*>(rv + o4) : 0u;
                kk[u] = valid ? *reinterpret_cast<const uint32_t*>(rk + o4) : 0u;
                bb[u] = __byte_perm(bb[u], 0u, swap_sel);   // low half: row 2 pr + flip
                vv[u] = __byte_perm(vv[u], 0u, swap_sel);
                kk[u] = __byte_perm(kk[u], 0u, swap_sel);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[st]);   // this warp's reads of the stage are done
        if (++st == AG_NS) { st = 0; rph ^= 1u; }
        // the operand buffer was last read by the MMAs of iteration it - 2
        if (it >= 2 && !mbar_wait(&mma_done[ob], ((it - 2) >> 1) & 1, p.wait_ns)) ok = false;

        // ---- build the 7 operand tiles of this chunk: products packed over
        // the row pair, pieces packed over token pairs ----
        {
            uint32_t t[AG_NTILE][2][4];   // [tile][row of the pair][4 x bf16x2 along the tokens]
#pragma unroll
            for (int u2 = 0; u2 < 4; ++u2) {
                uint32_t eh[2][2], em[2][2], el[2][2];   // [token of the pair][row]: pieces of w beta v
                uint32_t jh[2][2], jm[2][2];             //                                 of w k^2
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int u = 2 * u2 + e;
                    const float2 w2 = make_float2(wt[u], wt[u]);
                    const float2 bf = make_float2(__uint_as_float(bb[u] << 16), __uint_as_float(bb[u] & 0xffff0000u));
                    const float2 vf = make_float2(__uint_as_float(vv[u] << 16), __uint_as_float(vv[u] & 0xffff0000u));
                    const float2 kf = make_float2(__uint_as_float(kk[u] << 16), __uint_as_float(kk[u] & 0xffff0000u));
                    split3(__fmul2_rn(__fmul2_rn(w2, bf), vf), eh[e], em[e], el[e]);
                    if (!ETA_ONLY)   // k^2 is exact in fp32 (16 significant bits)
                        split2(__fmul2_rn(w2, __fmul2_rn(kf, kf)), jh[e], jm[e]);
                }
                const int u = 2 * u2;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t sel = r ? 0x7632u : 0x5410u;   // row r's halves of two tokens
                    if (!ETA_ONLY) {
                        t[0][r][u2] = __byte_perm(bb[u], bb[u + 1], sel);
                        t[5][r][u2] = pack_hi(jh[0][r], jh[1][r]);
                        t[6][r][u2] = pack_hi(jm[0][r], jm[1][r]);
                    }
                    t[1][r][u2] = pack_hi(eh[0][r], eh[1][r]);
                    t[2][r][u2] = pack_hi(em[0][r], em[1][r]);
                    t[3][r][u2] = pack_hi(el[0][r], el[1][r]);
                    t[4][r][u2] = __byte_perm(kk[u], kk[u + 1], sel);
                }
            }
            unsigned char* o = ops + ob * AG_OPS;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int rho = 2 * pr + (r ^ static_cast<int>(flip));
                const int off = ((rho >> 3) * (AG_KC / 8) + kg) * 128 + (rho & 7) * 16;   // core matrix (rho/8, kg)
#pragma unroll
                for (int tile = ETA_ONLY ? 1 : 0; tile < (ETA_ONLY ? 5 : AG_NTILE_BUILT); ++tile)
                    *reinterpret_cast<uint4*>(o + tile * AG_TILE + off) =
                        make_uint4(t[tile][r][0], t[tile][r][1], t[tile][r][2], t[tile][r][3]);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&ops_full[ob]);   // operands written
    }

    // ---- end state and scale of the part -------------------------------------
    if (nch > 0 && !mbar_wait(&mma_done[(nch - 1) & 1], ((nch - 1) >> 1) & 1, p.wait_ns)) ok = false;
    if (tid == 0) {
        // Z = L, the part's total decay exponent
        int R;
        float W;
        if (!(Z.hi < 1073741824.f)) {              // decays to 0 (or NaN): 2^-R underflows
            R = 1 << 30;
            W = 1.f;
        } else if (!(Z.hi > -1073741824.f)) {      // growth beyond any float
            R = -(1 << 30);
            W = 1.f;
        } else {
            float fl, f;
            xs_floor_frac(Z, fl, f);
            R = static_cast<int>(fl);
            W = exp2f(f);
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
            if constexpr (WIDE) {
                // J[row][c0 + j] = pieces' sum at columns c0 + j and 128 + c0 + j;
                // eta^T: lane `row` is the key column, columns 256 + c0 + j
                // (and 384 + c0 + j) the value rows c0 + j
                const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + half * 2 * AG_D + c0;
                float v[32], u[32];
                if (ETA_ONLY && half == 0) {   // J: not accumulated
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = u[j] = 0.f;
                } else {
                    tmem_ld32(ta, v);
                    tmem_ld32(ta + AG_D, u);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = nch == 0 ? 0.f : (v[j] + u[j]) * W;
                float* base = p.agg + (static_cast<long long>(part) * p.BH + bh) * 2 * S + half * S;
                if (half == 0) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(base + static_cast<long long>(row) * AG_D + c0 + j) =
                            make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)   // a warp writes 32 consecutive key columns of a row
                        base[static_cast<long long>(c0 + j) * AG_D + row] = v[j];
                }
                continue;
            }
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
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
    if (!ok) record_error(&g_diag_error, KDN_ERR_TIMEOUT);
}

}  // namespace
}  // namespace diag
}  // namespace kdn
