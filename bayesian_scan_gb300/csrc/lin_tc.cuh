// lin_tc.cuh -- the non-metaplastic limit on the tensor cores, for d_k = d_v
// = 128 and bf16 inputs ("Learning to Remember, Learn, and Forget in
// Attention-Based Models", Metodologia 4: with the importance held at I_prior
// the update is decayed linear attention).  Included by diag_impl.cuh.
//
// What is computed, per head: with S = I_prior mu (d_v x d_k, fp32),
//     S_t = alpha_t S_{t-1} + (beta_t . v_t) k_t^T,   o_t = S_t q_t / I_prior.
// How: chunks of C = 64 tokens.  With g_t = sum_{r <= t} log alpha_r inside a
// chunk (g_t <= 0), the chunk's outputs and end state are
//     o_t = [ sum_{s <= t} e^{g_t - g_s} (q_t . k_s) Vb_s  +  e^{g_t} S q_t ] / I_prior
//     S'  = e^{g_C} S + sum_s e^{g_C - g_s} Vb_s k_s^T,      Vb_s = beta_s . v_s,
// five matrix products per chunk, all with M = 128 rows on the tensor cores
// (tcgen05.mma kind::f16, bf16 operands staged in shared memory as 8 x
// 16-byte core matrices, fp32 accumulators in tensor memory):
//     P^T  [s x t] = K Q^T            (K padded to 128 rows; rows >= 64 unused)
//     Oi^T [i x t] = S Q^T            (S as hi + lo bf16 halves, read from
//                                      tensor memory as the A operand: 2 products)
//     Oa^T [i x t] = Vb^T P^T         (Vb and P as hi + lo halves: 3 products)
//     S   [i x j] += (w . Vb)^T K     (w_s = e^{g_C - g_s}; hi + lo: 2 products)
// The hi + lo splits keep every operand to ~2^-16 relative (one bf16 product
// alone loses ~2^-9, which fails the 2e-3 bar on o); q, k are bf16 inputs and
// exact.  Q and K are copied from the raw rows into K-major tiles ([token x
// j], 16-byte pieces of 8 consecutive j); the same tile of K is the state
// product's MN-major B operand, and Vb, w . Vb are built straight from the
// raw rows of beta and v as MN-major A operands in that layout, so no
// operand is transposed on the CUDA cores.  S lives in tensor memory for the
// whole sequence; once per chunk each warp reads its lanes and columns,
// writes the hi/lo halves back into tensor memory as packed bf16 pairs (the
// Oi product reads its A operand there, which leaves shared memory room for
// 64-token chunks) and scales S by e^{g_C} in place before the state product
// adds the chunk.  The P product is issued as soon as the Q and K tiles
// exist; warps 0, 1, 4, 5 copy its result to shared memory after the other
// tiles are built, and warps 1-4 turn it into the masked, decayed hi/lo
// operand of the Oa product while thread 0 issues the Oi and state products;
// thread 32 issues the Oa product.  One thread issues a tcgen05.mma about
// every 47 cycles, so the N = 64 products run at about 52 cycles each and
// the 36 products after the operand barrier take about 2000 cycles.  Warp 7 issues the 1-D
// bulk copies of the next chunk's q and k as soon as the Q and K tiles exist
// and of its v and beta once the operands are built, and computes the decay
// exponents one chunk ahead.
// All waits are bounded.

namespace kdn {
namespace lintc {
namespace {

constexpr int LD = 128;            // d_k = d_v
constexpr int LC = 64;             // tokens per chunk
constexpr int LTHREADS = 256;
constexpr uint32_t LTMEM_COLS = 512;
// tensor memory columns: S (fp32), its hi / lo bf16 halves as packed pairs
// (the A operand of the Oi product), the Oa and Oi accumulators, P^T
constexpr uint32_t COL_S = 0, COL_SH = 128, COL_SL = 192, COL_OA = 256, COL_OI = 320, COL_P = 384;
constexpr float LOG2E_L = 1.4426950408889634f;
// shared memory (bytes); K-major operand tiles: element (row r, k) at
// (r / 8) * SBO + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2
constexpr int RAW1 = LC * LD * 2;                 // one input array of a chunk
constexpr int RAW_STAGE = 4 * RAW1;               // q, k, v, beta (one stage)
constexpr int OFF_RAW = 0;
constexpr int OFF_KB = OFF_RAW + RAW_STAGE;       // [s x j], read as 128 rows by the P product
constexpr int OFF_QB = OFF_KB + LC * LD * 2;      // [t x j]
constexpr int OFF_VH = OFF_QB + LC * LD * 2;      // Vb [s x i] hi, lo (MN-major A operand)
constexpr int OFF_AW = OFF_VH + 2 * LD * LC * 2;  // w . Vb [s x i] hi, lo (MN-major A operand)
constexpr int OFF_P = OFF_AW + 2 * LD * LC * 2;   // [t x s] hi, lo
constexpr int OFF_PRAW = OFF_P + 2 * LC * LC * 2; // [t][s] fp32 copy of P^T
constexpr int PRAW_LD = LC + 4;
constexpr int OFF_MISC = OFF_PRAW + LC * PRAW_LD * 4;
constexpr int SBO_J = (LD / 8) * 128;             // K = 128 (j)
constexpr int SBO_C = (LC / 8) * 128;             // K = 64 (s)
constexpr int LSMEM = OFF_MISC + 2048;
static_assert(OFF_KB + (LD / 8) * SBO_J <= LSMEM, "the P product's 128-row read of K stays in shared memory");
static_assert(LSMEM <= 227 * 1024, "shared memory");

struct LinArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* beta;
    const __nv_bfloat16* d;
    const float* A;
    float Ip;
    const float* mu0;      // part 0's initial mean, or null
    const float* agg;      // start states of parts 1.. (carry pass output), or null
    float* out;
    float* final_mu;       // or null
    long long BH;
    int H, T, part_len;
    long long wait_ns;
};

// 2^x by the hardware approximation (MUFU ex2); results below the normal
// range flush to zero.  The library exp2f takes a slow path for the large
// negative arguments that fast decay gives, which cost more than the rest of
// the P operand's build.
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// hi + lo bf16 halves of a pair (x0, x1), packed two per 32-bit word: hi is
// x truncated to bf16 (exact, an integer mask), lo the rest x - hi (exact in
// fp32, below 2^-7 |x|) rounded to bf16, so hi + lo is within 2^-16 |x|.
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const uint32_t b0 = __float_as_uint(x0) & 0xffff0000u, b1 = __float_as_uint(x1) & 0xffff0000u;
    hi = (b0 >> 16) | b1;
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __uint_as_float(b0), x1 - __uint_as_float(b1));
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// D (TMEM) = A (TMEM, bf16 pairs packed per column, lane = row) * B^T (smem)
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t v[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

template <int D_>
__global__ void __launch_bounds__(LTHREADS, 1) lin_tc_kernel(const LinArgs p) {
    static_assert(D_ == LD, "d_k = d_v = 128");
    extern __shared__ __align__(128) unsigned char smem[];
    // per chunk (double-buffered by chunk parity): g_t, e^{g_t}, e^{g_C - g_t}, then e^{g_C}
    float* s_gall = reinterpret_cast<float*>(smem + OFF_MISC);       // [2][3][LC]
    float* s_eglall = s_gall + 2 * 3 * LC;                           // [2] (+2 pad)
    uint64_t* raw_qk = reinterpret_cast<uint64_t*>(s_eglall + 4);   // q, k of a chunk landed
    uint64_t* raw_bv = raw_qk + 1;                                     // v, beta of a chunk landed
    uint64_t* bar_p = raw_bv + 1;
    uint64_t* bar_o = bar_p + 1;
    uint32_t* holder = reinterpret_cast<uint32_t*>(bar_o + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long bh = blockIdx.x;
    const int part = blockIdx.y;
    const int T = p.T;
    const int tb = min(T, part * p.part_len);
    const int te = min(T, tb + p.part_len);
    const int nch = (te - tb + LC - 1) / LC;
    const long long S2 = static_cast<long long>(LD) * LD;
    const float Ah = p.A[bh % p.H];
    bool ok = true;

    // One thread: raw inputs of chunk c into the stage, in two halves with a
    // barrier each, so that q and k of the next chunk are fetched as soon as
    // this chunk's Q and K tiles exist.
    auto issue = [&](int c, bool qk) {
        const int t0 = tb + c * LC, n = min(LC, te - t0);
        const uint32_t bytes = static_cast<uint32_t>(n * LD * 2);
        const long long off = (bh * T + t0) * LD;
        unsigned char* dst = smem + OFF_RAW;
        uint64_t* bar = qk ? raw_qk : raw_bv;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(bar, 2 * bytes);
        if (qk) {
            bulk_g2s(dst, p.q + off, bytes, bar);
            bulk_g2s(dst + RAW1, p.k + off, bytes, bar);
        } else {
            bulk_g2s(dst + 2 * RAW1, p.v + off, bytes, bar);
            bulk_g2s(dst + 3 * RAW1, p.beta + off, bytes, bar);
        }
    };

    if (tid == 0) {
        mbar_init(raw_qk, 1);
        mbar_init(raw_bv, 1);
        mbar_init(bar_p, 1);
        mbar_init(bar_o, 2);   // two issuing threads commit per chunk
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(holder, LTMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *holder;
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const int row = 32 * q4 + lane;          // its TMEM lane = state row i
    const int cbase = (warp >> 2) * 64;      // its half of the state's columns
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);

    // ---- initial state S = I_prior mu_start into tensor memory ---------------
    {
        const float* src = nullptr;
        float scale = p.Ip;
        if (part > 0) {
            src = p.agg + (static_cast<long long>(part - 1) * p.BH + bh) * 2 * S2 + S2;   // eta part
            scale = 1.f;
        } else if (p.mu0) {
            src = p.mu0 + bh * S2;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (src) x = *reinterpret_cast<const float4*>(src + static_cast<long long>(row) * LD + cbase + 32 * h + j);
                v[j] = x.x * scale;
                v[j + 1] = x.y * scale;
                v[j + 2] = x.z * scale;
                v[j + 3] = x.w * scale;
            }
            tmem_st32(tl + COL_S + cbase + 32 * h, v);
        }
        tmem_wait_st();
    }

    constexpr uint32_t IDESC_T = umma_idesc_bf16_f32(128, LC);    // N = 64 tokens
    constexpr uint32_t IDESC_OA = umma_idesc_bf16_f32(128, LC, true);          // A = Vb^T MN-major
    constexpr uint32_t IDESC_S = umma_idesc_bf16_f32(128, LD, true, true);     // A = (w Vb)^T, B = K: MN-major
    // Warp 7 keeps the raw-input copies and the decay exponents one chunk
    // ahead (threads 0 and 32 issue the MMAs): exponents of chunk c from the
    // d of its tokens (dn0: token lane, dn1: token 32 + lane), into buffer c & 1.
    __nv_bfloat16 dn0 = __float2bfloat16_rn(0.f), dn1 = dn0;
    auto load_d = [&](int c) {
        const int t0 = tb + c * LC, n = min(LC, te - t0);
        dn0 = __float2bfloat16_rn(0.f);
        dn1 = dn0;
        if (lane < n) dn0 = p.d[bh * T + t0 + lane];
        if (32 + lane < n) dn1 = p.d[bh * T + t0 + 32 + lane];
    };
    auto exponents = [&](int c) {   // warp 7
        const int t0 = tb + c * LC, n = min(LC, te - t0);
        float a0 = lane < n ? -Ah * __bfloat162float(dn0) : 0.f;
        float a1 = 32 + lane < n ? -Ah * __bfloat162float(dn1) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, a0, o);
            const float y1 = __shfl_up_sync(0xffffffffu, a1, o);
            if (lane >= o) {
                a0 += y0;
                a1 += y1;
            }
        }
        a1 += __shfl_sync(0xffffffffu, a0, 31);
        const float gl = __shfl_sync(0xffffffffu, a1, 31);
        float* g = s_gall + (c & 1) * 3 * LC;
        g[lane] = a0;
        g[32 + lane] = a1;
        g[LC + lane] = expf(a0);
        g[LC + 32 + lane] = expf(a1);
        g[2 * LC + lane] = expf(gl - a0);
        g[2 * LC + 32 + lane] = expf(gl - a1);
        if (lane == 0) s_eglall[c & 1] = expf(gl);
        if (c + 1 < nch) load_d(c + 1);
    };
    if (warp == 7 && nch > 0) {
        if (lane == 0) {
            issue(0, true);
            issue(0, false);
        }
        load_d(0);
        exponents(0);
    }
    __syncthreads();   // chunk 0's exponents

    const uint32_t sbase = smem_addr(smem);
    auto dj = [&](int off, int ks) { return umma_desc_kmajor(sbase + off + ks * 256, 128, SBO_J); };
    auto dc = [&](int off, int ks) { return umma_desc_kmajor(sbase + off + ks * 256, 128, SBO_C); };
    // MN-major [s x (i or j)] tiles in the Q/K tile layout: 16-byte pieces of
    // 8 consecutive i (or j) of one token, core matrices 128 bytes apart along
    // i and SBO_J along s; a K = 16 step is two core matrices along s
    auto dm = [&](int off, int ks) { return umma_desc_mnmajor(sbase + off + ks * 2 * SBO_J, SBO_J, 128); };
    float* praw = reinterpret_cast<float*>(smem + OFF_PRAW);

    for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        const int t0 = tb + c * LC, n = min(LC, te - t0);
        const float* s_g = s_gall + st * 3 * LC;
        const float* s_eg = s_g + LC;
        const float* s_w = s_g + 2 * LC;
        if (!mbar_wait(raw_qk, c & 1, p.wait_ns)) ok = false;
        const unsigned char* rq = smem + OFF_RAW;
        const unsigned char* rk = rq + RAW1;
        const unsigned char* rv = rq + 2 * RAW1;
        const unsigned char* rbt = rq + 3 * RAW1;
        // ---- Q and K tiles [token x j] (16-byte pieces), then the P product.
        // A warp instruction moves 8 tokens x 4 of their 16-byte pieces,
        // chosen in a checkerboard (piece (a + 2 b + u) mod 8 of token a for
        // lane 8 b + a), so that both the row reads (bank group = piece mod 8)
        // and the core-matrix writes (bank group = token mod 8) hit each bank
        // group exactly four times ----
        static_assert(LC * (LD / 8) == 4 * LTHREADS, "four pieces per thread");
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int combo = warp + 8 * it, tg = combo >> 2, u = combo & 3;
            const int a = lane & 7, b = lane >> 3;
            const int t = 8 * tg + a, jc = 8 * (u >> 1) + ((a + 2 * b + (u & 1)) & 7);
            const int off = tg * SBO_J + jc * 128 + a * 16;
            uint4 qv = make_uint4(0u, 0u, 0u, 0u), kv = qv;
            if (t < n) {
                qv = *reinterpret_cast<const uint4*>(rq + t * LD * 2 + jc * 16);
                kv = *reinterpret_cast<const uint4*>(rk + t * LD * 2 + jc * 16);
            }
            *reinterpret_cast<uint4*>(smem + OFF_QB + off) = qv;
            *reinterpret_cast<uint4*>(smem + OFF_KB + off) = kv;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();   // Q, K tiles written
        if (tid == 0) {
            tc_fence_after_sync();
            // P^T [s x t] = K Q^T
#pragma unroll
            for (int ks = 0; ks < LD / 16; ++ks)
                umma_bf16(tmem + COL_P, dj(OFF_KB, ks), dj(OFF_QB, ks), IDESC_T, ks > 0 ? 1u : 0u);
            umma_commit(bar_p);
        }
        if (warp == 7 && lane == 0 && c + 1 < nch) issue(c + 1, true);   // q, k consumed
        if (!mbar_wait(raw_bv, c & 1, p.wait_ns)) ok = false;
        // ---- Vb = beta . v and w . Vb [s x i], hi and lo: the A operands of
        // the Oa and state products, MN-major (read as Vb^T), built piece by
        // piece from the raw rows in the Q/K tiles' checkerboard (K itself is
        // the state product's MN-major B operand) ----
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int combo = warp + 8 * it, tg = combo >> 2, u = combo & 3;
            const int a = lane & 7, b = lane >> 3;
            const int s_ = 8 * tg + a, ic = 8 * (u >> 1) + ((a + 2 * b + (u & 1)) & 7);
            const int off = tg * SBO_J + ic * 128 + a * 16;
            uint4 bq = make_uint4(0u, 0u, 0u, 0u), vq = bq;
            if (s_ < n) {
                bq = *reinterpret_cast<const uint4*>(rbt + s_ * LD * 2 + ic * 16);
                vq = *reinterpret_cast<const uint4*>(rv + s_ * LD * 2 + ic * 16);
            }
            const float ws = s_w[s_];
            const uint32_t bw[4] = {bq.x, bq.y, bq.z, bq.w}, vw[4] = {vq.x, vq.y, vq.z, vq.w};
            uint32_t vh[4], vl[4], ah[4], al[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {   // elements i = 8 ic + 2 e, + 1 (low, high halves)
                const float x0 = __uint_as_float(bw[e] << 16) * __uint_as_float(vw[e] << 16);
                const float x1 = __uint_as_float(bw[e] & 0xffff0000u) * __uint_as_float(vw[e] & 0xffff0000u);
                split_pair(x0, x1, vh[e], vl[e]);
                split_pair(ws * x0, ws * x1, ah[e], al[e]);
            }
            *reinterpret_cast<uint4*>(smem + OFF_VH + off) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
            *reinterpret_cast<uint4*>(smem + OFF_VH + LD * LC * 2 + off) = make_uint4(vl[0], vl[1], vl[2], vl[3]);
            *reinterpret_cast<uint4*>(smem + OFF_AW + off) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
            *reinterpret_cast<uint4*>(smem + OFF_AW + LD * LC * 2 + off) = make_uint4(al[0], al[1], al[2], al[3]);
        }
        // ---- P^T (TMEM lanes 0-63) to shared memory as fp32: warps 0, 1, 4,
        // 5 (the two lane quarters), 32 tokens each ----
        if (q4 < 2) {
            if (!mbar_wait(bar_p, c & 1, p.wait_ns)) ok = false;
            tc_fence_after_sync();
            float pv[32];
            const int tcol = (warp >> 2) * 32;
            tmem_ld32(tl + COL_P + tcol, pv);   // lane s = row: P^T[s][t]
#pragma unroll
            for (int t = 0; t < 32; ++t) praw[(tcol + t) * PRAW_LD + row] = pv[t];
        }
        // ---- S: its hi/lo bf16 halves into tensor memory (the A operand of
        // the Oi product), then S *= e^{g_C} in place ----
        {
            const float egl = s_eglall[st];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[32];
                tmem_ld32(tl + COL_S + cbase + 32 * h, v);
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) split_pair(v[2 * e], v[2 * e + 1], hi[e], lo[e]);
                const uint32_t pc0 = (cbase + 32 * h) / 2;   // packed column of this j range
                tmem_st16u(tl + COL_SH + pc0, hi);
                tmem_st16u(tl + COL_SL + pc0, lo);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= egl;
                tmem_st32(tl + COL_S + cbase + 32 * h, v);
            }
            tmem_wait_st();
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before_sync();
        __syncthreads();   // tiles built, raw stage consumed, S split and scaled, P^T copied
        if (warp == 7 && lane == 0 && c + 1 < nch) issue(c + 1, false);   // v, beta consumed
        if (tid == 0) {
            tc_fence_after_sync();
            // Oi^T [i x t] = (S hi + S lo) Q^T, S from tensor memory
#pragma unroll
            for (int ks = 0; ks < LD / 16; ++ks) {
                umma_bf16_ta(tmem + COL_OI, tmem + COL_SH + 8 * ks, dj(OFF_QB, ks), IDESC_T, ks > 0 ? 1u : 0u);
                umma_bf16_ta(tmem + COL_OI, tmem + COL_SL + 8 * ks, dj(OFF_QB, ks), IDESC_T, 1u);
            }
            // S [i x j] += (w Vb hi + w Vb lo)^T K
#pragma unroll
            for (int ks = 0; ks < LC / 16; ++ks) {
                umma_bf16(tmem + COL_S, dm(OFF_AW, ks), dm(OFF_KB, ks), IDESC_S, 1u);
                umma_bf16(tmem + COL_S, dm(OFF_AW + LD * LC * 2, ks), dm(OFF_KB, ks), IDESC_S, 1u);
            }
            umma_commit(bar_o);
        }
        // ---- the masked, decayed P as the hi/lo operand of the Oa product,
        // on warps 1-4 (token t = idx / 2, 32 source tokens each) ----
        if (warp >= 1 && warp <= 4) {
            const int idx = tid - 32, t = idx >> 1, sb = 32 * (idx & 1);
            const float gt = s_g[t];
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int s0 = sb + 8 * g8;
                const float4 pa = *reinterpret_cast<const float4*>(praw + t * PRAW_LD + s0);
                const float4 pb = *reinterpret_cast<const float4*>(praw + t * PRAW_LD + s0 + 4);
                const float4 ga = *reinterpret_cast<const float4*>(s_g + s0);
                const float4 gb = *reinterpret_cast<const float4*>(s_g + s0 + 4);
                const float pvv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
                const float gsv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int s_ = s0 + u;
                    x[u] = (s_ <= t && t < n && s_ < n) ? pvv[u] * ex2_approx((gt - gsv[u]) * LOG2E_L) : 0.f;
                }
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split_pair(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
                const int off = (t >> 3) * SBO_C + (s0 >> 3) * 128 + (t & 7) * 16;
                *reinterpret_cast<uint4*>(smem + OFF_P + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(smem + OFF_P + LC * LC * 2 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync 1, 128;" ::: "memory");   // P operand ready (warps 1-4)
            if (tid == 32) {
                // a second issuing thread, so that this product does not wait
                // behind thread 0's issue of the two products above
                tc_fence_after_sync();
                // Oa^T [i x t] = Vb hi P hi + Vb hi P lo + Vb lo P hi
#pragma unroll
                for (int ks = 0; ks < LC / 16; ++ks) {
                    umma_bf16(tmem + COL_OA, dm(OFF_VH, ks), dc(OFF_P, ks), IDESC_OA, ks > 0 ? 1u : 0u);
                    umma_bf16(tmem + COL_OA, dm(OFF_VH, ks), dc(OFF_P + LC * LC * 2, ks), IDESC_OA, 1u);
                    umma_bf16(tmem + COL_OA, dm(OFF_VH + LD * LC * 2, ks), dc(OFF_P, ks), IDESC_OA, 1u);
                }
                umma_commit(bar_o);
            }
        }
        if (warp == 7 && c + 1 < nch) exponents(c + 1);   // buffer (c+1)&1 is unused in chunk c
        if (!mbar_wait(bar_o, c & 1, p.wait_ns)) ok = false;
        tc_fence_after_sync();
        // ---- outputs: o_t[i] = (Oa + e^{g_t} Oi) / I_prior; the warps of a
        // lane quarter take 32 tokens each ----
        {
            const int tb32 = (warp >> 2) * 32;
            float oa[32], oi[32];
            tmem_ld32(tl + COL_OA + tb32, oa);
            tmem_ld32(tl + COL_OI + tb32, oi);
            const float rI = 1.f / p.Ip;
            float* dst = p.out + (bh * T + t0 + tb32) * LD + row;
#pragma unroll
            for (int t = 0; t < 32; ++t)
                if (tb32 + t < n) dst[static_cast<long long>(t) * LD] = (oa[t] + s_eg[tb32 + t] * oi[t]) * rI;
        }
        tc_fence_before_sync();
        __syncthreads();   // accumulators read; shared operands free; next exponents ready
    }

    // ---- end state mu_T = S / I_prior ----------------------------------------
    if (p.final_mu && part == static_cast<int>(gridDim.y) - 1) {
        tc_fence_after_sync();
        const float rI = 1.f / p.Ip;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[32];
            tmem_ld32(tl + COL_S + cbase + 32 * h, v);
            float* dst = p.final_mu + bh * S2 + static_cast<long long>(row) * LD + cbase + 32 * h;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(v[j] * rI, v[j + 1] * rI, v[j + 2] * rI, v[j + 3] * rI);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, LTMEM_COLS);
    if (!ok) record_error(&kdn::diag::g_diag_error, KDN_ERR_TIMEOUT);
}

}  // namespace
}  // namespace lintc
}  // namespace kdn
