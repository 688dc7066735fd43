// mobius_device.cuh -- device building blocks of the Moebius precision scan
//     lambda_t = (a_t lambda_{t-1} + b_t) / (c_t lambda_{t-1} + d_t)
// ("Kalman Linear Attention (KLA)", Metodologia 2, "Parallelizzazione tramite
// Trasformazioni di Moebius"), shared by the Moebius kernels and the
// diagonal-scan kernel that runs the per-head lambda in its own launch.
//
// Step t is the 2x2 matrix M_t = [[a_t, b_t], [c_t, d_t]]; applying M_1 then
// M_2 is the product M_2 M_1, and lambda_t = P_t(lambda_0) with P_t = M_t ...
// M_1.  lambda depends only on the ratio of the homogeneous coordinates, so
// every composed matrix is rescaled by an exact power of two (its largest
// entry into [1, 2)): no overflow or underflow, no rounding.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "kdn_device.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace mob {

struct Mat {
    float a, b, c, d;  // [[a, b], [c, d]]
};

__device__ __forceinline__ Mat identity() { return {1.f, 0.f, 0.f, 1.f}; }

// L * R (apply R first, then L)
__device__ __forceinline__ Mat mul(const Mat& L, const Mat& R) {
    Mat o;
    o.a = fmaf(L.a, R.a, L.b * R.c);
    o.b = fmaf(L.a, R.b, L.b * R.d);
    o.c = fmaf(L.c, R.a, L.d * R.c);
    o.d = fmaf(L.c, R.b, L.d * R.d);
    return o;
}

// Scale by an exact power of two so that the largest |entry| lies in [1, 2):
// the factor is built from the exponent field of the largest magnitude.  A
// zero matrix stays zero; a largest entry at or above 2^126 is brought into
// [1, 4) (the factor stays a normal number); infinities stay infinite and
// NaN propagates through the products.
__device__ __forceinline__ Mat normalize(const Mat& m) {
    const float mx = fmaxf(fmaxf(fabsf(m.a), fabsf(m.b)), fmaxf(fabsf(m.c), fabsf(m.d)));
    const uint32_t e = min(__float_as_uint(mx) & 0x7f800000u, 0x7e800000u);   // biased exponent E <= 253
    const float s = __uint_as_float(0x7f000000u - e);                           // 2^(127 - E)
    return {m.a * s, m.b * s, m.c * s, m.d * s};
}

__device__ __forceinline__ float apply(const Mat& m, float lam) {
    return fmaf(m.a, lam, m.b) / fmaf(m.c, lam, m.d);
}

__device__ __forceinline__ Mat shfl_up(const Mat& m, int off) {
    return {__shfl_up_sync(0xffffffffu, m.a, off), __shfl_up_sync(0xffffffffu, m.b, off),
            __shfl_up_sync(0xffffffffu, m.c, off), __shfl_up_sync(0xffffffffu, m.d, off)};
}

// Sequence walk with NT threads (a multiple of 32): tiles of NT * 8 steps.
constexpr int WALK_VPT = 8;          // steps per thread
constexpr int WALK_STAGES = 2;
template <int NT>
struct Walk {
    static constexpr int WARPS = NT / 32;
    static constexpr int TILE = NT * WALK_VPT;
    static constexpr int STAGE_FLOATS = 4 * TILE;
    // dynamic shared memory: the coefficient stages, then their mbarriers
    static constexpr int SMEM = WALK_STAGES * STAGE_FLOATS * 4 + WALK_STAGES * 8;
};

// One walker of G: walker `w` owns the sequences w, w + G, w + 2G, ... of
// [N, T] (rows 16-byte aligned, T % 4 == 0) and walks their tiles in order:
//   * the coefficients of the next tile of its stream are in flight as 1-D
//     bulk copies (one per coefficient array, completing on an mbarrier)
//     while the current tile is scanned;
//   * each thread owns 8 consecutive steps: it composes them as a balanced
//     tree; a warp-shuffle scan and the warp totals give its exclusive
//     prefix, and it evaluates its 8 outputs sequentially from the lambda at
//     its first step;
//   * lambda at the start of the next tile is the last output of this one,
//     so consecutive tiles continue exactly from the value that was written.
// Two barriers per tile; the per-tile shared words (warp totals, carried
// lambda) are double-buffered by tile parity.  A bounded wait that runs out
// records KDN_ERR_TIMEOUT in *err, stops the walk, and waits (bounded) for the
// copies still in flight before returning.  Every thread of the CTA calls it.
template <int NT>
__device__ __forceinline__ void mobius_walk(const float* __restrict__ A, const float* __restrict__ B,
                                            const float* __restrict__ C, const float* __restrict__ D,
                                            const float* __restrict__ lambda0, float* __restrict__ out,
                                            long long N, long long T, int tiles_per_seq, long long w,
                                            long long G, long long wait_ns, unsigned char* smem,
                                            int* err) {
    using WK = Walk<NT>;
    constexpr int TILE = WK::TILE, SF = WK::STAGE_FLOATS, WARPS = WK::WARPS;
    float* buf = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + WALK_STAGES * SF * 4);
    __shared__ Mat s_warp[2][WARPS];
    __shared__ float s_lam[2];
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long nseq = w < N ? (N - 1 - w) / G + 1 : 0;
    const long long ntiles = nseq * tiles_per_seq;

    // producer state (thread 0): next stream tile to issue
    long long iss_i = 0, iss_seq = w;
    int iss_part = 0, iss_st = 0;
    auto issue_next = [&]() {
        const long long t0 = static_cast<long long>(iss_part) * TILE;
        const long long n = min(static_cast<long long>(TILE), T - t0);
        const uint32_t bytes = static_cast<uint32_t>(n * 4);
        const long long off = iss_seq * T + t0;
        float* dst = buf + iss_st * SF;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&full[iss_st], 4 * bytes);
        bulk_g2s(dst, A + off, bytes, &full[iss_st]);
        bulk_g2s(dst + TILE, B + off, bytes, &full[iss_st]);
        bulk_g2s(dst + 2 * TILE, C + off, bytes, &full[iss_st]);
        bulk_g2s(dst + 3 * TILE, D + off, bytes, &full[iss_st]);
        ++iss_i;
        if (++iss_part == tiles_per_seq) { iss_part = 0; iss_seq += G; }
        if (++iss_st == WALK_STAGES) iss_st = 0;
    };

    if (tid == 0) {
        for (int st = 0; st < WALK_STAGES; ++st) mbar_init(&full[st], 1);
        mbar_init_fence();
        while (iss_i < WALK_STAGES && iss_i < ntiles) issue_next();
        s_abort = 0;
    }
    __syncthreads();

    long long seq = w;
    int part = 0, st = 0;
    uint32_t phase = 0;
    long long i = 0;
    for (; i < ntiles; ++i) {
        const int par = static_cast<int>(i & 1);
        if (!mbar_wait(&full[st], phase, wait_ns)) {
            record_error(err, KDN_ERR_TIMEOUT);
            s_abort = 1;
        }
        const long long t_first = static_cast<long long>(part) * TILE + tid * WALK_VPT;
        const int nvalid = static_cast<int>(max(0LL, min(static_cast<long long>(WALK_VPT), T - t_first)));

        // ---- 1. this thread's 8 steps from shared memory -----------------
        Mat m[WALK_VPT];
        {
            const float* sb = buf + st * SF + tid * WALK_VPT;
#pragma unroll
            for (int h = 0; h < WALK_VPT / 4; ++h) {
                const float4 x = *reinterpret_cast<const float4*>(sb + 4 * h);
                const float4 y = *reinterpret_cast<const float4*>(sb + TILE + 4 * h);
                const float4 z = *reinterpret_cast<const float4*>(sb + 2 * TILE + 4 * h);
                const float4 u = *reinterpret_cast<const float4*>(sb + 3 * TILE + 4 * h);
                m[4 * h + 0] = {x.x, y.x, z.x, u.x};
                m[4 * h + 1] = {x.y, y.y, z.y, u.y};
                m[4 * h + 2] = {x.z, y.z, z.z, u.z};
                m[4 * h + 3] = {x.w, y.w, z.w, u.w};
            }
#pragma unroll
            for (int s2 = 0; s2 < WALK_VPT; ++s2)
                if (s2 >= nvalid) m[s2] = identity();   // past the end of the sequence
        }
        __syncthreads();   // stage consumed: refill it with the next stream tile
        // s_abort is only set during the waits above (before this barrier) or
        // in the next tile's waits (after the barrier below): all threads read
        // the same value here
        if (s_abort) break;
        if (tid == 0 && iss_i < ntiles) issue_next();
        // lambda at the start of the tile: lambda_0 for the first tile of a
        // sequence, else the last output of the previous tile (written after
        // the previous tile's second barrier)
        const float lam_start = part == 0 ? __ldg(lambda0 + seq) : s_lam[par];

        // ---- 2. compose (balanced tree, later steps on the left) and scan --
        Mat tree[WALK_VPT];
#pragma unroll
        for (int k = 0; k < WALK_VPT; ++k) tree[k] = m[k];
#pragma unroll
        for (int wd = WALK_VPT; wd > 1; wd /= 2)
#pragma unroll
            for (int k = 0; k < wd / 2; ++k) tree[k] = normalize(mul(tree[2 * k + 1], tree[2 * k]));
        Mat P = tree[0];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const Mat Q = shfl_up(P, off);
            if (lane >= off) P = normalize(mul(P, Q));
        }
        Mat lane_excl = shfl_up(P, 1);
        if (lane == 0) lane_excl = identity();
        if (lane == 31) s_warp[par][warp] = P;
        __syncthreads();
        Mat warp_excl = identity();
        for (int wp = 0; wp < warp; ++wp) warp_excl = normalize(mul(s_warp[par][wp], warp_excl));
        const Mat thread_excl = normalize(mul(lane_excl, warp_excl));

        // ---- 3. outputs ------------------------------------------------------
        float lam = apply(thread_excl, lam_start);
        float res[WALK_VPT];
#pragma unroll
        for (int s2 = 0; s2 < WALK_VPT; ++s2) {
            lam = __fdividef(fmaf(m[s2].a, lam, m[s2].b), fmaf(m[s2].c, lam, m[s2].d));
            res[s2] = lam;
        }
        if (tid == NT - 1) s_lam[par ^ 1] = lam;   // carry (unused after a sequence's last tile)
        float* po = out + seq * T + t_first;
        if (nvalid == WALK_VPT) {
#pragma unroll
            for (int h = 0; h < WALK_VPT / 4; ++h)
                __stcs(reinterpret_cast<float4*>(po) + h,
                       make_float4(res[4 * h], res[4 * h + 1], res[4 * h + 2], res[4 * h + 3]));
        } else {
#pragma unroll
            for (int s2 = 0; s2 < WALK_VPT; ++s2)
                if (s2 < nvalid) __stcs(po + s2, res[s2]);
        }
        if (++part == tiles_per_seq) { part = 0; seq += G; }
        if (++st == WALK_STAGES) { st = 0; phase ^= 1u; }
    }
    // after an abort, wait (bounded) for the copies still in flight into this CTA
    if (s_abort && tid == 0) {
        for (long long k = i; k < iss_i; ++k)
            mbar_wait(&full[k % WALK_STAGES], static_cast<uint32_t>((k / WALK_STAGES) & 1), wait_ns);
    }
}

}  // namespace mob
}  // namespace kdn
