// mobius_scan.cu -- parallel prefix scan of the Moebius precision recursion
//     lambda_t = (a_t lambda_{t-1} + b_t) / (c_t lambda_{t-1} + d_t)
// ("Kalman Linear Attention (KLA)", Metodologia 2, "Parallelizzazione tramite
// Trasformazioni di Moebius": the maps compose associatively, so the
// recursion admits an O(T)-work, O(log T)-depth prefix scan).
//
// Each step is the 2x2 matrix M_t = [[a_t, b_t], [c_t, d_t]]; applying M_1
// then M_2 is the product M_2 M_1, and lambda_t = P_t(lambda_0) with
// P_t = M_t ... M_1.  Because lambda only depends on the ratio of the
// homogeneous coordinates, every composed matrix is rescaled by an exact
// power of two (its largest entry into [1, 2)), which removes overflow and
// underflow without rounding.
//
// Two kernels:
//  * mobius_scan_kernel (few sequences, or rows that are not 16-byte
//    aligned): one CTA per tile of 2048 consecutive steps of a sequence.
//    1. each thread loads 8 consecutive steps and composes them in order;
//    2. a warp-shuffle inclusive scan composes the 32 per-thread matrices;
//    3. warp totals meet in shared memory for the block-level carry;
//    4. tiles of the same sequence are chained with a decoupled look-back: a
//       tile publishes its aggregate matrix as soon as it is known, then walks
//       back over predecessors (composing aggregates) until it finds a
//       published inclusive value lambda, and publishes its own inclusive
//       lambda.  Tiles are numbered by an atomic ticket so that every tile's
//       predecessors were scheduled before it; every wait on a flag is
//       bounded by GPU time and records KDN_ERR_TIMEOUT instead of hanging;
//    5. each thread evaluates its 8 outputs sequentially from the lambda at
//       its first step (the exclusive prefix applied to the tile's carry).
//  * mobius_seq_kernel (at least as many sequences as resident CTAs): a
//    persistent CTA owns whole sequences and streams their tiles (described
//    at the kernel).
// Memory traffic is the algorithmic minimum (16 B in, 4 B out per step); the
// kernels are bound by HBM bandwidth once the sequences fill the GPU.
#include <cstdint>
#include <cuda_runtime.h>

#include <mutex>

#include "kdn_device.cuh"
#include "kdn_internal.h"
#include "mobius_device.cuh"

namespace kdn {
namespace {

constexpr int MB_THREADS = 256;
constexpr int MB_VPT = 8;                       // steps per thread
constexpr int MB_TILE = MB_THREADS * MB_VPT;    // steps per CTA
constexpr int MB_WARPS = MB_THREADS / 32;

constexpr unsigned int FLAG_AGG = 1u;           // aggregate matrix published
constexpr unsigned int FLAG_PRE = 2u;           // inclusive lambda published

__device__ int g_mobius_error = 0;

using mob::apply;
using mob::identity;
using mob::Mat;
using mob::mul;
using mob::normalize;
using mob::shfl_up;

struct LookbackScratch {
    unsigned long long* ticket;   // tile ticket counter (zeroed per launch)
    unsigned int* flags;          // [num_tiles], zeroed per launch
    float4* agg;                  // [num_tiles] aggregate matrix (a, b, c, d)
    float* pre;                   // [num_tiles] inclusive lambda at the tile end
};

// Bounded wait for a tile flag; returns 0 on timeout.
__device__ __forceinline__ unsigned int wait_flag(const unsigned int* f, long long limit_ns) {
    unsigned int v = ld_acquire_u32(f);
    if (v) return v;
    const unsigned long long t0 = globaltimer_ns();
    unsigned int sleep = 32;
    while (true) {
        __nanosleep(sleep);
        if (sleep < 1024) sleep <<= 1;
        v = ld_acquire_u32(f);
        if (v) return v;
        if (static_cast<long long>(globaltimer_ns() - t0) > limit_ns) return 0;
    }
}

template <bool VEC, bool LOOKBACK>
__global__ void __launch_bounds__(MB_THREADS)
mobius_scan_kernel(const float* __restrict__ A, const float* __restrict__ B,
                   const float* __restrict__ C, const float* __restrict__ D,
                   const float* __restrict__ lambda0, float* __restrict__ out,
                   long long T, long long tiles_per_seq, LookbackScratch sc,
                   long long wait_ns, long long stall_tile) {
    __shared__ long long s_tile;
    __shared__ Mat s_warp[MB_WARPS];
    __shared__ float s_lam;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    long long tile;
    if (LOOKBACK) {
        if (tid == 0) s_tile = static_cast<long long>(atomicAdd(sc.ticket, 1ull));
        __syncthreads();
        tile = s_tile;
    } else {
        tile = blockIdx.x;
    }
    const long long seq = tile / tiles_per_seq;
    const long long part = tile - seq * tiles_per_seq;
    const long long t_first = part * MB_TILE + static_cast<long long>(tid) * MB_VPT;
    const long long base = seq * T;

    // ---- 1. load 8 steps and compose them in order ----------------------
    float ca[MB_VPT], cb[MB_VPT], cc[MB_VPT], cd[MB_VPT];
    if (VEC && t_first + MB_VPT <= T) {
        const float4* pa = reinterpret_cast<const float4*>(A + base + t_first);
        const float4* pb = reinterpret_cast<const float4*>(B + base + t_first);
        const float4* pc = reinterpret_cast<const float4*>(C + base + t_first);
        const float4* pd = reinterpret_cast<const float4*>(D + base + t_first);
#pragma unroll
        for (int h = 0; h < MB_VPT / 4; ++h) {
            const float4 x = __ldcs(pa + h), y = __ldcs(pb + h), z = __ldcs(pc + h),
                         w = __ldcs(pd + h);
            ca[4 * h + 0] = x.x; ca[4 * h + 1] = x.y; ca[4 * h + 2] = x.z; ca[4 * h + 3] = x.w;
            cb[4 * h + 0] = y.x; cb[4 * h + 1] = y.y; cb[4 * h + 2] = y.z; cb[4 * h + 3] = y.w;
            cc[4 * h + 0] = z.x; cc[4 * h + 1] = z.y; cc[4 * h + 2] = z.z; cc[4 * h + 3] = z.w;
            cd[4 * h + 0] = w.x; cd[4 * h + 1] = w.y; cd[4 * h + 2] = w.z; cd[4 * h + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int s = 0; s < MB_VPT; ++s) {
            const long long t = t_first + s;
            const bool in = t < T;
            ca[s] = in ? __ldcs(A + base + t) : 1.f;
            cb[s] = in ? __ldcs(B + base + t) : 0.f;
            cc[s] = in ? __ldcs(C + base + t) : 0.f;
            cd[s] = in ? __ldcs(D + base + t) : 1.f;
        }
    }
    Mat P = {ca[0], cb[0], cc[0], cd[0]};
#pragma unroll
    for (int s = 1; s < MB_VPT; ++s) P = normalize(mul(Mat{ca[s], cb[s], cc[s], cd[s]}, P));
    P = normalize(P);

    // ---- 2. warp inclusive scan (later steps on the left) ---------------
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const Mat Q = shfl_up(P, off);
        if (lane >= off) P = normalize(mul(P, Q));
    }
    Mat lane_excl = shfl_up(P, 1);
    if (lane == 0) lane_excl = identity();
    if (lane == 31) s_warp[warp] = P;
    __syncthreads();

    // ---- 3. block carry: exclusive prefix of the earlier warps -----------
    Mat warp_excl = identity();
    for (int w = 0; w < warp; ++w) warp_excl = normalize(mul(s_warp[w], warp_excl));
    const Mat thread_excl = normalize(mul(lane_excl, warp_excl));

    // ---- 4. look-back across the tiles of this sequence ------------------
    if (tid == 0) {
        Mat agg = identity();
        for (int w = 0; w < MB_WARPS; ++w) agg = normalize(mul(s_warp[w], agg));
        const bool stalled = LOOKBACK && tile == stall_tile;   // fault injection
        float lam;
        if (!LOOKBACK || part == 0) {
            lam = lambda0[seq];
        } else {
            if (!stalled) {
                sc.agg[tile] = make_float4(agg.a, agg.b, agg.c, agg.d);
                __threadfence();
                st_release_u32(sc.flags + tile, FLAG_AGG);
            }
            Mat acc = identity();
            long long j = tile - 1;
            while (true) {
                const unsigned int f = wait_flag(sc.flags + j, wait_ns);
                if (f == 0) {                      // predecessor never published
                    record_error(&g_mobius_error, KDN_ERR_TIMEOUT);
                    lam = apply(acc, lambda0[seq]);
                    break;
                }
                if (f == FLAG_PRE) {
                    lam = apply(acc, __ldcg(sc.pre + j));
                    break;
                }
                const float4 g = __ldcg(sc.agg + j);
                acc = normalize(mul(acc, Mat{g.x, g.y, g.z, g.w}));
                --j;
            }
        }
        if (LOOKBACK && !stalled) {
            sc.pre[tile] = apply(agg, lam);
            __threadfence();
            st_release_u32(sc.flags + tile, FLAG_PRE);
        }
        s_lam = lam;
    }
    __syncthreads();

    // ---- 5. outputs: sequential recursion from this thread's start ------
    float lam = apply(thread_excl, s_lam);
    float res[MB_VPT];
#pragma unroll
    for (int s = 0; s < MB_VPT; ++s) {
        lam = fmaf(ca[s], lam, cb[s]) / fmaf(cc[s], lam, cd[s]);
        res[s] = lam;
    }
    if (VEC && t_first + MB_VPT <= T) {
        float4* po = reinterpret_cast<float4*>(out + base + t_first);
#pragma unroll
        for (int h = 0; h < MB_VPT / 4; ++h)
            __stcs(po + h, make_float4(res[4 * h], res[4 * h + 1], res[4 * h + 2], res[4 * h + 3]));
    } else {
#pragma unroll
        for (int s = 0; s < MB_VPT; ++s)
            if (t_first + s < T) __stcs(out + base + t_first + s, res[s]);
    }
}

// ---------------------------------------------------------------------------
// Sequence-per-CTA kernel for 16-byte aligned rows (T % 4 == 0), chosen by
// mobius_choose_seq (many sequences, or short ones).  A persistent grid of at
// most SQ_CTAS_PER_SM CTAs per SM gives CTA b the sequences b, b + G, b + 2G,
// ... (G = grid size) and walks their tiles in order (mob::mobius_walk), so no
// cross-CTA look-back (and no scratch) is needed.
constexpr int SQ_THREADS = 256;
constexpr int SQ_CTAS_PER_SM = 3;
static_assert(mob::Walk<SQ_THREADS>::TILE == MB_TILE, "both kernels count tiles of the same length");

__host__ __device__ constexpr int sq_smem_bytes() { return mob::Walk<SQ_THREADS>::SMEM; }

__global__ void __launch_bounds__(SQ_THREADS, SQ_CTAS_PER_SM)
mobius_seq_kernel(const float* __restrict__ A, const float* __restrict__ B,
                  const float* __restrict__ C, const float* __restrict__ D,
                  const float* __restrict__ lambda0, float* __restrict__ out, long long N,
                  long long T, int tiles_per_seq, long long wait_ns) {
    extern __shared__ __align__(128) unsigned char smem[];
    mob::mobius_walk<SQ_THREADS>(A, B, C, D, lambda0, out, N, T, tiles_per_seq, blockIdx.x, gridDim.x,
                                 wait_ns, smem, &g_mobius_error);
}

template <bool VEC, bool LB>
cudaError_t launch(const float* a, const float* b, const float* c, const float* d,
                   const float* lam0, float* out, long long T, long long tps, long long tiles,
                   LookbackScratch sc, cudaStream_t st, long long wait_ns, long long stall) {
    mobius_scan_kernel<VEC, LB><<<static_cast<unsigned>(tiles), MB_THREADS, 0, st>>>(
        a, b, c, d, lam0, out, T, tps, sc, wait_ns, stall);
    return cudaGetLastError();
}

}  // namespace

// Resident CTA slots of the sequence-per-CTA kernel on the current device
// (SMs x CTAs per SM); -1 on a CUDA error.
int mobius_seq_slots() {
    static int occ_cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    if (occ_cache[dev] == 0) {
        const int smem = sq_smem_bytes();
        if (cudaFuncSetAttribute(mobius_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return -1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mobius_seq_kernel, SQ_THREADS, smem) !=
            cudaSuccess)
            return -1;
        occ_cache[dev] = n > 0 ? n : 1;
    }
    return sm_count() * occ_cache[dev];
}

// Whether a scan of N sequences x tps tiles runs on the sequence-per-CTA
// kernel (needs 16-byte aligned rows).  It takes no scratch and no look-back,
// but each CTA walks its tiles one after another.  It is chosen when every
// resident CTA has sequences to stream; for fewer sequences the two kernels'
// costs are compared with a model fitted to GB300 timings (microseconds): the
// walk costs about 3.5 + 1.6 tps; the look-back kernel about 9 + 0.0224 per
// tile of the grid + 0.31 per look-back hop, and never less than 19 when it
// allocates its scratch (allocation, flag clearing and release on the
// stream) or 9 when the scratch is the library's fixed array (flag clearing
// and the launch: kdn_mobius_scan_noalloc, measured 9.0 us for 1 x 4096 and
// 11.5 us for 1 x 16384 steps against 16.7 us for the walk).  Single-tile
// sequences need no look-back and stay on the tile kernel.
bool mobius_choose_seq(long long N, long long tps, bool vec, int slots, bool fixed_scratch = false) {
    if (!vec || slots <= 0 || tps < 2) return false;
    if (N >= slots) return true;
    const double n = static_cast<double>(N), t = static_cast<double>(tps);
    const double walk = 3.5 + 1.6 * t;
    const double lookback = fmax(fixed_scratch ? 9.0 : 19.0, 9.0 + 0.0224 * n * t + 0.31 * t);
    return walk <= lookback;
}

void mobius_plan(long long N, long long T, int* kernels, size_t* scratch) {
    const long long tps = (T + MB_TILE - 1) / MB_TILE;
    const long long tiles = N * tps;
    *kernels = (N > 0 && T > 0) ? 1 : 0;
    *scratch = 0;
    const int slots = (T % 4 == 0) ? mobius_seq_slots() : -1;
    if (tps > 1 && !mobius_choose_seq(N, tps, T % 4 == 0, slots)) {
        const size_t zero_bytes = (8 + 4 * static_cast<size_t>(tiles) + 15) & ~size_t(15);
        *scratch = zero_bytes + 16 * static_cast<size_t>(tiles) + 4 * tiles;
    }
}

kdn_status mobius_launch(const float* a, const float* b, const float* c, const float* d,
                         const float* lambda0, float* out, long long N, long long T,
                         cudaStream_t stream, long long wait_ns, long long stall_tile) {
    if (N == 0 || T == 0) return KDN_OK;
    const long long tps = (T + MB_TILE - 1) / MB_TILE;
    const long long tiles = N * tps;
    if (tiles > 0x7fffffffLL) return KDN_ERR_INVALID_ARG;
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool vec = (T % 4 == 0) && aligned16(a) && aligned16(b) && aligned16(c) &&
                     aligned16(d) && aligned16(out);
    LookbackScratch sc{nullptr, nullptr, nullptr, nullptr};
    void* scratch = nullptr;
    cudaError_t e;
    const bool lookback = tps > 1;
    const int slots = vec ? mobius_seq_slots() : 0;
    if (slots < 0) return KDN_ERR_CUDA;
    const bool use_seq = mobius_choose_seq(N, tps, vec, slots);
    if (lookback && !use_seq) {
        // [ticket u64][flags u32 x tiles] (zeroed) | [agg float4 x tiles][pre f32 x tiles]
        const size_t zero_bytes = (8 + 4 * static_cast<size_t>(tiles) + 15) & ~size_t(15);
        const size_t bytes = zero_bytes + 16 * static_cast<size_t>(tiles) + 4 * tiles;
        e = cudaMallocAsync(&scratch, bytes, stream);
        if (e != cudaSuccess) return from_cuda(e);
        char* p = static_cast<char*>(scratch);
        sc.ticket = reinterpret_cast<unsigned long long*>(p);
        sc.flags = reinterpret_cast<unsigned int*>(p + 8);
        sc.agg = reinterpret_cast<float4*>(p + zero_bytes);
        sc.pre = reinterpret_cast<float*>(p + zero_bytes + 16 * tiles);
        e = cudaMemsetAsync(scratch, 0, zero_bytes, stream);
        if (e != cudaSuccess) {
            cudaFreeAsync(scratch, stream);
            return from_cuda(e);
        }
    }
    if (use_seq) {
        // many sequences: one persistent CTA per resident slot, each owning whole sequences
        // one persistent CTA per resident slot (at most one per sequence)
        mobius_seq_kernel<<<static_cast<unsigned>(min(static_cast<long long>(slots), N)), SQ_THREADS,
                            sq_smem_bytes(), stream>>>(a, b, c, d, lambda0, out, N, T,
                                                       static_cast<int>(tps), wait_ns);
        e = cudaGetLastError();
    } else if (lookback) {
        e = vec ? launch<true, true>(a, b, c, d, lambda0, out, T, tps, tiles, sc, stream, wait_ns, stall_tile)
                : launch<false, true>(a, b, c, d, lambda0, out, T, tps, tiles, sc, stream, wait_ns, stall_tile);
    } else {
        e = vec ? launch<true, false>(a, b, c, d, lambda0, out, T, tps, tiles, sc, stream, wait_ns, -1)
                : launch<false, false>(a, b, c, d, lambda0, out, T, tps, tiles, sc, stream, wait_ns, -1);
    }
    if (scratch) {
        const cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e == cudaSuccess) e = ef;
    }
    return from_cuda(e);
}

cudaError_t mobius_take_device_error(int* status) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_mobius_error, sizeof(int));
    if (e != cudaSuccess) return e;
    if (v != 0) e = cudaMemcpyToSymbol(g_mobius_error, &zero, sizeof(int));
    *status = v;
    return e;
}

}  // namespace kdn

// ---------------------------------------------------------------------------
// Allocation-free variant (kdn_mobius_scan_noalloc).
//
// Some callers must not allocate device memory during a call: for example a
// process whose framework reserved the GPU's memory up front, so that the
// default memory pool has nothing left to give, or a latency-critical loop in
// which allocator calls are not allowed.  For them the look-back scratch of a
// multi-tile scan lives in the fixed array below, part of the library's
// device image: every GPU that loads the library holds these 1 MiB until the
// process exits.  Host code cannot use the array's name as a device address,
// so set-up fetches the address once per device with cudaGetSymbolAddress.
namespace kdn {

static __device__ __align__(256) unsigned char g_kdn_noalloc_scratch[1u << 20];

namespace {
constexpr size_t kNoAllocBytes = sizeof(g_kdn_noalloc_scratch);
std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of the array on the current device (set-up on first use).
cudaError_t noalloc_base(void** base) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_kdn_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_addr[dev] = p;
    }
    *base = g_noalloc_addr[dev];
    return cudaSuccess;
}
}  // namespace

long long mobius_noalloc_max_tiles() {
    // largest t with round16(8 + 4 t) + 20 t <= kNoAllocBytes
    long long t = static_cast<long long>(kNoAllocBytes) / 24;
    while (t > 0 && (((8 + 4 * static_cast<size_t>(t) + 15) & ~size_t(15)) + 20 * static_cast<size_t>(t)) > kNoAllocBytes) --t;
    return t;
}

kdn_status mobius_launch_noalloc(const float* a, const float* b, const float* c, const float* d,
                                 const float* lambda0, float* out, long long N, long long T,
                                 cudaStream_t stream, long long wait_ns) {
    if (N == 0 || T == 0) return KDN_OK;
    const long long tps = (T + MB_TILE - 1) / MB_TILE;
    const long long tiles = N * tps;
    if (tiles > 0x7fffffffLL) return KDN_ERR_INVALID_ARG;
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool vec = (T % 4 == 0) && aligned16(a) && aligned16(b) && aligned16(c) &&
                     aligned16(d) && aligned16(out);
    LookbackScratch sc{nullptr, nullptr, nullptr, nullptr};
    cudaError_t e;
    const int slots = vec ? mobius_seq_slots() : 0;
    if (slots < 0) return KDN_ERR_CUDA;
    // the walk takes no scratch: it also serves aligned calls whose look-back
    // would need more tiles than the fixed array holds
    if (mobius_choose_seq(N, tps, vec, slots, true) ||
        (vec && slots > 0 && tps > 1 && tiles > mobius_noalloc_max_tiles())) {   // no scratch at all
        mobius_seq_kernel<<<static_cast<unsigned>(min(static_cast<long long>(slots), N)), SQ_THREADS,
                            sq_smem_bytes(), stream>>>(a, b, c, d, lambda0, out, N, T,
                                                       static_cast<int>(tps), wait_ns);
        return from_cuda(cudaGetLastError());
    }
    if (tps > 1) {
        if (tiles > mobius_noalloc_max_tiles()) return KDN_ERR_INVALID_ARG;
        void* base = nullptr;
        e = noalloc_base(&base);
        if (e != cudaSuccess) return from_cuda(e);
        const size_t zero_bytes = (8 + 4 * static_cast<size_t>(tiles) + 15) & ~size_t(15);
        char* p = static_cast<char*>(base);
        sc.ticket = reinterpret_cast<unsigned long long*>(p);
        sc.flags = reinterpret_cast<unsigned int*>(p + 8);
        sc.agg = reinterpret_cast<float4*>(p + zero_bytes);
        sc.pre = reinterpret_cast<float*>(p + zero_bytes + 16 * tiles);
        // the array keeps the previous call's contents: clear ticket and flags
        e = cudaMemsetAsync(base, 0, zero_bytes, stream);
        if (e != cudaSuccess) return from_cuda(e);
        e = vec ? launch<true, true>(a, b, c, d, lambda0, out, T, tps, tiles, sc, stream, wait_ns, -1)
                : launch<false, true>(a, b, c, d, lambda0, out, T, tps, tiles, sc, stream, wait_ns, -1);
    } else {
        e = vec ? launch<true, false>(a, b, c, d, lambda0, out, T, tps, tiles, sc, stream, wait_ns, -1)
                : launch<false, false>(a, b, c, d, lambda0, out, T, tps, tiles, sc, stream, wait_ns, -1);
    }
    return from_cuda(e);
}

}  // namespace kdn
