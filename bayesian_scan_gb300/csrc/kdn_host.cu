// kdn_host.cu -- entry points that take every tensor in host memory
// (kdn_diag_scan_fwd_host, kdn_mobius_scan_host).
//
// The work is cut into chunks that are pipelined over six streams: the
// caller's stream runs the kernels, four internal streams copy later chunks'
// inputs in while chunk c is scanned, another copies chunk c-1's outputs
// out (or the scan writes them straight into page-locked host memory).  The
// diagonal scan is cut into groups of whole batches when it has four or
// more (independent, contiguous in host memory; see diag_host_batches),
// else along the tokens (every head of a chunk runs in one launch, so the
// GPU stays full), carrying the state from one chunk to the next on the
// device through the scan's own final-state / initial-state interface; the
// Moebius scan is cut along the sequences, which are independent.  Host buffers should be page-locked for the copies
// to run asynchronously; pageable memory works, with the copies serialised.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kdn.h"
#include "kdn_internal.h"

namespace kdn {
namespace {

constexpr int kMaxDev = 64;

// Streams for the copies in (one stream runs back-to-back pitched
// host-to-device copies at about 130 GB/s on GB300, several reach the link's
// ~200 GB/s), one per input array of a chunk, and one for the copies out.
constexpr int kIn = 4;
struct CopyStreams {
    cudaStream_t in[kIn] = {};
    cudaStream_t out = nullptr;
};
CopyStreams g_streams[kMaxDev];
std::mutex g_streams_mu;

// The two copy streams of the current device (created once per device).
cudaError_t copy_streams(CopyStreams* cs) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_streams_mu);
    CopyStreams& s = g_streams[dev];
    if (!s.out) {
        CopyStreams n;
        cudaStream_t* all[] = {&n.in[0], &n.in[1], &n.in[2], &n.in[3], &n.out};
        for (cudaStream_t* p : all) {
            e = cudaStreamCreateWithFlags(p, cudaStreamNonBlocking);
            if (e != cudaSuccess) {
                for (cudaStream_t* q : all)
                    if (*q) cudaStreamDestroy(*q);
                return e;
            }
        }
        s = n;
    }
    *cs = s;
    return cudaSuccess;
}

// The host-buffer calls' device scratch comes from a memory pool of the
// library's own (one per device, created on first use) that keeps freed
// memory instead of releasing it to CUDA at every synchronisation: a
// call then reuses the previous call's buffers.  The pool holds at most the
// largest scratch one call needed.
cudaMemPool_t g_pools[kMaxDev] = {};

cudaError_t host_pool(cudaMemPool_t* pool) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_streams_mu);
    if (!g_pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        e = cudaMemPoolCreate(&p, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = ~0ull;
        e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return e;
        }
        g_pools[dev] = p;
    }
    *pool = g_pools[dev];
    return cudaSuccess;
}

// Chunk buffers in flight: with three, the copies of chunk c+2 run while
// chunk c is scanned and neither the copy streams nor the scan wait on each
// other in steady state (two leave both idle part of the time).
constexpr int kBufs = 3;

// Events of the chunk buffers (copies in on either copy stream, scan, copies
// out) and of the start, released on scope exit.
struct ChunkEvents {
    cudaEvent_t in[kBufs][kIn] = {}, comp[kBufs] = {}, out[kBufs] = {}, start = nullptr;
    cudaError_t create() {
        cudaError_t e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
        for (int b = 0; b < kBufs && e == cudaSuccess; ++b) {
            cudaEvent_t* all[] = {&in[b][0], &in[b][1], &in[b][2], &in[b][3], &comp[b], &out[b]};
            for (cudaEvent_t* ev : all)
                if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        }
        return e;
    }
    ~ChunkEvents() {
        if (start) cudaEventDestroy(start);
        for (int b = 0; b < kBufs; ++b) {
            cudaEvent_t all[] = {in[b][0], in[b][1], in[b][2], in[b][3], comp[b], out[b]};
            for (cudaEvent_t ev : all)
                if (ev) cudaEventDestroy(ev);
        }
    }
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Chunks of a host-buffer call (token ranges of a diagonal scan, groups of
// Moebius sequences).  The first chunk's copies run before any scan and the
// last chunk's scan after every copy, which favours more chunks, but every
// chunk's scan has its fixed costs: on the 65536-token context with its
// Moebius scan, 8 chunks gave 8.2e7 tokens/s end to end, 16 and 24 less
// (6.7e7 to 8.1e7, varying from run to run).
constexpr int kHostChunks = 8;

// Tokens per chunk of a host-buffer diagonal scan: about kHostChunks chunks,
// at least 512 tokens, a multiple of 16.
int diag_chunk_tokens(int T) {
    int tc = (T + kHostChunks - 1) / kHostChunks;
    tc = (tc + 15) / 16 * 16;
    if (tc < 512) tc = 512;
    return tc < T ? tc : T;
}

// Propagates the first error; keeps going so that every queued operation
// stays ordered before the final free and synchronisation.
struct Status {
    cudaError_t e = cudaSuccess;
    kdn_status k = KDN_OK;
    void cuda(cudaError_t x) {
        if (e == cudaSuccess && k == KDN_OK && x != cudaSuccess) e = x;
    }
    void kdn(kdn_status x) {
        if (e == cudaSuccess && k == KDN_OK && x != KDN_OK) k = x;
    }
    bool ok() const { return e == cudaSuccess && k == KDN_OK; }
    kdn_status result() const { return k != KDN_OK ? k : from_cuda(e); }
};

}  // namespace

// Batches: with four or more, the call is cut into about eight groups of
// whole batches (every head of a group, all its tokens, in one launch that
// fills the GPU through the token split).  A group's inputs are contiguous
// in host memory, so they travel as 1-D copies on one stream in group
// order: group 0 has the link to itself and the copies run back to back,
// where token chunks need pitched copies spread over several streams and
// let the first chunk share the link with the next two.  No state is
// carried between groups.  The outputs are staged on the device and copied
// out per group: written by the scan through the host mapping while the
// next groups' inputs come in, they held each group's scan to ~0.5 ms
// against ~0.36 ms (GB300, 750M-shaped layer: 3.7 ms per call against 4.2).
kdn_status diag_host_batches(const DiagArgs& h, cudaStream_t st, long long wait_ns) {
    const int B = h.B, H = h.H, T = h.T, dk = h.dk, dv = h.dv;
    const size_t es = h.dtype == KDN_BF16 ? 2 : 4;
    const size_t S = static_cast<size_t>(dv) * dk;
    const int gb = (B + 7) / 8;                 // batches per group
    const int ng = (B + gb - 1) / gb;
    const size_t gbh = static_cast<size_t>(gb) * H;   // heads per (full) group

    CopyStreams cs;
    cudaError_t e = copy_streams(&cs);
    if (e != cudaSuccess) return from_cuda(e);
    ChunkEvents ev;
    e = ev.create();
    if (e != cudaSuccess) return from_cuda(e);

    // device layout: kBufs group buffer sets, then A
    const size_t qk_b = align256(gbh * T * dk * es);
    const size_t vb_b = align256(gbh * T * dv * es);
    const size_t d_b = align256(gbh * T * es);
    const size_t o_b = align256(gbh * T * dv * 4);
    const size_t init_b = align256(gbh * S * 4);
    const size_t fs_b = align256(2 * gbh * S * 4);
    const size_t set_b = 2 * qk_b + 2 * vb_b + d_b + o_b + (h.I0 ? init_b : 0) + (h.mu0 ? init_b : 0) + fs_b;
    const size_t a_b = align256(static_cast<size_t>(H) * 4);
    cudaMemPool_t pool = nullptr;
    e = host_pool(&pool);
    if (e != cudaSuccess) return from_cuda(e);
    char* base = nullptr;
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&base), kBufs * set_b + a_b, pool, st);
    if (e != cudaSuccess) return from_cuda(e);
    float* A_d = reinterpret_cast<float*>(base + kBufs * set_b);

    Status s;
    s.cuda(cudaMemcpyAsync(A_d, h.A, static_cast<size_t>(H) * 4, cudaMemcpyHostToDevice, st));
    s.cuda(cudaEventRecord(ev.start, st));
    for (cudaStream_t x : {cs.in[0], cs.out}) s.cuda(cudaStreamWaitEvent(x, ev.start, 0));

    const size_t BHs = static_cast<size_t>(B) * H;
    for (int g = 0; g < ng && s.ok(); ++g) {
        const int b = g % kBufs;
        const int nb = (B - g * gb < gb) ? B - g * gb : gb;
        const size_t bh0 = static_cast<size_t>(g) * gbh, nbh = static_cast<size_t>(nb) * H;
        char* set = base + b * set_b;
        char* dq = set;
        char* dkp = dq + qk_b;
        char* dvp = dkp + qk_b;
        char* dbp = dvp + vb_b;
        char* dd = dbp + vb_b;
        float* dout = reinterpret_cast<float*>(dd + d_b);
        char* tail = dd + d_b + o_b;
        float* I0_d = h.I0 ? reinterpret_cast<float*>(tail) : nullptr;
        float* mu0_d = h.mu0 ? reinterpret_cast<float*>(tail + (h.I0 ? init_b : 0)) : nullptr;
        float* fs_d = reinterpret_cast<float*>(tail + (h.I0 ? init_b : 0) + (h.mu0 ? init_b : 0));
        // buffer b was last read by the scan of group g - kBufs and its final
        // state by that group's copy out
        if (g >= kBufs) {
            s.cuda(cudaStreamWaitEvent(cs.in[0], ev.comp[b], 0));
            s.cuda(cudaStreamWaitEvent(cs.in[0], ev.out[b], 0));
        }
        auto in1d = [&](void* dst, const void* src, size_t off, size_t bytes) {
            s.cuda(cudaMemcpyAsync(dst, static_cast<const char*>(src) + off, bytes, cudaMemcpyHostToDevice, cs.in[0]));
        };
        in1d(dq, h.q, bh0 * T * dk * es, nbh * T * dk * es);
        in1d(dkp, h.k, bh0 * T * dk * es, nbh * T * dk * es);
        in1d(dd, h.d, bh0 * T * es, nbh * T * es);
        in1d(dvp, h.v, bh0 * T * dv * es, nbh * T * dv * es);
        in1d(dbp, h.beta, bh0 * T * dv * es, nbh * T * dv * es);
        if (I0_d) in1d(I0_d, h.I0, bh0 * S * 4, nbh * S * 4);
        if (mu0_d) in1d(mu0_d, h.mu0, bh0 * S * 4, nbh * S * 4);
        s.cuda(cudaEventRecord(ev.in[b][0], cs.in[0]));
        s.cuda(cudaStreamWaitEvent(st, ev.in[b][0], 0));
        if (g >= kBufs) s.cuda(cudaStreamWaitEvent(st, ev.out[b], 0));
        DiagArgs a = h;
        a.B = nb;
        a.q = dq;
        a.k = dkp;
        a.v = dvp;
        a.beta = dbp;
        a.d = dd;
        a.d_ld = 0;
        a.A = A_d;
        a.I0 = I0_d;
        a.mu0 = mu0_d;
        a.out = dout;
        a.out_ld = 0;
        a.final_state = h.final_state ? fs_d : nullptr;
        if (s.ok()) s.kdn(a.dtype == KDN_BF16 ? diag_launch_bf16(a, st, wait_ns) : diag_launch_f32(a, st, wait_ns));
        s.cuda(cudaEventRecord(ev.comp[b], st));
        // outputs of group g: out, then mu_T and I_T into their halves of
        // final_state
        s.cuda(cudaStreamWaitEvent(cs.out, ev.comp[b], 0));
        s.cuda(cudaMemcpyAsync(h.out + bh0 * T * dv, dout, nbh * T * dv * 4, cudaMemcpyDeviceToHost, cs.out));
        if (h.final_state) {
            s.cuda(cudaMemcpyAsync(h.final_state + bh0 * S, fs_d, nbh * S * 4, cudaMemcpyDeviceToHost, cs.out));
            s.cuda(cudaMemcpyAsync(h.final_state + BHs * S + bh0 * S, fs_d + nbh * S, nbh * S * 4,
                                   cudaMemcpyDeviceToHost, cs.out));
        }
        s.cuda(cudaEventRecord(ev.out[b], cs.out));
    }
    // every copy is ordered before the release and the final synchronisation
    for (int b = 0; b < kBufs; ++b) {
        if (ng > b) {
            cudaStreamWaitEvent(st, ev.in[b][0], 0);
            cudaStreamWaitEvent(st, ev.out[b], 0);
        }
    }
    s.cuda(cudaFreeAsync(base, st));
    s.cuda(cudaStreamSynchronize(st));
    return s.result();
}

kdn_status diag_host(const DiagArgs& h, cudaStream_t st, long long wait_ns) {
    if (h.B >= 4 && h.T > 0 && !h.lin && h.d_ld == 0 && h.out_ld == 0) return diag_host_batches(h, st, wait_ns);
    const int B = h.B, H = h.H, T = h.T, dk = h.dk, dv = h.dv;
    const size_t es = h.dtype == KDN_BF16 ? 2 : 4;
    const long long BH = static_cast<long long>(B) * H;
    const size_t S = static_cast<size_t>(dv) * dk;
    const int Tc = T > 0 ? diag_chunk_tokens(T) : 0;
    const int nc = T > 0 ? (T + Tc - 1) / Tc : 0;

    CopyStreams cs;
    cudaError_t e = copy_streams(&cs);
    if (e != cudaSuccess) return from_cuda(e);
    ChunkEvents ev;
    e = ev.create();
    if (e != cudaSuccess) return from_cuda(e);

    // device layout: two chunk buffer sets, two carried states, A, I0, mu0
    const size_t qk_b = align256(BH * static_cast<size_t>(Tc) * dk * es);
    const size_t vb_b = align256(BH * static_cast<size_t>(Tc) * dv * es);
    const size_t o_b = align256(BH * static_cast<size_t>(Tc) * dv * 4);
    const size_t set_b = 2 * qk_b + 2 * vb_b + o_b;
    const size_t st_b = align256(2 * BH * S * 4);
    const size_t a_b = align256(static_cast<size_t>(H) * 4);
    const size_t init_b = align256(BH * S * 4);
    const size_t dall_b = align256(BH * static_cast<size_t>(T) * es);   // the whole d
    const size_t total = kBufs * set_b + 2 * st_b + a_b + dall_b + (h.I0 ? init_b : 0) + (h.mu0 ? init_b : 0);
    cudaMemPool_t pool = nullptr;
    e = host_pool(&pool);
    if (e != cudaSuccess) return from_cuda(e);
    char* base = nullptr;
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&base), total, pool, st);
    if (e != cudaSuccess) return from_cuda(e);
    auto set = [&](int b) { return base + b * set_b; };
    char* state[2] = {base + kBufs * set_b, base + kBufs * set_b + st_b};
    float* A_d = reinterpret_cast<float*>(base + kBufs * set_b + 2 * st_b);
    char* d_all = base + kBufs * set_b + 2 * st_b + a_b;
    char* tail = d_all + dall_b;
    float* I0_d = h.I0 ? reinterpret_cast<float*>(tail) : nullptr;
    float* mu0_d = h.mu0 ? reinterpret_cast<float*>(tail + (h.I0 ? init_b : 0)) : nullptr;

    Status s;
    if (T > 0) s.cuda(cudaMemcpyAsync(A_d, h.A, static_cast<size_t>(H) * 4, cudaMemcpyHostToDevice, st));
    if (I0_d) s.cuda(cudaMemcpyAsync(I0_d, h.I0, BH * S * 4, cudaMemcpyHostToDevice, st));
    if (mu0_d) s.cuda(cudaMemcpyAsync(mu0_d, h.mu0, BH * S * 4, cudaMemcpyHostToDevice, st));
    // the copy streams start after the allocation
    s.cuda(cudaEventRecord(ev.start, st));
    for (cudaStream_t x : {cs.in[0], cs.in[1], cs.in[2], cs.in[3], cs.out}) s.cuda(cudaStreamWaitEvent(x, ev.start, 0));

    // A page-locked host `out` is written by the scan itself through its
    // device mapping (no copy-engine traffic back); other memory is staged
    // and copied out per chunk.
    float* out_mapped = nullptr;
    if (T > 0) {
        cudaPointerAttributes pa;
        // (the scan stores 16-byte row quads: the mapping must be 16-byte aligned)
        if (cudaPointerGetAttributes(&pa, h.out) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
            pa.devicePointer && (reinterpret_cast<uintptr_t>(pa.devicePointer) & 15u) == 0)
            out_mapped = static_cast<float*>(pa.devicePointer);
        cudaGetLastError();
    }
    const char* hq = static_cast<const char*>(h.q);
    const char* hk = static_cast<const char*>(h.k);
    const char* hv = static_cast<const char*>(h.v);
    const char* hb = static_cast<const char*>(h.beta);
    // all of d in one contiguous copy (its per-chunk slices are too short for
    // an efficient pitched copy); the scan reads each chunk's slice in place
    if (T > 0) s.cuda(cudaMemcpyAsync(d_all, h.d, BH * static_cast<size_t>(T) * es, cudaMemcpyHostToDevice, cs.in[0]));
    for (int c = 0; c < nc && s.ok(); ++c) {
        const int b = c % kBufs;
        const int t0 = c * Tc, n = (T - t0 < Tc) ? T - t0 : Tc;
        char* in = set(b);
        char* dq = in;
        char* dkp = in + qk_b;
        char* dvp = in + 2 * qk_b;
        char* dbp = in + 2 * qk_b + vb_b;
        float* dout = reinterpret_cast<float*>(in + 2 * qk_b + 2 * vb_b);
        // inputs of chunk c (buffer b was last read by chunk c - 2)
        // (buffer b was last read by the scan of chunk c - kBufs)
        if (c >= kBufs)
            for (int i = 0; i < kIn; ++i) s.cuda(cudaStreamWaitEvent(cs.in[i], ev.comp[b], 0));
        auto rows_in = [&](char* dst, const char* src, size_t row_elems, cudaStream_t cpy) {
            const size_t w = static_cast<size_t>(n) * row_elems * es;
            s.cuda(cudaMemcpy2DAsync(dst, w, src + static_cast<size_t>(t0) * row_elems * es,
                                     static_cast<size_t>(T) * row_elems * es, w, BH,
                                     cudaMemcpyHostToDevice, cpy));
        };
        rows_in(dq, hq, dk, cs.in[0]);
        rows_in(dkp, hk, dk, cs.in[1]);
        rows_in(dvp, hv, dv, cs.in[2]);
        rows_in(dbp, hb, dv, cs.in[3]);
        for (int i = 0; i < kIn; ++i) s.cuda(cudaEventRecord(ev.in[b][i], cs.in[i]));
        // scan of chunk c from the state chunk c - 1 left
        for (int i = 0; i < kIn; ++i) s.cuda(cudaStreamWaitEvent(st, ev.in[b][i], 0));
        if (c >= kBufs) s.cuda(cudaStreamWaitEvent(st, ev.out[b], 0));
        DiagArgs a = h;
        a.q = dq;
        a.k = dkp;
        a.v = dvp;
        a.beta = dbp;
        a.d = d_all + static_cast<size_t>(t0) * es;
        a.d_ld = T;
        a.A = A_d;
        if (c == 0) {
            a.I0 = I0_d;
            a.mu0 = mu0_d;
        } else {
            const float* prev = reinterpret_cast<const float*>(state[(c - 1) & 1]);
            a.mu0 = prev;
            a.I0 = prev + BH * S;
        }
        if (out_mapped) {
            a.out = out_mapped + static_cast<size_t>(t0) * dv;
            a.out_ld = T;
        } else {
            a.out = dout;
        }
        a.final_state = reinterpret_cast<float*>(state[c & 1]);
        a.T = n;
        if (s.ok()) s.kdn(a.dtype == KDN_BF16 ? diag_launch_bf16(a, st, wait_ns)
                                              : diag_launch_f32(a, st, wait_ns));
        s.cuda(cudaEventRecord(ev.comp[b], st));
        // outputs of chunk c
        s.cuda(cudaStreamWaitEvent(cs.out, ev.comp[b], 0));
        if (!out_mapped) {
            const size_t w = static_cast<size_t>(n) * dv * 4;
            s.cuda(cudaMemcpy2DAsync(h.out + static_cast<size_t>(t0) * dv, static_cast<size_t>(T) * dv * 4, dout,
                                     w, w, BH, cudaMemcpyDeviceToHost, cs.out));
        }
        s.cuda(cudaEventRecord(ev.out[b], cs.out));
    }
    if (h.final_state && s.ok()) {
        if (nc > 0) {
            s.cuda(cudaMemcpyAsync(h.final_state, state[(nc - 1) & 1], 2 * BH * S * 4,
                                   cudaMemcpyDeviceToHost, st));
        } else {
            // no tokens: the final state is the initial one
            DiagArgs a = h;
            a.A = A_d;
            a.I0 = I0_d;
            a.mu0 = mu0_d;
            a.out = nullptr;
            a.final_state = reinterpret_cast<float*>(state[0]);
            a.T = 0;
            s.kdn(a.dtype == KDN_BF16 ? diag_launch_bf16(a, st, wait_ns) : diag_launch_f32(a, st, wait_ns));
            s.cuda(cudaMemcpyAsync(h.final_state, state[0], 2 * BH * S * 4, cudaMemcpyDeviceToHost, st));
        }
    }
    // every copy is ordered before the release and the final synchronisation
    for (int b = 0; b < kBufs; ++b) {
        if (nc > b) {
            for (int i = 0; i < kIn; ++i) cudaStreamWaitEvent(st, ev.in[b][i], 0);
            cudaStreamWaitEvent(st, ev.out[b], 0);
        }
    }
    s.cuda(cudaFreeAsync(base, st));
    s.cuda(cudaStreamSynchronize(st));
    return s.result();
}

kdn_status mobius_host(const float* ha, const float* hb, const float* hc, const float* hd,
                       const float* hl, float* hout, long long N, long long T, cudaStream_t st,
                       long long wait_ns) {
    if (N == 0 || T == 0) return KDN_OK;
    // groups of whole sequences: about kHostChunks, each with at least 16 MB
    // of coefficients (smaller scans run as one group)
    long long G = (N + kHostChunks - 1) / kHostChunks;
    const long long min_rows = (16LL << 20) / (16 * T) + 1;
    if (G < min_rows) G = min_rows;
    if (G > N) G = N;
    const int ng = static_cast<int>((N + G - 1) / G);
    CopyStreams cs;
    cudaError_t e = copy_streams(&cs);
    if (e != cudaSuccess) return from_cuda(e);
    ChunkEvents ev;
    e = ev.create();
    if (e != cudaSuccess) return from_cuda(e);
    const size_t coef_b = align256(static_cast<size_t>(G) * T * 4);
    const size_t lam_b = align256(static_cast<size_t>(G) * 4);
    const size_t set_b = 5 * coef_b + lam_b;   // a, b, c, d, out, lambda0
    cudaMemPool_t pool = nullptr;
    e = host_pool(&pool);
    if (e != cudaSuccess) return from_cuda(e);
    char* base = nullptr;
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&base), kBufs * set_b, pool, st);
    if (e != cudaSuccess) return from_cuda(e);
    Status s;
    s.cuda(cudaEventRecord(ev.start, st));
    for (cudaStream_t x : {cs.in[0], cs.in[1], cs.in[2], cs.in[3], cs.out}) s.cuda(cudaStreamWaitEvent(x, ev.start, 0));
    for (int g = 0; g < ng && s.ok(); ++g) {
        const int b = g % kBufs;
        const long long r0 = g * G, rows = (N - r0 < G) ? N - r0 : G;
        const size_t bytes = static_cast<size_t>(rows) * T * 4;
        char* set = base + b * set_b;
        float* dco[4] = {reinterpret_cast<float*>(set), reinterpret_cast<float*>(set + coef_b),
                         reinterpret_cast<float*>(set + 2 * coef_b), reinterpret_cast<float*>(set + 3 * coef_b)};
        float* dout = reinterpret_cast<float*>(set + 4 * coef_b);
        float* dlam = reinterpret_cast<float*>(set + 5 * coef_b);
        if (g >= kBufs)
            for (int i = 0; i < kIn; ++i) s.cuda(cudaStreamWaitEvent(cs.in[i], ev.comp[b], 0));
        const float* hco[4] = {ha, hb, hc, hd};
        for (int i = 0; i < 4; ++i)
            s.cuda(cudaMemcpyAsync(dco[i], hco[i] + r0 * T, bytes, cudaMemcpyHostToDevice, cs.in[i]));
        s.cuda(cudaMemcpyAsync(dlam, hl + r0, static_cast<size_t>(rows) * 4, cudaMemcpyHostToDevice, cs.in[0]));
        for (int i = 0; i < kIn; ++i) s.cuda(cudaEventRecord(ev.in[b][i], cs.in[i]));
        for (int i = 0; i < kIn; ++i) s.cuda(cudaStreamWaitEvent(st, ev.in[b][i], 0));
        if (g >= kBufs) s.cuda(cudaStreamWaitEvent(st, ev.out[b], 0));
        if (s.ok()) s.kdn(mobius_launch(dco[0], dco[1], dco[2], dco[3], dlam, dout, rows, T, st, wait_ns, -1));
        s.cuda(cudaEventRecord(ev.comp[b], st));
        s.cuda(cudaStreamWaitEvent(cs.out, ev.comp[b], 0));
        s.cuda(cudaMemcpyAsync(hout + r0 * T, dout, bytes, cudaMemcpyDeviceToHost, cs.out));
        s.cuda(cudaEventRecord(ev.out[b], cs.out));
    }
    for (int b = 0; b < kBufs; ++b) {
        if (ng > b) {
            for (int i = 0; i < kIn; ++i) cudaStreamWaitEvent(st, ev.in[b][i], 0);
            cudaStreamWaitEvent(st, ev.out[b], 0);
        }
    }
    s.cuda(cudaFreeAsync(base, st));
    s.cuda(cudaStreamSynchronize(st));
    return s.result();
}

}  // namespace kdn
