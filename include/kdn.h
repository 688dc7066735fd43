/*
 * kdn.h -- C ABI of the GB300 (sm_103a) uncertainty-tracked linear-attention
 * scans.  Plain pointers and sizes only; no C++ or framework types.
 *
 * Two operations:
 *
 *  kdn_diag_scan_fwd -- the diagonal metaplastic update of
 *    "Learning to Remember, Learn, and Forget in Attention-Based Models"
 *    (Metodologia 1: forget gate alpha_t = exp(-A d_t); Metodologia 2: the
 *    closed-form update of the importance I_t and the mean mu_t), per head a
 *    d_v x d_k state, with readout o_t = mu_t q_t (the posterior mean read by
 *    the query, "Kalman Linear Attention (KLA)", Metodologia 1, "Readout"):
 *        I_t  = alpha_t I_{t-1} + (1-alpha_t) I_prior + beta_t (x) k_t^2
 *        mu_t = alpha_t (I_{t-1}/I_t) . mu_{t-1} + (1/I_t) . [(beta_t . v_t) (x) k_t]
 *        o_t[i] = sum_j mu_t[i][j] q_t[j]
 *    with beta_t on the value axis: (beta (x) k^2)[i][j] = beta_i k_j^2 and
 *    ((beta . v) (x) k)[i][j] = beta_i v_i k_j.
 *
 *  kdn_mobius_scan -- the precision recursion of "Kalman Linear Attention
 *    (KLA)", Metodologia 2 ("Parallelizzazione tramite Trasformazioni di
 *    Moebius"):
 *        lambda_t = (a_t lambda_{t-1} + b_t) / (c_t lambda_{t-1} + d_t),
 *    computed as a parallel prefix scan of 2x2 matrix products.
 *
 * Conventions shared by every entry point:
 *  - All tensors are dense, row-major (C order) and contiguous.  Device
 *    pointers must point to memory of the current CUDA device; they are
 *    read/written asynchronously on `stream` (a cudaStream_t, or NULL for the
 *    legacy default stream).  The call returns as soon as the work is queued.
 *  - The caller owns every buffer.  Entry points may take short-lived
 *    stream-ordered scratch from the device's default memory pool
 *    (cudaMallocAsync / cudaFreeAsync on `stream`); the library holds no other
 *    device memory besides one error word per device, the fixed array of
 *    kdn_mobius_scan_noalloc and the pool of the host-buffer calls.
 *  - Errors detectable on the host (null pointers, bad sizes, unsupported
 *    head dimensions, misaligned pointers) are returned before anything is
 *    launched.  Launch failures return KDN_ERR_CUDA.  Errors found by a
 *    kernel (a bounded wait that ran out) are recorded in a per-device error
 *    word and reported by kdn_get_device_error().
 *  - Values are not checked: non-finite inputs or non-positive Moebius
 *    denominators propagate as IEEE inf/nan.
 */
#ifndef KDN_H_
#define KDN_H_

#if defined(__GNUC__) || defined(__clang__)
#define KDN_API __attribute__((visibility("default")))
#else
#define KDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDN_OK = 0,
    KDN_ERR_INVALID_ARG = -1,  /* null pointer, size out of range, misalignment */
    KDN_ERR_UNSUPPORTED = -2,  /* head dimension or dtype not supported */
    KDN_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
    KDN_ERR_TIMEOUT = -4,      /* a bounded device-side wait ran out */
    KDN_ERR_ALLOC = -5         /* scratch allocation failed */
} kdn_status;

typedef enum {
    KDN_F32 = 0,   /* IEEE binary32 */
    KDN_BF16 = 1   /* bfloat16 */
} kdn_dtype;

/*
 * kdn_diag_scan_fwd -- forward diagonal metaplastic scan with readout.
 *
 *   q, k       [B,H,T,dk]  in_dtype   query and key of each token-head
 *   v, beta    [B,H,T,dv]  in_dtype   value and input-dependent importance
 *   d          [B,H,T]     in_dtype   gate input; alpha_t = exp(-A[h] d_t)
 *   A          [H]         fp32       per-head gate rate
 *   I_prior                fp32       prior importance (> 0)
 *   I0, mu0    [B,H,dv,dk] fp32 or NULL   initial importance and mean; both
 *                          NULL => I_0 = I_prior, mu_0 = 0.  If exactly one is
 *                          NULL, that one takes its default.
 *   out        [B,H,T,dv]  fp32       o_t = mu_t q_t (after the token's update)
 *   final_state [2,B,H,dv,dk] fp32 or NULL   mu_T then I_T; feeding them back
 *                          as mu0/I0 of a call on the following tokens gives
 *                          the same result as one call over all tokens.
 *   B >= 1, H >= 1, T >= 0.  T = 0 writes only final_state (= the initial
 *   state); q, k, v, beta, d, A and out are then not read and may be NULL.
 *   dk, dv in {16, 32, 64, 128}, B*H*T*max(dk,dv) < 2^62.
 *   Pointers must be 16-byte aligned.  in_dtype is KDN_F32 or KDN_BF16.
 *
 * Arithmetic: fp32 state and accumulation.  The library computes the same
 * recurrence in the equivalent information form eta = I . mu with exact
 * power-of-two rescaling (the kernel source documents the rescaling); results match the
 * fp64 definition to a few fp32 ulps times the sequence's conditioning.
 */
KDN_API kdn_status kdn_diag_scan_fwd(const void* q, const void* k, const void* v,
                             const void* beta, const void* d, const float* A,
                             float I_prior, const float* I0, const float* mu0,
                             float* out, float* final_state,
                             int B, int H, int T, int dk, int dv,
                             kdn_dtype in_dtype, void* stream);

/*
 * kdn_diag_mobius_scan_fwd -- kdn_diag_scan_fwd and, in the same launch, the
 * per-head precision recursion of "Kalman Linear Attention (KLA)",
 * Metodologia 2 ("Parallelizzazione tramite Trasformazioni di Moebius"):
 * one lambda sequence per head over the same T tokens,
 *     lambda_t = (a_t lambda_{t-1} + b_t) / (c_t lambda_{t-1} + d_t).
 *
 *   q ... final_state   as for kdn_diag_scan_fwd
 *   ma, mb, mc, md  [B*H, T] fp32   the coefficients a, b, c, d of each head
 *                   (row b*H + h)
 *   lambda0         [B*H]    fp32   lambda_0 of each head
 *   lambda_out      [B*H, T] fp32   lambda_1 .. lambda_T of each head
 *   Sizes and errors as for kdn_diag_scan_fwd; the Moebius pointers must be
 *   4-byte aligned and are required when T > 0.
 *
 * When T % 4 == 0 and ma, mb, mc, md, lambda_out are 16-byte aligned, the
 * lambda sequences are walked by extra CTAs of the diagonal scan's full-pass
 * grid, placed after the scan's CTAs so that they fill the CTA slots its last
 * wave leaves free; otherwise the Moebius scan runs as its own launch after
 * the scan (same results, same stream).  lambda equals kdn_mobius_scan on the
 * same coefficients (the same tile composition and sequential evaluation).
 */
KDN_API kdn_status kdn_diag_mobius_scan_fwd(const void* q, const void* k, const void* v,
                                    const void* beta, const void* d, const float* A,
                                    float I_prior, const float* I0, const float* mu0,
                                    float* out, float* final_state,
                                    const float* ma, const float* mb, const float* mc,
                                    const float* md, const float* lambda0, float* lambda_out,
                                    int B, int H, int T, int dk, int dv,
                                    kdn_dtype in_dtype, void* stream);

/*
 * kdn_lin_scan_fwd -- the non-metaplastic limit of kdn_diag_scan_fwd: the
 * importance is held at I_prior ("Learning to Remember, Learn, and Forget in
 * Attention-Based Models", Metodologia 4, Unificazione Teorica: Mamba2 is the
 * case I_t = I_prior), so per head and token
 *     mu_t = alpha_t mu_{t-1} + (beta_t . v_t) (x) k_t / I_prior,
 *     o_t[i] = sum_j mu_t[i][j] q_t[j],        alpha_t = exp(-A d_t)
 * (decayed linear attention with a per-token scalar decay).
 *
 *   q, k, v, beta, d, A, I_prior   as for kdn_diag_scan_fwd
 *   mu0       [B,H,dv,dk] fp32 or NULL (mu_0 = 0)
 *   out       [B,H,T,dv] fp32
 *   final_mu  [B,H,dv,dk] fp32 or NULL   mu_T (feeding it back as mu0 of a
 *             call on the following tokens gives one call's result)
 *   Sizes, alignment and errors as for kdn_diag_scan_fwd.
 *
 * Same kernels as the diagonal scan with the importance update and the
 * per-element division taken out (two FP32 FMA per state element and token:
 * the write and the readout); long sequences with few heads are split into
 * token parts the same way.
 */
KDN_API kdn_status kdn_lin_scan_fwd(const void* q, const void* k, const void* v,
                            const void* beta, const void* d, const float* A,
                            float I_prior, const float* mu0, float* out,
                            float* final_mu, int B, int H, int T, int dk, int dv,
                            kdn_dtype in_dtype, void* stream);

/*
 * kdn_diag_scan_bwd -- backward pass of kdn_diag_scan_fwd (the pages' kernels
 * serve training on GPUs: "Learning to Remember, Learn, and Forget in
 * Attention-Based Models", Contributi Chiave).  For the scalar
 *     L = sum grad_out . out + sum dmu_T . mu_T + sum dI_T . I_T
 * of the forward call with the same inputs, writes dL/d(input) for every
 * input.  The forward is recomputed inside the call (nothing from a forward
 * call is needed).
 *
 *   q, k, v, beta, d, A, I_prior, I0, mu0   as for kdn_diag_scan_fwd
 *   grad_out          [B,H,T,dv] fp32   dL/d out
 *   grad_final_state  [2,B,H,dv,dk] fp32 or NULL   dL/d mu_T then dL/d I_T
 *                                    (NULL: the final state is not used)
 *   grad_q, grad_k    [B,H,T,dk] fp32   written
 *   grad_v, grad_beta [B,H,T,dv] fp32   written
 *   grad_d            [B,H,T]    fp32   written
 *   grad_A            [H] fp32 or NULL  written: summed over the batch
 *   grad_init_state   [2,B,H,dv,dk] fp32 or NULL   written: dL/d mu_0 then
 *                     dL/d I_0 (of the initial state used, given or default)
 *   I_prior gets no gradient (a fixed hyperparameter).
 *
 *   B >= 1, H >= 1, T >= 0; dk, dv in {16, 32, 64, 128};
 *   B*H*T*max(dk,dv)^2 < 2^62.  Array pointers 16-byte aligned (d and A:
 *   element-aligned; grad_d, grad_A: 4-byte aligned).  With T = 0 only
 *   grad_init_state (= grad_final_state) and grad_A (= 0) are written.
 *
 * Scratch ("workspace"): kdn_diag_scan_bwd_workspace gives its size, about
 * B*H*T*dv*dk + 8*B*H*T*dv bytes (every 8th token's state, and per-column-
 * block row sums; 16*B*H*T*dv for the latter when so few heads that the call
 * takes 16-column blocks, B*H*dk/32*2 <= the current device's SM count).
 * With workspace == NULL the call takes it from the
 * stream-ordered allocator (cudaMallocAsync, freed on the stream before
 * return; KDN_ERR_ALLOC if it cannot be had); otherwise workspace is a
 * 256-byte aligned device buffer of at least that many bytes, owned by the
 * caller and in use until the call's work on the stream completes
 * (KDN_ERR_INVALID_ARG if smaller or unaligned).  Each CTA owns all of its
 * SM's tensor memory while it runs.  Arithmetic: fp32 (the information form
 * eta = I mu, J = I - I_prior); results are deterministic (fixed summation
 * order).
 */
KDN_API kdn_status kdn_diag_scan_bwd(const void* q, const void* k, const void* v,
                             const void* beta, const void* d, const float* A,
                             float I_prior, const float* I0, const float* mu0,
                             const float* grad_out, const float* grad_final_state,
                             float* grad_q, float* grad_k, float* grad_v,
                             float* grad_beta, float* grad_d, float* grad_A,
                             float* grad_init_state,
                             int B, int H, int T, int dk, int dv,
                             kdn_dtype in_dtype, void* workspace,
                             long long workspace_bytes, void* stream);

/* Bytes of workspace kdn_diag_scan_bwd needs for these sizes on the current
 * device (no GPU work; it reads the device's SM count). */
KDN_API kdn_status kdn_diag_scan_bwd_workspace(int B, int H, int T, int dk, int dv,
                                       long long* workspace_bytes);

/*
 * kdn_mobius_scan -- lambda_t = (a_t lambda_{t-1} + b_t) / (c_t lambda_{t-1} + d_t)
 * for N independent sequences.
 *
 *   a, b, c, d [N,T] fp32   coefficients of step t (index t = 0..T-1)
 *   lambda0    [N]   fp32   initial value of each sequence
 *   out        [N,T] fp32   lambda_1..lambda_T (lambda0 is not repeated)
 *   N >= 0, T >= 0, N*T < 2^62; pointers 4-byte aligned (16-byte alignment
 *   with T % 4 == 0 enables the vector path).
 *
 * Sequences are cut into tiles of 2048 steps.  With T % 4 == 0 and 16-byte
 * aligned buffers, multi-tile sequences normally run on persistent CTAs that
 * each own whole sequences, with no scratch.  A few long sequences (too few
 * to fill the GPU, each long enough that walking it tile by tile costs more
 * than a look-back) and unaligned rows instead chain the tiles of a sequence
 * by a cross-block look-back that uses stream-ordered scratch
 * (cudaMallocAsync; KDN_ERR_ALLOC if it cannot be had).  kdn_mobius_scan_plan
 * tells which for given sizes.
 */
KDN_API kdn_status kdn_mobius_scan(const float* a, const float* b, const float* c,
                           const float* d, const float* lambda0, float* out,
                           long long N, long long T, void* stream);

/*
 * kdn_diag_step -- one token of kdn_diag_scan_fwd's update for B x H heads
 * whose state is kept on the device between calls (batched decoding), the
 * state read and overwritten in place.  The same equations for T = 1:
 *     alpha = exp(-A d); I' = alpha I + (1 - alpha) I_prior + beta_i k_j^2;
 *     mu' = (alpha I mu + beta_i v_i k_j) / I';  o_i = sum_j mu'_ij q_j.
 *
 *   q, k     [B,H,dk]  in_dtype     v, beta [B,H,dv] in_dtype   d [B,H] in_dtype
 *   A        [H] fp32               I_prior scalar
 *   state    [2,B,H,dv,dk] fp32, 16-byte aligned: mu then I (the layout of
 *            kdn_diag_scan_fwd's final_state and of its mu0 / I0); read and
 *            overwritten with the state after the token
 *   out      [B,H,dv] fp32
 *
 * Equal to kdn_diag_scan_fwd with T = 1, mu0 = state[0], I0 = state[1] and
 * final_state = state, up to rounding.  The step reads and writes each state
 * element once (16 bytes) and is bound by HBM bandwidth.  Asynchronous on
 * `stream`; no scratch.
 */
KDN_API kdn_status kdn_diag_step(const void* q, const void* k, const void* v, const void* beta,
                                 const void* d, const float* A, float I_prior, float* state,
                                 float* out, int B, int H, int dk, int dv, kdn_dtype in_dtype,
                                 void* stream);

/*
 * kdn_diag_scan_fwd_host -- kdn_diag_scan_fwd with every tensor (inputs,
 * A, I0, mu0, out, final_state) in host memory: same arguments, layouts and
 * results; pointers need only their element alignment.  The call returns when
 * the results are in host memory.
 *
 * With B >= 4 the call is cut into about eight groups of whole batches,
 * pipelined over three device buffers: a group's inputs (contiguous in host
 * memory) are copied in on an internal stream, in group order, while
 * earlier groups are scanned on `stream`, and each group's out and final
 * state are copied back on another internal stream.  With B < 4 the tokens
 * are cut into about eight chunks (at least 512 tokens each) instead: later
 * chunks' inputs come in on internal streams while chunk c is scanned,
 * outputs go straight into page-locked 16-byte aligned host memory from the
 * scan (or are copied back), and the state passes from chunk to chunk on
 * the device.  Page-locked host buffers (cudaHostAlloc, cudaHostRegister,
 * pinned framework tensors) let the copies overlap the scan; pageable
 * buffers give the same results with serialised copies.  Device memory for
 * three groups or chunks (and, for chunks, the carried states and d) comes,
 * stream-ordered on `stream`, from a memory pool of the library's own (one
 * per device) that keeps freed memory for the next host-buffer call instead
 * of releasing it to CUDA: after a call the pool holds up to the largest
 * scratch a host-buffer call has needed (about three groups' inputs,
 * outputs and states; 0.31 GB for 8 x 16 heads x 4096 tokens at d = 128).
 * KDN_ERR_ALLOC if the memory cannot be had.
 */
KDN_API kdn_status kdn_diag_scan_fwd_host(const void* q, const void* k, const void* v,
                                          const void* beta, const void* d, const float* A,
                                          float I_prior, const float* I0, const float* mu0,
                                          float* out, float* final_state, int B, int H, int T,
                                          int dk, int dv, kdn_dtype in_dtype, void* stream);

/*
 * kdn_mobius_scan_host -- kdn_mobius_scan with a, b, c, d, lambda0 and out in
 * host memory; returns when out is written.  The sequences are cut into
 * groups (about eight, at least 16 MB of coefficients each) whose copies in
 * and out overlap the scans of their neighbours, as for
 * kdn_diag_scan_fwd_host; scratch from the same library pool.
 */
KDN_API kdn_status kdn_mobius_scan_host(const float* a, const float* b, const float* c,
                                        const float* d, const float* lambda0, float* out,
                                        long long N, long long T, void* stream);

/*
 * kdn_diag_scan_plan -- how kdn_diag_scan_fwd would run these sizes on the
 * current device, without launching anything: `parts` = token ranges the
 * sequence is split into (1 = no split), `kernels` = kernels one call
 * launches, `scratch_bytes` = stream-ordered scratch one call takes.  Any
 * output pointer may be NULL.  Needs a CUDA device (occupancy query).
 */
KDN_API kdn_status kdn_diag_scan_plan(int B, int H, int T, int dk, int dv, kdn_dtype in_dtype,
                                      int* parts, int* kernels, long long* scratch_bytes);

/*
 * kdn_mobius_scan_plan -- kernels one kdn_mobius_scan call launches and the
 * scratch bytes it takes (plus one cudaMemsetAsync of part of the scratch
 * when scratch_bytes > 0), for 16-byte aligned buffers on the current device
 * (the choice between the look-back and the sequence-per-CTA kernel depends
 * on the device's resident CTA count).
 */
KDN_API kdn_status kdn_mobius_scan_plan(long long N, long long T, int* kernels,
                                        long long* scratch_bytes);

/*
 * kdn_mobius_scan_noalloc -- kdn_mobius_scan for callers that must not
 * allocate device memory during a call (for instance a process whose
 * framework reserved the GPU's memory up front, or a latency-critical loop
 * where allocator calls are not allowed).  The pages have no counterpart:
 * this is an interface variant, not part of the method.
 *
 * Same arguments, layouts and results as kdn_mobius_scan.  The look-back
 * scratch lives in a fixed 1 MiB array inside the library's device image,
 * which every GPU that loads the library holds until the process exits; no
 * cudaMalloc/cudaMallocAsync/cudaFree is called.  Limit: a call that needs
 * look-back scratch may use at most 43690 tiles, N * ceil(T / 2048) <= 43690;
 * larger calls return KDN_ERR_INVALID_ARG without launching.  A call needs
 * look-back scratch when T > 2048 and the sequence-walk kernel does not take
 * it.  That kernel needs T % 4 == 0 and a, b, c, d, out 16-byte aligned (an
 * offset view of a larger tensor may not be); on such rows it is chosen when
 * the sequences fill the GPU, when a cost model prefers it, or when the
 * look-back would need more tiles than the array holds.  So only calls with
 * T % 4 != 0 or unaligned rows can meet the limit.  The cost model counts no
 * allocation for this entry point, so it may pick the look-back where
 * kdn_mobius_scan would walk (kdn_mobius_scan_plan reports the allocating
 * entry point's choice).
 * The first call on a device fetches the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls share the one array: calls whose executions overlap on the GPU
 * (for example on two streams) race and give wrong results; serialise them.
 */
KDN_API kdn_status kdn_mobius_scan_noalloc(const float* a, const float* b, const float* c,
                                           const float* d, const float* lambda0, float* out,
                                           long long N, long long T, void* stream);

/* Human-readable name of a status code (static string). */
KDN_API const char* kdn_status_string(kdn_status s);

/*
 * kdn_get_device_error -- synchronises `stream`, then reads and clears the
 * current device's error word.  Returns KDN_OK if no kernel recorded an
 * error since the last call, else the recorded status (e.g.
 * KDN_ERR_TIMEOUT), or KDN_ERR_CUDA if synchronisation failed.
 */
KDN_API kdn_status kdn_get_device_error(void* stream);

/*
 * kdn_set_wait_limit_ns -- upper bound, in nanoseconds of GPU time, on any
 * single device-side wait of later launches (default 2e9).  A wait that runs
 * out records KDN_ERR_TIMEOUT and the kernel carries on without blocking.
 * Values <= 0 restore the default.
 */
KDN_API void kdn_set_wait_limit_ns(long long ns);

/*
 * kdn_debug_stall_mobius_tile -- fault injection for tests.  For the next
 * kdn_mobius_scan launches, the block that takes look-back tile `tile`
 * (0-based, in scheduling order) never publishes its result, so its
 * successor's wait must run out (KDN_ERR_TIMEOUT) instead of hanging.
 * A negative value (the default) disables the injection.
 */
KDN_API void kdn_debug_stall_mobius_tile(long long tile);

/* Library version string, e.g. "kdn 0.1.0 sm_103a". */
KDN_API const char* kdn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDN_H_ */
