/*
 * linattn.h — C ABI of the GB300 (sm_103a) normalized linear attention
 * library (liblinattn.so).
 *
 * The method: similarity sim(q, k) = phi(q)^T phi(k) with the feature map
 * phi(x) = ELU(x) + 1 (alpha = 1: x + 1 for x > 0, exp(x) otherwise),
 * applied separately to every query and key vector.  Keys and values are
 * summarized in a state S = sum_j phi(k_j) v_j^T ([m, d_v], m = d_k) and a
 * normalizer z = sum_j phi(k_j) ([m]); a query reads
 *     o = phi(q)^T S / (phi(q)^T z + eps).
 * Sources: "线性注意力从头到尾讲清楚" (lilfry09.github.io) §4 (eps-normalized
 * read), §5 (matrix form), §7 (causal recurrence), §8 (phi = elu + 1,
 * [B,H,N,.] layout); "Linear Attention Math" (aicassindra.com), "The
 * associativity trick, written out", "The recurrent form", "Feature maps:
 * elu+1"; "Linear Attention: Accumulating KV in a Fixed-Size State"
 * (ai-systems-engineering.com), "Summarize state updates and reads with
 * equations".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers are DEVICE pointers on the current CUDA device, except where a
 * comment says otherwise.  Tensors are contiguous row-major, last index
 * fastest:
 *     q, k : [B, H, N, d_k]        v, out : [B, H, N, d_v]
 *     S    : [B, H, d_k, d_v]      z      : [B, H, d_k]
 * (the decode step drops the N axis).  Rows of S are key-feature
 * components, columns value components.  q, k, v have the dtype given by
 * `dt`; out, S and z are always float32.
 *
 * Ownership: the caller owns every buffer.  The library keeps no pointer
 * after a call returns and never frees caller memory.  `out` must not
 * overlap q, k, v, S or z.  Calls only enqueue work on `stream` (a
 * cudaStream_t; NULL = the legacy default stream) and never synchronize
 * the host; errors raised by kernels that were enqueued successfully
 * surface at the caller's next synchronization.
 *
 * Errors: every entry point validates its arguments before touching the
 * GPU and returns a la_status; nothing is launched on error and no output
 * is modified.  LA_ERR_INVALID_VALUE: a NULL pointer where data is
 * needed, B, H, N < 0, d_k or d_v <= 0, or eps negative / not finite.
 * LA_ERR_UNSUPPORTED: d_k or d_v not in {32, 64, 128}, or an unknown
 * dtype.  LA_ERR_MISALIGNED: a pointer not 16-byte aligned.
 * LA_ERR_NO_DEVICE: no usable CUDA device.  LA_ERR_OUT_OF_MEMORY:
 * stream-ordered scratch could not be allocated.  LA_ERR_LAUNCH: a kernel
 * launch failed (cudaGetLastError).
 *
 * Thread safety: calls may be made concurrently from several host threads;
 * the only shared state is a per-device table of attributes filled once.
 */
#ifndef LINATTN_H
#define LINATTN_H

#if defined(__GNUC__)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LA_F32 = 0,  /* q, k, v are float32 */
  LA_BF16 = 1  /* q, k, v are bfloat16 */
} la_dtype;

typedef enum {
  LA_OK = 0,
  LA_ERR_INVALID_VALUE = 1,
  LA_ERR_UNSUPPORTED = 2,
  LA_ERR_MISALIGNED = 3,
  LA_ERR_OUT_OF_MEMORY = 4,
  LA_ERR_LAUNCH = 5,
  LA_ERR_TIMEOUT = 6,
  LA_ERR_NO_DEVICE = 7,
  LA_ERR_TOO_LARGE = 8
} la_status;

/*
 * Global (non-causal) linear attention: every position reads the state of
 * the whole sequence,
 *     S = sum_{j<N} phi(k_j) v_j^T,  z = sum_{j<N} phi(k_j),
 *     out_i = phi(q_i)^T S / (phi(q_i)^T z + eps)      for every i.
 * Source: "线性注意力从头到尾讲清楚" §5 (matrix form) and §8 (the einsum
 * sketch); "Linear Attention Math", "The associativity trick, written out".
 *
 * q, k: [B,H,N,d_k]; v: [B,H,N,d_v] (dtype dt).  out: [B,H,N,d_v] float32,
 * written.  S: [B,H,d_k,d_v], z: [B,H,d_k] float32, OVERWRITTEN with the
 * whole-sequence state (the zero state when N == 0).  May allocate
 * stream-ordered scratch on `stream`.  B*H == 0 is a no-op returning LA_OK.
 */
LA_API la_status la_global(const void *q, const void *k, const void *v, float *out, float *S, float *z,
                    int B, int H, int N, int d_k, int d_v, float eps, la_dtype dt, void *stream);

/*
 * Causal prefill: position t reads the prefix state that INCLUDES token t,
 *     S_t = S_{t-1} + phi(k_t) v_t^T,  z_t = z_{t-1} + phi(k_t),
 *     out_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps),   S_{-1} = 0, z_{-1} = 0.
 * Source: "线性注意力从头到尾讲清楚" §7; "Linear Attention Math", "The
 * recurrent form"; "Linear Attention: Accumulating KV in a Fixed-Size
 * State" (token t joins the state before its query reads it).  Computed in
 * chunks ("Linear Attention: From Pairwise Reads to a Recurrent State",
 * "A recurrence need not force token-serial training").
 *
 * Arguments as la_global.  S, z are OVERWRITTEN with the final prefix state
 * S_{N-1}, z_{N-1}, ready to be passed to la_decode_step.
 */
LA_API la_status la_causal(const void *q, const void *k, const void *v, float *out, float *S, float *z,
                    int B, int H, int N, int d_k, int d_v, float eps, la_dtype dt, void *stream);

/*
 * Causal prefill that continues from a given state: as la_causal, but the
 * recurrence starts from the caller's S, z instead of zero (chunked prefill
 * continuation; N new tokens appended to a sequence whose state is S, z).
 * S, z are read, then OVERWRITTEN with the state after the N new tokens.
 * With N == 0 the state is left unchanged.
 * Source: the causal recurrence above applied to a persistent state
 * ("线性注意力从头到尾讲清楚" §7, last paragraph: only S_t, z_t are kept).
 */
LA_API la_status la_causal_with_state(const void *q, const void *k, const void *v, float *out, float *S,
                               float *z, int B, int H, int N, int d_k, int d_v, float eps,
                               la_dtype dt, void *stream);

/*
 * la_causal without any device memory allocation.  The pages have no
 * counterpart to this call; it exists for callers that must not allocate
 * device memory once they are running: serving runtimes that reserve all of
 * their memory up front and forbid allocation after warm-up (so that memory
 * use and latency stay flat), and processes in which another framework's
 * caching allocator already holds nearly all device memory, so that a
 * stream-ordered allocation made by la_causal could fail mid-run.
 *
 * Same arguments, results and errors as la_causal.  The partial states that
 * la_causal allocates per call (for long sequences split into segments: at
 * most two 128x128 fp32 states per first-pass CTA, at most one CTA per SM) live here
 * in one fixed 20 MiB device array inside the library instead; every GPU
 * that loads the library keeps that array until the process exits.  It holds
 * the partial states of 158 first-pass CTAs.  The planner gives the first pass
 * at most one CTA per SM, so on a GB300 (152 SMs) every problem fits; only on
 * a device with more than 158 SMs can a problem need more (B * H * (segments
 * - 1) > 158), and there the call returns LA_ERR_TOO_LARGE and launches
 * nothing.  All calls share the array, so
 * calls whose work overlaps on the GPU (different streams, or different host
 * threads on the same device) race on it and give wrong results: order them.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Everything else is enqueued on `stream`; the
 * leading-token pass runs on `stream` too (no second stream is used).
 */
LA_API la_status la_causal_noalloc(const void *q, const void *k, const void *v, float *out, float *S,
                                   float *z, int B, int H, int N, int d_k, int d_v, float eps, la_dtype dt,
                                   void *stream);

/*
 * Positive random features (FAVOR+): for every row x of x ([B,H,N,d]) and the
 * m projections w_r (the rows of W, [m, d]),
 *     phi[b,h,t,r] = exp(w_r . x - |x|^2 / 2) / sqrt(m),
 * so that E[phi(q) . phi(k)] = exp(q . k) for w_r ~ N(0, I).  Source:
 * "Linear Attention Math", "Feature maps: elu+1 and positive random
 * features"; "线性注意力从头到尾讲清楚" §9 (approximating the softmax kernel
 * exp(q^T k / sqrt(d_k)): scale q and k by d_k^(-1/4) first).  W is an input
 * (random or orthogonal random projections, drawn by the caller).
 *
 * x: [B,H,N,d], W: [m,d], phi: [B,H,N,m], all of dtype dt (phi is written).
 * d in {32, 64, 128}; m in {32, 64, 128, 256} (the page notes that more
 * features give a closer approximation; m = 256 is m = 2d at d = 128).
 * Tensor cores for bf16 with m in {128, 256} and d in {64, 128} (one launch
 * per 128 features, each reading x); CUDA cores otherwise.  Allocates
 * nothing.  Errors as la_causal.
 * The features feed la_causal_features (or la_global / la_causal with any
 * caller-side map) as phi(q), phi(k).
 */
LA_API la_status la_favor_features(const void *x, const void *W, void *phi, int B, int H, int N, int d, int m,
                                   la_dtype dt, void *stream);

/*
 * Causal prefill on features the caller has already applied: as la_causal
 * with phi the identity, i.e. out_t = phi_q_t^T S_t / (phi_q_t^T z_t + eps),
 * S_t = sum_{j<=t} phi_k_j v_j^T, z_t = sum_{j<=t} phi_k_j.  For any
 * non-negative feature map, e.g. la_favor_features ("Linear Attention Math",
 * "Feature maps: elu+1 and positive random features": the normalized read
 * needs non-negative features).  phi_q, phi_k: [B,H,N,m] (dtype dt, m in
 * {32, 64, 128}, or 256 with d_v <= 128); S: [B,H,m,d_v]; z: [B,H,m]; other
 * arguments, results and errors as la_causal.  The tensor-core path (bf16,
 * m = d_v = 128) takes the features as given, so no leading tokens are
 * recomputed in fp32; every other size runs the exact fp32 CUDA-core pass
 * (32-token chunks at m = 256, where a 64-token chunk and the 128 KB state
 * would not fit in shared memory).
 */
LA_API la_status la_causal_features(const void *phi_q, const void *phi_k, const void *v, float *out, float *S,
                                    float *z, int B, int H, int N, int m, int d_v, float eps, la_dtype dt,
                                    void *stream);

/*
 * Global (non-causal) read on features the caller has already applied: as
 * la_global with phi the identity.  Arguments, results and errors as
 * la_causal_features.  Computed in fp32 on CUDA cores: the tensor-core
 * global read takes the state as one bf16 operand, which heavy-tailed
 * features (a few keys dominating each read while the state sums all of
 * them) do not tolerate.
 */
LA_API la_status la_global_features(const void *phi_q, const void *phi_k, const void *v, float *out, float *S,
                                    float *z, int B, int H, int N, int m, int d_v, float eps, la_dtype dt,
                                    void *stream);

/*
 * Retention: the causal recurrence with an explicit per-head decay and no
 * denominator,
 *     S_t = gamma_h S_{t-1} + k_t v_t^T,   out_t = q_t^T S_t,   S_{-1} = 0,
 * q and k used as given (no feature map), the read taken after the update as
 * in la_causal.  Source: "Linear Attention Math", "The kernel cousins: SSMs
 * and RetNet" (linear attention plus a decay gamma < 1, fixed or one per
 * head, without the denominator).  The pages' gated normalization that
 * replaces the denominator is a separate layer on top of out and is not
 * part of this call.
 *
 * q, k: [B,H,N,d_k]; v: [B,H,N,d_v] (dtype dt); out: [B,H,N,d_v] float32;
 * S: [B,H,d_k,d_v] float32, OVERWRITTEN with S_{N-1} (zeroed when N == 0).
 * gamma: HOST array of H floats, head h (of every batch row) decaying by
 * gamma[h]; read during the call only.
 *
 * Supported: dt LA_F32 or LA_BF16, d_k and d_v each 32, 64 or 128, H <= 128,
 * every gamma[h] in [0, 1] (gamma = 0 keeps only the current token);
 * anything else returns LA_ERR_UNSUPPORTED.  LA_ERR_INVALID_VALUE for a NULL
 * gamma or a gamma that is not finite; other errors as la_causal.
 *
 * Two kernels serve it.  bf16 with d_k == d_v == 128 on an sm_103 device and
 * every gamma[h] >= 0.75 runs on the tensor cores: that chunked kernel weighs
 * a key 128 tokens ahead by gamma^-128, which must stay well inside float
 * range, and it allocates stream-ordered scratch on `stream` for long
 * sequences split into segments.  Everything else runs on CUDA cores, exact
 * fp32 in 64-token chunks whose decay powers never exceed 1, one CTA per
 * head, allocating nothing.
 */
LA_API la_status la_retention(const void *q, const void *k, const void *v, float *out, float *S,
                              const float *gamma, int B, int H, int N, int d_k, int d_v, la_dtype dt,
                              void *stream);

/*
 * Retention continuing from a given state: as la_retention, but the
 * recurrence starts from the caller's S, which is read and then OVERWRITTEN
 * with the state after the N new tokens (N == 0 leaves it unchanged).
 */
LA_API la_status la_retention_with_state(const void *q, const void *k, const void *v, float *out, float *S,
                                         const float *gamma, int B, int H, int N, int d_k, int d_v,
                                         la_dtype dt, void *stream);

/*
 * Gradient of la_causal / la_causal_with_state.  The pages name training
 * through the chunked causal form ("Linear Attention: From Pairwise Reads to
 * a Recurrent State", "A recurrence need not force token-serial training")
 * but write no backward pass; this is the derivative of the causal
 * definition above.  With den_t = phi(q_t)^T z_t + eps, o_t the output and
 * dO_t its upstream gradient:
 *     gnum_t = dO_t / den_t,   gden_t = -(dO_t . o_t) / den_t
 *     dq_t = (S_t gnum_t + z_t gden_t) * phi'(q_t)
 *     dk_j = (U_j v_j + u_j) * phi'(k_j),   dv_j = U_j^T phi(k_j)
 *     U_j = dS + sum_{t >= j} phi(q_t) gnum_t^T,   u_j = dz + sum_{t >= j} phi(q_t) gden_t
 * and the initial state's gradient is (U_0, u_0).  phi'(x) = 1 for x > 0,
 * exp(x) otherwise.
 *
 * q, k: [B,H,N,d_k]; v: [B,H,N,d_v] (dtype dt), the forward's inputs.
 * dout: [B,H,N,d_v] float32, the gradient of the forward's out.  S0, z0
 * (nullable, each independently; NULL = zero): the forward's initial state.
 * dS, dz (nullable; NULL = zero): the gradient of the forward's final state.
 * dq, dk: [B,H,N,d_k], dv: [B,H,N,d_v] float32, written.  dS0: [B,H,d_k,d_v],
 * dz0: [B,H,d_k] float32 (nullable), written with the initial state's gradient.
 * The forward output is neither read nor formed: dO_t . o_t comes from the
 * state read dO S^T and the chunk's scores.  Allocates stream-ordered scratch
 * on `stream`: B*H*(N*(d_v+1) + 2*64*64*ceil(N/64)) floats (gnum, gden, and
 * each 64-token chunk's masked scores and score gradients), plus, when heads
 * are cut into segments, at most 4 * (SM count) * (d_k*d_v + d_k) floats of
 * segment part sums.  Errors as la_causal; every non-NULL pointer must be
 * 16-byte aligned.  B*H == 0 is a no-op.
 */
LA_API la_status la_causal_backward(const void *q, const void *k, const void *v, const float *dout,
                                    const float *S0, const float *z0, const float *dS, const float *dz,
                                    float *dq, float *dk, float *dv, float *dS0, float *dz0, int B, int H,
                                    int N, int d_k, int d_v, float eps, la_dtype dt, void *stream);

/*
 * One recurrent decode step per (b,h) on a persistent state: update, then
 * read the updated state,
 *     S += phi(k) v^T;  z += phi(k);  out = phi(q)^T S / (phi(q)^T z + eps).
 * Source: "线性注意力从头到尾讲清楚" §7 (inference keeps only S_t, z_t);
 * "Linear Attention Math", "The recurrent form" (O(1) time and memory per
 * generated token).
 *
 * q, k: [B,H,d_k]; v: [B,H,d_v] (dtype dt).  out: [B,H,d_v] float32,
 * written.  S: [B,H,d_k,d_v], z: [B,H,d_k] float32, read and written IN
 * PLACE.  Allocates nothing.
 */
LA_API la_status la_decode_step(const void *q, const void *k, const void *v, float *out, float *S,
                         float *z, int B, int H, int d_k, int d_v, float eps, la_dtype dt,
                         void *stream);

/*
 * One recurrent retention step per (b,h) on a persistent state: decay,
 * update, then read,
 *     S = gamma_h S + k v^T;   out = q^T S,
 * q and k used as given, no normalizer.  Source: "Linear Attention Math",
 * "The kernel cousins: SSMs and RetNet" (the recurrent form of retention).
 * Continues the state left by la_retention / la_retention_with_state.
 *
 * q, k: [B,H,d_k]; v: [B,H,d_v] (dtype dt).  out: [B,H,d_v] float32,
 * written.  S: [B,H,d_k,d_v] float32, read and written IN PLACE.  gamma:
 * HOST array of H floats (head h decays by gamma[h]), read during the call.
 * Allocates nothing.
 *
 * Supported: dt LA_F32 or LA_BF16; d_k, d_v in {32, 64, 128}; H <= 128;
 * every gamma[h] in [0, 1] (else LA_ERR_UNSUPPORTED).  LA_ERR_INVALID_VALUE
 * for a NULL pointer or a gamma that is not finite; LA_ERR_MISALIGNED for a
 * pointer that is not 16-byte aligned.  B*H == 0 is a no-op returning LA_OK.
 */
LA_API la_status la_retention_decode_step(const void *q, const void *k, const void *v, float *out, float *S,
                                          const float *gamma, int B, int H, int d_k, int d_v, la_dtype dt,
                                          void *stream);

/*
 * Synchronizes `stream`, then reads and clears the library's device status
 * word on the current device.  Returns LA_ERR_TIMEOUT if a bounded
 * device-side wait inside one of the library's kernels gave up since the
 * last check, LA_ERR_LAUNCH if a kernel refused to run on this device
 * configuration (its shared-memory base was not 1024-byte aligned); in both
 * cases that call's outputs are not valid.  LA_OK otherwise, or the error
 * of the synchronization itself.
 */
LA_API la_status la_device_status(void *stream);

/*
 * Diagnostics, for measuring the carry of the causal prefill: fixes how many
 * segments each head is cut into by the tensor-core passes of la_causal,
 * la_causal_with_state, la_causal_features and la_retention (1 = one CTA
 * carries each head's state through all of its chunks; G > 1 = G segments
 * whose starting states come from the first pass over the earlier ones),
 * clamped to the number of 128-token chunks.  0 restores the planner's
 * choice (enough segments to cover the SMs once, at least 4 chunks each).
 * Process-wide; results are the same up to rounding for every value.
 * la_causal_noalloc ignores it.  LA_ERR_INVALID_VALUE outside [0, 4096].
 */
LA_API la_status la_diag_force_segments(int segments);
/*
 * Testing only: exercises the bounded-wait failure path on the GPU without a
 * fault.  Arms a one-shot injection taken by the NEXT launch of the
 * tensor-core causal pass (la_causal, la_causal_with_state or
 * la_causal_noalloc with bf16 inputs and d_k = d_v = 128), from any host
 * thread: in that launch the first CTA (segment 0 of head 0) does not issue
 * the key load of chunk `chunk` (128-token chunks of its segment), and every
 * mbarrier wait of the launch gives up after wait_us microseconds instead of
 * 4 s.  The waits that depend on the missing load run out; the CTA raises its
 * abort word, drains the copies and tensor-core work already issued, frees its
 * tensor memory and exits, and the next la_device_status returns
 * LA_ERR_TIMEOUT.  That call's outputs are not valid; later calls are
 * unaffected.  If the chunk does not exist in that launch nothing is left out.
 * LA_ERR_INVALID_VALUE for chunk < 0 or wait_us outside [1, 1000000].  No
 * counterpart in the pages: it tests this library's error reporting.
 */
LA_API la_status la_test_inject_missing_load(int chunk, unsigned int wait_us);
/* Static English description of a status code (never NULL). */
LA_API const char *la_status_string(la_status s);

/* Library ABI version: (major << 16) | minor. */
LA_API int la_version(void);

/*
 * Diagnostics: name and description of the CUDA runtime error behind the
 * last LA_ERR_LAUNCH / LA_ERR_OUT_OF_MEMORY / LA_ERR_NO_DEVICE returned to
 * the calling host thread ("no error" if none).  Static storage; never NULL.
 */
LA_API const char *la_last_error_detail(void);

/*
 * Diagnostics: number of kernels this library has enqueued in this process
 * (all devices, all threads; a relaxed atomic counter incremented at every
 * successful launch).  Read it before and after a region to count the
 * library's launches inside it.
 */
LA_API unsigned long long la_kernel_launches(void);

/* Kernels whose device time la_profile_read reports. */
typedef enum {
  LA_KERNEL_CAUSAL_MAIN = 0,   /* tensor-core causal pass (bf16, d_k = d_v = 128) */
  LA_KERNEL_CAUSAL_STATE = 1,  /* its state-only first pass over earlier segments */
  LA_KERNEL_EXACT_HEAD = 2,    /* exact fp32 pass over each head's leading tokens */
  LA_KERNEL_CAUSAL_SIMT = 3,   /* fp32 chunked causal kernel (other shapes) */
  LA_KERNEL_GLOBAL_STATE = 4,  /* global form: state build */
  LA_KERNEL_GLOBAL_READ = 5,   /* global form: read */
  LA_KERNEL_DECODE = 6,         /* recurrent decode step */
  LA_KERNEL_RETENTION_MAIN = 7,   /* tensor-core retention pass */
  LA_KERNEL_RETENTION_STATE = 8,  /* its first pass over earlier segments */
  LA_KERNEL_RETENTION_DECODE = 9, /* recurrent retention step */
  LA_KERNEL_BACKWARD = 10,        /* causal backward */
  LA_KERNEL_FAVOR = 11,           /* positive random features */
  LA_KERNEL_GLOBAL_FUSED = 12     /* global form in one pass: a CTA per head (d = 64, heads >= 80 % of SMs) */
} la_kernel;

/*
 * Diagnostics: per-kernel device time.  la_profile_enable(1) clears the
 * totals and from then on brackets every launch of this library with a CUDA
 * event pair recorded on the launch's own stream (two event creations and
 * records per launch: host cost only, nothing is added to the kernels);
 * la_profile_enable(0) stops recording.  la_profile_read waits for the
 * recorded pairs to complete and returns, for one kernel, the summed
 * milliseconds between its events and the number of timed launches since
 * the last enable.  A kernel that shares the GPU with a concurrent one (the
 * exact leading-token pass runs beside the tensor-core pass) is timed as it
 * ran, contention included.  Thread-safe.  Errors: LA_ERR_INVALID_VALUE for an
 * unknown kernel or NULL outputs; a failed event query maps like a launch
 * error (the totals still hold the pairs that completed).
 */
LA_API la_status la_profile_enable(int on);
LA_API la_status la_profile_read(la_kernel kernel, double *ms_total, long long *launches);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
