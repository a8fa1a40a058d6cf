/*
 * pathattn.h -- C ABI of libpathattn.so, the PaTH attention forward pass on
 * one NVIDIA GB300 (sm_103a).
 *
 * The operation (from "PaTH Attention: Position Encoding via Accumulating
 * Householder Transformations", discussion slides for arXiv:2505.16381v2,
 * frame "PaTH inserts a learned transformation along every path"):
 *
 *   H_t   = I - beta_t w_t w_t^T            (||w_t|| = 1, beta_t in [0, 2])
 *   s_ij  = scale * k_j^T H_{j+1} ... H_i q_i  [+ sum_{s=j+1}^{i} log f_s]
 *   o_i   = sum_{j<=i} softmax_j(s_ij) v_j,   lse_i = log sum_{j<=i} exp(s_ij)
 *
 * The bracketed gate term is the PaTH-FoX forget gate (frame "FoX adds a
 * separate mechanism for forgetting"); it is added outside the scale.
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense, contiguous, row-major: q, k, v, w, out are
 *     [B, H, T, d]; beta, logf, lse are [B, H, T].
 *   - Device pointers must be 16-byte aligned and live on the current device.
 *   - dtype selects the element type of q, k, v, w and out: PATH_DTYPE_BF16
 *     (fp32 accumulation, tensor cores) or PATH_DTYPE_F32 (fp32 throughout).
 *     beta, logf and lse are always fp32.
 *   - d must be 64 or 128; B, H, T >= 1; B*H*T*d must fit in 2^31 - 1 rows*cols
 *     per operand index space (checked).
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Launches are
 *     asynchronous on that stream; nothing here synchronises the device except
 *     where a function says so.
 *   - Inputs are never written.  The caller owns every pointer it passes.
 *   - Errors are returned as path_status_t values; no function throws or
 *     aborts.  Argument checks happen before any CUDA call.
 */
#ifndef PATHATTN_H
#define PATHATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PATH_OK = 0,
  PATH_ERR_INVALID_ARG = -1, /* NULL or misaligned pointer, bad size, bad dtype */
  PATH_ERR_UNSUPPORTED = -2, /* valid but not supported here (e.g. d not 64/128, not sm_103) */
  PATH_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
  PATH_ERR_TIMEOUT = -4,     /* a kernel's bounded wait expired (device status word) */
  PATH_ERR_OOM = -5          /* workspace allocation failed */
} path_status_t;

typedef enum { PATH_DTYPE_F32 = 0, PATH_DTYPE_BF16 = 1 } path_dtype_t;

/*
 * path_attn_fwd -- the PaTH / PaTH-FoX causal attention forward pass.
 *
 * Defined by the slides' frames "PaTH inserts a learned transformation along
 * every path" (logits and softmax readout) and "FoX adds a separate mechanism
 * for forgetting" (gate); computed blockwise as in frames "A triangular
 * representation makes paths computable", "A right-to-left scan accumulates
 * cross-block paths" and "Backup: fix orientation before implementing UT
 * products".
 *
 *   q, k, v, w  device, [B,H,T,d], dtype      read only
 *   beta        device, [B,H,T], fp32          read only; values in [0, 2]
 *   logf        device, [B,H,T], fp32, or NULL (NULL = plain PaTH, no gate)
 *   scale       multiplies k_j^T (...) q_i only (e.g. 1/sqrt(d))
 *   out         device, [B,H,T,d], dtype       written
 *   lse         device, [B,H,T], fp32, or NULL; natural-log normaliser
 *
 * The library takes a stream-ordered workspace on `stream` from its own
 * memory pool (cached across calls) and returns it, stream-ordered, before
 * returning.  Returns PATH_ERR_OOM if it cannot.  Device-side wait timeouts
 * are reported by path_attn_device_status(), not by this call.
 */
int path_attn_fwd(const void* q, const void* k, const void* v, const void* w,
                  const float* beta, const float* logf, float scale, void* out,
                  float* lse, int B, int H, int T, int d, int dtype, void* stream);

/*
 * path_attn_fwd_host -- the same operation on HOST buffers (same shapes and
 * dtypes as path_attn_fwd).  Copies the inputs to the current device, runs
 * path_attn_fwd on `stream`, copies out (and lse if non-NULL) back and
 * synchronises `stream` before returning.  The (b, h) problems go in up to
 * four slices: copies in and out run on two library-owned copy streams and
 * overlap the computation of other slices.  Host buffers may be pageable;
 * page-locked buffers make the copies faster and let them overlap.  Device
 * buffers come from the library's pool and are returned before the call ends.
 */
int path_attn_fwd_host(const void* q, const void* k, const void* v, const void* w,
                       const float* beta, const float* logf, float scale, void* out,
                       float* lse, int B, int H, int T, int d, int dtype, void* stream);

/*
 * path_attn_fwd_partial -- partial PaTH: PaTH on the first r of the d head
 * dimensions, no position encoding on the other d - r (the authors' proposal
 * in the OpenReview discussion, sections "Efficiency" and "NoPE not included
 * as a baseline"; the choice of the first r coordinates is this library's):
 *   s_ij = scale * (ka_j^T G_{j+1} ... G_i qa_i + kb_j^T qb_i) [+ gate],
 *   G_t = I_r - beta_t u_t u_t^T,  q = (qa, qb), k = (ka, kb), qa, ka in R^r.
 * Arguments as path_attn_fwd except w, which is u: device, [B,H,T,r], dtype,
 * any alignment (NULL allowed when r == 0), and 0 <= r <= d.  A transition
 * that is the identity outside the first r coordinates gives exactly these
 * logits.  For bf16 with d = 128, r = 64 and u 16-byte aligned, dedicated
 * kernels run: the preparation reads u with zeros past column r and the
 * attention carries only the first r coordinates of the running query
 * through the transitions (one MMA of width C + r per key chunk instead of
 * C + d); about 1.13x faster than path_attn_fwd at B=2 H=16 T=16384.  Every
 * other case widens u with zeros to [B,H,T,d] in a stream-ordered buffer (two
 * copy operations) and runs the PaTH kernels, costing what path_attn_fwd
 * costs plus that copy.
 */
int path_attn_fwd_partial(const void* q, const void* k, const void* v, const void* w,
                          const float* beta, const float* logf, float scale, void* out,
                          float* lse, int B, int H, int T, int d, int r, int dtype, void* stream);

/*
 * path_attn_bwd -- gradients of a path_attn_fwd call: with a loss L whose
 * gradients with respect to out and lse are dout and dlse, returns
 * dq, dk, dv, dw = dL/d(q, k, v, w), dbeta = dL/dbeta and (PaTH-FoX)
 * dlogf = dL/dlog f.  The pages time the forward and backward together
 * (OpenReview discussion, section "Efficiency Evaluation") and define only
 * the forward ("PaTH Attention: ..." slides, frames "PaTH inserts a learned
 * transformation along every path", "FoX adds a separate mechanism for
 * forgetting"); these are the exact derivatives of that forward, taken
 * through its blockwise form (frames "A triangular representation makes paths
 * computable", "A right-to-left scan accumulates cross-block paths").
 *
 *   q, k, v, w, beta, logf, scale, B, H, T, d, dtype   as given to path_attn_fwd
 *   out   device, [B,H,T,d], dtype      the forward's output
 *   lse   device, [B,H,T], fp32         the forward's lse (required)
 *   dout  device, [B,H,T,d], dtype      dL/dout
 *   dlse  device, [B,H,T], fp32, or NULL (taken as zero)
 *   dq, dk, dv, dw   device, [B,H,T,d], dtype (written)
 *   dbeta device, [B,H,T], fp32 (written)
 *   dlogf device, [B,H,T], fp32 (written), required iff logf is not NULL
 * All arrays 16-byte aligned, outputs distinct from inputs.  The call reruns
 * the forward's chunk preparation, then walks every chunk pair; the walked
 * queries X_b^(c) and their gradients are kept for each pair c < b, so the
 * stream-ordered scratch from the library's pool grows as T^2 d / C
 * (path_attn_bwd_workspace_bytes reports it).  Errors as path_attn_fwd.
 */
int path_attn_bwd(const void* q, const void* k, const void* v, const void* w,
                  const float* beta, const float* logf, float scale, const void* out,
                  const float* lse, const void* dout, const float* dlse, void* dq, void* dk,
                  void* dv, void* dw, float* dbeta, float* dlogf, int B, int H, int T, int d,
                  int dtype, void* stream);

/* Bytes of stream-ordered scratch one path_attn_bwd call takes from the pool. */
int path_attn_bwd_workspace_bytes(int B, int H, int T, int d, int dtype, int with_gate,
                                  size_t* bytes);

/*
 * Decoding with keys rewritten in place (slides' frame "Decoding updates
 * historical keys in place").  A decoder keeps, per (b, h), a key cache in
 * which row j < t holds k_j carried to the latest token t - 1,
 * H_{t-1} ... H_{j+1} k_j, a value cache, and (PaTH-FoX) the gate prefix
 * lam_j = sum_{s<=j} log f_s.  Token t rewrites every cached key
 * k_j <- k_j - beta_t w_t (w_t^T k_j), appends k_t, v_t, lam_t, and reads out
 *   o_t = sum_{j<=t} softmax_j(scale * k_j^T q_t + lam_t - lam_j) v_j,
 * which equals row t of path_attn_fwd over tokens 0..t.
 *
 * Cache layout (caller-owned device memory, 16-byte aligned):
 *   kcache    [B,H,Tmax,d] fp32  (fp32 whatever dtype is: each key is rewritten
 *             once per later token, and rounding would compound)
 *   vcache    [B,H,Tmax,d] dtype
 *   lamcache  [B,H,Tmax]   fp32, natural log; used only with a gate (else NULL)
 *
 * path_attn_prefill -- path_attn_fwd over a prompt of T tokens (same
 * arguments and results) that also fills rows 0..T-1 of the caches: kcache
 * with every key carried to token T - 1, vcache with v, lamcache (iff logf is
 * not NULL) with the prefix sums.  Rows >= T are not touched.  Requires
 * T <= Tmax.  The cached keys come from the forward's chunk factors: the keys
 * of chunk c carried to the chunk end, times the product of the transitions of
 * the later chunks (frames "Backup: fix orientation before implementing UT
 * products" and "A right-to-left scan accumulates cross-block paths").
 */
int path_attn_prefill(const void* q, const void* k, const void* v, const void* w,
                      const float* beta, const float* logf, float scale, void* out,
                      float* lse, float* kcache, void* vcache, float* lamcache, int Tmax,
                      int B, int H, int T, int d, int dtype, void* stream);

/*
 * path_attn_decode_step -- one decoding step for every (b, h).
 *
 *   q, k, v, w  device, [B,H,d], dtype     the new token of each (b, h)
 *   beta        device, [B,H], fp32;  logf: device, [B,H], fp32, or NULL
 *   kcache, vcache, lamcache   as above; for batch row b, rows < pos[b] are
 *               the cache (rewritten in place), row pos[b] receives the new
 *               key, value and gate prefix.  lamcache is required iff logf is
 *               not NULL.
 *   pos         device, [B], int32: position t of the new token of batch row
 *               b (= its number of cached tokens); rows may differ
 *   max_len     host int, 1 <= max_len <= Tmax; every pos[b] must be below
 *               it.  It sizes the launch: the key cache is cut into spans
 *               covering rows [0, max_len - 1).
 *   out         device, [B,H,d], dtype;  lse: device, [B,H], fp32, or NULL
 *
 * One kernel launch on `stream` (after a memset of B*H ints) and a small
 * stream-ordered scratch ([B*H][spans][d+2] fp32 + B*H ints) from the
 * library's pool; the last CTA of each head merges that head's spans.  A pos[b] outside
 * [0, max_len) is only visible on the device: that batch row's out and lse
 * become NaN, its cache rows are left as they were, and
 * path_attn_device_status() then returns PATH_ERR_INVALID_ARG.
 */
int path_attn_decode_step(const void* q, const void* k, const void* v, const void* w,
                          const float* beta, const float* logf, float scale, float* kcache,
                          void* vcache, float* lamcache, const int* pos, int max_len,
                          void* out, float* lse, int B, int H, int Tmax, int d, int dtype,
                          void* stream);

/*
 * path_producer_fwd -- the producer of w and beta from the hidden states x
 * (slides' frame "PaTH inserts a learned transformation along every path":
 * low-rank projection, width-3 convolution, L2 normalization, beta = 2
 * sigmoid(u^T x + b); OpenReview section "Model Architecture Details": per
 * head, low-rank).  This library's readings of what the pages leave open:
 *   p_t  = Wu (Wd x_t)                      (no bias)
 *   z_t  = cw[:,0] p_{t-2} + cw[:,1] p_{t-1} + cw[:,2] p_t
 *          (per channel, causal, p = 0 before the sequence start, no activation)
 *   w_t  = z_t / max(|z_t|, 1e-12)          per head (d channels)
 *   beta_t[h] = 2 sigmoid(Ub[h] . x_t + bb[h])
 *
 *   x     device, [B,T,Dm], dtype           Wd: device, [R,Dm], dtype
 *   Wu    device, [H*d,R], dtype            cw: device, [H*d,3], fp32
 *   Ub    device, [H,Dm], dtype             bb: device, [H], fp32
 *   w     device, [B,H,T,d], dtype (out)    beta: device, [B,H,T], fp32 (out)
 * The outputs are laid out as path_attn_fwd's w and beta inputs.  Arrays
 * other than cw and bb must be 16-byte aligned.  Supported: d = 64 or 128;
 * Dm a multiple of 64 up to 32768; R a multiple of 16 up to 128; R + H up to
 * 128 (PATH_ERR_UNSUPPORTED otherwise).  Two kernel
 * launches and a [B*T][R] fp32 stream-ordered scratch from the library's pool.
 */
int path_producer_fwd(const void* x, const void* Wd, const void* Wu, const float* cw,
                      const void* Ub, const float* bb, void* w, float* beta, int B, int T,
                      int Dm, int H, int d, int R, int dtype, void* stream);

/* Human-readable name of a path_status_t value (static storage). */
const char* path_attn_status_string(int status);

/* Text of the last CUDA error seen by this thread inside the library (empty
 * if none); valid until the next call on this thread. */
const char* path_attn_last_error(void);

/* Library version: major*10000 + minor*100 + patch. */
int path_attn_version(void);

/*
 * Bytes of workspace path_attn_fwd takes for this problem (host arithmetic
 * only; touches no device).  Returns PATH_OK and writes *bytes, or an error
 * for invalid sizes.
 */
int path_attn_workspace_bytes(int B, int H, int T, int d, int dtype, int with_gate,
                              size_t* bytes);

/* Chunk length C used by the blockwise algorithm for (d, dtype): 128 for
 * bf16, 64 for fp32.  Returns a negative status for unsupported input. */
int path_attn_chunk_size(int d, int dtype);

/*
 * Device status word of `device` (0 = no error since the last clear; a
 * negative path_status_t otherwise: PATH_ERR_TIMEOUT if a kernel's bounded
 * wait expired, PATH_ERR_INVALID_ARG if path_attn_decode_step met a position
 * outside its bounds).  Synchronises that device first.  clear != 0 resets
 * the word.
 */
int path_attn_device_status(int device, int clear);

/*
 * Per-kernel timing with CUDA events recorded on the launch stream around each
 * kernel of path_attn_fwd.  path_attn_timing_enable(1) starts recording (and
 * clears the totals); path_attn_timing_read() synchronises on the recorded
 * events and returns the summed milliseconds of the chunk-preparation kernels
 * and of the attention kernel, and the number of path_attn_fwd calls timed.
 * Any output pointer may be NULL.  Timing off by default.
 */
int path_attn_timing_enable(int enable);
int path_attn_timing_read(double* prep_ms, double* attn_ms, long* calls);

/*
 * The same for path_attn_bwd (while timing is enabled): phase_ms[0..6]
 * receives the summed milliseconds of its seven phases, in launch order:
 * chunk preparation, the per-row D_i, the X walk, the key pass, the G walk,
 * the dF reduction, and the chunk pass with the gate scan (for fp32 inputs
 * the row kernels appear as one phase, the dF slot).  Either pointer may be
 * NULL; calls receives the number of path_attn_bwd calls timed.
 */
int path_attn_bwd_timing_read(double* phase_ms, long* calls);

/*
 * Number of kernel launches one path_attn_fwd call makes for this problem
 * (host arithmetic only).
 */
int path_attn_launches_per_call(int d, int dtype, int with_gate);

/* The same for one path_attn_bwd call at sequence length T (memsets not counted). */
int path_attn_bwd_launches_per_call(int T, int d, int dtype, int with_gate);

/*
 * path_attn_debug_factors -- diagnostics: run only the chunk preparation and
 * copy its per-chunk factors (frame "Backup: fix orientation before
 * implementing UT products") into caller buffers, for tests.  With C =
 * path_attn_chunk_size(d, dtype), Np = ceil(T / C), Tp = Np * C, BH = B * H:
 *   kr   [BH, Tp, d]    dtype  boundary-adjusted keys  k_j through H_{j+1}..H_last
 *   ql   [BH, Tp, d]    fp32   boundary-adjusted queries q_i through H_i..H_first
 *   ngt  [BH, Np, d, d] dtype  -(W^T U W)^T of each chunk (the transition is
 *                              q <- q + q ngt^T ... i.e. q^T F^T = q^T + q^T ngt^T)
 *   sdt  [BH, Np, C, C] fp32   intra-chunk log2-domain logits, transposed:
 *                              sdt[.., j, i] = log2(e) * (scale * At_ij + gate_ij)
 *                              for j <= i, -inf above the diagonal
 *   lam2 [BH, Tp]       fp32   log2(e) * cumulative sum of logf (NULL when
 *                              logf is NULL)
 * Tokens past T are padding with beta = 0.  Asynchronous on `stream`.
 */
int path_attn_debug_factors(const void* q, const void* k, const void* w, const float* beta,
                            const float* logf, float scale, int B, int H, int T, int d,
                            int dtype, void* kr, float* ql, void* ngt, float* sdt,
                            float* lam2, void* stream);

/*
 * path_attn_debug_wait_timeout -- diagnostics for the failure path: launches
 * on `stream` a one-thread kernel that waits, with the same bounded wait the
 * attention kernel uses, on a barrier nothing arrives at, for limit_ns
 * nanoseconds (1 .. 2e9).  The wait expires and the kernel records the
 * timeout in the device status word, which path_attn_device_status() then
 * reports as PATH_ERR_TIMEOUT (and clears).  Nothing faults; the context
 * stays usable.
 */
int path_attn_debug_wait_timeout(unsigned long long limit_ns, void* stream);

/*
 * path_attn_set_transition_form -- how the bf16 forward at d = 64 carries
 * the running query across a key chunk ("PaTH Attention ..." slides, frames
 * "A triangular representation makes paths computable" and "A right-to-left
 * scan accumulates cross-block paths": crossing chunk c multiplies the query
 * by I - W_c^T U_c W_c).  A library switch for measuring the two forms; they
 * compute the same values up to rounding.
 *   form 0 (default)  dense: q <- q + q ngt_c^T with the d x d matrix
 *                     ngt_c = -(W_c^T U_c W_c)^T from the preparation, fused
 *                     with the logits into one MMA of width C + d.
 *   form 1            low-rank, as the slides write it: q <- q - (q W_c^T)(U_c W_c):
 *                     [S | Y] = Qw [kr_c ; W_c]^T in one MMA of width 2C, Y
 *                     rounded to bf16 in shared memory, then Qm += Y (-(U W)_c)
 *                     (K = C); the preparation also stores -(U W)_c in bf16.
 * Other dtypes, d = 128 (where the low-rank form's tensor-memory operands, S,
 * Y, Qm, O, Qw and P, would need 640 of the 512 columns), partial PaTH, prefill
 * and path_attn_fwd_noalloc always use the dense form.  Process-wide; returns
 * PATH_ERR_INVALID_ARG for any other value.
 */
int path_attn_set_transition_form(int form);

/*
 * path_attn_fwd_noalloc -- path_attn_fwd for callers that cannot allocate
 * device memory.  The paper has no counterpart; this is a library interface.
 *
 * Some callers must not call cudaMalloc (or any allocating routine): a host
 * framework that has already reserved the device's memory for its own
 * allocator, where an extra allocation would fail or fragment that pool, or
 * a steady-state serving loop with a fixed memory budget.  This entry runs
 * the same kernels as path_attn_fwd but takes its workspace from a static
 * device array of PATH_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library, so
 * it allocates nothing.  The array belongs to the library's host-API module:
 * with lazy module loading (the CUDA default) only GPUs on which this entry
 * (or path_attn_noalloc_status) has been called hold it; under eager module
 * loading (CUDA_MODULE_LOADING=EAGER) every device on which the library
 * creates or uses a context holds it, whatever entry is called.  A GPU that
 * holds it keeps it until the process exits.
 *
 *   Arguments as path_attn_fwd, plus
 *   status  device int, or NULL: set to 0 at the start of the call, and to a
 *           non-zero value by a kernel whose bounded wait expired.  With
 *           NULL the kernels report into a second static word of the
 *           library, which path_attn_noalloc_status() reads.
 *
 * Problems whose workspace (path_attn_workspace_bytes) exceeds the array are
 * rejected with PATH_ERR_UNSUPPORTED before any launch; the message says how
 * many bytes were needed.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  All calls share the one array, which
 * keeps the last call's contents: calls that may overlap on the GPU (other
 * streams, other host threads) race on it and must be serialised by the
 * caller.  Asynchronous on `stream`.
 */
#define PATH_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int path_attn_fwd_noalloc(const void* q, const void* k, const void* v, const void* w,
                          const float* beta, const float* logf, float scale, void* out,
                          float* lse, int* status, int B, int H, int T, int d, int dtype,
                          void* stream);

/*
 * path_attn_noalloc_status -- reads the static status word that
 * path_attn_fwd_noalloc's kernels write when it was called with status NULL.
 * The paper has no counterpart; this is a library interface.
 *
 * Selects `device` for the call (the previous device is restored),
 * synchronises it, copies the word to the host and, if `clear` is non-zero,
 * resets it to 0.  Allocates nothing.  Returns PATH_OK when no bounded wait
 * expired since the word was last reset (every path_attn_fwd_noalloc call
 * with status NULL resets it at its start), PATH_ERR_TIMEOUT when one did,
 * PATH_ERR_UNSUPPORTED on a device other than sm_103a, PATH_ERR_CUDA on a
 * CUDA error.
 */
int path_attn_noalloc_status(int device, int clear);

#ifdef __cplusplus
}
#endif

#endif /* PATHATTN_H */
