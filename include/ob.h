/*
 * ob.h -- C ABI of the GB300 (sm_103a) library for the 1-bit Adam / APMSqueeze
 * compression-stage optimizer step.
 *
 * What the step computes (sources named by page title and section):
 *   - "1-bit Adam: Communication Efficient Large-Scale Training with Adam's Convergence
 *     Speed" (paper review), "Proposed method": Adam warm-up at full precision, then
 *     momentum SGD preconditioned by the variance frozen after the warm-up, with
 *     error-compensated 1-bit compression of the momentum.
 *   - "APMSqueeze: A Communication Efficient Adam-Preconditioned Momentum SGD
 *     Algorithm" (paper review), "Proposed method": m_t compressed, v_t frozen.
 *   - "DeepSpeed 1-bit Adam training guide" (tutorial page), §1 (one sign bit per
 *     value), §3.5 (exp_avg_mask), §4 (step() phases; compressed_allreduce with a
 *     worker_error and a server_error per GPU; update = exp_avg/(sqrt(exp_avg_sq)+eps)
 *     then weight decay and learning rate), §6.2 (bias_correction), §7 (errors reset
 *     when a checkpoint is loaded).
 *   - "LoCo: Low-Bit Communication Adaptor for Large-scale Model Training", "Method"
 *     (moving average of past compensation errors, low-bit compression, then sync).
 *
 * Data-parallel model. W workers are simulated as a leading batch dimension on one
 * GPU. The exchange of compressed momentum (worker -> server chunk, server -> every
 * worker) is a gather of packed words inside device memory: no inter-GPU collective.
 * Server j owns the elements [j*n/W, (j+1)*n/W).
 *
 * Conventions shared by every entry point:
 *   - n      elements of the flat parameter buffer; n % (W*256) == 0 (pad the buffer:
 *            pad elements with g = 0, x = 0, m = 0, v = 1 behave like any other), and
 *            W*n < 2^40 (every 256-element group of every row is numbered in 32 bits).
 *   - W      simulated workers, 1..16.
 *   - chunk  elements per scale; chunk % 256 == 0 and (n/W) % chunk == 0. Chunk k is
 *            elements [k*chunk, (k+1)*chunk), the same chunks for workers and servers.
 *   - Arrays are row-major; a [W][n] array holds worker w's row at offset w*n.
 *   - Device pointers must be 16-byte aligned (OB_EALIGN otherwise); the workspace
 *     256-byte aligned.
 *   - All device memory belongs to the caller. The library never allocates device
 *     memory; it keeps only the host-side context.
 *   - Every call is asynchronous on the given stream (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and returns without synchronizing, except where
 *     stated. Arguments are checked before anything is enqueued; a rejected call
 *     enqueues nothing. Launch failures map to OB_ECUDA.
 *   - A context is bound to the CUDA device current at ob_init and must be used with
 *     that device current. A context is not thread-safe.
 *   - Packed signs: bit t of 32-bit word k is element 32*k + t; the bit is 1 when the
 *     value is >= 0 (sign(0) = +1, -0.0 included).
 *   - Scales: one float per (row, chunk), the chunk's RMS sqrt(sum z^2 / chunk).
 *   - Arithmetic: float32 state; every element-wise operation is a single IEEE
 *     round-to-nearest float32 operation (no contraction into FMA), in the order the
 *     step is written below; chunk sums of squares are accumulated with compensation
 *     and combined in double in a fixed order, so results are deterministic.
 *
 * Error-buffer representation (read this before touching worker_err / server_err):
 *   to stream each buffer once per step, worker_err[w][i] stores the worker's
 *   pre-compression value z of the previous step and the workspace keeps that step's
 *   chunk scales S; the true residual is e = z - S*sign(z), rebuilt on the fly at the
 *   next step. server_err stores y likewise. All-zero buffers with a zeroed workspace
 *   mean "errors are zero". ob_export_state writes the true residuals.
 */
#ifndef OB_H
#define OB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ob_ctx ob_ctx;

enum {
    OB_OK = 0,
    OB_EINVAL = -1,   /* bad size, dtype, NULL pointer, or wrong device current */
    OB_ECUDA = -2,    /* a CUDA call or launch failed; ob_last_cuda_error() has the code */
    OB_ENOTIMPL = -3, /* valid request that this library does not implement */
    OB_EALIGN = -4,   /* a pointer is not aligned as required */
    OB_ESCRATCH = -5  /* problem too large for the fixed no-allocation scratch array */
};

enum { OB_F32 = 0, OB_F16 = 1, OB_BF16 = 2 };   /* gradient storage formats */

/* Kernel ids for ob_profile_read. OB_K_SCALES is the copy of a step's chunk scales into
 * the "previous" slots; it runs as a kernel of its own only when the scales are many
 * (short chunks), otherwise inside the update kernel. */
enum {
    OB_K_WORKER = 0, OB_K_SERVER = 1, OB_K_UPDATE = 2, OB_K_WARMUP = 3,
    OB_K_LOCO_ABSMAX = 4, OB_K_LOCO_QUANT = 5, OB_K_LOCO_SERVER = 6,
    OB_K_MASK = 7, OB_K_EXPORT = 8, OB_K_SCALES = 9, OB_K_COUNT = 10
};

/* ---- context ------------------------------------------------------------------------ */

/*
 * Create a context for an n-element buffer, W workers and `chunk` elements per scale,
 * with Adam's b1, b2, eps and the learning rate lr (weight decay 0, bias correction
 * off, as in the tutorial page's BERT configurations, §6.2). Queries the current
 * device and, when there is one, opts the worker and server kernels into the dynamic
 * shared memory they launch with on that device (OB_ECUDA if that fails); allocates host
 * memory only.
 * Contexts on different devices, or used from different host threads, are independent.
 * Returns OB_EINVAL for sizes outside the rules above or non-finite hyper-parameters;
 * *out is set only on OB_OK.
 */
int ob_init(int64_t n, int32_t W, int64_t chunk, float b1, float b2, float eps, float lr,
            ob_ctx **out);

/* Release the host context (and any profiling events). NULL is accepted. */
void ob_destroy(ob_ctx *ctx);

/*
 * Bytes of the device workspace the caller must provide to the 1-bit calls (packed
 * signs, scales, momentum-mask bits, partial sums, counters). The workspace holds
 * state between steps (the previous scales and the counters): zero it once before
 * first use (ob_workspace_init or a memset) and keep it with its error buffers.
 */
size_t ob_workspace_bytes(const ob_ctx *ctx);

/* Zero the whole workspace on the stream (a cudaMemsetAsync). */
int ob_workspace_init(ob_ctx *ctx, void *ws, void *stream);

int ob_set_lr(ob_ctx *ctx, float lr);

/*
 * Weight decay and bias correction, tutorial page §4 and §6.2. The update becomes
 * u = m/(sqrt(v)+eps) + weight_decay*x; x -= lr*u. With bias_correction != 0 the
 * warm-up step divides m and v by (1 - b1^t) and (1 - b2^t), t = the step count (see
 * ob_set_step); the compression stage keeps the frozen v unchanged and uses m as
 * received, matching the frozen-preconditioner update. Returns OB_EINVAL for a
 * negative or non-finite weight decay.
 */
int ob_set_options(ob_ctx *ctx, float weight_decay, int bias_correction);

/* Steps taken so far (each warm-up, compressed or LoCo call adds one). For resume. */
int ob_set_step(ob_ctx *ctx, int64_t step);
int64_t ob_get_step(const ob_ctx *ctx);

/*
 * Momentum mask, tutorial page §3.5: mask01 is a device float array [n] of 0/1; after
 * the compressed exchange, momentum is multiplied by it (positions with 0 keep zero
 * momentum; errors are not masked). Packs it into bits in the workspace. mask01 ==
 * NULL clears the mask. The mask is not part of any saved state (it is supplied again
 * on every run, §3.5).
 */
int ob_set_mask(ob_ctx *ctx, const float *mask01, void *ws, void *stream);

/* ---- steps ---------------------------------------------------------------------------- */

/*
 * Full-precision warm-up step (plain Adam), tutorial page §3.1 and §4; "1-bit Adam"
 * review, "Proposed method". grads [W][n] in `dtype`. With gbar = (sum over w of g_w)/W:
 *   m = b1*m + (1-b1)*gbar;  v = b2*v + (1-b2)*gbar^2;  x -= lr*(m/(sqrt(v)+eps) [+wd*x])
 * (bias correction as set by ob_set_options). Error buffers are not touched. ws is the
 * 1-bit workspace (only its launch bookkeeping is used).
 */
int ob_warmup_step(ob_ctx *ctx, const void *grads, int dtype, float *x, float *m, float *v,
                   void *ws, void *stream);

/*
 * Compression-stage step, tutorial page §3.5 and §4; "1-bit Adam" and "APMSqueeze"
 * reviews, "Proposed method". grads [W][n] in `dtype`; x, m [n] updated; v [n] read
 * only (frozen); worker_err [W][n] and server_err [n] in the representation described
 * at the top of this file. Per element i of chunk k:
 *   worker w:  p = b1*m + (1-b1)*g_w;  z = p + e_w;  S_wk = rms(z over chunk k);
 *              send sign(z), S_wk;  e_w = z - S_wk*sign(z)
 *   server:    a = (sum over w ascending of S_wk*sign_w)/W;  y = a + e_s;
 *              T_k = rms(y over chunk k);  send sign(y), T_k;  e_s = y - T_k*sign(y)
 *   all:       m = T_k*sign(y) [* mask];  x -= lr*(m/(sqrt(v)+eps) [+wd*x])
 * Three kernels on the stream: worker compress, server average/recompress, update; a
 * fourth (OB_K_SCALES) moves the step's chunk scales into the "previous" slots when
 * they are more than 4096 (short chunks), which the update does itself otherwise. They
 * are launched with programmatic dependent launch: each may be scheduled while the
 * kernel before it on the stream finishes, and waits for it before touching memory, so
 * stream order holds as for ordinary launches.
 */
int ob_compressed_step(ob_ctx *ctx, const void *grads, int dtype, float *x, float *m,
                       const float *v, float *worker_err, float *server_err, void *ws,
                       void *stream);

/*
 * The same step with the gradients in HOST memory: copies grads_host ([W][n] in dtype,
 * pinned for full speed) into the caller's device buffer grads_dev, runs the step, and
 * copies the step's compressed result -- the server's packed signs (n/32 words) and
 * scales (n/chunk floats), i.e. what every worker receives -- into sbits_host and
 * sscale_host. The host-to-device copy runs on a stream the context owns: it waits only
 * until no earlier worker pass of this context still reads grads_dev, and `stream` waits
 * for the copy before the step's kernels. So a caller that alternates two device
 * buffers between consecutive calls overlaps the next step's gradient copy with this
 * step's kernels. The copies back run on `stream`. The host buffers must stay valid
 * until `stream` has passed this call's work.
 */
int ob_compressed_step_host(ob_ctx *ctx, const void *grads_host, void *grads_dev, int dtype,
                            float *x, float *m, const float *v, float *worker_err,
                            float *server_err, void *ws, uint32_t *sbits_host,
                            float *sscale_host, void *stream);

/*
 * LoCo step, "LoCo" page, "Method". Per worker w and element i of chunk k:
 *   c = g_w + ratio*e~_w;  s_wk = max|c| over chunk / L;  q = clamp(rint(c/s_wk), -L, L)
 *   (q = 0 when s_wk = 0), L = 2^(bits-1) - 1;  e~_w = beta*e~_w + (1-beta)*(c - q*s_wk)
 * then gbar = (sum over w of q*s_wk)/W drives a plain Adam step on x, m, v (not
 * frozen). bits is 4 (two codes per byte, even element in the low nibble, two's
 * complement) or 8 (one signed byte). loco_err [W][n] float holds e~ (zero at start).
 * loco_ws must hold ob_loco_workspace_bytes(ctx, bits) bytes, zeroed before first use.
 * Chunks of up to 4096 elements are quantized in one pass that also finds their absmax
 * (profiled as OB_K_LOCO_QUANT; OB_K_LOCO_ABSMAX then records no launch), and a second
 * pass averages the codes and takes the Adam step (OB_K_LOCO_SERVER). Longer chunks take
 * a separate absmax pass first, then one pass that quantizes every worker's row and takes
 * the Adam step (profiled as OB_K_LOCO_QUANT; OB_K_LOCO_SERVER then records no launch);
 * its codes never leave the registers unless ob_set_loco_codes asks for them. The
 * results are the same either way. The scales are always stored in loco_ws.
 */
int ob_loco_step(ob_ctx *ctx, const void *grads, int dtype, float *x, float *m, float *v,
                 float *loco_err, float beta, int bits, void *loco_ws, void *stream);

/*
 * The LoCo compensation ratio ("LoCo" page, key design item 2: the proportion of the
 * compensation applied to the gradient is tuned per model and data): c = g + ratio*e~ in
 * ob_loco_step, ratio in [0, 1], 1 when never set (ratio 1 is the plain c = g + e~).
 * OB_EINVAL outside that range.
 */
int ob_set_loco_ratio(ob_ctx *ctx, float ratio);

/*
 * Whether ob_loco_step stores the codes in loco_ws (laid out as above, at the start of
 * the workspace) when the chunks are longer than 4096 elements: 0 (the default) keeps
 * them in registers, saving their W*bits/8 bytes per element of DRAM writes; 1 stores
 * them too, for inspection. Short chunks always store them. OB_EINVAL unless keep is 0
 * or 1.
 */
int ob_set_loco_codes(ob_ctx *ctx, int keep);
size_t ob_loco_workspace_bytes(const ob_ctx *ctx, int bits);

/* ---- state ----------------------------------------------------------------------------- */

/*
 * Reset both error buffers and the scales they depend on, as loading a checkpoint does
 * (tutorial page §7). worker_err [W][n] and server_err [n] are zeroed, and the
 * workspace's previous-scale slots too. The mask is kept.
 */
int ob_reset_errors(ob_ctx *ctx, float *worker_err, float *server_err, void *ws, void *stream);

/*
 * Write the true residuals: ew_out[w][i] = worker_err[w][i] - S*sign(worker_err[w][i])
 * and es_out[i] likewise with the server scales. For checkpoints and tests.
 */
int ob_export_state(ob_ctx *ctx, const float *worker_err, const float *server_err,
                    const void *ws, float *ew_out, float *es_out, void *stream);

/*
 * Device pointers into the workspace after a compressed step: worker signs [W][n/32],
 * worker scales [W][n/chunk], server signs [n/32], server scales [n/chunk]. Any output
 * pointer may be NULL. Enqueues nothing.
 */
int ob_debug_views(const ob_ctx *ctx, const void *ws, const uint32_t **wbits,
                   const float **wscale, const uint32_t **sbits, const float **sscale);

/* ---- measurement ------------------------------------------------------------------------ */

/*
 * With enable != 0, every kernel launch is bracketed by CUDA events recorded on the
 * launch stream. ob_profile_read synchronizes those events and reports, for one kernel
 * id, the summed duration in milliseconds and the launch count since profiling was
 * enabled (or last reset with ob_profile(ctx, 1)).
 */
int ob_profile(ob_ctx *ctx, int enable);
int ob_profile_read(ob_ctx *ctx, int kernel, double *total_ms, int64_t *launches);

/* Kernels this context has launched in total. */
int64_t ob_launch_count(const ob_ctx *ctx);

/*
 * Synchronize the stream, then copy the workspace's status word to *status: 0 when every
 * kernel finished normally; 1 when a kernel gave up waiting for a shared-memory pipeline
 * stage (every such wait is bounded, about two seconds). A non-zero status means the
 * step's outputs are not valid; re-initialise the workspace (ob_workspace_init) and the
 * error buffers before continuing.
 */
int ob_read_status(ob_ctx *ctx, const void *ws, unsigned *status, void *stream);

/*
 * Self-test of the failure detection above (the pages have no counterpart). Enqueues one
 * warp that waits, at most limit_ns nanoseconds (1 .. 2e9), on a shared-memory barrier
 * that nothing completes -- the situation of a pipeline stage whose copy never lands.
 * The wait runs out, the warp sets status 1 in the workspace's status word and returns;
 * nothing is copied, nothing faults, and the device stays usable. Read the result with
 * ob_read_status; ob_workspace_init clears it. With ws == NULL the warp sets the status
 * word of the no-allocation worker pass instead (read with ob_noalloc_read_status).
 * OB_EINVAL for a limit outside the range.
 */
int ob_selftest_wait(ob_ctx *ctx, void *ws, uint64_t limit_ns, void *stream);

/* Text for a status code; the last CUDA error number seen by this thread. */
const char *ob_strerror(int code);
int ob_last_cuda_error(void);

/* ---- a worker pass that allocates nothing ------------------------------------------------ */

/*
 * For callers that cannot allocate device memory themselves: a host runtime that
 * reserves all device memory up front and hands it out from its own arena (with no room
 * left for a separate workspace), or an embedding in which the caller has no device
 * allocator at all, only buffers that someone else owns.
 *
 * The pages have no counterpart of this entry point: it is a packaging of the worker
 * pass of ob_compressed_step (momentum, error compensation, sign packing and chunk
 * scales, the first of that step's three kernels), running the same kernel with the
 * same launch shape, so its outputs are bit-identical to that pass's.
 *
 * The caller passes every input and output; only the kernel's scratch (one double per
 * warp range, row and touched chunk, plus one arrival counter per chunk) lives in a
 * fixed array of OB_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU
 * that loads the library keeps until the process exits. Sizes whose scratch would not
 * fit -- many tiny chunks over a large buffer -- return OB_ESCRATCH and enqueue nothing.
 * The call itself never calls cudaMalloc, cudaFree or any allocating routine.
 *
 *   grads        [W][n] in dtype                    (input)
 *   m            [n] momentum of the previous step   (input)
 *   worker_err   [W][n] previous z in, this step's z out (the representation described
 *                at the top of this file)
 *   scale_prev   [W][n/chunk] scales of the previous step (input; zeros at the start)
 *   wbits        [W][n/32] packed signs               (output)
 *   scale_out    [W][n/chunk] this step's scales      (output)
 * An output that shares any byte with another of these buffers is rejected (OB_EINVAL).
 *
 * The scratch array is shared by every call in the process: calls whose kernels could
 * run at the same time on the GPU (different streams, or different host threads) race
 * on it and must be serialized by the caller. Each call clears the counters it needs
 * before its kernel runs; the rest of the array keeps whatever the last call left.
 *
 * The device address of the array is looked up (cudaGetSymbolAddress) by the first call
 * on each device, with that device current, and again whenever the device's context has
 * changed since (after a device reset the library's module may be loaded at another
 * address). Make that first call before any stream capture begins.
 *
 * Failures: a bounded pipeline wait that runs out (see ob_read_status) leaves this
 * call's outputs invalid and sets a status word kept in the array's last 256 bytes,
 * which no call clears. ob_noalloc_read_status synchronizes the stream, reports the word
 * (0: every such call since the last read finished normally; 1: a wait ran out) and
 * clears it.
 */
#define OB_NOALLOC_SCRATCH_BYTES (4u << 20)
int ob_worker_compress_noalloc(ob_ctx *ctx, const void *grads, int dtype, const float *m,
                               float *worker_err, const float *scale_prev, uint32_t *wbits,
                               float *scale_out, void *stream);
int ob_noalloc_read_status(ob_ctx *ctx, unsigned *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* OB_H */
