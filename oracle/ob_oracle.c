/*
 * CPU oracle for the 1-bit Adam / APMSqueeze compression-stage optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this
 * file: it exists so that tests, the package's smoke check and the benchmark's CPU
 * baseline can compare the CUDA kernels with a plain, slow, obviously correct
 * restatement of the method. It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Sources (the method as the pages state it):
 *  [1BA]  "1-bit Adam: Communication Efficient Large-Scale Training with Adam's
 *         Convergence Speed" (paper review), "Proposed method" bullets: full-precision
 *         Adam warm-up, then 1-bit compressed momentum SGD preconditioned by the
 *         variance frozen after the warm-up; error compensation on the momentum.
 *  [APM]  "APMSqueeze: A Communication Efficient Adam-Preconditioned Momentum SGD
 *         Algorithm" (paper review), "Proposed method": m_t is compressed, v_t frozen.
 *  [DS]   "DeepSpeed 1-bit Adam 训练优化 ... 完整配置指南" (tutorial page), sections
 *         §1 (one sign bit per value), §3.5 (exp_avg_mask), §4 (step() phases,
 *         compressed_allreduce with worker_error / server_error, update formula),
 *         §6.2 (bias_correction false, weight_decay), §7 (errors reset on load).
 *  [LoCo] "LoCo: Low-Bit Communication Adaptor for Large-scale Model Training",
 *         "Method" (moving average of past compensation errors compensates the
 *         gradient before low-bit compression, then synchronisation).
 *
 * Details the pages leave open, and the reading taken here:
 *  - scale of a chunk: its RMS, sqrt(sum z^2 / C), summed in double over ascending
 *    indices and rounded once to float; sign(0) = +1, i.e. the bit is (z >= 0.0f);
 *  - the residual uses the transmitted sign: e = z - S*sign(z);
 *  - the server averages the W decompressed workers: (sum over w ascending) / W;
 *  - one scale per chunk of C consecutive elements, the same chunks on the worker and
 *    the server side; the chunk of element i is i / C;
 *  - all state is float32, every operation a single IEEE float32 operation with
 *    round-to-nearest-even in the order written (the file must be compiled with
 *    -ffp-contract=off and without fast-math); reductions are in double;
 *  - weight decay is added to the update before the learning rate
 *    (u <- u + wd*x; x <- x - lr*u); bias correction (warm-up only) divides m and v by
 *    (1 - b^t) with the factors given by the caller;
 *  - LoCo: c = g + ratio*e~ (ratio: the share of the averaged error compensated into
 *    the gradient, a knob tuned per model and data ["LoCo", key design 2]; 1 by
 *    default), s = absmax(c over chunk)/L, q = clamp(rint(c/s), -L, L) with
 *    L = 2^(bits-1) - 1 (q = 0 when s = 0), e = c - q*s, e~ <- beta*e~ + (1-beta)*e,
 *    then an (unfrozen) Adam step on the mean of the dequantized gradients.
 *
 * Bit layout of packed signs: bit t of 32-bit word k is element 32*k + t.
 * LoCo 4-bit codes: two codes per byte, element 2j in the low nibble, two's complement.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_F32 0
#define ORA_F16 1
#define ORA_BF16 2

/* ---- gradient storage formats ------------------------------------------------ */

/* IEEE 754 binary16 -> binary32. Every binary16 value is exactly representable. */
static float ora_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    float mag;
    if (expo == 0) {
        mag = ldexpf((float)frac, -24);                 /* zero or subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(frac + 1024), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of a binary32 word. */
static float ora_bf16_to_float(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

static float ora_grad(const void *g, int dtype, int64_t idx)
{
    if (dtype == ORA_F16) return ora_half_to_float(((const uint16_t *)g)[idx]);
    if (dtype == ORA_BF16) return ora_bf16_to_float(((const uint16_t *)g)[idx]);
    return ((const float *)g)[idx];
}

/* Exported so that the tests can check the decoders against numpy's casts. */
void ora_decode_grads(const void *g, int dtype, int64_t count, float *out)
{
    for (int64_t i = 0; i < count; ++i) out[i] = ora_grad(g, dtype, i);
}

/* ---- the 1-bit compressor [DS §1, §4] ------------------------------------------ */

/* sign(0) = +1: the transmitted bit is 1 exactly when z >= 0 (so -0.0 also gives 1). */
static int ora_sign_bit(float z)
{
    return z >= 0.0f;
}

static float ora_signed(float scale, int bit)
{
    return bit ? scale : -scale;
}

/* RMS of one chunk: sqrt(sum z^2 / C), the sum in double over ascending index. */
float ora_chunk_scale(const float *z, int64_t C)
{
    double sum = 0.0;
    for (int64_t i = 0; i < C; ++i) sum += (double)z[i] * (double)z[i];
    return (float)sqrt(sum / (double)C);
}

/* Pack n signs (n a multiple of 32) into n/32 words. */
void ora_pack_signs(const float *z, int64_t n, uint32_t *words)
{
    for (int64_t k = 0; k < n / 32; ++k) {
        uint32_t word = 0;
        for (int t = 0; t < 32; ++t)
            if (ora_sign_bit(z[32 * k + t])) word |= (uint32_t)1 << t;
        words[k] = word;
    }
}

/* Decompress: element i is +scale or -scale of its chunk by its sign bit. */
void ora_unpack(const uint32_t *words, const float *scales, int64_t n, int64_t C, float *out)
{
    for (int64_t i = 0; i < n; ++i) {
        int bit = (int)((words[i / 32] >> (i % 32)) & 1u);
        out[i] = ora_signed(scales[i / C], bit);
    }
}

/*
 * Compress n values in chunks of C: sign bits, one scale per chunk, and the residual
 * that the compression discards (resid = z - S*sign), which becomes the new error.
 */
void ora_onebit_compress(const float *z, int64_t n, int64_t C,
                         uint32_t *words, float *scales, float *resid)
{
    for (int64_t k = 0; k < n / C; ++k) scales[k] = ora_chunk_scale(z + k * C, C);
    ora_pack_signs(z, n, words);
    for (int64_t i = 0; i < n; ++i)
        resid[i] = z[i] - ora_signed(scales[i / C], ora_sign_bit(z[i]));
}

/* ---- the preconditioned update [DS §4; 1BA "Proposed method"] -------------------- */

/* u = m / (sqrt(v) + eps); u += wd*x; x -= lr*u. */
static float ora_apply_update(float x, float m, float v, float eps, float lr, float wd)
{
    float denom = sqrtf(v) + eps;
    float u = m / denom;
    if (wd != 0.0f) {
        float decay = wd * x;
        u = u + decay;
    }
    float delta = lr * u;
    return x - delta;
}

/* ---- compression-stage step [DS §3.5, §4; 1BA; APM] ----------------------------- *
 *
 * Inputs: grads [W][n] (dtype), x, m, v [n] float, worker_err [W][n], server_err [n]
 * (canonical errors, zero at the first compressed step), mask [n] bytes (0/1) or NULL.
 * Outputs (all caller-allocated): the pre-compression buffers z [W][n], worker words
 * [W][n/32], worker scales [W][n/C], the server's pre-compression buffer y [n], server
 * words [n/32], server scales [n/C]. x, m, worker_err and server_err are updated in
 * place; v is read only (frozen after the warm-up).
 *
 * identity != 0 replaces both compressions by the identity (send z exactly, zero
 * residual): the uncompressed reference point of the method.
 */
int ora_compressed_step(int64_t n, int32_t W, int64_t C,
                        float b1, float eps, float lr, float wd,
                        const void *grads, int dtype,
                        float *x, float *m, const float *v,
                        float *worker_err, float *server_err,
                        const uint8_t *mask, int identity,
                        float *z, uint32_t *wwords, float *wscales,
                        float *y, uint32_t *swords, float *sscales)
{
    if (n <= 0 || W <= 0 || C <= 0 || n % 32 != 0 || n % C != 0) return -1;
    const float c1 = 1.0f - b1;
    const int64_t nchunks = n / C;

    /* worker side: momentum of this worker's gradient, plus its error, then compress */
    for (int32_t w = 0; w < W; ++w) {
        float *zw = z + (int64_t)w * n;
        float *ew = worker_err + (int64_t)w * n;
        for (int64_t i = 0; i < n; ++i) {
            float g = ora_grad(grads, dtype, (int64_t)w * n + i);
            float old_part = b1 * m[i];
            float new_part = c1 * g;
            float p = old_part + new_part;      /* exp_avg.mul_(b1).add_(1-b1, grad) */
            zw[i] = p + ew[i];                  /* error compensation on the momentum */
        }
        if (identity) {
            for (int64_t k = 0; k < nchunks; ++k) wscales[(int64_t)w * nchunks + k] = 0.0f;
            ora_pack_signs(zw, n, wwords + (int64_t)w * (n / 32));
            for (int64_t i = 0; i < n; ++i) ew[i] = 0.0f;
        } else {
            ora_onebit_compress(zw, n, C, wwords + (int64_t)w * (n / 32),
                                wscales + (int64_t)w * nchunks, ew);
        }
    }

    /* server side: average the W decompressed workers, add the server error, compress */
    for (int64_t i = 0; i < n; ++i) {
        float acc = 0.0f;
        for (int32_t w = 0; w < W; ++w) {
            float sent;
            if (identity) {
                sent = z[(int64_t)w * n + i];
            } else {
                int bit = (int)((wwords[(int64_t)w * (n / 32) + i / 32] >> (i % 32)) & 1u);
                sent = ora_signed(wscales[(int64_t)w * nchunks + i / C], bit);
            }
            acc = acc + sent;
        }
        float avg = acc / (float)W;
        y[i] = avg + server_err[i];
    }
    float *mom = (float *)malloc((size_t)n * sizeof(float));
    if (!mom) return -2;
    if (identity) {
        for (int64_t k = 0; k < nchunks; ++k) sscales[k] = 0.0f;
        ora_pack_signs(y, n, swords);
        for (int64_t i = 0; i < n; ++i) {
            mom[i] = y[i];
            server_err[i] = 0.0f;
        }
    } else {
        ora_onebit_compress(y, n, C, swords, sscales, server_err);
        ora_unpack(swords, sscales, n, C, mom);
    }

    /* every worker receives the same averaged momentum: it replaces exp_avg */
    for (int64_t i = 0; i < n; ++i) {
        float mi = mom[i];
        if (mask) {
            float keep = mask[i] ? 1.0f : 0.0f;
            mi = mi * keep;                     /* exp_avg.mul_(exp_avg_mask) [DS §3.5] */
        }
        m[i] = mi;
        x[i] = ora_apply_update(x[i], mi, v[i], eps, lr, wd);
    }
    free(mom);
    return 0;
}

/* ---- full-precision warm-up step (plain Adam) [DS §3.1, §4; 1BA; APM] ----------- *
 *
 * The W gradients are averaged (the full-precision AllReduce), then Adam updates m, v
 * and x. bc1 and bc2 are the bias-correction divisors (1 - b1^t, 1 - b2^t) or 1 when
 * bias correction is off. Errors are not touched.
 */
int ora_warmup_step(int64_t n, int32_t W, float b1, float b2, float eps, float lr, float wd,
                    float bc1, float bc2, const void *grads, int dtype,
                    float *x, float *m, float *v)
{
    if (n <= 0 || W <= 0) return -1;
    const float c1 = 1.0f - b1;
    const float c2 = 1.0f - b2;
    const int corrected = (bc1 != 1.0f) || (bc2 != 1.0f);
    for (int64_t i = 0; i < n; ++i) {
        float acc = 0.0f;
        for (int32_t w = 0; w < W; ++w) acc = acc + ora_grad(grads, dtype, (int64_t)w * n + i);
        float gbar = acc / (float)W;

        float m_old = b1 * m[i];
        float m_new = c1 * gbar;
        m[i] = m_old + m_new;

        float sq = gbar * gbar;
        float v_old = b2 * v[i];
        float v_new = c2 * sq;
        v[i] = v_old + v_new;

        float mh = m[i], vh = v[i];
        if (corrected) {
            mh = mh / bc1;
            vh = vh / bc2;
        }
        x[i] = ora_apply_update(x[i], mh, vh, eps, lr, wd);
    }
    return 0;
}

/* ---- LoCo low-bit step [LoCo "Method"] ------------------------------------------ *
 *
 * loco_err [W][n] holds each worker's moving average of past compensation errors.
 * Per worker: compensate the gradient with `ratio` times that average (LoCo page, key
 * design item 2: the proportion of compensation is tuned), quantize per chunk to
 * `bits`-bit signed codes with an absmax
 * scale, update the moving average with this step's compression error. Then the mean
 * of the W dequantized gradients drives a plain Adam step (m, v and x updated).
 * codes: [W][n*bits/8] bytes (bits = 4: two codes per byte, even element in the low
 * nibble; bits = 8: one signed byte per element); scales [W][n/C].
 */
int ora_loco_step(int64_t n, int32_t W, int64_t C, int bits,
                  float b1, float b2, float eps, float lr, float wd, float beta, float ratio,
                  const void *grads, int dtype,
                  float *x, float *m, float *v, float *loco_err,
                  uint8_t *codes, float *scales)
{
    if (n <= 0 || W <= 0 || C <= 0 || n % C != 0 || n % 2 != 0) return -1;
    if (bits != 4 && bits != 8) return -3;
    const int levels = (1 << (bits - 1)) - 1;
    const float flevels = (float)levels;
    const float keep = 1.0f - beta;
    const int64_t nchunks = n / C;
    const int64_t code_bytes = n * bits / 8;
    float *c = (float *)malloc((size_t)n * sizeof(float));
    int8_t *q = (int8_t *)malloc((size_t)W * (size_t)n);
    if (!c || !q) {
        free(c);
        free(q);
        return -2;
    }

    for (int32_t w = 0; w < W; ++w) {
        float *et = loco_err + (int64_t)w * n;
        int8_t *qw = q + (int64_t)w * n;
        for (int64_t i = 0; i < n; ++i) {
            float comp = ratio * et[i];
            c[i] = ora_grad(grads, dtype, (int64_t)w * n + i) + comp;
        }
        for (int64_t k = 0; k < nchunks; ++k) {
            float amax = 0.0f;
            for (int64_t i = k * C; i < (k + 1) * C; ++i) {
                float a = fabsf(c[i]);
                if (a > amax) amax = a;
            }
            float s = amax / flevels;
            scales[(int64_t)w * nchunks + k] = s;
            for (int64_t i = k * C; i < (k + 1) * C; ++i) {
                int qi = 0;
                if (s > 0.0f) {
                    float r = rintf(c[i] / s);
                    if (r > flevels) r = flevels;
                    if (r < -flevels) r = -flevels;
                    qi = (int)r;
                }
                qw[i] = (int8_t)qi;
                float deq = (float)qi * s;
                float e = c[i] - deq;
                float old_part = beta * et[i];
                float new_part = keep * e;
                et[i] = old_part + new_part;
            }
        }
        uint8_t *cw = codes + (int64_t)w * code_bytes;
        if (bits == 8) {
            for (int64_t i = 0; i < n; ++i) cw[i] = (uint8_t)qw[i];
        } else {
            for (int64_t j = 0; j < n / 2; ++j)
                cw[j] = (uint8_t)(((uint8_t)qw[2 * j] & 0x0f) | (((uint8_t)qw[2 * j + 1] & 0x0f) << 4));
        }
    }

    const float c1 = 1.0f - b1;
    const float c2 = 1.0f - b2;
    for (int64_t i = 0; i < n; ++i) {
        float acc = 0.0f;
        for (int32_t w = 0; w < W; ++w) {
            float deq = (float)q[(int64_t)w * n + i] * scales[(int64_t)w * nchunks + i / C];
            acc = acc + deq;
        }
        float gbar = acc / (float)W;
        float m_old = b1 * m[i];
        float m_new = c1 * gbar;
        m[i] = m_old + m_new;
        float sq = gbar * gbar;
        float v_old = b2 * v[i];
        float v_new = c2 * sq;
        v[i] = v_old + v_new;
        x[i] = ora_apply_update(x[i], m[i], v[i], eps, lr, wd);
    }
    free(c);
    free(q);
    return 0;
}
