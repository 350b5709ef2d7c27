// C ABI of the compression-stage library: argument checks, workspace layout, launch
// configuration and launches on the caller's stream. See include/ob.h for the contract.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/ob.h"
#include "ob_internal.h"
#include "ob_tma.cuh"

using namespace ob;

namespace {

thread_local int g_last_cuda = 0;

constexpr size_t kAlignWs = 256;
// LoCo chunks up to this many elements take the one-pass absmax + quantize kernel: the
// chunks its warps hold in flight together (a few tens of MB) stay in the L2 between
// their two reads.
constexpr int64_t kLocoOnePassMaxChunk = 4096;
constexpr int kWarpsPerBlock = kBlock / 32;

size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
    size_t wbits, sbits, mask, s_prev, s_next, t_prev, t_next, wpart, spart, wcnt, scnt, status, total;
};

struct Rec {
    int kernel;
    cudaEvent_t a, b;
};

}  // namespace

struct ob_ctx {
    int64_t n = 0, C = 0, nchunks = 0;
    int W = 0;
    float b1 = 0, b2 = 0, eps = 0, lr = 0, wd = 0;
    float loco_ratio = 1.0f;    // LoCo: share of the averaged error compensated into g
    bool loco_codes = false;    // LoCo, long chunks: also store the codes
    int bias_correction = 0;
    int64_t step = 0;
    int device = -1;
    int sms = 152;
    int smem_budget = 232448;   // opt-in shared memory per block
    Part ptw[3]{};              // worker partition per gradient type
    int wpr[3]{};               // worker warps per range (warps per block, or 1)
    Part pts{};                 // server partition
    int grid_s = 0;
    int grid_u = 0;             // update kernel: one resident wave
    int loco_occ_a[3] = {};     // resident blocks per SM of the LoCo absmax pass (per gradient type)
    int loco_occ_f[3][2] = {};  // the same for the one-pass short-chunk kernel (and code width)
    int loco_occ_qs[3][2] = {}; // and for the long-chunk quantize + server kernel (0 = not asked)
    Layout lay{};
    bool has_mask = false;
    int64_t launches = 0;
    bool profiling = false;
    std::vector<Rec> recs;
    std::vector<cudaEvent_t> spare;
    double prof_ms[OB_K_COUNT] = {};
    int64_t prof_n[OB_K_COUNT] = {};
    // host-gradient path: a copy stream, an event for "copy landed", and per device
    // gradient buffer an event recorded after the last worker pass that read it
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t copied = nullptr;
    std::vector<std::pair<const void*, cudaEvent_t>> buffer_read;
};

namespace {

int cuda_fail(cudaError_t e)
{
    g_last_cuda = (int)e;
    return OB_ECUDA;
}

int check_ptr(const void* p, size_t align)
{
    if (!p) return OB_EINVAL;
    if (reinterpret_cast<uintptr_t>(p) % align) return OB_EALIGN;
    return OB_OK;
}

// The device the context was created on must be current.
int check_device(const ob_ctx* c)
{
    int d = -1;
    const cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return cuda_fail(e);
    return d == c->device ? OB_OK : OB_EINVAL;
}

cudaEvent_t take_event(ob_ctx* c)
{
    if (!c->spare.empty()) {
        cudaEvent_t e = c->spare.back();
        c->spare.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Launch wrapper: counts launches and, when profiling, brackets them with events.
template <typename F>
int launch(ob_ctx* c, int kernel, cudaStream_t s, F&& f)
{
    cudaEvent_t a = nullptr, b = nullptr;
    if (c->profiling) {
        a = take_event(c);
        b = take_event(c);
        if (a && b) cudaEventRecord(a, s);
    }
    const cudaError_t e = f();
    if (e != cudaSuccess) return cuda_fail(e);
    ++c->launches;
    if (a && b) {
        cudaEventRecord(b, s);
        c->recs.push_back(Rec{kernel, a, b});
    }
    return OB_OK;
}

int stream_grid(const ob_ctx* c) { return c->sms * 8; }

// Worker/server grids: all resident blocks, rounded down to a power of two per SM so
// that P (a multiple of the SM count times a power of two) splits evenly over warps.
int pow2_floor(int v)
{
    int p = 1;
    while (p * 2 <= v) p *= 2;
    return v < 1 ? 1 : p;
}

Layout make_layout(int64_t n, int W, int64_t nch, int64_t wpart_doubles, int64_t spart_doubles)
{
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = up(off + bytes, kAlignWs);
        return at;
    };
    L.wbits = take((size_t)W * (n / 8));
    L.sbits = take((size_t)n / 8);
    L.mask = take((size_t)n / 8);
    L.s_prev = take((size_t)W * nch * 4);
    L.s_next = take((size_t)W * nch * 4);
    L.t_prev = take((size_t)nch * 4);
    L.t_next = take((size_t)nch * 4);
    L.wpart = take((size_t)wpart_doubles * 8);
    L.spart = take((size_t)spart_doubles * 8);
    L.wcnt = take((size_t)nch * 4);
    L.scnt = take((size_t)nch * 4);
    L.status = take(4);
    L.total = off;
    return L;
}

template <typename T>
T* at(void* ws, size_t off)
{
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

int check_grads(const ob_ctx* c, const void* g, int dtype)
{
    if (dtype != OB_F32 && dtype != OB_F16 && dtype != OB_BF16) return OB_EINVAL;
    return check_ptr(g, 16);
}

int grad_bytes(int dtype) { return dtype == OB_F32 ? 4 : 2; }

// P contiguous ranges of 256-element groups (at most one per group), and J, the most
// chunks any one range touches.
Part make_part(int64_t n, int64_t chunk, int64_t want)
{
    Part pt{};
    pt.NG = n / 256;
    pt.CG = chunk / 256;
    pt.nchunks = n / chunk;
    pt.P = want < pt.NG ? (want < 1 ? 1 : want) : pt.NG;
    int64_t J = 1;
    for (int64_t q = 0; q < pt.P; ++q) {
        const int64_t g0 = q * pt.NG / pt.P, g1 = (q + 1) * pt.NG / pt.P;
        const int64_t span = (g1 - 1) / pt.CG - g0 / pt.CG + 1;
        if (span > J) J = span;
    }
    pt.J = J;
    return pt;
}

bool finite(float v) { return std::isfinite(v); }

// The no-allocation path's scratch array (defined at the end of this file).
constexpr size_t kNoallocStatusOff = OB_NOALLOC_SCRATCH_BYTES - 256;   // its status word
int noalloc_scratch(int dev, void** out);

}  // namespace

extern "C" {

int ob_init(int64_t n, int32_t W, int64_t chunk, float b1, float b2, float eps, float lr,
            ob_ctx** out)
{
    if (!out) return OB_EINVAL;
    if (W < 1 || W > 16 || n <= 0 || chunk <= 0) return OB_EINVAL;
    if (n % ((int64_t)W * 256) != 0) return OB_EINVAL;
    if (chunk % 256 != 0 || (n / W) % chunk != 0) return OB_EINVAL;
    if ((int64_t)W * (n / 256) >= (1ll << 32)) return OB_EINVAL;   // group indices fit 32 bits
    if (!finite(b1) || !finite(b2) || !finite(eps) || !finite(lr)) return OB_EINVAL;
    if (b1 < 0.0f || b1 >= 1.0f || b2 < 0.0f || b2 >= 1.0f || eps < 0.0f) return OB_EINVAL;

    ob_ctx* c = new (std::nothrow) ob_ctx();
    if (!c) return OB_EINVAL;
    c->n = n;
    c->W = W;
    c->C = chunk;
    c->nchunks = n / chunk;
    c->b1 = b1;
    c->b2 = b2;
    c->eps = eps;
    c->lr = lr;

    // Device facts; on a machine without a GPU the context can still be created (for
    // argument checks), sized for a 152-SM part, and every launch will fail.
    int dev = -1, sms = 0, smem = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0 &&
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess) {
        c->device = dev;
        c->sms = sms;
        c->smem_budget = smem;
    } else {
        cudaGetLastError();
        c->device = -1;
        c->sms = 152;
        c->smem_budget = 232448;
    }
    // the worker kernels' shared-memory opt-in is a per-context property of the device:
    // set here, for this device, so contexts on several devices (and host threads) each
    // have it without a process-wide flag
    if (c->device >= 0) {
        cudaError_t e = prepare_worker(W, c->smem_budget);
        if (e == cudaSuccess) e = prepare_server(W);
        if (e == cudaSuccess) e = prepare_loco();
        if (e != cudaSuccess) {
            delete c;
            return cuda_fail(e);
        }
    }
    // worker: one block per SM, one range per block
    int64_t wpart = 0;
    for (int dt = 0; dt < 3; ++dt) {
        const WorkerConfig wc = worker_config(W, dt, c->smem_budget);
        // one range per block with interleaved warps while a block range spans at most a
        // couple of chunks; one range per warp for short chunks
        Part blocks = make_part(n, chunk, (int64_t)c->sms);
        if (blocks.J <= 2) {
            c->ptw[dt] = blocks;
            c->wpr[dt] = wc.warps_per_block;
        } else {
            c->ptw[dt] = make_part(n, chunk, (int64_t)c->sms * wc.warps_per_block);
            c->wpr[dt] = 1;
        }
        const int64_t need = (int64_t)W * c->ptw[dt].P * c->wpr[dt] * c->ptw[dt].J;
        if (need > wpart) wpart = need;
    }
    // server: all resident blocks, a power of two per SM
    int occ = c->device >= 0 ? occupancy_server(W) : 0;
    occ = pow2_floor(occ > 0 ? occ : 2);
    c->grid_s = c->sms * occ;
    // one range per warp, but at least four groups per range: on small buffers fewer,
    // longer ranges leave fewer partials to combine per chunk (measured faster)
    const int64_t srv_ranges = (int64_t)c->grid_s * kWarpsPerBlock;
    const int64_t srv_cap = (n / 256) / 4 > 0 ? (n / 256) / 4 : 1;
    c->pts = make_part(n, chunk, srv_ranges < srv_cap ? srv_ranges : srv_cap);
    const int occ_u = c->device >= 0 ? occupancy_update() : 0;
    c->grid_u = c->sms * (occ_u > 0 ? occ_u : 2);
    c->lay = make_layout(n, W, c->nchunks, wpart, c->pts.P * c->pts.J);
    *out = c;
    return OB_OK;
}

void ob_destroy(ob_ctx* c)
{
    if (!c) return;
    for (auto& r : c->recs) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    for (auto e : c->spare) cudaEventDestroy(e);
    for (auto& b : c->buffer_read) cudaEventDestroy(b.second);
    if (c->copied) cudaEventDestroy(c->copied);
    if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
    delete c;
}

size_t ob_workspace_bytes(const ob_ctx* c) { return c ? c->lay.total : 0; }

int ob_workspace_init(ob_ctx* c, void* ws, void* stream)
{
    if (!c) return OB_EINVAL;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    const cudaError_t e = cudaMemsetAsync(ws, 0, c->lay.total, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    c->has_mask = false;
    return OB_OK;
}

int ob_set_lr(ob_ctx* c, float lr)
{
    if (!c || !finite(lr)) return OB_EINVAL;
    c->lr = lr;
    return OB_OK;
}

int ob_set_options(ob_ctx* c, float weight_decay, int bias_correction)
{
    if (!c || !finite(weight_decay) || weight_decay < 0.0f) return OB_EINVAL;
    c->wd = weight_decay;
    c->bias_correction = bias_correction ? 1 : 0;
    return OB_OK;
}

int ob_set_loco_ratio(ob_ctx* c, float ratio)
{
    if (!c || !finite(ratio) || ratio < 0.0f || ratio > 1.0f) return OB_EINVAL;
    c->loco_ratio = ratio;
    return OB_OK;
}

int ob_set_loco_codes(ob_ctx* c, int keep)
{
    if (!c || (keep != 0 && keep != 1)) return OB_EINVAL;
    c->loco_codes = keep != 0;
    return OB_OK;
}

int ob_set_step(ob_ctx* c, int64_t step)
{
    if (!c || step < 0) return OB_EINVAL;
    c->step = step;
    return OB_OK;
}

int64_t ob_get_step(const ob_ctx* c) { return c ? c->step : -1; }

int ob_set_mask(ob_ctx* c, const float* mask01, void* ws, void* stream)
{
    if (!c) return OB_EINVAL;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    if (mask01 == nullptr) {
        c->has_mask = false;
        return OB_OK;
    }
    if (int r = check_ptr(mask01, 16)) return r;
    if (int r = check_device(c)) return r;
    MaskArgs a{mask01, at<uint32_t>(ws, c->lay.mask), c->n};
    const cudaStream_t s = (cudaStream_t)stream;
    if (int r = launch(c, OB_K_MASK, s, [&] { return launch_mask(a, stream_grid(c), s); })) return r;
    c->has_mask = true;
    return OB_OK;
}

int ob_warmup_step(ob_ctx* c, const void* grads, int dtype, float* x, float* m, float* v, void* ws,
                   void* stream)
{
    if (!c) return OB_EINVAL;
    if (int r = check_grads(c, grads, dtype)) return r;
    for (const void* p : {(const void*)x, (const void*)m, (const void*)v})
        if (int r = check_ptr(p, 16)) return r;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    const int64_t t = c->step + 1;
    WarmupArgs a{};
    a.g = grads;
    a.x = x;
    a.m = m;
    a.v = v;
    a.n = c->n;
    a.W = c->W;
    a.b1 = c->b1;
    a.c1 = 1.0f - c->b1;
    a.b2 = c->b2;
    a.c2 = 1.0f - c->b2;
    a.eps = c->eps;
    a.lr = c->lr;
    a.wd = c->wd;
    a.bc1 = 1.0f;
    a.bc2 = 1.0f;
    a.corrected = 0;
    if (c->bias_correction) {
        // (1 - b^t) in double, rounded once to float32
        a.bc1 = (float)(1.0 - std::pow((double)c->b1, (double)t));
        a.bc2 = (float)(1.0 - std::pow((double)c->b2, (double)t));
        a.corrected = (a.bc1 != 1.0f || a.bc2 != 1.0f) ? 1 : 0;
    }
    const cudaStream_t s = (cudaStream_t)stream;
    if (int r = launch(c, OB_K_WARMUP, s, [&] { return launch_warmup(dtype, a, stream_grid(c), s); })) return r;
    c->step = t;
    return OB_OK;
}

static int compressed_step_impl(ob_ctx* c, const void* grads, int dtype, float* x, float* m,
                                const float* v, float* worker_err, float* server_err, void* ws,
                                void* stream, cudaEvent_t after_worker);

int ob_compressed_step(ob_ctx* c, const void* grads, int dtype, float* x, float* m, const float* v,
                       float* worker_err, float* server_err, void* ws, void* stream)
{
    return compressed_step_impl(c, grads, dtype, x, m, v, worker_err, server_err, ws, stream, nullptr);
}

static int compressed_step_impl(ob_ctx* c, const void* grads, int dtype, float* x, float* m,
                                const float* v, float* worker_err, float* server_err, void* ws,
                                void* stream, cudaEvent_t after_worker)
{
    if (!c) return OB_EINVAL;
    if (int r = check_grads(c, grads, dtype)) return r;
    for (const void* p : {(const void*)x, (const void*)m, (const void*)v, (const void*)worker_err,
                          (const void*)server_err})
        if (int r = check_ptr(p, 16)) return r;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    const cudaStream_t s = (cudaStream_t)stream;
    const Layout& L = c->lay;

    WorkerArgs wa{};
    wa.g = grads;
    wa.m = m;
    wa.zbuf = worker_err;
    wa.wbits = at<uint32_t>(ws, L.wbits);
    wa.s_prev = at<float>(ws, L.s_prev);
    wa.s_next = at<float>(ws, L.s_next);
    wa.part = at<double>(ws, L.wpart);
    wa.cnt = at<unsigned>(ws, L.wcnt);
    wa.status = at<unsigned>(ws, L.status);
    wa.pt = c->ptw[dtype];
    wa.interleave = c->wpr[dtype] > 1 ? 1 : 0;
    wa.cg_div = make_fastdiv((uint32_t)(c->C / 256));
    wa.n = c->n;
    wa.C = c->C;
    wa.b1 = c->b1;
    wa.c1 = 1.0f - c->b1;
    const int grid_w = c->sms;
    if (int r = launch(c, OB_K_WORKER, s, [&] {
            return launch_worker(c->W, dtype, wa, grid_w, s, c->smem_budget);
        }))
        return r;
    if (after_worker) {
        const cudaError_t e = cudaEventRecord(after_worker, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }

    ServerArgs sa{};
    sa.wbits = wa.wbits;
    sa.s_next = wa.s_next;
    sa.ybuf = server_err;
    sa.sbits = at<uint32_t>(ws, L.sbits);
    sa.t_prev = at<float>(ws, L.t_prev);
    sa.t_next = at<float>(ws, L.t_next);
    sa.part = at<double>(ws, L.spart);
    sa.cnt = at<unsigned>(ws, L.scnt);
    sa.pt = c->pts;
    sa.n = c->n;
    sa.C = c->C;
    if (int r = launch(c, OB_K_SERVER, s, [&] { return launch_server(c->W, sa, c->grid_s, s); })) return r;

    UpdateArgs ua{};
    ua.sbits = sa.sbits;
    ua.t_next = sa.t_next;
    ua.maskbits = c->has_mask ? at<uint32_t>(ws, L.mask) : nullptr;
    ua.v = v;
    ua.x = x;
    ua.m = m;
    ua.s_prev = at<float>(ws, L.s_prev);
    ua.s_next = wa.s_next;
    ua.t_prev = at<float>(ws, L.t_prev);
    ua.NG = c->pts.NG;
    ua.CG = c->pts.CG;
    ua.nscales_w = (int64_t)c->W * c->nchunks;
    ua.nchunks = c->nchunks;
    ua.cg_div = make_fastdiv((uint32_t)(c->C / 256));
    ua.lr = c->lr;
    ua.eps = c->eps;
    ua.wd = c->wd;
    // the update's first block moves a few scales itself; many get a kernel of their own
    const UpdateArgs moves = ua;
    const bool many = ua.nscales_w + ua.nchunks > 16 * kBlock;
    if (many) ua.nscales_w = ua.nchunks = 0;
    if (int r = launch(c, OB_K_UPDATE, s, [&] { return launch_update(ua, c->grid_u, s); })) return r;
    if (many)
        if (int r = launch(c, OB_K_SCALES, s, [&] { return launch_scales(moves, stream_grid(c), s); })) return r;
    c->step += 1;
    return OB_OK;
}

int ob_compressed_step_host(ob_ctx* c, const void* grads_host, void* grads_dev, int dtype, float* x,
                            float* m, const float* v, float* worker_err, float* server_err, void* ws,
                            uint32_t* sbits_host, float* sscale_host, void* stream)
{
    if (!c || !grads_host || !sbits_host || !sscale_host) return OB_EINVAL;
    if (int r = check_grads(c, grads_dev, dtype)) return r;
    for (const void* p : {(const void*)x, (const void*)m, (const void*)v, (const void*)worker_err,
                          (const void*)server_err})
        if (int r = check_ptr(p, 16)) return r;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    const cudaStream_t s = (cudaStream_t)stream;
    const size_t gbytes = (size_t)c->W * (size_t)c->n * grad_bytes(dtype);
    cudaError_t e = cudaSuccess;
    if (!c->copy_stream) {
        e = cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->copied, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    // the event that marks the last worker pass reading this device buffer
    cudaEvent_t read_done = nullptr;
    for (auto& b : c->buffer_read)
        if (b.first == grads_dev) read_done = b.second;
    if (!read_done) {
        if (c->buffer_read.size() >= 8) {           // forget the oldest buffer
            cudaEventSynchronize(c->buffer_read.front().second);
            cudaEventDestroy(c->buffer_read.front().second);
            c->buffer_read.erase(c->buffer_read.begin());
        }
        e = cudaEventCreateWithFlags(&read_done, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e);
        c->buffer_read.emplace_back(grads_dev, read_done);
    }
    // copy on the copy stream once the buffer is free; the step waits for the copy
    e = cudaStreamWaitEvent(c->copy_stream, read_done, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(grads_dev, grads_host, gbytes, cudaMemcpyHostToDevice, c->copy_stream);
    if (e == cudaSuccess) e = cudaEventRecord(c->copied, c->copy_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c->copied, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    if (int r = compressed_step_impl(c, grads_dev, dtype, x, m, v, worker_err, server_err, ws, stream, read_done))
        return r;
    e = cudaMemcpyAsync(sbits_host, at<uint32_t>(ws, c->lay.sbits), (size_t)c->n / 8, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemcpyAsync(sscale_host, at<float>(ws, c->lay.t_next), (size_t)c->nchunks * 4,
                        cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return OB_OK;
}

size_t ob_loco_workspace_bytes(const ob_ctx* c, int bits)
{
    if (!c || (bits != 4 && bits != 8)) return 0;
    size_t off = up((size_t)c->W * (size_t)c->n * bits / 8, kAlignWs);   // codes
    off = up(off + (size_t)c->W * c->nchunks * 4, kAlignWs);               // scales
    off = up(off + (size_t)c->W * c->nchunks * 4, kAlignWs);               // absmax bits
    return off;
}

int ob_loco_step(ob_ctx* c, const void* grads, int dtype, float* x, float* m, float* v, float* loco_err,
                 float beta, int bits, void* loco_ws, void* stream)
{
    if (!c) return OB_EINVAL;
    if (bits != 4 && bits != 8) return OB_ENOTIMPL;
    if (!finite(beta) || beta < 0.0f || beta > 1.0f) return OB_EINVAL;
    if (int r = check_grads(c, grads, dtype)) return r;
    for (const void* p : {(const void*)x, (const void*)m, (const void*)v, (const void*)loco_err})
        if (int r = check_ptr(p, 16)) return r;
    if (int r = check_ptr(loco_ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    const cudaStream_t s = (cudaStream_t)stream;
    const size_t codes_b = up((size_t)c->W * (size_t)c->n * bits / 8, kAlignWs);
    const size_t scale_b = up((size_t)c->W * c->nchunks * 4, kAlignWs);
    LocoArgs a{};
    a.g = grads;
    a.err = loco_err;
    a.codes = at<uint8_t>(loco_ws, 0);
    a.scale = at<float>(loco_ws, codes_b);
    a.amax_bits = at<unsigned>(loco_ws, codes_b + scale_b);
    a.x = x;
    a.m = m;
    a.v = v;
    a.n = c->n;
    a.C = c->C;
    a.nchunks = c->nchunks;
    a.NG = c->n / 256;
    a.ng_div = make_fastdiv((uint32_t)a.NG);
    a.cg_div = make_fastdiv((uint32_t)(c->C / 256));
    a.W = c->W;
    a.bits = bits;
    a.ratio = c->loco_ratio;
    a.keep_codes = c->loco_codes ? 1 : 0;
    a.beta = beta;
    a.keep = 1.0f - beta;
    a.b1 = c->b1;
    a.c1 = 1.0f - c->b1;
    a.b2 = c->b2;
    a.c2 = 1.0f - c->b2;
    a.eps = c->eps;
    a.lr = c->lr;
    a.wd = c->wd;
    const int bi = bits == 4 ? 0 : 1;
    const int grid = c->sms * 4;
    if (c->C <= kLocoOnePassMaxChunk) {
        // short chunks: absmax and quantize in one pass, each warp owning whole chunks
        if (!c->loco_occ_f[dtype][bi]) c->loco_occ_f[dtype][bi] = occupancy_loco_fused(dtype, bits, c->C);
        const int grid_f = c->sms * (c->loco_occ_f[dtype][bi] > 0 ? c->loco_occ_f[dtype][bi] : 2);
        if (int r = launch(c, OB_K_LOCO_QUANT, s, [&] { return launch_loco_fused(dtype, a, grid_f, s); })) return r;
        if (int r = launch(c, OB_K_LOCO_SERVER, s, [&] { return launch_loco_server(a, grid, s); })) return r;
        c->step += 1;
        return OB_OK;
    }
    const cudaError_t e = cudaMemsetAsync(a.amax_bits, 0, (size_t)c->W * c->nchunks * 4, s);
    if (e != cudaSuccess) return cuda_fail(e);
    // the absmax pass (a contiguous range per warp), then one pass that quantizes every row
    // and takes the server step (a contiguous range per block, its warps taking the groups
    // in turn): each one resident wave
    if (!c->loco_occ_a[dtype]) c->loco_occ_a[dtype] = occupancy_loco_absmax(dtype);
    if (!c->loco_occ_qs[dtype][bi]) c->loco_occ_qs[dtype][bi] = occupancy_loco_qs(dtype, bits, c->W);
    const int grid_a = c->sms * (c->loco_occ_a[dtype] > 0 ? c->loco_occ_a[dtype] : 2);
    const int grid_qs = c->sms * (c->loco_occ_qs[dtype][bi] > 0 ? c->loco_occ_qs[dtype][bi] : 1);
    if (int r = launch(c, OB_K_LOCO_ABSMAX, s, [&] { return launch_loco_absmax(dtype, a, grid_a, s); })) return r;
    if (int r = launch(c, OB_K_LOCO_QUANT, s, [&] { return launch_loco_qs(dtype, a, grid_qs, s); })) return r;
    c->step += 1;
    return OB_OK;
}

int ob_reset_errors(ob_ctx* c, float* worker_err, float* server_err, void* ws, void* stream)
{
    if (!c) return OB_EINVAL;
    if (int r = check_ptr(worker_err, 16)) return r;
    if (int r = check_ptr(server_err, 16)) return r;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    const cudaStream_t s = (cudaStream_t)stream;
    const Layout& L = c->lay;
    cudaError_t e = cudaMemsetAsync(worker_err, 0, (size_t)c->W * c->n * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(server_err, 0, (size_t)c->n * 4, s);
    // previous and next scales of both sides (contiguous: s_prev .. t_next)
    if (e == cudaSuccess) e = cudaMemsetAsync(at<char>(ws, L.s_prev), 0, L.wpart - L.s_prev, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return OB_OK;
}

int ob_export_state(ob_ctx* c, const float* worker_err, const float* server_err, const void* ws,
                    float* ew_out, float* es_out, void* stream)
{
    if (!c) return OB_EINVAL;
    for (const void* p : {(const void*)worker_err, (const void*)server_err, (const void*)ew_out,
                          (const void*)es_out})
        if (int r = check_ptr(p, 16)) return r;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    ExportArgs a{};
    a.zbuf = worker_err;
    a.ybuf = server_err;
    a.s_prev = at<float>(const_cast<void*>(ws), c->lay.s_prev);
    a.t_prev = at<float>(const_cast<void*>(ws), c->lay.t_prev);
    a.ew_out = ew_out;
    a.es_out = es_out;
    a.n = c->n;
    a.C = c->C;
    a.nchunks = c->nchunks;
    a.W = c->W;
    const cudaStream_t s = (cudaStream_t)stream;
    return launch(c, OB_K_EXPORT, s, [&] { return launch_export(a, stream_grid(c), s); });
}

int ob_debug_views(const ob_ctx* c, const void* ws, const uint32_t** wbits, const float** wscale,
                   const uint32_t** sbits, const float** sscale)
{
    if (!c) return OB_EINVAL;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    void* w = const_cast<void*>(ws);
    if (wbits) *wbits = at<uint32_t>(w, c->lay.wbits);
    if (wscale) *wscale = at<float>(w, c->lay.s_next);
    if (sbits) *sbits = at<uint32_t>(w, c->lay.sbits);
    if (sscale) *sscale = at<float>(w, c->lay.t_next);
    return OB_OK;
}

int ob_profile(ob_ctx* c, int enable)
{
    if (!c) return OB_EINVAL;
    for (auto& r : c->recs) {
        c->spare.push_back(r.a);
        c->spare.push_back(r.b);
    }
    c->recs.clear();
    for (int k = 0; k < OB_K_COUNT; ++k) {
        c->prof_ms[k] = 0.0;
        c->prof_n[k] = 0;
    }
    c->profiling = enable != 0;
    return OB_OK;
}

int ob_profile_read(ob_ctx* c, int kernel, double* total_ms, int64_t* launches)
{
    if (!c || kernel < 0 || kernel >= OB_K_COUNT) return OB_EINVAL;
    for (auto& r : c->recs) {
        const cudaError_t e = cudaEventSynchronize(r.b);
        if (e != cudaSuccess) return cuda_fail(e);
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
            c->prof_ms[r.kernel] += ms;
            c->prof_n[r.kernel] += 1;
        }
        c->spare.push_back(r.a);
        c->spare.push_back(r.b);
    }
    c->recs.clear();
    if (total_ms) *total_ms = c->prof_ms[kernel];
    if (launches) *launches = c->prof_n[kernel];
    return OB_OK;
}

int64_t ob_launch_count(const ob_ctx* c) { return c ? c->launches : -1; }

int ob_selftest_wait(ob_ctx* c, void* ws, uint64_t limit_ns, void* stream)
{
    if (!c || limit_ns == 0 || limit_ns > kWaitLimitNs) return OB_EINVAL;
    if (ws != nullptr)
        if (int r = check_ptr(ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    unsigned* status = nullptr;
    if (ws != nullptr) {
        status = at<unsigned>(ws, c->lay.status);
    } else {
        void* scratch = nullptr;    // the no-allocation path's status word
        if (int r = noalloc_scratch(c->device, &scratch)) return r;
        status = at<unsigned>(scratch, kNoallocStatusOff);
    }
    const cudaError_t e = launch_wait_probe(status, limit_ns, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    c->launches += 1;
    return OB_OK;
}

int ob_read_status(ob_ctx* c, const void* ws, unsigned* status, void* stream)
{
    if (!c || !status) return OB_EINVAL;
    if (int r = check_ptr(ws, kAlignWs)) return r;
    if (int r = check_device(c)) return r;
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(status, at<unsigned>(const_cast<void*>(ws), c->lay.status), 4,
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    return OB_OK;
}

const char* ob_strerror(int code)
{
    switch (code) {
        case OB_OK: return "ok";
        case OB_EINVAL: return "invalid argument (size, dtype, null pointer or wrong device)";
        case OB_ECUDA: return "CUDA call or kernel launch failed";
        case OB_ENOTIMPL: return "not implemented";
        case OB_EALIGN: return "pointer not aligned (16 bytes; workspace 256 bytes)";
        case OB_ESCRATCH: return "too large for the fixed no-allocation scratch (OB_NOALLOC_SCRATCH_BYTES)";
    }
    return "unknown status";
}

int ob_last_cuda_error(void) { return g_last_cuda; }

}  // extern "C"

// ---- worker pass without any allocation ------------------------------------------------------
//
// For callers that cannot allocate device memory themselves (a runtime that hands out
// every byte of device memory from its own arena, or a caller with no allocator at
// all): the worker kernel's scratch -- per-range partial sums and per-chunk arrival
// counters -- lives in this fixed array instead of a caller-provided workspace. Every
// GPU that loads the library holds the array until the process exits. Its last 256
// bytes hold a status word that only ob_noalloc_read_status clears.
//
// Host code may not use the array's name as an address: it only stands for the symbol
// there. The device address is looked up with cudaGetSymbolAddress, with the device
// current, the first time a context of the driver is seen on that device, and again if
// that context changes (a device reset unloads the module, which may come back at
// another address).

static __device__ __align__(256) unsigned char g_noalloc_scratch[OB_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct NoallocSlot {
    unsigned long long ctx_id = 0;   // driver context the address belongs to (0: none yet)
    void* addr = nullptr;
};

std::mutex g_noalloc_mu;
NoallocSlot g_noalloc[kMaxDevices];

// The current driver context's unique id (never reused within a process), through the
// driver's entry points as the runtime exposes them; 0 if unavailable.
unsigned long long current_context_id()
{
    using GetCurrent = int (*)(void**);
    using GetId = int (*)(void*, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        cudaGetLastError();
    });
    void* ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
    return id;
}

// Device address of the scratch array on `dev` (which must be current).
int noalloc_scratch(int dev, void** out)
{
    if (dev < 0 || dev >= kMaxDevices) return OB_EINVAL;
    // id 0: no context is current on this thread yet; the lookup below makes the
    // device's primary context current, and the id is taken again after it
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot& slot = g_noalloc[dev];
    if (!slot.addr || id == 0 || slot.ctx_id != id) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        slot.addr = p;
        slot.ctx_id = id != 0 ? id : current_context_id();
    }
    *out = slot.addr;
    return OB_OK;
}

// [p, p + bytes) and [q, q + qbytes) share a byte.
bool overlap(const void* p, size_t bytes, const void* q, size_t qbytes)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + qbytes && b < a + bytes;
}

}  // namespace

extern "C" {

int ob_worker_compress_noalloc(ob_ctx* c, const void* grads, int dtype, const float* m, float* worker_err,
                               const float* scale_prev, uint32_t* wbits, float* scale_out, void* stream)
{
    if (!c) return OB_EINVAL;
    if (int r = check_grads(c, grads, dtype)) return r;
    for (const void* p : {(const void*)m, (const void*)worker_err, (const void*)scale_prev,
                          (const void*)wbits, (const void*)scale_out})
        if (int r = check_ptr(p, 16)) return r;
    // every output is disjoint from every other buffer (worker_err is updated in place)
    const size_t Wn = (size_t)c->W * (size_t)c->n;
    const size_t sc_bytes = (size_t)c->W * (size_t)c->nchunks * 4;
    struct Buf {
        const void* p;
        size_t bytes;
    };
    const Buf bufs[] = {{grads, Wn * grad_bytes(dtype)}, {m, (size_t)c->n * 4}, {worker_err, Wn * 4},
                        {scale_prev, sc_bytes}, {wbits, Wn / 8}, {scale_out, sc_bytes}};
    for (int o : {2, 4, 5})
        for (int i = 0; i < 6; ++i)
            if (i != o && overlap(bufs[o].p, bufs[o].bytes, bufs[i].p, bufs[i].bytes)) return OB_EINVAL;
    // scratch: partial sums [W][P][warps per range][J] doubles, then one counter per chunk;
    // the status word sits apart, in the array's last 256 bytes
    const Part& pt = c->ptw[dtype];
    const size_t part_bytes = up((size_t)c->W * pt.P * c->wpr[dtype] * pt.J * 8, kAlignWs);
    const size_t cnt_bytes = up((size_t)c->nchunks * 4, 16);
    if (part_bytes + cnt_bytes > kNoallocStatusOff) return OB_ESCRATCH;
    if (int r = check_device(c)) return r;
    void* scratch = nullptr;
    if (int r = noalloc_scratch(c->device, &scratch)) return r;
    const cudaStream_t s = (cudaStream_t)stream;
    unsigned* cnt = at<unsigned>(scratch, part_bytes);
    // the counters must start at zero; the partials are written before they are read
    const cudaError_t e = cudaMemsetAsync(cnt, 0, cnt_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e);

    WorkerArgs wa{};
    wa.g = grads;
    wa.m = m;
    wa.zbuf = worker_err;
    wa.wbits = wbits;
    wa.s_prev = scale_prev;
    wa.s_next = scale_out;
    wa.part = at<double>(scratch, 0);
    wa.cnt = cnt;
    wa.status = at<unsigned>(scratch, kNoallocStatusOff);
    wa.pt = pt;
    wa.interleave = c->wpr[dtype] > 1 ? 1 : 0;
    wa.cg_div = make_fastdiv((uint32_t)(c->C / 256));
    wa.n = c->n;
    wa.C = c->C;
    wa.b1 = c->b1;
    wa.c1 = 1.0f - c->b1;
    const int grid_w = c->sms;
    return launch(c, OB_K_WORKER, s, [&] { return launch_worker(c->W, dtype, wa, grid_w, s, c->smem_budget); });
}

int ob_noalloc_read_status(ob_ctx* c, unsigned* status, void* stream)
{
    if (!c || !status) return OB_EINVAL;
    if (int r = check_device(c)) return r;
    void* scratch = nullptr;
    if (int r = noalloc_scratch(c->device, &scratch)) return r;
    const cudaStream_t s = (cudaStream_t)stream;
    unsigned* word = at<unsigned>(scratch, kNoallocStatusOff);
    cudaError_t e = cudaMemcpyAsync(status, word, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, 4, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    return OB_OK;
}

}  // extern "C"
