// C ABI of libgdr.so: argument validation, lowering to kernel parameters and
// dispatch.  Every check runs on the host before anything is launched; the
// only device state the library owns is the per-device status word below.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "gdr_internal.h"

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int ok() {
    g_err.clear();
    return GDR_OK;
}

// Sticky error bits set by kernels (GDR_STATUS_*), one word per device.
__device__ unsigned int g_gdr_status;

std::mutex g_status_mu;
unsigned *g_status_ptr[64];

// Device address of this device's status word (cached; host-side symbol names
// are not device addresses).
int status_ptr(unsigned **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(GDR_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_gdr_status);
        if (e != cudaSuccess)
            return fail(GDR_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
        g_status_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_status_ptr[dev];
    return GDR_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dim(int K) { return K == 16 || K == 32 || K == 64 || K == 128; }

int esize(int dtype) { return dtype == GDR_BF16 ? 2 : 4; }

// Checks shared by every call that touches the pool.
int check_pool(const gdr_step_args *a, const char *fn) {
    if (!a) return fail(GDR_ERR_INVALID_ARG, "%s: args is NULL", fn);
    if (a->batch < 0) return fail(GDR_ERR_INVALID_ARG, "%s: batch %d < 0", fn, a->batch);
    if (a->nv <= 0 || a->nk <= 0)
        return fail(GDR_ERR_INVALID_ARG, "%s: nv=%d, nk=%d must be positive", fn, a->nv, a->nk);
    if (a->nv % a->nk != 0)
        return fail(GDR_ERR_INVALID_ARG, "%s: nv=%d is not a multiple of nk=%d", fn, a->nv, a->nk);
    if (a->V != a->K && a->V != 2 * a->K && !(2 * a->V == a->K && a->K >= 32))
        return fail(GDR_ERR_UNSUPPORTED, "%s: V=%d must be K=%d, 2K, or K/2 with K >= 32", fn, a->V, a->K);
    if (!supported_dim(a->K))
        return fail(GDR_ERR_UNSUPPORTED, "%s: K=%d not in {16,32,64,128}", fn, a->K);
    if (a->state_dtype != GDR_F32 && a->state_dtype != GDR_BF16)
        return fail(GDR_ERR_UNSUPPORTED, "%s: state_dtype %d", fn, a->state_dtype);
    if (a->batch == 0) return GDR_OK;
    if (!a->state || !a->slot_idx)
        return fail(GDR_ERR_INVALID_ARG, "%s: state/slot_idx is NULL", fn);
    if (a->max_slots <= 0) return fail(GDR_ERR_INVALID_ARG, "%s: max_slots %lld", fn, (long long)a->max_slots);
    if (a->state_vdim_stride != 1)
        return fail(GDR_ERR_UNSUPPORTED, "%s: state_vdim_stride must be 1 (got %lld)", fn,
                    (long long)a->state_vdim_stride);
    if (a->state_slot_stride <= 0 || a->state_head_stride <= 0 || a->state_kdim_stride <= 0)
        return fail(GDR_ERR_INVALID_ARG, "%s: state strides must be positive", fn);
    const long long es = esize(a->state_dtype);
    if (!aligned16(a->state) || (a->state_slot_stride * es) % 16 || (a->state_head_stride * es) % 16 ||
        (a->state_kdim_stride * es) % 16)
        return fail(GDR_ERR_UNSUPPORTED, "%s: state base and strides must be 16-byte aligned", fn);
    return GDR_OK;
}

// Checks for calls that read tokens and write output (fwd, verify, snapshots).
int check_step(const gdr_step_args *a, const char *fn) {
    int rc = check_pool(a, fn);
    if (rc) return rc;
    if (a->total_tokens < 0) return fail(GDR_ERR_INVALID_ARG, "%s: total_tokens < 0", fn);
    if (a->total_tokens >= (1ll << 31))
        return fail(GDR_ERR_UNSUPPORTED, "%s: total_tokens must be < 2^31", fn);
    if (a->batch > 0 && !a->offsets) return fail(GDR_ERR_INVALID_ARG, "%s: offsets is NULL", fn);
    if (a->total_tokens > 0) {
        if (!a->qkv || !a->decay || !a->beta || !a->out)
            return fail(GDR_ERR_INVALID_ARG, "%s: qkv/decay/beta/out is NULL", fn);
        if (a->qkv_seq_stride <= 0 || a->qkv_chan_stride <= 0 || a->tok_seq_stride <= 0 ||
            a->tok_head_stride <= 0 || a->out_seq_stride <= 0 || a->out_vdim_stride <= 0)
            return fail(GDR_ERR_INVALID_ARG, "%s: token/output strides must be positive", fn);
    }
    if (!(a->eps >= 0.0f)) return fail(GDR_ERR_INVALID_ARG, "%s: eps must be >= 0", fn);
    if (a->beta_vdim_stride < 0)
        return fail(GDR_ERR_INVALID_ARG, "%s: beta_vdim_stride < 0", fn);
    if (a->beta_vdim_stride > 0 && a->total_tokens > 0 && (a->beta_seq_stride <= 0 || a->beta_head_stride <= 0))
        return fail(GDR_ERR_INVALID_ARG, "%s: per-element beta strides must be positive", fn);
    return GDR_OK;
}

gdr::StepParams lower(const gdr_step_args *a, unsigned *status) {
    gdr::StepParams p{};
    p.batch = a->batch;
    p.nv = a->nv;
    p.nk = a->nk;
    p.r = a->nv / a->nk;
    p.decay_is_log = a->decay_is_log ? 1 : 0;
    p.l2norm = a->use_qk_l2norm ? 1 : 0;
    p.T = a->total_tokens;
    p.qkv = a->qkv;
    p.qkv_ss = a->qkv_seq_stride;
    p.qkv_cs = a->qkv_chan_stride;
    p.decay = a->decay;
    p.beta = a->beta;
    p.tok_ss = a->tok_seq_stride;
    p.tok_hs = a->tok_head_stride;
    p.bpv = a->beta_vdim_stride > 0 ? 1 : 0;
    p.beta_ss = a->beta_seq_stride;
    p.beta_hs = a->beta_head_stride;
    p.beta_vs = a->beta_vdim_stride;
    p.beta_vec = (p.bpv && a->beta_vdim_stride == 1 && aligned16(a->beta) && a->beta_seq_stride % 4 == 0 &&
                  a->beta_head_stride % 4 == 0) ? 1 : 0;
    p.scale = a->scale > 0.0f ? a->scale : (float)(1.0 / std::sqrt((double)a->K));
    p.eps = a->eps;
    p.out = a->out;
    p.out_ss = a->out_seq_stride;
    p.out_vs = a->out_vdim_stride;
    p.state = a->state;
    p.st_slot = a->state_slot_stride;
    p.st_head = a->state_head_stride;
    p.st_k = a->state_kdim_stride;
    p.max_slots = a->max_slots;
    p.slot_idx = a->slot_idx;
    p.offsets = a->offsets;
    p.qkv_vec = (a->qkv_chan_stride == 1 && aligned16(a->qkv) && a->qkv_seq_stride % 4 == 0) ? 1 : 0;
    p.out_vec = (a->out_vdim_stride == 1 && aligned16(a->out) && a->out_seq_stride % 4 == 0) ? 1 : 0;
    p.state_in = a->state;
    p.state_out = a->state;
    p.dense = 0;
    p.status = status;
    return p;
}

// Forward and verify rows of at most this many tokens (by the caller's
// max_row_len promise) run on the pipelined short-row kernel; longer or
// unknown lengths on the general one.  Snapshot passes always take the general
// kernel, which stores each snapshot straight from registers (measured faster
// than staging it through shared memory), as does per-element beta.
constexpr long long kShortRowMax = 64;

cudaError_t launch_rows(const gdr::StepParams &p, const gdr_step_args *a, gdr::Mode mode, const gdr::RingParams &rp,
                        const gdr::SnapParams &sp, cudaStream_t s) {
    const bool bf16 = a->state_dtype == GDR_BF16;
    if (!p.bpv && a->V == a->K && mode != gdr::Mode::Snap && a->max_row_len >= 1 && a->max_row_len <= kShortRowMax) {
        bool used = false;
        cudaError_t e = gdr::launch_short(p, a->K, bf16, mode, rp, sp, a->max_row_len, s, &used);
        if (used || e != cudaSuccess) return e;
    }
    return gdr::launch_chain(p, a->K, a->V, bf16, mode, rp, sp, a->max_row_len, s);
}

// The forward dispatch shared by gdr_fwd and gdr_fwd_host (arguments checked).
cudaError_t launch_fwd(const gdr_step_args *a, unsigned *status, cudaStream_t s) {
    const gdr::StepParams p = lower(a, status);
    if (a->max_row_len == 1 && !p.bpv && a->V == a->K) return gdr::launch_decode(p, a->K, a->state_dtype == GDR_BF16, s);
    return launch_rows(p, a, gdr::Mode::Fwd, gdr::RingParams{}, gdr::SnapParams{}, s);
}

// Row groups of gdr_fwd_host: the default count and the limit.
constexpr int kHostChunksAuto = 3;
constexpr int kHostMaxChunks = 16;

// Events that order gdr_fwd_host's copies and kernels across streams: one set
// per host thread and device, created on first use and kept until exit.
struct HostEvents {
    cudaEvent_t start, end, in[kHostMaxChunks], done[kHostMaxChunks];
};

int host_events(HostEvents **out) {
    static thread_local HostEvents *sets[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(GDR_ERR_CUDA, "device ordinal %d out of range", dev);
    if (!sets[dev]) {
        HostEvents *h = new HostEvents;
        cudaEvent_t *all[2 + 2 * kHostMaxChunks];
        int n = 0;
        all[n++] = &h->start;
        all[n++] = &h->end;
        for (int c = 0; c < kHostMaxChunks; ++c) {
            all[n++] = &h->in[c];
            all[n++] = &h->done[c];
        }
        for (int i = 0; i < n; ++i) {
            e = cudaEventCreateWithFlags(all[i], cudaEventDisableTiming);
            if (e != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaEventDestroy(*all[j]);
                delete h;
                return fail(GDR_ERR_CUDA, "cudaEventCreateWithFlags: %s", cudaGetErrorString(e));
            }
        }
        sets[dev] = h;
    }
    *out = sets[dev];
    return GDR_OK;
}

int launched(cudaError_t e, const char *fn) {
    if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
    return ok();
}

// Ring checks; writers (the verify pass) need a 16-byte aligned ring, the fold
// reads any element-aligned ring.
int check_ring(int32_t ring_dtype, int64_t ring_rows, int32_t ring_len, int64_t record_stride,
               const void *ring, const int32_t *ring_slot_idx, int K, int V, int r, int batch,
               bool writer, const char *fn) {
    if (ring_dtype != GDR_F32 && ring_dtype != GDR_BF16)
        return fail(GDR_ERR_UNSUPPORTED, "%s: ring_dtype %d (GDR_F32 or GDR_BF16)", fn, ring_dtype);
    if (ring_len < 1 || ring_len > 32)
        return fail(GDR_ERR_UNSUPPORTED, "%s: ring_len %d not in [1, 32]", fn, ring_len);
    const int need = gdr_ring_record_elements(K, V, r);
    const int mult = ring_dtype == GDR_BF16 ? 8 : 4;  // records start on 16 bytes
    if (record_stride < need || record_stride % mult)
        return fail(GDR_ERR_INVALID_ARG, "%s: record_stride %lld must be a multiple of %d and >= %d", fn,
                    (long long)record_stride, mult, need);
    if (batch > 0 && (!ring || !ring_slot_idx || ring_rows <= 0))
        return fail(GDR_ERR_INVALID_ARG, "%s: ring/ring_slot_idx NULL or ring_rows <= 0", fn);
    const uintptr_t align = writer ? 16 : (ring_dtype == GDR_BF16 ? 2 : 4);
    if (batch > 0 && (reinterpret_cast<uintptr_t>(ring) % align))
        return fail(GDR_ERR_UNSUPPORTED, "%s: ring must be %d-byte aligned", fn, (int)align);
    return GDR_OK;
}

int check_inter(const gdr_step_args *a, const void *inter, int64_t s_slot, int64_t s_tok,
                int64_t s_head, int32_t n_inter, const char *fn) {
    if (a->batch == 0) return GDR_OK;
    if (!inter) return fail(GDR_ERR_INVALID_ARG, "%s: intermediate buffer is NULL", fn);
    if (n_inter < 1) return fail(GDR_ERR_INVALID_ARG, "%s: n_inter %d < 1", fn, n_inter);
    if (s_slot <= 0 || s_tok <= 0 || s_head <= 0)
        return fail(GDR_ERR_INVALID_ARG, "%s: intermediate strides must be positive", fn);
    const long long es = esize(a->state_dtype);
    if (!aligned16(inter) || (s_slot * es) % 16 || (s_tok * es) % 16 || (s_head * es) % 16)
        return fail(GDR_ERR_UNSUPPORTED, "%s: intermediate base and strides must be 16-byte aligned", fn);
    return GDR_OK;
}

// ---- device-resident staging for gdr_fwd_host_noalloc ----------------------
// Some callers cannot allocate device memory at all: code that runs where an
// allocation would be an error (inside a stream capture with allocation
// forbidden, under a memory budget owned by someone else, or in a plug-in that
// only receives host buffers and a stream).  For them the staging buffers of
// the host-buffer forward pass live in this fixed array, one per device that
// loads the library, kept until the process exits.
constexpr size_t kNoAllocScratchBytes = 32u << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_gdr_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
unsigned char *g_noalloc_ptr[64];

// Device address of this device's staging array.  The symbol's name in host
// code is only a host-side stand-in, so the address is asked for once per
// device, with that device current, and cached.
int noalloc_scratch(unsigned char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(GDR_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_gdr_noalloc_scratch);
        if (e != cudaSuccess)
            return fail(GDR_ERR_CUDA, "cudaGetSymbolAddress(staging array): %s", cudaGetErrorString(e));
        g_noalloc_ptr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return GDR_OK;
}

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace

extern "C" {

const char *gdr_last_error(void) { return g_err.c_str(); }

int gdr_version(void) { return 100; }

int gdr_output_shape(int64_t total_tokens, int32_t nv, int32_t V, int64_t out_shape[2]) {
    if (!out_shape || total_tokens < 0 || nv <= 0 || V <= 0)
        return fail(GDR_ERR_INVALID_ARG, "gdr_output_shape: invalid arguments");
    out_shape[0] = total_tokens;
    out_shape[1] = (int64_t)nv * V;
    return ok();
}

int gdr_ring_record_elements(int32_t K, int32_t V, int32_t ratio) {
    if (K <= 0 || V <= 0 || ratio <= 0)
        return fail(GDR_ERR_INVALID_ARG, "gdr_ring_record_elements: invalid arguments");
    return K + ((ratio + 7) / 8) * 8 + ratio * V;
}

int gdr_fwd(const gdr_step_args *a, void *stream) {
    int rc = check_step(a, "gdr_fwd");
    if (rc) return rc;
    if (a->batch == 0) return ok();
    unsigned *st = nullptr;
    if ((rc = status_ptr(&st))) return rc;
    return launched(launch_fwd(a, st, static_cast<cudaStream_t>(stream)), "gdr_fwd");
}

int gdr_fwd_host(const gdr_step_args *a, const gdr_host_io *h, int32_t chunks, void *stream, void *h2d_stream,
                 void *d2h_stream) {
    const char *fn = "gdr_fwd_host";
    int rc = check_step(a, fn);
    if (rc) return rc;
    if (!h) return fail(GDR_ERR_INVALID_ARG, "%s: host is NULL", fn);
    if (a->batch == 0) return ok();
    if (!h->qkv || !h->decay || !h->beta || !h->slot_idx || !h->offsets || !h->out)
        return fail(GDR_ERR_INVALID_ARG, "%s: a host buffer is NULL", fn);
    const int64_t conv = 2ll * a->nk * a->K + (int64_t)a->nv * a->V, ow = (int64_t)a->nv * a->V;
    if (a->beta_vdim_stride > 0)
        return fail(GDR_ERR_UNSUPPORTED, "%s: beta must be [total_tokens, nv] (beta_vdim_stride 0)", fn);
    if (a->total_tokens > 0 &&
        (a->qkv_chan_stride != 1 || a->qkv_seq_stride != conv || a->tok_head_stride != 1 ||
         a->tok_seq_stride != a->nv || a->out_vdim_stride != 1 || a->out_seq_stride != ow))
        return fail(GDR_ERR_UNSUPPORTED, "%s: device token buffers must be dense", fn);
    const int32_t *off = h->offsets;
    if (off[0] < 0 || off[a->batch] > a->total_tokens)
        return fail(GDR_ERR_INVALID_ARG, "%s: offsets outside [0, total_tokens]", fn);
    for (int b = 0; b < a->batch; ++b)
        if (off[b + 1] < off[b]) return fail(GDR_ERR_INVALID_ARG, "%s: offsets not monotone at row %d", fn, b);
    unsigned *st = nullptr;
    if ((rc = status_ptr(&st))) return rc;
    HostEvents *ev = nullptr;
    if ((rc = host_events(&ev))) return rc;

    // groups of consecutive rows; with three or more groups the first and the
    // last get half the tokens of the others, since the first group's copy in
    // and the last group's copy out are the only copies nothing overlaps
    int nch = chunks > 0 ? chunks : kHostChunksAuto;
    if (nch > kHostMaxChunks) nch = kHostMaxChunks;
    if (nch > a->batch) nch = a->batch;
    int bound[kHostMaxChunks + 1];
    bound[0] = 0;
    const int64_t T0 = off[0], span = (int64_t)off[a->batch] - off[0];
    const int64_t parts = nch >= 3 ? 2 * nch - 2 : nch;  // in half-group units
    for (int c = 1; c < nch; ++c) {
        const int64_t upto = nch >= 3 ? 2 * c - 1 : c;      // half-group units before group c
        const int64_t target = T0 + span * upto / parts;
        int r = bound[c - 1] + 1;  // every group keeps at least one row
        while (r < a->batch - (nch - c) && off[r] < target) ++r;
        bound[c] = r;
    }
    bound[nch] = a->batch;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStream_t hs = h2d_stream ? static_cast<cudaStream_t>(h2d_stream) : cs;
    cudaStream_t ds = d2h_stream ? static_cast<cudaStream_t>(d2h_stream) : cs;
    cudaError_t e = cudaSuccess;
    auto cuda = [&](cudaError_t r) {
        if (e == cudaSuccess) e = r;
        return e == cudaSuccess;
    };
    auto order = [&](cudaStream_t from, cudaStream_t to, cudaEvent_t evt) {
        if (from == to) return true;
        return cuda(cudaEventRecord(evt, from)) && cuda(cudaStreamWaitEvent(to, evt, 0));
    };
    // the device buffers may still be in use by work queued earlier on `stream`
    if (!order(cs, hs, ev->start)) return fail(GDR_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    const size_t f4 = sizeof(float), i4 = sizeof(int32_t);
    // the small arrays (slots, offsets, decay, beta) go in whole with the first
    // group, since every copy has a fixed cost; qkv and out travel per group
    const int64_t T_lo = off[0], T_hi = off[a->batch];
    bool good = cuda(cudaMemcpyAsync(const_cast<int32_t *>(a->slot_idx), h->slot_idx, (size_t)a->batch * i4,
                                     cudaMemcpyHostToDevice, hs)) &&
                cuda(cudaMemcpyAsync(const_cast<int32_t *>(a->offsets), h->offsets, (size_t)(a->batch + 1) * i4,
                                     cudaMemcpyHostToDevice, hs));
    if (good && T_hi > T_lo)
        good = cuda(cudaMemcpyAsync(const_cast<float *>(a->decay) + T_lo * a->nv, h->decay + T_lo * a->nv,
                                    (size_t)((T_hi - T_lo) * a->nv) * f4, cudaMemcpyHostToDevice, hs)) &&
               cuda(cudaMemcpyAsync(const_cast<float *>(a->beta) + T_lo * a->nv, h->beta + T_lo * a->nv,
                                    (size_t)((T_hi - T_lo) * a->nv) * f4, cudaMemcpyHostToDevice, hs));
    if (!good) return fail(GDR_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    for (int c = 0; c < nch; ++c) {
        const int r0 = bound[c], r1 = bound[c + 1];
        const int64_t t0 = off[r0], t1 = off[r1];
        const int64_t nt = t1 - t0;
        if (nt > 0)
            good = cuda(cudaMemcpyAsync(const_cast<float *>(a->qkv) + t0 * conv, h->qkv + t0 * conv,
                                        (size_t)(nt * conv) * f4, cudaMemcpyHostToDevice, hs));
        good = good && order(hs, cs, ev->in[c]);
        if (good) {
            gdr_step_args g = *a;
            g.batch = r1 - r0;
            g.slot_idx = a->slot_idx + r0;
            g.offsets = a->offsets + r0;
            good = cuda(launch_fwd(&g, st, cs)) && order(cs, ds, ev->done[c]);
        }
        if (good && nt > 0)
            good = cuda(cudaMemcpyAsync(h->out + t0 * ow, a->out + t0 * ow, (size_t)(nt * ow) * f4,
                                        cudaMemcpyDeviceToHost, ds));
        if (!good) return fail(GDR_ERR_CUDA, "%s: group %d: %s", fn, c, cudaGetErrorString(e));
    }
    // `stream` passes the call only once every copy back has landed
    if (!order(ds, cs, ev->end)) return fail(GDR_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    return ok();
}

int gdr_fwd_host_noalloc(const gdr_step_args *a, const gdr_host_io *h, int32_t chunks, void *stream,
                         void *h2d_stream, void *d2h_stream) {
    const char *fn = "gdr_fwd_host_noalloc";
    if (!a) return fail(GDR_ERR_INVALID_ARG, "%s: args is NULL", fn);
    if (a->batch < 0 || a->total_tokens < 0 || a->nk <= 0 || a->nv <= 0 || a->K <= 0 || a->V <= 0)
        return fail(GDR_ERR_INVALID_ARG, "%s: sizes must be positive", fn);
    if (a->beta_vdim_stride > 0)
        return fail(GDR_ERR_UNSUPPORTED, "%s: beta must be [total_tokens, nv] (beta_vdim_stride 0)", fn);
    // the staging layout: qkv, decay, beta, out, slot_idx, offsets, each 256-byte aligned
    const int64_t T = a->total_tokens, conv = 2ll * a->nk * a->K + (int64_t)a->nv * a->V;
    const int64_t ow = (int64_t)a->nv * a->V;
    const size_t b_qkv = round256((size_t)(T * conv) * sizeof(float));
    const size_t b_tok = round256((size_t)(T * a->nv) * sizeof(float));
    const size_t b_out = round256((size_t)(T * ow) * sizeof(float));
    const size_t b_slot = round256((size_t)a->batch * sizeof(int32_t));
    const size_t b_off = round256((size_t)(a->batch + 1) * sizeof(int32_t));
    const size_t need = b_qkv + 2 * b_tok + b_out + b_slot + b_off;
    if (need > kNoAllocScratchBytes)
        return fail(GDR_ERR_UNSUPPORTED,
                    "%s: the call needs %zu bytes of staging, more than the library's fixed %zu-byte array "
                    "(use gdr_fwd_host with buffers of your own, or fewer tokens per call)",
                    fn, need, kNoAllocScratchBytes);
    unsigned char *base = nullptr;
    int rc = noalloc_scratch(&base);
    if (rc) return rc;
    gdr_step_args g = *a;
    unsigned char *q = base;
    g.qkv = reinterpret_cast<const float *>(q);
    g.qkv_seq_stride = conv;
    g.qkv_chan_stride = 1;
    q += b_qkv;
    g.decay = reinterpret_cast<const float *>(q);
    q += b_tok;
    g.beta = reinterpret_cast<const float *>(q);
    q += b_tok;
    g.tok_seq_stride = a->nv;
    g.tok_head_stride = 1;
    g.beta_seq_stride = g.beta_head_stride = g.beta_vdim_stride = 0;
    g.out = reinterpret_cast<float *>(q);
    g.out_seq_stride = ow;
    g.out_vdim_stride = 1;
    q += b_out;
    g.slot_idx = reinterpret_cast<const int32_t *>(q);
    q += b_slot;
    g.offsets = reinterpret_cast<const int32_t *>(q);
    // every staged byte a call reads is written by that call's own copies
    // first, so nothing needs clearing between calls
    return gdr_fwd_host(&g, h, chunks, stream, h2d_stream, d2h_stream);
}

int gdr_fwd_conv(const gdr_step_args *a, const gdr_conv_args *c, void *stream) {
    const char *fn = "gdr_fwd_conv";
    int rc = check_step(a, fn);
    if (rc) return rc;
    if (!c) return fail(GDR_ERR_INVALID_ARG, "%s: conv is NULL", fn);
    if (a->V != a->K) return fail(GDR_ERR_UNSUPPORTED, "%s: V=%d must equal K=%d", fn, a->V, a->K);
    if (a->beta_vdim_stride > 0)
        return fail(GDR_ERR_UNSUPPORTED, "%s: beta must be [total_tokens, nv] (beta_vdim_stride 0)", fn);
    if (c->width < 1 || c->width > 4) return fail(GDR_ERR_UNSUPPORTED, "%s: width %d not in [1, 4]", fn, c->width);
    if (c->activation != 0 && c->activation != 1)
        return fail(GDR_ERR_INVALID_ARG, "%s: activation %d (0 none, 1 SiLU)", fn, c->activation);
    if (!c->weight || c->weight_chan_stride <= 0 || c->weight_tap_stride <= 0)
        return fail(GDR_ERR_INVALID_ARG, "%s: weight is NULL or has a non-positive stride", fn);
    if (c->width > 1 && a->batch > 0 &&
        (!c->conv_state || c->state_slot_stride <= 0 || c->state_chan_stride <= 0 || c->state_tap_stride <= 0))
        return fail(GDR_ERR_INVALID_ARG, "%s: conv_state is NULL or has a non-positive stride", fn);
    if (a->batch == 0) return ok();
    unsigned *st = nullptr;
    if ((rc = status_ptr(&st))) return rc;
    const gdr::StepParams p = lower(a, st);
    gdr::ConvParams cv{};
    cv.width = c->width;
    cv.silu = c->activation;
    cv.w = c->weight;
    cv.w_cs = c->weight_chan_stride;
    cv.w_ts = c->weight_tap_stride;
    cv.bias = c->bias;
    cv.state = c->conv_state;
    cv.cs_slot = c->state_slot_stride;
    cv.cs_chan = c->state_chan_stride;
    cv.cs_tap = c->state_tap_stride;
    cv.channels = 2 * a->nk * a->K + a->nv * a->V;
    return launched(gdr::launch_chain_conv(p, cv, a->K, a->state_dtype == GDR_BF16, a->max_row_len,
                                           static_cast<cudaStream_t>(stream)),
                    fn);
}

int gdr_fwd_dense(const gdr_step_args *a, const void *initial_state, void *final_state, void *stream) {
    const char *fn = "gdr_fwd_dense";
    if (!a) return fail(GDR_ERR_INVALID_ARG, "%s: args is NULL", fn);
    // the dense buffers stand in for the pool: check them through a copy of the args
    gdr_step_args d = *a;
    d.state = initial_state ? const_cast<void *>(initial_state) : final_state;
    d.max_slots = a->batch > 0 ? a->batch : 1;
    static const int32_t kNoSlots = 0;
    d.slot_idx = &kNoSlots;  // not read in the dense mode
    int rc = check_step(&d, fn);
    if (rc) return rc;
    if (a->batch > 0 && !initial_state && !final_state)
        return fail(GDR_ERR_INVALID_ARG, "%s: initial_state and final_state are both NULL", fn);
    if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)))
        return fail(GDR_ERR_UNSUPPORTED, "%s: initial_state / final_state must be 16-byte aligned", fn);
    if (a->batch == 0) return ok();
    unsigned *st = nullptr;
    if ((rc = status_ptr(&st))) return rc;
    gdr::StepParams p = lower(&d, st);
    p.state = nullptr;
    p.slot_idx = nullptr;
    p.state_in = initial_state;
    p.state_out = final_state;
    p.dense = 1;
    const bool bf16 = a->state_dtype == GDR_BF16;
    return launched(gdr::launch_chain(p, a->K, a->V, bf16, gdr::Mode::Fwd, gdr::RingParams{}, gdr::SnapParams{},
                                      a->max_row_len, static_cast<cudaStream_t>(stream)),
                    fn);
}

int gdr_verify_ring(const gdr_step_args *a, void *ring, int32_t ring_dtype, int64_t ring_rows,
                    int32_t ring_len, int64_t record_stride, const int32_t *ring_slot_idx, void *stream) {
    int rc = check_step(a, "gdr_verify_ring");
    if (rc) return rc;
    if (a->beta_vdim_stride > 0)
        return fail(GDR_ERR_UNSUPPORTED, "gdr_verify_ring: beta must be [total_tokens, nv] (beta_vdim_stride 0)");
    if (a->V != a->K)
        return fail(GDR_ERR_UNSUPPORTED, "gdr_verify_ring: V=%d must equal K=%d", a->V, a->K);
    const int r = a->nv / a->nk;
    rc = check_ring(ring_dtype, ring_rows, ring_len, record_stride, ring, ring_slot_idx, a->K, a->V, r,
                    a->batch, true, "gdr_verify_ring");
    if (rc) return rc;
    if (a->batch == 0) return ok();
    unsigned *st = nullptr;
    if ((rc = status_ptr(&st))) return rc;
    const gdr::StepParams p = lower(a, st);
    gdr::RingParams rp{};
    rp.ring = ring;
    rp.bf16 = ring_dtype == GDR_BF16;
    rp.rows = ring_rows;
    rp.len = ring_len;
    rp.stride = record_stride;
    rp.ring_slot = ring_slot_idx;
    rp.alpha_off = a->K;
    rp.u_off = a->K + ((r + 7) / 8) * 8;
    return launched(launch_rows(p, a, gdr::Mode::Verify, rp, gdr::SnapParams{}, static_cast<cudaStream_t>(stream)),
                    "gdr_verify_ring");
}

int gdr_fold(const gdr_step_args *a, const void *ring, int32_t ring_dtype, int64_t ring_rows, int32_t ring_len,
             int64_t record_stride, const int32_t *ring_slot_idx, const int32_t *counts, void *stream) {
    int rc = check_pool(a, "gdr_fold");
    if (rc) return rc;
    if (a->V != a->K) return fail(GDR_ERR_UNSUPPORTED, "gdr_fold: V=%d must equal K=%d", a->V, a->K);
    const int r = a->nv / a->nk;
    rc = check_ring(ring_dtype, ring_rows, ring_len, record_stride, ring, ring_slot_idx, a->K, a->V, r,
                    a->batch, false, "gdr_fold");
    if (rc) return rc;
    if (a->batch == 0) return ok();
    if (!counts) return fail(GDR_ERR_INVALID_ARG, "gdr_fold: counts is NULL");
    unsigned *st = nullptr;
    if ((rc = status_ptr(&st))) return rc;
    gdr::FoldParams p{};
    p.batch = a->batch;
    p.nv = a->nv;
    p.nk = a->nk;
    p.r = r;
    p.state = a->state;
    p.st_slot = a->state_slot_stride;
    p.st_head = a->state_head_stride;
    p.st_k = a->state_kdim_stride;
    p.max_slots = a->max_slots;
    p.slot_idx = a->slot_idx;
    p.ring = ring;
    p.ring_bf16 = ring_dtype == GDR_BF16;
    p.ring_rows = ring_rows;
    p.ring_len = ring_len;
    p.stride = record_stride;
    p.ring_slot = ring_slot_idx;
    p.counts = counts;
    p.alpha_off = a->K;
    p.u_off = a->K + ((r + 7) / 8) * 8;
    p.status = st;
    return launched(gdr::launch_fold(p, a->K, a->state_dtype == GDR_BF16, static_cast<cudaStream_t>(stream)),
                    "gdr_fold");
}

int gdr_fwd_snapshots(const gdr_step_args *a, void *inter, int64_t inter_slot_stride, int64_t inter_token_stride,
                      int64_t inter_head_stride, int32_t n_inter, int32_t steps_per_token, void *stream) {
    int rc = check_step(a, "gdr_fwd_snapshots");
    if (rc) return rc;
    if (steps_per_token < 1) return fail(GDR_ERR_INVALID_ARG, "gdr_fwd_snapshots: steps_per_token < 1");
    rc = check_inter(a, inter, inter_slot_stride, inter_token_stride, inter_head_stride, n_inter,
                     "gdr_fwd_snapshots");
    if (rc) return rc;
    if (a->batch == 0) return ok();
    unsigned *st = nullptr;
    if ((rc = status_ptr(&st))) return rc;
    const gdr::StepParams p = lower(a, st);
    gdr::SnapParams sp{};
    sp.inter = inter;
    sp.s_slot = inter_slot_stride;
    sp.s_tok = inter_token_stride;
    sp.s_head = inter_head_stride;
    sp.n_inter = n_inter;
    sp.spt = steps_per_token;
    return launched(launch_rows(p, a, gdr::Mode::Snap, gdr::RingParams{}, sp, static_cast<cudaStream_t>(stream)),
                    "gdr_fwd_snapshots");
}

int gdr_rollback(const gdr_step_args *a, const void *inter, int64_t inter_slot_stride, int64_t inter_token_stride,
                 int64_t inter_head_stride, int32_t n_inter, const int32_t *accepted, void *stream) {
    int rc = check_pool(a, "gdr_rollback");
    if (rc) return rc;
    rc = check_inter(a, inter, inter_slot_stride, inter_token_stride, inter_head_stride, n_inter, "gdr_rollback");
    if (rc) return rc;
    if (a->batch == 0) return ok();
    if (!accepted) return fail(GDR_ERR_INVALID_ARG, "gdr_rollback: accepted is NULL");
    unsigned *st = nullptr;
    if ((rc = status_ptr(&st))) return rc;
    gdr::RollbackParams p{};
    p.batch = a->batch;
    p.nv = a->nv;
    p.state = a->state;
    p.st_slot = a->state_slot_stride;
    p.st_head = a->state_head_stride;
    p.st_k = a->state_kdim_stride;
    p.max_slots = a->max_slots;
    p.slot_idx = a->slot_idx;
    p.inter = inter;
    p.s_slot = inter_slot_stride;
    p.s_tok = inter_token_stride;
    p.s_head = inter_head_stride;
    p.n_inter = n_inter;
    p.accepted = accepted;
    p.status = st;
    return launched(gdr::launch_rollback(p, a->K, a->V, a->state_dtype == GDR_BF16, static_cast<cudaStream_t>(stream)),
                    "gdr_rollback");
}

int gdr_probe_fma(int32_t pattern, int32_t warps_per_subpartition, int32_t iterations, float *sink,
                  int64_t sink_elements, int32_t *ctas, void *stream) {
    if (pattern < 0 || pattern > 2 || warps_per_subpartition < 1 || warps_per_subpartition > 8 || iterations < 1 ||
        !sink || !ctas)
        return fail(GDR_ERR_INVALID_ARG, "gdr_probe_fma: invalid arguments");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "gdr_probe_fma: %s", cudaGetErrorString(e));
    if (sink_elements < (int64_t)sms * 128 * warps_per_subpartition)
        return fail(GDR_ERR_INVALID_ARG, "gdr_probe_fma: sink holds %lld floats, %lld needed", (long long)sink_elements,
                    (long long)sms * 128 * warps_per_subpartition);
    e = gdr::launch_probe_fma(pattern, warps_per_subpartition, iterations, sink, static_cast<cudaStream_t>(stream), ctas);
    if (e == cudaErrorInvalidConfiguration)
        return fail(GDR_ERR_UNSUPPORTED, "gdr_probe_fma: pattern %d does not fit %d warps per sub-partition in one SM",
                    pattern, warps_per_subpartition);
    return launched(e, "gdr_probe_fma");
}

int gdr_get_status(uint32_t *status, int32_t clear) {
    if (!status) return fail(GDR_ERR_INVALID_ARG, "gdr_get_status: status is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "gdr_get_status: %s", cudaGetErrorString(e));
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_gdr_status, sizeof v);
    if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "gdr_get_status: %s", cudaGetErrorString(e));
    if (clear) {
        const unsigned z = 0;
        e = cudaMemcpyToSymbol(g_gdr_status, &z, sizeof z);
        if (e != cudaSuccess) return fail(GDR_ERR_CUDA, "gdr_get_status: %s", cudaGetErrorString(e));
    }
    *status = v;
    return ok();
}

}  // extern "C"
