// C ABI of libsdm (declared and documented in include/sdm.h): argument checks, the workspace
// layout, and the launch sequence of the chunked write/read.
//
// Launch sequence of sdm_write_read (sparse-delta-memory 2.0.0, memory_ops.py module
// docstring "Forward"; the slabs follow _sdm_forward's bounded-memory no-grad steps):
//   status block cleared
//   for each slab of `ns` steps:        Phase 1 (one CTA per chunk), WY solve
//       for each step ti of the slab:   gather -> dual matmul -> DW
// Everything is queued on the caller's stream; nothing is allocated and nothing synchronizes.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

}  // namespace

namespace {
std::atomic<long long> g_wait_limit{kSpinLimit};
}  // namespace

long long wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

int set_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

namespace {

int cuda_fail(cudaError_t e, const char *what) {
    return fail(SDM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Checks the shape; fills d. Returns SDM_OK or a refusal (message set).
int check_shape(const sdm_shape *s, Dims &d) {
    if (!s) return fail(SDM_ERR_INVALID, "shape is NULL");
    if (s->P < 1) return fail(SDM_ERR_INVALID, "P must be >= 1, got %d", s->P);
    if (s->T < 1) return fail(SDM_ERR_INVALID, "T must be >= 1, got %d", s->T);
    if (s->C < kMinChunk || s->C > kMaxChunk)
        return fail(SDM_ERR_INVALID, "chunk size C must be in %d..%d, got %d", kMinChunk,
                    kMaxChunk, s->C);
    if (s->S < 1) return fail(SDM_ERR_INVALID, "S must be >= 1, got %d", s->S);
    if (s->W < 1 || s->W > kMaxWidth || s->R < 1 || s->R > kMaxWidth)
        return fail(SDM_ERR_INVALID, "W and R must be in 1..%d, got W=%d R=%d", kMaxWidth, s->W,
                    s->R);
    if (s->bank_dtype != SDM_F32 && s->bank_dtype != SDM_BF16)
        return fail(SDM_ERR_INVALID, "bank_dtype must be SDM_F32 (0) or SDM_BF16 (1), got %d",
                    s->bank_dtype);
    if (s->slab_steps < 0) return fail(SDM_ERR_INVALID, "slab_steps must be >= 0");
    if (s->flags & ~(SDM_FLAG_PER_STEP_KERNELS | SDM_FLAG_SNAPSHOT_BF16 | SDM_FLAG_TOKEN_GATE |
                     SDM_FLAG_SHARED_BANK | SDM_FLAG_SNAPSHOT_FP8))
        return fail(SDM_ERR_INVALID, "unknown flags 0x%x", (unsigned)s->flags);
    if ((s->flags & SDM_FLAG_SNAPSHOT_BF16) && (s->flags & SDM_FLAG_SNAPSHOT_FP8))
        return fail(SDM_ERR_INVALID, "SDM_FLAG_SNAPSHOT_BF16 and SDM_FLAG_SNAPSHOT_FP8 exclude each other");
    if (s->D != 32 && s->D != 64 && s->D != 128 && s->D != 256 && s->D != 512)
        return fail(SDM_ERR_UNSUPPORTED, "head_dim D=%d has no kernel (32, 64, 128, 256, 512)",
                    s->D);
    const long long Nt = (s->T + (long long)s->C - 1) / s->C;
    if ((long long)s->P * Nt * s->C >= (1LL << 31))
        return fail(SDM_ERR_INVALID, "P * ceil(T/C) * C = %lld token rows exceed 2^31 - 1",
                    (long long)s->P * Nt * s->C);
    d.P = s->P; d.T = s->T; d.C = s->C; d.S = s->S; d.D = s->D; d.W = s->W; d.R = s->R;
    d.Nt = (int)Nt;
    d.dtype = s->bank_dtype;
    d.bwd = 0;
    d.xp = d.C;
    d.per_step = ((s->flags & SDM_FLAG_PER_STEP_KERNELS) || !phase2_fused_fits(d)) ? 1 : 0;
    d.snapq = (s->flags & SDM_FLAG_SNAPSHOT_FP8)
                  ? 2 : (((s->flags & SDM_FLAG_SNAPSHOT_BF16) && d.dtype == SDM_F32) ? 1 : 0);
    d.gate = (s->flags & SDM_FLAG_TOKEN_GATE) ? 1 : 0;
    d.shared = (s->flags & SDM_FLAG_SHARED_BANK) ? 1 : 0;
    d.spin = wait_limit();
    return SDM_OK;
}

size_t per_chunk_bytes(const Dims &d) {
    const size_t CW = (size_t)d.C * d.W, CR = (size_t)d.C * d.R, CC = (size_t)d.C * d.C;
    const size_t dense =
        dense_gram(d) ? 4 * (CW + 1 + d.C + 3 * (size_t)d.C * dense_pitch(d.C)) : 0;
    const size_t pair = phase1_split(d) ? 4 * CW : 0;   // (g, k) pairs in place of k alone
    return 4 * (11 * CW + 4) + 4 * 3 * CR + 4 * 4 * CC + 24 + dense + pair;
}

int slab_steps(const Dims &d, int requested) {
    if (requested > 0) return requested < d.Nt ? requested : d.Nt;
    const size_t per_step = per_chunk_bytes(d) * d.P;
    if (per_step * d.Nt <= kSlabBudget) return d.Nt;
    long ns = (long)(kSlabBudget / per_step);
    // at least two chunks per SM, so that Phase 1 (a CTA per chunk, two fit on an SM) keeps
    // every SM busy with two chunks at once
    const long min_steps = (2L * kRefSms + d.P - 1) / d.P;
    if (ns < min_steps) ns = min_steps;
    if (ns < 1) ns = 1;
    return ns < d.Nt ? (int)ns : d.Nt;
}

}  // namespace

int phase1_ctas(const Dims &d, int ns) {
    const long N = (long)ns * d.P;
    if (phase1_split(d)) return (int)N;   // one CTA, and one scratch slot, per chunk
    const long cap = 2L * kRefSms;        // scratch on chip: two CTAs per SM
    return (int)(N < cap ? N : cap);
}

// Byte layout of the workspace (every array 256-byte aligned), in assignment order.
#define SDM_LAYOUT(F)                                                         \
    F(status, DevStatus, 1)                                                   \
    F(perm, int32_t, N * CW)                                                  \
    F(wdw, float, N * CW)                                                     \
    F(goff, int32_t, N * (CW + 4))                                            \
    F(ng4, int4, N)                                                           \
    F(p1sel, int32_t, N)                                                      \
    F(gord, int32_t, N * CW)                                                  \
    F(gslot, int32_t, N * CW)                                                 \
    F(gfac, float, N * CW)                                                    \
    F(ngroups, int32_t, N)                                                    \
    F(nvalid, int32_t, N)                                                     \
    F(minfo, int32_t, N * CW)                                                 \
    F(wsl, int32_t, N * CW)                                                   \
    F(rsl, int32_t, N * CR)                                                   \
    F(gw, float, N * CW)                                                      \
    F(qw, float, N * CR)                                                      \
    F(lw, float, N * CW)                                                      \
    F(lr, float, N * CR)                                                      \
    F(A, float, N * CC)                                                       \
    F(QK, float, N * CC)                                                      \
    F(X, float, N * CX)                                                       \
    F(QX, float, N * CX)                                                      \
    F(keys, unsigned long long, G * 2 * CW)                                   \
    F(inv, int32_t, G * CW)                                                   \
    F(lws, float, G * CW)                                                     \
    F(pgid, int32_t, G * CW)                                                  \
    F(pgs, int32_t, G * CW)                                                   \
    F(lend, float, G * CW)                                                    \
    F(kf, float, (1 - PS) * G * CW)                                           \
    F(gk, float2, PS * G * CW)                                                \
    F(rlo, int32_t, G * CR)                                                   \
    F(rhi, int32_t, G * CR)                                                   \
    F(dpos, int32_t, HS * G * CW)                                             \
    F(dref, float, HS * N * C)                                                \
    F(ndense, int32_t, HS * N)                                                \
    F(dka, float, HS * N * DCC)                                               \
    F(dkb, float, HS * N * DCC)                                               \
    F(dkq, float, HS * N * DCC)                                               \
    F(wkey, unsigned long long, B * N * CW)                                   \
    F(wlws, float, B * N * CW)                                                \
    F(wpgs, int32_t, B * N * CW)                                              \
    F(wpge, int32_t, B * N * CW)                                              \
    F(dwt, float, B * N * CW)                                                 \
    F(rkey, unsigned long long, B * N * CR)                                   \
    F(rgoff, int32_t, B * N * (CR + 1))                                       \
    F(rgslot, int32_t, B * N * CR)                                            \
    F(rng, int32_t, B * N)                                                    \
    F(rkeys, unsigned long long, B * G * 2 * CR)                              \
    F(bu, float, B * P * CD)                                                  \
    F(bup, float, B * P * CD)                                                 \
    F(bdret, float, B * P * CD)                                               \
    F(bdo, float, B * P * CD)                                                 \
    F(bdX, float, B * P * CC)                                                 \
    F(bdQX, float, B * P * CC)                                                \
    F(bdQK, float, B * P * CC)                                                \
    F(bT, float, B * P * CC)                                                  \
    F(bdA, float, B * P * CC)                                                 \
    F(bdb2, float, B * P * DT * C)                                            \
    F(bddw, float, B * P * CW)                                                \
    F(bdgw, float, B * P * CW)                                                \
    F(bdqw, float, B * P * CR)                                                \
    F(bdfac, float, B * P * CW)                                               \
    F(bdlam, float, B * P * CW)                                               \
    F(bdlr, float, B * P * CR)                                                \
    F(bdgate, float, B * GT * P * CW)                                         \
    F(ret, float, P * CD)                                                     \
    F(inter, float, P * CD)                                                   \
    F(dv, float, P * CD)

size_t layout_bytes(const Dims &d, int ns, int G_) {
    const size_t N = (size_t)ns * d.P, P = d.P, CW = (size_t)d.C * d.W, CR = (size_t)d.C * d.R,
                 CC = (size_t)d.C * d.C, CD = (size_t)d.C * d.D, G = G_, B = d.bwd ? 1 : 0,
                 C = d.C, DT = ((size_t)d.D + 31) / 32, CX = (size_t)d.C * d.xp,
                 GT = d.gate ? 1 : 0, HS = dense_gram(d) ? 1 : 0,
                 PS = phase1_split(d) ? 1 : 0,
                 DCC = (size_t)d.C * dense_pitch(d.C);
    size_t off = 0;
#define X_SIZE(name, type, count) off += up(sizeof(type) * (size_t)(count));
    SDM_LAYOUT(X_SIZE)
#undef X_SIZE
    return off;
}

Work layout_assign(const Dims &d, int ns, int G_, void *base) {
    const size_t N = (size_t)ns * d.P, P = d.P, CW = (size_t)d.C * d.W, CR = (size_t)d.C * d.R,
                 CC = (size_t)d.C * d.C, CD = (size_t)d.C * d.D, G = G_, B = d.bwd ? 1 : 0,
                 C = d.C, DT = ((size_t)d.D + 31) / 32, CX = (size_t)d.C * d.xp,
                 GT = d.gate ? 1 : 0, HS = dense_gram(d) ? 1 : 0,
                 PS = phase1_split(d) ? 1 : 0,
                 DCC = (size_t)d.C * dense_pitch(d.C);
    Work w;
    memset(&w, 0, sizeof(w));
    char *p = static_cast<char *>(base);
    size_t off = 0;
#define X_ASSIGN(name, type, count)                                   \
    w.name = reinterpret_cast<type *>(p + off);                       \
    off += up(sizeof(type) * (size_t)(count));
    SDM_LAYOUT(X_ASSIGN)
#undef X_ASSIGN
    w.ns = ns;
    w.G = G_;
    return w;
}

namespace {

struct Prepared {
    Dims d;
    int ns, G;
    size_t bytes;
};

int prepare(const sdm_shape *shape, Prepared &pr, int bwd = 0) {
    int rc = check_shape(shape, pr.d);
    if (rc) return rc;
    pr.d.bwd = bwd;
    pr.d.xp = x_row_pitch(pr.d);
    pr.ns = slab_steps(pr.d, shape->slab_steps);
    pr.G = phase1_ctas(pr.d, pr.ns);
    pr.bytes = layout_bytes(pr.d, pr.ns, pr.G);
    return SDM_OK;
}

int check_workspace(const Prepared &pr, void *ws, size_t bytes) {
    if (!ws) return fail(SDM_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) % kAlign)
        return fail(SDM_ERR_WORKSPACE, "workspace must be %zu-byte aligned", kAlign);
    if (bytes < pr.bytes)
        return fail(SDM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", bytes, pr.bytes);
    return SDM_OK;
}

// Events around every launch of a profiled call (one before each launch, one after the last).
struct Recorder {
    std::vector<cudaEvent_t> ev;
    std::vector<int> kind;
    cudaError_t mark(int k, cudaStream_t st) {
        cudaEvent_t e;
        cudaError_t err = cudaEventCreate(&e);
        if (err != cudaSuccess) return err;
        ev.push_back(e);
        if (k >= 0) kind.push_back(k);
        return cudaEventRecord(e, st);
    }
};

int check_inputs(const Inputs &in, bool need_bank) {
    if ((need_bank && !in.bank) || !in.ws || !in.kw || !in.g || !in.beta || !in.rs || !in.qw)
        return fail(SDM_ERR_INVALID, "a required input pointer is NULL");
    if (need_bank && (!in.v || !in.readings))
        return fail(SDM_ERR_INVALID, "v and readings must not be NULL");
    if (need_bank && (reinterpret_cast<uintptr_t>(in.bank) % 16 ||
                      reinterpret_cast<uintptr_t>(in.readings) % 16 ||
                      reinterpret_cast<uintptr_t>(in.v) % 16))
        return fail(SDM_ERR_INVALID, "bank, v and readings must be 16-byte aligned");
    return SDM_OK;
}

// The launch sequence of one forward call (see the file comment).
int run_forward(const Prepared &pr, const Inputs &in, void *workspace, cudaStream_t st,
                Recorder *rec, cudaEvent_t phase2_ready = nullptr) {
    const Dims &d = pr.d;
    Work w = layout_assign(d, pr.ns, pr.G, workspace);
    cudaError_t e = cudaMemsetAsync(w.status, 0, sizeof(DevStatus), st);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
#define SDM_LAUNCH(kind, call, what)                                                       \
    do {                                                                                   \
        if (rec && (e = rec->mark(kind, st)) != cudaSuccess) return cuda_fail(e, "event");  \
        if ((e = (call)) != cudaSuccess) return cuda_fail(e, what);                        \
    } while (0)
    for (int s0 = 0; s0 < d.Nt; s0 += pr.ns) {
        const int nsteps = (d.Nt - s0) < pr.ns ? (d.Nt - s0) : pr.ns;
        SDM_LAUNCH(SDM_KERNEL_PHASE1, launch_phase1(d, in, w, s0, nsteps, st), "phase1");
        SDM_LAUNCH(SDM_KERNEL_SOLVE, launch_solve(d, in, w, s0, nsteps, st), "solve");
        if (phase2_ready && s0 == 0 && (e = cudaStreamWaitEvent(st, phase2_ready, 0)) != cudaSuccess)
            return cuda_fail(e, "wait for v");
        if (!d.per_step) {
            SDM_LAUNCH(SDM_KERNEL_PHASE2, launch_phase2_fused(d, in, w, s0, nsteps, st),
                       "phase2");
            continue;
        }
        for (int ti = s0; ti < s0 + nsteps; ++ti) {
            SDM_LAUNCH(SDM_KERNEL_GATHER, launch_gather(d, in, w, s0, ti, st), "gather");
            SDM_LAUNCH(SDM_KERNEL_DUALMM, launch_dualmm(d, in, w, s0, ti, st), "dual matmul");
            SDM_LAUNCH(SDM_KERNEL_DW, launch_dw(d, in, w, s0, ti, st), "dw");
        }
    }
#undef SDM_LAUNCH
    if (rec && (e = rec->mark(-1, st)) != cudaSuccess) return cuda_fail(e, "event");
    return SDM_OK;
}

// Device copies of the host inputs, after the sdm_write_read workspace (256-byte aligned).
struct HostStage {
    size_t ws, kw, g, beta, v, rs, qw, valid, bytes;
};
HostStage host_stage(const Dims &d, size_t base) {
    const size_t PT = (size_t)d.P * d.T, es = d.dtype == SDM_BF16 ? 2 : 4;
    HostStage h;
    size_t o = up(base);
    h.ws = o; o = up(o + 4 * PT * d.W);
    h.kw = o; o = up(o + es * PT * d.W);
    h.g = o; o = up(o + 4 * PT * (d.gate ? 1 : d.W));
    h.beta = o; o = up(o + 4 * PT);
    h.v = o; o = up(o + es * PT * d.D);
    h.rs = o; o = up(o + 4 * PT * d.R);
    h.qw = o; o = up(o + es * PT * d.R);
    h.valid = o; o = up(o + 4 * (size_t)d.P);
    h.bytes = o;
    return h;
}

// The library's second stream on the current device (for the v copy of sdm_write_read_host).
std::mutex g_side_mu;
cudaStream_t g_side[64];
int side_stream(cudaStream_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(SDM_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(g_side_mu);
    if (!g_side[dev]) {
        e = cudaStreamCreateWithFlags(&g_side[dev], cudaStreamNonBlocking);
        if (e != cudaSuccess) return cuda_fail(e, "side stream");
    }
    *out = g_side[dev];
    return SDM_OK;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" {

const char *sdm_last_error(void) { return g_err; }

const char *sdm_version(void) { return "sdm-gb300 0.2 (sm_103a)"; }

long long sdm_set_wait_limit(long long polls) {
    const long long prev = g_wait_limit.load();
    g_wait_limit.store(polls < 1 ? kSpinLimit : polls);
    return prev;
}

size_t sdm_workspace_bytes(const sdm_shape *shape) {
    Prepared pr;
    if (prepare(shape, pr)) return 0;
    g_err[0] = 0;
    return pr.bytes;
}

int64_t sdm_launch_count(const sdm_shape *shape) {
    Prepared pr;
    if (prepare(shape, pr)) return 0;
    const int64_t slabs = (pr.d.Nt + pr.ns - 1) / pr.ns;
    // Phase 1 (+ its row kernel, + the dense-Gram kernel), per slab
    const int64_t p1 = phase1_split(pr.d) ? (dense_gram(pr.d) ? 3 : 2) : 1;
    return pr.d.per_step ? slabs * (p1 + 1) + (int64_t)pr.d.Nt * 3 : slabs * (p1 + 2);
}

int sdm_write_read(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                   const void *write_w, const float *log_decay, const float *beta,
                   const void *v, const int32_t *read_slots, const void *read_w,
                   const int32_t *valid_tokens, void *readings, void *workspace,
                   size_t workspace_bytes, void *stream) {
    Prepared pr;
    int rc = prepare(shape, pr);
    if (rc) return rc;
    Inputs in{bank, write_slots, write_w, log_decay, beta, v, read_slots, read_w, valid_tokens,
              readings, nullptr};
    if ((rc = check_inputs(in, true))) return rc;
    if ((rc = check_workspace(pr, workspace, workspace_bytes))) return rc;
    g_err[0] = 0;
    return run_forward(pr, in, workspace, static_cast<cudaStream_t>(stream), nullptr);
}

int sdm_profile_write_read(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                           const void *write_w, const float *log_decay, const float *beta,
                           const void *v, const int32_t *read_slots, const void *read_w,
                           const int32_t *valid_tokens, void *readings, void *workspace,
                           size_t workspace_bytes, float *kernel_ms, int32_t *launches,
                           void *stream) {
    Prepared pr;
    int rc = prepare(shape, pr);
    if (rc) return rc;
    Inputs in{bank, write_slots, write_w, log_decay, beta, v, read_slots, read_w, valid_tokens,
              readings, nullptr};
    if ((rc = check_inputs(in, true))) return rc;
    if ((rc = check_workspace(pr, workspace, workspace_bytes))) return rc;
    if (!kernel_ms || !launches) return fail(SDM_ERR_INVALID, "kernel_ms and launches must not be NULL");
    g_err[0] = 0;
    Recorder r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = run_forward(pr, in, workspace, st, &r);
    cudaError_t e = cudaStreamSynchronize(st);
    if (!rc && e != cudaSuccess) rc = cuda_fail(e, "profile synchronize");
    for (int k = 0; k < SDM_KERNEL_KINDS; ++k) { kernel_ms[k] = 0.f; launches[k] = 0; }
    if (!rc) {
        for (size_t i = 0; i + 1 < r.ev.size(); ++i) {
            float ms = 0.f;
            e = cudaEventElapsedTime(&ms, r.ev[i], r.ev[i + 1]);
            if (e != cudaSuccess) { rc = cuda_fail(e, "profile elapsed time"); break; }
            kernel_ms[r.kind[i]] += ms;
            launches[r.kind[i]] += 1;
        }
    }
    for (cudaEvent_t ev : r.ev) cudaEventDestroy(ev);
    return rc;
}

size_t sdm_saved_bytes(const sdm_shape *shape) {
    Dims d;
    if (check_shape(shape, d)) return 0;
    g_err[0] = 0;
    const size_t es = d.snapq == 2 ? 1 : ((d.dtype == SDM_BF16 || d.snapq) ? 2 : 4);
    return (size_t)d.Nt * d.P * d.C * d.W * d.D * es;
}

int sdm_write_read_save(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                        const void *write_w, const float *log_decay, const float *beta,
                        const void *v, const int32_t *read_slots, const void *read_w,
                        const int32_t *valid_tokens, void *readings, void *saved,
                        size_t saved_bytes, void *workspace, size_t workspace_bytes,
                        void *stream) {
    Prepared pr;
    int rc = prepare(shape, pr);
    if (rc) return rc;
    Inputs in{bank, write_slots, write_w, log_decay, beta, v, read_slots, read_w, valid_tokens,
              readings, saved};
    if ((rc = check_inputs(in, true))) return rc;
    if ((rc = check_workspace(pr, workspace, workspace_bytes))) return rc;
    const size_t need = sdm_saved_bytes(shape);
    if (!saved || saved_bytes < need || reinterpret_cast<uintptr_t>(saved) % 16)
        return fail(SDM_ERR_WORKSPACE, "saved buffer must hold %zu bytes, 16-byte aligned", need);
    g_err[0] = 0;
    return run_forward(pr, in, workspace, static_cast<cudaStream_t>(stream), nullptr);
}

size_t sdm_backward_workspace_bytes(const sdm_shape *shape) {
    Prepared pr;
    if (prepare(shape, pr, 1)) return 0;
    g_err[0] = 0;
    return pr.bytes;
}

int sdm_write_read_backward(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                            const void *write_w, const float *log_decay, const float *beta,
                            const void *v, const int32_t *read_slots, const void *read_w,
                            const int32_t *valid_tokens, const void *saved, size_t saved_bytes,
                            const void *grad_readings, float *grad_bank, float *grad_v,
                            float *grad_beta, float *grad_write_w, float *grad_log_decay,
                            float *grad_read_w, void *workspace, size_t workspace_bytes,
                            void *stream) {
    Prepared pr;
    int rc = prepare(shape, pr, 1);
    if (rc) return rc;
    Inputs in{bank, write_slots, write_w, log_decay, beta, v, read_slots, read_w, valid_tokens,
              const_cast<void *>(grad_readings), const_cast<void *>(saved)};
    if ((rc = check_inputs(in, true))) return rc;
    if ((rc = check_workspace(pr, workspace, workspace_bytes))) return rc;
    const size_t need = sdm_saved_bytes(shape);
    if (!saved || saved_bytes < need || reinterpret_cast<uintptr_t>(saved) % 16)
        return fail(SDM_ERR_WORKSPACE, "saved buffer must hold %zu bytes, 16-byte aligned", need);
    if (!grad_bank || !grad_v || !grad_beta || !grad_write_w || !grad_log_decay || !grad_read_w)
        return fail(SDM_ERR_INVALID, "gradient output pointers must not be NULL");
    if (reinterpret_cast<uintptr_t>(grad_bank) % 16)
        return fail(SDM_ERR_INVALID, "grad_bank must be 16-byte aligned");
    g_err[0] = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Dims &d = pr.d;
    Work w = layout_assign(d, pr.ns, pr.G, workspace);
    BwdOut o{grad_readings, grad_bank, grad_v, grad_beta, grad_write_w, grad_log_decay,
             grad_read_w};
    cudaError_t e = cudaMemsetAsync(w.status, 0, sizeof(DevStatus), st);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    const int nslabs = (d.Nt + pr.ns - 1) / pr.ns;
    for (int sl = nslabs - 1; sl >= 0; --sl) {
        const int s0 = sl * pr.ns;
        const int nsteps = (d.Nt - s0) < pr.ns ? (d.Nt - s0) : pr.ns;
        if ((e = launch_phase1(d, in, w, s0, nsteps, st)) != cudaSuccess) return cuda_fail(e, "phase1");
        if ((e = launch_solve(d, in, w, s0, nsteps, st)) != cudaSuccess) return cuda_fail(e, "solve");
        for (int ti = s0 + nsteps - 1; ti >= s0; --ti)
            if ((e = launch_backward_step(d, in, w, o, s0, ti, st)) != cudaSuccess)
                return cuda_fail(e, "backward step");
    }
    return SDM_OK;
}

int sdm_phase1_debug(const sdm_shape *shape, const int32_t *write_slots, const void *write_w,
                     const float *log_decay, const float *beta, const int32_t *read_slots,
                     const void *read_w, const int32_t *valid_tokens, int32_t *perm,
                     uint8_t *group_start, uint8_t *owner, int32_t *ngroups, float *lw,
                     float *gw, float *dw, float *lr, float *qw, float *A, float *QK, float *X,
                     float *QX, int32_t *dense_groups, void *workspace, size_t workspace_bytes,
                     void *stream) {
    Prepared pr;
    int rc = prepare(shape, pr);
    if (rc) return rc;
    Inputs in{nullptr, write_slots, write_w, log_decay, beta, nullptr, read_slots, read_w,
              valid_tokens, nullptr, nullptr};
    if ((rc = check_inputs(in, false))) return rc;
    if ((rc = check_workspace(pr, workspace, workspace_bytes))) return rc;
    if ((perm != nullptr) != (group_start != nullptr) || (perm != nullptr) != (owner != nullptr) ||
        (perm != nullptr) != (dw != nullptr))
        return fail(SDM_ERR_INVALID, "perm, group_start, owner and dw are requested together");
    g_err[0] = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Dims &d = pr.d;
    Work w = layout_assign(d, pr.ns, pr.G, workspace);
    const size_t CW = (size_t)d.C * d.W, CR = (size_t)d.C * d.R, CC = (size_t)d.C * d.C;
    cudaError_t e = cudaMemsetAsync(w.status, 0, sizeof(DevStatus), st);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    for (int s0 = 0; s0 < d.Nt; s0 += pr.ns) {
        const int nsteps = (d.Nt - s0) < pr.ns ? (d.Nt - s0) : pr.ns;
        const size_t N = (size_t)nsteps * d.P, n0 = (size_t)s0 * d.P;
        if ((e = launch_phase1(d, in, w, s0, nsteps, st)) != cudaSuccess) return cuda_fail(e, "phase1");
        if ((e = launch_solve(d, in, w, s0, nsteps, st)) != cudaSuccess) return cuda_fail(e, "solve");
        if (perm && (e = launch_debug_expand(d, w, (int)N, perm + n0 * CW, group_start + n0 * CW,
                                             owner + n0 * CW, dw + n0 * CW, st)) != cudaSuccess)
            return cuda_fail(e, "debug expand");
        struct { void *dst; const void *src; size_t per; } cp[] = {
            {ngroups, w.ngroups, 4}, {lw, w.lw, 4 * CW}, {gw, w.gw, 4 * CW},
            {lr, w.lr, 4 * CR}, {qw, w.qw, 4 * CR}, {A, w.A, 4 * CC}, {QK, w.QK, 4 * CC}};
        for (auto &c : cp) {
            if (!c.dst) continue;
            e = cudaMemcpyAsync(static_cast<char *>(c.dst) + n0 * c.per, c.src, N * c.per,
                                cudaMemcpyDeviceToDevice, st);
            if (e != cudaSuccess) return cuda_fail(e, "debug copy");
        }
        if (dense_groups) {
            e = dense_gram(d) ? cudaMemcpyAsync(dense_groups + n0, w.ndense, 4 * N,
                                                  cudaMemcpyDeviceToDevice, st)
                                : cudaMemsetAsync(dense_groups + n0, 0, 4 * N, st);
            if (e != cudaSuccess) return cuda_fail(e, "debug copy");
        }
        // X and QX rows at the workspace pitch -> dense [C][C]
        const float *xsrc[2] = {w.X, w.QX};
        float *xdst[2] = {X, QX};
        for (int m = 0; m < 2; ++m) {
            if (!xdst[m]) continue;
            e = cudaMemcpy2DAsync(xdst[m] + n0 * CC, 4 * (size_t)d.C, xsrc[m], 4 * (size_t)d.xp,
                                  4 * (size_t)d.C, N * d.C, cudaMemcpyDeviceToDevice, st);
            if (e != cudaSuccess) return cuda_fail(e, "debug copy");
        }
    }
    return SDM_OK;
}

int sdm_get_device_status(const void *workspace, sdm_device_status *status, void *stream) {
    if (!workspace || !status) return fail(SDM_ERR_INVALID, "workspace and status must not be NULL");
    DevStatus h;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    status->code = h.code;
    status->first_bad_token = h.first_bad_plus1 - 1;
    status->bad_slots = (int64_t)h.bad_slots;
    status->repeated_write_slots = (int64_t)h.repeated_write_slots;
    return SDM_OK;
}

size_t sdm_host_workspace_bytes(const sdm_shape *shape) {
    Prepared pr;
    if (prepare(shape, pr)) return 0;
    g_err[0] = 0;
    return host_stage(pr.d, pr.bytes).bytes;
}

int sdm_write_read_host(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                        const void *write_w, const float *log_decay, const float *beta,
                        const void *v, const int32_t *read_slots, const void *read_w,
                        const int32_t *valid_tokens, void *readings, void *workspace,
                        size_t workspace_bytes, void *stream) {
    Prepared pr;
    int rc = prepare(shape, pr);
    if (rc) return rc;
    const Dims &d = pr.d;
    const HostStage hs = host_stage(d, pr.bytes);
    if (!bank || !write_slots || !write_w || !log_decay || !beta || !v || !read_slots ||
        !read_w || !readings)
        return fail(SDM_ERR_INVALID, "a required pointer is NULL");
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % kAlign)
        return fail(SDM_ERR_WORKSPACE, "workspace must be %zu-byte aligned device memory", kAlign);
    if (workspace_bytes < hs.bytes)
        return fail(SDM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes,
                    hs.bytes);
    // readings: mapped page-locked host memory, written by the kernels through its device address
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, readings);
    if (e != cudaSuccess || at.type != cudaMemoryTypeHost || !at.devicePointer) {
        cudaGetLastError();
        return fail(SDM_ERR_INVALID, "readings must be mapped page-locked host memory");
    }
    void *rdev = at.devicePointer;
    if (reinterpret_cast<uintptr_t>(bank) % 16 || reinterpret_cast<uintptr_t>(rdev) % 16)
        return fail(SDM_ERR_INVALID, "bank and readings must be 16-byte aligned");
    g_err[0] = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream), side;
    if ((rc = side_stream(&side))) return rc;
    char *base = static_cast<char *>(workspace);
    const size_t PT = (size_t)d.P * d.T, es = d.dtype == SDM_BF16 ? 2 : 4;
    Inputs in{bank, reinterpret_cast<const int32_t *>(base + hs.ws), base + hs.kw,
              reinterpret_cast<const float *>(base + hs.g),
              reinterpret_cast<const float *>(base + hs.beta), base + hs.v,
              reinterpret_cast<const int32_t *>(base + hs.rs), base + hs.qw,
              valid_tokens ? reinterpret_cast<const int32_t *>(base + hs.valid) : nullptr, rdev,
              nullptr};
    cudaEvent_t ev_start = nullptr, ev_v = nullptr;
    auto done = [&](int r) {
        if (ev_start) cudaEventDestroy(ev_start);
        if (ev_v) cudaEventDestroy(ev_v);
        return r;
    };
    if ((e = cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&ev_v, cudaEventDisableTiming)) != cudaSuccess)
        return done(cuda_fail(e, "event"));
    // the inputs of Phase 1 and the solve on `stream`, then v on the side stream (after them,
    // so that the two copies do not share the link; v has Phase 1 and the solve to land)
    struct { size_t off; const void *src; size_t bytes; } cp[] = {
        {hs.ws, write_slots, 4 * PT * d.W}, {hs.kw, write_w, es * PT * d.W},
        {hs.g, log_decay, 4 * PT * (d.gate ? 1 : d.W)}, {hs.beta, beta, 4 * PT},
        {hs.rs, read_slots, 4 * PT * d.R},  {hs.qw, read_w, es * PT * d.R},
        {hs.valid, valid_tokens, 4 * (size_t)d.P}};
    // all of them mapped page-locked memory (16-byte aligned, whole 16-byte units): one copy
    // kernel reads them through their device addresses; otherwise one transfer per array
    HostCopyTable tab;
    tab.n = 0;
    bool mapped = true;
    for (auto &c : cp) {
        if (!c.src) continue;
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, c.src) != cudaSuccess || pa.type != cudaMemoryTypeHost ||
            !pa.devicePointer || (reinterpret_cast<uintptr_t>(pa.devicePointer) & 15) ||
            (c.bytes & 15)) {
            cudaGetLastError();
            mapped = false;
            break;
        }
        tab.src[tab.n] = static_cast<const uint4 *>(pa.devicePointer);
        tab.dst[tab.n] = reinterpret_cast<uint4 *>(base + c.off);
        tab.n16[tab.n] = (long long)(c.bytes / 16);
        ++tab.n;
    }
    if (mapped) {
        if ((e = launch_host_copy(tab, st)) != cudaSuccess) return done(cuda_fail(e, "input copy"));
    } else {
        for (auto &c : cp) {
            if (!c.src) continue;
            if ((e = cudaMemcpyAsync(base + c.off, c.src, c.bytes, cudaMemcpyHostToDevice, st)) !=
                cudaSuccess)
                return done(cuda_fail(e, "input copy"));
        }
    }
    if ((e = cudaEventRecord(ev_start, st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(side, ev_start, 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(base + hs.v, v, es * PT * d.D, cudaMemcpyHostToDevice, side)) !=
            cudaSuccess ||
        (e = cudaEventRecord(ev_v, side)) != cudaSuccess)
        return done(cuda_fail(e, "v copy"));
    return done(run_forward(pr, in, workspace, st, nullptr, ev_v));
}

}  // extern "C"
