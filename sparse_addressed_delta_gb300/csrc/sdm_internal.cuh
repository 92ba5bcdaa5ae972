// Internal declarations of libsdm: workspace layout, kernel argument blocks and small
// device helpers shared by the kernels. Nothing here is part of the C ABI (include/sdm.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sdm.h"

namespace sdm {

constexpr int kMinChunk = 16;
constexpr int kMaxChunk = 256;
constexpr int kMaxWidth = 256;
constexpr int kRefSms = 152;            // GB300 SM count: sizes grids and slabs (shape-only)
constexpr size_t kAlign = 256;
constexpr size_t kSlabBudget = size_t(256) << 20;   // per-chunk Phase-1 state held at once
constexpr size_t kPhase1SmemMax = 110 * 1024;        // Phase-1 scratch kept on chip up to this
                                                     // (two CTAs per SM); larger: split Phase 1
constexpr size_t kPipeSmemMax = 224 * 1024;          // pipelined Phase 2 when two stages fit
constexpr long kSpinLimit = 1L << 22;   // mbarrier polls before a wait gives up (seconds at most)
constexpr int32_t kNoEntry = INT32_MIN;  // Work::wsl / rsl: no entry
constexpr float kDenseSpan = 64.f;      // widest running log-decay range of a dense Gram group
constexpr int kDenseMinChunk = 128;     // smallest chunk whose large groups go dense
// row pitch (floats) of the dense Gram factors: C rounded up to 16 bytes
__host__ __device__ __forceinline__ int dense_pitch(int C) { return (C + 3) & ~3; }

// Device status block at the start of the workspace (sdm_device_status, with the first bad
// token stored +1 so that a zero fill means "none").
struct DevStatus {
    int32_t code;
    int32_t first_bad_plus1;
    unsigned long long bad_slots;
    unsigned long long repeated_write_slots;
};

struct Dims {
    int P, T, C, S, D, W, R, Nt;
    int dtype;   // SDM_F32 / SDM_BF16
    int per_step;   // 1: Phase 2 as three kernels per step; 0: one fused kernel per slab
    int bwd;        // 1: Phase 1 also keeps what the backward reads (sorted rows, read plan)
    int xp;         // row pitch (floats) of X and QX in the workspace: C + 4 for the pipelined
                    // Phase 2 (one bulk copy lands rows at a bank-conflict-free pitch), else C
    int snapq;      // snapshot elements: 0 the bank dtype, 1 bfloat16 (float32 banks),
                    // 2 float8_e4m3fn (either bank dtype)
    int gate;       // 1: one log-decay per token ([P, T]) instead of one per write entry
    int shared;     // 1: one [S, D] bank for all streams (disjoint slot sets), else [P*S, D]
    long long spin; // mbarrier polls before a kernel's wait for its copies gives up
                    // (kSpinLimit unless sdm_set_wait_limit changed it); the waits that
                    // drain a kernel's copies before it returns always use kSpinLimit
};

// polls a kernel's waits make before giving up (process-wide; sdm_set_wait_limit)
long long wait_limit();

// first bank row of stream p: its own block of S rows, or row 0 of a shared bank
__host__ __device__ __forceinline__ size_t stream_row0(const Dims &d, int p) {
    return d.shared ? 0 : (size_t)p * d.S;
}

inline int x_row_pitch(const Dims &d) { return (d.per_step || d.bwd) ? d.C : d.C + 4; }

// Device pointers of one slab's workspace. N = ns * P chunks; chunk n of the slab is step
// (step0 + n / P) of stream n % P.
struct Work {
    DevStatus *status;
    // Phase-1 outputs, per chunk
    int32_t *perm;      // [N][CW]   entry e = t*W + j at each sorted position
    float *wdw;         // [N][CW]   DW weight at each sorted position
    int32_t *goff;      // [N][CW+4] group start positions, goff[ngroups] = n_entries (the
                        //           stride keeps every chunk's row 16-byte aligned)
    int4 *ng4;          // [N]       (ngroups, hot groups, 0, 0) as one 16-byte word
    int32_t *p1sel;     // [N]       radix buffer holding the sorted write row (scratch in HBM)
    int32_t *gord;      // [N][CW]   DW order: the hot groups (>= kHotGroup members, or C/8 if
                        //           more, for the per-step DW), then the others by size,
                        //           largest first
    int32_t *gslot;     // [N][CW]   slot of each group
    float *gfac;        // [N][CW]   exp(lend) of each group
    int32_t *ngroups;   // [N]
    int32_t *nvalid;    // [N]       valid tokens of the chunk
    float *gw;          // [N][CW]   token-major gather weights of the writes
    float *qw;          // [N][CR]   token-major gather weights of the reads
    int32_t *minfo;     // [N][CW]   sorted position: t | j << 8 | head << 16 | tail << 17
    // token-major source of each entry's B0 piece for the pipelined Phase 2 (bulk-copied):
    // v >= 0 the bank row v; v = -1 - g: the new piece of group g of the same stream's previous
    // step in the slab (that step wrote the row); kNoEntry: no entry (slot outside [0, S) or a
    // token past the valid ones). Phase 1 writes the slots, the solve kernel the links.
    int32_t *wsl;       // [N][CW]
    int32_t *rsl;       // [N][CR]
    float *lw;          // [N][CW]   token-major running log-decay of the writes
    float *lr;          // [N][CR]   token-major running log-decay of the reads
    float *A, *QK;      // [N][C*C]
    float *X, *QX;      // [N][C][xp]
    // Phase-1 scratch, per Phase-1 CTA
    unsigned long long *keys;   // [G][2][CW]
    int32_t *inv;       // [G][CW]  sorted position of each entry
    float *lws;         // [G][CW]  running log-decay at each sorted position
    int32_t *pgid;      // [G][CW]  group id of each sorted position
    int32_t *pgs;       // [G][CW]  group start position of each sorted position
    float *lend;        // [G][CW]  log-decay total of each group
    float *kf;          // [G][CW]  write weight of each entry as float (0 for a bad slot);
                        //          chunks whose Phase-1 scratch is on chip only
    float2 *gk;         // [G][CW]  (log-decay, write weight) of each entry, entry order (0, 0
                        //          for a bad slot); chunks whose Phase-1 scratch is in HBM
    int32_t *rlo;       // [G][CR]  first write position of the read's slot group
    int32_t *rhi;       // [G][CR]  last write position at or before the read's token (-1: none)
    // dense Gram groups of the chunks whose Phase-1 scratch is in global memory (sized only
    // then): large groups whose pair sums are taken as the product of two per-token factors
    // around a reference log-decay of the group (k_gram_dense), DC = C of them at most
    int32_t *dpos;      // [G][CW]  dense index of each sorted position's group (-1: pair sums)
    float *dref;        // [N][DC]  reference log-decay of each dense group
    int32_t *ndense;    // [N]      dense groups of the chunk
    float *dka;         // [N][C][dense_pitch] sum over the token's writes of group h of
                        //           k exp(lw - ref)
    float *dkb;         // [N][C][dense_pitch] the same with exp(ref - lw)
    float *dkq;         // [N][C][dense_pitch] sum over the token's reads of group h of
                        //           q exp(lr - ref)
    // kept for the backward (sized only when Dims::bwd)
    unsigned long long *wkey;   // [N][CW]  sorted write keys (slot << 32 | t << 8 | j)
    float *wlws;        // [N][CW]   running log-decay at each sorted position
    int32_t *wpgs;      // [N][CW]   group start of each sorted position
    int32_t *wpge;      // [N][CW]   group end (exclusive) of each sorted position
    float *dwt;         // [N][CW]   token-major DW weights
    unsigned long long *rkey;   // [N][CR]  sorted read keys (slot << 32 | t << 8 | i)
    int32_t *rgoff;     // [N][CR+1] read group starts, rgoff[rng] = n_reads
    int32_t *rgslot;    // [N][CR]   slot of each read group
    int32_t *rng;       // [N]       read groups
    unsigned long long *rkeys;  // [G][2][CR] read sort scratch
    // backward step buffers (sized only when Dims::bwd)
    float *bu;          // [P][C*D]  delta_v recomputed
    float *bup;         // [P][C*D]  u_pre recomputed
    float *bdret;       // [P][C*D]  gradient of retrieved
    float *bdo;         // [P][C*D]  upstream readings gradient, zero past the valid tokens
    float *bdX;         // [P][C*C]  dX, then dX + QK^T dQX
    float *bdQX;        // [P][C*C]
    float *bdQK;        // [P][C*C]
    float *bT;          // [P][C*C]  X^T (dX + QK^T dQX)
    float *bdA;         // [P][C*C]  dL, then beta * dL (strictly lower)
    float *bdb2;        // [P][DT][C] per-column-tile partial <du_pre, v - retrieved>
    float *bddw;        // [P][CW]   <dB1[s], u_t> per write entry (token-major)
    float *bdgw;        // [P][CW]   <dretrieved_t, B0[s]> per write entry
    float *bdqw;        // [P][CR]   <dO_t, B0[r]> per read entry
    float *bdfac;       // [P][CW]   <dB1[s], B0[s]> at each group's head position
    float *bdlam;       // [P][CW]   d(log-decay running sum) at each sorted write position
    float *bdlr;        // [P][CR]   d(read running log-decay) at each sorted read position
    float *bdgate;      // [P][CW]   per-entry log-decay gradients of a per-token gate, summed
                        //           per token at the end of the step
    // Phase-2 step buffers
    float *ret;         // [P][C*D]
    float *inter;       // [P][C*D]
    float *dv;          // [P][C*D]
    int ns;             // steps per slab
    int G;              // Phase-1 CTAs
};

struct Inputs {
    void *bank;
    const int32_t *ws;
    const void *kw;
    const float *g;
    const float *beta;
    const void *v;
    const int32_t *rs;
    const void *qw;
    const int32_t *valid;   // may be null
    void *readings;
    void *snap;             // saving forward: [Nt*P][C*W][D] bank dtype, B0 rows of the written
                            // slots at their group's tail position; null otherwise
};

// Sets the thread's sdm_last_error() message; returns code.
int set_error(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));

// Outputs of the backward (all float32 except grad_readings, which is in the bank dtype).
struct BwdOut {
    const void *grad_readings;   // [P, T, D] upstream gradient of the readings
    float *grad_bank;            // [P*S, D] in: d/d(final bank); out: d/d(initial bank)
    float *grad_v;               // [P, T, D]
    float *grad_beta;            // [P, T]
    float *grad_write_w;         // [P, T, W]
    float *grad_log_decay;       // [P, T, W]
    float *grad_read_w;          // [P, T, R]
};

// ---------------------------------------------------------------------------------------
// host-side layout (api.cu)
// ---------------------------------------------------------------------------------------
size_t layout_bytes(const Dims &d, int ns, int G);
Work layout_assign(const Dims &d, int ns, int G, void *base);
int phase1_ctas(const Dims &d, int ns);

// ---------------------------------------------------------------------------------------
// launchers (one per kernel family); every one returns cudaGetLastError()
// ---------------------------------------------------------------------------------------
cudaError_t launch_phase1(const Dims &d, const Inputs &in, const Work &w, int step0, int nsteps,
                          cudaStream_t st);
cudaError_t launch_solve(const Dims &d, const Inputs &in, const Work &w, int step0, int nsteps,
                         cudaStream_t st);
cudaError_t launch_gather(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                          cudaStream_t st);
cudaError_t launch_dualmm(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                          cudaStream_t st);
cudaError_t launch_dw(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                      cudaStream_t st);
// the per-step dual matmul on tcgen05 tensor cores (C a multiple of 128); the gather then
// writes u_pre transposed ([P][D][C], K-major rows for the tensor cores)
__host__ __device__ inline bool dualmm_tc_fits(const Dims &d) {
    return d.per_step && d.C % 128 == 0 && d.D % 64 == 0;
}
cudaError_t launch_dualmm_tc(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                             cudaStream_t st);
cudaError_t launch_phase2_fused(const Dims &d, const Inputs &in, const Work &w, int step0,
                                int nsteps, cudaStream_t st);
size_t phase2_pipe_smem(const Dims &d);
// Phase-1 scratch in global memory: steps 3 and 4 run in a second kernel over row blocks
bool phase1_split(const Dims &d);
// chunks whose Phase-1 scratch is in global memory and whose large groups' Gram sums go dense
// (k_gram_dense): C >= kDenseMinChunk
bool dense_gram(const Dims &d);
// sdm_write_read_host: arrays copied from mapped page-locked host memory by one kernel
// (device addresses of the host pages; 16-byte aligned; sizes in 16-byte units)
struct HostCopyTable {
    const uint4 *src[8];
    uint4 *dst[8];
    long long n16[8];
    int n;
};
cudaError_t launch_host_copy(const HostCopyTable &t, cudaStream_t st);
bool phase2_fused_fits(const Dims &d);
cudaError_t launch_backward_step(const Dims &d, const Inputs &in, const Work &w,
                                 const BwdOut &o, int step0, int ti, cudaStream_t st);
cudaError_t launch_debug_expand(const Dims &d, const Work &w, int nchunks, int32_t *perm,
                                uint8_t *gstart, uint8_t *owner, float *dw_tok,
                                cudaStream_t st);

// ---------------------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Loads N consecutive elements of type T (N * sizeof(T) a power of two, 2..64 bytes,
// address aligned to it) as floats.
template <typename T, int N, bool NC>
__device__ __forceinline__ void load_vec(const T *p, float (&o)[N]) {
    constexpr int BYTES = N * (int)sizeof(T);
    static_assert(BYTES >= 2 && BYTES <= 64 && (BYTES & (BYTES - 1)) == 0, "vector size");
    if constexpr (BYTES >= 16) {
        constexpr int V = BYTES / 16;
        const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            uint4 u = NC ? __ldg(q + i) : q[i];
            const T *e = reinterpret_cast<const T *>(&u);
            constexpr int PER = 16 / (int)sizeof(T);
#pragma unroll
            for (int k = 0; k < PER; ++k) o[i * PER + k] = to_f32(e[k]);
        }
    } else if constexpr (BYTES == 8) {
        const uint2 *q = reinterpret_cast<const uint2 *>(p);
        uint2 u = NC ? __ldg(q) : *q;
        const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int k = 0; k < N; ++k) o[k] = to_f32(e[k]);
    } else if constexpr (BYTES == 4) {
        const unsigned *q = reinterpret_cast<const unsigned *>(p);
        unsigned u = NC ? __ldg(q) : *q;
        const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int k = 0; k < N; ++k) o[k] = to_f32(e[k]);
    } else {
        const unsigned short *q = reinterpret_cast<const unsigned short *>(p);
        unsigned short u = NC ? __ldg(q) : *q;
        o[0] = to_f32(*reinterpret_cast<const T *>(&u));
    }
}

template <typename T, int N>
__device__ __forceinline__ void store_vec(T *p, const float (&x)[N]) {
    constexpr int BYTES = N * (int)sizeof(T);
    static_assert(BYTES >= 2 && BYTES <= 64 && (BYTES & (BYTES - 1)) == 0, "vector size");
    alignas(16) T tmp[N];
#pragma unroll
    for (int k = 0; k < N; ++k) tmp[k] = from_f32<T>(x[k]);
    if constexpr (BYTES >= 16) {
        uint4 *q = reinterpret_cast<uint4 *>(p);
        const uint4 *s = reinterpret_cast<const uint4 *>(tmp);
#pragma unroll
        for (int i = 0; i < BYTES / 16; ++i) q[i] = s[i];
    } else if constexpr (BYTES == 8) {
        *reinterpret_cast<uint2 *>(p) = *reinterpret_cast<const uint2 *>(tmp);
    } else if constexpr (BYTES == 4) {
        *reinterpret_cast<unsigned *>(p) = *reinterpret_cast<const unsigned *>(tmp);
    } else {
        p[0] = tmp[0];
    }
}

// N consecutive float8_e4m3fn snapshot elements (N a power of two, 1..16; p aligned to N
// bytes): converted to nearest even, saturating at the largest finite value, and back
template <int N>
__device__ __forceinline__ void store_fp8(unsigned char *p, const float (&x)[N]) {
    alignas(16) unsigned char b[N < 2 ? 2 : N];
    if constexpr (N == 1) {
        b[0] = (unsigned char)__nv_cvt_float_to_fp8(x[0], __NV_SATFINITE, __NV_E4M3);
        p[0] = b[0];
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 2) {
            const __nv_fp8x2_storage_t two =
                __nv_cvt_float2_to_fp8x2(make_float2(x[c], x[c + 1]), __NV_SATFINITE, __NV_E4M3);
            b[c] = (unsigned char)(two & 0xff);
            b[c + 1] = (unsigned char)(two >> 8);
        }
        if constexpr (N == 2) *reinterpret_cast<unsigned short *>(p) = *reinterpret_cast<unsigned short *>(b);
        else if constexpr (N == 4) *reinterpret_cast<unsigned *>(p) = *reinterpret_cast<unsigned *>(b);
        else if constexpr (N == 8) *reinterpret_cast<uint2 *>(p) = *reinterpret_cast<uint2 *>(b);
        else *reinterpret_cast<uint4 *>(p) = *reinterpret_cast<uint4 *>(b);
    }
}

template <int N>
__device__ __forceinline__ void load_fp8(const unsigned char *p, float (&x)[N]) {
    alignas(16) unsigned char b[N < 2 ? 2 : N];
    if constexpr (N == 1) b[0] = p[0];
    else if constexpr (N == 2) *reinterpret_cast<unsigned short *>(b) = *reinterpret_cast<const unsigned short *>(p);
    else if constexpr (N == 4) *reinterpret_cast<unsigned *>(b) = *reinterpret_cast<const unsigned *>(p);
    else if constexpr (N == 8) *reinterpret_cast<uint2 *>(b) = *reinterpret_cast<const uint2 *>(p);
    else *reinterpret_cast<uint4 *>(b) = *reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int c = 0; c < N; ++c) {
        const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b[c], __NV_E4M3);
        x[c] = __half2float(__half(h));
    }
}

// Exact e / W for 0 <= e < 2^16 and 1 <= W <= 256 with m = ceil(2^24 / W): the rounding error
// of the reciprocal is below e / 2^24 < 1/256 <= 1/W, which never carries past an integer.
__host__ __device__ __forceinline__ unsigned div_magic(int W) {
    return (unsigned)(((1u << 24) + (unsigned)W - 1u) / (unsigned)W);
}
__device__ __forceinline__ int div_by(int e, unsigned magic) {
    return (int)(((unsigned long long)(unsigned)e * magic) >> 24);
}

__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gsrc) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// TF32 tensor-core product of a 16 x 8 tile, f32 accumulation (mma.sync m16n8k8, PTX ISA
// fragment layout: g = lane / 4, i = lane % 4; A: a0 (g, i), a1 (g + 8, i), a2 (g, i + 4),
// a3 (g + 8, i + 4); B: b0 (i, g), b1 (i + 4, g); C: c0 (g, 2i), c1 (g, 2i + 1), c2 (g + 8, 2i),
// c3 (g + 8, 2i + 1)). Float32 operands go through the 3xTF32 split (hi*lo + lo*hi + hi*hi).
// TF32 operand of a finite float: round to nearest, ties away from zero, on the bit pattern
// (add half a unit in the last of the ten kept mantissa bits to the magnitude, then clear the
// thirteen low bits; a carry into the exponent is the correct rounding up). Two integer
// operations, where the conversion instruction costs more inside the dual matmul's loop.
__device__ __forceinline__ unsigned to_tf32(float x) {
    return (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], const unsigned (&a)[4],
                                         const unsigned (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Bulk global -> shared copies completed on an mbarrier (the TMA unit moves the bytes; one
// thread issues a copy). Addresses 16-byte aligned, sizes multiples of 16.
__device__ __forceinline__ unsigned smem_u32(const void *p) {
    return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// arrive on `bar` once every cp.async this thread issued so far has landed (the arrival is
// counted in the barrier's initial count)
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(unsigned long long *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes,
                                         unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase of `parity` to complete; false if it did not within `limit` polls.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, unsigned parity,
                                                  long long limit = kSpinLimit) {
    for (long long it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// Orders this thread's earlier shared-memory accesses (generic proxy) before its later bulk
// copies (async proxy) into the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__host__ __device__ __forceinline__ int goff_stride(int CW) { return CW + 4; }

// Dynamic shared memory limit of a kernel (the driver keeps choosing the carveout: forcing the
// largest one measured slower for the pipelined Phase 2, whose gather uses the L1 that is left)
template <typename K>
inline void set_kernel_smem(K kern, size_t bytes) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
// a group with at least kHotGroup members is summed by a whole warp in the pipelined DW
constexpr int kHotGroup = 16;

__device__ __forceinline__ int chunk_valid(const int32_t *valid, int p, int T, int tok0, int C) {
    int v = valid ? valid[p] : T;
    v = v < 0 ? 0 : (v > T ? T : v);
    int n = v - tok0;
    return n < 0 ? 0 : (n > C ? C : n);
}

}  // namespace sdm
