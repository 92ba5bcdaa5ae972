// Phase 2 fused into one persistent kernel per slab: every CTA owns one stream p and one
// 16-byte slice of bank columns, and runs all the slab's steps for it (gather -> dual matmul ->
// DW, sparse-delta-memory 2.0.0, phase2_kernels.py module docstring).
//
// Why this is exact and needs no inter-CTA synchronization: given Phase 1 and the solve
// (which depend only on slots, weights and decays), every operation of Phase 2 acts on each
// bank column independently -- retrieved, inter, u = beta (v - retrieved), X u, QX u and the
// decay-and-write are all column-wise. A CTA therefore reads and writes only its own columns
// of its own stream's rows, step after step, and only ever waits on its own threads.
//
// The bank rows a step writes reach the next step without a memory round trip: the solve kernel
// links each entry of a chunk to the group of the previous step that writes its slot, and the
// DW keeps every group's new piece in shared memory; every other row is loaded from the bank
// one step early (it is final once the step before has ended: ordered by the closing barrier,
// plain loads, no read-only cache path). The kernel runs when two stages of per-step metadata
// fit in shared memory (launch_phase2_fused says whether); larger chunks use the per-step
// kernels of phase2.cu.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

template <typename BT>
struct Vec16 {                  // one 16-byte piece of a bank row
    static constexpr int N = 16 / sizeof(BT);
};

// Pipelined variant for chunks whose per-step metadata fits in shared memory twice: a
// producer warp brings the next step's slots/links, weights, member records, DW order, X and
// QX into the other stage with bulk copies (the TMA unit; part A, the slots and links, on its
// own mbarrier so that the early loads can start) and its v pieces and beta with cp.async,
// while the 16 compute warps run the current step. The gather keeps the B0 pieces of the
// written rows in shared memory; the dual matmul runs on the tensor cores; the DW gives each
// hot group a warp and every other group a thread, which sum the members in sorted order from
// shared memory and write the row once:
//   B[s] = (sum of dw * delta_v over the group, sorted order) + exp(lend) * B0[s].
// ---------------------------------------------------------------------------------------
constexpr int NT2 = 512;          // compute threads (16 warps)
constexpr int NW2 = NT2 / 32;
constexpr int NP2 = NT2 + 32;     // + one producer warp that only issues the stage copies

// barrier 1: the compute warps only (the producer warp never waits on it)
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NT2) : "memory");
}
__device__ __forceinline__ bool compute_sync_or(bool v) {
    unsigned r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
        " selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((unsigned)v), "n"(NT2)
        : "memory");
    return r != 0;
}

struct StageLayout {     // byte offsets inside one stage (every array 16-byte aligned)
    int wslot, wgw, rslot, rqw, minfo, mdw, gslot, gfac, goff, gord, scal, xs, qs, vpc, beta, bytes;
};

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline int x_pitch(int C) { return C + 4; }

__host__ __device__ inline StageLayout stage_layout(int C, int W, int R) {
    StageLayout L;
    const int CW = C * W, CR = C * R, XP = x_pitch(C);
    int o = 0;
    L.wslot = o; o = align16(o + 4 * CW);
    L.wgw = o; o = align16(o + 4 * CW);
    L.rslot = o; o = align16(o + 4 * CR);
    L.rqw = o; o = align16(o + 4 * CR);
    L.minfo = o; o = align16(o + 4 * CW);
    L.mdw = o; o = align16(o + 4 * CW);
    L.gslot = o; o = align16(o + 4 * CW);
    L.gfac = o; o = align16(o + 4 * CW);
    L.goff = o; o = align16(o + 4 * goff_stride(CW));
    L.gord = o; o = align16(o + 4 * CW);
    L.scal = o; o = align16(o + 16);
    L.xs = o; o = align16(o + 4 * C * XP);
    L.qs = o; o = align16(o + 4 * C * XP);
    L.vpc = o; o = align16(o + 16 * C);
    L.beta = o; o = align16(o + 4 * C);
    L.bytes = o;
    return L;
}

// Bytes the bulk copies of one stage move: part A (the entries' slots and links, which the
// previous step needs for its early loads) and part B (everything else before vpc; X and QX
// whole, padded rows)
__host__ __device__ inline unsigned stage_bytes_a(int C, int W, int R) {
    return (unsigned)(4 * (C * W + C * R));
}
__host__ __device__ inline unsigned stage_bytes_b(int C, int W, int R) {
    const int CW = C * W, CR = C * R;
    return (unsigned)(4 * (6 * CW + CR + goff_stride(CW)) + 16 + 2 * 4 * C * x_pitch(C));
}

// delta_v rows in shared memory are kDvPitch floats apart: 48 bytes spread a warp's random-row
// 16-byte reads over all eight 16-byte bank groups
constexpr int kDvPitch = 12;

// Bytes after the two stages: u_pre, inter [C][V] f32, delta_v [C][kDvPitch] f32, the B0 pieces
// [CW][16 B], the DW's new piece per group [CW][16 B] and the stage mbarriers (fullA[2],
// fullB[2], empty[2]).
__host__ __device__ inline int pipe_tail_bytes(int C, int W, int V) {
    return 2 * 4 * C * V + 4 * C * kDvPitch + 2 * 16 * C * W + 48;
}

// ---------------------------------------------------------------------------------------
// the per-step dual matmul runs on the tensor cores with mma.sync (to_tf32 / mma_tf32 in the
// internal header): a 64 x 64 by 64 x 8 product per CTA and step is far below a tcgen05 tile
// ---------------------------------------------------------------------------------------
template <typename BT>
__device__ __forceinline__ void piece_to_f32(const uint4 &u, float (&o)[16 / sizeof(BT)]) {
    if constexpr (sizeof(BT) == 2) {
        const unsigned wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = __uint_as_float(wv[i] << 16);
            o[2 * i + 1] = __uint_as_float(wv[i] & 0xffff0000u);
        }
    } else {
        o[0] = __uint_as_float(u.x);
        o[1] = __uint_as_float(u.y);
        o[2] = __uint_as_float(u.z);
        o[3] = __uint_as_float(u.w);
    }
}

// the 16-byte bank piece of V floats, rounded to the bank type exactly as store_vec does
template <typename BT>
__device__ __forceinline__ uint4 pack_piece(const float (&o)[16 / sizeof(BT)]) {
    alignas(16) BT tmp[16 / sizeof(BT)];
#pragma unroll
    for (int k = 0; k < (int)(16 / sizeof(BT)); ++k) tmp[k] = from_f32<BT>(o[k]);
    return *reinterpret_cast<const uint4 *>(tmp);
}

// a += w * x for two columns at once (one packed FFMA2, each half rounded like fmaf)
__device__ __forceinline__ void fma2(float &a0, float &a1, float w, float x0, float x1) {
    const float2 r = __ffma2_rn(make_float2(w, w), make_float2(x0, x1), make_float2(a0, a1));
    a0 = r.x;
    a1 = r.y;
}

template <int V>
__device__ __forceinline__ void add_piece(float (&acc)[V], float w, const float (&x)[V]) {
#pragma unroll
    for (int c = 0; c < V; c += 2) fma2(acc[c], acc[c + 1], w, x[c], x[c + 1]);
}

// Reduce-scatter of N values over the 2 * off lanes of a group (xor butterflies, off halving):
// at each level a lane keeps the half its lane bit selects and adds the partner's copy of it,
// so the levels move N/2, N/4, ... values instead of N. When one value is left, further
// levels add it across the remaining lanes and only the lowest of them emits it. Calls
// emit(index in 0..N-1, sum) for every value the lane ends up owning. Fixed order: bitwise
// reproducible.
template <int N, typename F>
__device__ __forceinline__ void reduce_scatter(float (&v)[N], int off, int lane, int base, F &&emit) {
    if constexpr (N == 1) {
        const int span = off;   // lanes below this bit hold copies after the butterflies
        for (; off > 0; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        if (span == 0 || (lane & (2 * span - 1)) == 0) emit(base, v[0]);
    } else {
        if (off == 0) {
#pragma unroll
            for (int i = 0; i < N; ++i) emit(base + i, v[i]);
            return;
        }
        const bool up = (lane & off) != 0;
        float h[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float send = up ? v[i] : v[i + N / 2];
            const float keep = up ? v[i + N / 2] : v[i];
            h[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        reduce_scatter<N / 2>(h, off >> 1, lane, base + (up ? N / 2 : 0), emit);
    }
}

template <typename BT>
__global__ void __launch_bounds__(NP2) k_phase2_pipe(Dims d, Inputs in, Work w, int step0,
                                                    int nsteps) {
    constexpr int V = Vec16<BT>::N;
    extern __shared__ __align__(16) unsigned char psm[];
    const int C = d.C, D = d.D, W = d.W, R = d.R, CW = C * W, CR = C * R;
    const int XP = x_pitch(C);
    const StageLayout L = stage_layout(C, W, R);
    const int slices = D / V;
    const int p = blockIdx.x / slices;
    const int c0 = (blockIdx.x - p * slices) * V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    float *us = reinterpret_cast<float *>(psm + 2 * L.bytes);   // [C][V]
    float *is = us + C * V;                                      // [C][V]
    float *dvs = is + C * V;                                     // [C][kDvPitch]
    uint4 *b0s = reinterpret_cast<uint4 *>(dvs + C * kDvPitch);  // [CW] B0 pieces (raw)
    uint4 *dwout = b0s + CW;                                      // [CW] new piece per group
    // fullA[st]: the slots/links of stage st landed (1 expect-tx arrival and their bytes);
    // fullB[st]: the rest landed (1 expect-tx arrival + 32 producer-lane cp.async arrivals and
    // the bulk bytes); empty[st]: the compute warps are done with stage st (1 arrival)
    unsigned long long *fullA = reinterpret_cast<unsigned long long *>(dwout + CW);
    unsigned long long *fullB = fullA + 2;
    unsigned long long *empty = fullA + 4;

    BT *bank = static_cast<BT *>(in.bank) + stream_row0(d, p) * D + c0;
    const BT *vin = static_cast<const BT *>(in.v);
    BT *out = static_cast<BT *>(in.readings);
    const unsigned S = (unsigned)d.S;
    int vp = in.valid ? in.valid[p] : d.T;
    vp = vp < 0 ? 0 : (vp > d.T ? d.T : vp);
    const unsigned magQ = div_magic(C / 4 > 0 ? C / 4 : 1);

    auto nvalid_of = [&](int ti) {
        const int r = vp - ti * C;
        return r < 0 ? 0 : (r > C ? C : r);
    };

    // stage st for step ls, issued by the producer warp: lanes 0 and 1 bulk-copy the slots and
    // links (part A), then lanes 0..10 the other workspace arrays (part B; 16-byte aligned chunk
    // offsets, C % 16 == 0); every lane cp.asyncs the v pieces and beta of its tokens and then
    // arrives on fullB[st] when those have landed
    auto issue = [&](int ls, int st) {
        unsigned char *b = psm + st * L.bytes;
        const int ti = step0 + ls;
        const int n = ls * d.P + p;
        const int nv = nvalid_of(ti);
        const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;
        unsigned long long *barA = fullA + st, *barB = fullB + st;
        if (lane == 0) {
            mbar_arrive_expect_tx(barA, stage_bytes_a(C, W, R));
            mbar_arrive_expect_tx(barB, stage_bytes_b(C, W, R));
        }
        __syncwarp();
        if (lane == 0) bulk_g2s(b + L.wslot, w.wsl + (size_t)n * CW, 4u * CW, barA);
        if (lane == 1) bulk_g2s(b + L.rslot, w.rsl + (size_t)n * CR, 4u * CR, barA);
        __syncwarp();
        if (lane < 11) {
            const void *src;
            int off, bytes;
            switch (lane) {
                case 0: src = w.gw + (size_t)n * CW; off = L.wgw; bytes = 4 * CW; break;
                case 1: src = w.qw + (size_t)n * CR; off = L.rqw; bytes = 4 * CR; break;
                case 2: src = w.minfo + (size_t)n * CW; off = L.minfo; bytes = 4 * CW; break;
                case 3: src = w.wdw + (size_t)n * CW; off = L.mdw; bytes = 4 * CW; break;
                case 4: src = w.gslot + (size_t)n * CW; off = L.gslot; bytes = 4 * CW; break;
                case 5: src = w.gfac + (size_t)n * CW; off = L.gfac; bytes = 4 * CW; break;
                case 6:
                    src = w.goff + (size_t)n * goff_stride(CW);
                    off = L.goff;
                    bytes = 4 * goff_stride(CW);
                    break;
                case 7: src = w.ng4 + n; off = L.scal; bytes = 16; break;
                case 8: src = w.X + (size_t)n * C * XP; off = L.xs; bytes = 4 * C * XP; break;
                case 9: src = w.gord + (size_t)n * CW; off = L.gord; bytes = 4 * CW; break;
                default: src = w.QX + (size_t)n * C * XP; off = L.qs; bytes = 4 * C * XP; break;
            }
            bulk_g2s(b + off, src, (unsigned)bytes, barB);
        }
        for (int t = lane; t < nv; t += 32) {
            cp_async16(b + L.vpc + 16 * t, vin + (tok0 + t) * D + c0);
            cp_async4(b + L.beta + 4 * t, in.beta + tok0 + t);
        }
        cp_async_mbar_arrive_noinc(barB);
    };
    // both parts of stage (ls & 1) for step ls, within `lim` polls each (the compute warps'
    // waits use the call's limit; the producer's drain before it leaves the default one)
    auto wait_stage = [&](int ls, long long lim) {
        const unsigned par = (unsigned)(ls >> 1) & 1u;
        return mbar_wait_bounded(fullA + (ls & 1), par, lim) &&
               mbar_wait_bounded(fullB + (ls & 1), par, lim);
    };

    if (tid == 0) {
        mbar_init(fullA, 1);
        mbar_init(fullA + 1, 1);
        mbar_init(fullB, 33);
        mbar_init(fullB + 1, 33);
        mbar_init(empty, 1);
        mbar_init(empty + 1, 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW2) {
        // producer: stage st is reissued once the compute warps released it (step ls - 2)
        int issued = 0;
        for (int ls = 0; ls < nsteps; ++ls) {
            const int st = ls & 1;
            if (ls >= 2 && !mbar_wait_bounded(empty + st, (unsigned)((ls - 2) >> 1) & 1u, d.spin)) {
                if (lane == 0) atomicCAS(&w.status->code, 0, (int)SDM_ERR_TIMEOUT);
                break;
            }
            issue(ls, st);
            issued = ls + 1;
        }
        // leave only after the last issued copies of both stages have landed
        for (int ls = issued - 2 < 0 ? 0 : issued - 2; ls < issued; ++ls) wait_stage(ls, kSpinLimit);
        cp_async_wait<0>();
        return;
    }

    // gather mapping: token gt = tid / tpt; the first half of its tpt lanes sum its write
    // entries and the second half its read entries (entry q = hl, hl + half, ... of the kind);
    // tpt is a power of two with tpt * C <= NT2 (C <= 256 gives tpt >= 2), so one pass covers
    // every token
    int tpt = NT2 / C;
    if (tpt > 32) tpt = 32;
    while (tpt & (tpt - 1)) tpt &= tpt - 1;
    const int half = tpt >> 1;
    const int sub = tid % tpt;
    const int gt = tid / tpt;
    const bool rd = sub >= half;     // this lane sums read entries (else write entries)
    const int hl = rd ? sub - half : sub;
    const int ne = rd ? R : W;       // entries of the lane's kind per token

    // The first PF entries of a lane are fetched one step ahead: while step ls computes, the
    // pieces of step ls + 1 are loaded into registers, except for entries linked to a group of
    // step ls (its slot is written there), which take that group's new piece from dwout. Every
    // other bank row is final for step ls + 1 once step ls - 1 has ended, so the early load
    // reads the right value.
    constexpr int PF = 4;
    uint4 pf[PF];
    int lk[PF];   // -2: no entry; -1: piece in pf; >= 0: dwout[lk]
    auto prefetch = [&](int ls_n, const unsigned char *bn) {
        const int nvn = nvalid_of(step0 + ls_n);
        const int32_t *sl = rd ? reinterpret_cast<const int32_t *>(bn + L.rslot) + gt * R
                               : reinterpret_cast<const int32_t *>(bn + L.wslot) + gt * W;
#pragma unroll
        for (int k = 0; k < PF; ++k) {
            const int q = hl + k * half;
            lk[k] = -2;
            if (gt < nvn && q < ne) {
                const int v = sl[q];
                if (v >= 0) {
                    lk[k] = -1;
                    pf[k] = *reinterpret_cast<const uint4 *>(bank + (size_t)v * D);
                } else if (v != kNoEntry) {
                    lk[k] = -1 - v;
                }
            }
        }
    };

    // the first stage; each later one is awaited by the step before it, ahead of its closing
    // barrier
    if (compute_sync_or(!wait_stage(0, d.spin))) {
        // a stage did not land: report and stop (the producer drains its own copies)
        if (tid == 0) atomicCAS(&w.status->code, 0, (int)SDM_ERR_TIMEOUT);
        return;
    }
    for (int ls = 0; ls < nsteps; ++ls) {
        const int st = ls & 1;
        const unsigned char *b = psm + st * L.bytes;
        const int32_t *swslot = reinterpret_cast<const int32_t *>(b + L.wslot);
        const float *swgw = reinterpret_cast<const float *>(b + L.wgw);
        const int32_t *srslot = reinterpret_cast<const int32_t *>(b + L.rslot);
        const float *srqw = reinterpret_cast<const float *>(b + L.rqw);
        const BT *svpc = reinterpret_cast<const BT *>(b + L.vpc);
        const float *sbeta = reinterpret_cast<const float *>(b + L.beta);
        const float *xs = reinterpret_cast<const float *>(b + L.xs);
        const float *qs = reinterpret_cast<const float *>(b + L.qs);
        const int32_t *sminfo = reinterpret_cast<const int32_t *>(b + L.minfo);
        const float *smdw = reinterpret_cast<const float *>(b + L.mdw);
        const int32_t *sgslot = reinterpret_cast<const int32_t *>(b + L.gslot);
        const float *sgfac = reinterpret_cast<const float *>(b + L.gfac);
        const int ti = step0 + ls;
        const int nv = nvalid_of(ti);
        const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;
        if (ls == 0) prefetch(0, b);

        // ---- gather (the write pieces are also kept as B0 for the DW) ----
        // each lane adds its entries in entry order: the PF early ones, then the rest fetched
        // now, GB at a time before any is used; a shuffle tree then sums the lanes of the kind
        {
            constexpr int GB = 4;
            float acc[V];
#pragma unroll
            for (int c = 0; c < V; ++c) acc[c] = 0.f;
            if (gt < nv) {
                const int32_t *sl = rd ? srslot + gt * R : swslot + gt * W;
                const float *wt = rd ? srqw + gt * R : swgw + gt * W;
                uint4 *b0 = b0s + gt * W;
#pragma unroll
                for (int k = 0; k < PF; ++k) {
                    const int q = hl + k * half;
                    if (q < ne) {
                        const uint4 u = lk[k] >= 0 ? dwout[lk[k]]
                                                   : (lk[k] == -1 ? pf[k] : make_uint4(0u, 0u, 0u, 0u));
                        if (!rd) b0[q] = u;
                        if (lk[k] != -2) {
                            float x[V];
                            piece_to_f32<BT>(u, x);
                            add_piece<V>(acc, wt[q], x);
                        }
                    }
                }
                for (int q0 = hl + PF * half; q0 < ne; q0 += GB * half) {
                    uint4 u[GB];
                    bool has[GB];
#pragma unroll
                    for (int k = 0; k < GB; ++k) {
                        const int q = q0 + k * half;
                        u[k] = make_uint4(0u, 0u, 0u, 0u);
                        has[k] = false;
                        if (q < ne) {
                            const int v = sl[q];
                            if (v >= 0) {
                                u[k] = *reinterpret_cast<const uint4 *>(bank + (size_t)v * D);
                                has[k] = true;
                            } else if (v != kNoEntry) {
                                u[k] = dwout[-1 - v];
                                has[k] = true;
                            }
                        }
                    }
#pragma unroll
                    for (int k = 0; k < GB; ++k) {
                        const int q = q0 + k * half;
                        if (q < ne) {
                            if (!rd) b0[q] = u[k];
                            if (has[k]) {
                                float x[V];
                                piece_to_f32<BT>(u[k], x);
                                add_piece<V>(acc, wt[q], x);
                            }
                        }
                    }
                }
            }
            // sum over the kind's lanes; each lane ends with a share of the V sums and writes
            // u_pre (write lanes: retrieved) or inter (read lanes) for it
            const bool live = gt < nv;
            const BT *vp16 = svpc + gt * V;
            const float bt = live ? sbeta[gt] : 0.f;
            reduce_scatter<V>(acc, half >> 1, lane, 0, [&](int idx, float x) {
                if (gt >= C) return;
                if (!rd) us[gt * V + idx] = live ? bt * (to_f32(vp16[idx]) - x) : 0.f;
                else is[gt * V + idx] = live ? x : 0.f;
            });
        }
        compute_sync();

        // ---- dual matmul on the tensor cores: one warp per (matrix, 16-row tile) ----
        // delta_v = X u_pre (matrix 0) and readings = QX u_pre + inter (matrix 1), over the
        // nv valid rows and k < nv (X and QX are zero past the diagonal and u_pre is zero past
        // nv). Float32 banks use the 3xTF32 split (hi*lo + lo*hi + hi*hi) for float32 accuracy.
        {
            const int g4 = lane >> 2, i4 = lane & 3;
            const int mt = (nv + 15) >> 4, kt = (nv + 7) >> 3;
            for (int job = warp; job < 2 * mt; job += NW2) {
                const int mat = job & 1, r0 = (job >> 1) * 16;
                const float *A = (mat ? qs : xs) + r0 * XP;
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                for (int k0 = 0; k0 < kt * 8; k0 += 8) {
                    const float af[4] = {A[g4 * XP + k0 + i4], A[(g4 + 8) * XP + k0 + i4],
                                         A[g4 * XP + k0 + i4 + 4], A[(g4 + 8) * XP + k0 + i4 + 4]};
                    const float bf[2] = {g4 < V ? us[(k0 + i4) * V + g4] : 0.f,
                                         g4 < V ? us[(k0 + i4 + 4) * V + g4] : 0.f};
                    unsigned ah[4], bh[2];
#pragma unroll
                    for (int q = 0; q < 4; ++q) ah[q] = to_tf32(af[q]);
                    bh[0] = to_tf32(bf[0]);
                    bh[1] = to_tf32(bf[1]);
                    if constexpr (sizeof(BT) == 4) {
                        unsigned al[4], bl[2];
#pragma unroll
                        for (int q = 0; q < 4; ++q) al[q] = to_tf32(af[q] - __uint_as_float(ah[q]));
                        bl[0] = to_tf32(bf[0] - __uint_as_float(bh[0]));
                        bl[1] = to_tf32(bf[1] - __uint_as_float(bh[1]));
                        mma_tf32(c, ah, bl);
                        mma_tf32(c, al, bh);
                    }
                    mma_tf32(c, ah, bh);
                }
                // c0 (g, 2i), c1 (g, 2i+1), c2 (g+8, 2i), c3 (g+8, 2i+1)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int t = r0 + g4 + (q >> 1) * 8, col = 2 * i4 + (q & 1);
                    if (col < V && t < C) {
                        const float val = t < nv ? c[q] : 0.f;
                        if (mat == 0) dvs[t * kDvPitch + col] = val;
                        else is[t * V + col] = t < nv ? val + is[t * V + col] : 0.f;
                    }
                }
            }
            // rows of whole 16-row tiles past nv were covered; rows from 16 * mt to C are padding
            for (int o = 16 * mt * V + tid; o < C * V; o += NT2) {
                dvs[(o / V) * kDvPitch + o % V] = 0.f;
                is[o] = 0.f;
            }
        }
        // ---- early loads of step ls + 1 (warps without a matmul tile start at once) ----
        bool ok_next = true;
        if (ls + 1 < nsteps) {
            // only part A (slots and links) is needed for the early loads
            ok_next = mbar_wait_bounded(fullA + (st ^ 1), (unsigned)((ls + 1) >> 1) & 1u, d.spin);
            if (ok_next) prefetch(ls + 1, psm + (st ^ 1) * L.bytes);
        }
        if (compute_sync_or(!ok_next)) {
            if (tid == 0) atomicCAS(&w.status->code, 0, (int)SDM_ERR_TIMEOUT);
            return;
        }
        for (int t = tid; t < C; t += NT2) {
            if ((size_t)ti * C + t >= (size_t)d.T) continue;
            float rd[V];
#pragma unroll
            for (int c = 0; c < V; ++c) rd[c] = is[t * V + c];
            store_vec<BT, V>(out + (tok0 + t) * D + c0, rd);
        }

        // ---- DW: B[s] = (sum of dw * delta_v over the group's members, sorted order) +
        //      exp(lend) * B0[s], one writer per written slot. A group of >= kHotGroup members
        //      gets a warp (lane l adds members l, l + 32, ..., then a fixed reduce-scatter);
        //      every other group a thread (members in order), in Phase 1's size order. ----
        {
            const int32_t *sgoff = reinterpret_cast<const int32_t *>(b + L.goff);
            const int4 sc = *reinterpret_cast<const int4 *>(b + L.scal);
            const int ng = nv > 0 ? sc.x : 0, nhot = nv > 0 ? sc.y : 0;
            const int32_t *sgord = reinterpret_cast<const int32_t *>(b + L.gord);
            // the group's row: B0 from the gather, the new piece to the bank and to dwout
            auto finish = [&](int g, int o1, const float (&acc)[V]) {
                const int tinf = sminfo[o1 - 1];
                const uint4 braw = b0s[(tinf & 255) * W + ((tinf >> 8) & 255)];
                float b0[V], o[V];
                piece_to_f32<BT>(braw, b0);
                const float fac = sgfac[g];
#pragma unroll
                for (int c = 0; c < V; ++c) o[c] = fmaf(fac, b0[c], acc[c]);
                const int sl = sgslot[g];
                if ((unsigned)sl < S) {
                    const uint4 packed = pack_piece<BT>(o);
                    *reinterpret_cast<uint4 *>(bank + (size_t)sl * D) = packed;
                    dwout[g] = packed;
                    if (in.snap) {
                        const size_t so = ((size_t)(ti * d.P + p) * CW + (o1 - 1)) * D + c0;
                        if (d.snapq == 2)      // float8_e4m3fn snapshot: V bytes
                            store_fp8<V>(static_cast<unsigned char *>(in.snap) + so, b0);
                        else if (d.snapq)      // float32 bank, bfloat16 snapshot: 4 columns, 8 bytes
                            store_vec<__nv_bfloat16, V>(static_cast<__nv_bfloat16 *>(in.snap) + so, b0);
                        else
                            *reinterpret_cast<uint4 *>(static_cast<BT *>(in.snap) + so) = braw;
                    }
                }
            };
            auto add_member = [&](int m, float (&acc)[V]) {
                const float wt = smdw[m];
                const float4 *dv4 =
                    reinterpret_cast<const float4 *>(dvs + (sminfo[m] & 255) * kDvPitch);
#pragma unroll
                for (int h = 0; h < V / 4; ++h) {
                    const float4 x = dv4[h];
                    fma2(acc[4 * h + 0], acc[4 * h + 1], wt, x.x, x.y);
                    fma2(acc[4 * h + 2], acc[4 * h + 3], wt, x.z, x.w);
                }
            };
            for (int h = warp; h < nhot; h += NW2) {
                const int g = sgord[h];
                const int o0 = sgoff[g], o1 = sgoff[g + 1];
                float acc[V];
#pragma unroll
                for (int c = 0; c < V; ++c) acc[c] = 0.f;
                for (int m = o0 + lane; m < o1; m += 32) add_member(m, acc);
                // a reduce-scatter leaves column c's sum on one lane, which finishes that column:
                // the V lanes store the piece together (one 16-byte segment per warp store)
                const int tinf = sminfo[o1 - 1];
                const int pos = (tinf & 255) * W + ((tinf >> 8) & 255);
                const float fac = sgfac[g];
                const int sl = sgslot[g];
                reduce_scatter<V>(acc, 16, lane, 0, [&](int c, float x) {
                    const BT b0 = reinterpret_cast<const BT *>(b0s + pos)[c];
                    const BT o = from_f32<BT>(fmaf(fac, to_f32(b0), x));
                    if ((unsigned)sl < S) {
                        bank[(size_t)sl * D + c] = o;
                        reinterpret_cast<BT *>(dwout + g)[c] = o;
                        if (in.snap) {
                            const size_t so = ((size_t)(ti * d.P + p) * CW + (o1 - 1)) * D + c0 + c;
                            if (d.snapq == 2) {
                                const float one[1] = {to_f32(b0)};
                                store_fp8<1>(static_cast<unsigned char *>(in.snap) + so, one);
                            } else if (d.snapq) {
                                static_cast<__nv_bfloat16 *>(in.snap)[so] = __float2bfloat16_rn(to_f32(b0));
                            } else {
                                static_cast<BT *>(in.snap)[so] = b0;
                            }
                        }
                    }
                });
            }
            // the other groups, largest first, so that a warp's lanes loop about equally long;
            // they start at the last thread, away from the warps that took a hot group
            for (int i = nhot + (NT2 - 1 - tid); i < ng; i += NT2) {
                const int g = sgord[i];
                const int o0 = sgoff[g], o1 = sgoff[g + 1];
                float acc[V];
#pragma unroll
                for (int c = 0; c < V; ++c) acc[c] = 0.f;
                int m = o0;
                for (; m + 4 <= o1; m += 4) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) add_member(m + q, acc);
                }
                for (; m < o1; ++m) add_member(m, acc);
                finish(g, o1, acc);
            }
        }
        const bool ok = ls + 1 < nsteps ? wait_stage(ls + 1, d.spin) : true;
        if (compute_sync_or(!ok)) {
            if (tid == 0) atomicCAS(&w.status->code, 0, (int)SDM_ERR_TIMEOUT);
            return;
        }
        if (tid == 0) mbar_arrive(empty + st);   // stage st may be refilled
    }
}

}  // namespace

size_t phase2_pipe_smem(const Dims &d) {
    const int V = d.dtype == SDM_BF16 ? 8 : 4;
    const StageLayout L = stage_layout(d.C, d.W, d.R);
    return (size_t)2 * L.bytes + (size_t)pipe_tail_bytes(d.C, d.W, V);
}

bool phase2_fused_fits(const Dims &d) {
    return d.C % 16 == 0 && phase2_pipe_smem(d) <= kPipeSmemMax;
}

namespace {

template <typename BT>
cudaError_t launch_pipe(const Dims &d, const Inputs &in, const Work &w, int step0, int nsteps,
                        cudaStream_t st, size_t smem) {
    const int grid = d.P * (d.D / (16 / (int)sizeof(BT)));
    auto kern = k_phase2_pipe<BT>;
    set_kernel_smem(kern, smem);
    kern<<<grid, NP2, smem, st>>>(d, in, w, step0, nsteps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_phase2_fused(const Dims &d, const Inputs &in, const Work &w, int step0,
                                int nsteps, cudaStream_t st) {
    const size_t pipe = phase2_pipe_smem(d);
    if (pipe > kPipeSmemMax || d.xp != x_pitch(d.C)) return cudaErrorInvalidConfiguration;
    if (d.dtype == SDM_BF16) return launch_pipe<__nv_bfloat16>(d, in, w, step0, nsteps, st, pipe);
    return launch_pipe<float>(d, in, w, step0, nsteps, st, pipe);
}

}  // namespace sdm
