// Phase 2 fused into one persistent kernel per slab: every CTA owns one stream p and one
// slice of VEC bank columns, and runs all the slab's steps for it (gather -> dual matmul ->
// DW, sparse-delta-memory 2.0.0, phase2_kernels.py module docstring).
//
// Why this is exact and needs no inter-CTA synchronization: given Phase 1 and the solve
// (which depend only on slots, weights and decays), every operation of Phase 2 acts on each
// bank column independently -- retrieved, inter, u = beta (v - retrieved), X u, QX u and the
// decay-and-write are all column-wise. A CTA therefore reads and writes only its own columns
// of its own stream's rows, step after step, and only ever waits on its own threads.
//
// Per step (chunk ti of stream p, nv valid tokens), with the CTA's columns c in [c0, c0+VEC):
//   gather  TPT threads per token split its W + R entries; each loads the VEC-column piece
//           (16 bytes) of each entry's bank row and accumulates in f32; the TPT partial sums
//           are combined by a fixed shuffle tree.
//   u_pre   beta_t (v_t - retrieved_t) in shared memory (0 for padding rows)
//   matmul  delta_v = X u_pre and readings = QX u_pre + inter, X and QX staged through
//           shared memory in column tiles; readings rounded once to the bank dtype
//   DW      one thread per group (distinct written slot): exp(lend) B0 + sum of its members'
//           dw * delta_v rows in sorted order, f32, one rounding at the store.
// The bank pieces a step writes are read back by the next step's gather through L1/L2 in
// the same CTA, ordered by the step's closing __syncthreads (no read-only cache path).
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int NT = 256;
constexpr int KT = 64;          // X / QX column tile staged in shared memory

template <typename BT>
struct Vec16 {                  // one 16-byte piece of a bank row
    static constexpr int N = 16 / sizeof(BT);
};

template <typename BT>
__global__ void __launch_bounds__(NT) k_phase2_fused(Dims d, Inputs in, Work w, int step0,
                                                     int nsteps) {
    constexpr int V = Vec16<BT>::N;          // columns per CTA
    extern __shared__ __align__(16) float fsm[];
    const int C = d.C, D = d.D, W = d.W, R = d.R;
    const int slices = D / V;
    const int p = blockIdx.x / slices;
    const int c0 = (blockIdx.x - p * slices) * V;
    const int tid = threadIdx.x;
    const int KP = KT + 1;                   // padded row of a staged X tile

    float *us = fsm;                          // [C][V]  u_pre
    float *is = us + C * V;                   // [C][V]  inter
    float *dvs = is + C * V;                  // [C][V]  delta_v
    float *xs = dvs + C * V;                  // [C][KP] X tile
    float *qs = xs + C * KP;                  // [C][KP] QX tile

    BT *bank = static_cast<BT *>(in.bank) + (size_t)p * d.S * D + c0;
    const BT *vin = static_cast<const BT *>(in.v);
    BT *out = static_cast<BT *>(in.readings);
    const unsigned S = (unsigned)d.S;

    // gather geometry: TPT threads per token (a power of two dividing 32)
    int tpt = NT / C;
    if (tpt > 32) tpt = 32;
    if (tpt < 1) tpt = 1;
    while (tpt & (tpt - 1)) tpt &= tpt - 1;
    const int tpb = NT / tpt;                 // tokens per pass
    const int sub = tid % tpt;

    for (int ls = 0; ls < nsteps; ++ls) {
        const int ti = step0 + ls;
        const int n = ls * d.P + p;
        const int nv = w.nvalid[n];
        const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;

        // ---- gather ----
        for (int tb = 0; tb < C; tb += tpb) {
            const int t = tb + tid / tpt;
            float ar[V], ai[V];
#pragma unroll
            for (int c = 0; c < V; ++c) { ar[c] = 0.f; ai[c] = 0.f; }
            if (t < nv) {
                const int32_t *ws = in.ws + (tok0 + t) * W;
                const int32_t *rs = in.rs + (tok0 + t) * R;
                const float *gw = w.gw + (size_t)n * C * W + (size_t)t * W;
                const float *qw = w.qw + (size_t)n * C * R + (size_t)t * R;
                int j = sub;
                for (; j + 3 * tpt < W; j += 4 * tpt) {
                    float x[4][V], wt[4];
                    int s[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) { s[u] = ws[j + u * tpt]; wt[u] = gw[j + u * tpt]; }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if ((unsigned)s[u] < S) load_vec<BT, V, false>(bank + (size_t)s[u] * D, x[u]);
                        else { wt[u] = 0.f;
#pragma unroll
                            for (int c = 0; c < V; ++c) x[u][c] = 0.f; }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int c = 0; c < V; ++c) ar[c] = fmaf(wt[u], x[u][c], ar[c]);
                }
                for (; j < W; j += tpt) {
                    const int s = ws[j];
                    if ((unsigned)s >= S) continue;
                    float x[V];
                    load_vec<BT, V, false>(bank + (size_t)s * D, x);
                    const float wt = gw[j];
#pragma unroll
                    for (int c = 0; c < V; ++c) ar[c] = fmaf(wt, x[c], ar[c]);
                }
                int i = sub;
                for (; i + 3 * tpt < R; i += 4 * tpt) {
                    float x[4][V], wt[4];
                    int s[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) { s[u] = rs[i + u * tpt]; wt[u] = qw[i + u * tpt]; }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if ((unsigned)s[u] < S) load_vec<BT, V, false>(bank + (size_t)s[u] * D, x[u]);
                        else { wt[u] = 0.f;
#pragma unroll
                            for (int c = 0; c < V; ++c) x[u][c] = 0.f; }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int c = 0; c < V; ++c) ai[c] = fmaf(wt[u], x[u][c], ai[c]);
                }
                for (; i < R; i += tpt) {
                    const int s = rs[i];
                    if ((unsigned)s >= S) continue;
                    float x[V];
                    load_vec<BT, V, false>(bank + (size_t)s * D, x);
                    const float wt = qw[i];
#pragma unroll
                    for (int c = 0; c < V; ++c) ai[c] = fmaf(wt, x[c], ai[c]);
                }
            }
            // fixed-order tree over the token's tpt consecutive lanes
            for (int off = tpt >> 1; off > 0; off >>= 1) {
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    ar[c] += __shfl_down_sync(0xffffffffu, ar[c], off, tpt);
                    ai[c] += __shfl_down_sync(0xffffffffu, ai[c], off, tpt);
                }
            }
            if (sub == 0 && t < C) {
                float u[V];
                if (t < nv) {
                    float vv[V];
                    load_vec<BT, V, false>(vin + (tok0 + t) * D + c0, vv);
                    const float b = in.beta[tok0 + t];
#pragma unroll
                    for (int c = 0; c < V; ++c) u[c] = b * (vv[c] - ar[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < V; ++c) { u[c] = 0.f; ai[c] = 0.f; }
                }
#pragma unroll
                for (int c = 0; c < V; ++c) { us[t * V + c] = u[c]; is[t * V + c] = ai[c]; }
            }
        }
        __syncthreads();

        // ---- dual matmul: outputs o = (row t, column c), o = tid + k * NT ----
        const float *X = w.X + (size_t)n * C * C;
        const float *QX = w.QX + (size_t)n * C * C;
        constexpr int MAXO = (kMaxChunk * V + NT - 1) / NT;
        float ax[MAXO], aq[MAXO];
#pragma unroll
        for (int k = 0; k < MAXO; ++k) { ax[k] = 0.f; aq[k] = 0.f; }
        const int nout = C * V;
        for (int k0 = 0; k0 < C; k0 += KT) {
            const int kw = (C - k0) < KT ? (C - k0) : KT;
            for (int idx = tid; idx < C * kw; idx += NT) {
                const int r = idx / kw, k = idx - r * kw;
                xs[r * KP + k] = X[(size_t)r * C + k0 + k];
                qs[r * KP + k] = QX[(size_t)r * C + k0 + k];
            }
            __syncthreads();
#pragma unroll
            for (int q = 0; q < MAXO; ++q) {
                const int o = tid + q * NT;
                if (o < nout) {
                    const int t = o / V, c = o - t * V;
                    float a = ax[q], b = aq[q];
                    for (int k = 0; k < kw; ++k) {
                        const float u = us[(k0 + k) * V + c];
                        a = fmaf(xs[t * KP + k], u, a);
                        b = fmaf(qs[t * KP + k], u, b);
                    }
                    ax[q] = a;
                    aq[q] = b;
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int q = 0; q < MAXO; ++q) {
            const int o = tid + q * NT;
            if (o < nout) {
                const int t = o / V;
                dvs[o] = t < nv ? ax[q] : 0.f;
                aq[q] = t < nv ? aq[q] + is[o] : 0.f;
            }
        }
        // write readings directly from the accumulators (each output element once)
#pragma unroll
        for (int q = 0; q < MAXO; ++q) {
            const int o = tid + q * NT;
            if (o < nout) {
                const int t = o / V, c = o - t * V;
                if ((size_t)ti * C + t < (size_t)d.T)
                    out[(tok0 + t) * D + c0 + c] = from_f32<BT>(aq[q]);
            }
        }

        // ---- DW ----
        const int ng = w.ngroups[n];
        const int CW = C * W;
        const int32_t *goff = w.goff + (size_t)n * (CW + 1);
        const int32_t *gslot = w.gslot + (size_t)n * CW;
        const float *gfac = w.gfac + (size_t)n * CW;
        const int32_t *perm = w.perm + (size_t)n * CW;
        const float *wdw = w.wdw + (size_t)n * CW;
        for (int g = tid; g < ng; g += NT) {
            const int o0 = goff[g], o1 = goff[g + 1];
            BT *row = bank + (size_t)gslot[g] * D;
            float acc[V];
            load_vec<BT, V, false>(row, acc);
            const float f = gfac[g];
#pragma unroll
            for (int c = 0; c < V; ++c) acc[c] *= f;
            for (int m = o0; m < o1; ++m) {
                const int t = perm[m] / W;
                const float wt = wdw[m];
                const float *dv = dvs + t * V;
#pragma unroll
                for (int c = 0; c < V; ++c) acc[c] = fmaf(wt, dv[c], acc[c]);
            }
            store_vec<BT, V>(row, acc);
        }
        __syncthreads();
    }
}

}  // namespace

size_t phase2_fused_smem(const Dims &d) {
    const int V = d.dtype == SDM_BF16 ? 8 : 4;
    return sizeof(float) * ((size_t)3 * d.C * V + (size_t)2 * d.C * (KT + 1));
}

cudaError_t launch_phase2_fused(const Dims &d, const Inputs &in, const Work &w, int step0,
                                int nsteps, cudaStream_t st) {
    const size_t smem = phase2_fused_smem(d);
    const int V = d.dtype == SDM_BF16 ? 8 : 4;
    const int grid = d.P * (d.D / V);
    if (d.dtype == SDM_BF16) {
        auto kern = k_phase2_fused<__nv_bfloat16>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, NT, smem, st>>>(d, in, w, step0, nsteps);
    } else {
        auto kern = k_phase2_fused<float>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, NT, smem, st>>>(d, in, w, step0, nsteps);
    }
    return cudaGetLastError();
}

}  // namespace sdm
