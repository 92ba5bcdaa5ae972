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
// The bank pieces a step writes are read back by the next step's gather through L1/L2 in the
// same CTA, ordered by the step's closing __syncthreads (no read-only cache path). The kernel
// runs when two stages of per-step metadata fit in shared memory (launch_phase2_fused says
// whether); larger chunks use the per-step kernels of phase2.cu.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

template <typename BT>
struct Vec16 {                  // one 16-byte piece of a bank row
    static constexpr int N = 16 / sizeof(BT);
};

// ---------------------------------------------------------------------------------------
// Pipelined variant for chunks whose per-step metadata fits in shared memory twice: the
// next step's slots, weights, v pieces, beta, X, QX and sorted member records are copied into
// the other stage with cp.async while the current step computes. The gather keeps the B0
// pieces of the written rows in shared memory, and the DW is a block-wide segmented scan over
// the sorted members (each thread a fixed run of positions, a fixed combine tree), so Zipf-hot
// groups are summed by many threads. The group's tail position writes the row:
//   B[s] = (sum of dw * delta_v over the group, scan order) + exp(lend) * B0[s].
// ---------------------------------------------------------------------------------------
constexpr int NT2 = 512;
constexpr int NW2 = NT2 / 32;

struct StageLayout {     // byte offsets inside one stage
    int wslot, wgw, rslot, rqw, vpc, beta, xs, qs, minfo, mdw, mslot, mfac, bytes;
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
    L.vpc = o; o = align16(o + 16 * C);
    L.beta = o; o = align16(o + 4 * C);
    L.xs = o; o = align16(o + 4 * C * XP);
    L.qs = o; o = align16(o + 4 * C * XP);
    L.minfo = o; o = align16(o + 4 * CW);
    L.mdw = o; o = align16(o + 4 * CW);
    L.mslot = o; o = align16(o + 4 * CW);
    L.mfac = o; o = align16(o + 4 * CW);
    L.bytes = o;
    return L;
}

// Bytes after the two stages: u_pre, inter, delta_v [C][V] f32, the B0 pieces [CW][16 B] and
// the scan's warp totals.
__host__ __device__ inline int pipe_tail_bytes(int C, int W, int V) {
    return 3 * 4 * C * V + 16 * C * W + NW2 * 4 * (V + 1) * 2;
}

// cp.async of nbytes (a multiple of 4) from global to shared, 16 bytes at a time when both
// ends are 16-byte aligned
__device__ __forceinline__ void copy_async(unsigned char *dst, const void *src, int nbytes, int tid,
                                           int nthr) {
    const unsigned char *s8 = static_cast<const unsigned char *>(src);
    if (((reinterpret_cast<uintptr_t>(s8) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
        const int n16 = nbytes >> 4;
        for (int i = tid; i < n16; i += nthr) cp_async16(dst + 16 * i, s8 + 16 * i);
        for (int i = n16 * 4 + tid; i < (nbytes >> 2); i += nthr) cp_async4(dst + 4 * i, s8 + 4 * i);
    } else {
        for (int i = tid; i < (nbytes >> 2); i += nthr) cp_async4(dst + 4 * i, s8 + 4 * i);
    }
}

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

template <typename BT>
__global__ void __launch_bounds__(NT2) k_phase2_pipe(Dims d, Inputs in, Work w, int step0,
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
    float *dvs = is + C * V;                                     // [C][V]
    uint4 *b0s = reinterpret_cast<uint4 *>(dvs + C * V);         // [CW] B0 pieces (raw)
    float *wtot = reinterpret_cast<float *>(b0s + CW);           // [NW2][V + 1] scan totals

    BT *bank = static_cast<BT *>(in.bank) + (size_t)p * d.S * D + c0;
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

    // cp.async of step ls's metadata into stage st (all threads)
    auto issue = [&](int ls, int st) {
        unsigned char *b = psm + st * L.bytes;
        const int ti = step0 + ls;
        const int n = ls * d.P + p;
        const int nv = nvalid_of(ti);
        const int nw = nv * W, nr = nv * R;
        const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;
        copy_async(b + L.wslot, in.ws + tok0 * W, 4 * nw, tid, NT2);
        copy_async(b + L.wgw, w.gw + (size_t)n * CW, 4 * nw, tid, NT2);
        copy_async(b + L.rslot, in.rs + tok0 * R, 4 * nr, tid, NT2);
        copy_async(b + L.rqw, w.qw + (size_t)n * CR, 4 * nr, tid, NT2);
        copy_async(b + L.beta, in.beta + tok0, 4 * nv, tid, NT2);
        copy_async(b + L.minfo, w.minfo + (size_t)n * CW, 4 * nw, tid, NT2);
        copy_async(b + L.mdw, w.wdw + (size_t)n * CW, 4 * nw, tid, NT2);
        copy_async(b + L.mslot, w.mslot + (size_t)n * CW, 4 * nw, tid, NT2);
        copy_async(b + L.mfac, w.mfac + (size_t)n * CW, 4 * nw, tid, NT2);
        for (int t = tid; t < nv; t += NT2)
            cp_async16(b + L.vpc + 16 * t, vin + (tok0 + t) * D + c0);
        const float *X = w.X + (size_t)n * C * C;
        const float *QX = w.QX + (size_t)n * C * C;
        if ((C & 3) == 0) {   // rows r < nv, whole rows, 16 bytes at a time
            const int q4 = C >> 2;
            for (int i = tid; i < nv * q4; i += NT2) {
                const int r = div_by(i, magQ), k = (i - r * q4) * 4;
                cp_async16(b + L.xs + 4 * (r * XP + k), X + (size_t)r * C + k);
                cp_async16(b + L.qs + 4 * (r * XP + k), QX + (size_t)r * C + k);
            }
        } else {
            for (int r = warp; r < nv; r += NW2)
                for (int k = lane; k < C; k += 32) {
                    cp_async4(b + L.xs + 4 * (r * XP + k), X + (size_t)r * C + k);
                    cp_async4(b + L.qs + 4 * (r * XP + k), QX + (size_t)r * C + k);
                }
        }
    };

    int tpt = NT2 / C;
    if (tpt > 32) tpt = 32;
    if (tpt < 1) tpt = 1;
    while (tpt & (tpt - 1)) tpt &= tpt - 1;
    const int tpb = NT2 / tpt;
    const int sub = tid % tpt;

    issue(0, 0);
    cp_async_commit();
    for (int ls = 0; ls < nsteps; ++ls) {
        const int st = ls & 1;
        if (ls + 1 < nsteps) {
            issue(ls + 1, st ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
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
        const int32_t *smslot = reinterpret_cast<const int32_t *>(b + L.mslot);
        const float *smfac = reinterpret_cast<const float *>(b + L.mfac);
        const int ti = step0 + ls;
        const int nv = nvalid_of(ti);
        const int nw = nv * W;
        const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;

        // ---- gather (the write pieces are also kept as B0 for the DW) ----
        // The token's W + R entries (writes first) are split over its tpt lanes; each lane
        // issues up to GB loads before using any, and adds them in entry order.
        constexpr int GB = 8;
        const int E = W + R;
        for (int tb = 0; tb < C; tb += tpb) {
            const int t = tb + tid / tpt;
            float ar[V], ai[V];
#pragma unroll
            for (int c = 0; c < V; ++c) { ar[c] = 0.f; ai[c] = 0.f; }
            if (t < nv) {
                const int32_t *wsl = swslot + t * W;
                const float *wg = swgw + t * W;
                const int32_t *rsl = srslot + t * R;
                const float *rq = srqw + t * R;
                for (int q0 = sub; q0 < E; q0 += GB * tpt) {
                    uint4 u[GB];
                    float wt[GB];
#pragma unroll
                    for (int k = 0; k < GB; ++k) {
                        const int q = q0 + k * tpt;
                        u[k] = make_uint4(0u, 0u, 0u, 0u);
                        wt[k] = 0.f;
                        if (q < E) {
                            const int sl = q < W ? wsl[q] : rsl[q - W];
                            if ((unsigned)sl < S) {
                                wt[k] = q < W ? wg[q] : rq[q - W];
                                u[k] = *reinterpret_cast<const uint4 *>(bank + (size_t)sl * D);
                            }
                        }
                    }
#pragma unroll
                    for (int k = 0; k < GB; ++k) {
                        const int q = q0 + k * tpt;
                        if (q < E) {
                            float x[V];
                            piece_to_f32<BT>(u[k], x);
                            if (q < W) {
                                b0s[t * W + q] = u[k];
#pragma unroll
                                for (int c = 0; c < V; ++c) ar[c] = fmaf(wt[k], x[c], ar[c]);
                            } else {
#pragma unroll
                                for (int c = 0; c < V; ++c) ai[c] = fmaf(wt[k], x[c], ai[c]);
                            }
                        }
                    }
                }
            }
            for (int off = tpt >> 1; off > 0; off >>= 1) {
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    ar[c] += __shfl_down_sync(0xffffffffu, ar[c], off, tpt);
                    ai[c] += __shfl_down_sync(0xffffffffu, ai[c], off, tpt);
                }
            }
            if (sub == 0 && t < C) {
                if (t < nv) {
                    const BT *vp16 = svpc + t * V;
                    const float bt = sbeta[t];
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        us[t * V + c] = bt * (to_f32(vp16[c]) - ar[c]);
                        is[t * V + c] = ai[c];
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < V; ++c) { us[t * V + c] = 0.f; is[t * V + c] = 0.f; }
                }
            }
        }
        __syncthreads();

        // ---- dual matmul: 8 lanes per row split k (k = ks, ks + 8, ...), tree-reduced ----
        {
            const int ks = tid & 7;
            for (int t0 = 0; t0 < C; t0 += NT2 / 8) {
                const int t = t0 + (tid >> 3);
                float ax[V], aq[V];
#pragma unroll
                for (int c = 0; c < V; ++c) { ax[c] = 0.f; aq[c] = 0.f; }
                if (t < nv) {
                    const float *xr = xs + t * XP, *qr = qs + t * XP;
                    for (int k = ks; k < nv; k += 8) {
                        const float xv = xr[k], qv = qr[k];
                        const float4 *up = reinterpret_cast<const float4 *>(us + k * V);
#pragma unroll
                        for (int h = 0; h < V / 4; ++h) {
                            const float4 u4 = up[h];
                            ax[4 * h + 0] = fmaf(xv, u4.x, ax[4 * h + 0]);
                            ax[4 * h + 1] = fmaf(xv, u4.y, ax[4 * h + 1]);
                            ax[4 * h + 2] = fmaf(xv, u4.z, ax[4 * h + 2]);
                            ax[4 * h + 3] = fmaf(xv, u4.w, ax[4 * h + 3]);
                            aq[4 * h + 0] = fmaf(qv, u4.x, aq[4 * h + 0]);
                            aq[4 * h + 1] = fmaf(qv, u4.y, aq[4 * h + 1]);
                            aq[4 * h + 2] = fmaf(qv, u4.z, aq[4 * h + 2]);
                            aq[4 * h + 3] = fmaf(qv, u4.w, aq[4 * h + 3]);
                        }
                    }
                }
#pragma unroll
                for (int off = 4; off > 0; off >>= 1) {
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        ax[c] += __shfl_down_sync(0xffffffffu, ax[c], off, 8);
                        aq[c] += __shfl_down_sync(0xffffffffu, aq[c], off, 8);
                    }
                }
                if (ks == 0 && t < C) {
                    float rd[V];
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        dvs[t * V + c] = t < nv ? ax[c] : 0.f;
                        rd[c] = t < nv ? aq[c] + is[t * V + c] : 0.f;
                    }
                    if ((size_t)ti * C + t < (size_t)d.T)
                        store_vec<BT, V>(out + (tok0 + t) * D + c0, rd);
                }
            }
        }
        __syncthreads();

        // ---- DW: segmented scan over the sorted members ----
        const int mpt = (nw + NT2 - 1) / NT2;
        const int m0 = tid * mpt, m1 = (m0 + mpt) < nw ? (m0 + mpt) : nw;
        float acc[V];
        int f = 0;
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] = 0.f;
        for (int m = m0; m < m1; ++m) {
            const int info = sminfo[m];
            const float wt = smdw[m];
            const float *dv = dvs + (info & 255) * V;
            if ((info >> 16) & 1) {
                f = 1;
#pragma unroll
                for (int c = 0; c < V; ++c) acc[c] = wt * dv[c];
            } else {
#pragma unroll
                for (int c = 0; c < V; ++c) acc[c] = fmaf(wt, dv[c], acc[c]);
            }
        }
        // inclusive scan of (f, acc) over the warp, then over the warps' totals
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int pf = __shfl_up_sync(0xffffffffu, f, off);
            float pv[V];
#pragma unroll
            for (int c = 0; c < V; ++c) pv[c] = __shfl_up_sync(0xffffffffu, acc[c], off);
            if (lane >= off) {
                if (!f) {
#pragma unroll
                    for (int c = 0; c < V; ++c) acc[c] = pv[c] + acc[c];
                }
                f |= pf;
            }
        }
        if (lane == 31) {
#pragma unroll
            for (int c = 0; c < V; ++c) wtot[warp * (V + 1) + c] = acc[c];
            wtot[warp * (V + 1) + V] = (float)f;
        }
        // exclusive value within the warp: the inclusive value of the lane before
        int ef = __shfl_up_sync(0xffffffffu, f, 1);
        float ev[V];
#pragma unroll
        for (int c = 0; c < V; ++c) ev[c] = __shfl_up_sync(0xffffffffu, acc[c], 1);
        if (lane == 0) {
            ef = 0;
#pragma unroll
            for (int c = 0; c < V; ++c) ev[c] = 0.f;
        }
        __syncthreads();
        if (warp == 0) {
            float tv[V];
            int tf = lane < NW2 ? (int)wtot[lane * (V + 1) + V] : 0;
#pragma unroll
            for (int c = 0; c < V; ++c) tv[c] = lane < NW2 ? wtot[lane * (V + 1) + c] : 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int pf = __shfl_up_sync(0xffffffffu, tf, off);
                float pv[V];
#pragma unroll
                for (int c = 0; c < V; ++c) pv[c] = __shfl_up_sync(0xffffffffu, tv[c], off);
                if (lane >= off) {
                    if (!tf) {
#pragma unroll
                        for (int c = 0; c < V; ++c) tv[c] = pv[c] + tv[c];
                    }
                    tf |= pf;
                }
            }
            // exclusive prefix of warp `lane`: inclusive value of warp lane-1
            float xv[V];
#pragma unroll
            for (int c = 0; c < V; ++c) xv[c] = __shfl_up_sync(0xffffffffu, tv[c], 1);
            if (lane < NW2) {
#pragma unroll
                for (int c = 0; c < V; ++c) wtot[NW2 * (V + 1) + lane * V + c] = lane ? xv[c] : 0.f;
            }
        }
        __syncthreads();
        // carry into this thread's run: the warp prefix combined with the lane prefix
        float run[V];
#pragma unroll
        for (int c = 0; c < V; ++c)
            run[c] = ef ? ev[c] : wtot[NW2 * (V + 1) + warp * V + c] + ev[c];
        for (int m = m0; m < m1; ++m) {
            const int info = sminfo[m];
            const float wt = smdw[m];
            const int t = info & 255;
            const float *dv = dvs + t * V;
            if ((info >> 16) & 1) {
#pragma unroll
                for (int c = 0; c < V; ++c) run[c] = wt * dv[c];
            } else {
#pragma unroll
                for (int c = 0; c < V; ++c) run[c] = fmaf(wt, dv[c], run[c]);
            }
            if ((info >> 17) & 1) {
                float b0[V], o[V];
                const uint4 braw = b0s[t * W + ((info >> 8) & 255)];
                piece_to_f32<BT>(braw, b0);
                if (in.snap)
                    *reinterpret_cast<uint4 *>(static_cast<BT *>(in.snap) +
                                               ((size_t)(ti * d.P + p) * CW + m) * D + c0) = braw;
                const float fac = smfac[m];
#pragma unroll
                for (int c = 0; c < V; ++c) o[c] = fmaf(fac, b0[c], run[c]);
                const int sl = smslot[m];
                if ((unsigned)sl < S) store_vec<BT, V>(bank + (size_t)sl * D, o);
            }
        }
        __syncthreads();
    }
}

}  // namespace

size_t phase2_pipe_smem(const Dims &d) {
    const int V = d.dtype == SDM_BF16 ? 8 : 4;
    const StageLayout L = stage_layout(d.C, d.W, d.R);
    return (size_t)2 * L.bytes + (size_t)pipe_tail_bytes(d.C, d.W, V);
}

bool phase2_fused_fits(const Dims &d) { return phase2_pipe_smem(d) <= kPipeSmemMax; }

cudaError_t launch_phase2_fused(const Dims &d, const Inputs &in, const Work &w, int step0,
                                int nsteps, cudaStream_t st) {
    const int V = d.dtype == SDM_BF16 ? 8 : 4;
    const int grid = d.P * (d.D / V);
    const size_t pipe = phase2_pipe_smem(d);
    if (pipe > kPipeSmemMax) return cudaErrorInvalidConfiguration;
    if (d.dtype == SDM_BF16) {
        auto kern = k_phase2_pipe<__nv_bfloat16>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pipe);
        kern<<<grid, NT2, pipe, st>>>(d, in, w, step0, nsteps);
    } else {
        auto kern = k_phase2_pipe<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pipe);
        kern<<<grid, NT2, pipe, st>>>(d, in, w, step0, nsteps);
    }
    return cudaGetLastError();
}

}  // namespace sdm
