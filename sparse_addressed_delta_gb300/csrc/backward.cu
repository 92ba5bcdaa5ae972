// Backward of the chunked SDM write/read (sparse-delta-memory 2.0.0 page, memory_ops.py module
// docstring, "Backward"; SDMWriteRead.backward's contract: gradients with respect to the bank,
// v, beta, the write and read weights and the log-decays, the bank restored exactly from the
// snapshot). The steps of the forward are undone from the last to the first; within a step the
// Phase-2 movers go first, then the products through the solve, then the Phase-1 quantities.
//
// Per step ti, in reverse (chunk quantities as in the forward; dB1 = gradient with respect
// to the bank after the chunk, held in grad_bank, which becomes dB0 in place):
//   restore   B0[s] = snapshot[s] for the chunk's written slots (the bank goes back one step)
//   gather    ret_t = sum_j gw_tj B0[s_tj],     du_t = sum_j dw_tj dB1[s_tj]
//   mm1       u_pre = beta (v - ret), u = X u_pre, du_pre = X^T du + QX^T dO,
//             dv = beta du_pre, dret = -beta du_pre, partials of <du_pre, v - ret>
//   mm2       dX = du u_pre^T, dQX = dO u_pre^T, dX += QK^T dQX, dQK = tril(dQX X^T),
//             dL = -strict_tril(X^T dX X^T), dA = beta dL, dbeta += <dL, A> per row
//   dots      ddw = <dB1[s], u_t>, dgw = <dret_t, B0[s]>, dqw = <dO_t, B0[r]>,
//             dfac = <dB1[s], B0[s]> per written slot
//   dB writes dB0[s] = exp(lend_s) dB1[s] + sum_members gw dret_t      (one warp per slot)
//   dB reads  dB0[r] += sum_members qw dO_t                             (one warp per slot)
//   phase 1   dk, dq and dg through gw, qw, dw, exp(lend), A and QK and the running sums Λ
// Every sum has a fixed order (lanes then a shuffle tree, or one owner walking its members),
// so the gradients are bitwise reproducible.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int NTB = 256;
constexpr int NWB = NTB / 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
    return __shfl_sync(0xffffffffu, v, 0);
}

__device__ __forceinline__ int local_n(const Dims &d, int step0, int ti, int p) {
    return (ti - step0) * d.P + p;
}

// ---------------------------------------------------------------------------------------
// restore: B0 rows of the written slots from the snapshot (one warp per group); a bfloat16
// (float32 banks) or float8_e4m3fn snapshot puts back the rounded rows
// ---------------------------------------------------------------------------------------
template <typename BT, int CPL>
__global__ void __launch_bounds__(NTB) k_b_restore(Dims d, Inputs in, Work w, int step0, int ti) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p = blockIdx.y, n = local_n(d, step0, ti, p);
    const int CW = d.C * d.W, D = d.D;
    const int ng = w.ngroups[n];
    const int32_t *goff = w.goff + (size_t)n * goff_stride(CW);
    const int32_t *gslot = w.gslot + (size_t)n * CW;
    BT *bank = static_cast<BT *>(in.bank) + stream_row0(d, p) * D + lane * CPL;
    // the snapshot is in the bank dtype, in bfloat16 (d.snapq 1, float32 banks) or in
    // float8_e4m3fn (d.snapq 2)
    const size_t s0 = (size_t)(ti * d.P + p) * CW * D + lane * CPL;
    const BT *snap = static_cast<const BT *>(in.snap) + s0;
    const __nv_bfloat16 *snaph = static_cast<const __nv_bfloat16 *>(in.snap) + s0;
    const unsigned char *snap8 = static_cast<const unsigned char *>(in.snap) + s0;
    for (int g = blockIdx.x * NWB + warp; g < ng; g += gridDim.x * NWB) {
        const int sl = gslot[g];
        if ((unsigned)sl >= (unsigned)d.S) continue;
        float x[CPL];
        const size_t ro = (size_t)(goff[g + 1] - 1) * D;
        if (d.snapq == 2) load_fp8<CPL>(snap8 + ro, x);
        else if (d.snapq) load_vec<__nv_bfloat16, CPL, false>(snaph + ro, x);
        else load_vec<BT, CPL, false>(snap + ro, x);
        store_vec<BT, CPL>(bank + (size_t)sl * D, x);
    }
}

// ---------------------------------------------------------------------------------------
// gather: ret and du rows (one warp per token, entries in order)
// ---------------------------------------------------------------------------------------
template <typename BT, int CPL>
__global__ void __launch_bounds__(NTB) k_b_gather(Dims d, Inputs in, Work w, const float *gbank,
                                                 int step0, int ti) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = d.C, D = d.D, W = d.W;
    const int gt = blockIdx.x * NWB + warp;
    if (gt >= d.P * C) return;
    const int p = gt / C, t = gt - p * C;
    const int n = local_n(d, step0, ti, p);
    const size_t row = ((size_t)p * C + t) * D + lane * CPL;
    if (t >= w.nvalid[n]) {   // rows past the valid tokens are zero (the C x C products read them)
        float z[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) z[c] = 0.f;
        store_vec<float, CPL>(w.ret + row, z);
        store_vec<float, CPL>(w.dv + row, z);
        return;
    }
    const size_t tok = (size_t)p * d.T + (size_t)ti * C + t;
    const int32_t *ws = in.ws + tok * W;
    const float *gw = w.gw + (size_t)n * C * W + (size_t)t * W;
    const float *dw = w.dwt + (size_t)n * C * W + (size_t)t * W;
    const BT *bank = static_cast<const BT *>(in.bank) + stream_row0(d, p) * D + lane * CPL;
    const float *gb = gbank + stream_row0(d, p) * D + lane * CPL;
    float ar[CPL], ad[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) { ar[c] = 0.f; ad[c] = 0.f; }
    for (int j = 0; j < W; ++j) {
        const int s = ws[j];
        if ((unsigned)s >= (unsigned)d.S) continue;
        float x[CPL], y[CPL];
        load_vec<BT, CPL, false>(bank + (size_t)s * D, x);
        load_vec<float, CPL, false>(gb + (size_t)s * D, y);
        const float a = gw[j], b = dw[j];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            ar[c] = fmaf(a, x[c], ar[c]);
            ad[c] = fmaf(b, y[c], ad[c]);
        }
    }
    store_vec<float, CPL>(w.ret + row, ar);
    store_vec<float, CPL>(w.dv + row, ad);   // w.dv holds du in the backward
}

// ---------------------------------------------------------------------------------------
// mm1: a 32-row x 32-column tile of u, u_pre, du_pre and the per-token outputs
// ---------------------------------------------------------------------------------------
constexpr int TM = 32, TN = 32;

template <typename BT>
__global__ void __launch_bounds__(NTB) k_b_mm1(Dims d, Inputs in, Work w, const void *grad_out,
                                              float *grad_v, int step0, int ti) {
    extern __shared__ __align__(16) float sm1[];
    const int C = d.C, D = d.D;
    const int m0 = blockIdx.x * TM, d0 = blockIdx.y * TN, p = blockIdx.z;
    const int n = local_n(d, step0, ti, p);
    const int nv = w.nvalid[n];
    const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;
    float *Up = sm1;               // [C][TN] u_pre
    float *Dd = Up + C * TN;       // [C][TN] du
    float *Do = Dd + C * TN;       // [C][TN] dO (zero past nv)
    float *Xr = Do + C * TN;       // [TM][C] X rows m0..
    float *Xc = Xr + TM * C;       // [C][TM] X[:, m0..]
    float *Qc = Xc + C * TM;       // [C][TM] QX[:, m0..]
    const float *X = w.X + (size_t)n * C * C;
    const float *QX = w.QX + (size_t)n * C * C;
    const BT *v = static_cast<const BT *>(in.v);
    const BT *go = static_cast<const BT *>(grad_out);
    const float *ret = w.ret + (size_t)p * C * D;
    const float *du = w.dv + (size_t)p * C * D;
    for (int idx = threadIdx.x; idx < C * TN; idx += NTB) {
        const int k = idx / TN, c = idx - k * TN, col = d0 + c;
        float up = 0.f, dd = 0.f, dob = 0.f;
        if (k < nv && col < D) {
            const size_t r = (tok0 + k) * D + col;
            up = in.beta[tok0 + k] * (to_f32(v[r]) - ret[(size_t)k * D + col]);
            dd = du[(size_t)k * D + col];
            dob = to_f32(go[r]);
        }
        Up[idx] = up;
        Dd[idx] = dd;
        Do[idx] = dob;
    }
    for (int idx = threadIdx.x; idx < TM * C; idx += NTB) {
        const int r = idx / C, k = idx - r * C;
        Xr[idx] = (m0 + r < C) ? X[(size_t)(m0 + r) * C + k] : 0.f;
        const int kk = idx / TM, mm = idx - kk * TM;     // column-block view of the same count
        Xc[idx] = (m0 + mm < C) ? X[(size_t)kk * C + m0 + mm] : 0.f;
        Qc[idx] = (m0 + mm < C) ? QX[(size_t)kk * C + m0 + mm] : 0.f;
    }
    __syncthreads();
    const int rr = threadIdx.x >> 3, cq = (threadIdx.x & 7) * 4;   // row, 4 columns
    const int m = m0 + rr;
    float au[4] = {}, adp[4] = {};
    for (int k = 0; k < C; ++k) {
        const float xr = Xr[rr * C + k], xc = Xc[k * TM + rr], qc = Qc[k * TM + rr];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            au[c] = fmaf(xr, Up[k * TN + cq + c], au[c]);
            adp[c] = fmaf(xc, Dd[k * TN + cq + c], adp[c]);
            adp[c] = fmaf(qc, Do[k * TN + cq + c], adp[c]);
        }
    }
    float part = 0.f;
    if (m < C) {
        const bool live = m < nv;
        const float b = live ? in.beta[tok0 + m] : 0.f;
        for (int c = 0; c < 4; ++c) {
            const int col = d0 + cq + c;
            if (col >= D) continue;
            const size_t o = ((size_t)p * C + m) * D + col;
            w.bu[o] = live ? au[c] : 0.f;
            w.bup[o] = Up[m * TN + cq + c];
            w.bdret[o] = live ? -b * adp[c] : 0.f;
            w.bdo[o] = Do[m * TN + cq + c];
            if (live) {
                const size_t r = (tok0 + m) * D + col;
                part = fmaf(adp[c], to_f32(v[r]) - ret[(size_t)m * D + col], part);
            }
            if ((size_t)ti * C + m < (size_t)d.T) grad_v[(tok0 + m) * D + col] = live ? b * adp[c] : 0.f;
        }
    }
    // row sum over the tile's 32 columns (8 lanes x 4), fixed tree
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) part += __shfl_down_sync(0xffffffffu, part, off, 8);
    if ((threadIdx.x & 7) == 0 && m < C)
        w.bdb2[((size_t)p * gridDim.y + blockIdx.y) * C + m] = part;
}

// ---------------------------------------------------------------------------------------
// batched GEMM: Out[b] = alpha op(A[b]) op(B[b]) (+ Out[b]), then a mask
// ---------------------------------------------------------------------------------------
struct GemmOp {
    const float *A, *B;
    float *Out;
    long long sa, sb, so;     // batch strides (elements)
    int lda, ldb, ldo;
    int ta, tb;               // 1: use the operand transposed
    int M, N, K;
    float alpha;
    int accum;                // 1: add into Out
    int mask;                 // 0 none, 1 lower incl. diagonal, 2 strictly lower
};

constexpr int GT = 64, GK = 16;
constexpr int GAP = GK + 4;     // A tile [64][GK] pitch: conflict-free fragment loads
constexpr int GBP = GT + 8;     // B tile [GK][64] pitch: conflict-free fragment loads
constexpr int GTHREADS = 128;   // 4 warps, a 32 x 32 quarter of the 64 x 64 tile each

// Batched GEMM on the tensor cores: mma.sync m16n8k8 with the 3xTF32 split (hi*lo + lo*hi +
// hi*hi), which keeps float32 accuracy; every output element sums its k terms in a fixed order.
__global__ void __launch_bounds__(GTHREADS) k_bgemm(GemmOp g) {
    __shared__ __align__(16) float As[GT * GAP];
    __shared__ __align__(16) float Bs[GK * GBP];
    const int b = blockIdx.z;
    const int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
    const float *A = g.A + b * g.sa;
    const float *B = g.B + b * g.sb;
    float *O = g.Out + b * g.so;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, i4 = lane & 3;
    const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;
    float acc[2][4][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;
    for (int k0 = 0; k0 < g.K; k0 += GK) {
        for (int idx = tid; idx < GK * GT; idx += GTHREADS) {
            // consecutive threads on the operand's contiguous index
            const int kk = g.ta ? idx / GT : idx % GK, mm = g.ta ? idx % GT : idx / GK;
            const int gm = m0 + mm, gk = k0 + kk;
            As[mm * GAP + kk] = (gm < g.M && gk < g.K)
                                    ? (g.ta ? A[(size_t)gk * g.lda + gm] : A[(size_t)gm * g.lda + gk])
                                    : 0.f;
            const int kb = g.tb ? idx % GK : idx / GT, nn = g.tb ? idx / GK : idx % GT;
            const int gn = n0 + nn, gkb = k0 + kb;
            Bs[kb * GBP + nn] = (gn < g.N && gkb < g.K)
                                    ? (g.tb ? B[(size_t)gn * g.ldb + gkb] : B[(size_t)gkb * g.ldb + gn])
                                    : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int ks = 0; ks < GK; ks += 8) {
            unsigned ah[2][4], al[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float *Ar = As + (wm + 16 * i + g4) * GAP + ks + i4;
                const float af[4] = {Ar[0], Ar[8 * GAP], Ar[4], Ar[8 * GAP + 4]};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ah[i][q] = to_tf32(af[q]);
                    al[i][q] = to_tf32(af[q] - __uint_as_float(ah[i][q]));
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float *Bc = Bs + (ks + i4) * GBP + wn + 8 * j + g4;
                const float bf[2] = {Bc[0], Bc[4 * GBP]};
                const unsigned bh[2] = {to_tf32(bf[0]), to_tf32(bf[1])};
                const unsigned bl[2] = {to_tf32(bf[0] - __uint_as_float(bh[0])),
                                        to_tf32(bf[1] - __uint_as_float(bh[1]))};
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    mma_tf32(acc[i][j], ah[i], bl);
                    mma_tf32(acc[i][j], al[i], bh);
                    mma_tf32(acc[i][j], ah[i], bh);
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = m0 + wm + 16 * i + g4 + (q >> 1) * 8;
                const int c = n0 + wn + 8 * j + 2 * i4 + (q & 1);
                if (r >= g.M || c >= g.N) continue;
                float v = g.alpha * acc[i][j][q];
                if (g.accum) v += O[(size_t)r * g.ldo + c];
                if ((g.mask == 1 && c > r) || (g.mask == 2 && c >= r)) v = 0.f;
                O[(size_t)r * g.ldo + c] = v;
            }
}

// dA = beta dL (strictly lower, in place) and grad_beta = <dL, A> per row + the mm1 partials
__global__ void __launch_bounds__(NTB) k_b_beta(Dims d, Inputs in, Work w, float *grad_beta,
                                               int step0, int ti, int dtiles) {
    const int p = blockIdx.x, n = local_n(d, step0, ti, p);
    const int C = d.C, nv = w.nvalid[n];
    const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;
    float *dA = w.bdA + (size_t)p * C * C;
    const float *A = w.A + (size_t)n * C * C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < C; t += NWB) {
        float s = 0.f;
        const float b = t < nv ? in.beta[tok0 + t] : 0.f;
        for (int u = lane; u < C; u += 32) {
            const float dl = (t < nv && u < t) ? dA[(size_t)t * C + u] : 0.f;
            s = fmaf(dl, A[(size_t)t * C + u], s);
            dA[(size_t)t * C + u] = b * dl;
        }
        s = warp_sum(s);
        if (lane == 0 && (size_t)ti * C + t < (size_t)d.T) {
            float b2 = 0.f;
            for (int k = 0; k < dtiles; ++k) b2 += w.bdb2[((size_t)p * dtiles + k) * C + t];
            grad_beta[tok0 + t] = t < nv ? s + b2 : 0.f;
        }
    }
}

// ---------------------------------------------------------------------------------------
// dots (one warp per entry)
// ---------------------------------------------------------------------------------------
template <typename BT, int CPL>
__global__ void __launch_bounds__(NTB) k_b_dots(Dims d, Inputs in, Work w, const float *gbank,
                                               int step0, int ti) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p = blockIdx.y, n = local_n(d, step0, ti, p);
    const int C = d.C, D = d.D, W = d.W, R = d.R, CW = C * W, CR = C * R;
    const int nv = w.nvalid[n];
    const int nw = nv * W, nr = nv * R, ng = w.ngroups[n];
    const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;
    const BT *bank = static_cast<const BT *>(in.bank) + stream_row0(d, p) * D + lane * CPL;
    const float *gb = gbank + stream_row0(d, p) * D + lane * CPL;
    const float *u = w.bu + (size_t)p * C * D + lane * CPL;
    const float *dret = w.bdret + (size_t)p * C * D + lane * CPL;
    const float *dO = w.bdo + (size_t)p * C * D + lane * CPL;
    const unsigned magW = div_magic(W), magR = div_magic(R);
    const int total = nw + nr + ng;
    for (int it = blockIdx.x * NWB + warp; it < total; it += gridDim.x * NWB) {
        if (it < nw) {
            const int e = it, t = div_by(e, magW);
            const int s = in.ws[tok0 * W + e];
            float a = 0.f, b = 0.f;
            if ((unsigned)s < (unsigned)d.S) {
                float x[CPL], y[CPL], uu[CPL], dr[CPL];
                load_vec<float, CPL, false>(gb + (size_t)s * D, y);
                load_vec<BT, CPL, false>(bank + (size_t)s * D, x);
                load_vec<float, CPL, false>(u + (size_t)t * D, uu);
                load_vec<float, CPL, false>(dret + (size_t)t * D, dr);
#pragma unroll
                for (int c = 0; c < CPL; ++c) { a = fmaf(y[c], uu[c], a); b = fmaf(dr[c], x[c], b); }
            }
            a = warp_sum(a);
            b = warp_sum(b);
            if (lane == 0) {
                w.bddw[(size_t)p * CW + e] = a;
                w.bdgw[(size_t)p * CW + e] = b;
            }
        } else if (it < nw + nr) {
            const int e = it - nw, t = div_by(e, magR);
            const int s = in.rs[tok0 * R + e];
            float a = 0.f;
            if ((unsigned)s < (unsigned)d.S) {
                float x[CPL], y[CPL];
                load_vec<BT, CPL, false>(bank + (size_t)s * D, x);
                load_vec<float, CPL, false>(dO + (size_t)t * D, y);
#pragma unroll
                for (int c = 0; c < CPL; ++c) a = fmaf(y[c], x[c], a);
            }
            a = warp_sum(a);
            if (lane == 0) w.bdqw[(size_t)p * CR + e] = a;
        } else {
            const int g = it - nw - nr;
            const int sl = w.gslot[(size_t)n * CW + g];
            float a = 0.f;
            if ((unsigned)sl < (unsigned)d.S) {
                float x[CPL], y[CPL];
                load_vec<BT, CPL, false>(bank + (size_t)sl * D, x);
                load_vec<float, CPL, false>(gb + (size_t)sl * D, y);
#pragma unroll
                for (int c = 0; c < CPL; ++c) a = fmaf(y[c], x[c], a);
            }
            a = warp_sum(a);
            if (lane == 0) w.bdfac[(size_t)p * CW + w.goff[(size_t)n * goff_stride(CW) + g]] = a;
        }
    }
}

// ---------------------------------------------------------------------------------------
// bank gradient: written slots, then read slots (one warp per group, members in order)
// ---------------------------------------------------------------------------------------
template <int CPL>
__global__ void __launch_bounds__(NTB) k_b_dbw(Dims d, Work w, float *gbank, int step0, int ti) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p = blockIdx.y, n = local_n(d, step0, ti, p);
    const int C = d.C, D = d.D, W = d.W, CW = C * W;
    const int ng = w.ngroups[n];
    const int32_t *goff = w.goff + (size_t)n * goff_stride(CW);
    const int32_t *gslot = w.gslot + (size_t)n * CW;
    const float *gfac = w.gfac + (size_t)n * CW;
    const int32_t *perm = w.perm + (size_t)n * CW;
    const float *gw = w.gw + (size_t)n * CW;
    const float *dret = w.bdret + (size_t)p * C * D + lane * CPL;
    float *gb = gbank + stream_row0(d, p) * D + lane * CPL;
    const unsigned magW = div_magic(W);
    for (int g = blockIdx.x * NWB + warp; g < ng; g += gridDim.x * NWB) {
        const int sl = gslot[g];
        if ((unsigned)sl >= (unsigned)d.S) continue;
        float acc[CPL];
        load_vec<float, CPL, false>(gb + (size_t)sl * D, acc);
        const float f = gfac[g];
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] *= f;
        for (int m = goff[g]; m < goff[g + 1]; ++m) {
            const int e = perm[m];
            float x[CPL];
            load_vec<float, CPL, false>(dret + (size_t)div_by(e, magW) * D, x);
            const float a = gw[e];
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = fmaf(a, x[c], acc[c]);
        }
        store_vec<float, CPL>(gb + (size_t)sl * D, acc);
    }
}

template <int CPL>
__global__ void __launch_bounds__(NTB) k_b_dbr(Dims d, Work w, float *gbank, int step0, int ti) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p = blockIdx.y, n = local_n(d, step0, ti, p);
    const int C = d.C, D = d.D, R = d.R, CR = C * R;
    const int ng = w.rng[n];
    const int32_t *goff = w.rgoff + (size_t)n * (CR + 1);
    const int32_t *gslot = w.rgslot + (size_t)n * CR;
    const unsigned long long *rkey = w.rkey + (size_t)n * CR;
    const float *qw = w.qw + (size_t)n * CR;
    const float *dO = w.bdo + (size_t)p * C * D + lane * CPL;
    float *gb = gbank + stream_row0(d, p) * D + lane * CPL;
    for (int g = blockIdx.x * NWB + warp; g < ng; g += gridDim.x * NWB) {
        const int sl = gslot[g];
        if ((unsigned)sl >= (unsigned)d.S) continue;
        float acc[CPL];
        load_vec<float, CPL, false>(gb + (size_t)sl * D, acc);
        for (int m = goff[g]; m < goff[g + 1]; ++m) {
            const unsigned low = (unsigned)rkey[m];
            const int t = (int)(low >> 8), e = t * R + (int)(low & 255u);
            float x[CPL];
            load_vec<float, CPL, false>(dO + (size_t)t * D, x);
            const float a = qw[e];
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = fmaf(a, x[c], acc[c]);
        }
        store_vec<float, CPL>(gb + (size_t)sl * D, acc);
    }
}

// ---------------------------------------------------------------------------------------
// Phase-1 backward: dk, dq, dg, in three launches per step (stage 0: reads, 1: writes, 2:
// groups; each stage needs the previous one's results for the whole chunk). A launch has
// gridDim.x CTAs per stream, each taking a contiguous share of the sorted entries, one warp per
// entry (a thread per group in stage 2).
// ---------------------------------------------------------------------------------------
template <typename WT>
__global__ void __launch_bounds__(NTB) k_b_phase1(Dims d, Inputs in, Work w, float *gk,
                                                 float *gg, float *gq, int step0, int ti,
                                                 int stage) {
    const int p = blockIdx.y, n = local_n(d, step0, ti, p);
    const int C = d.C, W = d.W, R = d.R, CW = C * W, CR = C * R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = w.nvalid[n], nw = nv * W, nr = nv * R;
    const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;
    const WT *kin = static_cast<const WT *>(in.kw) + tok0 * W;
    const WT *qin = static_cast<const WT *>(in.qw) + tok0 * R;
    const unsigned long long *wkey = w.wkey + (size_t)n * CW;
    const float *lws = w.wlws + (size_t)n * CW;
    const int32_t *pgs = w.wpgs + (size_t)n * CW;
    const int32_t *pge = w.wpge + (size_t)n * CW;
    const unsigned long long *rkey = w.rkey + (size_t)n * CR;
    const float *lr = w.lr + (size_t)n * CR;
    const float *qwv = w.qw + (size_t)n * CR;
    const float *dA = w.bdA + (size_t)p * C * C;
    const float *dQK = w.bdQK + (size_t)p * C * C;
    const float *ddw = w.bddw + (size_t)p * CW;
    const float *dgw = w.bdgw + (size_t)p * CW;
    const float *dqw = w.bdqw + (size_t)p * CR;
    const float *dfac = w.bdfac + (size_t)p * CW;
    float *dlam = w.bdlam + (size_t)p * CW;
    float *dlr = w.bdlr + (size_t)p * CR;
    const unsigned S = (unsigned)d.S;
    auto kval = [&](unsigned low) {   // write weight of a sorted write key's entry
        return to_f32(kin[(int)(low >> 8) * W + (int)(low & 255u)]);
    };
    // branch-free searches in a sorted key row, K at a time (the same probe count for all, so
    // the K searches overlap): upper bound (first key > target) or lower bound (first key >=)
    extern __shared__ int32_t bp1_found[];   // per entry of this CTA's share (see below)
    auto bounds = [&](const unsigned long long *row, int len0, const unsigned long long (&tg)[4],
                      bool upper, int (&res)[4]) {
        int base[4] = {0, 0, 0, 0};
        for (int len = len0; len > 1;) {
            const int half = len >> 1;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const unsigned long long v = row[base[k] + half - 1];
                if (upper ? v <= tg[k] : v < tg[k]) base[k] += half;
            }
            len -= half;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const unsigned long long v = len0 > 0 ? row[base[k]] : 0ull;
            res[k] = len0 > 0 ? base[k] + ((upper ? v <= tg[k] : v < tg[k]) ? 1 : 0) : 0;
        }
    };

    // this CTA's share [b0, b1) of the n entries of a stage
    auto share = [&](int cnt, int &b0, int &b1) {
        const int per = (cnt + gridDim.x - 1) / gridDim.x;
        b0 = blockIdx.x * per;
        b1 = b0 + per < cnt ? b0 + per : cnt;
    };
    int b0, b1;

    // (i) reads: dq and the gradient of their running log-decay
    if (stage == 0) {
    share(nr, b0, b1);
    // the last write of each read's slot at a token <= the read's (-1: none)
    for (int i0 = b0 + (int)threadIdx.x; i0 < b1; i0 += 4 * NTB) {
        unsigned long long tg[4];
        int res[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = i0 + k * NTB < b1 ? i0 + k * NTB : b0;
            const unsigned long long key = rkey[i];
            tg[k] = (key & 0xffffffff00000000ull) | (((unsigned)key >> 8) << 8) | 255u;
        }
        bounds(wkey, nw, tg, true, res);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = i0 + k * NTB;
            if (i >= b1) continue;
            const int pos = res[k] - 1;
            bp1_found[i - b0] =
                (pos >= 0 && (wkey[pos] >> 32) == (tg[k] >> 32)) ? pos : -1;
        }
    }
    __syncthreads();
    for (int rp = b0 + warp; rp < b1; rp += NWB) {
        const unsigned long long key = rkey[rp];
        const unsigned r = (unsigned)(key >> 32);
        const unsigned low = (unsigned)key;
        const int t = (int)(low >> 8), e = t * R + (int)(low & 255u);
        float dq = 0.f, dl = 0.f;
        if (r < S) {
            const float q = to_f32(qin[e]), l = lr[e];
            const int hi = bp1_found[rp - b0];
            float sum = 0.f;
            if (hi >= 0) {
                for (int m = pgs[hi] + lane; m <= hi; m += 32) {
                    const unsigned lb = (unsigned)wkey[m];
                    sum = fmaf(dQK[(size_t)t * C + (lb >> 8)], kval(lb) * expf(l - lws[m]), sum);
                }
            }
            sum = warp_sum(sum);
            const float el = expf(l);
            dq = dqw[e] * el + sum;
            dl = dqw[e] * qwv[e] + q * sum;
        }
        if (lane == 0) {
            gq[(tok0 + t) * R + (low & 255u)] = dq;
            dlr[rp] = dl;
        }
    }
    // padding tokens of the chunk: zero gradients
    if (blockIdx.x == 0) {
        const int tmax = (size_t)ti * C + C <= (size_t)d.T ? C : d.T - ti * C;
        for (int i = nr + threadIdx.x; i < tmax * R; i += NTB) gq[tok0 * R + i] = 0.f;
    }
    return;
    }
    // (ii) writes: dk and the gradient of their running log-decay
    if (stage == 1) {
    share(nw, b0, b1);
    // the sorted reads of each write's slot at tokens >= the write's: [r0, r1)
    for (int i0 = b0 + (int)threadIdx.x; i0 < b1; i0 += 2 * NTB) {
        unsigned long long tg[4];
        int res[4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = i0 + k * NTB < b1 ? i0 + k * NTB : b0;
            const unsigned long long key = wkey[i];
            const unsigned long long slot = key & 0xffffffff00000000ull;
            tg[2 * k] = slot | (((unsigned)key >> 8) << 8);
            tg[2 * k + 1] = slot | ((unsigned long long)C << 8);
        }
        bounds(rkey, nr, tg, false, res);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = i0 + k * NTB;
            if (i >= b1) continue;
            bp1_found[2 * (i - b0)] = res[2 * k];
            bp1_found[2 * (i - b0) + 1] = res[2 * k + 1];
        }
    }
    __syncthreads();
    for (int pa = b0 + warp; pa < b1; pa += NWB) {
        const unsigned long long key = wkey[pa];
        const unsigned s = (unsigned)(key >> 32);
        const unsigned low = (unsigned)key;
        const int ta = (int)(low >> 8), e = ta * W + (int)(low & 255u);
        float dk = 0.f, dlam_a = 0.f;
        if (s < S) {
            const float ka = kval(low), la = lws[pa];
            const int gs = pgs[pa], ge = pge[pa];
            const float lend = lws[ge - 1];
            float s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f;
            for (int m = gs + lane; m < pa; m += 32) {
                const unsigned lb = (unsigned)wkey[m];
                s1 = fmaf(dA[(size_t)ta * C + (lb >> 8)], kval(lb) * expf(la - lws[m]), s1);
            }
            for (int m = pa + 1 + lane; m < ge; m += 32) {
                const unsigned lc = (unsigned)wkey[m];
                s2 = fmaf(dA[(size_t)(lc >> 8) * C + ta], kval(lc) * expf(lws[m] - la), s2);
            }
            const int tnext = (pa + 1 < ge) ? (int)((unsigned)wkey[pa + 1] >> 8) : C;
            const int r0 = bp1_found[2 * (pa - b0)], r1 = bp1_found[2 * (pa - b0) + 1];
            for (int m = r0 + lane; m < r1; m += 32) {
                const unsigned lr_ = (unsigned)rkey[m];
                const int tr = (int)(lr_ >> 8), er = tr * R + (int)(lr_ & 255u);
                s3 = fmaf(dQK[(size_t)tr * C + ta], to_f32(qin[er]) * expf(lr[er] - la), s3);
                if (tr < tnext) s4 += dlr[m];
            }
            s1 = warp_sum(s1);
            s2 = warp_sum(s2);
            s3 = warp_sum(s3);
            s4 = warp_sum(s4);
            const float e1 = expf(la), e2 = expf(lend - la);
            dk = dgw[e] * e1 + ddw[e] * e2 + s1 + s2 + s3;
            dlam_a = dgw[e] * ka * e1 - ddw[e] * ka * e2 + ka * (s1 - s2 - s3) + s4;
        }
        if (lane == 0) {
            gk[(tok0 + ta) * W + (low & 255u)] = dk;
            dlam[pa] = dlam_a;
        }
    }
    if (blockIdx.x == 0) {
        const int tmax = (size_t)ti * C + C <= (size_t)d.T ? C : d.T - ti * C;
        for (int i = nw + threadIdx.x; i < tmax * W; i += NTB) gk[tok0 * W + i] = 0.f;
    }
    return;
    }
    // (iii) per group: the gradient of its total log-decay, then dg as suffix sums
    share(nw, b0, b1);
    for (int pa = b0 + threadIdx.x; pa < b1; pa += NTB) {
        if (pgs[pa] != pa) continue;              // one thread per group (its head)
        const unsigned s = (unsigned)(wkey[pa] >> 32);
        const int ge = pge[pa];
        float dend = 0.f;
        if (s < S) {
            const float lend = lws[ge - 1];
            for (int m = pa; m < ge; ++m) {
                const unsigned lb = (unsigned)wkey[m];
                const int eb = (int)(lb >> 8) * W + (int)(lb & 255u);
                dend = fmaf(ddw[eb], kval(lb) * expf(lend - lws[m]), dend);
            }
            dend = fmaf(dfac[pa], expf(lend), dend);
        }
        float run = dend;
        for (int m = ge - 1; m >= pa; --m) {
            const unsigned lb = (unsigned)wkey[m];
            run += dlam[m];
            const size_t ge_out = (size_t)(lb >> 8) * W + (lb & 255u);
            if (d.gate) w.bdgate[(size_t)p * CW + ge_out] = s < S ? run : 0.f;
            else gg[tok0 * W + ge_out] = s < S ? run : 0.f;
        }
    }
    if (blockIdx.x == 0) {
        const int tmax = (size_t)ti * C + C <= (size_t)d.T ? C : d.T - ti * C;
        for (int i = nw + threadIdx.x; i < tmax * W; i += NTB) {
            if (d.gate) w.bdgate[(size_t)p * CW + i] = 0.f;
            else gg[tok0 * W + i] = 0.f;
        }
    }
}

// per-token gate: the token's log-decay gradient is the sum of its W per-entry gradients, in
// entry order (one thread per token of the step's chunk)
__global__ void __launch_bounds__(NTB) k_b_gate(Dims d, Work w, float *gg, int ti) {
    const int p = blockIdx.y, CW = d.C * d.W;
    const int t = blockIdx.x * NTB + threadIdx.x;
    const int tmax = (size_t)ti * d.C + d.C <= (size_t)d.T ? d.C : d.T - ti * d.C;
    if (t >= tmax) return;
    const float *e = w.bdgate + (size_t)p * CW + (size_t)t * d.W;
    float sum = 0.f;
    for (int j = 0; j < d.W; ++j) sum += e[j];
    gg[(size_t)p * d.T + (size_t)ti * d.C + t] = sum;
}

template <typename T>
void set_smem(T kern, size_t bytes) {
    set_kernel_smem(kern, bytes);
}

void gemm(const GemmOp &g, int batch, cudaStream_t st) {
    dim3 grid((g.N + GT - 1) / GT, (g.M + GT - 1) / GT, batch);
    k_bgemm<<<grid, GTHREADS, 0, st>>>(g);
}

template <typename BT, int CPL>
cudaError_t backward_step(const Dims &d, const Inputs &in, const Work &w, const BwdOut &o,
                          int step0, int ti, cudaStream_t st) {
    const int P = d.P, C = d.C, D = d.D;
    int gx = (8 * kRefSms + P - 1) / P;
    const int grp_blocks = (d.C * d.W + NWB - 1) / NWB;
    if (gx > grp_blocks) gx = grp_blocks;
    if (gx < 1) gx = 1;
    k_b_restore<BT, CPL><<<dim3(gx, P), NTB, 0, st>>>(d, in, w, step0, ti);
    k_b_gather<BT, CPL><<<(P * C + NWB - 1) / NWB, NTB, 0, st>>>(d, in, w, o.grad_bank, step0, ti);
    const int dtiles = (D + TN - 1) / TN;
    const size_t smem1 = sizeof(float) * ((size_t)3 * C * TN + (size_t)3 * C * TM);
    set_smem(k_b_mm1<BT>, smem1);
    k_b_mm1<BT><<<dim3((C + TM - 1) / TM, dtiles, P), NTB, smem1, st>>>(d, in, w, o.grad_readings,
                                                                         o.grad_v, step0, ti);
    const long long cc = (long long)C * C, cd = (long long)C * D;
    const int n0 = (ti - step0) * P;
    const float *X = w.X + (size_t)n0 * cc, *QK = w.QK + (size_t)n0 * cc;
    // dX = du u_pre^T ; dQX = dO u_pre^T
    gemm({w.dv, w.bup, w.bdX, cd, cd, cc, D, D, C, 0, 1, C, C, D, 1.f, 0, 0}, P, st);
    gemm({w.bdo, w.bup, w.bdQX, cd, cd, cc, D, D, C, 0, 1, C, C, D, 1.f, 0, 0}, P, st);
    // dX += QK^T dQX ; dQK = tril(dQX X^T)
    gemm({QK, w.bdQX, w.bdX, cc, cc, cc, C, C, C, 1, 0, C, C, C, 1.f, 1, 0}, P, st);
    gemm({w.bdQX, X, w.bdQK, cc, cc, cc, C, C, C, 0, 1, C, C, C, 1.f, 0, 1}, P, st);
    // dL = -strict_tril(X^T dX X^T)
    gemm({X, w.bdX, w.bT, cc, cc, cc, C, C, C, 1, 0, C, C, C, 1.f, 0, 0}, P, st);
    gemm({w.bT, X, w.bdA, cc, cc, cc, C, C, C, 0, 1, C, C, C, -1.f, 0, 2}, P, st);
    k_b_beta<<<P, NTB, 0, st>>>(d, in, w, o.grad_beta, step0, ti, dtiles);
    const int ent_blocks = (C * (d.W + d.R) + C * d.W + NWB - 1) / NWB;
    int gd = (8 * kRefSms + P - 1) / P;
    if (gd > ent_blocks) gd = ent_blocks;
    k_b_dots<BT, CPL><<<dim3(gd, P), NTB, 0, st>>>(d, in, w, o.grad_bank, step0, ti);
    k_b_dbw<CPL><<<dim3(gx, P), NTB, 0, st>>>(d, w, o.grad_bank, step0, ti);
    int gr = (d.C * d.R + NWB - 1) / NWB;
    if (gr > gx) gr = gx;
    if (gr < 1) gr = 1;
    k_b_dbr<CPL><<<dim3(gr, P), NTB, 0, st>>>(d, w, o.grad_bank, step0, ti);
    // Phase-1 backward: about 8 entries per warp and stage (one warp walks an entry's members)
    const int per_cta = 8 * NWB;
    int gb = (d.C * (d.W > d.R ? d.W : d.R) + per_cta - 1) / per_cta;
    const int gmax = (8 * kRefSms + P - 1) / P;
    if (gb > gmax) gb = gmax;
    if (gb < 1) gb = 1;
    const int most = d.C * (d.W > d.R ? d.W : d.R);
    const size_t found_bytes = 2 * sizeof(int32_t) * (size_t)((most + gb - 1) / gb);
    set_smem(k_b_phase1<BT>, found_bytes);
    for (int stage = 0; stage < 3; ++stage)
        k_b_phase1<BT><<<dim3(gb, P), NTB, found_bytes, st>>>(
            d, in, w, o.grad_write_w, o.grad_log_decay, o.grad_read_w, step0, ti, stage);
    if (d.gate) k_b_gate<<<dim3((C + NTB - 1) / NTB, P), NTB, 0, st>>>(d, w, o.grad_log_decay, ti);
    return cudaGetLastError();
}

}  // namespace

#define SDM_DISPATCH_BWD(BT)                                                       \
    switch (d.D) {                                                                 \
        case 32: return backward_step<BT, 1>(d, in, w, o, step0, ti, st);          \
        case 64: return backward_step<BT, 2>(d, in, w, o, step0, ti, st);          \
        case 128: return backward_step<BT, 4>(d, in, w, o, step0, ti, st);         \
        case 256: return backward_step<BT, 8>(d, in, w, o, step0, ti, st);         \
        case 512: return backward_step<BT, 16>(d, in, w, o, step0, ti, st);        \
        default: return cudaErrorInvalidValue;                                     \
    }

cudaError_t launch_backward_step(const Dims &d, const Inputs &in, const Work &w,
                                 const BwdOut &o, int step0, int ti, cudaStream_t st) {
    if (d.dtype == SDM_BF16) { SDM_DISPATCH_BWD(__nv_bfloat16) }
    SDM_DISPATCH_BWD(float)
}

}  // namespace sdm
