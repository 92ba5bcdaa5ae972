// Phase 2 of the chunked SDM write/read: one step ti covers chunk ti of all P streams
// (sparse-delta-memory 2.0.0, phase2_kernels.py module docstring: "forward gather -> dual
// matmul -> DW"; the dual matmul's definition is the _sdm_dual_matmul docstring).
//
//   gather   retrieved[t] = sum_j gw[t][j] B[s_tj],  inter[t] = sum_i qw[t][i] B[r_ti]
//            (B = the bank at the start of the chunk), u_pre = beta (v - retrieved);
//            f32 rows [P][C][D] of u_pre and inter
//   dual mm  delta_v = X u_pre;  readings = QX u_pre + inter (TF32 tensor cores: tcgen05 in
//            dualmm_tc.cu when C is a multiple of 128, else mma.sync below)
//   DW       for every written slot s (one group of the sorted write row):
//            B[s] = exp(lend_s) B[s] + sum_{members m, sorted order} dw_m delta_v[t_m]
//            in f32, rounded once at the store; the group's single warp is the row's only
//            writer, so the step is deterministic without atomics.
//
// Rows of a warp: lane l holds columns [l*CPL, (l+1)*CPL) of a row (CPL = D / 32), so one
// warp-wide load moves a whole bank row with 4..64-byte vectors per lane.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kBlock = 256;           // threads of the gather and DW blocks
constexpr int kWarps = kBlock / 32;

// ---------------------------------------------------------------------------------------
// A lane's piece of a row: N consecutive elements of type T, held as raw 32-bit words and
// loaded with one vector load, then widened to float32 for the sums (a bfloat16 pair x of a
// word: low element = x << 16, high element = x & 0xffff0000).
// ---------------------------------------------------------------------------------------
template <typename T, int N>
struct Raw {
    static constexpr int BYTES = N * (int)sizeof(T);
    static constexpr int WORDS = BYTES >= 4 ? BYTES / 4 : 1;
    uint32_t u[WORDS];
};

template <typename T, int N>
__device__ __forceinline__ void raw_load(const T *p, Raw<T, N> &r) {
    constexpr int B = Raw<T, N>::BYTES;
    if constexpr (B >= 16) {
#pragma unroll
        for (int i = 0; i < B / 16; ++i) {
            const uint4 v = reinterpret_cast<const uint4 *>(p)[i];
            r.u[4 * i] = v.x; r.u[4 * i + 1] = v.y; r.u[4 * i + 2] = v.z; r.u[4 * i + 3] = v.w;
        }
    } else if constexpr (B == 8) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        r.u[0] = v.x; r.u[1] = v.y;
    } else if constexpr (B == 4) {
        r.u[0] = *reinterpret_cast<const uint32_t *>(p);
    } else {
        r.u[0] = *reinterpret_cast<const unsigned short *>(p);
    }
}

template <typename T, int N>
__device__ __forceinline__ void raw_zero(Raw<T, N> &r) {
#pragma unroll
    for (int i = 0; i < Raw<T, N>::WORDS; ++i) r.u[i] = 0u;
}

template <typename T, int N>
__device__ __forceinline__ void raw_widen(const Raw<T, N> &r, float (&x)[N]) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int c = 0; c < N; ++c) x[c] = __uint_as_float(r.u[c]);
    } else if constexpr (N == 1) {
        x[0] = __uint_as_float(r.u[0] << 16);
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 2) {
            x[c] = __uint_as_float(r.u[c / 2] << 16);
            x[c + 1] = __uint_as_float(r.u[c / 2] & 0xffff0000u);
        }
    }
}

// acc += w * x, two columns at a time with the packed FMA (each half rounded like fmaf)
template <int N>
__device__ __forceinline__ void axpy(float (&acc)[N], float w, const float (&x)[N]) {
    if constexpr (N == 1) {
        acc[0] = fmaf(w, x[0], acc[0]);
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 2) {
            const float2 r = __ffma2_rn(make_float2(w, w), make_float2(x[c], x[c + 1]),
                                        make_float2(acc[c], acc[c + 1]));
            acc[c] = r.x;
            acc[c + 1] = r.y;
        }
    }
}

// ---------------------------------------------------------------------------------------
// gather: WPT warps per token split the token's entries; their partial sums are added in
// warp order (a fixed order, WPT a function of the shape only)
// ---------------------------------------------------------------------------------------
template <typename BT, int CPL, int WPT>
__global__ void __launch_bounds__(kBlock) k_gather(Dims d, Inputs in, Work w, int step0, int ti) {
    constexpr int TPB = kWarps / WPT;
    __shared__ float part[(WPT > 1) ? kWarps : 1][2][(WPT > 1) ? 32 * CPL : 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tb = warp / WPT, sub = warp % WPT;
    const int C = d.C, D = d.D, W = d.W, R = d.R;
    const int gtok = blockIdx.x * TPB + tb;
    const int p = gtok / C, t = gtok - p * C;
    const int n = (ti - step0) * d.P + p;
    bool active = gtok < d.P * C;
    if (active) active = t < w.nvalid[n];

    float ar[CPL], ai[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) { ar[c] = 0.f; ai[c] = 0.f; }
    if (active) {
        const size_t tok = (size_t)p * d.T + (size_t)ti * C + t;
        const BT *bank = static_cast<const BT *>(in.bank) + stream_row0(d, p) * D + lane * CPL;
        const unsigned S = (unsigned)d.S;
        {
            const int32_t *ws = in.ws + tok * W;
            const float *gw = w.gw + (size_t)n * C * W + (size_t)t * W;
            const int j0 = sub * W / WPT, j1 = (sub + 1) * W / WPT;
            int j = j0;
            for (; j + 4 <= j1; j += 4) {
                int s[4];
                float wt[4], x[4][CPL];
#pragma unroll
                for (int u = 0; u < 4; ++u) { s[u] = ws[j + u]; wt[u] = gw[j + u]; }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if ((unsigned)s[u] < S) load_vec<BT, CPL, true>(bank + (size_t)s[u] * D, x[u]);
                    else {
#pragma unroll
                        for (int c = 0; c < CPL; ++c) x[u][c] = 0.f;
                        wt[u] = 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) axpy(ar, wt[u], x[u]);
            }
            for (; j < j1; ++j) {
                const int s = ws[j];
                if ((unsigned)s >= S) continue;
                float x[CPL];
                load_vec<BT, CPL, true>(bank + (size_t)s * D, x);
                axpy(ar, gw[j], x);
            }
        }
        {
            const int32_t *rs = in.rs + tok * R;
            const float *qw = w.qw + (size_t)n * C * R + (size_t)t * R;
            const int i0 = sub * R / WPT, i1 = (sub + 1) * R / WPT;
            int i = i0;
            for (; i + 4 <= i1; i += 4) {
                int s[4];
                float wt[4], x[4][CPL];
#pragma unroll
                for (int u = 0; u < 4; ++u) { s[u] = rs[i + u]; wt[u] = qw[i + u]; }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if ((unsigned)s[u] < S) load_vec<BT, CPL, true>(bank + (size_t)s[u] * D, x[u]);
                    else {
#pragma unroll
                        for (int c = 0; c < CPL; ++c) x[u][c] = 0.f;
                        wt[u] = 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) axpy(ai, wt[u], x[u]);
            }
            for (; i < i1; ++i) {
                const int s = rs[i];
                if ((unsigned)s >= S) continue;
                float x[CPL];
                load_vec<BT, CPL, true>(bank + (size_t)s * D, x);
                axpy(ai, qw[i], x);
            }
        }
    }
    const size_t row = ((size_t)p * C + t) * D + lane * CPL;
    // u_pre = beta (v - retrieved), kept for the dual matmul in place of retrieved
    auto finish = [&]() {
        const size_t tok = (size_t)p * d.T + (size_t)ti * C + t;
        float vv[CPL];
        load_vec<BT, CPL, false>(static_cast<const BT *>(in.v) + tok * D + lane * CPL, vv);
        const float bt = in.beta[tok];
#pragma unroll
        for (int c = 0; c < CPL; ++c) ar[c] = bt * (vv[c] - ar[c]);
        if (dualmm_tc_fits(d)) {   // u_pre transposed for the tensor-core dual matmul
            float *ut = w.ret + ((size_t)p * D + lane * CPL) * C + t;
#pragma unroll
            for (int c = 0; c < CPL; ++c) ut[(size_t)c * C] = ar[c];
        } else {
            store_vec<float, CPL>(w.ret + row, ar);
        }
        store_vec<float, CPL>(w.inter + row, ai);
    };
    // a padding token's u_pre column is zero for the tensor-core dual matmul, whose K-blocks
    // of 32 tokens reach past the valid ones (its X and QX entries there are 0)
    if (!active && gtok < d.P * C && sub == 0 && dualmm_tc_fits(d)) {
        float *ut = w.ret + ((size_t)p * D + lane * CPL) * C + t;
#pragma unroll
        for (int c = 0; c < CPL; ++c) ut[(size_t)c * C] = 0.f;
    }
    if constexpr (WPT == 1) {
        if (active) finish();
    } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            part[warp][0][lane * CPL + c] = ar[c];
            part[warp][1][lane * CPL + c] = ai[c];
        }
        __syncthreads();
        if (active && sub == 0) {
#pragma unroll
            for (int s = 1; s < WPT; ++s)
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    ar[c] += part[warp + s][0][lane * CPL + c];
                    ai[c] += part[warp + s][1][lane * CPL + c];
                }
            finish();
        }
    }
}

// ---------------------------------------------------------------------------------------
// dual matmul on the tensor cores: a 16-row x 64-column tile of delta_v = X u_pre and of
// readings = QX u_pre + inter of one chunk per CTA. X and QX rows and the u_pre tile are
// copied on chip (cp.async, 16 bytes at a time where aligned); 4 warps, each one matrix and
// four n8 tiles, mma.sync m16n8k8 TF32 (3xTF32 for float32 banks, as in the pipelined kernel).
// ---------------------------------------------------------------------------------------
constexpr int MM_R = 16, MM_N = 64, MM_T = 128;

__host__ __device__ inline int mm_kpad(int C) { return (C + 7) & ~7; }
__host__ __device__ inline int mm_apitch(int C) { return mm_kpad(C) + 4; }   // conflict-free A
constexpr int MM_UP = MM_N + 8;                                                // conflict-free B

template <typename BT>
__global__ void __launch_bounds__(MM_T) k_dualmm(Dims d, Inputs in, Work w, int step0, int ti) {
    extern __shared__ __align__(16) float dm_smem[];
    const int C = d.C, D = d.D, K = mm_kpad(C), AP = mm_apitch(C);
    const int m0 = blockIdx.x * MM_R, d0 = blockIdx.y * MM_N, p = blockIdx.z;
    const int n = (ti - step0) * d.P + p;
    const int nv = w.nvalid[n];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *Xs = dm_smem;                 // [16][AP]
    float *Qs = Xs + MM_R * AP;          // [16][AP]
    float *Us = Qs + MM_R * AP;          // [K][MM_UP]
    const float *X = w.X + (size_t)n * C * C;
    const float *QX = w.QX + (size_t)n * C * C;
    const float *U = w.ret + (size_t)p * C * D;
    const float *inter = w.inter + (size_t)p * C * D;
    const size_t tok0 = (size_t)p * d.T + (size_t)ti * C;

    // X, QX rows m0..m0+15 (zero past C and past column C), u_pre rows k < nv (zero beyond)
    const bool a16 = (C & 3) == 0;
    for (int idx = tid; idx < MM_R * K; idx += MM_T) {
        const int r = idx / K, k = idx - r * K, row = m0 + r;
        if (row < C && k < C) {
            if (a16) {
                if ((k & 3) == 0) {
                    cp_async16(Xs + r * AP + k, X + (size_t)row * C + k);
                    cp_async16(Qs + r * AP + k, QX + (size_t)row * C + k);
                }
            } else {
                cp_async4(Xs + r * AP + k, X + (size_t)row * C + k);
                cp_async4(Qs + r * AP + k, QX + (size_t)row * C + k);
            }
        } else {
            Xs[r * AP + k] = 0.f;
            Qs[r * AP + k] = 0.f;
        }
    }
    const int ncol = D - d0 < MM_N ? D - d0 : MM_N;
    for (int idx = tid; idx < K * (MM_N / 4); idx += MM_T) {
        const int k = idx / (MM_N / 4), c = (idx - k * (MM_N / 4)) * 4;
        if (k < nv && c < ncol) cp_async16(Us + k * MM_UP + c, U + (size_t)k * D + d0 + c);
        else *reinterpret_cast<float4 *>(Us + k * MM_UP + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    const int g4 = lane >> 2, i4 = lane & 3;
    const int mat = warp >> 1, nb = (warp & 1) * 4;          // this warp: matrix, first n8 tile
    const float *A = mat ? Qs : Xs;
    // independent accumulator chains: even and odd k-steps apart (h), and for float32 banks the
    // two small 3xTF32 terms apart from hi*hi (accs); summed once at the end in a fixed order
    constexpr int NS = sizeof(BT) == 4 ? 2 : 1;
    float acc[2][4][4], accs[NS][4][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[h][j][q] = 0.f;
#pragma unroll
    for (int h = 0; h < NS; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) accs[h][j][q] = 0.f;
    const int kend = mm_kpad(nv < C ? nv : C);                // u_pre is zero past nv
    for (int k00 = 0; k00 < kend; k00 += 16) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k0 = k00 + 8 * h;
            if (k0 >= kend) break;
            const float af[4] = {A[g4 * AP + k0 + i4], A[(g4 + 8) * AP + k0 + i4],
                                 A[g4 * AP + k0 + i4 + 4], A[(g4 + 8) * AP + k0 + i4 + 4]};
            unsigned ah[4], al[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) ah[q] = to_tf32(af[q]);
            if constexpr (sizeof(BT) == 4) {
#pragma unroll
                for (int q = 0; q < 4; ++q) al[q] = to_tf32(af[q] - __uint_as_float(ah[q]));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = (nb + j) * 8 + g4;
                const float bf[2] = {Us[(k0 + i4) * MM_UP + col], Us[(k0 + i4 + 4) * MM_UP + col]};
                unsigned bh[2] = {to_tf32(bf[0]), to_tf32(bf[1])};
                if constexpr (sizeof(BT) == 4) {
                    unsigned bl[2] = {to_tf32(bf[0] - __uint_as_float(bh[0])),
                                      to_tf32(bf[1] - __uint_as_float(bh[1]))};
                    mma_tf32(accs[h & (NS - 1)][j], ah, bl);
                    mma_tf32(accs[h & (NS - 1)][j], al, bh);
                }
                mma_tf32(acc[h][j], ah, bh);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc[0][j][q] += acc[1][j][q];
            if constexpr (sizeof(BT) == 4) acc[0][j][q] += accs[0][j][q] + accs[NS - 1][j][q];
        }

    BT *out = static_cast<BT *>(in.readings);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {                 // rows g4 and g4 + 8, two columns each
            const int row = m0 + g4 + 8 * h, col = d0 + (nb + j) * 8 + 2 * i4;
            if (row >= C || col >= D) continue;
            const bool live = row < nv;
            float o[2] = {live ? acc[0][j][2 * h] : 0.f, live ? acc[0][j][2 * h + 1] : 0.f};
            if (mat == 0) {
                store_vec<float, 2>(w.dv + ((size_t)p * C + row) * D + col, o);
            } else if ((size_t)ti * C + row < (size_t)d.T) {
                if (live) {
                    float it[2];
                    load_vec<float, 2, false>(inter + (size_t)row * D + col, it);
                    o[0] += it[0];
                    o[1] += it[1];
                }
                store_vec<BT, 2>(out + (tok0 + row) * D + col, o);
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// DW: every group (distinct written slot) of the step's P chunks.
//   B[s] = exp(lend_s) B0[s] + sum over the group's members, in sorted order, dw_m delta_v[t_m]
// in float32, rounded once at the store; one warp writes each element of the row.
// A CTA owns one chunk and one slice of DS = 32 CPS columns, and first copies the chunk's
// delta_v slice ([C][DS] float32, at most 128 KB) into shared memory: every delta_v row is read
// by every group that row's token writes (W groups), so from L2 those few rows would be
// requested by every SM at once. The hot groups (the first ones of the DW order Phase 1 wrote:
// at least max(kHotGroup, C/8) members) come first, a share of them per CTA, each summed by the
// whole CTA in rounds: their metadata, member records and B0 slices are staged in shared memory,
// a group's members are cut into chunks of 32 (sorted order), each warp sums one chunk, and the
// chunk sums are added to exp(lend) B0 in chunk order. A hot group summed by one warp would hold
// that warp (and the step) for its whole member list. The other groups go to the warps in a
// stride: a warp holds the metadata of 32 of its groups (lane l: group l, loaded one batch
// ahead), loads the B0 slices of U groups before adding any, and reads the members' delta_v
// from shared memory (member records 32 at a time, one batch ahead).
// ---------------------------------------------------------------------------------------
constexpr int DW_T = 1024;                   // threads per DW CTA (32 warps, 64 registers each)
constexpr int DW_W = DW_T / 32;
constexpr size_t kDwSmem = 128 * 1024;       // delta_v slice of a chunk in shared memory
constexpr int kDwHB = 16;                    // hot groups staged per round
constexpr int kDwRec = 2048;                 // member records staged per round

// the round's hot groups in shared memory (after the partial sums, B0 slices and records)
struct DwHot {
    int o0[kDwHB], nm[kDwHB], sl[kDwHB], roff[kDwHB + 1], toff[kDwHB + 1];
    float f[kDwHB];
    int cnt, big;
};

// dynamic shared memory of k_dw: delta_v slice [C][DS], partial sums [DW_W][DS], B0 slices
// [kDwHB][DS], records (token, weight) [kDwRec] x 2, DwHot
inline size_t dw_smem_bytes(int C, int DS) {
    return sizeof(float) * ((size_t)C * DS + (size_t)DW_W * DS + (size_t)kDwHB * DS) +
           8 * (size_t)kDwRec + sizeof(DwHot);
}

constexpr size_t kDwSmemMax = 200 * 1024;    // all of k_dw's shared memory

// columns per lane of a DW slice: the slice DS = 32 * CPS divides D, C * DS floats fit in
// kDwSmem and the whole layout in kDwSmemMax
inline int dw_cps(const Dims &d) {
    int ds = d.D;
    while (((size_t)d.C * ds * 4 > kDwSmem || dw_smem_bytes(d.C, ds) > kDwSmemMax) && ds > 32)
        ds >>= 1;
    return ds / 32;
}

template <typename BT, int CPS>
__global__ void __launch_bounds__(DW_T, 1) k_dw(Dims d, Inputs in, Work w, int step0, int ti, int cpp) {
    extern __shared__ __align__(16) float dvs[];       // [C][DS]
    constexpr int DS = 32 * CPS;
    constexpr int RB = CPS * (int)sizeof(BT);
    constexpr int U = RB >= 32 ? 1 : (RB >= 16 ? 2 : 4);   // B0 slices in flight per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int nsl = d.D / DS;
    const int pair = blockIdx.x / cpp, ck = blockIdx.x - pair * cpp;
    const int p = pair / nsl, cs = pair - p * nsl;
    const int n = (ti - step0) * d.P + p;
    const int C = d.C, D = d.D, W = d.W, CW = C * W;
    const int nv = w.nvalid[n];

    // the chunk's delta_v slice (rows past the valid tokens are never a member's)
    {
        const float *src = w.dv + (size_t)p * C * D + (size_t)cs * DS;
        constexpr int Q = DS / 4;                       // 16-byte pieces per row
        for (int i = tid; i < nv * Q; i += DW_T) {
            const int r = i / Q, q = i - r * Q;
            cp_async16(dvs + r * DS + q * 4, src + (size_t)r * D + q * 4);
        }
        cp_async_commit();
    }

    const int ng = w.ngroups[n];
    const int nhot = w.ng4[n].y;                       // gord positions [0, nhot): hot groups
    const int32_t *goff = w.goff + (size_t)n * goff_stride(CW);
    const int32_t *gslot = w.gslot + (size_t)n * CW;
    const int32_t *gord = w.gord + (size_t)n * CW;
    const float *gfac = w.gfac + (size_t)n * CW;
    const int32_t *perm = w.perm + (size_t)n * CW;
    const float *wdw = w.wdw + (size_t)n * CW;
    BT *bank = static_cast<BT *>(in.bank) + stream_row0(d, p) * D + (size_t)cs * DS + lane * CPS;
    const float *dvl = dvs + lane * CPS;
    const unsigned magic = div_magic(W);
    const int base = nhot + ck * DW_W + warp, stride = cpp * DW_W;
    const int mine = base < ng ? (ng - base + stride - 1) / stride : 0;
    const bool snap = in.snap != nullptr;

    // lane l: metadata of this warp's group q + l
    auto meta = [&](int q, int &sl, int &o0, int &o1, int &t1, float &f, float &w1) {
        sl = -1; o0 = o1 = t1 = 0; f = w1 = 0.f;
        if (q + lane < mine) {
            const int g = gord[base + (q + lane) * stride];
            sl = gslot[g];
            if ((unsigned)sl >= (unsigned)d.S) sl = -1;      // the dropped entries' group
            o0 = goff[g];
            o1 = goff[g + 1];
            f = gfac[g];
            t1 = div_by(perm[o0], magic);
            w1 = wdw[o0];
        }
    };
    int cslot, co0, co1, ct1, nslot, no0, no1, nt1;
    float cf, cw1, nf, nw1;
    meta(0, cslot, co0, co1, ct1, cf, cw1);
    meta(32, nslot, no0, no1, nt1, nf, nw1);
    cp_async_wait<0>();
    __syncthreads();

    // hot groups at gord positions ck, ck + cpp, ... (< nhot), by the whole CTA, in rounds:
    // a group's members split into chunks of 32 (in sorted order); the warps take the round's
    // chunks one each, and warp i adds group i's chunk sums to exp(lend) B0 in chunk order, so
    // every row is a fixed-order sum that depends on its own group alone
    {
        float *part = dvs + (size_t)C * DS;            // [DW_W][DS] chunk sums
        float *b0s = part + DW_W * DS;
        int *rec_t = reinterpret_cast<int *>(b0s + kDwHB * DS);
        float *rec_w = reinterpret_cast<float *>(rec_t + kDwRec);
        DwHot &hv = *reinterpret_cast<DwHot *>(rec_w + kDwRec);
        for (int h0 = 0; ck + h0 * cpp < nhot;) {
            if (warp == 0) {
                // the round: the next groups of this CTA whose records and chunks fit together;
                // a first group that alone does not fit is summed from global memory (big)
                const int q = ck + (h0 + lane) * cpp;
                const bool have = lane < kDwHB && q < nhot;
                int o0 = 0, nm = 0, sl = -1;
                float f = 0.f;
                if (have) {
                    const int g = gord[q];
                    o0 = goff[g];
                    nm = goff[g + 1] - o0;
                    sl = gslot[g];
                    if ((unsigned)sl >= (unsigned)d.S) sl = -1;
                    f = gfac[g];
                }
                int inc = nm, tinc = (nm + 31) >> 5;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, inc, off);
                    const int z = __shfl_up_sync(0xffffffffu, tinc, off);
                    if (lane >= off) { inc += y; tinc += z; }
                }
                const unsigned fit =
                    __ballot_sync(0xffffffffu, have && inc <= kDwRec && tinc <= DW_W);
                int cnt = __ffs(~fit) - 1;                 // leading lanes that fit
                const int big = cnt == 0 ? 1 : 0;          // lane 0 has a group (the loop test)
                if (big) cnt = 1;
                const int tot = big ? 0 : __shfl_sync(0xffffffffu, inc, cnt - 1);
                const int ttot = big ? DW_W : __shfl_sync(0xffffffffu, tinc, cnt - 1);
                if (lane < cnt) {
                    hv.o0[lane] = o0;
                    hv.nm[lane] = nm;
                    hv.sl[lane] = sl;
                    hv.f[lane] = f;
                    hv.roff[lane] = big ? 0 : inc - nm;
                    hv.toff[lane] = big ? 0 : tinc - ((nm + 31) >> 5);
                }
                if (lane == 0) {
                    hv.roff[cnt] = tot;
                    hv.toff[cnt] = ttot;
                    hv.cnt = cnt;
                    hv.big = big;
                }
            }
            __syncthreads();
            const int cnt = hv.cnt, big = hv.big, tot = hv.roff[cnt], ntask = hv.toff[cnt];
            for (int idx = tid; idx < tot; idx += DW_T) {
                int i = 0;
                while (i + 1 < cnt && hv.roff[i + 1] <= idx) ++i;
                const int pos = hv.o0[i] + (idx - hv.roff[i]);
                rec_t[idx] = div_by(perm[pos], magic);
                rec_w[idx] = wdw[pos];
            }
            if (warp < cnt && hv.sl[warp] >= 0) {
                Raw<BT, CPS> r;
                raw_load(bank + (size_t)hv.sl[warp] * D, r);
                float a[CPS];
                raw_widen(r, a);
#pragma unroll
                for (int c = 0; c < CPS; ++c) b0s[warp * DS + lane * CPS + c] = a[c];
            }
            __syncthreads();
            float acc[CPS];
#pragma unroll
            for (int c = 0; c < CPS; ++c) acc[c] = 0.f;
            if (!big) {
                // task `warp`: chunk warp - toff[i] of group i (records in shared memory)
                if (warp < ntask) {
                    int i = 0;
                    while (i + 1 < cnt && hv.toff[i + 1] <= warp) ++i;
                    const int m0 = (warp - hv.toff[i]) * 32;
                    const int m1 = hv.nm[i] - m0 < 32 ? hv.nm[i] : m0 + 32;
                    const int r0 = hv.roff[i];
                    for (int m = m0; m < m1; ++m) {
                        float x[CPS];
                        const float wv = rec_w[r0 + m];
                        load_vec<float, CPS, false>(dvl + rec_t[r0 + m] * DS, x);
                        axpy(acc, wv, x);
                    }
                }
            } else {
                // one large group: warp w sums its chunks w, w + DW_W, ... in order (records
                // from global memory)
                const int o0 = hv.o0[0], nm = hv.nm[0];
                for (int m0 = warp * 32; m0 < nm; m0 += DW_W * 32) {
                    int t = 0;
                    float wl = 0.f;
                    if (m0 + lane < nm) {
                        t = div_by(perm[o0 + m0 + lane], magic);
                        wl = wdw[o0 + m0 + lane];
                    }
                    const int mc = nm - m0 < 32 ? nm - m0 : 32;
                    for (int v = 0; v < mc; ++v) {
                        float x[CPS];
                        const int tv = __shfl_sync(0xffffffffu, t, v);
                        const float wv = __shfl_sync(0xffffffffu, wl, v);
                        load_vec<float, CPS, false>(dvl + tv * DS, x);
                        axpy(acc, wv, x);
                    }
                }
            }
            if (warp < ntask) {
#pragma unroll
                for (int c = 0; c < CPS; ++c) part[warp * DS + lane * CPS + c] = acc[c];
            }
            __syncthreads();
            if (warp < cnt && hv.sl[warp] >= 0) {
                const int i = warp;
                float b0[CPS], out[CPS];
                const float f = hv.f[i];
#pragma unroll
                for (int c = 0; c < CPS; ++c) {
                    b0[c] = b0s[i * DS + lane * CPS + c];
                    out[c] = b0[c] * f;
                }
                if (snap) {
                    const size_t so =
                        ((size_t)(ti * d.P + p) * CW + (hv.o0[i] + hv.nm[i] - 1)) * D +
                        (size_t)cs * DS + lane * CPS;
                    if (d.snapq == 2)
                        store_fp8<CPS>(static_cast<unsigned char *>(in.snap) + so, b0);
                    else if (d.snapq)
                        store_vec<__nv_bfloat16, CPS>(static_cast<__nv_bfloat16 *>(in.snap) + so, b0);
                    else
                        store_vec<BT, CPS>(static_cast<BT *>(in.snap) + so, b0);
                }
                for (int j = hv.toff[i]; j < hv.toff[i + 1]; ++j)
#pragma unroll
                    for (int c = 0; c < CPS; ++c) out[c] += part[j * DS + lane * CPS + c];
                store_vec<BT, CPS>(bank + (size_t)hv.sl[i] * D, out);
            }
            __syncthreads();
            h0 += cnt;
        }
    }

    for (int b = 0; b < mine; b += 32) {
        if (b > 0) {
            cslot = nslot; co0 = no0; co1 = no1; ct1 = nt1; cf = nf; cw1 = nw1;
            meta(b + 32, nslot, no0, no1, nt1, nf, nw1);
        }
        const int cnt = mine - b < 32 ? mine - b : 32;
        for (int k = 0; k < cnt; k += U) {
            Raw<BT, CPS> r[U];
            int sl[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                sl[u] = __shfl_sync(0xffffffffu, cslot, (k + u) & 31);
                if (k + u < cnt && sl[u] >= 0) raw_load(bank + (size_t)sl[u] * D, r[u]);
                else sl[u] = -1;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int o0 = __shfl_sync(0xffffffffu, co0, (k + u) & 31);
                const int o1 = __shfl_sync(0xffffffffu, co1, (k + u) & 31);
                const int t1 = __shfl_sync(0xffffffffu, ct1, (k + u) & 31);
                const float f = __shfl_sync(0xffffffffu, cf, (k + u) & 31);
                const float w1 = __shfl_sync(0xffffffffu, cw1, (k + u) & 31);
                if (sl[u] < 0) continue;                       // warp-uniform
                float acc[CPS], x[CPS];
                raw_widen(r[u], acc);
                if (snap) {
                    const size_t so = ((size_t)(ti * d.P + p) * CW + (o1 - 1)) * D +
                                      (size_t)cs * DS + lane * CPS;
                    if (d.snapq == 2)        // float8_e4m3fn snapshot
                        store_fp8<CPS>(static_cast<unsigned char *>(in.snap) + so, acc);
                    else if (d.snapq)        // float32 bank, bfloat16 snapshot
                        store_vec<__nv_bfloat16, CPS>(static_cast<__nv_bfloat16 *>(in.snap) + so, acc);
                    else
                        store_vec<BT, CPS>(static_cast<BT *>(in.snap) + so, acc);
                }
                load_vec<float, CPS, false>(dvl + t1 * DS, x);
#pragma unroll
                for (int c = 0; c < CPS; ++c) acc[c] = fmaf(w1, x[c], acc[c] * f);
                // further members in sorted order, records 32 at a time (the next 32 loaded one
                // batch ahead), 4 delta_v rows read at once
                int ct = 0;
                float cwv = 0.f;
                if (o0 + 1 + lane < o1) {
                    ct = div_by(perm[o0 + 1 + lane], magic);
                    cwv = wdw[o0 + 1 + lane];
                }
                for (int m = o0 + 1; m < o1; m += 32) {
                    int nt = 0;
                    float nwv = 0.f;
                    if (m + 32 + lane < o1) {
                        nt = div_by(perm[m + 32 + lane], magic);
                        nwv = wdw[m + 32 + lane];
                    }
                    const int mc = o1 - m < 32 ? o1 - m : 32;
                    for (int v0 = 0; v0 < mc; v0 += 4) {
                        float y[4][CPS], wv[4];
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int tv = __shfl_sync(0xffffffffu, ct, (v0 + v) & 31);
                            wv[v] = __shfl_sync(0xffffffffu, cwv, (v0 + v) & 31);
                            load_vec<float, CPS, false>(dvl + (v0 + v < mc ? tv : 0) * DS, y[v]);
                        }
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (v0 + v >= mc) break;
                            axpy(acc, wv[v], y[v]);
                        }
                    }
                    ct = nt;
                    cwv = nwv;
                }
                store_vec<BT, CPS>(bank + (size_t)sl[u] * D, acc);
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// debug: the plan's per-position flags and token-major DW weights of a slab's chunks
// ---------------------------------------------------------------------------------------
__global__ void k_debug_expand(Dims d, Work w, int32_t *perm_out, uint8_t *gs_out,
                               uint8_t *ow_out, float *dw_out) {
    const int n = blockIdx.x;
    const int CW = d.C * d.W;
    const int nw = w.nvalid[n] * d.W;
    const int ng = w.ngroups[n];
    const int32_t *perm = w.perm + (size_t)n * CW;
    const int32_t *goff = w.goff + (size_t)n * goff_stride(CW);
    const float *wdw = w.wdw + (size_t)n * CW;
    perm_out += (size_t)n * CW;
    gs_out += (size_t)n * CW;
    ow_out += (size_t)n * CW;
    dw_out += (size_t)n * CW;
    for (int i = threadIdx.x; i < CW; i += blockDim.x) {
        perm_out[i] = i < nw ? perm[i] : -1;
        gs_out[i] = 0;
        ow_out[i] = 0;
        dw_out[i] = 0.f;
    }
    __syncthreads();
    for (int g = threadIdx.x; g < ng; g += blockDim.x) {
        gs_out[goff[g]] = 1;
        ow_out[goff[g + 1] - 1] = 1;
    }
    for (int i = threadIdx.x; i < nw; i += blockDim.x) dw_out[perm[i]] = wdw[i];
}

// ---------------------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------------------
int gather_wpt(const Dims &d) {
    // warps per token: enough warps for the whole GPU, more of them for rows of 512 bytes or
    // more (32 warps per SM suit 256-byte rows, 64 the 512-byte ones)
    const long tokens = (long)d.P * d.C;
    const int row_bytes = d.D * (d.dtype == SDM_BF16 ? 2 : 4);
    const long target = (row_bytes >= 512 ? 64L : 32L) * kRefSms;
    int wpt = 1;
    while (wpt < 8 && tokens * wpt < target && 2 * wpt <= (d.W < d.R ? d.W : d.R)) wpt *= 2;
    return wpt;
}

template <typename BT, int CPL>
cudaError_t gather_cpl(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                       cudaStream_t st) {
    const int wpt = gather_wpt(d);
    const int tokens = d.P * d.C;
    const int tpb = kWarps / wpt;
    const int grid = (tokens + tpb - 1) / tpb;
    switch (wpt) {
        case 1: k_gather<BT, CPL, 1><<<grid, kBlock, 0, st>>>(d, in, w, step0, ti); break;
        case 2: k_gather<BT, CPL, 2><<<grid, kBlock, 0, st>>>(d, in, w, step0, ti); break;
        case 4: k_gather<BT, CPL, 4><<<grid, kBlock, 0, st>>>(d, in, w, step0, ti); break;
        default: k_gather<BT, CPL, 8><<<grid, kBlock, 0, st>>>(d, in, w, step0, ti); break;
    }
    return cudaGetLastError();
}

template <typename BT, int CPS>
cudaError_t dw_cps_launch(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                          cudaStream_t st) {
    // one 32-warp CTA per SM, the SMs shared out over the (chunk, slice) pairs in whole waves
    const size_t smem = dw_smem_bytes(d.C, 32 * CPS);
    const int pairs = d.P * (d.D / (32 * CPS));
    int cpp = kRefSms / pairs;
    const int need = (d.C * d.W + DW_W - 1) / DW_W;
    if (cpp > need) cpp = need;
    if (cpp < 1) cpp = 1;
    auto kern = k_dw<BT, CPS>;
    set_kernel_smem(kern, smem);
    kern<<<pairs * cpp, DW_T, smem, st>>>(d, in, w, step0, ti, cpp);
    return cudaGetLastError();
}

template <typename BT, int CPL>
cudaError_t dw_cpl(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                   cudaStream_t st) {
    switch (dw_cps(d)) {
        case 1: return dw_cps_launch<BT, 1>(d, in, w, step0, ti, st);
        case 2: return dw_cps_launch<BT, 2>(d, in, w, step0, ti, st);
        case 4: return dw_cps_launch<BT, 4>(d, in, w, step0, ti, st);
        case 8: return dw_cps_launch<BT, 8>(d, in, w, step0, ti, st);
        default: return dw_cps_launch<BT, 16>(d, in, w, step0, ti, st);
    }
}

}  // namespace

#define SDM_DISPATCH_D(FN, BT)                                      \
    switch (d.D) {                                                  \
        case 32: return FN<BT, 1>(d, in, w, step0, ti, st);         \
        case 64: return FN<BT, 2>(d, in, w, step0, ti, st);         \
        case 128: return FN<BT, 4>(d, in, w, step0, ti, st);        \
        case 256: return FN<BT, 8>(d, in, w, step0, ti, st);        \
        case 512: return FN<BT, 16>(d, in, w, step0, ti, st);       \
        default: return cudaErrorInvalidValue;                      \
    }

cudaError_t launch_gather(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                          cudaStream_t st) {
    if (d.dtype == SDM_BF16) { SDM_DISPATCH_D(gather_cpl, __nv_bfloat16) }
    SDM_DISPATCH_D(gather_cpl, float)
}

cudaError_t launch_dw(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                      cudaStream_t st) {
    if (d.dtype == SDM_BF16) { SDM_DISPATCH_D(dw_cpl, __nv_bfloat16) }
    SDM_DISPATCH_D(dw_cpl, float)
}

cudaError_t launch_dualmm(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                          cudaStream_t st) {
    if (dualmm_tc_fits(d)) return launch_dualmm_tc(d, in, w, step0, ti, st);
    const size_t smem =
        sizeof(float) * ((size_t)2 * MM_R * mm_apitch(d.C) + (size_t)mm_kpad(d.C) * MM_UP);
    dim3 grid((d.C + MM_R - 1) / MM_R, (d.D + MM_N - 1) / MM_N, d.P);
    if (d.dtype == SDM_BF16) {
        auto kern = k_dualmm<__nv_bfloat16>;
        set_kernel_smem(kern, smem);
        kern<<<grid, MM_T, smem, st>>>(d, in, w, step0, ti);
    } else {
        auto kern = k_dualmm<float>;
        set_kernel_smem(kern, smem);
        kern<<<grid, MM_T, smem, st>>>(d, in, w, step0, ti);
    }
    return cudaGetLastError();
}

cudaError_t launch_debug_expand(const Dims &d, const Work &w, int nchunks, int32_t *perm,
                                uint8_t *gstart, uint8_t *owner, float *dw_tok,
                                cudaStream_t st) {
    k_debug_expand<<<nchunks, kBlock, 0, st>>>(d, w, perm, gstart, owner, dw_tok);
    return cudaGetLastError();
}

}  // namespace sdm
