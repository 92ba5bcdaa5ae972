// The per-chunk WY solve (sparse-delta-memory 2.0.0, wy_solve.py module docstring):
//   X = (I + L)^-1 with L = tril(diag(beta) A, -1), and QX = QK X,
// both row-major [C, C] float32 (row pitch Dims::xp, padding zero) with +0 above the diagonal;
// rows and columns at or past the chunk's valid tokens are identity rows of X (zero rows of
// QX), so a ragged chunk is the leading block's inverse.
//
// The same CTA also links the chunk's entries to the previous step's groups for the pipelined
// Phase 2 (see below).
//
// Blocked forward substitution, one CTA (256 threads) per chunk, 16 x 16 blocks (nb = C/16):
//   1. the diagonal blocks D_i = (I + L_ii)^-1 are inverted at once, one thread per column
//      of a block (forward substitution inside 16 rows);
//   2. block row by block row, i = 1 .. nb-1:  T_ij = sum_{k=j}^{i-1} L_ik X_kj  (j < i, all
//      elements in parallel), then X_ij = -D_i T_ij;
//   3. QX_ij = sum_{k=j}^{i} QK_ik X_kj for every lower block, block row by block row.
// X lives in shared memory as packed lower blocks (nb(nb+1)/2 x 1 KB: 136 KB at C = 256); the
// current block row of L (or QK, when it is not copied on chip whole) and the T blocks are
// staged next to it; for C <= 32 the chunk's A and beta, and for C <= 64 its QK, are first
// copied on chip whole. In steps 2 and 3 a thread computes four adjacent columns of one row
// (one left-hand value and one 16-byte piece of an X row per four FMAs). Every product is full
// float32 FFMA in a fixed order: the inverse amplifies rounding, so no reduced-precision path.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int NTS = 256;
constexpr int BS = 16;                 // block size
constexpr int BB = BS * BS;            // floats per block
constexpr int LRP = BS + 1;            // row pitch of the staged L / QK blocks (no bank conflicts
constexpr int LB = BS * LRP;           // between the rows that one warp reads)

__host__ __device__ __forceinline__ int tri(int i) { return i * (i + 1) / 2; }

// links are written for the pipelined Phase 2 only
__host__ __device__ __forceinline__ bool solve_links(const Dims &d) { return !d.per_step && !d.bwd; }
// A, QK and beta of the chunk are copied on chip first for small chunks (one round of loads
// instead of one per block row); from C = 64 on the copies would cost more in CTAs per SM
// than they save
__host__ __device__ __forceinline__ bool solve_staged(const Dims &d) { return d.C <= 32 && d.C % 4 == 0; }
// QK alone (read only by the last phase, so its copy lands under the earlier ones) up to C = 64
__host__ __device__ __forceinline__ bool solve_staged_qk(const Dims &d) { return d.C <= 64 && d.C % 4 == 0; }
__host__ __device__ __forceinline__ int staged_pitch(int C) { return C + 4; }

// dynamic shared memory: X blocks, L/QK block row, T blocks; then (staged) A, QK [C][C+4] and
// beta [C]; then (links) the previous chunk's group slots [CW] and this chunk's entries
// [CW + CR]
struct SolveSmem {
    size_t a, q, beta, gsl, ent, bytes;
};
__host__ __device__ inline SolveSmem solve_layout(const Dims &d) {
    const int nb = (d.C + BS - 1) / BS;
    SolveSmem L;
    size_t o = sizeof(float) * ((size_t)(tri(nb) + nb) * BB + (size_t)nb * LB);
    L.a = L.q = L.beta = L.gsl = L.ent = o;
    const size_t m = sizeof(float) * (size_t)d.C * staged_pitch(d.C);
    if (solve_staged_qk(d)) {
        L.q = o; o += m;
    }
    if (solve_staged(d)) {
        L.a = o; o += m;
        L.beta = o; o += sizeof(float) * (size_t)d.C;
    }
    if (solve_links(d)) {
        const size_t CW = (size_t)d.C * d.W, CR = (size_t)d.C * d.R;
        L.gsl = o; o += sizeof(int32_t) * CW;
        L.ent = o; o += sizeof(int32_t) * (CW + CR);
    }
    L.bytes = o;
    return L;
}

__global__ void __launch_bounds__(NTS) k_solve(Dims d, Inputs in, Work w, int step0, int nsteps) {
    extern __shared__ __align__(16) float ssm[];
    unsigned char *sraw = reinterpret_cast<unsigned char *>(ssm);
    const SolveSmem SL = solve_layout(d);
    const int C = d.C;
    const int nb = (C + BS - 1) / BS;
    const int n = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int p = n % d.P, ti = step0 + n / d.P;
    const int nv = w.nvalid[n];
    const int nvb = (nv + BS - 1) / BS;          // block rows holding valid tokens
    const float *A = w.A + (size_t)n * C * C;
    const float *QK = w.QK + (size_t)n * C * C;
    const int xp = d.xp;
    float *X = w.X + (size_t)n * C * xp;
    float *QX = w.QX + (size_t)n * C * xp;
    const float *beta = in.beta + (size_t)p * d.T + (size_t)ti * C;
    float *Xp = ssm;                             // packed lower blocks of X
    float *Lr = Xp + tri(nb) * BB;               // current block row of L / QK  [nb][16][LRP]
    float *Tb = Lr + nb * LB;                    // T blocks                     [nb][16][16]

    // staged copies of the valid rows of QK (and for small chunks of A and beta): cp.async,
    // 16 bytes a copy, landing while the links and the first phases run
    const bool staged = solve_staged(d), staged_qk = solve_staged_qk(d);
    int ap = C, qp = C;
    if (staged_qk) {
        float *Qs = reinterpret_cast<float *>(sraw + SL.q);
        qp = staged_pitch(C);
        const int q4 = C / 4;
        for (int i = tid; i < nv * q4; i += NTS) {
            const int r = i / q4, k = (i - r * q4) * 4;
            cp_async16(Qs + r * qp + k, QK + (size_t)r * C + k);
        }
        QK = Qs;
    }
    if (staged) {
        float *As = reinterpret_cast<float *>(sraw + SL.a);
        float *bs = reinterpret_cast<float *>(sraw + SL.beta);
        ap = staged_pitch(C);
        const int q4 = C / 4;
        for (int i = tid; i < nv * q4; i += NTS) {
            const int r = i / q4, k = (i - r * q4) * 4;
            cp_async16(As + r * ap + k, A + (size_t)r * C + k);
        }
        for (int r = tid; r < nv; r += NTS) cp_async4(bs + r, beta + r);
        A = As;
        beta = bs;
    }
    cp_async_commit();

    // Links for the pipelined Phase 2 (every chunk after the first of the slab): an entry
    // whose slot the stream's previous step writes is pointed at that group's new piece
    // (-1 - g) instead of the bank row. The previous chunk's groups are sorted by slot; the
    // search runs in shared memory, four branch-free lower bounds at a time.
    if (solve_links(d) && n >= d.P) {
        const int CW = C * d.W, CR = C * d.R, NE = CW + CR, np = n - d.P;
        const int ngp = w.ngroups[np];
        int32_t *gsp = reinterpret_cast<int32_t *>(sraw + SL.gsl);
        int32_t *ent = reinterpret_cast<int32_t *>(sraw + SL.ent);
        int32_t *wsl = w.wsl + (size_t)n * CW;
        int32_t *rsl = w.rsl + (size_t)n * CR;
        for (int i = tid; i < ngp; i += NTS) gsp[i] = w.gslot[(size_t)np * CW + i];
        for (int i = tid; i < NE; i += NTS) ent[i] = i < CW ? wsl[i] : rsl[i - CW];
        __syncthreads();
        for (int i0 = tid; i0 < NE; i0 += 4 * NTS) {
            int v[4], base[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = i0 + k * NTS;
                v[k] = i < NE ? ent[i] : -1;
                base[k] = 0;
            }
            for (int len = ngp; len > 1;) {
                const int half = len >> 1;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (gsp[base[k] + half - 1] < v[k]) base[k] += half;
                len -= half;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = i0 + k * NTS;
                if (i >= NE || v[k] < 0 || ngp == 0) continue;
                // base is the last position whose predecessors are all < v
                const int lb = base[k] + (gsp[base[k]] < v[k] ? 1 : 0);
                if (lb < ngp && gsp[lb] == v[k]) {
                    if (i < CW) wsl[i] = -1 - lb;
                    else rsl[i - CW] = -1 - lb;
                }
            }
        }
    }
    if (staged) cp_async_wait<0>();
    __syncthreads();
    const bool qk_ready = !staged_qk || staged;   // else the QK copy is awaited before QX

    // L (or QK) element (R, K) of the chunk, zero outside the valid tokens
    auto lval = [&](int R, int K) {
        return (R < nv && K < R) ? beta[R] * A[(size_t)R * ap + K] : 0.f;
    };

    // 1. diagonal inverses: the diagonal blocks of L are staged (coalesced), then thread
    //    (block b, column c) substitutes down its column
    for (int e = tid; e < nvb * BB; e += NTS) {
        const int b = e / BB, rc = e - b * BB, r = rc / BS, c = rc - r * BS;
        Lr[b * LB + r * LRP + c] = lval(b * BS + r, b * BS + c);
    }
    __syncthreads();
    for (int job = tid; job < nvb * BS; job += NTS) {
        const int b = job / BS, c = job - b * BS;
        float *Dk = Xp + (tri(b) + b) * BB;
        const float *Lb = Lr + b * LB;
        float x[BS];
#pragma unroll
        for (int r = 0; r < BS; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < BS; ++r) {
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < BS; ++k)
                if (k < r) s = fmaf(Lb[r * LRP + k], x[k], s);
            if (r > c) x[r] = -s;
        }
#pragma unroll
        for (int r = 0; r < BS; ++r) Dk[r * BS + c] = x[r];
    }
    __syncthreads();

    // A thread computes a quad: four adjacent columns (c .. c+3) of one row r of block j, so one
    // left-hand value and one 16-byte piece of an X row feed four FMAs (k and m ascending, as a
    // plain dot product).
    auto quad = [](int qd, int &j, int &r, int &c) {
        j = qd >> 6;
        r = (qd >> 2) & 15;
        c = (qd & 3) * 4;
    };
    auto fma4 = [](float4 &s, float a, const float4 &x) {
        s.x = fmaf(a, x.x, s.x);
        s.y = fmaf(a, x.y, s.y);
        s.z = fmaf(a, x.z, s.z);
        s.w = fmaf(a, x.w, s.w);
    };

    // 2. block rows
    for (int i = 1; i < nvb; ++i) {
        for (int e = tid; e < i * BB; e += NTS) {
            const int k = e / BB, rc = e - k * BB, r = rc / BS, c = rc - r * BS;
            Lr[k * LB + r * LRP + c] = lval(i * BS + r, k * BS + c);
        }
        __syncthreads();
        for (int qd = tid; qd < i * 64; qd += NTS) {
            int j, r, c;
            quad(qd, j, r, c);
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k = j; k < i; ++k) {
                const float *Lk = Lr + k * LB + r * LRP;
                const float *Xk = Xp + (tri(k) + j) * BB + c;
#pragma unroll
                for (int m = 0; m < BS; ++m)
                    fma4(s, Lk[m], *reinterpret_cast<const float4 *>(Xk + m * BS));
            }
            *reinterpret_cast<float4 *>(Tb + j * BB + r * BS + c) = s;
        }
        __syncthreads();
        const float *Di = Xp + (tri(i) + i) * BB;
        for (int qd = tid; qd < i * 64; qd += NTS) {
            int j, r, c;
            quad(qd, j, r, c);
            const float *T = Tb + j * BB + c;
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int m = 0; m <= r; ++m)
                fma4(s, Di[r * BS + m], *reinterpret_cast<const float4 *>(T + m * BS));
            *reinterpret_cast<float4 *>(Xp + (tri(i) + j) * BB + r * BS + c) =
                make_float4(-s.x, -s.y, -s.z, -s.w);
        }
        __syncthreads();
    }

    // 3. QX, block row by block row; written out with X. QK is read from its staged copy when
    //    there is one, else its block row is staged like L's.
    if (!qk_ready) {
        cp_async_wait<0>();
        __syncthreads();
    }
    const bool vec = (xp & 3) == 0;     // X / QX rows are 16-byte aligned
    for (int i = 0; i < nb; ++i) {
        if (i < nvb) {
            const float *Qrow;
            int qpitch, qblock;
            if (staged_qk) {
                Qrow = QK + (size_t)i * BS * qp;   // valid rows, zero above the diagonal
                qpitch = qp;
                qblock = BS;
            } else {
                for (int e = tid; e < (i + 1) * BB; e += NTS) {
                    const int k = e / BB, rc = e - k * BB, r = rc / BS, c = rc - r * BS;
                    const int R = i * BS + r, K = k * BS + c;
                    Lr[k * LB + r * LRP + c] = (R < nv && K <= R) ? QK[(size_t)R * qp + K] : 0.f;
                }
                __syncthreads();
                Qrow = Lr;
                qpitch = LRP;
                qblock = LB;
            }
            for (int qd = tid; qd < (i + 1) * 64; qd += NTS) {
                int j, r, c;
                quad(qd, j, r, c);
                float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i * BS + r < nv) {
                    for (int k = j; k <= i; ++k) {
                        const float *Qk = Qrow + (size_t)k * qblock + r * qpitch;
                        const float *Xk = Xp + (tri(k) + j) * BB + c;
#pragma unroll
                        for (int m = 0; m < BS; ++m)
                            fma4(s, Qk[m], *reinterpret_cast<const float4 *>(Xk + m * BS));
                    }
                }
                *reinterpret_cast<float4 *>(Tb + j * BB + r * BS + c) = s;
            }
            __syncthreads();
        }
        // rows i*16 .. i*16+15 of X and QX: warp w takes rows w, w + 8; its lanes take
        // consecutive 16-byte pieces (or single columns when the pitch is not a multiple of 4)
        auto xq = [&](int r, int u, float &x, float &q) {
            const int t = i * BS + r;
            q = 0.f;
            if (u >= C) {
                x = 0.f;                       // pitch padding
            } else if (t < nv && u < nv) {
                const int j = u / BS;
                x = (u <= t) ? Xp[(tri(i) + j) * BB + r * BS + (u - j * BS)] : 0.f;
                if (j <= i) q = Tb[j * BB + r * BS + (u - j * BS)];
            } else {
                x = (t == u) ? 1.f : 0.f;
            }
        };
        for (int r = warp; r < BS; r += NTS / 32) {
            const int t = i * BS + r;
            if (t >= C) break;
            float *xrow = X + (size_t)t * xp, *qrow = QX + (size_t)t * xp;
            if (vec) {
                for (int u4 = lane * 4; u4 < xp; u4 += 128) {
                    float4 x, q;
                    xq(r, u4, x.x, q.x);
                    xq(r, u4 + 1, x.y, q.y);
                    xq(r, u4 + 2, x.z, q.z);
                    xq(r, u4 + 3, x.w, q.w);
                    *reinterpret_cast<float4 *>(xrow + u4) = x;
                    *reinterpret_cast<float4 *>(qrow + u4) = q;
                }
            } else {
                for (int u = lane; u < xp; u += 32) {
                    float x, q;
                    xq(r, u, x, q);
                    xrow[u] = x;
                    qrow[u] = q;
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace

size_t solve_smem_bytes(const Dims &d) { return solve_layout(d).bytes; }

cudaError_t launch_solve(const Dims &d, const Inputs &in, const Work &w, int step0, int nsteps,
                         cudaStream_t st) {
    const size_t smem = solve_smem_bytes(d);
    set_kernel_smem(k_solve, smem);
    k_solve<<<nsteps * d.P, NTS, smem, st>>>(d, in, w, step0, nsteps);
    return cudaGetLastError();
}

}  // namespace sdm
