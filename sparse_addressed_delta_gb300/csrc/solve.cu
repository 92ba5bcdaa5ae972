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
// current block row of L (or QK) and the T blocks are staged next to it. Every product is full
// float32 FFMA in a fixed order: the inverse amplifies rounding, so no reduced-precision path.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int NTS = 256;
constexpr int BS = 16;                 // block size
constexpr int BB = BS * BS;            // floats per block

__host__ __device__ __forceinline__ int tri(int i) { return i * (i + 1) / 2; }

__global__ void __launch_bounds__(NTS) k_solve(Dims d, Inputs in, Work w, int step0, int nsteps) {
    extern __shared__ __align__(16) float ssm[];
    const int C = d.C;
    const int nb = (C + BS - 1) / BS;
    const int n = blockIdx.x;
    const int tid = threadIdx.x;
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
    float *Lr = Xp + tri(nb) * BB;               // current block row of L / QK  [nb][16][16]
    float *Tb = Lr + nb * BB;                    // T blocks                     [nb][16][16]

    // Links for the pipelined Phase 2 (every chunk after the first of the slab): an entry
    // whose slot the stream's previous step writes is pointed at that group's new piece
    // (-1 - g) instead of the bank row. The previous chunk's groups are sorted by slot.
    if (!d.per_step && !d.bwd && n >= d.P) {
        const int CW = C * d.W, CR = C * d.R, np = n - d.P;
        const int ngp = w.ngroups[np];
        const int32_t *gsp = w.gslot + (size_t)np * CW;
        int32_t *wsl = w.wsl + (size_t)n * CW;
        int32_t *rsl = w.rsl + (size_t)n * CR;
        for (int i = tid; i < CW + CR; i += NTS) {
            int32_t *ent = i < CW ? wsl + i : rsl + (i - CW);
            const int v = *ent;
            if (v < 0) continue;
            int lo = 0, hi = ngp;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (gsp[mid] < v) lo = mid + 1; else hi = mid;
            }
            if (lo < ngp && gsp[lo] == v) *ent = -1 - lo;
        }
    }

    // L (or QK) element (R, K) of the chunk, zero outside the valid tokens
    auto lval = [&](int R, int K) {
        return (R < nv && K < R) ? beta[R] * A[(size_t)R * C + K] : 0.f;
    };

    // 1. diagonal inverses: thread (block b, column c) substitutes down its column
    for (int job = tid; job < nvb * BS; job += NTS) {
        const int b = job / BS, c = job - b * BS;
        float *Dk = Xp + (tri(b) + b) * BB;
        float x[BS];
#pragma unroll
        for (int r = 0; r < BS; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < BS; ++r) {
            const int R = b * BS + r;
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < BS; ++k)
                if (k < r) s = fmaf(lval(R, b * BS + k), x[k], s);
            if (r > c) x[r] = -s;
        }
#pragma unroll
        for (int r = 0; r < BS; ++r) Dk[r * BS + c] = x[r];
    }
    __syncthreads();

    // 2. block rows
    for (int i = 1; i < nvb; ++i) {
        for (int e = tid; e < i * BB; e += NTS) {
            const int k = e / BB, rc = e - k * BB, r = rc / BS, c = rc - r * BS;
            Lr[e] = lval(i * BS + r, k * BS + c);
        }
        __syncthreads();
        for (int e = tid; e < i * BB; e += NTS) {
            const int j = e / BB, rc = e - j * BB, r = rc / BS, c = rc - r * BS;
            float s = 0.f;
            for (int k = j; k < i; ++k) {
                const float *Lk = Lr + k * BB + r * BS;
                const float *Xk = Xp + (tri(k) + j) * BB + c;
#pragma unroll
                for (int m = 0; m < BS; ++m) s = fmaf(Lk[m], Xk[m * BS], s);
            }
            Tb[e] = s;
        }
        __syncthreads();
        const float *Di = Xp + (tri(i) + i) * BB;
        for (int e = tid; e < i * BB; e += NTS) {
            const int j = e / BB, rc = e - j * BB, r = rc / BS, c = rc - r * BS;
            const float *T = Tb + j * BB + c;
            float s = 0.f;
            for (int m = 0; m <= r; ++m) s = fmaf(Di[r * BS + m], T[m * BS], s);
            Xp[(tri(i) + j) * BB + rc] = -s;
        }
        __syncthreads();
    }

    // 3. QX, block row by block row; written out with X
    for (int i = 0; i < nb; ++i) {
        if (i < nvb) {
            for (int e = tid; e < (i + 1) * BB; e += NTS) {
                const int k = e / BB, rc = e - k * BB, r = rc / BS, c = rc - r * BS;
                const int R = i * BS + r, K = k * BS + c;
                Lr[e] = (R < nv && K <= R) ? QK[(size_t)R * C + K] : 0.f;
            }
            __syncthreads();
            for (int e = tid; e < (i + 1) * BB; e += NTS) {
                const int j = e / BB, rc = e - j * BB, r = rc / BS, c = rc - r * BS;
                float s = 0.f;
                for (int k = j; k <= i; ++k) {
                    const float *Qk = Lr + k * BB + r * BS;
                    const float *Xk = Xp + (tri(k) + j) * BB + c;
#pragma unroll
                    for (int m = 0; m < BS; ++m) s = fmaf(Qk[m], Xk[m * BS], s);
                }
                Tb[e] = s;
            }
            __syncthreads();
        }
        // rows i*16 .. i*16+15 of X and QX (consecutive threads on consecutive columns)
        for (int e = tid; e < BS * xp; e += NTS) {
            const int r = e / xp, u = e - r * xp, t = i * BS + r;
            if (t >= C) continue;
            if (u >= C) {   // pitch padding
                X[(size_t)t * xp + u] = 0.f;
                QX[(size_t)t * xp + u] = 0.f;
                continue;
            }
            float x, q = 0.f;
            if (t < nv && u < nv) {
                const int j = u / BS;
                x = (u <= t) ? Xp[(tri(i) + j) * BB + r * BS + (u - j * BS)] : 0.f;
                if (j <= i) q = Tb[j * BB + r * BS + (u - j * BS)];
            } else {
                x = (t == u) ? 1.f : 0.f;
            }
            X[(size_t)t * xp + u] = x;
            QX[(size_t)t * xp + u] = q;
        }
        __syncthreads();
    }
}

}  // namespace

size_t solve_smem_bytes(int C) {
    const int nb = (C + BS - 1) / BS;
    return sizeof(float) * (size_t)(tri(nb) + 2 * nb) * BB;
}

cudaError_t launch_solve(const Dims &d, const Inputs &in, const Work &w, int step0, int nsteps,
                         cudaStream_t st) {
    const size_t smem = solve_smem_bytes(d.C);
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(k_solve, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_solve<<<nsteps * d.P, NTS, smem, st>>>(d, in, w, step0, nsteps);
    return cudaGetLastError();
}

}  // namespace sdm
