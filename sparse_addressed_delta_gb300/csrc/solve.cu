// The per-chunk WY solve (sparse-delta-memory 2.0.0, wy_solve.py module docstring):
//   X = (I + L)^-1 with L = tril(diag(beta) A, -1), and QX = QK X,
// both dense row-major [C, C] float32 with +0 above the diagonal; rows and columns at or past
// the chunk's valid tokens are identity rows of X (zero rows of QX), so a ragged chunk is the
// leading block's inverse.
//
// GB300 design: one CTA per chunk, one thread per column of X. Column c of a unit lower
// triangular inverse depends only on itself (X[i][c] = -beta_i sum_{k=c}^{i-1} A[i][k] X[k][c]),
// so the threads never wait on one another; each keeps its column's nonzero part (rows c..C-1)
// in shared memory, packed as a triangle (C(C+1)/2 floats, 128.5 KB at C = 256). The rows of A
// and QK are read from L2/L1 with consecutive threads on consecutive columns. All arithmetic is
// full float32 FFMA: the inverse amplifies rounding, so no reduced-precision tensor path is used.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

__device__ __forceinline__ int tri_base(int c, int C) { return c * C - (c * (c - 1)) / 2; }

__global__ void __launch_bounds__(kMaxChunk) k_solve(Dims d, Inputs in, Work w, int step0,
                                                    int nsteps) {
    extern __shared__ float xs[];
    const int C = d.C;
    const int n = blockIdx.x;
    const int c = threadIdx.x;
    const int p = n % d.P, ti = step0 + n / d.P;
    const int nv = w.nvalid[n];
    const float *A = w.A + (size_t)n * C * C;
    const float *QK = w.QK + (size_t)n * C * C;
    float *X = w.X + (size_t)n * C * C;
    float *QX = w.QX + (size_t)n * C * C;
    const float *beta = in.beta + (size_t)p * d.T + (size_t)ti * C;
    float *xc = xs + tri_base(c, C);   // xc[i - c] = X[i][c], i >= c

    if (c < nv) {
        xc[0] = 1.f;
        for (int i = c + 1; i < nv; ++i) {
            const float *ai = A + (size_t)i * C;
            float acc = 0.f;
            for (int k = c; k < i; ++k) acc = fmaf(ai[k], xc[k - c], acc);
            xc[i - c] = -beta[i] * acc;
        }
    }
    // write X and QX row by row (consecutive threads on consecutive columns)
    for (int i = 0; i < C; ++i) {
        float x, qx = 0.f;
        if (i < nv && c < nv) {
            x = (c <= i) ? xc[i - c] : 0.f;
            if (c <= i) {
                const float *qi = QK + (size_t)i * C;
                for (int k = c; k <= i; ++k) qx = fmaf(qi[k], xc[k - c], qx);
            }
        } else {
            x = (i == c) ? 1.f : 0.f;
        }
        X[(size_t)i * C + c] = x;
        QX[(size_t)i * C + c] = qx;
    }
}

}  // namespace

cudaError_t launch_solve(const Dims &d, const Inputs &in, const Work &w, int step0, int nsteps,
                         cudaStream_t st) {
    const size_t smem = sizeof(float) * (size_t)d.C * (d.C + 1) / 2;
    cudaFuncSetAttribute(k_solve, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_solve<<<nsteps * d.P, d.C, smem, st>>>(d, in, w, step0, nsteps);
    return cudaGetLastError();
}

}  // namespace sdm
