// The per-chunk WY solve (sparse-delta-memory 2.0.0, wy_solve.py module docstring):
//   X = (I + L)^-1 with L = tril(diag(beta) A, -1), and QX = QK X,
// both dense row-major [C, C] float32 with +0 above the diagonal; rows and columns at or past
// the chunk's valid tokens are identity rows of X (zero rows of QX), so a ragged chunk is the
// leading block's inverse.
//
// GB300 design: one CTA per chunk, one thread per column of X. Column c of a unit lower
// triangular inverse depends only on itself (X[i][c] = -beta_i sum_{k=c}^{i-1} A[i][k] X[k][c]),
// so the threads never wait on one another; each keeps its column's nonzero part (rows c..C-1)
// in shared memory, packed as a triangle (C(C+1)/2 floats, 128.5 KB at C = 256). A and QK are
// staged in shared memory too when they fit (C <= 128), else read from L2 with consecutive
// threads on consecutive columns. Each dot product runs as four interleaved partial sums
// (fixed order) to break the FMA dependency chain. All arithmetic is full float32: the
// inverse amplifies rounding, so no reduced-precision tensor path is used.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

__device__ __forceinline__ int tri_base(int c, int C) { return c * C - (c * (c - 1)) / 2; }

// sum_{k=k0}^{k1-1} a[k] * xc[k - k0], four partial sums in a fixed order
__device__ __forceinline__ float dot4(const float *a, const float *x, int n) {
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    int k = 0;
    for (; k + 4 <= n; k += 4) {
        s0 = fmaf(a[k], x[k], s0);
        s1 = fmaf(a[k + 1], x[k + 1], s1);
        s2 = fmaf(a[k + 2], x[k + 2], s2);
        s3 = fmaf(a[k + 3], x[k + 3], s3);
    }
    for (; k < n; ++k) s0 = fmaf(a[k], x[k], s0);
    return (s0 + s1) + (s2 + s3);
}

template <bool STAGE>
__global__ void __launch_bounds__(kMaxChunk) k_solve(Dims d, Inputs in, Work w, int step0,
                                                    int nsteps) {
    extern __shared__ float sm[];
    const int C = d.C;
    const int n = blockIdx.x;
    const int c = threadIdx.x;
    const int p = n % d.P, ti = step0 + n / d.P;
    const int nv = w.nvalid[n];
    const float *Ag = w.A + (size_t)n * C * C;
    const float *QKg = w.QK + (size_t)n * C * C;
    float *X = w.X + (size_t)n * C * C;
    float *QX = w.QX + (size_t)n * C * C;
    const float *beta = in.beta + (size_t)p * d.T + (size_t)ti * C;
    float *xs = sm;                                    // packed triangle
    const int tri = C * (C + 1) / 2;
    const float *A = Ag, *QK = QKg;
    if (STAGE) {
        float *as = sm + ((tri + 3) & ~3);
        float *qs = as + C * C;
        for (int i = c; i < C * C; i += blockDim.x) { as[i] = Ag[i]; qs[i] = QKg[i]; }
        __syncthreads();
        A = as;
        QK = qs;
    }
    float *xc = xs + tri_base(c, C);   // xc[i - c] = X[i][c], i >= c

    if (c < nv) {
        xc[0] = 1.f;
        for (int i = c + 1; i < nv; ++i)
            xc[i - c] = -beta[i] * dot4(A + (size_t)i * C + c, xc, i - c);
    }
    // write X and QX row by row (consecutive threads on consecutive columns)
    for (int i = 0; i < C; ++i) {
        float x, qx = 0.f;
        if (i < nv && c < nv) {
            x = (c <= i) ? xc[i - c] : 0.f;
            if (c <= i) qx = dot4(QK + (size_t)i * C + c, xc, i - c + 1);
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
    const size_t tri = (size_t)d.C * (d.C + 1) / 2;
    const size_t staged = sizeof(float) * (((tri + 3) & ~size_t(3)) + 2 * (size_t)d.C * d.C);
    if (staged <= 200 * 1024) {
        if (staged > 48 * 1024)
            cudaFuncSetAttribute(k_solve<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)staged);
        k_solve<true><<<nsteps * d.P, d.C, staged, st>>>(d, in, w, step0, nsteps);
    } else {
        const size_t smem = sizeof(float) * tri;
        cudaFuncSetAttribute(k_solve<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        k_solve<false><<<nsteps * d.P, d.C, smem, st>>>(d, in, w, step0, nsteps);
    }
    return cudaGetLastError();
}

}  // namespace sdm
