// Exact top-k over product-key slots (sparse-delta-memory 2.0.0, product_key_topk.py: the
// product_key_topk docstring's selection rule), forward and backward; one CTA per row.
//
// A row holds F factors side by side (widths w_0..w_{F-1}); slot (c_0..c_{F-1}) scores the float32
// sum of its factor values in factor order (with bfloat16 input and F > 2 each partial sum is
// rounded to bfloat16 before the next factor is added) and has index
// lin = (..(c_0 w_1 + c_1) w_2 ..) w_{F-1} + c_{F-1}. Scores compare as float32 numbers, -0 below
// +0 and NaN as -inf.
//   1. each factor is ranked by a bitonic sort, in shared memory, of 64-bit keys: an order-
//      preserving image of the value above the column, descending (larger column first on
//      ties); only the first min(k, w_f) ranks are used;
//   2. stage 0 keeps the first n = min(k, w_0) ranks of factor 0; stage f keeps, of the pairs
//      (i, j) with i < n, j < m = min(k, w_f) and (i + 1)(j + 1) <= c = min(k, n m), the best c by
//      (score, i + j, i) descending: the pairs are enumerated from a prefix sum of
//      min(m, c / (i + 1)) over i (at most c (1 + ln c) of them, 1568 for c = 256) and sorted as
//      keys image(score) << 32 | (i + j) << 8 | i; the kept pairs in that order are the next
//      stage's ranks. With bfloat16 input and F > 2, a stage before the last compares the
//      bfloat16-rounded partial sum it passes on; the last compares the float32 sum;
//   3. the kept slots are sorted by lin (keys lin << 8 | rank) and written with
//      val = the score rounded to the input dtype.
// Backward: grad_raw[row][factor f column of slot t] += grad_val[row][t], in output order t,
// one thread per factor (its columns are its own), accumulated in shared memory.
#include <climits>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int PK_T = 256;
constexpr int PK_MAXF = 4;
constexpr int PK_MAXW = 4096;        // factor width
constexpr int PK_MAXK = 256;
constexpr int PK_MAXCAND = 2048;     // candidate pairs of a stage, padded to a power of two

struct PkArgs {
    int F, k, kk, ld;
    int w[PK_MAXF], off[PK_MAXF];
    long long rows;
};

// order-preserving 32-bit image of a float32: NaN as -inf, -0 below +0
__device__ __forceinline__ uint32_t fimage(float x) {
    uint32_t u = __float_as_uint(x);
    if (x != x) u = 0xff800000u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bf16_round_f(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// bitonic sort of n (a power of two) keys in shared memory; descending or ascending
__device__ void bitonic(unsigned long long *a, int n, bool desc) {
    for (int k = 2; k <= n; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int ij = i ^ j;
                if (ij > i) {
                    const unsigned long long x = a[i], y = a[ij];
                    const bool up = ((i & k) == 0) != desc;   // this pair sorts ascending
                    if (up ? x > y : x < y) { a[i] = y; a[ij] = x; }
                }
            }
            __syncthreads();
        }
}

__device__ __forceinline__ int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

template <typename T>
__global__ void __launch_bounds__(PK_T) k_pk_topk(const T *raw, PkArgs a, T *val, long long *lin) {
    __shared__ unsigned long long key[PK_MAXW];   // factor ranks / candidate pairs / final order
    __shared__ float sc[PK_MAXK], sc2[PK_MAXK], rv[PK_MAXK];
    __shared__ long long sl[PK_MAXK], sl2[PK_MAXK];
    __shared__ int rc[PK_MAXK], start[PK_MAXK + 1];
    const int tid = threadIdx.x;
    const long long row = blockIdx.x;
    const T *r = raw + row * a.ld;

    // ranks of factor f: the first min(k, w_f) columns in rc and their values in rv
    auto rank_factor = [&](int f) {
        const int w = a.w[f], np = pow2_at_least(w);
        for (int i = tid; i < np; i += PK_T)
            key[i] = i < w ? ((unsigned long long)fimage(to_f32(r[a.off[f] + i])) << 32) | (unsigned)i
                           : 0ull;
        __syncthreads();
        bitonic(key, np, true);
        const int m = w < a.k ? w : a.k;
        for (int j = tid; j < m; j += PK_T) {
            rc[j] = (int)(key[j] & 0xffffffffu);
            rv[j] = to_f32(r[a.off[f] + rc[j]]);
        }
        __syncthreads();
        return m;
    };

    int n = rank_factor(0);
    for (int i = tid; i < n; i += PK_T) { sc[i] = rv[i]; sl[i] = rc[i]; }
    __syncthreads();
    const bool round_partial = sizeof(T) == 2 && a.F > 2;
    for (int f = 1; f < a.F; ++f) {
        const int m = rank_factor(f);
        const int c = (long long)n * m < a.k ? n * m : a.k;
        // candidate pairs of row i: j < min(m, c / (i + 1)); their offsets by a scan (one warp)
        if (tid < 32) {
            int run = 0;
            for (int i0 = 0; i0 < n; i0 += 32) {
                const int i = i0 + tid;
                int cnt = 0;
                if (i < n) {
                    cnt = c / (i + 1);
                    cnt = cnt < m ? cnt : m;
                }
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += y;
                }
                if (i < n) start[i] = run + incl - cnt;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (tid == 0) start[n] = run;
        }
        __syncthreads();
        const int ncand = start[n], np = pow2_at_least(ncand);
        for (int q = tid; q < np; q += PK_T) {
            unsigned long long kq = 0ull;
            if (q < ncand) {
                int lo = 0, hi = n - 1;            // the row i with start[i] <= q < start[i + 1]
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (start[mid] <= q) lo = mid; else hi = mid - 1;
                }
                const int i = lo, j = q - start[i];
                float s = __fadd_rn(sc[i], rv[j]);
                if (round_partial && f < a.F - 1) s = bf16_round_f(s);
                kq = ((unsigned long long)fimage(s) << 32) | ((unsigned)(i + j) << 8) | (unsigned)i;
            }
            key[q] = kq;
        }
        __syncthreads();
        bitonic(key, np, true);
        for (int t = tid; t < c; t += PK_T) {
            const unsigned low = (unsigned)(key[t] & 0xffffffffu);
            const int i = (int)(low & 255u), j = (int)(low >> 8) - i;
            float s = __fadd_rn(sc[i], rv[j]);
            if (round_partial && f < a.F - 1) s = bf16_round_f(s);
            sc2[t] = s;
            sl2[t] = sl[i] * a.w[f] + rc[j];
        }
        __syncthreads();
        for (int t = tid; t < c; t += PK_T) { sc[t] = sc2[t]; sl[t] = sl2[t]; }
        __syncthreads();
        n = c;
    }
    // the kept slots by lin ascending
    const int np = pow2_at_least(n);
    for (int t = tid; t < np; t += PK_T)
        key[t] = t < n ? ((unsigned long long)sl[t] << 8) | (unsigned)t : ULLONG_MAX;
    __syncthreads();
    bitonic(key, np, false);
    for (int t = tid; t < n; t += PK_T) {
        const int src = (int)(key[t] & 255u);
        val[row * a.kk + t] = from_f32<T>(sc[src]);
        lin[row * a.kk + t] = sl[src];
    }
}

template <typename T>
__global__ void __launch_bounds__(32 * PK_MAXF) k_pk_backward(const long long *lin, const T *gval,
                                                             PkArgs a, float *graw) {
    extern __shared__ float acc[];     // [ld]
    const long long row = blockIdx.x;
    for (int i = threadIdx.x; i < a.ld; i += blockDim.x) acc[i] = 0.f;
    __syncthreads();
    const int f = threadIdx.x >> 5;
    if (f < a.F && (threadIdx.x & 31) == 0) {
        long long div = 1;
        for (int g = a.F - 1; g > f; --g) div *= a.w[g];
        for (int t = 0; t < a.kk; ++t) {
            const int col = (int)((lin[row * a.kk + t] / div) % a.w[f]);
            acc[a.off[f] + col] += to_f32(gval[row * a.kk + t]);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.ld; i += blockDim.x) graw[row * a.ld + i] = acc[i];
}

int pk_args(long long rows, const int *factors, int F, int k, PkArgs &a) {
    if (rows < 0 || rows > INT_MAX)
        return set_error(SDM_ERR_INVALID, "rows must be in 0..%d", INT_MAX);
    if (!factors || F < 1 || F > PK_MAXF)
        return set_error(SDM_ERR_INVALID, "F must be 1..%d with a factors array", PK_MAXF);
    if (k < 1 || k > PK_MAXK) return set_error(SDM_ERR_INVALID, "k must be 1..%d", PK_MAXK);
    a.F = F;
    a.k = k;
    a.rows = rows;
    a.ld = 0;
    long long prod = 1;
    for (int f = 0; f < F; ++f) {
        if (factors[f] < 1 || factors[f] > PK_MAXW)
            return set_error(SDM_ERR_UNSUPPORTED, "factor widths must be 1..%d, got %d", PK_MAXW,
                             factors[f]);
        a.w[f] = factors[f];
        a.off[f] = a.ld;
        a.ld += factors[f];
        prod *= factors[f];
    }
    a.kk = prod < k ? (int)prod : k;
    return SDM_OK;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" int sdm_product_key_topk(const void *raw, long long rows, const int *factors, int F,
                                    int k, int dtype, void *val, int64_t *lin, void *stream) {
    PkArgs a;
    int rc = pk_args(rows, factors, F, k, a);
    if (rc) return rc;
    if (dtype != SDM_F32 && dtype != SDM_BF16)
        return set_error(SDM_ERR_INVALID, "dtype must be SDM_F32 or SDM_BF16");
    if (rows > 0 && (!raw || !val || !lin))
        return set_error(SDM_ERR_INVALID, "raw, val and lin must not be NULL");
    if (rows == 0) return SDM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == SDM_BF16)
        k_pk_topk<__nv_bfloat16><<<(unsigned)rows, PK_T, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(raw), a, static_cast<__nv_bfloat16 *>(val),
            reinterpret_cast<long long *>(lin));
    else
        k_pk_topk<float><<<(unsigned)rows, PK_T, 0, st>>>(static_cast<const float *>(raw), a,
                                                          static_cast<float *>(val),
                                                          reinterpret_cast<long long *>(lin));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SDM_OK
                            : set_error(SDM_ERR_CUDA, "product-key top-k: %s", cudaGetErrorString(e));
}

extern "C" int sdm_product_key_topk_backward(const int64_t *lin, const void *grad_val,
                                             long long rows, const int *factors, int F, int k,
                                             int dtype, float *grad_raw, void *stream) {
    PkArgs a;
    int rc = pk_args(rows, factors, F, k, a);
    if (rc) return rc;
    if (dtype != SDM_F32 && dtype != SDM_BF16)
        return set_error(SDM_ERR_INVALID, "dtype must be SDM_F32 or SDM_BF16");
    if (rows > 0 && (!lin || !grad_val || !grad_raw))
        return set_error(SDM_ERR_INVALID, "lin, grad_val and grad_raw must not be NULL");
    if (rows == 0) return SDM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t smem = sizeof(float) * (size_t)a.ld;
    if (dtype == SDM_BF16) {
        auto kern = k_pk_backward<__nv_bfloat16>;
        set_kernel_smem(kern, smem);
        kern<<<(unsigned)rows, 32 * PK_MAXF, smem, st>>>(
            reinterpret_cast<const long long *>(lin), static_cast<const __nv_bfloat16 *>(grad_val),
            a, grad_raw);
    } else {
        auto kern = k_pk_backward<float>;
        set_kernel_smem(kern, smem);
        kern<<<(unsigned)rows, 32 * PK_MAXF, smem, st>>>(reinterpret_cast<const long long *>(lin),
                                                        static_cast<const float *>(grad_val), a,
                                                        grad_raw);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SDM_OK
                            : set_error(SDM_ERR_CUDA, "product-key backward: %s", cudaGetErrorString(e));
}
