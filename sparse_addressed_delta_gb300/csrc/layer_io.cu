// Layer I/O around the write/read (sparse-delta-memory 2.0.0, memory_ops.py "Layer I/O: head
// split / merge and the per-batch bank expand"):
//   head split   [B, T, H*CD] -> [B*H, T, CD]:  dst row (b*H + h)*T + t <- src row (b*T + t)*H + h
//   head merge   the inverse row permutation
//   bank expand  [S, D] -> [B, S, D]: every batch copy is the parameter bank
//   bank sum     [B, S, D] -> [S, D]: sum over the batch in float32, batch order, one rounding
// (the expand's adjoint, the gradient of the shared parameter bank).
// The permutations and the expand move whole rows: the results are bitwise copies. Rows are
// moved in 16-byte pieces when their length and the pointers allow it, else element by element.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kIoThreads = 256;

// dst row r <- src row of r, for the split (SPLIT) or the merge, for rows that do not split
// into whole 16-byte pieces: one warp per row, 2- or 4-byte elements (ne per row, es bytes)
template <bool SPLIT>
__global__ void __launch_bounds__(kIoThreads) k_head_perm(const unsigned char *src,
                                                          unsigned char *dst, long long rows,
                                                          int H, int T, int ne, int es) {
    const long long warps = (long long)gridDim.x * (kIoThreads / 32);
    const int lane = threadIdx.x & 31;
    for (long long r = (long long)blockIdx.x * (kIoThreads / 32) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        long long srow;
        if (SPLIT) {                       // r = (b*H + h)*T + t
            const long long t = r % T, bh = r / T, h = bh % H, b = bh / H;
            srow = (b * T + t) * H + h;
        } else {                           // r = (b*T + t)*H + h
            const long long h = r % H, bt = r / H, t = bt % T, b = bt / T;
            srow = (b * H + h) * T + t;
        }
        if (es == 2) {
            const unsigned short *s = reinterpret_cast<const unsigned short *>(src) + srow * ne;
            unsigned short *d = reinterpret_cast<unsigned short *>(dst) + r * ne;
            for (int i = lane; i < ne; i += 32) d[i] = s[i];
        } else {
            const unsigned *s = reinterpret_cast<const unsigned *>(src) + srow * ne;
            unsigned *d = reinterpret_cast<unsigned *>(dst) + r * ne;
            for (int i = lane; i < ne; i += 32) d[i] = s[i];
        }
    }
}

// the 16-byte path: one thread per 16-byte piece k of the destination (row k / n16, piece
// k % n16), so that short rows still keep every lane of a warp busy
template <bool SPLIT>
__global__ void __launch_bounds__(kIoThreads) k_head_perm16(const uint4 *src, uint4 *dst,
                                                           long long pieces, int H, int T,
                                                           int n16) {
    const long long stride = (long long)gridDim.x * kIoThreads;
    for (long long k = (long long)blockIdx.x * kIoThreads + threadIdx.x; k < pieces; k += stride) {
        const long long r = k / n16;
        const int i = (int)(k - r * n16);
        long long srow;
        if (SPLIT) {
            const long long t = r % T, bh = r / T, h = bh % H, b = bh / H;
            srow = (b * T + t) * H + h;
        } else {
            const long long h = r % H, bt = r / H, t = bt % T, b = bt / T;
            srow = (b * H + h) * T + t;
        }
        dst[k] = src[srow * n16 + i];
    }
}

// out[b][row] = param[row] for every batch copy b: a thread loads a 16-byte piece (or an
// element) once and stores it B times
template <bool VEC>
__global__ void __launch_bounds__(kIoThreads) k_bank_expand(const unsigned char *param,
                                                            unsigned char *out, int B,
                                                            long long units, int es) {
    const long long stride = (long long)gridDim.x * kIoThreads;
    for (long long u = (long long)blockIdx.x * kIoThreads + threadIdx.x; u < units; u += stride) {
        if (VEC) {
            const uint4 x = reinterpret_cast<const uint4 *>(param)[u];
            for (int b = 0; b < B; ++b) reinterpret_cast<uint4 *>(out)[(long long)b * units + u] = x;
        } else if (es == 2) {
            const unsigned short x = reinterpret_cast<const unsigned short *>(param)[u];
            for (int b = 0; b < B; ++b)
                reinterpret_cast<unsigned short *>(out)[(long long)b * units + u] = x;
        } else {
            const unsigned x = reinterpret_cast<const unsigned *>(param)[u];
            for (int b = 0; b < B; ++b) reinterpret_cast<unsigned *>(out)[(long long)b * units + u] = x;
        }
    }
}

// out[i] = sum over b of x[b][i] in float32 (b = 0, 1, ...), rounded once to T; V elements per
// thread (V * sizeof(T) = 16 bytes when the sizes allow it, else 1)
template <typename T, int V>
__global__ void __launch_bounds__(kIoThreads) k_bank_sum(const T *x, T *out, int B, long long n) {
    const long long stride = (long long)gridDim.x * kIoThreads;
    const long long groups = n / V;
    for (long long g = (long long)blockIdx.x * kIoThreads + threadIdx.x; g < groups; g += stride) {
        float acc[V];
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] = 0.f;
        for (int b = 0; b < B; ++b) {
            float v[V];
            load_vec<T, V, true>(x + (long long)b * n + g * V, v);
#pragma unroll
            for (int c = 0; c < V; ++c) acc[c] += v[c];
        }
        store_vec<T, V>(out + g * V, acc);
    }
}

int grid_for(long long work, int per_block) {
    const long long g = (work + per_block - 1) / per_block;
    const long long cap = 16LL * kRefSms;
    return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int io_status(cudaError_t e) {
    return e == cudaSuccess ? SDM_OK : set_error(SDM_ERR_CUDA, "layer I/O launch: %s",
                                                 cudaGetErrorString(e));
}

int head_perm(bool split, const void *src, void *dst, int B, int T, int H, int CD, int dtype,
              cudaStream_t st) {
    if (!src || !dst) return set_error(SDM_ERR_INVALID, "head split/merge: NULL pointer");
    if (B < 0 || T < 0 || H < 1 || CD < 0)
        return set_error(SDM_ERR_INVALID, "head split/merge: bad sizes B=%d T=%d H=%d CD=%d", B,
                         T, H, CD);
    if (dtype != SDM_F32 && dtype != SDM_BF16)
        return set_error(SDM_ERR_INVALID, "head split/merge: dtype must be SDM_F32 or SDM_BF16");
    const long long rows = (long long)B * H * T;
    if (rows == 0 || CD == 0) return SDM_OK;
    const int es = dtype == SDM_BF16 ? 2 : 4;
    const long long row_bytes = (long long)CD * es;
    const bool vec = row_bytes % 16 == 0 && aligned16(src) && aligned16(dst);
    const int n16 = (int)(row_bytes / 16);
    const int grid = grid_for(rows, kIoThreads / 32);
    auto s = static_cast<const unsigned char *>(src);
    auto d = static_cast<unsigned char *>(dst);
    if (vec) {
        const long long pieces = rows * n16;
        const int g16 = grid_for(pieces, kIoThreads);
        auto s16 = reinterpret_cast<const uint4 *>(s);
        auto d16 = reinterpret_cast<uint4 *>(d);
        if (split) k_head_perm16<true><<<g16, kIoThreads, 0, st>>>(s16, d16, pieces, H, T, n16);
        else k_head_perm16<false><<<g16, kIoThreads, 0, st>>>(s16, d16, pieces, H, T, n16);
    } else if (split) {
        k_head_perm<true><<<grid, kIoThreads, 0, st>>>(s, d, rows, H, T, CD, es);
    } else {
        k_head_perm<false><<<grid, kIoThreads, 0, st>>>(s, d, rows, H, T, CD, es);
    }
    return io_status(cudaGetLastError());
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" {

int sdm_head_split(const void *src, void *dst, int B, int T, int H, int CD, int dtype,
                   void *stream) {
    return head_perm(true, src, dst, B, T, H, CD, dtype, static_cast<cudaStream_t>(stream));
}

int sdm_head_merge(const void *src, void *dst, int B, int T, int H, int CD, int dtype,
                   void *stream) {
    return head_perm(false, src, dst, B, T, H, CD, dtype, static_cast<cudaStream_t>(stream));
}

int sdm_bank_expand(const void *param, void *out, int B, long long S, int D, int dtype,
                    void *stream) {
    if (!param || !out) return set_error(SDM_ERR_INVALID, "bank expand: NULL pointer");
    if (B < 0 || S < 0 || D < 0) return set_error(SDM_ERR_INVALID, "bank expand: bad sizes");
    if (dtype != SDM_F32 && dtype != SDM_BF16)
        return set_error(SDM_ERR_INVALID, "bank expand: dtype must be SDM_F32 or SDM_BF16");
    const int es = dtype == SDM_BF16 ? 2 : 4;
    const long long bytes = S * D * es;
    if (B == 0 || bytes == 0) return SDM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto p = static_cast<const unsigned char *>(param);
    auto o = static_cast<unsigned char *>(out);
    if (bytes % 16 == 0 && aligned16(param) && aligned16(out)) {
        const long long units = bytes / 16;
        k_bank_expand<true><<<grid_for(units, kIoThreads), kIoThreads, 0, st>>>(p, o, B, units, es);
    } else {
        const long long units = S * D;
        k_bank_expand<false><<<grid_for(units, kIoThreads), kIoThreads, 0, st>>>(p, o, B, units, es);
    }
    return io_status(cudaGetLastError());
}

int sdm_bank_sum(const void *x, void *out, int B, long long S, int D, int dtype, void *stream) {
    if (!x || !out) return set_error(SDM_ERR_INVALID, "bank sum: NULL pointer");
    if (B < 1 || S < 0 || D < 0) return set_error(SDM_ERR_INVALID, "bank sum: bad sizes");
    if (dtype != SDM_F32 && dtype != SDM_BF16)
        return set_error(SDM_ERR_INVALID, "bank sum: dtype must be SDM_F32 or SDM_BF16");
    const long long n = S * D;
    if (n == 0) return SDM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool vec = aligned16(x) && aligned16(out);
    if (dtype == SDM_BF16) {
        auto xi = static_cast<const __nv_bfloat16 *>(x);
        auto oo = static_cast<__nv_bfloat16 *>(out);
        if (vec && n % 8 == 0)
            k_bank_sum<__nv_bfloat16, 8><<<grid_for(n / 8, kIoThreads), kIoThreads, 0, st>>>(xi, oo, B, n);
        else
            k_bank_sum<__nv_bfloat16, 1><<<grid_for(n, kIoThreads), kIoThreads, 0, st>>>(xi, oo, B, n);
    } else {
        auto xi = static_cast<const float *>(x);
        auto oo = static_cast<float *>(out);
        if (vec && n % 4 == 0)
            k_bank_sum<float, 4><<<grid_for(n / 4, kIoThreads), kIoThreads, 0, st>>>(xi, oo, B, n);
        else
            k_bank_sum<float, 1><<<grid_for(n, kIoThreads), kIoThreads, 0, st>>>(xi, oo, B, n);
    }
    return io_status(cudaGetLastError());
}

}  // extern "C"
