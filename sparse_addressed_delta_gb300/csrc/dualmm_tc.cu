// The per-step dual matmul on the 5th-generation tensor cores (sparse-delta-memory 2.0.0,
// phase2_kernels.py, _sdm_dual_matmul docstring): for chunk p of step ti,
//   delta_v  = X  u_pre          [C, D]
//   readings = QX u_pre + inter  [C, D], rounded once to the bank dtype
// with u_pre zero past the chunk's valid tokens (rows past them are zero in both outputs).
//
// Used when C is a multiple of 128 (one M = 128 tile per 128 rows of X and QX). CTA (m-tile,
// n-tile, p) computes 128 rows x NT columns of both products: two float32 accumulators in
// tensor memory (2 NT columns), written by tcgen05.mma kind::tf32 (M = 128, N = NT, K = 8),
// issued by one thread, over K = the tokens the rows can see (X and QX are lower triangular)
// that are valid, in K-blocks of 32. The tensor memory accelerator copies each block's three
// tiles (128 rows of X and of QX, NT rows of u_pre transposed; 32 floats = 128 bytes of K per
// row) into shared memory with the 128-byte swizzle, which is the K-major layout the matrix
// descriptors read (8-row groups 1024 bytes apart; a K = 8 step is 32 bytes further along the
// row). NSTAGE blocks are in flight: a block's copies complete on its `full` mbarrier, and
// tcgen05.commit of its products on its `empty` mbarrier releases the stage for the block
// NSTAGE later. bfloat16 banks: one TF32 product (the tensor core reads the top 19 bits of each
// float); float32 banks: the 3xTF32 split (lo * hi + hi * lo + hi * hi, each operand's lo the
// part of it the TF32 read drops, formed in shared memory next to the tile) for float32
// accuracy. The epilogue: warp w reads accumulator lanes 32 w .. 32 w + 31 (one row per
// thread) with tcgen05.ld, adds inter and stores both rows. Every wait is bounded; a wait that
// gives up sets SDM_ERR_TIMEOUT in the device status, and the kernel still waits (with the
// default limit) for the copies and products it issued before freeing tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int TC_T = 128;        // threads: four warps, one per 32 accumulator lanes
constexpr int TC_M = 128;        // rows per CTA (one MMA M)
constexpr int TC_KB = 32;        // K per staged block: one 128-byte swizzle row of floats

// stage s: the X tile [128 x 32], the QX tile [128 x 32] and the u_pre tile [NT x 32] as the
// tensor memory accelerator writes them (128-byte swizzle), and for float32 banks the same
// three tiles again with the lo parts
template <int NT, int PARTS>
struct TcSmem {
    static constexpr int A_BYTES = TC_M * TC_KB * 4;
    static constexpr int B_BYTES = NT * TC_KB * 4;
    static constexpr int PART = 2 * A_BYTES + B_BYTES;
    static constexpr int STAGE = PARTS * PART;
    static constexpr int I_BYTES = TC_M * NT * 4;        // the inter tile [128][NT]
    static constexpr int NS0 = (212 * 1024 - I_BYTES) / STAGE;
    static constexpr int NSTAGE = NS0 > 8 ? 8 : (NS0 < 2 ? 2 : NS0);
    // + the alignment of the tiles to 1024 bytes, the barriers, flags and the tensor memory
    // address
    static constexpr size_t BYTES = (size_t)NSTAGE * STAGE + I_BYTES + 1024 + 16 * NSTAGE + 64;
};

// shared-memory matrix descriptor of a K-major tile with the 128-byte swizzle: start address,
// leading byte offset 16 (unused for this layout), stride byte offset 1024 (the next 8 rows),
// descriptor version 1, layout type 2 (128-byte swizzle)
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load2d(void *dst, const CUtensorMap *map, int x, int y,
                                           unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tc_commit(unsigned long long *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// x - (x with its 13 low mantissa bits cleared): the part of x the TF32 product drops
__device__ __forceinline__ float tf32_rest(float x) {
    return x - __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

template <typename BT, int NT>
__global__ void __launch_bounds__(TC_T, 1)
    k_dualmm_tc(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mq,
                const __grid_constant__ CUtensorMap mu, const __grid_constant__ CUtensorMap mi,
                Dims d, Inputs in, Work w, int step0, int ti) {
    constexpr int PARTS = sizeof(BT) == 4 ? 2 : 1;
    using L = TcSmem<NT, PARTS>;
    constexpr int NS = L::NSTAGE;
    extern __shared__ __align__(1024) unsigned char tsm_raw[];
    unsigned char *tsm = tsm_raw + ((1024u - (smem_u32(tsm_raw) & 1023u)) & 1023u);
    float *itile = reinterpret_cast<float *>(tsm + NS * L::STAGE);     // [128][NT]
    unsigned long long *full =
        reinterpret_cast<unsigned long long *>(tsm + NS * L::STAGE + L::I_BYTES);
    unsigned long long *empty = full + NS;
    unsigned long long *ibar = empty + NS;
    int *flag = reinterpret_cast<int *>(ibar + 1);   // [0] blocks issued, [1] loaded, [2] failed
    uint32_t *tslot = reinterpret_cast<uint32_t *>(flag + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x, nt = blockIdx.y, p = blockIdx.z;
    const int C = d.C, D = d.D, m0 = mt * TC_M, n0 = nt * NT;
    const int n = (ti - step0) * d.P + p;
    const int nv = w.nvalid[n];
    // K: the tokens these rows see (k <= row) that are valid
    const int kend = m0 + TC_M < nv ? m0 + TC_M : nv;
    const int nkb = kend > 0 ? (kend + TC_KB - 1) / TC_KB : 0;
    const int ya = n * C + m0, yb = p * D + n0;      // tile rows in the tensor maps

    const bool irows = m0 < nv;                      // live rows: the inter tile is read
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(ibar, 1);
        flag[0] = flag[1] = flag[2] = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tslot)),
                     "r"(2 * NT));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tslot;
    const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(NT >> 3) << 17) |
                           ((uint32_t)(TC_M >> 4) << 24);

    // the copies of K-block kb into stage kb % NS
    auto load = [&](int kb) {
        const int s = kb % NS;
        unsigned char *st = tsm + s * L::STAGE;
        mbar_arrive_expect_tx(full + s, (unsigned)L::PART);
        tma_load2d(st, &mx, kb * TC_KB, ya, full + s);
        tma_load2d(st + L::A_BYTES, &mq, kb * TC_KB, ya, full + s);
        tma_load2d(st + 2 * L::A_BYTES, &mu, kb * TC_KB, yb, full + s);
    };
    // the products of K-block kb (one thread), released on empty[kb % NS]
    auto mma = [&](int kb) {
        const int s = kb % NS;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t sa = smem_u32(tsm + s * L::STAGE);
#pragma unroll
        for (int ks = 0; ks < TC_KB / 8; ++ks) {
            const uint32_t kofs = ks * 32;               // K = 8 floats along the swizzled row
            const uint64_t ax = tc_desc(sa + kofs), aq = tc_desc(sa + L::A_BYTES + kofs);
            const uint64_t bh = tc_desc(sa + 2 * L::A_BYTES + kofs);
            const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
            if constexpr (PARTS == 2) {
                const uint32_t lb = sa + L::PART;
                const uint64_t axl = tc_desc(lb + kofs), aql = tc_desc(lb + L::A_BYTES + kofs);
                const uint64_t bl = tc_desc(lb + 2 * L::A_BYTES + kofs);
                tc_mma(tmem, axl, bh, idesc, acc);
                tc_mma(tmem, ax, bl, idesc, 1u);
                tc_mma(tmem, ax, bh, idesc, 1u);
                tc_mma(tmem + NT, aql, bh, idesc, acc);
                tc_mma(tmem + NT, aq, bl, idesc, 1u);
                tc_mma(tmem + NT, aq, bh, idesc, 1u);
            } else {
                tc_mma(tmem, ax, bh, idesc, acc);
                tc_mma(tmem + NT, aq, bh, idesc, acc);
            }
        }
        tc_commit(empty + s);
    };
    // the inter tile, for the epilogue
    if (tid == 32 && irows) {
        mbar_arrive_expect_tx(ibar, (unsigned)L::I_BYTES);
        tma_load2d(itile, &mi, n0, p * C + m0, ibar);
    }

    if constexpr (PARTS == 1) {
        // thread 32 copies, thread 0 issues the products as blocks land; a stage is copied
        // again once the products of the block NS earlier have read it
        if (tid == 32) {
            int kb = 0;
            for (; kb < nkb; ++kb) {
                const int s = kb % NS;
                if (kb >= NS && !mbar_wait_bounded(empty + s, (unsigned)((kb / NS) - 1) & 1u, d.spin))
                    break;
                load(kb);
            }
            flag[1] = kb;
            if (kb < nkb) flag[2] = 1;
        } else if (tid == 0) {
            int kb = 0;
            for (; kb < nkb; ++kb) {
                if (!mbar_wait_bounded(full + (kb % NS), (unsigned)(kb / NS) & 1u, d.spin)) break;
                mma(kb);
            }
            flag[0] = kb;
            if (kb < nkb) flag[2] = 1;
        }
    } else {
        // float32 banks: every thread forms the lo parts of a landed block before its products
        int nload = 0;                                   // blocks whose copies thread 0 issued
        if (tid == 0)
            for (; nload < NS && nload < nkb; ++nload) load(nload);
        int kb = 0;
        for (; kb < nkb; ++kb) {
            const int s = kb % NS;
            unsigned char *st = tsm + s * L::STAGE;
            const bool landed = mbar_wait_bounded(full + s, (unsigned)(kb / NS) & 1u, d.spin);
            if (!__syncthreads_and(landed)) break;      // one decision for the whole CTA
            const float *hi = reinterpret_cast<const float *>(st);
            float *lo = reinterpret_cast<float *>(st + L::PART);
            for (int i = tid; i < L::PART / 4; i += TC_T) lo[i] = tf32_rest(hi[i]);
            fence_proxy_async_smem();                    // the lo tiles, before the tensor cores
            __syncthreads();
            if (tid == 0) mma(kb);
            // stage s takes block kb + NS once the products of block kb have read it
            if (kb + NS < nkb) {
                bool freed = true;
                if (tid == 0) {
                    freed = mbar_wait_bounded(empty + s, (unsigned)(kb / NS) & 1u, d.spin);
                    if (freed) {
                        load(kb + NS);
                        nload = kb + NS + 1;
                    }
                }
                if (!__syncthreads_and(freed)) {
                    ++kb;
                    break;
                }
            }
        }
        if (tid == 0) {
            flag[0] = kb;
            flag[1] = nload;
            if (kb < nkb) flag[2] = 1;
        }
    }
    __syncthreads();
    const int issued = flag[0], loaded = flag[1];
    bool ok = flag[2] == 0;
    // every issued product done (the last commit covers the earlier ones), and after a give-up
    // every issued copy landed, before tensor memory is freed and the CTA leaves; the waits
    // after a give-up keep the default limit
    if (issued > 0) {
        const int last = issued - 1;
        const unsigned par = (unsigned)(last / NS) & 1u;
        bool done = mbar_wait_bounded(empty + (last % NS), par, ok ? d.spin : kSpinLimit);
        if (!done) done = mbar_wait_bounded(empty + (last % NS), par);
        ok = __syncthreads_and(ok && done);
    }
    if (irows) {
        bool got = mbar_wait_bounded(ibar, 0u, ok ? d.spin : kSpinLimit);
        if (!got) got = mbar_wait_bounded(ibar, 0u);
        ok = __syncthreads_and(ok && got);
    }
    if (!ok && tid == 0) {
        for (int kb = issued; kb < loaded; ++kb)
            mbar_wait_bounded(full + (kb % NS), (unsigned)(kb / NS) & 1u);
        atomicCAS(&w.status->code, 0, (int)SDM_ERR_TIMEOUT);
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    if (ok) {
        const int row = m0 + 32 * warp + lane;
        const bool live = row < nv;
        const size_t tok = (size_t)p * d.T + (size_t)ti * C + row;
        const bool out_row = (size_t)ti * C + row < (size_t)d.T;
        float *dvrow = w.dv + ((size_t)p * C + row) * D + n0;
        const float *irow = itile + (32 * warp + lane) * NT;
        BT *orow = static_cast<BT *>(in.readings) + tok * D + n0;
        constexpr int CW_ = NT < 32 ? NT : 32;          // accumulator columns per load
        for (int c0 = 0; c0 < NT; c0 += CW_) {
            uint32_t a[32], b[32];
            if (nkb > 0) {
                const uint32_t lanebase = (uint32_t)(32 * warp) << 16;
                if constexpr (CW_ == 32) {
                    tc_ld32(tmem + lanebase + c0, a);
                    tc_ld32(tmem + lanebase + NT + c0, b);
                } else {
                    tc_ld16(tmem + lanebase + c0, a);
                    tc_ld16(tmem + lanebase + NT + c0, b);
                }
            }
#pragma unroll
            for (int j = 0; j < CW_; j += 4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f), r = v;
                if (live) {
                    v = make_float4(__uint_as_float(a[j]), __uint_as_float(a[j + 1]),
                                    __uint_as_float(a[j + 2]), __uint_as_float(a[j + 3]));
                    const float4 it = *reinterpret_cast<const float4 *>(irow + c0 + j);
                    r = make_float4(__uint_as_float(b[j]) + it.x, __uint_as_float(b[j + 1]) + it.y,
                                    __uint_as_float(b[j + 2]) + it.z, __uint_as_float(b[j + 3]) + it.w);
                }
                *reinterpret_cast<float4 *>(dvrow + c0 + j) = v;
                if (out_row) {
                    const float rr[4] = {r.x, r.y, r.z, r.w};
                    store_vec<BT, 4>(orow + c0 + j, rr);
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * NT));
}

// The three tensor maps of a workspace and column tile (X and QX: [N C rows][xp] floats, box 32
// x 128; u_pre transposed: [P D rows][C] floats, box 32 x NT; 128-byte swizzle), encoded once
// per workspace address and shape (the calling thread's last ones are kept).
struct TcMaps {
    CUtensorMap x, q, u, i;
};

cudaError_t tc_maps(const Dims &d, const Work &w, int NT, const TcMaps *&out) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn,
                                                               12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    thread_local struct {
        const void *x, *q, *u, *i;
        int C, D, P, ns, xp, NT;
        TcMaps m;
    } cache = {};
    if (!(cache.x == w.X && cache.q == w.QX && cache.u == w.ret && cache.i == w.inter &&
          cache.C == d.C &&
          cache.D == d.D && cache.P == d.P && cache.ns == w.ns && cache.xp == d.xp &&
          cache.NT == NT)) {
        const cuuint64_t rows = (cuuint64_t)w.ns * d.P * d.C;
        const cuuint64_t dx[2] = {(cuuint64_t)d.xp, rows}, sx[1] = {(cuuint64_t)d.xp * 4};
        const cuuint64_t du[2] = {(cuuint64_t)d.C, (cuuint64_t)d.P * d.D},
                         su[1] = {(cuuint64_t)d.C * 4};
        const cuuint64_t di[2] = {(cuuint64_t)d.D, (cuuint64_t)d.P * d.C},
                         si[1] = {(cuuint64_t)d.D * 4};
        const cuuint32_t bx[2] = {TC_KB, TC_M}, bu[2] = {TC_KB, (cuuint32_t)NT},
                         bi[2] = {(cuuint32_t)NT, TC_M}, es[2] = {1, 1};
        auto enc = [&](CUtensorMap *m, void *base, const cuuint64_t *dim, const cuuint64_t *str,
                       const cuuint32_t *box, CUtensorMapSwizzle sw) {
            return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dim, str, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        };
        const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
        if (enc(&cache.m.x, w.X, dx, sx, bx, sw) != CUDA_SUCCESS ||
            enc(&cache.m.q, w.QX, dx, sx, bx, sw) != CUDA_SUCCESS ||
            enc(&cache.m.u, w.ret, du, su, bu, sw) != CUDA_SUCCESS ||
            enc(&cache.m.i, w.inter, di, si, bi, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS) {
            cache.x = nullptr;
            return cudaErrorInvalidValue;
        }
        cache.x = w.X; cache.q = w.QX; cache.u = w.ret; cache.i = w.inter;
        cache.C = d.C; cache.D = d.D; cache.P = d.P; cache.ns = w.ns; cache.xp = d.xp;
        cache.NT = NT;
    }
    out = &cache.m;
    return cudaSuccess;
}

template <typename BT, int NT>
cudaError_t launch_tc(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                      cudaStream_t st) {
    const TcMaps *m = nullptr;
    const cudaError_t e = tc_maps(d, w, NT, m);
    if (e != cudaSuccess) return e;
    constexpr size_t smem = TcSmem<NT, sizeof(BT) == 4 ? 2 : 1>::BYTES;
    auto kern = k_dualmm_tc<BT, NT>;
    set_kernel_smem(kern, smem);
    kern<<<dim3(d.C / TC_M, d.D / NT, d.P), TC_T, smem, st>>>(m->x, m->q, m->u, m->i, d, in, w,
                                                               step0, ti);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dualmm_tc(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                             cudaStream_t st) {
    // the widest column tile (64, 32 or 16) that still gives about one CTA per SM: the step's
    // products are small, and each CTA's time is its copies of X and QX tiles
    const long tiles = (long)d.P * (d.C / TC_M) * (d.D / 64);
    const int nt = tiles >= kRefSms ? 64 : (2 * tiles >= kRefSms ? 32 : 16);
    if (d.dtype == SDM_BF16) {
        if (nt == 64) return launch_tc<__nv_bfloat16, 64>(d, in, w, step0, ti, st);
        if (nt == 32) return launch_tc<__nv_bfloat16, 32>(d, in, w, step0, ti, st);
        return launch_tc<__nv_bfloat16, 16>(d, in, w, step0, ti, st);
    }
    if (nt == 64) return launch_tc<float, 64>(d, in, w, step0, ti, st);
    if (nt == 32) return launch_tc<float, 32>(d, in, w, step0, ti, st);
    return launch_tc<float, 16>(d, in, w, step0, ti, st);
}

}  // namespace sdm
