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
// that are valid, in K-blocks of 32 staged in shared memory twice over (the next block is
// loaded while the tensor cores work on the current ones; tcgen05.commit on the block's
// mbarrier releases its buffer). Operands are K-major with no swizzle: the canonical layout of
// 8-row x 16-byte core matrices, element (r, k) of a tile at ((r / 8) KB/4 + k / 4) 32 +
// (r % 8) 4 + k % 4 floats (KB = 32), i.e. core matrices 128 bytes apart along K (the leading
// byte offset) and 1024 bytes apart along the rows (the stride byte offset). X and QX rows are
// copied as they are; u_pre [k][n] is transposed into the B tile (n, k) while staging. bfloat16
// banks: one TF32 product (operands rounded to nearest on the bit pattern); float32 banks: the
// 3xTF32 split (lo * hi + hi * lo + hi * hi, each operand's hi its TF32 rounding and lo the
// rounded rest) for float32 accuracy. The epilogue: warp w reads accumulator lanes 32 w .. 32 w
// + 31 (one row per thread) with tcgen05.ld, adds inter and stores both rows. Every wait is
// bounded; a wait that gives up sets SDM_ERR_TIMEOUT in the device status, and the kernel still
// waits (with the default limit) for the products it issued before freeing tensor memory.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int TC_T = 128;        // threads: four warps, one per 32 accumulator lanes
constexpr int TC_M = 128;        // rows per CTA (one MMA M)
constexpr int TC_KB = 32;        // K per staged block (4 MMAs of K = 8)

__host__ __device__ constexpr int tc_tile_floats(int rows) { return rows * TC_KB; }

// stage s holds the X tile and the QX tile [128 x 32] and the B tile [NT x 32] (raw float32:
// the tensor core reads the TF32 truncation of each value, the "hi" part), and for float32
// banks the same three tiles again with the "lo" parts x - trunc_tf32(x)
template <int NT, int PARTS>
struct TcSmem {
    static constexpr int A = tc_tile_floats(TC_M), B = tc_tile_floats(NT);
    static constexpr int TILES = 2 * A + B;                      // floats of one part
    static constexpr int STAGE = PARTS * TILES;
    // K-blocks in flight: as many as about 220 KB of shared memory holds (one CTA per SM, so
    // that a CTA's loads overlap instead of taking a round trip per block)
    static constexpr int NS0 = (220 * 1024) / (int)(sizeof(float) * STAGE);
    static constexpr int NSTAGE = NS0 > 8 ? 8 : (NS0 < 2 ? 2 : NS0);
    static constexpr size_t BYTES = sizeof(float) * NSTAGE * STAGE + 64;
};

__device__ __forceinline__ int tc_off(int r, int k) {
    return ((r >> 3) * (TC_KB / 4) + (k >> 2)) * 32 + (r & 7) * 4 + (k & 3);
}

__device__ __forceinline__ uint64_t tc_desc(uint32_t addr) {
    // start address, leading byte offset 128 (next core matrix along K), stride byte offset
    // 1024 (next 8 rows), descriptor version 1, no swizzle
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46);
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

// 16 bytes global -> shared, the bytes past `src_bytes` (0..16) zero-filled
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// x - (x with its 13 low mantissa bits cleared): the part of x the TF32 product drops
__device__ __forceinline__ float tf32_rest(float x) {
    return x - __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

template <typename BT, int NT>
__global__ void __launch_bounds__(TC_T, 1) k_dualmm_tc(Dims d, Inputs in, Work w, int step0, int ti) {
    constexpr int PARTS = sizeof(BT) == 4 ? 2 : 1;
    using L = TcSmem<NT, PARTS>;
    constexpr int NS = L::NSTAGE;
    extern __shared__ __align__(1024) float tsm[];
    unsigned long long *bar = reinterpret_cast<unsigned long long *>(tsm + NS * L::STAGE);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + NS);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x, nt = blockIdx.y, p = blockIdx.z;
    const int C = d.C, D = d.D, m0 = mt * TC_M, n0 = nt * NT;
    const int n = (ti - step0) * d.P + p;
    const int nv = w.nvalid[n];
    const float *X = w.X + (size_t)n * C * d.xp;
    const float *QX = w.QX + (size_t)n * C * d.xp;
    const float *UT = w.ret + (size_t)p * D * C;     // u_pre transposed, [D][C]
    // K: the tokens these rows see (k <= row) that are valid
    const int kend = m0 + TC_M < nv ? m0 + TC_M : nv;
    const int nkb = kend > 0 ? (kend + TC_KB - 1) / TC_KB : 0;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bar + s, 1);
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

    // the copies of K-block kb into stage kb % NS (one commit group per block)
    auto load = [&](int kb) {
        if (kb < nkb) {
            float *st = tsm + (kb % NS) * L::STAGE;
            const int k0 = kb * TC_KB;
            for (int i = tid; i < TC_M * (TC_KB / 4); i += TC_T) {
                const int r = i >> 3, k = (i & 7) * 4;
                const size_t g = (size_t)(m0 + r) * d.xp + k0 + k;
                cp_async16(st + tc_off(r, k), X + g);
                cp_async16(st + L::A + tc_off(r, k), QX + g);
            }
            for (int i = tid; i < NT * (TC_KB / 4); i += TC_T) {
                const int c = i >> 3, k = (i & 7) * 4;
                int valid = nv - (k0 + k);
                valid = valid < 0 ? 0 : (valid > 4 ? 4 : valid);
                cp_async16_zfill(st + 2 * L::A + tc_off(c, k), UT + (size_t)(n0 + c) * C + k0 + k,
                                 4 * valid);
            }
        }
        cp_async_commit();
    };

    bool ok = true;
    int issued = 0;      // K-blocks whose products were issued (the same count in every thread)
    for (int kb = 0; kb < NS - 1; ++kb) load(kb);
    for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % NS;
        float *st = tsm + s * L::STAGE;
        cp_async_wait<NS - 2>();        // this thread's copies of block kb landed
        __syncthreads();                // everyone's
        if constexpr (PARTS == 2) {
            // the lo parts of the three tiles
            float *lo = st + L::TILES;
            for (int i = tid; i < L::TILES; i += TC_T) lo[i] = tf32_rest(st[i]);
            __syncthreads();
        }
        fence_proxy_async_smem();       // the tiles, before the tensor cores read them
        __syncthreads();
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t sa = smem_u32(st);
            for (int ks = 0; ks < TC_KB / 8; ++ks) {
                const uint32_t kofs = ks * 256;   // two 16-byte k-groups per K = 8
                const uint64_t ax = tc_desc(sa + kofs), aq = tc_desc(sa + 4 * L::A + kofs);
                const uint64_t bh = tc_desc(sa + 4 * 2 * L::A + kofs);
                const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
                if constexpr (PARTS == 2) {
                    const uint32_t lb = sa + 4 * L::TILES;
                    const uint64_t axl = tc_desc(lb + kofs), aql = tc_desc(lb + 4 * L::A + kofs);
                    const uint64_t bl = tc_desc(lb + 4 * 2 * L::A + kofs);
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
            tc_commit(bar + s);
        }
        issued = kb + 1;
        // block kb + NS - 1 goes into the stage block kb - 1 used: wait for its products
        const int nb = kb + NS - 1;
        if (kb >= 1 && nb < nkb) {
            const int pb = kb - 1;
            const bool landed = mbar_wait_bounded(bar + (pb % NS), (unsigned)(pb / NS) & 1u, d.spin);
            if (!__syncthreads_and(landed)) {            // one decision for the whole CTA
                ok = false;
                break;
            }
        }
        load(nb);
    }
    cp_async_wait<0>();
    // every issued product done (the last commit covers the earlier ones); after a give-up the
    // wait keeps the default limit, so that nothing is in flight when tensor memory is freed
    if (issued > 0) {
        const int last = issued - 1;
        const unsigned par = (unsigned)(last / NS) & 1u;
        bool landed = mbar_wait_bounded(bar + (last % NS), par, ok ? d.spin : kSpinLimit);
        if (!landed) landed = mbar_wait_bounded(bar + (last % NS), par);
        ok = __syncthreads_and(ok && landed);
    }
    if (!ok && tid == 0) atomicCAS(&w.status->code, 0, (int)SDM_ERR_TIMEOUT);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    if (ok) {
        const int row = m0 + 32 * warp + lane;
        const bool live = row < nv;
        const size_t tok = (size_t)p * d.T + (size_t)ti * C + row;
        const bool out_row = (size_t)ti * C + row < (size_t)d.T;
        float *dvrow = w.dv + ((size_t)p * C + row) * D + n0;
        const float *irow = w.inter + ((size_t)p * C + row) * D + n0;
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

template <typename BT, int NT>
cudaError_t launch_tc(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                      cudaStream_t st) {
    constexpr size_t smem = TcSmem<NT, sizeof(BT) == 4 ? 2 : 1>::BYTES;
    auto kern = k_dualmm_tc<BT, NT>;
    set_kernel_smem(kern, smem);
    kern<<<dim3(d.C / TC_M, d.D / NT, d.P), TC_T, smem, st>>>(d, in, w, step0, ti);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dualmm_tc(const Dims &d, const Inputs &in, const Work &w, int step0, int ti,
                             cudaStream_t st) {
    // the widest column tile (64, 32 or 16) that still gives about one CTA per SM: the step's
    // products are small, and each CTA's time is its loads of X and QX rows
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
