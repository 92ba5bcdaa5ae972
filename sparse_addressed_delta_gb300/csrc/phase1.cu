// Phase 1 of the chunked SDM write/read: the memory-independent quantities of every chunk
// (sparse-delta-memory 2.0.0, memory_ops.py module docstring, "Phase 1"; the sorted kind row
// and its groups are the phase2_kernels.py module docstring's "Determinism" paragraph).
//
// One CTA per chunk (a persistent grid walks the slab's chunks). For chunk (p, ti) with n
// valid tokens:
//   1. the n*W write entries e = t*W + j are sorted by (slot, e): a stable LSD radix sort on
//      the slot bits of 64-bit keys (slot << 32 | t << 8 | j), in shared memory when the
//      chunk's scratch fits (else in global scratch private to the CTA);
//   2. a group is a run of one slot in that row; its members are the slot's writes in token
//      order. A segmented scan of g along the row gives lw, the running log-decay of the slot
//      at each write (inclusive), and its group total lend;
//   3. gather weights gw = k exp(lw), DW weights dw = k exp(lend - lw), the group factor
//      exp(lend), and for each read entry (slot r, token t): lr = lw of the last write of r at
//      a token <= t (0 if none), qw = q exp(lr);
//   4. A[t][u] = sum over pairs of writes of one slot at tokens u < t of
//      k_t k_u exp(lw_t - lw_u), and QK[t][u] = the same over (read at t, write at u <= t)
//      with q_t and lr_t: one warp per row, its lanes over the earlier members of each group
//      (distinct tokens, so no two lanes add to one element), entries of the row in order;
//   5. (backward mode) the sorted write row with its running sums and group bounds, and the
//      read entries sorted by slot with their groups;
//   6. for the pipelined Phase 2: the slots of the entries (Work::wsl / rsl) and the DW order
//      of the groups (hot groups first, then by size).
// Every exponent is a difference of running log-decays of one slot; all sums run in a fixed
// order, so the outputs are bitwise reproducible.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int NT = 512;          // threads per Phase-1 CTA
constexpr int NW = NT / 32;

struct P1Smem {
    int hist[256];
    int base[256];
    int tile_total[256];
    int wcnt[NW][256];
    float wv[NW];
    int wf[NW];
    int wi[NW];
    float total_v;
    int total_i;
    float row[NW][kMaxChunk];
};

// One stable counting pass of the LSD radix sort: n keys from `in` to `out` by the 8-bit
// digit at `shift`. Tiles of NT keys keep their order: a key's rank among equal digits of its
// warp (match_any) plus the counts of earlier warps and earlier tiles.
__device__ void radix_pass(const unsigned long long *in, unsigned long long *out, int n,
                           int shift, P1Smem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 256; i += NT) sm.hist[i] = 0;
    for (int i = tid; i < NW * 256; i += NT) (&sm.wcnt[0][0])[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += NT) atomicAdd(&sm.hist[(int)((in[i] >> shift) & 255ull)], 1);
    __syncthreads();
    if (warp == 0) {
        int v[8], s = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) { v[k] = sm.hist[lane * 8 + k]; s += v[k]; }
        int incl = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        int run = incl - s;
#pragma unroll
        for (int k = 0; k < 8; ++k) { sm.base[lane * 8 + k] = run; run += v[k]; }
    }
    __syncthreads();
    for (int tile = 0; tile < n; tile += NT) {
        const int i = tile + tid;
        const bool ok = i < n;
        const unsigned long long key = ok ? in[i] : 0ull;
        const int d = ok ? (int)((key >> shift) & 255ull) : 256;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (ok && lane == __ffs(peers) - 1) sm.wcnt[warp][d] = __popc(peers);
        __syncthreads();
        for (int dd = tid; dd < 256; dd += NT) {
            int run = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                int c = sm.wcnt[w][dd];
                sm.wcnt[w][dd] = run;
                run += c;
            }
            sm.tile_total[dd] = run;
        }
        __syncthreads();
        if (ok) out[sm.base[d] + sm.wcnt[warp][d] + rank] = key;
        __syncthreads();
        for (int dd = tid; dd < 256; dd += NT) {
            sm.base[dd] += sm.tile_total[dd];
#pragma unroll
            for (int w = 0; w < NW; ++w) sm.wcnt[w][dd] = 0;
        }
        __syncthreads();
    }
}

// Block-wide inclusive scan of (segment head, value) pairs with a carried-in prefix; returns
// each thread's inclusive value and sets `carry` (all threads) to the last thread's value.
__device__ float seg_scan(bool head, float val, float carry_in, float &carry, P1Smem &sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int f = head ? 1 : 0;
    float v = val;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float pv = __shfl_up_sync(0xffffffffu, v, off);
        int pf = __shfl_up_sync(0xffffffffu, f, off);
        if (lane >= off) {
            if (!f) v = pv + v;
            f |= pf;
        }
    }
    if (lane == 31) { sm.wv[warp] = v; sm.wf[warp] = f; }
    __syncthreads();
    if (warp == 0) {
        float wv = lane < NW ? sm.wv[lane] : 0.f;
        int wf = lane < NW ? sm.wf[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            float pv = __shfl_up_sync(0xffffffffu, wv, off);
            int pf = __shfl_up_sync(0xffffffffu, wf, off);
            if (lane >= off) {
                if (!wf) wv = pv + wv;
                wf |= pf;
            }
        }
        float ev = __shfl_up_sync(0xffffffffu, wv, 1);
        int ef = __shfl_up_sync(0xffffffffu, wf, 1);
        float pre = (lane == 0) ? carry_in : (ef ? ev : carry_in + ev);
        if (lane < NW) sm.wv[lane] = pre;
        if (lane == NW - 1) sm.total_v = wf ? wv : carry_in + wv;
    }
    __syncthreads();
    float out = f ? v : sm.wv[warp] + v;
    carry = sm.total_v;
    __syncthreads();
    return out;
}

// Block-wide inclusive scan of ints with a carried-in prefix.
__device__ int int_scan(int val, int carry_in, int &carry, P1Smem &sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int v = val;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
    }
    if (lane == 31) sm.wi[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int wv = lane < NW ? sm.wi[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wv, off);
            if (lane >= off) wv += y;
        }
        int ex = __shfl_up_sync(0xffffffffu, wv, 1);
        if (lane < NW) sm.wi[lane] = carry_in + (lane == 0 ? 0 : ex);
        if (lane == NW - 1) sm.total_i = carry_in + wv;
    }
    __syncthreads();
    int out = sm.wi[warp] + v;
    carry = sm.total_i;
    __syncthreads();
    return out;
}

// Chunks whose scratch is in global memory work on tiles of G4 = 4 NT entries: four per
// thread, so that each thread has four global loads in flight and a tile costs one round of
// barriers for four times the entries.
constexpr int IT4 = 4;
constexpr int G4 = IT4 * NT;

// shared memory of those chunks after P1Smem: the per-(warp, digit) counts of a radix tile, and
// the scans' per-thread results
struct P1Big {
    int wc[NW][256];
    float tv[NT];
    int ti[NT];
};

// One stable counting pass of the LSD radix sort over tiles of G4 keys: warp w of the tile takes
// the IT4 x 32 keys from tile + IT4 32 w on (item k of lane l at + 32 k + l), so the order
// (warp, item, lane) is the position order. A warp ranks its items one after another against
// its own running count per digit (match_any within the item), then the counts of the earlier
// warps and tiles give each key its place.
__device__ void radix_pass4(const unsigned long long *in, unsigned long long *out, int n,
                            int shift, P1Smem &sm, P1Big &bg) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int *wcf = &bg.wc[0][0];
    for (int i = tid; i < 256; i += NT) sm.hist[i] = 0;
    for (int i = tid; i < NW * 256; i += NT) wcf[i] = 0;
    __syncthreads();
    for (int i0 = tid; i0 < n; i0 += G4) {
        unsigned long long kk[IT4];
#pragma unroll
        for (int k = 0; k < IT4; ++k) kk[k] = i0 + k * NT < n ? in[i0 + k * NT] : 0ull;
#pragma unroll
        for (int k = 0; k < IT4; ++k)
            if (i0 + k * NT < n) atomicAdd(&sm.hist[(int)((kk[k] >> shift) & 255ull)], 1);
    }
    __syncthreads();
    if (warp == 0) {
        int v[8], s = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) { v[k] = sm.hist[lane * 8 + k]; s += v[k]; }
        int incl = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        int run = incl - s;
#pragma unroll
        for (int k = 0; k < 8; ++k) { sm.base[lane * 8 + k] = run; run += v[k]; }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int tile = 0; tile < n; tile += G4) {
        const int wbase = tile + warp * (IT4 * 32);
        unsigned long long kk[IT4];
        int dg[IT4], rank[IT4];
#pragma unroll
        for (int k = 0; k < IT4; ++k) {
            const int i = wbase + k * 32 + lane;
            kk[k] = i < n ? in[i] : 0ull;
        }
#pragma unroll
        for (int k = 0; k < IT4; ++k) {
            const int i = wbase + k * 32 + lane;
            dg[k] = i < n ? (int)((kk[k] >> shift) & 255ull) : 256;
            const unsigned peers = __match_any_sync(0xffffffffu, dg[k]);
            const int before = dg[k] < 256 ? bg.wc[warp][dg[k]] : 0;
            rank[k] = before + __popc(peers & lt);
            __syncwarp();
            if (dg[k] < 256 && lane == __ffs(peers) - 1) bg.wc[warp][dg[k]] = before + __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        for (int dd = tid; dd < 256; dd += NT) {
            int run = 0;
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) {
                const int c = bg.wc[w2][dd];
                bg.wc[w2][dd] = run;
                run += c;
            }
            sm.tile_total[dd] = run;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < IT4; ++k)
            if (dg[k] < 256) out[sm.base[dg[k]] + bg.wc[warp][dg[k]] + rank[k]] = kk[k];
        __syncthreads();
        for (int dd = tid; dd < 256; dd += NT) sm.base[dd] += sm.tile_total[dd];
        for (int i = tid; i < NW * 256; i += NT) wcf[i] = 0;
        __syncthreads();
    }
}

__device__ __forceinline__ void report_bad_slot(DevStatus *st, int token) {
    atomicAdd(&st->bad_slots, 1ull);
    atomicCAS(&st->first_bad_plus1, 0, token + 1);
    st->code = SDM_ERR_DEVICE;
}

// Pointers and counts of one chunk for Phase-1 steps 3 and 4 (the sorted write row and the
// scratch of steps 1-2, in shared or global memory).
template <typename WT>
struct P1Chunk {
    const int32_t *rs;
    const WT *q;
    const unsigned long long *srt;
    const float2 *tkk;
    const int32_t *inv, *pgid, *pgs;
    const float *lws, *lend, *kf;
    int32_t *rlo, *rhi;
    float *wdw, *gw, *qw, *lr, *A, *QK, *dwt;
    int nv, nw, nr, C, W, R, S;
    // dense Gram groups (global-scratch chunks only; dpos null otherwise)
    const int32_t *dpos;
    const float *dref;
    float *dka, *dkb, *dkq;
    int nd;
    float *lw;          // token-major running log-decay of the writes (written by the Gram rows)
    const float2 *gk;   // (g, k) per entry when the scratch is in HBM (else k is in kf)
};

// 3a. weights of the sorted positions [pos0, pos1): gw = k exp(lw) (unless GW is false: the
// Gram rows write it token-major), dw = k exp(lend - lw)
template <typename WT, bool GW = true>
__device__ void p1_weights(const P1Chunk<WT> &c, int pos0, int pos1, int tid, int nthr) {
    for (int pos = pos0 + tid; pos < pos1; pos += nthr) {
        const float kk = c.tkk[pos].y;                 // the entry's k, in sorted order
        const float l = c.lws[pos];
        const float dwv = kk * expf(c.lend[c.pgid[pos]] - l);
        c.wdw[pos] = dwv;
        if (GW || c.dwt) {
            const unsigned low = (unsigned)c.srt[pos];
            const int e = (int)(low >> 8) * c.W + (int)(low & 255u);
            if (GW) c.gw[e] = kk * expf(l);
            if (c.dwt) c.dwt[e] = dwv;
        }
    }
}

// 3b. each read entry in [er_lo, er_hi) finds the last write of its slot at a token <= its own:
// an upper bound in the sorted write row, four reads per thread at a time, branch-free (the
// same probe count for all of them, so the four searches overlap); then lr and qw. With `smp`
// (every kSampleStep-th key of the row, nsmp of them, in shared memory) the bound is first
// found among the samples and then inside one window of kSampleStep - 1 keys; else over the
// whole row.
constexpr int kSampleStep = 64;
constexpr int kMaxSamples = kMaxChunk * kMaxWidth / kSampleStep;

template <typename WT, bool SAMPLED = false>
__device__ void p1_reads(const P1Chunk<WT> &c, int er_lo, int er_hi, int tid, int nthr,
                         const unsigned long long *smp = nullptr, int nsmp = 0) {
    const unsigned magR = div_magic(c.R);
    for (int er0 = er_lo + tid; er0 < er_hi; er0 += 4 * nthr) {
        unsigned long long target[4];
        int base[4], r[4], hi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int er = er0 + k * nthr;
            r[k] = er < er_hi ? c.rs[er] : -1;
            const int t = er < er_hi ? div_by(er, magR) : 0;
            target[k] = ((unsigned long long)(unsigned)r[k] << 32) | ((unsigned)t << 8) | 255u;
            base[k] = 0;
            hi[k] = c.nw;
        }
        int len0 = c.nw;
        if (SAMPLED && c.nw > 0) {
            // the number of samples <= target, then the window of row keys after the last such
            // sample and before the next (keys at or past hi count as above every target)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                int b = 0;
                for (int len = nsmp; len > 1;) {
                    const int half = len >> 1;
                    if (smp[b + half - 1] <= target[k]) b += half;
                    len -= half;
                }
                const int ns_le = b + (smp[b] <= target[k] ? 1 : 0);
                if (ns_le == 0) {
                    base[k] = 0;
                    hi[k] = 0;
                } else {
                    base[k] = (ns_le - 1) * kSampleStep + 1;
                    hi[k] = min(ns_le * kSampleStep, c.nw);
                }
            }
            len0 = kSampleStep - 1;
        }
        for (int len = len0; len > 1;) {
            const int half = len >> 1;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int ix = base[k] + half - 1;
                if (ix < hi[k] && c.srt[ix] <= target[k]) base[k] += half;
            }
            len -= half;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int er = er0 + k * nthr;
            if (er >= er_hi) continue;
            int lo = 0, hib = -1;
            float l = 0.f;
            const float qf = __int_as_float(c.rhi[er]);   // q, staged there by step 1
            const bool valid = (unsigned)r[k] < (unsigned)c.S;
            if (valid && c.nw > 0) {
                const int ub = base[k] + (base[k] < hi[k] && c.srt[base[k]] <= target[k] ? 1 : 0);
                const int pos = ub - 1;
                if (pos >= 0 && (int)(c.srt[pos] >> 32) == r[k]) {
                    hib = pos;
                    lo = c.pgs[pos];
                    l = c.lws[pos];
                    // a dense group's read: rlo = -1 - its dense index (no pair sums)
                    if (SAMPLED && c.dpos) {
                        const int dh = c.dpos[pos];
                        if (dh >= 0) lo = -1 - dh;
                    }
                }
            }
            c.rlo[er] = lo;
            c.rhi[er] = hib;
            c.lr[er] = l;
            c.qw[er] = valid ? qf * expf(l) : 0.f;
        }
    }
}

// Adds the dense-group values of one batch of a row's entries to the row's staged factors:
// lanes whose entry belongs to dense group dh >= 0 add v0 (and v1) at column dh of f0 (and
// f1). Lanes of one group (a repeated slot) are summed in lane order by the lowest of them, so
// every staged element is a fixed-order sum. `key` separates the two half-warp rows.
__device__ __forceinline__ void dense_stage(int dh, int key, float v0, float v1, float *f0,
                                            float *f1, int lane) {
    const bool dn = dh >= 0;
    const unsigned peers = __match_any_sync(0xffffffffu, dn ? (key << 16) | dh : -1 - lane);
    if (dn) {
        float s0 = 0.f, s1 = 0.f;
        for (unsigned m = peers; m; m &= m - 1u) {
            const int src = __ffs(m) - 1;
            s0 += __shfl_sync(peers, v0, src);
            s1 += __shfl_sync(peers, v1, src);
        }
        if (lane == __ffs(peers) - 1) {
            f0[dh] += s0;
            if (f1) f1[dh] += s1;
        }
    }
    __syncwarp();
}

// 4. rows [t0, t1) of A and QK. A warp takes two token rows at a time when both fit in its row
//    buffer (2 C <= kMaxChunk), one half-warp per row, else one row with all lanes. The row's
//    entries are looked up one per lane; entries with earlier members of their group (a ballot)
//    are then taken in entry order, the lanes of the row over those members (distinct tokens,
//    so no two lanes add to one element). (token, k) of every sorted position is kept in the
//    free radix buffer, next to its running log-decay. Entries of dense groups take no pair
//    sums here: they add their factors to the row's staged dense rows (dka, dkb from the
//    writes, dkq from the reads; `drow` holds 3 dense_pitch(C) floats per row), which
//    k_gram_dense multiplies out.
template <typename WT, bool TWO, int kPairAhead, bool WGL>
__device__ void p1_gram_rows(const P1Chunk<WT> &c, int t0, int t1, int warp, int nwarps, int lane,
                             float *row, float *drow) {
    const int C = c.C, W = c.W, R = c.R;
    constexpr int lpr = TWO ? 16 : 32;                  // lanes per row
    const int hsel = TWO ? lane >> 4 : 0;
    const int hl = lane & (lpr - 1);
    const unsigned hmask = TWO ? 0xffffu << (16 * hsel) : 0xffffffffu;
    constexpr int rpw = TWO ? 2 : 1;                    // rows per warp and pass
    float *rw = row + hsel * C;
    const int dp = dense_pitch(C);
    const int hp = kPairAhead > 1 && c.dpos ? (c.nd + 3) & ~3 : 0;   // staged dense columns
                                                     // (only the look-ahead variant stages)
    float *da = hp ? drow + hsel * 3 * dp : nullptr, *db = da + dp, *dq = db + dp;
    for (int tb = t0 + warp * rpw; tb < t1; tb += nwarps * rpw) {
        const int t = tb + hsel;
        const bool live = t < t1;                       // else this half only joins the shuffles
        const bool act = live && t < c.nv;
        for (int x = hl; x < C; x += lpr) rw[x] = 0.f;
        for (int x = hl; x < hp; x += lpr) { da[x] = 0.f; db[x] = 0.f; dq[x] = 0.f; }
        __syncwarp();
        for (int j0 = 0; j0 < W; j0 += lpr) {
            const int j = j0 + hl;
            float ka = 0.f, la = 0.f;
            int pos = 0, gs = 0, dh = -1;
            if (act && j < W) {
                const int e = t * W + j;
                ka = c.gk ? c.gk[e].y : c.kf[e];
                pos = c.inv[e];
                gs = c.pgs[pos];
                la = c.lws[pos];
                if (hp) dh = c.dpos[pos];
                if (WGL) {                   // the token-major running sum and gather weight
                    c.lw[e] = la;
                    c.gw[e] = ka * expf(la);
                }
            }
            if (hp) {
                float va = 0.f, vb = 0.f;
                if (dh >= 0) {
                    const float r = c.dref[dh];
                    va = ka * expf(la - r);
                    vb = ka * expf(r - la);
                }
                dense_stage(dh, hsel, va, vb, da, db, lane);
            }
            unsigned todo = __ballot_sync(0xffffffffu, ka != 0.f && pos > gs && dh < 0) & hmask;
            while (__any_sync(0xffffffffu, todo != 0u)) {
                // up to kPairAhead entries at a time: the first lane-stride of each one's
                // earlier members is loaded before any is added; the adds then run entry by
                // entry as before (members of one entry have distinct tokens, so no two lanes
                // add to one element, and each element sees the entries in row order)
                float kb[kPairAhead], lb[kPairAhead], l1[kPairAhead];
                int gb[kPairAhead], pe[kPairAhead];
                float2 tk1[kPairAhead];
#pragma unroll
                for (int u = 0; u < kPairAhead; ++u) {
                    const bool has = todo != 0u;
                    const int src = has ? __ffs(todo) - 1 : lane;
                    todo &= todo - 1u;
                    kb[u] = __shfl_sync(0xffffffffu, ka, src);
                    lb[u] = __shfl_sync(0xffffffffu, la, src);
                    const int pb = __shfl_sync(0xffffffffu, pos, src);
                    gb[u] = __shfl_sync(0xffffffffu, gs, src);
                    pe[u] = has ? pb : gb[u];
                    if (gb[u] + hl < pe[u]) {
                        tk1[u] = c.tkk[gb[u] + hl];
                        l1[u] = c.lws[gb[u] + hl];
                    }
                }
#pragma unroll
                for (int u = 0; u < kPairAhead; ++u) {
                    if (gb[u] + hl < pe[u])
                        rw[__float_as_int(tk1[u].x)] += kb[u] * tk1[u].y * expf(lb[u] - l1[u]);
                    for (int m = gb[u] + hl + lpr; m < pe[u]; m += lpr) {
                        const float2 tk = c.tkk[m];
                        rw[__float_as_int(tk.x)] += kb[u] * tk.y * expf(lb[u] - c.lws[m]);
                    }
                    __syncwarp();
                }
            }
        }
        if (live)
            for (int x = hl; x < C; x += lpr) c.A[(size_t)t * C + x] = rw[x];
        __syncwarp();
        for (int x = hl; x < C; x += lpr) rw[x] = 0.f;
        __syncwarp();
        for (int i0 = 0; i0 < R; i0 += lpr) {
            const int i = i0 + hl;
            float qa = 0.f, la = 0.f;
            int lo = 0, hi = -1;
            if (act && i < R) {
                const int er = t * R + i;
                lo = c.rlo[er];
                hi = c.rhi[er];
                if (hi >= 0) {
                    qa = to_f32(c.q[er]);
                    la = c.lr[er];
                }
            }
            if (hp) {
                const int dh = hi >= 0 && lo < 0 ? -1 - lo : -1;
                const float vq = dh >= 0 ? qa * expf(la - c.dref[dh]) : 0.f;
                dense_stage(dh, hsel, vq, 0.f, dq, nullptr, lane);
            }
            unsigned todo = __ballot_sync(0xffffffffu, hi >= 0 && lo >= 0) & hmask;
            while (__any_sync(0xffffffffu, todo != 0u)) {
                // as for the writes: kPairAhead read entries' first member loads in flight
                float qb[kPairAhead], lb[kPairAhead], l1[kPairAhead];
                int lob[kPairAhead], he[kPairAhead];
                float2 tk1[kPairAhead];
#pragma unroll
                for (int u = 0; u < kPairAhead; ++u) {
                    const bool has = todo != 0u;
                    const int src = has ? __ffs(todo) - 1 : lane;
                    todo &= todo - 1u;
                    qb[u] = __shfl_sync(0xffffffffu, qa, src);
                    lb[u] = __shfl_sync(0xffffffffu, la, src);
                    lob[u] = __shfl_sync(0xffffffffu, lo, src);
                    const int hib = __shfl_sync(0xffffffffu, hi, src);
                    he[u] = has ? hib : lob[u] - 1;
                    if (lob[u] + hl <= he[u]) {
                        tk1[u] = c.tkk[lob[u] + hl];
                        l1[u] = c.lws[lob[u] + hl];
                    }
                }
#pragma unroll
                for (int u = 0; u < kPairAhead; ++u) {
                    if (lob[u] + hl <= he[u])
                        rw[__float_as_int(tk1[u].x)] += qb[u] * tk1[u].y * expf(lb[u] - l1[u]);
                    for (int m = lob[u] + hl + lpr; m <= he[u]; m += lpr) {
                        const float2 tk = c.tkk[m];
                        rw[__float_as_int(tk.x)] += qb[u] * tk.y * expf(lb[u] - c.lws[m]);
                    }
                    __syncwarp();
                }
            }
        }
        if (live) {
            for (int x = hl; x < C; x += lpr) c.QK[(size_t)t * C + x] = rw[x];
            for (int x = hl; x < hp; x += lpr) {
                c.dka[(size_t)t * dp + x] = da[x];
                c.dkb[(size_t)t * dp + x] = db[x];
                c.dkq[(size_t)t * dp + x] = dq[x];
            }
        }
        __syncwarp();
    }
}

// AHEAD: Gram row entries whose first member loads are in flight at once; WGL: the rows also
// write the token-major lw and gw of their write entries
template <typename WT, int AHEAD, bool WGL>
__device__ __forceinline__ void p1_gram(const P1Chunk<WT> &c, int t0, int t1, int warp, int nwarps,
                                        int lane, float *row, float *drow) {
    if (2 * c.C <= kMaxChunk)
        p1_gram_rows<WT, true, AHEAD, WGL>(c, t0, t1, warp, nwarps, lane, row, drow);
    else
        p1_gram_rows<WT, false, AHEAD, WGL>(c, t0, t1, warp, nwarps, lane, row, drow);
}

// Dense Gram groups of a chunk whose scratch is in global memory. A group of n members costs
// about n^2 pair terms in the row kernel but a fixed C^2 multiply-adds as a dense factor, so the
// large groups go dense: those of at least thr members, thr the least of (C/8) << L
// (L = 0..7) that leaves at most C of them, in group order; of these, the ones whose running
// log-decays lie within kDenseSpan of each other (finite), with the middle of that range as the
// reference (so every factor exp(lw - ref), exp(ref - lw) is at most exp(kDenseSpan / 2)). Sets
// dpos of their members (the caller has set it to -1 at every position), dref and ndense.
__device__ void p1_dense_select(const int32_t *go, int ng, const float *lws, int C, int32_t *dpos,
                                float *dref, int32_t *ndense, P1Smem &sm, P1Big &bg) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NL = 8;
    const int thr0 = C / 8;
    if (tid <= NL) sm.hist[tid] = 0;
    __syncthreads();
    int cnt[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) cnt[l] = 0;
    for (int g = tid; g < ng; g += NT) {
        const int sz = go[g + 1] - go[g];
#pragma unroll
        for (int l = 0; l < NL; ++l) cnt[l] += sz >= (thr0 << l) ? 1 : 0;
    }
#pragma unroll
    for (int l = 0; l < NL; ++l) {
        int v = cnt[l];
#pragma unroll
        for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0 && v) atomicAdd(&sm.hist[l], v);
    }
    __syncthreads();
    int thr = -1;
    for (int l = 0; l < NL && thr < 0; ++l)
        if (sm.hist[l] <= C) thr = thr0 << l;
    if (thr < 0) {                     // cannot happen for distinct slots; no dense groups
        if (tid == 0) *ndense = 0;
        __syncthreads();
        return;
    }
    // the candidates, in any order, then ranked into group order
    int *list = bg.ti;
    int *sorted = &bg.wc[0][0];
    int *hidx = sorted + kMaxChunk;
    float *ref = reinterpret_cast<float *>(sorted + 2 * kMaxChunk);
    for (int g0 = 0; g0 < ng; g0 += NT) {
        const int g = g0 + tid;
        const bool take = g < ng && go[g + 1] - go[g] >= thr;
        const unsigned b = __ballot_sync(0xffffffffu, take);
        int base = 0;
        if (lane == 0 && b) base = atomicAdd(&sm.hist[NL], __popc(b));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (take) list[base + __popc(b & ((1u << lane) - 1u))] = g;
    }
    __syncthreads();
    const int nc = sm.hist[NL];
    if (tid < nc) {
        const int gi = list[tid];
        int r = 0;
        for (int j = 0; j < nc; ++j) r += list[j] < gi ? 1 : 0;
        sorted[r] = gi;
    }
    __syncthreads();
    // the range of each candidate's running log-decays, one warp per candidate
    for (int k = warp; k < nc; k += NW) {
        const int g = sorted[k];
        float mn = 3.0e38f, mx = -3.0e38f;
        bool bad = false;
        for (int pos = go[g] + lane; pos < go[g + 1]; pos += 32) {
            const float l = lws[pos];
            bad |= !(fabsf(l) <= 3.0e38f);           // NaN or infinite
            mn = fminf(mn, l);
            mx = fmaxf(mx, l);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            hidx[k] = !bad && mx - mn <= kDenseSpan ? 1 : 0;
            ref[k] = 0.5f * (mx + mn);
        }
    }
    __syncthreads();
    int h = -1;
    if (tid < nc && hidx[tid]) {
        h = 0;
        for (int j = 0; j < tid; ++j) h += hidx[j];
        dref[h] = ref[tid];
    }
    if (tid == 0) {
        int tot = 0;
        for (int j = 0; j < nc; ++j) tot += hidx[j];
        *ndense = tot;
    }
    __syncthreads();
    if (tid < nc) list[tid] = h;
    __syncthreads();
    for (int k = warp; k < nc; k += NW) {
        const int hk = list[k];
        if (hk < 0) continue;
        const int g = sorted[k];
        for (int pos = go[g] + lane; pos < go[g + 1]; pos += 32) dpos[pos] = hk;
    }
    __syncthreads();
}

template <typename WT>
__global__ void __launch_bounds__(NT, 2) k_phase1(Dims d, Inputs in, Work w, int step0, int nsteps,
                                               int scratch_in_smem) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    P1Smem &sm = *reinterpret_cast<P1Smem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = d.C, W = d.W, R = d.R, S = d.S;
    const int CW = C * W, CR = C * R, CC = C * C;
    const WT *kw = static_cast<const WT *>(in.kw);
    const WT *qwin = static_cast<const WT *>(in.qw);
    const int N = nsteps * d.P;
    const unsigned magW = div_magic(W), magR = div_magic(R);
    // sort keys are (slot << 32 | t << 8 | j): the low word orders like e = t*W + j, and the
    // token of an entry is a shift away
    auto ent_of = [W](unsigned low) { return (int)(low >> 8) * W + (int)(low & 255u); };
    const int bits = S <= 1 ? 0 : 32 - __clz(S - 1);
    const int passes = (bits + 7) / 8;

    // per-chunk scratch: in shared memory after P1Smem when it fits, else the CTA's slice of
    // the workspace (same layout either way)
    unsigned long long *keyA;
    int32_t *inv, *pgid, *pgs, *rlo, *rhi;
    int32_t *sgo = nullptr;   // group starts of the chunk on chip (else the chunk's goff row)
    float *lws, *lend, *kf = nullptr;
    float2 *gk = nullptr;      // (g, k) per entry (scratch in HBM)
    if (scratch_in_smem) {
        unsigned char *q = smem_raw + ((sizeof(P1Smem) + 15) & ~size_t(15));
        keyA = reinterpret_cast<unsigned long long *>(q); q += sizeof(unsigned long long) * 2 * CW;
        inv = reinterpret_cast<int32_t *>(q); q += 4 * (size_t)CW;
        pgid = reinterpret_cast<int32_t *>(q); q += 4 * (size_t)CW;
        pgs = reinterpret_cast<int32_t *>(q); q += 4 * (size_t)CW;
        lws = reinterpret_cast<float *>(q); q += 4 * (size_t)CW;
        lend = reinterpret_cast<float *>(q); q += 4 * (size_t)CW;
        kf = reinterpret_cast<float *>(q); q += 4 * (size_t)CW;
        rlo = reinterpret_cast<int32_t *>(q); q += 4 * (size_t)CR;
        rhi = reinterpret_cast<int32_t *>(q); q += 4 * (size_t)CR;
        sgo = reinterpret_cast<int32_t *>(q);
    } else {
        keyA = w.keys + (size_t)blockIdx.x * 2 * CW;
        inv = w.inv + (size_t)blockIdx.x * CW;
        pgid = w.pgid + (size_t)blockIdx.x * CW;
        pgs = w.pgs + (size_t)blockIdx.x * CW;
        lws = w.lws + (size_t)blockIdx.x * CW;
        lend = w.lend + (size_t)blockIdx.x * CW;
        gk = w.gk + (size_t)blockIdx.x * CW;
        rlo = w.rlo + (size_t)blockIdx.x * CR;
        rhi = w.rhi + (size_t)blockIdx.x * CR;
    }
    unsigned long long *keyB = keyA + CW;
    // chunks whose scratch lives in global memory leave steps 3 and 4 to k_phase1_rows (the
    // grid then has one CTA per chunk, so the scratch of chunk n stays in slot n), and work on
    // tiles of G4 entries with the counts and scan values after P1Smem
    const bool split = !scratch_in_smem;
    P1Big *bigp = reinterpret_cast<P1Big *>(smem_raw + ((sizeof(P1Smem) + 15) & ~size_t(15)));

    for (int n = blockIdx.x; n < N; n += gridDim.x) {
        const int p = n % d.P, ti = step0 + n / d.P;
        const int tok0 = ti * C;
        const int nv = chunk_valid(in.valid, p, d.T, tok0, C);
        const int nw = nv * W, nr = nv * R;
        const size_t tok_base = (size_t)p * d.T + tok0;
        const int32_t *ws = in.ws + tok_base * W;
        const int32_t *rs = in.rs + tok_base * R;
        const float *g = in.g + tok_base * (d.gate ? 1 : W);   // per entry, or per token
        const WT *k = kw + tok_base * W;
        const WT *q = qwin + tok_base * R;

        int32_t *perm = w.perm + (size_t)n * CW;
        float *wdw = w.wdw + (size_t)n * CW;
        int32_t *goff = w.goff + (size_t)n * goff_stride(CW);
        int32_t *go = scratch_in_smem ? sgo : goff;
        int32_t *gslot = w.gslot + (size_t)n * CW;
        float *gfac = w.gfac + (size_t)n * CW;
        float *gw = w.gw + (size_t)n * CW;
        float *qw = w.qw + (size_t)n * CR;
        float *lw = w.lw + (size_t)n * CW;
        float *lr = w.lr + (size_t)n * CR;
        int32_t *minfo = w.minfo + (size_t)n * CW;
        int32_t *wsl = w.wsl + (size_t)n * CW;
        int32_t *rsl = w.rsl + (size_t)n * CR;
        float *A = w.A + (size_t)n * CC;
        float *QK = w.QK + (size_t)n * CC;

        // 1. keys (a slot outside [0, S) is reported and sorted as slot S, after every real
        //    slot, with weight 0 and log-decay 0: it adds nothing anywhere and no DW writes it)
        int bad = 0;
        auto key_of = [&](int i, int sraw, float kraw, float graw) {
            int s = sraw;
            float kk = kraw;
            if ((unsigned)s >= (unsigned)S) {
                report_bad_slot(w.status, (int)(tok_base + i / W));
                s = S;
                kk = 0.f;
                bad = 1;
            }
            // k and g (0 if dropped), read in step 2: one (g, k) pair with the scratch in
            // HBM (a single random read per sorted position there), else two arrays on chip
            const float gg = s == S ? 0.f : graw;
            if (gk) {
                gk[i] = make_float2(gg, kk);
            } else {
                kf[i] = kk;
                pgs[i] = __float_as_int(gg);
            }
            wsl[i] = s < S ? s : kNoEntry;
            const int t = div_by(i, magW);
            keyA[i] = ((unsigned long long)(unsigned)s << 32) | ((unsigned)t << 8) |
                      (unsigned)(i - t * W);
        };
        auto read_of = [&](int i, int r, float qraw) {
            if ((unsigned)r >= (unsigned)S) report_bad_slot(w.status, (int)(tok_base + i / R));
            rsl[i] = (unsigned)r < (unsigned)S ? r : kNoEntry;
            rhi[i] = __float_as_int(qraw);   // q, read back in step 3
        };
        if (split) {
            // four entries per thread, their loads first
            for (int i0 = tid; i0 < nw; i0 += G4) {
                int sv[IT4];
                float kv[IT4], gv[IT4];
#pragma unroll
                for (int u = 0; u < IT4; ++u) {
                    const int i = i0 + u * NT;
                    if (i < nw) {
                        sv[u] = ws[i];
                        kv[u] = to_f32(k[i]);
                        gv[u] = g[d.gate ? div_by(i, magW) : i];
                    }
                }
#pragma unroll
                for (int u = 0; u < IT4; ++u)
                    if (i0 + u * NT < nw) key_of(i0 + u * NT, sv[u], kv[u], gv[u]);
            }
            for (int i0 = tid; i0 < nr; i0 += G4) {
                int rv[IT4];
                float qv[IT4];
#pragma unroll
                for (int u = 0; u < IT4; ++u) {
                    const int i = i0 + u * NT;
                    if (i < nr) { rv[u] = rs[i]; qv[u] = to_f32(q[i]); }
                }
#pragma unroll
                for (int u = 0; u < IT4; ++u)
                    if (i0 + u * NT < nr) read_of(i0 + u * NT, rv[u], qv[u]);
            }
        } else {
            for (int i = tid; i < nw; i += NT)
                key_of(i, ws[i], to_f32(k[i]), g[d.gate ? div_by(i, magW) : i]);
            for (int i = tid; i < nr; i += NT) read_of(i, rs[i], to_f32(q[i]));
        }
        // slot S may need one more radix digit than the real slots
        const int npass = __syncthreads_or(bad) ? (32 - __clz(S) + 7) / 8 : passes;
        unsigned long long *src = keyA, *dst = keyB;
        for (int ps = 0; ps < npass; ++ps) {
            if (split) radix_pass4(src, dst, nw, 32 + 8 * ps, sm, *bigp);
            else radix_pass(src, dst, nw, 32 + 8 * ps, sm);
            unsigned long long *t = src; src = dst; dst = t;
        }
        const unsigned long long *srt = src;
        float2 *tkk = reinterpret_cast<float2 *>(dst);   // (token bits, k) per sorted position

        // 2. groups and running log-decays along the sorted row
        float carry_v = 0.f;
        int carry_i = 0;
        if (split) {
            // tiles of G4 positions, four consecutive ones per thread: a thread-local segmented
            // scan, then one across the threads' aggregates, whose exclusive values (read from
            // shared memory) carry into each thread's positions before its first group head
            for (int tile = 0; tile < nw; tile += G4) {
                const int pos0 = tile + IT4 * tid;
                unsigned long long kk[IT4 + 2];          // positions pos0 - 1 .. pos0 + 4
#pragma unroll
                for (int u = 0; u < IT4 + 2; ++u) {
                    const int ps = pos0 - 1 + u;
                    kk[u] = (ps >= 0 && ps < nw) ? srt[ps] : ~0ull;
                }
                int e[IT4];
                float gv[IT4], kv[IT4];
                bool head[IT4], tail[IT4];
#pragma unroll
                for (int u = 0; u < IT4; ++u) {
                    const int ps = pos0 + u;
                    const bool ok = ps < nw;
                    const unsigned low = (unsigned)(kk[u + 1] & 0xffffffffu);
                    const int slot = (int)(kk[u + 1] >> 32);
                    e[u] = ok ? ent_of(low) : 0;
                    head[u] = ok && (ps == 0 || (int)(kk[u] >> 32) != slot);
                    tail[u] = ok && (ps == nw - 1 || (int)(kk[u + 2] >> 32) != slot);
                    const float2 pr = ok ? gk[e[u]] : make_float2(0.f, 0.f);
                    gv[u] = pr.x;
                    kv[u] = pr.y;
                }
                // thread-local inclusive values and head counts
                float lv[IT4];
                int hc[IT4];
                bool any_head = false;
                float run = 0.f;
                int hrun = 0;
#pragma unroll
                for (int u = 0; u < IT4; ++u) {
                    run = head[u] ? gv[u] : run + gv[u];
                    any_head |= head[u];
                    hrun += head[u] ? 1 : 0;
                    lv[u] = run;
                    hc[u] = hrun;
                }
                float cv;
                const float incl_v = seg_scan(any_head, run, carry_v, cv, sm);
                int ci;
                const int incl_i = int_scan(hrun, carry_i, ci, sm);
                bigp->tv[tid] = incl_v;
                bigp->ti[tid] = incl_i;
                __syncthreads();
                const float ex_v = tid == 0 ? carry_v : bigp->tv[tid - 1];
                const int ex_i = tid == 0 ? carry_i : bigp->ti[tid - 1];
                carry_v = cv;
                carry_i = ci;
                bool seen = false;
#pragma unroll
                for (int u = 0; u < IT4; ++u) {
                    const int ps = pos0 + u;
                    if (ps >= nw) break;
                    seen |= head[u];
                    const float l = seen ? lv[u] : ex_v + lv[u];
                    const int gid = ex_i + hc[u] - 1;
                    const unsigned low = (unsigned)(kk[u + 1] & 0xffffffffu);
                    const int slot = (int)(kk[u + 1] >> 32);
                    perm[ps] = e[u];
                    inv[e[u]] = ps;
                    tkk[ps] = make_float2(__int_as_float((int)(low >> 8)), kv[u]);
                    if (!head[u] && ((unsigned)kk[u] >> 8) == (low >> 8))
                        atomicAdd(&w.status->repeated_write_slots, 1ull);
                    lws[ps] = l;          // lw[e] is written token-major by k_phase1_rows
                    pgid[ps] = gid;
                    if (head[u]) {
                        goff[gid] = ps;
                        gslot[gid] = slot;
                    }
                    if (tail[u]) {
                        lend[gid] = l;
                        gfac[gid] = expf(l);
                    }
                    minfo[ps] = (int)(low >> 8) | (int)((low & 255u) << 8) | (head[u] ? 1 << 16 : 0) |
                                (tail[u] ? 1 << 17 : 0);
                }
                __syncthreads();
            }
        }
        for (int tile = 0; !split && tile < nw; tile += NT) {
            const int pos = tile + tid;
            const bool ok = pos < nw;
            unsigned long long key = ok ? srt[pos] : 0ull;
            const unsigned low = (unsigned)(key & 0xffffffffu);
            const int slot = (int)(key >> 32), e = ent_of(low);
            bool head = ok && (pos == 0 || (int)(srt[pos - 1] >> 32) != slot);
            float gv = 0.f;
            if (ok) {
                gv = __int_as_float(pgs[e]);
                perm[pos] = e;
                inv[e] = pos;
                tkk[pos] = make_float2(__int_as_float((int)(low >> 8)), kf[e]);
                if (!head && ((unsigned)srt[pos - 1] >> 8) == (low >> 8))
                    atomicAdd(&w.status->repeated_write_slots, 1ull);
            }
            float cv, lv;
            lv = seg_scan(head, gv, carry_v, cv, sm);
            carry_v = cv;
            int ci;
            int gid = int_scan(head ? 1 : 0, carry_i, ci, sm) - 1;
            carry_i = ci;
            if (ok) {
                lws[pos] = lv;
                lw[e] = lv;
                pgid[pos] = gid;
                if (head) {
                    goff[gid] = pos;
                    gslot[gid] = slot;
                    if (scratch_in_smem) sgo[gid] = pos;
                }
                const bool tail = (pos == nw - 1) || (int)(srt[pos + 1] >> 32) != slot;
                if (tail) {
                    lend[gid] = lv;
                    gfac[gid] = expf(lv);
                }
                minfo[pos] = (int)(low >> 8) | (int)((low & 255u) << 8) | (head ? 1 << 16 : 0) |
                             (tail ? 1 << 17 : 0);
            }
        }
        const int ng = carry_i;
        if (tid == 0) {
            w.ngroups[n] = ng;
            w.nvalid[n] = nv;
            goff[ng] = nw;
            if (scratch_in_smem) sgo[ng] = nw;
        }
        __syncthreads();
        // group start of every sorted position (one lookup instead of a chain later)
        int32_t *dpos = split && C >= kDenseMinChunk ? w.dpos + (size_t)blockIdx.x * CW : nullptr;
        if (split) {
            for (int p0 = tid; p0 < nw; p0 += G4) {
                int gid[IT4];
#pragma unroll
                for (int u = 0; u < IT4; ++u) gid[u] = p0 + u * NT < nw ? pgid[p0 + u * NT] : 0;
                int gs[IT4];
#pragma unroll
                for (int u = 0; u < IT4; ++u) gs[u] = p0 + u * NT < nw ? go[gid[u]] : 0;
#pragma unroll
                for (int u = 0; u < IT4; ++u)
                    if (p0 + u * NT < nw) {
                        pgs[p0 + u * NT] = gs[u];
                        if (dpos) dpos[p0 + u * NT] = -1;
                    }
            }
        } else {
            for (int pos = tid; pos < nw; pos += NT) pgs[pos] = go[pgid[pos]];
        }
        __syncthreads();
        if (dpos)
            p1_dense_select(go, ng, lws, C, dpos, w.dref + (size_t)n * C, w.ndense + n, sm, *bigp);

        const P1Chunk<WT> pc{rs, q, srt, tkk, inv, pgid, pgs, lws, lend, kf, rlo, rhi,
                             wdw, gw, qw, lr, A, QK,
                             d.bwd ? w.dwt + (size_t)n * CW : nullptr,
                             nv, nw, nr, C, W, R, S,
                             nullptr, nullptr, nullptr, nullptr, nullptr, 0, lw, nullptr};
        if (split) {
            // steps 3 and 4 run in k_phase1_rows, over many CTAs per chunk; it finds the
            // sorted row in the radix buffer recorded here
            if (tid == 0) w.p1sel[n] = srt == keyA ? 0 : 1;
        } else {
            // 3. weights and the reads' last writes; 4. the Gram rows
            p1_weights(pc, 0, nw, tid, NT);
            p1_reads(pc, 0, nr, tid, NT);
            __syncthreads();
            p1_gram<WT, 1, false>(pc, 0, C, warp, NW, lane, sm.row[warp], nullptr);
        }
        // tails of the per-entry rows past the valid entries (read by nothing but the debug
        // copy; written so that every output element is defined)
        if (d.bwd) {
            // 5. what the backward reads back: the sorted write row with its running log-decays
            //    and group bounds, and the read kind row sorted by (slot, t, i) with its groups
            for (int pos = tid; pos < nw; pos += NT) {
                const size_t o = (size_t)n * CW + pos;
                w.wkey[o] = srt[pos];
                w.wlws[o] = lws[pos];
                w.wpgs[o] = pgs[pos];
                w.wpge[o] = go[pgid[pos] + 1];
            }
            unsigned long long *rA = w.rkeys + (size_t)blockIdx.x * 2 * CR;
            unsigned long long *rB = rA + CR;
            int rbad = 0;
            for (int i = tid; i < nr; i += NT) {
                int sl = rs[i];
                if ((unsigned)sl >= (unsigned)S) { sl = S; rbad = 1; }
                const int t = div_by(i, magR);
                rA[i] = ((unsigned long long)(unsigned)sl << 32) | ((unsigned)t << 8) |
                        (unsigned)(i - t * R);
            }
            const int rpass = __syncthreads_or(rbad) ? (32 - __clz(S) + 7) / 8 : passes;
            unsigned long long *rsrc = rA, *rdst = rB;
            for (int ps = 0; ps < rpass; ++ps) {
                radix_pass(rsrc, rdst, nr, 32 + 8 * ps, sm);
                unsigned long long *tt = rsrc; rsrc = rdst; rdst = tt;
            }
            int32_t *rgoff = w.rgoff + (size_t)n * (CR + 1);
            int32_t *rgslot = w.rgslot + (size_t)n * CR;
            int rcarry = 0;
            for (int tile = 0; tile < nr; tile += NT) {
                const int pos = tile + tid;
                const bool ok = pos < nr;
                const unsigned long long key = ok ? rsrc[pos] : 0ull;
                const int sl = (int)(key >> 32);
                const bool head = ok && (pos == 0 || (int)(rsrc[pos - 1] >> 32) != sl);
                int ci;
                const int gid = int_scan(head ? 1 : 0, rcarry, ci, sm) - 1;
                rcarry = ci;
                if (ok) {
                    w.rkey[(size_t)n * CR + pos] = key;
                    if (head) { rgoff[gid] = pos; rgslot[gid] = sl; }
                }
            }
            if (tid == 0) { w.rng[n] = rcarry; rgoff[rcarry] = nr; }
            __syncthreads();
        }
        // 6. the DW order of Phase 2: the hot groups (at least hmin members) first, then the
        //    others by size, largest first (a counting sort over 1 + hmin size classes; the
        //    order inside a class is arbitrary, as a group's sum does not depend on which
        //    thread computes it). Warp-aggregated shared-memory atomics. The pipelined kernel
        //    gives each hot group a warp (hmin = kHotGroup); the per-step DW sums them with the
        //    whole CTA, which pays off from about C/8 members on (hmin = max(kHotGroup, C/8)).
        {
            const int hmin = d.per_step && C / 8 > kHotGroup ? C / 8 : kHotGroup;
            const int NB = hmin + 1;
            int *cnt = sm.hist, *cur = sm.hist + NB, *bas = sm.base;
            for (int i = tid; i < 2 * NB; i += NT) sm.hist[i] = 0;
            __syncthreads();
            auto digit = [&](int g) {
                const int sz = go[g + 1] - go[g];
                return sz >= hmin ? 0 : 1 + hmin - sz;
            };
            for (int g0 = 0; g0 < ng; g0 += NT) {
                const int g = g0 + tid;
                const int dig = g < ng ? digit(g) : NB;
                const unsigned peers = __match_any_sync(0xffffffffu, dig);
                if (dig < NB && lane == __ffs(peers) - 1) atomicAdd(&cnt[dig], __popc(peers));
            }
            __syncthreads();
            if (tid == 0) {
                int run = 0;
                for (int k = 0; k < NB; ++k) { bas[k] = run; run += cnt[k]; }
                w.ng4[n] = make_int4(ng, cnt[0], 0, 0);
            }
            __syncthreads();
            int32_t *gord = w.gord + (size_t)n * CW;
            for (int g0 = 0; g0 < ng; g0 += NT) {
                const int g = g0 + tid;
                const int dig = g < ng ? digit(g) : NB;
                const unsigned peers = __match_any_sync(0xffffffffu, dig);
                const int leader = __ffs(peers) - 1;
                int first = 0;
                if (dig < NB && lane == leader) first = atomicAdd(&cur[dig], __popc(peers));
                first = __shfl_sync(0xffffffffu, first, leader);
                if (dig < NB) gord[bas[dig] + first + __popc(peers & ((1u << lane) - 1u))] = g;
            }
        }
        for (int i = nw + tid; i < CW; i += NT) {
            perm[i] = -1; gw[i] = 0.f; lw[i] = 0.f; wdw[i] = 0.f; wsl[i] = kNoEntry;
        }
        for (int i = nr + tid; i < CR; i += NT) { qw[i] = 0.f; lr[i] = 0.f; rsl[i] = kNoEntry; }
        __syncthreads();
    }
}

// Steps 3 and 4 of the chunks whose scratch is in global memory: CTA (rb, n) takes a share of
// chunk n's sorted positions (weights), the reads of its KR token rows and those rows of A and
// QK. 8 warps, one row at a time each. BIG (C >= kDenseMinChunk): the chunk's large groups are
// dense (staged rows per warp), the reads search a sample of the sorted row first, and the
// Gram rows keep four entries' member loads in flight; shared memory (dynamic):
//   rows [8][kMaxChunk] float | BIG: drows [8][3 kMaxChunk] float, samples [kMaxSamples] u64
constexpr int KR = 16;          // token rows per CTA
constexpr int NTR = 256;

constexpr size_t rows_smem(bool big) {
    return sizeof(float) * (NTR / 32) * kMaxChunk +
           (big ? sizeof(float) * (NTR / 32) * 3 * kMaxChunk +
                      sizeof(unsigned long long) * kMaxSamples
                : 0);
}

template <typename WT, bool BIG>
__global__ void __launch_bounds__(NTR, BIG ? 4 : 6) k_phase1_rows(Dims d, Inputs in, Work w,
                                                                  int step0) {
    extern __shared__ __align__(16) unsigned char rsm[];
    float *rows = reinterpret_cast<float *>(rsm);
    float *drows = BIG ? rows + (NTR / 32) * kMaxChunk : nullptr;
    unsigned long long *smp =
        BIG ? reinterpret_cast<unsigned long long *>(drows + (NTR / 32) * 3 * kMaxChunk) : nullptr;
    const int n = blockIdx.y, rb = blockIdx.x, nrb = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = d.C, W = d.W, R = d.R, CW = C * W, CR = C * R, CC = C * C;
    const int p = n % d.P, ti = step0 + n / d.P;
    const int tok0 = ti * C;
    const int nv = chunk_valid(in.valid, p, d.T, tok0, C);
    const int nw = nv * W, nr = nv * R;
    const size_t tok_base = (size_t)p * d.T + tok0;
    const unsigned long long *keyA = w.keys + (size_t)n * 2 * CW;
    const unsigned long long *srt = w.p1sel[n] ? keyA + CW : keyA;
    const float2 *tkk = reinterpret_cast<const float2 *>(w.p1sel[n] ? keyA : keyA + CW);
    P1Chunk<WT> pc{in.rs + tok_base * R, static_cast<const WT *>(in.qw) + tok_base * R,
                         srt, tkk, w.inv + (size_t)n * CW, w.pgid + (size_t)n * CW,
                         w.pgs + (size_t)n * CW, w.lws + (size_t)n * CW, w.lend + (size_t)n * CW,
                         nullptr, w.rlo + (size_t)n * CR, w.rhi + (size_t)n * CR,
                         w.wdw + (size_t)n * CW, w.gw + (size_t)n * CW, w.qw + (size_t)n * CR,
                         w.lr + (size_t)n * CR, w.A + (size_t)n * CC, w.QK + (size_t)n * CC,
                         d.bwd ? w.dwt + (size_t)n * CW : nullptr,
                         nv, nw, nr, C, W, R, d.S,
                         nullptr, nullptr, nullptr, nullptr, nullptr, 0, w.lw + (size_t)n * CW,
                         w.gk + (size_t)n * CW};
    if (BIG && w.ndense[n] > 0) {
        pc.dpos = w.dpos + (size_t)n * CW;
        pc.dref = w.dref + (size_t)n * C;
        pc.dka = w.dka + (size_t)n * C * dense_pitch(C);
        pc.dkb = w.dkb + (size_t)n * C * dense_pitch(C);
        pc.dkq = w.dkq + (size_t)n * C * dense_pitch(C);
        pc.nd = w.ndense[n];
    }
    const int nsmp = BIG ? (nw + kSampleStep - 1) / kSampleStep : 0;
    if (BIG)
        for (int i = tid; i < nsmp; i += NTR) smp[i] = srt[(size_t)i * kSampleStep];
    const int per = (nw + nrb - 1) / nrb;
    const int pos0 = rb * per, pos1 = pos0 + per < nw ? pos0 + per : nw;
    p1_weights<WT, false>(pc, pos0, pos1, tid, NTR);
    __syncthreads();
    const int t0 = rb * KR, t1 = t0 + KR < C ? t0 + KR : C;
    const int r1 = (t1 < nv ? t1 : nv) * R;
    p1_reads<WT, BIG>(pc, t0 * R < r1 ? t0 * R : r1, r1, tid, NTR, smp, nsmp);
    __syncthreads();
    p1_gram<WT, BIG ? 4 : 1, true>(pc, t0, t1, warp, NTR / 32, lane, rows + warp * kMaxChunk,
                                   BIG ? drows + warp * 3 * kMaxChunk : nullptr);
}

// The dense groups' part of A and QK, after k_phase1_rows wrote the pair sums of the other
// groups: A[t][u] += sum_h dka[t][h] dkb[u][h] for u < t and QK[t][u] += sum_h dkq[t][h]
// dkb[u][h] for u <= t, h ascending (one fused multiply-add chain per element, so each element
// is a fixed-order sum). One CTA per 64 x 64 tile on or below the diagonal of a chunk; 256
// threads, 4 x 4 elements of both products each, the factors staged 16 columns at a time.
constexpr int GDT = 64, GDK = 16;

__global__ void __launch_bounds__(256) k_gram_dense(Dims d, Work w) {
    __shared__ __align__(16) float sa[GDK][GDT + 4];
    __shared__ __align__(16) float sq[GDK][GDT + 4];
    __shared__ __align__(16) float sb[GDK][GDT + 4];
    const int n = blockIdx.y;
    const int nd = w.ndense[n];
    if (nd == 0) return;
    const int C = d.C, dp = dense_pitch(C), hp = (nd + 3) & ~3;
    int ti = 0, rem = blockIdx.x;        // tile (ti, ui), ui <= ti, row-major over the triangle
    while (rem > ti) { rem -= ti + 1; ++ti; }
    const int t0 = ti * GDT, u0 = rem * GDT;
    const size_t fo = (size_t)n * C * dp;
    const float *ka = w.dka + fo, *kb = w.dkb + fo, *kq = w.dkq + fo;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int lr = tid >> 2, lk = (tid & 3) * 4;   // the element group this thread stages
    float accA[4][4], accQ[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) { accA[i][j] = 0.f; accQ[i][j] = 0.f; }
    for (int k0 = 0; k0 < hp; k0 += GDK) {
        const int k = k0 + lk;
        float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vq = va, vb = va;
        if (k < hp) {                    // hp and k are multiples of 4: the float4 is inside
            if (t0 + lr < C) {
                va = *reinterpret_cast<const float4 *>(ka + (size_t)(t0 + lr) * dp + k);
                vq = *reinterpret_cast<const float4 *>(kq + (size_t)(t0 + lr) * dp + k);
            }
            if (u0 + lr < C) vb = *reinterpret_cast<const float4 *>(kb + (size_t)(u0 + lr) * dp + k);
        }
        __syncthreads();
        sa[lk][lr] = va.x; sa[lk + 1][lr] = va.y; sa[lk + 2][lr] = va.z; sa[lk + 3][lr] = va.w;
        sq[lk][lr] = vq.x; sq[lk + 1][lr] = vq.y; sq[lk + 2][lr] = vq.z; sq[lk + 3][lr] = vq.w;
        sb[lk][lr] = vb.x; sb[lk + 1][lr] = vb.y; sb[lk + 2][lr] = vb.z; sb[lk + 3][lr] = vb.w;
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GDK; ++kk) {
            const float4 a4 = *reinterpret_cast<const float4 *>(&sa[kk][ty * 4]);
            const float4 q4 = *reinterpret_cast<const float4 *>(&sq[kk][ty * 4]);
            const float4 b4 = *reinterpret_cast<const float4 *>(&sb[kk][tx * 4]);
            const float a[4] = {a4.x, a4.y, a4.z, a4.w}, q[4] = {q4.x, q4.y, q4.z, q4.w};
            const float b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    accA[i][j] = fmaf(a[i], b[j], accA[i][j]);
                    accQ[i][j] = fmaf(q[i], b[j], accQ[i][j]);
                }
        }
    }
    float *A = w.A + (size_t)n * C * C, *QK = w.QK + (size_t)n * C * C;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= C) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int u = u0 + tx * 4 + j;
            if (u > t || u >= C) continue;
            if (u < t) A[(size_t)t * C + u] += accA[i][j];
            QK[(size_t)t * C + u] += accQ[i][j];
        }
    }
}

}  // namespace

size_t phase1_scratch_smem(const Dims &d) {
    const size_t CW = (size_t)d.C * d.W, CR = (size_t)d.C * d.R;
    return ((sizeof(P1Smem) + 15) & ~size_t(15)) + 8 * 2 * CW + 4 * 6 * CW + 4 * 2 * CR +
           4 * (CW + 4);   // + the group starts
}

bool phase1_split(const Dims &d) { return phase1_scratch_smem(d) > kPhase1SmemMax; }

namespace {
void launch_rows(void (*kern)(Dims, Inputs, Work, int), bool big, dim3 grid, const Dims &d,
                 const Inputs &in, const Work &w, int step0, cudaStream_t st) {
    const size_t smem = rows_smem(big);
    set_kernel_smem(kern, smem);
    kern<<<grid, NTR, smem, st>>>(d, in, w, step0);
}
}  // namespace

bool dense_gram(const Dims &d) { return phase1_split(d) && d.C >= kDenseMinChunk; }

cudaError_t launch_phase1(const Dims &d, const Inputs &in, const Work &w, int step0, int nsteps,
                          cudaStream_t st) {
    const size_t full = phase1_scratch_smem(d);
    const int in_smem = full <= kPhase1SmemMax ? 1 : 0;
    const size_t smem = in_smem ? full : ((sizeof(P1Smem) + 15) & ~size_t(15)) + sizeof(P1Big);
    const int grid = w.G;
    const dim3 rows_grid((d.C + KR - 1) / KR, nsteps * d.P);
    const bool big = dense_gram(d);
    if (d.dtype == SDM_BF16) {
        auto kern = k_phase1<__nv_bfloat16>;
        set_kernel_smem(kern, smem);
        kern<<<grid, NT, smem, st>>>(d, in, w, step0, nsteps, in_smem);
        if (!in_smem) launch_rows(big ? k_phase1_rows<__nv_bfloat16, true>
                                      : k_phase1_rows<__nv_bfloat16, false>,
                                  big, rows_grid, d, in, w, step0, st);
    } else {
        auto kern = k_phase1<float>;
        set_kernel_smem(kern, smem);
        kern<<<grid, NT, smem, st>>>(d, in, w, step0, nsteps, in_smem);
        if (!in_smem) launch_rows(big ? k_phase1_rows<float, true> : k_phase1_rows<float, false>,
                                  big, rows_grid, d, in, w, step0, st);
    }
    if (dense_gram(d)) {
        const int nt = (d.C + GDT - 1) / GDT;
        k_gram_dense<<<dim3(nt * (nt + 1) / 2, nsteps * d.P), 256, 0, st>>>(d, w);
    }
    return cudaGetLastError();
}

}  // namespace sdm
