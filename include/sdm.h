/*
 * sdm.h -- C ABI of libsdm.so, the GB300 (sm_103a) chunked sparse-delta-memory (SDM)
 * write/read.
 *
 * The operation (sparse-delta-memory 2.0.0, memory_ops.py: the SDMWriteRead docstring's
 * token loop and the module docstring's chunked form). P parallel streams of T tokens each
 * advance their own bank of S rows x D columns. Per token t of stream p, in order:
 *
 *     a_j    = B[s_j]                 j = 0..W-1, the token's W distinct write slots
 *     d_j    = exp(g_j) * a_j         only the written rows decay
 *     ret    = sum_j k_j * d_j        retrieved
 *     u      = beta * (v - ret)       delta_v
 *     B[s_j] = d_j + k_j * u          decay-and-write
 *     o      = sum_i q_i * B[r_i]     readings over the R read slots, after the write
 *
 * The library computes it in chunks of C tokens (Phase 1: per-slot log-decays, the dedup
 * plan, gather weights and the Gram matrices A and QK; the WY solve X = (I + tril(beta A,
 * -1))^-1, QX = QK X; Phase 2: Nt = ceil(T / C) sequential steps of gather, dual matmul and
 * decay-and-write), which reproduces the token loop up to floating-point rounding.
 *
 * Conventions shared by every entry point
 *   - Pointers named "device" are CUDA device pointers on the current device; "host" ones
 *     are ordinary host memory. The caller owns every buffer and the stream.
 *   - The library never allocates memory and never synchronizes, except where an entry
 *     point says so (sdm_get_device_status).
 *   - Arrays are dense row-major with the shapes given. "bank dtype" means float32
 *     (SDM_F32) or bfloat16 (SDM_BF16) elements, as set in sdm_shape.bank_dtype.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).
 *   - Every argument is checked before any work is queued; a refused call returns a
 *     negative sdm_status, queues nothing, and sdm_last_error() describes the reason.
 *   - Results are bitwise reproducible for fixed inputs, shape and GPU type: every bank
 *     row has one writer per step and every sum runs in a fixed order.
 */
#ifndef SDM_H
#define SDM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SDM_OK = 0,
    SDM_ERR_INVALID = -1,      /* bad argument: null pointer, size out of range */
    SDM_ERR_UNSUPPORTED = -2,  /* valid but not built: e.g. a head_dim without a kernel */
    SDM_ERR_CUDA = -3,         /* a CUDA runtime call failed (message in sdm_last_error) */
    SDM_ERR_TIMEOUT = -4,      /* device status: a bounded device-side wait gave up */
    SDM_ERR_WORKSPACE = -5,    /* workspace null, too small or not 256-byte aligned */
    SDM_ERR_DEVICE = -6        /* the device reported bad input (sdm_get_device_status) */
} sdm_status;

typedef enum { SDM_F32 = 0, SDM_BF16 = 1 } sdm_dtype;

/* Shape of one call (memory_ops.py, _Layout: P, T, C, Nt, W, R, head_dim).
 *   P  parallel streams, >= 1
 *   T  tokens per stream, >= 1
 *   C  chunk size, 16..256 (the pages' MIN_CHUNK..MAX_CHUNK)
 *   S  bank rows per stream, 1..2^31-1; stream p owns bank rows [p*S, (p+1)*S)
 *   D  columns per row (head_dim): 32, 64, 128, 256 or 512
 *   W  write slots per token, 1..256 (MAX_WIDTH); distinct within a token
 *   R  read slots per token, 1..256
 *   bank_dtype  SDM_F32 or SDM_BF16
 *   slab_steps  Phase-2 steps whose Phase-1 state is held at once; 0 = automatic: every
 *               step when the state of all of them fits in 256 MiB, else as many as fit but
 *               at least two chunks per SM (ceil(304 / P) steps), so the workspace does not
 *               grow with T. The results do not depend on it (Phase 1 and the solve are per
 *               chunk).
 *   flags       0, or any of SDM_FLAG_PER_STEP_KERNELS, SDM_FLAG_SNAPSHOT_BF16 or
 *               SDM_FLAG_SNAPSHOT_FP8, SDM_FLAG_TOKEN_GATE, SDM_FLAG_SHARED_BANK
 * P * ceil(T / C) * C must be below 2^31.
 *
 * Phase 2 runs as one persistent kernel per slab in which each CTA owns one stream and one
 * 16-byte slice of bank columns for all the slab's steps (the forward acts on every column
 * independently once Phase 1 and the solve are done), when two steps of its per-chunk
 * metadata fit in shared memory (about C * (W + R) <= 4K entries); otherwise, or with
 * SDM_FLAG_PER_STEP_KERNELS, as three kernels per step (gather, dual matmul, DW over all
 * streams), as the pages lay it out. Both are deterministic; their results differ only by
 * rounding. */
#define SDM_FLAG_PER_STEP_KERNELS 1
/* Snapshot of the saving forward in bfloat16 (memory_ops.py sdm_write_read: snapshot_quant
 * "bf16"; phase2_kernels.py SNAPSHOT_QUANT_MODES). On a float32 bank the saving forward stores
 * every snapshot row rounded to bfloat16 (to nearest even), which halves sdm_saved_bytes, and
 * the backward restores each written row to that rounded value and computes the gradients
 * from it: rows written by the call end at bf16(initial value) instead of their exact initial
 * value. On a bfloat16 bank the snapshot is bfloat16 already and the flag changes nothing.
 * sdm_write_read_save and sdm_write_read_backward must be given the same flag; the other
 * entry points ignore it. */
#define SDM_FLAG_SNAPSHOT_BF16 2
/* Snapshot of the saving forward in fp8 (memory_ops.py sdm_write_read: snapshot_quant "fp8";
 * phase2_kernels.py quant_row: a row of head_dim float8_e4m3fn elements, no scale). Each
 * snapshot element is the row's value (float32 for a float32 bank, the bfloat16 value for a
 * bfloat16 bank) converted to float8_e4m3fn, to nearest even, saturating at +-448 (the format
 * has no infinity), which makes sdm_saved_bytes a quarter (float32 banks) or half (bfloat16
 * banks) of the unquantized snapshot; the backward restores each written row to that rounded
 * value and computes the gradients from it. Not with SDM_FLAG_SNAPSHOT_BF16; like it, give
 * sdm_write_read_save and sdm_write_read_backward the same flag. */
#define SDM_FLAG_SNAPSHOT_FP8 16
/* One log-decay per token (memory_ops.py sdm_write_read: "g: [..., 1] per-token log-decay,
 * or [..., W] one per write"; key_weighted_decay False). log_decay is then [P, T] float32 and
 * applies to every row the token writes; the backward's grad_log_decay is [P, T], the sum of
 * the per-write gradients in write order. Every entry point takes it. */
#define SDM_FLAG_TOKEN_GATE 4
/* One bank shared by all P streams (memory_ops.py sdm_write_read: num_memory_slots 0 with
 * shared_bank=True): the bank (and the backward's grad_bank) is [S, D] instead of [P*S, D],
 * and slot ids are rows of it, in [0, S). The caller asserts that no two streams select the
 * same slot anywhere in the call; the library does not check it. With disjoint slot sets every
 * row still has one writer and the streams are independent problems, so the results are those
 * of the streams run one after another on the shared bank, and bitwise reproducible; if two
 * streams do share a slot the result is unspecified. */
#define SDM_FLAG_SHARED_BANK 8
typedef struct {
    int32_t P, T, C, S, D, W, R;
    int32_t bank_dtype;
    int32_t slab_steps;
    int32_t flags;
} sdm_shape;

/* Device status block, read by sdm_get_device_status. */
typedef struct {
    int32_t code;                  /* 0; SDM_ERR_DEVICE when a slot was out of range;
                                      SDM_ERR_TIMEOUT when a kernel's bounded wait on its own
                                      copies gave up (the kernel then returned early, and the
                                      bank and readings of the call are incomplete) */
    int32_t first_bad_token;       /* stream-major token index (p*T + t) of a bad slot, or -1 */
    int64_t bad_slots;             /* write/read entries whose slot was outside [0, S) */
    int64_t repeated_write_slots;  /* write entries repeating a slot of their own token */
} sdm_device_status;

/* Bytes of device workspace sdm_write_read needs for this shape (0 if the shape is
 * refused; sdm_last_error says why). Independent of T once T spans more steps than one
 * slab holds. */
size_t sdm_workspace_bytes(const sdm_shape *shape);

/* The chunked SDM write/read forward (memory_ops.py: sdm_write_read, no-grad call).
 *
 *   bank          device, [P*S, D] bank dtype; read and advanced in place to its final state
 *   write_slots   device, [P, T, W] int32, per-stream slot ids in [0, S), distinct per token
 *   write_w       device, [P, T, W] bank dtype, write weights k
 *   log_decay     device, [P, T, W] float32, g (one log-decay per write entry); [P, T]
 *                 with SDM_FLAG_TOKEN_GATE (one per token)
 *   beta          device, [P, T]    float32, write strength
 *   v             device, [P, T, D] bank dtype, values
 *   read_slots    device, [P, T, R] int32, slot ids in [0, S)
 *   read_w        device, [P, T, R] bank dtype, read weights q
 *   valid_tokens  device, [P] int32 in [0, T] (values outside are clamped to it), or NULL
 *                 for all T. Tokens t >= valid[p] are
 *                 padding: they touch no bank row, their inputs are never read, and their
 *                 readings rows are zero.
 *   readings      device, [P, T, D] bank dtype, written (every row)
 *   workspace     device, >= sdm_workspace_bytes(shape) bytes, 256-byte aligned; its
 *                 contents need no initialization and are scratch after the call
 *   stream        cudaStream_t the work is queued on
 *
 * Returns SDM_OK once the work is queued (asynchronous). A slot outside [0, S) is not
 * dereferenced: the entry is dropped, and the device status (sdm_get_device_status) reports
 * SDM_ERR_DEVICE; repeated write slots in a token are counted there (results for such a
 * token are unspecified). The bank, readings and inputs must not overlap; bank, v and
 * readings must be 16-byte aligned (SDM_ERR_INVALID otherwise). */
int sdm_write_read(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                   const void *write_w, const float *log_decay, const float *beta,
                   const void *v, const int32_t *read_slots, const void *read_w,
                   const int32_t *valid_tokens, void *readings, void *workspace,
                   size_t workspace_bytes, void *stream);

/* Bytes of the snapshot a saving forward keeps for the backward: the pre-write (chunk
 * start) row of every written slot of every chunk, Nt * P * C * W rows of D bank-dtype
 * elements (memory_ops.py: the snapshot of the saving forward, snapshot_quant "none"), of
 * D bfloat16 elements with SDM_FLAG_SNAPSHOT_BF16 (snapshot_quant "bf16"), or of D one-byte
 * float8_e4m3fn elements with SDM_FLAG_SNAPSHOT_FP8 (snapshot_quant "fp8"). */
size_t sdm_saved_bytes(const sdm_shape *shape);

/* The saving forward (memory_ops.py SDMWriteRead.forward): sdm_write_read plus the snapshot.
 * saved: device, >= sdm_saved_bytes(shape) bytes, 16-byte aligned, written (positions of
 * slots that are not written stay untouched). Same results as sdm_write_read. */
int sdm_write_read_save(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                        const void *write_w, const float *log_decay, const float *beta,
                        const void *v, const int32_t *read_slots, const void *read_w,
                        const int32_t *valid_tokens, void *readings, void *saved,
                        size_t saved_bytes, void *workspace, size_t workspace_bytes,
                        void *stream);

/* Bytes of device workspace sdm_write_read_backward needs (0 if refused). */
size_t sdm_backward_workspace_bytes(const sdm_shape *shape);

/* The backward (memory_ops.py SDMWriteRead.backward: the steps in reverse, the matmuls
 * through the solve and the Phase-1 backward), after sdm_write_read_save with the same shape
 * and inputs.
 *   bank           device [P*S, D]: in, the final bank the saving forward left; out, the
 *                  initial bank, restored exactly from the snapshot (with
 *                  SDM_FLAG_SNAPSHOT_BF16 on a float32 bank: every row a valid token writes
 *                  holds bf16(its initial value), the others their exact initial value)
 *   inputs         the forward's inputs, unchanged
 *   saved          the snapshot written by sdm_write_read_save
 *   grad_readings  device [P, T, D] bank dtype: dL/d(readings) (padding rows are ignored)
 *   grad_bank      device [P*S, D] float32, in place: in, dL/d(final bank) (zero if the loss
 *                  does not read the final bank); out, dL/d(initial bank)
 *   grad_v         device [P, T, D] float32, out
 *   grad_beta      device [P, T] float32, out
 *   grad_write_w   device [P, T, W] float32, out   (dL/dk)
 *   grad_log_decay device [P, T, W] float32, out   (dL/dg; [P, T] with SDM_FLAG_TOKEN_GATE)
 *   grad_read_w    device [P, T, R] float32, out   (dL/dq)
 * Gradients of padding tokens are zero. Asynchronous; deterministic. */
int sdm_write_read_backward(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                            const void *write_w, const float *log_decay, const float *beta,
                            const void *v, const int32_t *read_slots, const void *read_w,
                            const int32_t *valid_tokens, const void *saved, size_t saved_bytes,
                            const void *grad_readings, float *grad_bank, float *grad_v,
                            float *grad_beta, float *grad_write_w, float *grad_log_decay,
                            float *grad_read_w, void *workspace, size_t workspace_bytes,
                            void *stream);

/* Kernel families, in launch order within a slab: Phase 1 and the solve once per slab, then
 * the fused Phase-2 kernel once per slab, or (SDM_FLAG_PER_STEP_KERNELS) gather, dual matmul
 * and DW once per step. */
enum {
    SDM_KERNEL_PHASE1 = 0,
    SDM_KERNEL_SOLVE = 1,
    SDM_KERNEL_GATHER = 2,
    SDM_KERNEL_DUALMM = 3,
    SDM_KERNEL_DW = 4,
    SDM_KERNEL_PHASE2 = 5,   /* the fused Phase-2 kernel (gather + dual matmul + DW) */
    SDM_KERNEL_KINDS = 6
};

/* sdm_write_read with a CUDA event recorded before every kernel launch and after the last,
 * for per-kernel device times (same arguments and results). kernel_ms and launches are host
 * arrays of SDM_KERNEL_KINDS entries: the summed milliseconds between a launch's event and
 * the next one, and the launch count, of each kernel family. Creates and destroys its own
 * events and synchronizes the stream before returning: a measuring tool, not for CUDA graph
 * capture. */
int sdm_profile_write_read(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                           const void *write_w, const float *log_decay, const float *beta,
                           const void *v, const int32_t *read_slots, const void *read_w,
                           const int32_t *valid_tokens, void *readings, void *workspace,
                           size_t workspace_bytes, float *kernel_ms, int32_t *launches,
                           void *stream);

/* Phase 1 and the solve only, for every chunk of the call, with their outputs copied to
 * caller buffers (all device, float32 unless noted; N = P * ceil(T / C) chunks, chunk
 * n = ti * P + p is chunk ti of stream p, i.e. time-major as in phase2_kernels.py):
 *   perm        [N, C*W] int32   entry index e = t*W + j at each position of the chunk's
 *                                sorted write row (sorted by (slot, e)); -1 past the valid
 *                                entries
 *   group_start [N, C*W] uint8   1 where a group (a run of one slot) begins
 *   owner       [N, C*W] uint8   1 at the last entry of a group (the group's writer)
 *   ngroups     [N]      int32   groups (distinct written slots) of the chunk
 *   lw, gw, dw  [N, C*W]         per write entry, token-major: running log-decay of its
 *                                slot (inclusive), gather weight k*exp(lw), DW weight
 *                                k*exp(lend - lw)
 *   lr, qw      [N, C*R]         per read entry: running log-decay of its slot at its token,
 *                                gather weight q*exp(lr)
 *   A, QK, X, QX [N, C, C]       Gram matrices and the solve (X unit lower triangular, +0
 *                                above the diagonal; QX = QK X)
 *   dense_groups [N]     int32   groups of the chunk whose Gram pair sums were taken in the
 *                                dense factor form (0 where the chunk's scratch is on chip)
 * Any output pointer may be NULL (not copied). The workspace is the one sdm_write_read
 * takes for the same shape. The bank is not touched. */
int sdm_phase1_debug(const sdm_shape *shape, const int32_t *write_slots, const void *write_w,
                     const float *log_decay, const float *beta, const int32_t *read_slots,
                     const void *read_w, const int32_t *valid_tokens, int32_t *perm,
                     uint8_t *group_start, uint8_t *owner, int32_t *ngroups, float *lw,
                     float *gw, float *dw, float *lr, float *qw, float *A, float *QK, float *X,
                     float *QX, int32_t *dense_groups, void *workspace, size_t workspace_bytes,
                     void *stream);

/* Reads the device status block of the last call that used this workspace. Synchronizes
 * the stream. status: host pointer. Returns SDM_OK, or SDM_ERR_CUDA. The block's code is
 * SDM_ERR_DEVICE for a slot outside [0, S), or SDM_ERR_TIMEOUT when a kernel's bounded wait
 * for its own copies gave up (see sdm_set_wait_limit); the call's results are then
 * incomplete. */
int sdm_get_device_status(const void *workspace, sdm_device_status *status, void *stream);

/* Bytes of device workspace sdm_write_read_host needs: the sdm_write_read workspace plus a
 * device copy of the inputs (0 if the shape is refused). */
size_t sdm_host_workspace_bytes(const sdm_shape *shape);

/* The forward with its inputs and readings in host memory: what sdm_write_read computes, for a
 * caller whose data lives on the host (the sparse-delta-memory 2.0.0 memory_ops.py
 * sdm_write_read call with CPU tensors). The pages have no host-side variant; this one exists
 * so that one call covers the whole path including the transfers.
 *   - bank: device memory, advanced in place as in sdm_write_read.
 *   - write_slots ... valid_tokens: host memory, same layouts as sdm_write_read (valid_tokens
 *     may be NULL). Page-locked (pinned) memory lets the copies run asynchronously.
 *   - readings: page-locked host memory mapped into the device address space (cudaHostAlloc /
 *     cudaMallocHost, or cudaHostRegister with cudaHostRegisterMapped), [P, T, D] in the bank
 *     dtype, 16-byte aligned. The Phase-2 kernels store the readings straight into it; it is
 *     complete when the call's work on `stream` has finished. Other memory is refused with
 *     SDM_ERR_INVALID before any work.
 *   - workspace: device memory of at least sdm_host_workspace_bytes(shape) bytes, 256-byte
 *     aligned; it holds the device copy of the inputs.
 * The inputs other than v are copied on `stream` before Phase 1 (by one kernel reading the host
 * pages when all of them are mapped page-locked memory, else by one transfer each); v is copied
 * on a second, library-owned stream (created once per device) and joined before Phase 2, so
 * that its copy runs under Phase 1 and the solve. All work is ordered after the previous work on `stream` and
 * before later work on it; the call is asynchronous and may be captured in a CUDA graph. */
int sdm_write_read_host(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                        const void *write_w, const float *log_decay, const float *beta,
                        const void *v, const int32_t *read_slots, const void *read_w,
                        const int32_t *valid_tokens, void *readings, void *workspace,
                        size_t workspace_bytes, void *stream);

/* Number of kernel launches sdm_write_read queues for this shape (0 if refused). */
int64_t sdm_launch_count(const sdm_shape *shape);

/* Bytes of the static device scratch sdm_write_read_noalloc uses (16 MiB per GPU). */
#define SDM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* sdm_write_read for callers that cannot allocate device memory. The pages have no
 * counterpart: this entry point serves hosts that own every byte of device memory (an engine
 * or plugin host with its own pool, or a fixed-footprint or real-time service) and cannot call
 * cudaMalloc, or do not want to, as cudaMalloc may synchronize the device. Instead of a caller
 * workspace it uses one static device array of SDM_NOALLOC_SCRATCH_BYTES that lives in the
 * library; once loaded on a GPU it stays reserved there until the process exits. The caller
 * still provides the bank, the inputs and the readings (same arguments, layouts and results as
 * sdm_write_read, without workspace).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress, on the current
 *     device). Under the CUDA driver's lazy module loading (the default) the first lookup on
 *     a device is when the driver loads the array and reserves its 16 MiB there, and that
 *     load can fail like an allocation (SDM_ERR_CUDA). Make the first call at initialization
 *     time, and before any CUDA stream capture.
 *   - Phase-2 slabs are sized to fit the array (results do not depend on the slab size). A
 *     shape that does not fit even at one step per slab, or an explicit slab_steps that does
 *     not fit, is refused with SDM_ERR_WORKSPACE before any work.
 *   - Every call shares the one array, which keeps the last call's contents; the call clears
 *     what must start at zero itself. Calls whose work overlaps on the GPU (other streams,
 *     other host threads) race on the array: serialize them.
 *   - The device status of the last such call is read with sdm_noalloc_get_device_status
 *     (slots outside [0, S) are never dereferenced). */
int sdm_write_read_noalloc(const sdm_shape *shape, void *bank, const int32_t *write_slots,
                           const void *write_w, const float *log_decay, const float *beta,
                           const void *v, const int32_t *read_slots, const void *read_w,
                           const int32_t *valid_tokens, void *readings, void *stream);

/* The device status block of the last sdm_write_read_noalloc call on the current device (it
 * sits at the start of the static array). Synchronizes the stream. status: host pointer.
 * Returns SDM_OK, SDM_ERR_INVALID (status NULL) or SDM_ERR_CUDA. No counterpart on the pages. */
int sdm_noalloc_get_device_status(sdm_device_status *status, void *stream);

/* ---------------------------------------------------------------------------------------
 * Layer I/O around the write/read (memory_ops.py, "Layer I/O: head split / merge and the
 * per-batch bank expand"). All pointers are device pointers on the current device, dtype is
 * SDM_F32 or SDM_BF16, and the work is queued on stream (asynchronous). Each call returns
 * SDM_OK, or a negative sdm_status for a NULL pointer, bad sizes or a bad dtype (nothing
 * queued). Deterministic; the copies are bitwise.
 * --------------------------------------------------------------------------------------- */

/* Head split, rearrange 'b t (h k) -> (b h) t k': src [B, T, H*CD] -> dst [B*H, T, CD], i.e.
 * dst row (b*H + h)*T + t = src row (b*T + t)*H + h (rows of CD elements). src and dst must not
 * overlap. */
int sdm_head_split(const void *src, void *dst, int B, int T, int H, int CD, int dtype,
                   void *stream);

/* Head merge, the inverse: src [B*H, T, CD] -> dst [B, T, H*CD]. */
int sdm_head_merge(const void *src, void *dst, int B, int T, int H, int CD, int dtype,
                   void *stream);

/* Per-batch bank expand: out [B, S, D] = B copies of param [S, D] (the learned bank each
 * batch element starts from). */
int sdm_bank_expand(const void *param, void *out, int B, long long S, int D, int dtype,
                    void *stream);

/* Its adjoint: out [S, D] = sum over b of x [B, S, D], accumulated in float32 in batch order
 * and rounded once to the dtype (the gradient of the shared parameter bank). B >= 1. */
int sdm_bank_sum(const void *x, void *out, int B, long long S, int D, int dtype, void *stream);

/* ---------------------------------------------------------------------------------------
 * Product-key exact top-k, the slot selection upstream of the write/read
 * (product_key_topk.py: the product_key_topk docstring). A row of raw holds F factors side by
 * side (widths factors[0..F-1]); slot (c_0, .., c_{F-1}) scores the float32 sum of its factor
 * values in factor order (with bfloat16 input and F > 2 each partial sum rounded to bfloat16
 * before the next factor is added) and has index lin = (..(c_0 w_1 + c_1) w_2 ..) w_{F-1} +
 * c_{F-1}. Scores compare as float32, -0 below +0, NaN as -inf. Each factor is ranked by value
 * (larger column first on ties); stage 0 keeps the first min(k, w_0) ranks; stage f keeps the
 * best c = min(k, n m) pairs (i, j) of the previous stage's n ranks and the first
 * m = min(k, w_f) ranks of factor f with (i + 1)(j + 1) <= c, exact ties to the larger i + j,
 * then the larger i. With bfloat16 input and F > 2 an intermediate stage compares the rounded
 * partial sum it passes on. The kept kk = min(k, prod(factors)) slots are returned sorted by
 * lin, with val = the score rounded to the input dtype. Deterministic.
 *   raw      device [rows, sum(factors)], dtype SDM_F32 or SDM_BF16
 *   factors  host [F], 1 <= F <= 4, each width 1..4096
 *   k        1..256
 *   val      device [rows, kk], dtype
 *   lin      device [rows, kk] int64
 * Returns SDM_OK once queued on stream, or a negative sdm_status (nothing queued). */
int sdm_product_key_topk(const void *raw, long long rows, const int *factors, int F, int k,
                         int dtype, void *val, int64_t *lin, void *stream);

/* Its backward: grad_raw [rows, sum(factors)] float32 (device, written whole) =
 * the gradient of val reaching each factor column of each selected slot, added in output
 * order (the rounding of partial sums passes it unchanged). lin and grad_val [rows, kk] as the
 * forward returned / takes them (grad_val in dtype); factors, F and k as in the forward. */
int sdm_product_key_topk_backward(const int64_t *lin, const void *grad_val, long long rows,
                                  const int *factors, int F, int k, int dtype, float *grad_raw,
                                  void *stream);

/* Testing aid: the number of polls after which a kernel's bounded wait for its own bulk copies
 * gives up (default 2^22, seconds at most), for calls queued after this one, process-wide;
 * polls < 1 restores the default. A kernel whose wait gives up sets SDM_ERR_TIMEOUT in the
 * device status, waits (with the default limit) for the copies it has in flight, and returns
 * early, leaving that call's bank and readings incomplete. Returns the previous limit. The
 * pages have no counterpart: this exists so that the give-up path can be exercised without
 * a fault. */
long long sdm_set_wait_limit(long long polls);

/* Thread-local description of the last refused call or CUDA error ("" if none). */
const char *sdm_last_error(void);

/* Library version string. */
const char *sdm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDM_H */
