/*
 * invrope.h -- C ABI of the GB300 (sm_103a) inverse-RoPE + VHA postmix
 * library and its sparse-attention KV index remap.
 *
 * The operations are those of PaddleFleet pull request #1772, "Fuse HCA
 * inverse RoPE into the VHA postmix, and the sparse-attention KV index
 * remap" (cited below as [PR1772]):
 *
 *   [PR1772] English description, item 1 (fuse_inv_rope_into_vha_postmix):
 *     the HCA inverse RoPE rotates back only the trailing pe channels of each
 *     head of the attention output, and the ungrouped VHA postmix is an
 *     [nh, nh] GEMM over the head axis. The channel axis is therefore a pure
 *     N dimension and no full-width inv_rope(O) is needed.
 *   [PR1772] Chinese description, section 1: the weight gradient
 *     dM[h, h'] = sum_{t,c} dOut[t,h,c] * O_roped[t,h',c] over all tokens and
 *     the full channel axis.
 *   [PR1772] revision note: the input gradient is the postmix GEMM's input
 *     gradient pushed back through the rotation.
 *   [PR1772] English item 2 / Chinese section 2
 *     (sparse_attn_global_kv_idx_remap_fusion): per-batch-local -> flat-global
 *     KV column remap idx + b * seqlen_kv over a [b*sq, topk] table.
 *
 * Notation (all tensors dense, row-major, last index fastest):
 *   O, Y, dY, dO : bf16 [sq, nh, d], d = nope + pe, channel fastest.
 *   M, dM        : fp32 [nh, nh], row-major; Y[s,g,:] = sum_h M[g,h] X[s,h,:].
 *   positions    : row s sits at absolute position p = pos0 + s.
 *   rotary pairs : rotate-half, pair i = (nope+i, nope+i+pe/2), i < pe/2,
 *                  frequency f_i = theta^(-2i/pe), angle a = p * f_i.
 *   invrope      : (x1, x2) -> (x1 cos a + x2 sin a, x2 cos a - x1 sin a).
 *   rope         : (x1, x2) -> (x1 cos a - x2 sin a, x2 cos a + x1 sin a).
 *
 * Common contract of every call below:
 *   - Pointers are DEVICE pointers of the current CUDA device, owned by the
 *     caller. The library allocates no device memory at call time. Between
 *     calls it keeps cached device attributes and host-side caches, its
 *     loaded kernels, and library-owned device arrays that exist from module
 *     load until the process exits:
 *       . two arrays of 512 work-counter slots (8 KB each) for the forward
 *         and the remap, which hand out their work dynamically (thread blocks
 *         claim the next tile or chunk from their launch's slot);
 *       . the 8 MiB scratch array of invrope_postmix_bwd_noalloc (see there
 *         for how calls share it and must be ordered).
 *     Work-counter slots: a forward launch with at most two tiles per
 *     thread block, or a remap with no more chunks than thread blocks,
 *     claims nothing and takes no slot. Otherwise an eager launch takes the
 *     next of 256 slots in turn, a launch made while its stream is being captured into a CUDA
 *     graph the next of 256 other slots, which it keeps on every replay. A
 *     launch's thread blocks take their slot only when it is free or held by
 *     their own launch; the last block frees it. A launch that finds its
 *     slot held by another launch still running (more than 256 eager
 *     launches in flight at once, or two concurrent replays of captured
 *     launches that share a slot) claims nothing from it, records
 *     INVROPE_FAULT_SCHED_BUSY_FWD or _REMAP (see invrope_take_device_fault)
 *     and leaves its outputs undefined; it never disturbs the other launch.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Every call
 *     only enqueues work on `stream` and returns; nothing synchronises.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     rejected call enqueues nothing and returns a non-zero status.
 *   - A launch failure returns INVROPE_ERR_CUDA (the CUDA error is left for
 *     cudaGetLastError / invrope_last_cuda_error).
 *   - Kernel waits are bounded: a wait that runs out (about two seconds)
 *     records a fault code that invrope_take_device_fault() returns, and the
 *     kernel exits early instead of hanging. Outputs are then undefined.
 *   - The device must be compute capability 10.3 (GB300, sm_103a);
 *     otherwise calls return INVROPE_ERR_DEVICE.
 */
#ifndef INVROPE_H_
#define INVROPE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t == struct CUstream_st* */

typedef enum invrope_status {
  INVROPE_OK = 0,
  INVROPE_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, overlap */
  INVROPE_ERR_UNSUPPORTED = 2, /* valid shape outside what the kernels cover   */
  INVROPE_ERR_WORKSPACE = 3,   /* workspace missing or too small               */
  INVROPE_ERR_CUDA = 4,        /* a CUDA runtime / launch error                */
  INVROPE_ERR_DEVICE = 5       /* current device is not sm_103 (GB300)         */
} invrope_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* invrope_status_string(int status);

/* The last CUDA error code seen by the library on this thread (0 = none). */
int invrope_last_cuda_error(void);

/*
 * Forward of the fused inverse RoPE + ungrouped VHA postmix
 * ([PR1772] English item 1, Chinese section 1):
 *
 *   Y[s, g, :] = sum_h M[g, h] * invrope_{pos0+s}(O[s, h, :])
 *
 * O  : bf16 [sq, nh, d], input, 16-byte aligned.
 * M  : fp32 [nh, nh] row-major, input, 4-byte aligned.
 * Y  : bf16 [sq, nh, d], output (fully overwritten), 16-byte aligned; must
 *      not overlap O or M.
 * sq : rows (>= 0; 0 enqueues nothing). sq * nh must be < 2^31.
 * nh : heads, 1..128.
 * nope, pe : leading unrotated / trailing rotated channels; pe even >= 2,
 *      nope >= 0, d = nope + pe a multiple of 8. The pe channels must lie in
 *      one 64-channel-aligned block (nope / 64 == (d - 1) / 64), which holds
 *      for every DeepSeek-style split with pe <= 64 such as 448 + 64;
 *      otherwise INVROPE_ERR_UNSUPPORTED.
 * pos0 : absolute position of row 0 (>= 0); theta : rotary base (> 0, finite).
 * The head mix runs on the tensor cores with M split into two bf16 terms
 * (hi + lo) and fp32 accumulation; the rotation is applied to the fp32
 * accumulator, and Y is rounded to nearest-even bf16 once.
 */
int invrope_postmix_fwd(const void* O, const float* M, void* Y,
                        int64_t sq, int nh, int nope, int pe,
                        int64_t pos0, double theta,
                        struct CUstream_st* stream);

/*
 * Workspace bytes invrope_postmix_bwd needs on the CURRENT device for this
 * shape: fp32 [nh, nh] partials of dM, one per thread block and, for shapes
 * whose thread blocks hand out the last ~10% of their tiles dynamically (the
 * production split, nh = 64 with the pe block filling one 64-channel chunk),
 * one per such tail block; so it depends on the device's SM count. At most
 * 8 MiB for nh <= 64. Returns 0 when the shape is invalid or unsupported.
 */
size_t invrope_postmix_bwd_workspace_bytes(int64_t sq, int nh, int nope, int pe);

/*
 * Backward of invrope_postmix_fwd ([PR1772] Chinese section 1 and revision
 * note), in one pass over dY and O plus a small fixed-order reduction:
 *
 *   dO[s, h, :] = rope_{pos0+s}( sum_g M[g, h] * dY[s, g, :] )   (bf16)
 *   dM[g, h]    = sum_{s, c} dY[s, g, c] * X[s, h, c],  X = invrope(O) (fp32)
 *
 * dY, O : bf16 [sq, nh, d] inputs, 16-byte aligned.
 * M     : fp32 [nh, nh] input.
 * dO    : bf16 [sq, nh, d] output (overwritten), 16-byte aligned.
 * dM    : fp32 [nh, nh] output, OVERWRITTEN (not accumulated into).
 * workspace / workspace_bytes : caller-owned device scratch of at least
 *      invrope_postmix_bwd_workspace_bytes() bytes, 16-byte aligned; its
 *      contents on entry do not matter and are clobbered.
 * Outputs must not overlap each other, the inputs or the workspace.
 * Other arguments as in invrope_postmix_fwd. sq = 0 writes dM = 0.
 * dM is bitwise identical from run to run on the same device: each
 * partial covers a fixed range of tiles accumulated in a fixed order
 * (whichever thread block runs it), and the partials are summed in a fixed
 * order (compensated fp32) without atomics. The rotated pe operand of dM is
 * split into bf16 hi + lo terms so that dM is not limited by bf16 rounding of
 * X. Shapes that hand out tail blocks take one work-counter slot (see the
 * common contract) and may record INVROPE_FAULT_SCHED_BUSY_BWD.
 */
int invrope_postmix_bwd(const void* dY, const void* O, const float* M,
                        void* dO, float* dM,
                        void* workspace, size_t workspace_bytes,
                        int64_t sq, int nh, int nope, int pe,
                        int64_t pos0, double theta,
                        struct CUstream_st* stream);

/*
 * Forward with a grouped head mix and/or per-row positions. With gs = nh and
 * positions = NULL this is exactly invrope_postmix_fwd.
 *
 *   Y[s, k*gs + i, :] = sum_j M[k, i, j] * invrope_{p(s)}(O[s, k*gs + j, :])
 *   p(s) = pos0 + (positions ? positions[s] : s)
 *
 * Grouped mix: [PR1772] Chinese section 1 lists vha_postmix_grouped among the
 *      configurations its fused path hands back to the unfused code, without
 *      spelling the grouped mix out. It is read here as ng = nh / gs groups of
 *      gs consecutive heads, each mixed by its own [gs, gs] matrix (a
 *      block-diagonal [nh, nh] mix).
 * Positions: [PR1772] English item 1 runs the shard of a context-parallel
 *      split (positions are then not 0..sq-1), and the token axis may fold
 *      several sequences (positions restart per sequence); any int32 values
 *      are accepted, negative ones included (angles are taken mod 2 pi).
 * M         : fp32 [nh/gs, gs, gs] (row-major), input.
 * gs        : heads per group, 1 <= gs <= nh, nh % gs == 0.
 * positions : int32 [sq] DEVICE array, 4-byte aligned, or NULL; pos0 is
 *             added to every entry (pos0 >= 0).
 * Other arguments, errors and rounding as in invrope_postmix_fwd.
 */
int invrope_postmix_fwd_ex(const void* O, const float* M, void* Y,
                           int64_t sq, int nh, int gs, int nope, int pe,
                           const int32_t* positions, int64_t pos0, double theta,
                           struct CUstream_st* stream);

/*
 * Backward of invrope_postmix_fwd_ex (gs = nh, positions = NULL: exactly
 * invrope_postmix_bwd):
 *
 *   dO[s, k*gs + j, :] = rope_{p(s)}( sum_i M[k, i, j] * dY[s, k*gs + i, :] )
 *   dM[k, i, j]        = sum_{s, c} dY[s, k*gs + i, c] * X[s, k*gs + j, c]
 *
 * M, dM : fp32 [nh/gs, gs, gs]; dM is overwritten. The workspace is the
 *         same as for the ungrouped call (invrope_postmix_bwd_workspace_bytes).
 * Other arguments, errors and determinism as in invrope_postmix_bwd and
 * invrope_postmix_fwd_ex; positions must not overlap an output.
 */
int invrope_postmix_bwd_ex(const void* dY, const void* O, const float* M,
                           void* dO, float* dM,
                           void* workspace, size_t workspace_bytes,
                           int64_t sq, int nh, int gs, int nope, int pe,
                           const int32_t* positions, int64_t pos0, double theta,
                           struct CUstream_st* stream);

/*
 * Size of the fixed device scratch that invrope_postmix_bwd_noalloc uses in
 * place of a workspace: 8 MiB, i.e. up to 512 dM partials at nh = 64.
 */
#define INVROPE_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * invrope_postmix_bwd without a workspace argument, for callers that may not
 * allocate device memory on their call path (no cudaMalloc, no allocating
 * library call) and have no scratch buffer to pass: e.g. a runtime whose
 * device memory is all planned ahead, or a plugin interface that hands over
 * only inputs and outputs. It is not an operation of the pages (no
 * counterpart there); it computes exactly what invrope_postmix_bwd computes,
 * with the same kernels, arguments (minus the workspace) and results.
 *
 * Scratch: a file-scope device array of INVROPE_NOALLOC_SCRATCH_BYTES that
 * the library owns. Each device that loads the library's module keeps it until
 * the process exits. The library allocates nothing at call time.
 * Limit: shapes whose backward needs more than that
 *   (invrope_postmix_bwd_workspace_bytes(sq, nh, nope, pe) > 8 MiB, e.g.
 *   nh = 128 with 152 thread blocks) are refused with INVROPE_ERR_WORKSPACE;
 *   use invrope_postmix_bwd for those.
 * First call on a device: it looks up the array's device address with
 *   cudaGetSymbolAddress (with that device current), which may load the
 *   module; make this first call before any stream capture.
 * Sharing: all calls on a device use the same array and leave their partials
 *   in it. Nothing in it needs to start at zero (each call writes every
 *   partial it reads), but calls whose work overlaps on the GPU (e.g. on two
 *   streams at once) race on the array: order them.
 */
int invrope_postmix_bwd_noalloc(const void* dY, const void* O, const float* M,
                                void* dO, float* dM,
                                int64_t sq, int nh, int nope, int pe,
                                int64_t pos0, double theta,
                                struct CUstream_st* stream);

/*
 * Per-batch-local -> flat-global sparse-attention KV column remap
 * ([PR1772] English item 2, Chinese section 2), one pass over the table:
 *
 *   out[r, k] = idx[r, k] < 0 ? idx[r, k] : idx[r, k] + (r / sq) * seqlen_kv
 *
 * idx : int32 [rows, topk] input, 4-byte aligned.
 * out : int32 [rows, topk] output; may be idx itself (in place) but must not
 *       otherwise overlap it.
 * rows = b * sq (rows % sq == 0), topk >= 0, sq >= 1, seqlen_kv >= 0, and
 * b * seqlen_kv <= 2^31 so that every in-range index (0 <= idx < seqlen_kv)
 * maps into int32. Entries >= seqlen_kv are not clamped; the add wraps in
 * 32-bit two's complement. Bit-exact; an empty table enqueues nothing.
 */
int kv_idx_local_to_global(const int32_t* idx, int32_t* out,
                           int64_t rows, int topk, int64_t sq,
                           int64_t seqlen_kv, struct CUstream_st* stream);

/*
 * The same remap on an int64 table ([PR1772]'s remap tests build their tables
 * once per index dtype):
 *
 *   out[r, k] = idx[r, k] < 0 ? idx[r, k] : idx[r, k] + (r / sq) * seqlen_kv
 *
 * idx, out : int64 [rows, topk], 8-byte aligned; out may be idx itself.
 * rows = b * sq, topk >= 0, sq >= 1, seqlen_kv >= 0, and b * seqlen_kv <= 2^63
 * so that every in-range index maps into int64. Entries >= seqlen_kv are not
 * clamped; the add wraps in 64-bit two's complement. Bit-exact.
 */
int kv_idx_local_to_global_i64(const int64_t* idx, int64_t* out,
                               int64_t rows, int topk, int64_t sq,
                               int64_t seqlen_kv, struct CUstream_st* stream);

/*
 * Synchronises the current device, then returns in *fault the fault code
 * recorded by any kernel of this library on this device since the previous
 * call (0 = none) and clears it. A non-zero code means a bounded wait ran
 * out (code = role << 8 | barrier), or a launch found its work-counter slot
 * held by another launch (INVROPE_FAULT_SCHED_BUSY_*); the outputs of the
 * launches since the previous call are then undefined. After a non-zero code
 * every work-counter slot of the device is returned to the free state (no
 * call of this library may be running on the device at that point).
 */
#define INVROPE_FAULT_SCHED_BUSY_FWD 0x5C1
#define INVROPE_FAULT_SCHED_BUSY_REMAP 0x5C2
#define INVROPE_FAULT_SCHED_BUSY_BWD 0x5C3
int invrope_take_device_fault(int* fault);

/*
 * Test hook (library infrastructure, not an operation of the pages): marks
 * the work-counter slot that the next eager slot-taking forward (which = 0:
 * more than two tiles per thread block, or a backward that hands out tail
 * blocks) or slot-taking KV remap (which = 1: more chunks than thread
 * blocks) launch on the current device will take as held by the launch
 * tag `owner` (a synchronous host-to-device copy). With a non-zero owner
 * that no launch has, that next launch must find the slot busy, record
 * INVROPE_FAULT_SCHED_BUSY_FWD / _REMAP and leave its output undefined;
 * invrope_take_device_fault() then frees the slot again. Lets a test check
 * the collision path without running two launches at once.
 */
int invrope_debug_occupy_next_slot(int which, unsigned long long owner);

/*
 * Watchdog self-test: launches one thread block whose only mbarrier wait can
 * never complete (nothing arrives on it) and whose bounded wait gives up after
 * limit_us microseconds (1000..2000000), exactly as the kernels' waits do
 * after about two seconds. Synchronises the current device before and after;
 * returns in *fault the code the watchdog recorded, which must be
 * INVROPE_WATCHDOG_SELFTEST_CODE, and leaves the flag cleared and the CUDA
 * context usable. Library infrastructure, not an operation of the pages.
 */
#define INVROPE_WATCHDOG_SELFTEST_CODE 0x60A
int invrope_watchdog_selftest(int64_t limit_us, int* fault);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* INVROPE_H_ */
