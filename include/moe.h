/*
 * moe.h - C ABI of the GB300 (sm_103a) block-batched MXFP4 mixture-of-experts layer.
 *
 * The layer is the one described on "Run Kimi 3.1 locally on one GPU"
 * (argonautlabs.ai): each MoE layer has 896 experts, 16 are selected per token
 * (section "Read the experts the router needs"); experts are MXFP4, one
 * 17,547,264-byte file per expert, and the rest of the model is Q8_0 (section
 * "One GPU, three storage tiers"); a verification block of up to 16 rows reads
 * each expert once for all its rows and its rows run the same arithmetic as
 * plain single-row steps (section "A drafter that leaves the answer
 * unchanged").  "Run Kimi K3 and K3.1 Pro Locally" (computingforgeeks.com),
 * table in "Kimi K3 and K3.1 Pro in numbers", adds the 2 shared experts.
 *
 * One layer for a block of N rows is four calls on one stream:
 *   moe_route                       router GEMV (or caller logits), top-k,
 *                                   renormalised weights, grouping by expert
 *   moe_shared_experts_after_route  the 2 shared Q8_0 experts on every row,
 *                                   beside the routing (they need x only)
 *   moe_expert_block                every selected expert's SwiGLU MLP on its
 *                                   rows (MOE_MODE_ROUTED_ONLY |
 *                                   MOE_MODE_AFTER_SHARED), each expert's
 *                                   weights streamed from HBM once per block
 *   moe_combine                     out = bf16(residual + sum_j w_j y_j +
 *                                   sum_s shared_s)
 * (moe_expert_block alone also runs the shared experts, after the routing.)
 * q8_0_block_matmul is the stand-alone Q8_0 N-row matmul; moe_cache_* is the
 * device expert cache that holds routed experts in HBM slots filled from pinned
 * host memory, and moe_nvme_* the tier below it that reads expert slabs from
 * files into pinned host memory.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer unless it is documented as a
 *   host pointer (descriptors and pools are host structs).  The block's rows and
 *   the combine's residual and output (x of moe_route and moe_shared_experts*,
 *   residual and out of moe_combine) may instead point into pinned host memory,
 *   which the device addresses directly: the kernels then read the rows and write
 *   the output in place over the host link, with no copy launches.
 * - The caller owns every buffer.  No call allocates device memory.
 * - Every compute call is asynchronous on the given stream (a cudaStream_t
 *   passed as void*; NULL means the legacy default stream) and returns a
 *   status.  Argument errors are detected on the host before any launch and
 *   return MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED with nothing enqueued.
 * - Device-side failures (a bounded wait that ran out, a NaN logit) never trap:
 *   the kernel records a bit in the workspace's error word and finishes.  Read
 *   and clear it with moe_get_error().
 * - bf16 and fp16 values are passed as their 16-bit patterns (uint16_t).
 * - moe_expert_block, moe_shared_experts and moe_combine launch with
 *   programmatic dependent launch: their kernels may be scheduled while the
 *   previous kernel on the stream is still running, and wait for it to
 *   complete before they touch memory, so stream order holds as for plain
 *   launches; only the launch and the kernels' set-up overlap.  moe_route
 *   launches plainly and lets the next kernel be scheduled at once.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef MOE_API
#define MOE_API __attribute__((visibility("default")))
#endif

/* status codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1   /* NULL / misaligned pointer, bad size */
#define MOE_ERR_UNSUPPORTED 2   /* shape, row count or device not supported */
#define MOE_ERR_CUDA 3          /* a CUDA runtime call failed */
#define MOE_ERR_TIMEOUT 4       /* device error word: a bounded wait ran out */
#define MOE_ERR_NAN 5           /* device error word: a NaN logit was seen */
#define MOE_ERR_IO 6            /* a read of the NVMe expert tier failed */

/* bits of the device error word returned by moe_get_error */
#define MOE_EBIT_TIMEOUT 0x1u
#define MOE_EBIT_NAN 0x2u
#define MOE_EBIT_BAD_SLOT 0x4u

/* moe_expert_block modes */
#define MOE_MODE_DECODE 0       /* N <= 16: one arithmetic path for every N (row results
                                   do not depend on the other rows of the block) */
#define MOE_MODE_PREFILL 1      /* any N: block-scaled tensor-core path */
#define MOE_MODE_DEBUG_GU 0x100 /* also write g and u (before SwiGLU) to the workspace */
#define MOE_MODE_SHARED_ONLY 0x200 /* only the block's shared experts (writes shared_y) */
#define MOE_MODE_ROUTED_ONLY 0x400 /* only the routed experts (writes y_part); with a
                                      SHARED_ONLY call on the same workspace this does
                                      the work of one plain call, e.g. split over two
                                      streams that join before moe_combine */
#define MOE_MODE_AFTER_SHARED 0x800 /* with MOE_MODE_ROUTED_ONLY, for the call made
                                      right after moe_shared_experts_after_route on
                                      the same stream (which itself directly follows
                                      moe_route): the routed experts' kernel does not
                                      wait for the shared experts to complete before
                                      it starts (its CTAs run only once every CTA of
                                      the shared experts has seen the routing
                                      complete), only before it completes */

#define MOE_MODE_ORDERED 0x1000 /* routed experts in the order given by the workspace's
                                   uorder array (moe_ws_offsets.uorder: int32 [U], a
                                   permutation of 0..U-1, written by the caller after
                                   moe_route): position p works on expert uexp[uorder[p]].
                                   Only the schedule changes (e.g. experts already in a
                                   device cache first, those still uploading last); every
                                   output is bit-identical to the default order */

/* weight formats of a pool */
/* bits of a slot's ready flag (moe_expert_block's slot_ready; the device expert cache
   sets them as the slab's two upload chunks land) */
#define MOE_SLOT_GATE_UP 1u     /* gate and up planes (and their scales) are in the slot */
#define MOE_SLOT_DOWN 2u        /* down planes (and scales) are in the slot */
#define MOE_SLOT_READY 3u       /* the whole slab */

#define MOE_FMT_MXFP4 0
#define MOE_FMT_Q8_0 1

/* q8_0_block_matmul epilogues and input types */
#define MOE_EPI_NONE 0          /* y  = x W^T */
#define MOE_EPI_ACCUM 1         /* y += x W^T */
#define MOE_EPI_SWIGLU 2        /* y  = silu(x Wg^T) * (x Wu^T) */
#define MOE_DTYPE_BF16 0
#define MOE_DTYPE_F32 1

/*
 * Layer shape.  d_model = hidden size d, d_ff = expert width f, n_experts = E
 * routed experts, top_k = k experts per row, group = elements per scale.
 * Kimi K3.1: {7168, 1536, 896, 16, 32}.  Requirements: group == 32,
 * 1 <= top_k <= min(n_experts, 32), n_experts <= 1024, d_model % 256 == 0,
 * d_ff % 64 == 0, d_model % 64 == 0.
 */
typedef struct moe_desc {
    int32_t d_model;
    int32_t d_ff;
    int32_t n_experts;
    int32_t top_k;
    int32_t group;
} moe_desc;

/*
 * Expert slabs resident in ONE device allocation (host struct).
 *
 * Slot s starts at base + s * slot_bytes.  A slab is the expert's three
 * matrices in this order: gate [f][d], up [f][d], down [d][f], each stored as
 * its codes plane followed by its scales plane:
 *   MXFP4: codes [rows][K/2] bytes, two E2M1 codes per byte, the even-K element
 *          in the low nibble; scales [rows][K/32] E8M0 bytes (2^(s-127)).
 *          One slab is 3*d*f*(1/2 + 1/32) bytes (17,547,264 at d=7168, f=1536,
 *          the expert file size on "Run Kimi 3.1 locally on one GPU").
 *   Q8_0:  codes [rows][K] int8; scales [rows][K/32] fp16; 3*d*f*(1 + 2/32) bytes.
 * base must be 32-byte aligned and slot_bytes a multiple of 32 that is at
 * least the slab size.  The pool is read through TMA tensor maps that the
 * library encodes on the host from these fields.
 */
typedef struct moe_pool {
    const void* base;
    int64_t slot_bytes;
    int32_t n_slots;
    int32_t format;
} moe_pool;

/* Bytes of one slab of the given format for this shape. */
MOE_API size_t moe_slab_bytes(const moe_desc* desc, int32_t format);

/*
 * Workspace.  moe_workspace_size() gives the bytes a workspace for blocks of
 * up to n_rows_max rows needs (n_shared shared experts).  The caller
 * allocates it (256-byte aligned) and must zero it once before first use
 * (cudaMemset 0); the kernels leave it in that state after every layer.  A
 * workspace serves one layer at a time: layers that run concurrently need
 * their own.  The layout is opaque; moe_workspace_offsets() exposes the
 * parts tests inspect.
 */
MOE_API size_t moe_workspace_size(const moe_desc* desc, int32_t n_rows_max, int32_t n_shared);

typedef struct moe_ws_offsets {
    int64_t error_word;   /* uint32 */
    int64_t n_unique;     /* int32 U */
    int64_t uexp;         /* int32 [U] selected experts, ascending */
    int64_t uorder;       /* int32 [E] work order of MOE_MODE_ORDERED (caller-written) */
    int64_t off;          /* int32 [U+1] */
    int64_t pair;         /* int32 [N*k] row*k + slot, grouped by expert */
    int64_t dbg_g;        /* float [pairs][f] gate projection (MOE_MODE_DEBUG_GU) */
    int64_t dbg_u;        /* float [pairs][f] up projection   (MOE_MODE_DEBUG_GU) */
    int64_t h;            /* float [pairs][f] SwiGLU activations */
    int64_t shared_y;     /* float [n_shared][N][d] shared-expert outputs */
    int64_t timeline;     /* uint64 [4][2] kernel timeline: for the routing kernel
                             (moe_route with the router GEMV), the shared-expert kernel and
                             the routed-expert kernel (in that order; the fourth pair is
                             unused) the bitwise complement of the earliest CTA start and
                             the latest CTA end (%globaltimer ns) since the caller last
                             zeroed these 64 bytes; zero = no launch yet.  Zeroing them is
                             optional (they only serve timing) and must not overlap a
                             running layer. */
} moe_ws_offsets;

MOE_API int moe_workspace_offsets(const moe_desc* desc, int32_t n_rows_max, int32_t n_shared,
                          moe_ws_offsets* out /* host */);

/*
 * Routing (router GEMV -> top-k -> renormalised weights -> grouping).
 *
 * Pages: "Run Kimi 3.1 locally on one GPU", "Read the experts the router
 * needs" (16 of 896 selected); the router is BF16 ("Run Kimi K3 and K3.1 Pro
 * Locally", "Confirm the checkpoint format and size").  The routing function
 * itself is not on the pages; this library takes the plainest reading:
 *   logit[n][e] = sum_c x[n][c] * Wr[e][c]              (fp32 accumulate)
 *   idx[n][0..k)  = the k largest logits, larger first, equal logits by lower
 *                   index, NaN after every number (and MOE_EBIT_NAN is set)
 *   w[n][j]       = exp(l_j - l_0) / sum_i exp(l_i - l_0)  (softmax over the
 *                   selected k, i.e. softmax then renormalise; fp32)
 * and groups the block's (row, slot) pairs by expert for moe_expert_block.
 *
 *  n_rows      1..n_rows_max of the workspace; the GEMV path needs n_rows <= 32
 *              and d_model <= 8192
 *  x           bf16 [n_rows][d] activations, row-major; may be NULL only when
 *              logits_in is given and no moe_expert_block call follows
 *  w_router    bf16 [E][d] router matrix, row-major (ignored with logits_in)
 *  logits_in   fp32 [n_rows][E] logits to route on instead of the GEMV, or NULL
 *  logits_out  fp32 [n_rows][E] receives the GEMV logits, or NULL
 *  topk_idx    int32 [n_rows][k] selected experts in rank order (output)
 *  topk_w      fp32 [n_rows][k] their weights (output)
 *  ws          workspace (receives the grouping and prepared activations)
 */
MOE_API int moe_route(const moe_desc* desc, int32_t n_rows,
              const uint16_t* x, const uint16_t* w_router,
              const float* logits_in, float* logits_out,
              int32_t* topk_idx, float* topk_w,
              void* ws, int32_t n_rows_max, int32_t n_shared, void* stream);

/*
 * The shared experts alone, straight from the block's rows: they depend on x
 * only, not on the routing ("Run Kimi K3 and K3.1 Pro Locally": every token
 * also runs the 2 shared experts; their matmuls load each weight once for all
 * rows), so this call may run on a second stream while moe_route and the routed
 * experts run, joining before moe_combine.  It keeps its own copy of the
 * activations and its own counters in the workspace, so it never races with
 * moe_route or with the routed part of moe_expert_block (MOE_MODE_ROUTED_ONLY)
 * on the same workspace.  Any n_rows up to the workspace's n_rows_max: blocks
 * of up to 16 rows run on the TMA-fed tensor-core engine (one persistent
 * kernel), larger (prefill) blocks on three register-streaming launches (row
 * preparation, gate/up with SwiGLU, down) that read the weights from HBM once
 * and from L2 for every further 16 rows.  A row's result does not depend on
 * the other rows of its block (within each of the two size classes).
 *
 *  x        bf16 [n_rows][d] (device, 16-byte aligned)
 *  shared   pool of n_shared (1..8) Q8_0 shared experts in slots 0..n_shared-1
 *  Output: shared_y in the workspace (moe_ws_offsets.shared_y), the same values
 *  moe_expert_block writes there.  Errors as moe_expert_block.
 */
MOE_API int moe_shared_experts(const moe_desc* desc, int32_t n_rows, const uint16_t* x,
                       const moe_pool* shared, int32_t n_shared,
                       void* ws, int32_t n_rows_max, void* stream);

/*
 * moe_shared_experts for the launch that directly follows moe_route of the same
 * block on the same stream: its kernel starts while the routing runs (x must be
 * complete before moe_route is enqueued, as moe_route itself needs it) and
 * completes only after the routing has completed, so the next call on the
 * stream (moe_expert_block with MOE_MODE_ROUTED_ONLY, then moe_combine) sees
 * both.  One stream, no events: route -> shared experts -> routed experts ->
 * combine.  Arguments, output and errors as moe_shared_experts.
 */
MOE_API int moe_shared_experts_after_route(const moe_desc* desc, int32_t n_rows, const uint16_t* x,
                       const moe_pool* shared, int32_t n_shared,
                       void* ws, int32_t n_rows_max, void* stream);

/*
 * Every selected expert's SwiGLU MLP on the rows routed to it, plus the shared
 * experts on every row.  Pages: MXFP4 experts ("Run Kimi 3.1 locally on one
 * GPU", "One GPU, three storage tiers"), a block reads each expert once for
 * all its rows ("A drafter that leaves the answer unchanged"):
 *   g = x Wg^T, u = x Wu^T, h = silu(g) * u, y = h Wd^T   per (row, slot)
 * Each expert's slab is streamed from HBM once per call.  Must follow
 * moe_route on the same workspace and stream.
 *
 *  mode         MOE_MODE_DECODE (n_rows <= 16) or MOE_MODE_PREFILL, optionally
 *               | MOE_MODE_DEBUG_GU, and at most one of MOE_MODE_SHARED_ONLY /
 *               MOE_MODE_ROUTED_ONLY (both: MOE_ERR_INVALID_ARG); with
 *               MOE_MODE_ROUTED_ONLY, | MOE_MODE_AFTER_SHARED for the call right
 *               after moe_shared_experts_after_route (without ROUTED_ONLY:
 *               MOE_ERR_INVALID_ARG)
 *  routed       pool holding the routed experts (host struct, MXFP4)
 *  expert_slot  int32 [E] slot of each expert in `routed` (device)
 *  slot_ready   uint32 [routed->n_slots] flags, or NULL when every slot is
 *               resident: an expert's gate/up planes are read only after its
 *               flag has MOE_SLOT_GATE_UP, its down planes only after it has
 *               MOE_SLOT_DOWN (bounded waits; MOE_EBIT_TIMEOUT when one runs
 *               out); a resident slot holds MOE_SLOT_READY
 *  shared       pool of n_shared Q8_0 shared experts in slots 0..n_shared-1,
 *               or NULL with n_shared == 0
 *  y_part       fp32 [n_rows][k][d] output of each (row, slot)
 *  The shared experts' outputs go to the workspace (moe_ws_offsets.shared_y).
 */
MOE_API int moe_expert_block(const moe_desc* desc, int32_t n_rows, int32_t mode,
                     const moe_pool* routed, const int32_t* expert_slot,
                     const uint32_t* slot_ready,
                     const moe_pool* shared, int32_t n_shared,
                     void* ws, int32_t n_rows_max, float* y_part, void* stream);

/*
 * Weighted combine into the residual ("Run Kimi 3.1 locally on one GPU": each
 * token's 16 selected experts; "Run Kimi K3 and K3.1 Pro Locally", table in
 * "Kimi K3 and K3.1 Pro in numbers": plus 2 shared experts; the routed outputs
 * are weighted by the renormalised router weights and added, with the shared
 * experts' outputs, to the residual stream), in a fixed order per element:
 *   acc = 0; for j in 0..k-1: acc = fma(w[n][j], y[n][j][c], acc);
 *   for s in 0..n_shared-1: acc += shared_y[s][n][c];
 *   out[n][c] = bf16_rne(residual[n][c] + acc)
 *  residual  bf16 [n_rows][d];  y_part fp32 [n_rows][k][d];  topk_w fp32 [n_rows][k]
 *  shared_y  fp32 [n_shared][n_rows][d] or NULL;  out bf16 [n_rows][d]
 */
MOE_API int moe_combine(const moe_desc* desc, int32_t n_rows, const uint16_t* residual,
                const float* y_part, const float* topk_w,
                const float* shared_y, int32_t n_shared,
                uint16_t* out, void* stream);

/*
 * Stand-alone Q8_0 matmul of an N-row block: every weight is loaded from HBM
 * once for all rows ("Run Kimi 3.1 locally on one GPU": the spine's matrix
 * multiplies load each weight once for up to eight rows).  W[o][c] = q[o][c] *
 * fp16(d[o][c/32]).
 *  n_rows 1..16; k_in % 256 == 0; n_out % 64 == 0
 *  x       [n_rows][k_in], bf16 (x_dtype MOE_DTYPE_BF16) or fp32 (MOE_DTYPE_F32)
 *  q, d    int8 [n_out][k_in] and fp16 [n_out][k_in/32]; 32-byte aligned
 *  q2, d2  the up matrix for MOE_EPI_SWIGLU (same shape), else NULL
 *  y       fp32 [n_rows][n_out]
 *  ws      scratch of q8_0_workspace_size(n_rows, k_in, n_out) bytes, zeroed once
 *          before first use; a call leaves it ready for the next call of that shape
 * MOE_EPI_SWIGLU requires bf16 x.
 * Without SwiGLU, K may be split into ranges (more work items when n_out is small
 * for the GPU: 7168 -> 1536 has 24 blocks of 64 outputs).  The number of ranges
 * depends on k_in, n_out and the GPU's SM count, never on n_rows; the last range of
 * a 64-output block to finish adds the ranges' fp32 sums in range order, so every
 * row's result is the same in every block and from run to run.
 */
MOE_API size_t q8_0_workspace_size(int32_t n_rows, int32_t k_in, int32_t n_out);
MOE_API int q8_0_block_matmul(int32_t n_rows, int32_t k_in, int32_t n_out,
                      const void* x, int32_t x_dtype,
                      const int8_t* q, const uint16_t* d,
                      const int8_t* q2, const uint16_t* d2,
                      int32_t epilogue, float* y, void* ws, void* stream);

/*
 * q8_0_block_matmul without a caller-provided workspace, for callers that
 * cannot allocate device memory: a host process whose own pool allocator owns
 * all of HBM, or a latency-critical path where cudaMalloc/cudaFree (which can
 * synchronise the device) is not acceptable.  The pages have no counterpart of
 * this entry point; it is a deployment convenience of this library.
 *
 * Same arguments and results as q8_0_block_matmul, minus ws.  Its scratch is a
 * file-scope __device__ array of 2,789,376 bytes that every GPU loading this
 * library holds until the process exits; limits: n_rows <= 16 and
 * k_in <= 7168 (larger sizes return MOE_ERR_UNSUPPORTED before any launch).
 * It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  The address is kept per device together with the context it
 * belongs to: after a device reset (or any new primary context) the next call
 * looks it up again, so make that call outside a capture too.  Every call
 * shares the one array: the call clears the parts that must start at zero, but
 * calls that overlap on the GPU (different streams, or different host threads
 * on one device) race on it and must be serialised by the caller.  Device-side
 * errors (a bounded wait that ran out) accumulate in the array's error word
 * across calls; read and clear them with q8_0_noalloc_get_error.
 */
MOE_API int q8_0_block_matmul_noalloc(int32_t n_rows, int32_t k_in, int32_t n_out,
                                      const void* x, int32_t x_dtype,
                                      const int8_t* q, const uint16_t* d,
                                      const int8_t* q2, const uint16_t* d2,
                                      int32_t epilogue, float* y, void* stream);

/*
 * The device error word (MOE_EBIT_* bits) of q8_0_block_matmul_noalloc's static
 * array on the current device: every bit its calls set since the last read.
 * Synchronises `stream`, returns the word through *bits (host) and clears it.
 * Allocates nothing.  Returns MOE_OK, MOE_ERR_INVALID_ARG (bits NULL) or
 * MOE_ERR_CUDA.  Like the matmul call, it has no counterpart on the pages.
 */
MOE_API int q8_0_noalloc_get_error(void* stream, uint32_t* bits);

/*
 * Reads the workspace's device error word (synchronising `stream`), clears it,
 * and returns it through *bits (host).  Returns MOE_OK, or MOE_ERR_CUDA.
 */
MOE_API int moe_get_error(void* ws, void* stream, uint32_t* bits);

/* Number of SMs the persistent kernels size their grids for (0 if no device). */
MOE_API int32_t moe_device_sm_count(void);

/*
 * Device expert cache (host side).  A pool of n_slots device slots (the routed
 * pool of moe_expert_block) holds (layer, expert) slabs; misses are uploaded from
 * pinned host memory while the expert kernels run, which start on each expert's
 * work as its data lands (its ready flag, MOE_SLOT_* bits).
 *
 * Pages: "Run Kimi 3.1 locally on one GPU", section "One GPU, three storage
 * tiers" (experts streamed from the lower tier as the router asks for them; the
 * NVMe tier itself is out of scope, pinned host memory stands in for it).
 *
 * moe_cache_create: slot_base/slot_bytes/n_slots describe the device pool;
 *   slot_ready uint32 [n_slots] device flags (zeroed here); n_streams upload
 *   streams (0: planning only -- slot assignment and miss reporting without any
 *   CUDA call, pointers may be NULL); policy MOE_CACHE_LRU or
 *   MOE_CACHE_KEEP_MULTI_ROW (keep the experts used by two rows or more: evict
 *   the least recently used slot whose last block used it on one row, and when
 *   every candidate was used by several rows, the most recently used one).  The cache owns its streams and events.
 * moe_cache_request: the `count` distinct experts (host int32) one layer of a
 *   block needs, with the number of the block's rows using each (host int32, or
 *   NULL = 1) and each expert's pinned host slab (host array of pointers; unused
 *   when planning only).  Writes each expert's slot (host int32 [count]) and
 *   whether it was uploaded (host int32 [count], may be NULL).  For the misses it
 *   writes 0 to the victims' flags on compute_stream (after every earlier kernel
 *   there, so after every reader of the old slab), then on the upload streams
 *   copies gate+up, sets MOE_SLOT_GATE_UP, copies down, sets MOE_SLOT_READY.
 *   Launch the expert kernels for this layer on compute_stream after the call.
 *   count > n_slots: MOE_ERR_UNSUPPORTED.
 * moe_cache_sync waits for the uploads; moe_cache_destroy syncs and frees.
 */
#define MOE_CACHE_LRU 0
#define MOE_CACHE_KEEP_MULTI_ROW 1

typedef struct moe_cache moe_cache;

typedef struct moe_cache_stats {
    int64_t requests;
    int64_t hits;
    int64_t misses;
    int64_t evictions;
    int64_t bytes_uploaded;
} moe_cache_stats;

MOE_API int moe_cache_create(const moe_desc* desc, void* slot_base, int64_t slot_bytes, int32_t n_slots,
                     uint32_t* slot_ready, int32_t n_streams, int32_t policy, moe_cache** out /* host */);
MOE_API int moe_cache_request(moe_cache* cache, int32_t layer, int32_t count, const int32_t* experts,
                      const int32_t* rows, const void* const* host_src, int32_t* slot_out,
                      int32_t* miss_out, void* compute_stream);
MOE_API int moe_cache_stats_get(const moe_cache* cache, moe_cache_stats* out /* host */);

/* Which of `count` experts of `layer` hold a slot now (host int32 [count], 1 or 0),
   without touching the cache's state: a caller fetching misses from a lower tier
   asks this before moe_cache_request_staged. */
MOE_API int moe_cache_lookup(const moe_cache* cache, int32_t layer, int32_t count, const int32_t* experts,
                     int32_t* resident_out /* host */);

/*
 * moe_cache_request for slabs that are still being filled in host memory (by the
 * NVMe tier below): host_ready[i] points to a uint32 flag in pinned host memory
 * that receives MOE_SLOT_GATE_UP once the gate/up part of host_src[i] is in place
 * and MOE_SLOT_DOWN once the rest is.  Before each chunk's copy the upload stream
 * runs a host function that waits for the chunk's bit (bounded: 10 s), so the
 * call returns at once, the chunks move as soon as they have been read, and the
 * GPU never waits on host memory.  The NVMe tier sets both bits even when a read
 * fails (with MOE_NVME_FAILED).  Other arguments as moe_cache_request.
 */
MOE_API int moe_cache_request_staged(moe_cache* cache, int32_t layer, int32_t count, const int32_t* experts,
                      const int32_t* rows, const void* const* host_src,
                      const uint32_t* const* host_ready, int32_t* slot_out,
                      int32_t* miss_out, void* compute_stream);

/*
 * NVMe expert tier (host side).  The expert slabs live in files, one per drive,
 * each drive holding a replica of the same n_bodies slabs (slab b at byte offset
 * b * slab_stride).  Pages: "Run Kimi 3.1 locally on one GPU", section "Read the
 * experts the router needs" (experts on several NVMe drives read with O_DIRECT
 * into pinned memory, per-drive concurrency caps, replica choice by expected
 * completion time, decode fills in two chunks).
 *
 * moe_nvme_open: n_replicas files (the same slabs on each), depth reader threads
 *   per file (its cap on reads in flight).  O_DIRECT is used where the file system
 *   allows it and the read is 4 KiB aligned (buffer, offset, length), buffered
 *   reads otherwise.  Files shorter than the slabs they must hold: MOE_ERR_INVALID_ARG.
 * moe_nvme_read: queues the read of slab `body` into host memory dst (pinned, at
 *   least slab_bytes), first the bytes [0, first_bytes) then the rest, on the
 *   replica whose pending bytes plus this read, over its measured bandwidth, is
 *   smallest (*replica_out, may be NULL).  *flag (host) is zeroed, then gets
 *   MOE_SLOT_GATE_UP after the first chunk and MOE_SLOT_READY after the whole
 *   slab, plus MOE_NVME_FAILED if a read failed.  Returns at once.
 * moe_nvme_wait: host wait until (*flag & bits) == bits (MOE_ERR_TIMEOUT after
 *   timeout_ns; MOE_ERR_IO if the read failed).
 * moe_nvme_close waits for every queued read, then closes the files.
 */
#define MOE_NVME_FAILED 0x80000000u

typedef struct moe_nvme moe_nvme;

typedef struct moe_nvme_stats {
    int64_t reads;
    int64_t bytes;
    int64_t failures;
    int64_t pending_bytes;
    double bandwidth;      /* bytes/s, exponentially weighted over completed reads */
    double busy_seconds;   /* summed read time of its threads */
    int32_t direct;        /* 1 if the file was opened with O_DIRECT */
} moe_nvme_stats;

MOE_API int moe_nvme_open(const char* const* paths /* host */, int32_t n_replicas, int64_t slab_bytes,
                  int64_t slab_stride, int32_t n_bodies, int32_t depth, moe_nvme** out /* host */);
MOE_API int moe_nvme_read(moe_nvme* nvme, int32_t body, void* dst, int64_t first_bytes,
                  volatile uint32_t* flag, int32_t* replica_out);
MOE_API int moe_nvme_wait(const volatile uint32_t* flag, uint32_t bits, int64_t timeout_ns);
MOE_API int moe_nvme_stats_get(moe_nvme* nvme, int32_t replica, moe_nvme_stats* out /* host */);
MOE_API int moe_nvme_close(moe_nvme* nvme);
MOE_API int moe_cache_sync(moe_cache* cache);
MOE_API int moe_cache_destroy(moe_cache* cache);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
