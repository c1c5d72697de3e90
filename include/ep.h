/*
 * ep.h - C ABI of a single-GPU (GB300, sm_103a) MoE token layout, dispatch
 * and combine library.
 *
 * What it computes follows the DeepEP write-ups:
 *   - "DeepEP V1 (legacy) guide" (zskr.cn), section 5 (normal kernels:
 *     get_dispatch_layout, dispatch, combine), section 6 (low-latency
 *     kernels: fixed-shape receive buffer, receive counts, receive hook);
 *   - "How DeepEP enables hook-based overlapping" (instagit.com), sections
 *     "Two-Phase Kernel Architecture" and "Compute Stream vs. Communication
 *     Stream" (send and receive as two launches; the launch stream);
 *   - "DeepEP Ascend deep dive" (kongchang.com), sections "Two Transfers" and
 *     "Dispatch's Three Phases" (one copy per destination rank; the
 *     expert-major "expand" layout; the weighted top-k sum of combine).
 *
 * Expert-parallel ranks are logical partitions of one GPU's memory: R ranks,
 * E experts, expert e lives on rank e / (E / R). Tokens are split
 * contiguously over the R source ranks, so "source rank, then token index"
 * order is global token order.
 *
 * Conventions for every entry point:
 *   - Every pointer argument is a DEVICE pointer owned by the caller unless
 *     stated otherwise. The library never allocates or frees memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call only enqueues work on it and returns; nothing synchronises with
 *     the host. Outputs are ready when the stream reaches that point.
 *   - Return value: EP_OK, or a negative EP_ERR_* code for an error the host
 *     can see (bad argument, bad alignment, too-small workspace, a CUDA
 *     launch error). Nothing is enqueued when an argument error is returned.
 *     A call that makes two launches (the low-latency send, layout +
 *     dispatch in one call, an aligned dispatch with its padding fill) may
 *     have enqueued the first when the second fails with EP_ERR_CUDA.
 *   - `status` (may be NULL) points to one device int32. Kernels OR EP_ST_*
 *     bits into it for data-dependent conditions (an expert index out of
 *     range, a destination row beyond a buffer's capacity, ...). The
 *     offending row is skipped; no kernel traps. The caller zeroes it.
 *   - The combines, the low-latency send (up to 65536 entries) and the
 *     receive launch their first kernel as a programmatic dependent of the
 *     kernel before it on the stream: it may be scheduled while that kernel
 *     drains, and it waits for that kernel to complete before it reads or
 *     writes any memory, so stream order holds as for a plain launch. (If
 *     the kernel before it was itself launched by the caller with
 *     programmatic serialization and never waits for its own predecessor,
 *     that predecessor is not waited for either.)
 *   - BF16 data is passed as raw 16-bit words, E4M3 data as bytes.
 *   - Row buffers (x, receive buffers, expert outputs, out) must be 16-byte
 *     aligned, and hidden * element size must be a multiple of 16 bytes.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---------------------------------------------------- */
#define EP_OK 0
#define EP_ERR_INVALID_ARG (-1) /* null pointer, size out of range, E % R != 0, ... */
#define EP_ERR_ALIGNMENT (-2)   /* a row buffer is not 16-byte aligned */
#define EP_ERR_WORKSPACE (-3)   /* workspace missing or smaller than required */
#define EP_ERR_LL_CAPACITY (-4) /* low-latency: N / R tokens per rank exceed T */
#define EP_ERR_CUDA (-5)        /* a CUDA runtime call or launch failed */
#define EP_ERR_UNSUPPORTED (-6) /* device lacks a required feature */

/* ---- device status bits ---------------------------------------------- */
#define EP_ST_BAD_INDEX 0x1   /* a top-k index outside [-1, E): treated as -1 */
#define EP_ST_CAPACITY 0x2    /* a row did not fit the given buffer: skipped */
#define EP_ST_LL_OVERFLOW 0x4 /* low-latency: a row beyond an expert's R*T region */
#define EP_ST_TIMEOUT 0x8     /* a bounded in-kernel wait gave up */
#define EP_ST_NOT_SENT 0x10   /* low-latency receive without a matching send */
#define EP_ST_MISMATCH 0x20   /* low-latency shapes differ from those of the send */
#define EP_ST_WORKSPACE 0x40  /* the workspace's barrier count was not zero on entry */

/* ---- dispatch payload flags (the `fp8_flags` / `use_fp8` arguments) -------
 * 0: BF16 rows. EP_FP8: E4M3 rows with one fp32 scale per 128 channels,
 * s = amax / 448. EP_FP8_ROUND_SCALE: s raised to the next power of two, so
 * dequantisation is an exact shift. EP_FP8_UE8M0: power-of-two scales stored
 * as one UE8M0 byte 2^(b - 127) per 128 channels ([rows, H/128] bytes; viewed
 * as int32 [rows, H/512] they are four bytes per word, block b in byte b % 4),
 * s kept >= 2^-127. ("DeepEP V1 (legacy) guide", section 6.3: round_scale,
 * use_ue8m0.) The flag values 0 and 1 are the plain BF16 / FP8 choices. */
#define EP_FP8 0x1
#define EP_FP8_ROUND_SCALE 0x2
#define EP_FP8_UE8M0 0x4

/* ---- limits ---------------------------------------------------------- */
#define EP_MAX_EXPERTS 1024
#define EP_MAX_TOPK 32
#define EP_MAX_HIDDEN 16384

/*
 * The routing layout of one batch: the handle that dispatch and combine take.
 * The caller allocates every array and fills in the pointers and sizes;
 * ep_get_dispatch_layout writes the arrays. Reusing a filled handle skips the
 * layout ("cached dispatch", DeepEP V1 guide section 5.2(4)).
 *
 *   topk_idx              [N, K] int32  in: expert of each top-k slot, -1 = none
 *   num_tokens_per_rank   [R]    int32  tokens sent to each rank (one copy per rank)
 *   num_tokens_per_expert [E]    int32  (token, slot) pairs routed to each expert
 *   is_token_in_rank      [N, R] uint8  1 if some expert of the token lives on the rank
 *   rank_offset           [R+1]  int32  exclusive prefix sum of num_tokens_per_rank
 *   expert_offset         [E+1]  int32  exclusive prefix sum of num_tokens_per_expert
 *   rank_slot             [N, R] int32  row of the token in the per-rank buffer, or -1
 *   expert_slot           [N, K] int32  row of (token, slot) in the expert-major buffer, or -1
 *
 * Slots are deterministic: within a rank (or an expert) rows are in token
 * order (and top-k order for repeated experts), ranks (experts) in index
 * order.
 *
 * expert_alignment A > 1 pads every expert's segment of the expert-major
 * buffer to a multiple of A rows ("DeepEP Ascend deep dive", "Dispatch's
 * Three Phases": expert alignment to 128 rows for the grouped GEMM, empty rows
 * filled with zeros): expert_offset becomes the exclusive scan of the padded
 * lengths (num_tokens_per_expert stays the true count) and ep_dispatch zeroes
 * the padding rows (payload, scales, src = -1). Capacity then needs
 * N * K + E * (A - 1) rows in the worst case.
 */
typedef struct ep_layout {
  int32_t num_tokens;  /* N >= 0 */
  int32_t num_topk;    /* 1 <= K <= EP_MAX_TOPK */
  int32_t num_experts; /* 1 <= E <= EP_MAX_EXPERTS */
  int32_t num_ranks;   /* 1 <= R <= E, E % R == 0 */
  const int32_t* topk_idx;
  int32_t* num_tokens_per_rank;
  int32_t* num_tokens_per_expert;
  uint8_t* is_token_in_rank;
  int32_t* rank_offset;
  int32_t* expert_offset;
  int32_t* rank_slot;
  int32_t* expert_slot;
  int32_t expert_alignment; /* 0 or 1: expert segments packed; A > 1: each
                               expert's segment padded to a multiple of A rows */
} ep_layout_t;

/*
 * One receive buffer of ep_dispatch. Rows are packed: the per-rank buffer by
 * rank_offset, the expert-major buffer by expert_offset.
 *   x             [capacity, H]       BF16 words, or E4M3 bytes when use_fp8
 *   scales        [capacity, H/128]   fp32, or UE8M0 bytes with EP_FP8_UE8M0
 *                                     (FP8 only; may be NULL to skip)
 *   src_idx       [capacity]          int32, may be NULL. Per-rank buffer: the
 *                                     token index t. Expert-major: t * K + k.
 *   topk_idx      [capacity, K]       int32, may be NULL; per-rank buffer only:
 *                                     the local expert id (e - r * E/R) of each
 *                                     slot whose expert lives on this rank, else -1
 *   topk_weights  [capacity, K]       fp32, may be NULL; per-rank buffer only:
 *                                     the slot's router weight, or 0
 *   capacity      rows allocated; rows at or beyond it are skipped and flagged
 *                 EP_ST_CAPACITY. N * min(K, R) (per-rank) and N * K
 *                 (expert-major) always suffice without reading the counts.
 */
typedef struct ep_recv_buffer {
  void* x;
  void* scales;
  int32_t* src_idx;
  int32_t* topk_idx;
  float* topk_weights;
  int64_t capacity;
} ep_recv_buffer_t;

/* Library version (major * 10000 + minor * 100 + patch). */
int ep_version(void);

/* A short English description of a return code (negative) or of the lowest
 * set status bit (positive). Static storage; never NULL. */
const char* ep_error_string(int code_or_status);

/*
 * Bytes of device workspace ep_get_dispatch_layout needs for these sizes.
 * Depends only on the arguments (not on the device).
 */
size_t ep_layout_workspace_bytes(int num_tokens, int num_topk, int num_experts, int num_ranks);

/*
 * Routing layout: counts, the per-rank mask and deterministic prefix-sum
 * slots (DeepEP V1 guide section 5.2(1): get_dispatch_layout returns
 * num_tokens_per_rank, num_tokens_per_expert and is_token_in_rank; "DeepEP
 * Ascend deep dive", "Two Transfers": a rank receives a token once even when
 * several of its experts live there; "Dispatch's Three Phases", phase 3: the
 * receive-source map that combine follows back).
 *
 *   L          handle: sizes, topk_idx and the output arrays (see ep_layout_t)
 *   workspace  device scratch of at least ep_layout_workspace_bytes(...)
 *              bytes, 16-byte aligned, zero-filled before its first use (cudaMemset once at
 *              allocation). Every call leaves it as it needs to find it
 *              next time, so it is not cleared again between calls. Must
 *              not be used by another call in flight.
 *   status     EP_ST_BAD_INDEX when an index lies outside [-1, E) (the slot
 *              is treated as -1); EP_ST_TIMEOUT if an internal grid-wide wait
 *              gave up; EP_ST_WORKSPACE if the workspace was not zero-filled
 *              before its first use (or a previous call on it timed out).
 *              After either of the last two the outputs are invalid and the
 *              workspace must be zero-filled again.
 * Runs as one cooperative launch. The kernel releases programmatic dependents
 * at its start: a kernel the caller launches right after it with programmatic
 * stream serialization may begin at once and must wait on the grid dependency
 * (griddepcontrol.wait / cudaGridDependencySynchronize) before it reads any of
 * the layout's outputs. Kernels launched without that attribute are unaffected.
 */
int ep_get_dispatch_layout(const ep_layout_t* L, void* workspace, size_t workspace_bytes,
                           int32_t* status, void* stream);

/*
 * The routing layout for callers that cannot allocate device memory where
 * they need it: code inside a host framework whose caching allocator owns the
 * GPU's memory (a raw cudaMalloc bypasses its accounting and can fail once
 * the pool holds most of HBM), plug-ins that are handed only their input and
 * output buffers, and latency-critical loops where a cudaMalloc may
 * synchronise the device. The DeepEP write-ups have no counterpart of this
 * call; it is a convenience of this library.
 *
 * Same arguments and results as ep_get_dispatch_layout, without the
 * workspace: the scratch lives in a 1 MiB array of device memory that the
 * library holds on every GPU that loads it, until the process exits. Sizes
 * whose ep_layout_workspace_bytes(...) exceeds 1 MiB return EP_ERR_WORKSPACE
 * (for example E = R = 1024 with more than about 780,000 (token, slot)
 * entries); no call allocates or frees memory.
 *
 * The first call on a device looks up that array's device address (once per
 * device, with the device current); make that first call before any stream
 * capture. Every call shares the array and it keeps the last call's contents
 * (each call resets its barrier words first). Calls that overlap on the GPU,
 * such as calls on two streams with no ordering between them, race on it.
 */
int ep_get_dispatch_layout_noalloc(const ep_layout_t* L, int32_t* status, void* stream);

/*
 * Dispatch: copy each token's hidden row x[t] into the per-rank receive
 * buffer (row rank_slot[t, r] for every rank r of its mask: one copy per
 * rank) and into the expert-major buffer (row expert_slot[t, k] for every
 * unmasked slot k: one copy per chosen expert), optionally quantised once to
 * FP8 E4M3 with one fp32 scale per 128 channels: s = amax / 448 (round to
 * nearest), q = e4m3(x / s) rounded to nearest even and saturated to +-448;
 * an all-zero block has s = 0 and zero codes.
 * (DeepEP V1 guide sections 5.1 and 5.2(6); "DeepEP Ascend deep dive",
 * "Dispatch's Three Phases": the expert-major expand layout and FP8 E4M3 with
 * a scale travelling with each token.)
 *
 *   L             a handle filled by ep_get_dispatch_layout
 *   x             [N, hidden] BF16
 *   hidden        H: a multiple of 8 (BF16) or of 128 (FP8), <= EP_MAX_HIDDEN
 *   fp8_flags     0: rows are copied as BF16; EP_FP8 (optionally with
 *                 EP_FP8_ROUND_SCALE or EP_FP8_UE8M0): rows are E4M3 + scales
 *   topk_weights  [N, K] fp32; needed only for rank_buf->topk_weights
 *   rank_buf      per-rank receive buffer, or NULL to skip the per-rank copy
 *   expert_buf    expert-major receive buffer, or NULL to skip it
 *   status        EP_ST_CAPACITY for rows beyond a buffer's capacity
 */
int ep_dispatch(const ep_layout_t* L, const void* x, int hidden, int fp8_flags,
                const float* topk_weights, const ep_recv_buffer_t* rank_buf,
                const ep_recv_buffer_t* expert_buf, int32_t* status, void* stream);

/*
 * Layout and dispatch in one call: the same work, arguments, results, status
 * bits and error codes as ep_get_dispatch_layout(L, workspace,
 * workspace_bytes, status, stream) followed by ep_dispatch(L, x, hidden,
 * fp8_flags, topk_weights, rank_buf, expert_buf, status, stream). Every
 * argument of both is checked before anything is enqueued.
 * (The two steps of the DeepEP V1 guide, section 5.1: get_dispatch_layout,
 * then dispatch with its counts and mask.)
 *
 * The dispatch is launched as the programmatic dependent of the layout
 * (programmatic dependent launch): its blocks start while the layout runs,
 * bring in (and quantise) their token rows, and wait in-kernel for the layout
 * to complete before they read any slot. So x, topk_idx and topk_weights must
 * be ready when the call is enqueued, as for any stream-ordered call; nothing
 * else changes for the caller.
 * Receive buffers must exist before the call: size them for the worst case
 * (see ep_recv_buffer_t), since the counts are not known on the host.
 */
int ep_layout_dispatch(const ep_layout_t* L, void* workspace, size_t workspace_bytes,
                       const void* x, int hidden, int fp8_flags, const float* topk_weights,
                       const ep_recv_buffer_t* rank_buf, const ep_recv_buffer_t* expert_buf,
                       int32_t* status, void* stream);

/*
 * Combine: gather the expert outputs back along the dispatch path and take
 * the router-weighted sum: out[t] = bf16( sum over k = 0..K-1 with
 * expert_slot[t, k] >= 0 of w[t, k] * y[expert_slot[t, k]] ), accumulated in
 * fp32 with one fused multiply-add per term in slot order, starting from +0,
 * rounded once to BF16 (nearest even). A token with every slot masked gets +0.
 * ("DeepEP Ascend deep dive", "Two Transfers": results go back along the
 * same path and are weighted by router scores and summed; "DeepEP lesson 14",
 * practice task: out_i = sum_k w_ik * y_ik.)
 *
 *   L             a handle filled by ep_get_dispatch_layout
 *   expert_y      [y_rows, hidden] BF16 expert outputs in expert-major order
 *                 (row expert_slot[t, k] holds expert idx[t, k]'s output for t)
 *   y_rows        rows of expert_y; slots at or beyond it are skipped and
 *                 flagged EP_ST_CAPACITY
 *   hidden        a multiple of 8, <= EP_MAX_HIDDEN
 *   topk_weights  [N, K] fp32 router weights, or NULL for unit weights: the
 *                 unweighted sum of a token's expert-major rows is the
 *                 backward of dispatch ("DeepEP V1 (legacy) guide", section
 *                 5.1: the backward of dispatch is a combine)
 *   bias          [N, hidden] BF16 or NULL: added in fp32 after the weighted
 *                 sum, before the BF16 rounding (the shared expert's output
 *                 folded into the epilogue, "DeepEP Ascend deep dive",
 *                 "Combine: More Output, Same Cost")
 *   out           [N, hidden] BF16
 */
int ep_combine(const ep_layout_t* L, const void* expert_y, int64_t y_rows, int hidden,
               const float* topk_weights, const void* bias, void* out, int32_t* status,
               void* stream);

/*
 * Two-level combine, first level: each rank reduces its own experts' outputs
 * before sending one row per (token, rank) back (the shape of DeepEP's normal
 * combine(x, handle), whose x is one row per received token of each rank,
 * "DeepEP V1 (legacy) guide", section 5.1). For every (t, r) with
 * is_token_in_rank[t, r]: rank_out[rank_slot[t, r]] = bf16( sum over k in slot
 * order whose expert lives on r of w[t, k] * y[expert_slot[t, k]] ), the fp32
 * fused multiply-add chain of ep_combine.
 *
 *   L             a handle filled by ep_get_dispatch_layout (K <= EP_MAX_TOPK)
 *   expert_y      [y_rows, hidden] BF16 expert outputs, expert-major
 *   topk_weights  [N, K] fp32
 *   rank_out      [rank_rows, hidden] BF16, the per-rank layout
 */
int ep_combine_to_ranks(const ep_layout_t* L, const void* expert_y, int64_t y_rows, int hidden,
                        const float* topk_weights, void* rank_out, int64_t rank_rows,
                        int32_t* status, void* stream);

/*
 * Two-level combine, second level: out[t] = bf16( sum over ranks r ascending
 * with is_token_in_rank[t, r] of rank_y[rank_slot[t, r]] (+ bias) ), fp32
 * accumulation, one rounding. With rank_y from ep_combine_to_ranks this is the
 * whole combine with one intermediate BF16 rounding per rank.
 *
 *   rank_y   [rank_rows, hidden] BF16 per-rank rows
 *   bias     [N, hidden] BF16 or NULL, as for ep_combine
 *   out      [N, hidden] BF16
 */
int ep_combine_ranks(const ep_layout_t* L, const void* rank_y, int64_t rank_rows, int hidden,
                     const void* bias, void* out, int32_t* status, void* stream);

/*
 * Backward of combine ("DeepEP V1 (legacy) guide", section 5.1: the backward
 * of combine is a dispatch). For out[t] = sum_k w[t, k] y[expert_slot[t, k]]:
 *   grad_y[expert_slot[t, k]] = bf16( w[t, k] * grad_out[t] )   (fp32 product)
 *   grad_w[t, k]              = <grad_out[t], y[expert_slot[t, k]]>, fp32, in a
 *                               fixed order (deterministic), 0 for masked slots
 * The gradient of a combine bias is grad_out itself.
 *
 *   grad_out      [N, hidden] BF16
 *   expert_y      [y_rows, hidden] BF16 forward expert outputs (needed for grad_w)
 *   topk_weights  [N, K] fp32
 *   grad_y        [y_rows, hidden] BF16, or NULL to skip; rows that no slot
 *                 names (padding, capacity slack) are not written
 *   grad_w        [N, K] fp32, or NULL to skip
 */
int ep_combine_backward(const ep_layout_t* L, const void* grad_out, const void* expert_y, int64_t y_rows,
                        int hidden, const float* topk_weights, void* grad_y, float* grad_w,
                        int32_t* status, void* stream);

/*
 * Bytes of device workspace the low-latency calls need. The workspace
 * carries the routing from send to receive and combine (the "handle").
 */
size_t ep_ll_workspace_bytes(int num_tokens, int num_topk, int num_experts, int num_ranks,
                             int max_tokens_per_rank);

/*
 * Low-latency dispatch, send phase (DeepEP V1 guide section 6.1/6.3;
 * "How DeepEP enables hook-based overlapping", "Two-Phase Kernel
 * Architecture": the send phase runs at once, the receive phase when the
 * hook is called; "DeepEP lesson 14", low-latency call flow: receive buffer
 * [num_local_experts, num_max_dispatch_tokens_per_rank * num_ranks, hidden]).
 *
 * Tokens are split contiguously over R source ranks, n = N / R each, with
 * n <= T (else EP_ERR_LL_CAPACITY). Each (token, slot) with expert e >= 0 is
 * written to expert e's fixed region of recv_x: rows are packed in token
 * order at j = 0 .. count_e - 1 of [e][0 .. R*T). Rows j >= count_e are not
 * written. Seen from rank r, its experts' regions form the pages' per-rank
 * shape [E/R, R*T, H].
 *
 *   x            [N, hidden] BF16
 *   topk_idx     [N, K] int32, -1 = no expert
 *   fp8_flags    as for ep_dispatch (0 = BF16)
 *   recv_x       [E, R*T, hidden] BF16, or E4M3 with EP_FP8
 *   recv_scales  [E, R*T, hidden/128] fp32, or UE8M0 bytes (FP8 only)
 *   recv_src     [E, R*T] int32: global token index of each written row
 *   workspace    at least ep_ll_workspace_bytes(...) bytes, 16-byte aligned, zero-filled
 *                before its first use (as for ep_get_dispatch_layout: each
 *                send leaves its barrier words zero again); afterwards it
 *                holds the routing that receive and combine use, until the
 *                next send on it
 *   status       EP_ST_BAD_INDEX, EP_ST_TIMEOUT and EP_ST_WORKSPACE as for
 *                the layout
 * Slots of ranks masked in the workspace (shrink mode, ep_ll_update_mask)
 * are dropped. With E * R <= 16384, a batch of N * K <= 4096 entries is one
 * launch (every block finds its own token's slots from the whole routing
 * table; one block writes the counts and ranges), and a batch of up to 65536
 * entries with (N / R) * K <= 8192 is two: per-source-rank histograms, then
 * the row copies as their programmatic dependent (they load, count their own
 * source rank's earlier entries and quantise while the histograms are built,
 * then add the earlier source ranks' counts). Otherwise it is two launches:
 * the routing layout, then the row copies as its programmatic dependent. A
 * second launch may fail with EP_ERR_CUDA after the first was enqueued. The
 * rows are in place when the stream reaches the end of this call; the counts
 * are published by ep_ll_dispatch_recv.
 */
int ep_ll_dispatch_send(const void* x, const int32_t* topk_idx, int num_tokens, int num_topk,
                        int hidden, int num_experts, int num_ranks, int max_tokens_per_rank,
                        int fp8_flags, void* recv_x, void* recv_scales, int32_t* recv_src,
                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Low-latency dispatch, receive phase: the deferred second launch (the
 * "hook"). Publishes the per-expert receive counts and, per (expert, source
 * rank), the range of rows that came from that source. ("How DeepEP enables
 * hook-based overlapping", "Two-Phase Kernel Architecture": the receive phase
 * is a separate launch that runs when the hook is called; "DeepEP V1
 * (legacy) guide", section 6.3: the hook guarantees the rows have arrived and
 * returns recv_count, the tokens each local expert received.)
 *
 *   workspace     the workspace a send filled (same sizes)
 *   recv_count    [E] int32: rows received by each expert
 *   layout_range  [E, R] int64: (offset << 32) | count of the rows of expert
 *                 e that came from source rank s (offsets are an exclusive
 *                 scan over s; only rows inside the expert's R*T region are
 *                 counted, so with EP_ST_LL_OVERFLOW the ranges cover the
 *                 rows that landed); may be NULL
 *   cumulative_recv_stats  [E] int32 or NULL: each call adds recv_count to it
 *                 (the per-expert load statistics of "DeepEP V1 (legacy)
 *                 guide", section 6.3, cumulative_local_expert_recv_stats;
 *                 rank r's experts are entries [r*E/R, (r+1)*E/R))
 *   status        EP_ST_NOT_SENT if no send filled the workspace since the
 *                 last receive; EP_ST_MISMATCH if the sizes differ from it
 * Must be ordered after the send on the stream (same stream, or an event):
 * the kernel checks the workspace once and never waits on another launch.
 */
int ep_ll_dispatch_recv(void* workspace, size_t workspace_bytes, int num_tokens, int num_topk,
                        int num_experts, int num_ranks, int max_tokens_per_rank,
                        int32_t* recv_count, int64_t* layout_range, int32_t* cumulative_recv_stats,
                        int32_t* status, void* stream);

/*
 * Low-latency combine: out[t] = bf16( sum over k of w[t, k] * y[e][j(t, k)] )
 * with the same fp32 fused multiply-add chain in slot order as ep_combine,
 * where j(t, k) is the row the send gave (token, slot) in expert e's region.
 * (DeepEP V1 guide section 6.1, low_latency_combine; "DeepEP lesson 14",
 * low-latency call flow, step 4.)
 *
 *   expert_y      [E, R*T, hidden] BF16 expert outputs in the receive layout
 *   topk_weights  [N, K] fp32
 *   bias          [N, hidden] BF16 or NULL, as for ep_combine
 *   workspace     filled by the send of this batch (same sizes)
 *   out           [N, hidden] BF16
 *   status        EP_ST_NOT_SENT / EP_ST_MISMATCH as for the receive
 * Slots of ranks masked in the workspace now (shrink mode) are skipped.
 */
int ep_ll_combine(const void* expert_y, const float* topk_weights, const void* bias,
                  const void* workspace, size_t workspace_bytes, int num_tokens, int num_topk,
                  int hidden, int num_experts, int num_ranks, int max_tokens_per_rank, void* out,
                  int32_t* status, void* stream);

/*
 * Two-phase low-latency combine, send phase: the expert outputs go back to
 * their source tokens ("DeepEP V1 (legacy) guide", section 6.1:
 * low_latency_combine also returns a receive hook; "How DeepEP enables
 * hook-based overlapping", "Two-Phase Kernel Architecture"). On one GPU the
 * "transfer" gathers every routed row y[e][j(t, k)] into the token-major
 * staging row t * K + k; masked slots are not written.
 *
 *   expert_y   [E, R*T, hidden] BF16 expert outputs in the receive layout
 *   workspace  filled by the send of this batch (same sizes)
 *   staging    [N * K, hidden] BF16, caller-owned
 *   status     EP_ST_NOT_SENT / EP_ST_MISMATCH as for ep_ll_combine
 * The result of send followed by receive equals ep_ll_combine bit for bit
 * (same values, same fp32 fused multiply-add chain); the single-phase call
 * moves fewer bytes, the two-phase form lets other work run in between.
 */
int ep_ll_combine_send(const void* expert_y, const void* workspace, size_t workspace_bytes,
                       int num_tokens, int num_topk, int hidden, int num_experts, int num_ranks,
                       int max_tokens_per_rank, void* staging, int32_t* status, void* stream);

/*
 * Two-phase low-latency combine, receive phase (the hook): out[t] =
 * bf16( sum over unmasked k in slot order of w[t, k] * staging[t * K + k] ),
 * the same fp32 fused multiply-add chain as ep_combine.
 *
 *   staging       [N * K, hidden] BF16 written by ep_ll_combine_send
 *   topk_weights  [N, K] fp32
 *   bias          [N, hidden] BF16 or NULL, as for ep_combine
 *   workspace     the same workspace (it says which slots are masked)
 *   out           [N, hidden] BF16
 * Must be ordered after the send phase on the stream.
 */
int ep_ll_combine_recv(const void* staging, const float* topk_weights, const void* bias,
                       const void* workspace, size_t workspace_bytes, int num_tokens, int num_topk,
                       int hidden, int num_experts, int num_ranks, int max_tokens_per_rank,
                       void* out, int32_t* status, void* stream);

/*
 * Shrink mode: masking ranks of the low-latency path online ("DeepEP V1
 * (legacy) guide", section 6.4: low_latency_update_mask_buffer /
 * low_latency_query_mask_buffer / low_latency_clean_mask_buffer, used for
 * fault tolerance when a rank is lost).
 *
 * The low-latency workspace holds one int32 per rank, 0 (active) in a
 * zero-filled workspace, and it persists across sends. A masked rank neither
 * sends nor receives: a (token, slot) is dropped, exactly as if its index
 * were -1, when the rank holding its expert (e / (E/R)) or the token's source
 * rank (t / (N/R)) is masked. ep_ll_dispatch_send applies the mask as it
 * stands when the send runs (dropped slots are not written, counted or put in
 * the ranges); ep_ll_combine and both combine phases apply it as it stands
 * when they run, so a rank lost between send and combine is skipped there
 * too (a token of a masked source rank combines to +0).
 *
 *   workspace  a low-latency workspace (at least 256 + 4 * num_ranks bytes;
 *              normally the ep_ll_workspace_bytes(...) one the sends use)
 *   rank       0 <= rank < num_ranks; masked != 0 masks it, 0 restores it
 *   mask_out   [num_ranks] int32 device buffer: the current mask
 * Each call is one small launch on the stream, ordered like the others.
 */
int ep_ll_update_mask(void* workspace, size_t workspace_bytes, int num_ranks, int rank, int masked,
                      void* stream);
int ep_ll_query_mask(const void* workspace, size_t workspace_bytes, int num_ranks, int32_t* mask_out,
                     void* stream);
int ep_ll_clean_mask(void* workspace, size_t workspace_bytes, int num_ranks, void* stream);

/*
 * Element-wise fp32 -> FP8 E4M3 conversion (round to nearest even, saturated
 * to +-448, NaN -> NaN), the encoder the FP8 dispatch applies to x / s
 * (DeepEP V1 guide section 5.2(6)). n >= 0 elements; in and out device
 * pointers.
 */
int ep_fp8_e4m3_encode(const float* in, uint8_t* out, int64_t n, void* stream);

/*
 * FP8 quantisation of BF16 rows, exactly as the FP8 dispatch quantises a
 * token's row before copying it ("DeepEP V1 (legacy) guide", sections 5.2(6)
 * and 6.3: E4M3 data with one fp32 scale per 128 channels; round_scale,
 * use_ue8m0): per row and 128-channel block b, s_b = amax_b / 448 (fp32,
 * nearest; raised to the next power of two with EP_FP8_ROUND_SCALE or
 * EP_FP8_UE8M0, and kept >= 2^-127 with EP_FP8_UE8M0), q = e4m3(x / s_b) with
 * a correctly rounded division, rounded to nearest even and saturated to
 * +-448; an all-zero block has s = 0 and q = e4m3(x).
 *
 *   x          [rows, hidden] BF16, 16-byte aligned
 *   rows       >= 0
 *   hidden     a multiple of 128, <= EP_MAX_HIDDEN
 *   fp8_flags  EP_FP8, optionally with EP_FP8_ROUND_SCALE or EP_FP8_UE8M0
 *   q          [rows, hidden] E4M3 bytes, 16-byte aligned
 *   scales     [rows, hidden/128] fp32, or UE8M0 bytes with EP_FP8_UE8M0
 */
int ep_fp8_quantize(const void* x, int64_t rows, int hidden, int fp8_flags, uint8_t* q, void* scales,
                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
