// Kernel parameter blocks and launchers (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep.h"

namespace ep {

// Workspace header of the low-latency path: written by the send, checked by
// the receive and the combine.
struct LLHeader {
  unsigned long long magic;
  int32_t N, K, E, R, T, H, use_fp8, pad;
};
constexpr unsigned long long kMagicSent = 0x4C4C2D53454E5421ull;      // "LL-SENT!"
constexpr unsigned long long kMagicReceived = 0x4C4C2D5245435644ull;  // "LL-RECVD"

struct LayoutParams {
  const int32_t* idx;  // [N, K]
  int N, K, E, R, L;
  int tokens_per_cta;
  int align;                  // expert segments padded to a multiple of `align` rows (1: packed)
  uint32_t magic_L, magic_K;  // ceil(2^32 / d) for d = L, K (0 when d == 1): exact n / d for n < 2^20
  int bits_E, bits_R;         // bits of the largest expert / rank id
  // normal-mode outputs
  int32_t* per_rank;
  int32_t* per_expert;
  uint8_t* mask;
  int32_t* rank_off;
  int32_t* expert_off;
  int32_t* rank_slot;
  int32_t* expert_slot;  // low-latency mode: the slot map (row e * ll_cap + j)
  // low-latency mode outputs
  int64_t ll_cap;
  int64_t* ll_range;   // [E, R]
  LLHeader* ll_hdr;
  LLHeader hdr_value;
  const int32_t* rank_mask;  // low-latency shrink mode: [R], non-zero = masked (or null)
  int ll_src_entries;        // > 0: one-CTA low-latency form: source rank s holds entries
                             // [s * ll_src_entries, (s + 1) * ll_src_entries), on warps
  int ll_src_warps;          // [s * ll_src_warps, (s + 1) * ll_src_warps) (R * ll_src_warps <= 32)
  // scratch
  int32_t* ws_chunk;   // [G, C]
  unsigned* ws_barrier;
  int32_t* status;
};

struct DispatchParams {
  const uint16_t* x;  // [N, H] BF16
  int N, K, H, E, R, L;
  const int32_t* idx;
  const float* w;
  const int32_t* expert_slot;  // [N, K] destination rows (low-latency: slot map)
  const int32_t* rank_slot;    // [N, R] or null
  int fp8_flags;              // EP_FP8_ROUND_SCALE / EP_FP8_UE8M0 (FP8 kernel only)
  // per-rank buffer (null x: skip)
  uint8_t* rank_x;
  void* rank_scales;          // fp32, or UE8M0 bytes
  int32_t* rank_src;
  int32_t* rank_topk_idx;
  float* rank_topk_w;
  int64_t rank_cap;
  // expert-major buffer (null x: skip)
  uint8_t* exp_x;
  void* exp_scales;
  int32_t* exp_src;
  int64_t exp_cap;
  int exp_src_is_token;  // 1: exp_src[row] = t (low-latency recv_src); 0: t * K + k
  int overflow_bit;      // status bit for a row beyond exp_cap
  int32_t* status;
};

// The low-latency send without the layout kernel (ll_send_small_kernel, or
// ll_hist_kernel + ll_send_rows_kernel).
struct LLSendParams {
  const uint16_t* x;          // [N, H] BF16
  const int32_t* idx;         // [N, K]
  int N, K, H, E, R, L;
  int ns;                     // tokens per source rank (N / R)
  int64_t cap;                // R * T rows per expert region
  int fp8_flags;              // 0: BF16 rows; EP_FP8 (+ scale format flags)
  uint8_t* recv_x;            // [E, cap, H] BF16 words or E4M3 bytes
  void* recv_scales;          // [E, cap, H/128] fp32 or UE8M0 bytes (FP8), or null
  int32_t* recv_src;          // [E, cap] or null
  int32_t* count;             // [E] workspace: rows routed to each expert
  int64_t* range;             // [E, R] workspace: (offset << 32) | count per source rank
  int32_t* slot_map;          // [N, K] workspace: e * cap + j, or -1
  LLHeader* hdr;
  LLHeader hdr_value;
  const int32_t* rank_mask;   // [R] shrink mode, non-zero = masked
  int nsplit;                 // blocks per token, each one span of the row
  int span;                   // channels per span
  uint32_t magic_nsK, magic_L, magic_R;  // ceil(2^32 / d) for d = ns * K, L, R (0 when d == 1)
  int32_t* hist;              // [R, E] workspace: routed entries per (source rank, expert) (larger form)
  int32_t* status;
};

struct CombineParams {
  const uint16_t* y;     // [y_rows, H] BF16
  int64_t y_rows;
  const int32_t* slot;   // [N, K] rows of y, -1 = masked
  const float* w;        // [N, K]; null: every weight is 1
  const uint16_t* bias;  // [N, H] BF16 added after the weighted sum, or null
  uint16_t* out;         // [N, H]; gather mode: [N * K, H]
  int N, K, H;
  int token_major;       // read row t*K + k (for slot >= 0) instead of the slot value
  int gather;            // copy every routed row to out[t*K + k] instead of summing
  const LLHeader* ll_hdr;  // low-latency: the send's header (null in normal mode)
  LLHeader ll_expect;
  // low-latency shrink mode: slots of masked ranks are skipped (rank_mask null: none)
  const int32_t* rank_mask;  // [R]
  int64_t ll_cap;            // R * T rows per expert region
  int ll_L, ll_ns;           // experts per rank, tokens per source rank
  int32_t* status;
};

struct CombineRanksParams {
  const uint16_t* y;           // [y_rows, H] expert-major BF16 expert outputs
  int64_t y_rows;
  const int32_t* idx;          // [N, K]
  const int32_t* expert_slot;  // [N, K]
  const int32_t* rank_slot;    // [N, R]
  const float* w;              // [N, K]
  uint16_t* rank_out;          // [rank_rows, H]
  int64_t rank_rows;
  int N, K, H, E, R, L;
  int32_t* status;
};

struct CombineBwdParams {
  const uint16_t* grad_out;  // [N, H]
  const uint16_t* y;         // [y_rows, H] forward expert outputs, or null (no grad_w)
  int64_t y_rows;
  const int32_t* slot;       // [N, K]
  const float* w;            // [N, K]
  uint16_t* grad_y;          // [y_rows, H] or null
  float* grad_w;             // [N, K] or null
  int N, K, H;
  int32_t* status;
};

struct PadParams {
  const int32_t* expert_off;   // [E+1] aligned offsets
  const int32_t* per_expert;   // [E] true counts
  int E;
  uint8_t* x;                  // expert-major rows
  int64_t row_bytes;
  uint8_t* scales;             // scale rows or null
  int64_t scale_row_bytes;
  int32_t* src;                // or null
  int64_t cap;
  int32_t* status;
};

struct LLRecvParams {
  LLHeader* hdr;
  const int32_t* count;   // [E]
  const int64_t* range;   // [E, R]
  LLHeader expect;
  int32_t* recv_count;
  int64_t* layout_range;
  int32_t* stats;             // cumulative per-expert receive counts, or null
  int32_t* status;
};

// Host-side launch bookkeeping, asked of the runtime once per process
// (launch_cache.cu). current_device() is -1 on failure; the others return 0 /
// false on failure.
int current_device();
int device_sms(int dev);
bool device_cooperative(int dev);
cudaError_t ensure_dynamic_smem(const void* fn, int dev, size_t smem);  // raise the kernel's limit to >= smem
int blocks_per_sm(const void* fn, int dev, int threads, size_t smem);   // occupancy, 0 on failure

// The routing layout of ep_get_dispatch_layout: every check first (an error
// code, with nothing enqueued), then, when reset_barrier is set, a zero fill
// of the workspace's 256-byte barrier block, then the launch.
int layout_call(const ep_layout_t* L, void* workspace, size_t workspace_bytes, int32_t* status, cudaStream_t s,
                bool reset_barrier);

// Launchers: return cudaSuccess or the launch error.
size_t layout_smem_bytes(int E, int R, bool with_rank);
int layout_max_ctas(int E, int R, bool with_rank);  // co-resident limit (device-specific)
cudaError_t launch_layout(const LayoutParams& p, int G, bool with_rank, bool ll, cudaStream_t s);

// after_layout: the kernel just before on the stream is this library's
// layout, launched by the same call; the dispatch then starts as its
// programmatic dependent (rows loaded and quantised while the layout runs).
cudaError_t launch_dispatch(const DispatchParams& p, bool fp8, cudaStream_t s, bool after_layout = false);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_combine_to_ranks(const CombineRanksParams& p, cudaStream_t s);
cudaError_t launch_combine_backward(const CombineBwdParams& p, cudaStream_t s);
cudaError_t launch_pad_zero(const PadParams& p, cudaStream_t s);
// Forms of the low-latency send (ll_send_form): one launch for a small batch
// (N * K <= kLLSmallMaxEntries); a per-source histogram kernel and its
// dependent row kernel for a larger one (N * K <= kLLMidMaxEntries, (N / R) * K <=
// kLLMidMaxSourceEntries); both need E * R <= kLLSmallMaxTable. Otherwise
// the routing layout kernel and the dispatch kernel.
constexpr int kLLSmallMaxEntries = 4096;
constexpr int kLLSmallMaxTable = 16384;
constexpr int kLLMidMaxEntries = 65536;
constexpr int kLLMidMaxSourceEntries = 8192;
enum class LLSendForm { kSmall, kMid, kLayout };
LLSendForm ll_send_form(int N, int K, int E, int R);
cudaError_t launch_ll_send(LLSendParams p, cudaStream_t s);  // kSmall or kMid
cudaError_t launch_ll_mask(int32_t* mask, int R, int mode, int rank, int value, int32_t* out, cudaStream_t s);
cudaError_t launch_ll_recv(const LLRecvParams& p, int E, int R, cudaStream_t s);
cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, int64_t n, cudaStream_t s);
cudaError_t launch_quantize_rows(const uint16_t* x, int64_t rows, int H, int fp8_flags, uint8_t* q, void* scales,
                                 cudaStream_t s);

}  // namespace ep
