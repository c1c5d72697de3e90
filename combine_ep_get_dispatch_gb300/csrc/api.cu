// The C ABI declared in include/ep.h: argument checks, workspace carving and
// kernel launches. No entry point allocates, frees or synchronises.
#include <stdint.h>

#include "ep.h"
#include "kernels.cuh"

namespace {

using namespace ep;

constexpr int kVersion = 100;  // 0.1.0
constexpr int64_t kEntriesPerCta = 1024;  // (token, slot) entries per layout CTA (measured)
constexpr int kMaxLayoutCtas = 256;
// Low-latency batches up to this many (token, slot) entries take the one-CTA layout.
constexpr int64_t kLLOneCtaMaxEntries = 4096;

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool sizes_ok(int N, int K, int E, int R) {
  if (N < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS) return false;
  if (R < 1 || R > E || E % R != 0) return false;
  if (static_cast<int64_t>(N) * K > INT32_MAX || static_cast<int64_t>(N) * R > INT32_MAX) return false;
  return true;
}

bool hidden_ok(int H, int fp8_flags) {
  if (H < 8 || H > EP_MAX_HIDDEN || H % 8 != 0) return false;
  if ((fp8_flags & EP_FP8) && H % 128 != 0) return false;
  return true;
}

// 0, or EP_FP8 with optional EP_FP8_ROUND_SCALE / EP_FP8_UE8M0.
bool flags_ok(int f) {
  if (f & ~(EP_FP8 | EP_FP8_ROUND_SCALE | EP_FP8_UE8M0)) return false;
  if ((f & (EP_FP8_ROUND_SCALE | EP_FP8_UE8M0)) && !(f & EP_FP8)) return false;
  return true;
}

int layout_ctas_wanted(int N, int K) {
  const int64_t entries = static_cast<int64_t>(N) * K;
  int64_t g = (entries + kEntriesPerCta - 1) / kEntriesPerCta;
  if (g < 1) g = 1;
  if (g > kMaxLayoutCtas) g = kMaxLayoutCtas;
  return static_cast<int>(g);
}

// Layout workspace: [barrier 256 B][chunk counts G x C int32].
struct LayoutWs {
  size_t barrier, chunk, total;
};
LayoutWs layout_ws(int N, int K, int E, int R) {
  LayoutWs w;
  w.barrier = 0;
  w.chunk = 256;
  w.total = w.chunk + align256(sizeof(int32_t) * static_cast<size_t>(layout_ctas_wanted(N, K)) * (E + R));
  return w;
}

// Low-latency workspace: header, shrink-mode rank mask (at a fixed offset, so
// the mask calls need only R), counts, ranges, slot map, chunk counts, barrier.
constexpr size_t kLLMaskOffset = 256;
struct LLWs {
  size_t hdr, mask, count, range, slot, chunk, barrier, total;
};
LLWs ll_ws(int N, int K, int E, int R) {
  LLWs w;
  w.hdr = 0;
  w.mask = kLLMaskOffset;
  w.count = w.mask + align256(sizeof(int32_t) * R);
  w.range = w.count + align256(sizeof(int32_t) * E);
  w.slot = w.range + align256(sizeof(int64_t) * static_cast<size_t>(E) * R);
  w.chunk = w.slot + align256(sizeof(int32_t) * static_cast<size_t>(N) * K);
  w.barrier = w.chunk + align256(sizeof(int32_t) * static_cast<size_t>(R) * E);
  w.total = w.barrier + 256;
  return w;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

bool layout_ok(const ep_layout_t* L) {
  if (!L) return false;
  if (!sizes_ok(L->num_tokens, L->num_topk, L->num_experts, L->num_ranks)) return false;
  if (L->num_tokens > 0 && !L->topk_idx) return false;
  return true;
}

}  // namespace

extern "C" {

int ep_version(void) { return kVersion; }

const char* ep_error_string(int c) {
  switch (c) {
    case EP_OK: return "ok";
    case EP_ERR_INVALID_ARG: return "invalid argument";
    case EP_ERR_ALIGNMENT: return "row buffer not 16-byte aligned";
    case EP_ERR_WORKSPACE: return "workspace missing or too small";
    case EP_ERR_LL_CAPACITY: return "low-latency: tokens per rank exceed max_tokens_per_rank";
    case EP_ERR_CUDA: return "CUDA runtime or launch error";
    case EP_ERR_UNSUPPORTED: return "device lacks a required feature";
    default: break;
  }
  if (c > 0) {
    if (c & EP_ST_BAD_INDEX) return "status: top-k index outside [-1, num_experts)";
    if (c & EP_ST_CAPACITY) return "status: row beyond buffer capacity skipped";
    if (c & EP_ST_LL_OVERFLOW) return "status: low-latency expert region overflow";
    if (c & EP_ST_TIMEOUT) return "status: bounded in-kernel wait timed out";
    if (c & EP_ST_NOT_SENT) return "status: low-latency receive/combine without a send";
    if (c & EP_ST_MISMATCH) return "status: low-latency shapes differ from the send";
    if (c & EP_ST_WORKSPACE) return "status: workspace barrier count not zero on entry (zero-fill it)";
  }
  return "unknown code";
}

size_t ep_layout_workspace_bytes(int N, int K, int E, int R) {
  if (!sizes_ok(N, K, E, R)) return 0;
  return layout_ws(N, K, E, R).total;
}

}  // extern "C"

namespace {

// Checks and parameters of a normal-mode layout into the handle L. Returns
// EP_OK and fills p and G, or an error code (nothing is enqueued).
int layout_setup(const ep_layout_t* L, void* workspace, size_t workspace_bytes, int32_t* status, LayoutParams& p,
                 int& G) {
  if (!layout_ok(L)) return EP_ERR_INVALID_ARG;
  const int N = L->num_tokens, K = L->num_topk, E = L->num_experts, R = L->num_ranks;
  if (!L->num_tokens_per_rank || !L->num_tokens_per_expert || !L->rank_offset || !L->expert_offset)
    return EP_ERR_INVALID_ARG;
  if (L->expert_alignment < 0 || L->expert_alignment > (1 << 16)) return EP_ERR_INVALID_ARG;
  if (N > 0 && (!L->is_token_in_rank || !L->rank_slot || !L->expert_slot)) return EP_ERR_INVALID_ARG;
  const LayoutWs w = layout_ws(N, K, E, R);
  if (!workspace || workspace_bytes < w.total) return EP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EP_ERR_ALIGNMENT;
  G = layout_ctas_wanted(N, K);
  const int gmax = layout_max_ctas(E, R, true);
  if (gmax < 1) return EP_ERR_UNSUPPORTED;
  if (G > gmax) G = gmax;
  p = LayoutParams{};
  p.idx = L->topk_idx;
  p.N = N; p.K = K; p.E = E; p.R = R; p.L = E / R;
  p.tokens_per_cta = (N + G - 1) / G;
  if (p.tokens_per_cta < 1) p.tokens_per_cta = 1;
  p.per_rank = L->num_tokens_per_rank;
  p.per_expert = L->num_tokens_per_expert;
  p.mask = L->is_token_in_rank;
  p.rank_off = L->rank_offset;
  p.expert_off = L->expert_offset;
  p.rank_slot = L->rank_slot;
  p.expert_slot = L->expert_slot;
  p.align = L->expert_alignment > 1 ? L->expert_alignment : 1;
  p.ws_chunk = at<int32_t>(workspace, w.chunk);
  p.ws_barrier = at<unsigned>(workspace, w.barrier);
  p.status = status;
  return EP_OK;
}

// Checks and parameters of a dispatch through the handle L. Returns EP_OK and
// fills p (p.rank_x and p.exp_x both null: nothing to copy), or an error code.
int dispatch_setup(const ep_layout_t* L, const void* x, int hidden, int fp8_flags, const float* topk_weights,
                   const ep_recv_buffer_t* rank_buf, const ep_recv_buffer_t* expert_buf, int32_t* status,
                   DispatchParams& p) {
  if (!layout_ok(L) || !flags_ok(fp8_flags) || !hidden_ok(hidden, fp8_flags)) return EP_ERR_INVALID_ARG;
  const int use_fp8 = fp8_flags & EP_FP8;
  const int N = L->num_tokens, K = L->num_topk, E = L->num_experts, R = L->num_ranks;
  if (N > 0 && !x) return EP_ERR_INVALID_ARG;
  if (!aligned16(x)) return EP_ERR_ALIGNMENT;
  p = DispatchParams{};
  p.x = static_cast<const uint16_t*>(x);
  p.N = N; p.K = K; p.H = hidden; p.E = E; p.R = R; p.L = E / R;
  p.idx = L->topk_idx;
  p.w = topk_weights;
  p.status = status;
  p.overflow_bit = EP_ST_CAPACITY;
  p.fp8_flags = fp8_flags;
  if (rank_buf && rank_buf->x) {
    if (N > 0 && !L->rank_slot) return EP_ERR_INVALID_ARG;
    if (rank_buf->capacity < 0) return EP_ERR_INVALID_ARG;
    if (rank_buf->topk_weights && !topk_weights) return EP_ERR_INVALID_ARG;
    if (!aligned16(rank_buf->x) || (use_fp8 && rank_buf->scales && !aligned16(rank_buf->scales)))
      return EP_ERR_ALIGNMENT;
    p.rank_slot = L->rank_slot;
    p.rank_x = static_cast<uint8_t*>(rank_buf->x);
    p.rank_scales = use_fp8 ? rank_buf->scales : nullptr;
    p.rank_src = rank_buf->src_idx;
    p.rank_topk_idx = rank_buf->topk_idx;
    p.rank_topk_w = rank_buf->topk_weights;
    p.rank_cap = rank_buf->capacity;
  }
  if (expert_buf && expert_buf->x) {
    if (N > 0 && !L->expert_slot) return EP_ERR_INVALID_ARG;
    if (expert_buf->capacity < 0) return EP_ERR_INVALID_ARG;
    if (!aligned16(expert_buf->x) || (use_fp8 && expert_buf->scales && !aligned16(expert_buf->scales)))
      return EP_ERR_ALIGNMENT;
    p.expert_slot = L->expert_slot;
    p.exp_x = static_cast<uint8_t*>(expert_buf->x);
    p.exp_scales = use_fp8 ? expert_buf->scales : nullptr;
    p.exp_src = expert_buf->src_idx;
    p.exp_cap = expert_buf->capacity;
  }
  return EP_OK;
}

// The dispatch launch (after_layout: as the programmatic dependent of the
// layout launched just before by the same call), then, for an aligned layout,
// the zero-fill of the expert-major padding rows.
int dispatch_launch(const ep_layout_t* L, const DispatchParams& p, int fp8_flags, int32_t* status, cudaStream_t s,
                    bool after_layout) {
  if (!p.rank_x && !p.exp_x) return EP_OK;
  const int use_fp8 = fp8_flags & EP_FP8;
  const int rc = cuda_rc(launch_dispatch(p, use_fp8 != 0, s, after_layout));
  if (rc != EP_OK || !p.exp_x || L->expert_alignment <= 1) return rc;
  PadParams pp{};
  pp.expert_off = L->expert_offset;
  pp.per_expert = L->num_tokens_per_expert;
  pp.E = L->num_experts;
  pp.x = p.exp_x;
  pp.row_bytes = static_cast<int64_t>(p.H) * (use_fp8 ? 1 : 2);
  pp.scales = static_cast<uint8_t*>(p.exp_scales);
  pp.scale_row_bytes = static_cast<int64_t>(p.H / 128) * ((fp8_flags & EP_FP8_UE8M0) ? 1 : 4);
  pp.src = p.exp_src;
  pp.cap = p.exp_cap;
  pp.status = status;
  return cuda_rc(launch_pad_zero(pp, s));
}

}  // namespace

namespace ep {

int layout_call(const ep_layout_t* L, void* workspace, size_t workspace_bytes, int32_t* status, cudaStream_t s,
                bool reset_barrier) {
  LayoutParams p;
  int G = 0;
  const int rc = layout_setup(L, workspace, workspace_bytes, status, p, G);
  if (rc != EP_OK) return rc;
  if (reset_barrier && cudaMemsetAsync(p.ws_barrier, 0, 256, s) != cudaSuccess) return EP_ERR_CUDA;
  return cuda_rc(launch_layout(p, G, true, false, s));
}

}  // namespace ep

extern "C" {

int ep_get_dispatch_layout(const ep_layout_t* L, void* workspace, size_t workspace_bytes, int32_t* status,
                           void* stream) {
  return ep::layout_call(L, workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream), false);
}

int ep_dispatch(const ep_layout_t* L, const void* x, int hidden, int fp8_flags, const float* topk_weights,
                const ep_recv_buffer_t* rank_buf, const ep_recv_buffer_t* expert_buf, int32_t* status,
                void* stream) {
  DispatchParams p;
  const int rc = dispatch_setup(L, x, hidden, fp8_flags, topk_weights, rank_buf, expert_buf, status, p);
  if (rc != EP_OK) return rc;
  return dispatch_launch(L, p, fp8_flags, status, static_cast<cudaStream_t>(stream), false);
}

int ep_layout_dispatch(const ep_layout_t* L, void* workspace, size_t workspace_bytes, const void* x, int hidden,
                       int fp8_flags, const float* topk_weights, const ep_recv_buffer_t* rank_buf,
                       const ep_recv_buffer_t* expert_buf, int32_t* status, void* stream) {
  LayoutParams lp;
  DispatchParams dp;
  int G = 0;
  // The dispatch checks first: they need no device, the layout's ask for its
  // co-resident CTA limit.
  int rc = dispatch_setup(L, x, hidden, fp8_flags, topk_weights, rank_buf, expert_buf, status, dp);
  if (rc != EP_OK) return rc;
  rc = layout_setup(L, workspace, workspace_bytes, status, lp, G);
  if (rc != EP_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = cuda_rc(launch_layout(lp, G, true, false, s));
  if (rc != EP_OK) return rc;
  return dispatch_launch(L, dp, fp8_flags, status, s, true);
}

int ep_combine(const ep_layout_t* L, const void* expert_y, int64_t y_rows, int hidden,
               const float* topk_weights, const void* bias, void* out, int32_t* status, void* stream) {
  if (!layout_ok(L) || !hidden_ok(hidden, 0) || y_rows < 0) return EP_ERR_INVALID_ARG;
  const int N = L->num_tokens;
  // topk_weights may be NULL: a unit-weight sum (the backward of dispatch).
  if (N > 0 && (!L->expert_slot || !out || (!expert_y && y_rows > 0))) return EP_ERR_INVALID_ARG;
  if (!aligned16(expert_y) || !aligned16(out) || !aligned16(bias)) return EP_ERR_ALIGNMENT;
  CombineParams p{};
  p.y = static_cast<const uint16_t*>(expert_y);
  p.y_rows = y_rows;
  p.slot = L->expert_slot;
  p.w = topk_weights;
  p.bias = static_cast<const uint16_t*>(bias);
  p.out = static_cast<uint16_t*>(out);
  p.N = N; p.K = L->num_topk; p.H = hidden;
  p.status = status;
  return cuda_rc(launch_combine(p, static_cast<cudaStream_t>(stream)));
}

int ep_combine_to_ranks(const ep_layout_t* L, const void* expert_y, int64_t y_rows, int hidden,
                        const float* topk_weights, void* rank_out, int64_t rank_rows, int32_t* status,
                        void* stream) {
  if (!layout_ok(L) || !hidden_ok(hidden, 0) || y_rows < 0 || rank_rows < 0) return EP_ERR_INVALID_ARG;
  const int N = L->num_tokens;
  if (N > 0 && (!L->expert_slot || !L->rank_slot || !topk_weights || !rank_out || (!expert_y && y_rows > 0)))
    return EP_ERR_INVALID_ARG;
  if (!aligned16(expert_y) || !aligned16(rank_out)) return EP_ERR_ALIGNMENT;
  CombineRanksParams p{};
  p.y = static_cast<const uint16_t*>(expert_y);
  p.y_rows = y_rows;
  p.idx = L->topk_idx;
  p.expert_slot = L->expert_slot;
  p.rank_slot = L->rank_slot;
  p.w = topk_weights;
  p.rank_out = static_cast<uint16_t*>(rank_out);
  p.rank_rows = rank_rows;
  p.N = N; p.K = L->num_topk; p.H = hidden; p.E = L->num_experts; p.R = L->num_ranks;
  p.L = L->num_experts / L->num_ranks;
  p.status = status;
  return cuda_rc(launch_combine_to_ranks(p, static_cast<cudaStream_t>(stream)));
}

int ep_combine_ranks(const ep_layout_t* L, const void* rank_y, int64_t rank_rows, int hidden, const void* bias,
                     void* out, int32_t* status, void* stream) {
  if (!layout_ok(L) || !hidden_ok(hidden, 0) || rank_rows < 0) return EP_ERR_INVALID_ARG;
  const int N = L->num_tokens;
  if (N > 0 && (!L->rank_slot || !out || (!rank_y && rank_rows > 0))) return EP_ERR_INVALID_ARG;
  if (!aligned16(rank_y) || !aligned16(out) || !aligned16(bias)) return EP_ERR_ALIGNMENT;
  CombineParams p{};
  p.y = static_cast<const uint16_t*>(rank_y);
  p.y_rows = rank_rows;
  p.slot = L->rank_slot;  // [N, R]: the ranks play the role of the slots
  p.w = nullptr;          // unweighted sum
  p.bias = static_cast<const uint16_t*>(bias);
  p.out = static_cast<uint16_t*>(out);
  p.N = N; p.K = L->num_ranks; p.H = hidden;
  p.status = status;
  return cuda_rc(launch_combine(p, static_cast<cudaStream_t>(stream)));
}

int ep_combine_backward(const ep_layout_t* L, const void* grad_out, const void* expert_y, int64_t y_rows,
                        int hidden, const float* topk_weights, void* grad_y, float* grad_w, int32_t* status,
                        void* stream) {
  if (!layout_ok(L) || !hidden_ok(hidden, 0) || y_rows < 0) return EP_ERR_INVALID_ARG;
  const int N = L->num_tokens;
  if (N > 0 && (!L->expert_slot || !grad_out || !topk_weights)) return EP_ERR_INVALID_ARG;
  if (grad_w && !expert_y && y_rows > 0) return EP_ERR_INVALID_ARG;
  if (!aligned16(grad_out) || !aligned16(expert_y) || !aligned16(grad_y)) return EP_ERR_ALIGNMENT;
  if (!grad_y && !grad_w) return EP_OK;
  CombineBwdParams p{};
  p.grad_out = static_cast<const uint16_t*>(grad_out);
  p.y = static_cast<const uint16_t*>(expert_y);
  p.y_rows = y_rows;
  p.slot = L->expert_slot;
  p.w = topk_weights;
  p.grad_y = static_cast<uint16_t*>(grad_y);
  p.grad_w = grad_w;
  p.N = N; p.K = L->num_topk; p.H = hidden;
  p.status = status;
  return cuda_rc(launch_combine_backward(p, static_cast<cudaStream_t>(stream)));
}

size_t ep_ll_workspace_bytes(int N, int K, int E, int R, int T) {
  if (!sizes_ok(N, K, E, R) || T < 1) return 0;
  return ll_ws(N, K, E, R).total;
}

// The combine side of shrink mode: the mask as it stands when the combine runs.
static void set_ll_mask(CombineParams& p, void* ws, const LLWs& w, int N, int E, int R, int T) {
  p.rank_mask = at<int32_t>(ws, w.mask);
  p.ll_cap = static_cast<int64_t>(R) * T;
  p.ll_L = E / R;
  p.ll_ns = N / R > 0 ? N / R : 1;
}

static int ll_common_checks(int N, int K, int E, int R, int T) {
  if (!sizes_ok(N, K, E, R) || T < 1) return EP_ERR_INVALID_ARG;
  if (N % R != 0) return EP_ERR_INVALID_ARG;
  if (N / R > T) return EP_ERR_LL_CAPACITY;
  if (static_cast<int64_t>(E) * R * T > INT32_MAX) return EP_ERR_INVALID_ARG;
  return EP_OK;
}

int ep_ll_dispatch_send(const void* x, const int32_t* topk_idx, int N, int K, int H, int E, int R, int T,
                        int fp8_flags, void* recv_x, void* recv_scales, int32_t* recv_src, void* workspace,
                        size_t workspace_bytes, int32_t* status, void* stream) {
  int rc = ll_common_checks(N, K, E, R, T);
  if (rc != EP_OK) return rc;
  if (!flags_ok(fp8_flags) || !hidden_ok(H, fp8_flags)) return EP_ERR_INVALID_ARG;
  const int use_fp8 = fp8_flags & EP_FP8;
  if (!recv_x || (N > 0 && (!x || !topk_idx))) return EP_ERR_INVALID_ARG;
  if (use_fp8 && !recv_scales) return EP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(recv_x) || (use_fp8 && !aligned16(recv_scales))) return EP_ERR_ALIGNMENT;
  const LLWs w = ll_ws(N, K, E, R);
  if (!workspace || workspace_bytes < w.total) return EP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EP_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // Without the layout kernel when the routing table is small enough: a
  // small batch in one launch (each block derives its slots from the whole
  // routing table, one block publishes counts, ranges and header), a larger
  // one by a per-source histogram kernel and its dependent row kernel.
  if (ll_send_form(N, K, E, R) != LLSendForm::kLayout) {
    LLSendParams sp{};
    sp.x = static_cast<const uint16_t*>(x);
    sp.idx = topk_idx;
    sp.N = N; sp.K = K; sp.H = H; sp.E = E; sp.R = R; sp.L = E / R;
    sp.ns = N / R;
    sp.cap = static_cast<int64_t>(R) * T;
    sp.fp8_flags = fp8_flags;
    sp.recv_x = static_cast<uint8_t*>(recv_x);
    sp.recv_scales = use_fp8 ? recv_scales : nullptr;
    sp.recv_src = recv_src;
    sp.count = at<int32_t>(workspace, w.count);
    sp.range = at<int64_t>(workspace, w.range);
    sp.slot_map = at<int32_t>(workspace, w.slot);
    sp.hdr = at<LLHeader>(workspace, w.hdr);
    sp.hdr_value = LLHeader{kMagicSent, N, K, E, R, T, H, use_fp8, 0};
    sp.rank_mask = at<int32_t>(workspace, w.mask);
    sp.hist = at<int32_t>(workspace, w.chunk);  // [R, E]: the chunk-count area
    sp.status = status;
    return cuda_rc(launch_ll_send(sp, s));
  }

  const int gmax = layout_max_ctas(E, R, false);
  if (gmax < 1 || R > gmax) return EP_ERR_UNSUPPORTED;

  // A small batch runs the layout as one CTA with a group of g warps per
  // source rank (no grid barrier, no exchange of chunk counts through
  // memory); each source rank's entries must split evenly over its g warps
  // in whole multiples of 32.
  const int ns = N / R;
  int g = R <= 32 ? 32 / R : 0;
  while (g > 0 && (ns * K) % (32 * g) != 0) --g;
  const bool one_cta = N > 0 && g > 0 && static_cast<int64_t>(N) * K <= kLLOneCtaMaxEntries;
  LayoutParams lp{};
  lp.idx = topk_idx;
  lp.N = N; lp.K = K; lp.E = E; lp.R = R; lp.L = E / R;
  lp.tokens_per_cta = one_cta ? N : (ns > 0 ? ns : 1);
  lp.ll_src_entries = one_cta ? ns * K : 0;
  lp.ll_src_warps = one_cta ? g : 0;
  lp.per_expert = at<int32_t>(workspace, w.count);
  lp.expert_slot = at<int32_t>(workspace, w.slot);
  lp.ll_cap = static_cast<int64_t>(R) * T;
  lp.ll_range = at<int64_t>(workspace, w.range);
  lp.ll_hdr = at<LLHeader>(workspace, w.hdr);
  lp.hdr_value = LLHeader{kMagicSent, N, K, E, R, T, H, use_fp8, 0};
  lp.ws_chunk = at<int32_t>(workspace, w.chunk);
  lp.ws_barrier = at<unsigned>(workspace, w.barrier);
  lp.rank_mask = at<int32_t>(workspace, w.mask);
  lp.status = status;
  rc = cuda_rc(launch_layout(lp, one_cta ? 1 : R, false, true, s));
  if (rc != EP_OK) return rc;

  DispatchParams dp{};
  dp.x = static_cast<const uint16_t*>(x);
  dp.N = N; dp.K = K; dp.H = H; dp.E = E; dp.R = R; dp.L = E / R;
  dp.idx = topk_idx;
  dp.expert_slot = at<int32_t>(workspace, w.slot);
  dp.exp_x = static_cast<uint8_t*>(recv_x);
  dp.exp_scales = use_fp8 ? recv_scales : nullptr;
  dp.fp8_flags = fp8_flags;
  dp.exp_src = recv_src;
  dp.exp_cap = static_cast<int64_t>(E) * R * T;
  dp.exp_src_is_token = 1;
  dp.overflow_bit = EP_ST_LL_OVERFLOW;
  dp.status = status;
  return cuda_rc(launch_dispatch(dp, use_fp8 != 0, s, /*after_layout=*/true));
}

int ep_ll_dispatch_recv(void* workspace, size_t workspace_bytes, int N, int K, int E, int R, int T,
                        int32_t* recv_count, int64_t* layout_range, int32_t* cumulative_recv_stats,
                        int32_t* status, void* stream) {
  int rc = ll_common_checks(N, K, E, R, T);
  if (rc != EP_OK) return rc;
  if (!recv_count) return EP_ERR_INVALID_ARG;
  const LLWs w = ll_ws(N, K, E, R);
  if (!workspace || workspace_bytes < w.total) return EP_ERR_WORKSPACE;
  void* ws = workspace;
  LLRecvParams p{};
  p.hdr = at<LLHeader>(ws, w.hdr);
  p.count = at<int32_t>(ws, w.count);
  p.range = at<int64_t>(ws, w.range);
  p.expect = LLHeader{kMagicSent, N, K, E, R, T, 0, 0, 0};
  p.recv_count = recv_count;
  p.layout_range = layout_range;
  p.stats = cumulative_recv_stats;
  p.status = status;
  return cuda_rc(launch_ll_recv(p, E, R, static_cast<cudaStream_t>(stream)));
}

int ep_ll_combine(const void* expert_y, const float* topk_weights, const void* bias, const void* workspace,
                  size_t workspace_bytes, int N, int K, int H, int E, int R, int T, void* out, int32_t* status,
                  void* stream) {
  int rc = ll_common_checks(N, K, E, R, T);
  if (rc != EP_OK) return rc;
  if (!hidden_ok(H, 0)) return EP_ERR_INVALID_ARG;
  if (!expert_y || (N > 0 && (!topk_weights || !out))) return EP_ERR_INVALID_ARG;
  if (!aligned16(expert_y) || !aligned16(out) || !aligned16(bias)) return EP_ERR_ALIGNMENT;
  const LLWs w = ll_ws(N, K, E, R);
  if (!workspace || workspace_bytes < w.total) return EP_ERR_WORKSPACE;
  void* ws = const_cast<void*>(workspace);
  CombineParams p{};
  p.y = static_cast<const uint16_t*>(expert_y);
  p.y_rows = static_cast<int64_t>(E) * R * T;
  p.slot = at<int32_t>(ws, w.slot);
  p.w = topk_weights;
  p.bias = static_cast<const uint16_t*>(bias);
  p.out = static_cast<uint16_t*>(out);
  p.N = N; p.K = K; p.H = H;
  p.ll_hdr = at<LLHeader>(ws, w.hdr);
  p.ll_expect = LLHeader{kMagicSent, N, K, E, R, T, H, 0, 0};
  set_ll_mask(p, ws, w, N, E, R, T);
  p.status = status;
  return cuda_rc(launch_combine(p, static_cast<cudaStream_t>(stream)));
}

int ep_ll_combine_send(const void* expert_y, const void* workspace, size_t workspace_bytes, int N, int K, int H,
                       int E, int R, int T, void* staging, int32_t* status, void* stream) {
  int rc = ll_common_checks(N, K, E, R, T);
  if (rc != EP_OK) return rc;
  if (!hidden_ok(H, 0)) return EP_ERR_INVALID_ARG;
  if (!expert_y || (N > 0 && !staging)) return EP_ERR_INVALID_ARG;
  if (!aligned16(expert_y) || !aligned16(staging)) return EP_ERR_ALIGNMENT;
  const LLWs w = ll_ws(N, K, E, R);
  if (!workspace || workspace_bytes < w.total) return EP_ERR_WORKSPACE;
  void* ws = const_cast<void*>(workspace);
  CombineParams p{};
  p.y = static_cast<const uint16_t*>(expert_y);
  p.y_rows = static_cast<int64_t>(E) * R * T;
  p.slot = at<int32_t>(ws, w.slot);
  p.out = static_cast<uint16_t*>(staging);
  p.N = N; p.K = K; p.H = H;
  p.gather = 1;
  p.ll_hdr = at<LLHeader>(ws, w.hdr);
  p.ll_expect = LLHeader{kMagicSent, N, K, E, R, T, H, 0, 0};
  set_ll_mask(p, ws, w, N, E, R, T);
  p.status = status;
  return cuda_rc(launch_combine(p, static_cast<cudaStream_t>(stream)));
}

int ep_ll_combine_recv(const void* staging, const float* topk_weights, const void* bias, const void* workspace,
                       size_t workspace_bytes, int N, int K, int H, int E, int R, int T, void* out,
                       int32_t* status, void* stream) {
  int rc = ll_common_checks(N, K, E, R, T);
  if (rc != EP_OK) return rc;
  if (!hidden_ok(H, 0)) return EP_ERR_INVALID_ARG;
  if (N > 0 && (!staging || !topk_weights || !out)) return EP_ERR_INVALID_ARG;
  if (!aligned16(staging) || !aligned16(out) || !aligned16(bias)) return EP_ERR_ALIGNMENT;
  const LLWs w = ll_ws(N, K, E, R);
  if (!workspace || workspace_bytes < w.total) return EP_ERR_WORKSPACE;
  void* ws = const_cast<void*>(workspace);
  CombineParams p{};
  p.y = static_cast<const uint16_t*>(staging);
  p.y_rows = static_cast<int64_t>(N) * K;
  p.slot = at<int32_t>(ws, w.slot);
  p.token_major = 1;
  p.w = topk_weights;
  p.bias = static_cast<const uint16_t*>(bias);
  p.out = static_cast<uint16_t*>(out);
  p.N = N; p.K = K; p.H = H;
  p.ll_hdr = at<LLHeader>(ws, w.hdr);
  p.ll_expect = LLHeader{kMagicSent, N, K, E, R, T, H, 0, 0};
  set_ll_mask(p, ws, w, N, E, R, T);
  p.status = status;
  return cuda_rc(launch_combine(p, static_cast<cudaStream_t>(stream)));
}

static int ll_mask_call(void* workspace, size_t workspace_bytes, int R, int mode, int rank, int value,
                        int32_t* out, void* stream) {
  if (R < 1 || R > EP_MAX_EXPERTS) return EP_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kLLMaskOffset + sizeof(int32_t) * R) return EP_ERR_WORKSPACE;
  return cuda_rc(launch_ll_mask(at<int32_t>(workspace, kLLMaskOffset), R, mode, rank, value, out,
                                static_cast<cudaStream_t>(stream)));
}

int ep_ll_update_mask(void* workspace, size_t workspace_bytes, int num_ranks, int rank, int masked,
                      void* stream) {
  if (rank < 0 || rank >= num_ranks) return EP_ERR_INVALID_ARG;
  return ll_mask_call(workspace, workspace_bytes, num_ranks, 0, rank, masked ? 1 : 0, nullptr, stream);
}

int ep_ll_query_mask(const void* workspace, size_t workspace_bytes, int num_ranks, int32_t* mask_out,
                     void* stream) {
  if (!mask_out) return EP_ERR_INVALID_ARG;
  return ll_mask_call(const_cast<void*>(workspace), workspace_bytes, num_ranks, 1, 0, 0, mask_out, stream);
}

int ep_ll_clean_mask(void* workspace, size_t workspace_bytes, int num_ranks, void* stream) {
  return ll_mask_call(workspace, workspace_bytes, num_ranks, 2, 0, 0, nullptr, stream);
}

int ep_fp8_quantize(const void* x, int64_t rows, int hidden, int fp8_flags, uint8_t* q, void* scales,
                    void* stream) {
  if (!flags_ok(fp8_flags) || !(fp8_flags & EP_FP8) || !hidden_ok(hidden, fp8_flags) || rows < 0)
    return EP_ERR_INVALID_ARG;
  if (rows > 0 && (!x || !q || !scales)) return EP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q)) return EP_ERR_ALIGNMENT;
  return cuda_rc(launch_quantize_rows(static_cast<const uint16_t*>(x), rows, hidden, fp8_flags, q, scales,
                                      static_cast<cudaStream_t>(stream)));
}

int ep_fp8_e4m3_encode(const float* in, uint8_t* out, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return EP_ERR_INVALID_ARG;
  return cuda_rc(launch_e4m3_encode(in, out, n, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
