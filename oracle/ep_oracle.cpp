// Oracle for MoE token layout, dispatch and combine: TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU restatement of what the hot path
// computes. It is used by the tests, by the package's smoke check and by the
// benchmark's CPU baseline; nothing in the product path may call it. It shares
// no code, header, table or helper with the CUDA library: every encoder below
// is written from the format's definition.
//
// Sources (the DeepEP write-ups this project follows):
//  * "DeepEP Ascend deep dive" (kongchang.com), section "Two Transfers:
//    Dispatch and Combine": a token reaches a card once even when several of
//    its experts live there; combine weights each expert output by the router
//    score and sums. Section "Dispatch's Three Phases": tokens are cloned once
//    per chosen expert and reordered by expert (the "expand" layout); the
//    volume example 16,384 x 7,168 x 2 B x 6 copies.
//  * "DeepEP lesson 14" (hpc.payai.win), section "practice task": dispatch
//    appends (i, x_i) to expert e's queue for every (i, k) in order; combine
//    adds w_ik * f_e(x_i) for every k.
//  * "DeepEP V1 (legacy) guide" (zskr.cn), section 5.2(1): the layout returns
//    num_tokens_per_rank, num_tokens_per_expert and the is_token_in_rank mask;
//    section 5.2(6): FP8 data with float scales of shape [tokens, hidden/128];
//    section 6.1/6.3: low-latency receive buffer
//    [num_local_experts, num_ranks * max_tokens, hidden] plus per-expert
//    receive counts; -1 in topk_idx is a legal "no expert".
//
// Readings where the pages leave a step open (each one is listed with its
// reason in the design notes of this repository):
//  * expert e lives on rank e / (E / R) (contiguous blocks of experts);
//  * slots are assigned in (token, top-k) order: global token order is
//    source-rank-then-token order when tokens are split contiguously;
//  * an index outside [-1, E) is treated as masked and raises EP_BAD_INDEX;
//  * FP8: s = amax / 448 in fp32 (round to nearest), q = e4m3(x / s) with an
//    IEEE fp32 division, round to nearest even, saturating to +-448; an
//    all-zero block has s = 0 and q = e4m3(x) (signed zeros);
//  * combine: acc = +0, then acc = fmaf(w_k, y_k, acc) for k ascending over
//    unmasked slots, output BF16 rounded to nearest even.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fno-fast-math -shared -fPIC.
// The only fused multiply-add is the explicit std::fmaf of the combine.
// A second build of this same file with -fopenmp (libep_oracle_omp.so) runs
// the per-token row loops of dispatch and combine, the per-expert loop of the
// low-latency dispatch and the per-row loop of quantize_rows on every host
// core: those iterations write disjoint rows, so the results are identical;
// the layout stays sequential. It exists to time the oracle on all cores next
// to the plain build and to run the large exhaustive quantisation check.

#include <cmath>
#include <cstdint>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <cstring>
#include <utility>
#include <vector>

namespace {

// Data-dependent conditions, reported as bits of the returned status.
constexpr int kBadIndex = 1;   // an index outside [-1, E)
constexpr int kCapacity = 2;   // a destination row beyond the given capacity
constexpr int kLLOverflow = 4; // more than T tokens from one source rank

// ---------------------------------------------------------------- BF16 ----
// BF16 is the upper half of an IEEE binary32 word. Rounding to nearest even
// looks at the discarded lower half: above the midpoint rounds up, at the
// midpoint rounds to the even upper half. NaN stays NaN (made quiet).
uint16_t bf16_from_f32(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  const bool is_nan = (u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0;
  if (is_nan) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t upper = u >> 16;
  const uint32_t lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;
  return static_cast<uint16_t>(upper);
}

float f32_from_bf16(uint16_t h) {
  const uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// ---------------------------------------------------------------- E4M3 ----
// OCP 8-bit floating point, E4M3 ("fn": finite, no infinities): 1 sign bit,
// 4 exponent bits with bias 7, 3 mantissa bits. Exponent field 0 holds
// subnormals m * 2^-9; fields 1..15 hold (1 + m/8) * 2^(field - 7), except
// field 15 with m = 7, which is NaN. The largest finite value is 448.

double round_half_even(double y) {
  const double f = std::floor(y);
  const double d = y - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return std::fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

uint8_t e4m3_from_f32(float v) {
  if (std::isnan(v)) return 0x7F;
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(v));
  if (a >= 448.0) return sign | 0x7E;  // saturate to the largest finite value
  if (a < 0.015625) {                  // below 2^-6: quantum 2^-9
    const double n = round_half_even(a * 512.0);  // 0..8; 8 is the code of 2^-6
    return sign | static_cast<uint8_t>(n);
  }
  int e2;
  std::frexp(a, &e2);          // a = m * 2^e2 with m in [0.5, 1)
  const int ex = e2 - 1;       // floor(log2 a), in [-6, 8]
  const double quantum = std::ldexp(1.0, ex - 3);
  const double n = round_half_even(a / quantum);  // 8..16, exact division
  int code = ((ex + 7) << 3) + static_cast<int>(n) - 8;  // n == 16 carries
  if (code > 0x7E) code = 0x7E;
  return sign | static_cast<uint8_t>(code);
}

double e4m3_to_f64(uint8_t c) {
  const double s = (c & 0x80) ? -1.0 : 1.0;
  const int field = (c >> 3) & 0xF;
  const int m = c & 0x7;
  if (field == 15 && m == 7) return std::nan("");
  if (field == 0) return s * std::ldexp(static_cast<double>(m), -9);
  return s * std::ldexp(1.0 + m / 8.0, field - 7);
}

// Scale variants ("DeepEP V1 (legacy) guide", section 6.3: round_scale,
// use_ue8m0). Flag bits as in the library's dispatch flags.
constexpr int kFp8 = 1, kRoundScale = 2, kUe8m0 = 4;

// Smallest power of two >= s (s > 0), by frexp: s = m * 2^e with m in [0.5, 1).
float pow2_ceil(float s) {
  int e;
  const double m = std::frexp(static_cast<double>(s), &e);
  return static_cast<float>(m == 0.5 ? static_cast<double>(s) : std::ldexp(1.0, e));
}

// UE8M0 byte of a power of two s = 2^k: k + 127 (s = 0 -> 0).
uint8_t ue8m0_of(float s) {
  if (s == 0.0f) return 0;
  int e;
  std::frexp(static_cast<double>(s), &e);  // s = 0.5 * 2^e
  return static_cast<uint8_t>(e - 1 + 127);
}

// Per 128-channel block b of one BF16 row: amax_b = max |x|, s_b = amax_b / 448
// (fp32, round to nearest), q = e4m3(x / s_b). With round_scale, s_b is first
// raised to the next power of two; with UE8M0 it is also kept >= 2^-127 (the
// smallest UE8M0 value) when the block is not all zero.
void quantize_row(const uint16_t* x, int H, uint8_t* q, float* scales, int flags = kFp8) {
  for (int b = 0; b < H / 128; ++b) {
    float amax = 0.0f;
    for (int i = 0; i < 128; ++i) {
      const float a = std::fabs(f32_from_bf16(x[b * 128 + i]));
      if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    if ((flags & (kRoundScale | kUe8m0)) && s > 0.0f) s = pow2_ceil(s);
    if ((flags & kUe8m0) && amax > 0.0f && s < std::ldexp(1.0f, -127)) s = std::ldexp(1.0f, -127);
    scales[b] = s;
    for (int i = 0; i < 128; ++i) {
      const float xi = f32_from_bf16(x[b * 128 + i]);
      q[b * 128 + i] = (s > 0.0f) ? e4m3_from_f32(xi / s) : e4m3_from_f32(xi);
    }
  }
}

bool valid_expert(int32_t e, int E) { return e >= 0 && e < E; }

// Copy token t's already encoded row (BF16 or E4M3) into destination row
// `row` of a receive buffer, with its scales: fp32, or UE8M0 bytes.
void write_row(const uint8_t* payload, const float* scales, int H, int flags,
               void* dst_x, void* dst_scales, int64_t row) {
  const bool fp8 = flags & kFp8;
  const size_t row_bytes = static_cast<size_t>(H) * (fp8 ? 1 : 2);
  std::memcpy(static_cast<uint8_t*>(dst_x) + row * row_bytes, payload, row_bytes);
  if (!fp8 || !dst_scales) return;
  const int nsc = H / 128;
  if (flags & kUe8m0) {
    uint8_t* d = static_cast<uint8_t*>(dst_scales) + row * nsc;
    for (int b = 0; b < nsc; ++b) d[b] = ue8m0_of(scales[b]);
  } else {
    std::memcpy(static_cast<float*>(dst_scales) + row * nsc, scales, sizeof(float) * nsc);
  }
}

}  // namespace

extern "C" {

// Threads the row loops use: 1 in the plain build, the OpenMP team size in
// the all-core build (compiled from this same file with -fopenmp).
int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

uint16_t oracle_bf16_from_f32(float f) { return bf16_from_f32(f); }
uint8_t oracle_e4m3_from_f32(float f) { return e4m3_from_f32(f); }
double oracle_e4m3_to_f64(uint8_t c) { return e4m3_to_f64(c); }

void oracle_bf16_from_f32_n(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_from_f32(in[i]);
}

void oracle_e4m3_from_f32_n(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_from_f32(in[i]);
}

// rows x H BF16 -> rows x H E4M3 and rows x H/128 fp32 scales (flags: kFp8
// plus optional kRoundScale / kUe8m0).
void oracle_quantize_rows(const uint16_t* x, int64_t rows, int H, uint8_t* q, float* scales, int flags) {
  // Rows are independent: split over threads in the all-core build.
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    quantize_row(x + r * H, H, q + r * H, scales + r * (H / 128), flags | kFp8);
}

// fp32 power-of-two scales -> UE8M0 bytes.
void oracle_ue8m0_from_scales(const float* s, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ue8m0_of(s[i]);
}

// Routing layout.
//   per_expert[e]  = #{(t,k) : idx[t,k] == e}
//   mask[t,r]      = 1 if some k has a valid idx[t,k] on rank r (one copy per rank)
//   per_rank[r]    = sum_t mask[t,r]
//   expert_off, rank_off: exclusive prefix sums, length E+1 and R+1
//   expert_slot[t,k] = expert_off[e] + position of (t,k) in expert e's list
//   rank_slot[t,r]   = rank_off[r] + position of t in rank r's list
// Lists are built by visiting (t, k) in order, so they are in token order.
int oracle_layout(const int32_t* idx, int N, int K, int E, int R, int expert_alignment,
                  int32_t* per_rank, int32_t* per_expert, uint8_t* mask,
                  int32_t* rank_off, int32_t* expert_off,
                  int32_t* rank_slot, int32_t* expert_slot) {
  int status = 0;
  const int L = E / R;
  std::vector<std::vector<std::pair<int, int>>> expert_list(E);
  std::vector<std::vector<int>> rank_list(R);
  std::vector<char> seen(R);
  for (int t = 0; t < N; ++t) {
    std::fill(seen.begin(), seen.end(), 0);
    for (int k = 0; k < K; ++k) {
      const int32_t e = idx[static_cast<int64_t>(t) * K + k];
      if (e == -1) continue;
      if (!valid_expert(e, E)) { status |= kBadIndex; continue; }
      expert_list[e].push_back({t, k});
      const int r = e / L;
      if (!seen[r]) { seen[r] = 1; rank_list[r].push_back(t); }
    }
  }
  // With an alignment A > 1 each expert's segment is padded to a multiple of
  // A rows ("DeepEP Ascend deep dive", "Dispatch's Three Phases": expert
  // alignment to 128 for the grouped GEMM; the padding rows are zeros).
  const int A = expert_alignment > 1 ? expert_alignment : 1;
  expert_off[0] = 0;
  for (int e = 0; e < E; ++e) {
    per_expert[e] = static_cast<int32_t>(expert_list[e].size());
    const int32_t seg = (per_expert[e] + A - 1) / A * A;
    expert_off[e + 1] = expert_off[e] + seg;
  }
  rank_off[0] = 0;
  for (int r = 0; r < R; ++r) {
    per_rank[r] = static_cast<int32_t>(rank_list[r].size());
    rank_off[r + 1] = rank_off[r] + per_rank[r];
  }
  for (int64_t i = 0; i < static_cast<int64_t>(N) * K; ++i) expert_slot[i] = -1;
  for (int64_t i = 0; i < static_cast<int64_t>(N) * R; ++i) { rank_slot[i] = -1; mask[i] = 0; }
  for (int e = 0; e < E; ++e)
    for (size_t j = 0; j < expert_list[e].size(); ++j) {
      const auto [t, k] = expert_list[e][j];
      expert_slot[static_cast<int64_t>(t) * K + k] = expert_off[e] + static_cast<int32_t>(j);
    }
  for (int r = 0; r < R; ++r)
    for (size_t j = 0; j < rank_list[r].size(); ++j) {
      const int t = rank_list[r][j];
      rank_slot[static_cast<int64_t>(t) * R + r] = rank_off[r] + static_cast<int32_t>(j);
      mask[static_cast<int64_t>(t) * R + r] = 1;
    }
  return status;
}

// Dispatch: every token row goes once to each rank in its mask (per-rank
// receive buffer, rows packed by rank_off) and once per unmasked top-k slot to
// the expert-major buffer (rows packed by expert_off). In FP8 mode the row is
// quantised once and the same bytes and scales are written to every copy.
// Per-rank metadata: src[row] = t; topk_idx[row,k] = local expert id if
// expert k of t lives on that rank, else -1; topk_w[row,k] = w or 0.
// Expert-major metadata: src[row] = t*K + k. Any output pointer may be null.
int oracle_dispatch(const uint16_t* x, const int32_t* idx, const float* w,
                    int N, int K, int H, int E, int R, int flags,
                    const int32_t* rank_slot, const int32_t* expert_slot,
                    void* rank_x, void* rank_scales, int32_t* rank_src,
                    int32_t* rank_topk_idx, float* rank_topk_w, int64_t rank_cap,
                    void* exp_x, void* exp_scales, int32_t* exp_src, int64_t exp_cap) {
  const bool use_fp8 = flags & kFp8;
  int status = 0;
  const int L = E / R;
  // Tokens are independent (each writes only its own destination rows), so
  // the all-core build splits this loop over threads; the plain build runs
  // it in order. The results are the same either way.
#pragma omp parallel reduction(| : status)
  {
  std::vector<uint8_t> q(H);
  std::vector<float> sc(H / 128 > 0 ? H / 128 : 1);
#pragma omp for schedule(dynamic, 16)
  for (int t = 0; t < N; ++t) {
    const uint16_t* xt = x + static_cast<int64_t>(t) * H;
    const uint8_t* payload = reinterpret_cast<const uint8_t*>(xt);
    if (use_fp8) {
      quantize_row(xt, H, q.data(), sc.data(), flags);
      payload = q.data();
    }
    for (int r = 0; r < R; ++r) {
      const int32_t row = rank_slot[static_cast<int64_t>(t) * R + r];
      if (row < 0) continue;
      if (row >= rank_cap) { status |= kCapacity; continue; }
      if (rank_x) write_row(payload, sc.data(), H, flags, rank_x, rank_scales, row);
      if (rank_src) rank_src[row] = t;
      for (int k = 0; k < K; ++k) {
        const int32_t e = idx[static_cast<int64_t>(t) * K + k];
        const bool here = valid_expert(e, E) && e / L == r;
        if (rank_topk_idx) rank_topk_idx[static_cast<int64_t>(row) * K + k] = here ? e - r * L : -1;
        if (rank_topk_w) rank_topk_w[static_cast<int64_t>(row) * K + k] = here ? w[static_cast<int64_t>(t) * K + k] : 0.0f;
      }
    }
    for (int k = 0; k < K; ++k) {
      const int32_t row = expert_slot[static_cast<int64_t>(t) * K + k];
      if (row < 0) continue;
      if (row >= exp_cap) { status |= kCapacity; continue; }
      if (exp_x) write_row(payload, sc.data(), H, flags, exp_x, exp_scales, row);
      if (exp_src) exp_src[row] = t * K + k;
    }
  }
  }
  return status;
}

// Combine: out[t] = bf16( sum over k ascending with slot[t,k] >= 0 of
// w[t,k] * y[slot[t,k]] ), each term added with one fp32 fused multiply-add
// onto an accumulator that starts at +0. An optional bias row (the shared
// expert's output, "DeepEP Ascend deep dive", "Combine: More Output, Same
// Cost") is added in fp32 after the last term, before the one BF16 rounding.
// w may be null: every weight is 1.
int oracle_combine(const uint16_t* y, int64_t y_rows, const int32_t* slot, const float* w,
                   const uint16_t* bias, int N, int K, int H, uint16_t* out) {
  int status = 0;
  // Tokens are independent: split over threads in the all-core build.
#pragma omp parallel reduction(| : status)
  {
  std::vector<float> acc(H);
#pragma omp for schedule(dynamic, 16)
  for (int t = 0; t < N; ++t) {
    std::fill(acc.begin(), acc.end(), 0.0f);
    for (int k = 0; k < K; ++k) {
      const int32_t row = slot[static_cast<int64_t>(t) * K + k];
      if (row < 0) continue;
      if (row >= y_rows) { status |= kCapacity; continue; }
      const float wk = w ? w[static_cast<int64_t>(t) * K + k] : 1.0f;
      const uint16_t* yr = y + static_cast<int64_t>(row) * H;
      for (int h = 0; h < H; ++h) acc[h] = std::fmaf(wk, f32_from_bf16(yr[h]), acc[h]);
    }
    if (bias)
      for (int h = 0; h < H; ++h) acc[h] = acc[h] + f32_from_bf16(bias[static_cast<int64_t>(t) * H + h]);
    for (int h = 0; h < H; ++h) out[static_cast<int64_t>(t) * H + h] = bf16_from_f32(acc[h]);
  }
  }
  return status;
}

// Combine backward (training reuse, "DeepEP V1 (legacy) guide" 5.1: the
// backward of combine is a dispatch). For out[t] = sum_k w[t,k] y[slot[t,k]]:
//   grad_y[slot[t,k]] = bf16( w[t,k] * grad_out[t] )          (fp32 product)
//   grad_w[t,k]       = sum_h grad_out[t,h] * y[slot[t,k],h]  (double here;
//                        the library's fp32 sum is checked within its bound)
// Masked slots get nothing (grad_w = 0).
int oracle_combine_backward(const uint16_t* grad_out, const uint16_t* y, int64_t y_rows, const int32_t* slot,
                            const float* w, int N, int K, int H, uint16_t* grad_y, double* grad_w) {
  int status = 0;
  for (int t = 0; t < N; ++t)
    for (int k = 0; k < K; ++k) {
      const int64_t tk = static_cast<int64_t>(t) * K + k;
      const int32_t row = slot[tk];
      if (grad_w) grad_w[tk] = 0.0;
      if (row < 0) continue;
      if (row >= y_rows) { status |= kCapacity; continue; }
      const uint16_t* g = grad_out + static_cast<int64_t>(t) * H;
      if (grad_y)
        for (int h = 0; h < H; ++h)
          grad_y[static_cast<int64_t>(row) * H + h] = bf16_from_f32(w[tk] * f32_from_bf16(g[h]));
      if (grad_w && y) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
          acc += static_cast<double>(f32_from_bf16(g[h])) * f32_from_bf16(y[static_cast<int64_t>(row) * H + h]);
        grad_w[tk] = acc;
      }
    }
  return status;
}

// Two-level combine, first level (the expert layer's reduction on each rank,
// as in DeepEP's normal combine(x, handle), "DeepEP V1 (legacy) guide" 5.1):
// for every (t, r) in the mask, rank_out[rank_slot[t,r]] = bf16( sum over k
// ascending whose expert lives on r of w[t,k] * y[expert_slot[t,k]] ).
int oracle_combine_to_ranks(const uint16_t* y, int64_t y_rows, const int32_t* idx, const int32_t* expert_slot,
                            const int32_t* rank_slot, const float* w, int N, int K, int E, int R, int H,
                            uint16_t* rank_out, int64_t rank_rows) {
  int status = 0;
  const int L = E / R;
  std::vector<float> acc(H);
  for (int t = 0; t < N; ++t)
    for (int r = 0; r < R; ++r) {
      const int32_t orow = rank_slot[static_cast<int64_t>(t) * R + r];
      if (orow < 0) continue;
      if (orow >= rank_rows) { status |= kCapacity; continue; }
      std::fill(acc.begin(), acc.end(), 0.0f);
      for (int k = 0; k < K; ++k) {
        const int64_t tk = static_cast<int64_t>(t) * K + k;
        const int32_t e = idx[tk];
        if (!valid_expert(e, E) || e / L != r) continue;
        const int32_t row = expert_slot[tk];
        if (row < 0) continue;
        if (row >= y_rows) { status |= kCapacity; continue; }
        for (int h = 0; h < H; ++h)
          acc[h] = std::fmaf(w[tk], f32_from_bf16(y[static_cast<int64_t>(row) * H + h]), acc[h]);
      }
      for (int h = 0; h < H; ++h) rank_out[static_cast<int64_t>(orow) * H + h] = bf16_from_f32(acc[h]);
    }
  return status;
}

// Two-phase low-latency combine, send half: the output row of every routed
// (token, slot) is copied back to the token-major staging row t*K + k.
int oracle_gather_rows(const uint16_t* y, int64_t y_rows, const int32_t* slot, int N, int K, int H,
                       uint16_t* staging) {
  int status = 0;
  for (int t = 0; t < N; ++t)
    for (int k = 0; k < K; ++k) {
      const int64_t tk = static_cast<int64_t>(t) * K + k;
      const int32_t row = slot[tk];
      if (row < 0) continue;
      if (row >= y_rows) { status |= kCapacity; continue; }
      std::memcpy(staging + tk * H, y + static_cast<int64_t>(row) * H, sizeof(uint16_t) * H);
    }
  return status;
}

// Two-phase low-latency combine, receive half: the weighted sum of the
// staged rows t*K + k over the slots the send did route (slot[t,k] >= 0), in
// slot order, one fused multiply-add per term, BF16 at the end.
int oracle_combine_staged(const uint16_t* staging, const int32_t* slot, const float* w, int N, int K, int H,
                          uint16_t* out) {
  std::vector<float> acc(H);
  for (int t = 0; t < N; ++t) {
    std::fill(acc.begin(), acc.end(), 0.0f);
    for (int k = 0; k < K; ++k) {
      const int64_t tk = static_cast<int64_t>(t) * K + k;
      if (slot[tk] < 0) continue;
      const float wk = w[tk];
      for (int h = 0; h < H; ++h) acc[h] = std::fmaf(wk, f32_from_bf16(staging[tk * H + h]), acc[h]);
    }
    for (int h = 0; h < H; ++h) out[static_cast<int64_t>(t) * H + h] = bf16_from_f32(acc[h]);
  }
  return 0;
}

// Low-latency dispatch. Tokens are split contiguously over R source ranks,
// n_s = N / R each (n_s <= T). The receive buffer of expert e is the fixed
// region [e][0 .. R*T) of recv_x [E, R*T, H]; the rank owning e sees it as
// its local expert e - r*L, i.e. [L, R*T, H] per rank. Expert e's received
// rows are packed at j = 0 .. count-1 in token order; rows at j >= count are
// not written.
//   recv_count[e]      = number of (t,k) routed to e
//   recv_src[e, j]     = global token index of row j
//   layout_range[e, s] = (offset << 32) | count for the rows from source s
//   slot_map[t, k]     = e * R*T + j, or -1 if masked
int oracle_ll_dispatch(const uint16_t* x, const int32_t* idx, int N, int K, int H,
                       int E, int R, int T, int flags,
                       void* recv_x, void* recv_scales, int32_t* recv_src,
                       int32_t* recv_count, int64_t* layout_range, int32_t* slot_map) {
  int status = 0;
  const int n_s = N / R;
  if (n_s > T) status |= kLLOverflow;
  const int64_t cap = static_cast<int64_t>(R) * T;
  std::vector<std::vector<std::pair<int, int>>> expert_list(E);
  for (int t = 0; t < N; ++t)
    for (int k = 0; k < K; ++k) {
      const int32_t e = idx[static_cast<int64_t>(t) * K + k];
      slot_map[static_cast<int64_t>(t) * K + k] = -1;
      if (e == -1) continue;
      if (!valid_expert(e, E)) { status |= kBadIndex; continue; }
      expert_list[e].push_back({t, k});
    }
  // Experts are independent (each fills only its own region): split over
  // threads in the all-core build.
#pragma omp parallel reduction(| : status)
  {
  std::vector<uint8_t> q(H);
  std::vector<float> sc(H / 128 > 0 ? H / 128 : 1);
#pragma omp for schedule(dynamic, 1)
  for (int e = 0; e < E; ++e) {
    recv_count[e] = static_cast<int32_t>(expert_list[e].size());
    std::vector<int64_t> count_from(R, 0);
    for (size_t j = 0; j < expert_list[e].size(); ++j) {
      const auto [t, k] = expert_list[e][j];
      if (static_cast<int64_t>(j) >= cap) { status |= kLLOverflow; continue; }
      const int64_t row = static_cast<int64_t>(e) * cap + static_cast<int64_t>(j);
      const uint16_t* xt = x + static_cast<int64_t>(t) * H;
      const uint8_t* payload = reinterpret_cast<const uint8_t*>(xt);
      if (flags & kFp8) { quantize_row(xt, H, q.data(), sc.data(), flags); payload = q.data(); }
      write_row(payload, sc.data(), H, flags, recv_x, recv_scales, row);
      recv_src[row] = t;
      slot_map[static_cast<int64_t>(t) * K + k] = static_cast<int32_t>(row);
      const int s = (n_s > 0) ? t / n_s : 0;
      if (s < R) count_from[s] += 1;
    }
    int64_t offset = 0;
    for (int s = 0; s < R; ++s) {
      layout_range[static_cast<int64_t>(e) * R + s] = (offset << 32) | count_from[s];
      offset += count_from[s];
    }
  }
  }
  return status;
}

// Shrink mode ("DeepEP V1 (legacy) guide", section 6.4: a rank can be masked
// out online with low_latency_update_mask_buffer and restored with
// low_latency_clean_mask_buffer). A masked rank neither sends nor receives,
// so a (token, slot) is dropped, exactly as if its index were -1, when the
// rank holding its expert (e / L) or the token's source rank (t / n_s, n_s =
// N / R) is masked. Out-of-range indices are left as they are (the dispatch
// reports them).
int oracle_ll_mask_routing(const int32_t* idx, int N, int K, int E, int R, const int32_t* rank_mask,
                           int32_t* out) {
  const int L = E / R;
  const int n_s = N / R;
  for (int t = 0; t < N; ++t)
    for (int k = 0; k < K; ++k) {
      const int64_t tk = static_cast<int64_t>(t) * K + k;
      const int32_t e = idx[tk];
      out[tk] = e;
      if (!valid_expert(e, E)) continue;
      const int src = n_s > 0 ? t / n_s : 0;
      if (rank_mask[e / L] != 0 || (src < R && rank_mask[src] != 0)) out[tk] = -1;
    }
  return 0;
}

// The same rule applied when the combine runs to a low-latency slot map
// (entries e * R*T + j, or -1): the mask may have changed since the send.
int oracle_ll_mask_slot_map(const int32_t* slot_map, int N, int K, int E, int R, int T,
                            const int32_t* rank_mask, int32_t* out) {
  const int L = E / R;
  const int n_s = N / R;
  const int64_t cap = static_cast<int64_t>(R) * T;
  for (int t = 0; t < N; ++t)
    for (int k = 0; k < K; ++k) {
      const int64_t tk = static_cast<int64_t>(t) * K + k;
      const int32_t row = slot_map[tk];
      out[tk] = row;
      if (row < 0) continue;
      const int e = static_cast<int>(row / cap);
      const int src = n_s > 0 ? t / n_s : 0;
      if (rank_mask[e / L] != 0 || (src < R && rank_mask[src] != 0)) out[tk] = -1;
    }
  return 0;
}

}  // extern "C"
