// Dispatch on sm_103a: scatter each token's hidden row into the per-rank and
// expert-major receive buffers (and, for the low-latency send, into the
// fixed per-expert regions), optionally quantised once to FP8 E4M3 with one
// fp32 scale per 128 channels.
//
// What it computes ("DeepEP V1 (legacy) guide", sections 5.1 and 5.2(6);
// "DeepEP Ascend deep dive", "Two Transfers" and "Dispatch's Three Phases"):
//   per-rank rows   rank_x[rank_slot[t, r]] = row(t) for each rank r in t's mask
//   expert rows     exp_x[expert_slot[t, k]] = row(t) for each unmasked slot k
//   FP8 row(t)      per block b of 128 channels: s_b = amax_b / 448 (fp32,
//                   nearest), q = e4m3_rn_satfinite(x / s_b); s_b = 0 -> q = e4m3(x)
//
// Design (HBM-bound, write-heavy: one row read, ~R'+K' rows written).
// BF16: a warp per token and one shared-memory row per warp. Lane 0 brings
// the row in with one bulk TMA copy (cp.async.bulk global->shared, completion
// on an mbarrier); every destination row is one bulk TMA store
// (cp.async.bulk shared->global) issued by the lane that owns that
// destination, so the copy engine generates the addresses and the SM issues
// ~R'+K' instructions per token. Grid: one token per warp; the block
// scheduler hands out blocks as earlier ones retire, which balances tokens
// with many copies against tokens with few.
// FP8: bulk TMA in, quantised in place in shared memory, bulk TMA out (see
// dispatch_fp8_kernel below): one token per block of four warps, one bulk
// store per destination row.
#include "common.cuh"
#include "kernels.cuh"

namespace ep {

namespace {

constexpr int kMaxWarps = 4;

__host__ __device__ inline unsigned round_up(unsigned v, unsigned a) { return (v + a - 1) / a * a; }

// Shared memory of one warp: one staged BF16 row (2H bytes, rounded to 128).
__host__ __device__ inline unsigned bf16_row_bytes(int H) { return round_up(static_cast<unsigned>(H) * 2u, 128u); }

constexpr unsigned kBarBytes = 128;  // one mbarrier per warp

// A warp per token, one token per warp: lane 0 brings the row in with one
// bulk TMA copy completing on the warp's mbarrier; every destination row then
// leaves by one bulk TMA store from the same shared row. The block scheduler
// balances the work: with a grid of one token per warp, blocks retiring as
// their rows leave, the 16384-token workload ran 12 % faster than on a
// persistent grid (whose warps each own a fixed share of the tokens, so the
// grid waits for the warp whose tokens have the most copies).
__global__ void __launch_bounds__(kMaxWarps * 32) dispatch_bf16_kernel(const DispatchParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, W = blockDim.x >> 5;
  const int H = p.H, K = p.K, R = p.R, L = p.L, E = p.E;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * W + w;
  if (t >= p.N) return;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem) + w;
  uint8_t* src = smem + kBarBytes + static_cast<size_t>(w) * bf16_row_bytes(H);
  const unsigned xbytes = static_cast<unsigned>(H) * 2u;
  const unsigned obytes = xbytes;
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, xbytes);
    bulk_g2s(src, p.x + t * H, xbytes, bar);
  }
  __syncwarp();

  // The slots come from the layout: under a programmatic dependent launch
  // this kernel may have started before the layout finished (the row load
  // above needs nothing from it).
  grid_dependency_wait();
  // This lane's top-k slot (lane < K): expert, weight and expert-major row;
  // and its first rank's per-rank row. Every lookup goes out before any
  // store (a store through a pointer that may alias would hold back the
  // loads after it).
  int e_k = -1;
  float w_k = 0.0f;
  int32_t erow = -1;
  if (lane < K) {
    e_k = __ldg(p.idx + t * K + lane);
    if (p.w) w_k = __ldg(p.w + t * K + lane);
    if (p.exp_x) erow = __ldcg(p.expert_slot + t * K + lane);
  }
  int32_t rrow0 = (p.rank_x && lane < R) ? __ldcg(p.rank_slot + t * R + lane) : -1;
  const int rank_k = (e_k >= 0 && e_k < E) ? e_k / L : -1;
  const int local_k = e_k - rank_k * L;
  if (erow >= p.exp_cap) {
    flag(p.status, p.overflow_bit);
    erow = -1;
  }
  if (erow >= 0 && p.exp_src)
    p.exp_src[erow] = p.exp_src_is_token ? static_cast<int32_t>(t) : static_cast<int32_t>(t * K + lane);

  // Every lane sees the row land itself (its stores read it); the warp
  // leaves together if any lane's bounded wait gave up.
  const bool ok = mbar_wait(bar, 0, p.status);
  if (!__all_sync(0xffffffffu, ok)) {
    // Timed out: the row load may still be in flight into this warp's
    // shared row. Let it land (bounded) before the block can exit and its
    // shared memory go to another block; no store has been issued yet.
    if (lane == 0) mbar_drain(bar, 0);
    __syncwarp();
    return;
  }

  // Expert-major copies.
  if (erow >= 0) bulk_s2g(p.exp_x + static_cast<int64_t>(erow) * obytes, src, obytes);

  // Per-rank copies: lane owns ranks lane, lane + 32, ...
  if (p.rank_x) {
    for (int r0 = 0; r0 < R; r0 += 32) {
      const int r = r0 + lane;
      int32_t rrow = r0 == 0 ? rrow0 : ((r < R) ? __ldcg(p.rank_slot + t * R + r) : -1);
      if (rrow >= p.rank_cap) {
        flag(p.status, EP_ST_CAPACITY);
        rrow = -1;
      }
      if (rrow >= 0) {
        bulk_s2g(p.rank_x + static_cast<int64_t>(rrow) * obytes, src, obytes);
        if (p.rank_src) p.rank_src[rrow] = static_cast<int32_t>(t);
      }
      if (p.rank_topk_idx || p.rank_topk_w) {
        for (int kk = 0; kk < K; ++kk) {
          const int rk = __shfl_sync(0xffffffffu, rank_k, kk);
          const int lk = __shfl_sync(0xffffffffu, local_k, kk);
          const float wk = __shfl_sync(0xffffffffu, w_k, kk);
          if (rrow >= 0) {
            const bool here = rk == r;
            if (p.rank_topk_idx) p.rank_topk_idx[static_cast<int64_t>(rrow) * K + kk] = here ? lk : -1;
            if (p.rank_topk_w) p.rank_topk_w[static_cast<int64_t>(rrow) * K + kk] = here ? wk : 0.0f;
          }
        }
      }
    }
  }
  bulk_commit();
  // The shared row must outlive the stores' reads of it.
  bulk_wait_read<0>();
}

// ---- FP8 dispatch ---------------------------------------------------------------
// A block of four warps per token. Thread 0 brings the token's BF16 row into
// shared memory with one bulk TMA load (the whole row in flight at once); the
// warps then quantise it in place, 512 channels per warp per step: lanes own
// 16 consecutive channels (8 lanes = one 128-channel block), take the block's
// max by shuffles, divide by the scale (correctly rounded) and convert to
// E4M3, writing the codes over the front of the staged row. As soon as a
// step's 2048 channels are quantised they leave by one bulk store
// (cp.async.bulk shared->global) per destination row, while the next step is
// quantised; the scales follow with plain stores (a UE8M0 scale row is not a
// multiple of 16 bytes). Launched with at most 105 KB of staged rows per SM
// (7 tokens of hidden 7168): every first-wave block loads its row at once, so
// the cap shortens the read burst and the synchronous quantisation before the
// first stores (measured on GB300: the 4096-token hidden-7168 dispatch went
// from 85 to 79 us with the three changes; the PM-sampled DRAM timeline had
// shown ~8 us without traffic between the first wave's loads and its stores).
// Measured on GB300 (all bit-identical): the row loaded through registers one
// step ahead (each token then waits out ~14 load latencies behind the write
// traffic); a separate E4M3 row (fewer tokens in flight); one warp per token
// (each token's chain of load, quantisation and stores is longer, so the
// kernel's ramp and tail are too: four warps took the 4096-token FP8
// dispatches from 90.1 to 86.0 us and 79.9 to 74.2 us).
constexpr int kF8Warps = 4;                  // warps per token (one token per block)
constexpr size_t kF8StagedBytesPerSM = 105 * 1024;  // see launch_fp8
constexpr size_t kF8MaxBlocksPerSM = 10;
constexpr size_t kSmemPerSM = 228 * 1024;            // shared memory of one SM
constexpr size_t kSmemReservedPerBlock = 1024;       // the runtime's share of it per block
constexpr int kF8MaxDest = 2 * EP_MAX_TOPK;  // <= K expert copies + <= K rank copies

// Smallest power of two >= s for s >= 0 (exact on the bit pattern; a
// subnormal m * 2^-149 rounds to the next power of two of m).
__device__ __forceinline__ float pow2_ceil(float s) {
  unsigned u = __float_as_uint(s);
  if (u == 0u) return s;
  if ((u & 0x7F800000u) == 0u) return __uint_as_float(u == 1u ? 1u : (1u << (32 - __clz(u - 1u))));
  if (u & 0x007FFFFFu) u = (u & 0xFF800000u) + 0x00800000u;
  return __uint_as_float(u);
}

// UE8M0 byte 2^(b - 127) of a power-of-two scale >= 2^-127 (0 for s = 0).
__device__ __forceinline__ uint8_t ue8m0_byte(float s) {
  return static_cast<uint8_t>((__float_as_uint(s) >> 23) & 0xFFu);
}

// Packed fp32 pairs (lo in the low word): the sm_100-family f32x2
// arithmetic, one instruction for two IEEE fp32 operations.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return pack_e4m3x2(a, b) | (pack_e4m3x2(c, d) << 16);
}

// Per half of two packed BF16 pairs: max(|a|, |b|) (exact, as any max is),
// with a sign bit the caller drops.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The sign bits of four BF16 values (two packed pairs, in channel order)
// placed at bit 7 of four code bytes.
__device__ __forceinline__ uint32_t bf16_signs4(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, 0x7531) & 0x80808080u;
}

// 16 BF16 channels of one lane -> 16 E4M3 codes; the 8 lanes of a 128-channel
// block share the block's scale s = amax / 448, raised to a power of two with
// EP_FP8_ROUND_SCALE, and also kept >= 2^-127 with EP_FP8_UE8M0 (all 32 lanes
// must call it).
__device__ __forceinline__ uint4 quantize16(const uint4& v0, const uint4& v1, float& sc, int flags) {
  float f[16];
  f[0] = bf16_lo(v0.x); f[1] = bf16_hi(v0.x); f[2] = bf16_lo(v0.y); f[3] = bf16_hi(v0.y);
  f[4] = bf16_lo(v0.z); f[5] = bf16_hi(v0.z); f[6] = bf16_lo(v0.w); f[7] = bf16_hi(v0.w);
  f[8] = bf16_lo(v1.x); f[9] = bf16_hi(v1.x); f[10] = bf16_lo(v1.y); f[11] = bf16_hi(v1.y);
  f[12] = bf16_lo(v1.z); f[13] = bf16_hi(v1.z); f[14] = bf16_lo(v1.w); f[15] = bf16_hi(v1.w);
  uint32_t m2 = bf16x2_absmax(v0.x, v0.y);
  m2 = bf16x2_absmax(m2, v0.z);
  m2 = bf16x2_absmax(m2, v0.w);
  m2 = bf16x2_absmax(m2, v1.x);
  m2 = bf16x2_absmax(m2, v1.y);
  m2 = bf16x2_absmax(m2, v1.z);
  m2 = bf16x2_absmax(m2, v1.w);
  // (fmaxf returns the other operand for a NaN: a NaN channel is left out of
  // the amax, as when the maximum is taken over each channel in turn from 0.)
  float m = fmaxf(0.0f, fmaxf(__uint_as_float((m2 << 16) & 0x7FFFFFFFu), __uint_as_float(m2 & 0x7FFF0000u)));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  sc = __fdiv_rn(m, 448.0f);
  if ((flags & (EP_FP8_ROUND_SCALE | EP_FP8_UE8M0)) && sc > 0.0f) sc = pow2_ceil(sc);
  if ((flags & EP_FP8_UE8M0) && m > 0.0f) sc = fmaxf(sc, __uint_as_float(0x00400000u));  // 2^-127
  if (sc > 0.0f) {
    if (sc >= 0x1p-92f && sc <= 0x1p126f) {
      // x / s, correctly rounded, from one correctly rounded reciprocal
      // y = 1/s per block: q0 = x * y is within an ulp of x / s, the
      // remainder x - s * q0 is exact by a fused multiply-add, and
      // q0 + remainder * y rounds to x / s (Markstein's correction step,
      // "Computation of elementary functions on the IBM RISC System/6000
      // processor", IBM J. Res. Dev. 34(1), 1990). The remainder is exact
      // only if it does not underflow: for |x / s| >= 2^-11 (below that
      // every E4M3 code is a zero) it is a multiple of 2^(e_s - 57), which
      // s >= 2^-92 keeps at or above 2^-149; s <= 2^126 keeps y normal.
      // Smaller or larger scales take the IEEE division. Two channels per
      // instruction (packed fp32 pairs, each lane rounded as its own fp32
      // operation). The codes take x's sign at the end: the correction
      // turns -0 / s into +0, every other quotient already has it. A device
      // test compares every (x, amax) pair of BF16 inputs with the oracle's
      // IEEE division.
      const float y = __frcp_rn(sc);
      const uint64_t y2 = pack_f32x2(y, y), ns2 = pack_f32x2(-sc, -sc);
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const uint64_t x2 = pack_f32x2(f[i], f[i + 1]);
        const uint64_t q0 = mul_f32x2(x2, y2);
        const uint64_t r = fma_f32x2(ns2, q0, x2);
        unpack_f32x2(fma_f32x2(r, y2, q0), f[i], f[i + 1]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = __fdiv_rn(f[i], sc);
    }
  }
  // Each code takes its input's sign bit: it changes only the +0 that the
  // correction step makes of -0 / s (a quotient's sign is x's otherwise, and
  // the codes of s = 0 are x's own).
  uint4 q;
  q.x = e4m3x4(f[0], f[1], f[2], f[3]) | bf16_signs4(v0.x, v0.y);
  q.y = e4m3x4(f[4], f[5], f[6], f[7]) | bf16_signs4(v0.z, v0.w);
  q.z = e4m3x4(f[8], f[9], f[10], f[11]) | bf16_signs4(v1.x, v1.y);
  q.w = e4m3x4(f[12], f[13], f[14], f[15]) | bf16_signs4(v1.z, v1.w);
  return q;
}

// Shared memory of one warp: the staged row (2H bytes: BF16 in, then E4M3
// codes in its first H bytes, the source of the bulk stores), the row's
// H/128 scales and its destination rows (expert-major rows first, then
// per-rank rows).
__host__ __device__ inline unsigned f8_row_bytes(int H) { return round_up(static_cast<unsigned>(H) * 2u, 128u); }
__host__ __device__ inline unsigned f8_warp_bytes(int H) {
  return f8_row_bytes(H) + round_up(static_cast<unsigned>(H / 128) * 4u + kF8MaxDest * 4u, 128u);
}

// Destination rows of token t, listed in the warp's shared `drow` (expert-
// major rows first, then per-rank rows), with each row's metadata written
// (source index; per-rank local top-k ids and weights). Returns the number
// of rows and sets `ne` to the expert-major ones. All 32 lanes call it; e_k
// and w_k are lane k's expert and weight (lane < K).
__device__ __forceinline__ int f8_destinations(const DispatchParams& p, int64_t t, int lane, int e_k, float w_k,
                                               int32_t* drow, int& ne) {
  const int K = p.K, R = p.R, L = p.L, E = p.E;
  // Every lookup goes out before any store below: the stores go through
  // pointers the compiler must assume may alias the slot arrays, so a load
  // issued after one waits for it.
  int32_t erow = (lane < K && p.exp_x) ? __ldcg(p.expert_slot + t * K + lane) : -1;
  int32_t rrow = (p.rank_x && lane < R) ? __ldcg(p.rank_slot + t * R + lane) : -1;
  // This slot's rank and local expert id, for the per-rank top-k metadata.
  const int rank_k = (e_k >= 0 && e_k < E) ? e_k / L : -1;
  const int local_k = e_k - rank_k * L;
  if (erow >= p.exp_cap) {
    flag(p.status, p.overflow_bit);
    erow = -1;
  }
  if (erow >= 0 && p.exp_src)
    p.exp_src[erow] = p.exp_src_is_token ? static_cast<int32_t>(t) : static_cast<int32_t>(t * K + lane);
  const unsigned vm = __ballot_sync(0xffffffffu, erow >= 0);
  if (erow >= 0) drow[__popc(vm & lanemask_lt())] = erow;
  ne = __popc(vm);
  int n = ne;
  if (p.rank_x) {
    for (int rb = 0; rb < R; rb += 32) {
      const int r = rb + lane;
      if (rb > 0) rrow = (r < R) ? __ldcg(p.rank_slot + t * R + r) : -1;
      if (rrow >= p.rank_cap) {
        flag(p.status, EP_ST_CAPACITY);
        rrow = -1;
      }
      const unsigned rm = __ballot_sync(0xffffffffu, rrow >= 0);
      // at most K ranks hold a copy of one token; the list has room for K more
      if (rrow >= 0) {
        const int pos = n + __popc(rm & lanemask_lt());
        if (pos < kF8MaxDest) drow[pos] = rrow;
        if (p.rank_src) p.rank_src[rrow] = static_cast<int32_t>(t);
      }
      n = min(n + __popc(rm), kF8MaxDest);
      if (p.rank_topk_idx || p.rank_topk_w) {
        for (int kk = 0; kk < K; ++kk) {
          const int rk = __shfl_sync(0xffffffffu, rank_k, kk);
          const int lk = __shfl_sync(0xffffffffu, local_k, kk);
          const float wk = __shfl_sync(0xffffffffu, w_k, kk);
          if (rrow >= 0) {
            const bool here = rk == r;
            if (p.rank_topk_idx) p.rank_topk_idx[static_cast<int64_t>(rrow) * K + kk] = here ? lk : -1;
            if (p.rank_topk_w) p.rank_topk_w[static_cast<int64_t>(rrow) * K + kk] = here ? wk : 0.0f;
          }
        }
      }
    }
  }
  return n;
}

// kLateDest: the destinations are looked up after the row is quantised, behind
// a wait for the preceding grid (the layout, when the two are launched as a
// programmatic dependent pair), so the row's load and quantisation overlap
// the layout. Otherwise the lookups go first, while the row is in flight.
template <bool kLateDest>
__global__ void __launch_bounds__(kF8Warps * 32) dispatch_fp8_kernel(const DispatchParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_n, s_ne;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int H = p.H, K = p.K;
  const int nsc = H / 128;
  const int64_t t = blockIdx.x;  // one token per block
  if (t >= p.N) return;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  uint8_t* row = smem + kBarBytes;
  float* scales = reinterpret_cast<float*>(row + f8_row_bytes(H));
  int32_t* drow = reinterpret_cast<int32_t*>(scales + nsc);
  const unsigned xbytes = static_cast<unsigned>(H) * 2u;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, xbytes);
    bulk_g2s(row, p.x + t * H, xbytes, bar);
  }
  // Every thread waits on the mbarrier below: none may touch it before
  // thread 0 has initialised it.
  __syncthreads();
  // Warp 0 looks up the destinations (all 32 lanes take part).
  int e_k = -1;
  float w_k = 0.0f;
  if (w == 0 && lane < K) {
    e_k = __ldg(p.idx + t * K + lane);
    if (p.w) w_k = __ldg(p.w + t * K + lane);
  }
  if (!kLateDest && w == 0) {
    grid_dependency_wait();
    int ne = 0;
    const int n = f8_destinations(p, t, lane, e_k, w_k, drow, ne);
    if (lane == 0) {
      s_n = n;
      s_ne = ne;
    }
  }
  // Every thread sees the row land itself (it reads the row); the block
  // leaves together if any thread's bounded wait gave up.
  const bool ok = mbar_wait(bar, 0, p.status);
  if (!__syncthreads_and(ok)) {
    // Timed out: the row load may still be in flight into this block's
    // shared row. Let it land (bounded) before the block exits and its
    // shared memory goes to another block; no store has been issued yet.
    if (tid == 0) mbar_drain(bar, 0);
    __syncthreads();
    return;
  }
  // Step c0 covers channels [c0, c0 + kStep), 512 per warp. Its codes go to
  // bytes [c0, c0 + kStep) of the row, which later steps never read; the
  // barrier keeps them from overwriting this step's own inputs.
  constexpr int kStep = 512 * kF8Warps;
  int seg_lo = 0;
  for (int c0 = 0; c0 < H; c0 += kStep) {
    const int c = c0 + w * 512 + lane * 16;
    uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
    if (c < H) {
      v0 = *reinterpret_cast<const uint4*>(row + 2 * c);
      v1 = *reinterpret_cast<const uint4*>(row + 2 * c + 16);
    }
    __syncthreads();
    float sc;
    const uint4 q = quantize16(v0, v1, sc, p.fp8_flags);
    if (c < H) {
      *reinterpret_cast<uint4*>(row + c) = q;
      if ((lane & 7) == 0) scales[c >> 7] = sc;
    }
    const int hi = c0 + kStep;
    if (!kLateDest && hi < H) {
      fence_proxy_async_smem();
      __syncthreads();
      const int n = s_n, ne = s_ne;
      for (int d = tid; d < n; d += kF8Warps * 32) {
        uint8_t* base = d < ne ? p.exp_x : p.rank_x;
        bulk_s2g(base + static_cast<int64_t>(drow[d]) * H + seg_lo, row + seg_lo, static_cast<unsigned>(hi - seg_lo));
      }
      bulk_commit();
      seg_lo = hi;
    }
  }
  if (kLateDest && w == 0) {
    grid_dependency_wait();
    int ne = 0;
    const int n = f8_destinations(p, t, lane, e_k, w_k, drow, ne);
    if (lane == 0) {
      s_n = n;
      s_ne = ne;
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  const int n = s_n, ne = s_ne;
  // One bulk store per destination row, spread over the block's threads.
  for (int d = tid; d < n; d += kF8Warps * 32) {
    uint8_t* base = d < ne ? p.exp_x : p.rank_x;
    bulk_s2g(base + static_cast<int64_t>(drow[d]) * H + seg_lo, row + seg_lo, static_cast<unsigned>(H - seg_lo));
  }
  bulk_commit();
  const bool ue8m0 = p.fp8_flags & EP_FP8_UE8M0;
  for (int d = 0; d < n; ++d) {
    void* sbase = d < ne ? p.exp_scales : p.rank_scales;
    if (!sbase) continue;
    const int64_t r0 = static_cast<int64_t>(drow[d]) * nsc;
    if (ue8m0)
      for (int b = tid; b < nsc; b += kF8Warps * 32) static_cast<uint8_t*>(sbase)[r0 + b] = ue8m0_byte(scales[b]);
    else
      for (int b = tid; b < nsc; b += kF8Warps * 32) static_cast<float*>(sbase)[r0 + b] = scales[b];
  }
  // The shared row must outlive the stores' reads of it (each thread waits
  // for the stores it issued).
  bulk_wait_read<0>();
}

// ---- low-latency send without the layout kernel ------------------------------------
// The layout kernel of the general send computes every slot with a grid-wide
// scan and costs a decode-sized batch ~15 us before any row can leave. The
// slot of (token t, slot k) routed to expert e is
//   j = pre[e][s] + #{(t', k') before (t, k) in source rank s = t / ns,
//                     routed to e},
// where pre[e][s] counts e's entries from the source ranks before s. Two
// forms compute it without the layout:
//   small batch (N * K <= 4096, E * R <= 16384): one launch. Block 0 (the
//     table block) counts the routed entries per (expert, source rank) in
//     shared memory and publishes the per-expert counts, the per-(expert,
//     source) ranges and the header that the receive phase and the combine
//     read; every other block counts the entries of all earlier tokens itself
//     (a few KB, from L2), so it needs nothing from the table block.
//   larger batch (N * K <= 65536, E * R <= 16384, a source rank's entries
//     <= 8192): two launches. A histogram kernel, one block per source rank,
//     counts that source's routed entries per expert (hist[s][e]); the row
//     kernel is its programmatic dependent: its blocks start at once, count
//     the earlier entries of their own source rank, bring in (and quantise)
//     their rows, and only then wait for the histograms and add pre[e][s] =
//     sum over s' < s of hist[s'][e] for their own experts; its block 0
//     publishes the counts, ranges and header from the histograms.
// A row block copies span sp of token t's row: one bulk TMA load in, FP8
// quantisation in place, one bulk store per slot to row e * cap + j of the
// fixed receive buffer. Shrink mode: entries of masked ranks (the expert's, or
// the token's source) are dropped, exactly as in the layout of the general
// send; so are indices outside [-1, E) (flagged by the table).
constexpr int kLLRowThreads = 128;
constexpr int kLLHistThreads = 256;  // the histogram kernel of the larger form
constexpr int kLLSmallBlocksPerSM = 2;
constexpr int kLLMaxRanks = 128;  // E * R <= kLLSmallMaxTable with R <= E gives R <= 128

// n / d by a multiply-high with magic = ceil(2^32 / d) (magic 0 stands for
// d == 1): exact whenever n * d <= 2^32 (n, d >= 0).
__device__ __forceinline__ int div_magic(int n, uint32_t magic) {
  return magic ? static_cast<int>(__umulhi(static_cast<unsigned>(n), magic)) : n;
}

// Entries idx[i0 + j] for j < n, thread tid taking j = tid, tid + NT, ...,
// kBatch loads in flight per thread before any of them is used (a store to
// shared memory or a shared atomic between two loads would otherwise keep the
// next load from being issued early: the pointers may alias).
template <int kBatch, typename F>
__device__ __forceinline__ void for_entries(const int32_t* idx, int i0, int n, int tid, int NT, F&& use) {
  for (int b = tid; b < n; b += kBatch * NT) {
    int v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = b + u * NT;
      v[u] = j < n ? __ldg(idx + i0 + j) : 0;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = b + u * NT;
      if (j < n) use(j, v[u]);
    }
  }
}

// The table of the small form (all threads of the block): counts per
// (expert, source rank) from the routing table, then per-expert counts, the
// per-(expert, source) ranges and the header. hist: shared memory of
// E * (R + 1) + E ints (a row of R + 1 per expert, so the scan over source
// ranks, one thread per expert, is free of bank conflicts).
__device__ void ll_table(const LLSendParams& p, int32_t* hist) {
  __shared__ int s_mask[kLLMaxRanks];
  const int tid = threadIdx.x, NT = blockDim.x;
  const int K = p.K, E = p.E, R = p.R, RP = R + 1;
  int32_t* tot = hist + E * RP;  // [E]
  const int NK = p.N * K;
  const int m = (tid < R && p.rank_mask) ? __ldg(p.rank_mask + tid) : 0;
  if (tid < R) s_mask[tid] = m;
  for (int i = tid; i < E * RP; i += NT) hist[i] = 0;
  const bool any_masked = __syncthreads_or(m != 0);
  bool bad = false;
  for_entries<16>(p.idx, 0, NK, tid, NT, [&](int i, int e) {
    if (e == -1) return;
    if (e < 0 || e >= E) {
      bad = true;
      return;
    }
    const int src = div_magic(i, p.magic_nsK);
    if (any_masked && (s_mask[src] != 0 || s_mask[div_magic(e, p.magic_L)] != 0)) return;
    atomicAdd(&hist[e * RP + src], 1);
  });
  if (__syncthreads_or(bad) && tid == 0) flag(p.status, EP_ST_BAD_INDEX);
  for (int e = tid; e < E; e += NT) {
    int off = 0;
    for (int s = 0; s < R; ++s) {
      const int c = hist[e * RP + s];
      hist[e * RP + s] = off;
      off += c;
    }
    tot[e] = off;
    p.count[e] = off;
  }
  __syncthreads();
  // Rows j >= cap overflow the region (only repeated experts in a row can
  // get there): a range covers the rows that landed.
  for (int i = tid; i < E * R; i += NT) {
    const int e = div_magic(i, p.magic_R), s = i - e * R;
    const int off = hist[e * RP + s];
    const int64_t lo = min(static_cast<int64_t>(off), p.cap);
    const int64_t hi = min(static_cast<int64_t>(s + 1 < R ? hist[e * RP + s + 1] : tot[e]), p.cap);
    p.range[i] = (lo << 32) | (hi - lo);
  }
  if (tid == 0) *p.hdr = p.hdr_value;
}

// The same counts, ranges and header for the larger form, from the
// per-source histograms p.hist [R, E]: a thread per expert runs the prefix
// over source ranks, eight counts loaded at a time.
__device__ void ll_table_from_hist(const LLSendParams& p) {
  const int tid = threadIdx.x, NT = blockDim.x;
  const int E = p.E, R = p.R;
  for (int e = tid; e < E; e += NT) {
    int off = 0;
    for (int s0 = 0; s0 < R; s0 += 8) {
      int c[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) c[u] = s0 + u < R ? __ldcg(p.hist + static_cast<int64_t>(s0 + u) * E + e) : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (s0 + u >= R) break;
        const int64_t lo = min(static_cast<int64_t>(off), p.cap);
        const int64_t hi = min(static_cast<int64_t>(off) + c[u], p.cap);
        p.range[static_cast<int64_t>(e) * R + s0 + u] = (lo << 32) | (hi - lo);
        off += c[u];
      }
    }
    p.count[e] = off;
  }
  if (tid == 0) *p.hdr = p.hdr_value;
}

// The larger form's histogram of source rank s = blockIdx.x: hist[s][e] =
// routed entries of that source for expert e (entries of masked ranks
// dropped; indices outside [-1, E) flagged). hist: shared memory of E ints.
__device__ void ll_source_hist(const LLSendParams& p, int32_t* hist) {
  __shared__ int s_mask[kLLMaxRanks];
  const int tid = threadIdx.x, NT = blockDim.x;
  const int E = p.E, R = p.R, s = blockIdx.x, nsK = p.ns * p.K;
  const int m = (tid < R && p.rank_mask) ? __ldg(p.rank_mask + tid) : 0;
  if (tid < R) s_mask[tid] = m;
  for (int e = tid; e < E; e += NT) hist[e] = 0;
  const bool any_masked = __syncthreads_or(m != 0);
  const bool src_masked = any_masked && s_mask[s] != 0;
  bool bad = false;
  for_entries<8>(p.idx, s * nsK, nsK, tid, NT, [&](int, int e) {
    if (e == -1) return;
    if (e < 0 || e >= E) {
      bad = true;
      return;
    }
    if (src_masked || (any_masked && s_mask[div_magic(e, p.magic_L)] != 0)) return;
    atomicAdd(&hist[e], 1);
  });
  if (__syncthreads_or(bad) && tid == 0) flag(p.status, EP_ST_BAD_INDEX);
  for (int e = tid; e < E; e += NT) p.hist[static_cast<int64_t>(s) * E + e] = hist[e];
}

// Span sp of token t's row (all kLLRowThreads threads of the block). kMid:
// the larger form (count within the own source rank, then wait for the table
// kernel and add its prefix); otherwise the small form (count over every
// earlier token).
template <bool kFp8, int KMAX, bool kMid>
__device__ void ll_row(const LLSendParams& p, int t, int sp, uint8_t* smem) {
  __shared__ int s_e[KMAX], s_cnt[KMAX];
  __shared__ int32_t s_row[KMAX];
  __shared__ int s_mask[kLLMaxRanks];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, NT = kLLRowThreads;
  const int K = p.K, E = p.E, R = p.R;
  const int c0 = sp * p.span, c1 = min(p.H, c0 + p.span);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  uint8_t* row = smem + kBarBytes;
  float* scales = reinterpret_cast<float*>(row + round_up(static_cast<unsigned>(p.span) * 2u, 128u));
  int32_t* s_ent = reinterpret_cast<int32_t*>(scales + p.span / 128);  // the counted entries
  const unsigned in_bytes = static_cast<unsigned>(c1 - c0) * 2u;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, in_bytes);
    bulk_g2s(row, p.x + static_cast<int64_t>(t) * p.H + c0, in_bytes, bar);
  }
  // Every load this block needs goes out together: the entries to count
  // (staged in shared memory), the token's own slots and the rank mask.
  const int src_t = t / p.ns;
  const int tK = t * K;
  const int i0 = kMid ? src_t * p.ns * K : 0;  // first entry counted
  for_entries<8>(p.idx, i0, tK - i0, tid, NT, [&](int j, int v) { s_ent[j] = v; });
  if (tid < K) {
    s_e[tid] = __ldg(p.idx + tK + tid);
    s_cnt[tid] = 0;
  }
  const int m = (tid < R && p.rank_mask) ? __ldg(p.rank_mask + tid) : 0;
  if (tid < R) s_mask[tid] = m;
  // Publishes the mbarrier's initialisation (every thread waits on it
  // below), the entries, the slots' experts and the mask.
  const bool any_masked = __syncthreads_or(m != 0);
  const bool src_masked = any_masked && s_mask[src_t] != 0;
  int key[KMAX], cnt[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    const int e = k < K ? s_e[k] : -1;
    const bool ok = e >= 0 && e < E && !(any_masked && (src_masked || s_mask[div_magic(e, p.magic_L)] != 0));
    key[k] = ok ? e : -1;
    cnt[k] = 0;
  }
  // Earlier entries from unmasked source ranks that name each key.
  for (int i = i0 + tid; i < tK; i += NT) {
    const int x = s_ent[i - i0];
    if (x < 0) continue;
    if (!kMid && any_masked && s_mask[div_magic(i, p.magic_nsK)] != 0) continue;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) cnt[k] += (x == key[k]) ? 1 : 0;
  }
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    if (k >= K) break;
    const int c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(cnt[k])));
    if (lane == 0 && c) atomicAdd(&s_cnt[k], c);
  }
  // Every thread sees the span land itself (it reads it); the block leaves
  // together if any thread's bounded wait gave up, after the load in flight
  // has landed (bounded). The barrier also publishes the counts.
  const bool ok = mbar_wait(bar, 0, p.status);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) mbar_drain(bar, 0);
    __syncthreads();
    return;
  }
  const int n = c1 - c0;
  if (kFp8) {
    // In place, as in dispatch_fp8_kernel: a step reads 512 channels per warp
    // into registers, the block barrier, then the codes go over bytes that
    // no later step reads.
    for (int q0 = 0; q0 < n; q0 += 512 * (kLLRowThreads / 32)) {
      const int c = q0 + w * 512 + lane * 16;
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
      if (c < n) {
        v0 = *reinterpret_cast<const uint4*>(row + 2 * c);
        v1 = *reinterpret_cast<const uint4*>(row + 2 * c + 16);
      }
      __syncthreads();
      float sc;
      const uint4 q = quantize16(v0, v1, sc, p.fp8_flags);
      if (c < n) {
        *reinterpret_cast<uint4*>(row + c) = q;
        if ((lane & 7) == 0) scales[c >> 7] = sc;
      }
    }
  }
  // The larger form: the histograms' sum over the earlier source ranks for
  // each of the token's experts, pairs (k, s') spread over the block.
  __shared__ int s_pre[KMAX];
  if (kMid) {
    if (tid < K) s_pre[tid] = 0;
    grid_dependency_wait();
    __syncthreads();
    const int KS = K * src_t;
    for (int q0 = tid; q0 < KS; q0 += 4 * NT) {
      int c[4], kk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + u * NT;
        c[u] = 0;
        kk[u] = 0;
        if (q < KS) {
          const int k = q / src_t, s2 = q - k * src_t;
          const int e = s_e[k];
          kk[u] = k;
          if (e >= 0 && e < E) c[u] = __ldcg(p.hist + static_cast<int64_t>(s2) * E + e);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c[u]) atomicAdd(&s_pre[kk[u]], c[u]);
    }
    __syncthreads();
  }
  if (tid < K) {
    const int e0 = s_e[tid];
    const bool ok0 = e0 >= 0 && e0 < E && !(any_masked && (src_masked || s_mask[div_magic(e0, p.magic_L)] != 0));
    const int e = ok0 ? e0 : -1;
    int32_t r = -1;
    if (e >= 0) {
      // The token's own earlier slots naming the same expert (a slot equal
      // to a valid key is valid itself).
      int j = s_cnt[tid] + (kMid ? s_pre[tid] : 0);
      for (int k2 = 0; k2 < tid; ++k2) j += (s_e[k2] == e) ? 1 : 0;
      if (j < p.cap)
        r = static_cast<int32_t>(static_cast<int64_t>(e) * p.cap + j);
      else
        flag(p.status, EP_ST_LL_OVERFLOW);
    }
    s_row[tid] = r;
    if (sp == 0) {
      p.slot_map[tK + tid] = r;
      if (r >= 0 && p.recv_src) p.recv_src[r] = t;
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  const int eb = kFp8 ? 1 : 2;
  for (int k = tid; k < K; k += NT) {
    const int32_t r = s_row[k];
    if (r >= 0)
      bulk_s2g(p.recv_x + (static_cast<int64_t>(r) * p.H + c0) * eb, row, static_cast<unsigned>(n * eb));
  }
  bulk_commit();
  if (kFp8 && p.recv_scales) {
    const int nsc = n / 128, b0 = c0 / 128, nall = p.H / 128;
    const bool ue8m0 = p.fp8_flags & EP_FP8_UE8M0;
    for (int i = tid; i < K * nsc; i += NT) {
      const int k = i / nsc, bb = i - k * nsc;
      const int32_t r = s_row[k];
      if (r < 0) continue;
      const int64_t at = static_cast<int64_t>(r) * nall + b0 + bb;
      if (ue8m0)
        static_cast<uint8_t*>(p.recv_scales)[at] = ue8m0_byte(scales[bb]);
      else
        static_cast<float*>(p.recv_scales)[at] = scales[bb];
    }
  }
  // The shared span must outlive the stores' reads of it.
  bulk_wait_read<0>();
}

// The small form: block 0 is the table, block 1 + t * nsplit + sp a row span.
template <bool kFp8, int KMAX>
__global__ void __launch_bounds__(kLLRowThreads) ll_send_small_kernel(const LLSendParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  // Launched as a programmatic dependent of the kernel before it on the
  // stream (which may have produced x or the routing): wait for it first.
  grid_dependency_wait();
  launch_dependents();
  if (blockIdx.x == 0) {
    ll_table(p, reinterpret_cast<int32_t*>(smem));
    return;
  }
  const int b = blockIdx.x - 1;
  ll_row<kFp8, KMAX, false>(p, b / p.nsplit, b % p.nsplit, smem);
}

// The larger form: the histogram kernel (one block per source rank) releases
// its dependent row kernel at once.
__global__ void __launch_bounds__(kLLHistThreads) ll_hist_kernel(const LLSendParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  grid_dependency_wait();  // launched as a programmatic dependent, like the small form
  launch_dependents();
  ll_source_hist(p, reinterpret_cast<int32_t*>(smem));
}

// Block 0 publishes counts, ranges and header once the histograms are in;
// block 1 + t * nsplit + sp is a row span.
template <bool kFp8, int KMAX>
__global__ void __launch_bounds__(kLLRowThreads) ll_send_rows_kernel(const LLSendParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  if (blockIdx.x == 0) {
    grid_dependency_wait();
    ll_table_from_hist(p);
    return;
  }
  const int b = blockIdx.x - 1;
  ll_row<kFp8, KMAX, true>(p, b / p.nsplit, b % p.nsplit, smem);
}

// Launch `fn` with one parameter block; with `pdl`, as the dependent
// of a programmatic pair (it may start before the kernel ahead of it on the
// stream completes, and waits for that kernel in-kernel).
template <typename Params>
cudaError_t launch_ex(void (*fn)(Params), unsigned grid, unsigned threads, size_t smem, cudaStream_t s, bool pdl,
                      const Params& p) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

// One token per block (N <= INT32_MAX fits the grid's x limit): blocks
// retire as their rows leave and the block scheduler hands the next tokens
// to the freed slots.
cudaError_t launch_fp8(const DispatchParams& p, cudaStream_t s, bool pdl) {
  if (p.N <= 0) return cudaSuccess;
  // At most kF8StagedBytesPerSM of staged rows, and kF8MaxBlocksPerSM
  // blocks, per SM: every block of the first wave loads its row at once, so
  // this caps the first wave's read burst (and its synchronous quantisation)
  // before the first stores; the request for more shared memory than a
  // block needs is what caps it. Measured on GB300 (4096 tokens at hidden
  // 7168: 6 / 7 / 8 blocks 79.8 / 77.8 / 81.1 us; 8192 tokens at hidden
  // 4096: 9 / 10 / 11 / 12 blocks 71.3 / 70.6 / 70.9 / 71.5 us).
  size_t smem = kBarBytes + f8_warp_bytes(p.H);
  size_t blocks = kF8StagedBytesPerSM / smem;
  if (blocks > kF8MaxBlocksPerSM) blocks = kF8MaxBlocksPerSM;
  if (blocks >= 1 && blocks < kSmemPerSM / (smem + kSmemReservedPerBlock)) {
    const size_t capped = kSmemPerSM / blocks - kSmemReservedPerBlock - 256;
    if (capped > smem) smem = capped;
  }
  void (*fn)(DispatchParams) = pdl ? dispatch_fp8_kernel<true> : dispatch_fp8_kernel<false>;
  const cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), current_device(), smem);
  if (err != cudaSuccess) return err;
  return launch_ex(fn, static_cast<unsigned>(p.N), kF8Warps * 32, smem, s, pdl, p);
}

cudaError_t launch_bf16(const DispatchParams& p, cudaStream_t s, bool pdl) {
  if (p.N <= 0) return cudaSuccess;
  const unsigned rb = bf16_row_bytes(p.H);
  const int dev = current_device();
  const int sms = device_sms(dev);
  // Up to 4 warps per CTA; a batch with fewer tokens than 4 per SM uses
  // fewer, so its rows spread over more SMs (and their copy engines).
  int W = kMaxWarps;
  while (W > 1 && static_cast<int64_t>(W) * sms > p.N * 2) W >>= 1;
  const unsigned budget = 200u * 1024u;
  while (W > 1 && kBarBytes + W * rb > budget) --W;
  const size_t smem = kBarBytes + static_cast<size_t>(W) * rb;
  void (*fn)(DispatchParams) = dispatch_bf16_kernel;
  const cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), dev, smem);
  if (err != cudaSuccess) return err;
  // One token per warp (N <= INT32_MAX: the grid fits the x limit).
  const int64_t grid = (p.N + W - 1) / W;
  return launch_ex(fn, static_cast<unsigned>(grid), W * 32, smem, s, pdl, p);
}

template <bool kFp8, int KMAX>
cudaError_t launch_ll_rows_variant(const LLSendParams& p, unsigned grid, size_t smem, cudaStream_t s, bool mid) {
  if (!mid) {
    void (*fn)(LLSendParams) = ll_send_small_kernel<kFp8, KMAX>;
    const cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), current_device(), smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(fn, dim3(grid), dim3(kLLRowThreads), smem, s, /*dependent=*/true, p);
  }
  void (*fn)(LLSendParams) = ll_send_rows_kernel<kFp8, KMAX>;
  const cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), current_device(), smem);
  if (err != cudaSuccess) return err;
  return launch_ex(fn, grid, kLLRowThreads, smem, s, /*pdl=*/true, p);
}

}  // namespace

LLSendForm ll_send_form(int N, int K, int E, int R) {
  if (N <= 0 || static_cast<int64_t>(E) * R > kLLSmallMaxTable) return LLSendForm::kLayout;
  const int64_t NK = static_cast<int64_t>(N) * K;
  if (NK <= kLLSmallMaxEntries) return LLSendForm::kSmall;
  if (NK <= kLLMidMaxEntries && static_cast<int64_t>(N / R) * K <= kLLMidMaxSourceEntries) return LLSendForm::kMid;
  return LLSendForm::kLayout;
}

// Blocks per token: about kLLSmallBlocksPerSM blocks per SM over the batch,
// each a span of whole 16-byte BF16 groups (8 channels) or, for FP8, whole
// 128-channel scale blocks. p.hist: the [R, E] per-source histograms of the
// larger form (workspace).
cudaError_t launch_ll_send(LLSendParams p, cudaStream_t s) {
  const LLSendForm form = ll_send_form(p.N, p.K, p.E, p.R);
  if (form == LLSendForm::kLayout) return cudaErrorInvalidValue;
  const bool mid = form == LLSendForm::kMid;
  const bool fp8 = p.fp8_flags & EP_FP8;
  const int sms = device_sms(current_device());
  const int gran = fp8 ? 128 : 8;
  const int units = p.H / gran;
  int nsplit = (kLLSmallBlocksPerSM * sms + p.N - 1) / p.N;
  nsplit = nsplit < 1 ? 1 : (nsplit > units ? units : nsplit);
  const int span_units = (units + nsplit - 1) / nsplit;
  p.span = span_units * gran;
  p.nsplit = (units + span_units - 1) / span_units;
  auto magic = [](int d) { return d > 1 ? static_cast<uint32_t>(((uint64_t(1) << 32) + d - 1) / d) : 0u; };
  p.magic_nsK = magic(p.ns * p.K);
  p.magic_L = magic(p.L);
  p.magic_R = magic(p.R);
  // Row block: the staged span, its FP8 scales, the entries it counts.
  const size_t counted = mid ? static_cast<size_t>(p.ns) * p.K : static_cast<size_t>(p.N) * p.K;
  const size_t row_smem = kBarBytes + round_up(static_cast<unsigned>(p.span) * 2u, 128u) +
                          static_cast<size_t>(p.span / 128) * 4u + sizeof(int32_t) * counted;
  const size_t table_smem = sizeof(int32_t) * (static_cast<size_t>(p.E) * (p.R + 1) + p.E);
  if (mid) {
    if (!p.hist) return cudaErrorInvalidValue;
    const cudaError_t lerr = launch_kernel(ll_hist_kernel, dim3(p.R), dim3(kLLHistThreads), sizeof(int32_t) * p.E,
                                           s, /*dependent=*/true, p);
    if (lerr != cudaSuccess) return lerr;
  }
  // Block 0 of the larger form's row kernel needs no shared table.
  const size_t smem = mid ? row_smem : (row_smem > table_smem ? row_smem : table_smem);
  const unsigned grid = 1u + static_cast<unsigned>(p.N) * static_cast<unsigned>(p.nsplit);
  if (p.K <= 8)
    return fp8 ? launch_ll_rows_variant<true, 8>(p, grid, smem, s, mid)
               : launch_ll_rows_variant<false, 8>(p, grid, smem, s, mid);
  return fp8 ? launch_ll_rows_variant<true, EP_MAX_TOPK>(p, grid, smem, s, mid)
             : launch_ll_rows_variant<false, EP_MAX_TOPK>(p, grid, smem, s, mid);
}

// Zero the padding rows of an aligned expert-major buffer: rows
// [expert_off[e] + count[e], expert_off[e+1]) of each expert e (payload,
// scales, src = -1). Block (e, s) writes the s-th of kPadSlices interleaved
// shares of expert e's padding, so the work spreads over the whole GPU.
constexpr int kPadSlices = 8;

__global__ void __launch_bounds__(256) pad_zero_kernel(const PadParams p) {
  const int e = blockIdx.x;
  const int64_t lo = static_cast<int64_t>(__ldg(p.expert_off + e)) + __ldg(p.per_expert + e);
  int64_t hi = __ldg(p.expert_off + e + 1);
  if (hi > p.cap) {
    if (threadIdx.x == 0 && blockIdx.y == 0) flag(p.status, EP_ST_CAPACITY);
    hi = p.cap;
  }
  if (hi <= lo) return;
  const int64_t first = static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x;
  const int64_t step = static_cast<int64_t>(gridDim.y) * blockDim.x;
  const int64_t vpr = p.row_bytes / 16;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t i = first; i < (hi - lo) * vpr; i += step) reinterpret_cast<uint4*>(p.x + lo * p.row_bytes)[i] = z;
  if (p.scales)
    for (int64_t i = first; i < (hi - lo) * p.scale_row_bytes; i += step) p.scales[lo * p.scale_row_bytes + i] = 0;
  if (p.src)
    for (int64_t r = lo + first; r < hi; r += step) p.src[r] = -1;
}

cudaError_t launch_pad_zero(const PadParams& p, cudaStream_t s) {
  if (p.E <= 0) return cudaSuccess;
  pad_zero_kernel<<<dim3(p.E, kPadSlices), 256, 0, s>>>(p);
  return cudaGetLastError();
}

// Rows to E4M3 + scales with the dispatch's quantiser: a warp per 512
// channels of a row, lanes owning 16 channels (8 lanes per scale block).
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows, int H,
                                                            int flags, uint8_t* __restrict__ q, void* scales) {
  const int lane = threadIdx.x & 31;
  const int per_row = (H + 511) / 512;
  const int64_t nw = rows * per_row;
  const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const bool ue8m0 = flags & EP_FP8_UE8M0;
  for (int64_t wi = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; wi < nw; wi += stride) {
    const int64_t r = wi / per_row;
    const int c = static_cast<int>(wi - r * per_row) * 512 + lane * 16;
    uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
    if (c < H) {
      v0 = __ldg(reinterpret_cast<const uint4*>(x + r * H + c));
      v1 = __ldg(reinterpret_cast<const uint4*>(x + r * H + c + 8));
    }
    float sc;
    const uint4 qq = quantize16(v0, v1, sc, flags);
    if (c < H) {
      *reinterpret_cast<uint4*>(q + r * H + c) = qq;
      if ((lane & 7) == 0) {
        const int64_t at = r * (H / 128) + (c >> 7);
        if (ue8m0)
          static_cast<uint8_t*>(scales)[at] = ue8m0_byte(sc);
        else
          static_cast<float*>(scales)[at] = sc;
      }
    }
  }
}

cudaError_t launch_quantize_rows(const uint16_t* x, int64_t rows, int H, int fp8_flags, uint8_t* q, void* scales,
                                 cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int64_t warps = rows * ((H + 511) / 512);
  const int64_t cap = static_cast<int64_t>(device_sms(current_device())) * 64;
  const int64_t blocks = (warps + 7) / 8;
  quantize_rows_kernel<<<static_cast<unsigned>(blocks < cap ? blocks : cap), 256, 0, s>>>(x, rows, H, fp8_flags, q,
                                                                                          scales);
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const DispatchParams& p, bool fp8, cudaStream_t s, bool after_layout) {
  return fp8 ? launch_fp8(p, s, after_layout) : launch_bf16(p, s, after_layout);
}

}  // namespace ep
