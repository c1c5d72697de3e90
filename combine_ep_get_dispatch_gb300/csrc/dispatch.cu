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
  // This lane's top-k slot (lane < K): expert, weight and expert-major row.
  int e_k = -1;
  float w_k = 0.0f;
  int32_t erow = -1;
  if (lane < K) {
    e_k = __ldg(p.idx + t * K + lane);
    if (p.w) w_k = __ldg(p.w + t * K + lane);
    if (p.exp_x) {
      erow = __ldcg(p.expert_slot + t * K + lane);
      if (erow >= p.exp_cap) {
        flag(p.status, p.overflow_bit);
        erow = -1;
      }
      if (erow >= 0 && p.exp_src)
        p.exp_src[erow] = p.exp_src_is_token ? static_cast<int32_t>(t) : static_cast<int32_t>(t * K + lane);
    }
  }

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
      int32_t rrow = (r < R) ? __ldcg(p.rank_slot + t * R + r) : -1;
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
          const int ek = __shfl_sync(0xffffffffu, e_k, kk);
          const float wk = __shfl_sync(0xffffffffu, w_k, kk);
          if (rrow >= 0) {
            const bool here = ek >= 0 && ek < E && ek / L == r;
            if (p.rank_topk_idx) p.rank_topk_idx[static_cast<int64_t>(rrow) * K + kk] = here ? ek - r * L : -1;
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
// max by shuffles, divide by the scale (IEEE) and convert to E4M3, writing the
// codes over the front of the staged row. Each destination row then leaves by
// one bulk store (cp.async.bulk shared->global), and the scales follow with
// plain stores (a UE8M0 scale row is not a multiple of 16 bytes). At 14.9 KB
// of shared memory per token about 14 tokens are in flight per SM.
// Measured on GB300 (all bit-identical): the row loaded through registers one
// step ahead (each token then waits out ~14 load latencies behind the write
// traffic); a separate E4M3 row (fewer tokens in flight); one warp per token
// (each token's chain of load, quantisation and stores is longer, so the
// kernel's ramp and tail are too: four warps took the 4096-token FP8
// dispatches from 90.1 to 86.0 us and 79.9 to 74.2 us).
constexpr int kF8Warps = 4;                  // warps per token (one token per block)
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

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return pack_e4m3x2(a, b) | (pack_e4m3x2(c, d) << 16);
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
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(f[i]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  sc = __fdiv_rn(m, 448.0f);
  if ((flags & (EP_FP8_ROUND_SCALE | EP_FP8_UE8M0)) && sc > 0.0f) sc = pow2_ceil(sc);
  if ((flags & EP_FP8_UE8M0) && m > 0.0f) sc = fmaxf(sc, __uint_as_float(0x00400000u));  // 2^-127
  if (sc > 0.0f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __fdiv_rn(f[i], sc);
  }
  uint4 q;
  q.x = e4m3x4(f[0], f[1], f[2], f[3]);
  q.y = e4m3x4(f[4], f[5], f[6], f[7]);
  q.z = e4m3x4(f[8], f[9], f[10], f[11]);
  q.w = e4m3x4(f[12], f[13], f[14], f[15]);
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
  int32_t erow = -1;
  if (lane < K && p.exp_x) {
    erow = __ldcg(p.expert_slot + t * K + lane);
    if (erow >= p.exp_cap) {
      flag(p.status, p.overflow_bit);
      erow = -1;
    }
    if (erow >= 0 && p.exp_src)
      p.exp_src[erow] = p.exp_src_is_token ? static_cast<int32_t>(t) : static_cast<int32_t>(t * K + lane);
  }
  const unsigned vm = __ballot_sync(0xffffffffu, erow >= 0);
  if (erow >= 0) drow[__popc(vm & lanemask_lt())] = erow;
  ne = __popc(vm);
  int n = ne;
  if (p.rank_x) {
    for (int rb = 0; rb < R; rb += 32) {
      const int r = rb + lane;
      int32_t rrow = (r < R) ? __ldcg(p.rank_slot + t * R + r) : -1;
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
          const int ek = __shfl_sync(0xffffffffu, e_k, kk);
          const float wk = __shfl_sync(0xffffffffu, w_k, kk);
          if (rrow >= 0) {
            const bool here = ek >= 0 && ek < E && ek / L == r;
            if (p.rank_topk_idx) p.rank_topk_idx[static_cast<int64_t>(rrow) * K + kk] = here ? ek - r * L : -1;
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
  // Step c0 covers channels [c0, c0 + 512 * kF8Warps), 512 per warp. Its codes
  // go to bytes [c0, c0 + 512 * kF8Warps) of the row, which later steps never
  // read; the barrier keeps them from overwriting this step's own inputs.
  for (int c0 = 0; c0 < H; c0 += 512 * kF8Warps) {
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
    bulk_s2g(base + static_cast<int64_t>(drow[d]) * H, row, static_cast<unsigned>(H));
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

// Launch `fn` with one DispatchParams argument; with `pdl`, as the dependent
// of a programmatic pair (it may start before the kernel ahead of it on the
// stream completes, and waits for that kernel in-kernel).
cudaError_t launch_ex(void (*fn)(DispatchParams), unsigned grid, unsigned threads, size_t smem, cudaStream_t s,
                      bool pdl, const DispatchParams& p) {
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
  const size_t smem = kBarBytes + f8_warp_bytes(p.H);
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

}  // namespace

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

cudaError_t launch_dispatch(const DispatchParams& p, bool fp8, cudaStream_t s, bool after_layout) {
  return fp8 ? launch_fp8(p, s, after_layout) : launch_bf16(p, s, after_layout);
}

}  // namespace ep
