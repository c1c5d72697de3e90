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
// Each warp owns a token at a time and a two-stage shared-memory row buffer.
// Lane 0 brings the next token's BF16 row in with one bulk TMA copy
// (cp.async.bulk global->shared, completion on an mbarrier) while the current
// row is written out. For FP8 the warp quantises the staged row in shared
// memory (half a warp per 128-channel block, shuffle max, IEEE division,
// cvt.rn.satfinite.e4m3x2) into a second two-stage buffer. Every destination
// row is then one bulk TMA store (cp.async.bulk shared->global) issued by the
// lane that owns that destination: the copy engine generates the addresses,
// the SM issues ~R'+K' instructions per token. Grid: persistent, a multiple
// of the SM count.
#include "common.cuh"
#include "kernels.cuh"

namespace ep {

namespace {

constexpr int kMaxWarps = 4;

struct WarpSmem {
  unsigned row_bf16;   // bytes of one staged BF16 row (2H)
  unsigned row_q;      // bytes of one quantised row (H), FP8 only
  unsigned row_s;      // bytes of one scale row (H/128 * 4, rounded to 16), FP8 only
  unsigned per_warp;   // total bytes per warp, 128-aligned
};

__host__ __device__ inline unsigned round_up(unsigned v, unsigned a) { return (v + a - 1) / a * a; }

__host__ __device__ inline WarpSmem warp_smem(int H, bool fp8) {
  WarpSmem w;
  w.row_bf16 = round_up(static_cast<unsigned>(H) * 2u, 128u);
  w.row_q = fp8 ? round_up(static_cast<unsigned>(H), 128u) : 0u;
  w.row_s = fp8 ? round_up(static_cast<unsigned>(H / 128) * 4u, 128u) : 0u;
  w.per_warp = 2u * (w.row_bf16 + w.row_q + w.row_s);
  return w;
}

constexpr unsigned kBarBytes = 128;  // 2 mbarriers per warp, up to 8 warps

// Quantise one staged BF16 row (H channels) into E4M3 codes and fp32 scales.
// Half a warp per 128-channel block: lane j of the half holds channels
// [8j, 8j+8) of the block.
__device__ __forceinline__ void quantize_row_smem(const uint8_t* src, uint8_t* q, float* sc, int H,
                                                  int lane) {
  const int half = lane >> 4, j = lane & 15;
  const int nblk = H / 128;
  // Warp-uniform trip count: both halves run every iteration (the shuffles
  // name the whole warp); a half past the last block only idles.
  for (int b0 = 0; b0 < nblk; b0 += 2) {
    const int b = b0 + half;
    const bool active = b < nblk;
    float f[8];
    if (active) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + b * 256 + j * 16);
      f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
      f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
      f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
      f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.0f;
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!active) continue;
    const float s = __fdiv_rn(m, 448.0f);
    if (s > 0.0f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = __fdiv_rn(f[i], s);
    }
    uint2 out;
    out.x = pack_e4m3x2(f[0], f[1]) | (pack_e4m3x2(f[2], f[3]) << 16);
    out.y = pack_e4m3x2(f[4], f[5]) | (pack_e4m3x2(f[6], f[7]) << 16);
    *reinterpret_cast<uint2*>(q + b * 128 + j * 8) = out;
    if (j == 0) sc[b] = s;
  }
}

template <bool kFP8>
__global__ void __launch_bounds__(kMaxWarps * 32) dispatch_kernel(const DispatchParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, W = blockDim.x >> 5;
  const int H = p.H, K = p.K, R = p.R, L = p.L, E = p.E;
  const WarpSmem ws = warp_smem(H, kFP8);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem) + 2 * w;
  uint8_t* wb = smem + kBarBytes + static_cast<size_t>(w) * ws.per_warp;
  // Stage s of each buffer: BF16 row at wb + s*rb, E4M3 row at qbase + s*rq,
  // scales at sbase + s*rs.
  const unsigned rb = ws.row_bf16, rq = ws.row_q, rs = ws.row_s;
  uint8_t* const qbase = wb + 2 * rb;
  uint8_t* const sbase = wb + 2 * rb + 2 * rq;

  const unsigned xbytes = static_cast<unsigned>(H) * 2u;
  const unsigned obytes = kFP8 ? static_cast<unsigned>(H) : xbytes;
  const unsigned sbytes = static_cast<unsigned>(H / 128) * 4u;
  const bool scale_bulk = kFP8 && (sbytes % 16u == 0u);
  const int64_t nsc = H / 128;

  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int64_t N = p.N;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * W + w;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * W;
  if (gw < N && lane == 0) {
    mbar_arrive_expect_tx(&bar[0], xbytes);
    bulk_g2s(wb, p.x + gw * H, xbytes, &bar[0]);
  }

  unsigned parity = 0;
  unsigned pending = (gw < N) ? 1u : 0u;  // bit s: a load into stage[s] is in flight
  int it = 0;
  for (int64_t t = gw; t < N; t += nw, ++it) {
    const int s = it & 1;
    const int64_t tn = t + nw;
    if (tn < N) {
      if (kFP8)
        fence_proxy_async_smem();  // quantisation reads of stage s^1 precede the refill
      else
        bulk_wait_read<0>();       // the stores of the previous token read stage s^1
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar[s ^ 1], xbytes);
        bulk_g2s(wb + (s ^ 1) * rb, p.x + tn * H, xbytes, &bar[s ^ 1]);
      }
      pending |= 1u << (s ^ 1);
    }

    // This lane's top-k slot (lane < K): expert, weight and expert-major row.
    int e_k = -1;
    float w_k = 0.0f;
    int32_t erow = -1;
    if (lane < K) {
      e_k = __ldg(p.idx + t * K + lane);
      if (p.w) w_k = __ldg(p.w + t * K + lane);
      if (p.exp_x) {
        erow = __ldg(p.expert_slot + t * K + lane);
        if (erow >= p.exp_cap) {
          flag(p.status, p.overflow_bit);
          erow = -1;
        }
        if (erow >= 0 && p.exp_src)
          p.exp_src[erow] = p.exp_src_is_token ? static_cast<int32_t>(t) : static_cast<int32_t>(t * K + lane);
      }
    }

    if (!mbar_wait(&bar[s], (parity >> s) & 1u, p.status)) break;
    parity ^= 1u << s;
    pending &= ~(1u << s);

    const uint8_t* src = wb + s * rb;
    const float* scl = nullptr;
    if (kFP8) {
      bulk_wait_read<1>();  // the stores of two tokens ago read E4M3 row and scales s
      __syncwarp();
      uint8_t* qs = qbase + s * rq;
      float* ss = reinterpret_cast<float*>(sbase + s * rs);
      quantize_row_smem(wb + s * rb, qs, ss, H, lane);
      fence_proxy_async_smem();
      __syncwarp();
      src = qs;
      scl = ss;
    }

    // Expert-major copies.
    if (erow >= 0) {
      bulk_s2g(p.exp_x + static_cast<int64_t>(erow) * obytes, src, obytes);
      if (kFP8 && p.exp_scales) {
        if (scale_bulk)
          bulk_s2g(p.exp_scales + static_cast<int64_t>(erow) * nsc, scl, sbytes);
        else
          for (int64_t b = 0; b < nsc; ++b) p.exp_scales[erow * nsc + b] = scl[b];
      }
    }

    // Per-rank copies: lane owns ranks lane, lane + 32, ...
    if (p.rank_x) {
      for (int rb = 0; rb < R; rb += 32) {
        const int r = rb + lane;
        int32_t rrow = (r < R) ? __ldg(p.rank_slot + t * R + r) : -1;
        if (rrow >= p.rank_cap) {
          flag(p.status, EP_ST_CAPACITY);
          rrow = -1;
        }
        if (rrow >= 0) {
          bulk_s2g(p.rank_x + static_cast<int64_t>(rrow) * obytes, src, obytes);
          if (kFP8 && p.rank_scales) {
            if (scale_bulk)
              bulk_s2g(p.rank_scales + static_cast<int64_t>(rrow) * nsc, scl, sbytes);
            else
              for (int64_t b = 0; b < nsc; ++b) p.rank_scales[rrow * nsc + b] = scl[b];
          }
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
  }
  // Only after a timed-out wait can a load still be in flight: give it a
  // bounded chance to land before the block's shared memory is released.
  for (int st = 0; st < 2; ++st)
    if (pending & (1u << st)) mbar_wait(&bar[st], (parity >> st) & 1u, p.status);
  bulk_wait<0>();
}

template <bool kFP8>
cudaError_t launch_impl(const DispatchParams& p, cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  const WarpSmem ws = warp_smem(p.H, kFP8);
  int W = kMaxWarps;
  const unsigned budget = 200u * 1024u;
  while (W > 1 && kBarBytes + W * ws.per_warp > budget) --W;
  const size_t smem = kBarBytes + static_cast<size_t>(W) * ws.per_warp;
  const void* fn = reinterpret_cast<const void*>(&dispatch_kernel<kFP8>);
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, W * 32, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t need = (p.N + W - 1) / W;
  const int64_t full = static_cast<int64_t>(per_sm) * sms;
  const int grid = static_cast<int>(need < full ? need : full);
  dispatch_kernel<kFP8><<<grid, W * 32, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dispatch(const DispatchParams& p, bool fp8, cudaStream_t s) {
  return fp8 ? launch_impl<true>(p, s) : launch_impl<false>(p, s);
}

}  // namespace ep
