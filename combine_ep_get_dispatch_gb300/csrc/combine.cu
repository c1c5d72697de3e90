// Combine on sm_103a: gather each token's expert outputs back and take the
// router-weighted top-k sum.
//
// What it computes ("DeepEP Ascend deep dive", "Two Transfers": results come
// back along the same path and are weighted by router score and summed;
// "DeepEP lesson 14", practice task: out_i = sum_k w_ik * y_ik):
//   out[t] = bf16_rn( fma(w[t,K-1], y[slot[t,K-1]], ... fma(w[t,0], y[slot[t,0]], +0)) )
// over unmasked slots, in slot order, one fp32 fused multiply-add per term.
//
// Design (HBM-bound, read-heavy: K rows read, one row written per token).
// One block per token. The token's slots and weights go to
// shared memory once; each thread then owns 16-byte vectors of the row and,
// for up to 8 slots at a time, issues all their loads before the FMAs, so K
// independent 16-byte reads per thread are in flight. The rows are read once,
// with an L2 evict-first policy (measured 5 % faster on 4096-token batches
// than plain non-coherent loads; no change at 16384). The reduction happens
// in registers as the rows arrive: no intermediate buffer, no second pass.
#include "common.cuh"
#include "kernels.cuh"

namespace ep {

namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 8;

// Barrier `id` (1..15; 0 is __syncthreads) over the first `threads` threads
// of the block (a multiple of 32, whole warps).
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void fma8(float* acc, float w, const uint4& v) {
  acc[0] = __fmaf_rn(w, bf16_lo(v.x), acc[0]);
  acc[1] = __fmaf_rn(w, bf16_hi(v.x), acc[1]);
  acc[2] = __fmaf_rn(w, bf16_lo(v.y), acc[2]);
  acc[3] = __fmaf_rn(w, bf16_hi(v.y), acc[3]);
  acc[4] = __fmaf_rn(w, bf16_lo(v.z), acc[4]);
  acc[5] = __fmaf_rn(w, bf16_hi(v.z), acc[5]);
  acc[6] = __fmaf_rn(w, bf16_lo(v.w), acc[6]);
  acc[7] = __fmaf_rn(w, bf16_hi(v.w), acc[7]);
}

__device__ __forceinline__ bool same_shape(const LLHeader& a, const LLHeader& b) {
  return a.N == b.N && a.K == b.K && a.E == b.E && a.R == b.R && a.T == b.T;
}

// The first N - tail tokens are one work item each (the whole row); each of
// the last `tail` tokens is nchunk items, equal spans of its row. Splitting
// the tail shortens the blocks that run while the grid drains; a small batch
// is all tail (it spreads over more SMs). Blocks take items in order.
// kGather copies each routed row to its own output row t*K + k instead of
// summing (the send half of the two-phase low-latency combine).
template <bool kGather>
__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineParams p, int64_t tail, int nchunk) {
  // The token's routed slots in order: expert row, weight, slot index; and
  // the weights by slot.
  __shared__ int32_t s_row[EP_MAX_TOPK], s_k[EP_MAX_TOPK];
  __shared__ float s_w[EP_MAX_TOPK], s_wk[EP_MAX_TOPK];
  __shared__ int s_ok, s_nv;
  const int tid = threadIdx.x, lane = tid & 31;
  const int K = p.K, H = p.H;
  // Launched as a programmatic dependent: nothing is touched before the
  // kernel ahead of it on the stream has completed.
  grid_dependency_wait();
  if (p.ll_hdr) {
    if (tid == 0) {
      const LLHeader h = *p.ll_hdr;
      int ok = (h.magic == kMagicSent || h.magic == kMagicReceived) ? 1 : 0;
      if (!ok) {
        if (blockIdx.x == 0) flag(p.status, EP_ST_NOT_SENT);
      } else if (!same_shape(h, p.ll_expect)) {
        ok = 0;
        if (blockIdx.x == 0) flag(p.status, EP_ST_MISMATCH);
      }
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) return;
  }
  const int nvec = H / 8;
  const int span = (nvec + nchunk - 1) / nchunk;
  const int64_t head = p.N - tail;
  const int64_t items = head + tail * nchunk;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    int64_t t = it;
    int v0 = 0, v1 = nvec;
    if (it >= head) {
      const int64_t j = it - head;
      t = head + j / nchunk;
      v0 = static_cast<int>(j - (t - head) * nchunk) * span;
      v1 = min(nvec, v0 + span);
    }
    // Warp 0 lists the routed slots in slot order (masked ones dropped), so
    // every row load below is useful and all of them go out in one round
    // whenever a token has at most kChunk routed slots. K <= 32: a lane per
    // slot. Warp 1 fetches the weights meanwhile (by slot), and warp 0 copies
    // them into list order once both warps are past the named barrier.
    if (tid < 32) {
      const int k = lane;
      int32_t row = k < K ? __ldg(p.slot + t * K + k) : -1;
      // Low-latency shrink mode: skip the slots of ranks masked now (the
      // expert's rank, from its region e = row / (R*T), or the token's source).
      if (row >= 0 && p.rank_mask &&
          (__ldg(p.rank_mask + static_cast<int>(row / p.ll_cap) / p.ll_L) != 0 ||
           __ldg(p.rank_mask + static_cast<int>(t / p.ll_ns)) != 0))
        row = -1;
      if (row >= 0 && p.token_major) row = static_cast<int32_t>(t * K + k);
      if (row >= p.y_rows) {
        flag(p.status, EP_ST_CAPACITY);
        row = -1;
      }
      const unsigned m = __ballot_sync(0xffffffffu, row >= 0);
      const int pos = __popc(m & lanemask_lt());
      if (row >= 0) {
        s_row[pos] = row;
        s_k[pos] = k;
      }
      if (lane == 0) s_nv = __popc(m);
      if (!kGather) {
        named_barrier_sync(1, 64);
        if (row >= 0) s_w[pos] = s_wk[k];
      }
    } else if (!kGather && tid < 64) {
      if (lane < K) s_wk[lane] = p.w ? __ldg(p.w + t * K + lane) : 1.0f;
      named_barrier_sync(1, 64);
    }
    __syncthreads();
    const int nv = s_nv;
    for (int v = v0 + tid; v < v1; v += kThreads) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      for (int i0 = 0; i0 < nv; i0 += kChunk) {
        uint4 yv[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
          if (i0 + j < nv)
            yv[j] = ld_stream_v4(reinterpret_cast<const uint4*>(p.y + static_cast<int64_t>(s_row[i0 + j]) * H) + v);
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          const int i = i0 + j;
          if (i >= nv) break;
          if (kGather)
            reinterpret_cast<uint4*>(p.out + (t * K + s_k[i]) * H)[v] = yv[j];
          else
            fma8(acc, s_w[i], yv[j]);
        }
      }
      if (kGather) continue;
      if (p.bias) {
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(p.bias + t * H) + v);
        acc[0] += bf16_lo(b.x); acc[1] += bf16_hi(b.x);
        acc[2] += bf16_lo(b.y); acc[3] += bf16_hi(b.y);
        acc[4] += bf16_lo(b.z); acc[5] += bf16_hi(b.z);
        acc[6] += bf16_lo(b.w); acc[7] += bf16_hi(b.w);
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      reinterpret_cast<uint4*>(p.out + t * H)[v] = o;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  // One block per token (the hardware scheduler hands blocks to SMs as they
  // free up), at most eight resident per SM (64 registers). The tokens past
  // the last multiple of eight per SM (the last partial wave) are split into
  // as many spans as a row has 128-vector groups, so the blocks still running
  // while the grid drains are short; measured against whole-token blocks:
  // -1.6 us on 16384 tokens at hidden 7168, -2.7 us on 4096. A batch with
  // fewer tokens than that splits every row, up to the same limit.
  const int sms = device_sms(current_device());
  const int nvec = p.H / 8;
  const int most = (nvec + kThreads - 1) / kThreads;
  const int64_t want = static_cast<int64_t>(sms) * 8;
  int nchunk = most;
  int64_t tail = p.N % want;
  if (p.N < want) {
    nchunk = static_cast<int>((want + p.N - 1) / p.N);
    if (nchunk > most) nchunk = most;
    tail = p.N;
  }
  if (nchunk <= 1) {
    nchunk = 1;
    tail = 0;
  }
  const int64_t items = (p.N - tail) + tail * nchunk;
  const int64_t cap = int64_t(1) << 30;
  const int grid = static_cast<int>(items < cap ? items : cap);
  return launch_kernel(p.gather ? combine_kernel<true> : combine_kernel<false>, dim3(grid), dim3(kThreads), 0, s,
                       /*dependent=*/true, p, tail, nchunk);
}

// ---- two-level combine, first level --------------------------------------------
// For every (token, rank) of the mask: rank_out[rank_slot[t, r]] = bf16( sum
// over k ascending whose expert lives on r of w[t, k] * y[expert_slot[t, k]] )
// (the reduction DeepEP's expert layer does on each rank before combine).
// One block per token; the K slots are grouped by rank in shared memory and
// each rank's chain runs in slot order (for K <= 8 from registers, after one
// round of loads of all the token's rows).
__global__ void __launch_bounds__(kThreads) combine_to_ranks_kernel(const CombineRanksParams p) {
  __shared__ int32_t s_row[EP_MAX_TOPK], s_rank[EP_MAX_TOPK], s_out[EP_MAX_TOPK];
  __shared__ float s_w[EP_MAX_TOPK];
  const int tid = threadIdx.x;
  const int K = p.K, H = p.H, E = p.E, L = p.L, R = p.R;
  const int nvec = H / 8;
  for (int64_t t = blockIdx.x; t < p.N; t += gridDim.x) {
    if (tid < K) {
      const int e = __ldg(p.idx + t * K + tid);
      int32_t row = __ldg(p.expert_slot + t * K + tid);
      const float wk = __ldg(p.w + t * K + tid);
      const bool ok = e >= 0 && e < E && row >= 0;
      if (ok && row >= p.y_rows) {
        flag(p.status, EP_ST_CAPACITY);
        row = -1;
      }
      const int r = (ok && row >= 0) ? e / L : -1;
      s_rank[tid] = r;
      s_row[tid] = row;
      s_w[tid] = wk;
      int32_t orow = -1;
      if (r >= 0) {
        orow = __ldg(p.rank_slot + t * R + r);
        if (orow >= p.rank_rows) {
          flag(p.status, EP_ST_CAPACITY);
          orow = -1;
        }
      }
      s_out[tid] = orow;
    }
    __syncthreads();
    if (K <= kChunk) {
      // All of the token's rows are loaded at once for a vector; each rank's
      // chain then runs from registers, in slot order.
      for (int v = tid; v < nvec; v += kThreads) {
        uint4 yv[kChunk];
#pragma unroll
        for (int k = 0; k < kChunk; ++k)
          if (k < K && s_rank[k] >= 0)
            yv[k] = ld_stream_v4(reinterpret_cast<const uint4*>(p.y + static_cast<int64_t>(s_row[k]) * H) + v);
#pragma unroll
        for (int k0 = 0; k0 < kChunk; ++k0) {
          if (k0 >= K) break;
          const int r = s_rank[k0];
          if (r < 0 || s_out[k0] < 0) continue;
          bool first = true;
          for (int k = 0; k < k0; ++k) first &= s_rank[k] != r;
          if (!first) continue;
          float acc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
          for (int k = 0; k < kChunk; ++k)
            if (k >= k0 && k < K && s_rank[k] == r) fma8(acc, s_w[k], yv[k]);
          uint4 o;
          o.x = pack_bf16x2(acc[0], acc[1]);
          o.y = pack_bf16x2(acc[2], acc[3]);
          o.z = pack_bf16x2(acc[4], acc[5]);
          o.w = pack_bf16x2(acc[6], acc[7]);
          reinterpret_cast<uint4*>(p.rank_out + static_cast<int64_t>(s_out[k0]) * H)[v] = o;
        }
      }
      __syncthreads();
      continue;
    }
    for (int k0 = 0; k0 < K; ++k0) {
      const int r = s_rank[k0];
      if (r < 0) continue;
      bool first = true;
      for (int k = 0; k < k0; ++k) first &= s_rank[k] != r;
      if (!first || s_out[k0] < 0) continue;
      uint16_t* orow = p.rank_out + static_cast<int64_t>(s_out[k0]) * H;
      for (int v = tid; v < nvec; v += kThreads) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int k = k0; k < K; ++k) {
          if (s_rank[k] != r) continue;
          const uint4 yv = __ldg(reinterpret_cast<const uint4*>(p.y + static_cast<int64_t>(s_row[k]) * H) + v);
          fma8(acc, s_w[k], yv);
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4*>(orow)[v] = o;
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_combine_to_ranks(const CombineRanksParams& p, cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  const int64_t cap = int64_t(1) << 30;
  combine_to_ranks_kernel<<<static_cast<int>(p.N < cap ? p.N : cap), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

// ---- combine backward --------------------------------------------------------------
// For out[t] = sum_k w[t,k] y[slot[t,k]]: grad_y[slot[t,k]] = bf16(w[t,k] *
// grad_out[t]) (the backward of combine is a dispatch of the weighted
// gradient) and grad_w[t,k] = <grad_out[t], y[slot[t,k]]> in fp32: each
// thread chains its vectors' products with fused multiply-adds, then a fixed
// shuffle / shared-memory tree sums the threads, so the result is the same on
// every run. One block per token.
__global__ void __launch_bounds__(kThreads) combine_backward_kernel(const CombineBwdParams p) {
  __shared__ int32_t s_row[EP_MAX_TOPK];
  __shared__ float s_w[EP_MAX_TOPK];
  __shared__ float s_red[kThreads / 32][kChunk];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K, H = p.H, nvec = H / 8;
  for (int64_t t = blockIdx.x; t < p.N; t += gridDim.x) {
    if (tid < K) {
      int32_t row = __ldg(p.slot + t * K + tid);
      const float wk = __ldg(p.w + t * K + tid);
      if (row >= p.y_rows) {
        flag(p.status, EP_ST_CAPACITY);
        row = -1;
      }
      s_row[tid] = row;
      s_w[tid] = wk;
    }
    __syncthreads();
    const uint4* g_row = reinterpret_cast<const uint4*>(p.grad_out + t * H);
    for (int k0 = 0; k0 < K; k0 += kChunk) {
      float dot[kChunk];
#pragma unroll
      for (int j = 0; j < kChunk; ++j) dot[j] = 0.0f;
      for (int v = tid; v < nvec; v += kThreads) {
        const uint4 g = __ldg(g_row + v);
        // All of this chunk's row loads go out first (before the gradient
        // stores, which the compiler could not move loads across).
        uint4 yv_all[kChunk];
        if (p.grad_w && p.y) {
#pragma unroll
          for (int j = 0; j < kChunk; ++j) {
            const int k = k0 + j;
            const int32_t row = (k < K) ? s_row[k] : -1;
            if (row >= 0)
              yv_all[j] = ld_stream_v4(reinterpret_cast<const uint4*>(p.y + static_cast<int64_t>(row) * H) + v);
          }
        }
        const float gf[8] = {bf16_lo(g.x), bf16_hi(g.x), bf16_lo(g.y), bf16_hi(g.y),
                             bf16_lo(g.z), bf16_hi(g.z), bf16_lo(g.w), bf16_hi(g.w)};
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          const int k = k0 + j;
          const int32_t row = (k < K) ? s_row[k] : -1;
          if (row < 0) continue;
          if (p.grad_y) {
            const float wk = s_w[k];
            uint4 o;
            o.x = pack_bf16x2(__fmul_rn(wk, gf[0]), __fmul_rn(wk, gf[1]));
            o.y = pack_bf16x2(__fmul_rn(wk, gf[2]), __fmul_rn(wk, gf[3]));
            o.z = pack_bf16x2(__fmul_rn(wk, gf[4]), __fmul_rn(wk, gf[5]));
            o.w = pack_bf16x2(__fmul_rn(wk, gf[6]), __fmul_rn(wk, gf[7]));
            reinterpret_cast<uint4*>(p.grad_y + static_cast<int64_t>(row) * H)[v] = o;
          }
          if (p.grad_w && p.y) {
            const uint4 yv = yv_all[j];
            dot[j] = __fmaf_rn(gf[0], bf16_lo(yv.x), dot[j]);
            dot[j] = __fmaf_rn(gf[1], bf16_hi(yv.x), dot[j]);
            dot[j] = __fmaf_rn(gf[2], bf16_lo(yv.y), dot[j]);
            dot[j] = __fmaf_rn(gf[3], bf16_hi(yv.y), dot[j]);
            dot[j] = __fmaf_rn(gf[4], bf16_lo(yv.z), dot[j]);
            dot[j] = __fmaf_rn(gf[5], bf16_hi(yv.z), dot[j]);
            dot[j] = __fmaf_rn(gf[6], bf16_lo(yv.w), dot[j]);
            dot[j] = __fmaf_rn(gf[7], bf16_hi(yv.w), dot[j]);
          }
        }
      }
      if (p.grad_w) {
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          float d = dot[j];
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          if (lane == 0) s_red[warp][j] = d;
        }
        __syncthreads();
        if (tid < kChunk && k0 + tid < K) {
          float d = 0.0f;
          for (int ww = 0; ww < kThreads / 32; ++ww) d += s_red[ww][tid];
          p.grad_w[t * K + k0 + tid] = (s_row[k0 + tid] >= 0 && p.y) ? d : 0.0f;
        }
        __syncthreads();
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_combine_backward(const CombineBwdParams& p, cudaStream_t s) {
  if (p.N <= 0) return cudaSuccess;
  const int64_t cap = int64_t(1) << 30;
  combine_backward_kernel<<<static_cast<int>(p.N < cap ? p.N : cap), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ep
