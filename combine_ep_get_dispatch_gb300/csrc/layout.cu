// Routing layout on sm_103a: counts, the per-rank mask and deterministic
// prefix-sum slots in one cooperative launch.
//
// What it computes ("DeepEP V1 (legacy) guide", section 5.2(1); "DeepEP
// Ascend deep dive", "Two Transfers" and "Dispatch's Three Phases"):
//   per_expert[e]      #{(t, k): idx[t, k] == e}
//   mask[t, r]         some slot of t names an expert of rank r (one copy per rank)
//   per_rank[r]        sum over t of mask[t, r]
//   expert_slot[t, k]  expert_off[e] + #{(t', k') < (t, k) in (token, slot) order with idx == e}
//   rank_slot[t, r]    rank_off[r] + #{t' < t with mask[t', r]}
//
// Design. The (token, slot) entries are cut into G contiguous chunks, one
// per CTA, and each chunk into 16 contiguous warp ranges. A warp walks its
// range 32 entries at a time; __match_any_sync groups the lanes that name the
// same expert (or, for ranks, the first slot of a token on that rank), so the
// rank of an entry among equal keys in the window is a popcount and one
// leader lane bumps the warp's private counter: no atomics, and the order is
// (token, slot) order by construction. Pass 1 counts; the per-chunk totals
// go to global memory; one bounded grid barrier; every CTA then sums the
// chunk totals before it (its prefix) and all of them (the totals), scans the
// totals over experts and ranks, and pass 2 repeats the walk, now writing
// slots. Launch-bound: the work is a few hundred KB of int32 traffic.
#include "common.cuh"
#include "kernels.cuh"

namespace ep {

constexpr int kLayoutThreads = 512;
constexpr int kLayoutWarps = kLayoutThreads / 32;

// Exclusive scan of a[0..n) in shared memory, in place; returns the total.
// All threads of the block must call it.
__device__ int block_exclusive_scan(int32_t* a, int n, int32_t* warp_tmp) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (n + kLayoutThreads - 1) / kLayoutThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += a[i];
  int v = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) warp_tmp[w] = v;
  __syncthreads();
  if (w == 0) {
    int x = lane < kLayoutWarps ? warp_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < kLayoutWarps) warp_tmp[lane] = x;
  }
  __syncthreads();
  int run = (w > 0 ? warp_tmp[w - 1] : 0) + v - s;
  const int total = warp_tmp[kLayoutWarps - 1];
  for (int i = lo; i < hi; ++i) {
    const int x = a[i];
    a[i] = run;
    run += x;
  }
  __syncthreads();
  return total;
}

template <bool kRank, bool kLL>
__global__ void __launch_bounds__(kLayoutThreads) layout_kernel(const LayoutParams p) {
  extern __shared__ int32_t sm[];
  const int E = p.E, R = p.R, K = p.K, L = p.L;
  const int C = E + (kRank ? R : 0);
  int32_t* hist = sm;                        // [16][C]: counts, then running slots
  int32_t* base = hist + kLayoutWarps * C;   // [C]: this chunk's prefix over earlier chunks
  int32_t* tot = base + C;                   // [C]: totals, then their exclusive scan
  int32_t* own = tot + C;                    // [C]: this chunk's own count
  int32_t* tmp = own + C;                    // [32]

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int cta = blockIdx.x, G = gridDim.x;
  const int64_t N = p.N;
  const int64_t t0 = min(N, static_cast<int64_t>(cta) * p.tokens_per_cta);
  const int64_t t1 = min(N, t0 + p.tokens_per_cta);
  const int64_t a0 = t0 * K, a1 = t1 * K;
  const int64_t per_warp = ((a1 - a0 + kLayoutWarps * 32 - 1) / (kLayoutWarps * 32)) * 32;
  const int64_t wa0 = min(a1, a0 + w * per_warp), wa1 = min(a1, wa0 + per_warp);

  for (int i = tid; i < kLayoutWarps * C; i += kLayoutThreads) hist[i] = 0;
  if (kRank) {
    for (int64_t i = t0 * R + tid; i < t1 * R; i += kLayoutThreads) {
      p.mask[i] = 0;
      p.rank_slot[i] = -1;
    }
  }
  __syncthreads();

  int32_t* my = hist + w * C;

  // Pass 1: per-warp counts.
  bool bad = false;
  for (int64_t b = wa0; b < wa1; b += 32) {
    const int64_t i = b + lane;
    const bool in = i < wa1;
    const int e = in ? __ldg(p.idx + i) : -1;
    const bool valid = in && e >= 0 && e < E;
    bad |= in && e != -1 && !valid;
    const unsigned pe = __match_any_sync(0xffffffffu, valid ? e : -2 - lane);
    if (valid && lane == __ffs(pe) - 1) my[e] += __popc(pe);
    if (kRank) {
      const int r = valid ? e / L : -1;
      bool first = valid;
      if (valid) {
        const int64_t t = i / K;
        for (int64_t j = t * K; j < i; ++j) {
          const int e2 = __ldg(p.idx + j);
          if (e2 >= 0 && e2 < E && e2 / L == r) first = false;
        }
      }
      const unsigned pr = __match_any_sync(0xffffffffu, first ? r : -2 - lane);
      if (first && lane == __ffs(pr) - 1) my[E + r] += __popc(pr);
    }
    __syncwarp();
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag(p.status, EP_ST_BAD_INDEX);
  __syncthreads();

  // Per column: exclusive prefix over warps; the chunk's total goes out.
  for (int col = tid; col < C; col += kLayoutThreads) {
    int run = 0;
    for (int ww = 0; ww < kLayoutWarps; ++ww) {
      const int v = hist[ww * C + col];
      hist[ww * C + col] = run;
      run += v;
    }
    own[col] = run;
    p.ws_chunk[static_cast<int64_t>(cta) * C + col] = run;
  }
  if (G > 1)
    grid_barrier(p.ws_barrier, static_cast<unsigned>(G), p.status);
  else
    __syncthreads();

  // Prefix over earlier chunks and totals over all chunks.
  for (int col = tid; col < C; col += kLayoutThreads) {
    int pre = 0, total = 0;
    for (int c = 0; c < G; ++c) {
      const int v = __ldcg(p.ws_chunk + static_cast<int64_t>(c) * C + col);
      pre += (c < cta) ? v : 0;
      total += v;
    }
    base[col] = pre;
    tot[col] = total;
    if (cta == 0) {
      if (col < E)
        p.per_expert[col] = total;
      else
        p.per_rank[col - E] = total;
    }
  }
  __syncthreads();
  const int total_e = block_exclusive_scan(tot, E, tmp);
  const int total_r = kRank ? block_exclusive_scan(tot + E, R, tmp) : 0;
  if (cta == 0 && !kLL) {
    for (int e = tid; e <= E; e += kLayoutThreads) p.expert_off[e] = (e < E) ? tot[e] : total_e;
    if (kRank)
      for (int r = tid; r <= R; r += kLayoutThreads) p.rank_off[r] = (r < R) ? tot[E + r] : total_r;
  }
  if (kLL) {
    // Chunks are source ranks here: (offset << 32) | count of expert e's rows from source `cta`.
    for (int e = tid; e < E; e += kLayoutThreads)
      p.ll_range[static_cast<int64_t>(e) * R + cta] =
          (static_cast<int64_t>(base[e]) << 32) | static_cast<int64_t>(own[e]);
    if (cta == 0 && tid == 0) *p.ll_hdr = p.hdr_value;
  }
  // Running counters: warp prefix + chunk prefix (+ global offset in normal mode).
  for (int i = tid; i < kLayoutWarps * C; i += kLayoutThreads) {
    const int col = i % C;
    hist[i] += base[col] + (kLL ? 0 : tot[col]);
  }
  __syncthreads();

  // Pass 2: slots.
  bool overflow = false;
  for (int64_t b = wa0; b < wa1; b += 32) {
    const int64_t i = b + lane;
    const bool in = i < wa1;
    const int e = in ? __ldg(p.idx + i) : -1;
    const bool valid = in && e >= 0 && e < E;
    const unsigned pe = __match_any_sync(0xffffffffu, valid ? e : -2 - lane);
    const int slot = valid ? my[e] + __popc(pe & lanemask_lt()) : -1;
    int r = -1, rslot = -1;
    bool first = false;
    unsigned pr = 0;
    if (kRank) {
      r = valid ? e / L : -1;
      first = valid;
      if (valid) {
        const int64_t t = i / K;
        for (int64_t j = t * K; j < i; ++j) {
          const int e2 = __ldg(p.idx + j);
          if (e2 >= 0 && e2 < E && e2 / L == r) first = false;
        }
      }
      pr = __match_any_sync(0xffffffffu, first ? r : -2 - lane);
      rslot = first ? my[E + r] + __popc(pr & lanemask_lt()) : -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(pe) - 1) my[e] += __popc(pe);
    if (kRank && first && lane == __ffs(pr) - 1) my[E + r] += __popc(pr);
    __syncwarp();
    if (in) {
      if (kLL) {
        int32_t row = -1;
        if (valid) {
          if (slot < p.ll_cap)
            row = static_cast<int32_t>(static_cast<int64_t>(e) * p.ll_cap + slot);
          else
            overflow = true;
        }
        p.expert_slot[i] = row;
      } else {
        p.expert_slot[i] = slot;
      }
      if (kRank && first) {
        const int64_t t = i / K;
        p.rank_slot[t * R + r] = rslot;
        p.mask[t * R + r] = 1;
      }
    }
  }
  if (kLL && __any_sync(0xffffffffu, overflow) && lane == 0) flag(p.status, EP_ST_LL_OVERFLOW);
}

size_t layout_smem_bytes(int E, int R, bool with_rank) {
  const int C = E + (with_rank ? R : 0);
  return sizeof(int32_t) * (static_cast<size_t>(kLayoutWarps) * C + 3 * C + 32);
}

template <bool kRank, bool kLL>
static const void* layout_fn() {
  return reinterpret_cast<const void*>(&layout_kernel<kRank, kLL>);
}

static const void* pick_layout(bool with_rank, bool ll) {
  if (ll) return with_rank ? layout_fn<true, true>() : layout_fn<false, true>();
  return with_rank ? layout_fn<true, false>() : layout_fn<false, false>();
}

int layout_max_ctas(int E, int R, bool with_rank) {
  int dev = 0, sms = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (!coop) return 0;
  const size_t smem = layout_smem_bytes(E, R, with_rank);
  int best = 0;
  for (int ll = 0; ll < 2; ++ll) {
    const void* fn = pick_layout(with_rank, ll != 0);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kLayoutThreads, smem) != cudaSuccess)
      return 0;
    const int n = per_sm * sms;
    best = (ll == 0) ? n : (n < best ? n : best);
  }
  return best;
}

cudaError_t launch_layout(const LayoutParams& p, int G, bool with_rank, bool ll, cudaStream_t s) {
  const size_t smem = layout_smem_bytes(p.E, p.R, with_rank);
  const void* fn = pick_layout(with_rank, ll);
  cudaError_t err =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  if (G > 1) {
    err = cudaMemsetAsync(p.ws_barrier, 0, sizeof(unsigned), s);
    if (err != cudaSuccess) return err;
  }
  LayoutParams q = p;
  void* args[] = {&q};
  return cudaLaunchCooperativeKernel(fn, dim3(G), dim3(kLayoutThreads), args, smem, s);
}

}  // namespace ep
