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
// per CTA (up to 32 warps), and each chunk into contiguous warp ranges. A CTA
// first stages its chunk's indices in shared memory in one coalesced pass,
// coding each entry as (expert, rank, first-slot-of-the-token-on-that-rank;
// the flag from the token's earlier slots, neighbours of the entry's own
// index); divisions by E/R and K are multiply-highs. Pass 1 counts per warp with
// shared-memory atomics. One thread per column then walks the warps' counts,
// leaving each warp its prefix (a shuffle scan per column across the warps
// was bound by shuffle throughput: 2.2 of the kernel's 13.3 us at 16384
// tokens, against 0.6 us for the walk); the chunk totals go to global
// memory; one bounded grid barrier (cooperative launch); every CTA then sums
// the chunk totals before it (its prefix) and all of them (the totals), and
// warp 0 scans the totals over experts and ranks in one pass. Pass 2 walks the
// warp's range 32 entries at a time: ballots on the key bits give each lane
// the lanes with the same expert (rank); its slot is the warp's running count
// plus the chunk prefix and the global offset plus its position among them (a
// popcount), and one leader bumps the warp's counter. No atomics decide an
// order: slots follow (token, slot) order by construction. The kernel is
// bound by instruction latency, not memory: the traffic is a few hundred KB
// of int32.
// Low latency: chunks are source ranks. A small batch instead runs as one CTA
// in which a group of g warps holds each source rank's entries: the walk
// over the warps then gives the prefix over source ranks, and no grid barrier
// or exchange through memory is needed (nor with a single chunk in normal
// mode).
#include "common.cuh"
#include "kernels.cuh"

namespace ep {

constexpr int kMaxLayoutThreads = 1024;

// Exclusive scan of a[0..n) in shared memory by warp 0 (lane l scans a run
// of ceil(n / 32) entries, a shuffle scan joins the runs); returns the total
// to every thread. a[] must be complete; all threads must call it.
__device__ int warp0_exclusive_scan(int32_t* a, int n, int32_t* tmp) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (n + 31) / 32;
    const int lo = min(n, lane * per), hi = min(n, lo + per);
    int s = 0;
    for (int i = lo; i < hi; ++i) s += a[i];
    int v = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    int run = v - s;
    for (int i = lo; i < hi; ++i) {
      const int x = a[i];
      a[i] = run;
      run += x;
    }
    if (lane == 31) tmp[0] = v;
  }
  __syncthreads();
  return tmp[0];
}

// Entry code of one (token, slot): -1 for "no expert" (masked, or an index
// outside [-1, E)), else e | r << 10 | first << 20, where r is expert e's
// rank and `first` says that this slot is the token's first one on rank r
// (the slot that carries the token's per-rank copy).
constexpr int kFirstBit = 1 << 20;
__device__ __forceinline__ int code_e(int c) { return c & 1023; }
__device__ __forceinline__ int code_r(int c) { return (c >> 10) & 1023; }

// Lanes of the warp whose `key` equals this lane's, among lanes with `valid`
// set (0 for an invalid lane): one ballot per key bit. Keys lie in
// [0, 2^nbits). All lanes must call it (nbits warp-uniform).
__device__ __forceinline__ unsigned warp_peers(int key, bool valid, int nbits) {
  unsigned m = __ballot_sync(0xffffffffu, valid);
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (key >> b) & 1;
    const unsigned v = __ballot_sync(0xffffffffu, bit);
    m &= bit ? v : ~v;
  }
  return valid ? m : 0u;
}

// n / d for 0 <= n < 2^20 by a multiply-high with magic = ceil(2^32 / d)
// (magic 0 stands for d == 1); exact in that range for d <= 4096.
__device__ __forceinline__ int fast_div(int n, uint32_t magic) {
  return magic ? static_cast<int>(__umulhi(static_cast<unsigned>(n), magic)) : n;
}

template <bool kRank>
__device__ __forceinline__ int entry_code_global(const LayoutParams& p, int64_t i, bool& bad) {
  const int e = __ldg(p.idx + i);
  if (e == -1) return -1;
  if (e < 0 || e >= p.E) {
    bad = true;
    return -1;
  }
  const int r = e / p.L;
  int code = e | (r << 10);
  if (kRank) {
    bool first = true;
    const int64_t t = i / p.K;
    for (int64_t j = t * p.K; j < i; ++j) {
      const int e2 = __ldg(p.idx + j);
      if (e2 >= 0 && e2 < p.E && e2 / p.L == r) first = false;
    }
    if (first) code |= kFirstBit;
  }
  return code;
}

// Low-latency shrink mode: an entry is dropped (as if its index were -1) when
// its source rank (the CTA's chunk, or its warp range in the one-CTA form) or
// the rank holding its expert is masked.
template <bool kLL>
__device__ __forceinline__ bool ll_drop(const LayoutParams& p, int code, bool src_masked) {
  if (!kLL || code < 0 || !p.rank_mask) return false;
  return src_masked || __ldg(p.rank_mask + code_r(code)) != 0;
}

template <bool kRank, bool kLL, bool kStaged>
__global__ void __launch_bounds__(kMaxLayoutThreads) layout_kernel(const LayoutParams p) {
  extern __shared__ int32_t sm[];
  const int E = p.E, R = p.R, K = p.K;
  const int C = E + (kRank ? R : 0);
  const int NT = blockDim.x, W = NT >> 5;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int cta = blockIdx.x, G = gridDim.x;
  const int64_t N = p.N;
  const int64_t t0 = min(N, static_cast<int64_t>(cta) * p.tokens_per_cta);
  const int64_t t1 = min(N, t0 + p.tokens_per_cta);
  const int64_t a0 = t0 * K;
  const int n_ent = static_cast<int>((t1 - t0) * K);    // entries of this chunk
  const int per_warp = ((n_ent + W * 32 - 1) / (W * 32)) * 32;
  const int wa0 = min(n_ent, w * per_warp), wa1 = min(n_ent, wa0 + per_warp);

  const int CP = C | 1;                // odd row stride: conflict-free column access across warps
  int32_t* hist = sm;                  // [W][CP]: per-warp counts, then running slots
  int32_t* base = hist + W * CP;       // [C]: this chunk's prefix over earlier chunks
  int32_t* tot = base + C;             // [C]: totals, then their exclusive scan
  int32_t* own = tot + C;              // [C]: this chunk's own count
  int32_t* tmp = own + C;              // [32]
  const int PS = max(4 * NT, C);      // >= P * C for either prefix path below
  int32_t* part = tmp + 32;            // [2][PS]: partial sums over chunks
  int32_t* scode = part + 2 * PS;      // [tokens_per_cta * K]: entry codes (kStaged)

  // The low-latency send's dispatch may start now: it loads and quantises its
  // rows, then waits for this grid to finish before it reads any slot.
  launch_dependents();
  bool bad = false;
  // The barrier's generation, read before any block can have arrived.
  const unsigned gen0 = (G > 1 && tid == 0) ? barrier_generation(p.ws_barrier) : 0u;
  // Low-latency shrink mode: a masked source rank sends nothing. An entry's
  // source rank is this CTA's chunk or, in the one-CTA form (where source
  // ranks are warp groups), the warp group that holds entry li.
  const bool warp_src = kLL && p.ll_src_entries > 0;
  const bool cta_src_masked = kLL && p.rank_mask && !warp_src && __ldg(p.rank_mask + cta) != 0;
  auto src_masked = [&](int li) -> bool {
    if (!kLL || !p.rank_mask) return false;
    return warp_src ? __ldg(p.rank_mask + li / p.ll_src_entries) != 0 : cta_src_masked;
  };
  for (int i = tid; i < W * CP; i += NT) hist[i] = 0;
  if (kStaged) {
    // One coalesced pass over the chunk's indices; each entry's rank is
    // computed once here. In rank mode the entry also reads its token's
    // earlier slots (neighbours of its own index, from L1) and marks itself
    // when it is the token's first slot on its rank.
    for (int li = tid; li < n_ent; li += NT) {
      const int e = __ldg(p.idx + a0 + li);
      int code = -1;
      if (e != -1) {
        if (e >= 0 && e < E)
          code = e | (fast_div(e, p.magic_L) << 10);
        else
          bad = true;
      }
      if (kRank && code >= 0) {
        // a0 is a multiple of K, so li % K is the slot (li < 2^20 here)
        const int k = li - fast_div(li, p.magic_K) * K;
        bool first = true;
#pragma unroll 4
        for (int kk = 1; kk <= k; ++kk) {
          const int e2 = __ldg(p.idx + a0 + li - kk);
          if (e2 >= 0 && e2 < E && fast_div(e2, p.magic_L) == code_r(code)) first = false;
        }
        if (first) code |= kFirstBit;
      }
      scode[li] = ll_drop<kLL>(p, code, code >= 0 && src_masked(li)) ? -1 : code;
    }
  }
  __syncthreads();

  int32_t* my = hist + w * CP;

  // Pass 1: per-warp counts (shared-memory atomics: counting needs no order).
  for (int li = wa0 + lane; li < wa1; li += 32) {
    int code = kStaged ? scode[li] : entry_code_global<kRank>(p, a0 + li, bad);
    if (!kStaged && ll_drop<kLL>(p, code, code >= 0 && src_masked(li))) code = -1;
    if (code >= 0) {
      atomicAdd(&my[code_e(code)], 1);
      if (kRank && (code & kFirstBit)) atomicAdd(&my[E + code_r(code)], 1);
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag(p.status, EP_ST_BAD_INDEX);
  __syncthreads();

  // Per column: exclusive prefix over warps, one thread per column walking
  // the warps' counts (consecutive threads, consecutive columns: no bank
  // conflict; eight loads in flight at a time); the chunk's total goes out.
  for (int col = tid; col < C; col += NT) {
    const bool ranges = warp_src && col < E;
    const int g = ranges ? p.ll_src_warps : 1;
    int run = 0, lo = 0;
    for (int w0 = 0; w0 < W; w0 += 8) {
      int x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = (w0 + u < W) ? hist[(w0 + u) * CP + col] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int w2 = w0 + u;
        if (w2 < W) hist[w2 * CP + col] = run;
        if (ranges && w2 < W && w2 % g == 0) lo = run;
        run += x[u];
        if (ranges && w2 < W && w2 % g == g - 1) {
          // One-CTA low-latency form: warps [s*g, (s+1)*g) hold source rank
          // s, so its range of expert col is (prefix before its first warp,
          // count up to the end of its last warp).
          const int64_t l = min(static_cast<int64_t>(lo), p.ll_cap);
          const int64_t h = min(static_cast<int64_t>(run), p.ll_cap);
          p.ll_range[static_cast<int64_t>(col) * R + w2 / g] = (l << 32) | (h - l);
        }
      }
    }
    own[col] = run;
    if (G > 1) p.ws_chunk[static_cast<int64_t>(cta) * C + col] = run;
  }
  if (G > 1)
    grid_barrier(p.ws_barrier, static_cast<unsigned>(G), gen0, p.status);
  else
    __syncthreads();
  // Clear this chunk's rows of the mask and the rank slots now, after the
  // barrier (whose fence then need not wait for these stores); the block
  // synchronisations below order them before pass 2 writes its entries.
  if (kRank) {
    for (int64_t i = t0 * R + tid; i < t1 * R; i += NT) {
      p.mask[i] = 0;
      p.rank_slot[i] = -1;
    }
  }

  // Prefix over earlier chunks and totals over all chunks (four columns per
  // 16-byte load when C % 4 == 0). One CTA: no other chunks, the totals are
  // its own counts.
  const int CV = (C % 4 == 0) ? C / 4 : 0;   // 16-byte column groups
  const int P = CV ? max(1, min(NT / CV, G)) : max(1, min(NT / C, G));
  // Column totals and this chunk's prefix land in tot[] / base[]; cta 0 also
  // writes the counts. Aligned layouts scan the padded segment lengths (the
  // counts stay true).
  auto put = [&](int col, int pre, int total) {
    base[col] = pre;
    if (cta == 0) {
      if (col < E)
        p.per_expert[col] = total;
      else
        p.per_rank[col - E] = total;
    }
    if (p.align > 1 && col < E) total = (total + p.align - 1) / p.align * p.align;
    tot[col] = total;
  };
  // Up to 64 chunks: an octet of lanes per group of four columns, each lane
  // summing every eighth chunk (at most eight loads, all in flight at once);
  // shuffles reduce the octet. More chunks: P threads per column group, each
  // summing every P-th chunk, partial sums reduced through shared memory.
  constexpr int kOct = 8;
  if (G > 1 && CV && CV * kOct <= NT && G <= 8 * kOct) {
    const int4* chunk4 = reinterpret_cast<const int4*>(p.ws_chunk);
    const bool act = tid < CV * kOct;  // whole octets: CV * kOct is a multiple of 8
    const int cv = tid / kOct, pp = tid % kOct;
    int4 pre = make_int4(0, 0, 0, 0), total = pre;
    if (act) {
      int4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = (pp + u * kOct < G) ? __ldcg(chunk4 + static_cast<int64_t>(pp + u * kOct) * CV + cv)
                                   : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool before = pp + u * kOct < cta;
        pre.x += before ? v[u].x : 0; pre.y += before ? v[u].y : 0;
        pre.z += before ? v[u].z : 0; pre.w += before ? v[u].w : 0;
        total.x += v[u].x; total.y += v[u].y; total.z += v[u].z; total.w += v[u].w;
      }
    }
#pragma unroll
    for (int o = 1; o < kOct; o <<= 1) {
      pre.x += __shfl_xor_sync(0xffffffffu, pre.x, o); pre.y += __shfl_xor_sync(0xffffffffu, pre.y, o);
      pre.z += __shfl_xor_sync(0xffffffffu, pre.z, o); pre.w += __shfl_xor_sync(0xffffffffu, pre.w, o);
      total.x += __shfl_xor_sync(0xffffffffu, total.x, o); total.y += __shfl_xor_sync(0xffffffffu, total.y, o);
      total.z += __shfl_xor_sync(0xffffffffu, total.z, o); total.w += __shfl_xor_sync(0xffffffffu, total.w, o);
    }
    if (act && pp == 0) {
      put(4 * cv, pre.x, total.x); put(4 * cv + 1, pre.y, total.y);
      put(4 * cv + 2, pre.z, total.z); put(4 * cv + 3, pre.w, total.w);
    }
  } else {
    if (G > 1 && CV) {
      const int4* chunk4 = reinterpret_cast<const int4*>(p.ws_chunk);
      for (int j = tid; j < P * CV; j += NT) {
        const int cv = j % CV, pp = j / CV;
        int4 pre = make_int4(0, 0, 0, 0), total = pre;
        for (int c = pp; c < G; c += 8 * P) {
          int4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            v[u] = (c + u * P < G) ? __ldcg(chunk4 + static_cast<int64_t>(c + u * P) * CV + cv) : make_int4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const bool before = c + u * P < cta;
            pre.x += before ? v[u].x : 0; pre.y += before ? v[u].y : 0;
            pre.z += before ? v[u].z : 0; pre.w += before ? v[u].w : 0;
            total.x += v[u].x; total.y += v[u].y; total.z += v[u].z; total.w += v[u].w;
          }
        }
        const int col = 4 * cv;  // part[pp * C + col .. col + 3]
        part[pp * C + col] = pre.x; part[pp * C + col + 1] = pre.y;
        part[pp * C + col + 2] = pre.z; part[pp * C + col + 3] = pre.w;
        part[PS + pp * C + col] = total.x; part[PS + pp * C + col + 1] = total.y;
        part[PS + pp * C + col + 2] = total.z; part[PS + pp * C + col + 3] = total.w;
      }
    }
    for (int j = tid; G > 1 && !CV && j < P * C; j += NT) {
      const int col = j % C, pp = j / C;
      int pre = 0, total = 0, c = pp;
      for (; c + 7 * P < G; c += 8 * P) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcg(p.ws_chunk + static_cast<int64_t>(c + u * P) * C + col);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          pre += (c + u * P < cta) ? v[u] : 0;
          total += v[u];
        }
      }
      for (; c < G; c += P) {
        const int v = __ldcg(p.ws_chunk + static_cast<int64_t>(c) * C + col);
        pre += (c < cta) ? v : 0;
        total += v;
      }
      part[j] = pre;  // j < P * C <= PS
      part[PS + j] = total;
    }
    if (G > 1) __syncthreads();
    for (int col = tid; col < C; col += NT) {
      int pre = 0, total = own[col];
      if (G > 1) {
        total = 0;
        for (int pp = 0; pp < P; ++pp) {
          pre += part[pp * C + col];
          total += part[PS + pp * C + col];
        }
      }
      put(col, pre, total);
    }
  }
  __syncthreads();
  // One scan over the expert and the rank columns together (by warp 0); a
  // rank column's offset is its prefix minus the expert total.
  const int total_c = warp0_exclusive_scan(tot, C, tmp);
  const int total_e = kRank ? tot[E] : total_c;
  const int total_r = total_c - total_e;
  if (cta == 0 && !kLL) {
    for (int e = tid; e <= E; e += NT) p.expert_off[e] = (e < E) ? tot[e] : total_e;
    if (kRank)
      for (int r = tid; r <= R; r += NT) p.rank_off[r] = (r < R) ? tot[E + r] - total_e : total_r;
  }
  if (kLL) {
    // Chunks are source ranks here: (offset << 32) | count of expert e's rows
    // from source `cta` (the one-CTA form wrote its ranges in the column scan).
    // Rows at j >= ll_cap overflow the region (only repeated experts in a
    // row get there); a range covers the rows that landed.
    for (int e = tid; !warp_src && e < E; e += NT) {
      const int64_t lo = min(static_cast<int64_t>(base[e]), p.ll_cap);
      const int64_t hi = min(static_cast<int64_t>(base[e]) + own[e], p.ll_cap);
      p.ll_range[static_cast<int64_t>(e) * R + cta] = (lo << 32) | (hi - lo);
    }
    if (cta == 0 && tid == 0) *p.ll_hdr = p.hdr_value;
  }

  // Pass 2: slots, in (token, slot) order within the warp's range.
  bool overflow = false, bad2 = false;
  for (int b = wa0; b < wa1; b += 32) {
    const int li = b + lane;
    const bool in = li < wa1;
    int code = in ? (kStaged ? scode[li] : entry_code_global<kRank>(p, a0 + li, bad2)) : -1;
    if (!kStaged && ll_drop<kLL>(p, code, code >= 0 && src_masked(li))) code = -1;
    const bool valid = code >= 0;
    const int e = code_e(code);
    const unsigned pe = warp_peers(e, valid, p.bits_E);
    // warp prefix (running) + chunk prefix (+ global offset in normal mode)
    const int slot = valid ? my[e] + base[e] + (kLL ? 0 : tot[e]) + __popc(pe & lanemask_lt()) : -1;
    const bool first = kRank && valid && (code & kFirstBit);
    const int r = code_r(code);
    unsigned pr = 0;
    int rslot = -1;
    if (kRank) {
      pr = warp_peers(r, first, p.bits_R);
      rslot = first ? my[E + r] + base[E + r] + (kLL ? 0 : tot[E + r] - total_e) + __popc(pr & lanemask_lt()) : -1;
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
        p.expert_slot[a0 + li] = row;
      } else {
        p.expert_slot[a0 + li] = slot;
      }
      if (kRank && first) {
        // fast_div is exact below 2^20, which bounds a staged chunk
        const int64_t t = t0 + (kStaged ? fast_div(li, p.magic_K) : li / K);
        p.rank_slot[t * R + r] = rslot;
        p.mask[t * R + r] = 1;
      }
    }
  }
  if (kLL && __any_sync(0xffffffffu, overflow) && lane == 0) flag(p.status, EP_ST_LL_OVERFLOW);
}

// ---- host side ---------------------------------------------------------------
constexpr size_t kMaxStagedEntries = 24576;  // 96 KB of entry codes per CTA
constexpr int kVariants = 8;                 // kRank x kLL x kStaged
constexpr size_t kHistBudget = 96 * 1024;    // per-warp counters

// Threads per block: as many warps (up to 32) as the per-warp counters allow.
// (Fewer warps for small chunks were measured slower on a 128-token batch.)
static int layout_threads(int E, int R, bool with_rank) {
  const size_t C = static_cast<size_t>(E) + (with_rank ? R : 0);
  int W = 32;
  while (W > 4 && static_cast<size_t>(W) * C * sizeof(int32_t) > kHistBudget) W >>= 1;
  return W * 32;
}

static size_t layout_smem(int E, int R, bool with_rank, int threads, size_t staged_entries) {
  const size_t C = static_cast<size_t>(E) + (with_rank ? R : 0);
  const size_t CP = C | 1;
  const size_t W = threads / 32;
  const size_t PS = C > 4 * static_cast<size_t>(threads) ? C : 4 * static_cast<size_t>(threads);
  return sizeof(int32_t) * (W * CP + 3 * C + 32 + 2 * PS + staged_entries);
}

size_t layout_smem_bytes(int E, int R, bool with_rank) {
  return layout_smem(E, R, with_rank, layout_threads(E, R, with_rank), 0);
}

static const void* layout_fn(bool rank, bool ll, bool staged) {
  const void* fns[kVariants] = {
      reinterpret_cast<const void*>(&layout_kernel<false, false, false>),
      reinterpret_cast<const void*>(&layout_kernel<false, false, true>),
      reinterpret_cast<const void*>(&layout_kernel<false, true, false>),
      reinterpret_cast<const void*>(&layout_kernel<false, true, true>),
      reinterpret_cast<const void*>(&layout_kernel<true, false, false>),
      reinterpret_cast<const void*>(&layout_kernel<true, false, true>),
      reinterpret_cast<const void*>(&layout_kernel<true, true, false>),
      reinterpret_cast<const void*>(&layout_kernel<true, true, true>),
  };
  return fns[(rank ? 4 : 0) + (ll ? 2 : 0) + (staged ? 1 : 0)];
}

static cudaError_t prepare(int dev, bool rank, bool ll, bool staged, size_t smem) {
  return ensure_dynamic_smem(layout_fn(rank, ll, staged), dev, smem);
}

static int coresident(int dev, bool rank, bool ll, bool staged, int threads, size_t smem) {
  if (prepare(dev, rank, ll, staged, smem) != cudaSuccess) return 0;
  return blocks_per_sm(layout_fn(rank, ll, staged), dev, threads, smem) * device_sms(dev);
}

int layout_max_ctas(int E, int R, bool with_rank) {
  const int dev = current_device();
  if (dev < 0 || !device_cooperative(dev)) return 0;
  const int threads = layout_threads(E, R, with_rank);
  const size_t smem = layout_smem(E, R, with_rank, threads, 0);
  const int a = coresident(dev, with_rank, false, false, threads, smem);
  const int b = coresident(dev, with_rank, true, false, threads, smem);
  return a < b ? a : b;
}

cudaError_t launch_layout(const LayoutParams& p, int G, bool with_rank, bool ll, cudaStream_t s) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorNoDevice;
  // The one-CTA low-latency form runs ll_src_warps warps per source rank.
  const int threads = p.ll_src_entries > 0 ? p.R * p.ll_src_warps * 32 : layout_threads(p.E, p.R, with_rank);
  const size_t entries = static_cast<size_t>(p.tokens_per_cta) * p.K;
  bool staged = entries <= kMaxStagedEntries;
  size_t smem = layout_smem(p.E, p.R, with_rank, threads, staged ? entries : 0);
  if (staged && coresident(dev, with_rank, ll, true, threads, smem) < G) {
    staged = false;
    smem = layout_smem(p.E, p.R, with_rank, threads, 0);
  }
  const cudaError_t err = prepare(dev, with_rank, ll, staged, smem);
  if (err != cudaSuccess) return err;
  LayoutParams q = p;
  q.magic_L = p.L > 1 ? static_cast<uint32_t>(((uint64_t(1) << 32) + p.L - 1) / p.L) : 0u;
  q.magic_K = p.K > 1 ? static_cast<uint32_t>(((uint64_t(1) << 32) + p.K - 1) / p.K) : 0u;
  q.bits_E = 0;
  while ((1 << q.bits_E) < p.E) ++q.bits_E;
  q.bits_R = 0;
  while ((1 << q.bits_R) < p.R) ++q.bits_R;
  void* args[] = {&q};
  return cudaLaunchCooperativeKernel(layout_fn(with_rank, ll, staged), dim3(G), dim3(threads), args, smem, s);
}

}  // namespace ep
