// Low-latency receive phase and the element-wise E4M3 encoder.
//
// The receive phase is the deferred second launch of the low-latency
// dispatch ("How DeepEP enables hook-based overlapping", "Two-Phase Kernel
// Architecture": the receive phase runs when the hook is called; "DeepEP V1
// (legacy) guide", section 6.3: the hook guarantees the data has arrived and
// the per-expert receive counts are returned). On one GPU the send already
// placed the rows; the receive checks that a send with the same shapes
// filled the workspace, then publishes the per-expert counts and the
// per-(expert, source rank) ranges, and marks the workspace consumed. It
// never waits on another launch: it must be ordered after the send on the
// stream.
#include "common.cuh"
#include "kernels.cuh"

namespace ep {

namespace {

constexpr int kRecvThreads = 1024;
constexpr int kRecvUnroll = 8;  // ranges per thread with their loads in flight together

// One block (E <= 1024 = one expert per thread). Every load of the first
// round goes out before the header has been checked: the header, this
// thread's count and running statistic, and up to kRecvUnroll of its ranges;
// only the stores wait for the check. Larger range tables are copied in
// further rounds of kRecvUnroll loads, then kRecvUnroll stores. The header is
// marked consumed last; later launches on the stream see it.
__global__ void __launch_bounds__(kRecvThreads) ll_recv_kernel(const LLRecvParams p, int E, int R) {
  __shared__ int s_ok;
  const int tid = threadIdx.x;
  // Launched as a programmatic dependent (the send before it drains while
  // this block is scheduled): wait for it before reading the workspace, and
  // let the next kernel on the stream be scheduled at once.
  grid_dependency_wait();
  launch_dependents();
  LLHeader h{};
  if (tid == 0) h = *p.hdr;  // written by an earlier launch on this stream
  const int32_t c = tid < E ? p.count[tid] : 0;
  const int32_t acc = (tid < E && p.stats) ? p.stats[tid] : 0;
  const int64_t n = p.layout_range ? static_cast<int64_t>(E) * R : 0;
  constexpr int64_t kRound = static_cast<int64_t>(kRecvThreads) * kRecvUnroll;
  int64_t r[kRecvUnroll];
#pragma unroll
  for (int u = 0; u < kRecvUnroll; ++u) {
    const int64_t i = static_cast<int64_t>(u) * kRecvThreads + tid;
    r[u] = i < n ? p.range[i] : 0;
  }
  if (tid == 0) {
    int ok = 1;
    if (h.magic != kMagicSent) {
      ok = 0;
      flag(p.status, EP_ST_NOT_SENT);
    } else if (h.N != p.expect.N || h.K != p.expect.K || h.E != p.expect.E || h.R != p.expect.R ||
               h.T != p.expect.T) {
      ok = 0;
      flag(p.status, EP_ST_MISMATCH);
    }
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  if (tid < E) {
    p.recv_count[tid] = c;
    if (p.stats) p.stats[tid] = acc + c;  // one block: no other writer
  }
  for (int64_t b = 0; b < n; b += kRound) {
    if (b > 0) {
#pragma unroll
      for (int u = 0; u < kRecvUnroll; ++u) {
        const int64_t i = b + static_cast<int64_t>(u) * kRecvThreads + tid;
        r[u] = i < n ? p.range[i] : 0;
      }
    }
#pragma unroll
    for (int u = 0; u < kRecvUnroll; ++u) {
      const int64_t i = b + static_cast<int64_t>(u) * kRecvThreads + tid;
      if (i < n) p.layout_range[i] = r[u];
    }
  }
  __syncthreads();
  if (tid == 0) p.hdr->magic = kMagicReceived;
}

// Shrink-mode mask buffer: mode 0 sets mask[rank] = value, 1 copies the mask
// to out, 2 clears it.
__global__ void ll_mask_kernel(int32_t* mask, int R, int mode, int rank, int value, int32_t* out) {
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    if (mode == 0 && i == rank) mask[i] = value;
    if (mode == 1) out[i] = mask[i];
    if (mode == 2) mask[i] = 0;
  }
}

__global__ void e4m3_encode_kernel(const float* __restrict__ in, uint8_t* __restrict__ out, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint8_t>(pack_e4m3x2(in[i], 0.0f) & 0xFFu);
}

}  // namespace

cudaError_t launch_ll_recv(const LLRecvParams& p, int E, int R, cudaStream_t s) {
  return launch_kernel(ll_recv_kernel, dim3(1), dim3(kRecvThreads), 0, s, /*dependent=*/true, p, E, R);
}

cudaError_t launch_ll_mask(int32_t* mask, int R, int mode, int rank, int value, int32_t* out, cudaStream_t s) {
  ll_mask_kernel<<<1, 256, 0, s>>>(mask, R, mode, rank, value, out);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int sms = device_sms(current_device());
  const int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  e4m3_encode_kernel<<<static_cast<int>(blocks < cap ? blocks : cap), 256, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

}  // namespace ep
