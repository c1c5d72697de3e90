// Device helpers shared by the sm_103a kernels of this library.
//
// Inline PTX for the Blackwell data-movement primitives used on the hot path:
// the bulk (non-tensor) TMA copies global -> shared (completing on an
// mbarrier) and shared -> global (bulk groups), the async-proxy fence, the
// streaming row load, the programmatic-dependent-launch controls, and the
// acquire loads of the bounded grid-wide barrier.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ep.h"

namespace ep {

// Wait limits, in nanoseconds of the GPU's global timer. A wait that exceeds
// its limit sets EP_ST_TIMEOUT and returns; no kernel of this library can
// wait forever. Every wait here normally ends within microseconds (a row
// landing in shared memory, the other blocks of a cooperative grid arriving),
// so one second means something is wrong. kDrainLimitNs bounds the second
// wait a block makes for its own bulk copy still in flight before it leaves
// (the copy depends on no other block and lands unless its address is bad).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s
constexpr unsigned long long kDrainLimitNs = 4000000000ull;  // 4 s

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void flag(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ---- mbarrier ------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete: false (and
// EP_ST_TIMEOUT) after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      flag(status, EP_ST_TIMEOUT);
      return false;
    }
  }
  return true;
}

// After a timed-out mbar_wait, before the block gives up its shared memory:
// wait (with backoff, up to kDrainLimitNs) for the bulk load that targets it,
// so the copy cannot land in memory a later block owns.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, unsigned parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity) && global_ns() - t0 <= kDrainLimitNs) __nanosleep(1000);
}

// ---- bulk TMA copies -----------------------------------------------------
// global -> shared, completion counted on an mbarrier (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global, tracked in this thread's current bulk group.
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- loads ----------------------------------------------------------------
// A 16-byte load of data read exactly once: no L1 allocation, and first in
// line for eviction from L2 (an evict-first access policy), so the stream of
// rows does not push out data that is still wanted.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile(
      "{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---- programmatic dependent launch ---------------------------------------------
// A kernel launched with programmatic stream serialization may start while
// the kernel before it on the stream is still running, once every block of
// that kernel has issued launch_dependents (or exited). Before it reads what
// that kernel writes it must wait for it: grid_dependency_wait returns once
// the preceding grid has completed and its memory is visible. In a launch
// without the attribute the wait returns at once.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `fn` on stream s. With `dependent`, as a programmatic dependent of
// the kernel before it on the stream: it may be scheduled while that kernel
// drains, so its launch latency hides behind that kernel's tail, and it must
// call grid_dependency_wait() before it touches any memory (which makes it
// ordered exactly as a plain launch would be).
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*fn)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool dependent,
                          Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, static_cast<Args&&>(args)...);
}

// ---- grid-wide barrier (cooperative launches only) --------------------------
// One barrier per launch over two words that persist across launches: bar[0]
// counts arrivals and is zero between launches, bar[1] is a generation
// number. Thread 0 of every block reads the generation early in the launch
// (barrier_generation), before it can change; the last block to arrive
// bumps the generation, which releases the others, and then clears the count.
// So a workspace that was zero-filled once needs no reset between calls. A
// block whose arrival count comes back >= nblocks found leftover words (a
// workspace never zero-filled, or one an aborted launch left behind): it
// flags EP_ST_WORKSPACE and does not wait. Waits are bounded (kWaitLimitNs):
// on expiry the block flags EP_ST_TIMEOUT and goes on; every access after
// the barrier stays inside the caller's arrays, so the outputs are merely
// wrong, and the status says so.
// A relaxed read: the generation cannot change before this block arrives, so
// no ordering is needed, and the thread does not stall on it until the wait.
__device__ __forceinline__ unsigned barrier_generation(const unsigned* bar) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar + 1));
  return v;
}

__device__ __forceinline__ void grid_barrier(unsigned* bar, unsigned nblocks, unsigned gen0, int32_t* status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this block's writes are visible before its arrival
    const unsigned old = atomicAdd(&bar[0], 1u);
    if (old >= nblocks) {
      flag(status, EP_ST_WORKSPACE);
    } else if (old == nblocks - 1) {
      __threadfence();
      atomicAdd(&bar[1], 1u);
      // Every block has arrived, none reads the count again in this launch,
      // and the next launch starts after this one completes: the reset is a
      // plain store after the release, off the others' critical path.
      *reinterpret_cast<volatile unsigned*>(&bar[0]) = 0u;
    } else {
      const unsigned long long t0 = global_ns();
      while (ld_acquire_u32(bar + 1) == gen0) {
        if (global_ns() - t0 > kWaitLimitNs) {
          flag(status, EP_ST_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
    }
    // (The acquire load that saw the new generation orders this block's
    // later reads; they read the chunk counts from L2.)
  }
  __syncthreads();
}

// ---- number formats --------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> two BF16 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Two fp32 -> two E4M3 codes (round to nearest even, saturating), `lo` in the
// low byte. The PTX form puts its first source operand in the upper byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("{\n\t.reg .b16 t;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"
      "mov.b16 %0, t;\n\t}"
      : "=h"(d)
      : "f"(hi), "f"(lo));
  return d;
}

}  // namespace ep
