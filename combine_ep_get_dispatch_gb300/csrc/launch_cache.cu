// Host-side launch bookkeeping, cached per process.
//
// Every entry point runs on the host before it enqueues its kernel, and on a
// decode-sized batch that host time is as long as the kernels themselves. The
// answers to the questions a launch asks do not change while the process
// runs: a device's SM count and cooperative-launch support, how many blocks
// of a kernel fit on one SM for a given block size and shared memory, and
// whether a kernel's dynamic shared-memory limit has already been raised. So
// each is asked of the runtime once and remembered. The tables are guarded by
// one mutex; the attribute and occupancy queries run outside it, the
// shared-memory limit call inside it (see ensure_dynamic_smem).
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.cuh"

namespace ep {

namespace {

struct DeviceInfo {
  bool known = false;
  int sms = 0;
  int coop = 0;
};

constexpr int kMaxDevices = 64;

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
std::map<std::tuple<const void*, int, int, size_t>, int> g_occupancy;  // (fn, dev, threads, smem)
std::map<std::pair<const void*, int>, size_t> g_smem_limit;            // (fn, dev) -> limit set

const DeviceInfo* device_info(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_dev[dev].known) return &g_dev[dev];
  }
  DeviceInfo d;
  if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
  if (cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) return nullptr;
  d.known = true;
  std::lock_guard<std::mutex> lock(g_mutex);
  g_dev[dev] = d;
  return &g_dev[dev];
}

}  // namespace

int current_device() {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

int device_sms(int dev) {
  const DeviceInfo* d = device_info(dev);
  return d ? d->sms : 0;
}

bool device_cooperative(int dev) {
  const DeviceInfo* d = device_info(dev);
  return d && d->coop != 0;
}

// The check, the runtime call and the record happen under one lock: two
// threads raising the same kernel's limit to different values must leave the
// runtime at the value the table records (otherwise the smaller call could
// land last while the table kept the larger one).
cudaError_t ensure_dynamic_smem(const void* fn, int dev, size_t smem) {
  std::lock_guard<std::mutex> lock(g_mutex);
  size_t& v = g_smem_limit[{fn, dev}];
  if (v >= smem) return cudaSuccess;
  const cudaError_t err =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  v = smem;
  return cudaSuccess;
}

int blocks_per_sm(const void* fn, int dev, int threads, size_t smem) {
  const auto key = std::make_tuple(fn, dev, threads, smem);
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    const auto it = g_occupancy.find(key);
    if (it != g_occupancy.end()) return it->second;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  g_occupancy[key] = per_sm;
  return per_sm;
}

}  // namespace ep
