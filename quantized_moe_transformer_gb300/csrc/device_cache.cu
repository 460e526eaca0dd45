// Per-device launch bookkeeping: the dynamic shared-memory limit raised for a
// kernel and each device's SM count. cudaFuncSetAttribute acts on the current
// device only, so a process that drives several GPUs must raise the limit once
// per (device, kernel); both tables are keyed by the current device and
// guarded by one mutex.
#include <mutex>

#include "kernels.cuh"

namespace qmoe {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxEntries = 512;

struct AttrEntry {
  int dev;
  const void* fn;
  size_t smem;  // largest dynamic shared memory size set so far
  int carveout;
};

std::mutex g_mu;
AttrEntry g_attr[kMaxEntries];
int g_n_attr = 0;
int g_sms[kMaxDevices];

}  // namespace

cudaError_t ensure_kernel_smem(const void* fn, size_t smem, int carveout) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  int i = 0;
  while (i < g_n_attr && !(g_attr[i].dev == dev && g_attr[i].fn == fn)) ++i;
  if (i == g_n_attr) {
    if (g_n_attr == kMaxEntries) return cudaErrorInvalidValue;
    g_attr[i] = AttrEntry{dev, fn, 0, -1};
    ++g_n_attr;
  }
  AttrEntry& a = g_attr[i];
  if (carveout >= 0 && a.carveout != carveout) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
    if (e != cudaSuccess) return e;
    a.carveout = carveout;
  }
  // the default limit is 48 KB minus the kernel's static shared memory, so
  // every dynamic size a launch asks for is set explicitly the first time
  if (smem > a.smem) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    a.smem = smem;
  }
  return cudaSuccess;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sms[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = v > 0 ? v : 1;
  }
  return g_sms[dev];
}

}  // namespace qmoe
