// qmoe_moe_forward_noalloc: the routed-MoE layer with library-owned scratch.
//
// Some callers cannot allocate device memory at all: plugin interfaces that
// hand an operator only its input and output buffers, or threads that must not
// call cudaMalloc because it can synchronise the whole device. For them this
// entry point takes its scratch from a fixed array in device memory that the
// library declares at file scope, so the caller passes only inputs and
// outputs.
//
// The array holds QMOE_NOALLOC_SCRATCH_BYTES (8 MiB) on every GPU that loads
// the library, until the process exits. Host code cannot use the array's name
// as a device address, so the first call on each device looks the address up
// with cudaGetSymbolAddress (with that device current) and keeps it.
#include <atomic>

#include "kernels.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[QMOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::atomic<void*> g_scratch_addr[kMaxDev];

// Device address of this device's scratch array (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return QMOE_ERR_CUDA;
  void* p = g_scratch_addr[dev].load();
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QMOE_ERR_CUDA;
    g_scratch_addr[dev].store(p);
  }
  *out = p;
  return QMOE_OK;
}

}  // namespace

extern "C" int qmoe_moe_forward_noalloc(const qmoe_moe_desc* d, const float* X, const float* R, float* out,
                                        int T, qmoe_stream_t stream) {
  if (T < 0) return QMOE_ERR_ARG;
  if (T == 0) return qmoe_moe_forward(d, X, R, nullptr, nullptr, out, 0, nullptr, 0, stream);
  const size_t need = qmoe_moe_workspace_bytes(d, T);
  if (need == 0)  // invalid descriptor: let the regular entry point name the problem
    return qmoe_moe_forward(d, X, R, nullptr, nullptr, out, T, nullptr, 0, stream);
  if (need > (size_t)QMOE_NOALLOC_SCRATCH_BYTES) return QMOE_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int r = scratch_address(&scratch);
  if (r != QMOE_OK) return r;
  // Every scratch byte a call reads is written earlier in the same call, so
  // nothing needs clearing between calls.
  return qmoe_moe_forward(d, X, R, nullptr, nullptr, out, T, scratch, (size_t)QMOE_NOALLOC_SCRATCH_BYTES,
                          stream);
}
