// static_ws.cu -- the decode layer for callers that cannot allocate device
// memory.
//
// Some callers of a decode step have no way to obtain a workspace: a host
// application that hands this library only its activation and weight buffers
// and keeps every other byte of device memory under its own accounting, or a
// latency-critical token loop that must not enter the CUDA allocator between
// tokens.  For them lily_moe_decode_static() runs exactly the work of
// lily_moe_decode() with its scratch memory taken from one fixed array that
// the library declares at file scope.  The array is created when the library
// is loaded on a device and stays there, at its full size, until the process
// exits.
#include <mutex>

#include "common.cuh"

namespace lily {
namespace {

// Largest scratch the static variant can use.  1 MiB covers a decode step of
// up to 8 rows at d_model 2048 / d_ff 512 (about 0.7 MiB); bigger shapes are
// refused (LILY_ERR_WORKSPACE_TOO_SMALL).
constexpr size_t kStaticScratchBytes = 1u << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The array's name in host code is only a host-side handle; the device
// address differs per device and is looked up once per device.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LILY_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LILY_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return LILY_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return LILY_OK;
}

}  // namespace
}  // namespace lily

extern "C" int lily_moe_decode_static(const lily_moe_dims* dims, const void* x,
                                      const lily_moe_weights* weights, lily_moe_routing* routing,
                                      void* y, void* stream) {
  using namespace lily;
  if (!dims) return LILY_ERR_INVALID_ARG;
  const size_t need = lily_moe_workspace_bytes(dims);
  if (need == 0) return lily_moe_check_dims(dims);
  // more rows than the decode path takes is a shape error, whatever the size
  if (dims->T > 8) return LILY_ERR_UNSUPPORTED_SHAPE;
  if (need > kStaticScratchBytes) return LILY_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  int rc = scratch_address(&ws);
  if (rc) return rc;
  // The array keeps whatever the previous call left in it.  Only its first
  // 256 bytes (status word and grid-barrier counters) must start at zero; the
  // rest is fully rewritten by every call.
  if (cudaMemsetAsync(ws, 0, 256, (cudaStream_t)stream) != cudaSuccess) return LILY_ERR_CUDA;
  return lily_moe_decode(dims, x, weights, routing, y, ws, kStaticScratchBytes, stream);
}
