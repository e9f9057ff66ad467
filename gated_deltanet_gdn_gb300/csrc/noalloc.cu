// gdn_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate device
// memory. The residual records the forward passes between its two kernels live in a
// fixed array compiled into the library instead of a caller-provided buffer.
#include <cstdint>
#include <mutex>

#include "../../include/gdn.h"
#include "kernels.h"

namespace gdn {
namespace {

// Scratch for the forward's residual records. Every GPU that loads the library holds
// these GDN_NOALLOC_SCRATCH_BYTES until the process exits. Host code must never pass
// this symbol to a kernel (on the host it only names a stand-in); it passes the device
// address obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_fwd_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
void* g_scratch_addr[MAX_DEVICES];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device, resolved once per device
// with that device current. NULL if the runtime cannot resolve it.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_chunk_fwd_noalloc(const gdn_dims* dims, const void* q, const void* k,
                                     const void* v, const void* g, const void* beta,
                                     const float* h0, float scale, void* out, float* h_final,
                                     void* stream) {
  if (!dims) return GDN_ERR_INVALID_ARG;
  // 0 for an empty problem or for dims the forward rejects (it reports why below)
  const size_t need = gdn_chunk_residual_bytes(dims);
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = gdn::scratch_address();
    if (!scratch) return GDN_ERR_CUDA;
  }
  // The residual records are written in full by the first kernel before the second
  // reads them, so nothing in the shared array needs clearing between calls.
  return gdn_chunk_fwd(dims, q, k, v, g, beta, h0, scale, out, h_final, scratch, stream);
}
