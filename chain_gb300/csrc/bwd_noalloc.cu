// bwd_noalloc.cu -- the attention backward for callers that cannot
// allocate device memory (chain_bwd_noalloc in include/chain.h).
//
// chain_bwd keeps an fp32 row term D (one value per query row) in a
// scratch workspace the caller passes in.  Here that
// scratch is a fixed array compiled into the library instead, so a caller
// with no allocator at hand (a pre-reserved memory pool it cannot reach, a
// plugin that must not grow the device footprint, a loop that cannot take
// the device-wide synchronisation of cudaMalloc) can still run the
// backward.  Nothing in this file allocates: the array exists from the
// moment the library's module is loaded on a device until the process ends.
#include <mutex>

#include "../../include/chain.h"
#include "internal.h"

namespace chain {

// 32 MiB, shared by every call on a device.  Host code must not use the
// symbol's address directly (on the host it names a stand-in, not device
// memory); the device address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CHAIN_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};
}  // namespace

}  // namespace chain

extern "C" int chain_bwd_noalloc(const chain_tensor_t *dO, const chain_tensor_t *A,
                                 const chain_tensor_t *B, const chain_tensor_t *C,
                                 const chain_tensor_t *O, const chain_tensor_t *LSE, int f,
                                 int mask, float scale, chain_tensor_t *dA, chain_tensor_t *dB,
                                 chain_tensor_t *dC, void *stream) {
  using namespace chain;
  // Sized by the chain f names: an MLP whose X and W2 share one shape would
  // otherwise be sized as attention.
  const size_t need = chain_bwd_workspace_size_f(A, C, f);
  if (need == 0) return CHAIN_ERR_ARG;
  if (need > CHAIN_NOALLOC_SCRATCH_BYTES) return CHAIN_ERR_SCRATCH_LIMIT;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return CHAIN_ERR_DEVICE;
  void *scratch = nullptr;
  {
    // Set-up on the first call for this device (the device is current).
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr)
        return record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  // Same checks and kernels as chain_bwd.  Every call rewrites what it
  // later reads (D for every query row of the attention backward; H and dT
  // of every row of the MLP backward), so what an earlier call left in the
  // array is never read.
  return chain_bwd(dO, A, B, C, O, LSE, f, mask, scale, dA, dB, dC, scratch,
                   CHAIN_NOALLOC_SCRATCH_BYTES, stream);
}
