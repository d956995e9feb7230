// topk_noalloc.cu -- dsa_topk_noalloc: the top-K selection of dsa_topk for
// callers that cannot allocate device memory.
//
// Who needs it: code handed a stream but no allocator (a plugin inside a host
// framework that owns all device memory), real-time threads that must not
// take the allocator's locks or risk its latency, and deployments whose
// device memory is carved up ahead of time so that no call may grow it.  For
// them this entry point keeps its scratch (the status word and, for rows
// longer than one block, the per-block winners) in one fixed array that is
// part of the library image: nothing is allocated or freed per call.
//
// The array is DSA_TOPK_NOALLOC_SCRATCH_BYTES bytes on every GPU that loads
// the library and stays there until the process exits.  Host code reaches it
// only through the device address that cudaGetSymbolAddress returns, looked
// up once per device with that device current (the name of the array in host
// code is a host-side stand-in, never a device address).
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "dsa.h"
#include "dsa_internal.cuh"

namespace dsa {

static __device__ __align__(256) unsigned char g_topk_scratch[DSA_TOPK_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; the first call
// on a device looks it up and caches it for the life of the process (a
// cudaDeviceReset of that device would leave the cached address stale, which
// the header tells callers not to do between calls).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return set_error(DSA_ERR_CUDA, std::string("topk_noalloc: cudaGetDevice: ") +
                                       cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(DSA_ERR_UNSUPPORTED, "topk_noalloc: device index out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess || !p)
      return set_error(DSA_ERR_CUDA, std::string("topk_noalloc: cudaGetSymbolAddress: ") +
                                         cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_topk_noalloc_scratch_bytes(void) { return sizeof(g_topk_scratch); }

extern "C" int dsa_topk_noalloc(const float* scores, int64_t ld, const int32_t* n_eligible,
                                int Nq, int K, int32_t* idx, dsa_stream_t stream) {
  if (Nq < 0 || ld < 1 || K < 1 || K > 65536)
    return set_error(DSA_ERR_INVALID, "topk_noalloc: need Nq >= 0, ld >= 1, 1 <= K <= 65536");
  if (!scores || !n_eligible || !idx)
    return set_error(DSA_ERR_INVALID, "topk_noalloc: NULL pointer");
  const size_t need = topk_ws(Nq, (long long)ld, K);
  if (need > (size_t)DSA_TOPK_NOALLOC_SCRATCH_BYTES)
    return set_error(DSA_ERR_WORKSPACE,
                     "topk_noalloc: this problem needs " + std::to_string(need) +
                         " bytes of scratch, more than the fixed " +
                         std::to_string((size_t)DSA_TOPK_NOALLOC_SCRATCH_BYTES) +
                         "; call dsa_topk with a workspace of your own instead");
  void* ws = nullptr;
  int rc = scratch_address(&ws);
  if (rc) return rc;
  if (Nq == 0) return DSA_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents.  Only the status word must
  // start at zero; the block winners are written before they are read.
  cudaError_t e = cudaMemsetAsync(ws, 0, kWsHeader, s);
  if (e != cudaSuccess)
    return set_error(DSA_ERR_CUDA, std::string("topk_noalloc: ") + cudaGetErrorString(e));
  TopkParams p{};
  p.scores = scores;
  p.ld = (long long)ld;
  p.n_elig = n_eligible;
  p.Nq = Nq;
  p.K = K;
  p.idx = idx;
  p.status = reinterpret_cast<int*>(ws);
  return launch_topk(p, ws, (size_t)DSA_TOPK_NOALLOC_SCRATCH_BYTES, s);
}
