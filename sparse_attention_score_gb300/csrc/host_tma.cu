// host_tma.cu -- TMA tensor-map encoding on the host.  The driver entry point
// is fetched through the runtime, so libdsa.so does not link libcuda itself.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <utility>

#include "dsa_internal.cuh"

namespace dsa {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_tmap_2d(CUtensorMap* map, const void* base, bool one_byte, uint64_t inner_elems,
                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return set_error(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {inner_elems, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, one_byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed with " + std::to_string((int)r));
  return DSA_OK;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  static std::mutex m;
  static std::map<int, int> counts;
  std::lock_guard<std::mutex> lock(m);
  auto it = counts.find(dev);
  if (it != counts.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  counts[dev] = n;
  return n;
}

int max_active_clusters(const void* kernel, int threads, size_t smem, int cs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::mutex m;
  static std::map<std::tuple<const void*, int, int, size_t, int>, int> known;
  std::lock_guard<std::mutex> lock(m);
  const auto key = std::make_tuple(kernel, dev, cs, smem, threads);
  auto it = known.find(key);
  if (it != known.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();  // clear the error state: that launch takes the plain path
    return 0;
  }
  known[key] = n;
  return n;
}

int ensure_dynamic_smem(const void* kernel, int bytes, const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return set_error(DSA_ERR_CUDA, std::string(what) + ": cudaGetDevice: " + cudaGetErrorString(e));
  // function attributes belong to a device's context: one record per
  // (kernel, device), the largest size set so far
  static std::mutex m;
  static std::map<std::pair<const void*, int>, int> done;
  std::lock_guard<std::mutex> lock(m);
  const auto key = std::make_pair(kernel, dev);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return DSA_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess)
    return set_error(DSA_ERR_CUDA, std::string(what) + ": cudaFuncSetAttribute(" +
                                       std::to_string(bytes) + " bytes): " + cudaGetErrorString(e));
  done[key] = bytes;
  return DSA_OK;
}

}  // namespace dsa
