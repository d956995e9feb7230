// device_common.cuh -- small device helpers shared by the kernels of libdsa.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

// Programmatic dependent launch: kernels of this library are launched so that
// the next kernel in the stream may start while this one finishes.  A kernel
// lets its dependents start with launch_dependents() and, before it reads any
// global memory another kernel may have written, waits for the previous grid
// with grid_dependency_wait() (a no-op when launched without the attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier over every thread of every CTA of the thread-block cluster, with
// release / acquire at cluster scope: global writes before it are visible to
// the cluster's threads after it.  A kernel that takes it passes it exactly
// once in every thread, after all its own waits, so it cannot block past them.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void flag_status(int* status, int bit) {
  if (status) atomicOr(status, bit);
}

// Paged layout: physical row of logical position p of sequence b, or -1 when
// the page id is outside [0, nb) ("Day-0 Adaptation of Trillion-Parameter MoE
// Models on Domestic GPUs", section 3 (2): pages contiguous inside, an index
// table jumping between pages).
__device__ __forceinline__ long long phys_row(const int32_t* bt, int maxb, int bs, int nb, int b,
                                              long long p) {
  long long slot = p / bs;
  if (slot >= maxb) return -1;
  int page = __ldg(&bt[(long long)b * maxb + slot]);
  if (page < 0 || page >= nb) return -1;
  return (long long)page * bs + (p - slot * bs);
}

// Order-preserving map of an fp32 score onto uint32 (larger score -> larger
// key).  -0.0 is canonicalised to +0.0 so that the two tie; NaN maps to 0,
// below every other value.
__device__ __forceinline__ uint32_t score_key(float x) {
  if (x != x) return 0u;
  if (x == 0.0f) x = 0.0f;
  uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Two FP8 E4M3 codes (low byte first) -> two floats, via the cuda_fp8.h
// conversion intrinsic.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t v) {
  return __uint_as_float(((uint32_t)v) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace dsa
