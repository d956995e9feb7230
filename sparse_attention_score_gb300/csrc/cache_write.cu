// cache_write.cu -- store new K/V rows and indexer-key rows into the paged
// caches through the block table.
//
// "Day-0 Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI
// Accelerators", section 4: the KV cache is written in the block layout, and
// the layout written at prefill must match exactly the addresses the decode
// gather reads.  Both sides use phys_row() of device_common.cuh.
//
// One warp per new row: 16-byte copies, lanes over the row's granules
// (1152 bytes = 72 granules for the latent rows, 128 bytes for an FP8 indexer
// key), grid-stride over the rows.  Memory-bound: 2 x the row bytes; the
// grid is one warp per row, capped at 16 blocks of 8 warps per SM.
#include <cuda_runtime.h>

#include <string>

#include "device_common.cuh"
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kWarps = 8;

struct CacheWriteParams {
  LayoutDev lay;
  const int32_t* seq;
  const int32_t* pos;
  int N;
  const uint4* kv_new;  // [N][kv_g] granules
  uint4* kv_pool;
  int kv_g;             // granules per row
  long long kv_stride_g;
  const uint4* kidx_new;
  uint4* kidx_pool;
  int kidx_g;
  int* status;
  int seq_const;  // seq NULL with pos given: every row in this sequence
};

// Granules a lane holds in registers (rows up to 32 * kHeld granules, i.e.
// 2 KB, are loaded in one go; longer rows fall back to a loop).
constexpr int kHeld = 4;

// Every load of a row is issued before its destination is known: the source
// granules depend only on the row number, so they travel while the
// sequence / position / block-table chain resolves.
__global__ void __launch_bounds__(kWarps * 32, 5) k_cache_write(CacheWriteParams p) {
  grid_dependency_wait();
  launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const long long nw = (long long)gridDim.x * kWarps;
  for (long long i = gw; i < p.N; i += nw) {
    // append form (seq / pos NULL): row i is the newest position of sequence i
    const int b = p.seq ? __ldg(&p.seq[i]) : (p.pos ? p.seq_const : (int)i);
    long long ps = -1;
    if (p.pos)
      ps = __ldg(&p.pos[i]);
    else if (b >= 0 && b < p.lay.batch)
      ps = (long long)__ldg(&p.lay.seq_lens[b]) - 1;
    uint4 v[kHeld];
    uint4 vi = make_uint4(0, 0, 0, 0);
    const uint4* src = p.kv_new ? p.kv_new + i * p.kv_g : nullptr;
#pragma unroll
    for (int j = 0; j < kHeld; ++j) {
      const int g = lane + 32 * j;
      v[j] = (src && g < p.kv_g) ? __ldg(&src[g]) : make_uint4(0, 0, 0, 0);
    }
    const uint4* srci = p.kidx_new ? p.kidx_new + i * p.kidx_g : nullptr;
    if (srci && lane < p.kidx_g) vi = __ldg(&srci[lane]);
    long long row = -1;
    if (b >= 0 && b < p.lay.batch && ps >= 0) row = phys_row(p.lay.bt, p.lay.maxb, p.lay.bs, p.lay.nb, b, ps);
    if (row < 0) {
      if (lane == 0) flag_status(p.status, DSA_STATUS_BAD_BLOCK);
      continue;
    }
    if (src) {
      uint4* dst = p.kv_pool + row * p.kv_stride_g;
#pragma unroll
      for (int j = 0; j < kHeld; ++j) {
        const int g = lane + 32 * j;
        if (g < p.kv_g) dst[g] = v[j];
      }
      for (int g = lane + 32 * kHeld; g < p.kv_g; g += 32) dst[g] = __ldg(&src[g]);
    }
    if (srci) {
      uint4* dst = p.kidx_pool + row * p.kidx_g;
      if (lane < p.kidx_g) dst[lane] = vi;
      for (int g = lane + 32; g < p.kidx_g; g += 32) dst[g] = __ldg(&srci[g]);
    }
  }
}

bool aligned16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

}  // namespace

int cache_write(const LayoutDev& lay, const int32_t* seq, const int32_t* pos, int N,
                const void* kv_new, int row_elems, void* kv_pool, long long kv_row_stride,
                const void* kidx_new, int D_i, int kidx_dtype, void* kidx_pool, int* status,
                cudaStream_t s, int seq_const) {
  if (N < 0) return set_error(DSA_ERR_INVALID, "cache_write: N < 0");
  if (N == 0) return DSA_OK;
  if ((seq == nullptr) != (pos == nullptr) && !(seq == nullptr && seq_const >= 0))
    return set_error(DSA_ERR_INVALID, "cache_write: give both seq and pos, or neither (append)");
  if (!seq && !pos && N > lay.batch)
    return set_error(DSA_ERR_INVALID, "cache_write: append form needs N <= batch");
  if (!kv_new && !kidx_new) return set_error(DSA_ERR_INVALID, "cache_write: nothing to write");
  CacheWriteParams p{};
  p.lay = lay;
  p.seq = seq;
  p.pos = pos;
  p.N = N;
  p.status = status;
  p.seq_const = seq_const;
  if (kv_new) {
    if (!kv_pool) return set_error(DSA_ERR_INVALID, "cache_write: kv_pool is NULL");
    if (row_elems < 8 || row_elems % 8 || kv_row_stride < row_elems || kv_row_stride % 8)
      return set_error(DSA_ERR_INVALID,
                       "cache_write: row_elems and kv_row_stride must be multiples of 8, "
                       "stride >= row_elems");
    if (!aligned16(kv_new) || !aligned16(kv_pool))
      return set_error(DSA_ERR_INVALID, "cache_write: kv_new / kv_pool must be 16-byte aligned");
    p.kv_new = reinterpret_cast<const uint4*>(kv_new);
    p.kv_pool = reinterpret_cast<uint4*>(kv_pool);
    p.kv_g = row_elems / 8;
    p.kv_stride_g = kv_row_stride / 8;
  }
  if (kidx_new) {
    if (!kidx_pool) return set_error(DSA_ERR_INVALID, "cache_write: kidx_pool is NULL");
    if (kidx_dtype != DSA_BF16 && kidx_dtype != DSA_FP8_E4M3)
      return set_error(DSA_ERR_INVALID, "cache_write: kidx_dtype must be DSA_BF16 or DSA_FP8_E4M3");
    const long long bytes = (long long)D_i * (kidx_dtype == DSA_BF16 ? 2 : 1);
    if (D_i < 1 || bytes % 16)
      return set_error(DSA_ERR_INVALID, "cache_write: an indexer-key row must be a multiple of 16 bytes");
    if (!aligned16(kidx_new) || !aligned16(kidx_pool))
      return set_error(DSA_ERR_INVALID, "cache_write: kidx_new / kidx_pool must be 16-byte aligned");
    p.kidx_new = reinterpret_cast<const uint4*>(kidx_new);
    p.kidx_pool = reinterpret_cast<uint4*>(kidx_pool);
    p.kidx_g = (int)(bytes / 16);
  }
  long long grid = (N + kWarps - 1) / kWarps;
  const long long cap = 16LL * sm_count();
  if (grid > cap) grid = cap;
  const cudaError_t e = launch_pdl(k_cache_write, dim3((unsigned)grid), dim3(kWarps * 32), 0, s, p);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("cache_write");
}

}  // namespace dsa
