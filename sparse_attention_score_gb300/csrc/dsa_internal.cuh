// dsa_internal.cuh -- parameter blocks and launcher declarations shared by the
// translation units of libdsa.so (never installed, never seen by callers).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>

#include "dsa.h"

namespace dsa {

// Bytes reserved at the head of every workspace: the status word and small
// self-resetting counters.
constexpr size_t kWsHeader = 256;

struct LayoutDev {
  int bs, nb, maxb, batch, max_len;
  const int32_t* bt;
  const int32_t* seq_lens;
};

struct IndexParams {
  LayoutDev lay;
  const void* q_idx;
  const float* w;
  const void* kidx;
  int dtype, H, D;
  const int32_t* q_seq;
  const int32_t* q_pos;
  int seq_const;  // >= 0: every query belongs to this sequence (q_seq ignored)
  int Nq;
  float* scores;
  long long ld;
  int* status;
  // optional per-tile mask over positions [128 t, 128 t + 128) of query r,
  // skip[r * skip_stride + t]: 0 score the tile, kSkipInf leave it out
  // (scores -inf, keys not read), kSkipKeep leave it out and its scores as
  // they are
  const uint8_t* skip;
  long long skip_stride;
};

constexpr uint8_t kSkipInf = 1, kSkipKeep = 2;

struct TopkParams {
  const float* scores;
  long long ld;
  const int32_t* n_elig;
  int Nq, K;
  int32_t* idx;
  int* status;
};

struct AttnParams {
  LayoutDev lay;
  const __nv_bfloat16* q;
  const __nv_bfloat16* kp;
  long long ks;
  const __nv_bfloat16* vp;
  long long vs;
  int Hq, Dqk, Dv;
  const int32_t* q_seq;  // NULL: query r is sequence r (decode) / sequence 0 (prefill)
  int seq_const;         // q_seq NULL: every query in this sequence (>= 0), or query r in sequence r (-1)
  const int32_t* q_pos;  // NULL or [Nq]: causal bound of each query (prefill)
  int Nq;
  const int32_t* idx;
  int K;
  float scale_log2;  // sm_scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  int* status;
  float* part_o;   // [Nq][S][Hq][Dv] unnormalised partial outputs
  float* part_ml;  // [Nq][S][Hq][2] (running max in log2 units, sum)
  int S;           // splits of the K selected rows
};

// Launch with the programmatic-stream-serialization attribute (the kernel must
// call grid_dependency_wait() before reading inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same launch with its CTAs grouped in clusters of `cs` along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               int cs, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cs;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// selftest.cu
int bounded_wait_selftest(int expire, unsigned long long limit_ns, int* status, cudaStream_t s);

// cache_write.cu
int cache_write(const LayoutDev& lay, const int32_t* seq, const int32_t* pos, int N,
                const void* kv_new, int row_elems, void* kv_pool, long long kv_row_stride,
                const void* kidx_new, int D_i, int kidx_dtype, void* kidx_pool, int* status,
                cudaStream_t s, int seq_const = -1);

// host-side bookkeeping (dsa_api.cu)
void count_launch(int n = 1);
int set_error(int code, const std::string& msg);
int check_launch(const char* what);

// host_tma.cu: 2D TMA map with 128-byte swizzle over rows of `inner_elems`
// elements (1-byte elements if one_byte, else bf16), rows `row_stride_bytes`
// apart; box of box_inner x box_rows.
int make_tmap_2d(CUtensorMap* map, const void* base, bool one_byte, uint64_t inner_elems,
                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);
int sm_count();  // of the current device
// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device (once per kernel and device, thread-safe); DSA_ERR_CUDA on failure.
int ensure_dynamic_smem(const void* kernel, int bytes, const char* what);
// Largest number of clusters of `cs` CTAs (1-D, `threads` each, `smem` bytes of
// dynamic shared memory) of `kernel` resident at once on the current device;
// 0 if the query fails.  Answers are recorded per (kernel, device, shape).
int max_active_clusters(const void* kernel, int threads, size_t smem, int cs);

// launchers: return DSA_OK / DSA_ERR_*
int launch_index_score(const IndexParams& p, cudaStream_t s);
// tensor-core indexer (FP8 E4M3, H_i = 64, D_i = 128, block size 64)
bool index_tc_eligible(const IndexParams& p);
int launch_index_tc(const IndexParams& p, cudaStream_t s);
// tensor-core prefill indexer (queries of one sequence sharing key tiles)
bool index_prefill_tc_eligible(const IndexParams& p);
int launch_index_prefill_tc(const IndexParams& p, cudaStream_t s);
bool index_score_supported(int dtype, int H, int D);
size_t index_score_ws(int Nq, int H, int D, long long ld);

int launch_topk(const TopkParams& p, void* ws, size_t ws_bytes, cudaStream_t s);

// index_bounds.cu: per-page bounds of the indexer keys, and the decode
// indexer that leaves out tiles which cannot reach the top-K.  The bounded
// call counts skipped and bounded tiles in two uint64 of its workspace header.
constexpr size_t kBoundedCounters = 64;
int index_bounds_update(const LayoutDev& lay, const int32_t* seq, const int32_t* pos, int N,
                        const void* kidx, int D, int dtype, void* kbound, int* status,
                        cudaStream_t s);
size_t index_bounded_ws(int B, long long ld, int K);
int index_score_bounded(IndexParams p, const void* kbound, int K, void* ws, cudaStream_t s);
// shared-memory block top-K (topk_smem.cu)
bool topk_smem_eligible(long long ld, int K);
size_t topk_smem_ws(int Nq, long long ld, int K);
int launch_topk_smem(const TopkParams& p, void* ws, cudaStream_t s);
size_t topk_ws(int Nq, long long ld, int K);

int launch_attn(AttnParams p, bool decode, void* ws, size_t ws_bytes, cudaStream_t s);
// tensor-core attention (64 heads, latent 576/512 rows shared by K and V)
bool attn_tc_eligible(const AttnParams& p);
size_t attn_tc_ws(int Nq);
int launch_attn_tc(const AttnParams& p, void* ws, cudaStream_t s);
bool attn_supported(int Hq, int Dqk, int Dv);
size_t attn_ws(int Nq, int Hq, int Dqk, int Dv, int K, bool decode);

}  // namespace dsa
