// dsa_api.cu -- the C ABI of libdsa.so: argument validation, workspace
// checks, dispatch to the kernels, error reporting.  Declarations and the
// contract of every entry point are in include/dsa.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <string>

#include "dsa.h"
#include "dsa_internal.cuh"

namespace dsa {

static std::atomic<uint64_t> g_launches{0};
static thread_local std::string g_last_error;

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int set_error(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(DSA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return DSA_OK;
}

static int check_layout(const dsa_paged_layout* L, LayoutDev* out) {
  if (!L) return set_error(DSA_ERR_INVALID, "layout is NULL");
  if (!L->block_table || !L->seq_lens)
    return set_error(DSA_ERR_INVALID, "layout.block_table / seq_lens is NULL");
  if (L->block_size < 1 || L->block_size > 1024)
    return set_error(DSA_ERR_INVALID, "layout.block_size must be in 1..1024");
  if (L->num_blocks < 1 || L->max_blocks_per_seq < 1 || L->batch < 1)
    return set_error(DSA_ERR_INVALID, "layout.num_blocks/max_blocks_per_seq/batch must be >= 1");
  if (L->max_seq_len < 0 ||
      (long long)L->max_seq_len > (long long)L->max_blocks_per_seq * L->block_size)
    return set_error(DSA_ERR_INVALID,
                     "layout.max_seq_len must be in 0..max_blocks_per_seq*block_size");
  out->bs = L->block_size;
  out->nb = L->num_blocks;
  out->maxb = L->max_blocks_per_seq;
  out->batch = L->batch;
  out->max_len = L->max_seq_len;
  out->bt = L->block_table;
  out->seq_lens = L->seq_lens;
  return DSA_OK;
}

static int check_ws(void* ws, size_t have, size_t need) {
  if (!ws) return set_error(DSA_ERR_WORKSPACE, "workspace is NULL");
  if (((uintptr_t)ws) & 255u) return set_error(DSA_ERR_WORKSPACE, "workspace not 256-byte aligned");
  if (have < need)
    return set_error(DSA_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) +
                                            " bytes, got " + std::to_string(have));
  return DSA_OK;
}

static bool aligned16(const void* p) { return (((uintptr_t)p) & 15u) == 0; }

}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_version(void) { return 100; }

uint64_t dsa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* dsa_last_error_string(void) { return g_last_error.c_str(); }

int dsa_get_status(void* ws, dsa_stream_t stream, int32_t* status, int clear) {
  if (!ws || !status) return set_error(DSA_ERR_INVALID, "dsa_get_status: NULL argument");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws, 0, sizeof v, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess)
    return set_error(DSA_ERR_CUDA, std::string("dsa_get_status: ") + cudaGetErrorString(e));
  *status = v;
  return DSA_OK;
}

size_t dsa_index_score_workspace_size(int Nq, int H_i, int D_i, int64_t ld) {
  return index_score_ws(Nq, H_i, D_i, (long long)ld);
}

static int index_common(const dsa_paged_layout* layout, const void* q_idx, const float* w,
                        const void* kidx_pool, int dtype, int H_i, int D_i,
                        const int32_t* q_seq, const int32_t* q_pos, int seq_const, int Nq,
                        float* scores, int64_t ld, void* ws, size_t ws_bytes,
                        dsa_stream_t stream, int* status = nullptr) {
  IndexParams p{};
  int rc = check_layout(layout, &p.lay);
  if (rc) return rc;
  if (Nq < 0 || ld < 1) return set_error(DSA_ERR_INVALID, "index_score: Nq < 0 or ld < 1");
  if (!q_idx || !w || !kidx_pool || !scores)
    return set_error(DSA_ERR_INVALID, "index_score: NULL tensor pointer");
  if (seq_const >= layout->batch)
    return set_error(DSA_ERR_INVALID, "index_score_prefill: seq out of range");
  if (!index_score_supported(dtype, H_i, D_i))
    return set_error(DSA_ERR_UNSUPPORTED,
                     "index_score: supported dtype BF16/FP8_E4M3, H_i 1..128, D_i 32/64/128");
  if (!aligned16(q_idx) || !aligned16(kidx_pool))
    return set_error(DSA_ERR_INVALID, "index_score: q_idx / kidx_pool must be 16-byte aligned");
  rc = check_ws(ws, ws_bytes, index_score_ws(Nq, H_i, D_i, (long long)ld));
  if (rc) return rc;
  p.q_idx = q_idx;
  p.w = w;
  p.kidx = kidx_pool;
  p.dtype = dtype;
  p.H = H_i;
  p.D = D_i;
  p.q_seq = q_seq;
  p.q_pos = q_pos;
  p.seq_const = seq_const;
  p.Nq = Nq;
  p.scores = scores;
  p.ld = (long long)ld;
  p.status = status ? status : reinterpret_cast<int*>(ws);
  return launch_index_score(p, reinterpret_cast<cudaStream_t>(stream));
}

int dsa_index_score(const dsa_paged_layout* layout, const void* q_idx, const float* w,
                    const void* kidx_pool, int dtype, int H_i, int D_i, const int32_t* q_seq,
                    const int32_t* q_pos, int Nq, float* scores, int64_t ld, void* ws,
                    size_t ws_bytes, dsa_stream_t stream) {
  return index_common(layout, q_idx, w, kidx_pool, dtype, H_i, D_i, q_seq, q_pos, -1, Nq, scores,
                      ld, ws, ws_bytes, stream);
}

size_t dsa_index_score_prefill_workspace_size(int Nq, int H_i, int D_i, int64_t ld) {
  return index_score_ws(Nq, H_i, D_i, (long long)ld);
}

int dsa_index_score_prefill(const dsa_paged_layout* layout, int seq, const void* q_idx,
                            const float* w, const void* kidx_pool, int dtype, int H_i, int D_i,
                            const int32_t* q_pos, int Nq, float* scores, int64_t ld, void* ws,
                            size_t ws_bytes, dsa_stream_t stream) {
  if (seq < 0) return set_error(DSA_ERR_INVALID, "index_score_prefill: seq < 0");
  return index_common(layout, q_idx, w, kidx_pool, dtype, H_i, D_i, nullptr, q_pos, seq, Nq,
                      scores, ld, ws, ws_bytes, stream);
}

size_t dsa_topk_workspace_size(int Nq, int64_t ld, int K) {
  return topk_ws(Nq, (long long)ld, K);
}

static int topk_common(const float* scores, int64_t ld, const int32_t* n_eligible, int Nq, int K,
                       int32_t* idx, void* ws, size_t ws_bytes, dsa_stream_t stream,
                       int* status = nullptr) {
  if (Nq < 0 || ld < 1 || K < 1 || K > 65536)
    return set_error(DSA_ERR_INVALID, "topk: need Nq >= 0, ld >= 1, 1 <= K <= 65536");
  if (!scores || !n_eligible || !idx) return set_error(DSA_ERR_INVALID, "topk: NULL pointer");
  int rc = check_ws(ws, ws_bytes, topk_ws(Nq, (long long)ld, K));
  if (rc) return rc;
  TopkParams p{};
  p.scores = scores;
  p.ld = (long long)ld;
  p.n_elig = n_eligible;
  p.Nq = Nq;
  p.K = K;
  p.idx = idx;
  p.status = status ? status : reinterpret_cast<int*>(ws);
  return launch_topk(p, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int dsa_topk(const float* scores, int64_t ld, const int32_t* n_eligible, int Nq, int K,
             int32_t* idx, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  return topk_common(scores, ld, n_eligible, Nq, K, idx, ws, ws_bytes, stream);
}

// ------------------------------------------------------------- bounds --
size_t dsa_index_bounds_update_workspace_size(void) { return kWsHeader; }

int dsa_index_bounds_update(const dsa_paged_layout* layout, const int32_t* seq,
                            const int32_t* pos, int N, const void* kidx_pool, int D_i,
                            int idx_dtype, void* kbound_pool, void* ws, size_t ws_bytes,
                            dsa_stream_t stream) {
  LayoutDev lay;
  int rc = check_layout(layout, &lay);
  if (rc) return rc;
  if (!kidx_pool || !kbound_pool)
    return set_error(DSA_ERR_INVALID, "index_bounds_update: NULL pool");
  if ((seq == nullptr) != (pos == nullptr) || N < 0)
    return set_error(DSA_ERR_INVALID, "index_bounds_update: seq and pos both or neither, N >= 0");
  if ((idx_dtype != DSA_BF16 && idx_dtype != DSA_FP8_E4M3) || (D_i != 32 && D_i != 64 && D_i != 128))
    return set_error(DSA_ERR_UNSUPPORTED,
                     "index_bounds_update: dtype BF16/FP8_E4M3, D_i 32/64/128");
  rc = check_ws(ws, ws_bytes, kWsHeader);
  if (rc) return rc;
  return index_bounds_update(lay, seq, pos, seq ? N : 0, kidx_pool, D_i, idx_dtype, kbound_pool,
                             reinterpret_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream));
}

size_t dsa_index_score_bounded_workspace_size(int B, int H_i, int D_i, int64_t ld, int K) {
  (void)H_i;
  (void)D_i;
  if (B < 1 || ld < 1 || K < 1) return kWsHeader;
  return index_bounded_ws(B, (long long)ld, K);
}

int dsa_index_score_bounded(const dsa_paged_layout* layout, const void* q_idx, const float* w,
                            const void* kidx_pool, int idx_dtype, int H_i, int D_i,
                            const void* kbound_pool, int K, float* scores, int64_t ld, void* ws,
                            size_t ws_bytes, dsa_stream_t stream) {
  IndexParams p{};
  int rc = check_layout(layout, &p.lay);
  if (rc) return rc;
  if (ld < 1 || K < 1 || K > 65536)
    return set_error(DSA_ERR_INVALID, "index_score_bounded: need ld >= 1, 1 <= K <= 65536");
  if (!q_idx || !w || !kidx_pool || !kbound_pool || !scores)
    return set_error(DSA_ERR_INVALID, "index_score_bounded: NULL tensor pointer");
  if (!index_score_supported(idx_dtype, H_i, D_i))
    return set_error(DSA_ERR_UNSUPPORTED,
                     "index_score_bounded: supported dtype BF16/FP8_E4M3, H_i 1..128, D_i 32/64/128");
  if (!aligned16(q_idx) || !aligned16(kidx_pool))
    return set_error(DSA_ERR_INVALID,
                     "index_score_bounded: q_idx / kidx_pool must be 16-byte aligned");
  const int B = layout->batch;
  if (B > 65535)  // the candidate gather puts the batch on the grid's y dimension
    return set_error(DSA_ERR_UNSUPPORTED, "index_score_bounded: batch > 65535");
  rc = check_ws(ws, ws_bytes, index_bounded_ws(B, (long long)ld, K));
  if (rc) return rc;
  p.q_idx = q_idx;
  p.w = w;
  p.kidx = kidx_pool;
  p.dtype = idx_dtype;
  p.H = H_i;
  p.D = D_i;
  p.seq_const = -1;
  p.Nq = B;
  p.scores = scores;
  p.ld = (long long)ld;
  p.status = reinterpret_cast<int*>(ws);
  return index_score_bounded(p, kbound_pool, K, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dsa_index_bounded_stats(void* ws, dsa_stream_t stream, uint64_t* tiles_skipped,
                            uint64_t* tiles_bounded) {
  if (!ws || !tiles_skipped || !tiles_bounded)
    return set_error(DSA_ERR_INVALID, "index_bounded_stats: NULL pointer");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned long long h[2] = {0ull, 0ull};
  cudaError_t e = cudaMemcpyAsync(h, reinterpret_cast<char*>(ws) + kBoundedCounters, sizeof(h),
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  *tiles_skipped = h[0];
  *tiles_bounded = h[1];
  return DSA_OK;
}

size_t dsa_cache_write_workspace_size(void) { return kWsHeader; }

int dsa_cache_write(const dsa_paged_layout* layout, const int32_t* seq, const int32_t* pos, int N,
                    const void* kv_new, int row_elems, void* kv_pool, int64_t kv_row_stride,
                    const void* kidx_new, int D_i, int kidx_dtype, void* kidx_pool, void* ws,
                    size_t ws_bytes, dsa_stream_t stream) {
  LayoutDev lay;
  int rc = check_layout(layout, &lay);
  if (rc) return rc;
  rc = check_ws(ws, ws_bytes, kWsHeader);
  if (rc) return rc;
  return cache_write(lay, seq, pos, N, kv_new, row_elems, kv_pool, (long long)kv_row_stride,
                     kidx_new, D_i, kidx_dtype, kidx_pool, reinterpret_cast<int*>(ws),
                     reinterpret_cast<cudaStream_t>(stream));
}

static int attn_common(const dsa_paged_layout* layout, const void* q, const void* k_pool,
                       int64_t k_row_stride, const void* v_pool, int64_t v_row_stride, int Hq,
                       int Dqk, int Dv, const int32_t* q_seq, const int32_t* q_pos, int Nq,
                       const int32_t* idx, int K,
                       float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes,
                       dsa_stream_t stream, bool decode, int* status = nullptr,
                       int seq_const = -2) {
  AttnParams p{};
  int rc = check_layout(layout, &p.lay);
  if (rc) return rc;
  if (Nq < 0 || K < 1) return set_error(DSA_ERR_INVALID, "sparse_attn: Nq < 0 or K < 1");
  if (Nq > 65535) return set_error(DSA_ERR_UNSUPPORTED, "sparse_attn: Nq > 65535");
  if (!q || !k_pool || !v_pool || !idx || !out)
    return set_error(DSA_ERR_INVALID, "sparse_attn: NULL tensor pointer");
  if (k_row_stride < Dqk || v_row_stride < Dv || (k_row_stride % 8) || (v_row_stride % 8))
    return set_error(DSA_ERR_INVALID,
                     "sparse_attn: row strides must cover Dqk/Dv and be multiples of 8");
  if (!attn_supported(Hq, Dqk, Dv))
    return set_error(DSA_ERR_UNSUPPORTED,
                     "sparse_attn: supported Hq 1..64, Dqk/Dv multiples of 8, Dv <= 512");
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return set_error(DSA_ERR_INVALID, "sparse_attn: q / k_pool / v_pool must be 16-byte aligned");
  if (!(sm_scale > 0.0f) || sm_scale != sm_scale)
    return set_error(DSA_ERR_INVALID, "sparse_attn: sm_scale must be a positive number");
  rc = check_ws(ws, ws_bytes, attn_ws(Nq, Hq, Dqk, Dv, K, decode));
  if (rc) return rc;
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.kp = reinterpret_cast<const __nv_bfloat16*>(k_pool);
  p.ks = (long long)k_row_stride;
  p.vp = reinterpret_cast<const __nv_bfloat16*>(v_pool);
  p.vs = (long long)v_row_stride;
  p.Hq = Hq;
  p.Dqk = Dqk;
  p.Dv = Dv;
  p.q_seq = q_seq;
  p.q_pos = q_pos;
  p.seq_const = seq_const >= -1 ? seq_const : (decode ? -1 : 0);
  p.Nq = Nq;
  p.idx = idx;
  p.K = K;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = status ? status : reinterpret_cast<int*>(ws);
  return launch_attn(p, decode, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t dsa_sparse_attn_decode_workspace_size(int B, int Hq, int Dqk, int Dv, int K) {
  return attn_ws(B, Hq, Dqk, Dv, K, true);
}

int dsa_sparse_attn_decode(const dsa_paged_layout* layout, const void* q, const void* k_pool,
                           int64_t k_row_stride, const void* v_pool, int64_t v_row_stride,
                           int Hq, int Dqk, int Dv, const int32_t* idx, int K, float sm_scale,
                           void* out, float* lse, void* ws, size_t ws_bytes,
                           dsa_stream_t stream) {
  int B = layout ? layout->batch : 0;
  return attn_common(layout, q, k_pool, k_row_stride, v_pool, v_row_stride, Hq, Dqk, Dv, nullptr,
                     nullptr, B, idx, K, sm_scale, out, lse, ws, ws_bytes, stream, true);
}

size_t dsa_sparse_attn_prefill_workspace_size(int Nq, int Hq, int Dqk, int Dv, int K) {
  return attn_ws(Nq, Hq, Dqk, Dv, K, false);
}

int dsa_sparse_attn_prefill(const dsa_paged_layout* layout, const void* q, const void* k_pool,
                            int64_t k_row_stride, const void* v_pool, int64_t v_row_stride,
                            int Hq, int Dqk, int Dv, const int32_t* q_seq,
                            const int32_t* q_pos, int Nq, const int32_t* idx, int K,
                            float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes,
                            dsa_stream_t stream) {
  return attn_common(layout, q, k_pool, k_row_stride, v_pool, v_row_stride, Hq, Dqk, Dv, q_seq,
                     q_pos, Nq, idx, K, sm_scale, out, lse, ws, ws_bytes, stream, false);
}

int dsa_selftest_bounded_wait(int expire, uint64_t limit_ns, void* ws, size_t ws_bytes,
                              dsa_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000ull)
    return set_error(DSA_ERR_INVALID, "selftest_bounded_wait: limit_ns must be in [1 us, 1 s]");
  int rc = check_ws(ws, ws_bytes, kWsHeader);
  if (rc) return rc;
  return bounded_wait_selftest(expire ? 1 : 0, (unsigned long long)limit_ns,
                               reinterpret_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- steps --
// A step workspace: the step's status header, then one region per stage
// (each region 256-byte aligned and laid out as that stage's own workspace).
// Every stage ORs its status bits into the step's word at offset 0.
static size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

struct StepLayout {
  size_t off_index, off_topk, off_attn, total;
};

static StepLayout step_layout(int Nq, int H_i, int D_i, int64_t ld, int Hq, int Dqk, int Dv, int K,
                              bool decode) {
  StepLayout L;
  L.off_index = kWsHeader;
  L.off_topk = L.off_index + round256(index_score_ws(Nq, H_i, D_i, (long long)ld));
  L.off_attn = L.off_topk + round256(topk_ws(Nq, (long long)ld, K));
  L.total = L.off_attn + round256(attn_ws(Nq, Hq, Dqk, Dv, K, decode));
  return L;
}

static int step_cache_write(const dsa_paged_layout* layout, int seq_const, const int32_t* pos,
                            int N, const void* k_new, void* k_pool, int64_t k_row_stride, int Dqk,
                            const void* v_new, void* v_pool, int64_t v_row_stride, int Dv,
                            const void* kidx_new, void* kidx_pool, int idx_dtype, int D_i,
                            int* status, cudaStream_t s) {
  LayoutDev lay;
  int rc = check_layout(layout, &lay);
  if (rc) return rc;
  if (k_new || kidx_new) {
    rc = cache_write(lay, nullptr, pos, N, k_new, Dqk, k_pool, (long long)k_row_stride, kidx_new,
                     D_i, idx_dtype, kidx_pool, status, s, seq_const);
    if (rc) return rc;
  }
  if (v_new)
    rc = cache_write(lay, nullptr, pos, N, v_new, Dv, v_pool, (long long)v_row_stride, nullptr, 0,
                     0, nullptr, status, s, seq_const);
  return rc;
}

size_t dsa_decode_step_workspace_size(int B, int H_i, int D_i, int64_t ld, int Hq, int Dqk,
                                      int Dv, int K) {
  return step_layout(B, H_i, D_i, ld, Hq, Dqk, Dv, K, true).total;
}

int dsa_decode_step(const dsa_paged_layout* layout, const void* k_new, void* k_pool,
                    int64_t k_row_stride, const void* v_new, void* v_pool, int64_t v_row_stride,
                    const void* kidx_new, void* kidx_pool, int idx_dtype, const void* q_idx,
                    const float* w, int H_i, int D_i, const void* q, int Hq, int Dqk, int Dv,
                    int K, float sm_scale, float* scores, int64_t ld, int32_t* idx, void* out,
                    float* lse, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  if (!layout) return set_error(DSA_ERR_INVALID, "decode_step: NULL layout");
  const int B = layout->batch;
  const StepLayout L = step_layout(B, H_i, D_i, ld, Hq, Dqk, Dv, K, true);
  int rc = check_ws(ws, ws_bytes, L.total);
  if (rc) return rc;
  char* base = reinterpret_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = step_cache_write(layout, -1, nullptr, B, k_new, k_pool, k_row_stride, Dqk, v_new, v_pool,
                        v_row_stride, Dv, kidx_new, kidx_pool, idx_dtype, D_i, status, s);
  if (rc) return rc;
  rc = index_common(layout, q_idx, w, kidx_pool, idx_dtype, H_i, D_i, nullptr, nullptr, -1, B,
                    scores, ld, base + L.off_index, L.off_topk - L.off_index, stream, status);
  if (rc) return rc;
  rc = topk_common(scores, ld, layout->seq_lens, B, K, idx, base + L.off_topk,
                   L.off_attn - L.off_topk, stream, status);
  if (rc) return rc;
  return attn_common(layout, q, k_pool, k_row_stride, v_pool, v_row_stride, Hq, Dqk, Dv, nullptr,
                     nullptr, B, idx, K, sm_scale, out, lse, base + L.off_attn,
                     L.total - L.off_attn, stream, true, status);
}

size_t dsa_prefill_step_workspace_size(int Nq, int H_i, int D_i, int64_t ld, int Hq, int Dqk,
                                       int Dv, int K) {
  return step_layout(Nq, H_i, D_i, ld, Hq, Dqk, Dv, K, false).total;
}

int dsa_prefill_step(const dsa_paged_layout* layout, int seq, const int32_t* q_pos,
                     const int32_t* n_eligible, int Nq, const void* k_new,
                     void* k_pool, int64_t k_row_stride, const void* v_new, void* v_pool,
                     int64_t v_row_stride, const void* kidx_new, void* kidx_pool, int idx_dtype,
                     const void* q_idx, const float* w, int H_i, int D_i, const void* q, int Hq,
                     int Dqk, int Dv, int K, float sm_scale, float* scores, int64_t ld,
                     int32_t* idx, void* out, float* lse, void* ws, size_t ws_bytes,
                     dsa_stream_t stream) {
  if (!layout) return set_error(DSA_ERR_INVALID, "prefill_step: NULL layout");
  if (seq < 0 || seq >= layout->batch)
    return set_error(DSA_ERR_INVALID, "prefill_step: seq out of range");
  if (!q_pos || !n_eligible)
    return set_error(DSA_ERR_INVALID, "prefill_step: q_pos and n_eligible are required");
  const StepLayout L = step_layout(Nq, H_i, D_i, ld, Hq, Dqk, Dv, K, false);
  int rc = check_ws(ws, ws_bytes, L.total);
  if (rc) return rc;
  char* base = reinterpret_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = step_cache_write(layout, seq, q_pos, Nq, k_new, k_pool, k_row_stride, Dqk, v_new, v_pool,
                        v_row_stride, Dv, kidx_new, kidx_pool, idx_dtype, D_i, status, s);
  if (rc) return rc;
  rc = index_common(layout, q_idx, w, kidx_pool, idx_dtype, H_i, D_i, nullptr, q_pos, seq, Nq,
                    scores, ld, base + L.off_index, L.off_topk - L.off_index, stream, status);
  if (rc) return rc;
  rc = topk_common(scores, ld, n_eligible, Nq, K, idx, base + L.off_topk,
                   L.off_attn - L.off_topk, stream, status);
  if (rc) return rc;
  return attn_common(layout, q, k_pool, k_row_stride, v_pool, v_row_stride, Hq, Dqk, Dv, nullptr,
                     q_pos, Nq, idx, K, sm_scale, out, lse, base + L.off_attn,
                     L.total - L.off_attn, stream, false, status, seq);
}

// ---------------------------------------------------------- chunked step --
// The prefill step without the score matrix: queries are scored and selected
// a chunk at a time; a chunk's scores go to one scratch region of the
// workspace, sized for one chunk, which the next chunk overwrites.  With the
// default chunk the scratch (<= kChunkScoreBytes) stays in L2 between the
// indexer that writes it and the top-K that reads it.
constexpr size_t kChunkScoreBytes = 48ull << 20;

static int prefill_chunk_rows(int Nq, int64_t ld, int chunk) {
  long long c = chunk > 0 ? chunk : (long long)(kChunkScoreBytes / ((size_t)(ld > 0 ? ld : 1) * 4));
  if (chunk <= 0) c = c / 16 * 16;  // whole blocks of the prefill indexer
  if (c < 16) c = 16;
  if (c > Nq) c = Nq;
  if (c < 1) c = 1;
  return (int)c;
}

struct ChunkLayout {
  size_t off_index, off_topk, off_attn, off_scores, total;
  int C;
};

static ChunkLayout chunk_layout(int Nq, int H_i, int D_i, int64_t ld, int Hq, int Dqk, int Dv,
                                int K, int chunk) {
  ChunkLayout L;
  L.C = prefill_chunk_rows(Nq, ld, chunk);
  L.off_index = kWsHeader;
  L.off_topk = L.off_index + round256(index_score_ws(L.C, H_i, D_i, (long long)ld));
  L.off_attn = L.off_topk + round256(topk_ws(L.C, (long long)ld, K));
  L.off_scores = L.off_attn + round256(attn_ws(Nq, Hq, Dqk, Dv, K, false));
  L.total = L.off_scores + round256((size_t)L.C * (size_t)ld * sizeof(float));
  return L;
}

size_t dsa_prefill_step_chunked_workspace_size(int Nq, int H_i, int D_i, int64_t ld, int Hq,
                                               int Dqk, int Dv, int K, int chunk) {
  if (Nq < 1 || ld < 1) return kWsHeader;
  return chunk_layout(Nq, H_i, D_i, ld, Hq, Dqk, Dv, K, chunk).total;
}

int dsa_prefill_step_chunked(const dsa_paged_layout* layout, int seq, const int32_t* q_pos,
                             const int32_t* n_eligible, int Nq, const void* k_new, void* k_pool,
                             int64_t k_row_stride, const void* v_new, void* v_pool,
                             int64_t v_row_stride, const void* kidx_new, void* kidx_pool,
                             int idx_dtype, const void* q_idx, const float* w, int H_i, int D_i,
                             const void* q, int Hq, int Dqk, int Dv, int K, float sm_scale,
                             int64_t ld, int chunk, int32_t* idx, void* out, float* lse, void* ws,
                             size_t ws_bytes, dsa_stream_t stream) {
  if (!layout) return set_error(DSA_ERR_INVALID, "prefill_step_chunked: NULL layout");
  if (seq < 0 || seq >= layout->batch)
    return set_error(DSA_ERR_INVALID, "prefill_step_chunked: seq out of range");
  if (!q_pos || !n_eligible || !q_idx || !w || !idx)
    return set_error(DSA_ERR_INVALID, "prefill_step_chunked: NULL pointer");
  if (Nq < 0 || ld < 1 || chunk < 0)
    return set_error(DSA_ERR_INVALID, "prefill_step_chunked: need Nq >= 0, ld >= 1, chunk >= 0");
  if (idx_dtype != DSA_BF16 && idx_dtype != DSA_FP8_E4M3)
    return set_error(DSA_ERR_UNSUPPORTED, "prefill_step_chunked: idx_dtype BF16 or FP8_E4M3");
  if (Nq == 0) return DSA_OK;
  const ChunkLayout L = chunk_layout(Nq, H_i, D_i, ld, Hq, Dqk, Dv, K, chunk);
  int rc = check_ws(ws, ws_bytes, L.total);
  if (rc) return rc;
  char* base = reinterpret_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(ws);
  float* scratch = reinterpret_cast<float*>(base + L.off_scores);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = step_cache_write(layout, seq, q_pos, Nq, k_new, k_pool, k_row_stride, Dqk, v_new, v_pool,
                        v_row_stride, Dv, kidx_new, kidx_pool, idx_dtype, D_i, status, s);
  if (rc) return rc;
  const size_t qrow = (size_t)H_i * D_i * (idx_dtype == DSA_FP8_E4M3 ? 1 : 2);
  for (int r0 = 0; r0 < Nq; r0 += L.C) {
    const int n = Nq - r0 < L.C ? Nq - r0 : L.C;
    rc = index_common(layout, reinterpret_cast<const char*>(q_idx) + (size_t)r0 * qrow, w + (size_t)r0 * H_i,
                      kidx_pool, idx_dtype, H_i, D_i, nullptr, q_pos + r0, seq, n, scratch, ld,
                      base + L.off_index, L.off_topk - L.off_index, stream, status);
    if (rc) return rc;
    rc = topk_common(scratch, ld, n_eligible + r0, n, K, idx + (size_t)r0 * K, base + L.off_topk,
                     L.off_attn - L.off_topk, stream, status);
    if (rc) return rc;
  }
  return attn_common(layout, q, k_pool, k_row_stride, v_pool, v_row_stride, Hq, Dqk, Dv, nullptr,
                     q_pos, Nq, idx, K, sm_scale, out, lse, base + L.off_attn,
                     L.off_scores - L.off_attn, stream, false, status, seq);
}

}  // extern "C"
