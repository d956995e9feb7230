// index_score.cu -- stage 1 of the DSA path: the lightweight indexer score.
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (1): every historical position is scored against the query through
// a low-dimension indexer key; the score is read as
//     s[r][p] = sum_h w[r][h] * max(0, q_idx[r][h] . k_idx[p])
// over the causal positions p <= q_pos[r], p < L_b; -inf elsewhere in the row.
//
// This file holds the CUDA-core kernel, used for every shape the tensor-core
// kernel (index_tc.cu) does not cover; it is exact for integer-valued inputs
// (fp32 accumulation of integers < 2^24).
#include "device_common.cuh"
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kGenThreads = 128;

template <int DT>
__device__ __forceinline__ float load_code(const void* base, long long i) {
  if (DT == DSA_BF16) return bf16_bits_to_float(__ldg((const uint16_t*)base + i));
  const uint8_t v = __ldg((const uint8_t*)base + i);
  return e4m3x2_to_float2((uint16_t)v).x;
}

// Load D consecutive codes starting at element `off` (16-byte aligned rows).
template <int D, int DT>
__device__ __forceinline__ void load_row(const void* base, long long off, float (&k)[D]) {
  if (DT == DSA_BF16) {
    const uint4* src = reinterpret_cast<const uint4*>((const uint16_t*)base + off);
#pragma unroll
    for (int v = 0; v < D / 8; ++v) {
      uint4 u = __ldg(src + v);
      uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        k[v * 8 + 2 * j] = __uint_as_float(w4[j] << 16);
        k[v * 8 + 2 * j + 1] = __uint_as_float(w4[j] & 0xffff0000u);
      }
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>((const uint8_t*)base + off);
#pragma unroll
    for (int v = 0; v < D / 16; ++v) {
      uint4 u = __ldg(src + v);
      uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 lo = e4m3x2_to_float2((uint16_t)(w4[j] & 0xffffu));
        float2 hi = e4m3x2_to_float2((uint16_t)(w4[j] >> 16));
        k[v * 16 + 4 * j + 0] = lo.x;
        k[v * 16 + 4 * j + 1] = lo.y;
        k[v * 16 + 4 * j + 2] = hi.x;
        k[v * 16 + 4 * j + 3] = hi.y;
      }
    }
  }
}

// One thread per position; grid (ceil(ld/128), Nq).  The query's indexer
// heads and weights sit in shared memory and are read as broadcasts.  Each
// thread's sequence length, causal bound and block-table entry are loaded
// before the heads (none depends on another), so the chain to its key row is
// one load deep.
template <int D, int DT>
__global__ void __launch_bounds__(kGenThreads) k_index_score_generic(IndexParams a) {
  extern __shared__ float sm[];
  const int H = a.H;
  grid_dependency_wait();
  launch_dependents();
  const int r = blockIdx.y;
  // a CTA covers one 128-position tile; a tile the caller left out is -inf
  static_assert(kGenThreads == 128, "one skip-mask tile per CTA");
  if (a.skip) {
    const uint8_t m = __ldg(&a.skip[(long long)r * a.skip_stride + blockIdx.x]);
    if (m != 0) {
      const long long p = (long long)blockIdx.x * kGenThreads + threadIdx.x;
      if (m == kSkipInf && p < a.ld) a.scores[(long long)r * a.ld + p] = -INFINITY;
      return;
    }
  }
  const long long p = (long long)blockIdx.x * kGenThreads + threadIdx.x;
  const int b = a.seq_const >= 0 ? a.seq_const : (a.q_seq ? __ldg(&a.q_seq[r]) : r);
  const bool b_ok = b >= 0 && b < a.lay.batch;
  long long L = 0, qp = 0;
  int page = -1;
  if (b_ok) {
    L = __ldg(&a.lay.seq_lens[b]);
    if (a.q_pos) qp = __ldg(&a.q_pos[r]);
    const long long slot = p / a.lay.bs;
    if (p < a.ld && slot < a.lay.maxb) page = __ldg(&a.lay.bt[(long long)b * a.lay.maxb + slot]);
  }
  float* qs = sm;
  float* ws = sm + H * D;
  for (int i = threadIdx.x; i < H * D; i += blockDim.x)
    qs[i] = load_code<DT>(a.q_idx, (long long)r * H * D + i);
  for (int i = threadIdx.x; i < H; i += blockDim.x) ws[i] = __ldg(&a.w[(long long)r * H + i]);
  __syncthreads();

  if (p >= a.ld) return;
  float out = -INFINITY;
  if (b_ok) {
    const long long cap = (long long)a.lay.maxb * a.lay.bs;
    if (L > cap || L > a.ld) {
      if (p == 0) flag_status(a.status, DSA_STATUS_BAD_LENGTH);
      L = L < cap ? L : cap;
    }
    long long last = a.q_pos ? qp : L - 1;
    if (last > L - 1) last = L - 1;
    if (p <= last) {
      // phys_row with the entry loaded above
      const long long row =
          page >= 0 && page < a.lay.nb ? (long long)page * a.lay.bs + p % a.lay.bs : -1;
      if (row < 0) {
        flag_status(a.status, DSA_STATUS_BAD_BLOCK);
      } else {
        float k[D];
        load_row<D, DT>(a.kidx, row * D, k);
        float s = 0.0f;
        for (int h = 0; h < H; ++h) {
          float dot = 0.0f;
#pragma unroll
          for (int d = 0; d < D; ++d) dot = fmaf(qs[h * D + d], k[d], dot);
          s = fmaf(ws[h], fmaxf(dot, 0.0f), s);
        }
        out = s + 0.0f;  // -0.0 -> +0.0
      }
    }
  } else if (p == 0) {
    flag_status(a.status, DSA_STATUS_BAD_INDEX);
  }
  a.scores[(long long)r * a.ld + p] = out;
}

template <int D, int DT>
int launch_generic(const IndexParams& p, cudaStream_t s) {
  const size_t smem = sizeof(float) * ((size_t)p.H * D + p.H);
  auto kern = k_index_score_generic<D, DT>;
  const int arc = ensure_dynamic_smem((const void*)kern, 96 * 1024, "index_score");
  if (arc) return arc;
  dim3 grid((unsigned)((p.ld + kGenThreads - 1) / kGenThreads), (unsigned)p.Nq);
  const cudaError_t e = launch_pdl(kern, grid, dim3(kGenThreads), smem, s, p);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("index_score");
}

}  // namespace

bool index_score_supported(int dtype, int H, int D) {
  return (dtype == DSA_BF16 || dtype == DSA_FP8_E4M3) && H >= 1 && H <= 128 &&
         (D == 32 || D == 64 || D == 128);
}

size_t index_score_ws(int, int, int, long long) { return kWsHeader; }

int launch_index_score(const IndexParams& p, cudaStream_t s) {
  if (p.Nq == 0) return DSA_OK;
  if (p.seq_const >= 0 && index_prefill_tc_eligible(p)) return launch_index_prefill_tc(p, s);
  if (p.seq_const < 0 && index_tc_eligible(p)) return launch_index_tc(p, s);
  if (p.Nq > 65535) return set_error(DSA_ERR_UNSUPPORTED, "index_score: Nq > 65535 for this shape");
  if (p.dtype == DSA_BF16) {
    if (p.D == 32) return launch_generic<32, DSA_BF16>(p, s);
    if (p.D == 64) return launch_generic<64, DSA_BF16>(p, s);
    return launch_generic<128, DSA_BF16>(p, s);
  }
  if (p.D == 32) return launch_generic<32, DSA_FP8_E4M3>(p, s);
  if (p.D == 64) return launch_generic<64, DSA_FP8_E4M3>(p, s);
  return launch_generic<128, DSA_FP8_E4M3>(p, s);
}

}  // namespace dsa
