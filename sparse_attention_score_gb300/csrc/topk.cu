// topk.cu -- stage 2 of the DSA path: exact top-K with the lower-position tie
// rule.
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (1): top-K without a global sort, as block-wise scoring,
// intra-block reduction and a cross-block merge; "Day-0 Adaptation of
// Ultra-Large-Scale MoE Models on Heterogeneous AI Accelerators", section 4:
// equal scores resolve deterministically (here: the lower position wins).
//
// Method (radix select on order-preserving 32-bit keys):
//   1. per radix digit (8 bits, most significant first) every block of
//      positions contributes to a 256-bin histogram of the keys that still
//      match the selected prefix (block-wise scoring + intra-block reduction);
//   2. the digit holding the K-th largest key is found from the histogram's
//      suffix counts (merge), narrowing the prefix; after four digits the exact
//      threshold key T and the number `need` of keys equal to T to keep are
//      known;
//   3. one ordered sweep keeps every key > T and the first `need` keys == T in
//      position order, writing positions ascending (a bitmask-and-prefix-count
//      compaction over each block of positions).
#include "device_common.cuh"
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kTopkThreads = 1024;
constexpr int kWarps = kTopkThreads / 32;

// Block-wide exclusive scan of one flag per thread; returns the prefix and
// writes the block total to *total.  `sh` holds kWarps ints.
__device__ __forceinline__ int block_excl_scan(bool flag, int* sh, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) sh[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = sh[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    sh[lane] = incl - v;
    if (lane == 31) sh[kWarps] = incl;
  }
  __syncthreads();
  *total = sh[kWarps];
  return sh[warp] + in_warp;
}

// One CTA per row; keys are re-read from global memory (L2) on every pass.
// Used only for rows too long for the shared-memory block kernel (topk_smem.cu).
__global__ void __launch_bounds__(kTopkThreads) k_topk_rowwise(TopkParams a) {
  __shared__ int hist[256];
  grid_dependency_wait();
  launch_dependents();
  __shared__ int scan_sh[kWarps + 1];
  __shared__ uint32_t sel_digit;
  __shared__ int sel_above;

  const int r = blockIdx.x;
  const float* row = a.scores + (long long)r * a.ld;
  int32_t* out = a.idx + (long long)r * a.K;
  long long n = __ldg(&a.n_elig[r]);
  if (n < 0) n = 0;
  if (n > a.ld) {
    if (threadIdx.x == 0) flag_status(a.status, DSA_STATUS_BAD_LENGTH);
    n = a.ld;
  }
  const int K = a.K;
  const long long m = n < K ? n : K;

  uint32_t T = 0;       // threshold key
  long long need = 0;   // keys equal to T to keep
  const bool take_all = (m == n);
  if (!take_all) {
    uint32_t prefix = 0, mask = 0;
    long long remaining = m;  // how many of the keys matching `prefix` to keep
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
      for (long long i = threadIdx.x; i < n; i += kTopkThreads) {
        const uint32_t k = score_key(__ldg(&row[i]));
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // suffix sums over 256 bins, 8 bins per lane, highest digit first
        const int lane = threadIdx.x;
        int loc[8];
        int s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          loc[j] = hist[255 - (lane * 8 + j)];
          s += loc[j];
        }
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        int before = incl - s;  // keys in strictly higher bins than this lane's first
        const long long rem = remaining;
        bool mine = before < rem && incl >= rem;
        if (mine) {
          int acc = before;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (acc + loc[j] >= rem) {
              sel_digit = 255u - (uint32_t)(lane * 8 + j);
              sel_above = acc;
              break;
            }
            acc += loc[j];
          }
        }
      }
      __syncthreads();
      remaining -= sel_above;
      prefix |= sel_digit << shift;
      mask |= 255u << shift;
      __syncthreads();
    }
    T = prefix;
    need = remaining;
  }

  // ordered compaction: keep keys > T, and the first `need` keys == T
  long long written = 0, eq_seen = 0;
  for (long long base = 0; base < n; base += kTopkThreads) {
    const long long i = base + threadIdx.x;
    bool keep = false, eq = false;
    if (i < n) {
      if (take_all) {
        keep = true;
      } else {
        const uint32_t k = score_key(__ldg(&row[i]));
        keep = k > T;
        eq = (k == T);
      }
    }
    if (!take_all) {
      int eq_total;
      const int eq_rank = block_excl_scan(eq, scan_sh, &eq_total);
      if (eq && eq_seen + eq_rank < need) keep = true;
      eq_seen += eq_total;
    }
    int total;
    const int pos = block_excl_scan(keep, scan_sh, &total);
    if (keep && written + pos < K) out[written + pos] = (int32_t)i;
    written += total;
  }
  for (long long j = m + threadIdx.x; j < K; j += kTopkThreads) out[j] = -1;
}

}  // namespace

size_t topk_ws(int Nq, long long ld, int K) {
  return kWsHeader + (topk_smem_eligible(ld, K) ? topk_smem_ws(Nq, ld, K) : 0);
}

int launch_topk(const TopkParams& p, void* ws, size_t, cudaStream_t s) {
  if (p.Nq == 0) return DSA_OK;
  if (topk_smem_eligible(p.ld, p.K)) return launch_topk_smem(p, ws, s);
  k_topk_rowwise<<<p.Nq, kTopkThreads, 0, s>>>(p);
  count_launch();
  return check_launch("topk");
}

}  // namespace dsa
