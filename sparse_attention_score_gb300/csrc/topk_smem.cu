// topk_smem.cu -- exact top-K with the lower-position tie rule, one row chunk
// per CTA held in shared memory.
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (1): top-K as "block-wise scoring + intra-block reduction +
// cross-block merge" without a global sort; "Day-0 Adaptation of
// Ultra-Large-Scale MoE Models on Heterogeneous AI Accelerators", section 4:
// equal scores resolve deterministically (the lower position wins).
//
// A row of n scores is cut into blocks of at most kCap positions.
//   block step  : one CTA loads its block as order-preserving 32-bit keys into
//                 shared memory and finds the exact K-th largest key T of the
//                 block by three radix histograms (11 + 11 + 10 bits), all in
//                 shared memory; the quota of keys equal to T is taken in
//                 position order.  Kept positions are written in ascending
//                 order by warp segments with one block-wide prefix.
//   merge step  : when a row spans several blocks, the union of the blocks'
//                 winners (which contains the row's exact top-K: anything that
//                 beats a global winner inside its own block beats it
//                 globally) is selected again by the same code, reading the
//                 keys from the workspace.
// Rows of at most kCap positions need one launch; longer rows two.
#include "device_common.cuh"
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCap = 49152;  // keys per CTA in shared memory (192 KB)

struct Shared {
  int hist[2048];
  int scan[kWarps + 1];
  int wgt[kWarps], weq[kWarps];
  int sel_bin, sel_above;
  int chunk_off[33];
};

// Inclusive block scan of one int per thread; returns the inclusive value.
__device__ __forceinline__ int block_incl_scan(int v, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = sh[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    sh[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const int r = incl + sh[warp];
  __syncthreads();
  return r;
}

// One radix pass over the keys matching (prefix, mask): histogram of the
// `bits`-wide digit at `shift`, then the digit that holds the remaining-th
// largest key.  Updates prefix/mask/remaining.
__device__ __forceinline__ void radix_pass(const uint32_t* keys, int cnt, int shift, int bits,
                                           uint32_t& prefix, uint32_t& mask, int& remaining,
                                           Shared& sh) {
  const int nb = 1 << bits;
  for (int i = threadIdx.x; i < nb; i += kThreads) sh.hist[i] = 0;
  __syncthreads();
  // Scores concentrate in a few digits (integer scores share an exponent), so
  // equal bins of a warp are combined first: one shared atomic per distinct bin.
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < cnt; base += kThreads) {
    const int i = base + threadIdx.x;
    uint32_t k = 0;
    bool m = false;
    if (i < cnt) {
      k = keys[i];
      m = (k & mask) == prefix;
    }
    const unsigned active = __ballot_sync(0xffffffffu, m);
    if (m) {
      const uint32_t bin = (k >> shift) & (uint32_t)(nb - 1);
      const unsigned peers = __match_any_sync(active, bin);
      if (lane == __ffs(peers) - 1) atomicAdd(&sh.hist[bin], __popc(peers));
    }
  }
  __syncthreads();
  // thread t owns bins nb-1-2t and nb-2-2t (highest digits first)
  const int b0 = nb - 1 - 2 * (int)threadIdx.x, b1 = b0 - 1;
  const int h0 = b0 >= 0 ? sh.hist[b0] : 0;
  const int h1 = b1 >= 0 ? sh.hist[b1] : 0;
  const int incl = block_incl_scan(h0 + h1, sh.scan);
  const int before = incl - h0 - h1;
  if (before < remaining && incl >= remaining) {
    if (before + h0 >= remaining) {
      sh.sel_bin = b0;
      sh.sel_above = before;
    } else {
      sh.sel_bin = b1;
      sh.sel_above = before + h0;
    }
  }
  __syncthreads();
  remaining -= sh.sel_above;
  prefix |= (uint32_t)sh.sel_bin << shift;
  mask |= (uint32_t)(nb - 1) << shift;
  __syncthreads();
}

struct Job {
  const float* scores;  // block mode: row base
  long long start;      // block mode: first position of the block
  int cnt;              // keys in this CTA
  int K;                // keys to keep
  int32_t* out_pos;     // destination of kept positions (ascending)
  uint32_t* out_key;    // block mode with merge pending: kept keys too
  const int32_t* cand_pos;  // merge mode: positions of the loaded keys (chunked)
};

// Emit the kept positions in ascending order.  pos_of(i) maps a key index to
// its position.
template <typename PosOf>
__device__ __forceinline__ void emit(const uint32_t* keys, int cnt, uint32_t T, int need,
                                     bool take_all, int32_t* out_pos, uint32_t* out_key,
                                     PosOf pos_of, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = ((cnt + kThreads - 1) / kThreads) * 32;
  const int s0 = warp * seg, s1 = min(cnt, s0 + seg);
  int gt = 0, eq = 0;
  if (!take_all) {
    for (int i = s0 + lane; i < s1; i += 32) {
      const uint32_t k = keys[i];
      gt += k > T;
      eq += k == T;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, o);
      eq += __shfl_xor_sync(0xffffffffu, eq, o);
    }
  } else {
    gt = max(0, s1 - s0);
  }
  if (lane == 0) {
    sh.wgt[warp] = gt;
    sh.weq[warp] = eq;
  }
  __syncthreads();
  if (warp == 0) {
    const int g = sh.wgt[lane], e = sh.weq[lane];
    int gi = g, ei = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t1 = __shfl_up_sync(0xffffffffu, gi, o);
      const int t2 = __shfl_up_sync(0xffffffffu, ei, o);
      if (lane >= o) {
        gi += t1;
        ei += t2;
      }
    }
    sh.wgt[lane] = gi - g;  // exclusive
    sh.weq[lane] = ei - e;
  }
  __syncthreads();
  const int eq_off = sh.weq[warp];
  const int quota = take_all ? 0 : max(0, min(eq, need - eq_off));
  int w = sh.wgt[warp] + (take_all ? 0 : min(eq_off, need));
  int eq_seen = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = s0; base < s1; base += 32) {
    const int i = base + lane;
    bool keep = false, is_eq = false;
    uint32_t k = 0;
    if (i < s1) {
      k = keys[i];
      keep = take_all || k > T;
      is_eq = !take_all && k == T;
    }
    const unsigned eqb = __ballot_sync(0xffffffffu, is_eq);
    if (is_eq && eq_seen + __popc(eqb & lt) < quota) keep = true;
    eq_seen += __popc(eqb);
    const unsigned kb = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int o = w + __popc(kb & lt);
      out_pos[o] = pos_of(i);
      if (out_key) out_key[o] = k;
    }
    w += __popc(kb);
  }
}

// mode 0: block step writing final indices (row fits one block)
// mode 1: block step writing the block's winners to the workspace
// mode 2: merge step over a row's block winners
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    k_topk_block(TopkParams a, int nchunks, uint32_t* cand_key, int32_t* cand_pos, int* cand_cnt) {
  extern __shared__ uint32_t keys[];
  __shared__ Shared sh;
  grid_dependency_wait();
  launch_dependents();
  const int r = kMode == 2 ? blockIdx.x : blockIdx.y;
  const int c = kMode == 2 ? 0 : blockIdx.x;
  long long n = __ldg(&a.n_elig[r]);
  if (n < 0) n = 0;
  if (n > a.ld) {
    if (threadIdx.x == 0 && c == 0) flag_status(a.status, DSA_STATUS_BAD_LENGTH);
    n = a.ld;
  }
  const int K = a.K;
  int cnt;
  long long start = 0;
  if (kMode != 2) {
    start = (long long)c * kCap;
    const long long rem = n - start;
    cnt = (int)(rem < 0 ? 0 : (rem > kCap ? kCap : rem));
    const float* src = a.scores + (long long)r * a.ld + start;
    for (int i = threadIdx.x; i < cnt; i += kThreads) keys[i] = score_key(__ldg(&src[i]));
  } else {
    if (threadIdx.x == 0) {
      int off = 0;
      for (int j = 0; j < nchunks; ++j) {
        sh.chunk_off[j] = off;
        off += __ldg(&cand_cnt[(long long)r * nchunks + j]);
      }
      sh.chunk_off[nchunks] = off;
    }
    __syncthreads();
    cnt = sh.chunk_off[nchunks];
    for (int j = 0; j < nchunks; ++j) {
      const int o = sh.chunk_off[j], m = sh.chunk_off[j + 1] - o;
      const uint32_t* src = cand_key + ((long long)r * nchunks + j) * K;
      for (int i = threadIdx.x; i < m; i += kThreads) keys[o + i] = __ldg(&src[i]);
    }
  }
  __syncthreads();

  const int keep_n = cnt < K ? cnt : K;
  const bool take_all = keep_n == cnt;
  uint32_t prefix = 0, mask = 0;
  int remaining = keep_n;
  if (!take_all) {
    radix_pass(keys, cnt, 21, 11, prefix, mask, remaining, sh);
    radix_pass(keys, cnt, 10, 11, prefix, mask, remaining, sh);
    radix_pass(keys, cnt, 0, 10, prefix, mask, remaining, sh);
  }

  if (kMode == 0) {
    int32_t* out = a.idx + (long long)r * K;
    emit(keys, cnt, prefix, remaining, take_all, out, (uint32_t*)nullptr,
         [&](int i) { return (int32_t)(start + i); }, sh);
    for (int j = keep_n + threadIdx.x; j < K; j += kThreads) out[j] = -1;
  } else if (kMode == 1) {
    const long long slot = (long long)r * nchunks + c;
    emit(keys, cnt, prefix, remaining, take_all, cand_pos + slot * K, cand_key + slot * K,
         [&](int i) { return (int32_t)(start + i); }, sh);
    if (threadIdx.x == 0) cand_cnt[slot] = keep_n;
  } else {
    int32_t* out = a.idx + (long long)r * K;
    const int32_t* cp = cand_pos + (long long)r * nchunks * K;
    emit(keys, cnt, prefix, remaining, take_all, out, (uint32_t*)nullptr,
         [&](int i) {
           int j = 0;
           while (j + 1 < nchunks && sh.chunk_off[j + 1] <= i) ++j;
           return __ldg(&cp[(long long)j * K + (i - sh.chunk_off[j])]);
         },
         sh);
    for (int j = keep_n + threadIdx.x; j < K; j += kThreads) out[j] = -1;
  }
}

template <int kMode>
void set_smem_attr() {
  static bool done = false;
  if (!done) {
    cudaFuncSetAttribute(k_topk_block<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kCap * (int)sizeof(uint32_t));
    done = true;
  }
}

}  // namespace

int topk_chunks(long long ld) { return (int)((ld + kCap - 1) / kCap); }

bool topk_smem_eligible(long long ld, int K) {
  const int nch = topk_chunks(ld);
  return nch <= 32 && (nch == 1 || (long long)nch * K <= kCap);
}

size_t topk_smem_ws(int Nq, long long ld, int K) {
  const int nch = topk_chunks(ld);
  if (nch <= 1) return 0;
  return (size_t)Nq * nch * ((size_t)K * 8 + 4) + 256;
}

int launch_topk_smem(const TopkParams& p, void* ws, cudaStream_t s) {
  const int nch = topk_chunks(p.ld);
  const size_t smem = kCap * sizeof(uint32_t);
  if (nch == 1) {
    set_smem_attr<0>();
    const cudaError_t e = launch_pdl(k_topk_block<0>, dim3(1, p.Nq), dim3(kThreads), smem, s, p, 1,
                                     (uint32_t*)nullptr, (int32_t*)nullptr, (int*)nullptr);
    count_launch();
    if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
    return check_launch("topk");
  }
  char* base = (char*)ws + kWsHeader;
  const size_t nslot = (size_t)p.Nq * nch;
  uint32_t* ckey = reinterpret_cast<uint32_t*>(base);
  int32_t* cpos = reinterpret_cast<int32_t*>(base + nslot * p.K * 4);
  int* ccnt = reinterpret_cast<int*>(base + nslot * p.K * 8);
  set_smem_attr<1>();
  set_smem_attr<2>();
  cudaError_t e = launch_pdl(k_topk_block<1>, dim3(nch, p.Nq), dim3(kThreads), smem, s, p, nch,
                             ckey, cpos, ccnt);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  int rc = check_launch("topk (blocks)");
  if (rc) return rc;
  e = launch_pdl(k_topk_block<2>, dim3(p.Nq), dim3(kThreads), smem, s, p, nch, ckey, cpos, ccnt);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("topk (merge)");
}

}  // namespace dsa
