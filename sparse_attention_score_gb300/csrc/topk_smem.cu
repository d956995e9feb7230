// topk_smem.cu -- exact top-K with the lower-position tie rule, one row chunk
// per CTA held in shared memory.
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (1): the selection is made inside blocks of positions and the
// blocks' results are then combined, with no sort of a whole row; "Day-0
// Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI Accelerators",
// section 4:
// equal scores resolve deterministically (the lower position wins).
//
// A row of n scores is cut into as few blocks of at most kCap positions as
// hold it.  (Cutting short rows further, to spread 32 decode rows over more
// SMs, measured slower: 35 us against 21 us for rows of up to 32 K.)
//   block step  : one CTA loads its block as order-preserving 32-bit keys into
//                 shared memory and finds the exact K-th largest key T of the
//                 block by radix histograms of up to 11 bits, all in shared
//                 memory; the quota of keys equal to T is taken in position
//                 order.  Kept positions are written in ascending order by
//                 warp segments with one block-wide prefix.
//   merge step  : when a row spans several blocks, the union of the blocks'
//                 winners contains the row's exact top-K (anything that beats
//                 a global winner inside its own block beats it globally).
//                 Each block also stores its own K-th largest key; the row's
//                 K-th largest key is at least the largest of those, B, so
//                 only winners >= B take part.  A second kernel (one CTA per
//                 row) selects again over them in shared memory and writes
//                 the positions in block order, which is position order.
// A row that fits one block takes one launch; other rows two.
#include "device_common.cuh"
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCap = 49152;  // keys per CTA in shared memory (192 KB)

constexpr int kWords = kCap / 32;  // one bit per key

constexpr int kMaxBlocks = 32;  // blocks per row (the merge reads one bound per lane)

struct Shared {
  int hist[2048];
  uint32_t gtm[kWords], eqm[kWords];  // per 32 keys: which are > T, which == T
  uint32_t scan[kWarps + 1];
  int wgt[kWarps], weq[kWarps];
  int sel_bin, sel_above;
  uint32_t bound;  // merge: the row's bound on its K-th largest key
  int fcnt;
};

// 16-byte asynchronous global -> shared copy (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}

// Inclusive block scan of one unsigned value per thread (sums wrap modulo
// 2^32, which packed counts rely on); returns the inclusive value.
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = sh[lane];
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    sh[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const uint32_t r = incl + sh[warp];
  __syncthreads();
  return r;
}

// One radix digit: histogram of the `bits`-wide digit at `shift` over the keys
// matching (prefix, mask), then the digit holding the remaining-th largest
// key.  Updates prefix/mask/remaining.  Keys are read four at a time; the
// digits below the bits shared by every key of the block are diverse enough
// that plain shared atomics rarely collide.
// Also returns, over the keys matching (prefix, mask) on entry, the OR and the
// AND of their bits: where the two agree below the digit, every candidate
// shares those bits, and so does the threshold.
__device__ __forceinline__ void radix_pass(const uint32_t* keys, int cnt, int shift, int bits,
                                           uint32_t& prefix, uint32_t& mask, int& remaining,
                                           uint32_t& cand_or, uint32_t& cand_and, Shared& sh) {
  const int nb = 1 << bits;
  for (int i = threadIdx.x; i < nb; i += kThreads) sh.hist[i] = 0;
  __syncthreads();
  const uint4* k4 = reinterpret_cast<const uint4*>(keys);
  const int n4 = (cnt + 3) >> 2;  // the array has room for three keys past cnt
  const uint32_t dm = (uint32_t)(nb - 1);
  uint32_t c_or = 0u, c_and = 0xFFFFFFFFu;
#pragma unroll 4
  for (int j = threadIdx.x; j < n4; j += kThreads) {
    const uint4 v = k4[j];
    const int i0 = 4 * j;
    if ((v.x & mask) == prefix) {
      atomicAdd(&sh.hist[(v.x >> shift) & dm], 1);
      c_or |= v.x;
      c_and &= v.x;
    }
    if (i0 + 1 < cnt && (v.y & mask) == prefix) {
      atomicAdd(&sh.hist[(v.y >> shift) & dm], 1);
      c_or |= v.y;
      c_and &= v.y;
    }
    if (i0 + 2 < cnt && (v.z & mask) == prefix) {
      atomicAdd(&sh.hist[(v.z >> shift) & dm], 1);
      c_or |= v.z;
      c_and &= v.z;
    }
    if (i0 + 3 < cnt && (v.w & mask) == prefix) {
      atomicAdd(&sh.hist[(v.w >> shift) & dm], 1);
      c_or |= v.w;
      c_and &= v.w;
    }
  }
  c_or = __reduce_or_sync(0xffffffffu, c_or);
  c_and = __reduce_and_sync(0xffffffffu, c_and);
  if ((threadIdx.x & 31) == 0) {
    sh.wgt[threadIdx.x >> 5] = (int)c_or;
    sh.weq[threadIdx.x >> 5] = (int)c_and;
  }
  __syncthreads();
  cand_or = __reduce_or_sync(0xffffffffu, (uint32_t)sh.wgt[threadIdx.x & 31]);
  cand_and = __reduce_and_sync(0xffffffffu, (uint32_t)sh.weq[threadIdx.x & 31]);
  // thread t owns bins nb-1-2t and nb-2-2t (highest digits first)
  const int b0 = nb - 1 - 2 * (int)threadIdx.x, b1 = b0 - 1;
  const int h0 = b0 >= 0 ? sh.hist[b0] : 0;
  const int h1 = b1 >= 0 ? sh.hist[b1] : 0;
  const int incl = (int)block_incl_scan((uint32_t)(h0 + h1), sh.scan);
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
  mask |= dm << shift;
  __syncthreads();
}

// Minimum and maximum key over the block (every thread gets both).
__device__ __forceinline__ void block_min_max(uint32_t& lo, uint32_t& hi, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    sh.wgt[warp] = (int)lo;
    sh.weq[warp] = (int)hi;
  }
  __syncthreads();
  lo = __reduce_min_sync(0xffffffffu, (uint32_t)sh.wgt[lane]);
  hi = __reduce_max_sync(0xffffffffu, (uint32_t)sh.weq[lane]);
  __syncthreads();
}

// Exact K-th largest key: the bits shared by every key (from the block's
// minimum and maximum) are fixed at once, the rest in digits of up to 11 bits.
// On return `prefix` is the threshold key T and `remaining` the number of keys
// equal to T to keep.
__device__ __forceinline__ void select_threshold(const uint32_t* keys, int cnt, uint32_t kmin,
                                                 uint32_t kmax, uint32_t& prefix, int& remaining,
                                                 Shared& sh) {
  uint32_t mask = 0;
  prefix = 0;
  if (kmin == kmax) {
    prefix = kmax;  // every key ties: T is that key
    return;
  }
  const int hb = 31 - __clz(kmin ^ kmax);  // highest bit where keys differ
  mask = hb == 31 ? 0u : ~((2u << hb) - 1u);
  prefix = kmax & mask;
  int hi = hb;
  while (hi >= 0) {
    const int bits = hi + 1 < 11 ? hi + 1 : 11;
    const int shift = hi + 1 - bits;
    uint32_t cand_or, cand_and;
    radix_pass(keys, cnt, shift, bits, prefix, mask, remaining, cand_or, cand_and, sh);
    // the bits below this digit, where every candidate agrees, need no pass
    // (integer-valued scores leave their low mantissa bits zero)
    const uint32_t below = shift > 0 ? (1u << shift) - 1u : 0u;
    if (below && ((cand_or ^ cand_and) & below) == 0u) {
      prefix |= cand_and & below;
      mask |= below;
      break;
    }
    hi = shift - 1;
  }
}

// Emit the kept positions in ascending order: every key > T and the first
// `need` keys == T (position order); all keys when take_all.  pos_of(i) maps
// a key index to its position.  One pass over the keys builds two bit masks
// per 32 consecutive keys (a warp ballot each: > T, == T); one block scan of
// the packed per-word counts (greater | equal << 16) then gives every word its
// output offset and its rank among the equal keys, and each thread writes the
// kept positions of its two words.  Every key is read once.
template <typename PosOf>
__device__ __forceinline__ void emit(const uint32_t* keys, int cnt, uint32_t T, int need,
                                     bool take_all, int32_t* out_pos, uint32_t* out_key,
                                     PosOf pos_of, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwords = (cnt + 31) >> 5;
  for (int wd = warp; wd < nwords; wd += kWarps) {
    const int i = wd * 32 + lane;
    const uint32_t k = i < cnt ? keys[i] : 0u;
    const bool in = i < cnt;
    const uint32_t g = __ballot_sync(0xffffffffu, in && (take_all || k > T));
    const uint32_t e = __ballot_sync(0xffffffffu, in && !take_all && k == T);
    if (lane == 0) {
      sh.gtm[wd] = g;
      sh.eqm[wd] = e;
    }
  }
  __syncthreads();
  // thread t owns words 2t and 2t + 1
  const int w0 = 2 * (int)threadIdx.x, w1 = w0 + 1;
  const uint32_t g0 = w0 < nwords ? sh.gtm[w0] : 0u, e0 = w0 < nwords ? sh.eqm[w0] : 0u;
  const uint32_t g1 = w1 < nwords ? sh.gtm[w1] : 0u, e1 = w1 < nwords ? sh.eqm[w1] : 0u;
  // packed (greater | equal << 16): each field stays below kCap < 2^16, so the
  // sums never carry between fields; unsigned, since equal << 16 may pass 2^31
  const uint32_t c0 = (uint32_t)__popc(g0) | ((uint32_t)__popc(e0) << 16);
  const uint32_t c1 = (uint32_t)__popc(g1) | ((uint32_t)__popc(e1) << 16);
  const uint32_t incl = block_incl_scan(c0 + c1, sh.scan);
  uint32_t before = incl - c0 - c1;  // packed counts of the earlier words
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int wd = h ? w1 : w0;
    if (wd >= nwords) break;
    const uint32_t g = h ? g1 : g0;
    uint32_t e = h ? e1 : e0;
    const int gt_before = (int)(before & 0xFFFFu), eq_before = (int)(before >> 16);
    // keep the first (need - eq_before) keys == T of this word
    int keep_eq = need - eq_before;
    uint32_t ek = 0u;
    for (; keep_eq > 0 && e; --keep_eq) {
      const uint32_t lowest = e & (0u - e);
      ek |= lowest;
      e ^= lowest;
    }
    uint32_t m = g | ek;
    int o = gt_before + min(max(need, 0), eq_before);
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1;
      const int i = wd * 32 + b;
      out_pos[o] = pos_of(i);
      if (out_key) out_key[o] = keys[i];
      ++o;
    }
    before += h ? 0 : c0;
  }
}

// Merge of row r's block winners (one CTA per row).  The winners sit in the
// workspace as [block][K] slots; they are loaded into shared memory in that
// layout, each key raised by one, with 0 in the slots that hold nothing or a
// key below the row's bound, so that every winner outranks every empty slot.
// The selection and the ordered write are then those of the block step, over
// slot indices: block order, then position order within a block, which is
// ascending position order.
__global__ void __launch_bounds__(kThreads, 1)
    k_topk_merge(TopkParams a, int nchunks, const uint32_t* cand_key, const int32_t* cand_pos,
                 const int* cand_cnt, const uint32_t* cand_kth) {
  extern __shared__ uint4 keys_raw[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(keys_raw);
  __shared__ Shared sh;
  __shared__ int s_cnt[kMaxBlocks];
  grid_dependency_wait();
  launch_dependents();
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K;
  const long long base = (long long)r * nchunks * K;
  if (warp == 0) {
    uint32_t b = 0u;
    int m = 0;
    if (lane < nchunks) {
      b = __ldg(&cand_kth[(long long)r * nchunks + lane]);
      m = __ldg(&cand_cnt[(long long)r * nchunks + lane]);
      s_cnt[lane] = m;
    }
    b = __reduce_max_sync(0xffffffffu, b);
    if (lane == 0) sh.bound = b;
  }
  __syncthreads();
  const uint32_t bound = sh.bound;
  const int total = nchunks * K;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  int real = 0;
  // slot q of block j keeps its key, raised by one, if it holds a winner at
  // or above the bound (keys stay below 2^32 - 1: the largest is that of +inf)
  auto take = [&](uint32_t v, int q, int cnt) -> uint32_t {
    const bool in = q < cnt && v >= bound;
    real += in ? 1 : 0;
    return in ? v + 1u : 0u;
  };
  const uint32_t* src = cand_key + base;
  if ((K & 3) == 0 && (((uintptr_t)src) & 15u) == 0) {
    // every slot in flight at once (16-byte copies; the slots past a block's
    // count hold stale words and are cleared below), then the keys are
    // filtered in place; four keys of one 16-byte word share their block
    const int n4 = total >> 2;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int j = threadIdx.x; j < n4; j += kThreads) cp_async16(keys + 4 * j, s4 + j);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    uint4* k4 = reinterpret_cast<uint4*>(keys);
#pragma unroll 4
    for (int j = threadIdx.x; j < n4; j += kThreads) {
      const int i = 4 * j;
      const int b = i / K, q = i - b * K;
      const int cnt = s_cnt[b];
      uint4 v = k4[j];
      v.x = take(v.x, q, cnt);
      v.y = take(v.y, q + 1, cnt);
      v.z = take(v.z, q + 2, cnt);
      v.w = take(v.w, q + 3, cnt);
      k4[j] = v;
      kmin = min(min(kmin, min(v.x, v.y)), min(v.z, v.w));
      kmax = max(max(kmax, max(v.x, v.y)), max(v.z, v.w));
    }
  } else {
#pragma unroll 4
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const int j = i / K, q = i - j * K;
      const uint32_t k = take(q < s_cnt[j] ? __ldg(&cand_key[base + i]) : 0u, q, s_cnt[j]);
      keys[i] = k;
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
  }
  // number of winners >= bound (a block-wide sum through the scan buffer)
  real = __reduce_add_sync(0xffffffffu, real);
  if (lane == 0) sh.scan[warp] = (uint32_t)real;
  block_min_max(kmin, kmax, sh);  // includes the barrier after the loads
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < kWarps; ++w) t += (int)sh.scan[w];
    sh.fcnt = t;
  }
  __syncthreads();
  const int fcnt = sh.fcnt;
  const int keep_n = fcnt < K ? fcnt : K;
  uint32_t T = 0u;  // every non-empty slot holds a key > 0
  int need = 0;
  if (keep_n < fcnt) {
    need = keep_n;
    select_threshold(keys, total, kmin, kmax, T, need, sh);
  }
  // the kept slots' indices, in output order, over the keys (emit reads every
  // key before its first write); then their positions, all loads in flight
  int32_t* sel = reinterpret_cast<int32_t*>(keys);
  emit(keys, total, T, need, false, sel, (uint32_t*)nullptr, [](int i) { return i; }, sh);
  __syncthreads();
  int32_t* out = a.idx + (long long)r * K;
#pragma unroll 4
  for (int j = threadIdx.x; j < K; j += kThreads)
    out[j] = j < keep_n ? __ldg(&cand_pos[base + sel[j]]) : -1;
}

// Grid: x = row (up to 2^31 - 1 rows), y = block of the row.
// mode 0: the row is one block; writes the final indices
// mode 1: block `blockIdx.y` of `nchunks` blocks of `blk` positions; writes
//         the block's winners, their count and the block's K-th largest key
//         (0 when the block has fewer than K positions) to the workspace
template <int kMode>
__global__ void __launch_bounds__(kThreads, 2)
    k_topk_block(TopkParams a, int nchunks, int blk, uint32_t* cand_key, int32_t* cand_pos,
                 int* cand_cnt, uint32_t* cand_kth) {
  extern __shared__ uint4 keys_raw[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(keys_raw);
  __shared__ Shared sh;
  grid_dependency_wait();
  launch_dependents();
  const int r = blockIdx.x;
  const int c = blockIdx.y;
  long long n = __ldg(&a.n_elig[r]);
  if (n < 0) n = 0;
  if (n > a.ld) {
    if (threadIdx.x == 0 && c == 0) flag_status(a.status, DSA_STATUS_BAD_LENGTH);
    n = a.ld;
  }
  const int K = a.K;
  const long long start = (long long)c * blk;
  const long long rem = n - start;
  const int cnt = (int)(rem < 0 ? 0 : (rem > blk ? blk : rem));
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  {
    const float* src = a.scores + (long long)r * a.ld + start;
    if ((((uintptr_t)src) & 15u) == 0) {
      // the whole block in flight at once (16-byte copies), then the scores
      // are turned into keys in place
      const int n4 = cnt >> 2;
      const float4* s4 = reinterpret_cast<const float4*>(src);
      for (int j = threadIdx.x; j < n4; j += kThreads) cp_async16(keys + 4 * j, s4 + j);
      for (int i = 4 * n4 + threadIdx.x; i < cnt; i += kThreads)
        keys[i] = __float_as_uint(__ldg(&src[i]));
      asm volatile("cp.async.wait_all;" ::: "memory");
      __syncthreads();
      uint4* k4 = reinterpret_cast<uint4*>(keys);
#pragma unroll 4
      for (int j = threadIdx.x; j < n4; j += kThreads) {
        uint4 v = k4[j];
        v.x = score_key(__uint_as_float(v.x));
        v.y = score_key(__uint_as_float(v.y));
        v.z = score_key(__uint_as_float(v.z));
        v.w = score_key(__uint_as_float(v.w));
        k4[j] = v;
        kmin = min(min(kmin, min(v.x, v.y)), min(v.z, v.w));
        kmax = max(max(kmax, max(v.x, v.y)), max(v.z, v.w));
      }
      for (int i = 4 * n4 + threadIdx.x; i < cnt; i += kThreads) {
        const uint32_t k = score_key(__uint_as_float(keys[i]));
        keys[i] = k;
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    } else {
#pragma unroll 8
      for (int i = threadIdx.x; i < cnt; i += kThreads) {
        const uint32_t k = score_key(__ldg(&src[i]));
        keys[i] = k;
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    }
  }
  block_min_max(kmin, kmax, sh);  // includes the barrier after the loads

  const int keep_n = cnt < K ? cnt : K;
  const bool take_all = keep_n == cnt;
  uint32_t T = 0;
  int need = keep_n;
  if (!take_all) select_threshold(keys, cnt, kmin, kmax, T, need, sh);

  if (kMode == 0) {
    int32_t* out = a.idx + (long long)r * K;
    emit(keys, cnt, T, need, take_all, out, (uint32_t*)nullptr,
         [&](int i) { return (int32_t)(start + i); }, sh);
    for (int j = keep_n + threadIdx.x; j < K; j += kThreads) out[j] = -1;
  } else {
    const long long slot = (long long)r * nchunks + c;
    emit(keys, cnt, T, need, take_all, cand_pos + slot * K, cand_key + slot * K,
         [&](int i) { return (int32_t)(start + i); }, sh);
    if (threadIdx.x == 0) {
      cand_cnt[slot] = keep_n;
      cand_kth[slot] = cnt >= K ? (take_all ? kmin : T) : 0u;
    }
  }
}

template <int kMode>
int set_smem_attr() {
  return ensure_dynamic_smem((const void*)k_topk_block<kMode>, (kCap + 4) * (int)sizeof(uint32_t),
                             "topk");
}

}  // namespace

int topk_chunks(long long ld) { return (int)((ld + kCap - 1) / kCap); }

bool topk_smem_eligible(long long ld, int K) {
  const int nch = topk_chunks(ld);
  return nch <= kMaxBlocks && (nch == 1 || (long long)nch * K <= kCap);
}

size_t topk_smem_ws(int Nq, long long ld, int K) {
  const int nch = topk_chunks(ld);
  if (nch <= 1) return 0;
  // winners' keys and positions [Nq][nch][K], then counts and K-th keys [Nq][nch]
  const size_t nslot = (size_t)Nq * nch;
  return nslot * (size_t)K * 8 + nslot * 8 + 256;
}

int launch_topk_smem(const TopkParams& p, void* ws, cudaStream_t s) {
  const int nch = topk_chunks(p.ld);
  if (nch == 1) {
    // a row shorter than the cap needs only its own keys in shared memory,
    // so that two CTAs (two rows) share an SM
    const int arc = set_smem_attr<0>();
    if (arc) return arc;
    const size_t smem0 = (size_t)((p.ld + 4 + 3) & ~3LL) * sizeof(uint32_t);
    const cudaError_t e = launch_pdl(k_topk_block<0>, dim3(p.Nq, 1), dim3(kThreads), smem0, s, p,
                                     1, (int)p.ld, (uint32_t*)nullptr, (int32_t*)nullptr,
                                     (int*)nullptr, (uint32_t*)nullptr);
    count_launch();
    if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
    return check_launch("topk");
  }
  // block length: a multiple of 4 keys, so that blocks of a 16-byte aligned
  // row start 16-byte aligned
  const long long blk = ((p.ld + nch - 1) / nch + 3) & ~3LL;
  char* base = (char*)ws + kWsHeader;
  const size_t nslot = (size_t)p.Nq * nch;
  uint32_t* ckey = reinterpret_cast<uint32_t*>(base);
  int32_t* cpos = reinterpret_cast<int32_t*>(base + nslot * p.K * 4);
  int* ccnt = reinterpret_cast<int*>(base + nslot * p.K * 8);
  uint32_t* ckth = reinterpret_cast<uint32_t*>(ccnt + nslot);
  int rc = set_smem_attr<1>();
  if (rc) return rc;
  cudaError_t e = launch_pdl(k_topk_block<1>, dim3(p.Nq, nch), dim3(kThreads),
                             (size_t)(blk + 4) * sizeof(uint32_t), s, p, nch, (int)blk, ckey, cpos,
                             ccnt, ckth);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  rc = check_launch("topk (blocks)");
  if (rc) return rc;
  rc = ensure_dynamic_smem((const void*)k_topk_merge, (kCap + 4) * (int)sizeof(uint32_t),
                           "topk (merge)");
  if (rc) return rc;
  e = launch_pdl(k_topk_merge, dim3(p.Nq), dim3(kThreads),
                 (size_t)((long long)nch * p.K + 4) * sizeof(uint32_t), s, p, nch,
                 (const uint32_t*)ckey, (const int32_t*)cpos, (const int*)ccnt,
                 (const uint32_t*)ckth);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("topk (merge)");
}

}  // namespace dsa
