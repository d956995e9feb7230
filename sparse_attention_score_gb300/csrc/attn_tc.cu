// attn_tc.cu -- tensor-core sparse attention for the latent multi-query cache
// (64 query heads, 576-dim K rows whose first 512 dims are V, bf16).
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (2)-(3) and "Day-0 Adaptation of Ultra-Large-Scale MoE Models on
// Heterogeneous AI Accelerators", section 4 (cache gather + sparse attention):
// every query attends, exactly, over its own selected rows only, gathered from
// the paged cache through the block table.
//
// Work unit: a tile of 128 selected rows of one query.  Per tile:
//   QK  S^T[128 rows x 64 heads] = K_rows[128 x 576] . Q^T      (TMEM, fp32)
//       A = gathered rows, K-major, 9 chunks of 64 dims (128-byte swizzle);
//       B = the query's 64 heads, K-major; 36 tcgen05.mma kind::f16, K = 16.
//   softmax (4 warps, one TMEM lane = one row per thread): per-head tile max
//       by a transposing butterfly over the warp plus a 4-warp exchange;
//       running max kept per head, raised only when a tile exceeds it by more
//       than 2^8, in which case O is rescaled in TMEM; P = 2^(z - m) in bf16.
//   PV  O^T[512 dv x 64 heads] += V^T[512 x 128 rows] . P^T[128 rows x 64]
//       A = V^T (the first 512 dims of the same rows, MN-major), B = P^T
//       (MN-major, one 128-byte row per KV row); 4 blocks of 128 dv.
// P is rounded to bf16 once for the PV MMA when the query has more than
// kSplitRows usable rows; the softmax denominators sum the fp32 values, so
// each weight of the output's average of V rows is within 2^-9 (relative) of
// its exact value and lse keeps fp32 accuracy.  A query with fewer rows has a
// peaked softmax and an output close to a few single V rows, so there P is
// kept as bf16 hi + lo (two PV passes, the remainder written over the bf16
// part once the first pass has read it) and the output is exact up to its
// final bf16 store.
// The tiles of all queries are laid end to end and split evenly over one CTA
// per SM.  A query whose tiles span several CTAs leaves one unnormalised
// partial (O, m, l) per CTA in the workspace and these are merged:
// M = max m_s,  l = sum l_s 2^(m_s - M),  O = sum O_s 2^(m_s - M) / l.
// When every query is split evenly over two or four CTAs (a decode batch: 16
// tiles per query over four CTAs of four), those CTAs form one thread-block
// cluster: after a cluster barrier each CTA merges its share of the query's
// dv from the partials in L2.  Otherwise a second small kernel merges them.
//
// Warp roles (448 threads):
//   warps 0-3 and 10-13 softmax, and at the end of each query segment O out
//   of TMEM: two warps per TMEM lane quadrant, one for heads 0-31 and one for
//   heads 32-63, which halves the softmax's share of the per-tile chain;
//   warps 4-7 producer: the tile's 9 chunks of 128 rows by 16-byte cp.async
//   into the 128-byte swizzled layout, 8 consecutive threads per 128-byte
//   row chunk (rows of 1152 bytes anywhere in the pool); the tile stays
//   resident from QK to PV, each chunk slot refilled for the next tile as
//   soon as its last MMA is done (chunks 0-7 after their PV block, chunk 8,
//   needed by QK only and taken last, after the PV: from the softmax to the
//   PV its slot holds P^T);
//   warp 8 TMEM owner and MMA issuer; warp 9 loads the query's Q (72 KB) by
//   TMA once per query, resident while the CTA works on that query.
// Selected rows that are padding, past the sequence, non-causal or behind a
// bad block id are copied as zeros and masked to -inf.
// Every wait is bounded (DSA_STATUS_TIMEOUT, then the CTA winds down).
#include "device_common.cuh"
#include "dsa_internal.cuh"
#include "sm100.cuh"

namespace dsa {

namespace {

using namespace sm100;

constexpr int kHq = 64, kDqk = 576, kDv = 512;
constexpr int kRows = 128;
constexpr int kChunks = kDqk / 64;           // 9 K chunks of 64 dims; the first 8 are V
constexpr int kChunkBytes = kRows * 128;     // 64 dims x 128 rows, bf16
constexpr int kCopyLag = 2;                  // producer: copy groups in flight before an arrival
constexpr int kQChunkBytes = kHq * 128;      // 8 KB
constexpr int kThreads = 448;         // softmax 0-3 + 10-13, producer 4-7, MMA 8, Q loader 9
constexpr int kSoftmaxThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // two 64-column S^T buffers
constexpr uint32_t kColO = 128;  // four 64-column O^T blocks
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kSplitRows = 512;  // queries with at most this many rows: P as hi + lo
constexpr int kMaxCtas = 160;
constexpr uint32_t kIdescQK = instr_desc(128, kHq, 1, 1, 0, 0);
constexpr uint32_t kIdescPV = instr_desc(128, kHq, 1, 1, 1, 1);
constexpr int kPSlot = kChunks - 1;  // chunk 8 (QK only): its slot holds P^T from softmax to PV
constexpr int kMergeBatch = 4;  // partial slots read per round trip by a merge

struct __align__(1024) Smem {
  // the tile's rows, chunks 0-7 resident from QK to PV; once QK is done,
  // chunk 8's slot holds P^T (one 128-byte row of 64 bf16 heads per row)
  uint8_t kv[kChunks][kChunkBytes];
  uint8_t q[kChunks][kQChunkBytes];  // the current query's Q, loaded once per query
  uint64_t kfull[kChunks], kempty[kChunks], qfull, qempty, phidone, plofull;
  uint64_t sfull[2], sempty[2], pfull, pempty, ofull, ofree, smsync, prsync, done, vfull[2];
  int rowtab[kRows];     // physical rows of the producer's current tile
  int valid[2][kRows];   // usable rows of tiles u (slot u % 2), for the softmax
  uint32_t tmem_base;
  int abort;
  int rescale[3], slow[3];  // per tile u: slot u % 3
  float redm[4][kHq], reds[4][kHq];
  float m_used[kHq], fscale[kHq], l_run[kHq], l_inv[kHq];
};

static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory of k_attn_tc");

struct Geo {
  int Tq;     // tiles per query (uniform item grid)
  long long total;
  int G;
  long long lo, hi;
  // 32-bit divisions whenever the products fit (every workload here): a
  // 64-bit division is a long instruction sequence on the GPU.
  __host__ __device__ long long lo_of(int c) const {
    const unsigned long long p = (unsigned long long)c * (unsigned long long)total;
    if (p < (1ull << 32)) return (long long)((uint32_t)p / (uint32_t)G);
    return (long long)(p / (unsigned long long)G);
  }
  // tile index x -> query index (x / Tq)
  __host__ __device__ long long query_of(long long x) const {
    return x < (1ll << 32) ? (long long)((uint32_t)x / (uint32_t)Tq) : x / Tq;
  }
  __host__ __device__ int cta_of(long long x) const {
    const unsigned long long p = (unsigned long long)x * (unsigned long long)G;
    int c = (p < (1ull << 32) && total < (1ll << 32)) ? (int)((uint32_t)p / (uint32_t)total)
                                                      : (int)(p / (unsigned long long)total);
    while (c + 1 < G && lo_of(c + 1) <= x) ++c;
    while (c > 0 && lo_of(c) > x) --c;
    return c;
  }
};

struct Seg {
  int r;
  int t0, t1;   // items [t0, t1) of query r in this CTA
  int act_end;  // active tiles are [t0, act_end)
  long long n;  // valid rows of query r
  int b;
  long long L;  // sequence length (clamped)
  long long qp; // causal bound (inclusive), or -1
  bool complete;
  __device__ int active() const { return act_end > t0 ? act_end - t0 : 0; }
};

__device__ __forceinline__ Seg make_seg(const AttnParams& a, const Geo& g, int r) {
  Seg s;
  s.r = r;
  const long long base = (long long)r * g.Tq;
  s.t0 = (int)(g.lo > base ? g.lo - base : 0);
  s.t1 = (int)min((long long)g.Tq, g.hi - base);
  s.complete = (s.t0 == 0 && s.t1 == g.Tq);
  s.b = a.q_seq ? __ldg(&a.q_seq[r]) : (a.seq_const >= 0 ? a.seq_const : r);
  s.n = 0;
  s.L = 0;
  s.qp = -1;
  if (s.b >= 0 && s.b < a.lay.batch) {
    long long L = __ldg(&a.lay.seq_lens[s.b]);
    const long long cap = (long long)a.lay.maxb * a.lay.bs;
    if (L > cap) L = cap;
    if (L < 0) L = 0;
    s.L = L;
    long long n = a.K < L ? a.K : L;
    if (a.q_pos) {
      s.qp = __ldg(&a.q_pos[r]);
      if (s.qp + 1 < n) n = s.qp + 1 > 0 ? s.qp + 1 : 0;
    }
    s.n = n;
  } else {
    s.b = -1;
  }
  const int act = (int)((s.n + kRows - 1) / kRows);
  s.act_end = min(s.t1, act);
  return s;
}

// Selected position of entry j of a query (-1: none / padding).
__device__ __forceinline__ int sel_pos(const AttnParams& a, const Seg& s, long long j) {
  if (j >= s.n || s.b < 0) return -1;
  return __ldg(&a.idx[(long long)s.r * a.K + j]);
}

// Physical row of a selected position, or -1 if it is not usable.
__device__ __forceinline__ long long pos_row(const AttnParams& a, const Seg& s, int p, bool flag) {
  if (p < 0) return -1;
  if (p >= s.L || (s.qp >= 0 && p > s.qp)) {
    if (flag) flag_status(a.status, DSA_STATUS_BAD_INDEX);
    return -1;
  }
  const long long row = phys_row(a.lay.bt, a.lay.maxb, a.lay.bs, a.lay.nb, s.b, p);
  if (row < 0 && flag) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
  return row;
}

// Active tiles of this CTA in order (segments without active tiles skipped).
struct Walker {
  int r, r_last, t;
  Seg s;
  bool ok;
  __device__ void settle(const AttnParams& a, const Geo& g) {
    while (ok && t >= s.act_end) {
      if (++r > r_last) { ok = false; break; }
      s = make_seg(a, g, r);
      t = s.t0;
    }
  }
  __device__ void init(const AttnParams& a, const Geo& g, int r0, int r1) {
    r = r0;
    r_last = r1;
    ok = r0 <= r1;
    if (ok) {
      s = make_seg(a, g, r);
      t = s.t0;
      settle(a, g);
    }
  }
  __device__ void next(const AttnParams& a, const Geo& g) {
    ++t;
    settle(a, g);
  }
};

__device__ __forceinline__ void fail(Smem& sm, int* status) {
  sm.abort = 1;
  flag_status(status, DSA_STATUS_TIMEOUT);
}

// Transposing butterfly over a warp: on entry v[0..31] hold one value per
// column for this lane's row; returns, in lane l, the reduction over the 32
// lanes (rows) of column l.  31 shuffles for 32 columns.
template <bool kMax>
__device__ __forceinline__ float butterfly32(float (&v)[32], int lane) {
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int o = 16 >> st;
    const int n = 32 >> st;  // live values
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// Barrier among the 128 threads of one warp group, built on an mbarrier so
// that it is bounded like every other wait (a plain bar.sync would block
// forever if a sibling warp had given up).
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, volatile int* abort) {
  mbar_arrive(bar);
  const bool ok = warp_wait(bar, phase, abort);
  phase ^= 1;
  return ok;
}

// 16-byte asynchronous global -> shared copy; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Merge of the cluster's query, this CTA's share of its dv, from the CS
// partial slots 2 c (c = the cluster's CTAs, in order), with the arithmetic
// and order of k_attn_tc_merge (one round of CS <= kMergeBatch slots), so the
// output is the same bit for bit.  Thread st: head st / 4; its (m, l) pairs
// are read once and each of its two rounds has all 16 float4 loads in flight.
// The share's float4 k * 4 + st % 4 of the head belong to the thread, so four
// neighbouring threads read 64 contiguous bytes.
template <int CS>
__device__ __forceinline__ void merge_cluster_share(const AttnParams& a, const Geo& g,
                                                    const float* part_o, const float* part_ml,
                                                    int st) {
  static_assert(CS >= 2 && CS <= kMergeBatch, "one merge round");
  constexpr int kN4 = kDv / CS / 4;   // float4 of the share per head
  constexpr int kPer = kN4 / 4;       // of them per thread
  constexpr int kRound = 16 / CS;     // per thread per round: 16 loads in flight
  const int rank = (int)(blockIdx.x % (unsigned)CS);
  const int c0 = (int)blockIdx.x - rank;
  const int r = (int)g.query_of(g.lo_of(c0));
  const int h = st >> 2, part = st & 3;
  const int dv0 = rank * (kDv / CS);
  float2 ml[CS];
#pragma unroll
  for (int j = 0; j < CS; ++j)
    ml[j] = __ldcg(reinterpret_cast<const float2*>(part_ml + ((size_t)2 * (c0 + j) * kHq + h) * 2));
  float M = -INFINITY;
#pragma unroll
  for (int j = 0; j < CS; ++j)
    if (ml[j].y > 0.0f) M = fmaxf(M, ml[j].x);
  float w[CS], L = 0.0f;
#pragma unroll
  for (int j = 0; j < CS; ++j) {
    w[j] = (M > -INFINITY && ml[j].y > 0.0f) ? exp2f(ml[j].x - M) : 0.0f;
    if (M > -INFINITY && ml[j].y > 0.0f) L = fmaf(ml[j].y, w[j], L);
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  __nv_bfloat16* o = a.out + ((size_t)r * kHq + h) * kDv + dv0;
#pragma unroll
  for (int k0 = 0; k0 < kPer; k0 += kRound) {
    float4 v[CS][kRound];
#pragma unroll
    for (int j = 0; j < CS; ++j)
#pragma unroll
      for (int k = 0; k < kRound; ++k)
        v[j][k] = __ldcg(reinterpret_cast<const float4*>(
                             part_o + ((size_t)2 * (c0 + j) * kHq + h) * kDv + dv0) +
                         (k0 + k) * 4 + part);
#pragma unroll
    for (int k = 0; k < kRound; ++k) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < CS; ++j) {
        if (M > -INFINITY && ml[j].y > 0.0f) {
          acc.x = fmaf(w[j], v[j][k].x, acc.x); acc.y = fmaf(w[j], v[j][k].y, acc.y);
          acc.z = fmaf(w[j], v[j][k].z, acc.z); acc.w = fmaf(w[j], v[j][k].w, acc.w);
        }
      }
      __nv_bfloat162 p0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(o + 4 * ((k0 + k) * 4 + part)) =
          make_uint2(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1));
    }
  }
  if (a.lse && rank == 0 && part == 0)
    a.lse[(size_t)r * kHq + h] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap map_q, AttnParams a, float* part_o,
              float* part_ml, int ccs) {
  extern __shared__ uint8_t smraw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Geo g;
  g.Tq = (a.K + kRows - 1) / kRows;
  g.total = (long long)a.Nq * g.Tq;
  g.G = gridDim.x;
  g.lo = g.lo_of(blockIdx.x);
  g.hi = g.lo_of(blockIdx.x + 1);
  const int r_first = (int)g.query_of(g.lo);
  const int r_last = g.hi > g.lo ? (int)g.query_of(g.hi - 1) : r_first - 1;
  launch_dependents();

  if (threadIdx.x == 0) {
    sm.abort = 0;
    for (int i = 0; i < 3; ++i) sm.rescale[i] = sm.slow[i] = 0;
    for (int i = 0; i < kChunks; ++i) {
      mbar_init(&sm.kfull[i], 128);
      mbar_init(&sm.kempty[i], 1);
    }
    mbar_init(&sm.qfull, 1);
    mbar_init(&sm.qempty, 1);
    mbar_init(&sm.phidone, 1);
    mbar_init(&sm.plofull, kSoftmaxThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.sfull[i], 1);
      mbar_init(&sm.sempty[i], kSoftmaxThreads);
    }
    mbar_init(&sm.pfull, kSoftmaxThreads);
    mbar_init(&sm.pempty, 1);
    mbar_init(&sm.ofull, 1);
    mbar_init(&sm.ofree, kSoftmaxThreads);
    mbar_init(&sm.smsync, kSoftmaxThreads);
    mbar_init(&sm.prsync, 128);
    mbar_init(&sm.done, 1);
    mbar_init(&sm.vfull[0], 128);
    mbar_init(&sm.vfull[1], 128);
    fence_mbar_init();
  }
  if (threadIdx.x < kHq) {
    sm.m_used[threadIdx.x] = -INFINITY;
    sm.l_run[threadIdx.x] = 0.0f;
    sm.fscale[threadIdx.x] = 1.0f;
  }
  if (warp == 8) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 9 && lane == 0) tma_prefetch_desc(&map_q);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  grid_dependency_wait();  // everything below reads inputs of earlier kernels

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ producer --
    // Each 128-byte row chunk is copied by 8 consecutive threads (16 B each),
    // so a warp instruction moves four whole rows; thread t copies granule
    // t % 8 of rows t / 8 + 16 i.  The tile's physical rows are looked up
    // once (thread t: row t) into a shared table, and each thread keeps its
    // eight rows in registers for the tile's nine chunks (a shared-memory
    // load issued behind pending copies waits for them).  Every slot is
    // refilled as soon as it is released.  Completion is tracked by copy
    // groups: cp.async.mbarrier.arrive.noinc arrivals were measured to cap
    // one SM's copies at about a third of the rate of groups.
    const int pt = threadIdx.x - 128;
    const int gq = pt & 7, r0 = pt >> 3;
    const char* kv = reinterpret_cast<const char*>(a.kp);
    uint32_t ps = 0;
    bool ok = true;
    Walker w;
    w.init(a, g, r_first, r_last);
    int u = 0;
    int p_cur = w.ok ? sel_pos(a, w.s, (long long)w.t * kRows + pt) : -1;
    while (w.ok && ok) {
      const long long row_cur = pos_row(a, w.s, p_cur, true);
      Walker nx = w;
      nx.next(a, g);
      const int p_next = nx.ok ? sel_pos(a, nx.s, (long long)nx.t * kRows + pt) : -1;
      if (!group_sync(&sm.prsync, ps, &sm.abort)) { ok = false; break; }
      sm.rowtab[pt] = (int)row_cur;
      // The softmax of tile u reads valid[u % 2]; the slot is written again
      // for tile u + 2 only after this producer has passed the slot waits of
      // tile u + 1, i.e. after PV(u), which follows that softmax.
      sm.valid[u & 1][pt] = row_cur >= 0 ? 1 : 0;
      mbar_arrive(&sm.vfull[u & 1]);
      if (!group_sync(&sm.prsync, ps, &sm.abort)) { ok = false; break; }
      int prows[kRows / 16];
#pragma unroll
      for (int k = 0; k < kRows / 16; ++k) prows[k] = sm.rowtab[r0 + 16 * k];
      // One copy group per chunk; chunk i's full barrier gets one plain
      // arrival per thread once its group has landed, checked when chunk
      // i + 2 has been issued (and for the last two at the end of the tile).
      // Every slot wait of this tile depends only on the previous tile's
      // chunks, all of which have been arrived, so the lag cannot deadlock.
#pragma unroll 1
      for (int i = 0; i < kChunks && ok; ++i) {
        const int c = i;
        if (u > 0 && !warp_wait(&sm.kempty[c], (u - 1) & 1, &sm.abort)) { ok = false; break; }
        uint8_t* base = sm.kv[c];
#pragma unroll
        for (int k = 0; k < kRows / 16; ++k) {
          const int r = r0 + 16 * k;
          const int prow = prows[k];
          const char* src = prow >= 0 ? kv + (size_t)prow * (kDqk * 2) + c * 128 + gq * 16 : kv;
          cp_async16(base + r * 128 + ((gq ^ (r & 7)) << 4), src, prow >= 0 ? 16u : 0u);
        }
        cp_async_commit();
        if (i >= kCopyLag) {
          cp_async_wait<kCopyLag>();
          mbar_arrive(&sm.kfull[i - kCopyLag]);
        }
      }
      if (!ok) break;
      cp_async_wait<0>();
#pragma unroll
      for (int i = kChunks - kCopyLag; i < kChunks; ++i) mbar_arrive(&sm.kfull[i]);
      p_cur = p_next;
      w = nx;
      ++u;
    }
    cp_async_wait<0>();
    if (!ok) fail(sm, a.status);
  } else if (warp == 9) {
    // ----------------------------------------------------------- Q loader --
    if (lane == 0) {
      Walker w;
      w.init(a, g, r_first, r_last);
      int nq = 0, cur = -1;
      bool ok = true;
      while (w.ok && ok) {
        if (w.r != cur) {  // a new query: its Q replaces the previous one's after its last QK
          cur = w.r;
          if (nq > 0 && !mbar_wait(&sm.qempty, (nq - 1) & 1, &sm.abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.qfull, kChunks * kQChunkBytes);
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(sm.q[c], &map_q, &sm.qfull, 64 * c, w.r * kHq);
          ++nq;
        }
        w.next(a, g);
      }
      if (!ok) fail(sm, a.status);
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int u = 0, sa = 0, ns = 0, cur_r = -1;  // ns: tiles with P as hi + lo so far
      bool ok = true;
      Walker w;
      w.init(a, g, r_first, r_last);
      while (w.ok && ok) {
        const bool first = (w.t == w.s.t0), last = (w.t == w.s.act_end - 1);
        if (w.r != cur_r) {
          cur_r = w.r;
          ++sa;
          if (!mbar_wait(&sm.qfull, (sa - 1) & 1, &sm.abort)) { ok = false; break; }
        }
        if (!mbar_wait(&sm.sempty[u & 1], ((u >> 1) & 1) ^ 1, &sm.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dS = tbase + kColS + 64 * (u & 1);
        for (int c = 0; c < kChunks; ++c) {
          if (!mbar_wait(&sm.kfull[c], u & 1, &sm.abort)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // the copies' writes, seen by the tensor cores
          tc_fence_after();
          const uint32_t a0 = smem_u32(sm.kv[c]), b0 = smem_u32(sm.q[c]);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16(dS, smem_desc(a0 + 32 * k, 16, 1024, kSwizzle128B),
                    smem_desc(b0 + 32 * k, 16, 1024, kSwizzle128B), kIdescQK,
                    (c + k) > 0 ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(&sm.sfull[u & 1]);
        if (last) mma_commit(&sm.qempty);  // this query's Q is read for the last time
        // PV of this tile once the softmax has written P^T (into chunk 8's slot)
        if (!mbar_wait(&sm.pfull, u & 1, &sm.abort)) { ok = false; break; }
        if (first && sa > 1 && !mbar_wait(&sm.ofree, (sa - 2) & 1, &sm.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t pt = smem_u32(sm.kv[kPSlot]);
        const bool split = w.s.n <= kSplitRows;
        // split: the bf16 part first, then (once the softmax has written it
        // over the first) the remainder, releasing the V chunks
        for (int pass = split ? 0 : 1; pass < 2 && ok; ++pass) {
          if (pass == 1 && split) {
            mma_commit(&sm.phidone);
            if (!mbar_wait(&sm.plofull, ns & 1, &sm.abort)) { ok = false; break; }
            tc_fence_after();
            ++ns;
          }
          for (int blk = 0; blk < kDv / 128; ++blk) {
            const uint32_t v0 = smem_u32(sm.kv[2 * blk]);  // chunks 2blk, 2blk+1 are 16 KB apart
            const uint32_t d = tbase + kColO + 64 * blk;
#pragma unroll
            for (int k = 0; k < kRows / 16; ++k)
              mma_f16(d, smem_desc(v0 + 2048 * k, kChunkBytes, 1024, kSwizzle128B),
                      smem_desc(pt + 2048 * k, 8192, 1024, kSwizzle128B), kIdescPV,
                      (first && k == 0 && pass == (split ? 0 : 1)) ? 0u : 1u);
            if (pass == 1) {
              mma_commit(&sm.kempty[2 * blk]);
              mma_commit(&sm.kempty[2 * blk + 1]);
            }
          }
        }
        if (!ok) break;
        mma_commit(&sm.kempty[kPSlot]);  // P^T read: chunk 8's slot may take the next tile
        mma_commit(&sm.pempty);
        if (last) mma_commit(&sm.ofull);
        ++u;
        w.next(a, g);
      }
      if (!ok) fail(sm, a.status);
      mma_commit(&sm.done);
      mbar_wait(&sm.done, 0, &sm.abort, 100000000ull);
    }
  } else {
    // ------------------------------------------------- softmax + finalize --
    // Thread = TMEM lane = row of the tile (and dv lane of O at the end).
    // Two warps per TMEM lane quadrant: warps 0-3 take the heads 0-31 (the
    // first 32 columns of S and of each O block), warps 10-13 heads 32-63.
    const int quad = warp & 3;
    const int half = warp >= 10 ? 1 : 0;
    const int row = quad * 32 + lane;
    const uint32_t lanes = (uint32_t)(quad * 32) << 16;
    const float c = a.scale_log2;
    int u = 0, sa = 0, ns = 0;  // ns: tiles with P as hi + lo so far
    uint32_t sp = 0;
    bool ok = true;
    for (int r = r_first; r <= r_last && ok; ++r) {
      const Seg s = make_seg(a, g, r);
      const int pslot = 2 * blockIdx.x + (((long long)r * g.Tq > g.lo) ? 1 : 0);
      float* po = part_o + (size_t)pslot * kHq * kDv;
      float* pml = part_ml + (size_t)pslot * kHq * 2;
      __nv_bfloat16* out = a.out + (size_t)r * kHq * kDv;
      if (s.active() == 0) {
        if (s.complete) {
          for (int i = row + 128 * half; i < kHq * kDv; i += 256) out[i] = __float2bfloat16(0.0f);
          if (a.lse && half == 0 && row < kHq) a.lse[(size_t)r * kHq + row] = -INFINITY;
        } else if (half == 0 && row < kHq) {
          pml[2 * row] = -INFINITY;
          pml[2 * row + 1] = 0.0f;
        }
        continue;
      }
      // lane l of this warp accumulates, over the warp's 32 rows of every
      // tile, the softmax denominator of head 32 * half + l
      float l_acc = 0.0f;
      for (int t = s.t0; t < s.act_end; ++t) {
        // usable rows of the tile, as the producer looked them up
        if (!warp_wait(&sm.vfull[u & 1], (u >> 1) & 1, &sm.abort)) { ok = false; break; }
        const bool valid = sm.valid[u & 1][row] != 0;
        if (!warp_wait(&sm.sfull[u & 1], (u >> 1) & 1, &sm.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t ta = tbase + lanes + kColS + 64 * (u & 1);
        float z[32];  // scores of this row for the warp's 32 heads, log2 units
        {
          uint32_t raw[32];
          tmem_ld_32cols(ta + 32 * half, raw);
          tmem_wait_ld();
          bool exc = false;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            z[i] = valid ? __uint_as_float(raw[i]) * c : -INFINITY;
            // a head's running max is raised only when a score exceeds it by
            // more than 2^8 (the first usable row of a query always does)
            exc |= z[i] > sm.m_used[32 * half + i] + kRescaleLog2;
          }
          if (__any_sync(0xffffffffu, exc) && lane == 0) atomicOr(&sm.slow[u % 3], 1);
        }
        // slot (u + 1) % 3 was last read in tile u - 2, before every thread
        // arrived at tile u - 1's barrier; it is set again in tile u + 1,
        // after this thread's arrival at tile u's barrier
        if (half == 0 && row == 0) {
          sm.slow[(u + 1) % 3] = 0;
          sm.rescale[(u + 1) % 3] = 0;
        }
        if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }
        const bool slow = sm.slow[u % 3] != 0;
        bool resc = false;
        if (slow) {
          // per-head maximum of the tile over all 128 rows, then the new
          // running maxima and their rescale factors (thread h: head h)
          // (the butterfly consumes z; it is read again from TMEM below, so
          // that the rare path holds no second copy of the row in registers)
          sm.redm[quad][32 * half + lane] = butterfly32<true>(z, lane);
          if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }
          if (half == 0 && row < kHq) {
            const int h = row;
            const float mt = fmaxf(fmaxf(sm.redm[0][h], sm.redm[1][h]),
                                   fmaxf(sm.redm[2][h], sm.redm[3][h]));
            const float mo = sm.m_used[h];
            float mn = mo, f = 1.0f;
            if (mt > mo + kRescaleLog2 || (mo == -INFINITY && mt > -INFINITY)) {
              mn = mt;
              if (mo > -INFINITY) {
                f = exp2f(mo - mn);
                sm.rescale[u % 3] = 1;
              }
            }
            sm.m_used[h] = mn;
            sm.fscale[h] = f;
          }
          if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }
          resc = sm.rescale[u % 3] != 0;
          l_acc *= sm.fscale[32 * half + lane];
          uint32_t raw[32];
          tmem_ld_32cols(ta + 32 * half, raw);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = valid ? __uint_as_float(raw[i]) * c : -INFINITY;
        }
        // the previous PV must be done before P^T (and, if needed, O) change
        if (!warp_wait(&sm.pempty, (u & 1) ^ 1, &sm.abort)) { ok = false; break; }
        tc_fence_after();
        if (resc) {
#pragma unroll 1
          for (int q = half; q < 8; q += 2) {
            const uint32_t to = tbase + lanes + kColO + 64 * (q >> 1) + 32 * (q & 1);
            uint32_t raw[32];
            tmem_ld_32cols(to, raw);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              raw[i] = __float_as_uint(__uint_as_float(raw[i]) * sm.fscale[32 * (q & 1) + i]);
            tmem_st_32cols(to, raw);
          }
          tmem_wait_st();
        }
        // P = 2^(z - m) in bf16 (hi + lo for short queries) into this row of
        // P^T; the denominators add the fp32 values
        const bool split = s.n <= kSplitRows;
        uint8_t* rp = sm.kv[kPSlot] + row * 128;  // QK is done with chunk 8 (sfull)
        uint32_t lw[16];
        {
          float v[32];
          uint32_t hw[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            // branch-free: an unusable row gives 2^-inf = 0 (a usable row makes
            // every head's running max finite)
            const float m0 = sm.m_used[32 * half + i], m1 = sm.m_used[32 * half + i + 1];
            const float p0 = ex2_approx(valid ? z[i] - m0 : -INFINITY);
            const float p1 = ex2_approx(valid ? z[i + 1] - m1 : -INFINITY);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
            const float2 hf = __bfloat1622float2(hi);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
            v[i] = p0;
            v[i + 1] = p1;
            hw[i / 2] = *reinterpret_cast<const uint32_t*>(&hi);
            lw[i / 2] = *reinterpret_cast<const uint32_t*>(&lo);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int off = ((4 * half + k) ^ (row & 7)) << 4;
            *reinterpret_cast<uint4*>(rp + off) =
                make_uint4(hw[4 * k], hw[4 * k + 1], hw[4 * k + 2], hw[4 * k + 3]);
          }
          l_acc += butterfly32<false>(v, lane);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.sempty[u & 1]);
        mbar_arrive(&sm.pfull);
        if (split) {
          // the remainder, over the bf16 part once the PV has read that
          if (!warp_wait(&sm.phidone, ns & 1, &sm.abort)) { ok = false; break; }
          ++ns;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int off = ((4 * half + k) ^ (row & 7)) << 4;
            *reinterpret_cast<uint4*>(rp + off) =
                make_uint4(lw[4 * k], lw[4 * k + 1], lw[4 * k + 2], lw[4 * k + 3]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&sm.plofull);
        }
        ++u;
      }
      if (!ok) break;
      // ---- finalize the query segment: O out of TMEM ----
      sm.reds[quad][32 * half + lane] = l_acc;
      if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }  // all partial sums
      if (half == 0 && row < kHq) {
        const int h = row;
        const float l = (sm.reds[0][h] + sm.reds[1][h]) + (sm.reds[2][h] + sm.reds[3][h]);
        sm.l_run[h] = l;
        sm.l_inv[h] = l > 0.0f ? 1.0f / l : 0.0f;
      }
      if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }  // l_run final
      if (!warp_wait(&sm.ofull, sa & 1, &sm.abort)) { ok = false; break; }
      tc_fence_after();
      // this warp's 32 heads' 1 / l, read once for the four dv blocks
      float inv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) inv[i] = s.complete ? sm.l_inv[32 * half + i] : 0.0f;
#pragma unroll 1
      for (int q = half; q < 8; q += 2) {
        const int blk = q >> 1;
        uint32_t raw[32];
        tmem_ld_32cols(tbase + lanes + kColO + 64 * blk + 32 * half, raw);
        tmem_wait_ld();
        const int dv = blk * 128 + row;
        if (s.complete) {
          __nv_bfloat16* o = out + (size_t)(32 * half) * kDv + dv;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            o[(size_t)i * kDv] = __float2bfloat16(__uint_as_float(raw[i]) * inv[i]);
        } else {
          float* o = po + (size_t)(32 * half) * kDv + dv;
#pragma unroll
          for (int i = 0; i < 32; ++i) o[(size_t)i * kDv] = __uint_as_float(raw[i]);
        }
      }
      if (half == 0 && row < kHq) {
        const float m = sm.m_used[row], l = sm.l_run[row];
        if (s.complete) {
          if (a.lse)
            a.lse[(size_t)r * kHq + row] =
                l > 0.0f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
        } else {
          pml[2 * row] = m;
          pml[2 * row + 1] = l;
        }
        // head h's statistics are read by thread h only; reset them before
        // the barrier after which the next query's first tile reads m_used
        sm.m_used[row] = -INFINITY;
        sm.l_run[row] = 0.0f;
        sm.fscale[row] = 1.0f;
      }
      tc_fence_before();
      mbar_arrive(&sm.ofree);
      if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }  // stats read, reset
      ++sa;
      ok = ok && !sm.abort;
    }
    if (!ok) fail(sm, a.status);
  }

  if (ccs > 1) {
    // every query split over this cluster's CTAs: all partials written, then
    // each CTA merges its share (the softmax warps' 256 threads)
    cluster_sync_all();
    if (warp < 4 || warp >= 10) {
      const int st = (warp < 4 ? warp : warp - 6) * 32 + lane;
      if (ccs == 2)
        merge_cluster_share<2>(a, g, part_o, part_ml, st);
      else
        merge_cluster_share<4>(a, g, part_o, part_ml, st);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// Merge of the queries whose tiles span several CTAs.  Grid (16 head groups,
// Y): with by_query, row y is query y (skipped when it lies inside one CTA);
// otherwise row y is CTA boundary y + 1, which handles the query containing
// it when it is the first boundary inside that query.  The first form is
// used when there are fewer queries than boundaries, so that no block of the
// grid is idle.  Each thread owns two float4 of dv for one of the group's 4
// heads and reads, for up to kMergeBatch slots at a time, the slot's (m, l)
// and its two partial float4 in one go: a query split over at most
// kMergeBatch CTAs (a decode query over four CTAs of four tiles) is merged
// after a single round trip.  Slots beyond the first batch are folded in with
// a running maximum.  Four slots per batch keep the kernel at 80 registers,
// three blocks per SM.
constexpr int kMergeHeads = 4;

__global__ void __launch_bounds__(256) k_attn_tc_merge(AttnParams a, Geo g, const float* part_o,
                                                       const float* part_ml, int by_query) {
  grid_dependency_wait();
  launch_dependents();
  int r;
  long long first;
  if (by_query) {
    r = blockIdx.y;
    first = (long long)r * g.Tq;
  } else {
    const int c = blockIdx.y + 1;
    const long long bnd = g.lo_of(c);
    r = (int)g.query_of(bnd);
    first = (long long)r * g.Tq;
    if (bnd == first) return;
    if (g.lo_of(c - 1) > first) return;  // an earlier boundary of this query merges it
  }
  const int c0 = g.cta_of(first), c1 = g.cta_of(first + g.Tq - 1);
  if (c1 == c0) return;  // not split: the attention kernel wrote this query
  const int ns = c1 - c0 + 1;
  const int h = blockIdx.x * kMergeHeads + (threadIdx.x >> 6);  // 64 threads per head
  const int q4 = threadIdx.x & 63;                               // float4 q4 and q4 + 64 of dv
  float M = -INFINITY, L = 0.0f;
  float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
  for (int j0 = 0; j0 < ns; j0 += kMergeBatch) {
    const int nb = min(kMergeBatch, ns - j0);
    float2 ml[kMergeBatch];
    float4 v0[kMergeBatch], v1[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      if (j < nb) {
        const int cc = c0 + j0 + j;
        const int ps = 2 * cc + ((first > g.lo_of(cc)) ? 1 : 0);
        ml[j] = __ldcg(reinterpret_cast<const float2*>(part_ml + ((size_t)ps * kHq + h) * 2));
        const float4* src =
            reinterpret_cast<const float4*>(part_o + ((size_t)ps * kHq + h) * kDv) + q4;
        v0[j] = __ldcg(src);
        v1[j] = __ldcg(src + 64);
      }
    }
    float Mb = M;
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      if (j < nb && ml[j].y > 0.0f) Mb = fmaxf(Mb, ml[j].x);
    if (Mb == -INFINITY) continue;
    const float f = M > -INFINITY ? exp2f(M - Mb) : 0.0f;
    L *= f;
    acc0.x *= f; acc0.y *= f; acc0.z *= f; acc0.w *= f;
    acc1.x *= f; acc1.y *= f; acc1.z *= f; acc1.w *= f;
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      if (j < nb && ml[j].y > 0.0f) {
        const float w = exp2f(ml[j].x - Mb);
        L = fmaf(ml[j].y, w, L);
        acc0.x = fmaf(w, v0[j].x, acc0.x); acc0.y = fmaf(w, v0[j].y, acc0.y);
        acc0.z = fmaf(w, v0[j].z, acc0.z); acc0.w = fmaf(w, v0[j].w, acc0.w);
        acc1.x = fmaf(w, v1[j].x, acc1.x); acc1.y = fmaf(w, v1[j].y, acc1.y);
        acc1.z = fmaf(w, v1[j].z, acc1.z); acc1.w = fmaf(w, v1[j].w, acc1.w);
      }
    }
    M = Mb;
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  __nv_bfloat16* o = a.out + ((size_t)r * kHq + h) * kDv + 4 * q4;
  __nv_bfloat162 p[4] = {__floats2bfloat162_rn(acc0.x * inv, acc0.y * inv),
                         __floats2bfloat162_rn(acc0.z * inv, acc0.w * inv),
                         __floats2bfloat162_rn(acc1.x * inv, acc1.y * inv),
                         __floats2bfloat162_rn(acc1.z * inv, acc1.w * inv)};
  *reinterpret_cast<uint2*>(o) = make_uint2(*reinterpret_cast<uint32_t*>(&p[0]),
                                            *reinterpret_cast<uint32_t*>(&p[1]));
  *reinterpret_cast<uint2*>(o + 256) = make_uint2(*reinterpret_cast<uint32_t*>(&p[2]),
                                                  *reinterpret_cast<uint32_t*>(&p[3]));
  if (a.lse && q4 == 0)
    a.lse[(size_t)r * kHq + h] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

bool attn_tc_eligible(const AttnParams& p) {
  // the merge stores four bf16 at a time: out must be 8-byte aligned
  return p.Hq == kHq && p.Dqk == kDqk && p.Dv == kDv && p.kp == p.vp && p.ks == kDqk &&
         p.vs == kDqk && p.Nq >= 1 && ((uintptr_t)p.out & 7u) == 0 &&
         (long long)p.lay.nb * p.lay.bs < (1LL << 31) - 1;
}

size_t attn_tc_ws(int) {
  return kWsHeader + sizeof(float) * 2 * kMaxCtas * kHq * (kDv + 2);
}

int launch_attn_tc(const AttnParams& p, void* ws, cudaStream_t s) {
  CUtensorMap mq;
  int rc = make_tmap_2d(&mq, p.q, false, kDqk, (uint64_t)p.Nq * kHq, kDqk * 2, 64, kHq);
  if (rc) return rc;
  float* part_ml = reinterpret_cast<float*>((char*)ws + kWsHeader);
  float* part_o = part_ml + (size_t)2 * kMaxCtas * kHq * 2;
  const size_t smem = sizeof(Smem) + 1024;
  rc = ensure_dynamic_smem((const void*)k_attn_tc, (int)smem, "sparse_attn (tensor cores)");
  if (rc) return rc;
  Geo g;
  g.Tq = (p.K + kRows - 1) / kRows;
  g.total = (long long)p.Nq * g.Tq;
  long long grid = sm_count();
  if (grid > kMaxCtas) grid = kMaxCtas;
  if (grid > g.total) grid = g.total;
  // As few CTAs as give every CTA the same largest share: with 512 tiles on
  // 152 SMs some CTA takes 4 tiles either way, and 128 CTAs of exactly 4 keep
  // each CTA inside one query (one finalize, fewer partials to merge).
  const long long per = (g.total + grid - 1) / grid;
  grid = (g.total + per - 1) / per;
  g.G = (int)grid;
  g.lo = g.hi = 0;
  // every query on exactly cs whole CTAs (2 or 4), all clusters resident at
  // once: the merge runs inside the attention kernel
  int ccs = 0;
  if (grid >= 2 && grid * per == g.total && g.Tq % per == 0) {
    const int cs = (int)(g.Tq / per);
    if ((cs == 2 || cs == 4) &&
        (long long)max_active_clusters((const void*)k_attn_tc, kThreads, smem, cs) * cs >= grid)
      ccs = cs;
  }
  cudaError_t e;
  if (ccs) {
    e = launch_pdl_cluster(k_attn_tc, dim3((unsigned)grid), dim3(kThreads), smem, ccs, s, mq, p,
                           part_o, part_ml, ccs);
  } else {
    e = launch_pdl(k_attn_tc, dim3((unsigned)grid), dim3(kThreads), smem, s, mq, p, part_o,
                   part_ml, 0);
  }
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  rc = check_launch("sparse_attn (tensor cores)");
  if (rc || grid < 2 || ccs) return rc;
  const int by_query = p.Nq <= grid - 1 ? 1 : 0;
  e = launch_pdl(k_attn_tc_merge,
                 dim3(kHq / kMergeHeads, (unsigned)(by_query ? p.Nq : grid - 1)), dim3(256), 0, s,
                 p, g, (const float*)part_o, (const float*)part_ml, by_query);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("sparse_attn merge");
}

}  // namespace dsa
