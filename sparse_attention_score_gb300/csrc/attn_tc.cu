// attn_tc.cu -- tensor-core sparse attention for the latent multi-query cache
// (64 query heads, 576-dim K rows whose first 512 dims are V, bf16).
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (2)-(3) and "Day-0 Adaptation of Ultra-Large-Scale MoE Models on
// Heterogeneous AI Accelerators", section 4 (cache gather + sparse attention):
// every query attends, exactly, over its own selected rows only, gathered from
// the paged cache through the block table.
//
// Work unit: a tile of 64 selected rows of one query.  Per tile:
//   QK  S[128 x 64 rows] = Q[128 x 576] . K_rows[64 x 576]^T    (TMEM, fp32)
//       A = the query's 64 heads as M rows 0-63 (a Q chunk from the ring;
//       M rows 64-127 read whatever follows in shared memory and land in TMEM
//       lanes nobody reads), B = the gathered rows; both K-major in 9 chunks
//       of 64 dims (128-byte swizzle); 36 tcgen05.mma kind::f16 (K = 16).
//       One TMEM lane holds one head, so the softmax is thread-local: thread
//       h keeps head h's running max m (raised only when a tile exceeds it by
//       more than 2^8; O is rescaled in TMEM then) and running sum l.
//       P = 2^(z - m) is split into bf16 hi + lo and l sums hi + lo exactly,
//       so the only rounding left in the output is its final bf16 store.
//   PV  O^T[512 dv x 64 heads] += V^T[512 x 64 rows] . P^T[64 rows x 64]
//       A = V^T (the first 512 dims of the same rows, MN-major), B = P^T
//       (K-major, one 128-byte line per head); 4 blocks of 128 dv, hi and lo.
// The rows of two tiles are resident at once (two buffers), and the MMA warp
// issues QK of tile u before PV of tile u-1: the gathers of the next tile,
// the tensor cores and the softmax of the current tile run at the same time.
// The tiles of all queries are laid end to end and split evenly over one CTA
// per SM.  A query whose tiles span several CTAs leaves one unnormalised
// partial (O, m, l) per CTA in the workspace and a second small kernel merges
// them:  M = max m_s,  l = sum l_s 2^(m_s - M),  O = sum O_s 2^(m_s - M) / l.
//
// Warp roles (320 threads):
//   warps 0-3 softmax (warps 0-1 own the 64 heads; all four rescale O and
//   read it out of TMEM, one TMEM lane quadrant each);
//   warps 4-7 producer: a tile's 9 chunks of 64 rows by 16-byte cp.async
//   into the swizzled layout, 8 consecutive threads per 128-byte row chunk
//   (rows of 1152 bytes anywhere in the pool); each chunk's full barrier is
//   armed by the copies themselves, so the producer never waits for its
//   own loads, only for a slot to be released;
//   warp 8 TMEM owner and MMA issuer; warp 9 streams Q's chunks from L2 by
//   TMA through a six-slot ring.
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
constexpr int kRows = 64;                    // selected rows per tile (MMA N of QK)
constexpr int kChunks = kDqk / 64;           // 9 chunks of 64 dims; the first 8 are V
constexpr int kChunkBytes = kRows * 128;     // 64 rows x 128 B
constexpr int kQRing = 4;                    // Q chunks in flight
constexpr int kQChunkBytes = kHq * 128;      // 8 KB (M rows 0-63 of the A operand)
constexpr int kPBytes = kHq * 128;           // P^T: one 128-byte line (64 rows) per head
constexpr int kThreads = 352;
constexpr int kPrefetchAhead = 3;  // tiles the L2 prefetch runs ahead of the producer
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // two 64-column S buffers (lanes = heads)
constexpr uint32_t kColO = 128;  // four 64-column O^T blocks (lanes = dv)
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxCtas = 160;
constexpr uint32_t kIdescQK = instr_desc(128, kRows, 1, 1, 0, 0);
constexpr uint32_t kIdescPV = instr_desc(128, kHq, 1, 1, 1, 0);
// Chunk order within a tile: chunk 8 (needed by QK only) first, because its
// slot is the first one a tile releases.
__device__ __forceinline__ int chunk_at(int i) { return i == 0 ? 8 : i - 1; }

struct __align__(1024) Smem {
  uint8_t kv[2][kChunks][kChunkBytes];  // two tile buffers
  uint8_t q[kQRing][kQChunkBytes];      // Q chunks streamed from L2
  uint8_t phi[2][kPBytes];              // P^T per tile parity: bf16 part (phi[0]
  uint8_t plo[2][kPBytes];              // is also the M rows 64-127 of the last Q
                                        // slot), bf16 remainder
  uint64_t kfull[2][kChunks], kempty[2][kChunks], qfull[kQRing], qempty[kQRing];
  uint64_t sfull[2], sempty[2], vfull[2], pfull[2], pempty[2], ofull, ofree, smsync, prsync,
      done;
  unsigned long long vmask[2];  // usable rows of the tiles in the two buffers
  int rowtab[kRows];            // physical rows of the producer's current tile
  uint32_t tmem_base;
  int abort;
  int prod_tile;         // tile the producer is on (read by the prefetcher)
  int resc_tile[2];      // last tile (per S buffer) whose softmax raised a max
  float fscale[2][kHq];  // per S buffer: O rescale factor of each head
  float l_inv[kHq];
};

struct Geo {
  int Tq;     // tiles per query (uniform item grid)
  long long total;
  int G;
  long long lo, hi;
  __host__ __device__ long long lo_of(int c) const { return (long long)c * total / G; }
  __host__ __device__ int cta_of(long long x) const {
    int c = (int)(x * G / total);
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
  s.b = a.q_seq ? __ldg(&a.q_seq[r]) : (a.seq0 ? 0 : r);
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
// One arrival on `bar` once every cp.async this thread has issued so far has
// landed; the thread does not wait (the arrival counts toward the barrier's
// expected count).  The consumer makes the data visible to the tensor cores
// with a proxy fence after its wait.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap map_q, AttnParams a, float* part_o,
              float* part_ml) {
  extern __shared__ uint8_t smraw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Geo g;
  g.Tq = (a.K + kRows - 1) / kRows;
  g.total = (long long)a.Nq * g.Tq;
  g.G = gridDim.x;
  g.lo = g.lo_of(blockIdx.x);
  g.hi = g.lo_of(blockIdx.x + 1);
  const int r_first = (int)(g.lo / g.Tq);
  const int r_last = g.hi > g.lo ? (int)((g.hi - 1) / g.Tq) : r_first - 1;
  launch_dependents();

  if (threadIdx.x == 0) {
    sm.abort = 0;
    sm.prod_tile = 0;
    sm.resc_tile[0] = sm.resc_tile[1] = -1;
    for (int b = 0; b < 2; ++b)
      for (int i = 0; i < kChunks; ++i) {
        mbar_init(&sm.kfull[b][i], 128);  // one copy-tracking arrival per producer thread
        mbar_init(&sm.kempty[b][i], 1);
      }
    for (int i = 0; i < kQRing; ++i) {
      mbar_init(&sm.qfull[i], 1);
      mbar_init(&sm.qempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.sfull[i], 1);
      mbar_init(&sm.sempty[i], kHq);
      mbar_init(&sm.vfull[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.pfull[i], 128);
      mbar_init(&sm.pempty[i], 1);
    }
    mbar_init(&sm.ofull, 1);
    mbar_init(&sm.ofree, 128);
    mbar_init(&sm.smsync, 128);
    mbar_init(&sm.prsync, 128);
    mbar_init(&sm.done, 1);
    fence_mbar_init();
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
    // once (threads 0-63: one row each) into a shared table.
    const int pt = threadIdx.x - 128;
    const int gq = pt & 7, r0 = pt >> 3;
    const char* kv = reinterpret_cast<const char*>(a.kp);
    uint32_t ps = 0;
    bool ok = true;
    Walker w;
    w.init(a, g, r_first, r_last);
    int u = 0;
    int p_cur = (w.ok && pt < kRows) ? sel_pos(a, w.s, (long long)w.t * kRows + pt) : -1;
    while (w.ok && ok) {
      const int bufi = u & 1;
      const long long row_cur = pt < kRows ? pos_row(a, w.s, p_cur, false) : -1;
      Walker nx = w;
      nx.next(a, g);
      const int p_next =
          (nx.ok && pt < kRows) ? sel_pos(a, nx.s, (long long)nx.t * kRows + pt) : -1;
      if (!group_sync(&sm.prsync, ps, &sm.abort)) { ok = false; break; }
      if (pt == 0) *(volatile int*)&sm.prod_tile = u;
      if (pt < kRows) sm.rowtab[pt] = (int)row_cur;
      if (!group_sync(&sm.prsync, ps, &sm.abort)) { ok = false; break; }
      int rows[kRows / 16];
#pragma unroll
      for (int k = 0; k < kRows / 16; ++k) rows[k] = sm.rowtab[r0 + 16 * k];
      // usable rows of this tile for the softmax (bit r: row r)
      unsigned long long vmask = 0;
      if (pt < 32) {
        const unsigned lo = __ballot_sync(0xffffffffu, sm.rowtab[pt] >= 0);
        const unsigned hi = __ballot_sync(0xffffffffu, sm.rowtab[pt + 32] >= 0);
        vmask = ((unsigned long long)hi << 32) | lo;
      }
      for (int i = 0; i < kChunks && ok; ++i) {
        const int c = chunk_at(i);
        if (u >= 2 && !warp_wait(&sm.kempty[bufi][c], ((u >> 1) - 1) & 1, &sm.abort)) {
          ok = false;
          break;
        }
        if (i == 1 && pt == 0) {
          // chunk 0's slot is released by the PV of this buffer's previous
          // tile, after the softmax finished with its mask: the mask is free
          sm.vmask[bufi] = vmask;
          mbar_arrive(&sm.vfull[bufi]);
        }
        uint8_t* base = sm.kv[bufi][c];
#pragma unroll
        for (int k = 0; k < kRows / 16; ++k) {
          const int r = r0 + 16 * k;
          const int prow = rows[k];
          const char* src = prow >= 0 ? kv + (size_t)prow * (kDqk * 2) + c * 128 + gq * 16 : kv;
          cp_async16(base + r * 128 + ((gq ^ (r & 7)) << 4), src, prow >= 0 ? 16u : 0u);
        }
        cp_async_arrive(&sm.kfull[bufi][c]);
      }
      p_cur = p_next;
      w = nx;
      ++u;
    }
    cp_async_wait<0>();
    if (!ok) fail(sm, a.status);
  } else if (warp == 10) {
    // --------------------------------------------------------- L2 prefetch --
    // The rows of the next tiles are pulled into L2 (one bulk prefetch per
    // 1152-byte row) a few tiles ahead of the producer, so that its copies,
    // which can only be in flight for one tile buffer, see L2 latency rather
    // than HBM latency under load.  A hint only: on a stall it just stops.
    const char* kv = reinterpret_cast<const char*>(a.kp);
    // the Q rows of this CTA's queries first (contiguous, 64 x 1152 bytes
    // each): every tile streams its query's Q chunks again
    {
      const char* qb = reinterpret_cast<const char*>(a.q);
      const long long qbytes = (long long)kHq * kDqk * 2;
      for (int r = r_first; r <= r_last; ++r)
        for (long long o = (long long)lane * 4096; o < qbytes; o += 32 * 4096) {
          const long long n = qbytes - o < 4096 ? qbytes - o : 4096;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(qb + (size_t)r * qbytes + o),
                       "r"((uint32_t)n)
                       : "memory");
        }
    }
    Walker w;
    w.init(a, g, r_first, r_last);
    int u = 0;
    const uint64_t t0 = globaltimer_ns();
    bool live = true;
    while (w.ok && live) {
      while (u > *(volatile int*)&sm.prod_tile + kPrefetchAhead) {
        if (*(volatile int*)&sm.abort || globaltimer_ns() - t0 > 2000000000ull) {
          live = false;
          break;
        }
        __nanosleep(256);
      }
      if (!live) break;
      for (int j = lane; j < kRows; j += 32) {
        const long long row = pos_row(a, w.s, sel_pos(a, w.s, (long long)w.t * kRows + j), false);
        if (row >= 0) {
          const char* src = kv + (size_t)row * (kDqk * 2);
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(kDqk * 2)
                       : "memory");
        }
      }
      w.next(a, g);
      ++u;
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- Q loader --
    if (lane == 0) {
      Walker w;
      w.init(a, g, r_first, r_last);
      int qs = 0;
      bool ok = true;
      while (w.ok && ok) {
        for (int i = 0; i < kChunks; ++i, ++qs) {
          const int slot = qs % kQRing;
          if (qs >= kQRing && !mbar_wait(&sm.qempty[slot], ((qs / kQRing) - 1) & 1, &sm.abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.qfull[slot], kQChunkBytes);
          tma_load_2d(sm.q[slot], &map_q, &sm.qfull[slot], 64 * chunk_at(i), w.r * kHq);
        }
        w.next(a, g);
      }
      if (!ok) fail(sm, a.status);
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------- MMA issuer --
    // Two cursors, served as their inputs arrive: PV of the oldest tile whose
    // P^T is ready (first: it releases a KV buffer), else the next chunk of
    // QK (up to two tiles ahead).  QK of the next tile thus runs while the
    // softmax of the current one does, and PV never waits for later loads.
    if (lane == 0) {
      struct TileInfo { int seg; bool first, last; };
      TileInfo info[4];
      Walker w;
      w.init(a, g, r_first, r_last);
      int u_qk = 0, i_qk = 0, qs = 0, cur_r = -1, sa = 0, u_pv = 0;
      bool qk_all = !w.ok, ok = true;
      uint64_t t_prog = globaltimer_ns();
      uint32_t spins = 0;
      while (ok && !(qk_all && u_pv == u_qk)) {
        bool prog = false;
        if (u_pv < u_qk) {
          const TileInfo ti = info[u_pv & 3];
          const int pb = u_pv & 1;
          if (mbar_try_wait(&sm.pfull[pb], (u_pv >> 1) & 1) &&
              (!ti.first || ti.seg == 0 || mbar_try_wait(&sm.ofree, (ti.seg - 1) & 1))) {
            tc_fence_after();
            const uint32_t ph = smem_u32(sm.phi[pb]), pl = smem_u32(sm.plo[pb]);
            for (int blk = 0; blk < kDv / 128; ++blk) {
              const uint32_t v0 = smem_u32(sm.kv[pb][2 * blk]);  // chunks 2blk, 2blk+1: 8 KB apart
              const uint32_t d = tbase + kColO + 64 * blk;
#pragma unroll
              for (int k = 0; k < kRows / 16; ++k) {
                const uint64_t va = smem_desc(v0 + 2048 * k, kChunkBytes, 1024, kSwizzle128B);
                mma_f16(d, va, smem_desc(ph + 32 * k, 16, 1024, kSwizzle128B), kIdescPV,
                        (ti.first && k == 0) ? 0u : 1u);
                mma_f16(d, va, smem_desc(pl + 32 * k, 16, 1024, kSwizzle128B), kIdescPV, 1u);
              }
              mma_commit(&sm.kempty[pb][2 * blk]);
              mma_commit(&sm.kempty[pb][2 * blk + 1]);
            }
            mma_commit(&sm.pempty[pb]);
            if (ti.last) mma_commit(&sm.ofull);
            ++u_pv;
            prog = true;
          }
        }
        if (!prog && !qk_all && u_qk < u_pv + 2) {
          const int bufi = u_qk & 1;
          const int c = chunk_at(i_qk), slot = qs % kQRing;
          // S buffer free (the softmax of tile u_qk - 2 has read it), then
          // this chunk's Q and rows
          bool ready = i_qk > 0 || mbar_try_wait(&sm.sempty[bufi], ((u_qk >> 1) & 1) ^ 1);
          ready = ready && mbar_try_wait(&sm.qfull[slot], (qs / kQRing) & 1) &&
                  mbar_try_wait(&sm.kfull[bufi][c], (u_qk >> 1) & 1);
          if (ready) {
            if (i_qk == 0) {
              if (w.r != cur_r) {
                cur_r = w.r;
                ++sa;
              }
              info[u_qk & 3] = TileInfo{sa - 1, w.t == w.s.t0, w.t == w.s.act_end - 1};
            }
            fence_proxy_async_smem();  // the copies' writes, seen by the tensor cores
            tc_fence_after();
            const uint32_t dS = tbase + kColS + 64 * bufi;
            const uint32_t a0 = smem_u32(sm.q[slot]), b0 = smem_u32(sm.kv[bufi][c]);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f16(dS, smem_desc(a0 + 32 * k, 16, 1024, kSwizzle128B),
                      smem_desc(b0 + 32 * k, 16, 1024, kSwizzle128B), kIdescQK,
                      (i_qk + k) > 0 ? 1u : 0u);
            mma_commit(&sm.qempty[slot]);
            if (c == kChunks - 1) mma_commit(&sm.kempty[bufi][c]);  // QK only
            ++qs;
            if (++i_qk == kChunks) {
              mma_commit(&sm.sfull[bufi]);
              i_qk = 0;
              ++u_qk;
              w.next(a, g);
              qk_all = !w.ok;
            }
            prog = true;
          }
        }
        if (prog) {
          spins = 0;
        } else if ((++spins & 255u) == 0) {
          // bounded: give up after 2 s without progress, or when another
          // role has
          const uint64_t now = globaltimer_ns();
          if (spins == 256) t_prog = now;
          if (sm.abort || now - t_prog > 2000000000ull) ok = false;
        }
      }
      if (!ok) fail(sm, a.status);
      mma_commit(&sm.done);
      mbar_wait(&sm.done, 0, &sm.abort, 100000000ull);
    }
  } else {
    // ------------------------------------------------- softmax + finalize --
    // Thread h < 64 (warps 0-1) owns head h: its S row is TMEM lane h.  All
    // four warps take part in rescaling O^T and in reading it out (lane = dv
    // within a 128-dv block).  Loops over 32-column groups stay rolled.
    const int t = threadIdx.x;
    const bool owner = t < kHq;
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
    const float c = a.scale_log2;
    int u = 0, sa = 0;
    uint32_t sp = 0;
    bool ok = true;
    float m = -INFINITY, l = 0.0f;  // running max (log2 units) and sum of head t
    for (int r = r_first; r <= r_last && ok; ++r) {
      const Seg s = make_seg(a, g, r);
      const int pslot = 2 * blockIdx.x + (((long long)r * g.Tq > g.lo) ? 1 : 0);
      float* po = part_o + (size_t)pslot * kHq * kDv;
      float* pml = part_ml + (size_t)pslot * kHq * 2;
      __nv_bfloat16* out = a.out + (size_t)r * kHq * kDv;
      if (s.active() == 0) {
        if (s.complete) {
          for (int i = t; i < kHq * kDv; i += 128) out[i] = __float2bfloat16(0.0f);
          if (a.lse && owner) a.lse[(size_t)r * kHq + t] = -INFINITY;
        } else if (owner) {
          pml[2 * t] = -INFINITY;
          pml[2 * t + 1] = 0.0f;
        }
        continue;
      }
      for (int tt = s.t0; tt < s.act_end; ++tt) {
        const int bufi = u & 1;
        float f = 1.0f;
        unsigned long long vm = 0;
        const uint32_t ta = tbase + lanes + kColS + 64 * bufi;
        if (owner) {
          if (!warp_wait(&sm.sfull[bufi], (u >> 1) & 1, &sm.abort) ||
              !warp_wait(&sm.vfull[bufi], (u >> 1) & 1, &sm.abort)) {
            ok = false;
          } else {
            tc_fence_after();
            vm = sm.vmask[bufi];
            // pass 1: the tile's max for this head
            float mt = -INFINITY;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t raw[32];
              tmem_ld_32cols(ta + 32 * half, raw);
              tmem_wait_ld();
              const unsigned vb = (unsigned)(vm >> (32 * half));
#pragma unroll
              for (int j = 0; j < 32; ++j)
                mt = fmaxf(mt, ((vb >> j) & 1u) ? __uint_as_float(raw[j]) * c : -INFINITY);
            }
            if (mt > m + kRescaleLog2 || (m == -INFINITY && mt > -INFINITY)) {
              if (m > -INFINITY) {
                f = exp2f(m - mt);
                sm.resc_tile[bufi] = u;
              }
              m = mt;
            }
            sm.fscale[bufi][t] = f;
          }
        }
        if (!group_sync(&sm.smsync, sp, &sm.abort) || !ok) { ok = false; break; }
        // fscale and the flag are per S buffer: the next writer of this
        // buffer's entries (tile u + 2) starts only after every thread has
        // passed tile u + 1's barrier
        const bool resc = sm.resc_tile[bufi] == u;
        // O changes only after PV of the previous tile is done (u > 0 here:
        // a segment's first tile never rescales)
        if (resc && !warp_wait(&sm.pempty[bufi ^ 1], ((u - 1) >> 1) & 1, &sm.abort)) {
          ok = false;
          break;
        }
        // this P^T buffer is free once PV of tile u - 2 is done
        if (!warp_wait(&sm.pempty[bufi], ((u >> 1) & 1) ^ 1, &sm.abort)) { ok = false; break; }
        tc_fence_after();
        if (resc) {
#pragma unroll 1
          for (int q = 0; q < 8; ++q) {
            const uint32_t to = tbase + lanes + kColO + 64 * (q >> 1) + 32 * (q & 1);
            uint32_t raw[32];
            tmem_ld_32cols(to, raw);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              raw[i] = __float_as_uint(__uint_as_float(raw[i]) * sm.fscale[bufi][32 * (q & 1) + i]);
            tmem_st_32cols(to, raw);
          }
          tmem_wait_st();
        }
        if (owner) {
          // pass 2: P = 2^(z - m) as bf16 hi + lo, one 128-byte line of P^T
          // per head; l sums exactly what the MMAs multiply.  S is read a
          // second time (it stays in TMEM until sempty).
          float lt = 0.0f;
          uint8_t* rh = sm.phi[bufi] + t * 128;
          uint8_t* rl = sm.plo[bufi] + t * 128;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t raw[32];
            tmem_ld_32cols(ta + 32 * half, raw);
            tmem_wait_ld();
            const unsigned vb = (unsigned)(vm >> (32 * half));
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              // branch-free: an unusable row gives 2^-inf = 0 (a usable row
              // makes the running max finite)
              const float p0 =
                  ex2_approx(((vb >> j) & 1u) ? __uint_as_float(raw[j]) * c - m : -INFINITY);
              const float p1 = ex2_approx(
                  ((vb >> (j + 1)) & 1u) ? __uint_as_float(raw[j + 1]) * c - m : -INFINITY);
              const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
              const float2 hf = __bfloat1622float2(hi);
              const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
              const float2 lf = __bfloat1622float2(lo);
              lt += (hf.x + lf.x) + (hf.y + lf.y);
              hw[j / 2] = *reinterpret_cast<const uint32_t*>(&hi);
              lw[j / 2] = *reinterpret_cast<const uint32_t*>(&lo);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int off = ((4 * half + k) ^ (t & 7)) << 4;
              *reinterpret_cast<uint4*>(rh + off) =
                  make_uint4(hw[4 * k], hw[4 * k + 1], hw[4 * k + 2], hw[4 * k + 3]);
              *reinterpret_cast<uint4*>(rl + off) =
                  make_uint4(lw[4 * k], lw[4 * k + 1], lw[4 * k + 2], lw[4 * k + 3]);
            }
          }
          l = l * f + lt;
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&sm.sempty[bufi]);  // S buffer read for the last time
        }
        tc_fence_before();
        mbar_arrive(&sm.pfull[bufi]);  // all four warps: P^T written and O rescaled
        ++u;
      }
      if (!ok) break;
      // ---- finalize the query segment: O out of TMEM ----
      if (owner) sm.l_inv[t] = l > 0.0f ? 1.0f / l : 0.0f;
      if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }
      if (!warp_wait(&sm.ofull, sa & 1, &sm.abort)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int q = 0; q < 8; ++q) {
        const int blk = q >> 1, half = q & 1;
        uint32_t raw[32];
        tmem_ld_32cols(tbase + lanes + kColO + 64 * blk + 32 * half, raw);
        tmem_wait_ld();
        const int dv = blk * 128 + t;
        if (s.complete) {
          __nv_bfloat16* o = out + (size_t)(32 * half) * kDv + dv;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            o[(size_t)i * kDv] = __float2bfloat16(__uint_as_float(raw[i]) * sm.l_inv[32 * half + i]);
        } else {
          float* o = po + (size_t)(32 * half) * kDv + dv;
#pragma unroll
          for (int i = 0; i < 32; ++i) o[(size_t)i * kDv] = __uint_as_float(raw[i]);
        }
      }
      if (owner) {
        if (s.complete) {
          if (a.lse)
            a.lse[(size_t)r * kHq + t] = l > 0.0f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
        } else {
          pml[2 * t] = m;
          pml[2 * t + 1] = l;
        }
        m = -INFINITY;
        l = 0.0f;
      }
      tc_fence_before();
      mbar_arrive(&sm.ofree);
      if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }  // l_inv reusable
      ++sa;
      ok = ok && !sm.abort;
    }
    if (!ok) fail(sm, a.status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// Merge of the queries whose tiles span several CTAs.  Grid (8 head groups,
// G): CTA column c handles the query that contains the boundary lo(c) when c
// is the first boundary inside that query.
__global__ void __launch_bounds__(256) k_attn_tc_merge(AttnParams a, Geo g, const float* part_o,
                                                       const float* part_ml) {
  grid_dependency_wait();
  launch_dependents();
  const int c = blockIdx.y + 1;
  const long long bnd = g.lo_of(c);
  if (bnd % g.Tq == 0) return;
  const int r = (int)(bnd / g.Tq);
  const long long first = (long long)r * g.Tq;
  if (g.lo_of(c - 1) > first) return;  // an earlier boundary of this query merges it
  const int c0 = g.cta_of(first), c1 = g.cta_of(first + g.Tq - 1);
  const int h0 = blockIdx.x * 8;
  __shared__ float wgt[8][kMaxCtas + 1], lpart[8][kMaxCtas + 1];
  __shared__ float lsum[8], mmax[8];
  const int ns = c1 - c0 + 1;
  // (m, l) of every slot and head of this group, loaded all at once
  for (int i = threadIdx.x; i < ns * 8; i += blockDim.x) {
    const int cc = c0 + i / 8, hh = i % 8;
    const int ps = 2 * cc + ((first > g.lo_of(cc)) ? 1 : 0);
    const float2 ml =
        __ldcg(reinterpret_cast<const float2*>(part_ml + ((size_t)ps * kHq + h0 + hh) * 2));
    wgt[hh][i / 8] = ml.y > 0.0f ? ml.x : -INFINITY;
    lpart[hh][i / 8] = ml.y;
  }
  __syncthreads();
  {
    // warp hh: M = max m_s, weights 2^(m_s - M), L = sum l_s 2^(m_s - M)
    const int hh = threadIdx.x >> 5, ln = threadIdx.x & 31;
    float M = -INFINITY;
    for (int j = ln; j < ns; j += 32) M = fmaxf(M, wgt[hh][j]);
    M = warp_max(M);
    float L = 0.0f;
    for (int j = ln; j < ns; j += 32) {
      const float mj = wgt[hh][j];
      const float w = mj > -INFINITY ? exp2f(mj - M) : 0.0f;
      L += lpart[hh][j] * w;
      wgt[hh][j] = w;
    }
    L = warp_sum(L);
    if (ln == 0) {
      lsum[hh] = L;
      mmax[hh] = M;
    }
  }
  __syncthreads();
  // thread t owns outputs t + 256 k (k < 16): head k/2, dv t + 256 (k & 1);
  // every slot's 16 loads are independent, so they overlap
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
  for (int cc = c0; cc <= c1; ++cc) {
    const int ps = 2 * cc + ((first > g.lo_of(cc)) ? 1 : 0);
    const float* src = part_o + ((size_t)ps * kHq + h0) * kDv + threadIdx.x;
    float val[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) val[k] = __ldcg(src + (size_t)(k >> 1) * kDv + 256 * (k & 1));
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float w = wgt[k >> 1][cc - c0];
      acc[k] = w > 0.0f ? fmaf(w, val[k], acc[k]) : acc[k];
    }
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int hh = k >> 1, dv = threadIdx.x + 256 * (k & 1);
    const float L = lsum[hh];
    a.out[((size_t)r * kHq + h0 + hh) * kDv + dv] = __float2bfloat16(L > 0.0f ? acc[k] / L : 0.0f);
  }
  if (a.lse && threadIdx.x < 8) {
    const float L = lsum[threadIdx.x];
    a.lse[(size_t)r * kHq + h0 + threadIdx.x] =
        L > 0.0f ? (mmax[threadIdx.x] + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
}

}  // namespace

bool attn_tc_eligible(const AttnParams& p) {
  return p.Hq == kHq && p.Dqk == kDqk && p.Dv == kDv && p.kp == p.vp && p.ks == kDqk &&
         p.vs == kDqk && p.Nq >= 1 &&
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
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  Geo g;
  g.Tq = (p.K + kRows - 1) / kRows;
  g.total = (long long)p.Nq * g.Tq;
  long long grid = sm_count();
  if (grid > kMaxCtas) grid = kMaxCtas;
  if (grid > g.total) grid = g.total;
  g.G = (int)grid;
  g.lo = g.hi = 0;
  cudaError_t e =
      launch_pdl(k_attn_tc, dim3((unsigned)grid), dim3(kThreads), smem, s, mq, p, part_o, part_ml);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  rc = check_launch("sparse_attn (tensor cores)");
  if (rc || grid < 2) return rc;
  e = launch_pdl(k_attn_tc_merge, dim3(kHq / 8, (unsigned)(grid - 1)), dim3(256), 0, s, p, g,
                 (const float*)part_o, (const float*)part_ml);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("sparse_attn merge");
}

}  // namespace dsa
