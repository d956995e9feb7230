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
// The tiles of all queries are laid end to end and split evenly over one CTA
// per SM.  A query whose tiles span several CTAs leaves one unnormalised
// partial (O, m, l) per CTA in the workspace; the CTA that finishes last
// (atomic counter, no waiting) merges them:
//   M = max m_s,  l = sum l_s 2^(m_s - M),  O = sum O_s 2^(m_s - M) / l.
//
// Warp roles (320 threads):
//   warps 0-3 softmax; warps 4-7 epilogue (O out of TMEM, partials, merge);
//   warp 8 producer (TMA: Q, then per tile 9 K chunks and, one tile later, the
//   8 V chunks again, rows gathered four at a time with tile::gather4);
//   warp 9 TMEM owner and MMA issuer.  QK of tile i is issued before PV of
//   tile i-1, so the softmax of one tile overlaps the MMAs of the next.
// Selected rows that are padding, past the sequence, non-causal or behind a
// bad block id are read as zeros (out-of-range TMA rows) and masked to -inf.
// Every wait is bounded (DSA_STATUS_TIMEOUT, then the CTA winds down).
#include "device_common.cuh"
#include "dsa_internal.cuh"
#include "sm100.cuh"

namespace dsa {

namespace {

using namespace sm100;

constexpr int kHq = 64, kDqk = 576, kDv = 512;
constexpr int kRows = 128;
constexpr int kChunkBytes = kRows * 128;     // 64 dims x 128 rows, bf16
constexpr int kPairBytes = 2 * kChunkBytes;  // two chunks at a fixed 16 KB stride
constexpr int kRing = 3;                     // pair slots
constexpr int kQChunks = kDqk / 64;          // 9
constexpr int kQChunkBytes = kHq * 128;      // 8 KB
constexpr int kPBytes = kRows * 128;         // P^T: 64 heads (128 B) per row
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // two 64-column S^T buffers
constexpr uint32_t kColO = 128;  // four 64-column O^T blocks
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxCtas = 160;
constexpr uint32_t kIdescQK = instr_desc(128, kHq, 1, 1, 0, 0);
constexpr uint32_t kIdescPV = instr_desc(128, kHq, 1, 1, 1, 1);

struct __align__(1024) Smem {
  uint8_t q[kQChunks][kQChunkBytes];
  uint8_t ring[kRing][kPairBytes];
  uint8_t pt[2][kPBytes];
  uint64_t qfull, qempty, full[kRing], empty[kRing], sfull[2], sempty[2], pfull[2], pempty[2];
  uint64_t pvdone, ofull, ofree, statfull, statempty, done, smsync, epsync;
  uint32_t tmem_base;
  int abort;
  int rescale[2];
  int combine;
  float redm[4][kHq], reds[4][kHq];
  float m_used[kHq], fscale[kHq], l_run[kHq];
  float stat_m[kHq], stat_l[kHq];
};

struct Geo {
  int Tq;     // tiles per query (uniform item grid)
  long long total;
  int G;
  long long lo, hi;
  __device__ long long lo_of(int c) const { return (long long)c * total / G; }
  __device__ int cta_of(long long x) const {
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

// Physical row of selected entry j of a query, or -1 if it is not usable.
__device__ __forceinline__ long long sel_row(const AttnParams& a, const Seg& s, long long j,
                                             bool flag) {
  if (j >= s.n || s.b < 0) return -1;
  const int p = __ldg(&a.idx[(long long)s.r * a.K + j]);
  if (p < 0) return -1;
  if (p >= s.L || (s.qp >= 0 && p > s.qp)) {
    if (flag) flag_status(a.status, DSA_STATUS_BAD_INDEX);
    return -1;
  }
  const long long row = phys_row(a.lay.bt, a.lay.maxb, a.lay.bs, a.lay.nb, s.b, p);
  if (row < 0 && flag) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
  return row;
}

__device__ __forceinline__ void fail(Smem& sm, int* status) {
  sm.abort = 1;
  flag_status(status, DSA_STATUS_TIMEOUT);
}

// Transposing butterfly over a warp: on entry v[0..63] hold one value per head
// for this lane's row; on exit v[0], v[1] hold the reduction over the 32 lanes
// for heads hb, hb + 1, hb = 32 b4 + 16 b3 + 8 b2 + 4 b1 + 2 b0 (lane bits).
template <bool kMax>
__device__ __forceinline__ void butterfly(float (&v)[kHq], int lane) {
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int o = 16 >> st;
    const int n = kHq >> st;  // live values
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
}

__device__ __forceinline__ int butterfly_head(int lane) {
  return 32 * ((lane >> 4) & 1) + 16 * ((lane >> 3) & 1) + 8 * ((lane >> 2) & 1) +
         4 * ((lane >> 1) & 1) + 2 * (lane & 1);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
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

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_q,
              AttnParams a, float* part_o, float* part_ml, int* counters) {
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
  const int oob_row = a.lay.nb * a.lay.bs;  // read as zeros by TMA

  if (threadIdx.x == 0) {
    sm.abort = 0;
    sm.rescale[0] = sm.rescale[1] = 0;
    mbar_init(&sm.qfull, 1);
    mbar_init(&sm.qempty, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.sfull[i], 1);
      mbar_init(&sm.sempty[i], 128);
      mbar_init(&sm.pfull[i], 128);
      mbar_init(&sm.pempty[i], 1);
    }
    mbar_init(&sm.pvdone, 1);
    mbar_init(&sm.ofull, 1);
    mbar_init(&sm.ofree, 128);
    mbar_init(&sm.statfull, 32);
    mbar_init(&sm.statempty, 128);
    mbar_init(&sm.done, 1);
    mbar_init(&sm.smsync, 128);
    mbar_init(&sm.epsync, 128);
    fence_mbar_init();
  }
  if (threadIdx.x < kHq) {
    sm.m_used[threadIdx.x] = -INFINITY;
    sm.l_run[threadIdx.x] = 0.0f;
  }
  if (warp == 9) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&map_kv);
    tma_prefetch_desc(&map_q);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ producer --
    int slot = 0;
    uint32_t phase = 0;
    int issued = 0, sa = 0;
    uint32_t issued_parity[kRing];
    int rk[4], rv[4];
    bool have_prev = false, ok = true;
    auto load_pairs = [&](int first_chunk, int nchunks, const int (&rows)[4]) -> bool {
      for (int c = first_chunk; c < first_chunk + nchunks; c += 2) {
        const int nc = min(2, first_chunk + nchunks - c);
        bool w = true;
        if (lane == 0) {
          w = mbar_wait(&sm.empty[slot], phase ^ 1, &sm.abort);
          if (w) mbar_arrive_expect_tx(&sm.full[slot], nc * kChunkBytes);
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) return false;
        for (int i = 0; i < nc; ++i)
          tma_gather4(sm.ring[slot] + i * kChunkBytes + lane * 512, &map_kv, &sm.full[slot],
                      64 * (c + i), rows[0], rows[1], rows[2], rows[3]);
        issued_parity[slot] = phase;
        ++issued;
        if (++slot == kRing) {
          slot = 0;
          phase ^= 1;
        }
      }
      return true;
    };
    for (int r = r_first; r <= r_last && ok; ++r) {
      const Seg s = make_seg(a, g, r);
      if (s.active() == 0) continue;
      bool w = true;
      if (lane == 0) {
        if (sa > 0) w = mbar_wait(&sm.qempty, (sa - 1) & 1, &sm.abort);
        if (w) {
          mbar_arrive_expect_tx(&sm.qfull, kQChunks * kQChunkBytes);
          for (int c = 0; c < kQChunks; ++c)
            tma_load_2d(sm.q[c], &map_q, &sm.qfull, 64 * c, r * kHq);
        }
      }
      if (!__shfl_sync(0xffffffffu, w, 0)) {
        ok = false;
        break;
      }
      for (int t = s.t0; t < s.act_end; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const long long row = sel_row(a, s, (long long)t * kRows + lane * 4 + e, false);
          rk[e] = row < 0 ? oob_row : (int)row;
        }
        if (!load_pairs(0, kQChunks, rk)) { ok = false; break; }
        if (have_prev && !load_pairs(0, kDv / 64, rv)) { ok = false; break; }
#pragma unroll
        for (int e = 0; e < 4; ++e) rv[e] = rk[e];
        have_prev = true;
      }
      ++sa;
    }
    if (ok && have_prev) ok = load_pairs(0, kDv / 64, rv);
    if (!ok && lane == 0) fail(sm, a.status);
    if (lane == 0) {
      const int pend = issued < kRing ? issued : kRing;
      for (int i = 0; i < pend; ++i) {
        const int st = (slot - 1 - i + 2 * kRing) % kRing;
        mbar_wait(&sm.full[st], issued_parity[st], &sm.abort, 100000000ull);
      }
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0;
      int u = 0, sa = 0;
      bool ok = true;
      struct Prev { int u, seg; bool first, last; } prev{0, 0, false, false};
      bool have_prev = false;
      auto consume = [&]() -> bool {
        if (!mbar_wait(&sm.full[slot], phase, &sm.abort)) return false;
        tc_fence_after();
        return true;
      };
      auto release = [&]() {
        mma_commit(&sm.empty[slot]);
        if (++slot == kRing) {
          slot = 0;
          phase ^= 1;
        }
      };
      auto do_pv = [&](const Prev& p) -> bool {
        if (!mbar_wait(&sm.pfull[p.u & 1], (p.u >> 1) & 1, &sm.abort)) return false;
        if (p.first && p.seg > 0 && !mbar_wait(&sm.ofree, (p.seg - 1) & 1, &sm.abort)) return false;
        tc_fence_after();
        const uint32_t pt0 = smem_u32(sm.pt[p.u & 1]);
        for (int blk = 0; blk < kDv / 128; ++blk) {
          if (!consume()) return false;
          const uint32_t v0 = smem_u32(sm.ring[slot]);
#pragma unroll
          for (int k = 0; k < kRows / 16; ++k) {
            mma_f16(tbase + kColO + 64 * blk, smem_desc(v0 + 2048 * k, kChunkBytes, 1024, kSwizzle128B),
                    smem_desc(pt0 + 2048 * k, 8192, 1024, kSwizzle128B), kIdescPV,
                    (p.first && k == 0) ? 0u : 1u);
          }
          release();
        }
        mma_commit(&sm.pempty[p.u & 1]);
        mma_commit(&sm.pvdone);
        if (p.last) mma_commit(&sm.ofull);
        return true;
      };
      for (int r = r_first; r <= r_last && ok; ++r) {
        const Seg s = make_seg(a, g, r);
        if (s.active() == 0) continue;
        if (!mbar_wait(&sm.qfull, sa & 1, &sm.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t q0 = smem_u32(sm.q[0]);
        for (int t = s.t0; t < s.act_end; ++t) {
          if (!mbar_wait(&sm.sempty[u & 1], ((u >> 1) & 1) ^ 1, &sm.abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t dS = tbase + kColS + 64 * (u & 1);
          for (int c = 0; c < kQChunks && ok; c += 2) {
            if (!consume()) { ok = false; break; }
            const uint32_t a0 = smem_u32(sm.ring[slot]);
            for (int i = 0; i < 2 && c + i < kQChunks; ++i) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                mma_f16(dS, smem_desc(a0 + i * kChunkBytes + 32 * k, 16, 1024, kSwizzle128B),
                        smem_desc(q0 + (c + i) * kQChunkBytes + 32 * k, 16, 1024, kSwizzle128B),
                        kIdescQK, (c + i + k) > 0 ? 1u : 0u);
              }
            }
            release();
          }
          if (!ok) break;
          mma_commit(&sm.sfull[u & 1]);
          if (t == s.act_end - 1) mma_commit(&sm.qempty);
          if (have_prev && !do_pv(prev)) { ok = false; break; }
          prev = Prev{u, sa, t == s.t0, t == s.act_end - 1};
          have_prev = true;
          ++u;
        }
        ++sa;
      }
      if (ok && have_prev) ok = do_pv(prev);
      if (!ok) fail(sm, a.status);
      mma_commit(&sm.done);
      mbar_wait(&sm.done, 0, &sm.abort, 100000000ull);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------- softmax --
    const int row = threadIdx.x;  // TMEM lane = row of the tile
    const int hb = butterfly_head(lane);
    const float c = a.scale_log2;
    int u = 0, sa = 0;
    uint32_t sp = 0;
    bool ok = true;
    for (int r = r_first; r <= r_last && ok; ++r) {
      const Seg s = make_seg(a, g, r);
      if (s.active() == 0) continue;
      for (int t = s.t0; t < s.act_end; ++t) {
        const bool valid = sel_row(a, s, (long long)t * kRows + row, true) >= 0;
        if (!warp_wait(&sm.sfull[u & 1], (u >> 1) & 1, &sm.abort)) { ok = false; break; }
        tc_fence_after();
        float z[kHq], v[kHq];
        {
          uint32_t raw[32];
          const uint32_t ta = tbase + ((uint32_t)(warp * 32) << 16) + kColS + 64 * (u & 1);
          tmem_ld_32cols(ta, raw);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) z[h] = valid ? __uint_as_float(raw[h]) * c : -INFINITY;
          tmem_ld_32cols(ta + 32, raw);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) z[32 + h] = valid ? __uint_as_float(raw[h]) * c : -INFINITY;
        }
        tc_fence_before();
        mbar_arrive(&sm.sempty[u & 1]);
        // per-head tile max
#pragma unroll
        for (int h = 0; h < kHq; ++h) v[h] = z[h];
        butterfly<true>(v, lane);
        sm.redm[warp][hb] = v[0];
        sm.redm[warp][hb + 1] = v[1];
        if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }
        if (warp == 0) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = hb + e;
            const float mt = fmaxf(fmaxf(sm.redm[0][h], sm.redm[1][h]),
                                   fmaxf(sm.redm[2][h], sm.redm[3][h]));
            const float mo = sm.m_used[h];
            float mn = mo, f = 1.0f;
            if (mt > mo + kRescaleLog2 || (mo == -INFINITY && mt > -INFINITY)) {
              mn = mt;
              if (mo > -INFINITY) {
                f = exp2f(mo - mn);
                sm.rescale[u & 1] = 1;
              }
            }
            sm.m_used[h] = mn;
            sm.fscale[h] = f;
          }
        }
        if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }
        const bool resc = sm.rescale[u & 1] != 0;
        if (threadIdx.x == 0) sm.rescale[(u + 1) & 1] = 0;
#pragma unroll
        for (int h = 0; h < kHq; ++h) {
          const float mu = sm.m_used[h];
          z[h] = (mu == -INFINITY) ? 0.0f : exp2f(z[h] - mu);
        }
        if (resc) {
          // O (tiles before this one) must be complete before it is rescaled
          if (!warp_wait(&sm.pvdone, (u - 1) & 1, &sm.abort)) { ok = false; break; }
          tc_fence_after();
          for (int blk = 0; blk < kDv / 128; ++blk) {
            for (int half = 0; half < 2; ++half) {
              uint32_t raw[32];
              const uint32_t ta = tbase + ((uint32_t)(warp * 32) << 16) + kColO + 64 * blk + 32 * half;
              tmem_ld_32cols(ta, raw);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                raw[i] = __float_as_uint(__uint_as_float(raw[i]) * sm.fscale[32 * half + i]);
              tmem_st_32cols(ta, raw);
            }
          }
          tmem_wait_st();
          tc_fence_before();
        }
        // P^T row: 64 heads as bf16, 128-byte row, 16-byte granules swizzled
        if (!warp_wait(&sm.pempty[u & 1], ((u >> 1) & 1) ^ 1, &sm.abort)) { ok = false; break; }
        {
          uint8_t* prow = sm.pt[u & 1] + row * 128;
#pragma unroll
          for (int gq = 0; gq < 8; ++gq) {
            uint4 pk;
            pk.x = pack_bf16(z[8 * gq + 0], z[8 * gq + 1]);
            pk.y = pack_bf16(z[8 * gq + 2], z[8 * gq + 3]);
            pk.z = pack_bf16(z[8 * gq + 4], z[8 * gq + 5]);
            pk.w = pack_bf16(z[8 * gq + 6], z[8 * gq + 7]);
            *reinterpret_cast<uint4*>(prow + ((gq ^ (row & 7)) << 4)) = pk;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&sm.pfull[u & 1]);
        // per-head tile sum (of the fp32 probabilities)
#pragma unroll
        for (int h = 0; h < kHq; ++h) v[h] = z[h];
        butterfly<false>(v, lane);
        sm.reds[warp][hb] = v[0];
        sm.reds[warp][hb + 1] = v[1];
        if (!group_sync(&sm.smsync, sp, &sm.abort)) { ok = false; break; }
        const bool last = (t == s.act_end - 1);
        if (warp == 0) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = hb + e;
            sm.l_run[h] = sm.l_run[h] * sm.fscale[h] +
                          ((sm.reds[0][h] + sm.reds[1][h]) + (sm.reds[2][h] + sm.reds[3][h]));
          }
          if (last) {
            // hand the segment's statistics to the epilogue, then reset
            if (sa > 0 && !warp_wait(&sm.statempty, (sa - 1) & 1, &sm.abort)) {
              ok = false;
            } else {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int h = hb + e;
                sm.stat_m[h] = sm.m_used[h];
                sm.stat_l[h] = sm.l_run[h];
                sm.m_used[h] = -INFINITY;
                sm.l_run[h] = 0.0f;
              }
              __syncwarp();
              mbar_arrive(&sm.statfull);
            }
          }
        }
        ++u;
      }
      ++sa;
      ok = ok && !sm.abort;
    }
    if (!ok) fail(sm, a.status);
  } else {
    // ------------------------------------------------------------ epilogue --
    const int e = threadIdx.x - 128;  // 0..127
    const int quad = warp - 4;
    int sa = 0;
    uint32_t ep = 0;
    bool ok = true;
    for (int r = r_first; r <= r_last && ok; ++r) {
      const Seg s = make_seg(a, g, r);
      const int pslot = 2 * blockIdx.x + (((long long)r * g.Tq > g.lo) ? 1 : 0);
      float* po = part_o + (size_t)pslot * kHq * kDv;
      float* pml = part_ml + (size_t)pslot * kHq * 2;
      __nv_bfloat16* out = a.out + (size_t)r * kHq * kDv;
      if (s.active() > 0) {
        if (!warp_wait(&sm.ofull, sa & 1, &sm.abort) ||
            !warp_wait(&sm.statfull, sa & 1, &sm.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int blk = 0; blk < kDv / 128; ++blk) {
          const int dv = blk * 128 + quad * 32 + lane;
          for (int half = 0; half < 2; ++half) {
            uint32_t raw[32];
            tmem_ld_32cols(tbase + ((uint32_t)(quad * 32) << 16) + kColO + 64 * blk + 32 * half, raw);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int h = 32 * half + i;
              const float o = __uint_as_float(raw[i]);
              if (s.complete) {
                const float l = sm.stat_l[h];
                out[(size_t)h * kDv + dv] = __float2bfloat16(l > 0.0f ? o / l : 0.0f);
              } else {
                po[(size_t)h * kDv + dv] = o;
              }
            }
          }
        }
        if (e < kHq) {
          const float m = sm.stat_m[e], l = sm.stat_l[e];
          if (s.complete) {
            if (a.lse) a.lse[(size_t)r * kHq + e] =
                l > 0.0f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
          } else {
            pml[2 * e] = m;
            pml[2 * e + 1] = l;
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.ofree);
        mbar_arrive(&sm.statempty);
        ++sa;
      } else {
        if (s.complete) {
          for (int i = e; i < kHq * kDv; i += 128) out[i] = __float2bfloat16(0.0f);
          if (a.lse && e < kHq) a.lse[(size_t)r * kHq + e] = -INFINITY;
        } else if (e < kHq) {
          pml[2 * e] = -INFINITY;
          pml[2 * e + 1] = 0.0f;
        }
      }
      if (!s.complete) {
        // last CTA to finish this query merges the partials
        __threadfence();
        if (!group_sync(&sm.epsync, ep, &sm.abort)) { ok = false; break; }
        const long long first = (long long)r * g.Tq;
        const int c0 = g.cta_of(first), c1 = g.cta_of(first + g.Tq - 1);
        if (e == 0) {
          const int old = atomicAdd(&counters[r], 1);
          sm.combine = (old == c1 - c0) ? 1 : 0;
        }
        if (!group_sync(&sm.epsync, ep, &sm.abort)) { ok = false; break; }
        if (sm.combine) {
          __threadfence();
          float wsum[kHq];
          float mmax[kHq];
#pragma unroll 4
          for (int h = 0; h < kHq; ++h) {
            mmax[h] = -INFINITY;
            wsum[h] = 0.0f;
          }
          for (int cc = c0; cc <= c1; ++cc) {
            const int ps = 2 * cc + ((first > g.lo_of(cc)) ? 1 : 0);
            const float* ml = part_ml + (size_t)ps * kHq * 2;
            for (int h = 0; h < kHq; ++h)
              if (__ldcg(&ml[2 * h + 1]) > 0.0f) mmax[h] = fmaxf(mmax[h], __ldcg(&ml[2 * h]));
          }
          for (int cc = c0; cc <= c1; ++cc) {
            const int ps = 2 * cc + ((first > g.lo_of(cc)) ? 1 : 0);
            const float* ml = part_ml + (size_t)ps * kHq * 2;
            for (int h = 0; h < kHq; ++h) {
              const float l = __ldcg(&ml[2 * h + 1]);
              if (l > 0.0f) wsum[h] += l * exp2f(__ldcg(&ml[2 * h]) - mmax[h]);
            }
          }
          for (int dv = e; dv < kDv; dv += 128) {
            for (int h = 0; h < kHq; ++h) {
              float acc = 0.0f;
              for (int cc = c0; cc <= c1; ++cc) {
                const int ps = 2 * cc + ((first > g.lo_of(cc)) ? 1 : 0);
                const float l = __ldcg(&part_ml[((size_t)ps * kHq + h) * 2 + 1]);
                if (l > 0.0f) {
                  const float wgt = exp2f(__ldcg(&part_ml[((size_t)ps * kHq + h) * 2]) - mmax[h]);
                  acc = fmaf(wgt, __ldcg(&part_o[((size_t)ps * kHq + h) * kDv + dv]), acc);
                }
              }
              out[(size_t)h * kDv + dv] =
                  __float2bfloat16(wsum[h] > 0.0f ? acc / wsum[h] : 0.0f);
            }
          }
          if (a.lse && e < kHq)
            a.lse[(size_t)r * kHq + e] =
                wsum[e] > 0.0f ? (mmax[e] + log2f(wsum[e])) * 0.6931471805599453f : -INFINITY;
          if (!group_sync(&sm.epsync, ep, &sm.abort)) { ok = false; break; }
          if (e == 0) counters[r] = 0;
        }
      }
      ok = ok && !sm.abort;
    }
    if (!ok) fail(sm, a.status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

bool attn_tc_eligible(const AttnParams& p) {
  return p.Hq == kHq && p.Dqk == kDqk && p.Dv == kDv && p.kp == p.vp && p.ks == kDqk &&
         p.vs == kDqk && p.Nq >= 1 &&
         (long long)p.lay.nb * p.lay.bs < (1LL << 31) - 1;
}

size_t attn_tc_ws(int Nq) {
  const size_t counters = (((size_t)Nq * sizeof(int)) + 255) & ~size_t(255);
  return kWsHeader + counters + sizeof(float) * 2 * kMaxCtas * kHq * (kDv + 2);
}

int launch_attn_tc(const AttnParams& p, void* ws, cudaStream_t s) {
  CUtensorMap mkv, mq;
  int rc = make_tmap_2d(&mkv, p.kp, false, kDqk, (uint64_t)p.lay.nb * p.lay.bs, kDqk * 2, 64, 1);
  if (rc) return rc;
  rc = make_tmap_2d(&mq, p.q, false, kDqk, (uint64_t)p.Nq * kHq, kDqk * 2, 64, kHq);
  if (rc) return rc;
  int* counters = reinterpret_cast<int*>((char*)ws + kWsHeader);
  const size_t cbytes = (((size_t)p.Nq * sizeof(int)) + 255) & ~size_t(255);
  float* part_ml = reinterpret_cast<float*>((char*)ws + kWsHeader + cbytes);
  float* part_o = part_ml + (size_t)2 * kMaxCtas * kHq * 2;
  const size_t smem = sizeof(Smem) + 1024;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  const long long total = (long long)p.Nq * ((p.K + kRows - 1) / kRows);
  long long grid = sm_count();
  if (grid > kMaxCtas) grid = kMaxCtas;
  if (grid > total) grid = total;
  k_attn_tc<<<(unsigned)grid, kThreads, smem, s>>>(mkv, mq, p, part_o, part_ml, counters);
  count_launch();
  return check_launch("sparse_attn (tensor cores)");
}

}  // namespace dsa
