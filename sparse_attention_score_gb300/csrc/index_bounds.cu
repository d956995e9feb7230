// index_bounds.cu -- block-level bounds of the indexer keys, and the decode
// indexer score that uses them to leave out tiles which cannot reach the
// top-K.
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (3): decode-time index selection is incremental, reusing the
// index structure of earlier steps and computing only what the new position
// needs.  The structure kept here is, per page of the indexer-key cache and
// per key dimension d, the largest and the smallest key over the page's
// cached positions, stored as key codes in kbound[page][0][d] and
// kbound[page][1][d].  A cache write touches only the pages it writes, so
// after a decode step's append one page per sequence is recomputed.
//
// For a query with indexer heads q_h and weights w_h, every cached position
// p of a page satisfies lo_h <= q_h . k_p <= hi_h with
//     hi_h = sum_d max(q_hd kmax_d, q_hd kmin_d),
//     lo_h = sum_d min(q_hd kmax_d, q_hd kmin_d),
// so its score s(p) = sum_h w_h relu(q_h . k_p) is at most
//     UB = sum_h (w_h >= 0 ? w_h relu(hi_h) : w_h relu(lo_h)).
// A 128-position tile is bounded through the union of its two pages' key
// ranges, plus a margin for fp32 rounding (2^-12 of sum_h |w_h| sum_d |q_hd|
// max_d |k_d|, far above the rounding of either sum).
//
// Bounded scoring of one decode query per sequence (the exact top-K of the
// scores it leaves equals that of the full score row):
//   1. the bound of every tile of the query's sequence;
//   2. the M = ceil(K / 128) + 1 tiles with the largest bounds are scored
//      (they hold at least K positions unless the sequence is shorter), and
//      tau = the K-th largest of their scores is at most the K-th largest
//      score of the whole row;
//   3. every other tile whose bound is below tau is left out (scores -inf,
//      keys not read): each of its positions scores below the row's K-th
//      largest, so it is in no top-K and no tie; the remaining tiles are
//      scored.  Both scoring passes are the ordinary indexer kernels with a
//      tile mask, so every score that is computed is the same number.
#include "device_common.cuh"
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kTile = 128;  // positions per tile (two pages of 64)

template <int DT>
__device__ __forceinline__ float key_value(uint16_t code) {
  if (DT == DSA_BF16) return __uint_as_float(((uint32_t)code) << 16);
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

template <int DT>
__device__ __forceinline__ uint16_t load_key(const void* base, long long i) {
  if (DT == DSA_BF16) return __ldg(reinterpret_cast<const uint16_t*>(base) + i);
  return __ldg(reinterpret_cast<const uint8_t*>(base) + i);
}

template <int DT>
__device__ __forceinline__ void store_key(void* base, long long i, uint16_t code) {
  if (DT == DSA_BF16) reinterpret_cast<uint16_t*>(base)[i] = code;
  else reinterpret_cast<uint8_t*>(base)[i] = (uint8_t)code;
}

// One warp per page: the per-dimension largest and smallest key over the
// page's cached positions.  seq == NULL: every page slot of every sequence
// (item = b * maxb + slot); else the page of row i, recomputed by the last
// row of each run of rows in the same page (every touched page at least once).
template <int DT>
__global__ void __launch_bounds__(256) k_bounds_update(LayoutDev lay, const int32_t* seq,
                                                      const int32_t* pos, int N, const void* kidx,
                                                      int D, void* kbound, int* status) {
  grid_dependency_wait();
  launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long nitems = seq ? (long long)N : (long long)lay.batch * lay.maxb;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long it = warp0; it < nitems; it += nwarps) {
    int b;
    long long slot;
    if (seq) {
      b = __ldg(&seq[it]);
      const long long p = __ldg(&pos[it]);
      if (b < 0 || b >= lay.batch || p < 0) continue;
      slot = p / lay.bs;
      if (it + 1 < N) {
        const int b2 = __ldg(&seq[it + 1]);
        const long long p2 = __ldg(&pos[it + 1]);
        if (b2 == b && p2 >= 0 && p2 / lay.bs == slot) continue;  // a later row redoes the page
      }
    } else {
      b = (int)(it / lay.maxb);
      slot = it - (long long)b * lay.maxb;
    }
    long long L = __ldg(&lay.seq_lens[b]);
    const long long cap = (long long)lay.maxb * lay.bs;
    if (L > cap) L = cap;
    if (slot >= lay.maxb || slot * lay.bs >= L) continue;
    const int page = __ldg(&lay.bt[(long long)b * lay.maxb + slot]);
    if (page < 0 || page >= lay.nb) {
      if (lane == 0) flag_status(status, DSA_STATUS_BAD_BLOCK);
      continue;
    }
    const long long nv = L - slot * lay.bs < lay.bs ? L - slot * lay.bs : lay.bs;
    for (int d = lane; d < D; d += 32) {
      float mx = -INFINITY, mn = INFINITY;
      uint16_t cmx = 0, cmn = 0;
      for (long long r = 0; r < nv; ++r) {
        const uint16_t c = load_key<DT>(kidx, ((long long)page * lay.bs + r) * D + d);
        const float v = key_value<DT>(c);
        if (v > mx || r == 0) {
          mx = v;
          cmx = c;
        }
        if (v < mn || r == 0) {
          mn = v;
          cmn = c;
        }
      }
      store_key<DT>(kbound, ((long long)page * 2 + 0) * D + d, cmx);
      store_key<DT>(kbound, ((long long)page * 2 + 1) * D + d, cmn);
    }
  }
}

struct BoundedWs {
  float* ub;        // [B][nt] tile bounds
  int32_t* ntiles;  // [B]
  int32_t* sel;     // [B][M] tiles scored first
  void* ws_sel;
  size_t ws_sel_bytes;
  uint8_t* mask;    // [B][nt]
  float* cand;      // [B][M * 128] their scores
  int32_t* ncand;   // [B]
  int32_t* cidx;    // [B][K]
  void* ws_cand;
  size_t ws_cand_bytes;
  unsigned long long* counters;  // skipped tiles, tiles (in the workspace header)
  size_t total;
};

__host__ __device__ inline size_t r256(size_t n) { return (n + 255) & ~(size_t)255; }

inline int first_tiles(int K) { return (K + kTile - 1) / kTile + 1; }

inline BoundedWs bounded_layout(void* ws, int B, long long ld, int K) {
  BoundedWs w{};
  const long long nt = (ld + kTile - 1) / kTile;
  const int M = first_tiles(K);
  char* base = reinterpret_cast<char*>(ws);
  size_t off = kWsHeader;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off += r256(bytes);
    return p;
  };
  w.ub = reinterpret_cast<float*>(take(sizeof(float) * (size_t)B * nt));
  w.ntiles = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)B));
  w.sel = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)B * M));
  w.ws_sel_bytes = topk_ws(B, nt, M);
  w.ws_sel = take(w.ws_sel_bytes);
  w.mask = reinterpret_cast<uint8_t*>(take((size_t)B * nt));
  w.cand = reinterpret_cast<float*>(take(sizeof(float) * (size_t)B * M * kTile));
  w.ncand = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)B));
  w.cidx = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)B * K));
  w.ws_cand_bytes = topk_ws(B, (long long)M * kTile, K);
  w.ws_cand = take(w.ws_cand_bytes);
  w.counters = base ? reinterpret_cast<unsigned long long*>(base + kBoundedCounters) : nullptr;
  w.total = off;
  return w;
}

// Eligible positions of decode query b (sequence b, all cached positions).
__device__ __forceinline__ long long decode_n(const LayoutDev& lay, long long ld, int b) {
  long long L = __ldg(&lay.seq_lens[b]);
  const long long cap = (long long)lay.maxb * lay.bs;
  if (L > cap) L = cap;
  if (L > ld) L = ld;
  return L > 0 ? L : 0;
}

constexpr int kBoundWarps = 8;       // 256 threads
constexpr int kTilesPerBlock = 16;  // one load of the query's heads per 16 tiles

// grid (ceil(nt / 16), B), 256 threads: warp w bounds tiles 16 blockIdx.x + w
// and + w + 8 of sequence b.  A tile is bounded through the union of its
// pages' key ranges (per dimension the larger maximum and the smaller
// minimum), one bound per tile.  Shared memory: the query's heads transposed
// (q[d][h], consecutive heads adjacent), the weights, sum_d |q_hd| per head,
// and per warp the tile's decoded range.  Per head and dimension the two sums
// are four FMAs over the sign parts of q:
//   hi = q+ . kmax + q- . kmin,  lo = q- . kmax + q+ . kmin;
// the rounding margin is 2^-12 sum_h |w_h| (sum_d |q_hd|) max_d |k_d|.
template <int DT>
__global__ void __launch_bounds__(256)
    k_tile_bounds(IndexParams a, const void* kbound, long long nt, float* ub, int32_t* ntiles,
                  unsigned long long* counters) {
  extern __shared__ float smb[];
  grid_dependency_wait();
  launch_dependents();
  const int H = a.H, D = a.D, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* qT = smb;                     // [D][H]
  float* wsh = qT + D * H;             // [H]
  float* qabs = wsh + H;               // [H]: sum_d |q_hd|
  float* pb = qabs + H + warp * 2 * D; // this warp's tile: kmax [0, D), kmin [D, 2D)
  const long long n = decode_n(a.lay, a.ld, b);
  const long long tiles = (n + kTile - 1) / kTile;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    ntiles[b] = (int32_t)tiles;
    if (b == 0) counters[0] = counters[1] = 0ull;
  }
  // element (h, d) goes to qT[d * H + h]: consecutive threads take
  // consecutive heads, so the shared-memory stores do not collide
  for (int i = threadIdx.x; i < H * D; i += blockDim.x) {
    const int d = i / H, h = i - d * H;
    qT[i] = key_value<DT>(load_key<DT>(a.q_idx, ((long long)b * H + h) * D + d));
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) wsh[h] = __ldg(&a.w[(long long)b * H + h]);
  __syncthreads();
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    float sa = 0.0f;
    for (int d = 0; d < D; ++d) sa += fabsf(qT[d * H + h]);
    qabs[h] = sa;
  }
  __syncthreads();
  for (int k = warp; k < kTilesPerBlock; k += kBoundWarps) {
    const long long t = (long long)blockIdx.x * kTilesPerBlock + k;
    if (t >= nt) break;
    float best = -INFINITY;
    if (t < tiles) {
      bool bad = false;
      float kabs = 0.0f;  // this lane's part of max_d |k_d|
      for (int d = lane; d < D; d += 32) {
        pb[d] = -INFINITY;
        pb[D + d] = INFINITY;
      }
      for (int pg = 0; pg < 2; ++pg) {
        const long long slot = t * 2 + pg;
        if (slot * a.lay.bs >= n) break;
        const int page = __ldg(&a.lay.bt[(long long)b * a.lay.maxb + slot]);
        if (page < 0 || page >= a.lay.nb) {  // the indexer flags it; never leave it out
          bad = true;
          break;
        }
        for (int d = lane; d < D; d += 32) {
          const float kx = key_value<DT>(load_key<DT>(kbound, (long long)page * 2 * D + d));
          const float kn = key_value<DT>(load_key<DT>(kbound, (long long)page * 2 * D + D + d));
          pb[d] = fmaxf(pb[d], kx);
          pb[D + d] = fminf(pb[D + d], kn);
          kabs = fmaxf(kabs, fmaxf(fabsf(kx), fabsf(kn)));
        }
      }
      if (bad) {
        best = INFINITY;
      } else {
        kabs = warp_max(kabs);
        __syncwarp();
        float ubw = 0.0f, absw = 0.0f;
        for (int h = lane; h < H; h += 32) {
          float hi = 0.0f, lo = 0.0f;
#pragma unroll 8
          for (int d = 0; d < D; ++d) {
            const float q = qT[d * H + h];
            const float qp = fmaxf(q, 0.0f), qn = fminf(q, 0.0f);
            const float kx = pb[d], kn = pb[D + d];
            hi = fmaf(qp, kx, fmaf(qn, kn, hi));
            lo = fmaf(qn, kx, fmaf(qp, kn, lo));
          }
          const float wh = wsh[h];
          ubw += wh >= 0.0f ? wh * fmaxf(hi, 0.0f) : wh * fmaxf(lo, 0.0f);
          absw += fabsf(wh) * qabs[h];
        }
        const float u = warp_sum(ubw), m = warp_sum(absw);
        best = u + m * kabs * (1.0f / 4096.0f);
      }
      __syncwarp();
    }
    if (lane == 0) ub[(long long)b * nt + t] = best;
  }
}

// grid B, 256 threads: pass-1 mask: the selected tiles scored, the others
// left as they are.
__global__ void __launch_bounds__(256) k_mask_first(const int32_t* sel, int M, long long nt,
                                                   uint8_t* mask) {
  grid_dependency_wait();
  launch_dependents();
  const int b = blockIdx.x;
  for (long long t = threadIdx.x; t < nt; t += blockDim.x) mask[(long long)b * nt + t] = kSkipKeep;
  __syncthreads();
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    const int t = __ldg(&sel[(long long)b * M + j]);
    if (t >= 0 && t < nt) mask[(long long)b * nt + t] = 0;
  }
}

// grid (M, B), 128 threads: the scores of selected tile j, -inf past the
// sequence or for an empty selection slot.
__global__ void __launch_bounds__(128) k_gather_first(IndexParams a, const int32_t* sel, int M,
                                                     float* cand, int32_t* ncand) {
  grid_dependency_wait();
  launch_dependents();
  const int j = blockIdx.x, b = blockIdx.y;
  const long long n = decode_n(a.lay, a.ld, b);
  const int t = __ldg(&sel[(long long)b * M + j]);
  const long long p = (long long)t * kTile + threadIdx.x;
  float v = -INFINITY;
  if (t >= 0 && p < n) v = a.scores[(long long)b * a.ld + p];
  cand[((long long)b * M + j) * kTile + threadIdx.x] = v;
  if (j == 0 && threadIdx.x == 0) ncand[b] = M * kTile;
}

// grid B, 1024 threads: tau = the K-th largest first-pass score (-inf when
// fewer than K were scored), then the pass-2 mask: tiles scored in pass 1
// kept, the others left out when their bound is below tau, else scored.
__global__ void __launch_bounds__(1024) k_mask_second(const float* cand, const int32_t* cidx, int M,
                                                    int K, const float* ub, const int32_t* ntiles,
                                                    long long nt, uint8_t* mask,
                                                    unsigned long long* counters) {
  __shared__ float red[32];
  __shared__ int redn[32];
  grid_dependency_wait();
  launch_dependents();
  const int b = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float mn = INFINITY;
  int missing = 0;
  for (int j = threadIdx.x; j < K; j += blockDim.x) {
    const int c = __ldg(&cidx[(long long)b * K + j]);
    if (c < 0) missing = 1;
    else mn = fminf(mn, cand[(long long)b * M * kTile + c]);
  }
  mn = warp_min(mn);
  missing = __reduce_or_sync(0xffffffffu, missing);
  if (lane == 0) {
    red[warp] = mn;
    redn[warp] = missing;
  }
  __syncthreads();
  float tau = red[0];
  int miss = redn[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
    tau = fminf(tau, red[w]);
    miss |= redn[w];
  }
  if (miss || tau != tau) tau = -INFINITY;  // fewer than K scored (or NaN): leave nothing out
  const long long tiles = __ldg(&ntiles[b]);
  int skipped = 0;
  for (long long t = threadIdx.x; t < nt; t += blockDim.x) {
    uint8_t m = kSkipKeep;
    if (t < tiles) {
      if (mask[(long long)b * nt + t] == 0) {
        m = kSkipKeep;  // scored in pass 1
      } else if (ub[(long long)b * nt + t] < tau) {
        m = kSkipInf;
        ++skipped;
      } else {
        m = 0;
      }
    }
    mask[(long long)b * nt + t] = m;
  }
  skipped = __reduce_add_sync(0xffffffffu, skipped);
  if (lane == 0 && skipped) atomicAdd(&counters[0], (unsigned long long)skipped);
  if (threadIdx.x == 0) atomicAdd(&counters[1], (unsigned long long)tiles);
}

template <int DT>
int launch_bounds_update(const LayoutDev& lay, const int32_t* seq, const int32_t* pos, int N,
                         const void* kidx, int D, void* kbound, int* status, cudaStream_t s) {
  const long long items = seq ? (long long)N : (long long)lay.batch * lay.maxb;
  if (items <= 0) return DSA_OK;
  long long blocks = (items + 7) / 8;  // 8 warps per block
  const long long cap = 16LL * sm_count();
  if (blocks > cap) blocks = cap;
  k_bounds_update<DT><<<(unsigned)blocks, 256, 0, s>>>(lay, seq, pos, N, kidx, D, kbound, status);
  count_launch();
  return check_launch("index_bounds_update");
}

}  // namespace

int index_bounds_update(const LayoutDev& lay, const int32_t* seq, const int32_t* pos, int N,
                        const void* kidx, int D, int dtype, void* kbound, int* status,
                        cudaStream_t s) {
  if (dtype == DSA_BF16)
    return launch_bounds_update<DSA_BF16>(lay, seq, pos, N, kidx, D, kbound, status, s);
  return launch_bounds_update<DSA_FP8_E4M3>(lay, seq, pos, N, kidx, D, kbound, status, s);
}

size_t index_bounded_ws(int B, long long ld, int K) {
  return bounded_layout(nullptr, B, ld, K).total;
}

int index_score_bounded(IndexParams p, const void* kbound, int K, void* ws, cudaStream_t s) {
  const int B = p.Nq;
  if (B == 0) return DSA_OK;
  const long long nt = (p.ld + kTile - 1) / kTile;
  const int M = first_tiles(K);
  const BoundedWs w = bounded_layout(ws, B, p.ld, K);
  // 1. tile bounds
  {
    const size_t smem =
        sizeof(float) * ((size_t)p.D * p.H + 2 * (size_t)p.H + kBoundWarps * 2 * (size_t)p.D);
    dim3 grid((unsigned)((nt + kTilesPerBlock - 1) / kTilesPerBlock), (unsigned)B);
    if (p.dtype == DSA_BF16) {
      int rc =
          ensure_dynamic_smem((const void*)k_tile_bounds<DSA_BF16>, (int)smem, "index_bounded");
      if (rc) return rc;
      k_tile_bounds<DSA_BF16>
          <<<grid, 32 * kBoundWarps, smem, s>>>(p, kbound, nt, w.ub, w.ntiles, w.counters);
    } else {
      int rc = ensure_dynamic_smem((const void*)k_tile_bounds<DSA_FP8_E4M3>, (int)smem,
                                   "index_bounded");
      if (rc) return rc;
      k_tile_bounds<DSA_FP8_E4M3>
          <<<grid, 32 * kBoundWarps, smem, s>>>(p, kbound, nt, w.ub, w.ntiles, w.counters);
    }
    count_launch();
    int rc = check_launch("index_bounded (tile bounds)");
    if (rc) return rc;
  }
  // 2. the M tiles with the largest bounds, scored first
  {
    TopkParams t{};
    t.scores = w.ub;
    t.ld = nt;
    t.n_elig = w.ntiles;
    t.Nq = B;
    t.K = M;
    t.idx = w.sel;
    t.status = p.status;
    int rc = launch_topk(t, w.ws_sel, w.ws_sel_bytes, s);
    if (rc) return rc;
  }
  k_mask_first<<<B, 256, 0, s>>>(w.sel, M, nt, w.mask);
  count_launch();
  int rc = check_launch("index_bounded (first mask)");
  if (rc) return rc;
  IndexParams p1 = p;
  p1.skip = w.mask;
  p1.skip_stride = nt;
  rc = launch_index_score(p1, s);
  if (rc) return rc;
  // 3. tau from the first tiles, then the rest of the row
  k_gather_first<<<dim3(M, B), kTile, 0, s>>>(p, w.sel, M, w.cand, w.ncand);
  count_launch();
  rc = check_launch("index_bounded (gather)");
  if (rc) return rc;
  {
    TopkParams t{};
    t.scores = w.cand;
    t.ld = (long long)M * kTile;
    t.n_elig = w.ncand;
    t.Nq = B;
    t.K = K;
    t.idx = w.cidx;
    t.status = p.status;
    rc = launch_topk(t, w.ws_cand, w.ws_cand_bytes, s);
    if (rc) return rc;
  }
  k_mask_second<<<B, 1024, 0, s>>>(w.cand, w.cidx, M, K, w.ub, w.ntiles, nt, w.mask, w.counters);
  count_launch();
  rc = check_launch("index_bounded (second mask)");
  if (rc) return rc;
  return launch_index_score(p1, s);
}

}  // namespace dsa
