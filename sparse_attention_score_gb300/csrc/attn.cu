// attn.cu -- stage 3 of the DSA path: exact softmax attention over the
// selected positions, their K/V rows gathered through the block table.
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (3) (prefill and decode paths) and "Day-0 Adaptation of
// Ultra-Large-Scale MoE Models on Heterogeneous AI Accelerators", section 4
// (cache gather + sparse attention).  For query r, head h and selected rows j:
//     z_j = sm_scale * q[r][h] . K_j,   out = sum_j softmax(z)_j V_j.
// Softmax runs online in fp32 (log2 domain).  The K selected rows of a query
// may be split into S ranges processed by different CTAs; each writes an
// unnormalised partial (o, m, l) and these are merged:
//     M = max_s m_s,  l = sum_s l_s 2^(m_s - M),  o = sum_s o_s 2^(m_s - M) / l.
// With S <= 8 the S CTAs of a query form one thread-block cluster and merge
// inside the kernel after a cluster barrier (CTA s: heads s, s + S, ...);
// otherwise a combine kernel merges them.  Both merges do the same arithmetic
// in the same order.
//
// This file holds the CUDA-core kernel, used for every shape the tensor-core
// kernel (attn_tc.cu) does not cover.
#include "device_common.cuh"
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kRowChunk = kAttnThreads;  // selected rows looked up per pass
constexpr int kMaxTile = 32;             // rows per K/V tile (one per lane)
constexpr int kSmemLimit = 227 * 1024;   // opt-in shared memory per CTA
constexpr int kMaxSplits = 64;

// 16-byte global -> shared copy; with ok false nothing is read and the
// destination is zero-filled (the source must still be a valid address).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool ok) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
               "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_prev() {  // all groups but the newest done
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 u = __bfloat1622float2(x[i]), v = __bfloat1622float2(y[i]);
    acc = fmaf(u.x, v.x, acc);
    acc = fmaf(u.y, v.y, acc);
  }
  return acc;
}

// Shared memory of k_attn_generic for tiles of T rows.
__host__ __device__ inline size_t generic_smem(int Hq, int Dqk, int Dv, int T) {
  return (size_t)Hq * Dqk * 2 + (size_t)2 * T * ((Dqk + 8) + Dv) * 2 +
         (size_t)kRowChunk * 8 + 2 * kMaxTile * 4;
}

// Merge of head h of query r from its S partials: one warp takes the (m, l)
// of split s in lane s % 32 (S <= 64), then the weights and the denominator
// are shared and every thread combines dims d, d + nthreads, ...  Partials
// written by other CTAs of the kernel are read from L2.
__device__ __forceinline__ void merge_head(const AttnParams& a, int r, int h, int S,
                                           float* wsh, float* lsum_sh, float* mmax_sh) {
  const int Hq = a.Hq, Dv = a.Dv;
  if (threadIdx.x < 32) {  // lane s holds splits s and s + 32
    const int lane = threadIdx.x;
    float ms[2], ls[2];
    float M = -INFINITY;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int s = lane + 32 * u;
      ms[u] = -INFINITY;
      ls[u] = 0.0f;
      if (s < S) {
        const float* pml = a.part_ml + (((long long)r * S + s) * Hq + h) * 2;
        ms[u] = __ldcg(pml);
        ls[u] = __ldcg(pml + 1);
        if (ls[u] > 0.0f) M = fmaxf(M, ms[u]);
      }
    }
    M = warp_max(M);
    float lsum = 0.0f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int s = lane + 32 * u;
      const float wgt = ls[u] > 0.0f ? exp2f(ms[u] - M) : 0.0f;
      if (s < S) wsh[s] = wgt;
      lsum += ls[u] * wgt;
    }
    lsum = warp_sum(lsum);
    if (lane == 0) {
      *lsum_sh = lsum;
      *mmax_sh = M;
    }
  }
  __syncthreads();
  const float lsum = *lsum_sh;
  const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
  for (int d = threadIdx.x; d < Dv; d += blockDim.x) {
    float acc = 0.0f;
    for (int s = 0; s < S; ++s)
      acc = fmaf(wsh[s], __ldcg(&a.part_o[(((long long)r * S + s) * Hq + h) * Dv + d]), acc);
    a.out[((long long)r * Hq + h) * Dv + d] = __float2bfloat16(acc * inv);
  }
  if (a.lse && threadIdx.x == 0)
    a.lse[(long long)r * Hq + h] =
        lsum > 0.0f ? (*mmax_sh + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
  __syncthreads();  // wsh and the sums are rewritten for the next head
}

// The same merge inside the kernel for a cluster of S <= 8 CTAs: CTA `split`
// merges heads split, split + S, ... of query r all at once.  Warp w takes
// the weights of its heads w, w + 8, ... (as merge_head's first warp does);
// then each thread takes one (head, dim) at a time with all S partial values
// loaded before the fma chain, which runs in merge_head's order.  scratch:
// 10 Hq floats of the CTA's dynamic shared memory, free once the tiles are
// done (the kernel's smallest dynamic allocation, 3.3 KB, holds 40 B x 64).
constexpr int kClusterMax = 8;
__device__ __forceinline__ void merge_heads_cluster(const AttnParams& a, int r, int split, int S,
                                                    float* scratch) {
  const int Hq = a.Hq, Dv = a.Dv;
  float* wsh = scratch;                 // [Hq][kClusterMax]
  float* lsum_sh = wsh + Hq * kClusterMax;
  float* mmax_sh = lsum_sh + Hq;
  const int nh = split < Hq ? (Hq - split + S - 1) / S : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int hh = warp; hh < nh; hh += kAttnWarps) {
    const int h = split + hh * S;
    float ms = -INFINITY, ls = 0.0f, M = -INFINITY;
    if (lane < S) {
      const float* pml = a.part_ml + (((long long)r * S + lane) * Hq + h) * 2;
      ms = __ldcg(pml);
      ls = __ldcg(pml + 1);
      if (ls > 0.0f) M = ms;
    }
    M = warp_max(M);
    const float wgt = ls > 0.0f ? exp2f(ms - M) : 0.0f;
    if (lane < S) wsh[hh * kClusterMax + lane] = wgt;
    // merge_head's lane value (its second split, s + 32, is empty here)
    const float lsum = warp_sum(ls * wgt);
    if (lane == 0) {
      lsum_sh[hh] = lsum;
      mmax_sh[hh] = M;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nh * Dv; i += kAttnThreads) {
    const int hh = i / Dv, d = i - hh * Dv, h = split + hh * S;
    float v[kClusterMax];
#pragma unroll
    for (int s = 0; s < kClusterMax; ++s)
      v[s] = s < S ? __ldcg(&a.part_o[(((long long)r * S + s) * Hq + h) * Dv + d]) : 0.0f;
    float acc = 0.0f;
#pragma unroll
    for (int s = 0; s < kClusterMax; ++s)
      if (s < S) acc = fmaf(wsh[hh * kClusterMax + s], v[s], acc);
    const float lsum = lsum_sh[hh];
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
    a.out[((long long)r * Hq + h) * Dv + d] = __float2bfloat16(acc * inv);
    if (a.lse && d == 0)
      a.lse[(long long)r * Hq + h] =
          lsum > 0.0f ? (mmax_sh[hh] + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
  }
}

// grid (S, Nq): CTA (split, r) takes its range of query r's selected rows in
// tiles of T rows.  The page-table lookups of up to 256 rows run at once (one
// thread per row); the K/V rows of tile t+1 are copied (cp.async) while tile
// t is scored.  Warp w owns heads w, w+8, ...: in scoring lane t owns row t of
// the tile, in the P.V product lane l owns output dims 2l, 2l+1, 2l+64, ...
template <int HPW, int DVP>
__global__ void __launch_bounds__(kAttnThreads) k_attn_generic(AttnParams a, int T, int ccs) {
  extern __shared__ __align__(16) unsigned char smraw[];
  const int Hq = a.Hq, Dqk = a.Dqk, Dv = a.Dv;
  const int KS = Dqk + 8;  // padded K row: 16-byte reads of consecutive rows hit distinct banks
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smraw);  // [Hq][Dqk]
  __nv_bfloat16* ksm = qs + (size_t)Hq * Dqk;                   // [2][T][KS]
  __nv_bfloat16* vsm = ksm + (size_t)2 * T * KS;                // [2][T][Dv]
  long long* rows = reinterpret_cast<long long*>(vsm + (size_t)2 * T * Dv);  // [kRowChunk]
  int* valid = reinterpret_cast<int*>(rows + kRowChunk);                     // [2][kMaxTile]
  grid_dependency_wait();
  launch_dependents();

  const int r = blockIdx.y, split = blockIdx.x, S = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = a.q_seq ? __ldg(&a.q_seq[r]) : (a.seq_const >= 0 ? a.seq_const : r);
  const bool b_ok = b >= 0 && b < a.lay.batch;

  for (int i = threadIdx.x; i < Hq * Dqk / 8; i += kAttnThreads)
    reinterpret_cast<uint4*>(qs)[i] =
        __ldg(reinterpret_cast<const uint4*>(a.q + (long long)r * Hq * Dqk) + i);

  const int per = (a.K + S - 1) / S;
  const int j0 = split * per, j1 = min(a.K, j0 + per);
  long long L = b_ok ? (long long)__ldg(&a.lay.seq_lens[b]) : 0;
  if (a.q_pos) {
    const long long qp = (long long)__ldg(&a.q_pos[r]) + 1;  // positions <= q_pos
    if (qp < L) L = qp;
  }

  // rows[t] = physical row of selected entry j0 + c * kRowChunk + t, or -1
  auto lookup = [&](int c) {
    const int j = j0 + c * kRowChunk + threadIdx.x;
    long long row = -1;
    if (j < j1) {
      const int p = __ldg(&a.idx[(long long)r * a.K + j]);
      if (!b_ok) {
        if (j == j0) flag_status(a.status, DSA_STATUS_BAD_INDEX);
      } else if (p >= 0) {
        if (p >= L) {
          flag_status(a.status, DSA_STATUS_BAD_INDEX);
        } else {
          row = phys_row(a.lay.bt, a.lay.maxb, a.lay.bs, a.lay.nb, b, p);
          if (row < 0) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
        }
      }
    }
    rows[threadIdx.x] = row;
  };
  const int kp8 = Dqk >> 3, vp8 = Dv >> 3;
  auto issue = [&](int tt) {
    const int bb = tt & 1, base = (tt * T) % kRowChunk;
    const int nt = min(T, j1 - (j0 + tt * T));
    for (int i = threadIdx.x; i < T * kp8; i += kAttnThreads) {
      const int t = i / kp8, c = i - t * kp8;
      const long long row = t < nt ? rows[base + t] : -1;
      cp_async16(ksm + ((size_t)bb * T + t) * KS + c * 8,
                 row >= 0 ? a.kp + row * a.ks + c * 8 : a.kp, row >= 0);
    }
    for (int i = threadIdx.x; i < T * vp8; i += kAttnThreads) {
      const int t = i / vp8, c = i - t * vp8;
      const long long row = t < nt ? rows[base + t] : -1;
      cp_async16(vsm + ((size_t)bb * T + t) * Dv + c * 8,
                 row >= 0 ? a.vp + row * a.vs + c * 8 : a.vp, row >= 0);
    }
    if (threadIdx.x < T)
      valid[bb * kMaxTile + threadIdx.x] = threadIdx.x < nt && rows[base + threadIdx.x] >= 0;
    cp_async_commit();
  };

  float m[HPW], l[HPW];
  float2 o[HPW][DVP];
#pragma unroll
  for (int i = 0; i < HPW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.0f;  // this lane's share of the sum
#pragma unroll
    for (int k = 0; k < DVP; ++k) o[i][k] = make_float2(0.0f, 0.0f);
  }

  const int ntile = j1 > j0 ? (j1 - j0 + T - 1) / T : 0;
  const int tpc = kRowChunk / T;  // tiles per lookup pass
  if (ntile > 0) {
    lookup(0);
    __syncthreads();
    issue(0);
  }
  for (int tt = 0; tt < ntile; ++tt) {
    if (tt + 1 < ntile) {
      if ((tt + 1) % tpc == 0) {  // rows[] was last read by issue(tt), before the syncs below
        lookup((tt + 1) / tpc);
        __syncthreads();
      }
      issue(tt + 1);
    } else {
      cp_async_commit();  // empty group: wait_group 1 then covers tile tt
    }
    cp_async_wait_prev();
    __syncthreads();

    const int bb = tt & 1;
    const __nv_bfloat16* kt = ksm + (size_t)bb * T * KS;
    const __nv_bfloat16* vt = vsm + (size_t)bb * T * Dv;
    float acc[HPW];
#pragma unroll
    for (int i = 0; i < HPW; ++i) acc[i] = 0.0f;
    const bool rv = lane < T && valid[bb * kMaxTile + lane];
    if (lane < T) {
      const uint4* kr = reinterpret_cast<const uint4*>(kt + (size_t)lane * KS);
      for (int c = 0; c < kp8; ++c) {
        const uint4 kv = kr[c];
#pragma unroll
        for (int i = 0; i < HPW; ++i) {
          const int h = warp + kAttnWarps * i;
          if (h < Hq)
            acc[i] = dot8(reinterpret_cast<const uint4*>(qs + (size_t)h * Dqk)[c], kv, acc[i]);
        }
      }
    }
    float pr[HPW];
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      pr[i] = 0.0f;
      const float z = rv ? acc[i] * a.scale_log2 : -INFINITY;
      const float mt = warp_max(z);
      if (mt == -INFINITY) continue;  // no valid row in this tile (warp-uniform)
      const float mn = fmaxf(m[i], mt);
      const float c = exp2f(m[i] - mn);
      pr[i] = exp2f(z - mn);
      l[i] = l[i] * c + pr[i];
#pragma unroll
      for (int k = 0; k < DVP; ++k) {
        o[i][k].x *= c;
        o[i][k].y *= c;
      }
      m[i] = mn;
    }
    for (int t = 0; t < T; ++t) {
      float2 v[DVP];
#pragma unroll
      for (int k = 0; k < DVP; ++k) {
        const int d = 2 * lane + 64 * k;
        v[k] = d < Dv ? __bfloat1622float2(
                            *reinterpret_cast<const __nv_bfloat162*>(vt + (size_t)t * Dv + d))
                      : make_float2(0.0f, 0.0f);
      }
#pragma unroll
      for (int i = 0; i < HPW; ++i) {
        const float pt = __shfl_sync(0xffffffffu, pr[i], t);
#pragma unroll
        for (int k = 0; k < DVP; ++k) {
          o[i][k].x = fmaf(pt, v[k].x, o[i][k].x);
          o[i][k].y = fmaf(pt, v[k].y, o[i][k].y);
        }
      }
    }
    __syncthreads();  // buffer bb is refilled by issue(tt + 2)
  }

#pragma unroll
  for (int i = 0; i < HPW; ++i) {
    const int h = warp + kAttnWarps * i;
    if (h >= Hq) continue;
    const float lt = warp_sum(l[i]);
    if (S == 1) {
      const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
      __nv_bfloat16* dst = a.out + ((long long)r * Hq + h) * Dv;
#pragma unroll
      for (int k = 0; k < DVP; ++k) {
        const int d = 2 * lane + 64 * k;
        if (d < Dv) {  // two scalar stores: out need only be 2-byte aligned
          dst[d] = __float2bfloat16(o[i][k].x * inv);
          dst[d + 1] = __float2bfloat16(o[i][k].y * inv);
        }
      }
      if (a.lse && lane == 0)
        a.lse[(long long)r * Hq + h] =
            lt > 0.0f ? (m[i] + log2f(lt)) * 0.6931471805599453f : -INFINITY;
    } else {
      float* po = a.part_o + (((long long)r * S + split) * Hq + h) * Dv;
#pragma unroll
      for (int k = 0; k < DVP; ++k) {
        const int d = 2 * lane + 64 * k;
        if (d < Dv) *reinterpret_cast<float2*>(po + d) = o[i][k];
      }
      if (lane == 0) {
        float* pml = a.part_ml + (((long long)r * S + split) * Hq + h) * 2;
        pml[0] = m[i];
        pml[1] = lt;
      }
    }
  }
  if (ccs > 1) {
    // this cluster is query r's S CTAs: every partial is written once all
    // pass the barrier (which also ends this CTA's use of its tile buffers);
    // CTA `split` then merges heads split, split + S, ...
    cluster_sync_all();
    merge_heads_cluster(a, r, split, S, reinterpret_cast<float*>(smraw));
  }
}

// grid (Hq, Nq): merge the S partials of one (query, head).
__global__ void __launch_bounds__(128) k_attn_combine(AttnParams a) {
  grid_dependency_wait();
  launch_dependents();
  __shared__ float wsh[kMaxSplits];
  __shared__ float lsum_sh, mmax_sh;
  merge_head(a, blockIdx.y, blockIdx.x, a.S, wsh, &lsum_sh, &mmax_sh);
}

// Splits of a query's K rows: enough CTAs for two per SM, each at least one
// full tile of rows.
int choose_splits(int Nq, int K) {
  int s = (2 * 152 + Nq - 1) / (Nq > 0 ? Nq : 1);
  int maxs = K / kMaxTile;
  if (maxs < 1) maxs = 1;
  if (s > maxs) s = maxs;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s < 1) s = 1;
  return s;
}

// *merged: the splits were merged inside the kernel (clusters of S <= 8 CTAs,
// every query's cluster resident at once), so no combine launch is needed.
template <int HPW, int DVP>
int launch_generic(const AttnParams& p, cudaStream_t s, bool* merged) {
  auto kern = k_attn_generic<HPW, DVP>;
  int T = kMaxTile;  // largest tile whose double buffer fits
  while (T > 1 && generic_smem(p.Hq, p.Dqk, p.Dv, T) > (size_t)kSmemLimit) T >>= 1;
  const size_t smem = generic_smem(p.Hq, p.Dqk, p.Dv, T);
  const int arc = ensure_dynamic_smem((const void*)kern, (int)smem, "sparse_attn");
  if (arc) return arc;
  *merged = p.S >= 2 && p.S <= kClusterMax &&
            max_active_clusters((const void*)kern, kAttnThreads, smem, p.S) >= p.Nq;
  const cudaError_t e =
      *merged ? launch_pdl_cluster(kern, dim3(p.S, p.Nq), dim3(kAttnThreads), smem, p.S, s, p, T,
                                   p.S)
              : launch_pdl(kern, dim3(p.S, p.Nq), dim3(kAttnThreads), smem, s, p, T, 0);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("sparse_attn");
}

template <int HPW>
int launch_dv(const AttnParams& p, cudaStream_t s, bool* merged) {
  const int dvp = (p.Dv + 63) / 64;  // bf16 pairs per lane
  if (dvp <= 1) return launch_generic<HPW, 1>(p, s, merged);
  if (dvp <= 2) return launch_generic<HPW, 2>(p, s, merged);
  if (dvp <= 4) return launch_generic<HPW, 4>(p, s, merged);
  return launch_generic<HPW, 8>(p, s, merged);
}

}  // namespace

bool attn_supported(int Hq, int Dqk, int Dv) {
  return Hq >= 1 && Hq <= 64 && Dqk >= 8 && Dv >= 8 && Dqk % 8 == 0 && Dv % 8 == 0 &&
         Dv <= 512 && (size_t)Hq * Dqk * 2 + 4 * (Dqk + Dv) <= 200 * 1024;
}

size_t attn_ws(int Nq, int Hq, int Dqk, int Dv, int K, bool) {
  const int S = choose_splits(Nq, K);
  size_t generic = kWsHeader;
  if (S > 1) generic += sizeof(float) * (size_t)Nq * S * Hq * ((size_t)Dv + 2);
  size_t tc = 0;
  if (Hq == 64 && Dqk == 576 && Dv == 512) tc = attn_tc_ws(Nq);
  return generic > tc ? generic : tc;
}

int launch_attn(AttnParams p, bool /*decode*/, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (p.Nq == 0) return DSA_OK;
  if (attn_tc_eligible(p) && ws_bytes >= attn_tc_ws(p.Nq)) return launch_attn_tc(p, ws, s);
  p.S = choose_splits(p.Nq, p.K);
  if (p.S > 1) {
    p.part_o = reinterpret_cast<float*>((char*)ws + kWsHeader);
    p.part_ml = p.part_o + (size_t)p.Nq * p.S * p.Hq * p.Dv;
  }
  const int hpw = (p.Hq + kAttnWarps - 1) / kAttnWarps;
  bool merged = false;
  int rc;
  if (hpw <= 1) rc = launch_dv<1>(p, s, &merged);
  else if (hpw <= 2) rc = launch_dv<2>(p, s, &merged);
  else if (hpw <= 4) rc = launch_dv<4>(p, s, &merged);
  else rc = launch_dv<8>(p, s, &merged);
  if (rc != DSA_OK || p.S == 1 || merged) return rc;
  const cudaError_t e = launch_pdl(k_attn_combine, dim3(p.Hq, p.Nq), dim3(128), 0, s, p);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("sparse_attn combine");
}

}  // namespace dsa
