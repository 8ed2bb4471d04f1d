// topk_em.cu -- the M-step of approximate top-k EM (the "GMMXX" README's
// training option approx_top_k: every point keeps only its k largest
// component logits in the E-step and its responsibilities are normalised over
// those k; k >= K is exact EM), on the EM step of "Flash-GMM: A
// Memory-Efficient Kernel for Scalable Soft Clustering", section 2.
//
// The E-step is the top-m pass (m = k): per point the k largest
// responsibilities r_ij (normalised over all K) and their components c_ij.
// Normalising over the kept k is a division by the row sum, since
// r_ij / sum_j r_ij = exp(l_ij) / sum_j exp(l_ij).  The statistics are then
// sparse: point i adds to k components only.  They are gathered, not
// scattered, so that every sum has one fixed order:
//   1. tk_count:  a stable counting sort of the N k (point, component) pairs
//                 by component.  Points are cut into tiles of kTkTile; one
//                 warp walks one tile in point order and counts its pairs
//                 per component (counts[c][t]).
//   2. tk_scan:   per component, the exclusive prefix over tiles; the total.
//   3. tk_base:   the exclusive prefix over components (pair offsets) and the
//                 chunking of every component's pairs into runs of kTkChunk.
//   4. tk_fill:   the warp of each tile walks it again and writes every pair
//                 (point, normalised responsibility) to its slot: within a
//                 component, pairs are ordered by point index.
//   5. tk_stats:  one CTA per chunk (a run of one component's pairs), one
//                 thread per feature: pass 1 sums r and r x, pass 2 sums
//                 r (x - mu')^2 with the new mean (the two-pass variance).
//   6. tk_final:  one CTA per component sums its chunks in order (fp64) and
//                 writes log pi, mu (pass 1) or the variance (pass 2), with the
//                 floor, the regulariser and the empty-component rule.
// Every step reads the pairs and the data rows they name; nothing depends on
// the order in which CTAs or warps run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gmm_kernels.cuh"

namespace gmm {

namespace {

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Component of pair q, or -1 for a pair beyond the end or an index out of range.
__device__ __forceinline__ int pair_comp(const int32_t* __restrict__ idx, int64_t q, int64_t q_end, int K) {
  if (q >= q_end) return -1;
  const int c = __ldg(idx + q);
  return (c >= 0 && c < K) ? c : -1;
}

// One warp per tile: counts[c * T + t] = pairs of tile t with component c.
// The warp owns column t alone, so plain read-modify-writes suffice; the
// warp barrier orders them between steps.
__global__ void __launch_bounds__(256) tk_count_kernel(const int32_t* __restrict__ idx, int64_t N, int k, int K,
                                                       int64_t T, int32_t* __restrict__ counts) {
  const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int64_t q0 = t * kTkTile * k;
  const int64_t q1 = (t + 1) * kTkTile < N ? (t + 1) * kTkTile * k : N * k;
  for (int64_t b = q0; b < q1; b += 32) {
    const int c = pair_comp(idx, b + lane, q1, K);
    const unsigned grp = __match_any_sync(0xffffffffu, c);
    if (c >= 0 && lane == 31 - __clz(grp)) counts[static_cast<int64_t>(c) * T + t] += __popc(grp);
    __syncwarp();
  }
}

// One CTA per component: exclusive prefix of counts[c][0 .. T) in place,
// the total into tot[c].
__global__ void __launch_bounds__(256) tk_scan_kernel(int32_t* __restrict__ counts, int64_t T,
                                                      int32_t* __restrict__ tot) {
  __shared__ int32_t wsum[8];
  __shared__ int32_t carry;
  const int c = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* row = counts + static_cast<int64_t>(c) * T;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int64_t b = 0; b < T; b += 256) {
    const int64_t t = b + tid;
    const int32_t v = t < T ? row[t] : 0;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int32_t before = carry;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    if (t < T) row[t] = before + x - v;
    __syncthreads();
    if (tid == 255) carry = before + x;
    __syncthreads();
  }
  if (tid == 0) tot[c] = carry;
}

// One CTA of 1024 threads: base[c] = sum of tot over components below c
// (base[K] = all pairs); chunk_base[c] = chunks of kTkChunk pairs of the
// components below c (chunk_base[K] = all chunks).
__global__ void __launch_bounds__(1024) tk_base_kernel(const int32_t* __restrict__ tot, int K,
                                                       int64_t* __restrict__ base, int32_t* __restrict__ chunk_base) {
  __shared__ int64_t sp[1024];
  __shared__ int32_t sc[1024];
  const int tid = threadIdx.x;
  const int per = (K + 1023) / 1024;
  const int c0 = tid * per;
  int64_t p = 0;
  int32_t ch = 0;
  for (int c = c0; c < c0 + per && c < K; ++c) {
    p += tot[c];
    ch += (tot[c] + kTkChunk - 1) / kTkChunk;
  }
  sp[tid] = p;
  sc[tid] = ch;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int64_t a = tid >= o ? sp[tid - o] : 0;
    const int32_t b = tid >= o ? sc[tid - o] : 0;
    __syncthreads();
    sp[tid] += a;
    sc[tid] += b;
    __syncthreads();
  }
  p = sp[tid] - p;
  ch = sc[tid] - ch;
  for (int c = c0; c < c0 + per && c < K; ++c) {
    base[c] = p;
    chunk_base[c] = ch;
    p += tot[c];
    ch += (tot[c] + kTkChunk - 1) / kTkChunk;
  }
  if (tid == 1023) {
    base[K] = sp[1023];
    chunk_base[K] = sc[1023];
  }
}

// One warp per tile, the same walk as tk_count: every pair goes to
// base[c] + (pairs of c in earlier tiles) + (pairs of c earlier in this
// tile).  counts[c][t] (the exclusive prefix) is advanced as the cursor.
// The responsibility is normalised over the point's k kept components.
__global__ void __launch_bounds__(256) tk_fill_kernel(const int32_t* __restrict__ idx, const float* __restrict__ resp,
                                                      int64_t N, int k, int K, int64_t T,
                                                      int32_t* __restrict__ counts, const int64_t* __restrict__ base,
                                                      uint32_t* __restrict__ pt, float* __restrict__ rw) {
  const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int64_t q0 = t * kTkTile * k;
  const int64_t q1 = (t + 1) * kTkTile < N ? (t + 1) * kTkTile * k : N * k;
  for (int64_t b = q0; b < q1; b += 32) {
    const int64_t q = b + lane;
    const int c = pair_comp(idx, q, q1, K);
    const unsigned grp = __match_any_sync(0xffffffffu, c);
    int32_t cur = 0;
    if (c >= 0) {
      const int64_t i = q / k;
      const float* row = resp + i * k;
      float s = 0.f;
      for (int j = 0; j < k; ++j) s += __ldg(row + j);
      const float r = __ldg(resp + q);
      cur = counts[static_cast<int64_t>(c) * T + t];
      const int64_t pos = base[c] + cur + __popc(grp & lanemask_lt());
      pt[pos] = static_cast<uint32_t>(i);
      rw[pos] = s > 0.f ? r / s : 0.f;
    }
    __syncwarp();
    if (c >= 0 && lane == 31 - __clz(grp)) counts[static_cast<int64_t>(c) * T + t] = cur + __popc(grp);
    __syncwarp();
  }
}

// The component whose chunks include chunk `ch` (chunk_base is
// non-decreasing; empty components own no chunk).
__device__ __forceinline__ int chunk_owner(const int32_t* __restrict__ chunk_base, int K, int ch) {
  int lo = 0, hi = K - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (chunk_base[mid] <= ch) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <bool XB>
__device__ __forceinline__ float load_x(const void* X, int64_t off) {
  if constexpr (XB) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(X)[off]);
  else return __ldg(reinterpret_cast<const float*>(X) + off);
}

// One CTA per chunk, thread d = feature d.  PASS 1: part[ch][d] = sum r x_d,
// part[ch][D] = sum r.  PASS 2: part[ch][d] = sum r (x_d - mu'_d)^2.  Four
// interleaved fp32 accumulators per thread (pair j goes to accumulator
// j mod 4), added in a fixed order at the end.
template <bool XB, int PASS>
__global__ void __launch_bounds__(128) tk_stats_kernel(const void* __restrict__ X, int D, int K,
                                                       const int64_t* __restrict__ base,
                                                       const int32_t* __restrict__ chunk_base,
                                                       const uint32_t* __restrict__ pt, const float* __restrict__ rw,
                                                       const float* __restrict__ new_means,
                                                       double* __restrict__ part) {
  const int ch = blockIdx.x;
  if (ch >= chunk_base[K]) return;
  const int c = chunk_owner(chunk_base, K, ch);
  const int64_t q0 = base[c] + static_cast<int64_t>(ch - chunk_base[c]) * kTkChunk;
  const int64_t q1 = min(q0 + kTkChunk, base[c + 1]);
  const int d = threadIdx.x;
  const bool on = d < D;
  const float mu = (PASS == 2 && on) ? new_means[static_cast<int64_t>(c) * D + d] : 0.f;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  int64_t q = q0;
  for (; q + 8 <= q1; q += 8) {
    uint32_t i[8];
    float r[8], x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      i[j] = __ldg(pt + q + j);
      r[j] = __ldg(rw + q + j);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = on ? load_x<XB>(X, static_cast<int64_t>(i[j]) * D + d) : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if constexpr (PASS == 1) {
        a[j & 3] = fmaf(r[j], x[j], a[j & 3]);
        s[j & 3] += r[j];
      } else {
        const float y = x[j] - mu;
        a[j & 3] = fmaf(r[j] * y, y, a[j & 3]);
      }
    }
  }
  for (int j = 0; q < q1; ++q, ++j) {
    const uint32_t i = __ldg(pt + q);
    const float r = __ldg(rw + q);
    const float x = on ? load_x<XB>(X, static_cast<int64_t>(i) * D + d) : 0.f;
    if constexpr (PASS == 1) {
      a[j & 3] = fmaf(r, x, a[j & 3]);
      s[j & 3] += r;
    } else {
      const float y = x - mu;
      a[j & 3] = fmaf(r * y, y, a[j & 3]);
    }
  }
  double* out = part + static_cast<int64_t>(ch) * (D + 1);
  if (on) out[d] = (static_cast<double>(a[0]) + a[1]) + (static_cast<double>(a[2]) + a[3]);
  if (PASS == 1 && d == 0) out[D] = (static_cast<double>(s[0]) + s[1]) + (static_cast<double>(s[2]) + s[3]);
}

// One CTA per component, thread d = feature d: the component's chunk
// partials summed in chunk order.
//   PASS 1: N_k; log pi_k = log(N_k / N) (-inf and the old mean when
//           N_k < 1e-30); mu'_kd = S1_kd / N_k.  N_k is kept in nk[c].
//   PASS 2: s2 = S2 / N_k (diagonal), or sum_d S2_d / (D N_k) (spherical);
//           new variance max(s2, var_floor) + reg_covar (the old one when
//           N_k < 1e-30).
template <int PASS>
__global__ void __launch_bounds__(128) tk_final_kernel(const double* __restrict__ part,
                                                       const int32_t* __restrict__ chunk_base, int64_t N, int D,
                                                       int cov_diag, float reg_covar, float var_floor,
                                                       const float* means, const float* vars, double* __restrict__ nk,
                                                       float* new_log_weights, float* new_means, float* new_vars) {
  __shared__ double red[128];
  const int c = blockIdx.x, d = threadIdx.x;
  const int ch0 = chunk_base[c], ch1 = chunk_base[c + 1];
  double sd = 0.0, s0 = 0.0;
  for (int ch = ch0; ch < ch1; ++ch) {
    const double* p = part + static_cast<int64_t>(ch) * (D + 1);
    if (d < D) sd += p[d];
    if (PASS == 1) s0 += p[D];
  }
  constexpr double kEmpty = 1e-30;
  if constexpr (PASS == 1) {
    const bool empty = !(s0 >= kEmpty);
    if (d == 0) {
      nk[c] = s0;
      new_log_weights[c] = empty ? -INFINITY : static_cast<float>(log(s0 / static_cast<double>(N)));
    }
    if (d < D) {
      const int64_t o = static_cast<int64_t>(c) * D + d;
      new_means[o] = empty ? means[o] : static_cast<float>(sd / s0);
    }
  } else {
    const double n = nk[c];
    const bool empty = !(n >= kEmpty);
    if (cov_diag) {
      if (d < D) {
        const int64_t o = static_cast<int64_t>(c) * D + d;
        new_vars[o] = empty ? vars[o] : static_cast<float>(fmax(sd / n, static_cast<double>(var_floor)) + reg_covar);
      }
    } else {
      red[d] = d < D ? sd : 0.0;
      __syncthreads();
      if (d == 0) {
        double t = 0.0;
        for (int e = 0; e < D; ++e) t += red[e];
        new_vars[c] = empty ? vars[c]
                            : static_cast<float>(fmax(t / (static_cast<double>(D) * n), static_cast<double>(var_floor)) +
                                                 reg_covar);
      }
    }
  }
}

}  // namespace

const void* topk_handle(TopkKernel id, bool xb) {
  switch (id) {
    case TK_COUNT: return reinterpret_cast<const void*>(&tk_count_kernel);
    case TK_SCAN: return reinterpret_cast<const void*>(&tk_scan_kernel);
    case TK_BASE: return reinterpret_cast<const void*>(&tk_base_kernel);
    case TK_FILL: return reinterpret_cast<const void*>(&tk_fill_kernel);
    case TK_STATS1:
      return xb ? reinterpret_cast<const void*>(&tk_stats_kernel<true, 1>)
                : reinterpret_cast<const void*>(&tk_stats_kernel<false, 1>);
    case TK_STATS2:
      return xb ? reinterpret_cast<const void*>(&tk_stats_kernel<true, 2>)
                : reinterpret_cast<const void*>(&tk_stats_kernel<false, 2>);
    case TK_FINAL1: return reinterpret_cast<const void*>(&tk_final_kernel<1>);
    case TK_FINAL2: return reinterpret_cast<const void*>(&tk_final_kernel<2>);
  }
  return nullptr;
}

}  // namespace gmm
