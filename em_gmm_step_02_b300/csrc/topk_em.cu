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
//                 by component.  Points are cut into tiles (4096 points, more
//                 when K times the number of tiles would pass 2^25); one warp
//                 walks one tile in point order and counts its pairs per
//                 component in shared memory (counts[t][c]).
//   2. tk_scan:   per component, the exclusive prefix over tiles; the total.
//   3. tk_base:   the exclusive prefix over components (pair offsets) and the
//                 chunking of every component's pairs into runs of kTkChunk.
//   4. tk_fill:   the warp of each tile walks it again and writes every pair
//                 (point, normalised responsibility) to its slot: within a
//                 component, pairs are ordered by point index.
//   5. tk_stats:  one CTA per chunk (a run of one component's pairs), one
//                 thread per feature, one pass: sum r, sum r (x - s) and
//                 sum r (x - s)^2 about a shift s inside the chunk (the row
//                 of its largest responsibility).
//   6. tk_final:  one CTA per component combines its chunks in order (fp64)
//                 into N_k, the mean and the second moment about the mean
//                 (the pairwise-combination form of the variance), then
//                 writes log pi, mu and the variance with the floor, the
//                 regulariser and the empty-component rule.
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

// One warp (one CTA of 32 threads) per tile: counts[t * K + c] = pairs of
// tile t with component c, counted in a table of K ints in shared memory
// (dynamic, K * 4 bytes).  The warp walks its tile in point order; lanes with
// equal components form a group whose highest lane adds the group's size; the
// warp barrier orders the table updates between steps.
__global__ void __launch_bounds__(32) tk_count_kernel(const int32_t* __restrict__ idx, int64_t N, int k, int K,
                                                      int64_t T, int tile, int32_t* __restrict__ counts) {
  extern __shared__ int32_t table[];
  const int64_t t = blockIdx.x;
  const int lane = threadIdx.x;
  for (int c = lane; c < K; c += 32) table[c] = 0;
  __syncwarp();
  const int64_t q0 = t * tile * k;
  const int64_t q1 = (t + 1) * tile < N ? (t + 1) * tile * k : N * k;
  for (int64_t b = q0; b < q1; b += 32) {
    const int c = pair_comp(idx, b + lane, q1, K);
    const unsigned grp = __match_any_sync(0xffffffffu, c);
    if (c >= 0 && lane == 31 - __clz(grp)) table[c] += __popc(grp);
    __syncwarp();
  }
  int32_t* row = counts + t * K;
  for (int c = lane; c < K; c += 32) row[c] = table[c];
}

// Per component c, the exclusive prefix of counts[0 .. T)[c] over the tiles,
// in place, and the total into tot[c].  One CTA of 32 x 32 threads per 32
// components: thread (x, y) takes component 32 * blockIdx.x + x and the y-th
// segment of the tiles (loads of one tile row are consecutive); the segment
// sums are scanned in segment order, then each segment is rewritten.
__global__ void __launch_bounds__(1024) tk_scan_kernel(int32_t* __restrict__ counts, int K, int64_t T,
                                                       int32_t* __restrict__ tot) {
  __shared__ int32_t seg_sum[32][33];
  const int x = threadIdx.x & 31, y = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + x;
  const int64_t S = (T + 31) / 32;
  const int64_t t0 = y * S, t1 = min(T, t0 + S);
  int32_t s = 0;
  if (c < K)
    for (int64_t t = t0; t < t1; ++t) s += counts[t * K + c];
  seg_sum[y][x] = s;
  __syncthreads();
  if (y == 0) {
    int32_t run = 0;
    for (int g = 0; g < 32; ++g) {
      const int32_t v = seg_sum[g][x];
      seg_sum[g][x] = run;
      run += v;
    }
    if (c < K) tot[c] = run;
  }
  __syncthreads();
  int32_t run = seg_sum[y][x];
  if (c < K)
    for (int64_t t = t0; t < t1; ++t) {
      const int32_t v = counts[t * K + c];
      counts[t * K + c] = run;
      run += v;
    }
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

// One warp (one CTA of 32 threads) per tile, the same walk as tk_count: every
// pair goes to base[c] + (pairs of c in earlier tiles) + (pairs of c earlier
// in this tile).  The tile's row of the scanned counts is the cursor table in
// shared memory (K ints).  The responsibility is normalised over the point's k
// kept components.
__global__ void __launch_bounds__(32) tk_fill_kernel(const int32_t* __restrict__ idx, const float* __restrict__ resp,
                                                     int64_t N, int k, int K, int64_t T, int tile,
                                                     const int32_t* __restrict__ counts,
                                                     const int64_t* __restrict__ base, uint32_t* __restrict__ pt,
                                                     float* __restrict__ rw) {
  extern __shared__ int32_t table[];
  const int64_t t = blockIdx.x;
  const int lane = threadIdx.x;
  const int32_t* row = counts + t * K;
  for (int c = lane; c < K; c += 32) table[c] = row[c];
  __syncwarp();
  const int64_t q0 = t * tile * k;
  const int64_t q1 = (t + 1) * tile < N ? (t + 1) * tile * k : N * k;
  for (int64_t b = q0; b < q1; b += 32) {
    const int64_t q = b + lane;
    const int c = pair_comp(idx, q, q1, K);
    const unsigned grp = __match_any_sync(0xffffffffu, c);
    int32_t cur = 0;
    if (c >= 0) {
      const int64_t i = q / k;
      const float* rrow = resp + i * k;
      float s = 0.f;
      for (int j = 0; j < k; ++j) s += __ldg(rrow + j);
      const float r = __ldg(resp + q);
      cur = table[c];
      const int64_t pos = base[c] + cur + __popc(grp & lanemask_lt());
      pt[pos] = static_cast<uint32_t>(i);
      rw[pos] = s > 0.f ? r / s : 0.f;
    }
    __syncwarp();
    if (c >= 0 && lane == 31 - __clz(grp)) table[c] = cur + __popc(grp);
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

// One CTA per chunk, thread d = feature d, one pass over the chunk's pairs.
// The sums are taken about a shift inside the chunk -- the data row of the
// chunk's largest responsibility (the first such pair among equals) -- so that
// the second moment about the final mean is formed without cancellation:
//   part[ch] = [W, S1_0 .. S1_{D-1}, S2_0 .. S2_{D-1}, s_0 .. s_{D-1}],
//   W = sum r, S1_d = sum r (x_d - s_d), S2_d = sum r (x_d - s_d)^2.
// Four interleaved fp32 accumulators per thread (pair j goes to accumulator
// j mod 4), added in a fixed order at the end.
template <bool XB>
__global__ void __launch_bounds__(128) tk_stats_kernel(const void* __restrict__ X, int D, int K,
                                                       const int64_t* __restrict__ base,
                                                       const int32_t* __restrict__ chunk_base,
                                                       const uint32_t* __restrict__ pt, const float* __restrict__ rw,
                                                       double* __restrict__ part) {
  __shared__ float s_best[4];
  __shared__ int64_t s_pos[4];
  const int ch = blockIdx.x;
  if (ch >= chunk_base[K]) return;
  const int c = chunk_owner(chunk_base, K, ch);
  const int64_t q0 = base[c] + static_cast<int64_t>(ch - chunk_base[c]) * kTkChunk;
  const int64_t q1 = min(q0 + kTkChunk, base[c + 1]);
  const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
  const bool on = d < D;

  // the chunk's largest responsibility (lowest position among equals)
  float best = -1.f;
  int64_t bpos = q0;
  for (int64_t q = q0 + d; q < q1; q += 128) {
    const float r = __ldg(rw + q);
    if (r > best) {
      best = r;
      bpos = q;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int64_t op = __shfl_xor_sync(0xffffffffu, bpos, o);
    if (ob > best || (ob == best && op < bpos)) {
      best = ob;
      bpos = op;
    }
  }
  if (lane == 0) {
    s_best[warp] = best;
    s_pos[warp] = bpos;
  }
  __syncthreads();
  best = s_best[0];
  bpos = s_pos[0];
  for (int w = 1; w < 4; ++w)
    if (s_best[w] > best || (s_best[w] == best && s_pos[w] < bpos)) {
      best = s_best[w];
      bpos = s_pos[w];
    }
  const float sh = on ? load_x<XB>(X, static_cast<int64_t>(__ldg(pt + bpos)) * D + d) : 0.f;

  float a1[4] = {0.f, 0.f, 0.f, 0.f};
  float a2[4] = {0.f, 0.f, 0.f, 0.f};
  float w[4] = {0.f, 0.f, 0.f, 0.f};
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
      const float y = x[j] - sh;
      const float ry = r[j] * y;
      a1[j & 3] += ry;
      a2[j & 3] = fmaf(ry, y, a2[j & 3]);
      w[j & 3] += r[j];
    }
  }
  for (int j = 0; q < q1; ++q, ++j) {
    const uint32_t i = __ldg(pt + q);
    const float r = __ldg(rw + q);
    const float y = (on ? load_x<XB>(X, static_cast<int64_t>(i) * D + d) : 0.f) - sh;
    const float ry = r * y;
    a1[j & 3] += ry;
    a2[j & 3] = fmaf(ry, y, a2[j & 3]);
    w[j & 3] += r;
  }
  double* out = part + static_cast<int64_t>(ch) * (3 * D + 1);
  if (d == 0) out[0] = (static_cast<double>(w[0]) + w[1]) + (static_cast<double>(w[2]) + w[3]);
  if (on) {
    out[1 + d] = (static_cast<double>(a1[0]) + a1[1]) + (static_cast<double>(a1[2]) + a1[3]);
    out[1 + D + d] = (static_cast<double>(a2[0]) + a2[1]) + (static_cast<double>(a2[2]) + a2[3]);
    out[1 + 2 * D + d] = sh;
  }
}

// The same statistics with 16-byte loads, for rows whose size is a multiple
// of 16 bytes (bf16: D % 8 == 0; float32: D % 4 == 0).  A row is read by
// TPR = D / V threads of V features each; the CTA's 128 threads form
// G = 128 / TPR row groups, and group g takes the chunk's pairs g, g + G,
// g + 2G, ... in order.  The groups' sums are added in group order (fp64) at
// the end, so every sum still has one fixed order.
template <bool XB>
__global__ void __launch_bounds__(128) tk_stats_vec_kernel(const void* __restrict__ X, int D, int K,
                                                           const int64_t* __restrict__ base,
                                                           const int32_t* __restrict__ chunk_base,
                                                           const uint32_t* __restrict__ pt,
                                                           const float* __restrict__ rw, double* __restrict__ part) {
  constexpr int V = XB ? 8 : 4;              // features per 16-byte load
  __shared__ float s_best[4];
  __shared__ int64_t s_pos[4];
  __shared__ float s_a1[128 * V];            // [group][feature]
  __shared__ float s_a2[128 * V];
  __shared__ float s_w[128];
  const int ch = blockIdx.x;
  if (ch >= chunk_base[K]) return;
  const int c = chunk_owner(chunk_base, K, ch);
  const int64_t q0 = base[c] + static_cast<int64_t>(ch - chunk_base[c]) * kTkChunk;
  const int64_t q1 = min(q0 + kTkChunk, base[c + 1]);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int TPR = D / V;
  const int G = 128 / TPR;
  const int g = tid / TPR, u = tid % TPR;
  const bool on = g < G;

  // the chunk's largest responsibility (lowest position among equals)
  float best = -1.f;
  int64_t bpos = q0;
  for (int64_t q = q0 + tid; q < q1; q += 128) {
    const float r = __ldg(rw + q);
    if (r > best) {
      best = r;
      bpos = q;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int64_t op = __shfl_xor_sync(0xffffffffu, bpos, o);
    if (ob > best || (ob == best && op < bpos)) {
      best = ob;
      bpos = op;
    }
  }
  if (lane == 0) {
    s_best[warp] = best;
    s_pos[warp] = bpos;
  }
  __syncthreads();
  best = s_best[0];
  bpos = s_pos[0];
  for (int w = 1; w < 4; ++w)
    if (s_best[w] > best || (s_best[w] == best && s_pos[w] < bpos)) {
      best = s_best[w];
      bpos = s_pos[w];
    }

  auto load_row = [&](uint32_t i, float* x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(X) +
                                                         (static_cast<int64_t>(i) * D + u * V) * (XB ? 2 : 4)));
    if constexpr (XB) {
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w4[e] << 16);
        x[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
      }
    } else {
      x[0] = __uint_as_float(v.x);
      x[1] = __uint_as_float(v.y);
      x[2] = __uint_as_float(v.z);
      x[3] = __uint_as_float(v.w);
    }
  };

  float sh[V], a1[V], a2[V];
  float w = 0.f;
#pragma unroll
  for (int e = 0; e < V; ++e) a1[e] = a2[e] = 0.f;
  if (on) {
    load_row(__ldg(pt + bpos), sh);
    int64_t q = q0 + g;
    for (; q + 3 * G < q1; q += 4 * G) {
      uint32_t i[4];
      float r[4];
      float x[4][V];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        i[j] = __ldg(pt + q + j * G);
        r[j] = __ldg(rw + q + j * G);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) load_row(i[j], x[j]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float y = x[j][e] - sh[e];
          const float ry = r[j] * y;
          a1[e] += ry;
          a2[e] = fmaf(ry, y, a2[e]);
        }
        w += r[j];
      }
    }
    for (; q < q1; q += G) {
      float x[V];
      const float r = __ldg(rw + q);
      load_row(__ldg(pt + q), x);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float y = x[e] - sh[e];
        const float ry = r * y;
        a1[e] += ry;
        a2[e] = fmaf(ry, y, a2[e]);
      }
      w += r;
    }
#pragma unroll
    for (int e = 0; e < V; ++e) {
      s_a1[g * D + u * V + e] = a1[e];
      s_a2[g * D + u * V + e] = a2[e];
    }
    if (u == 0) s_w[g] = w;
  }
  __syncthreads();
  double* out = part + static_cast<int64_t>(ch) * (3 * D + 1);
  if (tid == 0) {
    double tw = 0.0;
    for (int gg = 0; gg < G; ++gg) tw += s_w[gg];
    out[0] = tw;
  }
  for (int d = tid; d < D; d += 128) {
    double t1 = 0.0, t2 = 0.0;
    for (int gg = 0; gg < G; ++gg) {
      t1 += s_a1[gg * D + d];
      t2 += s_a2[gg * D + d];
    }
    out[1 + d] = t1;
    out[1 + D + d] = t2;
  }
  // the shift of feature d, from the thread that loaded it (group 0)
  if (g == 0) {
#pragma unroll
    for (int e = 0; e < V; ++e) out[1 + 2 * D + u * V + e] = sh[e];
  }
}

// One CTA per component, thread d = feature d: the component's chunks
// combined in chunk order in fp64 (each chunk's sums are about its own shift
// s_c):
//   N_k  = sum_c W_c;  log pi_k = log(N_k / N);
//   mu_d = sum_c (S1_cd + W_c s_cd) / N_k;
//   M2_d = sum_c [S2_cd + 2 (s_cd - mu_d) S1_cd + W_c (s_cd - mu_d)^2]
//        = sum_i r_i (x_id - mu_d)^2;
//   variance M2_d / N_k (diagonal) or sum_d M2_d / (D N_k) (spherical), then
//   max(., var_floor) + reg_covar.  N_k < 1e-30: log pi = -inf, mean and
//   variance kept.
__global__ void __launch_bounds__(128) tk_final_kernel(const double* __restrict__ part,
                                                       const int32_t* __restrict__ chunk_base, int64_t N, int D,
                                                       int cov_diag, float reg_covar, float var_floor,
                                                       const float* means, const float* vars,
                                                       float* new_log_weights, float* new_means, float* new_vars) {
  __shared__ double red[128];
  const int c = blockIdx.x, d = threadIdx.x;
  const int ch0 = chunk_base[c], ch1 = chunk_base[c + 1];
  const int64_t stride = 3 * D + 1;
  double W = 0.0, t1 = 0.0;
  for (int ch = ch0; ch < ch1; ++ch) {
    const double* p = part + ch * stride;
    W += p[0];
    if (d < D) t1 += p[1 + d] + p[0] * p[1 + 2 * D + d];
  }
  constexpr double kEmpty = 1e-30;
  const bool empty = !(W >= kEmpty);
  const double iw = 1.0 / W;   // one fp64 division per thread (fp64 is slow here), then products
  const double mu = d < D ? t1 * iw : 0.0;
  double m2 = 0.0;
  if (!empty && d < D) {
    for (int ch = ch0; ch < ch1; ++ch) {
      const double* p = part + ch * stride;
      const double e = p[1 + 2 * D + d] - mu;
      m2 += p[1 + D + d] + 2.0 * e * p[1 + d] + p[0] * e * e;
    }
  }
  if (d == 0) new_log_weights[c] = empty ? -INFINITY : static_cast<float>(log(W / static_cast<double>(N)));
  if (d < D) {
    const int64_t o = static_cast<int64_t>(c) * D + d;
    new_means[o] = empty ? means[o] : static_cast<float>(mu);
  }
  if (cov_diag) {
    if (d < D) {
      const int64_t o = static_cast<int64_t>(c) * D + d;
      new_vars[o] = empty ? vars[o] : static_cast<float>(fmax(m2 * iw, static_cast<double>(var_floor)) + reg_covar);
    }
  } else {
    red[d] = d < D ? m2 : 0.0;
    __syncthreads();
    if (d == 0) {
      double t = 0.0;
      for (int e = 0; e < D; ++e) t += red[e];
      new_vars[c] = empty ? vars[c]
                          : static_cast<float>(fmax(t * iw / static_cast<double>(D), static_cast<double>(var_floor)) +
                                               reg_covar);
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
    case TK_STATS:
      return xb ? reinterpret_cast<const void*>(&tk_stats_kernel<true>)
                : reinterpret_cast<const void*>(&tk_stats_kernel<false>);
    case TK_STATS_VEC:
      return xb ? reinterpret_cast<const void*>(&tk_stats_vec_kernel<true>)
                : reinterpret_cast<const void*>(&tk_stats_vec_kernel<false>);
    case TK_FINAL: return reinterpret_cast<const void*>(&tk_final_kernel);
  }
  return nullptr;
}

}  // namespace gmm
