// topm_refine.cu -- the top-m responsibilities recomputed from the direct form
// of the Gaussian log-density ("Flash-GMM: A Memory-Efficient Kernel for
// Scalable Soft Clustering", section 2: log pi_k + log N(x | mu_k, Sigma_k)
// with the squared distance (x - mu)^2 / s2, not its expansion).
//
// The top-m pass ranks components by logits from the tensor cores, where the
// expanded form [x, x^2] . [mu / s2, -1 / (2 s2)] carries a rounding error
// that grows with x^2 / s2 (sharply fitted components).  Its candidates are
// kept; their logits are recomputed here in fp32 from x, mu and s2:
//   l'_k = c_k - 1/2 sum_d (x_d - mu_kd)^2 / s2_kd,
//   c_k  = log pi_k - 1/2 sum_d log(2 pi s2_kd),
// and the mass the pass gave the candidates, R = sum_j r_j (all K
// normalised), is redistributed among them by the recomputed logits:
//   r'_j = R exp(l'_j) / sum_i exp(l'_i),
// then the list is sorted again (descending, equal values by the lower
// component).  R itself is the pass's; at fitted parameters it is 1 up to
// the non-candidates' share.  A point's log-likelihood becomes
// log sum_j exp(l'_j) - log R.  The host runs these kernels after the pass
// when gmm_opts.topm_refine asks for them (by default on the PRECISE path)
// and the covariance is spherical or diagonal.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "gmm_kernels.cuh"

namespace gmm {

namespace {

// Per-component rows of the refinement, padded to kMaxD features:
// pm[k][d] = (mu_kd, 1 / s2_kd) for d < D (spherical: s2_k for every d) and
// (0, 0) beyond, so that padding adds nothing to the distance; cdir[k] = c_k
// (-inf for a dead component, log pi_k = -inf).  One block of kMaxD threads
// per component.
__global__ void __launch_bounds__(kMaxD) refine_params_kernel(const float* __restrict__ log_weights,
                                                              const float* __restrict__ means,
                                                              const float* __restrict__ vars, int D, int cov_diag,
                                                              float2* __restrict__ pm, float* __restrict__ cdir) {
  __shared__ double red[kMaxD];
  const int k = blockIdx.x, d = threadIdx.x;
  double lg = 0.0;
  float2 e = make_float2(0.f, 0.f);
  if (d < D) {
    const int64_t o = static_cast<int64_t>(k) * D + d;
    const double v = cov_diag ? vars[o] : vars[k];
    e = make_float2(means[o], static_cast<float>(1.0 / v));
    lg = log(2.0 * 3.14159265358979323846 * v);
  }
  pm[static_cast<int64_t>(k) * kMaxD + d] = e;
  red[d] = lg;
  __syncthreads();
  if (d == 0) {
    double s = 0.0;
    for (int i = 0; i < D; ++i) s += red[i];
    const float lw = log_weights[k];
    cdir[k] = lw == -INFINITY ? -INFINITY : static_cast<float>(static_cast<double>(lw) - 0.5 * s);
  }
}

// Features 16 h + 2 q and 16 h + 2 q + 1 (h = 0..7) of row n (0 past D or
// for n >= N), fetched into w and turned into floats by decode_x16 when they
// are used, so that the loads of the next point stay in flight meanwhile: the
// eight lanes of a group read 32 (bf16) or 64 (float32) contiguous bytes per
// load.  VEC: one 4- or 8-byte load per pair (D even, X aligned to the pair;
// bf16 pairs stay packed in w[2 h]); otherwise element loads, as float bits.
template <bool XB, bool VEC>
__device__ __forceinline__ void fetch_x16(const void* X, int64_t n, int64_t N, int D, int q, uint32_t (&w)[16]) {
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const int d = 16 * h + 2 * q;
    uint32_t w0 = 0, w1 = 0;
    if (n < N) {
      if constexpr (VEC && XB) {
        if (d < D)
          w0 = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(X) + n * D + d));
      } else if constexpr (VEC) {
        if (d < D) {
          const float2 u = __ldg(reinterpret_cast<const float2*>(reinterpret_cast<const float*>(X) + n * D + d));
          w0 = __float_as_uint(u.x);
          w1 = __float_as_uint(u.y);
        }
      } else if constexpr (XB) {
        const __nv_bfloat16* row = reinterpret_cast<const __nv_bfloat16*>(X) + n * D;
        if (d < D) w0 = __float_as_uint(__bfloat162float(row[d]));
        if (d + 1 < D) w1 = __float_as_uint(__bfloat162float(row[d + 1]));
      } else {
        const float* row = reinterpret_cast<const float*>(X) + n * D;
        if (d < D) w0 = __float_as_uint(row[d]);
        if (d + 1 < D) w1 = __float_as_uint(row[d + 1]);
      }
    }
    w[2 * h] = w0;
    w[2 * h + 1] = w1;
  }
}

template <bool XB, bool VEC>
__device__ __forceinline__ void decode_x16(const uint32_t (&w)[16], float (&v)[16]) {
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if constexpr (VEC && XB) {
      v[2 * h] = __uint_as_float(w[2 * h] << 16);
      v[2 * h + 1] = __uint_as_float(w[2 * h] & 0xffff0000u);
    } else {
      v[2 * h] = __uint_as_float(w[2 * h]);
      v[2 * h + 1] = __uint_as_float(w[2 * h + 1]);
    }
  }
}

// Eight lanes per point (lane q of the group holds the feature pairs 8 h + q,
// h = 0..7, so that the group reads one 128-byte line of a candidate's row
// per load), four points per warp; the next point's candidate list, row of X
// and responsibilities are loaded while the current one is refined.  Every lane of a group ends with the whole sorted
// list; lane q writes entries q and q + 8.  With ll_part set, each block
// writes the sum over its points of  log sum_j exp(l'_j) - log R  (the
// point's log-likelihood: the candidates carry the share R of the density).
template <bool XB, bool VEC, int MAXM>
__global__ void __launch_bounds__(256, MAXM >= 8 ? 2 : 3) refine_kernel(const void* __restrict__ X, int64_t N, int D, int K, int m,
                                                        const float4* __restrict__ pm,
                                                        const float* __restrict__ cdir, float* __restrict__ resp,
                                                        int32_t* __restrict__ idx, double* __restrict__ ll_part) {
  __shared__ double red[8];
  const int lane = threadIdx.x & 31, g = lane >> 3, q = lane & 7;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5) * 4;
  int64_t n = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * 4 + g;
  int32_t cn[MAXM];
  float rn[MAXM];
  uint32_t wn[16];
#pragma unroll
  for (int j = 0; j < MAXM; ++j) {
    cn[j] = (j < m && n < N) ? idx[n * m + j] : -1;
    rn[j] = (j < m && n < N) ? resp[n * m + j] : 0.f;
  }
  fetch_x16<XB, VEC>(X, n, N, D, q, wn);
  double acc = 0.0;
  for (; n - g < N; n += stride) {
    const bool valid = n < N;
    int32_t c[MAXM];
    float r[MAXM];
    float x[16];
#pragma unroll
    for (int j = 0; j < MAXM; ++j) {
      c[j] = cn[j];
      r[j] = rn[j];
    }
    decode_x16<XB, VEC>(wn, x);
    const int64_t nn = n + stride;
#pragma unroll
    for (int j = 0; j < MAXM; ++j) {
      cn[j] = (j < m && nn < N) ? idx[nn * m + j] : -1;
      rn[j] = (j < m && nn < N) ? resp[nn * m + j] : 0.f;
    }
    fetch_x16<XB, VEC>(X, nn, N, D, q, wn);
    float l[MAXM];
    float lmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < MAXM; ++j) {
      const int k = c[j];
      const bool live = j < m && k >= 0 && k < K;
      const float ck = live ? __ldg(cdir + k) : -INFINITY;
      float s = 0.f;
      if (live) {
        const float4* row = pm + static_cast<int64_t>(k) * (kMaxD / 2) + q;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          if (16 * h < D) {
            const float4 e = __ldg(row + 8 * h);   // (mu, 1/s2) of features 16 h + 2 q, 16 h + 2 q + 1
            const float y0 = x[2 * h] - e.x, y1 = x[2 * h + 1] - e.z;
            s = fmaf(y0 * y0, e.y, s);
            s = fmaf(y1 * y1, e.w, s);
          }
        }
      }
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      l[j] = ck > -INFINITY ? ck - 0.5f * s : -INFINITY;
      lmax = fmaxf(lmax, l[j]);
    }
    if (!valid) continue;
    float mass = 0.f;
#pragma unroll
    for (int j = 0; j < MAXM; ++j) mass += r[j];
    if (!(lmax > -INFINITY && mass > 0.f)) {
      if (q == 0) acc += -INFINITY;
      continue;
    }
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < MAXM; ++j) {
      l[j] = l[j] > -INFINITY ? expf(l[j] - lmax) : 0.f;
      z += l[j];
    }
    const float f = mass / z;
#pragma unroll
    for (int j = 0; j < MAXM; ++j) r[j] = j < m ? l[j] * f : -INFINITY;
    if (q == 0) acc += static_cast<double>(lmax) + static_cast<double>(logf(z)) - static_cast<double>(logf(mass));
    // descending r, equal values by the lower component (bubble passes over
    // compile-time positions keep the lists in registers; entries past m
    // hold -inf and stay last)
#pragma unroll
    for (int a = 0; a < MAXM - 1; ++a) {
#pragma unroll
      for (int b = 0; b < MAXM - 1 - a; ++b) {
        const bool sw = r[b] < r[b + 1] || (r[b] == r[b + 1] && c[b] > c[b + 1]);
        const float tr = sw ? r[b + 1] : r[b];
        const float ur = sw ? r[b] : r[b + 1];
        const int32_t tc = sw ? c[b + 1] : c[b];
        const int32_t uc = sw ? c[b] : c[b + 1];
        r[b] = tr;
        r[b + 1] = ur;
        c[b] = tc;
        c[b + 1] = uc;
      }
    }
#pragma unroll
    for (int j = 0; j < MAXM; ++j) {
      if (j < m && (j & 7) == q) {
        resp[n * m + j] = r[j];
        idx[n * m + j] = c[j];
      }
    }
  }
  if (ll_part) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += red[i];
      ll_part[blockIdx.x] = t;
    }
  }
}

template <bool XB, bool VEC>
const void* refine_fn(int maxm) {
  switch (maxm) {
    case 2: return reinterpret_cast<const void*>(&refine_kernel<XB, VEC, 2>);
    case 4: return reinterpret_cast<const void*>(&refine_kernel<XB, VEC, 4>);
    case 8: return reinterpret_cast<const void*>(&refine_kernel<XB, VEC, 8>);
    case 16: return reinterpret_cast<const void*>(&refine_kernel<XB, VEC, 16>);
  }
  return nullptr;
}

}  // namespace

const void* refine_params_handle() { return reinterpret_cast<const void*>(&refine_params_kernel); }

const void* refine_handle(bool xb, bool vec, int maxm) {
  return xb ? (vec ? refine_fn<true, true>(maxm) : refine_fn<true, false>(maxm))
            : (vec ? refine_fn<false, true>(maxm) : refine_fn<false, false>(maxm));
}

}  // namespace gmm
