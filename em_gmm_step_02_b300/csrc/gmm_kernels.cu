// gmm_kernels.cu -- the EM-step kernels for sm_103a.
//
// Method: "Flash-GMM: A Memory-Efficient Kernel for Scalable Soft Clustering",
// section 2 (E-step responsibilities through a log-sum-exp over K weighted
// Gaussian terms; M-step from responsibility-weighted sufficient statistics)
// and section 3 (a naive GPU EM stores and re-reads the N x K responsibility
// matrix; here it lives only in on-chip tiles).
//
// Data path of one EM step (diagonal covariance; spherical uses the same
// path with the variance repeated over the D dimensions):
//   prep     per component: operand image of [mu/s2, -1/(2 s2)] (scaled to
//            log2 units) and the constant c_k = log pi_k - 1/2 sum log(2 pi s2)
//            - 1/2 sum mu^2/s2.
//   fused    per 128-point tile, per 128-component slice (one CTA each, the
//            slices of one tile forming a thread-block cluster):
//              logits   l = [x, x^2] . [mu/s2, -1/(2 s2)]^T + c     (tcgen05, TMEM)
//              softmax  row max / sum in registers, slices combined through
//                       distributed shared memory, r = 2^(l - lse)
//              stats    [S1 | S2 | S0] += R^T [x | x^2 | 1]           (tcgen05, TMEM)
//            statistics leave tensor memory every few tiles into fp64
//            per-cluster partials; nothing of size N x K is ever stored.
//   finalize fixed-order fp64 reduction of the partials and the M-step.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "gmm_kernels.cuh"
#include "layout.cuh"
#include "ptx.cuh"
#include "common.cuh"
#include "transform.cuh"

namespace gmm {


// ============================================================== scan of |X|
__global__ void absmax_kernel(const void* __restrict__ X, int64_t n_elems, int x_bf16,
                              Meta* __restrict__ meta) {
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (x_bf16) {
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(X);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_elems; i += stride)
      m = fmaxf(m, fabsf(__bfloat162float(x[i])));
  } else {
    const float* x = static_cast<const float*>(X);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_elems; i += stride)
      m = fmaxf(m, fabsf(x[i]));
  }
  // NaN propagates as a huge bound (caught later as a range error).
  if (m != m) m = CUDART_INF_F;
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(&meta->absmax_bits, __float_as_uint(m));
}

// Vectorised scan for 16-byte aligned data (8 bf16 or 4 f32 per load).
__global__ void absmax_vec_kernel(const uint4* __restrict__ X, int64_t n_vec, int x_bf16,
                                  Meta* __restrict__ meta) {
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
    uint4 v = __ldg(X + i);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (x_bf16) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, fabsf(__uint_as_float(w[j])));
    }
  }
  if (m != m) m = CUDART_INF_F;
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(&meta->absmax_bits, __float_as_uint(m));
}

// ============================================================== meta
// shift = mean of the component means (per dimension; zero when use_shift is
// 0, which keeps bf16 data exact in fp16); scale = power of two that keeps
// |x'| <= 127, so that x'^2 and its fp16 pieces stay inside the fp16 range.
__global__ void meta_kernel(const float* __restrict__ means, int D, int K, int use_shift, float absmax_hint,
                            Meta* __restrict__ meta, uint32_t* __restrict__ status) {
  __shared__ float red[kMaxD];
  const int d = threadIdx.x;
  float sh = 0.f;
  if (d < D && use_shift) {
    double s = 0.0;
    for (int k = 0; k < K; ++k) s += static_cast<double>(means[static_cast<int64_t>(k) * D + d]);
    sh = static_cast<float>(s / K);
    if (!isfinite(sh)) {
      atomicOr(status, ST_NONFINITE);
      sh = 0.f;
    }
  }
  if (d < kMaxD) meta->shift[d] = sh;
  red[d] = fabsf(sh);
  __syncthreads();
  if (d == 0) {
    float bmax = 0.f;
    for (int i = 0; i < D; ++i) bmax = fmaxf(bmax, red[i]);
    const float xa = absmax_hint > 0.f ? absmax_hint : __uint_as_float(meta->absmax_bits);
    float bound = xa + bmax;
    float scale = 1.f;
    if (!(bound < 1e30f)) {
      atomicOr(status, ST_RANGE);
      bound = 1.f;
    }
    if (bound > 0.f) {
      int e = static_cast<int>(floorf(log2f(127.f / bound)));
      e = max(-100, min(100, e));
      scale = ldexpf(1.f, e);
      if (bound * scale > 127.5f) scale *= 0.5f;   // guard against rounding at the boundary
    }
    meta->scale = scale;
    meta->inv_scale = 1.f / scale;
    meta->bmax_bits = 0u;
  }
}

// ============================================================== bmax (FAST)
// Largest magnitude over all components and features of the logit
// coefficients mu'/s2' and 1/(2 s2') (log2 units; tied: (Sigma^-1 nu)_d /
// scale): FAST gives every parameter row the same power-of-two scale, so the
// accumulated logits need one multiplier only.  One block per component.
__global__ void bmax_kernel(const float* __restrict__ means, const float* __restrict__ vars, int D, int K,
                            int cov_diag, Meta* __restrict__ meta, const double* __restrict__ sinv) {
  const int k = blockIdx.x;
  const int d = threadIdx.x;   // blockDim.x == 128
  __shared__ double nu[kMaxD];
  __shared__ float red[128];
  float m = 0.f;
  if (cov_diag == 2) {
    if (k < K && d < D) nu[d] = static_cast<double>(means[static_cast<int64_t>(k) * D + d]) - meta->shift[d];
    __syncthreads();
    if (k < K && d < D) {
      double w = 0.0;
      for (int e = 0; e < D; ++e) w += sinv[static_cast<int64_t>(d) * D + e] * nu[e];
      m = static_cast<float>(fabs(w / meta->scale * kLog2e));
    }
  } else if (k < K && d < D) {
    const double sc = meta->scale;
    const double mup = (static_cast<double>(means[static_cast<int64_t>(k) * D + d]) - meta->shift[d]) * sc;
    const double vp = static_cast<double>(cov_diag ? vars[static_cast<int64_t>(k) * D + d] : vars[k]) * sc * sc;
    if (vp > 0.0) m = static_cast<float>(fmax(fabs(mup / vp), 0.5 / vp) * kLog2e);
  }
  if (!(m < 3e38f)) m = 0.f;   // non-finite parameters are reported by params_kernel
  red[d] = m;
  __syncthreads();
  for (int o = 64; o > 0; o >>= 1) {
    if (d < o) red[d] = fmaxf(red[d], red[d + o]);
    __syncthreads();
  }
  if (d == 0) atomicMax(&meta->bmax_bits, __float_as_uint(red[0]));
}

// ============================================================== params
// One block per (padded) component.  Builds that component's rows of the
// per-slice parameter operand images (fp16; PRECISE adds a second image
// holding the rounding remainder, so that hi + lo carries 22 bits):
//   columns [0, D)        mu'/s2' * log2(e)        (x-part)
//   columns [Dp, Dp + D)  -1/(2 s2') * log2(e)     (x^2-part)
// in the same swizzled K-major layout as the data tiles, and the logit
// constant in log2 units.  x' = (x - shift) * scale, s2' = s2 * scale^2.
//
// FAST: every row carries the same power-of-two scale (from bmax_kernel), and
// the constant is the one of the Gaussian that the fp16-rounded row describes
// exactly: with b1, b2 the rounded coefficients, that Gaussian has
// s2' = -log2(e) / (2 b2) and mu' = -b1 / (2 b2), so the logit is a properly
// normalised log-density and the rounding only moves mu and s2 by relative
// amounts of 2^-12 (instead of adding an offset to every logit of the row).
// The constant also goes, split into three fp16 pieces, into the 128 x 16
// constant operand of the slice (c_img), which turns it into one more K step
// of the logit contraction.
//
// Tied covariance (cov == 2; Sigma shared, its inverse `sinv` and log|Sigma|
// from tied_prep_kernel): the logit drops its per-point term
// -1/2 x'^T Sigma'^-1 x', which cancels in the responsibilities and is put
// back into the log-likelihood from the data's Gram matrix, and keeps
//   columns [0, D)        (Sigma^-1 (mu - shift))_d / scale * log2(e)
//   columns [Dp, Dp + D)  0
//   constant              (log pi - 1/2 (D log 2 pi + log|Sigma|
//                          + (mu - shift)^T Sigma^-1 (mu - shift))) * log2(e)
template <bool kFast>
__global__ void params_kernel(const float* __restrict__ log_weights, const float* __restrict__ means,
                              const float* __restrict__ vars, int D, int K, int cov_diag, int nch,
                              Meta* __restrict__ meta, uint8_t* __restrict__ p_img, uint8_t* __restrict__ c_img,
                              float* __restrict__ cadj, float* __restrict__ iscale,
                              uint32_t* __restrict__ status, const double* __restrict__ sinv,
                              const double* __restrict__ tied_logdet) {
  const int k = blockIdx.x;
  const int d = threadIdx.x;   // blockDim.x == 128
  const int Dp = nch * kAtomElems;
  __shared__ double red_c[128];
  __shared__ float red_m[128];
  const bool valid_k = k < K;
  double b1 = 0.0, b2 = 0.0, cpart = 0.0;
  bool bad = false;
  __shared__ double nu[kMaxD];
  const double sc = meta->scale;
  double v_nat = 1.0, mup = 0.0, vp = 1.0;
  if (cov_diag == 2) {
    // tied: nu = mu_k - shift, then b1 = Sigma^-1 nu / scale
    if (valid_k && d < D) {
      const float mu = means[static_cast<int64_t>(k) * D + d];
      bad = !isfinite(mu);
      nu[d] = static_cast<double>(mu) - meta->shift[d];
    }
    __syncthreads();
    if (valid_k && d < D) {
      double w = 0.0;
      for (int e = 0; e < D; ++e) w += sinv[static_cast<int64_t>(d) * D + e] * nu[e];
      b1 = w / sc * kLog2e;
      cpart = nu[d] * w;
    }
  } else if (valid_k && d < D) {
    const float mu = means[static_cast<int64_t>(k) * D + d];
    const float v = cov_diag ? vars[static_cast<int64_t>(k) * D + d] : vars[k];
    bad = !isfinite(mu) || !isfinite(v) || !(v > 0.f);
    mup = (static_cast<double>(mu) - meta->shift[d]) * sc;
    vp = static_cast<double>(v) * sc * sc;
    v_nat = v;
    b1 = mup / vp * kLog2e;
    b2 = -0.5 / vp * kLog2e;
    cpart = log(static_cast<double>(v)) + kLog2Pi + mup * mup / vp;
  }
  if (bad) atomicOr(status, ST_NONFINITE);
  // scale of the fp16 rows: FAST one for all components, PRECISE per component
  float s = 1.f;
  if (kFast) {
    const float bm = __uint_as_float(meta->bmax_bits);
    if (bm > 0.f) s = ldexpf(1.f, max(-120, min(120, static_cast<int>(floorf(log2f(16384.f / bm))))));
    if (k == 0 && d == 0) {
      meta->pscale = s;
      meta->pinv = 1.f / s;
    }
  }
  // FAST diagonal / spherical: the constant of the Gaussian the rounded row
  // describes, summed in log2 units (see above); otherwise the exact one
  const bool consistent = kFast && cov_diag != 2;
  if (consistent && valid_k && d < D) {
    const double h1 = __half2float(__float2half_rn(static_cast<float>(b1 * s))) / s;
    const double h2 = __half2float(__float2half_rn(static_cast<float>(b2 * s))) / s;
    if (h2 < 0.0) {
      const double vpe = -0.5 * kLog2e / h2;
      cpart = 0.5 * kLog2e * (kLog2Pi + log(vpe) - 2.0 * log(sc)) - h1 * h1 / (4.0 * h2);
    } else {
      cpart = 0.5 * kLog2e * (log(v_nat) + kLog2Pi + mup * mup / vp);
    }
  }
  red_c[d] = cpart;
  red_m[d] = static_cast<float>(fmax(fabs(b1), fabs(b2)));
  __syncthreads();
  for (int o = 64; o > 0; o >>= 1) {
    if (d < o) {
      red_c[d] += red_c[d + o];
      red_m[d] = fmaxf(red_m[d], red_m[d + o]);
    }
    __syncthreads();
  }
  if (!kFast && red_m[0] > 0.f) {
    int e = static_cast<int>(floorf(log2f(16384.f / red_m[0])));
    s = ldexpf(1.f, max(-120, min(120, e)));
  }
  const int slice = k / kSlice, row = k % kSlice;
  double cval = -CUDART_INF;   // logit constant, log2 units
  {
    const float lw = valid_k ? log_weights[k] : -CUDART_INF_F;
    if (d == 0 && valid_k && (lw != lw || lw == CUDART_INF_F)) atomicOr(status, ST_NONFINITE);
    if (valid_k && lw > -CUDART_INF_F) {
      if (consistent) {
        cval = static_cast<double>(lw) * kLog2e - red_c[0];
      } else {
        const double q = cov_diag == 2 ? static_cast<double>(D) * kLog2Pi + *tied_logdet + red_c[0] : red_c[0];
        cval = (static_cast<double>(lw) - 0.5 * q) * kLog2e;
      }
    }
  }
  if (d == 0) {
    cadj[k] = static_cast<float>(cval);
    iscale[k] = valid_k ? 1.f / s : 0.f;
  }
  if (kFast && d < 16) {
    // row `row` of the slice's constant operand: s * c in three fp16 pieces
    __half piece = __float2half_rn(0.f);
    if (d < 3) {
      if (cval == -CUDART_INF) {
        piece = d == 0 ? __float2half_rn(-CUDART_INF_F) : __float2half_rn(0.f);
      } else {
        double rem = cval * s;
        if (!(fabs(rem) < 65504.0 * 32768.0)) {
          atomicOr(status, ST_RANGE);
          rem = 0.0;
        }
        for (int i = 0; i <= d; ++i) {
          const __half h = __float2half_rn(static_cast<float>(ldexp(rem, -const_exp(i))));
          if (i == d) piece = h;
          rem -= ldexp(static_cast<double>(__half2float(h)), const_exp(i));
        }
      }
    }
    *reinterpret_cast<__half*>(c_img + static_cast<size_t>(slice) * kConstBytes + const_off(row, d)) = piece;
  }
  // write this component's row of the operand images (thread d owns column d)
  const int np = kFast ? 1 : 2;
  const size_t piece_bytes = static_cast<size_t>(2 * nch) * kChunkBytes;
  uint8_t* img = p_img + static_cast<size_t>(slice) * np * piece_bytes;
  if (d < Dp) {
    for (int part = 0; part < 2; ++part) {
      const double val = (valid_k && d < D) ? (part == 0 ? b1 : b2) : 0.0;
      const int c = part * nch + d / kAtomElems;
      const uint32_t off = c * kChunkBytes + sw128_off(row, (d % kAtomElems) / 8) + (d % 8) * 2;
      const float f = static_cast<float>(val * s);
      const __half hi = __float2half_rn(f);
      *reinterpret_cast<__half*>(img + off) = hi;
      if (!kFast) *reinterpret_cast<__half*>(img + piece_bytes + off) = __float2half_rn(f - __half2float(hi));
    }
  }
}

// ============================================================== top-m
// MODE_TOPM work on one tile, after the row normaliser `lse` (log2 units,
// over every component of the launch's K group) is known.  v[e] holds the
// logit (log2 units) of component kbase + 64h + e for row nl; mh is the
// maximum over those 64.
//  1. Each half-row keeps its MAXM best components.  A candidate is ranked by
//     the key (mh - logit) with its low six bits replaced by e: the order of
//     keys is the order of logits, and equal truncated values fall back to
//     the lower component index.  (Dropping six of the 23 mantissa bits moves
//     a logit by at most 2^-17 of its distance to mh: well below the error of
//     the logits themselves.)
//  2. The lists of every half-row of every CTA in the cluster meet in shared
//     memory; each CTA merges the rows r = rank (mod C): one warp per row, one
//     lane per list, m rounds of a warp-wide maximum of the list heads.
//  3. One K group: the final responsibilities 2^(logit - lse) and indices go
//     to the output.  Several K groups: the group's best logits and indices
//     go to the per-group buffers for the combine kernel.
template <int MAXM>
__device__ __forceinline__ void topm_tile(const FusedArgs& a, Small* S, uint8_t* lists, const float (&v)[64],
                                          float mh, float lse, int64_t n0, int nl, int h, int lane, int warp,
                                          int st, int rank, int C, int kbase, int j,
                                          volatile uint32_t* abort_flag) {
  float key[MAXM];
#pragma unroll
  for (int s = 0; s < MAXM; ++s) key[s] = __uint_as_float(0x7f7fffffu);
  const bool live = mh > -CUDART_INF_F;
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    const float d = live ? fminf(mh - v[e], 1e30f) : 1e30f;
    float c = __uint_as_float((__float_as_uint(d) & ~63u) | static_cast<uint32_t>(e));
#pragma unroll
    for (int s = 0; s < MAXM; ++s) {
      const float lo = fminf(c, key[s]);
      c = fmaxf(c, key[s]);
      key[s] = lo;
    }
  }
  float* lv = reinterpret_cast<float*>(lists);
  uint16_t* li = reinterpret_cast<uint16_t*>(lists + kBN * 2 * MAXM * 4);
  if (C > 1 && j > 0) mbar_wait_cluster(&S->tfree, (j - 1) & 1, abort_flag, a.status);
#pragma unroll
  for (int s = 0; s < MAXM; ++s) {
    const uint32_t b = __float_as_uint(key[s]);
    const float dd = __uint_as_float(b & ~63u);
    lv[(nl * 2 + h) * MAXM + s] = dd >= 1e29f ? -CUDART_INF_F : mh - dd;
    li[(nl * 2 + h) * MAXM + s] = static_cast<uint16_t>(kbase + 64 * h + static_cast<int>(b & 63u));
  }
  if (h == 0) S->lse_row[nl] = lse;
  named_bar_sync(1, 256);
  if (C > 1) {
    if (st == 0) {
      fence_acq_rel_cluster();
      const uint32_t bar = smem_u32(&S->tready);
      for (int r = 0; r < C; ++r) mbar_arrive_remote(mapa(bar, r));
    }
    mbar_wait_cluster(&S->tready, j & 1, abort_flag, a.status);
  }
  const int m = a.topm;
  const int nlists = 2 * C;
  const int w8 = warp - 4;
  const uint32_t lv_s = smem_u32(lv), li_s = smem_u32(li);
  for (int row = rank + C * w8; row < kBN; row += 8 * C) {
    float hv[MAXM];
    uint32_t hx[MAXM];
    if (lane < nlists) {
      const int cr = lane >> 1, hh = lane & 1;
      const int base = (row * 2 + hh) * MAXM;
      if (C > 1) {
#pragma unroll
        for (int s = 0; s < MAXM; ++s) {
          hv[s] = ld_cluster_f32(mapa(lv_s + 4u * (base + s), cr));
          hx[s] = ld_cluster_u16(mapa(li_s + 2u * (base + s), cr));
        }
      } else {
#pragma unroll
        for (int s = 0; s < MAXM; ++s) {
          hv[s] = lv[base + s];
          hx[s] = li[base + s];
        }
      }
    } else {
#pragma unroll
      for (int s = 0; s < MAXM; ++s) {
        hv[s] = -CUDART_INF_F;
        hx[s] = 0xFFFFu;
      }
    }
    float outv = -CUDART_INF_F;
    uint32_t outi = 0xFFFFu;
    for (int s = 0; s < m; ++s) {
      float bv = hv[0];
      uint32_t bi = hx[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const uint32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (lane < nlists && hx[0] == bi) {
#pragma unroll
        for (int u = 0; u + 1 < MAXM; ++u) {
          hv[u] = hv[u + 1];
          hx[u] = hx[u + 1];
        }
        hv[MAXM - 1] = -CUDART_INF_F;
        hx[MAXM - 1] = 0xFFFFu;
      }
      if (lane == s) {
        outv = bv;
        outi = bi;
      }
    }
    const int64_t n = n0 + row;
    if (lane < m && n < a.N) {
      if (a.topm_groups == 1) {
        const float lse_r = S->lse_row[row];
        a.topm_val[n * m + lane] = lse_r > -CUDART_INF_F ? ex2(outv - lse_r) : 0.f;
        a.topm_idx[n * m + lane] = static_cast<int32_t>(outi);
      } else {
        const int64_t o = (static_cast<int64_t>(blockIdx.y) * a.N + n) * m + lane;
        a.topm_val[o] = outv;
        a.topm_idx[o] = static_cast<int32_t>(outi);
      }
    }
  }
  named_bar_sync(1, 256);
  if (C > 1 && st == 0) {
    const uint32_t bar = smem_u32(&S->tfree);
    for (int r = 0; r < C; ++r) mbar_arrive_remote(mapa(bar, r));
  }
}

// Adds this thread's row of the statistics accumulator (tensor-memory lane =
// component; h = 0: S1 and S0, h = 1: S2) to its fp64 partial row.  Each
// element of the partials has one writer, so fire-and-forget fp64 reductions
// keep a fixed order of additions.
template <int DP>
__device__ __forceinline__ void flush_stats(double* prow, uint32_t taddr, int h, bool live) {
  const int c0 = h == 0 ? 0 : DP;
  for (int c = 0; c < DP; c += 16) {
    float w[16];
    tmem_ld16(taddr + c0 + c, w);
    tmem_wait_ld();
    if (live) {
#pragma unroll
      for (int e = 0; e < 16; ++e) red_add_f64(prow + c0 + c + e, static_cast<double>(w[e]));
    }
  }
  if (h == 0) {
    float w[16];
    tmem_ld16(taddr + 2 * DP, w);
    tmem_wait_ld();
    if (live) red_add_f64(prow + 2 * DP, static_cast<double>(w[0]));
  }
}

// The R operand of the statistics MMA is a ring of two slots of 32 points:
// the rows of lane quarter q of every tile go to slot q & 1, so each slot
// serves two quarters per tile (q and q ^ 2).  Quarter q of tile j may write
// once the MMA has read the slot's previous user: quarter q - 2 of tile j
// (q >= 2) or quarter q + 2 of tile j - 1 (q < 2).  Each quarter has its
// own pair of barriers (r_full[q]: its rows written; r_done[q]: its rows
// read), one phase per tile.  A writer's previous wait on r_done[q ^ 2] saw
// the phase before the one it waits for now, and the phase after needs this
// quarter's own write, so the parity test cannot be fooled by a phase two
// steps away.
__device__ __forceinline__ bool r_slot_wait(Small* S, int q, int j, volatile uint32_t* abort_flag,
                                            uint32_t* status) {
  if (q >= 2) return mbar_wait(&S->r_done[q - 2], static_cast<uint32_t>(j & 1), abort_flag, status);
  if (j > 0) return mbar_wait(&S->r_done[q + 2], static_cast<uint32_t>((j - 1) & 1), abort_flag, status);
  return true;
}

// ============================================================== FAST softmax warps
// The softmax warps of the FAST (single fp16 piece) EM, normaliser and
// statistics-given modes.  Per tile:
//   A(j): logits of tile j from tensor memory (released at once), row
//         maximum and sum over this CTA's 128 components, p = 2^(l - m + 10)
//         kept as packed fp16 pairs, and this CTA's row normaliser, pushed
//         to every CTA of the cluster.
//   B(j): the row normaliser over the whole cluster (or read from memory),
//         r * 2^10 = p * 2^(m - lse) by a packed multiply, the R tile for
//         the statistics MMA, and the periodic flush of the statistics.
// Two receive slots are safe: a CTA pushes tile t only after its B(t-1),
// which needs every CTA's push of t-1, which each makes only after its own
// B(t-2) has read the slot that tile t reuses.
// The two warps that share a lane quarter (one per column half) meet at a
// named barrier of their own.
template <typename CF>
__device__ __forceinline__ void softmax_fast(const FusedArgs& a, uint8_t* sm, Small* S,
                                             volatile uint32_t* abort_flag, int tid, int warp, int lane,
                                             int rank, int C, int tgroup, int n_tgroups, int my_tiles,
                                             uint32_t acc1, uint32_t acc2, int kbase, int kvalid) {
  const int st = tid - 128;
  const int q = warp & 3;                 // TMEM lane quarter
  const int h = (warp - 4) >> 2;          // column half
  const int nl = 32 * q + lane;           // point row inside the tile
  const int pbar = 3 + q;                 // named barrier of the pair of warps of this quarter
  const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
  const bool given = a.mode == MODE_GIVEN;
  const bool want_r = a.mode != MODE_LSE;
  const bool exch = C > 1 && !given;
  constexpr float kLog2R = 10.f;          // log2 of kRScale<1>()
  double ll = 0.0;
  float llf = 0.f;                        // fp32 part of ll, moved into ll at every flush
  const bool ll_row = h == 0 && (nl % C) == rank;   // rows shared among the CTAs of a cluster
  int flush_idx = 0;
  for (int j = 0; j < my_tiles; ++j) {
    // (no early exit on an abort: every wait returns at once after one, so the
    // loop runs out quickly and both warps of a pair meet at every barrier)
    // ---------------------------------------------------------------- A(j): local softmax
    float v[64];
    float m;
    {
      mbar_wait(&S->acc1_full, j & 1, abort_flag, a.status);
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float w[16];
        tmem_ld16(acc1 + lane_off + 64 * h + 16 * c, w);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[16 * c + e] = w[e];
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&S->acc1_empty);
      // logits (log2 units); padded and dead components have cadj = -inf
      float mq[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int e4 = 0; e4 < 16; ++e4) {
        const float4 sc = *reinterpret_cast<const float4*>(&S->iscale[64 * h + 4 * e4]);
        const float4 cc = *reinterpret_cast<const float4*>(&S->cadj[64 * h + 4 * e4]);
        v[4 * e4 + 0] = fmaf(v[4 * e4 + 0], sc.x, cc.x);
        v[4 * e4 + 1] = fmaf(v[4 * e4 + 1], sc.y, cc.y);
        v[4 * e4 + 2] = fmaf(v[4 * e4 + 2], sc.z, cc.z);
        v[4 * e4 + 3] = fmaf(v[4 * e4 + 3], sc.w, cc.w);
        mq[0] = fmaxf(mq[0], v[4 * e4 + 0]);
        mq[1] = fmaxf(mq[1], v[4 * e4 + 1]);
        mq[2] = fmaxf(mq[2], v[4 * e4 + 2]);
        mq[3] = fmaxf(mq[3], v[4 * e4 + 3]);
      }
      S->pair_m[h][nl] = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      named_bar_sync(pbar, 64);
      m = fmaxf(S->pair_m[0][nl], S->pair_m[1][nl]);
    }
    uint32_t pk[32];                      // p = 2^(l - m + 10), packed fp16 pairs
    float lse_loc;
    {
      float sq[4] = {0.f, 0.f, 0.f, 0.f};
      if (m > -CUDART_INF_F) {
        const float mo = m - kLog2R;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2(v[2 * i] - mo);
          const float p1 = ex2(v[2 * i + 1] - mo);
          sq[i & 3] += p0 + p1;
          pk[i] = pack_f16x2(p0, p1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = 0u;
      }
      S->pair_s[h][nl] = (sq[0] + sq[1]) + (sq[2] + sq[3]);
      named_bar_sync(pbar, 64);
      const float tot = S->pair_s[0][nl] + S->pair_s[1][nl];
      lse_loc = tot > 0.f ? m + lg2(tot) - kLog2R : -CUDART_INF_F;
    }
    // push this CTA's row normalisers of tile j to every CTA of the cluster;
    // both threads of a row hold the value and share the stores (ranks of
    // their own parity); each store completes 4 transaction bytes on the
    // destination's slot barrier
    if (exch) {
      const uint32_t dst = smem_u32(&S->xrecv[j & 1][rank][nl]);
      const uint32_t bar = smem_u32(&S->xready[j & 1]);
#pragma unroll
      for (int r2 = 0; r2 < 4; ++r2) {
        const int r = 2 * r2 + h;
        if (r < C) st_async_f32(mapa(dst, r), lse_loc, mapa(bar, r));
      }
    }
    // ---------------------------------------------------------------- B(j): normalise, R tile
    const int64_t pn = static_cast<int64_t>(tgroup + j * n_tgroups) * kBN + nl;
    const float pm = m;
    const float plse = lse_loc;
    {
      const int jj = j;
      const bool valid = pn < a.N;
      const bool early_r = want_r && exch && q < 2 && jj > 0;
      float lse = plse;
      if (given) {
        lse = valid ? __ldg(a.lse_in + pn) : -CUDART_INF_F;
      } else if (C > 1) {
        // quarters 0-1 wait for their R slot (freed by the previous tile's
        // quarters 2-3) here, where the wait overlaps the exchange
        if (early_r) r_slot_wait(S, q, jj, abort_flag, a.status);
        const int slot = jj & 1;
        if (st == 0) mbar_arrive_expect_tx(&S->xready[slot], static_cast<uint32_t>(C * kBN * 4));
        mbar_wait(&S->xready[slot], (jj >> 1) & 1, abort_flag, a.status);
        float vals[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) vals[r] = r < C ? S->xrecv[slot][r][nl] : -CUDART_INF_F;
        float mx = vals[0];
#pragma unroll
        for (int r = 1; r < 8; ++r) mx = fmaxf(mx, vals[r]);
        float s2 = 0.f;
        if (mx > -CUDART_INF_F) {
#pragma unroll
          for (int r = 0; r < 8; ++r) s2 += ex2(vals[r] - mx);
        }
        lse = s2 > 0.f ? mx + lg2(s2) : -CUDART_INF_F;
      }
      if (!want_r) {
        if (rank == 0 && h == 0 && valid) a.lse_part[static_cast<int64_t>(blockIdx.y) * a.N + pn] = lse;
      } else {
        if (a.mode == MODE_EM && ll_row && valid) llf += lse;
        const float f = (valid && lse > -CUDART_INF_F && pm > -CUDART_INF_F) ? ex2(pm - lse) : 0.f;
        const __half2 f2 = __float2half2_rn(f);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          __half2 x = *reinterpret_cast<__half2*>(&pk[i]);
          x = __hmul2(x, f2);
          pk[i] = *reinterpret_cast<uint32_t*>(&x);
        }
        // this quarter's 32 rows go to R slot q & 1 once the statistics MMA
        // has read the quarter two before (with an exchange, quarters 0-1
        // have waited for that already)
        if (!early_r) r_slot_wait(S, q, jj, abort_flag, a.status);
        uint8_t* rbase = sm + CF::kOffR + h * 8192 + (q & 1) * kRSlotBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 w;
          w.x = pk[4 * c]; w.y = pk[4 * c + 1]; w.z = pk[4 * c + 2]; w.w = pk[4 * c + 3];
          *reinterpret_cast<uint4*>(rbase + sw128_off(lane, c)) = w;
        }
        fence_proxy_async_smem();
        mbar_arrive(&S->r_full[q]);
        // statistics leave tensor memory at the end of a flush period
        if (((jj + 1) % a.flush_tiles == 0) || (jj + 1 == my_tiles)) {
          ll += static_cast<double>(llf);
          llf = 0.f;
          mbar_wait(&S->acc2_full, flush_idx & 1, abort_flag, a.status);
          tc_fence_after();
          flush_stats<CF::kDp>(a.part + (static_cast<int64_t>(tgroup) * a.K_pad + kbase + 32 * q + lane) * a.F,
                               acc2 + lane_off, h, 32 * q + lane < kvalid);
          tc_fence_before();
          mbar_arrive(&S->acc2_empty);
          ++flush_idx;
        }
      }
    }
  }
  // log-likelihood partial of this CTA
  if (a.mode == MODE_EM) {
    ll += static_cast<double>(llf);
    for (int o = 16; o > 0; o >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, o);
    if (lane == 0) S->ll_red[warp - 4] = ll;
    named_bar_sync(1, 256);
    if (st == 0) {
      double tot = 0.0;
      for (int i = 0; i < 8; ++i) tot += S->ll_red[i];
      a.ll_part[tgroup * C + rank] = tot * kLn2;
    }
  }
}

// ============================================================== fused kernel
// kTopm: the MODE_TOPM instantiation; the others run MODE_EM, MODE_LSE and
// MODE_GIVEN.  Keeping the top-m code out of the EM instantiations keeps their
// register allocation for the softmax.
template <int NP, int NCH, int NST, bool kTopm>
__global__ void __launch_bounds__(416, 1) fused_em_kernel(const FusedArgs a) {
  using CF = Cfg<NP, NCH, NST>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Small* S = reinterpret_cast<Small*>(sm + CF::kOffSmall);
  volatile uint32_t* abort_flag = &S->abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool given = a.mode == MODE_GIVEN;
  const bool stats = a.mode == MODE_EM || a.mode == MODE_GIVEN;
  const int C = a.C;

  // ---- which slice / which tiles
  int rank, slice, tgroup, n_tgroups;
  if (given) {
    rank = 0;
    slice = blockIdx.x;
    tgroup = blockIdx.y;
    n_tgroups = gridDim.y;
  } else {
    rank = C > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    slice = blockIdx.y * C + rank;
    tgroup = blockIdx.x / C;
    n_tgroups = gridDim.x / C;
  }
  const int kbase = slice * kSlice;
  const int kvalid = max(0, min(kSlice, a.K - kbase));
  // every logit column is computed: padded components have zero operand rows
  // and a -inf constant, so their logits are -inf whatever tensor memory held
  const int n1 = kSlice;
  int my_tiles = 0;
  if (tgroup < a.n_tiles) my_tiles = (a.n_tiles - 1 - tgroup) / n_tgroups + 1;

  // ---- set-up
  if (tid == 0) {
    S->abort_flag = 0;
    S->poll_limit = a.max_polls ? a.max_polls : kMaxPolls;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S->full_a[i], 128);
      for (int g = 0; g < 8; ++g) mbar_init(&S->empty_g[i][g], 1);
      mbar_init(&S->xready[i], 1);
    }
    mbar_init(&S->p_full, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&S->pfull[i], 1);
      mbar_init(&S->pempty[i], 1);
    }
    mbar_init(&S->acc1_full, 1);
    mbar_init(&S->acc1_empty, 256);
    for (int q = 0; q < 4; ++q) {
      mbar_init(&S->r_full[q], 64);
      mbar_init(&S->r_done[q], 1);
    }
    mbar_init(&S->acc2_full, 1);
    mbar_init(&S->acc2_empty, 256);
    mbar_init(&S->drain, 1);
    mbar_init(&S->tready, C);
    mbar_init(&S->tfree, C);
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(&S->tmem_base, 512);
    tmem_relinquish();
  }
  if (tid >= 128 && tid < 384) {
    const int j = tid - 128;
    if (j < kSlice) {
      S->cadj[j] = a.cadj[kbase + j];
      S->iscale[j] = a.iscale[kbase + j];
    }
  }
  if (tid < 128) {
    // the all-ones operand that turns the statistics MMA into a row count
    const uint32_t one2 = 0x3C003C00u;   // pairs of fp16 1.0
    uint32_t* ones = reinterpret_cast<uint32_t*>(sm + CF::kOffOnes);
    for (int i = tid; i < 512; i += 128) ones[i] = one2;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if (C > 1 && !given) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = S->tmem_base;
  const uint32_t acc1 = tmem + CF::kAcc1Col;
  const uint32_t acc2 = tmem + CF::kAcc2Col;

  const uint32_t sA = smem_u32(sm + CF::kOffA);
  const uint32_t sP = smem_u32(sm + CF::kOffP);
  const uint32_t sR = smem_u32(sm + CF::kOffR);
  const uint32_t sOnes = smem_u32(sm + CF::kOffOnes);
  constexpr uint32_t kAbType = 0u;   // fp16 operands (PRECISE: hi and lo pieces)

  // FAST EM: the softmax warps hold a tile's logits and responsibilities in
  // registers; the transform warpgroup gives up 16 registers a thread so that
  // the two softmax warpgroups get 8 more each (per SM sub-partition: one
  // transform warp, two softmax warps, 512 registers moved either way).
  constexpr bool kRegSplit = NP == 1 && !kTopm;
  if (warp < 4) {
    // ================================================= transform warps
    if constexpr (kRegSplit) regs_release<112>();
    if (a.x_bf16) transform_warps<CF, Small, NP, NCH, NST, true, kTopm>(a, sm, S, abort_flag, tid, tgroup, n_tgroups, my_tiles);
    else transform_warps<CF, Small, NP, NCH, NST, false, kTopm>(a, sm, S, abort_flag, tid, tgroup, n_tgroups, my_tiles);
  } else if (warp < 12 && NP == 1 && !kTopm) {
    // ================================================= softmax warps (FAST EM)
    if constexpr (kRegSplit) regs_claim<136>();
    softmax_fast<CF>(a, sm, S, abort_flag, tid, warp, lane, rank, C, tgroup, n_tgroups, my_tiles, acc1, acc2,
                     kbase, kvalid);
  } else if (warp < 12) {
    // ================================================= softmax warps (PRECISE, top-m)
    const int st = tid - 128;            // 0..255
    const int q = warp & 3;              // TMEM lane quarter
    const int h = (warp - 4) >> 2;       // column half
    const int nl = 32 * q + lane;        // point row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    double ll = 0.0;
    float llf = 0.f;              // fp32 part of ll, moved into ll at every flush
    // the rows of a tile share the log-likelihood work among the CTAs of a cluster
    const bool ll_row = h == 0 && (nl % C) == rank;
    int flush_idx = 0;
    int j = 0;
    for (int t = tgroup; j < my_tiles; t += n_tgroups, ++j) {
      // all 256 threads agree on stopping (waits return at once after an abort,
      // so every thread reaches this check)
      if ((j & 7) == 0 && bar_red_or(1, 256, *abort_flag != 0)) break;
      const int64_t n = static_cast<int64_t>(t) * kBN + nl;
      const bool valid = n < a.N;
      mbar_wait(&S->acc1_full, j & 1, abort_flag, a.status);
      tc_fence_after();
      float v[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float w[16];
        tmem_ld16(acc1 + lane_off + 64 * h + 16 * c, w);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[16 * c + e] = w[e];
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&S->acc1_empty);
      // logits (log2 units) and the row maximum; padded and dead components
      // have cadj = -inf (and a zero operand row), so their logit is -inf
      float m = -CUDART_INF_F;
#pragma unroll
      for (int e4 = 0; e4 < 16; ++e4) {
        const float4 sc = *reinterpret_cast<const float4*>(&S->iscale[64 * h + 4 * e4]);
        const float4 cc = *reinterpret_cast<const float4*>(&S->cadj[64 * h + 4 * e4]);
        v[4 * e4 + 0] = fmaf(v[4 * e4 + 0], sc.x, cc.x);
        v[4 * e4 + 1] = fmaf(v[4 * e4 + 1], sc.y, cc.y);
        v[4 * e4 + 2] = fmaf(v[4 * e4 + 2], sc.z, cc.z);
        v[4 * e4 + 3] = fmaf(v[4 * e4 + 3], sc.w, cc.w);
        m = fmaxf(fmaxf(m, fmaxf(v[4 * e4 + 0], v[4 * e4 + 1])), fmaxf(v[4 * e4 + 2], v[4 * e4 + 3]));
      }
      S->pair_m[h][nl] = m;
      named_bar_sync(1, 256);
      m = fmaxf(S->pair_m[0][nl], S->pair_m[1][nl]);
      const float mh = S->pair_m[h][nl];   // maximum over this half (MODE_TOPM keys)
      float ssum = 0.f;
      if (kTopm) {
#pragma unroll
        for (int e = 0; e < 64; ++e) ssum += m == -CUDART_INF_F ? 0.f : ex2(v[e] - m);
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float p = m == -CUDART_INF_F ? 0.f : ex2(v[e] - m);
          v[e] = p;
          ssum += p;
        }
      }
      S->pair_s[h][nl] = ssum;
      named_bar_sync(1, 256);
      ssum = S->pair_s[0][nl] + S->pair_s[1][nl];
      const float lse_loc = ssum > 0.f ? m + lg2(ssum) : -CUDART_INF_F;
      float lse = lse_loc;
      if (given) {
        lse = valid ? __ldg(a.lse_in + n) : -CUDART_INF_F;
      } else if (C > 1) {
        // Every CTA of the cluster pushes its row normalisers into slot j & 1 of
        // every CTA (itself included); the slot's barrier completes when all
        // C * 128 floats have landed.  Two slots suffice: a CTA pushes tile
        // j + 2 only after every CTA has pushed tile j + 1, which each does
        // only after all of its threads have read slot j & 1 for tile j.
        const int slot = j & 1;
        if (h == 0) {
          const uint32_t dst = smem_u32(&S->xrecv[slot][rank][nl]);
          const uint32_t bar = smem_u32(&S->xready[slot]);
#pragma unroll
          for (int r = 0; r < 8; ++r)
            if (r < C) st_async_f32(mapa(dst, r), lse_loc, mapa(bar, r));
        }
        if (st == 0) mbar_arrive_expect_tx(&S->xready[slot], static_cast<uint32_t>(C * kBN * 4));
        mbar_wait(&S->xready[slot], (j >> 1) & 1, abort_flag, a.status);
        float vals[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) vals[r] = r < C ? S->xrecv[slot][r][nl] : -CUDART_INF_F;
        float mx = vals[0];
#pragma unroll
        for (int r = 1; r < 8; ++r) mx = fmaxf(mx, vals[r]);
        float s2 = 0.f;
        if (mx > -CUDART_INF_F) {
#pragma unroll
          for (int r = 0; r < 8; ++r) s2 += ex2(vals[r] - mx);
        }
        lse = s2 > 0.f ? mx + lg2(s2) : -CUDART_INF_F;
      }
      if (a.mode == MODE_LSE) {
        if (rank == 0 && h == 0 && valid) a.lse_part[static_cast<int64_t>(blockIdx.y) * a.N + n] = lse;
        continue;
      }
      if constexpr (kTopm) {
        if (a.topm_groups > 1) {
          if (rank == 0 && h == 0 && valid) a.lse_part[static_cast<int64_t>(blockIdx.y) * a.N + n] = lse;
        } else if (ll_row && valid) {
          llf += lse;
        }
        // candidate lists: the second data stage (unused in this mode), or the
        // R tile area of the single-stage configuration
        uint8_t* lists = NST == 2 ? sm + CF::kOffA + CF::kStageBytes : sm + CF::kOffR;
        const int64_t n0 = static_cast<int64_t>(t) * kBN;
        switch (a.topm_max) {
          case 2: topm_tile<2>(a, S, lists, v, mh, lse, n0, nl, h, lane, warp, st, rank, C, kbase, j, abort_flag); break;
          case 4: topm_tile<4>(a, S, lists, v, mh, lse, n0, nl, h, lane, warp, st, rank, C, kbase, j, abort_flag); break;
          case 8: topm_tile<8>(a, S, lists, v, mh, lse, n0, nl, h, lane, warp, st, rank, C, kbase, j, abort_flag); break;
          default: topm_tile<16>(a, S, lists, v, mh, lse, n0, nl, h, lane, warp, st, rank, C, kbase, j, abort_flag); break;
        }
        continue;
      }
      if (a.mode == MODE_EM && ll_row && valid) llf += lse;
      // r is stored as r * kRScale in fp16 so that small responsibilities stay
      // out of the fp16 subnormal range; finalize divides the statistics back.
      const float rscale = kRScale<NP>();
      const float f = (valid && lse > -CUDART_INF_F && m > -CUDART_INF_F) ? ex2(m - lse) * rscale : 0.f;
      // responsibilities of this quarter's rows into R slot q & 1, once the
      // statistics MMA has read the quarter two before
      r_slot_wait(S, q, j, abort_flag, a.status);
      const int nr = lane;                 // row inside the 32-point slot
      uint8_t* rbase = sm + CF::kOffR + h * 8192 + (q & 1) * kRSlotBytes;
      if constexpr (NP == 1) {
        // fp16 pairs of r * kRScale: the R tile
        uint32_t rw[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) rw[i] = pack_f16x2(v[2 * i] * f, v[2 * i + 1] * f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 w;
          w.x = rw[4 * c]; w.y = rw[4 * c + 1]; w.z = rw[4 * c + 2]; w.w = rw[4 * c + 3];
          *reinterpret_cast<uint4*>(rbase + sw128_off(nr, c)) = w;
        }
        fence_proxy_async_smem();
        mbar_arrive(&S->r_full[q]);
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) v[e] *= f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float* r8 = v + 8 * c;
          const uint32_t off = sw128_off(nr, c);
          float hi[8], lo[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            hi[e] = __half2float(__float2half_rn(r8[e]));
            lo[e] = r8[e] - hi[e];
          }
          uint4 w;
          w.x = pack_f16x2(hi[0], hi[1]); w.y = pack_f16x2(hi[2], hi[3]);
          w.z = pack_f16x2(hi[4], hi[5]); w.w = pack_f16x2(hi[6], hi[7]);
          *reinterpret_cast<uint4*>(rbase + off) = w;
          w.x = pack_f16x2(lo[0], lo[1]); w.y = pack_f16x2(lo[2], lo[3]);
          w.z = pack_f16x2(lo[4], lo[5]); w.w = pack_f16x2(lo[6], lo[7]);
          *reinterpret_cast<uint4*>(rbase + CF::kRBytes + off) = w;
        }
        fence_proxy_async_smem();
        mbar_arrive(&S->r_full[q]);
      }
      // statistics leave tensor memory at the end of a flush period
      const bool flush = ((j + 1) % a.flush_tiles == 0) || (j + 1 == my_tiles);
      if (flush && stats) {
        ll += static_cast<double>(llf);
        llf = 0.f;
        mbar_wait(&S->acc2_full, flush_idx & 1, abort_flag, a.status);
        tc_fence_after();
        // lanes = components 32q + lane; h = 0: S1 and S0, h = 1: S2
        const int kl = 32 * q + lane;
        double* prow = a.part + (static_cast<int64_t>(tgroup) * a.K_pad + kbase + kl) * a.F;
        const int c0 = h == 0 ? 0 : CF::kDp;
        // Each element of the partials has exactly one writer (this thread),
        // so fire-and-forget fp64 reductions keep a fixed order of additions
        // without waiting for the old value.
        for (int c = 0; c < CF::kDp; c += 16) {
          float w[16];
          tmem_ld16(acc2 + lane_off + c0 + c, w);
          tmem_wait_ld();
          if (kl < kvalid) {
#pragma unroll
            for (int e = 0; e < 16; ++e) red_add_f64(prow + c0 + c + e, static_cast<double>(w[e]));
          }
        }
        if (h == 0) {
          float w[16];
          tmem_ld16(acc2 + lane_off + 2 * CF::kDp, w);
          tmem_wait_ld();
          if (kl < kvalid) red_add_f64(prow + 2 * CF::kDp, static_cast<double>(w[0]));
        }
        tc_fence_before();
        mbar_arrive(&S->acc2_empty);
        ++flush_idx;
      }
    }
    // log-likelihood partial of this cluster (rank 0 only)
    if (a.mode == MODE_EM || (kTopm && a.topm_groups == 1)) {
      ll += static_cast<double>(llf);
      for (int o = 16; o > 0; o >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, o);
      if (lane == 0) S->ll_red[warp - 4] = ll;
      named_bar_sync(1, 256);
      if (st == 0) {
        double tot = 0.0;
        for (int i = 0; i < 8; ++i) tot += S->ll_red[i];
        a.ll_part[tgroup * C + rank] = tot * kLn2;
      }
    }
  } else {
    // ================================================= MMA warp
    if (lane == 0) {
      const size_t pbytes = static_cast<size_t>(NP) * CF::kPieceBytes;
      const uint8_t* src = a.p_img + static_cast<size_t>(slice) * pbytes;
      if constexpr (!CF::kStreamP) {
        mbar_arrive_expect_tx(&S->p_full, static_cast<uint32_t>(pbytes));
        for (size_t o = 0; o < pbytes; o += 16384)
          bulk_g2s(sm + CF::kOffP + o, src + o, 16384, &S->p_full);
        mbar_wait(&S->p_full, 0, abort_flag, a.status);
        tc_fence_after();
      }

      const uint32_t id1 = idesc_f16(kAbType, 0, 0, 128, n1);
      const uint32_t id2 = idesc_f16(kAbType, 1, 1, 128, 2 * CF::kDp);
      const uint32_t id0 = idesc_f16(kAbType, 1, 1, 128, 16);
      int flush_idx = 0;
      bool fresh = true;   // next statistics MMA starts a new accumulation
      const int nst = kTopm ? 1 : NST;   // MODE_TOPM: stage 1 holds the lists

      // Streamed parameter image (CF::kStreamP): every tile reads the slice's
      // image as a sequence of 8 chunks of 16 KB, chunk i = (piece i & 1,
      // column block i >> 1), through a ring of kPRing slots.  Sequence
      // number L = 8 * tile + i; slot L % kPRing, phase (L / kPRing) & 1.  A
      // slot is refilled once the MMAs of its previous chunk have completed
      // (tcgen05.commit to pempty); copies run two chunks ahead.
      const int n_chunks = CF::kStreamP ? 8 * my_tiles : 0;
      int n_copied = 0;
      auto issue_copy = [&](int L) {
        if (*abort_flag) return;
        const int s = L % CF::kPRing;
        if (L >= CF::kPRing)
          mbar_wait(&S->pempty[s], static_cast<uint32_t>((L / CF::kPRing - 1) & 1), abort_flag, a.status);
        const int i = L & 7;
        mbar_arrive_expect_tx(&S->pfull[s], static_cast<uint32_t>(kChunkBytes));
        bulk_g2s(sm + CF::kOffP + s * kChunkBytes, src + (i & 1) * CF::kPieceBytes + (i >> 1) * kChunkBytes,
                 kChunkBytes, &S->pfull[s]);
        n_copied = L + 1;
      };

      auto issue_g1 = [&](int jj) {
        const int s = jj % nst;
        const uint32_t stage = sA + s * CF::kStageBytes;
        uint32_t accf = 0;
        if constexpr (CF::kStreamP) {
          if (jj == 0) {
            if (n_chunks > 0) issue_copy(0);
            if (n_chunks > 1) issue_copy(1);
          }
          for (int i = 0; i < 8; ++i) {
            const int L = 8 * jj + i;
            const int ps = L % CF::kPRing;
            mbar_wait(&S->pfull[ps], static_cast<uint32_t>((L / CF::kPRing) & 1), abort_flag, a.status);
            tc_fence_after();
            const uint32_t pslot = sP + ps * kChunkBytes;
            const int c = i >> 1;                 // column block of [x | x^2]
            const int n_pa = (i & 1) ? 1 : 2;     // parameter hi: data hi and lo; parameter lo: data hi
            for (int pa = 0; pa < n_pa; ++pa)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sdesc_sw128(stage + pa * CF::kPieceBytes + c * kChunkBytes + 32 * kk, 16, 1024);
                const uint64_t bd = sdesc_sw128(pslot + 32 * kk, 16, 1024);
                mma_f16_ss(acc1, ad, bd, id1, accf);
                accf = 1;
              }
            mma_commit(&S->pempty[ps]);
            if (L + 2 < n_chunks) issue_copy(L + 2);
          }
        } else {
#pragma unroll
          for (int pr = 0; pr < (NP == 1 ? 1 : 3); ++pr) {
            const int pa = pr == 2 ? 1 : 0;      // data piece
            const int pp = pr == 1 ? 1 : 0;      // parameter piece
            for (int c = 0; c < 2 * NCH; ++c)
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sdesc_sw128(stage + pa * CF::kPieceBytes + c * kChunkBytes + 32 * kk, 16, 1024);
                const uint64_t bd = sdesc_sw128(sP + pp * CF::kPieceBytes + c * kChunkBytes + 32 * kk, 16, 1024);
                mma_f16_ss(acc1, ad, bd, id1, accf);
                accf = 1;
              }
          }
        }
        mma_commit(&S->acc1_full);
      };
      auto wait_a = [&](int jj) {
        mbar_wait(&S->full_a[jj % nst], (jj / nst) & 1, abort_flag, a.status);
        tc_fence_after();
      };

      if (my_tiles > 0) {
        wait_a(0);
        issue_g1(0);
        if (!stats)
          for (int g = 0; g < 8; ++g) mma_commit(&S->empty_g[0][g]);
      }
      for (int j = 0; j < my_tiles; ++j) {
        if (*abort_flag) break;
        const int s = j % NST;
        const bool next = j + 1 < my_tiles;
        if (NST == 2 || !stats) {
          if (next) {
            wait_a(j + 1);
            mbar_wait(&S->acc1_empty, j & 1, abort_flag, a.status);
            tc_fence_after();
            issue_g1(j + 1);
            if (!stats)
              for (int g = 0; g < 8; ++g) mma_commit(&S->empty_g[(j + 1) % nst][g]);
          }
        }
        if (stats) {
          const uint32_t stage = sA + s * CF::kStageBytes;
          if (fresh && flush_idx > 0) {
            mbar_wait(&S->acc2_empty, (flush_idx - 1) & 1, abort_flag, a.status);
            tc_fence_after();
          }
          // one lane quarter (32 points, R slot q & 1) at a time
          for (int q = 0; q < 4; ++q) {
            const uint32_t sRq = sR + (q & 1) * kRSlotBytes;
            mbar_wait(&S->r_full[q], static_cast<uint32_t>(j & 1), abort_flag, a.status);
            tc_fence_after();
            for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
              for (int pr = 0; pr < (NP == 1 ? 1 : 3); ++pr) {
                const int prr = pr == 2 ? 1 : 0;   // responsibility piece
                const int pf = pr == 1 ? 1 : 0;    // data piece
                const uint64_t ad = sdesc_sw128(sRq + prr * CF::kRBytes + 2048 * kk, 8192, 1024);
                const uint64_t bd = sdesc_sw128(stage + pf * CF::kPieceBytes + q * 4096 + 2048 * kk,
                                                kChunkBytes, 1024);
                mma_f16_ss(acc2, ad, bd, id2, fresh ? 0u : 1u);
                fresh = false;
              }
              // rows 16 (2 q + kk) .. +15 of the stage are no longer needed
              mma_commit(&S->empty_g[s][2 * q + kk]);
            }
            // S0: responsibilities against an all-ones operand (the same fp16
            // values as S1 and S2, summed in fp32 by the tensor core)
            bool fresh0 = (q == 0) && (j % a.flush_tiles == 0);
            for (int prr = 0; prr < NP; ++prr)
              for (int kk = 0; kk < 2; ++kk) {
                const uint64_t ad = sdesc_sw128(sRq + prr * CF::kRBytes + 2048 * kk, 8192, 1024);
                const uint64_t bd = sdesc_sw128(sOnes, kChunkBytes, 1024);
                mma_f16_ss(acc2 + 2 * CF::kDp, ad, bd, id0, fresh0 ? 0u : 1u);
                fresh0 = false;
              }
            mma_commit(&S->r_done[q]);
          }
          const bool flush = ((j + 1) % a.flush_tiles == 0) || (j + 1 == my_tiles);
          if (flush) {
            mma_commit(&S->acc2_full);
            ++flush_idx;
            fresh = true;
          }
          if (NST == 1 && next) {
            wait_a(j + 1);
            mbar_wait(&S->acc1_empty, j & 1, abort_flag, a.status);
            tc_fence_after();
            issue_g1(j + 1);
          }
        }
      }
      // every copy and tensor-core operation of this CTA completes before the
      // tensor memory and shared memory are released (bounded waits that do not
      // give up early after another wait has failed)
      if constexpr (CF::kStreamP) {
        // the copies still in flight after an early stop (at most the last
        // kPRing issued; each was awaited before use otherwise)
        for (int L = n_copied - CF::kPRing < 0 ? 0 : n_copied - CF::kPRing; L < n_copied; ++L)
          mbar_wait_final(&S->pfull[L % CF::kPRing], static_cast<uint32_t>((L / CF::kPRing) & 1), a.status);
      } else {
        mbar_wait_final(&S->p_full, 0, a.status);
      }
      mma_commit(&S->drain);
      mbar_wait_final(&S->drain, 0, a.status);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (C > 1 && !given) cluster_sync();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================== combine (K > 1024)
// lse[n] = log2 sum_g 2^(lse_part[g][n]); per-block log-likelihood partials.
__global__ void lse_combine_kernel(const float* __restrict__ lse_part, int n_groups, int64_t N,
                                   float* __restrict__ lse, double* __restrict__ ll_part) {
  __shared__ double red[8];
  double acc = 0.0;
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < N;
       n += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float mx = -CUDART_INF_F;
    for (int g = 0; g < n_groups; ++g) mx = fmaxf(mx, lse_part[static_cast<int64_t>(g) * N + n]);
    float s = 0.f;
    for (int g = 0; g < n_groups; ++g)
      s += mx == -CUDART_INF_F ? 0.f : ex2(lse_part[static_cast<int64_t>(g) * N + n] - mx);
    const float l = s > 0.f ? mx + lg2(s) : -CUDART_INF_F;
    lse[n] = l;
    acc += static_cast<double>(l);
  }
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += red[i];
    ll_part[blockIdx.x] = t * kLn2;
  }
}

// ============================================================== top-m combine (K > 1024)
// Per point: the normaliser over all K groups and the best m of the groups'
// candidate lists (each sorted, best first); ties go to the lower index.
__global__ void topm_combine_kernel(const float* __restrict__ lse_part, const float* __restrict__ gval,
                                    const int32_t* __restrict__ gidx, int n_groups, int64_t N, int m,
                                    float* __restrict__ resp_out, int32_t* __restrict__ idx_out,
                                    double* __restrict__ ll_part) {
  __shared__ double red[8];
  double acc = 0.0;
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < N;
       n += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float mx = -CUDART_INF_F;
    for (int g = 0; g < n_groups; ++g) mx = fmaxf(mx, lse_part[static_cast<int64_t>(g) * N + n]);
    float s = 0.f;
    if (mx > -CUDART_INF_F)
      for (int g = 0; g < n_groups; ++g) s += ex2(lse_part[static_cast<int64_t>(g) * N + n] - mx);
    const float lse = s > 0.f ? mx + lg2(s) : -CUDART_INF_F;
    acc += static_cast<double>(lse);
    float bv[16];
    int32_t bi[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      bv[u] = -CUDART_INF_F;
      bi[u] = 0x7fffffff;
    }
    for (int g = 0; g < n_groups; ++g) {
      const int64_t base = (static_cast<int64_t>(g) * N + n) * m;
      for (int c = 0; c < m; ++c) {
        float cv = gval[base + c];
        int32_t ci = gidx[base + c];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const bool better = cv > bv[u] || (cv == bv[u] && ci < bi[u]);
          const float tv = better ? bv[u] : cv;
          const int32_t ti = better ? bi[u] : ci;
          if (better) {
            bv[u] = cv;
            bi[u] = ci;
          }
          cv = tv;
          ci = ti;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (u < m) {
        resp_out[n * m + u] = lse > -CUDART_INF_F ? ex2(bv[u] - lse) : 0.f;
        idx_out[n * m + u] = bi[u];
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += red[i];
    ll_part[blockIdx.x] = t * kLn2;
  }
}

// Sum of n partial log-likelihoods in a fixed order (one thread).
__global__ void ll_total_kernel(const double* __restrict__ parts, int n, double* __restrict__ out) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < n; ++i) t += parts[i];
    *out = t;
  }
}

// ============================================================== finalize (M-step)
// One block per component; fixed-order fp64 reduction over tile groups.
__global__ void finalize_kernel(const double* __restrict__ part, int n_parts, int K_pad, int F, int Dp,
                                int D, int K, int64_t N, int cov_diag, float reg_covar, float var_floor,
                                double rscale,
                                const Meta* __restrict__ meta, const double* __restrict__ ll_part,
                                int n_ll, float* __restrict__ out_lw, float* __restrict__ out_mu,
                                float* __restrict__ out_var, const float* __restrict__ old_mu,
                                const float* __restrict__ old_var, double* __restrict__ ll_out,
                                double* __restrict__ tied_stats) {
  const int k = blockIdx.x;
  const int d = threadIdx.x;
  __shared__ double red[128];
  double S0 = 0.0;
  for (int g = 0; g < n_parts; ++g) S0 += part[(static_cast<int64_t>(g) * K_pad + k) * F + 2 * Dp];
  S0 /= rscale;   // the responsibility operand carries a power-of-two scale
  const bool empty = !(S0 >= 1e-30);
  const double isc = meta->inv_scale;
  double vd = 0.0;
  float keep_mu = 0.f, keep_var = 0.f;
  if (d < D) {
    keep_mu = old_mu[static_cast<int64_t>(k) * D + d];
    if (cov_diag != 2) keep_var = cov_diag ? old_var[static_cast<int64_t>(k) * D + d] : old_var[k];
  }
  __syncthreads();   // every old value is read before any output is written
  if (d < D) {
    double S1 = 0.0, S2 = 0.0;
    for (int g = 0; g < n_parts; ++g) {
      const double* row = part + (static_cast<int64_t>(g) * K_pad + k) * F;
      S1 += row[d];
      S2 += row[Dp + d];
    }
    S1 /= rscale;
    S2 /= rscale;
    const double m1 = S1 / S0;
    double v = (S2 / S0 - m1 * m1) * isc * isc;
    if (v < 0.0) v = 0.0;
    vd = v;
    const double mu = m1 * isc + meta->shift[d];
    out_mu[static_cast<int64_t>(k) * D + d] = empty ? keep_mu : static_cast<float>(mu);
    if (cov_diag == 2 && tied_stats) {
      // tied: N_k and nu_k = mu_k - shift for the shared covariance (empty: 0)
      double* ts = tied_stats + static_cast<int64_t>(k) * (D + 1);
      if (d == 0) ts[0] = empty ? 0.0 : S0;
      ts[1 + d] = empty ? 0.0 : m1 * isc;
    }
    if (cov_diag == 1) {
      const double vv = (v > var_floor ? v : static_cast<double>(var_floor)) + reg_covar;
      out_var[static_cast<int64_t>(k) * D + d] = empty ? keep_var : static_cast<float>(vv);
    }
  }
  if (cov_diag == 0) {
    red[d] = vd;
    __syncthreads();
    for (int o = 64; o > 0; o >>= 1) {
      if (d < o) red[d] += red[d + o];
      __syncthreads();
    }
    if (d == 0) {
      const double v = red[0] / D;
      const double vv = (v > var_floor ? v : static_cast<double>(var_floor)) + reg_covar;
      out_var[k] = empty ? keep_var : static_cast<float>(vv);
    }
  }
  if (d == 0) out_lw[k] = empty ? -CUDART_INF_F : static_cast<float>(log(S0 / static_cast<double>(N)));
  if (k == 0 && d == 0 && ll_out) {
    double t = 0.0;
    for (int i = 0; i < n_ll; ++i) t += ll_part[i];
    *ll_out = t;
  }
}

// ============================================================== tied covariance
// One shared D x D covariance Sigma (the "tied" type of the "GMMXX" README's
// "Covariance Coverage" table).  The E-step runs the fused kernel with the
// linear logits of params_kernel (cov == 2); these kernels supply Sigma^-1
// and log|Sigma|, the Gram matrix G = sum_i (x_i - shift)(x_i - shift)^T of
// the data, and the M-step of the shared covariance:
//   Sigma' = (G - sum_k N_k nu_k nu_k^T) / N,  nu_k = mu_k' - shift,
// which is sum_k sum_i r_ik (x_i - mu_k')(x_i - mu_k')^T / N because the
// responsibilities of a point sum to one; the dropped per-point term of the
// logits returns to the log-likelihood as -1/2 tr(Sigma^-1 G).

// One block of 128 threads with the Cholesky factor L of Sigma in shared
// memory (fp64, row-major, lower; D * (D + 1) * 8 bytes of dynamic shared memory):
// L (written to global memory, zero above the diagonal) and log|Sigma|.  A
// matrix that is not positive definite (or not finite) raises ST_NONFINITE.
__global__ void __launch_bounds__(128) tied_prep_kernel(const float* __restrict__ sigma, int D,
                                                        double* __restrict__ L, double* __restrict__ logdet,
                                                        uint32_t* __restrict__ status) {
  extern __shared__ double Ls[];
  // row stride D + 1: the threads of a step own different rows, and a
  // stride of D doubles would put all their accesses in one bank
  const int ld = D + 1;
  const int t = threadIdx.x;
  __shared__ int bad;
  if (t == 0) bad = 0;
  __syncthreads();
  for (int i = t; i < D * D; i += blockDim.x) {
    const float v = sigma[i];
    if (!isfinite(v)) bad = 1;
    Ls[(i / D) * ld + i % D] = v;
  }
  __syncthreads();
  // right-looking Cholesky: column j is final once the updates of the
  // columns before it have been applied; it then updates the trailing lower
  // triangle (thread t owns rows t, t + 128, ...; the updates of one row are
  // independent of each other, so fp64, which is slow on this GPU, runs at
  // its throughput rather than its latency)
  // (scalar fp64 work is slow here: one reciprocal per column, then
  // multiplications; the logarithms of the diagonal are taken in parallel)
  __shared__ double rdiag;
  for (int j = 0; j < D; ++j) {
    if (t == 0) {
      double a = Ls[j * ld + j];
      if (!(a > 0.0)) {
        bad = 1;
        a = 1.0;
      }
      const double r = sqrt(a);
      Ls[j * ld + j] = r;
      rdiag = 1.0 / r;
    }
    __syncthreads();
    const double rj = rdiag;
    for (int i = j + 1 + t; i < D; i += blockDim.x) Ls[i * ld + j] *= rj;
    __syncthreads();
    for (int i = j + 1 + t; i < D; i += blockDim.x) {
      const double lij = Ls[i * ld + j];
      for (int k = j + 1; k <= i; ++k) Ls[i * ld + k] -= lij * Ls[k * ld + j];
    }
    __syncthreads();
  }
  __shared__ double lgs[kMaxD];
  for (int j = t; j < D; j += blockDim.x) lgs[j] = log(Ls[j * ld + j]);
  __syncthreads();
  if (t == 0) {
    double lg = 0.0;
    for (int j = 0; j < D; ++j) lg += lgs[j];
    *logdet = 2.0 * lg;
    if (bad) atomicOr(status, ST_NONFINITE);
  }
  for (int i = t; i < D * D; i += blockDim.x) L[i] = (i % D) <= (i / D) ? Ls[(i / D) * ld + i % D] : 0.0;
}

// Column j of Sigma^-1 = L^-T L^-1 e_j, one block of 128 threads per column
// (fp64 is scarce on this GPU: spreading the D solves over D SMs keeps them
// short), with L copied to shared memory (row stride D + 1, D * (D + 1) * 8
// bytes of dynamic shared memory).  Forward then backward substitution; each
// step's dot product is split over the threads (thread t takes k = t,
// t + 128, ...) and summed in a fixed order (warp shuffles, then the four
// warps in order).
__global__ void __launch_bounds__(128) tied_inv_kernel(const double* __restrict__ L, int D,
                                                       double* __restrict__ sinv) {
  extern __shared__ double Ls[];
  __shared__ double y[kMaxD];
  __shared__ double rd[kMaxD];              // reciprocals of the diagonal
  __shared__ double wsum[4];
  const int ld = D + 1;
  const int j = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int i = t; i < D * D; i += 128) Ls[(i / D) * ld + i % D] = L[i];
  for (int i = t; i < D; i += 128) rd[i] = 1.0 / L[static_cast<int64_t>(i) * D + i];
  __syncthreads();
  auto block_sum = [&](double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) wsum[warp] = v;
    __syncthreads();
    const double s = (wsum[0] + wsum[1]) + (wsum[2] + wsum[3]);
    __syncthreads();
    return s;
  };
  for (int i = 0; i < D; ++i) {
    double part = 0.0;
    for (int k = t; k < i; k += 128) part += Ls[i * ld + k] * y[k];
    const double s = block_sum(part);
    if (t == 0) y[i] = ((i == j ? 1.0 : 0.0) - s) * rd[i];
    __syncthreads();
  }
  for (int i = D - 1; i >= 0; --i) {
    double part = 0.0;
    for (int k = i + 1 + t; k < D; k += 128) part += Ls[k * ld + i] * y[k];
    const double s = block_sum(part);
    if (t == 0) y[i] = (y[i] - s) * rd[i];
    __syncthreads();
  }
  for (int i = t; i < D; i += 128) sinv[static_cast<int64_t>(i) * D + j] = y[i];
}

// G = sum over the partials of the CTAs in a fixed order, in fp64, with the
// operand scale undone: the partials hold sums of (y * scale)(y * scale)^T.
__global__ void gram_reduce_kernel(const double* __restrict__ part, int n_parts, int D,
                                   const Meta* __restrict__ meta, double* __restrict__ G) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(D) * D) return;
  double s = 0.0;
  for (int p = 0; p < n_parts; ++p) s += part[static_cast<int64_t>(p) * D * D + e];
  const double is = meta->inv_scale;
  G[e] = s * is * is;
}

// Shared covariance of the M-step, one block of 16 x 16 threads per 16 x 16
// tile of Sigma' (thread = element (d, e)):
//   Sigma'_de = (G_de - sum_k N_k nu_kd nu_ke) / N, diagonal floored and
//   regularised.
// The components' (N_k, nu_k) rows are staged in shared memory 32 at a time,
// and every element sums over k in ascending order (fp64).  Block (0, 0) also
// subtracts 1/2 tr(Sigma^-1 G) from the log-likelihood (the logits' dropped
// per-point term), when ll is given.
__global__ void __launch_bounds__(256) sigma_tied_kernel(const double* __restrict__ G,
                                                         const double* __restrict__ tied_stats, int K, int D,
                                                         int64_t N, float reg_covar, float var_floor,
                                                         const double* __restrict__ sinv, double* __restrict__ ll,
                                                         float* __restrict__ out_sigma) {
  constexpr int kT = 16, kC = 32;
  __shared__ double a_s[kC][kT];   // N_k nu_kd, rows of this tile
  __shared__ double b_s[kC][kT];   // nu_ke, columns of this tile
  const int tx = threadIdx.x % kT, ty = threadIdx.x / kT;
  const int d = blockIdx.y * kT + ty, e = blockIdx.x * kT + tx;
  double s = 0.0;
  for (int k0 = 0; k0 < K; k0 += kC) {
    for (int i = threadIdx.x; i < kC * kT; i += 256) {
      const int kk = i / kT, c = i % kT;
      const int k = k0 + kk;
      const double* ts = tied_stats + static_cast<int64_t>(k) * (D + 1);
      const int dr = blockIdx.y * kT + c, ec = blockIdx.x * kT + c;
      a_s[kk][c] = (k < K && dr < D) ? ts[0] * ts[1 + dr] : 0.0;
      b_s[kk][c] = (k < K && ec < D) ? ts[1 + ec] : 0.0;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kC; ++kk) s += a_s[kk][ty] * b_s[kk][tx];
    __syncthreads();
  }
  if (d < D && e < D) {
    double v = (G[static_cast<int64_t>(d) * D + e] - s) / static_cast<double>(N);
    if (d == e) v = (v > var_floor ? v : static_cast<double>(var_floor)) + reg_covar;
    out_sigma[static_cast<int64_t>(d) * D + e] = static_cast<float>(v);
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && ll) {
    __shared__ double red[256];
    double t = 0.0;
    for (int i = threadIdx.x; i < D * D; i += 256) t += sinv[i] * G[i];
    red[threadIdx.x] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
      double tot = 0.0;
      for (int i = 0; i < 256; ++i) tot += red[i];
      *ll -= 0.5 * tot;
    }
  }
}

// ============================================================== threshold assignment
// The multi-assignment of "Flash-GMM" (conclusion; the posting-list use in
// its IVF experiments): every (point, component) pair whose responsibility
// reaches a threshold, as compressed rows.  Input: each point's m largest
// responsibilities in descending order (ties: lower index first) from the
// top-m pass.  Three kernels: per-point counts with a block-local exclusive
// scan, a scan of the block totals, and the scatter of the kept entries.

// cnt_i = number of j < m with resp[i][j] >= tau (a prefix of the sorted
// row).  offsets[i] <- exclusive scan of cnt within the block;
// block_tot[b] <- the block's total.
__global__ void __launch_bounds__(kThreshBlock) thresh_count_kernel(const float* __restrict__ resp, int64_t N,
                                                                   int m, float tau, int64_t* __restrict__ offsets,
                                                                   int64_t* __restrict__ block_tot) {
  __shared__ int32_t sc[kThreshBlock];
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreshBlock + threadIdx.x;
  int c = 0;
  if (i < N) {
    const float* r = resp + i * m;
    while (c < m && r[c] >= tau) ++c;
  }
  sc[threadIdx.x] = c;
  __syncthreads();
  // Hillis-Steele inclusive scan over the block
  for (int o = 1; o < kThreshBlock; o <<= 1) {
    const int v = threadIdx.x >= static_cast<unsigned>(o) ? sc[threadIdx.x - o] : 0;
    __syncthreads();
    sc[threadIdx.x] += v;
    __syncthreads();
  }
  if (i < N) offsets[i] = sc[threadIdx.x] - c;
  if (threadIdx.x == kThreshBlock - 1) block_tot[blockIdx.x] = sc[threadIdx.x];
}

// One block: block_tot[b] <- exclusive scan over b; block_tot[n_blocks] <- the
// total.  Chunks of 1024 with a running carry.
__global__ void __launch_bounds__(1024) thresh_scan_kernel(int64_t* __restrict__ block_tot, int64_t n_blocks) {
  __shared__ int64_t sc[1024];
  __shared__ int64_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < n_blocks; base += 1024) {
    const int64_t b = base + threadIdx.x;
    const int64_t v = b < n_blocks ? block_tot[b] : 0;
    sc[threadIdx.x] = v;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
      const int64_t u = threadIdx.x >= static_cast<unsigned>(o) ? sc[threadIdx.x - o] : 0;
      __syncthreads();
      sc[threadIdx.x] += u;
      __syncthreads();
    }
    if (b < n_blocks) block_tot[b] = carry + sc[threadIdx.x] - v;
    __syncthreads();
    if (threadIdx.x == 1023) carry += sc[1023];
    __syncthreads();
  }
  if (threadIdx.x == 0) block_tot[n_blocks] = carry;
}

// offsets[i] += its block's offset; offsets[N] = total; the kept entries go
// to idx_out / resp_out[offsets[i] ...] when the total fits `capacity`,
// otherwise nothing is written there and ST_CAPACITY is raised.
__global__ void __launch_bounds__(kThreshBlock) thresh_scatter_kernel(
    const float* __restrict__ resp, const int32_t* __restrict__ idx, int64_t N, int m, float tau,
    int64_t* __restrict__ offsets, const int64_t* __restrict__ block_tot, int64_t n_blocks,
    int32_t* __restrict__ idx_out, float* __restrict__ resp_out, int64_t capacity, uint32_t* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreshBlock + threadIdx.x;
  const int64_t total = block_tot[n_blocks];
  if (i == 0) {
    offsets[N] = total;
    if (total > capacity) atomicOr(status, ST_CAPACITY);
  }
  if (i >= N) return;
  const int64_t off = offsets[i] + block_tot[blockIdx.x];
  offsets[i] = off;
  if (total > capacity) return;
  const float* r = resp + i * m;
  const int32_t* k = idx + i * m;
  for (int j = 0; j < m && r[j] >= tau; ++j) {
    idx_out[off + j] = k[j];
    resp_out[off + j] = r[j];
  }
}

// Host-side handles of the kernels (launched from gmm_api.cu).
const void* kernel_handle(KernelId id) {
  switch (id) {
    case K_ABSMAX: return reinterpret_cast<const void*>(&absmax_kernel);
    case K_ABSMAX_VEC: return reinterpret_cast<const void*>(&absmax_vec_kernel);
    case K_META: return reinterpret_cast<const void*>(&meta_kernel);
    case K_PARAMS_FAST: return reinterpret_cast<const void*>(&params_kernel<true>);
    case K_PARAMS_PRECISE: return reinterpret_cast<const void*>(&params_kernel<false>);
    case K_FUSED_1_1_2: return reinterpret_cast<const void*>(&fused_em_kernel<1, 1, 2, false>);
    case K_FUSED_1_2_2: return reinterpret_cast<const void*>(&fused_em_kernel<1, 2, 2, false>);
    case K_FUSED_2_1_1: return reinterpret_cast<const void*>(&fused_em_kernel<2, 1, 1, false>);
    case K_FUSED_2_2_1: return reinterpret_cast<const void*>(&fused_em_kernel<2, 2, 1, false>);
    case K_TOPM_1_1_2: return reinterpret_cast<const void*>(&fused_em_kernel<1, 1, 2, true>);
    case K_TOPM_1_2_2: return reinterpret_cast<const void*>(&fused_em_kernel<1, 2, 2, true>);
    case K_TOPM_2_1_1: return reinterpret_cast<const void*>(&fused_em_kernel<2, 1, 1, true>);
    case K_TOPM_2_2_1: return reinterpret_cast<const void*>(&fused_em_kernel<2, 2, 1, true>);
    case K_LSE_COMBINE: return reinterpret_cast<const void*>(&lse_combine_kernel);
    case K_FINALIZE: return reinterpret_cast<const void*>(&finalize_kernel);
    case K_TOPM_COMBINE: return reinterpret_cast<const void*>(&topm_combine_kernel);
    case K_LL_TOTAL: return reinterpret_cast<const void*>(&ll_total_kernel);
    case K_THRESH_COUNT: return reinterpret_cast<const void*>(&thresh_count_kernel);
    case K_THRESH_SCAN: return reinterpret_cast<const void*>(&thresh_scan_kernel);
    case K_THRESH_SCATTER: return reinterpret_cast<const void*>(&thresh_scatter_kernel);
    case K_TIED_PREP: return reinterpret_cast<const void*>(&tied_prep_kernel);
    case K_TIED_INV: return reinterpret_cast<const void*>(&tied_inv_kernel);
    case K_GRAM_REDUCE: return reinterpret_cast<const void*>(&gram_reduce_kernel);
    case K_SIGMA_TIED: return reinterpret_cast<const void*>(&sigma_tied_kernel);
    case K_BMAX: return reinterpret_cast<const void*>(&bmax_kernel);
  }
  return nullptr;
}

}  // namespace gmm
