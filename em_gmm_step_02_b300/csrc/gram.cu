// gram.cu -- the data's Gram matrix G = sum_i y_i y_i^T, y = x - shift, on the
// tensor cores, for the tied-covariance model (one full D x D covariance
// shared by every component: the "GMMXX" README's "Covariance Coverage" table,
// tied, shape (D, D)).  The EM step needs G every call: the logits of a tied
// model drop the per-point term -1/2 y^T Sigma^-1 y, which returns to the
// log-likelihood as -1/2 tr(Sigma^-1 G), and the M-step forms the shared
// covariance from G and the new means.
//
// Per 128-point tile the transform warps write y' = y * scale (no squares) as fp16 into a
// data stage (the same 128-byte-swizzled layout as the EM kernels; PRECISE
// adds the rounding remainder as a second piece).  The stage is a K x MN
// matrix (K = points, MN = features) read as both operands of
//   G' += Y'^T Y'     (M = 128 features, N = Dp features, K = 16 points per step)
// (PRECISE: hi^T hi + hi^T lo + lo^T hi).  Accumulators alternate between two
// tensor-memory buffers, one per flush period; four flush warps add each
// period's sums to this CTA's fp64 partial (one writer per element), and
// gram_reduce_kernel sums the partials in a fixed order and undoes scale^2.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "gmm_kernels.cuh"
#include "layout.cuh"
#include "ptx.cuh"
#include "transform.cuh"

namespace gmm {

namespace {

struct GramSmall {
  uint64_t full_a[4];        // stage s filled (128 transform threads)
  uint64_t empty_g[4][8];    // stage s, 16-row group g read by the MMAs
  uint64_t acc_full[2];      // period sums complete in buffer b
  uint64_t acc_empty[2];     // buffer b read out (128 flush threads)
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t poll_limit;       // follows abort_flag (read by the bounded waits)
};

template <int NP, int NCH, int NST>
struct GramCfg {
  static constexpr int kDp = NCH * kAtomElems;
  static constexpr int kPieceBytes = NCH * kChunkBytes;       // y' for 128 rows (no squares)
  static constexpr int kStageBytes = NP * kPieceBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffSmall = NST * kStageBytes;
  static constexpr int kEnd = kOffSmall + static_cast<int>(sizeof(GramSmall));
};

constexpr int kGramThreads = 288;   // transform 0-3, MMA 4, flush 5-8

// Two CTAs per SM (256 tensor-memory columns each): twice the rows in flight
// from HBM.
template <int NP, int NCH, int NST, bool XB>
__global__ void __launch_bounds__(kGramThreads, 2) gram_tc_kernel(const FusedArgs a, double* __restrict__ part) {
  using CF = GramCfg<NP, NCH, NST>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GramSmall* S = reinterpret_cast<GramSmall*>(sm + CF::kOffSmall);
  volatile uint32_t* abort_flag = &S->abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tgroup = blockIdx.x, n_tgroups = gridDim.x;
  int my_tiles = 0;
  if (tgroup < a.n_tiles) my_tiles = (a.n_tiles - 1 - tgroup) / n_tgroups + 1;
  const int F = a.flush_tiles;

  if (tid == 0) {
    S->abort_flag = 0;
    S->poll_limit = a.max_polls ? a.max_polls : kMaxPolls;
    for (int i = 0; i < NST; ++i) {
      mbar_init(&S->full_a[i], 128);
      for (int g = 0; g < 8; ++g) mbar_init(&S->empty_g[i][g], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S->acc_full[i], 1);
      mbar_init(&S->acc_empty[i], 128);
    }
    mbar_init(&S->drain, 1);
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(&S->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S->tmem_base;

  if (warp < 4) {
    transform_warps<CF, GramSmall, NP, NCH, NST, XB, false, false>(a, sm, S, abort_flag, tid, tgroup, n_tgroups,
                                                                   my_tiles);
  } else if (warp == 4) {
    if (lane == 0) {
      const uint32_t sA = smem_u32(sm + CF::kOffA);
      const uint32_t idesc = idesc_f16(0, 1, 1, 128, CF::kDp);
      for (int j = 0; j < my_tiles; ++j) {
        if (*abort_flag) break;
        const int s = j % NST, p = j / F, b = p & 1;
        const bool first = j % F == 0;
        mbar_wait(&S->full_a[s], static_cast<uint32_t>((j / NST) & 1), abort_flag, a.status);
        if (first && p >= 2) mbar_wait(&S->acc_empty[b], static_cast<uint32_t>(((p >> 1) - 1) & 1), abort_flag, a.status);
        tc_fence_after();
        const uint32_t stage = sA + s * CF::kStageBytes;
        const uint32_t acc = tmem + 128u * static_cast<uint32_t>(b);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
          for (int pr = 0; pr < (NP == 1 ? 1 : 3); ++pr) {
            const int pa = pr == 2 ? 1 : 0;   // piece of the A side
            const int pb = pr == 1 ? 1 : 0;   // piece of the B side
            const uint64_t ad = sdesc_sw128(stage + pa * CF::kPieceBytes + 2048 * kk, kChunkBytes, 1024);
            const uint64_t bd = sdesc_sw128(stage + pb * CF::kPieceBytes + 2048 * kk, kChunkBytes, 1024);
            mma_f16_ss(acc, ad, bd, idesc, (first && kk == 0 && pr == 0) ? 0u : 1u);
          }
          // rows 16 kk .. 16 kk + 15 of the stage are no longer needed
          mma_commit(&S->empty_g[s][kk]);
        }
        if ((j + 1) % F == 0 || j + 1 == my_tiles) mma_commit(&S->acc_full[b]);
      }
      mma_commit(&S->drain);
      mbar_wait_final(&S->drain, 0, a.status);
    }
    __syncwarp();
  } else {
    // flush warps: lane quarter (warp & 3) of each period's buffer into the
    // CTA's partial G (row = feature of the lane, columns = features)
    const int q = warp & 3;
    const int i = 32 * q + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    double* prow = part + (static_cast<int64_t>(blockIdx.x) * a.D + i) * a.D;
    const int n_periods = my_tiles > 0 ? (my_tiles - 1) / F + 1 : 0;
    for (int p = 0; p < n_periods; ++p) {
      const int b = p & 1;
      mbar_wait(&S->acc_full[b], static_cast<uint32_t>((p >> 1) & 1), abort_flag, a.status);
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < CF::kDp; c += 16) {
        float w[16];
        tmem_ld16(tmem + 128u * static_cast<uint32_t>(b) + lane_off + c, w);
        tmem_wait_ld();
        if (i < a.D) {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (c + e < a.D) red_add_f64(prow + c + e, static_cast<double>(w[e]));
        }
      }
      tc_fence_before();
      mbar_arrive(&S->acc_empty[b]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int NP, int NCH, int NST>
const void* gram_fn_t(bool xb) {
  return xb ? reinterpret_cast<const void*>(&gram_tc_kernel<NP, NCH, NST, true>)
            : reinterpret_cast<const void*>(&gram_tc_kernel<NP, NCH, NST, false>);
}

}  // namespace

// Stages of y' only (no squares), sized for two CTAs per SM: FAST three
// stages, PRECISE (two pieces) two at D <= 64, one above.
const void* gram_handle(int np, int nch, bool xb) {
  if (np == 1) return nch == 1 ? gram_fn_t<1, 1, 3>(xb) : gram_fn_t<1, 2, 3>(xb);
  return nch == 1 ? gram_fn_t<2, 1, 2>(xb) : gram_fn_t<2, 2, 1>(xb);
}

size_t gram_smem(int np, int nch) {
  size_t b = np == 1 ? (nch == 1 ? GramCfg<1, 1, 3>::kEnd : GramCfg<1, 2, 3>::kEnd)
                     : (nch == 1 ? GramCfg<2, 1, 2>::kEnd : GramCfg<2, 2, 1>::kEnd);
  return b + 1024;
}

int gram_threads() { return kGramThreads; }

}  // namespace gmm
