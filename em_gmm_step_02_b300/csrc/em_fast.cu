// em_fast.cu -- the FAST (single fp16 piece) EM kernel for sm_103a, with two
// softmax teams working on alternating tiles.
//
// Method: "Flash-GMM: A Memory-Efficient Kernel for Scalable Soft Clustering",
// section 2 (E-step responsibilities through a log-sum-exp over the K weighted
// Gaussian terms; M-step from responsibility-weighted sufficient statistics);
// the N x K responsibility matrix exists only as on-chip tiles.
//
// One CTA owns a 128-component slice; the CTAs of a thread-block cluster own
// the slices of one component group and walk the same 128-point tiles.  Per
// CTA, sixteen warps:
//   warps 0-3    transform: X rows -> fp16 [x' | x'^2] in one of two data
//                stages (tile j uses stage j & 1).
//   warps 4-7    team 0 and warps 8-11 team 1: team t handles the tiles
//                j = t, t + 2, ...; thread = one point row (TMEM lane), all
//                128 components of the slice.  Per tile: an online
//                max / sum over four 32-column chunks of the logits
//                (p = 2^(l - M_c + 10) kept as packed fp16 pairs, M_c the
//                running maximum), the row normaliser pushed to every CTA of
//                the cluster, then r * 2^10 = p * 2^(M_c - lse) by a packed
//                multiply, written as the R tile.
//   warp 12      allocates tensor memory and issues every tcgen05.mma:
//                logits of tile j into buffer j & 1 (M = 128 points,
//                N = 128 components, K = 2 Dp + one 16-wide constant step),
//                then the statistics of tile j - 1
//                ([S1 | S2] += R^T [x' | x'^2], M = 128 components, N = 2 Dp).
//   warps 13-14  S0: column sums of each R quarter in fp32 (CUDA cores), the
//                count statistic that would otherwise need its own tensor
//                memory columns.
// Tensor memory: logits 2 x 128 columns, statistics 2 Dp columns.
// Statistics leave tensor memory every `flush_tiles` tiles into fp64
// per-cluster partials (one writer per element, fixed order of additions).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "common.cuh"
#include "gmm_kernels.cuh"
#include "layout.cuh"
#include "ptx.cuh"
#include "transform.cuh"

namespace gmm {

namespace {

struct FastSmall {
  float xrecv[2][8][kBN];    // per team: row normalisers pushed by each CTA of the cluster
  double ll_red[8];
  uint64_t full_a[2];        // stage s filled (128 transform threads)
  uint64_t empty_g[2][8];    // stage s, 16-row group g read by the statistics MMA
  uint64_t p_full;           // parameter image and constant operand loaded
  uint64_t acc_full[2];      // logits of team t's current tile in buffer t
  uint64_t acc_empty[2];     // team t has read its logits (128 threads)
  uint64_t r_full[2][4];     // team t, lane quarter q written to its R slot (32 threads)
  uint64_t r_done[2][4];     // team t, quarter q read by the statistics MMA and both S0 warps
  uint64_t acc2_full[2];     // statistics of flush period f complete (barrier f & 1)
  uint64_t acc2_empty;       // statistics read out (the 128 threads of the flushing team)
  uint64_t xready[2];        // team t's receive slot filled by every CTA of the cluster
  uint64_t xfree[2];         // team t's slot in every CTA read (4 warps x C CTAs)
  uint64_t cready[2];        // MODE_TOPM: candidate lists of team t's rows received from every CTA
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t poll_limit;       // follows abort_flag (read by the bounded waits)
};

// Shared-memory plan: [stage 0 | stage 1 | parameter image | constant operand |
// ones operand | R ring | FastSmall].
template <int NCH>
struct FastCfg {
  static constexpr int kDp = NCH * kAtomElems;
  static constexpr int kPieceBytes = 2 * NCH * kChunkBytes;   // [x | x^2] for 128 rows
  static constexpr int kStageBytes = kPieceBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffP = 2 * kStageBytes;
  static constexpr int kOffC = kOffP + kPieceBytes;
  static constexpr int kOffOnes = kOffC + kConstBytes;
  static constexpr int kOffR = kOffOnes + kConstBytes;
  static constexpr int kRBytes = 4 * kRSlotBytes;            // 2 slots x 32 points x 128 components
  static constexpr int kOffSmall = kOffR + kRBytes;
  static constexpr int kEnd = kOffSmall + static_cast<int>(sizeof(FastSmall));
  static constexpr uint32_t kAccCol = 0;      // logit buffers at columns 0 and 128
  static constexpr uint32_t kStatCol = 256;   // [S1 | S2]
};

constexpr float kLog2R = 10.f;   // log2 of the responsibility scale (r is stored as r * 2^10)

// Slot-ring wait of team t's lane quarter q before it writes tile j (team
// index jj = j >> 1) into R slot q & 1.  The slot's previous user is quarter
// q - 2 of the same tile (q >= 2; same team, barrier phase jj) or quarter
// q + 2 of tile j - 1 (q < 2; the other team, its phase (j - 1) >> 1).  In
// both cases this warp's previous wait on that barrier was for the phase just
// before (tile j - 2 of the same barrier), so a parity test cannot be fooled
// by a phase two steps away.
__device__ __forceinline__ void r_slot_wait2(FastSmall* S, int t, int q, int j, volatile uint32_t* abort_flag,
                                             uint32_t* status) {
  if (q >= 2) {
    mbar_wait(&S->r_done[t][q - 2], static_cast<uint32_t>((j >> 1) & 1), abort_flag, status);
  } else if (j > 0) {
    mbar_wait(&S->r_done[t ^ 1][q + 2], static_cast<uint32_t>(((j - 1) >> 1) & 1), abort_flag, status);
  }
}

// Adds this thread's row of the statistics accumulator (tensor-memory lane =
// component, columns [S1 | S2]) to its fp64 partial row.
template <int DP>
__device__ __forceinline__ void flush_stats2(double* prow, uint32_t taddr, bool live) {
#pragma unroll 1
  for (int c = 0; c < 2 * DP; c += 16) {
    float w[16];
    tmem_ld16(taddr + c, w);
    tmem_wait_ld();
    if (live) {
#pragma unroll
      for (int e = 0; e < 16; ++e) red_add_f64(prow + c + e, static_cast<double>(w[e]));
    }
  }
}

// ------------------------------------------------------------------ teams
template <typename CF, int MODE>
__device__ __forceinline__ void team_loop(const FusedArgs& a, uint8_t* sm, FastSmall* S, volatile uint32_t* abort_flag,
                                          int t, int warp, int lane, int rank, int C, int tgroup, int n_tgroups,
                                          int my_tiles, uint32_t tmem, int kbase, int kvalid) {
  const int q = warp & 3;                    // TMEM lane quarter
  const int nl = 32 * q + lane;              // point row inside the tile
  const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
  const uint32_t acc = tmem + CF::kAccCol + 128u * static_cast<uint32_t>(t);
  constexpr bool given = MODE == MODE_GIVEN;
  constexpr bool lse_only = MODE == MODE_LSE;
  const bool exch = C > 1 && !given;
  const float is = a.meta->pinv;             // log2 units per accumulator unit
  const bool ll_row = MODE == MODE_EM && (nl % C) == rank;
  double ll = 0.0;
  float llf = 0.f;
  // MODE_GIVEN: the row normaliser of the team's next tile is loaded one tile
  // ahead, off the critical path of the current one
  auto lse_of = [&](int jt) {
    const int64_t nn = static_cast<int64_t>(tgroup + jt * n_tgroups) * kBN + nl;
    return (jt < my_tiles && nn < a.N) ? __ldg(a.lse_in + nn) : -CUDART_INF_F;
  };
  float lse_next = 0.f;
  if constexpr (given) lse_next = lse_of(t);
  for (int j = t; j < my_tiles; j += 2) {
    const int jj = j >> 1;
    const int64_t n = static_cast<int64_t>(tgroup + j * n_tgroups) * kBN + nl;
    const bool valid = n < a.N;
    uint32_t pk[64];                         // packed fp16 pairs of p (chunk c: pk[16c .. 16c + 15])
    float Mc[4];                             // running row maximum (accumulator units) after chunk c
    float lse;                               // row normaliser, log2 units
    float lse_cur = 0.f;
    if constexpr (given) {
      lse_cur = lse_next;
      lse_next = lse_of(j + 2);
    }
    mbar_wait(&S->acc_full[t], static_cast<uint32_t>(jj & 1), abort_flag, a.status);
    tc_fence_after();
    if constexpr (given) {
      // normaliser over all components from memory: r * 2^10 directly
      lse = valid ? lse_cur : -CUDART_INF_F;
      const float off = lse > -CUDART_INF_F ? kLog2R - lse : -CUDART_INF_F;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[32], w[32];
        tmem_ld32(acc + lane_off + 64 * h, v);
        tmem_ld32(acc + lane_off + 64 * h + 32, w);
        tmem_wait_ld();
        if (h == 1) {
          tc_fence_before();
          mbar_arrive(&S->acc_empty[t]);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          pk[32 * h + e] = pack_f16x2(ex2(fmaf(v[2 * e], is, off)), ex2(fmaf(v[2 * e + 1], is, off)));
          pk[32 * h + 16 + e] = pack_f16x2(ex2(fmaf(w[2 * e], is, off)), ex2(fmaf(w[2 * e + 1], is, off)));
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) Mc[c] = 0.f;
    } else if constexpr (lse_only) {
      // ---- this CTA's normaliser only: online max and sum over 32-column
      // chunks, nothing kept for a responsibility tile
      float M = -CUDART_INF_F;
      float ssum = 0.f;                      // sum of 2^(l - M) (log2 units)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float w0[32], w1[32];
        tmem_ld32(acc + lane_off + 64 * h, w0);
        tmem_ld32(acc + lane_off + 64 * h + 32, w1);
        tmem_wait_ld();
        if (h == 1) {
          tc_fence_before();
          mbar_arrive(&S->acc_empty[t]);
        }
        float mq[4] = {w0[0], w0[1], w0[2], w0[3]};
#pragma unroll
        for (int e = 4; e < 32; e += 4) {
          mq[0] = fmaxf(mq[0], w0[e]);
          mq[1] = fmaxf(mq[1], w0[e + 1]);
          mq[2] = fmaxf(mq[2], w0[e + 2]);
          mq[3] = fmaxf(mq[3], w0[e + 3]);
        }
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          mq[0] = fmaxf(mq[0], w1[e]);
          mq[1] = fmaxf(mq[1], w1[e + 1]);
          mq[2] = fmaxf(mq[2], w1[e + 2]);
          mq[3] = fmaxf(mq[3], w1[e + 3]);
        }
        const float Mn = fmaxf(M, fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])));
        if (Mn > M && M > -CUDART_INF_F) ssum *= ex2((M - Mn) * is);
        M = Mn;
        if (M > -CUDART_INF_F) {
          const float off = -M * is;
          float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            sq[e & 3] += ex2(fmaf(w0[e], is, off));
            sq[(e + 2) & 3] += ex2(fmaf(w1[e], is, off));
          }
          ssum += (sq[0] + sq[1]) + (sq[2] + sq[3]);
        }
      }
      lse = ssum > 0.f ? M * is + lg2(ssum) : -CUDART_INF_F;
      if (exch) {
        if (jj > 0) mbar_wait_cluster(&S->xfree[t], static_cast<uint32_t>((jj - 1) & 1), abort_flag, a.status);
        const uint32_t dst = smem_u32(&S->xrecv[t][rank][nl]);
        const uint32_t bar = smem_u32(&S->xready[t]);
        for (int r = 0; r < C; ++r) st_async_f32(mapa(dst, r), lse, mapa(bar, r));
        if (q == 0 && lane == 0) mbar_arrive_expect_tx(&S->xready[t], static_cast<uint32_t>(C * kBN * 4));
        mbar_wait_cluster(&S->xready[t], static_cast<uint32_t>(jj & 1), abort_flag, a.status);
        float vals[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) vals[r] = r < C ? S->xrecv[t][r][nl] : -CUDART_INF_F;
        __syncwarp();
        if (lane < C) mbar_arrive_remote_relaxed(mapa(smem_u32(&S->xfree[t]), static_cast<uint32_t>(lane)));
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
      // K group of this CTA: the slice itself without clusters (slice-major grid)
      const int64_t kgroup = C == 1 ? blockIdx.x : blockIdx.y;
      if (rank == 0 && valid) a.lse_part[kgroup * a.N + n] = lse;
      continue;
    } else {
      // ---- local online softmax over this CTA's 128 components
      float M = -CUDART_INF_F;
      float ssum = 0.f;                      // sum of 2^(l - M + 10)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[64];
        {
          float w0[32], w1[32];
          tmem_ld32(acc + lane_off + 64 * h, w0);
          tmem_ld32(acc + lane_off + 64 * h + 32, w1);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            v[e] = w0[e];
            v[32 + e] = w1[e];
          }
        }
        if (h == 1) {
          // the logit buffer is free for tile j + 2
          tc_fence_before();
          mbar_arrive(&S->acc_empty[t]);
        }
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 2 * h + c2;
          float mq[4] = {v[32 * c2], v[32 * c2 + 1], v[32 * c2 + 2], v[32 * c2 + 3]};
#pragma unroll
          for (int e = 4; e < 32; e += 4) {
            mq[0] = fmaxf(mq[0], v[32 * c2 + e]);
            mq[1] = fmaxf(mq[1], v[32 * c2 + e + 1]);
            mq[2] = fmaxf(mq[2], v[32 * c2 + e + 2]);
            mq[3] = fmaxf(mq[3], v[32 * c2 + e + 3]);
          }
          const float Mn = fmaxf(M, fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])));
          if (Mn > M && M > -CUDART_INF_F) ssum *= ex2((M - Mn) * is);
          M = Mn;
          Mc[c] = M;
          if (M > -CUDART_INF_F) {
            const float off = kLog2R - M * is;
            float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p0 = ex2(fmaf(v[32 * c2 + 2 * e], is, off));
              const float p1 = ex2(fmaf(v[32 * c2 + 2 * e + 1], is, off));
              sq[e & 3] += p0 + p1;
              pk[16 * c + e] = pack_f16x2(p0, p1);
            }
            ssum += (sq[0] + sq[1]) + (sq[2] + sq[3]);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[16 * c + e] = 0u;
          }
        }
      }
      const float lse_loc = ssum > 0.f ? M * is + lg2(ssum) - kLog2R : -CUDART_INF_F;
      lse = lse_loc;
      if (exch) {
        // push this CTA's row normaliser to every CTA of the cluster (once each
        // has read the slot's previous contents), then combine the C values
        if (jj > 0) mbar_wait_cluster(&S->xfree[t], static_cast<uint32_t>((jj - 1) & 1), abort_flag, a.status);
        const uint32_t dst = smem_u32(&S->xrecv[t][rank][nl]);
        const uint32_t bar = smem_u32(&S->xready[t]);
        for (int r = 0; r < C; ++r) st_async_f32(mapa(dst, r), lse_loc, mapa(bar, r));
        if (q == 0 && lane == 0) mbar_arrive_expect_tx(&S->xready[t], static_cast<uint32_t>(C * kBN * 4));
        mbar_wait_cluster(&S->xready[t], static_cast<uint32_t>(jj & 1), abort_flag, a.status);
        float vals[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) vals[r] = r < C ? S->xrecv[t][r][nl] : -CUDART_INF_F;
        // this warp has read its rows of the slot: tell every CTA of the
        // cluster (lane r signals CTA r).  The values are consumed below before
        // anything else happens, and a peer's next push into this slot waits
        // for the signal, so no release fence is needed.
        __syncwarp();
        if (lane < C) mbar_arrive_remote_relaxed(mapa(smem_u32(&S->xfree[t]), static_cast<uint32_t>(lane)));
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
      if (ll_row && valid) llf += lse;
      // r * 2^10 = p * 2^(M_c * is - lse)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float f = (valid && lse > -CUDART_INF_F && Mc[c] > -CUDART_INF_F) ? ex2(Mc[c] * is - lse) : 0.f;
        const __half2 f2 = __float2half2_rn(f);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          __half2 x = *reinterpret_cast<__half2*>(&pk[16 * c + e]);
          x = __hmul2(x, f2);
          pk[16 * c + e] = *reinterpret_cast<uint32_t*>(&x);
        }
      }
    }
    if constexpr (given) if (!valid) {
#pragma unroll
      for (int i = 0; i < 64; ++i) pk[i] = 0u;
    }
    // ---- R: this quarter's 32 rows into slot q & 1 (both 64-component halves)
    r_slot_wait2(S, t, q, j, abort_flag, a.status);
    uint8_t* rbase = sm + CF::kOffR + (q & 1) * kRSlotBytes;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 w;
        w.x = pk[32 * h + 4 * c];
        w.y = pk[32 * h + 4 * c + 1];
        w.z = pk[32 * h + 4 * c + 2];
        w.w = pk[32 * h + 4 * c + 3];
        *reinterpret_cast<uint4*>(rbase + h * 2 * kRSlotBytes + sw128_off(lane, c)) = w;
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&S->r_full[t][q]);
    // ---- statistics leave tensor memory at the end of a flush period
    if (((j + 1) % a.flush_tiles == 0) || (j + 1 == my_tiles)) {
      ll += static_cast<double>(llf);
      llf = 0.f;
      // Period f ends at tile j and is read out by the team of that tile.  Its
      // barrier (f & 1) serves every other period, so the phase wanted is
      // f >> 1; phase (f >> 1) - 1 (period f - 2) is complete by now, because
      // the statistics of period f - 1 started only after it was read out.
      const int fidx = j / a.flush_tiles;
      mbar_wait(&S->acc2_full[fidx & 1], static_cast<uint32_t>((fidx >> 1) & 1), abort_flag, a.status);
      tc_fence_after();
      const int kl = 32 * q + lane;
      flush_stats2<CF::kDp>(a.part + (static_cast<int64_t>(tgroup) * a.K_pad + kbase + kl) * a.F,
                            tmem + CF::kStatCol + lane_off, kl < kvalid);
      tc_fence_before();
      mbar_arrive(&S->acc2_empty);
    }
  }
  // log-likelihood partial of this CTA (both teams)
  if constexpr (MODE == MODE_EM) {
    ll += static_cast<double>(llf);
    for (int o = 16; o > 0; o >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, o);
    if (lane == 0) S->ll_red[warp - 4] = ll;
    named_bar_sync(1, 256);
    if (warp == 4 && lane == 0) {
      double tot = 0.0;
      for (int i = 0; i < 8; ++i) tot += S->ll_red[i];
      a.ll_part[tgroup * C + rank] = tot * kLn2;
    }
  }
}



// a, b: ascending lists of MAXM keys.  Leaves in a the MAXM smallest of the
// two, ascending: a[i] = min(a[i], b[MAXM - 1 - i]) is a bitonic sequence that
// holds them, which half-cleaners of stride MAXM/2, ..., 1 then sort.
template <int MAXM>
__device__ __forceinline__ void bitonic_keep_min(float (&a)[MAXM], const float (&b)[MAXM]) {
#pragma unroll
  for (int i = 0; i < MAXM; ++i) a[i] = fminf(a[i], b[MAXM - 1 - i]);
#pragma unroll
  for (int stride = MAXM / 2; stride >= 1; stride >>= 1)
#pragma unroll
    for (int i = 0; i < MAXM; ++i)
      if ((i & stride) == 0) {
        const float lo = fminf(a[i], a[i + stride]);
        const float hi = fmaxf(a[i], a[i + stride]);
        a[i] = lo;
        a[i + stride] = hi;
      }
}

// Merge four keys into a sorted list of MAXM, keeping the MAXM smallest
// (ascending).  The four are first sorted (a five-comparator network); then,
// as in bitonic_keep_min with the four padded by +inf to MAXM, the list's tail
// takes the elementwise minimum with the four reversed (only the two smallest
// matter when MAXM = 2) and half-cleaners sort the resulting bitonic sequence.
// Per key this costs 5.5 (MAXM = 4) or 9.5 (MAXM = 8) min/max operations
// instead of 2 MAXM for an insertion into the sorted list.
template <int MAXM>
__device__ __forceinline__ void merge_four(float (&a)[MAXM], float q0, float q1, float q2, float q3) {
  auto ce = [](float& x, float& y) {
    const float lo = fminf(x, y);
    y = fmaxf(x, y);
    x = lo;
  };
  ce(q0, q1);
  ce(q2, q3);
  ce(q0, q2);
  ce(q1, q3);
  ce(q1, q2);
  const float q[4] = {q0, q1, q2, q3};
  constexpr int kTail = MAXM < 4 ? MAXM : 4;
#pragma unroll
  for (int i = 0; i < kTail; ++i) a[MAXM - 1 - i] = fminf(a[MAXM - 1 - i], q[i]);
#pragma unroll
  for (int stride = MAXM / 2; stride >= 1; stride >>= 1)
#pragma unroll
    for (int i = 0; i < MAXM; ++i)
      if ((i & stride) == 0) ce(a[i], a[i + stride]);
}

// ------------------------------------------------------------------ top-m teams
// MODE_TOPM: each point's m largest responsibilities (over every component of
// the launch's K group) and their components, best first, ties to the lower
// index ("Flash-GMM", conclusion: multi-assignment read off the final
// responsibilities).  Per tile and row (team thread):
//   1. all 128 logits of the slice from tensor memory, the row maximum M, the
//      local normaliser, and the slice's MAXM best candidates, ranked by a key
//      (M - logit with its low seven bits replaced by the column: the order of
//      keys is the order of logits, equal truncated values fall back to the
//      lower column; truncation moves a logit by at most 2^-16 of its distance
//      to M);
//   2. the normaliser goes to every CTA of the cluster, the candidates (logit
//      in log2 units, component) to the CTA that finalises the row
//      (rank = row mod C);
//   3. the finalising CTA merges the C sorted lists and writes 2^(logit - lse)
//      and the components (one K group), or the group's best logits and its
//      normaliser (several K groups, merged by topm_combine_kernel).
// The candidate lists live in the R area (no statistics in this mode).
template <typename CF, int MAXM>
__device__ __forceinline__ void topm_team_loop(const FusedArgs& a, uint8_t* sm, FastSmall* S,
                                               volatile uint32_t* abort_flag, int t, int warp, int lane, int rank,
                                               int C, int tgroup, int n_tgroups, int my_tiles, uint32_t tmem,
                                               int kbase) {
  const int q = warp & 3;
  const int nl = 32 * q + lane;
  const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
  const uint32_t acc = tmem + CF::kAccCol + 128u * static_cast<uint32_t>(t);
  const float is = a.meta->pinv;
  const int rpc = kBN / C;                     // rows each CTA finalises
  const bool mine = (nl % C) == rank;
  const int m = a.topm;
  // candidate lists of team t: [source rank][row slot][MAXM] x (logit bits, component)
  uint8_t* cand = sm + CF::kOffR + t * (kBN * MAXM * 8);
  double ll = 0.0;
  float llf = 0.f;
  for (int j = t; j < my_tiles; j += 2) {
    const int jj = j >> 1;
    const int64_t n = static_cast<int64_t>(tgroup + j * n_tgroups) * kBN + nl;
    const bool valid = n < a.N;
    // pass 1: the row maximum
    float M;
    mbar_wait(&S->acc_full[t], static_cast<uint32_t>(jj & 1), abort_flag, a.status);
    tc_fence_after();
    {
      float v[128];
      tmem_ld32(acc + lane_off + 0, *reinterpret_cast<float(*)[32]>(v));
      tmem_ld32(acc + lane_off + 32, *reinterpret_cast<float(*)[32]>(v + 32));
      tmem_ld32(acc + lane_off + 64, *reinterpret_cast<float(*)[32]>(v + 64));
      tmem_ld32(acc + lane_off + 96, *reinterpret_cast<float(*)[32]>(v + 96));
      tmem_wait_ld();
      float mq[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
      for (int e = 4; e < 128; e += 4) {
        mq[0] = fmaxf(mq[0], v[e]);
        mq[1] = fmaxf(mq[1], v[e + 1]);
        mq[2] = fmaxf(mq[2], v[e + 2]);
        mq[3] = fmaxf(mq[3], v[e + 3]);
      }
      M = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
    }
    // pass 2, one 32-column chunk at a time (a loop, to keep the code small):
    // the normaliser's sum, and the slice's MAXM best keys in four independent
    // streams (column 32 c + e goes to stream e & 3) whose sorted lists are
    // then merged by bitonic networks; keys ascend, so the lists hold the
    // smallest keys = largest logits
    float key[4][MAXM];
#pragma unroll
    for (int st = 0; st < 4; ++st)
#pragma unroll
      for (int s = 0; s < MAXM; ++s) key[st][s] = __uint_as_float(0x7f7fffffu);
    const bool live = M > -CUDART_INF_F;
    const float off = live ? kLog2R - M * is : 0.f;
    float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float v[32];
      tmem_ld32(acc + lane_off + 32 * c, v);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        if (live) sq[e & 3] += ex2(fmaf(v[e], is, off));
        const float d = live ? fminf(M - v[e], 1e30f) : 1e30f;
        v[e] = __uint_as_float((__float_as_uint(d) & ~127u) | static_cast<uint32_t>(32 * c + e));
      }
      // stream st takes columns st, st + 4, ..., st + 28 of the chunk, in two
      // groups of four
#pragma unroll
      for (int st = 0; st < 4; ++st)
#pragma unroll
        for (int g = 0; g < 2; ++g)
          merge_four<MAXM>(key[st], v[st + 16 * g], v[st + 16 * g + 4], v[st + 16 * g + 8], v[st + 16 * g + 12]);
    }
    // the logit buffer is free for tile j + 2
    tc_fence_before();
    mbar_arrive(&S->acc_empty[t]);
    const float ssum = (sq[0] + sq[1]) + (sq[2] + sq[3]);
    const float lse_loc = ssum > 0.f ? M * is + lg2(ssum) - kLog2R : -CUDART_INF_F;
    if (C > 1) {
      if (jj > 0) mbar_wait_cluster(&S->xfree[t], static_cast<uint32_t>((jj - 1) & 1), abort_flag, a.status);
      const uint32_t dst = smem_u32(&S->xrecv[t][rank][nl]);
      const uint32_t bar = smem_u32(&S->xready[t]);
      for (int r = 0; r < C; ++r) st_async_f32(mapa(dst, r), lse_loc, mapa(bar, r));
      if (q == 0 && lane == 0) {
        mbar_arrive_expect_tx(&S->xready[t], static_cast<uint32_t>(C * kBN * 4));
        mbar_arrive_expect_tx(&S->cready[t], static_cast<uint32_t>(kBN * MAXM * 8));
      }
    }
    bitonic_keep_min<MAXM>(key[0], key[1]);
    bitonic_keep_min<MAXM>(key[2], key[3]);
    bitonic_keep_min<MAXM>(key[0], key[2]);
    // candidates in log2 units with their components
    float cv[MAXM];
    uint32_t ci[MAXM];
#pragma unroll
    for (int s = 0; s < MAXM; ++s) {
      const uint32_t b = __float_as_uint(key[0][s]);
      const float dd = __uint_as_float(b & ~127u);
      cv[s] = dd >= 1e29f ? -CUDART_INF_F : (M - dd) * is;
      ci[s] = static_cast<uint32_t>(kbase) + (b & 127u);
    }
    float lse = lse_loc;
    if (C > 1) {
      const int fin = nl % C;
      const uint32_t cdst = smem_u32(cand + ((rank * rpc + nl / C) * MAXM) * 8);
      const uint32_t cbar = mapa(smem_u32(&S->cready[t]), static_cast<uint32_t>(fin));
#pragma unroll
      for (int s = 0; s < MAXM; ++s)
        st_async_v2(mapa(cdst + 8u * s, static_cast<uint32_t>(fin)), __float_as_uint(cv[s]), ci[s], cbar);
      mbar_wait_cluster(&S->xready[t], static_cast<uint32_t>(jj & 1), abort_flag, a.status);
      float vals[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) vals[r] = r < C ? S->xrecv[t][r][nl] : -CUDART_INF_F;
      float mx = vals[0];
#pragma unroll
      for (int r = 1; r < 8; ++r) mx = fmaxf(mx, vals[r]);
      float s2 = 0.f;
      if (mx > -CUDART_INF_F) {
#pragma unroll
        for (int r = 0; r < 8; ++r) s2 += ex2(vals[r] - mx);
      }
      lse = s2 > 0.f ? mx + lg2(s2) : -CUDART_INF_F;
      mbar_wait_cluster(&S->cready[t], static_cast<uint32_t>(jj & 1), abort_flag, a.status);
      if (mine) {
        // C-way merge of the sorted lists of this row (the lists' heads in
        // registers, the next entry of the list that gave the output read back)
        float hv[8];
        uint32_t hi[8];
        int hp[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          hp[r] = 0;
          if (r < C) {
            const uint2 w = *reinterpret_cast<const uint2*>(cand + ((r * rpc + nl / C) * MAXM) * 8);
            hv[r] = __uint_as_float(w.x);
            hi[r] = w.y;
          } else {
            hv[r] = -CUDART_INF_F;
            hi[r] = 0xFFFFFFFFu;
          }
        }
#pragma unroll
        for (int s = 0; s < MAXM; ++s) {
          if (s < m) {
            int best = 0;
            float bv = hv[0];
            uint32_t bi = hi[0];
#pragma unroll
            for (int r = 1; r < 8; ++r)
              if (hv[r] > bv || (hv[r] == bv && hi[r] < bi)) {
                best = r;
                bv = hv[r];
                bi = hi[r];
              }
            cv[s] = bv;
            ci[s] = bi;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              if (r == best) {
                ++hp[r];
                if (hp[r] < MAXM) {
                  const uint2 w = *reinterpret_cast<const uint2*>(cand + ((r * rpc + nl / C) * MAXM + hp[r]) * 8);
                  hv[r] = __uint_as_float(w.x);
                  hi[r] = w.y;
                } else {
                  hv[r] = -CUDART_INF_F;
                  hi[r] = 0xFFFFFFFFu;
                }
              }
            }
          }
        }
      }
      // this warp has read its slot rows and candidate lists
      __syncwarp();
      if (lane < C) mbar_arrive_remote_relaxed(mapa(smem_u32(&S->xfree[t]), static_cast<uint32_t>(lane)));
    }
    if (mine && valid) {
      if (a.topm_groups == 1) {
        llf += lse;
#pragma unroll
        for (int s = 0; s < MAXM; ++s) {
          if (s < m) {
            a.topm_val[n * m + s] = lse > -CUDART_INF_F ? ex2(cv[s] - lse) : 0.f;
            a.topm_idx[n * m + s] = static_cast<int32_t>(ci[s]);
          }
        }
      } else {
        a.lse_part[static_cast<int64_t>(blockIdx.y) * a.N + n] = lse;
        const int64_t o = (static_cast<int64_t>(blockIdx.y) * a.N + n) * m;
#pragma unroll
        for (int s = 0; s < MAXM; ++s) {
          if (s < m) {
            a.topm_val[o + s] = cv[s];
            a.topm_idx[o + s] = static_cast<int32_t>(ci[s]);
          }
        }
      }
    }
  }
  // log-likelihood partial of this CTA (one K group)
  if (a.topm_groups == 1) {
    ll += static_cast<double>(llf);
    for (int o = 16; o > 0; o >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, o);
    if (lane == 0) S->ll_red[warp - 4] = ll;
    named_bar_sync(1, 256);
    if (warp == 4 && lane == 0) {
      double tot = 0.0;
      for (int i = 0; i < 8; ++i) tot += S->ll_red[i];
      a.ll_part[tgroup * C + rank] = tot * kLn2;
    }
  }
}

// ------------------------------------------------------------------ S0 warps
// Warp 13 + h sums components 64 h + 2 lane and + 1 of every R quarter (fp32,
// the same fp16 values the statistics MMA reads) and adds the sums to the
// count column of the partials at the end of each flush period.
template <typename CF>
__device__ __forceinline__ void s0_loop(const FusedArgs& a, uint8_t* sm, FastSmall* S, volatile uint32_t* abort_flag,
                                        int h, int lane, int tgroup, int my_tiles, int kbase, int kvalid) {
  float s0a = 0.f, s0b = 0.f;
  const uint32_t col = static_cast<uint32_t>(lane >> 2);   // 16-byte chunk of the row
  const uint32_t within = static_cast<uint32_t>(lane & 3) * 4u;
  for (int j = 0; j < my_tiles; ++j) {
    const int t = j & 1, jj = j >> 1;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      mbar_wait(&S->r_full[t][q], static_cast<uint32_t>(jj & 1), abort_flag, a.status);
      const uint8_t* base = sm + CF::kOffR + h * 2 * kRSlotBytes + (q & 1) * kRSlotBytes;
      float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int r = 0; r < 32; ++r) {
        const __half2 x = *reinterpret_cast<const __half2*>(base + sw128_off(r, col) + within);
        const float2 f = __half22float2(x);
        pa[r & 3] += f.x;
        pb[r & 3] += f.y;
      }
      s0a += (pa[0] + pa[1]) + (pa[2] + pa[3]);
      s0b += (pb[0] + pb[1]) + (pb[2] + pb[3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S->r_done[t][q]);
    }
    if (((j + 1) % a.flush_tiles == 0) || (j + 1 == my_tiles)) {
      const int kl = 64 * h + 2 * lane;
      double* prow = a.part + (static_cast<int64_t>(tgroup) * a.K_pad + kbase + kl) * a.F + 2 * CF::kDp;
      if (kl < kvalid) red_add_f64(prow, static_cast<double>(s0a));
      if (kl + 1 < kvalid) red_add_f64(prow + a.F, static_cast<double>(s0b));
      s0a = 0.f;
      s0b = 0.f;
    }
  }
}

// ------------------------------------------------------------------ MMA warp
template <typename CF, bool stats>
__device__ __forceinline__ void mma_loop(const FusedArgs& a, uint8_t* sm, FastSmall* S, volatile uint32_t* abort_flag,
                                         int slice, int my_tiles, uint32_t tmem, int n1) {
  const uint32_t sA = smem_u32(sm + CF::kOffA);
  const uint32_t sP = smem_u32(sm + CF::kOffP);
  const uint32_t sC = smem_u32(sm + CF::kOffC);
  const uint32_t sOnes = smem_u32(sm + CF::kOffOnes);
  const uint32_t sR = smem_u32(sm + CF::kOffR);
  const uint32_t idl = idesc_f16(0, 0, 0, 128, n1);
  const uint32_t ids = idesc_f16(0, 1, 1, 128, 2 * CF::kDp);
  const uint32_t stat = tmem + CF::kStatCol;
  int fidx = 0;
  bool fresh = true;

  auto issue_logits = [&](int j) {
    const uint32_t stage = sA + (j & 1) * CF::kStageBytes;
    const uint32_t acc = tmem + CF::kAccCol + 128u * static_cast<uint32_t>(j & 1);
    uint32_t accf = 0;
    for (int c = 0; c < 2 * (CF::kDp / kAtomElems); ++c)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // K steps wholly inside the zero padding beyond D add nothing
        if ((c % (CF::kDp / kAtomElems)) * kAtomElems + 16 * kk >= a.D) continue;
        const uint64_t ad = sdesc_sw128(stage + c * kChunkBytes + 32 * kk, 16, 1024);
        const uint64_t bd = sdesc_sw128(sP + c * kChunkBytes + 32 * kk, 16, 1024);
        mma_f16_ss(acc, ad, bd, idl, accf);
        accf = 1;
      }
    // the logit constant: one more K step
    mma_f16_ss(acc, sdesc_none(sOnes, kConstLbo, kConstSbo), sdesc_none(sC, kConstLbo, kConstSbo), idl, 1);
    mma_commit(&S->acc_full[j & 1]);
    if (!stats)
      for (int g = 0; g < 8; ++g) mma_commit(&S->empty_g[j & 1][g]);
  };
  auto issue_stats = [&](int j) {
    const int t = j & 1, jj = j >> 1;
    const uint32_t stage = sA + t * CF::kStageBytes;
    if (fresh && fidx > 0) {
      mbar_wait(&S->acc2_empty, static_cast<uint32_t>((fidx - 1) & 1), abort_flag, a.status);
      tc_fence_after();
    }
    for (int q = 0; q < 4; ++q) {
      const uint32_t sRq = sR + (q & 1) * kRSlotBytes;
      mbar_wait(&S->r_full[t][q], static_cast<uint32_t>(jj & 1), abort_flag, a.status);
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint64_t ad = sdesc_sw128(sRq + 2048 * kk, 2 * kRSlotBytes, 1024);
        const uint64_t bd = sdesc_sw128(stage + q * 4096 + 2048 * kk, kChunkBytes, 1024);
        mma_f16_ss(stat, ad, bd, ids, fresh ? 0u : 1u);
        fresh = false;
        // rows 16 (2 q + kk) .. +15 of the stage are no longer needed
        mma_commit(&S->empty_g[t][2 * q + kk]);
      }
      mma_commit(&S->r_done[t][q]);
    }
    if (((j + 1) % a.flush_tiles == 0) || (j + 1 == my_tiles)) {
      mma_commit(&S->acc2_full[fidx & 1]);
      ++fidx;
      fresh = true;
    }
  };

  for (int j = 0; j < my_tiles; ++j) {
    if (*abort_flag) break;
    mbar_wait(&S->full_a[j & 1], static_cast<uint32_t>((j >> 1) & 1), abort_flag, a.status);
    if (j >= 2) mbar_wait(&S->acc_empty[j & 1], static_cast<uint32_t>(((j >> 1) - 1) & 1), abort_flag, a.status);
    tc_fence_after();
    issue_logits(j);
    if (stats && j >= 1) issue_stats(j - 1);
  }
  if (stats && my_tiles > 0 && !*abort_flag) issue_stats(my_tiles - 1);
}

// ------------------------------------------------------------------ kernel
template <int NCH, int MODE, int MAXM>
__global__ void __launch_bounds__(512, 1) em_fast_kernel(const FusedArgs a) {
  using CF = FastCfg<NCH>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FastSmall* S = reinterpret_cast<FastSmall*>(sm + CF::kOffSmall);
  volatile uint32_t* abort_flag = &S->abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr bool given = MODE == MODE_GIVEN;
  constexpr bool stats = MODE == MODE_EM || MODE == MODE_GIVEN;
  const int C = a.C;

  // The statistics pass, and the normaliser pass without clusters, launch
  // slice-major (blockIdx.x = slice): the CTAs that run at the same time share
  // their point tiles, which then come from L2 once per tile group instead of
  // once per slice.
  int rank, slice, tgroup, n_tgroups;
  if (given || (MODE == MODE_LSE && C == 1)) {
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
  // all 128 logit columns are computed: padded and dead components carry a
  // -inf constant, which the tensor core propagates to their logits
  const int n1 = kSlice;
  int my_tiles = 0;
  if (tgroup < a.n_tiles) my_tiles = (a.n_tiles - 1 - tgroup) / n_tgroups + 1;

  if (tid == 0) {
    S->abort_flag = 0;
    S->poll_limit = a.max_polls ? a.max_polls : kMaxPolls;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S->full_a[i], 128);
      for (int g = 0; g < 8; ++g) mbar_init(&S->empty_g[i][g], 1);
      mbar_init(&S->acc_full[i], 1);
      mbar_init(&S->acc_empty[i], 128);
      for (int q = 0; q < 4; ++q) {
        mbar_init(&S->r_full[i][q], 32);
        mbar_init(&S->r_done[i][q], 3);
      }
      mbar_init(&S->xready[i], 1);
      mbar_init(&S->xfree[i], 4 * C);
      mbar_init(&S->cready[i], 1);
    }
    mbar_init(&S->p_full, 1);
    mbar_init(&S->acc2_full[0], 1);
    mbar_init(&S->acc2_full[1], 1);
    mbar_init(&S->acc2_empty, 128);
    mbar_init(&S->drain, 1);
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(&S->tmem_base, 512);
    tmem_relinquish();
  }
  if (tid < 128) {
    // the data side of the constant K step: 2^15, 2^4, 2^-7 in columns 0..2
    // of every row (fp16 bit patterns), zeros elsewhere
    uint4* ones = reinterpret_cast<uint4*>(sm + CF::kOffOnes);
    for (int i = tid; i < kConstBytes / 16; i += 128) {
      const bool first = ((i * 16) / kConstLbo) % 2 == 0;
      ones[i] = first ? make_uint4(0x4C007800u, 0x00002000u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if (C > 1 && !given) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = S->tmem_base;

  // Register split of the 512 threads launched at 128 registers (65,536 in
  // all): transform warpgroup 112, the two softmax teams kTeamRegs, the MMA /
  // S0 warpgroup kRestRegs, with 128 (112 + 2 kTeamRegs + kRestRegs) <= 65,536,
  // i.e. 2 kTeamRegs + kRestRegs <= 400.  Per mode the teams take what their
  // loop needs and the rest goes to the MMA warpgroup (each choice is the one
  // without spills under -Xptxas -v).
  constexpr int kTeamRegs = MODE == MODE_EM ? 160 : MODE == MODE_GIVEN ? 136 : 144;
  constexpr int kRestRegs = MODE == MODE_EM ? 72 : MODE == MODE_GIVEN ? 120 : 104;
  static_assert(2 * kTeamRegs + kRestRegs <= 400, "register split exceeds the launch's registers");
  const int wg = warp >> 2;
  if (wg == 0) {
    regs_release<112>();
    if (a.x_bf16) transform_warps<CF, FastSmall, 1, NCH, 2, true, false>(a, sm, S, abort_flag, tid, tgroup, n_tgroups, my_tiles);
    else transform_warps<CF, FastSmall, 1, NCH, 2, false, false>(a, sm, S, abort_flag, tid, tgroup, n_tgroups, my_tiles);
  } else if (wg <= 2) {
    regs_claim<kTeamRegs>();
    if constexpr (MODE == MODE_TOPM)
      topm_team_loop<CF, MAXM>(a, sm, S, abort_flag, wg - 1, warp, lane, rank, C, tgroup, n_tgroups, my_tiles, tmem,
                               kbase);
    else
      team_loop<CF, MODE>(a, sm, S, abort_flag, wg - 1, warp, lane, rank, C, tgroup, n_tgroups, my_tiles, tmem, kbase,
                          kvalid);
  } else {
    regs_release<kRestRegs>();
    if (warp == 12) {
      if (lane == 0) {
        const uint32_t pbytes = static_cast<uint32_t>(CF::kPieceBytes);
        mbar_arrive_expect_tx(&S->p_full, pbytes + kConstBytes);
        const uint8_t* src = a.p_img + static_cast<size_t>(slice) * pbytes;
        for (uint32_t o = 0; o < pbytes; o += 16384) bulk_g2s(sm + CF::kOffP + o, src + o, 16384, &S->p_full);
        bulk_g2s(sm + CF::kOffC, a.c_img + static_cast<size_t>(slice) * kConstBytes, kConstBytes, &S->p_full);
        mbar_wait(&S->p_full, 0, abort_flag, a.status);
        tc_fence_after();
        mma_loop<CF, stats>(a, sm, S, abort_flag, slice, my_tiles, tmem, n1);
        // every copy and tensor-core operation of this CTA completes before
        // the tensor memory and shared memory are released (bounded waits
        // that do not give up early after another wait has failed)
        mbar_wait_final(&S->p_full, 0, a.status);
        mma_commit(&S->drain);
        mbar_wait_final(&S->drain, 0, a.status);
      }
      __syncwarp();
    } else if ((warp == 13 || warp == 14) && stats) {
      s0_loop<CF>(a, sm, S, abort_flag, warp - 13, lane, tgroup, my_tiles, kbase, kvalid);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (C > 1 && !given) cluster_sync();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int NCH>
const void* emfast_handle_nch(int mode, int maxm) {
  switch (mode) {
    case MODE_LSE: return reinterpret_cast<const void*>(&em_fast_kernel<NCH, MODE_LSE, 0>);
    case MODE_GIVEN: return reinterpret_cast<const void*>(&em_fast_kernel<NCH, MODE_GIVEN, 0>);
    case MODE_TOPM:
      if (maxm <= 2) return reinterpret_cast<const void*>(&em_fast_kernel<NCH, MODE_TOPM, 2>);
      if (maxm <= 4) return reinterpret_cast<const void*>(&em_fast_kernel<NCH, MODE_TOPM, 4>);
      return reinterpret_cast<const void*>(&em_fast_kernel<NCH, MODE_TOPM, 8>);
    // the single-pass EM step runs on the fused kernel (gmm_kernels.cu), which
    // measured faster than this kernel in that mode
    default: return nullptr;
  }
}

const void* emfast_handle(int nch, int mode, int maxm) {
  return nch == 1 ? emfast_handle_nch<1>(mode, maxm) : emfast_handle_nch<2>(mode, maxm);
}

size_t emfast_smem(int nch) {
  return (nch == 1 ? FastCfg<1>::kEnd : FastCfg<2>::kEnd) + 1024;
}

}  // namespace gmm
