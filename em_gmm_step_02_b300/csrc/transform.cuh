// transform.cuh -- the transform warps of the EM kernels: each 128-point tile
// of X becomes the fp16 operand pieces [x' | x'^2] (PRECISE: hi and lo parts
// of each) in the 128-byte-swizzled K-major layout of a data stage.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "common.cuh"
#include "gmm_kernels.cuh"
#include "layout.cuh"
#include "ptx.cuh"

namespace gmm {

// ============================================================== data transform
// 16-byte load that bypasses L1 (each data tile is read once per SM).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// The four transform warps turn each 128-point tile of X into the two fp16
// operand pieces [x' | x'^2] (PRECISE: hi and lo parts of each), with
// x' = (x - shift) * scale, in the swizzled K-major layout of the data stage.
// Thread `tid` owns one 8-feature unit of every RPP-th row.  All loads of a
// tile are issued together (and, when the registers allow, one tile ahead)
// so that the whole tile is in flight at once.
// kSq = false writes x' only (the Gram matrix needs no squares; its stage
// holds one 64-feature block column per atom and no x'^2 part).
template <typename CF, typename SmallT, int NP, int NCH, int NST, bool XB, bool kTopm, bool kSq = true>
__device__ __forceinline__ void transform_warps(const FusedArgs& a, uint8_t* sm, SmallT* S,
                                                volatile uint32_t* abort_flag, int tid, int tgroup,
                                                int n_tgroups, int my_tiles) {
  constexpr int UPR = 8 * NCH;               // 8-feature units per row
  constexpr int RPP = 128 / UPR;             // rows per pass of the 128 threads
  constexpr int NPASS = 128 / RPP;
  constexpr int W = XB ? 4 : 8;              // 32-bit words per unit
  constexpr int NBATCH = (XB || NCH == 1) ? 1 : 2;
  constexpr int NB = NPASS / NBATCH;
  const int ch = tid % UPR;
  const int r0 = tid / UPR;
  const int d0 = ch * 8;
  const Meta* meta = a.meta;
  const float scale = meta->scale;
  float nshift[8];                           // -shift * scale
#pragma unroll
  for (int e = 0; e < 8; ++e) nshift[e] = d0 + e < a.D ? -meta->shift[d0 + e] * scale : 0.f;
  const bool vec = (a.D % 8) == 0;
  const bool unit_in = d0 < a.D;
  uint32_t buf[NB][W];

  auto load_batch = [&](int t, int b) {
#pragma unroll
    for (int p = 0; p < NB; ++p) {
      const int row = r0 + RPP * (b * NB + p);
      const int64_t n = static_cast<int64_t>(t) * kBN + row;
#pragma unroll
      for (int e = 0; e < W; ++e) buf[p][e] = 0u;
      if (n < a.N && unit_in) {
        if constexpr (XB) {
          const uint16_t* xr = static_cast<const uint16_t*>(a.X) + n * a.D + d0;
          if (vec) {
            const uint4 v = ldg_stream_v4(xr);
            buf[p][0] = v.x; buf[p][1] = v.y; buf[p][2] = v.z; buf[p][3] = v.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (d0 + e < a.D) buf[p][e >> 1] |= static_cast<uint32_t>(__ldg(xr + e)) << (16 * (e & 1));
          }
        } else {
          const float* xr = static_cast<const float*>(a.X) + n * a.D + d0;
          if (vec) {
            const uint4 v0 = ldg_stream_v4(xr);
            const uint4 v1 = ldg_stream_v4(xr + 4);
            buf[p][0] = v0.x; buf[p][1] = v0.y; buf[p][2] = v0.z; buf[p][3] = v0.w;
            buf[p][4] = v1.x; buf[p][5] = v1.y; buf[p][6] = v1.z; buf[p][7] = v1.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (d0 + e < a.D) buf[p][e] = __float_as_uint(__ldg(xr + e));
          }
        }
      }
    }
  };

  auto store_batch = [&](int t, int b, uint8_t* stage, int s, int use) {
#pragma unroll
    for (int p = 0; p < NB; ++p) {
      const int i = b * NB + p;
      const int row = r0 + RPP * i;
      // rows 16g..16g+15 of the stage are free once the statistics MMA of the
      // stage's previous tile has consumed them
      if ((RPP * i) % 16 == 0 && use > 0)
        mbar_wait(&S->empty_g[s][(RPP * i) / 16], (use - 1) & 1, abort_flag, a.status);
      const bool valid = static_cast<int64_t>(t) * kBN + row < a.N;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v;
        if constexpr (XB) v = __uint_as_float((e & 1) ? (buf[p][e >> 1] & 0xffff0000u) : (buf[p][e >> 1] << 16));
        else v = __uint_as_float(buf[p][e]);
        // bf16 data in FAST are never shifted, and rows beyond N were loaded as
        // zeros, so the plain scaling already leaves those rows zero
        if constexpr (XB && NP == 1) x[e] = v * scale;
        else x[e] = valid ? fmaf(v, scale, nshift[e]) : 0.f;
      }
      const uint32_t off = (ch / 8) * kChunkBytes + sw128_off(row, ch % 8);
      const uint32_t off2 = off + NCH * kChunkBytes;
      if constexpr (NP == 1) {
        uint4 hx, hq;
        hx.x = pack_f16x2(x[0], x[1]); hx.y = pack_f16x2(x[2], x[3]);
        hx.z = pack_f16x2(x[4], x[5]); hx.w = pack_f16x2(x[6], x[7]);
        if (XB) {
          // bf16 data scaled by a power of two are exact in fp16, so the
          // fp16 square of the packed value rounds the exact x'^2 once
          hq.x = sq_f16x2(hx.x); hq.y = sq_f16x2(hx.y); hq.z = sq_f16x2(hx.z); hq.w = sq_f16x2(hx.w);
        } else {
          hq.x = pack_f16x2(x[0] * x[0], x[1] * x[1]); hq.y = pack_f16x2(x[2] * x[2], x[3] * x[3]);
          hq.z = pack_f16x2(x[4] * x[4], x[5] * x[5]); hq.w = pack_f16x2(x[6] * x[6], x[7] * x[7]);
        }
        *reinterpret_cast<uint4*>(stage + off) = hx;
        if constexpr (kSq) *reinterpret_cast<uint4*>(stage + off2) = hq;
      } else {
        float xh[8], xl[8], qh[8], ql[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          xh[e] = __half2float(__float2half_rn(x[e]));
          xl[e] = x[e] - xh[e];
          const float q = x[e] * x[e];
          qh[e] = __half2float(__float2half_rn(q));
          ql[e] = q - qh[e];
        }
        uint4 v;
        v.x = pack_f16x2(xh[0], xh[1]); v.y = pack_f16x2(xh[2], xh[3]);
        v.z = pack_f16x2(xh[4], xh[5]); v.w = pack_f16x2(xh[6], xh[7]);
        *reinterpret_cast<uint4*>(stage + off) = v;
        if constexpr (kSq) {
          v.x = pack_f16x2(qh[0], qh[1]); v.y = pack_f16x2(qh[2], qh[3]);
          v.z = pack_f16x2(qh[4], qh[5]); v.w = pack_f16x2(qh[6], qh[7]);
          *reinterpret_cast<uint4*>(stage + off2) = v;
        }
        v.x = pack_f16x2(xl[0], xl[1]); v.y = pack_f16x2(xl[2], xl[3]);
        v.z = pack_f16x2(xl[4], xl[5]); v.w = pack_f16x2(xl[6], xl[7]);
        *reinterpret_cast<uint4*>(stage + CF::kPieceBytes + off) = v;
        if constexpr (kSq) {
          v.x = pack_f16x2(ql[0], ql[1]); v.y = pack_f16x2(ql[2], ql[3]);
          v.z = pack_f16x2(ql[4], ql[5]); v.w = pack_f16x2(ql[6], ql[7]);
          *reinterpret_cast<uint4*>(stage + CF::kPieceBytes + off2) = v;
        }
      }
    }
  };

  const int nst = kTopm ? 1 : NST;
  if (NBATCH == 1 && my_tiles > 0) load_batch(tgroup, 0);
  int t = tgroup;
#pragma unroll 1
  for (int j = 0; j < my_tiles; ++j, t += n_tgroups) {
    // (no early exit on an abort: every wait below returns at once after one,
    // so the loop runs out quickly and every barrier still sees all its threads)
    const int s = j % nst, use = j / nst;
    uint8_t* stage = sm + CF::kOffA + s * CF::kStageBytes;
#pragma unroll
    for (int b = 0; b < NBATCH; ++b) {
      if (NBATCH > 1) load_batch(t, b);
      store_batch(t, b, stage, s, use);
    }
    fence_proxy_async_smem();
    mbar_arrive(&S->full_a[s]);
    if (NBATCH == 1 && j + 1 < my_tiles) load_batch(t + n_tgroups, 0);
  }
}

}  // namespace gmm
