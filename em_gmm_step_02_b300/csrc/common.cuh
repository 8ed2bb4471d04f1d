// common.cuh -- small device helpers shared by the EM-step kernels: constants
// in log2 units, fast base-2 exponent and logarithm, fp16 packing, and the
// fire-and-forget fp64 reduction used for the partial statistics.
#pragma once
#include <cuda_fp16.h>
#include <cstdint>

namespace gmm {

constexpr double kLog2e = 1.4426950408889634073599246810019;
constexpr double kLn2 = 0.69314718055994530941723212145818;
constexpr double kLog2Pi = 1.8378770664093454835606594728112;  // ln(2 pi)

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool cond) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"(static_cast<uint32_t>(cond)), "r"(id), "r"(nthreads) : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void red_add_f64(double* p, double v) {
  asm volatile("red.global.add.f64 [%0], %1;" :: "l"(p), "d"(v) : "memory");
}

__device__ __forceinline__ uint32_t sq_f16x2(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  h = __hmul2(h, h);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace gmm
