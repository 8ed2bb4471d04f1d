// selftest.cu -- diagnostic: one tensor-core contraction on operands given
// as ready-made shared-memory images, used by the tests to check the
// descriptor encodings and the tensor-memory read-back layout that the EM
// kernels rely on.  Not part of the EM data path.
#include <cuda_runtime.h>
#include <cstdint>

#include "layout.cuh"
#include "ptx.cuh"

using namespace gmm;

namespace {

constexpr int kOperandBytes = 64 * 1024;  // each operand buffer

// variant bit 0: 0 = both operands K-major (M=128, N=128, K=64)
//                1 = both operands MN-major (M=128, N=256, K=64)
// variant bit 1: 0 = fp16, 1 = bf16
// variant 4:     both operands K-major without swizzling (the layout of the
//                logit constant step), fp16, M=128, N=128, K=16
__global__ void __launch_bounds__(128, 1)
selftest_mma_kernel(int variant, const uint4* __restrict__ a_img, const uint4* __restrict__ b_img,
                    float* __restrict__ d_out, uint32_t* __restrict__ status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = base;
  uint8_t* sb = base + kOperandBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + 2 * kOperandBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 2 * kOperandBytes + 64);
  __shared__ uint32_t abort_flag[2];   // abort flag, poll limit

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool nosw = variant == 4;
  const bool mn = !nosw && (variant & 1) != 0;
  const uint32_t ab_type = nosw ? 0u : (variant >> 1) & 1;
  const int N = mn ? 256 : 128;
  const int a_bytes = nosw ? kConstBytes : 16384;   // 64 x 128 or 128 x 64 sixteen-bit elements
  const int b_bytes = nosw ? kConstBytes : (mn ? 32768 : 16384);

  for (int i = tid; i < a_bytes / 16; i += 128) reinterpret_cast<uint4*>(sa)[i] = a_img[i];
  for (int i = tid; i < b_bytes / 16; i += 128) reinterpret_cast<uint4*>(sb)[i] = b_img[i];
  fence_proxy_async_smem();
  if (tid == 0) {
    abort_flag[0] = 0;
    abort_flag[1] = kMaxPolls;
    mbar_init(bar, 1);
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    const uint32_t idesc = idesc_f16(ab_type, mn ? 1u : 0u, mn ? 1u : 0u, 128, N);
    if (nosw) {
      mma_f16_ss(tmem, sdesc_none(smem_u32(sa), kConstLbo, kConstSbo), sdesc_none(smem_u32(sb), kConstLbo, kConstSbo),
                 idesc, 0);
    }
    for (int k = 0; k < (nosw ? 0 : 4); ++k) {
      uint64_t ad, bd;
      if (!mn) {
        ad = sdesc_sw128(smem_u32(sa) + 32u * k, 16, 1024);
        bd = sdesc_sw128(smem_u32(sb) + 32u * k, 16, 1024);
      } else {
        ad = sdesc_sw128(smem_u32(sa) + 2048u * k, 8192, 1024);
        bd = sdesc_sw128(smem_u32(sb) + 2048u * k, 8192, 1024);
      }
      mma_f16_ss(tmem, ad, bd, idesc, k > 0);
    }
    mma_commit(bar);
  }
  __syncwarp();
  mbar_wait(bar, 0, abort_flag, status);
  tc_fence_after();
  const int row = warp * 32 + lane;
  for (int c = 0; c < N; c += 16) {
    float v[16];
    tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
    tmem_wait_ld();
    for (int j = 0; j < 16; ++j) d_out[row * N + c + j] = v[j];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

extern "C" int gmm_selftest_mma(int variant, const void* a_img, const void* b_img, float* d_out,
                                unsigned int* status, void* stream) {
  const size_t smem = 2 * kOperandBytes + 1024 + 1024;
  cudaError_t e = cudaFuncSetAttribute(selftest_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return -4;
  selftest_mma_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
      variant, static_cast<const uint4*>(a_img), static_cast<const uint4*>(b_img), d_out, status);
  e = cudaGetLastError();
  return e == cudaSuccess ? 0 : -4;
}
