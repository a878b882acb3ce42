// wp_chain.cu -- the elementwise passes of the unfused dynamic-LoRA chain (the "exact" tier).
//
// sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM", Motivation and
// Modifications: before the fused design, a dynamic LoRA layer ran the base linear, then
// x @ A^T, then that @ B^T, then one multiplication per scale (alpha/rank, adapter strength,
// request scale), then the add onto the base output, every intermediate a BF16 tensor; the
// PR's exact tier keeps that chain and only skips multiplications by exactly 1.0.  The
// GEMMs of the chain run on the library's tensor-core kernel; the two passes here are the
// chain's elementwise steps:
//
//   scale:  d = bf16(d * c)           (d bf16, c an fp32 scale)
//   add:    Y = bf16(Y + d)           (Y bf16, d bf16 or fp32)
//
// Each result is the correctly rounded (round-to-nearest-even) bf16 of the exact value: the
// product or sum is formed exactly in double (8 + 24 significant bits, or the sum of two
// such values a few binades apart), narrowed to float by round-to-odd (truncate, then set
// the last bit when anything was dropped) and only then rounded to bf16, a single rounding
// in effect (a round-to-odd step with at least two spare bits does not disturb a later
// round-to-nearest).
//
// HBM-bound: per element 2 (scale) or 4-6 (add) bytes read and 2 written; each thread moves
// 8 consecutive columns of one row with 16-byte loads and stores.
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_ptx.cuh"

namespace wp {

namespace {

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// round-to-nearest-even bf16 of a double, through a round-to-odd float
__device__ __forceinline__ uint16_t bf16_of_double(double x) {
  float f = __double2float_rz(x);
  if (static_cast<double>(f) != x) f = __uint_as_float(__float_as_uint(f) | 1u);
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

__global__ void __launch_bounds__(256) chain_kernel(const ChainParams q) {
  const long long oct = q.N >> 3;                       // 8-column units per row
  const long long units = q.T * oct;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < units; u += stride) {
    const long long row = u / oct;
    const long long col = (u - row * oct) << 3;
    uint16_t* y = q.Y + row * q.ldy + col;
    const uint4 y4 = *reinterpret_cast<const uint4*>(y);
    const uint32_t yw[4] = {y4.x, y4.y, y4.z, y4.w};
    float dv[8];
    if (q.mode == kChainAdd && q.d_f32) {
      const float* dp = static_cast<const float*>(q.d) + row * q.ldd + col;
      const float4 a = *reinterpret_cast<const float4*>(dp);
      const float4 b = *reinterpret_cast<const float4*>(dp + 4);
      dv[0] = a.x; dv[1] = a.y; dv[2] = a.z; dv[3] = a.w; dv[4] = b.x; dv[5] = b.y; dv[6] = b.z; dv[7] = b.w;
    } else if (q.mode == kChainAdd) {
      const uint4 d4 = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(q.d) + row * q.ldd + col);
      const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        dv[2 * k] = bf16_to_f32(dw[k] & 0xffffu);
        dv[2 * k + 1] = bf16_to_f32(dw[k] >> 16);
      }
    }
    uint32_t ow[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint16_t o[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        // element 2k is the low half of word k, element 2k + 1 the high half
        const double v = static_cast<double>(bf16_to_f32(j ? (yw[k] >> 16) : (yw[k] & 0xffffu)));
        const double r = q.mode == kChainScale ? v * static_cast<double>(q.c)
                                               : v + static_cast<double>(dv[2 * k + j]);
        o[j] = bf16_of_double(r);
      }
      ow[k] = static_cast<uint32_t>(o[0]) | (static_cast<uint32_t>(o[1]) << 16);
    }
    *reinterpret_cast<uint4*>(y) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  }
}

}  // namespace

int launch_chain(const ChainParams& q, cudaStream_t stream) {
  const long long units = q.T * (q.N >> 3);
  if (units <= 0) return WP_OK;
  long long blocks = (units + 255) / 256;
  const long long cap = static_cast<long long>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  chain_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(q);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace wp
