// wp_bwd.cu -- helper kernels of the closed-form LoRA backward.
//
// Unsloth fast_lora walkthrough, sections 2 and 4: the backward of Y = X W^T + s (X A^T) B^T
// is written out by hand, dX = dY W + s (dY B) A, dA = s (dY B)^T X, dB = s dY^T (X A^T),
// with only X kept from the forward and the 4-bit weight dequantised when W is needed.
// The large contraction (dX, including G = dY B) runs on the fused tensor-core kernel and the
// two reductions over tokens (dA, dB) on the token-contraction kernel (wp_tokgemm.cu); the
// kernels here prepare the dX pass's operands:
//
//   transpose_bf16_kernel    dst[c, r] = src[r, c]                (B^T, A^T operands)
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_ptx.cuh"

namespace wp {

namespace {

int check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace

// 64 x 64 tiles through shared memory; 256 threads.  Both loops are unrolled so that a
// thread's 16 loads are all in flight before its first shared-memory store.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ src,
                                                             long long ld_s, int R, int C,
                                                             uint16_t* __restrict__ dst,
                                                             long long ld_d) {
  __shared__ uint16_t tile[64][65];
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
#pragma unroll
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int rr = i / 64, cc = i % 64;
    const int r = r0 + rr, c = c0 + cc;
    tile[rr][cc] = (r < R && c < C) ? src[(long long)r * ld_s + c] : 0;
  }
  __syncthreads();
#pragma unroll
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int cc = i / 64, rr = i % 64;
    const int r = r0 + rr, c = c0 + cc;
    if (r < R && c < C) dst[(long long)c * ld_d + r] = tile[rr][cc];
  }
}

int launch_transpose_bf16(const void* src, long long ld_s, int R, int C, void* dst, long long ld_d,
                          cudaStream_t stream) {
  if (R <= 0 || C <= 0) return WP_OK;
  dim3 grid((C + 63) / 64, (R + 63) / 64);
  transpose_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(src), ld_s, R, C,
                                                  static_cast<uint16_t*>(dst), ld_d);
  return check_launch();
}


}  // namespace wp
