// wp_bwd.cu -- helper kernels of the closed-form LoRA backward.
//
// Unsloth fast_lora walkthrough, sections 2 and 4: the backward of Y = X W^T + s (X A^T) B^T
// is written out by hand, dX = dY W + s (dY B) A, dA = s (dY B)^T X, dB = s dY^T (X A^T),
// with only X kept from the forward and the 4-bit weight dequantised when W is needed.
// The large contraction (dX, including G = dY B) runs on the fused tensor-core kernel and the
// two reductions over tokens (dA, dB) on the token-contraction kernel (wp_tokgemm.cu); the
// kernels here prepare the dX pass's operands:
//
//   transpose_bf16_kernel    dst[c, r] = src[r, c]                (W^T, B^T, A^T operands)
//   nf4_dequant_t_kernel     dst[k, n] = bf16(fl32(level[q[n, k]]) * absmax[n, k / 64])
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_ptx.cuh"

namespace wp {

namespace {

__device__ __forceinline__ uint16_t to_bf16(float v) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
  return h;
}

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

// W [N, K] 4-bit (row-major codes, element 2k in the high nibble of byte k; one fp32 scale
// per 64 elements) -> W^T [K, N] bf16.  Tile: 64 rows of W x 128 elements of K.  Each
// thread decodes 8 consecutive elements of one row (4 code bytes, one block scale) into
// a K-major shared tile; the write-out sends 8 consecutive n of one k per 16-byte store.
__global__ void __launch_bounds__(256) nf4_dequant_t_kernel(const uint8_t* __restrict__ codes,
                                                            const float* __restrict__ absmax,
                                                            int N, int K, const NF4Table tab,
                                                            uint16_t* __restrict__ dst,
                                                            long long ld_d) {
  __shared__ __align__(16) uint16_t tile[128][64 + 8];    // [k][n], rows padded by 16 bytes
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = tab.level[threadIdx.x];
  __syncthreads();
  const int n0 = blockIdx.y * 64, k0 = blockIdx.x * 128;
  for (int e = threadIdx.x; e < 64 * 16; e += 256) {         // 64 rows x 16 groups of 8
    const int rr = e % 64, g = e / 64;                      // lanes on rows: conflict-free stores
    const int n = n0 + rr, k = k0 + 8 * g;
    uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (n < N && k < K) {                                   // K % 64 == 0: all 8 exist
      const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + static_cast<long long>(n) * (K / 2) + k / 2);
      const float am = absmax[static_cast<long long>(n) * (K / 64) + k / 64];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = (w >> (8 * b)) & 0xFFu;
        v[2 * b] = to_bf16(lv[byte >> 4] * am);             // element k + 2b
        v[2 * b + 1] = to_bf16(lv[byte & 0xFu] * am);       // element k + 2b + 1
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) tile[8 * g + q][rr] = v[q];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 128 * 8; e += 256) {         // 128 k x 8 groups of 8 n
    const int kk = e / 8, g = e % 8;
    const int k = k0 + kk, n = n0 + 8 * g;
    if (k >= K || n >= N) continue;
    const uint4 w = *reinterpret_cast<const uint4*>(&tile[kk][8 * g]);
    if (n + 8 <= N) {
      *reinterpret_cast<uint4*>(dst + static_cast<long long>(k) * ld_d + n) = w;   // ld_d % 8 == 0
    } else {
      const uint16_t* h = &tile[kk][8 * g];
      for (int q = 0; q < N - n; ++q) dst[static_cast<long long>(k) * ld_d + n + q] = h[q];
    }
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

int launch_nf4_dequant_t(const void* codes, const float* absmax, int N, int K, const NF4Table& tab,
                         void* dst, long long ld_d, cudaStream_t stream) {
  dim3 grid((K + 127) / 128, (N + 63) / 64);
  nf4_dequant_t_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(codes), absmax, N, K,
                                                 tab, static_cast<uint16_t*>(dst), ld_d);
  return check_launch();
}

}  // namespace wp
