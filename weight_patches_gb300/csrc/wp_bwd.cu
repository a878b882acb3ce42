// wp_bwd.cu -- helper kernels of the closed-form LoRA backward.
//
// Unsloth fast_lora walkthrough, sections 2 and 4: the backward of Y = X W^T + s (X A^T) B^T
// is written out by hand, dX = dY W + s (dY B) A, dA = s (dY B)^T X, dB = s dY^T (X A^T),
// with only X kept from the forward and the 4-bit weight dequantised when W is needed.
// The large contraction (dX, including G = dY B) runs on the fused tensor-core kernel; the
// kernels here prepare its operands and compute the two skinny reductions over tokens:
//
//   transpose_bf16_kernel    dst[c, r] = src[r, c]                (W^T, B^T, A^T operands)
//   nf4_dequant_t_kernel     dst[k, n] = bf16(fl32(level[q[n, k]]) * absmax[n, k / 64])
//   skinny_partial_kernel    part[c, i, j] = sum_{t in chunk c} P[t, i] Q[t, j]   (fp32)
//   skinny_finish_kernel     out = scale * sum_c part[c]  (fixed order: deterministic)
#include <cuda_runtime.h>

#include "wp_internal.h"

namespace wp {

namespace {

__device__ __forceinline__ float ld_f32(const void* p, int dtype, long long i) {
  if (dtype == WP_FP32) return static_cast<const float*>(p)[i];
  return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16);
}

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

// 64 x 64 tiles through shared memory; 256 threads.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ src,
                                                             long long ld_s, int R, int C,
                                                             uint16_t* __restrict__ dst,
                                                             long long ld_d) {
  __shared__ uint16_t tile[64][65];
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int rr = i / 64, cc = i % 64;
    const int r = r0 + rr, c = c0 + cc;
    tile[rr][cc] = (r < R && c < C) ? src[(long long)r * ld_s + c] : 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int cc = i / 64, rr = i % 64;
    const int r = r0 + rr, c = c0 + cc;
    if (r < R && c < C) dst[(long long)c * ld_d + r] = tile[rr][cc];
  }
}

// W [N, K] 4-bit (row-major codes, element 2k in the high nibble of byte k; one fp32 scale
// per 64 elements) -> W^T [K, N] bf16.  Tiles of 64 rows of W x 128 elements of K.
__global__ void __launch_bounds__(256) nf4_dequant_t_kernel(const uint8_t* __restrict__ codes,
                                                            const float* __restrict__ absmax,
                                                            int N, int K, const NF4Table tab,
                                                            uint16_t* __restrict__ dst,
                                                            long long ld_d) {
  __shared__ uint16_t tile[64][129];
  const int n0 = blockIdx.y * 64, k0 = blockIdx.x * 128;
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {         // 64 rows x 64 bytes
    const int rr = i / 64, bb = i % 64;
    const int n = n0 + rr, k = k0 + 2 * bb;
    uint16_t lo = 0, hi = 0;
    if (n < N && k < K) {
      const uint8_t byte = codes[(long long)n * (K / 2) + k / 2];
      const float am = absmax[(long long)n * (K / 64) + k / 64];
      hi = to_bf16(tab.level[byte >> 4] * am);                 // element k
      lo = to_bf16(tab.level[byte & 0xF] * am);                // element k + 1
    }
    tile[rr][2 * bb] = hi;
    tile[rr][2 * bb + 1] = lo;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 128; i += 256) {
    const int kk = i / 64, rr = i % 64;
    const int n = n0 + rr, k = k0 + kk;
    if (n < N && k < K) dst[(long long)k * ld_d + n] = tile[rr][kk];
  }
}

// part[c, i, j] = sum over t in [c * tc, (c + 1) * tc) of P[t, i] * Q[t, j], j < R <= 64.
// One thread per column i of P; Q's rows for the chunk are staged in shared memory.
__global__ void __launch_bounds__(128) skinny_partial_kernel(const void* __restrict__ P, int p_dtype,
                                                             long long ldp, int T, int M,
                                                             const float* __restrict__ Q,
                                                             long long ldq, int R, int tc,
                                                             float* __restrict__ part) {
  constexpr int kTT = 32;                                      // token rows per step
  __shared__ float qs[kTT][64];
  const int i = blockIdx.x * 128 + threadIdx.x;
  const int c = blockIdx.y;
  const int t_begin = c * tc, t_end = min(T, t_begin + tc);
  float acc[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) acc[j] = 0.f;
  for (int t0 = t_begin; t0 < t_end; t0 += kTT) {
    const int nt = min(kTT, t_end - t0);
    __syncthreads();
    for (int e = threadIdx.x; e < kTT * 64; e += 128) {
      const int tt = e / 64, j = e % 64;
      qs[tt][j] = (tt < nt && j < R) ? Q[(long long)(t0 + tt) * ldq + j] : 0.f;
    }
    __syncthreads();
    if (i < M) {
      for (int tt = 0; tt < nt; ++tt) {
        const float pv = ld_f32(P, p_dtype, (long long)(t0 + tt) * ldp + i);
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (j < R) acc[j] = fmaf(pv, qs[tt][j], acc[j]);
      }
    }
  }
  if (i < M) {
    float* out = part + ((long long)c * M + i) * R;
#pragma unroll
    for (int j = 0; j < 64; ++j)
      if (j < R) out[j] = acc[j];
  }
}

// out[i, j] (or out[j, i] when transposed) = scale * sum_{c = 0..nc-1} part[c, i, j].
__global__ void __launch_bounds__(256) skinny_finish_kernel(const float* __restrict__ part, int nc,
                                                            int M, int R, float scale,
                                                            float* __restrict__ out, long long ldo,
                                                            int transposed) {
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  if (e >= (long long)M * R) return;
  const int i = static_cast<int>(e / R), j = static_cast<int>(e % R);
  float sum = 0.f;
  for (int c = 0; c < nc; ++c) sum += part[((long long)c * M + i) * R + j];
  sum *= scale;
  if (transposed)
    out[(long long)j * ldo + i] = sum;
  else
    out[(long long)i * ldo + j] = sum;
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

int skinny_chunks(int T, int M) {
  const int col_blocks = (M + 127) / 128;
  int want = (4 * device_sm_count() + col_blocks - 1) / col_blocks;   // ~4 CTAs per SM
  int max_by_rows = (T + 255) / 256;                                  // at least 256 rows per chunk
  int nc = want < max_by_rows ? want : max_by_rows;
  return nc < 1 ? 1 : nc;
}

int launch_skinny(const void* P, int p_dtype, long long ldp, int T, int M, const float* Q,
                  long long ldq, int R, float scale, float* part, float* out, long long ldo,
                  bool transposed, cudaStream_t stream) {
  if (T <= 0 || M <= 0 || R <= 0) return WP_OK;
  if (R > 64) return WP_ERR_UNSUPPORTED;
  const int nc = skinny_chunks(T, M);
  const int tc = (T + nc - 1) / nc;
  dim3 grid((M + 127) / 128, nc);
  skinny_partial_kernel<<<grid, 128, 0, stream>>>(P, p_dtype, ldp, T, M, Q, ldq, R, tc, part);
  int rc = check_launch();
  if (rc != WP_OK) return rc;
  const long long n = (long long)M * R;
  skinny_finish_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(part, nc, M, R, scale, out, ldo,
                                                                         transposed ? 1 : 0);
  return check_launch();
}

}  // namespace wp
