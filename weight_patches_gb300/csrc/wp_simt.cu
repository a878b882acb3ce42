// wp_simt.cu -- FP32 CUDA-core kernels.
//
// sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM",
// Modifications: an FP32 adapter on BF16 activations keeps its GEMMs in FP32 and is
// added once.  Two kernels serve that rule and the all-FP32 layer:
//
//   rank_proj_kernel   H[t, off_a + j] = s_a * sum_k X[t, k] A_a[j, k]     (FP32 FMA)
//   f32_linear_kernel  Y[t, o] = sum_k X[t, k] W[o, k] + bias[o]
//                                + sum_a sum_j H[t, off_a + j] B_a[o - c0_a, j]
//
// Products and sums are true FP32 (no TF32, no bf16 operands beyond the exact
// widening of stored bf16 inputs).  The rank projection also feeds the tensor-core
// kernel's epilogue when an FP32 adapter rides on a bf16 layer.
#include <cuda_runtime.h>

#include "wp_internal.h"

namespace wp {

namespace {

__device__ __forceinline__ float load_as_f32(const void* p, int dtype, long long i) {
  if (dtype == WP_FP32) return static_cast<const float*>(p)[i];
  return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16);
}

__device__ __forceinline__ void store_from_f32(void* p, int dtype, long long i, float v) {
  if (dtype == WP_FP32) {
    static_cast<float*>(p)[i] = v;
  } else {
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
    static_cast<uint16_t*>(p)[i] = h;
  }
}

constexpr int kTile = 64;
constexpr int kKc = 32;

}  // namespace

// One block: 32 token rows x 64 rank columns of H (all adapters concatenated).
__global__ void __launch_bounds__(256) rank_proj_kernel(const H32Params p) {
  __shared__ float xs[32][kKc + 1];
  __shared__ float as[64][kKc + 1];
  const int t0 = blockIdx.x * 32;
  const int c0 = blockIdx.y * 64;
  const int tid = threadIdx.x;
  const int c_lo = c0 + (tid & 63);   // this thread's rank column
  const int r_lo = tid >> 6;          // rows r_lo, r_lo + 4, ..., (8 rows)
  int ad = -1;
  for (int a = 0; a < p.n_ad; ++a)
    if (c_lo >= p.h_off[a] && c_lo < p.h_off[a] + p.rank[a]) ad = a;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < p.K; k0 += kKc) {
    for (int idx = tid; idx < 32 * kKc; idx += 256) {
      const int r = idx / kKc, k = idx % kKc;
      const int t = t0 + r, kk = k0 + k;
      xs[r][k] = (t < p.T && kk < p.K) ? load_as_f32(p.X, p.x_dtype, (long long)t * p.ldx + kk) : 0.f;
    }
    for (int idx = tid; idx < 64 * kKc; idx += 256) {
      const int c = c0 + idx / kKc, k = idx % kKc;
      const int kk = k0 + k;
      float v = 0.f;
      if (kk < p.K) {
        for (int a = 0; a < p.n_ad; ++a)
          if (c >= p.h_off[a] && c < p.h_off[a] + p.rank[a])
            v = load_as_f32(p.A[a], p.a_dtype[a], (long long)(c - p.h_off[a]) * p.lda[a] + kk);
      }
      as[c - c0][k] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < kKc; ++k) {
      const float av = as[c_lo - c0][k];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(xs[r_lo + 4 * i][k], av, acc[i]);
    }
    __syncthreads();
  }
  if (ad < 0 || c_lo >= p.h_cols) return;
  const float s = p.s[ad];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + r_lo + 4 * i;
    if (t < p.T) p.H[(long long)t * p.h_cols + c_lo] = s * acc[i];
  }
}

// One block: 64 x 64 outputs, 256 threads, 4 x 4 per thread.
__global__ void __launch_bounds__(256) f32_linear_kernel(const F32Params p, const float* H,
                                                          int h_cols) {
  __shared__ float xs[kTile][kKc + 1];
  __shared__ float ws[kTile][kKc + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int row0 = blockIdx.y * kTile, col0 = blockIdx.x * kTile;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  if (p.W) {
    for (int k0 = 0; k0 < p.K; k0 += kKc) {
      for (int idx = threadIdx.x; idx < kTile * kKc; idx += 256) {
        const int r = idx / kKc, k = idx % kKc;
        const int kk = k0 + k;
        const int t = row0 + r, o = col0 + r;
        xs[r][k] = (t < p.T && kk < p.K) ? load_as_f32(p.X, p.x_dtype, (long long)t * p.ldx + kk) : 0.f;
        ws[r][k] = (o < p.N && kk < p.K) ? load_as_f32(p.W, p.w_dtype, (long long)o * p.ldw + kk) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int k = 0; k < kKc; ++k) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = xs[ty * 4 + i][k];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = ws[tx * 4 + j][k];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = row0 + ty * 4 + i;
    if (t >= p.T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int o = col0 + tx * 4 + j;
      if (o >= p.N) continue;
      float v = acc[i][j];
      if (p.bias) v += load_as_f32(p.bias, p.bias_dtype, o);
      int off = 0;
      for (int a = 0; a < p.n_ad; ++a) {
        const F32Adapter& ad = p.ad[a];
        if (o >= p.col_begin[a] && o < p.col_end[a]) {
          const long long brow = (long long)(o - p.col_begin[a]) * ad.ldb;
          const float* hrow = H + (long long)t * h_cols + off;
          for (int jj = 0; jj < ad.rank; ++jj)
            v = fmaf(hrow[jj], load_as_f32(ad.B, ad.b_dtype, brow + jj), v);
        }
        off += ad.rank;
      }
      store_from_f32(p.Y, p.y_dtype, (long long)t * p.ldy + o, v);
    }
  }
}

int launch_h32(const H32Params& p, cudaStream_t stream) {
  if (p.T <= 0 || p.n_ad <= 0) return WP_OK;
  dim3 grid((p.T + 31) / 32, (p.h_cols + 63) / 64);
  rank_proj_kernel<<<grid, 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int launch_f32_linear(const F32Params& p, const float* H, int h_cols, cudaStream_t stream) {
  if (p.T <= 0 || p.N <= 0) return WP_OK;
  dim3 grid((p.N + kTile - 1) / kTile, (p.T + kTile - 1) / kTile);
  f32_linear_kernel<<<grid, 256, 0, stream>>>(p, H, h_cols);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace wp
