// wp_merge.cu -- the elementwise halves of a LoRA merge into a 4-bit NormalFloat weight.
//
// piper-offload docs, "LoRA merge" and "Quantized weight support": a plain floating-point
// weight takes the update in place (addmm_); a bitsandbytes NF4 weight is dequantised,
// takes every LoRA of the target as one staged update, and is re-encoded once, with
// deterministic round-to-nearest on request.  The library does that as
//   U = fl32(W_eff)                          nf4_to_f32_kernel
//   U = s_p * (B_p A_p) + U  per adapter     the fused kernel's merge epilogue
//   (codes, absmax) = requantise(U)           nf4_requant_kernel
// with W_eff = bf16(fl32(level[q]) * absmax) as everywhere else, and the requantisation of a
// 64-element block: absmax' = max |u|, x = fl32(u / absmax'), code = the number of level
// midpoints fl32((level[k] + level[k+1]) / 2) that x exceeds (the nearest level; a value on a
// midpoint takes the lower code); an all-zero block keeps scale 0 and the code of level 0.
// Both kernels are HBM-bound: 8 elements per thread, 16-byte fp32 loads/stores.
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_nf4.cuh"
#include "wp_ptx.cuh"

namespace wp {

namespace {

__global__ void __launch_bounds__(256) nf4_to_f32_kernel(const uint8_t* codes, const float* absmax, long long n8,
                                                         NF4Table tab, float* U) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < n8; u += stride) {
    const uint32_t c4 = *reinterpret_cast<const uint32_t*>(codes + u * 4);   // 8 codes
    const float am = absmax[u >> 3];                                        // 8 octets per block
    float v[8];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = (c4 >> (8 * b)) & 0xffu;
      // element 2b in the high nibble, 2b + 1 in the low nibble
      const float w0 = tab.level[byte >> 4] * am, w1 = tab.level[byte & 0xfu] * am;
      uint16_t h0, h1;
      asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h0) : "f"(w0));
      asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h1) : "f"(w1));
      v[2 * b] = __uint_as_float(static_cast<uint32_t>(h0) << 16);
      v[2 * b + 1] = __uint_as_float(static_cast<uint32_t>(h1) << 16);
    }
    float4* dst = reinterpret_cast<float4*>(U + u * 8);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// 8 threads per 64-element block (consecutive lanes), the block's absmax by shuffles.
__global__ void __launch_bounds__(256) nf4_requant_kernel(const float* U, long long n8, NF4Table tab,
                                                          uint8_t* codes, float* absmax) {
  float mid[15];
#pragma unroll
  for (int k = 0; k < 15; ++k) mid[k] = __fmul_rn(__fadd_rn(tab.level[k], tab.level[k + 1]), 0.5f);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // every lane of a warp runs the same number of iterations (n8 is a multiple of 8 and the
  // stride a multiple of 32), so the shuffles below always see all 8 lanes of a block
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u - (threadIdx.x & 31) < n8;
       u += stride) {
    const bool live = u < n8;
    float v[8];
    if (live) {
      const float4 a = reinterpret_cast<const float4*>(U + u * 8)[0];
      const float4 b = reinterpret_cast<const float4*>(U + u * 8)[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    uint32_t c4 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t q = 7;                                   // level 0 for an all-zero block
      if (m > 0.f) {
        q = nf4_code_of(__fdiv_rn(v[i], m), mid);
      }
      // element 2b in the high nibble of byte b
      c4 |= q << (8 * (i >> 1) + ((i & 1) ? 0 : 4));
    }
    if (live) {
      *reinterpret_cast<uint32_t*>(codes + u * 4) = c4;
      if ((u & 7) == 0) absmax[u >> 3] = m;
    }
  }
}

}  // namespace

int launch_nf4_to_f32(const void* codes, const float* absmax, long long numel, const NF4Table& tab, float* U,
                      cudaStream_t stream) {
  const long long n8 = numel / 8;
  if (n8 <= 0) return WP_OK;
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  nf4_to_f32_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const uint8_t*>(codes), absmax,
                                                                       n8, tab, U);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

// The stochastic form: a thread per 64-element block (rows of U are whole blocks), the block's
// level cells in shared memory.
__global__ void __launch_bounds__(128) nf4_requant_stochastic_kernel(const float* U, long long nblk,
                                                                     const __grid_constant__ NF4LevelCells lc,
                                                                     uint8_t* codes, float* absmax, uint32_t k0,
                                                                     uint32_t k1) {
  __shared__ uint32_t s_l[4 * kCodeCells];
  for (int c = threadIdx.x; c < kCodeCells; c += blockDim.x) {
    s_l[c] = __float_as_uint(lc.next_l[c]);
    s_l[kCodeCells + c] = static_cast<uint32_t>(lc.base[c]);
    s_l[2 * kCodeCells + c] = __float_as_uint(lc.prev_l[c]);
    s_l[3 * kCodeCells + c] = __float_as_uint(lc.after_l[c]);
  }
  __syncthreads();
  const uint32_t cells = smem_u32(s_l);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long bk = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; bk < nblk; bk += stride) {
    float u[64];
    const float4* src = reinterpret_cast<const float4*>(U + bk * 64);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 v = src[i];
      u[4 * i] = v.x;
      u[4 * i + 1] = v.y;
      u[4 * i + 2] = v.z;
      u[4 * i + 3] = v.w;
    }
    uint32_t cw[8];
    const float m = nf4_requant_block_stochastic(u, cells, static_cast<unsigned long long>(bk) * 64, k0, k1, cw);
    uint4* dst = reinterpret_cast<uint4*>(codes + bk * 32);
    dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    absmax[bk] = m;
  }
}

int launch_nf4_requant_stochastic(const float* U, long long numel, const NF4Table& tab, void* codes,
                                  float* absmax, uint64_t seed, cudaStream_t stream) {
  const long long nblk = numel / 64;
  if (nblk <= 0) return WP_OK;
  NF4LevelCells lc;
  if (!nf4_level_cells(tab, &lc)) return WP_ERR_UNSUPPORTED;
  long long blocks = (nblk + 127) / 128;
  const long long cap = static_cast<long long>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  nf4_requant_stochastic_kernel<<<static_cast<unsigned>(blocks), 128, 0, stream>>>(
      U, nblk, lc, static_cast<uint8_t*>(codes), absmax, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int launch_nf4_requant(const float* U, long long numel, const NF4Table& tab, void* codes, float* absmax,
                       cudaStream_t stream) {
  const long long n8 = numel / 8;
  if (n8 <= 0) return WP_OK;
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  nf4_requant_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(U, n8, tab, static_cast<uint8_t*>(codes),
                                                                        absmax);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

// The code search by cells: cell c holds [-1 + c/16, -1 + (c+1)/16), 32 cells over [-1, 1)
// and a 33rd from 1.  The midpoints (fp32, as the kernels form them) below a
// cell's lower end count into its base code; the first midpoint at or above it is the one a
// value in the cell is compared against.  False if a cell holds two midpoints (one compare
// cannot resolve it); the NF4 midpoints are at least 0.08 apart, so no cell holds two.
bool nf4_code_cells(const NF4Table& tab, NF4Cells* cells) {
  float mid[15];
  for (int k = 0; k < 15; ++k) mid[k] = (tab.level[k] + tab.level[k + 1]) * 0.5f;
  for (int k = 0; k + 1 < 15; ++k)
    if (!(mid[k] < mid[k + 1])) return false;
  for (int c = 0; c < kCodeCells; ++c) {
    const float lo = -1.0f + static_cast<float>(c) / 16.0f, hi = lo + 1.0f / 16.0f;
    int base = 0;
    while (base < 15 && mid[base] < lo) ++base;
    if (base + 1 < 15 && mid[base + 1] < hi) return false;
    cells->base[c] = base;
    cells->next_mid[c] = base < 15 ? mid[base] : 2.0f;
  }
  return true;
}

// The stochastic re-encoding's cells (the same 33 cells): the first level at or above a cell's
// start, its index, the level before it and the level after it.  False if a cell holds two
// levels.
bool nf4_level_cells(const NF4Table& tab, NF4LevelCells* cells) {
  for (int k = 0; k + 1 < 16; ++k)
    if (!(tab.level[k] < tab.level[k + 1])) return false;
  for (int c = 0; c < kCodeCells; ++c) {
    const float lo = -1.0f + static_cast<float>(c) / 16.0f, hi = lo + 1.0f / 16.0f;
    int base = 0;
    while (base < 16 && tab.level[base] < lo) ++base;
    if (base + 1 < 16 && tab.level[base + 1] < hi) return false;
    cells->base[c] = base;
    cells->next_l[c] = base < 16 ? tab.level[base] : 2.0f;
    cells->prev_l[c] = base > 0 ? tab.level[base - 1] : -2.0f;
    cells->after_l[c] = base + 1 < 16 ? tab.level[base + 1] : 2.0f;
  }
  return true;
}

}  // namespace wp
