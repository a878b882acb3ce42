// wp_patch.cu -- dense LoRA payloads applied in place.
//
// FastVideo API docs, fastvideo.models.loader.lora_patch, DenseLoRAPatch:
//   apply_to (.diff / .diff_b):  param = cast(fp32(param) + fp32(payload) * k)
//   replacement_for (.set_weight): param = cast(fp32(payload) * k)
// The sum is taken in float32 whatever the operand types are, and the caller casts
// back to the parameter's dtype.  Here the product and the sum are two separate
// round-to-nearest float32 operations (explicit __fmul_rn / __fadd_rn, so the
// compiler cannot contract them into an FMA) and the cast back to bf16 is
// round-to-nearest-even, which makes the result bit-exact against the float32
// definition.  The kernel is HBM-bound: 16-byte vector loads and stores, four of each in
// flight per thread, a grid of a few CTAs per SM striding over the tensor.
//
// The same add folds the legacy lora_B.bias vectors of older adapters into a layer's bias
// (bias_fold_kernel): for the forward's epilogue (kept in fp32) and for the merge (rounded
// once to the bias's dtype).
#include <cuda_runtime.h>

#include "wp_internal.h"

namespace wp {

namespace {

__device__ __forceinline__ float widen(const void* p, int dtype, long long i) {
  if (dtype == WP_FP32) return static_cast<const float*>(p)[i];
  return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16);
}

__device__ __forceinline__ uint16_t to_bf16(float v) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
  return h;
}

__device__ __forceinline__ float combine(float p, float d, float k, int kind) {
  const float scaled = __fmul_rn(d, k);
  return kind == WP_PATCH_ADD ? __fadd_rn(p, scaled) : scaled;
}

}  // namespace

__device__ __forceinline__ uint4 patch8(uint4 d, uint4 pv, int kind, float k) {
  const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
  const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
  uint32_t out[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float d_lo = __uint_as_float(dw[w] << 16), d_hi = __uint_as_float(dw[w] & 0xFFFF0000u);
    const float p_lo = __uint_as_float(pw[w] << 16), p_hi = __uint_as_float(pw[w] & 0xFFFF0000u);
    const uint16_t lo = to_bf16(combine(p_lo, d_lo, k, kind));
    const uint16_t hi = to_bf16(combine(p_hi, d_hi, k, kind));
    out[w] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void __launch_bounds__(256) bias_fold_kernel(const BiasFoldParams p) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= p.N) return;
  float v = p.bias ? widen(p.bias, p.bias_dtype, n) : 0.f;
  for (int i = 0; i < p.n; ++i) {
    const int j = n - p.ad[i].col0;
    if (j >= 0 && j < p.ad[i].cols) v = combine(v, widen(p.ad[i].v, p.ad[i].dtype, j), p.ad[i].s, WP_PATCH_ADD);
  }
  if (p.out) {
    p.out[n] = v;
  } else if (p.bias_dtype == WP_FP32) {
    static_cast<float*>(p.bias)[n] = v;
  } else {
    static_cast<uint16_t*>(p.bias)[n] = to_bf16(v);
  }
}

int launch_bias_fold(const BiasFoldParams& p, cudaStream_t stream) {
  if (p.N <= 0) return WP_OK;
  bias_fold_kernel<<<(p.N + 255) / 256, 256, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

// bf16 parameter, bf16 payload, 8 elements (16 bytes) per vector; each thread keeps four
// vectors of each operand in flight (their loads issued before any arithmetic).
__global__ void __launch_bounds__(256) dense_patch_bf16_vec(uint16_t* __restrict__ param,
                                                            const uint16_t* __restrict__ payload,
                                                            long long n8, int kind, float k) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const uint4* src = reinterpret_cast<const uint4*>(payload);
  uint4* dst = reinterpret_cast<uint4*>(param);
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 d[4], pv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      d[u] = src[i + u * stride];
      pv[u] = kind == WP_PATCH_ADD ? dst[i + u * stride] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) dst[i + u * stride] = patch8(d[u], pv[u], kind, k);
  }
  for (; i < n8; i += stride) {
    const uint4 pv = kind == WP_PATCH_ADD ? dst[i] : make_uint4(0, 0, 0, 0);
    dst[i] = patch8(src[i], pv, kind, k);
  }
}

// Any dtype pair, one element per thread per step (tails and unaligned tensors).
__global__ void __launch_bounds__(256) dense_patch_scalar(void* __restrict__ param, int pdt,
                                                          const void* __restrict__ payload, int ydt,
                                                          long long begin, long long n, int kind,
                                                          float k) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = begin + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float d = widen(payload, ydt, i);
    const float p = kind == WP_PATCH_ADD ? widen(param, pdt, i) : 0.f;
    const float r = combine(p, d, k, kind);
    if (pdt == WP_FP32)
      static_cast<float*>(param)[i] = r;
    else
      static_cast<uint16_t*>(param)[i] = to_bf16(r);
  }
}

int launch_dense_patch(void* param, int pdt, const void* payload, int ydt, long long n, int kind,
                       float k, cudaStream_t stream) {
  if (n <= 0) return WP_OK;
  const int sms = device_sm_count();
  long long done = 0;
  const bool vec = pdt == WP_BF16 && ydt == WP_BF16 &&
                   (reinterpret_cast<uintptr_t>(param) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(payload) & 15) == 0;
  if (vec && n >= 8) {
    const long long n8 = n / 8;
    long long blocks = (n8 + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    dense_patch_bf16_vec<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<uint16_t*>(param), static_cast<const uint16_t*>(payload), n8, kind, k);
    done = n8 * 8;
  }
  if (done < n) {
    long long blocks = (n - done + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    dense_patch_scalar<<<(unsigned)blocks, 256, 0, stream>>>(param, pdt, payload, ydt, done, n,
                                                              kind, k);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace wp
