// wp_swiglu.cu -- the SwiGLU backward of the LoRA MLP, one elementwise pass.
//
// Unsloth fast_lora walkthrough, section 4 (LoRA_MLP backward): the gradient DW that
// reaches h = f(e) g through the down projection becomes, in one kernel, h itself (for the
// down adapter's gradients), the gradient at g and the gradient at e:
//   f  = e sigmoid(e),  h = f g,
//   dg = DW f,          de = DW g sigmoid(e) (1 + e (1 - sigmoid(e))).
// Inputs are bf16 (DW, and the e | g the forward saved); every product is a separate
// round-to-nearest float32 operation and each output is rounded to bf16 once.  de and dg
// are written side by side (de | dg), the stacked gate/up output gradient that the
// grouped backward of the gate/up linears takes as dY.
//
// HBM-bound: per element 6 bytes read and 4 (6 with h) written; each thread moves 8
// consecutive columns of one row with 16-byte loads and stores, the grid strides over
// the rows x column-octets of the whole matrix with a few CTAs per SM.
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_ptx.cuh"

namespace wp {

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const SwigluBwdParams q) {
  const long long oct = q.F >> 3;                       // 8-column units per row
  const long long units = q.T * oct;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < units; u += stride) {
    const long long row = u / oct;
    const long long col = (u - row * oct) << 3;
    const uint4 dh4 = ld_stream(q.dh + row * q.ld_dh + col);
    const uint4 e4 = ld_stream(q.eg + row * q.ld_eg + col);
    const uint4 g4 = ld_stream(q.eg + row * q.ld_eg + q.F + col);
    const uint32_t dhw[4] = {dh4.x, dh4.y, dh4.z, dh4.w};
    const uint32_t ew[4] = {e4.x, e4.y, e4.z, e4.w};
    const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
    uint32_t de[4], dg[4], hh[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float o_de[2], o_dg[2], o_h[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        // element 2k is the low half of word k, element 2k + 1 the high half
        const float dw = __uint_as_float(j ? (dhw[k] & 0xffff0000u) : (dhw[k] << 16));
        const float e = __uint_as_float(j ? (ew[k] & 0xffff0000u) : (ew[k] << 16));
        const float g = __uint_as_float(j ? (gw[k] & 0xffff0000u) : (gw[k] << 16));
        const float sg = sigmoid_f32(e);
        const float f = silu_f32(e);
        o_h[j] = __fmul_rn(f, g);
        o_dg[j] = __fmul_rn(dw, f);
        // f'(e) = sigmoid(e) (1 + e (1 - sigmoid(e)))
        const float fp = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(e, __fsub_rn(1.0f, sg))));
        o_de[j] = __fmul_rn(__fmul_rn(dw, g), fp);
      }
      de[k] = pack_bf16x2(o_de[0], o_de[1]);
      dg[k] = pack_bf16x2(o_dg[0], o_dg[1]);
      hh[k] = pack_bf16x2(o_h[0], o_h[1]);
    }
    uint16_t* out = q.deg + row * q.ld_deg + col;
    st_global_v4(out, de[0], de[1], de[2], de[3]);
    st_global_v4(out + q.F, dg[0], dg[1], dg[2], dg[3]);
    if (q.h) st_global_v4(q.h + row * q.ld_h + col, hh[0], hh[1], hh[2], hh[3]);
  }
}

}  // namespace

int launch_swiglu_bwd(const SwigluBwdParams& q, cudaStream_t stream) {
  const int sms = device_sm_count();
  const long long units = q.T * (q.F >> 3);
  long long blocks = (units + 255) / 256;
  const long long cap = static_cast<long long>(sms) * 8;   // 8 CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  swiglu_bwd_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(q);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace wp
