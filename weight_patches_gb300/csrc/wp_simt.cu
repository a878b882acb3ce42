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

#include <algorithm>
#include <cstdint>

#include "wp_internal.h"
#include "wp_ptx.cuh"

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

}  // namespace

// s * X A^T for skinny A (a few to a few hundred rank columns).  One block: 32 token
// rows x CW rank columns (adapters concatenated), 4 warps.  A lane owns two rows
// (r and r + 4 of its warp's 8) and one 8-wide k segment of each 64-wide K chunk; the
// chunk of A sits in shared memory as [segment][k][column], each segment's block padded
// by 16 bytes so that the 8 segments a warp reads at once fall in distinct banks (lanes
// of one segment read the same address: a broadcast).  At the end the 8 segment partial
// sums of a row are combined by a fixed butterfly (reduce-scatter over shuffles), so the
// result does not depend on timing.
template <int CW, bool kXf32>
__global__ void __launch_bounds__(128) rank_proj_kernel(const H32Params p) {
  constexpr int kKC = 64;
  constexpr int kSeg = 8 * CW + 4;            // floats per segment block, padded
  constexpr int kSlots = CW / 8;              // A quads (4 consecutive k) per thread per chunk
  __shared__ __align__(16) float As[8 * kSeg];
  __shared__ float col_s[CW];
  __shared__ int col_ok[CW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c0 = blockIdx.x * CW;
  const int s8 = lane & 7;

  if (tid < CW) {
    const int col = c0 + tid;
    int ok = 0;
    float sc = 0.f;
    for (int a = 0; a < p.n_ad; ++a)
      if (col < p.h_cols && col >= p.h_off[a] && col < p.h_off[a] + p.rank[a]) { ok = 1; sc = p.s[a]; }
    col_s[tid] = sc;
    col_ok[tid] = ok;
  }

  // this thread's A quads: column c0 + (e >> 4), k offset 4 * (e & 15) within a chunk
  const char* asrc[kSlots];
  long long ald[kSlots];
  int adt[kSlots];
  bool avec[kSlots];
#pragma unroll
  for (int i = 0; i < kSlots; ++i) {
    const int e = tid + 128 * i;
    const int col = c0 + (e >> 4);
    asrc[i] = nullptr; ald[i] = 0; adt[i] = WP_BF16; avec[i] = false;
    for (int a = 0; a < p.n_ad; ++a) {
      if (col < p.h_cols && col >= p.h_off[a] && col < p.h_off[a] + p.rank[a]) {
        const int es = p.a_dtype[a] == WP_FP32 ? 4 : 2;
        asrc[i] = static_cast<const char*>(p.A[a]) + static_cast<long long>(col - p.h_off[a]) * p.lda[a] * es;
        ald[i] = p.lda[a];
        adt[i] = p.a_dtype[a];
        avec[i] = p.a_vec[a] != 0;
      }
    }
  }

  float areg[kSlots][4];
  auto load_a = [&](int k0) {
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const int k = k0 + 4 * ((tid + 128 * i) & 15);
#pragma unroll
      for (int j = 0; j < 4; ++j) areg[i][j] = 0.f;
      if (!asrc[i]) continue;
      if (adt[i] == WP_FP32) {
        const float* a = reinterpret_cast<const float*>(asrc[i]);
        if (avec[i] && k + 3 < p.K) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(a + k));
          areg[i][0] = v.x; areg[i][1] = v.y; areg[i][2] = v.z; areg[i][3] = v.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) if (k + j < p.K) areg[i][j] = a[k + j];
        }
      } else {
        const uint16_t* a = reinterpret_cast<const uint16_t*>(asrc[i]);
        if (avec[i] && k + 3 < p.K) {
          const uint2 v = __ldg(reinterpret_cast<const uint2*>(a + k));
          areg[i][0] = __uint_as_float(v.x << 16); areg[i][1] = __uint_as_float(v.x & 0xffff0000u);
          areg[i][2] = __uint_as_float(v.y << 16); areg[i][3] = __uint_as_float(v.y & 0xffff0000u);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (k + j < p.K) areg[i][j] = __uint_as_float(static_cast<uint32_t>(a[k + j]) << 16);
        }
      }
    }
  };
  auto store_a = [&]() {
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const int e = tid + 128 * i;
      const int c = e >> 4, k4 = e & 15;
#pragma unroll
      for (int j = 0; j < 4; ++j) As[(k4 >> 1) * kSeg + ((k4 & 1) * 4 + j) * CW + c] = areg[i][j];
    }
  };

  float xr[2][8];
  auto load_x = [&](int rb, int k0) {
    const int k = k0 + 8 * s8;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = rb * 32 + warp * 8 + (lane >> 3) + 4 * h;
#pragma unroll
      for (int j = 0; j < 8; ++j) xr[h][j] = 0.f;
      if (t >= p.T) continue;
      if (kXf32) {
        const float* x = static_cast<const float*>(p.X) + static_cast<long long>(t) * p.ldx;
        if (p.x_vec && k + 7 < p.K) {
          const float4 u = __ldg(reinterpret_cast<const float4*>(x + k));
          const float4 v = __ldg(reinterpret_cast<const float4*>(x + k + 4));
          xr[h][0] = u.x; xr[h][1] = u.y; xr[h][2] = u.z; xr[h][3] = u.w;
          xr[h][4] = v.x; xr[h][5] = v.y; xr[h][6] = v.z; xr[h][7] = v.w;
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) if (k + j < p.K) xr[h][j] = x[k + j];
        }
      } else {
        const uint16_t* x = static_cast<const uint16_t*>(p.X) + static_cast<long long>(t) * p.ldx;
        if (p.x_vec && k + 7 < p.K) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(x + k));
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            xr[h][2 * j] = __uint_as_float(w[j] << 16);
            xr[h][2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (k + j < p.K) xr[h][j] = __uint_as_float(static_cast<uint32_t>(x[k + j]) << 16);
        }
      }
    }
  };

  const int row_blocks = (p.T + 31) / 32;
  for (int rb = blockIdx.y; rb < row_blocks; rb += gridDim.y) {
    float acc[2][CW];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int c = 0; c < CW; ++c) acc[h][c] = 0.f;
    load_a(0);
    load_x(rb, 0);
    for (int k0 = 0; k0 < p.K; k0 += kKC) {
      __syncthreads();                      // the previous chunk is no longer read
      store_a();
      __syncthreads();
      float xc[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 8; ++j) xc[h][j] = xr[h][j];
      if (k0 + kKC < p.K) {                 // next chunk in flight during the FMAs
        load_a(k0 + kKC);
        load_x(rb, k0 + kKC);
      }
      const float* as = As + s8 * kSeg;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int c4 = 0; c4 < CW / 4; ++c4) {
          const float4 a = *reinterpret_cast<const float4*>(as + kk * CW + 4 * c4);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            acc[h][4 * c4 + 0] = fmaf(xc[h][kk], a.x, acc[h][4 * c4 + 0]);
            acc[h][4 * c4 + 1] = fmaf(xc[h][kk], a.y, acc[h][4 * c4 + 1]);
            acc[h][4 * c4 + 2] = fmaf(xc[h][kk], a.z, acc[h][4 * c4 + 2]);
            acc[h][4 * c4 + 3] = fmaf(xc[h][kk], a.w, acc[h][4 * c4 + 3]);
          }
        }
      }
    }
    // combine the 8 segments: after the butterfly each lane of a row's 8 holds CW/8 sums
#pragma unroll
    for (int step = 0; step < 3; ++step) {
      const int m = 4 >> step;
      const int half = (CW / 2) >> step;
      const bool hi = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float keep = hi ? acc[h][i + half] : acc[h][i];
          const float send = hi ? acc[h][i] : acc[h][i + half];
          acc[h][i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
    }
    const int cofs = ((lane >> 2) & 1) * (CW / 2) + ((lane >> 1) & 1) * (CW / 4) + (lane & 1) * (CW / 8);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = rb * 32 + warp * 8 + (lane >> 3) + 4 * h;
      if (t >= p.T) continue;
#pragma unroll
      for (int i = 0; i < CW / 8; ++i) {
        const int c = cofs + i;
        if (col_ok[c]) p.H[static_cast<long long>(t) * p.h_cols + c0 + c] = col_s[c] * acc[h][i];
      }
    }
  }
}

// One block: 128 x 128 outputs, 256 threads, 8 x 8 per thread (rows ty*4 + {0..3} and
// 64 + ty*4 + {0..3}, columns tx*4 + {0..3} and 64 + tx*4 + {0..3}).  K goes 8 at a time
// through two shared-memory buffers holding the X and W tiles K-major ([k][row]), so a thread
// reads its 8 X and 8 W values of one k with four 16-byte loads (the X ones a broadcast
// across the warp) and issues 64 fmas for them; the next K slice's global loads are in flight
// in registers meanwhile (4 consecutive k of one row per thread, one vector load when the rows
// allow it).  Each output's sum over k runs in k order from 0 in fp32 fmas; then the bias and
// the adapters' H B^T terms, rank by rank in adapter order, as fmas onto it.
constexpr int kSM = 128, kSN = 128, kSK = 8;

// 4 consecutive elements of a row as fp32 (vec: one 8- or 16-byte load; else one by one,
// zero past k_end)
template <bool kF32>
__device__ __forceinline__ void load4(const void* base, long long off, int k, int k_end, bool vec, float (&v)[4]) {
  if (kF32) {
    const float* q = static_cast<const float*>(base) + off;
    if (vec) {
      const float4 f = *reinterpret_cast<const float4*>(q);
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = k + i < k_end ? q[i] : 0.f;
    }
  } else {
    const uint16_t* q = static_cast<const uint16_t*>(base) + off;
    if (vec) {
      const uint2 h = *reinterpret_cast<const uint2*>(q);
      v[0] = __uint_as_float(h.x << 16); v[1] = __uint_as_float(h.x & 0xffff0000u);
      v[2] = __uint_as_float(h.y << 16); v[3] = __uint_as_float(h.y & 0xffff0000u);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = k + i < k_end ? __uint_as_float(static_cast<uint32_t>(q[i]) << 16) : 0.f;
    }
  }
}

template <bool kXF32, bool kWF32>
__global__ void __launch_bounds__(256, 2) f32_linear_kernel(const F32Params p, const float* H, int h_cols,
                                                             int vec) {
  __shared__ __align__(16) float xs[2][kSK][kSM];
  __shared__ __align__(16) float ws[2][kSK][kSN];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int row0 = blockIdx.y * kSM, col0 = blockIdx.x * kSN;
  const int lr = tid >> 1, lk = (tid & 1) * 4;    // the slice loads: row lr, k offsets lk .. lk + 3
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  if (p.W) {
    float xr[4], wr[4];
    const int t = row0 + lr, o = col0 + lr;
    auto gload = [&](int k0) {
      const int k = k0 + lk;
      if (t < p.T && k < p.K) {
        load4<kXF32>(p.X, static_cast<long long>(t) * p.ldx + k, k, p.K, vec != 0, xr);
      } else {
        xr[0] = xr[1] = xr[2] = xr[3] = 0.f;
      }
      if (o < p.N && k < p.K) {
        load4<kWF32>(p.W, static_cast<long long>(o) * p.ldw + k, k, p.K, vec != 0, wr);
      } else {
        wr[0] = wr[1] = wr[2] = wr[3] = 0.f;
      }
    };
    auto sstore = [&](int buf) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xs[buf][lk + q][lr] = xr[q];
        ws[buf][lk + q][lr] = wr[q];
      }
    };
    gload(0);
    sstore(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < p.K; k0 += kSK) {
      const bool more = k0 + kSK < p.K;
      if (more) gload(k0 + kSK);
#pragma unroll
      for (int k = 0; k < kSK; ++k) {
        const float4 a0 = *reinterpret_cast<const float4*>(&xs[buf][k][ty * 4]);
        const float4 a1 = *reinterpret_cast<const float4*>(&xs[buf][k][64 + ty * 4]);
        const float4 b0 = *reinterpret_cast<const float4*>(&ws[buf][k][tx * 4]);
        const float4 b1 = *reinterpret_cast<const float4*>(&ws[buf][k][64 + tx * 4]);
        const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      if (more) sstore(buf ^ 1);
      __syncthreads();
      buf ^= 1;
    }
  }

  // epilogue: bias, then each adapter's rank terms in order, for all 64 outputs at once
  int trow[8], ocol[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) trow[i] = row0 + (i < 4 ? ty * 4 + i : 60 + ty * 4 + i);
#pragma unroll
  for (int j = 0; j < 8; ++j) ocol[j] = col0 + (j < 4 ? tx * 4 + j : 60 + tx * 4 + j);
  if (p.bias) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float bj = ocol[j] < p.N ? load_as_f32(p.bias, p.bias_dtype, ocol[j]) : 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i][j] += bj;
    }
  }
  int off = 0;
  for (int a = 0; a < p.n_ad; ++a) {
    const F32Adapter& ad = p.ad[a];
    bool in[8], any = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      in[j] = ocol[j] < p.N && ocol[j] >= p.col_begin[a] && ocol[j] < p.col_end[a];
      any = any || in[j];
    }
    if (any) {
      for (int jj = 0; jj < ad.rank; ++jj) {
        float h[8], bb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = trow[i] < p.T ? H[static_cast<long long>(trow[i]) * h_cols + off + jj] : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          bb[j] = in[j] ? load_as_f32(ad.B, ad.b_dtype, static_cast<long long>(ocol[j] - p.col_begin[a]) * ad.ldb + jj)
                        : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (in[j]) acc[i][j] = fmaf(h[i], bb[j], acc[i][j]);
      }
    }
    off += ad.rank;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (trow[i] >= p.T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (ocol[j] < p.N) store_from_f32(p.Y, p.y_dtype, static_cast<long long>(trow[i]) * p.ldy + ocol[j], acc[i][j]);
  }
}

int launch_h32(const H32Params& p0, cudaStream_t stream) {
  if (p0.T <= 0 || p0.n_ad <= 0) return WP_OK;
  // vector loads where every row start is aligned: 8 elements of X, 4 of A
  H32Params p = p0;
  const auto aligned = [](const void* ptr, long long ld, int bytes, int align) {
    return reinterpret_cast<uintptr_t>(ptr) % align == 0 && (ld * bytes) % align == 0;
  };
  const int xb = p.x_dtype == WP_FP32 ? 4 : 2;
  p.x_vec = aligned(p.X, p.ldx, xb, 16);
  for (int a = 0; a < p.n_ad; ++a) {
    const int ab = p.a_dtype[a] == WP_FP32 ? 4 : 2;
    p.a_vec[a] = aligned(p.A[a], p.lda[a], ab, 4 * ab);
  }
  const int cw = p.h_cols <= 16 ? 16 : 32;
  dim3 grid((p.h_cols + cw - 1) / cw, std::min((p.T + 31) / 32, 65535));
  if (p.x_dtype == WP_FP32) {
    if (cw == 16) rank_proj_kernel<16, true><<<grid, 128, 0, stream>>>(p);
    else rank_proj_kernel<32, true><<<grid, 128, 0, stream>>>(p);
  } else {
    if (cw == 16) rank_proj_kernel<16, false><<<grid, 128, 0, stream>>>(p);
    else rank_proj_kernel<32, false><<<grid, 128, 0, stream>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

namespace {

__device__ __forceinline__ void split3_bf16(float x, uint16_t* h) {
  uint16_t a;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(a) : "f"(x));
  const float r1 = x - __uint_as_float(static_cast<uint32_t>(a) << 16);     // exact
  uint16_t b;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b) : "f"(r1));
  const float r2 = r1 - __uint_as_float(static_cast<uint32_t>(b) << 16);    // exact
  uint16_t c;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(c) : "f"(r2));
  h[0] = a; h[1] = b; h[2] = c;
}

}  // namespace

// One block per row: rows [0, 2 half) are the packed A rows, the rest the B-piece rows of
// the FP32 adapters (adapter by adapter); threads take 8 consecutive elements each.
// Block 0 also clears the row-block flags of the forward kernel that follows.
__global__ void __launch_bounds__(256) rank_pack_kernel(const PackParams p) {
  // the fused kernel that follows may start its set-up now; it waits for this grid to
  // finish before it touches the packed rows, the B pieces or the flags
  grid_launch_dependents();
  const int htot = 2 * p.half;
  const int arows = htot * p.npass;
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < p.n_flags; i += blockDim.x) p.flags[i] = 0u;
  for (int vr = blockIdx.y; vr < p.rows_total; vr += gridDim.y) {
    if (vr < arows) {
      // packed A row pr of pass pr / htot: find the adapter and rank column it holds (rows
      // past the pass's adapters are zero)
      const int pr = vr;
      const bool first_half = pr % htot < p.half;
      int da = -1, u = 0;
      for (int a = 0; a < p.n_ad; ++a) {
        const int base = first_half ? p.ad[a].hoff : p.ad[a].hoff2;
        if (pr >= base && pr < base + p.ad[a].pw / 2) {
          da = a;
          u = pr - base + (first_half ? 0 : p.ad[a].pw / 2);
        }
      }
      const bool split3 = da >= 0 && p.ad[da].split3;
      const int i = split3 ? u / p.ad[da].rp : 0;
      const int j = split3 ? u % p.ad[da].rp : u;
      const bool live = da >= 0 && j < p.ad[da].r;
      const void* srcA = live ? p.ad[da].A : nullptr;
      const long long lda = live ? p.ad[da].lda : 0;
      uint16_t* dst = p.Ap + static_cast<long long>(pr) * p.ldk;
      for (int k0 = (blockIdx.x * blockDim.x + threadIdx.x) * 8; k0 < p.ldk; k0 += gridDim.x * blockDim.x * 8) {
        uint16_t h8[8];
        if (!live) {
#pragma unroll
          for (int e = 0; e < 8; ++e) h8[e] = 0;
        } else if (split3) {
          const float* src = static_cast<const float*>(srcA) + j * lda;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            uint16_t h[3] = {0, 0, 0};
            if (k0 + e < p.K) split3_bf16(src[k0 + e], h);
            h8[e] = h[i];
          }
        } else {
          const uint16_t* src = static_cast<const uint16_t*>(srcA) + j * lda;
#pragma unroll
          for (int e = 0; e < 8; ++e) h8[e] = k0 + e < p.K ? src[k0 + e] : uint16_t(0);
        }
        uint4 w;
        w.x = h8[0] | (uint32_t(h8[1]) << 16); w.y = h8[2] | (uint32_t(h8[3]) << 16);
        w.z = h8[4] | (uint32_t(h8[5]) << 16); w.w = h8[6] | (uint32_t(h8[7]) << 16);
        *reinterpret_cast<uint4*>(dst + k0) = w;     // ldk % 8 == 0, Ap 16-byte aligned
      }
    } else {
      // B-piece row: (adapter, output row o) in order
      int f = vr - arows;
      for (int a = 0; a < p.n_ad; ++a) {
        const PackAdapter& d = p.ad[a];
        if (!d.split3) continue;
        if (f >= d.out) { f -= d.out; continue; }
        const int rp = d.rp;
        uint16_t* row = d.Bs + static_cast<long long>(f) * 6 * rp;
        for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < rp; j += gridDim.x * blockDim.x) {
          uint16_t h[3] = {0, 0, 0};
          if (j < d.r) split3_bf16(d.B[f * d.ldb + j], h);
          row[j] = h[0]; row[rp + j] = h[1]; row[2 * rp + j] = h[0];
          row[3 * rp + j] = h[2]; row[4 * rp + j] = h[1]; row[5 * rp + j] = h[0];
        }
        break;
      }
    }
  }
}

int launch_rank_pack(const PackParams& p0, cudaStream_t stream) {
  PackParams p = p0;
  p.rows_total = 2 * p.half * p.npass;
  for (int a = 0; a < p.n_ad; ++a)
    if (p.ad[a].split3) p.rows_total += p.ad[a].out;
  if (p.rows_total == 0 && p.n_flags == 0) return WP_OK;
  dim3 grid(std::max(1, std::min((p.ldk + 2047) / 2048, 4)), std::max(1, std::min(p.rows_total, 65535)));
  rank_pack_kernel<<<grid, 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int launch_f32_linear(const F32Params& p, const float* H, int h_cols, cudaStream_t stream) {
  if (p.T <= 0 || p.N <= 0) return WP_OK;
  dim3 grid((p.N + kSN - 1) / kSN, std::min((p.T + kSM - 1) / kSM, 65535));
  // vector loads of 4 consecutive K elements: every row start and K itself 4-element aligned
  const auto aligned = [](const void* ptr, long long ld, int bytes) {
    return reinterpret_cast<uintptr_t>(ptr) % (4 * bytes) == 0 && ld % 4 == 0;
  };
  const int xb = p.x_dtype == WP_FP32 ? 4 : 2, wb = p.w_dtype == WP_FP32 ? 4 : 2;
  const int vec = p.K % 4 == 0 && aligned(p.X, p.ldx, xb) && (!p.W || aligned(p.W, p.ldw, wb)) ? 1 : 0;
  const bool xf = p.x_dtype == WP_FP32, wf = !p.W || p.w_dtype == WP_FP32;
  if (xf && wf) f32_linear_kernel<true, true><<<grid, 256, 0, stream>>>(p, H, h_cols, vec);
  else if (xf) f32_linear_kernel<true, false><<<grid, 256, 0, stream>>>(p, H, h_cols, vec);
  else if (wf) f32_linear_kernel<false, true><<<grid, 256, 0, stream>>>(p, H, h_cols, vec);
  else f32_linear_kernel<false, false><<<grid, 256, 0, stream>>>(p, H, h_cols, vec);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace wp
