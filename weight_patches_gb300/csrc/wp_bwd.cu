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
//   skinny_partial_kernel    part[c, i, j] = sum_{t in chunk c} P[t, i] Q[t, j]   (fp32, FFMA)
//   skinny_finish_kernel     out = scale * sum_c part[c]  (fixed order: deterministic)
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

// part[c, i, j] = sum over t in [c * tc, (c + 1) * tc) of P[t, i] * Q[t, j], j < R; P bf16.
// RP = R rounded up to 16.  A block owns 512 columns of P and one chunk of token rows; the
// rows stream through a 3-stage shared-memory ring by cp.async (32 rows x 1 KiB of P and
// the same 32 rows of Q per stage, zero-filled past the chunk, past M and past R), so that
// about 64 KiB per block are in flight.  Thread t owns columns 2t, 2t+1 of the block and
// all RP sums of each (FFMA); Q is read as 16-byte broadcasts.
namespace {
constexpr int kSkCols = 512;      // columns of P per block (1 KiB of bf16 per row)
constexpr int kSkRows = 32;       // token rows per stage
constexpr int kSkStages = 3;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
}  // namespace

template <int RP>
__global__ void __launch_bounds__(256) skinny_partial_kernel(const uint16_t* __restrict__ P, long long ldp,
                                                             int T, int M, const float* __restrict__ Q,
                                                             long long ldq, int R, int tc,
                                                             float* __restrict__ part) {
  extern __shared__ __align__(16) uint8_t sk_smem[];
  uint8_t* ptile = sk_smem;                                           // [stage][row][1 KiB]
  float* qtile = reinterpret_cast<float*>(sk_smem + kSkStages * kSkRows * kSkCols * 2);   // [stage][row][RP]
  const int tid = threadIdx.x;
  const int c0 = blockIdx.x * kSkCols;
  const int c = blockIdx.y;
  const int t_begin = c * tc, t_end = min(T, t_begin + tc);
  const int n_steps = (t_end - t_begin + kSkRows - 1) / kSkRows;

  // stage s <- rows [t_begin + step * 32, +32): each thread copies 4 x 16 B of P and
  // (32 * RP / 256) floats of Q
  auto issue = [&](int step, int st) {
    const int t0 = t_begin + step * kSkRows;
    const uint32_t pbase = smem_u32(ptile + st * kSkRows * kSkCols * 2);
#pragma unroll
    for (int q = 0; q < (kSkRows * kSkCols * 2 / 16) / 256; ++q) {
      const int e = tid + 256 * q;
      const int row = e / (kSkCols / 8), u = e % (kSkCols / 8);     // 64 units of 16 B per row
      const int t = t0 + row, col = c0 + 8 * u;
      const bool ok = t < t_end && col < M;                           // M % 8 == 0
      const uint16_t* src = ok ? P + static_cast<long long>(t) * ldp + col : P;
      cp_async16(pbase + row * kSkCols * 2 + u * 16, src, ok ? 16u : 0u);
    }
    const uint32_t qbase = smem_u32(qtile + st * kSkRows * RP);
#pragma unroll
    for (int q = 0; q < (kSkRows * RP) / 256 + ((kSkRows * RP) % 256 ? 1 : 0); ++q) {
      const int e = tid + 256 * q;
      if (e >= kSkRows * RP) break;
      const int row = e / RP, j = e % RP;
      const int t = t0 + row;
      const bool ok = t < t_end && j < R;
      const float* src = ok ? Q + static_cast<long long>(t) * ldq + j : Q;
      cp_async4(qbase + e * 4, src, ok ? 4u : 0u);
    }
  };

  float acc[2][RP];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int j = 0; j < RP; ++j) acc[h][j] = 0.f;

#pragma unroll
  for (int s = 0; s < kSkStages - 1; ++s) {
    if (s < n_steps) issue(s, s);
    cp_async_commit();
  }
  for (int step = 0; step < n_steps; ++step) {
    const int nxt = step + kSkStages - 1;
    if (nxt < n_steps) issue(nxt, nxt % kSkStages);
    cp_async_commit();
    cp_async_wait<kSkStages - 1>();                 // this thread's copies of `step` landed
    __syncthreads();                                // and everyone else's
    const int st = step % kSkStages;
    const uint8_t* pt = ptile + st * kSkRows * kSkCols * 2;
    const float* qt = qtile + st * kSkRows * RP;
#pragma unroll 4
    for (int row = 0; row < kSkRows; ++row) {       // rows past the chunk are zero
      const uint32_t w = *reinterpret_cast<const uint32_t*>(pt + row * kSkCols * 2 + tid * 4);
      const float p0 = __uint_as_float(w << 16), p1 = __uint_as_float(w & 0xffff0000u);
#pragma unroll
      for (int j4 = 0; j4 < RP / 4; ++j4) {
        const float4 qv = *reinterpret_cast<const float4*>(qt + row * RP + 4 * j4);
        acc[0][4 * j4 + 0] = fmaf(p0, qv.x, acc[0][4 * j4 + 0]);
        acc[0][4 * j4 + 1] = fmaf(p0, qv.y, acc[0][4 * j4 + 1]);
        acc[0][4 * j4 + 2] = fmaf(p0, qv.z, acc[0][4 * j4 + 2]);
        acc[0][4 * j4 + 3] = fmaf(p0, qv.w, acc[0][4 * j4 + 3]);
        acc[1][4 * j4 + 0] = fmaf(p1, qv.x, acc[1][4 * j4 + 0]);
        acc[1][4 * j4 + 1] = fmaf(p1, qv.y, acc[1][4 * j4 + 1]);
        acc[1][4 * j4 + 2] = fmaf(p1, qv.z, acc[1][4 * j4 + 2]);
        acc[1][4 * j4 + 3] = fmaf(p1, qv.w, acc[1][4 * j4 + 3]);
      }
    }
    __syncthreads();                                // the stage may be refilled next
  }
  cp_async_wait<0>();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = c0 + 2 * tid + h;
    if (i >= M) continue;
    float* out = part + ((long long)c * M + i) * R;
#pragma unroll
    for (int j = 0; j < RP; ++j)
      if (j < R) out[j] = acc[h][j];
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
  const int col_blocks = (M + kSkCols - 1) / kSkCols;
  int want = (2 * device_sm_count() + col_blocks - 1) / col_blocks;   // ~2 CTAs per SM
  int max_by_rows = (T + 255) / 256;                                  // at least 256 rows per chunk
  int nc = want < max_by_rows ? want : max_by_rows;
  return nc < 1 ? 1 : nc;
}

namespace {
template <int RP>
int launch_skinny_rp(const uint16_t* P, long long ldp, int T, int M, const float* Q, long long ldq,
                     int R, int nc, int tc, float* part, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kSkStages) * kSkRows * (kSkCols * 2 + RP * 4);
  cudaError_t e = cudaFuncSetAttribute(skinny_partial_kernel<RP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  dim3 grid((M + kSkCols - 1) / kSkCols, nc);
  skinny_partial_kernel<RP><<<grid, 256, smem, stream>>>(P, ldp, T, M, Q, ldq, R, tc, part);
  return check_launch();
}
}  // namespace

int launch_skinny(const void* P, int p_dtype, long long ldp, int T, int M, const float* Q,
                  long long ldq, int R, float scale, float* part, float* out, long long ldo,
                  bool transposed, cudaStream_t stream) {
  if (T <= 0 || M <= 0 || R <= 0) return WP_OK;
  if (R > 64 || p_dtype != WP_BF16 || M % 8 || ldp % 8) return WP_ERR_UNSUPPORTED;
  const int nc = skinny_chunks(T, M);
  const int tc = (T + nc - 1) / nc;
  const uint16_t* p = static_cast<const uint16_t*>(P);
  int rc = R <= 16   ? launch_skinny_rp<16>(p, ldp, T, M, Q, ldq, R, nc, tc, part, stream)
           : R <= 32 ? launch_skinny_rp<32>(p, ldp, T, M, Q, ldq, R, nc, tc, part, stream)
                     : launch_skinny_rp<64>(p, ldp, T, M, Q, ldq, R, nc, tc, part, stream);
  if (rc != WP_OK) return rc;
  const long long n = (long long)M * R;
  skinny_finish_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(part, nc, M, R, scale, out, ldo,
                                                                         transposed ? 1 : 0);
  return check_launch();
}

}  // namespace wp
