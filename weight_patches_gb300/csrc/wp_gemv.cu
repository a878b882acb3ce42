// wp_gemv.cu -- the dynamic LoRA linear for one to four tokens on the CUDA cores, against a
// 4-bit NormalFloat or a bf16 base weight (Unsloth fast_lora walkthrough, section 3: the 4-bit
// weight is dequantised inside the matmul; LoRA, section 4.1: the low-rank branch X A^T is
// formed from the same X).  With so few tokens the product is a matrix-vector one: every
// weight element is used T times, so the work is streaming the weight from HBM once (and, for
// 4 bits, turning its codes into bf16 values), not a contraction worth the tensor cores.
//
// Each warp owns 32 consecutive weight rows at a time, one per lane, and a ring of stages it
// fills itself by TMA (128 B x 32 rows in the 128-byte swizzle: 256 codes or 64 bf16 values
// a row; for 4 bits also the rows' 4 fp32 block scales), so a lane reads its row's 16-byte
// units without bank conflicts and no role waits on another.  A lane builds the 16 values bf16(level * absmax) of a 64-element block in two byte
// planes and looks its codes up with byte permutes (the same W_eff the tensor-core paths put
// in their operand tiles), then multiplies them by X read from shared memory, the same address
// in every lane (a broadcast), with mixed-precision fmas (bf16 pairs in, fp32 sums): the
// integer pipe, which carries the permutes, is the kernel's bound, so nothing else goes there.
// Sums are fp32 per lane; a block of warps shares one
// K range (a split) whose X it holds.  The adapters' A rows go one row per warp, lanes along
// K, reduced by shuffles.  Partial sums land in the layout the small-token reduce reads.
#include <atomic>

#include "wp_internal.h"
#include "wp_nf4.cuh"
#include "wp_ptx.cuh"

namespace wp {
namespace {

// Bounded wait by every lane of a warp; the warp agrees on the outcome.  False: the budget
// ran out in some lane (the status records WP_ERR_TIMEOUT).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          int* status) {
  const uint32_t a = smem_u32(bar);
  bool ok = true;
  if (!mbar_try_wait(a, parity)) {
    SpinBudget budget;
    while (!mbar_try_wait(a, parity)) {
      if (budget.spent(timeout_ns)) {
        ok = false;
        break;
      }
    }
  }
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) atomicExch(status, kErrTimeout);
  return ok;
}

// acc + w.lo * x.lo + w.hi * x.hi for two bf16 pairs: the mixed-precision fma (bf16 operands,
// fp32 addend and result, one rounding each), the same as fp32 fmas of the widened values.
__device__ __forceinline__ float fma_bf16x2(uint32_t w, uint32_t x, float acc) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %1;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
      : "+f"(acc)
      : "r"(w), "r"(x));
  return acc;
}

// The 16 values of a block in two byte planes (lo / hi: low and high bytes of entries 4j..4j+3).
__device__ __forceinline__ void block_table(float am, const float (&lv)[16], uint32_t (&lo)[4],
                                            uint32_t (&hi)[4]) {
  uint32_t e[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) e[k] = pack_bf16x2(lv[2 * k] * am, lv[2 * k + 1] * am);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    lo[j] = prmt(e[2 * j], e[2 * j + 1], 0x6420u);
    hi[j] = prmt(e[2 * j], e[2 * j + 1], 0x7531u);
  }
}

// kNF4: 4-bit codes and block scales, 256 K elements per stage; else bf16 rows, 64 per stage
template <int kT, bool kNF4>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_kernel(const __grid_constant__ GemvMaps maps,
                                                               const GemvParams p) {
  constexpr int kStageK = kNF4 ? kGemvStageK : 64;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.splits;
  const int jb = blockIdx.x / p.splits;
  const int nbs = gridDim.x / p.splits;           // the host launches a multiple of the splits
  const int k0 = split * p.ks_len;
  const int klen = min(p.ks_len, p.K - k0);

  uint8_t* codes = sbase + warp * kGemvStages * kGemvCodeBytes;
  uint8_t* ams = sbase + kGemvWarps * kGemvStages * kGemvCodeBytes + warp * kGemvStages * kGemvAmBytes;
  uint16_t* xs = reinterpret_cast<uint16_t*>(sbase + kGemvWarps * kGemvStages * (kGemvCodeBytes + kGemvAmBytes));
  uint64_t* bars = reinterpret_cast<uint64_t*>(xs + kT * p.ks_len) + warp * kGemvStages;  // ks_len % 256 == 0

  if (lane == 0) {
    for (int s = 0; s < kGemvStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  // X of this split, [t][k - k0] bf16
  for (int i = threadIdx.x; i < kT * klen / 8; i += blockDim.x) {
    const int t = i / (klen / 8);
    const int k = (i - t * (klen / 8)) * 8;
    *reinterpret_cast<uint4*>(xs + t * p.ks_len + k) =
        __ldg(reinterpret_cast<const uint4*>(p.X + t * p.ldx + k0 + k));
  }
  __syncthreads();

  const int gw = jb * kGemvWarps + warp;          // this warp among its split's warps
  const int wstride = nbs * kGemvWarps;
  const int units = p.ngW + p.R16;
  float* part = p.part + static_cast<long long>(split) * p.T * p.ldp;

  // ---- weight rows: flat sequence of (unit, stage) over this warp's 32-row groups
  const int ns = klen / kStageK;
  const int my_w = gw < p.ngW ? (p.ngW - gw + wstride - 1) / wstride : 0;
  const int n_it = my_w * ns;
  int issued = 0;
  auto issue = [&](int it) {
    const int g = gw + (it / ns) * wstride;
    const int kk = k0 + (it % ns) * kStageK;
    const int s = it % kGemvStages;
    if (kNF4) {
      mbar_arrive_expect_tx(&bars[s], kGemvCodeBytes + kGemvAmBytes);
      tma_load_2d(codes + s * kGemvCodeBytes, &maps.wq, kk / 2, g * 32, &bars[s]);
      tma_load_2d(ams + s * kGemvAmBytes, &maps.am, kk / 64, g * 32, &bars[s]);
    } else {
      mbar_arrive_expect_tx(&bars[s], kGemvCodeBytes);
      tma_load_2d(codes + s * kGemvCodeBytes, &maps.w, kk, g * 32, &bars[s]);
    }
  };
  if (lane == 0)
    for (int it = 0; it < kGemvStages - 1 && it < n_it; ++it) issue(it);
  issued = min(n_it, kGemvStages - 1);

  float lv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) lv[i] = p.nf4_code[i];
  float acc[kT][2];
#pragma unroll
  for (int t = 0; t < kT; ++t) acc[t][0] = acc[t][1] = 0.f;

  bool ok = true;
  for (int it = 0; it < n_it; ++it) {
    if (issued < n_it) {
      // the slot refilled here was read in the previous iteration, by every lane
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(issued);
      }
      ++issued;
    }
    const int s = it % kGemvStages;
    if (!warp_wait(&bars[s], (it / kGemvStages) & 1, p.timeout_ns, p.status)) {
      ok = false;
      // settle the copies still in flight into this warp's slots before leaving
      for (int j = it; j < issued; ++j)
        if (!warp_wait(&bars[j % kGemvStages], (j / kGemvStages) & 1, p.timeout_ns, p.status)) break;
      break;
    }
    const int st = it % ns;
    const uint8_t* crow = codes + s * kGemvCodeBytes + lane * 128;
    if (!kNF4) {
      // bf16 row: 64 elements in 8 units of 8
#pragma unroll
      for (int unit = 0; unit < 8; ++unit) {
        const uint4 wv = *reinterpret_cast<const uint4*>(crow + ((unit ^ (lane & 7)) << 4));
        const int e0 = st * kStageK + unit * 8;
#pragma unroll
        for (int t = 0; t < kT; ++t) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * p.ks_len + e0);
          float& a = acc[t][unit & 1];
          a = fma_bf16x2(wv.x, xv.x, a);
          a = fma_bf16x2(wv.y, xv.y, a);
          a = fma_bf16x2(wv.z, xv.z, a);
          a = fma_bf16x2(wv.w, xv.w, a);
        }
      }
    } else {
    const uint4 amv = *reinterpret_cast<const uint4*>(ams + s * kGemvAmBytes + lane * 16);
    const float am4[4] = {__uint_as_float(amv.x), __uint_as_float(amv.y), __uint_as_float(amv.z),
                          __uint_as_float(amv.w)};
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      uint32_t lo[4], hi[4];
      block_table(am4[blk], lv, lo, hi);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int unit = blk * 2 + half;
        const uint4 cw4 = *reinterpret_cast<const uint4*>(crow + ((unit ^ (lane & 7)) << 4));
        const uint32_t cw[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t c = cw[u];
          const uint32_t sel = c & 0x77777777u;
          const uint32_t pick = ((c >> 1) & 0x44444444u) | 0x32103210u;
          uint32_t o[4];
          lookup4(sel, pick, lo, hi, o[0], o[1]);
          lookup4(sel >> 16, pick >> 16, lo, hi, o[2], o[3]);
          const int e0 = st * kStageK + unit * 32 + u * 8;
#pragma unroll
          for (int t = 0; t < kT; ++t) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * p.ks_len + e0);
            float& a = acc[t][u & 1];
            a = fma_bf16x2(o[0], xv.x, a);
            a = fma_bf16x2(o[1], xv.y, a);
            a = fma_bf16x2(o[2], xv.z, a);
            a = fma_bf16x2(o[3], xv.w, a);
          }
        }
      }
    }
    }
    if (st == ns - 1) {
      const int n = (gw + (it / ns) * wstride) * 32 + lane;
      if (n < p.N) {
#pragma unroll
        for (int t = 0; t < kT; ++t) part[static_cast<long long>(t) * p.ldp + n] = acc[t][0] + acc[t][1];
      }
#pragma unroll
      for (int t = 0; t < kT; ++t) acc[t][0] = acc[t][1] = 0.f;
    }
  }
  if (!ok) return;

  // ---- adapter A rows: one row per unit, lanes along K, then a shuffle reduction
  const int first_a = gw < p.ngW ? gw + my_w * wstride : gw;
  for (int u = first_a; u < units; u += wstride) {
    const int ar = u - p.ngW;
    int a = 0;
    while (a + 1 < p.n_ad && ar >= p.a_off[a + 1]) ++a;
    const int j = ar - p.a_off[a];
    float sum[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) sum[t] = 0.f;
    if (j < p.rank[a]) {
      const uint16_t* row = p.A[a] + j * p.lda[a] + k0;
      for (int kk = lane * 8; kk < klen; kk += 256) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + kk));
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < kT; ++t) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * p.ks_len + kk);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) sum[t] = fma_bf16x2(wv[k], xw[k], sum[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < kT; ++t)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum[t] += __shfl_xor_sync(0xffffffffu, sum[t], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < kT; ++t) part[static_cast<long long>(t) * p.ldp + p.N + ar] = sum[t];
    }
  }
}

// A 16-byte load of weight bytes read once: not kept in L1.
__device__ __forceinline__ uint4 ld_once_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_once_f32(const float* p) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// The 4-bit weight against one token by plain loads.  The TMA ring above pays the
// copy engine per row of every box (32 rows of 128 code bytes and 32 rows of 16 scale
// bytes a stage), which held the weight stream to about half the HBM rate.  Here a warp
// takes whole 2048-element slices of a row: lane l loads the 32 code bytes of elements
// [64 l, 64 l + 64) of the slice (one 64-element block, so one scale and one 16-entry table
// per lane and row) with two 16-byte loads, the warp's loads covering 1 KiB of the row, and
// keeps its 64 X values in registers for every row it takes (two tokens' would not fit
// beside the ring without spilling, so two to four tokens stay on the kernel above).  A split is one slice (K must
// be a multiple of 2048); the row's slice sum is a shuffle reduction, written where the
// small-token reduce reads the K splits.  Rows go two at a time through a three-deep ring of
// registers, so four rows' loads are in flight while two are computed.
template <int kT>
__global__ void __launch_bounds__(kGemvLdWarps * 32, 2) gemv_nf4_ld_kernel(const GemvParams p,
                                                                             const uint8_t* __restrict__ codes,
                                                                             const float* __restrict__ absmax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.splits;
  const int jb = blockIdx.x / p.splits;
  const int nbs = gridDim.x / p.splits;           // the host launches a multiple of the splits
  const int kl = split * kGemvLdSlice + lane * 64;    // this lane's 64 elements
  uint32_t xw[kT][32];                            // X pairs (elements 2i, 2i + 1) of them
#pragma unroll
  for (int t = 0; t < kT; ++t)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.X + t * p.ldx + kl + 8 * i));
      xw[t][4 * i] = v.x; xw[t][4 * i + 1] = v.y; xw[t][4 * i + 2] = v.z; xw[t][4 * i + 3] = v.w;
    }
  float lv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) lv[i] = p.nf4_code[i];
  const int gw = jb * kGemvLdWarps + warp;
  const int wstride = nbs * kGemvLdWarps;
  float* part = p.part + static_cast<long long>(split) * p.T * p.ldp;
  const long long row_bytes = p.K / 2, row_blocks = p.K / 64;

  struct Rows {
    uint4 c[2][2];    // [row][16-byte half]
    float am[2];
  };
  // rows gw + (2 j + i) wstride, i = 0, 1 (past the last row: zeros, nothing read)
  auto load = [&](Rows& b, int j) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = gw + (2 * j + i) * wstride;
      if (r < p.N) {
        const uint8_t* src = codes + static_cast<long long>(r) * row_bytes + kl / 2;
        b.c[i][0] = ld_once_v4(src);
        b.c[i][1] = ld_once_v4(src + 16);
        b.am[i] = ld_once_f32(absmax + static_cast<long long>(r) * row_blocks + kl / 64);
      } else {
        b.c[i][0] = b.c[i][1] = make_uint4(0u, 0u, 0u, 0u);
        b.am[i] = 0.f;
      }
    }
  };
  auto compute = [&](const Rows& b, int j) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = gw + (2 * j + i) * wstride;
      uint32_t lo[4], hi[4];
      block_table(b.am[i], lv, lo, hi);
      const uint32_t cw[8] = {b.c[i][0].x, b.c[i][0].y, b.c[i][0].z, b.c[i][0].w,
                              b.c[i][1].x, b.c[i][1].y, b.c[i][1].z, b.c[i][1].w};
      float acc[kT][2];
#pragma unroll
      for (int t = 0; t < kT; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t c = cw[u];
        const uint32_t sel = c & 0x77777777u;
        const uint32_t pick = ((c >> 1) & 0x44444444u) | 0x32103210u;
        uint32_t o[4];
        lookup4(sel, pick, lo, hi, o[0], o[1]);
        lookup4(sel >> 16, pick >> 16, lo, hi, o[2], o[3]);
#pragma unroll
        for (int t = 0; t < kT; ++t) {
          float& a = acc[t][u & 1];
          a = fma_bf16x2(o[0], xw[t][4 * u], a);
          a = fma_bf16x2(o[1], xw[t][4 * u + 1], a);
          a = fma_bf16x2(o[2], xw[t][4 * u + 2], a);
          a = fma_bf16x2(o[3], xw[t][4 * u + 3], a);
        }
      }
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        float sum = acc[t][0] + acc[t][1];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0 && r < p.N) part[static_cast<long long>(t) * p.ldp + r] = sum;
      }
    }
  };
  const int nrows = gw < p.N ? (p.N - gw + wstride - 1) / wstride : 0;
  const int npr = (nrows + 1) / 2;                // row pairs of this warp
  Rows b0, b1, b2;
  load(b0, 0);
  load(b1, 1);
  for (int j = 0; j < npr; j += 3) {
    load(b2, j + 2);
    compute(b0, j);
    if (j + 1 >= npr) break;
    load(b0, j + 3);
    compute(b1, j + 1);
    if (j + 2 >= npr) break;
    load(b1, j + 4);
    compute(b2, j + 2);
  }

  // adapter A rows (bf16): the same lane slices, one row per warp
  for (int ar = gw; ar < p.R16; ar += wstride) {
    int a = 0;
    while (a + 1 < p.n_ad && ar >= p.a_off[a + 1]) ++a;
    const int j = ar - p.a_off[a];
    float sum[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) sum[t] = 0.f;
    if (j < p.rank[a]) {
      const uint16_t* row = p.A[a] + j * p.lda[a] + kl;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + 8 * i));
#pragma unroll
        for (int t = 0; t < kT; ++t) {
          sum[t] = fma_bf16x2(v.x, xw[t][4 * i], sum[t]);
          sum[t] = fma_bf16x2(v.y, xw[t][4 * i + 1], sum[t]);
          sum[t] = fma_bf16x2(v.z, xw[t][4 * i + 2], sum[t]);
          sum[t] = fma_bf16x2(v.w, xw[t][4 * i + 3], sum[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kT; ++t) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum[t] += __shfl_xor_sync(0xffffffffu, sum[t], o);
      if (lane == 0) part[static_cast<long long>(t) * p.ldp + p.N + ar] = sum[t];
    }
  }
}

template <int kT, bool kNF4>
int launch_t(const GemvMaps& maps, const GemvParams& p, int grid, size_t smem, cudaStream_t stream) {
  auto kern = gemv_kernel<kT, kNF4>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) {
    kern<<<grid, kGemvWarps * 32, smem, stream>>>(maps, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

template <int kT, bool kNF4>
int occupancy_t(size_t smem) {
  int n = 0;
  if (cudaFuncSetAttribute(gemv_kernel<kT, kNF4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<kT, kNF4>, kGemvWarps * 32, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace

size_t gemv_smem_bytes(int T, int ks_len) {
  return 1024 + static_cast<size_t>(kGemvWarps) * kGemvStages * (kGemvCodeBytes + kGemvAmBytes) +
         static_cast<size_t>(T) * ks_len * 2 + kGemvWarps * kGemvStages * 8;
}

int gemv_blocks_per_sm(int T, bool nf4, size_t smem) {
  // the answer depends on T, the weight type and the shared memory alone; kept per 1 KiB
  static std::atomic<int> cache[2][kGemvMaxT + 1][kSmemLimit / 1024 + 2];
  if (T < 1 || T > kGemvMaxT || smem > static_cast<size_t>(kSmemLimit)) return 0;
  std::atomic<int>& c = cache[nf4 ? 1 : 0][T][(smem + 1023) / 1024];
  int n = c.load(std::memory_order_relaxed);
  if (n != 0) return n > 0 ? n : 0;
  if (nf4) {
    switch (T) {
      case 1: n = occupancy_t<1, true>(smem); break;
      case 2: n = occupancy_t<2, true>(smem); break;
      case 3: n = occupancy_t<3, true>(smem); break;
      default: n = occupancy_t<4, true>(smem); break;
    }
  } else {
    switch (T) {
      case 1: n = occupancy_t<1, false>(smem); break;
      case 2: n = occupancy_t<2, false>(smem); break;
      case 3: n = occupancy_t<3, false>(smem); break;
      default: n = occupancy_t<4, false>(smem); break;
    }
  }
  c.store(n > 0 ? n : -1, std::memory_order_relaxed);
  return n;
}

int launch_gemv_ld(const GemvParams& p, const void* codes, const float* absmax, int grid, cudaStream_t stream) {
  if (grid < 1) return WP_OK;
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  if (p.T != 1) return WP_ERR_UNSUPPORTED;
  gemv_nf4_ld_kernel<1><<<grid, kGemvLdWarps * 32, 0, stream>>>(p, c, absmax);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int launch_gemv(const GemvMaps& maps, const GemvParams& p, bool nf4, int grid, size_t smem,
                cudaStream_t stream) {
  if (grid < 1) return WP_OK;
  if (nf4) {
    switch (p.T) {
      case 1: return launch_t<1, true>(maps, p, grid, smem, stream);
      case 2: return launch_t<2, true>(maps, p, grid, smem, stream);
      case 3: return launch_t<3, true>(maps, p, grid, smem, stream);
      case 4: return launch_t<4, true>(maps, p, grid, smem, stream);
      default: return WP_ERR_UNSUPPORTED;
    }
  }
  switch (p.T) {
    case 1: return launch_t<1, false>(maps, p, grid, smem, stream);
    case 2: return launch_t<2, false>(maps, p, grid, smem, stream);
    case 3: return launch_t<3, false>(maps, p, grid, smem, stream);
    case 4: return launch_t<4, false>(maps, p, grid, smem, stream);
    default: return WP_ERR_UNSUPPORTED;
  }
}

}  // namespace wp
