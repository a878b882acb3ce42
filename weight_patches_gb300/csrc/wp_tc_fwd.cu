// wp_tc_fwd.cu -- the fused dynamic-LoRA linear on the sm_103a tensor cores.
//
//   Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T        (per column group)
//
// sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM",
// Modifications: the combined scale multiplies the rank-wide intermediate X A^T, the
// second low-rank GEMM accumulates straight onto the base output so the [T, out]
// delta never exists, the bias belongs to the base GEMM's epilogue, stacked q/k/v
// (gate/up) adapters take one update per column group, and an FP32 adapter keeps its
// FP32 GEMMs and is added once.  Here all of it happens inside one persistent kernel:
//
//   * tiles are 128 (tokens) x 256 (output columns); each CTA owns a contiguous range
//     of tiles ordered (row block, group, column tile), so consecutive tiles share
//     their X row block and their group's adapters;
//   * when a CTA enters a new (row block, group) "unit" it first runs a rank pass: a
//     K-loop over the X row block against A_p (N = r_p) that leaves H_p = X A_p^T in
//     tensor memory; the epilogue warps scale it by the runtime s_p, round it once to
//     bf16 and park it in shared memory in the MMA operand layout;
//   * every tile then runs its base K-loop (X W^T into a 128x256 fp32 accumulator in
//     tensor memory) followed by the second contraction H~ B_tile^T into the same
//     accumulator, so the low-rank update costs K = r extra MMA steps per tile and the
//     rank pass costs r / (tiles per unit * 256) of the base work;
//   * the epilogue (8 warps) drains the accumulator to registers, frees tensor memory
//     for the next tile, adds the bias and the FP32 adapters' terms
//     (sum_j (s X A32^T)[t, j] * B32[o, j] with FFMA, before the single rounding),
//     and writes bf16 or fp32.
//
// Warp roles: warp 0 issues TMA loads, warp 1 issues tcgen05.mma (one thread each),
// warps 2..9 are the epilogue.  Operands are K-major bf16 in the 128-byte swizzle
// layout, one 64-element K slice per pipeline stage.  Every mbarrier wait is bounded
// (wall clock); on expiry the CTA records WP_ERR_TIMEOUT, waits for its own copies in
// flight, frees tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_ptx.cuh"

namespace wp {

static __device__ int g_tc_status;

namespace {

struct Tile {
  int m, g, j;
};

__device__ __forceinline__ Tile decode_tile(const TcParams& p, int L) {
  Tile t;
  const int mg = L / p.nt_g;
  t.j = L - mg * p.nt_g;
  t.m = mg / p.G;
  t.g = mg - t.m * p.G;
  return t;
}

__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

}  // namespace

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_fused_fwd_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base_addr - raw_addr);

  const int S = p.stages;
  uint8_t* hbuf = sbase + S * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(hbuf + p.hchunks * kHChunkBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* acc_full = bars + 2 * S;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* h_full = acc_full + 2;
  uint64_t* h_ready = acc_full + 3;
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 8);
    mbar_init(h_full, 1);
    mbar_init(h_ready, 8);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.x);
    if (p.has_base) tma_prefetch_desc(&maps.w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_acc = tmem;             // columns [0, 256)
  const uint32_t tmem_h = tmem + kBN;         // columns [256, 512)

  const long long total = p.total_tiles;
  const int t_begin = static_cast<int>(blockIdx.x * total / gridDim.x);
  const int t_end = static_cast<int>((blockIdx.x + 1) * total / gridDim.x);
  const uint64_t tmo = p.timeout_ns;
  int* status = &g_tc_status;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued[16];
      for (int s = 0; s < S; ++s) issued[s] = 0;
      bool ok = true;
      for (int L = t_begin; L < t_end && ok; ++L) {
        const Tile t = decode_tile(p, L);
        const int a0 = p.ad_begin[t.g], a1 = p.ad_begin[t.g + 1];
        const bool lora = a1 > a0;
        const bool new_unit = (L == t_begin) || (t.j == 0);
        const int m0 = t.m * kBM;
        if (lora && new_unit) {
          uint32_t bytes = kATileBytes;
          for (int a = a0; a < a1; ++a) bytes += p.ad[a].rpad16 * 128;
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!(ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, tmo, status))) break;
            uint8_t* st = sbase + stage * kStageBytes;
            mbar_arrive_expect_tx(&full[stage], bytes);
            tma_load_2d(st, &maps.x, kb * kBK, m0, &full[stage]);
            for (int a = a0; a < a1; ++a)
              tma_load_2d(st + kATileBytes + p.ad[a].chunk_off * 64 * 128, &maps.a[a], kb * kBK, 0,
                          &full[stage]);
            ++issued[stage];
            if (++stage == S) { stage = 0; phase ^= 1; }
          }
        }
        if (ok && p.has_base) {
          const int n_row0 = t.g * p.out_g + t.j * kBN;
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!(ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, tmo, status))) break;
            uint8_t* st = sbase + stage * kStageBytes;
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            tma_load_2d(st, &maps.x, kb * kBK, m0, &full[stage]);
            tma_load_2d(st + kATileBytes, &maps.w, kb * kBK, n_row0, &full[stage]);
            ++issued[stage];
            if (++stage == S) { stage = 0; phase ^= 1; }
          }
        }
        if (ok && lora) {
          for (int a = a0; a < a1 && ok; ++a) {
            for (int c = 0; c < p.ad[a].nchunks; ++c) {
              if (!(ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, tmo, status))) break;
              uint8_t* st = sbase + stage * kStageBytes;
              mbar_arrive_expect_tx(&full[stage], kBTileBytes);
              tma_load_2d(st + kATileBytes, &maps.b[a], c * 64, t.j * kBN, &full[stage]);
              ++issued[stage];
              if (++stage == S) { stage = 0; phase ^= 1; }
            }
          }
        }
      }
      if (!ok) {
        // Wait (bounded) for the copies this thread put in flight before the CTA exits.
        for (int s = 0; s < S; ++s) {
          if (issued[s] == 0) continue;
          const uint32_t par = static_cast<uint32_t>((issued[s] - 1) & 1);
          const uint32_t a = smem_u32(&full[s]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, par) && globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      uint32_t unit_phase = 0;
      const uint32_t idesc_acc = idesc_bf16_f32(kBM, kBN);
      const uint32_t hbuf_addr = smem_u32(hbuf);
      bool ok = true;
      for (int L = t_begin; L < t_end && ok; ++L) {
        const Tile t = decode_tile(p, L);
        const int a0 = p.ad_begin[t.g], a1 = p.ad_begin[t.g + 1];
        const bool lora = a1 > a0;
        const bool new_unit = (L == t_begin) || (t.j == 0);
        if (lora && new_unit) {
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!(ok = mbar_wait(&full[stage], phase, abort_flag, tmo, status))) break;
            tc_fence_after();
            const uint32_t st = smem_u32(sbase + stage * kStageBytes);
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint64_t adesc = sw128_kmajor_desc(st + kk * 32);
              for (int a = a0; a < a1; ++a) {
                const uint64_t bdesc =
                    sw128_kmajor_desc(st + kATileBytes + p.ad[a].chunk_off * 64 * 128 + kk * 32);
                mma_bf16(tmem_h + p.ad[a].chunk_off * 64, adesc, bdesc,
                         idesc_bf16_f32(kBM, p.ad[a].rpad16), (kb | kk) != 0);
              }
            }
            mma_commit(&empty[stage]);
            if (++stage == S) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          mma_commit(h_full);
        }
        if (!(p.has_base || lora)) continue;
        if (!(ok = mbar_wait(acc_empty, acc_phase ^ 1, abort_flag, tmo, status))) break;
        tc_fence_after();
        bool accum = false;
        if (p.has_base) {
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!(ok = mbar_wait(&full[stage], phase, abort_flag, tmo, status))) break;
            tc_fence_after();
            const uint32_t st = smem_u32(sbase + stage * kStageBytes);
            for (int kk = 0; kk < kBK / 16; ++kk) {
              mma_bf16(tmem_acc, sw128_kmajor_desc(st + kk * 32),
                       sw128_kmajor_desc(st + kATileBytes + kk * 32), idesc_acc,
                       (accum || kk > 0) ? 1u : 0u);
            }
            accum = true;
            mma_commit(&empty[stage]);
            if (++stage == S) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
        }
        if (lora) {
          if (new_unit) {
            if (!(ok = mbar_wait(h_ready, unit_phase, abort_flag, tmo, status))) break;
            tc_fence_after();
            unit_phase ^= 1;
          }
          for (int a = a0; a < a1 && ok; ++a) {
            for (int c = 0; c < p.ad[a].nchunks; ++c) {
              if (!(ok = mbar_wait(&full[stage], phase, abort_flag, tmo, status))) break;
              tc_fence_after();
              const uint32_t st = smem_u32(sbase + stage * kStageBytes);
              const int kext = min(64, p.ad[a].rpad16 - 64 * c);
              const uint32_t hchunk = hbuf_addr + (p.ad[a].chunk_off + c) * kHChunkBytes;
              for (int kk = 0; kk < kext / 16; ++kk) {
                mma_bf16(tmem_acc, sw128_kmajor_desc(hchunk + kk * 32),
                         sw128_kmajor_desc(st + kATileBytes + kk * 32), idesc_acc,
                         (accum || kk > 0) ? 1u : 0u);
              }
              accum = true;
              mma_commit(&empty[stage]);
              if (++stage == S) { stage = 0; phase ^= 1; }
            }
          }
          if (!ok) break;
        }
        mma_commit(acc_full);
        acc_phase ^= 1;
      }
      // Make sure every MMA this thread issued has finished before TMEM is freed.
      mma_commit(drain);
      const uint32_t a = smem_u32(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (8 warps)
    const int e = warp - 2;
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int half = e >> 2;                // which 128 of the 256 tile columns
    const int row_in_tile = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t hbuf_addr = smem_u32(hbuf);
    uint32_t acc_phase = 0;
    uint32_t unit_phase = 0;
    for (int L = t_begin; L < t_end; ++L) {
      const Tile t = decode_tile(p, L);
      const int a0 = p.ad_begin[t.g], a1 = p.ad_begin[t.g + 1];
      const bool lora = a1 > a0;
      const bool new_unit = (L == t_begin) || (t.j == 0);
      if (lora && new_unit) {
        // every lane waits; the warp proceeds only if all lanes saw the phase, so the
        // .sync.aligned TMEM loads below are always executed by the whole warp
        if (!__all_sync(0xffffffffu, mbar_wait(h_full, unit_phase, abort_flag, tmo, status))) break;
        tc_fence_after();
        unit_phase ^= 1;
        for (int a = a0; a < a1; ++a) {
          const float s = p.ad[a].s;
          const int units = p.ad[a].rpad16 >> 3;
          for (int u = half; u < units; u += 2) {
            uint32_t r[8];
            tmem_ld8(tmem_h + lane_base + p.ad[a].chunk_off * 64 + u * 8, r);
            const uint32_t w0 = pack_bf16x2(u2f(r[0]) * s, u2f(r[1]) * s);
            const uint32_t w1 = pack_bf16x2(u2f(r[2]) * s, u2f(r[3]) * s);
            const uint32_t w2 = pack_bf16x2(u2f(r[4]) * s, u2f(r[5]) * s);
            const uint32_t w3 = pack_bf16x2(u2f(r[6]) * s, u2f(r[7]) * s);
            const int chunk = p.ad[a].chunk_off + (u >> 3);
            const int unit16 = (u & 7) ^ (row_in_tile & 7);
            st_shared_v4(hbuf_addr + chunk * kHChunkBytes + row_in_tile * 128 + unit16 * 16, w0,
                         w1, w2, w3);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(h_ready);
      }

      float acc[128];
      const bool any_mma = p.has_base || lora;
      if (any_mma) {
        if (!__all_sync(0xffffffffu, mbar_wait(acc_full, acc_phase, abort_flag, tmo, status))) break;
        tc_fence_after();
        acc_phase ^= 1;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem_acc + lane_base + half * 128 + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[c * 32 + i] = u2f(r[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) acc[i] = 0.f;
      }

      const int row = t.m * kBM + row_in_tile;
      const int col_in_group0 = t.j * kBN + half * 128;     // first column of this thread
      const int gcol0 = t.g * p.out_g + col_in_group0;      // same, in Y
      const int ncols = min(128, p.out_g - col_in_group0);  // valid columns (may be <= 0)
      if (ncols <= 0) continue;

      if (p.bias) {
        if (p.bias_f32) {
          const float* b = static_cast<const float*>(p.bias) + gcol0;
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i < ncols) acc[i] += b[i];
        } else {
          const uint16_t* b = static_cast<const uint16_t*>(p.bias) + gcol0;
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i < ncols) acc[i] += bf16_to_f32(b[i]);
        }
      }

      if (p.n_ad32 > 0 && row < p.T) {
        for (int a = 0; a < p.n_ad32; ++a) {
          if (p.ad32[a].group != t.g) continue;
          const float* hrow = p.h32 + static_cast<long long>(row) * p.h32_cols + p.ad32[a].h_off;
          const int r = p.ad32[a].rank;
          const float* Bm = p.ad32[a].B;
          const long long ldb = p.ad32[a].ldb;
          for (int jj = 0; jj < r; ++jj) {
            const float h = hrow[jj];
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (i < ncols) acc[i] = fmaf(h, Bm[static_cast<long long>(col_in_group0 + i) * ldb + jj], acc[i]);
          }
        }
      }

      if (row < p.T) {
        if (p.y_f32) {
          float* yrow = static_cast<float*>(p.Y) + static_cast<long long>(row) * p.ldy + gcol0;
#pragma unroll
          for (int v = 0; v < 32; ++v)
            if (v * 4 < ncols)
              st_global_v4(yrow + v * 4, f2u(acc[4 * v]), f2u(acc[4 * v + 1]), f2u(acc[4 * v + 2]),
                           f2u(acc[4 * v + 3]));
        } else {
          uint16_t* yrow = static_cast<uint16_t*>(p.Y) + static_cast<long long>(row) * p.ldy + gcol0;
#pragma unroll
          for (int v = 0; v < 16; ++v)
            if (v * 8 < ncols)
              st_global_v4(yrow + v * 8, pack_bf16x2(acc[8 * v], acc[8 * v + 1]),
                           pack_bf16x2(acc[8 * v + 2], acc[8 * v + 3]),
                           pack_bf16x2(acc[8 * v + 4], acc[8 * v + 5]),
                           pack_bf16x2(acc[8 * v + 6], acc[8 * v + 7]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int launch_tc_fwd(const TcMaps& maps, const TcParams& p, int grid, size_t smem_bytes,
                  cudaStream_t stream) {
  cudaError_t ea = cudaFuncSetAttribute(tc_fused_fwd_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (ea != cudaSuccess) {
    set_last_cuda_error(ea);
    return WP_ERR_CUDA;
  }
  tc_fused_fwd_kernel<<<grid, kTcThreads, smem_bytes, stream>>>(maps, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int tc_fwd_status(int reset) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int));
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  if (reset && v != 0) {
    int z = 0;
    cudaMemcpyToSymbol(g_tc_status, &z, sizeof(int));
  }
  return v;
}

}  // namespace wp
