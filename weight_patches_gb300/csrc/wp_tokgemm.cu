// wp_tokgemm.cu -- contractions over the token index on the tensor cores, for the
// closed-form backward's adapter gradients (Unsloth fast_lora walkthrough, sections 2 and 4):
//   dB_g = s_g dY_g^T H_g      dA_g = (s_g G_g)^T X
// Both are D[m, n] = sum_t A[t, m] B[t, n] with A = dY or X ([T, M] bf16, row-major) and B the
// rank-wide operand ([T, N] bf16: every group's columns, as a high and a low bf16 piece of the
// fp32 values, zero-padded to N = 128 or 256).  The token index is the outer index of both, so
// the operands are MN-major: TMA brings boxes of 64 tokens x 64 columns in the 128-byte swizzle
// layout (each token a 128-byte row, 8 tokens a 1 KiB atom), and the tcgen05 descriptors step
// 8192 bytes between 64-column chunks and 1024 bytes between 8-token groups.  A CTA pair owns
// 256 rows of D (each CTA 128, its TMEM lanes) and all N columns; the tokens are split into
// ranges so the (256-row block, token range) units spread over the pairs, and each unit writes
// fp32 partial sums that a finishing kernel adds in a fixed order (so the result does not
// depend on the launch geometry), together with the two pieces, the scale and the transposition.
#include <cuda.h>
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_ptx.cuh"

namespace wp {

namespace {

constexpr int kTgABytes = 2 * 64 * 128;          // this CTA's 128 rows of D: two 64-column boxes


__global__ void __launch_bounds__(192, 1) tokgemm_kernel(const __grid_constant__ TokGemmMaps maps,
                                                         const __grid_constant__ TokGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base_addr - raw_addr);
  const int S = p.stages;
  const int bbytes = p.N / 2 * 128;                    // this CTA's half of B: N/2 columns
  const int SB = kTgABytes + bbytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + S * SB);
  uint64_t* full = bars;                  // [S] leader: both CTAs' bytes landed
  uint64_t* empty = bars + S;             // [S] both: the pair MMAs consumed the stage
  uint64_t* acc_full = bars + 2 * S;      // [2]
  uint64_t* acc_empty = acc_full + 2;     // [2] leader: both epilogues drained it
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();
  const bool leader = cta == 0;
  const uint32_t tmem_cols = 2 * static_cast<uint32_t>(p.N);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], 8);          // 4 epilogue warps x 2 CTAs
    mbar_init(&acc_empty[1], 8);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, tmem_cols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const uint64_t tmo = p.timeout_ns;
  int* status = p.status;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t keep = l2_evict_last();     // the narrow B: read by every unit
      const uint64_t once = l2_evict_first();    // A: each token range of a row block once
      int stage = 0;
      uint32_t phase = 0;
      int issued[kMaxStages];
      for (int s = 0; s < kMaxStages; ++s) issued[s] = 0;
      bool ok = true;
      for (int u = pair; u < p.units && ok; u += npairs) {
        const int mt = u / p.splits, ks = u - mt * p.splits;
        const int kb0 = ks * p.kb_per_split, kb1 = min(p.k_blocks, kb0 + p.kb_per_split);
        const int m0 = mt * 256 + static_cast<int>(cta) * 128;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!(ok = mbar_wait_cluster(&empty[stage], phase ^ 1, abort_flag, tmo, status))) break;
          uint8_t* st = sbase + stage * SB;
          const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2u * static_cast<uint32_t>(SB));
          tma_load_2d_pair_hint(st, &maps.a, m0, kb * 64, fb, once);
          tma_load_2d_pair_hint(st + kTgABytes / 2, &maps.a, m0 + 64, kb * 64, fb, once);
          for (int c = 0; c < p.N / 128; ++c)
            tma_load_2d_pair_hint(st + kTgABytes + c * 8192, &maps.b, static_cast<int>(cta) * (p.N / 2) + c * 64,
                                  kb * 64, fb, keep);
          ++issued[stage];
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        for (int s = 0; s < S; ++s) {
          if (issued[s] == 0 || !leader) continue;
          const uint32_t a = smem_u32(&full[s]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait_cluster(a, static_cast<uint32_t>((issued[s] - 1) & 1)) &&
                 globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t nuse[2] = {0, 0};
      int count = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16_f32_mn(256, static_cast<uint32_t>(p.N));
      const uint32_t stage_base = smem_u32(sbase);
      for (int u = pair; u < p.units && ok; u += npairs) {
        const int mt = u / p.splits, ks = u - mt * p.splits;
        const int kb0 = ks * p.kb_per_split, kb1 = min(p.k_blocks, kb0 + p.kb_per_split);
        const int b = count & 1;
        if (!(ok = mbar_wait_cluster(&acc_empty[b], (nuse[b] & 1) ^ 1, abort_flag, tmo, status))) break;
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!(ok = mbar_wait(&full[stage], phase, abort_flag, tmo, status))) break;
          tc_fence_after();
          const uint32_t st = stage_base + stage * SB;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // 16 tokens per MMA: two 8-token groups of 1 KiB
            mma_bf16_pair(tmem + b * p.N, sw128_mnmajor_desc(st + kk * 2048),
                          sw128_mnmajor_desc(st + kTgABytes + kk * 2048), idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          mma_commit_pair_mc(&empty[stage], 0x3);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair_mc(&acc_full[b], 0x3);
        ++nuse[b];
        ++count;
      }
      mma_commit_pair_mc(drain, 0x1);
      const uint32_t a = smem_u32(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait_cluster(a, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    // thread = one row of D (its TMEM lane); all N columns as fp32 partial sums
    const int q = warp & 3;
    const int row_in_cta = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t acc_empty_l[2] = {mapa_shared(smem_u32(&acc_empty[0]), 0),
                                     mapa_shared(smem_u32(&acc_empty[1]), 0)};
    uint32_t nuse[2] = {0, 0};
    int count = 0;
    for (int u = pair; u < p.units; u += npairs) {
      const int mt = u / p.splits, ks = u - mt * p.splits;
      const int b = count & 1;
      const bool okw = mbar_wait_cluster(&acc_full[b], nuse[b] & 1, abort_flag, tmo, status);
      if (!__all_sync(0xffffffffu, okw)) break;
      tc_fence_after();
      const int m = mt * 256 + static_cast<int>(cta) * 128 + row_in_cta;
      float* dst = p.part + (static_cast<long long>(ks) * p.M + m) * p.N;
#pragma unroll 1
      for (int c = 0; c < p.N / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + b * p.N + lane_base + c * 32, r);
        if (m < p.M) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(dst + c * 32)[i] =
                make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                            __uint_as_float(r[4 * i + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_l[b]);
      ++nuse[b];
      ++count;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, tmem_cols);
  }
}

// fp32 [T, R] (row pitch ld) -> bf16 pieces [T, N]: column off[g] + j of group g (j < r[g])
// gets hi = bf16(v) in column roff16[g] + j and lo = bf16(v - hi) in column R16 + roff16[g] + j;
// every other column is zero.
// A block takes kPieceRows token rows; thread c owns output column c of every one of them (its
// group, rank column and piece worked out once), so loads and stores are contiguous along c.
constexpr int kPieceRows = 8;

__global__ void __launch_bounds__(256) pieces_kernel(const float* src, long long ld, int T, int N,
                                                     TokPieceMap pm, uint16_t* dst) {
  const int c = threadIdx.x;
  const int piece = c >= pm.R16 ? 1 : 0;
  const int cc = c - piece * pm.R16;
  int col = -1;                                   // the source column, or -1 for a zero
  if (c < N && cc < pm.R16)
    for (int g = 0; g < pm.G; ++g) {
      const int j = cc - pm.roff16[g];
      if (j >= 0 && j < pm.r[g]) col = pm.off[g] + j;
    }
  for (int i = 0; i < kPieceRows; ++i) {
    const long long t = static_cast<long long>(blockIdx.x) * kPieceRows + i;
    if (t >= T || c >= N) break;
    uint16_t out = 0;
    if (col >= 0) {
      const float v = src[t * ld + col];
      uint16_t hi;
      asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(hi) : "f"(v));
      if (piece == 0) {
        out = hi;
      } else {
        const float rest = __fsub_rn(v, __uint_as_float(static_cast<uint32_t>(hi) << 16));
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(out) : "f"(rest));
      }
    }
    dst[t * N + c] = out;
  }
}

// out_g[j, i] (transposed) or out_g[m, j]: scale * sum over splits of (hi + lo columns), rows
// [row0, row0 + rows) of D for group g, in a fixed order.  A block takes kFinRows rows and all r
// columns: loads along j (contiguous in the partial sums), every split's loads issued before
// any is added (in split order); the transposed form goes through shared memory so that its
// stores run along m.
constexpr int kFinRows = 16;
constexpr int kFinMaxR = 128;

__global__ void __launch_bounds__(256) tok_finish_kernel(const float* part, int M, int N, int splits, int R16,
                                                         int roff16, int r, int row0, int rows, float scale,
                                                         float* out, long long ldo, int transposed) {
  __shared__ float tile[kFinRows][kFinMaxR + 1];
  const int m0 = blockIdx.x * kFinRows;
  const int nm = min(kFinRows, rows - m0);
  for (int idx = threadIdx.x; idx < nm * r; idx += blockDim.x) {
    const int mm = idx / r, j = idx - mm * r;
    const long long m = row0 + m0 + mm;
    float acc = 0.f;
    for (int k0 = 0; k0 < splits; k0 += 4) {
      float hi[4], lo[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float* pr = part + (static_cast<long long>(min(k0 + q, splits - 1)) * M + m) * N;
        hi[q] = pr[roff16 + j];
        lo[q] = pr[R16 + roff16 + j];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (k0 + q < splits) acc += __fadd_rn(hi[q], lo[q]);
    }
    const float v = __fmul_rn(acc, scale);
    if (transposed)
      tile[mm][j] = v;
    else
      out[static_cast<long long>(m0 + mm) * ldo + j] = v;
  }
  if (transposed) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < nm * r; idx += blockDim.x) {
      const int j = idx / nm, mm = idx - j * nm;
      out[static_cast<long long>(j) * ldo + m0 + mm] = tile[mm][j];
    }
  }
}

}  // namespace

int tokgemm_max_pairs(size_t smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(tokgemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * 256);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, tokgemm_kernel, &cfg);
  if (e != cudaSuccess || n <= 0) n = device_sm_count() / 2;
  return n;
}

int launch_tokgemm(const TokGemmMaps& maps, const TokGemmParams& p, int pairs, size_t smem_bytes,
                   cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaFuncSetAttribute(tokgemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, tokgemm_kernel, maps, p);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int launch_pieces(const float* src, long long ld, int T, int N, const TokPieceMap& pm, uint16_t* dst,
                  cudaStream_t stream) {
  if (T <= 0 || N <= 0) return WP_OK;
  if (N > 256) return WP_ERR_UNSUPPORTED;
  const long long blocks = (static_cast<long long>(T) + kPieceRows - 1) / kPieceRows;
  if (blocks > 0x7FFFFFFFLL) return WP_ERR_UNSUPPORTED;
  pieces_kernel<<<static_cast<unsigned>(blocks), N, 0, stream>>>(src, ld, T, N, pm, dst);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int launch_tok_finish(const float* part, int M, int N, int splits, int R16, int roff16, int r, int row0, int rows,
                      float scale, float* out, long long ldo, bool transposed, cudaStream_t stream) {
  if (rows <= 0 || r <= 0 || splits <= 0) return WP_OK;
  if (r > kFinMaxR) return WP_ERR_UNSUPPORTED;
  const int blocks = (rows + kFinRows - 1) / kFinRows;
  tok_finish_kernel<<<blocks, 256, 0, stream>>>(part, M, N, splits, R16, roff16, r, row0, rows, scale, out, ldo,
                                                transposed ? 1 : 0);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace wp
