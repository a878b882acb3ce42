// wp_skinny.cu -- the LoRA linear for a few tokens (T <= 64), as decode and small-batch
// serving calls it.
//
//   Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T
//
// With T this small the weight dominates the traffic (InvokeAI sidecar-patch article,
// section 五: a quantised layer keeps its 4-bit weight and runs it through the small-batch
// kernel), so the pass streams W once across every SM.  The tensor cores still do the
// products: the MMA is swapped, D^T = W X^T, with 128 weight rows as the M = 128 operand
// and the tokens, rounded up to 16, as its width; the A rows of every adapter, one
// adapter after another at 16-aligned row offsets (16-row TMA boxes straight from each
// adapter, zero past its rank), ride as extra row blocks, so X A^T comes out of the same
// pass.  A unit of work is (128-row block, K
// range); K is split so that the units fill the machine.  Per CTA: warp 0 issues the TMA
// loads, warp 1 the single-CTA MMAs (two 64-column accumulators in tensor memory, so the
// epilogue of one unit overlaps the next), warps 2..5 write fp32 partial sums, and with a
// 4-bit weight warps 6..21 dequantise the tiles in shared memory, four groups of four
// taking every fourth K step, a thread per weight row (as the large-T kernel does).  The second kernel, one block per (token, 256 output columns), sums the K splits
// in a fixed order, forms the token's H~ = bf16(s X A^T), adds the bias and H~ B^T in
// fp32 and rounds once.
#include <cuda.h>
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_nf4.cuh"
#include "wp_ptx.cuh"

namespace wp {

namespace {

constexpr int kWTileBytes = 128 * kBK * 2;   // 128 weight (or A) rows x 64 K, bf16

struct Unit {
  int rb, ks, kb0, kb1;
  bool a_blk;   // a block of packed A rows rather than weight rows
};

__device__ __forceinline__ Unit unit_of(const SkinnyParams& p, int u) {
  Unit t;
  t.rb = u / p.splits;
  t.ks = u - t.rb * p.splits;
  t.kb0 = t.ks * p.kb_per_split;
  t.kb1 = min(p.k_blocks, t.kb0 + p.kb_per_split);
  t.a_blk = t.rb >= p.nbW;
  return t;
}

template <bool kNF4>
__global__ void __launch_bounds__(kNF4 ? kSkinnyThreadsNF4 : kSkinnyThreads, 1)
    skinny_kernel(const __grid_constant__ SkinnyMaps maps, const __grid_constant__ SkinnyParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base_addr - raw_addr);

  // stage: [W (or A) rows 16 KiB | X rows 8 KiB | 4-bit codes 4 KiB | block scales 2 KiB]
  const int S = p.stages;
  const int SB = p.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + S * SB);
  uint64_t* full = bars;                  // [S] TMA bytes landed
  uint64_t* empty = bars + S;             // [S] the MMAs are done with the stage
  uint64_t* wfull = bars + 2 * S;         // [S] 4-bit W: every dequantisation warp is done
                                          //     with this use (tile written if any)
  uint64_t* acc_full = bars + 3 * S;      // [2] accumulator ready
  uint64_t* acc_empty = acc_full + 2;     // [2] the epilogue has read it
  uint64_t* drain = acc_full + 4;         //     every MMA issued has finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&wfull[s], 16);           // 16 dequantisation warps
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], 4);          // 4 epilogue warps
    mbar_init(&acc_empty[1], 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);           // two accumulators of 64 columns
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t tmo = p.timeout_ns;
  int* status = p.status;
  // the reduction kernel may be scheduled now; its dependency wait still waits for the
  // whole of this grid (partial sums included)
  if (threadIdx.x == 0) grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t keep = l2_evict_last();      // X and the A rows: read by every CTA
      const uint64_t once = l2_evict_first();     // the weight: read once
      int stage = 0;
      uint32_t phase = 0;
      int issued[kMaxStages];
      for (int s = 0; s < kMaxStages; ++s) issued[s] = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const Unit t = unit_of(p, u);
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!(ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, tmo, status))) break;
          uint8_t* st = sbase + stage * SB;
          const bool codes = kNF4 && !t.a_blk;
          // A block: the 16-row pieces of the adapters inside it (rows of the block that no
          // adapter covers are never read by the epilogue)
          const int a0 = (t.rb - p.nbW) * 128;
          uint32_t a_bytes = 0;
          if (t.a_blk)
            for (int i = 0; i < p.n_ad; ++i) {
              const int lo = max(a0, p.a_off[i]), hi = min(a0 + 128, p.a_off[i + 1]);
              if (hi > lo) a_bytes += static_cast<uint32_t>(hi - lo) * 128;
            }
          const uint32_t tx = static_cast<uint32_t>(p.Tp) * 128 +
                              (codes ? kRawBytes + (p.am_tma ? kAmBytes : 0) : t.a_blk ? a_bytes : kWTileBytes);
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_2d_hint(st + kWTileBytes, &maps.x, kb * kBK, 0, &full[stage], keep);
          if (t.a_blk) {
            for (int i = 0; i < p.n_ad; ++i) {
              const int lo = max(a0, p.a_off[i]), hi = min(a0 + 128, p.a_off[i + 1]);
              for (int r0 = lo; r0 < hi; r0 += 16)
                tma_load_2d_hint(st + (r0 - a0) * 128, &maps.a[i], kb * kBK, r0 - p.a_off[i], &full[stage], keep);
            }
          } else if (codes) {
            uint8_t* raw = st + kWTileBytes + kSkinnyXBytes;
            tma_load_2d_hint(raw, &maps.wq, kb * (kBK / 2), t.rb * 128, &full[stage], once);
            if (p.am_tma) tma_load_2d_hint(raw + kRawBytes, &maps.am, kb & ~3, t.rb * 128, &full[stage], once);
          } else {
            tma_load_2d_hint(st, &maps.w, kb * kBK, t.rb * 128, &full[stage], once);
          }
          ++issued[stage];
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // wait (bounded) for the copies in flight before the CTA exits
        for (int s = 0; s < S; ++s) {
          if (issued[s] == 0) continue;
          const uint32_t a = smem_u32(&full[s]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, static_cast<uint32_t>((issued[s] - 1) & 1)) &&
                 globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t nuse[2] = {0, 0};
      int count = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(p.Tp));
      const uint32_t stage_base = smem_u32(sbase);
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const Unit t = unit_of(p, u);
        const int b = count & 1;
        if (!(ok = mbar_wait(&acc_empty[b], (nuse[b] & 1) ^ 1, abort_flag, tmo, status))) break;
        tc_fence_after();
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!(ok = mbar_wait(&full[stage], phase, abort_flag, tmo, status))) break;
          if (kNF4 && !(ok = mbar_wait(&wfull[stage], phase, abort_flag, tmo, status))) break;
          tc_fence_after();
          const uint32_t st = stage_base + stage * SB;
          const uint64_t ad = sw128_kmajor_desc(st);
          const uint64_t bd = sw128_kmajor_desc(st + kWTileBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16(tmem + b * 64, ad + 2 * kk, bd + 2 * kk, idesc, (kb > t.kb0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit(&acc_full[b]);
        ++nuse[b];
        ++count;
      }
      // every MMA issued must finish before tensor memory is freed
      mma_commit(drain);
      const uint32_t a = smem_u32(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue (4 warps)
    // thread = one row of the block (its TMEM lane), Tp token columns
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t nuse[2] = {0, 0};
    int count = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      const Unit t = unit_of(p, u);
      const int b = count & 1;
      const bool ok = mbar_wait(&acc_full[b], nuse[b] & 1, abort_flag, tmo, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int lrow = q * 32 + lane;
      long long grow;
      bool valid;
      if (t.a_blk) {
        const int ar = (t.rb - p.nbW) * 128 + lrow;
        valid = ar < p.R16;
        grow = static_cast<long long>(p.N) + ar;
      } else {
        const int wr = t.rb * 128 + lrow;
        valid = wr < p.N;
        grow = wr;
      }
      float* dst = p.part + static_cast<long long>(t.ks) * p.T * p.ldp + grow;
      // 8 token columns per TMEM load, written as soon as they arrive
#pragma unroll 1
      for (int c = 0; c < p.Tp / 8; ++c) {
        uint32_t r8[8];
        tmem_ld8(tmem + b * 64 + lane_base + c * 8, r8);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (c * 8 + i < p.T) dst[(c * 8 + i) * p.ldp] = __uint_as_float(r8[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++nuse[b];
      ++count;
    }
  } else if (kNF4) {
    // ------------------------------------------------------------ 4-bit dequantisation
    // four groups of 128 threads take every fourth K step of the weight blocks; thread r
    // of a group owns row r of the block (one 64-element absmax block per K step).  Every
    // warp waits on every stage use and arrives on its wfull, after its tile if the use is
    // one of its group's, so that no parity wait can pass or fall behind a phase
    const int group = (threadIdx.x - kSkinnyThreads) >> 7;
    const int r = (threadIdx.x - kSkinnyThreads) & 127;
    uint32_t kc = 0;                                 // weight-block K steps seen
    float lv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lv[i] = p.nf4_code[i];
    const int kb64 = p.K / 64;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const Unit t = unit_of(p, u);
      const int wrow = t.rb * 128 + r;
      const bool wrow_ok = !t.a_blk && wrow < p.N;
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_flag, tmo, status));
        if (!ok) break;
        const bool mine = !t.a_blk && static_cast<int>(kc++ & 3u) == group;
        if (mine) {
          uint8_t* st = sbase + stage * SB;
          const uint8_t* raw = st + kWTileBytes + kSkinnyXBytes;
          const float am = p.am_tma ? reinterpret_cast<const float*>(raw + kRawBytes)[r * 4 + (kb & 3)]
                                    : (wrow_ok ? __ldg(p.absmax + static_cast<long long>(wrow) * kb64 + kb) : 0.f);
          nf4_dequant_row(raw + r * 32, am, lv, smem_u32(st), r);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&wfull[stage]);
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Sum of the K splits, H~ = bf16(s X A^T), bias and H~ B^T, one rounding.  Block
// (c, tb): output columns [256 c, 256 c + 256) of tokens [16 tb, 16 tb + 16).  It first forms
// those tokens' H~ in shared memory; each thread then finishes one column for the 16
// tokens, reading its B rows 8 ranks at a time and each H~ entry as a shared-memory
// broadcast.  Launched as a programmatic dependent of skinny_kernel: everything before the
// dependency wait overlaps the end of that kernel.
constexpr int kReduceT = 16;
constexpr int kMaxSplits = 8;                 // the host never splits K further

__global__ void __launch_bounds__(256) skinny_reduce_kernel(const SkinnyReduceParams q) {
  __shared__ __align__(16) uint16_t hs[kReduceT * kHCols];
  const int t0 = blockIdx.y * kReduceT;
  const int nt = min(kReduceT, q.T - t0);
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const long long sstride = static_cast<long long>(q.T) * q.ldp;
  const float* part = q.part + static_cast<long long>(t0) * q.ldp;
  float bias = 0.f;
  if (q.bias && n < q.N)
    bias = q.bias_f32 ? static_cast<const float*>(q.bias)[n]
                      : __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(q.bias)[n]) << 16);
  grid_dependency_wait();
#pragma unroll 4
  for (int idx = threadIdx.x; idx < nt * q.R16; idx += blockDim.x) {
    const int t = idx / q.R16;
    const int j = idx - t * q.R16;
    // the splits' loads are independent: issued together, summed in order
    float hv[kMaxSplits];
#pragma unroll
    for (int ks = 0; ks < kMaxSplits; ++ks) hv[ks] = ks < q.splits ? part[ks * sstride + t * q.ldp + q.N + j] : 0.f;
    float h = 0.f;
#pragma unroll
    for (int ks = 0; ks < kMaxSplits; ++ks) h += hv[ks];
    float s = 0.f;
    for (int a = 0; a < q.n_ad; ++a)
      if (j >= q.ad[a].toff && j < q.ad[a].toff + q.ad[a].rank) s = q.ad[a].s;
    uint16_t hb;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(hb) : "f"(s * h));
    hs[t * q.R16 + j] = hb;
  }
  __syncthreads();
  if (n >= q.N) return;
  float acc[kReduceT];
#pragma unroll
  for (int t = 0; t < kReduceT; ++t) acc[t] = 0.f;
  if (q.has_w) {
#pragma unroll
    for (int ks = 0; ks < kMaxSplits; ++ks) {
      if (ks < q.splits) {
#pragma unroll
        for (int t = 0; t < kReduceT; ++t)
          if (t < nt) acc[t] += part[ks * sstride + t * q.ldp + n];
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kReduceT; ++t) acc[t] += bias;
  const int g = n / q.out_g;
  const int col = n - g * q.out_g;
  for (int a = 0; a < q.n_ad; ++a) {
    if (q.ad[a].group != g) continue;
    const uint16_t* Brow = q.ad[a].B + static_cast<long long>(col) * q.ad[a].ldb;
    const int rank = q.ad[a].rank;
    for (int j0 = 0; j0 < rank; j0 += 8) {
      float b[8];
      if (q.ad[a].vec && j0 + 8 <= rank) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(Brow + j0));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          b[2 * k] = __uint_as_float(w[k] << 16);
          b[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          b[k] = j0 + k < rank ? __uint_as_float(static_cast<uint32_t>(Brow[j0 + k]) << 16) : 0.f;
      }
      // H~ columns past the rank are zero (s = 0 there), so whole groups of 8 are safe
#pragma unroll
      for (int t = 0; t < kReduceT; ++t) {
        if (t < nt) {
          const uint4 hv = *reinterpret_cast<const uint4*>(hs + t * q.R16 + q.ad[a].toff + j0);
          const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[t] = fmaf(__uint_as_float(hw[k] << 16), b[2 * k], acc[t]);
            acc[t] = fmaf(__uint_as_float(hw[k] & 0xffff0000u), b[2 * k + 1], acc[t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kReduceT; ++t) {
    if (t >= nt) break;
    const long long o = static_cast<long long>(t0 + t) * q.ldy + n;
    if (q.y_f32) {
      static_cast<float*>(q.Y)[o] = acc[t];
    } else {
      uint16_t yb;
      asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(yb) : "f"(acc[t]));
      static_cast<uint16_t*>(q.Y)[o] = yb;
    }
  }
}

template <bool kNF4>
int launch_impl(const SkinnyMaps& maps, const SkinnyParams& p, int grid, size_t smem, cudaStream_t stream) {
  auto kern = skinny_kernel<kNF4>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) {
    kern<<<grid, kNF4 ? kSkinnyThreadsNF4 : kSkinnyThreads, smem, stream>>>(maps, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace

int skinny_grid_ctas(size_t smem_bytes, bool nf4) {
  int n = 0;
  const cudaError_t e =
      nf4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, skinny_kernel<true>, kSkinnyThreadsNF4, smem_bytes)
          : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, skinny_kernel<false>, kSkinnyThreads, smem_bytes);
  if (e != cudaSuccess || n < 1) n = 1;
  return n * device_sm_count();
}

int launch_skinny(const SkinnyMaps& maps, const SkinnyParams& p, size_t smem_bytes, bool nf4,
                  cudaStream_t stream) {
  int grid = device_sm_count();
  if (grid > p.units) grid = p.units;
  if (grid < 1) return WP_OK;
  return nf4 ? launch_impl<true>(maps, p, grid, smem_bytes, stream)
             : launch_impl<false>(maps, p, grid, smem_bytes, stream);
}

int launch_skinny_reduce(const SkinnyReduceParams& q, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((q.N + 255) / 256, (q.T + kReduceT - 1) / kReduceT);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, skinny_reduce_kernel, q);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace wp
