// wp_merge_tile.cu -- one product pass of a LoRA merge:  Y = s (P Q^T) + R.
//
// piper-offload docs, "LoRA merge": a plain floating-point weight takes the adapter's update
// in place (an addmm_ on the weight); here P = B_p [out, r], Q = A_p^T [in, r] and R = Y = W
// (or an fp32 buffer carrying the sum of several adapters, or a 4-bit weight's W_eff).  Each
// element is fl32(fl32(s * acc) + R), acc the fp32 tensor-core sum over r.
//
// With K = r (a few hundred at most) the product is small; the pass is the weight's read and
// write.  So a CTA owns one 128 x 128 output tile and does one thing after another: the whole
// of both operand tiles by TMA (every K block under one barrier), the single-CTA MMAs into 128
// tensor-memory columns, and an epilogue of four warps, a thread per output row: the row's
// residual is pulled toward L2 while the operands land and read one 32-column slice ahead of
// its use, and the result goes straight to global memory in 16-byte stores.  The CTA's shared
// memory is padded so that at most four CTAs share an SM (their 4 x 128 tensor-memory columns
// fit the SM's 512), and the CTAs resident on an SM overlap one another's phases.
#include <cuda.h>
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_nf4.cuh"
#include "wp_ptx.cuh"

namespace wp {

namespace {

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t (&w)[4]) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(addr));
}

constexpr int kMT = 128;                          // tile rows
constexpr int kMTBox = kMT * kBK * 2;             // one 128-row x 64-K bf16 operand box: 16 KiB

// NT: tile columns (64, 128 or 256), the MMA's N and the tensor-memory columns a CTA holds
template <int NT>
__global__ void __launch_bounds__(128) merge_tile_kernel(const __grid_constant__ MergeTileMaps maps,
                                                         const __grid_constant__ MergeTileParams p) {
  constexpr int kQBox = NT * kBK * 2;             // one NT-row x 64-K box of Q
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sP = sbase;                            // [nk] boxes of P rows
  uint8_t* sQ = sbase + p.nk * kMTBox;            // [nk] boxes of Q rows
  const int esz = p.r_f32 ? 4 : 2;
  uint8_t* sR = sQ + p.nk * kQBox;                // staged: the residual tile, boxes of 128 B x 128 rows
  const int r_bytes = p.staged ? kMT * NT * esz : 0;
  uint64_t* full = reinterpret_cast<uint64_t*>(sR + r_bytes);                // operands landed
  uint64_t* done = full + 1;                      // the MMAs have finished
  uint64_t* rfull = full + 2;                     // staged: the residual tile landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int row0 = blockIdx.y * kMT, col0 = blockIdx.x * NT;
  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    mbar_init(done, 1);
    mbar_init(rfull, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    // both operand tiles, every K block (rows and K past the matrices read as zeros)
    const uint64_t keep = l2_evict_last();        // P and Q are read by a row / column of CTAs
    mbar_arrive_expect_tx(full, static_cast<uint32_t>(p.nk) * (kMTBox + kQBox));
    for (int kb = 0; kb < p.nk; ++kb) {
      tma_load_2d_hint(sP + kb * kMTBox, &maps.p, kb * kBK, row0, full, keep);
      tma_load_2d_hint(sQ + kb * kQBox, &maps.q, kb * kBK, col0, full, keep);
    }
    if (p.staged) {
      // the residual tile, read once: it lands while the MMAs run
      mbar_arrive_expect_tx(rfull, static_cast<uint32_t>(r_bytes));
      for (int b = 0; b < r_bytes / (kMT * 128); ++b)
        tma_load_2d_hint(sR + b * (kMT * 128), &maps.r, col0 + b * (128 / esz), row0, rfull, l2_evict_first());
    }
  }

  // this thread's output row; its residual heads for L2 while the operands land
  const int row = row0 + static_cast<int>(threadIdx.x);
  const bool row_ok = row < p.rows;
  const int ncol = min(NT, p.cols - col0);        // a multiple of 8
  const char* rrow = static_cast<const char*>(p.R) + (static_cast<long long>(row_ok ? row : 0) * p.ldr + col0) * esz;
  if (row_ok && !p.staged)
    for (int off = 0; off < ncol * esz; off += 128) prefetch_l2(rrow + off);

  bool issued = false;
  if (threadIdx.x == 0 && mbar_wait(full, 0, abort_flag, p.timeout_ns, p.status)) {
    tc_fence_after();
    const uint32_t idesc = idesc_bf16_f32(kMT, NT);
    for (int kb = 0; kb < p.nk; ++kb) {
      const uint64_t ad = sw128_kmajor_desc(smem_u32(sP + kb * kMTBox));
      const uint64_t bd = sw128_kmajor_desc(smem_u32(sQ + kb * kQBox));
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
    }
    mma_commit(done);
    issued = true;
  }
  // warp-uniform: the epilogue's tensor-memory loads are warp-collective
  const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, p.timeout_ns, p.status));
  tc_fence_after();
  // staged: the residual tile must have landed too (every thread waits: warp-uniform)
  const bool rok = !p.staged || __all_sync(0xffffffffu, mbar_wait(rfull, 0, abort_flag, p.timeout_ns, p.status));

  if (ok && rok && p.staged) {
    // s * acc + R in place in the residual tile: slice c of row rl is 32 elements, at byte
    // c * 32 * esz of the row, in the box of that 128-byte column block, its 16-byte units
    // stored at unit ^ (rl & 7) (the copy engine's 128-byte swizzle)
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int rl = static_cast<int>(threadIdx.x);
    const uint32_t rowbase = smem_u32(sR) + rl * 128;
#pragma unroll 1
    for (int c = 0; c < NT / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tmem + lane_base + c * 32, a);      // warp-collective: every lane, valid or not
      if (!row_ok || c * 32 >= ncol) continue;
      const int byte0 = c * 32 * esz;
      const uint32_t box = rowbase + (byte0 >> 7) * (kMT * 128);
      const int u0 = (byte0 & 127) >> 4;
      if (p.r_f32) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t addr = box + (((u0 + u) ^ (rl & 7)) << 4);
          uint32_t w[4];
          lds128(addr, w);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            w[k] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(a[4 * u + k]), p.s), __uint_as_float(w[k])));
          st_shared_v4(addr, w[0], w[1], w[2], w[3]);
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t addr = box + (((u0 + u) ^ (rl & 7)) << 4);
          uint32_t w[4];
          lds128(addr, w);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float lo = __fadd_rn(__fmul_rn(__uint_as_float(a[8 * u + 2 * k]), p.s), __uint_as_float(w[k] << 16));
            const float hi =
                __fadd_rn(__fmul_rn(__uint_as_float(a[8 * u + 2 * k + 1]), p.s), __uint_as_float(w[k] & 0xffff0000u));
            w[k] = pack_bf16x2(lo, hi);
          }
          st_shared_v4(addr, w[0], w[1], w[2], w[3]);
        }
      }
    }
  } else if (ok && !p.staged) {
    // the residual of 32-column slice c of this row into d: 4 x 16 bytes (bf16) or 8 (fp32)
    auto load_slice = [&](int c, uint4 (&d)[8]) {
      const int n = min(32, ncol - c * 32);
      const uint4* rp = reinterpret_cast<const uint4*>(rrow + c * 32 * esz);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < 2 * esz && i * (16 / esz) < n) d[i] = rp[i];
    };
    uint4 rnext[8], rcur[8];
    if (row_ok) load_slice(0, rnext);
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
    for (int c = 0; c < NT / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tmem + lane_base + c * 32, a);      // warp-collective: every lane, valid or not
      const int n = min(32, ncol - c * 32);
      if (!row_ok || n <= 0) continue;
#pragma unroll
      for (int i = 0; i < 8; ++i) rcur[i] = rnext[i];
      if (c + 1 < NT / 32 && ncol > (c + 1) * 32) load_slice(c + 1, rnext);
      float v[32];
      if (p.r_f32) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t w[4] = {rcur[i].x, rcur[i].y, rcur[i].z, rcur[i].w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            v[4 * i + k] = __fadd_rn(__fmul_rn(__uint_as_float(a[4 * i + k]), p.s), __uint_as_float(w[k]));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w[4] = {rcur[i].x, rcur[i].y, rcur[i].z, rcur[i].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * i + 2 * k] = __fadd_rn(__fmul_rn(__uint_as_float(a[8 * i + 2 * k]), p.s), __uint_as_float(w[k] << 16));
            v[8 * i + 2 * k + 1] =
                __fadd_rn(__fmul_rn(__uint_as_float(a[8 * i + 2 * k + 1]), p.s), __uint_as_float(w[k] & 0xffff0000u));
          }
        }
      }
      const long long yo = static_cast<long long>(row) * p.ldy + col0 + c * 32;
      if (p.y_f32) {
        float* y = static_cast<float*>(p.Y) + yo;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (4 * i < n) *reinterpret_cast<float4*>(y + 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      } else {
        uint16_t* y = static_cast<uint16_t*>(p.Y) + yo;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (8 * i >= n) continue;
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) w[k] = pack_bf16x2(v[8 * i + 2 * k], v[8 * i + 2 * k + 1]);
          *reinterpret_cast<uint4*>(y + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }

  fence_proxy_async_smem();                       // staged: the tile is read by the copy engine
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && p.staged && !*abort_flag) {
    // the tile leaves by TMA (rows and columns past the matrix are not written)
    const uint64_t once = l2_evict_first();
    for (int b = 0; b < r_bytes / (kMT * 128); ++b)
      tma_store_2d_hint(&maps.y, col0 + b * (128 / esz), row0, sR + b * (kMT * 128), once);
    bulk_commit();
    bulk_wait_all();
  }
  if (threadIdx.x == 0 && *abort_flag) {
    // after a timed-out wait: the copies (and MMAs) still in flight finish before the exit
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(full), 0) && globaltimer_ns() - t0 < 100000000ull) {
    }
    if (p.staged)
      while (!mbar_try_wait(smem_u32(rfull), 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    if (issued)
      while (!mbar_try_wait(smem_u32(done), 0) && globaltimer_ns() - t0 < 200000000ull) {
      }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, NT);
  }
}

template <int NT>
int launch_nt(const MergeTileMaps& maps, const MergeTileParams& p, cudaStream_t stream) {
  // shared memory padded so that at most 512 / NT CTAs share an SM (tensor memory)
  const size_t per_sm = 228 * 1024, per_cta_reserved = 1024;
  const size_t floor = per_sm / (512 / NT) - per_cta_reserved;
  size_t smem = 1024 + static_cast<size_t>(p.nk) * (kMTBox + NT * kBK * 2) +
                (p.staged ? static_cast<size_t>(kMT) * NT * (p.r_f32 ? 4 : 2) : 0) + 64;
  if (smem < floor) smem = floor;
  cudaError_t e = cudaFuncSetAttribute(merge_tile_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e == cudaSuccess) {
    const dim3 grid((p.cols + NT - 1) / NT, (p.rows + kMT - 1) / kMT);
    merge_tile_kernel<NT><<<grid, kMT, smem, stream>>>(maps, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace

namespace {

constexpr int kMNBoxP = 128 * kBK * 2;            // 128 B_p rows x 64 K: 16 KiB
constexpr int kMNBoxQ = 64 * kBK * 2;             // 64 A_p^T rows x 64 K: 8 KiB

__global__ void __launch_bounds__(128) merge_nf4_kernel(const __grid_constant__ MergeNF4Maps maps,
                                                        const __grid_constant__ MergeNF4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sP = sbase;                            // [nk_max] boxes of B_p rows
  uint8_t* sQ = sbase + p.nk_max * kMNBoxP;       // [nk_max] boxes of A_p^T rows
  uint64_t* full = reinterpret_cast<uint64_t*>(sQ + p.nk_max * kMNBoxQ);     // one phase per adapter
  uint64_t* done = full + 1;                      // one phase per adapter
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int blk = blockIdx.x;                     // the 64-column block
  const int row0 = blockIdx.y * 128, col0 = blk * 64;
  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  // this thread's block: row row0 + t, columns [col0, col0 + 64), dequantised to W_eff
  const int row = row0 + static_cast<int>(threadIdx.x);
  const bool row_ok = row < p.rows;
  const long long cb = static_cast<long long>(p.cols) / 64;        // blocks per row
  uint8_t* crow = p.codes + (static_cast<long long>(row_ok ? row : 0) * p.cols + col0) / 2;
  float u[64];
  {
    uint4 c0 = make_uint4(0, 0, 0, 0), c1 = make_uint4(0, 0, 0, 0);
    float am = 0.f;
    if (row_ok) {
      c0 = reinterpret_cast<const uint4*>(crow)[0];
      c1 = reinterpret_cast<const uint4*>(crow)[1];
      am = p.absmax[static_cast<long long>(row) * cb + blk];
    }
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    float lv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) lv[k] = p.tab.level[k];
    nf4_dequant_regs(cw, am, lv, u);
  }

  // each adapter in call order: operands by TMA, the MMAs, u = fl32(fl32(s * acc) + u).  Every
  // thread walks every adapter (the barriers below are uniform); after an abort nothing is
  // issued or read
  bool ok = true;
  uint32_t armed = 0, committed = 0;              // thread 0: phases of full / done it started
  for (int a = 0; a < p.n; ++a) {
    const uint32_t par = static_cast<uint32_t>(a & 1);
    if (threadIdx.x == 0 && !*abort_flag) {
      const uint64_t keep = l2_evict_last();
      mbar_arrive_expect_tx(full, static_cast<uint32_t>(p.nk[a]) * (kMNBoxP + kMNBoxQ));
      ++armed;
      for (int kb = 0; kb < p.nk[a]; ++kb) {
        tma_load_2d_hint(sP + kb * kMNBoxP, &maps.p[a], kb * kBK, row0, full, keep);
        tma_load_2d_hint(sQ + kb * kMNBoxQ, &maps.q[a], kb * kBK, col0, full, keep);
      }
      if (mbar_wait(full, par, abort_flag, p.timeout_ns, p.status)) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, 64);
        for (int kb = 0; kb < p.nk[a]; ++kb) {
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sP + kb * kMNBoxP));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sQ + kb * kMNBoxQ));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        mma_commit(done);
        ++committed;
      }
    }
    ok = ok && __all_sync(0xffffffffu, mbar_wait(done, par, abort_flag, p.timeout_ns, p.status));
    tc_fence_after();
    if (ok) {
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem + lane_base, r0);
      tmem_ld32(tmem + lane_base + 32, r1);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        u[i] = __fadd_rn(__fmul_rn(__uint_as_float(r0[i]), p.s[a]), u[i]);
        u[32 + i] = __fadd_rn(__fmul_rn(__uint_as_float(r1[i]), p.s[a]), u[32 + i]);
      }
    }
    // tensor memory and the operand tiles are free for the next adapter
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (ok && row_ok && !*abort_flag) {
    // requantise the block: absmax' = max |u|, x = fl32(u / absmax'), code = the number of
    // level midpoints x exceeds (an all-zero block keeps scale 0 and level 0's code)
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) m = fmaxf(m, fabsf(u[i]));
    float mid[15];
#pragma unroll
    for (int k = 0; k < 15; ++k) mid[k] = __fmul_rn(__fadd_rn(p.tab.level[k], p.tab.level[k + 1]), 0.5f);
    uint32_t cw[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint32_t c4 = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t q = 7;
        if (m > 0.f) {
          q = nf4_code_of(__fdiv_rn(u[8 * w + i], m), mid);
        }
        c4 |= q << (8 * (i >> 1) + ((i & 1) ? 0 : 4));
      }
      cw[w] = c4;
    }
    reinterpret_cast<uint4*>(crow)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    reinterpret_cast<uint4*>(crow)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    p.absmax[static_cast<long long>(row) * cb + blk] = m;
  }

  if (threadIdx.x == 0 && *abort_flag) {
    // after a timed-out wait: the last copies and MMAs started finish before the exit
    const uint64_t t0 = globaltimer_ns();
    if (armed > 0)
      while (!mbar_try_wait(smem_u32(full), (armed - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    if (committed > 0)
      while (!mbar_try_wait(smem_u32(done), (committed - 1) & 1u) && globaltimer_ns() - t0 < 200000000ull) {
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

}  // namespace

int launch_merge_nf4(const MergeNF4Maps& maps, const MergeNF4Params& p, cudaStream_t stream) {
  if (p.rows <= 0 || p.cols <= 0 || p.n <= 0) return WP_OK;
  if (p.n > kMaxAd || p.nk_max < 1 || p.nk_max > kMergeTileMaxK || p.cols % 64 != 0) return WP_ERR_UNSUPPORTED;
  size_t smem = 1024 + static_cast<size_t>(p.nk_max) * (kMNBoxP + kMNBoxQ) + 64;
  const size_t floor = 228 * 1024 / 8 - 1024;    // at most 8 CTAs of 64 TMEM columns per SM
  if (smem < floor) smem = floor;
  cudaError_t e = cudaFuncSetAttribute(merge_nf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e == cudaSuccess) {
    const dim3 grid(p.cols / 64, (p.rows + 127) / 128);
    merge_nf4_kernel<<<grid, 128, smem, stream>>>(maps, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int launch_merge_tile(const MergeTileMaps& maps, const MergeTileParams& p, cudaStream_t stream) {
  if (p.rows <= 0 || p.cols <= 0) return WP_OK;
  if (p.nk < 1 || p.nk > kMergeTileMaxK || p.cols % 8 != 0 || (p.nt != 64 && p.nt != 128 && p.nt != 256) ||
      (p.staged && (p.nt == 256 || p.r_f32 != p.y_f32)))
    return WP_ERR_UNSUPPORTED;
  return p.nt == 256 ? launch_nt<256>(maps, p, stream)
       : p.nt == 128 ? launch_nt<128>(maps, p, stream)
                     : launch_nt<64>(maps, p, stream);
}

}  // namespace wp
