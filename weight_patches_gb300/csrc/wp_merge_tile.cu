// wp_merge_tile.cu -- one product pass of a LoRA merge:  Y = s (P Q^T) + R.
//
// piper-offload docs, "LoRA merge": a plain floating-point weight takes the adapter's update
// in place (an addmm_ on the weight); here P = B_p [out, r], Q = A_p^T [in, r] and R = Y = W
// (or an fp32 buffer carrying the sum of several adapters, or a 4-bit weight's W_eff).  Each
// element is fl32(s * acc + R) (one fused multiply-add), acc the fp32 tensor-core sum over r.
//
// With K = r (a few hundred at most) the product is small; the pass is the weight's read and
// write.  So a CTA owns one 128 x 128 output tile and does one thing after another: the whole
// of both operand tiles by TMA (every K block under one barrier), the single-CTA MMAs into 128
// tensor-memory columns, and an epilogue of four warps, a thread per output row: the row's
// residual is pulled toward L2 while the operands land and read one 32-column slice ahead of
// its use, and the result goes straight to global memory in 16-byte stores.  The CTA's shared
// memory is padded so that at most four CTAs share an SM (their 4 x 128 tensor-memory columns
// fit the SM's 512), and the CTAs resident on an SM overlap one another's phases.
#include <algorithm>

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
            w[k] = __float_as_uint(__fmaf_rn(__uint_as_float(a[4 * u + k]), p.s, __uint_as_float(w[k])));
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
            const float lo = __fmaf_rn(__uint_as_float(a[8 * u + 2 * k]), p.s, __uint_as_float(w[k] << 16));
            const float hi =
                __fmaf_rn(__uint_as_float(a[8 * u + 2 * k + 1]), p.s, __uint_as_float(w[k] & 0xffff0000u));
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
            v[4 * i + k] = __fmaf_rn(__uint_as_float(a[4 * i + k]), p.s, __uint_as_float(w[k]));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w[4] = {rcur[i].x, rcur[i].y, rcur[i].z, rcur[i].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * i + 2 * k] = __fmaf_rn(__uint_as_float(a[8 * i + 2 * k]), p.s, __uint_as_float(w[k] << 16));
            v[8 * i + 2 * k + 1] =
                __fmaf_rn(__uint_as_float(a[8 * i + 2 * k + 1]), p.s, __uint_as_float(w[k] & 0xffff0000u));
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

// Persistent: a CTA takes the 128-row x 64-column tiles blockIdx.x, + gridDim.x, ... (row tile
// major, so the CTAs resident at one time share B_p's rows and sweep A_p^T's), and within a
// tile the adapters in call order.  Each (tile, adapter) job has an operand stage and a
// 64-column tensor-memory buffer of its own parity, so while the four warps work on job j the
// MMAs of job j + 1 run and the copies of job j + 2 are on their way; the next tile's codes
// are read into registers a whole tile ahead.  Thread 0 issues the copies and the MMAs
// between its share of the arithmetic.  The warps never wait for one another: a warp that has
// read its lanes of a buffer arrives on the buffer's "empty" barrier, and thread 0 waits there
// before the MMAs that overwrite it.
__global__ void __launch_bounds__(128, 4) merge_nf4_kernel(const __grid_constant__ MergeNF4Maps maps,
                                                           const __grid_constant__ MergeNF4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int stage_bytes = p.nk_max * (kMNBoxP + kMNBoxQ);       // [nk_max] B_p boxes, then A_p^T boxes
  uint64_t* full = reinterpret_cast<uint64_t*>(sbase + 2 * stage_bytes);   // [2] a stage's operands landed
  uint64_t* done = full + 2;                      // [2] a buffer's MMAs finished
  uint64_t* empty = full + 4;                     // [2] every warp has read a buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ uint32_t s_cells[2 * kCodeCells];    // the code search by cells: next midpoints, base codes

  const int warp = threadIdx.x >> 5;
  const int nb = p.cols / 64;                     // column blocks
  const int tiles = nb * ((p.rows + 127) / 128);
  const int ntile = blockIdx.x < tiles ? (tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  const int J = ntile * p.n;                      // this CTA's jobs
  const long long cb = static_cast<long long>(p.cols) / 64;     // blocks per row
  for (int c = threadIdx.x; c < kCodeCells; c += blockDim.x)
    s_cells[c] = __float_as_uint(p.cells.next_mid[c]), s_cells[kCodeCells + c] = static_cast<uint32_t>(p.cells.base[c]);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(full + i, 1);
      mbar_init(done + i, 1);
      mbar_init(empty + i, 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t cells_addr = smem_u32(s_cells);

  // thread 0's copies and MMAs; the jobs of a parity alternate on one stage and one buffer, so
  // job j waits on phase (j >> 1) & 1 of its barriers
  int tma_last0 = -1, tma_last1 = -1, mma_last0 = -1, mma_last1 = -1;   // the last job per parity
  auto issue_tma = [&](int j) {
    const int k = j / p.n, a = j - k * p.n, st = j & 1;
    const int t = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    const int row0 = (t / nb) * 128, col0 = (t % nb) * 64;
    uint8_t* sP = sbase + st * stage_bytes;
    uint8_t* sQ = sP + p.nk_max * kMNBoxP;
    const uint64_t keep = l2_evict_last();
    mbar_arrive_expect_tx(full + st, static_cast<uint32_t>(p.nk[a]) * (kMNBoxP + kMNBoxQ));
    (st ? tma_last1 : tma_last0) = j;
    for (int kb = 0; kb < p.nk[a]; ++kb) {
      tma_load_2d_hint(sP + kb * kMNBoxP, &maps.p[a], kb * kBK, row0, full + st, keep);
      tma_load_2d_hint(sQ + kb * kMNBoxQ, &maps.q[a], kb * kBK, col0, full + st, keep);
    }
  };
  auto issue_mma = [&](int j) {
    const int a = j % p.n, st = j & 1;
    if (!mbar_wait(full + st, static_cast<uint32_t>(j >> 1) & 1u, abort_flag, p.timeout_ns, p.status)) return;
    tc_fence_after();
    const uint8_t* sP = sbase + st * stage_bytes;
    const uint8_t* sQ = sP + p.nk_max * kMNBoxP;
    const uint32_t idesc = idesc_bf16_f32(128, 64);
    for (int kb = 0; kb < p.nk[a]; ++kb) {
      const uint64_t ad = sw128_kmajor_desc(smem_u32(sP + kb * kMNBoxP));
      const uint64_t bd = sw128_kmajor_desc(smem_u32(sQ + kb * kMNBoxQ));
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        mma_bf16(tmem + 64u * st, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
    }
    mma_commit(done + st);
    (st ? mma_last1 : mma_last0) = j;
  };
  if (threadIdx.x == 0) {
    if (J > 0) issue_tma(0);
    if (J > 1) issue_tma(1);
    if (J > 0) issue_mma(0);
  }

  // this thread's row of a tile: its 64-element block, 32 code bytes and a scale
  auto load_block = [&](int k, uint32_t (&cw)[8], float& am) {
    const int t = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    const int row = (t / nb) * 128 + static_cast<int>(threadIdx.x), blk = t % nb;
    if (row < p.rows) {
      const uint4* src = reinterpret_cast<const uint4*>(p.codes + (static_cast<long long>(row) * p.cols + blk * 64) / 2);
      const uint4 c0 = src[0], c1 = src[1];
      cw[0] = c0.x; cw[1] = c0.y; cw[2] = c0.z; cw[3] = c0.w;
      cw[4] = c1.x; cw[5] = c1.y; cw[6] = c1.z; cw[7] = c1.w;
      am = p.absmax[static_cast<long long>(row) * cb + blk];
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) cw[i] = 0;
      am = 0.f;
    }
  };
  uint32_t cwn[8];
  float amn = 0.f;
  if (ntile > 0) load_block(0, cwn, amn);

  bool bad = false;                               // warp-uniform
  for (int k = 0; k < ntile && !bad; ++k) {
    const int t = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    const int row = (t / nb) * 128 + static_cast<int>(threadIdx.x), blk = t % nb;
    float u[64];
    {
      uint32_t cw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) cw[i] = cwn[i];
      const float am = amn;
      if (k + 1 < ntile) load_block(k + 1, cwn, amn);
      float lv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) lv[i] = p.tab.level[i];
      nf4_dequant_regs(cw, am, lv, u);
    }
    for (int a = 0; a < p.n; ++a) {
      const int j = k * p.n + a, st = j & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(done + st, static_cast<uint32_t>(j >> 1) & 1u, abort_flag,
                                                        p.timeout_ns, p.status));
      if (!ok) {
        bad = true;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h) {               // 32 columns at a time: fewer live registers
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + 64u * st + 32u * h, r);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          u[32 * h + i] = __fmaf_rn(__uint_as_float(r[i]), p.s[a], u[32 * h + i]);
      }
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(empty + st);
      if (threadIdx.x == 0) {
        // stage st: MMA j (waited above) was its last reader; buffer st ^ 1: every warp has read
        // job j - 1 once its empty phase completes.  A failed wait raises the abort flag, which
        // every later wait sees.
        if (j + 2 < J) issue_tma(j + 2);
        if (j + 1 < J && (j == 0 || mbar_wait(empty + (st ^ 1), static_cast<uint32_t>((j - 1) >> 1) & 1u,
                                              abort_flag, p.timeout_ns, p.status)))
          issue_mma(j + 1);
      }
    }
    if (bad) break;
    if (row < p.rows) {
      // requantise: absmax' = max |u|, x = fl32(u / absmax'), code = the number of level
      // midpoints x exceeds; an all-zero block keeps scale 0 and level 0's code
      uint32_t cw[8];
      const float m = nf4_requant_block(u, cells_addr, cw);
      uint4* dst = reinterpret_cast<uint4*>(p.codes + (static_cast<long long>(row) * p.cols + blk * 64) / 2);
      dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
      p.absmax[static_cast<long long>(row) * cb + blk] = m;
    }
  }

  if (threadIdx.x == 0 && *abort_flag) {
    // after a timed-out wait: the copies and MMAs started finish before the exit
    const uint64_t t0 = globaltimer_ns();
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const int tl = st ? tma_last1 : tma_last0, ml = st ? mma_last1 : mma_last0;
      if (tl >= 0)
        while (!mbar_try_wait(smem_u32(full + st), static_cast<uint32_t>(tl >> 1) & 1u) &&
               globaltimer_ns() - t0 < 100000000ull) {
        }
      if (ml >= 0)
        while (!mbar_try_wait(smem_u32(done + st), static_cast<uint32_t>(ml >> 1) & 1u) &&
               globaltimer_ns() - t0 < 200000000ull) {
        }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// The wide form, for weights whose columns are a multiple of 256: one CTA per SM, sixteen
// warps, tiles of 128 rows x 256 columns.  Warp w reads tensor-memory lanes 32 (w % 4) on and
// owns column block w / 4 of the tile, a thread per row and block as above; one job per tile
// and adapter is a single 128 x 256 MMA.  The codes and scales move by TMA: the tile's 16 KiB
// of codes (128 B a row, 128-byte swizzle, so that the rows a warp reads fall in different
// banks) and its 2 KiB of scales (4 a row) land in one of s_c (3 or 4) shared-memory stages
// s_c - 2 tiles ahead, are requantised in place and leave by TMA stores, so that every global
// access is a whole-line transfer that no thread waits for.  Thread 0 issues the copies, the
// MMAs and the stores between its share of the arithmetic: at the top of job j the operands
// of job j + s_op and the MMAs of job j + 1, at a tile's first job the store of the tile before
// and the codes of a later tile into the stage stored a tile ago.  Operand stages s_op (1 or 2)
// and two 256-column accumulator buffers as above.
constexpr int kWCols = 256;                       // tile columns
constexpr int kWCodeBox = 128 * 128;              // 128 rows x 128 code bytes: 16 KiB
constexpr int kWAmBox = 128 * 16;                 // 128 rows x 4 scales: 2 KiB
constexpr int kWCodeStage = kWCodeBox + kWAmBox;  // 18 KiB (a multiple of 1 KiB)
constexpr int kWQBox = kWCols * kBK * 2;          // 256 A_p^T rows x 64 K: 32 KiB
constexpr int kWOpK = kMNBoxP + kWQBox;           // one K block of both operands: 48 KiB

__device__ __forceinline__ void lds128w(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr));
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__global__ void __launch_bounds__(512, 1) merge_nf4_wide_kernel(const __grid_constant__ MergeNF4Maps maps,
                                                                const __grid_constant__ MergeNF4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int op_bytes = p.nk_max * kWOpK;          // [nk_max] B_p boxes, then [nk_max] A_p^T boxes
  const int S_op = p.s_op, S_c = p.s_c;
  uint8_t* sC = sbase + S_op * op_bytes;          // [S_c] code stages: codes box, then scales box
  uint64_t* full = reinterpret_cast<uint64_t*>(sC + S_c * kWCodeStage);   // [2] operand stage landed
  uint64_t* done = full + 2;                      // [2] accumulator buffer's MMAs finished
  uint64_t* empty = full + 4;                     // [2] every warp has read an accumulator buffer
  uint64_t* cfull = full + 6;                     // [4] code stage landed
  uint64_t* cwritten = full + 10;                 // [4] every warp has written its requantised codes
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ uint32_t s_cells[2 * kCodeCells];    // the code search by cells: next midpoints, base codes

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = 32 * (warp & 3) + lane;           // row within the tile
  const int b = warp >> 2;                        // 64-column block within the tile
  const int nbw = p.cols / kWCols;
  const int tiles = nbw * ((p.rows + 127) / 128);
  const int ntile = blockIdx.x < tiles ? (tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  const int J = ntile * p.n;
  for (int c = threadIdx.x; c < kCodeCells; c += blockDim.x)
    s_cells[c] = __float_as_uint(p.cells.next_mid[c]), s_cells[kCodeCells + c] = static_cast<uint32_t>(p.cells.base[c]);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(full + i, 1);
      mbar_init(done + i, 1);
      mbar_init(empty + i, 16);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(cfull + i, 1);
      mbar_init(cwritten + i, 16);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t cells_addr = smem_u32(s_cells);

  auto tile_at = [&](int k, int& row0, int& tc) {
    const int t = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    row0 = (t / nbw) * 128;
    tc = t % nbw;
  };
  auto op_par = [&](int j) { return static_cast<uint32_t>(S_op == 2 ? (j >> 1) : j) & 1u; };
  // thread 0's issue state: how many jobs' operands, MMAs and tiles' codes it has started
  int op_issued = 0, mma_issued = 0, codes_issued = 0;
  auto issue_op = [&](int j) {
    const int k = j / p.n, a = j - k * p.n, os = S_op == 2 ? (j & 1) : 0;
    int row0, tc;
    tile_at(k, row0, tc);
    uint8_t* sP = sbase + os * op_bytes;
    uint8_t* sQ = sP + p.nk_max * kMNBoxP;
    const uint64_t keep = l2_evict_last();
    mbar_arrive_expect_tx(full + os, static_cast<uint32_t>(p.nk[a]) * kWOpK);
    for (int kb = 0; kb < p.nk[a]; ++kb) {
      tma_load_2d_hint(sP + kb * kMNBoxP, &maps.p[a], kb * kBK, row0, full + os, keep);
      tma_load_2d_hint(sQ + kb * kWQBox, &maps.q[a], kb * kBK, tc * kWCols, full + os, keep);
    }
    op_issued = j + 1;
  };
  auto issue_mma = [&](int j) {
    const int a = j % p.n, os = S_op == 2 ? (j & 1) : 0, tb = j & 1;
    if (!mbar_wait(full + os, op_par(j), abort_flag, p.timeout_ns, p.status)) return;
    tc_fence_after();
    const uint8_t* sP = sbase + os * op_bytes;
    const uint8_t* sQ = sP + p.nk_max * kMNBoxP;
    const uint32_t idesc = idesc_bf16_f32(128, kWCols);
    for (int kb = 0; kb < p.nk[a]; ++kb) {
      const uint64_t ad = sw128_kmajor_desc(smem_u32(sP + kb * kMNBoxP));
      const uint64_t bd = sw128_kmajor_desc(smem_u32(sQ + kb * kWQBox));
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        mma_bf16(tmem + static_cast<uint32_t>(kWCols * tb), ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
    }
    mma_commit(done + tb);
    mma_issued = j + 1;
  };
  const uint64_t stream_out = l2_evict_first();
  auto issue_codes = [&](int k) {
    const int cs = k % S_c;
    int row0, tc;
    tile_at(k, row0, tc);
    uint8_t* st = sC + cs * kWCodeStage;
    mbar_arrive_expect_tx(cfull + cs, kWCodeStage);
    tma_load_2d_hint(st, &maps.codes, tc * 128, row0, cfull + cs, stream_out);
    tma_load_2d_hint(st + kWCodeBox, &maps.am, tc * 4, row0, cfull + cs, stream_out);
    codes_issued = k + 1;
  };
  // the requantised tile k goes out once every warp has written it
  auto store_tile = [&](int k) {
    const int cs = k % S_c;
    if (!mbar_wait(cwritten + cs, static_cast<uint32_t>(k / S_c) & 1u, abort_flag, p.timeout_ns, p.status)) return;
    int row0, tc;
    tile_at(k, row0, tc);
    const uint8_t* st = sC + cs * kWCodeStage;
    tma_store_2d_hint(&maps.codes, tc * 128, row0, st, stream_out);
    tma_store_2d_hint(&maps.am, tc * 4, row0, st + kWCodeBox, stream_out);
    bulk_commit();
  };
  if (threadIdx.x == 0) {
    for (int k = 0; k < S_c && k < ntile; ++k) issue_codes(k);
    for (int j = 0; j < S_op && j < J; ++j) issue_op(j);
    if (J > 0) issue_mma(0);
  }

  bool bad = false;                               // warp-uniform
  for (int k = 0; k < ntile && !bad; ++k) {
    const int cs = k % S_c;
    const uint32_t st = smem_u32(sC + cs * kWCodeStage);
    const uint32_t sw = static_cast<uint32_t>(r & 7);
    const uint32_t a0 = st + r * 128 + (((2u * b) ^ sw) << 4), a1 = st + r * 128 + (((2u * b + 1u) ^ sw) << 4);
    const uint32_t aam = st + kWCodeBox + r * 16 + 4 * b;
    if (!__all_sync(0xffffffffu, mbar_wait(cfull + cs, static_cast<uint32_t>(k / S_c) & 1u, abort_flag,
                                           p.timeout_ns, p.status))) {
      bad = true;
      break;
    }
    float u[64];
    {
      uint32_t cw[8];
      lds128w(a0, cw[0], cw[1], cw[2], cw[3]);
      lds128w(a1, cw[4], cw[5], cw[6], cw[7]);
      float am;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(am) : "r"(aam));
      float lv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) lv[i] = p.tab.level[i];
      nf4_dequant_regs(cw, am, lv, u);
    }
    for (int a = 0; a < p.n; ++a) {
      const int j = k * p.n + a, tb = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(done + tb, static_cast<uint32_t>(j >> 1) & 1u, abort_flag,
                                             p.timeout_ns, p.status))) {
        bad = true;
        break;
      }
      tc_fence_after();
      if (threadIdx.x == 0) {
        // operand stage of job j: MMA j (waited above) was its last reader; accumulator
        // buffer tb ^ 1: free once every warp has read job j - 1.  A failed wait raises the
        // abort flag, which every later wait sees.
        if (j + S_op < J) issue_op(j + S_op);
        if (j + 1 < J && (j == 0 || mbar_wait(empty + (tb ^ 1), static_cast<uint32_t>((j - 1) >> 1) & 1u,
                                              abort_flag, p.timeout_ns, p.status)))
          issue_mma(j + 1);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(kWCols * tb + 64 * b + 32 * h), v);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          u[32 * h + i] = __fmaf_rn(__uint_as_float(v[i]), p.s[a], u[32 * h + i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + tb);
      if (threadIdx.x == 0 && a == 0 && !*abort_flag) {
        // the stage of tile k - 2 (stored a tile ago) takes the codes of tile k - 2 + S_c;
        // the requantised tile k - 1 goes out
        if (k >= 2 && k - 2 + S_c < ntile) {
          bulk_wait_read_0();
          issue_codes(k - 2 + S_c);
        }
        if (k >= 1) store_tile(k - 1);
      }
    }
    if (bad) break;
    // requantise (see merge_nf4_kernel) into the stage, in place
    uint32_t cw[8];
    const float m = nf4_requant_block(u, cells_addr, cw);
    sts128(a0, cw[0], cw[1], cw[2], cw[3]);
    sts128(a1, cw[4], cw[5], cw[6], cw[7]);
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(aam), "f"(m) : "memory");
    fence_proxy_async_smem();                     // the TMA store reads what this thread wrote
    __syncwarp();
    if (lane == 0) mbar_arrive(cwritten + cs);
  }

  if (threadIdx.x == 0) {
    if (!bad && !*abort_flag && ntile > 0) store_tile(ntile - 1);
    if (*abort_flag) {
      // after a timed-out wait: the copies and MMAs started finish before the exit
      const uint64_t t0 = globaltimer_ns();
      for (int k = codes_issued - S_c; k < codes_issued; ++k)
        if (k >= 0)
          while (!mbar_try_wait(smem_u32(cfull + k % S_c), static_cast<uint32_t>(k / S_c) & 1u) &&
                 globaltimer_ns() - t0 < 100000000ull) {
          }
      for (int j = op_issued - S_op; j < op_issued; ++j)
        if (j >= 0)
          while (!mbar_try_wait(smem_u32(full + (S_op == 2 ? (j & 1) : 0)), op_par(j)) &&
                 globaltimer_ns() - t0 < 150000000ull) {
          }
      for (int j = mma_issued - 2; j < mma_issued; ++j)
        if (j >= 0)
          while (!mbar_try_wait(smem_u32(done + (j & 1)), static_cast<uint32_t>(j >> 1) & 1u) &&
                 globaltimer_ns() - t0 < 200000000ull) {
          }
    }
    bulk_wait_all();                              // the stores have read shared memory and landed
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool merge_nf4_wide_plan(int nk_max, long long cols, int* s_op, int* s_c) {
  if (cols % kWCols != 0 || nk_max < 1 || nk_max > kMergeTileMaxK) return false;
  const long long budget = 227 * 1024 - 1024 - 128 - static_cast<long long>(kCodeCells) * 2 * sizeof(uint32_t);
  const long long op = static_cast<long long>(nk_max) * kWOpK;
  const int so = 2 * op + 2 * kWCodeStage <= budget ? 2 : 1;
  const long long sc = std::min<long long>(4, (budget - so * op) / kWCodeStage);
  if (sc < 3) return false;                      // the codes of tile k + s_c - 2 leave at tile k
  *s_op = so;
  *s_c = static_cast<int>(sc);
  return true;
}

int launch_merge_nf4(const MergeNF4Maps& maps, const MergeNF4Params& p, cudaStream_t stream) {
  if (p.rows <= 0 || p.cols <= 0 || p.n <= 0) return WP_OK;
  if (p.n > kMaxAd || p.nk_max < 1 || p.nk_max > kMergeTileMaxK || p.cols % 64 != 0) return WP_ERR_UNSUPPORTED;
  if (p.wide) {
    if (p.cols % kWCols != 0 || p.s_op < 1 || p.s_op > 2 || p.s_c < 3 || p.s_c > 4) return WP_ERR_UNSUPPORTED;
    const size_t smem = 1024 + static_cast<size_t>(p.s_op) * p.nk_max * kWOpK +
                        static_cast<size_t>(p.s_c) * kWCodeStage + 128;
    cudaError_t e = cudaFuncSetAttribute(merge_nf4_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess) {
      const long long tiles = static_cast<long long>(p.cols / kWCols) * ((p.rows + 127) / 128);
      const unsigned grid = static_cast<unsigned>(std::min<long long>(tiles, device_sm_count()));
      merge_nf4_wide_kernel<<<grid, 512, smem, stream>>>(maps, p);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
      set_last_cuda_error(e);
      return WP_ERR_CUDA;
    }
    return WP_OK;
  }
  size_t smem = 1024 + 2 * static_cast<size_t>(p.nk_max) * (kMNBoxP + kMNBoxQ) + 64;
  // at most 4 CTAs per SM: their 4 x 128 tensor-memory columns fill the SM's 512, and a fifth
  // CTA's allocation would wait for a persistent CTA to leave
  const size_t floor = 228 * 1024 / 4 - 1024 - kCodeCells * 2 * sizeof(uint32_t) - 16;
  if (smem < floor) smem = floor;
  cudaError_t e = cudaFuncSetAttribute(merge_nf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  // the whole shared-memory carveout, so that the CTAs the padding allows do fit
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(merge_nf4_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) {
    // CTAs per SM: the shared memory's count (each CTA also holds the static cell table and
    // the 1 KiB the driver reserves), at most 4; 128 threads x 128 registers allow 4 as well
    const size_t per_cta = smem + kCodeCells * 2 * sizeof(uint32_t) + 16 + 1024;
    const int per_sm = static_cast<int>(std::min<size_t>(4, 228 * 1024 / per_cta));
    const long long tiles = static_cast<long long>(p.cols / 64) * ((p.rows + 127) / 128);
    const long long cap = static_cast<long long>(device_sm_count()) * std::max(1, per_sm);
    const unsigned grid = static_cast<unsigned>(std::min(tiles, cap));
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
