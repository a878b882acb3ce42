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

// The cell tables in shared memory: the code search (next midpoints, base codes), then the
// stochastic re-encoding's level cells (next level, its index, the level before, the level
// after), kCodeCells words each.
constexpr int kCellWords = 6 * kCodeCells;
constexpr size_t kCellBytes = kCellWords * sizeof(uint32_t);
__device__ __forceinline__ void fill_cells(uint32_t* t, int c, const MergeNF4Params& p) {
  t[c] = __float_as_uint(p.cells.next_mid[c]);
  t[kCodeCells + c] = static_cast<uint32_t>(p.cells.base[c]);
  t[2 * kCodeCells + c] = __float_as_uint(p.lcells.next_l[c]);
  t[3 * kCodeCells + c] = static_cast<uint32_t>(p.lcells.base[c]);
  t[4 * kCodeCells + c] = __float_as_uint(p.lcells.prev_l[c]);
  t[5 * kCodeCells + c] = __float_as_uint(p.lcells.after_l[c]);
}

// Persistent: a CTA takes the 128-row x 64-column tiles blockIdx.x, + gridDim.x, ... (row tile
// major, so the CTAs resident at one time share B_p's rows and sweep A_p^T's), and within a
// tile the adapters in call order.  Each (tile, adapter) job has an operand stage and a
// 64-column tensor-memory buffer of its own parity, so while the four warps work on job j the
// MMAs of job j + 1 run and the copies of job j + 2 are on their way; the next tile's codes
// are read into registers a whole tile ahead.  Thread 0 issues the copies and the MMAs
// between its share of the arithmetic.  The warps never wait for one another: a warp that has
// read its lanes of a buffer arrives on the buffer's "empty" barrier, and thread 0 waits there
// before the MMAs that overwrite it.
template <bool kStoch>
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
  __shared__ uint32_t s_cells[kCellWords];        // the code search by cells, then the level cells

  const int warp = threadIdx.x >> 5;
  const int nb = p.cols / 64;                     // column blocks
  const int tiles = nb * ((p.rows + 127) / 128);
  const int ntile = blockIdx.x < tiles ? (tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  const int J = ntile * p.n;                      // this CTA's jobs
  const long long cb = static_cast<long long>(p.cols) / 64;     // blocks per row
  for (int c = threadIdx.x; c < kCodeCells; c += blockDim.x)
    fill_cells(s_cells, c, p);
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
    if (J > 0 && !(p.hold && J == 1)) issue_mma(0);   // hold: the last job's MMAs never come
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
        // (hold: the last job's MMAs never come)
        if (j + 1 < J && !(p.hold && j + 1 == J - 1) &&
            (j == 0 ||
             mbar_wait(empty + (st ^ 1), static_cast<uint32_t>((j - 1) >> 1) & 1u, abort_flag, p.timeout_ns, p.status)))
          issue_mma(j + 1);
      }
    }
    if (bad) break;
    if (row < p.rows) {
      // requantise: absmax' = max |u|, x = fl32(u / absmax'), code = the number of level
      // midpoints x exceeds; an all-zero block keeps scale 0 and level 0's code
      uint32_t cw[8];
      const long long e0 = static_cast<long long>(row) * p.cols + blk * 64;
      const float m = kStoch ? nf4_requant_block_stochastic(u, cells_addr + 8 * kCodeCells, e0, p.seed_lo, p.seed_hi, cw)
                             : nf4_requant_block(u, cells_addr, cw);
      uint4* dst = reinterpret_cast<uint4*>(p.codes + e0 / 2);
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
// compute warps and a producer warp, tiles of 128 rows x 256 columns.  Compute warp w reads
// tensor-memory lanes 32 (w % 4) on and owns column block w / 4 of the tile, a thread per row
// and block as above; one job per tile and adapter is a single 128 x 256 MMA.
//
// A CTA takes a contiguous run of groups, a group being 4 tiles side by side (128 x 1024;
// fewer at a row's end), in row-major order.  Everything moves by TMA, in as few box rows as
// the layouts allow (the copy engine's time goes by rows):
//   codes   one 128 x 128-byte box per tile (128-byte swizzle, so that the rows a warp reads
//           fall in different banks), in and out through a ring of s_c stages, loaded s_c - 3
//           tiles ahead;
//   scales  one 128 x 16-float box per group, in and out (a ring of three group buffers);
//   B_p     the 128 rows x r of every adapter once per group (K-major, 64-wide K boxes, two
//           group buffers);
//   A_p     per job, read where it lies ([r, in] row-major: the MMA's B operand MN-major), four
//           boxes of 64 columns x kbox rows (kbox = r rounded up to 16, at most 64), a ring of
//           s_a stages.
// The producer's lane 0 issues all copies and MMAs and the stores, waiting only on barriers;
// the compute warps wait for their tile's codes and scales and for each job's accumulator,
// release the accumulator buffer per warp (empty) and report the tile written (cwritten).
constexpr int kWCols = 256;                       // tile columns
constexpr int kWCodeBox = 128 * 128;              // 128 rows x 128 code bytes: 16 KiB
constexpr int kWAmBox = 128 * 64;                 // a group's scales: 128 rows x 16 floats, 8 KiB
constexpr int kWAmRing = 3;
constexpr int kWMaxSA = 4, kWMaxSC = 8;
constexpr int kWThreads = 17 * 32;

__device__ __forceinline__ void lds128w(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr));
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <bool kStoch>
__global__ void __launch_bounds__(kWThreads, 1) merge_nf4_wide_kernel(const __grid_constant__ MergeNF4Maps maps,
                                                                      const __grid_constant__ MergeNF4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sbase = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int S_a = p.s_a, S_c = p.s_c;
  uint8_t* sB = sbase;                            // [2] groups' B_p boxes, [adapter][K block] of 16 KiB
  uint8_t* sA = sB + 2 * p.b_bytes;               // [S_a] jobs' A_p boxes, [K block][column group]
  uint8_t* sC = sA + S_a * p.a_bytes;             // [S_c] tiles' codes
  uint8_t* sM = sC + S_c * kWCodeBox;             // [3] groups' scales
  uint64_t* fullA = reinterpret_cast<uint64_t*>(sM + kWAmRing * kWAmBox);   // [4] A_p stage landed
  uint64_t* done = fullA + kWMaxSA;               // [2] accumulator buffer's MMAs finished
  uint64_t* empty = done + 2;                     // [2] every compute warp has read a buffer
  uint64_t* cfull = empty + 2;                    // [8] code stage landed
  uint64_t* cwritten = cfull + kWMaxSC;           // [8] every compute warp has written its codes
  uint64_t* bfull = cwritten + kWMaxSC;           // [2] a group's B_p landed
  uint64_t* mfull = bfull + 2;                    // [3] a group's scales landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mfull + kWAmRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ uint32_t s_cells[kCellWords];        // the code search by cells, then the level cells

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nbw = p.cols / kWCols, ngc = (nbw + 3) / 4, nrt = (p.rows + 127) / 128;
  const long long G = static_cast<long long>(ngc) * nrt;
  const int g0 = static_cast<int>(G * blockIdx.x / gridDim.x), g1 = static_cast<int>(G * (blockIdx.x + 1) / gridDim.x);
  auto tiles_before = [&](int g) { return (g / ngc) * nbw + min((g % ngc) * 4, nbw); };
  const int T0 = tiles_before(g0), ntile = tiles_before(g1) - T0, J = ntile * p.n;
  // tile k of this CTA: global tile T0 + k, row-major; its group (counted from this CTA's
  // first) and its place in the group
  auto group_of = [&](int k) { const int t = T0 + k; return (t / nbw) * ngc + (t % nbw) / 4 - g0; };
  auto pos_of = [&](int k) { return ((T0 + k) % nbw) & 3; };
  auto last_in_group = [&](int k) { const int tc = (T0 + k) % nbw; return (tc & 3) == 3 || tc == nbw - 1; };

  for (int c = threadIdx.x; c < kCodeCells; c += blockDim.x)
    fill_cells(s_cells, c, p);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kWMaxSA; ++i) mbar_init(fullA + i, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(done + i, 1);
      mbar_init(empty + i, 16);
      mbar_init(bfull + i, 1);
    }
    for (int i = 0; i < kWMaxSC; ++i) {
      mbar_init(cfull + i, 1);
      mbar_init(cwritten + i, 16);
    }
    for (int i = 0; i < kWAmRing; ++i) mbar_init(mfull + i, 1);
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

  if (warp == 16) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t keep = l2_evict_last(), stream_out = l2_evict_first();
      int a_last = -1, mma_last = -1, codes_last = -1, b_last = -1, m_last = -1;   // for the drain
      auto tile_at = [&](int k, int& row0, int& tc) {
        row0 = ((T0 + k) / nbw) * 128;
        tc = (T0 + k) % nbw;
      };
      auto load_codes = [&](int k) {
        int row0, tc;
        tile_at(k, row0, tc);
        const int cs = k % S_c;
        mbar_arrive_expect_tx(cfull + cs, kWCodeBox);
        tma_load_2d_hint(sC + cs * kWCodeBox, &maps.codes, tc * 128, row0, cfull + cs, stream_out);
        codes_last = k;
      };
      auto load_scales = [&](int k) {             // the group starting at tile k
        int row0, tc;
        tile_at(k, row0, tc);
        const int gl = group_of(k), ms = gl % kWAmRing;
        mbar_arrive_expect_tx(mfull + ms, kWAmBox);
        tma_load_2d_hint(sM + ms * kWAmBox, &maps.am, (tc / 4) * 16, row0, mfull + ms, stream_out);
        m_last = gl;
      };
      auto load_b = [&](int k) {                  // every adapter's B_p rows of the group at tile k
        int row0, tc;
        tile_at(k, row0, tc);
        const int gl = group_of(k), bs = gl & 1;
        mbar_arrive_expect_tx(bfull + bs, static_cast<uint32_t>(p.b_bytes));
        for (int a = 0; a < p.n; ++a)
          for (int kb = 0; kb < p.nk[a]; ++kb)
            tma_load_2d_hint(sB + bs * p.b_bytes + (p.boff[a] + kb) * kMNBoxP, &maps.p[a], kb * kBK, row0, bfull + bs,
                             keep);
        b_last = gl;
      };
      auto load_a = [&](int j) {
        const int k = j / p.n, a = j - k * p.n, st = j % S_a, kbox = p.kbox[a];
        int row0, tc;
        tile_at(k, row0, tc);
        uint8_t* dst = sA + st * p.a_bytes;
        mbar_arrive_expect_tx(fullA + st, static_cast<uint32_t>(p.nk[a] * 4 * kbox * 128));
        for (int kb = 0; kb < p.nk[a]; ++kb)
          for (int g = 0; g < 4; ++g)
            tma_load_2d_hint(dst + (kb * 4 + g) * kbox * 128, &maps.q[a], tc * kWCols + 64 * g, kb * kbox, fullA + st,
                             keep);
        a_last = j;
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return mbar_wait(bar, parity, abort_flag, p.timeout_ns, p.status);
      };
      auto issue_mma = [&](int j) {
        const int k = j / p.n, a = j - k * p.n, st = j % S_a, tb = j & 1, gl = group_of(k);
        const uint8_t* bb = sB + (gl & 1) * p.b_bytes + p.boff[a] * kMNBoxP;
        const uint8_t* ab = sA + st * p.a_bytes;
        const int kbox = p.kbox[a];
        const uint32_t idesc = idesc_bf16_f32_bmn(128, kWCols);
        for (int kb = 0; kb < p.nk[a]; ++kb) {
          const uint64_t ad = sw128_kmajor_desc(smem_u32(bb + kb * kMNBoxP));
          for (int kk = 0; kk < kbox / 16; ++kk) {
            const uint64_t bd = sw128_mnmajor_desc_lbo(smem_u32(ab + kb * 4 * kbox * 128 + kk * 2048), kbox * 128);
            mma_bf16(tmem + static_cast<uint32_t>(kWCols * tb), ad + 2 * kk, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
        }
        mma_commit(done + tb);
        mma_last = j;
      };
      // the requantised tile k goes out once every compute warp has written it, with its
      // group's scales after the group's last tile
      auto store_tile = [&](int k) {
        const int cs = k % S_c;
        if (!wait(cwritten + cs, static_cast<uint32_t>(k / S_c) & 1u)) return;
        int row0, tc;
        tile_at(k, row0, tc);
        tma_store_2d_hint(&maps.codes, tc * 128, row0, sC + cs * kWCodeBox, stream_out);
        if (last_in_group(k))
          tma_store_2d_hint(&maps.am, (tc / 4) * 16, row0, sM + (group_of(k) % kWAmRing) * kWAmBox, stream_out);
        bulk_commit();
      };

      if (ntile > 0) {
        for (int k = 0; k < S_c - 3 && k < ntile; ++k) load_codes(k);
        load_scales(0);
        load_b(0);
        for (int j = 0; j < S_a - 1 && j < J; ++j) load_a(j);
      }
      for (int k = 0; k < ntile && !*abort_flag; ++k) {
        if (k >= 2) store_tile(k - 2);
        const int kc = k + S_c - 3;               // the codes of tile kc into the stage of tile kc - S_c
        if (kc < ntile) {
          if (kc >= S_c) bulk_wait_read_le1();
          load_codes(kc);
        }
        if (k + 1 < ntile && pos_of(k + 1) == 0) {
          // the next group: its B_p buffer's last readers are the MMAs up to job k n - 1, its
          // scale buffer's last store has been issued (three groups back)
          if (k > 0 && !wait(done + ((k * p.n - 1) & 1), static_cast<uint32_t>((k * p.n - 1) >> 1) & 1u)) break;
          load_b(k + 1);
          bulk_wait_read_0();
          load_scales(k + 1);
        }
        for (int a = 0; a < p.n && !*abort_flag; ++a) {
          const int j = k * p.n + a;
          if (j >= 2 && !wait(empty + (j & 1), static_cast<uint32_t>((j - 2) >> 1) & 1u)) break;
          if (!wait(fullA + j % S_a, static_cast<uint32_t>(j / S_a) & 1u)) break;
          if (a == 0 && (k == 0 || pos_of(k) == 0) &&
              !wait(bfull + (group_of(k) & 1), static_cast<uint32_t>(group_of(k) >> 1) & 1u))
            break;
          tc_fence_after();
          if (!(p.hold && j == J - 1)) issue_mma(j);   // hold: the last job's MMAs never come
          // the A_p stage of job j - 1 takes job j + S_a - 1 once MMA j - 1 has finished
          const int ja = j + S_a - 1;
          if (ja < J) {
            if (j >= 1 && !wait(done + ((j - 1) & 1), static_cast<uint32_t>((j - 1) >> 1) & 1u)) break;
            load_a(ja);
          }
        }
      }
      if (!*abort_flag) {
        if (ntile >= 2) store_tile(ntile - 2);
        if (ntile >= 1) store_tile(ntile - 1);
      }
      if (*abort_flag) {
        // after a timed-out wait: the copies and MMAs started finish before the exit
        const uint64_t t0 = globaltimer_ns();
        auto drain = [&](uint64_t* bar, uint32_t parity) {
          while (!mbar_try_wait(smem_u32(bar), parity) && globaltimer_ns() - t0 < 200000000ull) {
          }
        };
        for (int k = max(0, codes_last - S_c + 1); k <= codes_last; ++k)
          drain(cfull + k % S_c, static_cast<uint32_t>(k / S_c) & 1u);
        for (int j = max(0, a_last - S_a + 1); j <= a_last; ++j) drain(fullA + j % S_a, static_cast<uint32_t>(j / S_a) & 1u);
        for (int g = max(0, b_last - 1); g <= b_last; ++g) drain(bfull + (g & 1), static_cast<uint32_t>(g >> 1) & 1u);
        for (int g = max(0, m_last - kWAmRing + 1); g <= m_last; ++g)
          drain(mfull + g % kWAmRing, static_cast<uint32_t>(g / kWAmRing) & 1u);
        for (int j = max(0, mma_last - 1); j <= mma_last; ++j) drain(done + (j & 1), static_cast<uint32_t>(j >> 1) & 1u);
      }
      bulk_wait_all();                            // the stores have read shared memory and landed
    }
  } else {
    // ------------------------------------------------------------------ compute warps
    const int r = 32 * (warp & 3) + lane;         // row within the tile
    const int b = warp >> 2;                      // 64-column block within the tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t cells_addr = smem_u32(s_cells);
    for (int k = 0; k < ntile; ++k) {
      const int cs = k % S_c, gl = group_of(k);
      const uint32_t st = smem_u32(sC + cs * kWCodeBox);
      const uint32_t sw = static_cast<uint32_t>(r & 7);
      const uint32_t a0 = st + r * 128 + (((2u * b) ^ sw) << 4), a1 = st + r * 128 + (((2u * b + 1u) ^ sw) << 4);
      const uint32_t aam = smem_u32(sM + (gl % kWAmRing) * kWAmBox) + r * 64 + (4 * pos_of(k) + b) * 4;
      bool ok = true;
      if (k == 0 || pos_of(k) == 0)
        ok = mbar_wait(mfull + gl % kWAmRing, static_cast<uint32_t>(gl / kWAmRing) & 1u, abort_flag, p.timeout_ns,
                       p.status);
      ok = ok && mbar_wait(cfull + cs, static_cast<uint32_t>(k / S_c) & 1u, abort_flag, p.timeout_ns, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
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
      bool bad = false;
      for (int a = 0; a < p.n; ++a) {
        const int j = k * p.n + a, tb = j & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(done + tb, static_cast<uint32_t>(j >> 1) & 1u, abort_flag,
                                               p.timeout_ns, p.status))) {
          bad = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(kWCols * tb + 64 * b + 32 * h), v);
#pragma unroll
          for (int i = 0; i < 32; ++i) u[32 * h + i] = __fmaf_rn(__uint_as_float(v[i]), p.s[a], u[32 * h + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + tb);
      }
      if (bad) break;
      // requantise (see merge_nf4_kernel) into the stage and the group's scales, in place
      uint32_t cw[8];
      float m;
      if (kStoch) {
        const int t = T0 + k;
        const long long e0 = static_cast<long long>((t / nbw) * 128 + r) * p.cols + (t % nbw) * kWCols + 64 * b;
        m = nf4_requant_block_stochastic(u, cells_addr + 8 * kCodeCells, e0, p.seed_lo, p.seed_hi, cw);
      } else {
        m = nf4_requant_block(u, cells_addr, cw);
      }
      sts128(a0, cw[0], cw[1], cw[2], cw[3]);
      sts128(a1, cw[4], cw[5], cw[6], cw[7]);
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(aam), "f"(m) : "memory");
      fence_proxy_async_smem();                   // the TMA stores read what this thread wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(cwritten + cs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool merge_nf4_wide_plan(const int* ranks, int n, long long cols, MergeNF4Params* p) {
  if (cols % kWCols != 0 || n < 1 || n > kMaxAd) return false;
  int boff = 0, a_bytes = 0;
  for (int a = 0; a < n; ++a) {
    const int r = ranks[a];
    if (r < 1 || r > kMergeTileMaxK * kBK) return false;
    p->kbox[a] = std::min(kBK, (r + 15) / 16 * 16);
    p->nk[a] = (r + p->kbox[a] - 1) / p->kbox[a];
    p->boff[a] = boff;
    boff += p->nk[a];
    a_bytes = std::max(a_bytes, p->nk[a] * 4 * p->kbox[a] * 128);
  }
  p->b_bytes = boff * kMNBoxP;
  p->a_bytes = a_bytes;
  const long long budget = 227 * 1024 - 1024 - 256 - static_cast<long long>(kCellBytes);
  const long long fixed = 2LL * p->b_bytes + static_cast<long long>(kWAmRing) * kWAmBox;
  for (int sa = 3; sa >= 2; --sa) {
    const long long sc = std::min<long long>(kWMaxSC, (budget - fixed - sa * static_cast<long long>(a_bytes)) / kWCodeBox);
    if (sc >= 4) {                                 // the codes of tile k + s_c - 3 go in at tile k
      p->s_a = sa;
      p->s_c = static_cast<int>(sc);
      return true;
    }
  }
  return false;
}

int launch_merge_nf4(const MergeNF4Maps& maps, const MergeNF4Params& p, cudaStream_t stream) {
  if (p.rows <= 0 || p.cols <= 0 || p.n <= 0) return WP_OK;
  if (p.n > kMaxAd || p.nk_max < 1 || p.nk_max > kMergeTileMaxK || p.cols % 64 != 0) return WP_ERR_UNSUPPORTED;
  if (p.wide) {
    if (p.cols % kWCols != 0 || p.s_a < 2 || p.s_a > kWMaxSA || p.s_c < 4 || p.s_c > kWMaxSC) return WP_ERR_UNSUPPORTED;
    const size_t smem = 1024 + 2 * static_cast<size_t>(p.b_bytes) + static_cast<size_t>(p.s_a) * p.a_bytes +
                        static_cast<size_t>(p.s_c) * kWCodeBox + static_cast<size_t>(kWAmRing) * kWAmBox + 256;
    auto kernel = p.stochastic ? merge_nf4_wide_kernel<true> : merge_nf4_wide_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) {
      const long long groups = static_cast<long long>((p.cols / kWCols + 3) / 4) * ((p.rows + 127) / 128);
      const unsigned grid = static_cast<unsigned>(std::min<long long>(groups, device_sm_count()));
      kernel<<<grid, kWThreads, smem, stream>>>(maps, p);
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
  const size_t floor = 228 * 1024 / 4 - 1024 - kCellBytes - 16;
  if (smem < floor) smem = floor;
  auto kernel = p.stochastic ? merge_nf4_kernel<true> : merge_nf4_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  // the whole shared-memory carveout, so that the CTAs the padding allows do fit
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) {
    // CTAs per SM: the shared memory's count (each CTA also holds the static cell table and
    // the 1 KiB the driver reserves), at most 4; 128 threads x 128 registers allow 4 as well
    const size_t per_cta = smem + kCellBytes + 16 + 1024;
    const int per_sm = static_cast<int>(std::min<size_t>(4, 228 * 1024 / per_cta));
    const long long tiles = static_cast<long long>(p.cols / 64) * ((p.rows + 127) / 128);
    const long long cap = static_cast<long long>(device_sm_count()) * std::max(1, per_sm);
    const unsigned grid = static_cast<unsigned>(std::min(tiles, cap));
    kernel<<<grid, 128, smem, stream>>>(maps, p);
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
