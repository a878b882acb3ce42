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
// pass.  A unit of work is (128-row block, K range); K is split so that the units fill
// the machine.  Per CTA: warp 0 issues the TMA loads, warp 1 the single-CTA MMAs (two
// 64-column accumulators in tensor memory, so the epilogue of one unit overlaps the
// next), warps 2..5 write fp32 partial sums, and with a 4-bit weight warps 6..21
// dequantise the tiles in shared memory: four groups of four warps, a thread per weight
// row, each group owning the stages of every fourth step.  A 4-bit step covers two K
// blocks: every hand-off between the roles (a barrier round trip of a few hundred cycles
// on this part) then moves twice the weight.  The 4-bit codes travel in a ring of their
// own that each group refills, as soon as it has read a slot, with the codes of the step
// a ring's length ahead, so the weight stream never waits on the producer.  The second
// kernel, one block per (16 tokens, 256 output columns), sums the K splits in a fixed
// order, forms the tokens' H~ = bf16(s X A^T), adds the bias and H~ B^T in fp32 and
// rounds once.
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

// Walks the weight steps of a CTA in issue order (its weight units come before its units of
// A rows, so the walk ends at the first A unit).
struct WIter {
  int u, kb, kb1, rb;
  bool more;
};

__device__ __forceinline__ void witer_unit(const SkinnyParams& p, WIter& it) {
  it.more = false;
  if (it.u < p.units) {
    const Unit t = unit_of(p, it.u);
    it.more = !t.a_blk;
    it.kb = t.kb0;
    it.kb1 = t.kb1;
    it.rb = t.rb;
  }
}

__device__ __forceinline__ void witer_start(const SkinnyParams& p, WIter& it) {
  it.u = blockIdx.x;
  witer_unit(p, it);
}

__device__ __forceinline__ void witer_next(const SkinnyParams& p, WIter& it) {
  if (!it.more) return;
  it.kb += p.kkb;
  if (it.kb >= it.kb1) {
    it.u += gridDim.x;
    witer_unit(p, it);
  }
}

template <bool kNF4>
__global__ void __launch_bounds__(kNF4 ? kSkinnyThreadsNF4 : kSkinnyThreads, 1)
    skinny_kernel(const __grid_constant__ SkinnyMaps maps, const __grid_constant__ SkinnyParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base_addr - raw_addr);

  // A step covers kkb 64-wide K blocks (1, or 2 with a 4-bit W).  stage = [kkb W (or A)
  // tiles of 16 KiB | kkb boxes of Tp X rows].  bf16 W: all of it comes by TMA.  4-bit W:
  // the W tiles are written by the stage's dequantisation group (stage s belongs to group
  // s % 4, S is 4 or 8), and the codes travel in a ring of slots [4-bit codes, kkb x 4 KiB |
  // block scales 2 KiB] that the groups refill themselves, R weight steps ahead of the one
  // they have just read.
  const int S = p.stages;
  const int SB = p.stage_bytes;
  const int kkb = kNF4 ? p.kkb : 1;
  const int XB = p.Tp * 128;                    // one box of X rows
  const int x_off = kkb * kWTileBytes;          // X boxes within a stage
  const int CSB = kkb * kRawBytes + (p.am_tma ? kAmBytes : 0);   // one code slot
  const int R = kNF4 ? p.code_slots : 1;
  uint8_t* codes = sbase + S * SB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(codes + (kNF4 ? R * CSB : 0));
  uint64_t* full = bars;                  // [S] TMA bytes landed: X, and W (bf16) or A rows
  uint64_t* empty = bars + S;             // [S] the MMAs are done with the stage
  uint64_t* wfull = bars + 2 * S;         // [S] 4-bit: the owning group has written the tile
                                          //     (or has nothing to write) and seen `full`
  uint64_t* code_full = bars + 3 * S;     // [R] 4-bit: codes (and scales) landed
  uint64_t* acc_full = code_full + R;     // [2] accumulator ready
  uint64_t* acc_empty = acc_full + 2;     // [2] the epilogue has read it
  uint64_t* drain = acc_full + 4;         //     every MMA issued has finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* c_uses = tmem_slot + 2;       // [R] 4-bit: copies issued into each code slot

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&wfull[s], 4);            // the 4 warps of the stage's dequantisation group
    }
    if (kNF4)
      for (int c = 0; c < R; ++c) {
        mbar_init(&code_full[c], 1);
        c_uses[c] = 0;
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

  // the A rows of A block `a0`: the 16-row pieces of the adapters inside it (rows of the
  // block that no adapter covers are never read by the epilogue)
  auto a_block_bytes = [&](int a0) {
    uint32_t bytes = 0;
    for (int i = 0; i < p.n_ad; ++i) {
      const int lo = max(a0, p.a_off[i]), hi = min(a0 + 128, p.a_off[i + 1]);
      if (hi > lo) bytes += static_cast<uint32_t>(hi - lo) * 128;
    }
    return bytes;
  };
  auto load_a_block = [&](uint8_t* dst, int a0, int kb, uint64_t* bar, uint64_t hint) {
    for (int i = 0; i < p.n_ad; ++i) {
      const int lo = max(a0, p.a_off[i]), hi = min(a0 + 128, p.a_off[i + 1]);
      for (int r0 = lo; r0 < hi; r0 += 16)
        tma_load_2d_hint(dst + (r0 - a0) * 128, &maps.a[i], kb * kBK, r0 - p.a_off[i], bar, hint);
    }
  };
  // bounded wait for the copies of a barrier's last armed phase (after an abort)
  auto settle = [](uint64_t* bar, uint32_t uses) {
    if (uses == 0) return;
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(a, (uses - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
    }
  };

  // the codes (and block scales) of weight step (rb, kb) into code slot c
  // (one box of kkb K blocks; the scale box of 4 blocks holds both of a 2-block step, which
  // starts at an even block)
  auto load_codes = [&](int c, int rb, int kb, uint64_t hint) {
    uint8_t* cs = codes + c * CSB;
    ++c_uses[c];
    mbar_arrive_expect_tx(&code_full[c], kkb * kRawBytes + (p.am_tma ? kAmBytes : 0));
    tma_load_2d_hint(cs, &maps.wq, kb * (kBK / 2), rb * 128, &code_full[c], hint);
    if (p.am_tma) tma_load_2d_hint(cs + kkb * kRawBytes, &maps.am, kb & ~3, rb * 128, &code_full[c], hint);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t keep = l2_evict_last();      // X and the A rows: read by every CTA
      const uint64_t once = l2_evict_first();     // the weight: read once
      bool ok = true;
      if (kNF4) {
        // the first R weight steps' codes; the dequantisation groups issue the rest
        WIter c;
        witer_start(p, c);
        for (int i = 0; i < R && c.more; ++i) {
          load_codes(i, c.rb, c.kb, once);
          witer_next(p, c);
        }
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t n_issued = 0;                  // stages filled so far (no per-stage array: local memory)
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const Unit t = unit_of(p, u);
        for (int kb = t.kb0; kb < t.kb1; kb += kkb) {
          if (!(ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, tmo, status))) break;
          uint8_t* st = sbase + stage * SB;
          const int a0 = (t.rb - p.nbW) * 128;
          // K blocks past K (the second block of a last 2-block step) read as zeros
          const uint32_t tx = static_cast<uint32_t>(kkb) *
                              (static_cast<uint32_t>(XB) +
                               (t.a_blk ? a_block_bytes(a0) : kNF4 ? 0u : static_cast<uint32_t>(kWTileBytes)));
          mbar_arrive_expect_tx(&full[stage], tx);
          for (int h = 0; h < kkb; ++h) {
            tma_load_2d_hint(st + x_off + h * XB, &maps.x, (kb + h) * kBK, 0, &full[stage], keep);
            if (t.a_blk) load_a_block(st + h * kWTileBytes, a0, kb + h, &full[stage], keep);
            else if (!kNF4) tma_load_2d_hint(st + h * kWTileBytes, &maps.w, (kb + h) * kBK, t.rb * 128, &full[stage], once);
          }
          ++n_issued;
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok)
        for (int s = 0; s < S; ++s)
          settle(&full[s], n_issued / S + (static_cast<uint32_t>(s) < n_issued % S ? 1u : 0u));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // waits for the stage's TMA bytes and, with a 4-bit W, for its dequantisation group
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int count = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(p.Tp));
      const uint32_t stage_base = smem_u32(sbase);
      // This thread's instructions between two MMAs are on the tensor core's critical path
      // (a 128 x Tp x 16 MMA is short): descriptors are the constant fields and the start
      // address (16-byte units) of stage 0's slots plus the stage's offset.
      const uint32_t u_w = stage_base >> 4, u_x = (stage_base + static_cast<uint32_t>(x_off)) >> 4;
      const uint32_t w_step = kWTileBytes >> 4, x_step = static_cast<uint32_t>(XB) >> 4;
      const uint32_t stage_units = static_cast<uint32_t>(SB) >> 4;
      uint32_t off = 0;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const Unit t = unit_of(p, u);
        const int b = count & 1;
        // unit `count` uses buffer count & 1, whose earlier uses number count >> 1
        if (!(ok = mbar_wait(&acc_empty[b], ((static_cast<uint32_t>(count) >> 1) & 1u) ^ 1u, abort_flag, tmo, status)))
          break;
        tc_fence_after();
        for (int kb = t.kb0; kb < t.kb1; kb += kkb) {
          if (kNF4 && !(ok = mbar_wait(&wfull[stage], phase, abort_flag, tmo, status))) break;
          if (!(ok = mbar_wait(&full[stage], phase, abort_flag, tmo, status))) break;
          tc_fence_after();
          for (int h = 0; h < kkb; ++h) {
            const uint64_t ad = kDescSw128K | (u_w + off + h * w_step);
            const uint64_t bd = kDescSw128K | (u_x + off + h * x_step);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16(tmem + b * 64, ad + 2 * kk, bd + 2 * kk, idesc, (kb > t.kb0 || h > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          off += stage_units;
          if (++stage == S) { stage = 0; phase ^= 1; off = 0; }
        }
        if (!ok) break;
        mma_commit(&acc_full[b]);
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
    int count = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      const Unit t = unit_of(p, u);
      const int b = count & 1;
      const bool ok = mbar_wait(&acc_full[b], (static_cast<uint32_t>(count) >> 1) & 1u, abort_flag, tmo, status);
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
      ++count;
    }
  } else if (kNF4) {
    // ------------------------------------------------------------ 4-bit dequantisation
    // Four groups of 128 threads; step j belongs to group j % 4, and so do all the uses of
    // its stage j % S (S is 4 or 8), so each group's waits see every phase of its stages'
    // barriers.  Thread r of a group owns row r of the step: kkb 64-element blocks.  A
    // weight step's codes sit in the ring slot of its weight-step index; once the whole
    // group has read them, the group's elected thread refills the slot with the codes of
    // the weight step R further on.  That slot's previous use is R >= S steps back, and the
    // stage wait has already seen the MMAs of every step S back, so the parity wait on the
    // slot cannot pass on a stale phase.  Lane 0 of each warp polls and the warp follows;
    // every exit is decided by a vote of the whole group, so no warp can leave the others
    // waiting at the group's named barrier.
    const int group = (threadIdx.x - kSkinnyThreads) >> 7;
    const int r = (threadIdx.x - kSkinnyThreads) & 127;
    const uint32_t gbar = 1u + static_cast<uint32_t>(group);      // named barrier of the group
    float lv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lv[i] = p.nf4_code[i];
    const int kb64 = p.K / 64;
    const uint64_t once = l2_evict_first();
    auto wait0 = [&](uint64_t* bar, uint32_t par) -> bool {
      bool w = true;
      if (lane == 0) w = mbar_wait(bar, par, abort_flag, tmo, status);
      __syncwarp();
      return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    };
    uint32_t j = 0;                                  // steps seen
    int s = 0;                                       // the next step's stage and its use parity
    uint32_t spar = 0;
    int cslot = 0;                                   // the next weight step's code slot and parity
    uint32_t cpar = 0;
    WIter ahead;                                     // the weight step R after the next one
    witer_start(p, ahead);
    for (int i = 0; i < R; ++i) witer_next(p, ahead);
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const Unit t = unit_of(p, u);
      const int wrow = t.rb * 128 + r;
      const bool wrow_ok = !t.a_blk && wrow < p.N;
      for (int kb = t.kb0; kb < t.kb1; kb += kkb) {
        const int st = s;
        const uint32_t st_par = spar;
        const int slot = cslot;
        const uint32_t slot_par = cpar;
        const bool mine = static_cast<int>(j & 3u) == group;
        ++j;
        if (++s == S) { s = 0; spar ^= 1u; }
        if (!t.a_blk && ++cslot == R) { cslot = 0; cpar ^= 1u; }
        if (!mine) {
          if (!t.a_blk) witer_next(p, ahead);
          continue;
        }
        bool w = wait0(&empty[st], st_par ^ 1u);
        if (!t.a_blk) w = w && wait0(&code_full[slot], slot_par);
        if (!(ok = named_bar_all(w, gbar, 128))) break;
        if (!t.a_blk) {
          const uint8_t* cs = codes + slot * CSB;
          const uint32_t tile = smem_u32(sbase + st * SB);
          for (int h = 0; h < kkb; ++h) {
            // a block past K (K blocks odd, last 2-block step) reads zero codes and scale
            const int k = kb + h;
            const float am = p.am_tma ? reinterpret_cast<const float*>(cs + kkb * kRawBytes)[r * 4 + (k & 3)]
                                      : (wrow_ok && k < kb64 ? __ldg(p.absmax + static_cast<long long>(wrow) * kb64 + k) : 0.f);
            nf4_dequant_row(cs + r * (32 * kkb), 2 * h, kkb == 2 ? (r >> 1) & 3 : (r >> 2) & 1, am, lv,
                            tile + h * kWTileBytes, r);
          }
          fence_proxy_async_smem();
          named_bar_sync(gbar, 128);                 // the slot is read and the tiles written
          if (r == 0 && ahead.more) load_codes(slot, ahead.rb, ahead.kb, once);
          witer_next(p, ahead);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&wfull[st]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // after an abort: the last copy into each code slot may still be in flight
  if (kNF4 && threadIdx.x == 0 && *abort_flag)
    for (int c = 0; c < R; ++c) settle(&code_full[c], c_uses[c]);
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
constexpr int kMaxSplits = 8;                 // partial sums loaded together per round

// sum_k p[k * stride] for k = 0 .. n - 1, added in k order from 0.  The loads go out
// kMaxSplits at a time with no condition between them (an index past the end reads the last
// split again and is not added), so they overlap instead of waiting for one another.
__device__ __forceinline__ float sum_splits(const float* p, long long stride, int n) {
  float sum = 0.f;
  for (int k0 = 0; k0 < n; k0 += kMaxSplits) {
    float v[kMaxSplits];
#pragma unroll
    for (int k = 0; k < kMaxSplits; ++k) v[k] = p[min(k0 + k, n - 1) * stride];
#pragma unroll
    for (int k = 0; k < kMaxSplits; ++k)
      if (k0 + k < n) sum += v[k];
  }
  return sum;
}

// The splits' partial sums of kNT tokens' columns, all loads of a group of splits issued
// before any is added (an index past the last token or split reads an existing entry, which
// is not added); each token's sum in split order from 0.
template <int kNT>
__device__ __forceinline__ void sum_splits_t(const float* p, long long stride, long long ldp, int n, int nt,
                                             float (&acc)[kNT]) {
  constexpr int kG = kNT >= 16 ? 4 : kMaxSplits;
  for (int k0 = 0; k0 < n; k0 += kG) {
    float v[kG][kNT];
#pragma unroll
    for (int k = 0; k < kG; ++k)
#pragma unroll
      for (int t = 0; t < kNT; ++t) v[k][t] = p[min(k0 + k, n - 1) * stride + min(t, nt - 1) * ldp];
#pragma unroll
    for (int k = 0; k < kG; ++k)
      if (k0 + k < n)
#pragma unroll
        for (int t = 0; t < kNT; ++t) acc[t] += v[k][t];
  }
}

// kNT: the tokens a block carries (the call's T when it is at most 4, 8 up to 8, else 16 per
// block row)
template <int kNT>
__global__ void __launch_bounds__(256) skinny_reduce_kernel(const SkinnyReduceParams q) {
  __shared__ __align__(16) uint16_t hs[kNT * kHCols];
  const int t0 = blockIdx.y * kNT;
  const int nt = min(kNT, q.T - t0);
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
    const float h = sum_splits(part + t * q.ldp + q.N + j, sstride, q.splits);
    float s = 0.f;
    for (int a = 0; a < q.n_ad; ++a)
      if (j >= q.ad[a].toff && j < q.ad[a].toff + q.ad[a].rank) s = q.ad[a].s;
    uint16_t hb;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(hb) : "f"(s * h));
    hs[t * q.R16 + j] = hb;
  }
  __syncthreads();
  if (n >= q.N) return;
  float acc[kNT];
#pragma unroll
  for (int t = 0; t < kNT; ++t) acc[t] = 0.f;
  if (q.has_w) sum_splits_t<kNT>(part + n, sstride, q.ldp, q.splits, nt, acc);
#pragma unroll
  for (int t = 0; t < kNT; ++t) acc[t] += bias;
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
      for (int t = 0; t < kNT; ++t) {
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
  for (int t = 0; t < kNT; ++t) {
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
  if (q.T <= 0 || q.N <= 0) return WP_OK;
  const int nt = q.T <= 4 ? q.T : (q.T <= 8 ? 8 : kReduceT);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((q.N + 255) / 256, (q.T + nt - 1) / nt);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  switch (nt) {
    case 1: e = cudaLaunchKernelEx(&cfg, skinny_reduce_kernel<1>, q); break;
    case 2: e = cudaLaunchKernelEx(&cfg, skinny_reduce_kernel<2>, q); break;
    case 3: e = cudaLaunchKernelEx(&cfg, skinny_reduce_kernel<3>, q); break;
    case 4: e = cudaLaunchKernelEx(&cfg, skinny_reduce_kernel<4>, q); break;
    case 8: e = cudaLaunchKernelEx(&cfg, skinny_reduce_kernel<8>, q); break;
    default: e = cudaLaunchKernelEx(&cfg, skinny_reduce_kernel<kReduceT>, q); break;
  }
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace wp
