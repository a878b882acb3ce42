// wp_tc_fwd.cu -- the fused dynamic-LoRA linear on the sm_103a tensor cores.
//
//   Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T        (per column group)
//
// sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM",
// Modifications: the combined scale multiplies the rank-wide intermediate X A^T, the
// second low-rank GEMM accumulates straight onto the base output so the [T, out]
// delta never exists, the bias belongs to the base GEMM's epilogue, stacked q/k/v
// (gate/up) adapters take one update per column group, and an FP32 adapter keeps its
// FP32 GEMMs and is added once.  Unsloth fast_lora walkthrough, section 3 (matmul_lora):
// a 4-bit base weight is dequantised into the matmul.  Here all of it happens inside one
// persistent kernel:
//
//   * a CTA pair (cluster of 2) computes 256 x 256 output tiles with tcgen05.mma
//     cta_group::2: each CTA stages its own 128 X rows and half of the weight tile, so
//     every SM receives 32 KiB of operands per 64-deep K step;
//   * output tiles are dealt round-robin to the pairs, so the pairs busy at any moment
//     share a few 256-row blocks of X and sweep W together (both stay in L2); per row
//     block m, a rank item computes X_m A^T for every adapter at once (one MMA of
//     N = total rank per K step), one or two rounds of tiles before the tiles of m;
//   * the rank item's epilogue scales X A^T by the runtime s_p, rounds it once to bf16
//     (H~) and writes it to a small [T, total rank] buffer, then releases a flag for row
//     block m; every tile of m waits for that flag before its second contraction
//     H~ B_tile^T (K = r), which TMA feeds like extra K steps and which accumulates onto
//     the base tile in tensor memory, so the [T, out] delta never leaves the SM;
//   * an FP32 adapter rides on the same path as bf16 pieces (A = a1 + a2 + a3, the same
//     for B and for s X A^T), keeping every product above 2^-24 of the leading one;
//   * two accumulator buffers (2 x 256 TMEM columns) let the epilogue of item n overlap
//     the MMAs of item n+1; the tile epilogue adds the bias (and, for FP32 adapters too
//     wide for the pieces, sum_j (s X A32^T)[t, j] B32[o, j] by FFMA) before the single
//     rounding and writes bf16 or fp32 rows through TMA bulk stores;
//   * with a 4-bit NormalFloat base weight, TMA brings the packed codes (32 bytes per row
//     per K step) and eight dequantisation warps per CTA turn them into the bf16 weight
//     tile in shared memory -- bf16(fl32(level[q]) * absmax) through a per-row, per-block
//     16-entry table and register byte permutes -- so no bf16 copy of W ever exists.
//
// Warp roles per CTA: warp 0 issues TMA loads (both CTAs), warp 1 allocates tensor
// memory (both CTAs) and issues the pair MMAs (leader CTA only), warps 2..5 are the
// epilogue (one token row per thread), warps 6..13 dequantise (4-bit weights only).
// Operands are K-major bf16 in the 128-byte swizzle layout.  Every wait (mbarrier or
// flag) is bounded (wall clock); on expiry the CTA records WP_ERR_TIMEOUT, waits for its
// own copies in flight, frees tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "wp_internal.h"
#include "wp_nf4.cuh"
#include "wp_ptx.cuh"

namespace wp {

static __device__ int g_tc_status;

namespace {

struct Tile {
  int m, g, j;
};

// Tile L in (row block, column group, column tile) order.
__device__ __forceinline__ Tile decode_tile(const TcParams& p, int L) {
  Tile t;
  const int mg = L / p.nt_g;
  t.j = L - mg * p.nt_g;
  t.m = mg / p.G;
  t.g = mg - t.m * p.G;
  return t;
}

// Work items of one pair.  Output tiles are dealt round-robin: round k of pair q is tile
// q + k * npairs.  The rank item of row block m belongs to pair (m + total_tiles) mod npairs
// (so the pairs with one tile fewer take rank items first) and runs at the start of that
// pair's round r(m) - rlead, where r(m) = floor(m * tpb / npairs) is the first round that
// can hold a tile of m (or as soon as the pair has no tiles left); with rank_first a pair's
// first rank item runs before its first tile.
// A tile of round k waits only for rank items of rounds < k, and every pair walks its
// items in order, so the schedule cannot deadlock while all pairs are resident.
struct Item {
  bool rank;   // rank item (X_m A^T of the adapters of one rank pass) rather than an output tile
  int m;       // row block
  int q;       // rank pass (rank items)
  Tile t;      // the tile (output items)
};

// Rank items are numbered i = m * npass + q (row block m, pass q); item i belongs to pair
// (i + total_tiles) mod npairs.  The walk is incremental: the next tile is the current one
// stepped by npairs in (row block, group, column tile) digits, and the round at which the
// next rank item is due is formed once per rank item, so that the threads on the tensor
// core's critical path divide nothing per item.
struct ItemIter {
  int k;        // tile rounds handed out so far
  int pos;      // position of the next tile: pair + k * npairs
  Tile t;       // the tile at pos (while pos < total_tiles)
  int m_next;   // next rank item this pair owns
  int due;      // the round at whose start item m_next runs
};

__device__ __forceinline__ int rank_item_due(const TcParams& p, int i, int npairs) {
  // rank_first: every pair opens with its first rank item.  The first round's tiles need
  // the H~ of the first row blocks by the end of their K loops, and a handful of pairs
  // computing those alone (from cold memory, like everyone else) finish well after that;
  // the host asks for it where those items' X rows stay in L2 until their tiles come.
  if (p.rank_first && i < npairs) return 0;
  const int m = p.npass == 1 ? i : i / p.npass;
  // (m >> m_shift) * tpb <= total_tiles < 2^31
  const uint32_t first = static_cast<uint32_t>((m >> p.m_shift) * p.G * p.nt_g) / static_cast<uint32_t>(npairs);
  return static_cast<int>(first) - p.rlead;
}

__device__ __forceinline__ ItemIter item_iter_begin(const TcParams& p, int pair, int npairs) {
  ItemIter s;
  s.k = 0;
  s.pos = pair;
  s.t = pair < p.total_tiles ? decode_tile(p, pair) : Tile{0, 0, 0};
  s.m_next = ((pair - p.total_tiles) % npairs + npairs) % npairs;
  s.due = p.n_ad > 0 ? rank_item_due(p, s.m_next, npairs) : 0;
  return s;
}

__device__ __forceinline__ bool next_item(ItemIter& s, const TcParams& p, int pair, int npairs,
                                          Item& it) {
  (void)pair;
  const int n_rank = p.r_blocks * p.npass;
  if (p.n_ad > 0 && s.m_next < n_rank && (s.due <= s.k || s.pos >= p.total_tiles)) {
    it.rank = true;
    it.m = p.npass == 1 ? s.m_next : s.m_next / p.npass;
    it.q = s.m_next - it.m * p.npass;
    it.t = Tile{0, 0, 0};
    s.m_next += npairs;
    if (s.m_next < n_rank) s.due = rank_item_due(p, s.m_next, npairs);
    return true;
  }
  if (s.pos >= p.total_tiles) return false;
  it.rank = false;
  it.q = 0;
  it.t = s.t;
  it.m = s.t.m;
  ++s.k;
  s.pos += npairs;
  // npairs = (step_m * G + step_g) * nt_g + step_j, with step_j < nt_g and step_g < G
  s.t.j += p.step_j;
  const int cj = s.t.j >= p.nt_g ? 1 : 0;
  s.t.j -= cj * p.nt_g;
  s.t.g += p.step_g + cj;
  const int cg = s.t.g >= p.G ? 1 : 0;
  s.t.g -= cg * p.G;
  s.t.m += p.step_m + cg;
  return true;
}

__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

constexpr uint16_t kBothCtas = 0x3;

// First weight row of this CTA's half of tile t: 128 consecutive rows of the tile's column
// group, or, for the SwiGLU front half, the tile's 128 gate rows (CTA 0) or up rows (CTA 1)
__device__ __forceinline__ int weight_row(const TcParams& p, const Tile& t, uint32_t cta) {
  return p.swiglu ? (cta ? p.out_g : 0) + t.j * 128 : t.g * p.out_g + t.j * kBN + static_cast<int>(cta) * 128;
}

__device__ __forceinline__ float bias_at(const TcParams& p, int col) {
  return p.bias_f32 ? static_cast<const float*>(p.bias)[col]
                    : bf16_to_f32(static_cast<const uint16_t*>(p.bias)[col]);
}

}  // namespace

// kF32: the epilogue also adds FP32 adapters by FFMA (those too wide to ride as bf16
// pieces); a separate instantiation so that the common kernels do not carry its registers.
template <bool kNF4, bool kF32>
__global__ void __launch_bounds__(kNF4 ? kTcThreadsNF4 : kTcThreads, 1)
    tc_fused_fwd_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
  constexpr int kEpiWarp0 = kNF4 ? 4 : 2;              // first epilogue warp
  constexpr int kEpiWarps = kNF4 ? 8 : 4;              // 4-bit W: one warpgroup per M half
  constexpr int kDeqWarp0 = kEpiWarp0 + kEpiWarps;     // 4-bit W: 12 dequantisation warps
  // token rows per pair tile: kMH halves of 256 rows, each with its own accumulator; a
  // 4-bit W's stage holds both halves' X rows ahead of the weight slot
  constexpr int kMH = kNF4 ? kMHalvesNF4 : 1;
  constexpr int kXBytes = kMH * kATileBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base_addr - raw_addr);

  // Stage s: [X rows (or H~ rows) 16 KiB | W half (or B) 16 KiB]; with a 4-bit W it also
  // holds [codes 4 KiB | block scales 2 KiB] and its W half is the dequantised tile.
  const int S = p.stages;
  const int SB = p.stage_bytes;
  const int R = kNF4 ? p.code_slots : 1;                // 4-bit W: codes ring slots
  uint8_t* codes = sbase + S * SB;                      // [R] codes | block scales
  uint8_t* stg = codes + (kNF4 ? R * kCodeSlotBytes : 0);   // 2 output staging buffers
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + 2 * kStgBytes);
  uint64_t* full = bars;                  // [S]  leader: TMA bytes of both CTAs landed
  uint64_t* empty = bars + S;             // [S]  both: the pair MMAs consumed the stage
  uint64_t* acc_full = bars + 2 * S;      // [2]  both: accumulator buffer ready
  uint64_t* acc_empty = acc_full + 2;     // [2]  leader: both epilogues drained it
  uint64_t* drain = acc_full + 4;         //      leader: every MMA issued has finished
  uint64_t* wfull = acc_full + 5;         // [S]  4-bit W, leader: every dequantisation warp of both
                                          //      CTAs is done with this use (tile written if any)
  uint64_t* code_full = wfull + S;        // [R]  4-bit W, local: a codes slot landed
  uint64_t* code_empty = code_full + R;   // [R]  4-bit W, local: its dequantisation group is done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(code_empty + R);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta = cluster_ctarank();
  const bool leader = cta == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&wfull[s], 24);           // 12 dequantisation warps x 2 CTAs
    }
    for (int s = 0; s < R; ++s) {
      mbar_init(&code_full[s], 1);
      mbar_init(&code_empty[s], 4);       // the 4 warps of one dequantisation group
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], 2 * kEpiWarps);   // every epilogue warp of both CTAs
    mbar_init(&acc_empty[1], 2 * kEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.x);
    if (p.has_base) tma_prefetch_desc(kNF4 ? &maps.wq : &maps.w);
    if (p.n_ad > 0) {
      tma_prefetch_desc(&maps.hq);
      tma_prefetch_desc(&maps.ap);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                          // peer barriers initialised before remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // 4-bit W: 24 warps launched at 80 registers (768 x 80 = 61440 in all); the warpgroups
  // re-balance that exact total: TMA/MMA 128 x 56, epilogue 256 x 104, dequantisation
  // 384 x 72 (each warpgroup runs one setmaxnreg at the top of its role branch)

  // Pair `pair` takes items pair, pair + npairs, pair + 2 npairs, ...
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const uint64_t tmo = p.timeout_ns;
  int* status = &g_tc_status;

  if (warp < kEpiWarp0) {
  if (kNF4) regs_dec<56>();                           // warpgroup 0: TMA, MMA, 2 idle warps
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint64_t keep = l2_evict_last();   // W, A, B and H~ are re-read by many tiles
      int stage = 0;
      uint32_t phase = 0;
      uint32_t n_issued = 0;                  // stages claimed and filled so far
      bool ok = true;
      // Claim the next stage once the MMAs have released it; the leader's full barrier
      // expects `tx` bytes from both CTAs.  (The leader's barrier address as both CTAs see
      // it is formed once: the claim sits between an MMA's release and the next loads.)
      const uint32_t full_l0 = mapa_shared(smem_u32(&full[0]), 0);
      auto claim = [&](uint32_t tx, uint8_t*& st, uint32_t& fb) -> bool {
        if (!mbar_wait_cluster(&empty[stage], phase ^ 1, abort_flag, tmo, status)) return false;
        st = sbase + stage * SB;
        fb = full_l0 + static_cast<uint32_t>(stage) * 8u;
        if (leader) mbar_arrive_expect_tx(&full[stage], tx);
        return true;
      };
      auto advance = [&]() {
        ++n_issued;
        if (++stage == S) { stage = 0; phase ^= 1; }
      };
      const uint32_t rank_tx = static_cast<uint32_t>(p.htot) * 128;   // packed A rows, both CTAs
      // 4-bit W: this CTA's codes and block scales of every base K step, in order, run
      // through their own ring up to R - 1 steps ahead of the stages (a second walk over the
      // same items), so that the dequantisation of a step waits only for its weight slot
      ItemIter citer = item_iter_begin(p, pair, npairs);
      Item cit;
      int c_kb = p.k_blocks, c_wrow = 0;
      uint32_t c_issued = 0;
      bool c_more = kNF4;
      auto issue_codes = [&]() -> bool {
        while (c_kb == p.k_blocks) {
          if (!next_item(citer, p, pair, npairs, cit)) { c_more = false; return true; }
          if (!cit.rank) {
            c_kb = 0;
            c_wrow = weight_row(p, cit.t, cta);
          }
        }
        const uint32_t slot = c_issued % static_cast<uint32_t>(R);
        // free once the group that dequantised the slot's previous step is done with it
        if (!mbar_wait(&code_empty[slot], ((c_issued / R) & 1u) ^ 1u, abort_flag, tmo, status)) return false;
        uint8_t* cs = codes + slot * kCodeSlotBytes;
        if (p.w_mn) {
          // W stored [in, out]: 64 rows of the step's K range x this CTA's 128 output columns
          // (64 bytes), and their block scales (a 16-byte box of four blocks holding both)
          mbar_arrive_expect_tx(&code_full[slot], kRawBytes + (p.am_tma ? kAmBytesMN : 0));
          tma_load_2d_hint(cs, &maps.wq, c_wrow / 2, c_kb * kBK, &code_full[slot], keep);
          if (p.am_tma)
            tma_load_2d_hint(cs + kRawBytes, &maps.am, (c_wrow / 64) & ~3, c_kb * kBK, &code_full[slot], keep);
        } else {
          mbar_arrive_expect_tx(&code_full[slot], kRawBytes + (p.am_tma ? kAmBytes : 0));
          tma_load_2d_hint(cs, &maps.wq, c_kb * (kBK / 2), c_wrow, &code_full[slot], keep);
          // the block scales of this K step and the next three (16-byte boxes)
          if (p.am_tma) tma_load_2d_hint(cs + kRawBytes, &maps.am, c_kb & ~3, c_wrow, &code_full[slot], keep);
        }
        ++c_kb;
        ++c_issued;
        return true;
      };
      for (int i = 0; i < R - 1 && c_more && ok; ++i) ok = issue_codes();
      // the operands packed by the kernel launched just before (packed A rows, B pieces,
      // cleared flags) are read only after that kernel has finished
      if (p.n_ad > 0) grid_dependency_wait();
      const int half = p.htot >> 1;
      ItemIter iter = item_iter_begin(p, pair, npairs);
      Item it;
      while (ok && next_item(iter, p, pair, npairs, it)) {
        if (it.rank) {
          const int x_row = it.m * kPairM + static_cast<int>(cta) * kBM;
          const int a_row = it.q * p.htot + static_cast<int>(cta) * half;   // the pass's packed rows
          // X rows of the block and this CTA's half of the pass's packed A rows (one box each)
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            uint8_t* st;
            uint32_t fb;
            if (!(ok = claim(2u * kATileBytes + rank_tx, st, fb))) break;
            tma_load_2d_pair(st, &maps.x, kb * kBK, x_row, fb);
            tma_load_2d_pair_hint(st + kATileBytes, &maps.ap, kb * kBK, a_row, fb, keep);
            advance();
          }
          continue;
        }
        const Tile& t = it.t;
        const int a0 = p.ad_begin[t.g], a1 = p.ad_begin[t.g + 1];
        // this CTA's X rows of the tile's first half; half h starts h * 256 rows further
        const int x_row = t.m * (kPairM * kMH) + static_cast<int>(cta) * kBM;
        const int blk0 = t.m * kMH;                           // the tile's 256-row blocks
        const int nblk = min(kMH, p.r_blocks - blk0);
        // the blocks' flags, read (relaxed) before the base K loop and used at its end, so
        // that the read's latency overlaps the base steps' loads (an acquire here would hold
        // back every later load until the flag's line came back); usually they are set
        uint32_t peek = p.flag_target;
        if (a1 > a0)
          for (int h = 0; h < nblk; ++h) peek = min(peek, ld_relaxed_gpu(p.flags + blk0 + h));
        if (p.has_base) {
          const int w_row = weight_row(p, t, cta);
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            uint8_t* st;
            uint32_t fb;
            // 4-bit W: only the X rows of both halves come with the stage; the
            // dequantisation warps write the weight slot (wfull) from the codes ring
            if (!(ok = claim(kNF4 ? 2u * kXBytes : 4u * kATileBytes, st, fb))) break;
            if (kNF4) {
              for (int h = 0; h < kMH; ++h)
                tma_load_2d_pair(st + h * kATileBytes, &maps.x, kb * kBK, x_row + h * kPairM, fb);
              advance();
              if (c_more && !(ok = issue_codes())) break;   // the step R - 1 ahead
              continue;
            } else {
              tma_load_2d_pair(st, &maps.x, kb * kBK, x_row, fb);
              if (p.w_mn) {
                // W stored [in, out]: the step's 64 K rows x this CTA's 128 output columns, as
                // two 64-column boxes (an MN-major operand)
                tma_load_2d_pair_hint(st + kATileBytes, &maps.w, w_row, kb * kBK, fb, keep);
                tma_load_2d_pair_hint(st + kATileBytes + kATileBytes / 2, &maps.w, w_row + 64, kb * kBK, fb, keep);
              } else {
                tma_load_2d_pair_hint(st + kATileBytes, &maps.w, kb * kBK, w_row, fb, keep);
              }
            }
            advance();
          }
          if (!ok) break;
        }
        if (a1 > a0) {
          // second contraction: H~ of the tile's rows (written by the rank items of its
          // blocks) and B
          if (peek >= p.flag_target) {
            fence_acq_rel_gpu();                 // the relaxed reads saw every release: acquire
          } else {
            for (int h = 0; h < nblk && ok; ++h)
              ok = flag_wait(p.flags + blk0 + h, p.flag_target, abort_flag, tmo, status);
          }
          if (!ok) break;
          fence_proxy_async_global();
          for (int a = a0; a < a1 && ok; ++a) {
            // SwiGLU: an adapter's B rows go to the CTA of its own half; the other CTA's
            // box starts past the last row, so TMA fills it with zeros
            const int b_row = !p.swiglu ? t.j * kBN + static_cast<int>(cta) * 128
                              : p.ad[a].group == static_cast<int>(cta) ? t.j * 128 : p.out_g + t.j * 128;
            for (int c = 0; c < p.ad[a].nchunks; ++c) {
              // a chunk with at most 32 ranks left travels in 32-rank boxes (half the bytes)
              const bool narrow = p.ad[a].rpad16 - 64 * c <= 32;
              const uint32_t box = narrow ? kATileBytes / 2 : kATileBytes;   // per CTA, per operand
              uint8_t* st;
              uint32_t fb;
              if (!(ok = claim(2u * (kMH + 1) * box, st, fb))) break;
              for (int h = 0; h < kMH; ++h)
                tma_load_2d_pair_hint(st + h * kATileBytes, narrow ? &maps.hq32 : &maps.hq, p.ad[a].toff + 64 * c,
                                      x_row + h * kPairM, fb, keep);
              tma_load_2d_pair_hint(st + kXBytes, narrow ? &maps.b32[a] : &maps.b[a], c * 64, b_row, fb, keep);
              advance();
            }
          }
        }
      }
      if (!ok) {
        // Wait (bounded) for the copies put in flight before the CTA exits: the pair's
        // copies complete on the leader's barriers, a 4-bit W's codes on code_full.
        for (int s = 0; s < S; ++s) {
          const uint32_t n = n_issued / S + (static_cast<uint32_t>(s) < n_issued % S ? 1u : 0u);
          if (n == 0 || !leader) continue;
          const uint32_t par = (n - 1) & 1u;
          const uint64_t t0 = globaltimer_ns();
          const uint32_t a = smem_u32(&full[s]);
          while (!mbar_try_wait_cluster(a, par) && globaltimer_ns() - t0 < 100000000ull) {
          }
        }
        for (int s = 0; s < R; ++s) {
          const uint32_t n = c_issued / R + (static_cast<uint32_t>(s) < c_issued % R ? 1u : 0u);
          if (n == 0) continue;
          const uint64_t t0 = globaltimer_ns();
          const uint32_t a = smem_u32(&code_full[s]);
          while (!mbar_try_wait(a, (n - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int count = 0;
      // item `count` uses accumulator buffer count & 1 (a 4-bit W's tile: buffer 0 always);
      // the parity of that buffer's earlier uses
      auto use_parity = [&]() -> uint32_t { return static_cast<uint32_t>(kNF4 ? count : (count >> 1)) & 1u; };
      const uint32_t idesc_acc = idesc_bf16_f32(kPairM, kBN);
      const uint32_t idesc_acc_mn = idesc_bf16_f32_bmn(kPairM, kBN);
      const uint32_t idesc_h = idesc_bf16_f32(kPairM, p.htot > 0 ? p.htot : 16);
      const uint32_t stage_base = smem_u32(sbase);
      bool ok = true;
      // This thread issues every MMA of the pair, so its instructions between two MMAs are
      // on the tensor core's critical path: a step's descriptors are the constant fields
      // and the start address (16-byte units, below 2^14 for any shared-memory address) of
      // its slot, stage 0's plus the stage's offset.
      const uint32_t u_x = stage_base >> 4;                     // X / H~ rows
      const uint32_t u_w = (stage_base + kXBytes) >> 4;         // W, packed A or B rows
      constexpr uint32_t kHalfStep = kATileBytes >> 4;          // next M half's X rows
      const uint32_t stage_units = static_cast<uint32_t>(SB) >> 4;
      // Operands of a step: A (X or H~ rows of each half) first, then B.  Every step
      // waits for the TMA bytes of both CTAs (full) and, with a 4-bit W, for the
      // dequantisation warps (wfull: the weight tile of a base step is written; on the
      // other steps it keeps every dequantisation warp in step).
      int s0 = 0;
      uint32_t off_next = 0;                  // descriptor offset of `stage`
      auto take = [&](uint32_t& off) -> bool {
        if (!mbar_wait(&full[stage], phase, abort_flag, tmo, status)) return false;
        if (kNF4 && !mbar_wait_cluster(&wfull[stage], phase, abort_flag, tmo, status)) return false;
        s0 = stage;
        off = off_next;
        off_next += stage_units;
        if (++stage == S) { stage = 0; phase ^= 1; off_next = 0; }
        tc_fence_after();
        return true;
      };
      auto give_back = [&]() { mma_commit_pair_mc(&empty[s0], kBothCtas); };
      ItemIter iter = item_iter_begin(p, pair, npairs);
      Item it;
      while (next_item(iter, p, pair, npairs, it)) {
        const int a0 = it.rank ? 0 : p.ad_begin[it.t.g];
        const int a1 = it.rank ? 0 : p.ad_begin[it.t.g + 1];
        if (!it.rank && !(p.has_base || a1 > a0)) continue;   // bias-only tile: no MMA
        const int b = kNF4 ? 0 : (count & 1);   // a 4-bit W's tile fills all 512 columns
        if (!(ok = mbar_wait_cluster(&acc_empty[b], use_parity() ^ 1u, abort_flag, tmo, status)))
          break;
        tc_fence_after();
        const uint32_t acc_t = tmem + b * kBN;
        if (it.rank) {
          // one MMA per K step covers every adapter: N = htot rank columns (the packed A
          // rows sit one X box further)
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            uint32_t off;
            if (!(ok = take(off))) break;
            const uint64_t ad = kDescSw128K | (u_x + off), rd = kDescSw128K | (u_x + off + kHalfStep);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_bf16_pair(acc_t, ad + 2 * kk, rd + 2 * kk, idesc_h, (kb | kk) != 0 ? 1u : 0u);
            give_back();
          }
        } else {
          if (p.has_base && !p.w_mn) {
            for (int kb = 0; kb < p.k_blocks; ++kb) {
              uint32_t off;
              if (!(ok = take(off))) break;
              const uint64_t ad = kDescSw128K | (u_x + off), bd = kDescSw128K | (u_w + off);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
                for (int h = 0; h < kMH; ++h)
                  mma_bf16_pair(acc_t + h * kBN, ad + h * kHalfStep + 2 * kk, bd + 2 * kk, idesc_acc,
                                (kb | kk) != 0 ? 1u : 0u);
              give_back();
            }
          } else if (p.has_base) {
            // W stored [in, out]: an MN-major weight slot, 2048 bytes per 16 K rows
            for (int kb = 0; kb < p.k_blocks; ++kb) {
              uint32_t off;
              if (!(ok = take(off))) break;
              const uint64_t ad = kDescSw128K | (u_x + off), bd = kDescSw128MN | (u_w + off);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
                for (int h = 0; h < kMH; ++h)
                  mma_bf16_pair(acc_t + h * kBN, ad + h * kHalfStep + 2 * kk, bd + kk * (2048 >> 4), idesc_acc_mn,
                                (kb | kk) != 0 ? 1u : 0u);
              give_back();
            }
          }
          bool accum = p.has_base != 0;
          for (int a = a0; a < a1 && ok; ++a) {
            for (int c = 0; c < p.ad[a].nchunks; ++c) {
              uint32_t off;
              if (!(ok = take(off))) break;
              const int kext = min(64, p.ad[a].rpad16 - 64 * c);
              const bool narrow = kext <= 32;              // 32-rank boxes, 64-byte swizzle
              const uint64_t bits = narrow ? kDescSw64K : kDescSw128K;
              const uint64_t ad = bits | (u_x + off), bd = bits | (u_w + off);
              for (int kk = 0; kk < kext / 16; ++kk)
#pragma unroll
                for (int h = 0; h < kMH; ++h)
                  mma_bf16_pair(acc_t + h * kBN, ad + h * kHalfStep + 2 * kk, bd + 2 * kk, idesc_acc,
                                (accum || kk > 0) ? 1u : 0u);
              accum = true;
              give_back();
            }
          }
        }
        if (!ok) break;
        mma_commit_pair_mc(&acc_full[b], kBothCtas);
        ++count;
      }
      // Every MMA this thread issued must finish before tensor memory is freed.
      mma_commit_pair_mc(drain, 0x1);
      const uint32_t a = smem_u32(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait_cluster(a, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  }
  } else if (warp < kDeqWarp0) {
    if (kNF4) regs_inc<104>();
    // ------------------------------------------------------------ epilogue
    // Output chunks of 128 bytes per row (64 bf16 or 32 fp32 columns) are staged in
    // 128-byte-swizzled shared buffers and written by TMA bulk stores (evict-first in L2);
    // a partial chunk at the end of a column group is written with plain stores.  bf16 W:
    // one warpgroup, two staging buffers used in turn.  4-bit W: warpgroup eg drains M
    // half eg of a tile through its own buffer, the other half at the same time (the tile
    // holds all of tensor memory, so the MMAs wait for both); rank items are read by
    // warpgroup 0.  Every wait outcome is OR-reduced over a warpgroup so that its warps
    // always leave together and never strand each other at a named barrier.
    const int eg = (warp - kEpiWarp0) >> 2;  // epilogue warpgroup
    const uint32_t bar_main = 1 + 2 * eg, bar_any = 2 + 2 * eg;
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int row_in_cta = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t stg_addr = smem_u32(stg);
    const bool elected = threadIdx.x == (kEpiWarp0 + 4 * eg) * 32;
    const int h_begin = kNF4 ? eg : 0, h_end = kNF4 ? eg + 1 : kMH;   // M halves drained here
    // staging buffer of chunk sidx, and the wait before reusing it
    auto stg_index = [&](uint32_t sidx) -> int { return kNF4 ? eg : static_cast<int>(sidx & 1); };
    auto stg_free = [&](uint32_t sidx) {
      if (kNF4) {
        if (sidx >= 1 && elected) bulk_wait_read_0();
      } else if (sidx >= 2 && elected) {
        bulk_wait_read_le1();
      }
    };
    const uint32_t acc_empty_l0 = mapa_shared(smem_u32(&acc_empty[0]), 0);   // buffer b: + 8 b
    const uint64_t stream_out = l2_evict_first();   // Y is written once: keep X and W in L2
    const int cw = p.y_f32 ? 32 : 64;               // columns per 128-byte row chunk
    int count = 0;
    auto use_parity = [&]() -> uint32_t { return static_cast<uint32_t>(kNF4 ? count : (count >> 1)) & 1u; };
    uint32_t sidx = 0;                              // staging chunks issued so far
    if (p.n_ad > 0) grid_dependency_wait();          // rank items release flags cleared by it
    ItemIter iter = item_iter_begin(p, pair, npairs);
    Item it;
    while (next_item(iter, p, pair, npairs, it)) {
      const int b = kNF4 ? 0 : (count & 1);
      if (it.rank && eg == 1) {
        // 4-bit W: warpgroup 1 has no rows of the rank item to read; it only counts the
        // item off the accumulator buffer, after the MMAs filled it
        const bool okw = mbar_wait_cluster(&acc_full[b], use_parity(), abort_flag, tmo, status);
        if (named_bar_any(!okw, bar_any, 128)) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_l0 + 8u * static_cast<uint32_t>(b));
        ++count;
        continue;
      }
      if (it.rank) {
        // s X A^T of every adapter -> bf16 H~ rows of this block in global memory (and
        // the fp32 values in h_out when asked), then the block's flag
        const bool okw = mbar_wait_cluster(&acc_full[b], use_parity(), abort_flag, tmo, status);
        if (named_bar_any(!okw, bar_any, 128)) break;
        tc_fence_after();
        const uint32_t h_t = tmem + b * kBN;
        const int row = it.m * kPairM + static_cast<int>(cta) * kBM + row_in_cta;
        const bool row_ok = row < p.T;
        uint16_t* hrow = p.hq + static_cast<long long>(row_ok ? row : 0) * p.hq_ld;
        for (int a = 0; a < p.n_ad; ++a) {
          if (p.ad[a].pass != it.q) continue;          // another pass's adapter
          const float s = p.ad[a].s;
          const int units = p.ad[a].pw >> 3;           // 8 rank columns per unit
          // TMEM column of unit u: the two halves of an adapter's columns may lie apart
          const int hu = units >> 1;
          auto col = [&](int u) { return u < hu ? p.ad[a].hoff + u * 8 : p.ad[a].hoff2 + (u - hu) * 8; };
          if (p.ad[a].split3) {
            // FP32 adapter: s X A^T = s (X a1^T + X a2^T + X a3^T) in fp32, split again into
            // bf16 pieces h1 + h2 + h3 and laid out as [h1 h1 h2 h1 h2 h3] against the
            // [b1 b2 b1 b3 b2 b1] of B: every product above 2^-24 of the leading one is kept
            const int pu = units / 3;                  // units per piece
            for (int u = 0; u < pu; ++u) {
              // the unit's three pieces under one TMEM wait (the fourth address repeats one)
              uint32_t q[32];
              const uint32_t ta[4] = {h_t + lane_base + col(u), h_t + lane_base + col(u + pu),
                                      h_t + lane_base + col(u + 2 * pu), h_t + lane_base + col(u)};
              tmem_ld8x4(ta, q);
              uint32_t w1[4], w2[4], w3[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float x0 = s * ((u2f(q[2 * i]) + u2f(q[8 + 2 * i])) + u2f(q[16 + 2 * i]));
                const float x1 = s * ((u2f(q[2 * i + 1]) + u2f(q[8 + 2 * i + 1])) + u2f(q[16 + 2 * i + 1]));
                w1[i] = pack_bf16x2(x0, x1);
                const float y0 = x0 - __uint_as_float(w1[i] << 16);
                const float y1 = x1 - __uint_as_float(w1[i] & 0xffff0000u);
                w2[i] = pack_bf16x2(y0, y1);
                w3[i] = pack_bf16x2(y0 - __uint_as_float(w2[i] << 16), y1 - __uint_as_float(w2[i] & 0xffff0000u));
              }
              if (row_ok) {
                auto put = [&](int k, const uint32_t* w) {
                  st_global_v4(hrow + p.ad[a].toff + (k * pu + u) * 8, w[0], w[1], w[2], w[3]);
                };
                put(0, w1); put(1, w1); put(2, w2); put(3, w1); put(4, w2); put(5, w3);
              }
            }
            continue;
          }
          for (int u0 = 0; u0 < units; u0 += 4) {
            // 32 ranks per TMEM load where the columns allow it, else four 8-column loads
            // under one wait (a unit past the adapter's last repeats the first); registers
            // are indexed by constants only, so that r stays out of local memory
            uint32_t r[32];
            const int n = min(4, units - u0);
            if (n == 4 && col(u0 + 3) == col(u0) + 24) {
              tmem_ld32(h_t + lane_base + col(u0), r);
            } else {
              uint32_t ta[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) ta[k] = h_t + lane_base + col(k < n ? u0 + k : u0);
              tmem_ld8x4(ta, r);
            }
            if (!row_ok) continue;
            if (p.h_out) {
              // keep s * X A^T in fp32 as well (the backward needs it for dA)
              float* ho = p.h_out + static_cast<long long>(row) * p.h_out_ld + p.ad[a].hout_off;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < n * 8 && u0 * 8 + i < p.ad[a].rank) ho[u0 * 8 + i] = u2f(r[i]) * s;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (k >= n) break;
              const uint32_t* q8 = r + k * 8;
              st_global_v4(hrow + p.ad[a].toff + (u0 + k) * 8, pack_bf16x2(u2f(q8[0]) * s, u2f(q8[1]) * s),
                           pack_bf16x2(u2f(q8[2]) * s, u2f(q8[3]) * s), pack_bf16x2(u2f(q8[4]) * s, u2f(q8[5]) * s),
                           pack_bf16x2(u2f(q8[6]) * s, u2f(q8[7]) * s));
            }
          }
        }
        // the accumulator is fully in registers: hand it back to the MMA
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_l0 + 8u * static_cast<uint32_t>(b));
        // H~ rows visible to the TMA loads of other pairs: every thread orders its stores
        // for the async proxy, the barrier gathers them, and one release counts this CTA in
        fence_proxy_async_global();
        named_bar_sync(bar_main, 128);
        if (elected) red_release_gpu_add(p.flags + it.m, 1u);
        ++count;
        continue;
      }
      const Tile& t = it.t;
      const int a0 = p.ad_begin[t.g], a1 = p.ad_begin[t.g + 1];
      const bool any_mma = p.has_base || a1 > a0;
      if (!kNF4 && p.resid) {
        // merge: pull this thread's residual rows toward L2 one tile ahead of their use (the
        // first tile's own rows too), so that they land while this tile is drained
        auto prefetch_tile = [&](const Tile& tt) {
          const int esz = p.resid_f32 ? 4 : 2;
          const int nbytes = min(kBN, p.out_g - tt.j * kBN) * esz;
          for (int h = h_begin; h < h_end; ++h) {
            const int row = tt.m * (kPairM * kMH) + h * kPairM + static_cast<int>(cta) * kBM + row_in_cta;
            if (row >= p.T) continue;
            const char* rp = static_cast<const char*>(p.resid) +
                             (static_cast<long long>(row) * p.ld_resid + tt.g * p.out_g + tt.j * kBN) * esz;
            for (int off = 0; off < nbytes; off += 128) prefetch_l2(rp + off);
            prefetch_l2(rp + nbytes - 1);
          }
        };
        if (count == 0) prefetch_tile(t);
        ItemIter peek = iter;                       // the iterator's state alone: a copy peeks
        Item nx;
        if (next_item(peek, p, pair, npairs, nx) && !nx.rank) prefetch_tile(nx.t);
      }
      if (any_mma) {
        const bool ok = mbar_wait_cluster(&acc_full[b], use_parity(), abort_flag, tmo, status);
        if (named_bar_any(!ok, bar_any, 128)) break;
        tc_fence_after();
      }
      if (p.swiglu) {
        // SwiGLU front half: accumulator columns [0, 128) hold e (gate) and [128, 256) g
        // (up) of the same output columns.  e and g are rounded to bf16 once -- they are
        // the two linears' outputs, written to eg when asked -- and h = silu(e) g is
        // rounded once; h chunks of 64 columns go out like the plain output.
        const int ncol = min(128, p.out_g - t.j * 128);
        const int nch = (ncol + 63) / 64;
#pragma unroll 1
        for (int h = h_begin; h < h_end; ++h) {
          const int row0 = t.m * (kPairM * kMH) + h * kPairM + static_cast<int>(cta) * kBM;
          const int row = row0 + row_in_cta;
          const bool row_ok = row < p.T;
          const uint32_t acc_t = tmem + (b + h) * kBN;
#pragma unroll 1
          for (int c = 0; c < nch; ++c) {
            const int cig = t.j * 128 + c * 64;            // first h column of the chunk
            const int ncols = min(64, p.out_g - cig);
            const bool full_chunk = ncols == 64;
            const uint32_t buf = stg_addr + stg_index(sidx) * kStgBytes;
            if (full_chunk) {
              stg_free(sidx);
              named_bar_sync(bar_main, 128);
            }
            // 16 columns at a time: e and g under one TMEM wait
#pragma unroll 1
            for (int sub = 0; sub < 4; ++sub) {
              const int c0 = c * 64 + sub * 16;            // column within the tile's 128
              uint32_t re[16], rg[16];
              tmem_ld16x2(acc_t + lane_base + c0, re, acc_t + lane_base + 128 + c0, rg);
              if (h == h_end - 1 && c == nch - 1 && sub == 3) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc_empty_l0 + 8u * static_cast<uint32_t>(b));
              }
              const int nc = min(16, ncols - sub * 16);
              const int col = cig + sub * 16;              // first column of the sub-chunk
              uint32_t eb[8], gb[8], hb[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float e0 = u2f(re[2 * i]), e1 = u2f(re[2 * i + 1]);
                float g0 = u2f(rg[2 * i]), g1 = u2f(rg[2 * i + 1]);
                if (p.bias && 2 * i < nc) {
                  e0 += bias_at(p, col + 2 * i); e1 += bias_at(p, col + 2 * i + 1);
                  g0 += bias_at(p, p.out_g + col + 2 * i); g1 += bias_at(p, p.out_g + col + 2 * i + 1);
                }
                eb[i] = pack_bf16x2(e0, e1);
                gb[i] = pack_bf16x2(g0, g1);
                hb[i] = pack_bf16x2(__fmul_rn(silu_f32(u2f(eb[i] << 16)), u2f(gb[i] << 16)),
                                    __fmul_rn(silu_f32(u2f(eb[i] & 0xffff0000u)), u2f(gb[i] & 0xffff0000u)));
              }
              if (p.eg && row_ok) {
                uint16_t* pe = p.eg + static_cast<long long>(row) * p.ld_eg + col;
#pragma unroll
                for (int u = 0; u < 2; ++u)
                  if (u * 8 < nc) {
                    st_global_v4_hint(pe + u * 8, eb[4 * u], eb[4 * u + 1], eb[4 * u + 2], eb[4 * u + 3], stream_out);
                    st_global_v4_hint(pe + p.out_g + u * 8, gb[4 * u], gb[4 * u + 1], gb[4 * u + 2], gb[4 * u + 3],
                                      stream_out);
                  }
              }
              if (full_chunk) {
                const uint32_t rowb = buf + row_in_cta * 128;
#pragma unroll
                for (int u = 0; u < 2; ++u)
                  st_shared_v4(rowb + (((sub * 2 + u) ^ (row_in_cta & 7)) * 16), hb[4 * u], hb[4 * u + 1],
                               hb[4 * u + 2], hb[4 * u + 3]);
              } else if (row_ok) {
                uint16_t* y = static_cast<uint16_t*>(p.Y) + static_cast<long long>(row) * p.ldy + col;
#pragma unroll
                for (int u = 0; u < 2; ++u)
                  if (u * 8 < nc)
                    st_global_v4_hint(y + u * 8, hb[4 * u], hb[4 * u + 1], hb[4 * u + 2], hb[4 * u + 3], stream_out);
              }
            }
            if (full_chunk) {
              fence_proxy_async_smem();
              named_bar_sync(bar_main, 128);
              if (elected && row0 < p.T) {
                tma_store_2d_hint(&maps.y, cig, row0, stg + stg_index(sidx) * kStgBytes, stream_out);
                bulk_commit();
              }
              ++sidx;
            }
          }
        }
        ++count;
        continue;
      }

      // valid chunks of this tile (the last tile of a group may be partial)
      const int nchunk = min(kBN / cw, (p.out_g - t.j * kBN + cw - 1) / cw);
      // merge: the residual of 32-column sub-chunk (cc, ss) of `row` into dst (4 x 16 bytes
      // bf16, 8 x 16 bytes fp32; the row pitch and the sub-chunk start are multiples of 8
      // elements), issued one sub-chunk ahead of its use so its latency overlaps the work
      const int esz_r = p.resid_f32 ? 4 : 2;
      auto load_res = [&](int row, int cc, int ss, uint4 (&dst)[8]) {
        const int cig2 = t.j * kBN + cc * cw + ss * 32;
        const int n2 = min(32, p.out_g - cig2);
        const uint4* rp = reinterpret_cast<const uint4*>(
            static_cast<const char*>(p.resid) +
            (static_cast<long long>(row) * p.ld_resid + t.g * p.out_g + cig2) * esz_r);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < 2 * esz_r && i * (16 / esz_r) < n2) dst[i] = rp[i];
      };
#pragma unroll 1
      for (int h = h_begin; h < h_end; ++h) {
      const int row0 = t.m * (kPairM * kMH) + h * kPairM + static_cast<int>(cta) * kBM;
      const int row = row0 + row_in_cta;
      const bool row_ok = row < p.T;
      const uint32_t acc_t = tmem + (b + h) * kBN;
      const bool res_row = !kNF4 && p.resid && row_ok;   // merges run on the bf16 instantiation
      uint4 rnext[8], rcur[8];
      if (res_row) load_res(row, 0, 0, rnext);
#pragma unroll 1
      for (int c = 0; c < nchunk; ++c) {
        const int cig = t.j * kBN + c * cw;                 // first column, within the group
        const int ncols = min(cw, p.out_g - cig);           // uniform across the warps
        const int gcol = t.g * p.out_g + cig;
        const bool full_chunk = ncols == cw;
        const uint32_t buf = stg_addr + stg_index(sidx) * kStgBytes;
        if (full_chunk) {
          // the staging buffer is free once the bulk store that last used it has read it
          stg_free(sidx);
          named_bar_sync(bar_main, 128);
        }
        // 32 columns at a time: TMEM -> registers -> bias / FP32 adapters -> staging
#pragma unroll 1
        for (int sub = 0; sub < cw / 32; ++sub) {
          const int c0 = sub * 32;                          // first column of the sub-chunk
          float v[32];
          if (any_mma) {
            uint32_t r[32];
            tmem_ld32(acc_t + lane_base + c * cw + c0, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = u2f(r[i]);
            if (h == h_end - 1 && c == nchunk - 1 && sub == cw / 32 - 1) {
              // the accumulator is fully in registers: hand it back to the MMA
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(acc_empty_l0 + 8u * static_cast<uint32_t>(b));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
          const int nc = min(32, ncols - c0);               // valid columns of the sub-chunk
          if (res_row && nc > 0) {
            // merge: s * acc + R, two fp32 roundings; this sub-chunk's R was loaded one
            // sub-chunk ago, the next one's load goes out now
#pragma unroll
            for (int i = 0; i < 8; ++i) rcur[i] = rnext[i];
            const int cn = sub + 1 < cw / 32 ? c : c + 1, sn = sub + 1 < cw / 32 ? sub + 1 : 0;
            if (cn < nchunk && t.j * kBN + cn * cw + sn * 32 < p.out_g) load_res(row, cn, sn, rnext);
            if (p.resid_f32) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if (4 * i < nc) {
                  const float4 r4 = make_float4(__uint_as_float(rcur[i].x), __uint_as_float(rcur[i].y),
                                                __uint_as_float(rcur[i].z), __uint_as_float(rcur[i].w));
                  v[4 * i] = __fadd_rn(__fmul_rn(v[4 * i], p.acc_scale), r4.x);
                  v[4 * i + 1] = __fadd_rn(__fmul_rn(v[4 * i + 1], p.acc_scale), r4.y);
                  v[4 * i + 2] = __fadd_rn(__fmul_rn(v[4 * i + 2], p.acc_scale), r4.z);
                  v[4 * i + 3] = __fadd_rn(__fmul_rn(v[4 * i + 3], p.acc_scale), r4.w);
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if (8 * i < nc) {
                  const uint4 r8 = rcur[i];
                  const uint32_t w[4] = {r8.x, r8.y, r8.z, r8.w};
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    v[8 * i + 2 * k] = __fadd_rn(__fmul_rn(v[8 * i + 2 * k], p.acc_scale), u2f(w[k] << 16));
                    v[8 * i + 2 * k + 1] = __fadd_rn(__fmul_rn(v[8 * i + 2 * k + 1], p.acc_scale), u2f(w[k] & 0xffff0000u));
                  }
                }
              }
            }
          }
          if (p.bias && nc > 0) {
            // 16-byte loads of the 32 bias values (the same for every row: broadcast)
            // where they all exist and the bias is aligned, single values otherwise
            if (p.bias_f32) {
              const float* bp = static_cast<const float*>(p.bias) + gcol + c0;
              if (nc == 32 && p.bias_vec) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 b4 = __ldg(reinterpret_cast<const float4*>(bp) + i);
                  v[4 * i] += b4.x; v[4 * i + 1] += b4.y; v[4 * i + 2] += b4.z; v[4 * i + 3] += b4.w;
                }
              } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (i < nc) v[i] += bp[i];
              }
            } else {
              const uint16_t* bp = static_cast<const uint16_t*>(p.bias) + gcol + c0;
              if (nc == 32 && p.bias_vec) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint4 b8 = __ldg(reinterpret_cast<const uint4*>(bp) + i);
                  const uint32_t w[4] = {b8.x, b8.y, b8.z, b8.w};
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    v[8 * i + 2 * k] += u2f(w[k] << 16);
                    v[8 * i + 2 * k + 1] += u2f(w[k] & 0xffff0000u);
                  }
                }
              } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (i < nc) v[i] += bf16_to_f32(bp[i]);
              }
            }
          }
          if (kF32 && p.n_ad32 > 0 && row_ok && nc > 0) {
            for (int a = 0; a < p.n_ad32; ++a) {
              if (p.ad32[a].group != t.g) continue;
              const float* hrow = p.h32 + static_cast<long long>(row) * p.h32_cols + p.ad32[a].h_off;
              const float* Bm = p.ad32[a].B + static_cast<long long>(cig + c0) * p.ad32[a].ldb;
              const long long ldb = p.ad32[a].ldb;
              // eight columns at a time: sum_j h[j] B[o, j] in fp32, then added once (B rows
              // are read by every thread of the warp: broadcast, L1-resident)
#pragma unroll
              for (int g8 = 0; g8 < 4; ++g8) {
                float dsum[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) dsum[i] = 0.f;
                if (p.ad32[a].vec4) {
#pragma unroll 1
                  for (int jj = 0; jj < p.ad32[a].rank; jj += 4) {
                    const float4 h4 = *reinterpret_cast<const float4*>(hrow + jj);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                      if (g8 * 8 + i < nc) {
                        const float4 b4 = __ldg(reinterpret_cast<const float4*>(Bm + (g8 * 8 + i) * ldb + jj));
                        dsum[i] = fmaf(h4.x, b4.x, dsum[i]);
                        dsum[i] = fmaf(h4.y, b4.y, dsum[i]);
                        dsum[i] = fmaf(h4.z, b4.z, dsum[i]);
                        dsum[i] = fmaf(h4.w, b4.w, dsum[i]);
                      }
                    }
                  }
                } else {
#pragma unroll 1
                  for (int jj = 0; jj < p.ad32[a].rank; ++jj) {
                    const float h = hrow[jj];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                      if (g8 * 8 + i < nc) dsum[i] = fmaf(h, Bm[(g8 * 8 + i) * ldb + jj], dsum[i]);
                  }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) v[g8 * 8 + i] += dsum[i];
              }
            }
          }
          if (full_chunk) {
            // four (bf16) or eight (fp32) 16-byte units of this row, 128-byte swizzled
            const uint32_t rowb = buf + row_in_cta * 128;
            if (cw == 64) {
#pragma unroll
              for (int u = 0; u < 4; ++u)
                st_shared_v4(rowb + (((sub * 4 + u) ^ (row_in_cta & 7)) * 16),
                             pack_bf16x2(v[8 * u], v[8 * u + 1]), pack_bf16x2(v[8 * u + 2], v[8 * u + 3]),
                             pack_bf16x2(v[8 * u + 4], v[8 * u + 5]), pack_bf16x2(v[8 * u + 6], v[8 * u + 7]));
            } else {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                st_shared_v4(rowb + ((u ^ (row_in_cta & 7)) * 16), f2u(v[4 * u]), f2u(v[4 * u + 1]),
                             f2u(v[4 * u + 2]), f2u(v[4 * u + 3]));
            }
          } else if (row_ok && nc > 0) {
            // partial chunk at the end of a group: plain stores, masked
            if (p.y_f32) {
              float* y = static_cast<float*>(p.Y) + static_cast<long long>(row) * p.ldy + gcol + c0;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (i * 4 < nc)
                  st_global_v4_hint(y + i * 4, f2u(v[4 * i]), f2u(v[4 * i + 1]), f2u(v[4 * i + 2]),
                                    f2u(v[4 * i + 3]), stream_out);
            } else {
              uint16_t* y = static_cast<uint16_t*>(p.Y) + static_cast<long long>(row) * p.ldy + gcol + c0;
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (i * 8 < nc)
                  st_global_v4_hint(y + i * 8, pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                    pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                    pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                    pack_bf16x2(v[8 * i + 6], v[8 * i + 7]), stream_out);
            }
          }
        }
        if (full_chunk) {
          fence_proxy_async_smem();
          named_bar_sync(bar_main, 128);
          if (elected && row0 < p.T) {                     // no store of rows past the end
            tma_store_2d_hint(&maps.y, gcol, row0, stg + stg_index(sidx) * kStgBytes, stream_out);
            bulk_commit();
          }
          ++sidx;
        }
      }
      }
      if (any_mma) {
        ++count;
      }
    }
    if (elected) bulk_wait_all();
  } else if (kNF4) {
    regs_dec<72>();
    // ------------------------------------------------------------ 4-bit dequantisation
    // Three groups of 128 threads take every third base K step (the CTA's running count
    // of them).  Thread d of a group owns row d of this CTA's 128 weight rows: for every
    // (row, K step) -- one 64-element absmax block -- it builds the 16 bf16 values
    // bf16(fl32(level[i]) * absmax) in registers, split into low-byte and high-byte planes,
    // and looks its 64 codes up four at a time with byte permutes; the result goes to the
    // stage's W slot in the 128-byte swizzle K-major layout.  The codes come from their own ring (loaded ahead), so a step waits only for
    // its slot: free once the MMAs released the stage's previous use (empty).  Every warp
    // waits on every use of every stage (so that no parity wait can pass a phase that has
    // not completed yet) and then arrives on the stage's wfull, after its tile if the use
    // is one of its group's K steps; the MMA waits for all 24 arrivals of every use, so
    // that no warp can fall two phases behind either.
    const int group = (threadIdx.x - kDeqWarp0 * 32) >> 7;
    const int r = (threadIdx.x - kDeqWarp0 * 32) & 127;
    uint32_t kc = 0;                                  // base K steps seen by this CTA
    const uint32_t wfull_l0 = mapa_shared(smem_u32(&wfull[0]), 0);   // leader's barriers
    float lv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lv[i] = p.nf4_code[i];
    const int kb64 = p.K / 64;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    auto slot_free = [&]() {                          // the stage's previous use released
      return mbar_wait_cluster(&empty[stage], phase ^ 1, abort_flag, tmo, status);
    };
    auto pass = [&]() {                               // a stage use this warp does not fill
      ok = __all_sync(0xffffffffu, slot_free());
      if (ok && lane == 0) mbar_arrive_remote(wfull_l0 + 8u * stage);
      if (++stage == S) { stage = 0; phase ^= 1; }
    };
    ItemIter iter = item_iter_begin(p, pair, npairs);
    Item it;
    while (ok && next_item(iter, p, pair, npairs, it)) {
      if (it.rank) {
        for (int kb = 0; kb < p.k_blocks && ok; ++kb) pass();
        continue;
      }
      const Tile& t = it.t;
      const int a0 = p.ad_begin[t.g], a1 = p.ad_begin[t.g + 1];
      // K-major: thread r dequantises weight row (output column) wrow, 64 K values per step.
      // W stored [in, out] (w_mn): thread r takes K row kb * 64 + (r & 63) of the step and the
      // 64 output columns mcol.. of half r >> 6 of this CTA's 128, written as row r of the
      // MN-major tile (the two 64-column halves 8 KiB apart)
      const int wrow = weight_row(p, t, cta) + r;
      const bool wrow_ok = wrow < p.N;
      const float* am_row = p.absmax + static_cast<long long>(wrow_ok ? wrow : 0) * kb64;
      const int mcol = weight_row(p, t, cta) + 64 * (r >> 6);
      const int mrow = r & 63;
      for (int kb = 0; kb < p.k_blocks && ok; ++kb, ++kc) {
        if (static_cast<int>(kc % 3u) != group) {       // another group's K step
          pass();
          continue;
        }
        const uint32_t slot = kc % static_cast<uint32_t>(R);   // its codes in the ring
        ok = slot_free() && mbar_wait(&code_full[slot], (kc / R) & 1u, abort_flag, tmo, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const uint8_t* raw = codes + slot * kCodeSlotBytes;                // codes | block scales
        // block scale: from the stage (TMA, no global load left in flight when this warp
        // releases the tile to the peer CTA) or, when the scales' rows are not 16-byte
        // multiples, straight from memory
        if (p.w_mn) {
          const int krow = kb * kBK + mrow;
          const float am = p.am_tma ? reinterpret_cast<const float*>(raw + kRawBytes)[mrow * 4 + ((mcol >> 6) & 3)]
                                    : ((krow < p.K && mcol < p.N)
                                           ? __ldg(p.absmax + static_cast<long long>(krow) * (p.N / 64) + mcol / 64)
                                           : 0.f);
          nf4_dequant_row(raw + mrow * 64, 2 * (r >> 6), (mrow >> 1) & 3, am, lv,
                          smem_u32(sbase + stage * SB + kXBytes), r);
        } else {
          const float am = p.am_tma ? reinterpret_cast<const float*>(raw + kRawBytes)[r * 4 + (kb & 3)]
                                    : (wrow_ok ? __ldg(am_row + kb) : 0.f);
          nf4_dequant_row(raw + r * 32, 0, (r >> 2) & 1, am, lv, smem_u32(sbase + stage * SB + kXBytes), r);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_remote(wfull_l0 + 8u * stage);
          mbar_arrive(&code_empty[slot]);
        }
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      for (int a = a0; a < a1 && ok; ++a)
        for (int c = 0; c < p.ad[a].nchunks && ok; ++c) pass();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();                          // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

namespace {

// attr must hold 2 entries; `pdl` lets the kernel start while the previous kernel of the
// stream (the operand pack) is still running.
template <bool kNF4>
cudaLaunchConfig_t pair_config(int grid, size_t smem_bytes, cudaStream_t stream,
                               cudaLaunchAttribute* attr, bool pdl = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kNF4 ? kTcThreadsNF4 : kTcThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  return cfg;
}

template <bool kNF4>
int max_pairs_impl(size_t smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(tc_fused_fwd_kernel<kNF4, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return 0;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config<kNF4>(2 * 256, smem_bytes, nullptr, attr);
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, tc_fused_fwd_kernel<kNF4, false>, &cfg);
  if (e != cudaSuccess || n <= 0) {
    if (e != cudaSuccess) set_last_cuda_error(e);
    n = device_sm_count() / 2;
  }
  return n;
}

template <bool kNF4, bool kF32>
int launch_impl(const TcMaps& maps, const TcParams& p, int grid, size_t smem_bytes,
                cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(tc_fused_fwd_kernel<kNF4, kF32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config<kNF4>(grid, smem_bytes, stream, attr, p.n_ad > 0);
  e = cudaLaunchKernelEx(&cfg, tc_fused_fwd_kernel<kNF4, kF32>, maps, p);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

}  // namespace

int tc_max_pairs(size_t smem_bytes, bool nf4) {
  static size_t cached_smem[2] = {0, 0};
  static int cached[2] = {0, 0};
  static int cached_dev[2] = {-1, -1};
  int dev = 0;
  cudaGetDevice(&dev);
  const int k = nf4 ? 1 : 0;
  if (cached_smem[k] == smem_bytes && cached_dev[k] == dev && cached[k] > 0) return cached[k];
  const int n = nf4 ? max_pairs_impl<true>(smem_bytes) : max_pairs_impl<false>(smem_bytes);
  cached_smem[k] = smem_bytes;
  cached[k] = n;
  cached_dev[k] = dev;
  return n;
}

int launch_tc_fwd(const TcMaps& maps, const TcParams& params, int grid, size_t smem_bytes,
                  cudaStream_t stream, bool nf4) {
  // the pairs' stride through the tiles, in (row block, group, column tile) digits
  TcParams p = params;
  const int npairs = grid / 2;
  p.step_j = p.step_g = p.step_m = 0;
  if (p.nt_g > 0 && p.G > 0 && npairs > 0) {
    p.step_j = npairs % p.nt_g;
    p.step_g = (npairs / p.nt_g) % p.G;
    p.step_m = npairs / p.nt_g / p.G;
  }
  const bool f32 = p.n_ad32 > 0;
  if (nf4)
    return f32 ? launch_impl<true, true>(maps, p, grid, smem_bytes, stream)
               : launch_impl<true, false>(maps, p, grid, smem_bytes, stream);
  return f32 ? launch_impl<false, true>(maps, p, grid, smem_bytes, stream)
             : launch_impl<false, false>(maps, p, grid, smem_bytes, stream);
}

int* tc_status_ptr() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_tc_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(ptr);
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
