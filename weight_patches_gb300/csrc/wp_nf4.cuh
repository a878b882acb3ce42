// wp_nf4.cuh -- 4-bit NormalFloat weights dequantised into a bf16 MMA operand tile in
// shared memory (Unsloth fast_lora walkthrough, section 3: the 4-bit base weight is
// dequantised into the matmul; the code layout and block scales follow the bitsandbytes
// NF4 format as the workloads store it: byte k of a row holds element 2k in its high
// nibble, one fp32 absmax per 64 consecutive elements).
//
// Value of code q in a block with scale a: bf16(fl32(level[q]) * a), rounded to nearest
// even.  A thread builds the 16 values of its (row, block) in registers, split into a
// low-byte and a high-byte plane, and looks its codes up four at a time with byte
// permutes; the result goes to the tile row in the 128-byte swizzle K-major layout (row r
// of the tile at r * 128 bytes, 16-byte unit u stored at unit u ^ (r & 7)).
#pragma once

#include <cstdint>

#include "wp_internal.h"

#include "wp_ptx.cuh"

namespace wp {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four 4-bit codes -> four bf16 values from a 16-entry table split into byte planes:
// lo[j] / hi[j] hold the low / high bytes of entries 4j..4j+3.  `sel` holds the codes' low
// three bits (a byte select into one half-table) and `pick`, per byte, 3210 plus 4 where the
// code's bit 3 points at the upper half-table; both in their low 16 bits, for the 16 bits
// of the packed stream as stored (byte k: element 2k in the high nibble), so the nibbles,
// low to high, are the codes of elements 1, 0, 3, 2.  Each plane is looked up in both
// half-tables, a third permute keeps the half the code points at, and the last two
// permutes interleave the planes back into element order.  Returns the words holding
// elements (0, 1) and (2, 3).
__device__ __forceinline__ void lookup4(uint32_t sel, uint32_t pick, const uint32_t (&lo)[4],
                                        const uint32_t (&hi)[4], uint32_t& out01, uint32_t& out23) {
  const uint32_t l = prmt(prmt(lo[0], lo[1], sel), prmt(lo[2], lo[3], sel), pick);
  const uint32_t h = prmt(prmt(hi[0], hi[1], sel), prmt(hi[2], hi[3], sel), pick);
  out01 = prmt(l, h, 0x4051u);
  out23 = prmt(l, h, 0x6273u);
}

// All 64 elements of one block: row `r` of the tile, one table for the 64 codes.
// `row` points at the row's codes in shared memory as the copy engine swizzled them: the
// block's two 16-byte halves are the row's 16-byte units unit0 and unit0 + 1, stored at
// unit ^ swz (the 32-byte swizzle of 32-byte rows: swz = (r >> 2) & 1; the 64-byte swizzle
// of 64-byte rows: swz = (r >> 1) & 3), which spreads the rows of a quarter-warp load over
// eight bank groups.  `am` is the block's scale, `lv` the 16 levels, `tile` the shared-
// memory address of the tile (row r at r * 128 bytes, 16-byte unit u stored at unit
// u ^ (r & 7): the 128-byte swizzle, K-major).
__device__ __forceinline__ void nf4_dequant_row(const uint8_t* row, int unit0, int swz, float am,
                                                const float (&lv)[16], uint32_t tile, int r) {
  uint32_t e[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) e[k] = pack_bf16x2(lv[2 * k] * am, lv[2 * k + 1] * am);
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    lo[j] = prmt(e[2 * j], e[2 * j + 1], 0x6420u);
    hi[j] = prmt(e[2 * j], e[2 * j + 1], 0x7531u);
  }
  const uint32_t dst = tile + r * 128;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint4 cw4 = *reinterpret_cast<const uint4*>(row + (((unit0 + half) ^ swz) << 4));
    const uint32_t cwords[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      // one word = 8 codes; the selectors of both 16-bit halves are formed together
      const uint32_t c = cwords[u];
      const uint32_t sel = c & 0x77777777u;
      const uint32_t pick = ((c >> 1) & 0x44444444u) | 0x32103210u;
      uint32_t o0, o1, o2, o3;
      lookup4(sel, pick, lo, hi, o0, o1);
      lookup4(sel >> 16, pick >> 16, lo, hi, o2, o3);
      const int unit = half * 4 + u;
      st_shared_v4(dst + ((unit ^ (r & 7)) * 16), o0, o1, o2, o3);
    }
  }
}

// All 64 elements of one block into registers as floats (the bf16 values W_eff), from its 32
// code bytes as stored (cw[0..7], byte k: element 2k in the high nibble), its scale and the 16
// levels: the same table and byte-permute lookups as nf4_dequant_row.
__device__ __forceinline__ void nf4_dequant_regs(const uint32_t (&cw)[8], float am, const float (&lv)[16],
                                                 float (&u)[64]) {
  uint32_t e[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) e[k] = pack_bf16x2(lv[2 * k] * am, lv[2 * k + 1] * am);
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    lo[j] = prmt(e[2 * j], e[2 * j + 1], 0x6420u);
    hi[j] = prmt(e[2 * j], e[2 * j + 1], 0x7531u);
  }
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t c = cw[w];
    const uint32_t sel = c & 0x77777777u;
    const uint32_t pick = ((c >> 1) & 0x44444444u) | 0x32103210u;
    uint32_t o[4];
    lookup4(sel, pick, lo, hi, o[0], o[1]);
    lookup4(sel >> 16, pick >> 16, lo, hi, o[2], o[3]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      u[8 * w + 2 * k] = __uint_as_float(o[k] << 16);
      u[8 * w + 2 * k + 1] = __uint_as_float(o[k] & 0xffff0000u);
    }
  }
}

// x = fl32(u / a) for a > 0 by Markstein's division (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// y = RN(1/a), q = RN(u y) is within an ulp of u / a, the residual e = u - a q is exact as one
// fused multiply-add, and RN(q + e y) is the correctly rounded quotient as long as nothing
// underflows.  For a in [2^-90, 2^90] and a quotient of magnitude 2^-5 or more (every level
// midpoint is further than that from zero) the residual is a multiple of 2^-141, so it is
// exact; a smaller quotient may come out an ulp off, which moves it across no midpoint.
// Outside that range scale_reciprocal gives 0 and the caller divides plainly instead.
__device__ __forceinline__ float div_by_scale(float u, float a, float y) {
  const float q = __fmul_rn(u, y);
  const float e = __fmaf_rn(-q, a, u);
  return __fmaf_rn(e, y, q);
}

// y for div_by_scale: RN(1/a) for a in [2^-90, 2^90], else 0 (the plain division).
__device__ __forceinline__ float scale_reciprocal(float a) {
  return a >= 0x1p-90f && a <= 0x1p90f ? __frcp_rn(a) : 0.f;
}

// max(a, b) with a NaN operand giving NaN (fmaxf drops it)
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// The 4-bit code of x in [-1, 1] (the number of level midpoints below it) by the cells of
// nf4_code_cells, held in shared memory at cells_addr as two word arrays of kCodeCells: the
// cells' next midpoints, then their base codes, for cell c = floor(16 x) + 16.  Two 4-byte
// tables rather than one of pairs: a warp's 32 lookups then fall in 32 different banks
// unless two lanes read cells 0 and 32.  The index comes from one fused multiply-add rounded
// down, RD(16 x + 2^23 + 16): the sum lies in [2^23, 2^24), where the float spacing is 1, so
// its bits are those of 2^23 plus c exactly.  kClamp: x may be a NaN, which lands outside the
// 33 cells and takes cell 0, whose compare fails (code 0, as nf4_code_of gives).
template <bool kClamp>
__device__ __forceinline__ uint32_t nf4_code_by_cells(float x, uint32_t cells_addr) {
  const uint32_t bits = __float_as_uint(__fmaf_rd(x, 16.0f, 8388624.0f));
  uint32_t addr;
  if (kClamp) {
    uint32_t c = bits - 0x4B000000u;
    c = c < static_cast<uint32_t>(kCodeCells) ? c : 0u;
    addr = cells_addr + 4u * c;
  } else {
    addr = 4u * bits + (cells_addr - 4u * 0x4B000000u);   // the same address, modulo 2^32
  }
  float next_mid;
  uint32_t base, gt;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(next_mid) : "r"(addr));
  asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(base) : "r"(addr), "n"(4 * kCodeCells));
  asm("set.gt.u32.f32 %0, %1, %2;" : "=r"(gt) : "f"(x), "f"(next_mid));   // all ones when above
  return base - gt;
}

// Requantise one block held in registers: absmax' = m = max |u| (m > 0), the codes of
// x = fl32(u / m) packed as stored (byte k: element 2k in the high nibble).  kFast: the
// quotient by div_by_scale with y = scale_reciprocal(m) != 0 and no NaN in the block; else the
// plain division and the NaN-safe cell index.
template <bool kFast>
__device__ __forceinline__ void nf4_requant_regs(const float (&u)[64], float m, float y, uint32_t cells_addr,
                                                 uint32_t (&cw)[8]) {
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t c4 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x = kFast ? div_by_scale(u[8 * w + i], m, y) : __fdiv_rn(u[8 * w + i], m);
      c4 += nf4_code_by_cells<!kFast>(x, cells_addr) << (8 * (i >> 1) + ((i & 1) ? 0 : 4));
    }
    cw[w] = c4;
  }
}

// The whole requantisation of a block: returns absmax' = max |u| (the largest of the other
// elements when some are NaN) and the codes, x = fl32(u / absmax') rounded to the nearest
// level (a value on a midpoint takes the lower code); an all-zero block keeps scale 0 and
// level 0's code.  One pass finds the maximum with a NaN kept, which sends such a block the
// plain way; the usual block takes the fast quotient once for all its elements.
__device__ __forceinline__ float nf4_requant_block(const float (&u)[64], uint32_t cells_addr, uint32_t (&cw)[8]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) m = fmax_nan(m, fabsf(u[i]));
  const bool nan_in = m != m;
  if (nan_in) {
    m = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) m = fmaxf(m, fabsf(u[i]));
  }
  const float y = nan_in ? 0.f : scale_reciprocal(m);
  if (y != 0.f) {
    nf4_requant_regs<true>(u, m, y, cells_addr, cw);
  } else if (m > 0.f) {
    nf4_requant_regs<false>(u, m, y, cells_addr, cw);
  } else {
#pragma unroll
    for (int w = 0; w < 8; ++w) cw[w] = 0x77777777u;
  }
  return m;
}

// ---------------------------------------------------------------- stochastic re-encoding
// Philox4x32-10 (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random numbers:
// as easy as 1, 2, 3", SC 2011): ten rounds of (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0,
// lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)) with the key advanced by the two Weyl
// constants between rounds.
__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c[0]), lo0 = 0xD2511F53u * c[0];
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]), lo1 = 0xCD9E8D57u * c[2];
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// The stochastic code of x in [-1, 1] with the element's draw U (23 bits), by the level cells
// of nf4_level_cells at cells_addr: four word arrays of kCodeCells (the first level at or
// above the cell's start, its index, the level before it and the level after it).  x equal
// to a level keeps that level's code; otherwise, between its neighbours lo < x < hi, the
// upper code when U w < d 2^23 (d = fl32(x - lo), w = fl32(hi - lo)); the fused multiply-add
// below has the sign of U w - d 2^23 exactly, both products being exact.  A NaN x takes code 0.
template <bool kClamp>
__device__ __forceinline__ uint32_t nf4_code_stochastic(float x, uint32_t U, uint32_t cells_addr) {
  const uint32_t bits = __float_as_uint(__fmaf_rd(x, 16.0f, 8388624.0f));
  uint32_t c = bits - 0x4B000000u;
  if (kClamp) c = c < static_cast<uint32_t>(kCodeCells) ? c : 0u;
  const uint32_t addr = cells_addr + 4u * c;
  float next_l, prev_l, after_l;
  uint32_t base;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(next_l) : "r"(addr));
  asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(base) : "r"(addr), "n"(4 * kCodeCells));
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(prev_l) : "r"(addr), "n"(8 * kCodeCells));
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(after_l) : "r"(addr), "n"(12 * kCodeCells));
  const bool gt = x > next_l;
  const float lo = gt ? next_l : prev_l, hi = gt ? after_l : next_l;
  const float d = __fsub_rn(x, lo), w = __fsub_rn(hi, lo);
  const float uf = __fsub_rn(__uint_as_float(0x4B000000u | U), 8388608.0f);      // U exactly
  const bool up = __fmaf_rn(uf, w, -__fmul_rn(d, 8388608.0f)) < 0.f;
  uint32_t code = x == next_l ? base : base + (gt ? 1u : 0u) + (up ? 1u : 0u) - 1u;
  if (kClamp && x != x) code = 0u;
  return code;
}

// The stochastic requantisation of a block whose first element has logical index e0 (a
// multiple of 4): absmax' and x exactly as nf4_requant_block, then each code sampled with
// the element's Philox draw (counter = e / 4, word e % 4, key = the seed's two words).
__device__ __forceinline__ float nf4_requant_block_stochastic(const float (&u)[64], uint32_t cells_addr,
                                                              unsigned long long e0, uint32_t k0, uint32_t k1,
                                                              uint32_t (&cw)[8]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) m = fmax_nan(m, fabsf(u[i]));
  const bool nan_in = m != m;
  if (nan_in) {
    m = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) m = fmaxf(m, fabsf(u[i]));
  }
  if (!(m > 0.f)) {
#pragma unroll
    for (int w = 0; w < 8; ++w) cw[w] = 0x77777777u;
    return m;
  }
  const float y = nan_in ? 0.f : scale_reciprocal(m);
  const unsigned long long q0 = e0 >> 2;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t c4 = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {                 // four elements per Philox call
      const unsigned long long q = q0 + 2 * w + h;
      uint32_t r[4] = {static_cast<uint32_t>(q), static_cast<uint32_t>(q >> 32), 0u, 0u};
      philox4x32_10(r, k0, k1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * h + j;                  // element 8 w + i
        const float v = u[8 * w + i];
        const float x = y != 0.f ? div_by_scale(v, m, y) : __fdiv_rn(v, m);
        const uint32_t code = y != 0.f ? nf4_code_stochastic<false>(x, r[j] >> 9, cells_addr)
                                       : nf4_code_stochastic<true>(x, r[j] >> 9, cells_addr);
        c4 += code << (8 * (i >> 1) + ((i & 1) ? 0 : 4));
      }
    }
    cw[w] = c4;
  }
  return m;
}

// The 4-bit code of x = u / absmax' (the nearest level): the number of level midpoints
// mid[k] = fl32((level[k] + level[k+1]) / 2) below x, a value on a midpoint taking the lower
// code; found by binary search over the increasing midpoints (four comparisons).
__device__ __forceinline__ uint32_t nf4_code_of(float x, const float (&mid)[15]) {
  uint32_t q = x > mid[7] ? 8u : 0u;
  q += x > (q ? mid[11] : mid[3]) ? 4u : 0u;
  const float t2 = (q & 8u) ? ((q & 4u) ? mid[13] : mid[9]) : ((q & 4u) ? mid[5] : mid[1]);
  q += x > t2 ? 2u : 0u;
  const float t10 = (q & 2u) ? ((q & 4u) ? mid[6] : mid[2]) : ((q & 4u) ? mid[4] : mid[0]);
  const float t11 = (q & 2u) ? ((q & 4u) ? mid[14] : mid[10]) : ((q & 4u) ? mid[12] : mid[8]);
  return q + (x > ((q & 8u) ? t11 : t10) ? 1u : 0u);
}

}  // namespace wp
