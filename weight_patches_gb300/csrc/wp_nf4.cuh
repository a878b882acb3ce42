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

#include "wp_ptx.cuh"

namespace wp {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four 4-bit codes -> four bf16 values from a 16-entry table split into byte planes:
// lo[j] / hi[j] hold the low / high bytes of entries 4j..4j+3.  `codes` is 16 bits of the
// packed stream as stored (byte k: element 2k in the high nibble), so its nibbles, low
// to high, are the codes of elements 1, 0, 3, 2.  Each plane is looked up in both
// half-tables (3-bit byte selects); a fourth permute keeps, per byte, the half the code's
// bit 3 points at; the last two permutes interleave the planes back into element order.
// Returns the words holding elements (0, 1) and (2, 3).
__device__ __forceinline__ void lookup4(uint32_t codes, const uint32_t (&lo)[4], const uint32_t (&hi)[4],
                                        uint32_t& out01, uint32_t& out23) {
  const uint32_t sel3 = codes & 0x7777u;
  const uint32_t pick = 0x3210u | ((codes >> 1) & 0x4444u);     // byte i from the upper half-table if code >= 8
  const uint32_t l = prmt(prmt(lo[0], lo[1], sel3), prmt(lo[2], lo[3], sel3), pick);
  const uint32_t h = prmt(prmt(hi[0], hi[1], sel3), prmt(hi[2], hi[3], sel3), pick);
  out01 = prmt(l, h, 0x4051u);
  out23 = prmt(l, h, 0x6273u);
}

// 32 consecutive elements of one 64-element block: half `hh` of row `r` of the tile.
// `codes16` points at the half's 16 code bytes, `am` is the block's scale, `lv` the 16
// levels, `tile` the shared-memory address of the tile.
__device__ __forceinline__ void nf4_dequant_half_row(const uint8_t* codes16, float am, const float (&lv)[16],
                                                     uint32_t tile, int r, int hh) {
  // table: entries 2k, 2k+1 packed in e[k]; byte planes lo/hi of entries 4j..4j+3
  uint32_t e[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) e[k] = pack_bf16x2(lv[2 * k] * am, lv[2 * k + 1] * am);
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    lo[j] = prmt(e[2 * j], e[2 * j + 1], 0x6420u);
    hi[j] = prmt(e[2 * j], e[2 * j + 1], 0x7531u);
  }
  const uint4 cw4 = *reinterpret_cast<const uint4*>(codes16);
  const uint32_t cwords[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
  const uint32_t dst = tile + r * 128;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    // 4 bytes = 8 codes of consecutive elements
    const uint32_t c = cwords[u];
    uint32_t o0, o1, o2, o3;
    lookup4(c & 0xFFFFu, lo, hi, o0, o1);
    lookup4(c >> 16, lo, hi, o2, o3);
    const int unit = hh * 4 + u;                    // 16-byte unit = 8 elements
    st_shared_v4(dst + ((unit ^ (r & 7)) * 16), o0, o1, o2, o3);
  }
}

// All 64 elements of one block: row `r` of the tile, one table for the 64 codes.
__device__ __forceinline__ void nf4_dequant_row(const uint8_t* codes32, float am, const float (&lv)[16],
                                                uint32_t tile, int r) {
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
    const uint4 cw4 = *reinterpret_cast<const uint4*>(codes32 + half * 16);
    const uint32_t cwords[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t c = cwords[u];
      uint32_t o0, o1, o2, o3;
      lookup4(c & 0xFFFFu, lo, hi, o0, o1);
      lookup4(c >> 16, lo, hi, o2, o3);
      const int unit = half * 4 + u;
      st_shared_v4(dst + ((unit ^ (r & 7)) * 16), o0, o1, o2, o3);
    }
  }
}

}  // namespace wp
