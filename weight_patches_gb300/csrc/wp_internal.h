// wp_internal.h -- launch descriptors shared by the C-ABI front (wp_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "weight_patches.h"

namespace wp {

// ------------------------------------------------------------------ tensor-core path
// A CTA pair (cluster of 2) computes a 256 x 256 output tile: each CTA owns 128 token
// rows (its TMEM lanes) and holds half of the weight tile's 256 rows as MMA operand.
constexpr int kBM = 128;            // token rows per CTA (TMEM lanes)
constexpr int kPairM = 256;         // token rows per CTA pair
constexpr int kBN = 256;            // output columns per tile (TMEM columns per buffer)
constexpr int kBK = 64;             // K per pipeline stage (one 128-byte swizzle atom)
constexpr int kMaxAd = 8;           // bf16 adapters per call (all groups)
constexpr int kMaxAd32 = 4;         // fp32 adapters per call
constexpr int kMaxGroups = 8;
constexpr int kHCols = 256;         // TMEM columns available for X A^T (one buffer)
constexpr int kATileBytes = kBM * kBK * 2;      // 16 KiB: this CTA's X rows
constexpr int kBHalfBytes = 128 * kBK * 2;      // 16 KiB: this CTA's half of a B tile
constexpr int kStgBytes = kBM * 128;            // output staging: 128 rows x 128 bytes
constexpr int kTcThreads = 192;     // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
// 4-bit W: warp 0 TMA, warp 1 MMA (warps 2..3 idle), warps 4..7 epilogue, warps 8..23
// dequantisation in two groups of 8 warps that take alternate K steps
constexpr int kTcThreadsNF4 = 768;
// 4-bit W: a pair tile covers 2 x 256 token rows (two accumulators of 256 TMEM columns,
// one buffer), so every dequantised weight tile feeds two MMAs
constexpr int kMHalvesNF4 = 2;
constexpr int kRawBytes = 128 * 32;             // 4-bit codes of 128 rows x 64 K per stage
constexpr int kAmBytes = 128 * 4 * 4;           // block scales of 128 rows x 4 K steps
constexpr int kAmBytesMN = 64 * 4 * 4;         // W stored [in, out]: 64 K rows x a 4-block box
constexpr int kCodeSlotBytes = kRawBytes + kAmBytes;
constexpr int kMaxCodeSlots = 8;
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 227 * 1024;

struct TcAdapter {
  int group;       // column group this adapter belongs to
  int rank;        // r
  int rpad16;      // r rounded up to 16 (MMA N for X A^T and K extent of the 2nd GEMM); for
                   // an FP32 adapter carried as bf16 pieces, 6 * rp (the width of its H~)
  int pw;          // rank-pass columns: rpad16, or 3 * rp for an FP32 adapter (X a_i^T, i=1..3)
  int split3;      // FP32 adapter as three bf16 pieces (rp = pw / 3 ranks per piece)
  int hoff;        // rank columns [0, pw/2) of this adapter: TMEM column = packed A row
  int hoff2;       // rank columns [pw/2, pw): TMEM column = packed A row (htot/2 + hoff)
  int toff;        // first column of this adapter's H~ (multiple of 16)
  int nchunks;     // ceil(r / 64)
  int hout_off;    // column of this adapter's s * X A^T in TcParams::h_out (if stored)
  int pass;        // rank pass whose MMA computes this adapter's X A^T (hoff, hoff2 within it)
  float s;         // combined scale, fp32
};

struct TcAdapter32 {
  int group;
  int rank;
  int h_off;             // column offset in the s * X A^T fp32 workspace matrix
  int ldb;               // row pitch of B (elements)
  int vec4;              // rank, pitch, offset and base all allow 16-byte loads
  const float* B;        // [out_g, r] fp32
};

struct TcParams {
  int T, K, N;                 // tokens, in_features, total out_features
  int out_g, G, nt_g;          // group width, groups, N-tiles per group
  int m_tiles, total_tiles, k_blocks;   // m_tiles counts tile rows (256 << m_shift token rows)
  int r_blocks;                // 256-row blocks: one rank item and one flag each
  int m_shift;                 // 4-bit W: 1 (a tile is two 256-row halves that share the
                               // dequantised weight tile), else 0
  int w_mn;                    // W stored [in, out] (the backward's dX pass reads the forward's
                               // W as it is): weight tiles are MN-major MMA operands; a 4-bit
                               // W's codes are [in rows, out / 2 bytes], blocks of 64 along out
  int rlead;                   // rank items run this many rounds of tiles ahead of their tiles
  int rank_first;              // every pair opens with its first rank item
  int step_j, step_g, step_m;  // the number of pairs in (row block, group, column tile) digits
                               // (set by the launcher)
  int has_base;
  int n_ad;                    // adapters on the tensor cores (bf16, or FP32 as pieces)
  int ad_begin[kMaxGroups + 1];
  int htot;                    // rank-item MMA width: twice the larger CTA half (<= 256)
  int npass;                   // rank passes per 256-row block: the adapters' rank columns in
                               // groups of at most 256 (htot wide each), one rank item per pass
  uint32_t flag_target;        // a block's H~ rows are complete when its flag reaches this
                               // (2 npass: one release per CTA per pass)
  int stages;
  int stage_bytes;             // bf16 W: 32 KiB; 4-bit W: 2 x 16 KiB X + 16 KiB dequantised W
  int code_slots;              // 4-bit W: ring of [4 KiB codes | 2 KiB block scales] slots, loaded
                               // ahead of the stages
  const float* absmax;         // 4-bit W: [N * K / 64] fp32 block scales
  int am_tma;                  // 4-bit W: block scales arrive by TMA with the codes
  float nf4_code[16];          // 4-bit W: the NormalFloat levels
  TcAdapter ad[kMaxAd];
  uint16_t* hq;                // [T, hq_ld] bf16: H~ = s X A^T of every adapter (toff columns)
  int hq_ld;
  uint32_t* flags;             // [r_blocks]: flag_target once both CTAs of every pass wrote the
                               // block's H~ rows
  int n_ad32;                  // fp32 adapters (epilogue FFMA)
  TcAdapter32 ad32[kMaxAd32];
  float* h_out;                // optional [T, h_out_ld] fp32: s * X A^T of the bf16 adapters
  int h_out_ld;
  const float* h32;            // [T, h32_cols] fp32: s * X A^T of the fp32 adapters
  int h32_cols;
  const void* bias;            // [N] or null
  int bias_f32;
  int bias_vec;                // bias 16-byte aligned: 16-byte loads of full sub-chunks
  // merge: the accumulator times acc_scale plus a per-element residual R [T, N] (bf16 or
  // fp32, may be Y itself: each element is read by the thread that writes it), in fp32
  float acc_scale;
  const void* resid;
  long long ld_resid;
  int resid_f32;
  void* Y;
  long long ldy;
  int y_f32;
  // SwiGLU front half: every tile holds 128 gate columns (CTA 0's weight rows) and the same
  // 128 up columns (CTA 1's); Y is h = silu(e) g [T, out_g]; eg, when set, receives the
  // bf16 e | g [T, 2 out_g] that the backward needs
  int swiglu;
  uint16_t* eg;
  long long ld_eg;
  unsigned long long timeout_ns;
};

struct TcMaps {
  CUtensorMap x;
  CUtensorMap w;
  CUtensorMap y;                 // output, 128-byte swizzled boxes of 128 rows
  CUtensorMap wq;                // 4-bit W codes: [N rows, K/2 bytes], boxes of 128 x 32 bytes
                                 // (w_mn: [K rows, N/2 bytes], boxes of 64 x 64 bytes)
  CUtensorMap am;                // 4-bit W block scales: [N rows, K/64] fp32, boxes of 128 x 4
                                 // (w_mn: [K rows, N/64], boxes of 64 x 4)
  CUtensorMap hq;                // H~ [T rows, hq_ld], boxes of 128 rows x 64 ranks
  CUtensorMap hq32;              // the same with boxes of 128 rows x 32 ranks (64-byte swizzle)
  CUtensorMap ap;                // packed A rows [npass htot, K]: boxes of htot/2 rows x 64
  CUtensorMap b[kMaxAd];
  CUtensorMap b32[kMaxAd];       // B with boxes of 128 rows x 32 ranks (64-byte swizzle)
};

// Number of CTA pairs that can be resident at once for this shared-memory size.
// SwiGLU backward, elementwise: from the gradient at h and the saved e | g, the gradients
// at e and g (written as de | dg, the stacked gate/up output gradient) and h itself
struct SwigluBwdParams {
  long long T, F;
  const uint16_t* dh; long long ld_dh;
  const uint16_t* eg; long long ld_eg;
  uint16_t* deg; long long ld_deg;
  uint16_t* h; long long ld_h;       // optional
};
int launch_swiglu_bwd(const SwigluBwdParams& q, cudaStream_t stream);

// ------------------------------------------------------------------ small-token path
// T <= 64 tokens: Y^T = W X^T with the weight rows as the 128-row MMA operand and the
// tokens (rounded up to 16) as its width, single-CTA tcgen05; the adapters' A rows
// (laid out one adapter after another at 16-aligned offsets) ride as extra row blocks, so X A^T comes
// out of the same pass.  K is split so that the units fill the SMs; a second kernel sums
// the splits, forms H~ = bf16(s X A^T), adds the bias and H~ B^T and rounds once.
constexpr int kSkinnyMaxT = 64;
constexpr int kSkinnyThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kSkinnyThreadsNF4 = 704;    // + warps 6..21 dequantisation (four groups of 4)
constexpr int kSkinnyXBytes = kSkinnyMaxT * 128;   // X rows of a stage (64 rows x 64 K bf16)
constexpr int kWTileBytesSkinny = 128 * 64 * 2;   // 128 weight (or A) rows x 64 K, bf16
constexpr int kSkinnyCodeSlots = 16;      // 4-bit W: most slots of the codes ring

struct SkinnyParams {
  int T, Tp;                   // tokens and the MMA width (T rounded up to 16)
  int K, k_blocks;
  int N;                       // output columns: weight rows, and the first A-row column
  int nbW, nbA;                // 128-row blocks of W and of the A rows
  int R16;                     // A rows: adapter i at rows [a_off[i], a_off[i] + ceil16(r_i))
  int n_ad;
  int a_off[kMaxAd + 1];       // a_off[n_ad] = R16
  int splits, kb_per_split, units;
  int kkb;                     // 64-wide K blocks per step (1, or 2 with a 4-bit W); kb_per_split
                               // is a multiple of it
  int am_tma;
  const float* absmax;
  float nf4_code[16];
  float* part;                 // [splits][T][ldp] fp32: W rows, then the A rows at N
  long long ldp;
  int stages, stage_bytes;     // 4-bit W: 4 or 8 stages (stage s written by group s % 4)
  int code_slots;              // 4-bit W: slots of the codes ring (0 for bf16)
  int* status;
  unsigned long long timeout_ns;
};

struct SkinnyMaps {
  CUtensorMap x, w, wq, am;
  CUtensorMap a[kMaxAd];       // adapter A [r, in], boxes of 16 rows x 64 K (rows past r read 0)
};

struct SkinnyReduceParams {
  int T, N, out_g, R16, splits, has_w;
  long long ldp;
  const float* part;
  const void* bias;
  int bias_f32;
  int n_ad;
  struct Ad {
    int group, rank, toff;
    int vec;                   // B rows 16-byte aligned: loaded 8 ranks at a time
    float s;
    const uint16_t* B;
    long long ldb;
  } ad[kMaxAd];
  void* Y;
  long long ldy;
  int y_f32;
};

int launch_skinny(const SkinnyMaps& maps, const SkinnyParams& p, size_t smem_bytes, bool nf4,
                  cudaStream_t stream);
int launch_skinny_reduce(const SkinnyReduceParams& q, cudaStream_t stream);
int skinny_grid_ctas(size_t smem_bytes, bool nf4);

// One to four tokens on the CUDA cores (wp_gemv.cu): each warp streams 32 weight rows, one per
// lane, through its own ring of TMA stages (4-bit W: 256 K elements of 32 rows, 4 KiB of codes
// in the 128-byte swizzle and 512 B of block scales; bf16 W: 64 K elements of 32 rows, 4 KiB in
// the same swizzle); X of the block's K range
// waits in shared memory as bf16.  It writes the partial sums skinny_reduce_kernel reads: the
// W rows at [split][t][n], the adapters' A rows at [split][t][N + a_off + j].
constexpr int kGemvMaxT = 4;
constexpr int kGemvWarps = 4;
constexpr int kGemvStages = 3;
constexpr int kGemvMaxSplits = 32;
constexpr int kGemvStageK = 256;
constexpr int kGemvCodeBytes = 32 * kGemvStageK / 2;   // 4 KiB
constexpr int kGemvAmBytes = 32 * kGemvStageK / 64 * 4;  // 512 B
constexpr int kGemvXBudget = 16384;                      // bf16 X elements a block holds (32 KiB)
// the plain-load 4-bit kernel for one token: 2048-element K splits, 8 warps a block
constexpr int kGemvLdSlice = 2048;
constexpr int kGemvLdWarps = 8;

struct GemvParams {
  int T, K, N;
  int splits, ks_len;          // K elements per split (a multiple of 256; the last one shorter)
  int ngW;                     // 32-row groups of W
  int R16;                     // A rows, each adapter padded to 16 (rows past the rank write 0)
  int n_ad;
  int a_off[kMaxAd + 1];
  int rank[kMaxAd];
  const uint16_t* A[kMaxAd];
  long long lda[kMaxAd];
  float nf4_code[16];
  const uint16_t* X;
  long long ldx;
  float* part;                 // [splits][T][ldp]
  long long ldp;
  int* status;
  unsigned long long timeout_ns;
};

struct GemvMaps {
  CUtensorMap w;               // bf16 W [N, K], boxes of 64 x 32 rows, 128-byte swizzle
  CUtensorMap wq;              // codes [N, K/2] u8, boxes of 128 B x 32 rows, 128-byte swizzle
  CUtensorMap am;              // block scales [N, K/64] fp32, boxes of 4 x 32 rows
};

size_t gemv_smem_bytes(int T, int ks_len);
int gemv_blocks_per_sm(int T, bool nf4, size_t smem_bytes);
int launch_gemv(const GemvMaps& maps, const GemvParams& p, bool nf4, int grid, size_t smem_bytes,
                cudaStream_t stream);
int launch_gemv_ld(const GemvParams& p, const void* codes, const float* absmax, int grid, cudaStream_t stream);
int* tc_status_ptr();

int tc_max_pairs(size_t smem_bytes, bool nf4);
int launch_tc_fwd(const TcMaps& maps, const TcParams& p, int grid, size_t smem_bytes,
                  cudaStream_t stream, bool nf4);
int tc_fwd_status(int reset);

// ------------------------------------------------------------------ fp32 CUDA-core path
struct F32Adapter {
  const void* A; int a_dtype; long long lda;   // [r, in]
  const void* B; int b_dtype; long long ldb;   // [out, r]
  int rank;
  float s;
};

struct F32Params {
  int T, K, N;
  const void* X; int x_dtype; long long ldx;
  const void* W; int w_dtype; long long ldw;   // may be null
  const void* bias; int bias_dtype;            // may be null
  void* Y; int y_dtype; long long ldy;
  int n_ad;
  F32Adapter ad[kMaxAd + kMaxAd32];
  int col_begin[kMaxAd + kMaxAd32];            // output column window of each adapter
  int col_end[kMaxAd + kMaxAd32];
};

// H: [T, h_cols] fp32 = s * X A^T of the adapters, in adapter order (rank_proj_kernel).
int launch_f32_linear(const F32Params& p, const float* H, int h_cols, cudaStream_t stream);

// s * X A^T of a list of adapters, written to an fp32 [T, h_cols] workspace matrix.
struct H32Params {
  int T, K;
  const void* X; int x_dtype; long long ldx;
  int x_vec;                       // X rows 16-byte aligned (vector loads allowed)
  int n_ad;
  const void* A[kMaxAd + kMaxAd32]; long long lda[kMaxAd + kMaxAd32];
  int a_dtype[kMaxAd + kMaxAd32];
  int a_vec[kMaxAd + kMaxAd32];    // 4-element runs of A aligned for one vector load
  int rank[kMaxAd + kMaxAd32], h_off[kMaxAd + kMaxAd32];
  float s[kMaxAd + kMaxAd32];
  float* H; int h_cols;
};
int launch_h32(const H32Params& p, cudaStream_t stream);

// Operands of the rank item, packed once per call.  Ap [htot, ldk] bf16 holds every
// adapter's A rows as the pair's MMA reads them: rows [0, htot/2) feed CTA 0 (rank columns
// [0, pw/2) of each adapter, from row hoff), rows [htot/2, htot) feed CTA 1 (columns
// [pw/2, pw), from row hoff2).  A bf16 adapter's column j is its row j (zero past r).  An
// FP32 adapter (A [r, K], B [out, r]) rides as bf16 pieces x = x1 + x2 + x3, each the
// rounding of what the previous ones leave: its column i * rp + j is piece i + 1 of its
// row j, and its B becomes Bs [out, 6 rp] = [b1 b2 b1 b3 b2 b1].
struct PackAdapter {
  const void* A; long long lda; int dtype;
  int r, pw, rp, hoff, hoff2, split3;   // hoff, hoff2: packed rows (pass q's rows start at q htot)
  const float* B; long long ldb; int out; uint16_t* Bs;   // FP32 adapters only
};
struct PackParams {
  int n_ad, K, ldk, half;        // half = htot / 2: the packed A rows are npass blocks of htot rows
  int npass;
  int rows_total;                // set by launch_rank_pack
  uint16_t* Ap;
  uint32_t* flags;               // row-block flags of the forward kernel, cleared here
  int n_flags;
  PackAdapter ad[kMaxAd];
};
int launch_rank_pack(const PackParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ backward helpers
struct NF4Table {
  float level[16];
};
// Token contractions for the backward's dA / dB on the tensor cores (wp_tokgemm.cu):
// part[split][m][n] = sum over the split's tokens t of A[t, m] B[t, n]
struct TokGemmParams {
  int T, M, N;                 // tokens, rows of D (A's columns), columns (128 or 256)
  int m_tiles, splits, kb_per_split, k_blocks, units;
  float* part;                 // [splits][M][N] fp32
  int stages;
  int* status;
  unsigned long long timeout_ns;
};
struct TokGemmMaps {
  CUtensorMap a, b;            // A [T, M], B [T, N]: boxes of 64 tokens x 64 columns, 128-byte swizzle
};
// column map of the rank-wide operand's bf16 pieces (see launch_pieces)
struct TokPieceMap {
  int G, R16;
  int roff16[kMaxGroups], off[kMaxGroups], r[kMaxGroups];
};
int tokgemm_max_pairs(size_t smem_bytes);
int launch_tokgemm(const TokGemmMaps& maps, const TokGemmParams& p, int pairs, size_t smem_bytes,
                   cudaStream_t stream);
int launch_pieces(const float* src, long long ld, int T, int N, const TokPieceMap& pm, uint16_t* dst,
                  cudaStream_t stream);
int launch_tok_finish(const float* part, int M, int N, int splits, int R16, int roff16, int r, int row0, int rows,
                      float scale, float* out, long long ldo, bool transposed, cudaStream_t stream);

// LoRA merge into a 4-bit weight (wp_merge.cu): W_eff as fp32, and the requantisation
// Legacy adapter bias vectors folded into one per-column vector (piper-offload docs,
// "LoRA merge": older adapters' lora_B.bias):  v[n] = fl32(bias[n]) and then, in order,
// v[n] = fl32(v[n] + fl32(s_p * vec_p[n - col0_p])) for each adapter p whose columns
// [col0_p, col0_p + cols_p) hold n.  out != nullptr: v goes there in fp32 (the forward's
// epilogue bias); else it is rounded to the bias's own dtype and written back (the merge).
struct BiasFoldParams {
  float* out;
  void* bias;                  // [N] or nullptr (forward only)
  int bias_dtype;
  int N, n;
  struct Vec {
    const void* v;
    int dtype;
    float s;
    int col0, cols;
  } ad[kMaxAd + kMaxAd32];
};
int launch_bias_fold(const BiasFoldParams& p, cudaStream_t stream);

// One merge pass on 128 x 128 output tiles, a CTA each: Y = fl32(s * acc + R) with
// acc = P Q^T, P [rows, r] and Q [cols, r] bf16 K-major (r <= kMergeTileMaxK * 64), R and Y
// [rows, cols] bf16 or fp32 (R may be Y), cols % 8 == 0, 16-byte aligned rows.
constexpr int kMergeTileMaxK = 4;
struct MergeTileParams {
  int rows, cols, nk;          // output shape; 64-wide K blocks of r
  int nt;                      // tile columns: 64, 128 or 256 (the Q box's rows)
  int staged;                  // R and Y of one dtype (nt 64 or 128): R in and Y out by TMA
  float s;
  const void* R;
  long long ldr;
  int r_f32;
  void* Y;
  long long ldy;
  int y_f32;
  int* status;
  unsigned long long timeout_ns;
};
struct MergeTileMaps {
  CUtensorMap p, q;            // boxes of 64 K x 128 (P) / nt (Q) rows, 128-byte swizzle
  CUtensorMap r, y;            // staged: boxes of 128 bytes x 128 rows, 128-byte swizzle
};
int launch_merge_tile(const MergeTileMaps& maps, const MergeTileParams& p, cudaStream_t stream);

// A whole 4-bit merge in one pass (ranks up to kMergeTileMaxK * 64), a thread per 64-element
// block: W_eff = bf16(fl32(level[q]) * absmax) in registers, u = fl32(s_p * acc_p + u) for
// each adapter in call order (acc_p = B_p A_p on the tensor cores), then the block
// requantised as nf4_requant_kernel does and written in place.  Two forms: one CTA per SM on
// 128 x 256 tiles whose codes and scales move by TMA (merge_nf4_wide_plan), else persistent
// CTAs on 128 x 64 tiles with plain loads and stores.
// The 4-bit code of x in [-1, 1] by cells of width 1/16: cell c = floor(16 x) + 16 holds at
// most one level midpoint (they are at least 0.08 apart), so the code is base[c] (the
// midpoints below the cell) plus one when x exceeds the cell's next midpoint next_mid[c] (the
// smallest midpoint at or above the cell's start; 2 when none).
constexpr int kCodeCells = 33;            // 32 cells of width 1/16 over [-1, 1), and x = 1
struct NF4Cells {
  float next_mid[kCodeCells];
  int base[kCodeCells];
};
bool nf4_code_cells(const NF4Table& tab, NF4Cells* cells);
// The stochastic re-encoding's cells (same width): per cell the first level at or above its
// start (2 when none), that level's index, the level before it (-2 when none) and the one after
// it (2 when none).  False if a cell holds two levels (the NF4 levels are at least 0.079 apart).
struct NF4LevelCells {
  float next_l[kCodeCells];
  int base[kCodeCells];
  float prev_l[kCodeCells];
  float after_l[kCodeCells];
};
bool nf4_level_cells(const NF4Table& tab, NF4LevelCells* cells);

struct MergeNF4Params {
  int rows, cols;              // W [rows, cols], cols % 64 == 0
  uint8_t* codes;              // [rows, cols / 2], rewritten
  float* absmax;               // [rows * cols / 64], rewritten
  NF4Table tab;
  NF4Cells cells;              // the code search by cells (nf4_code_cells)
  int hold;                    // test hook (lora_debug_hold_flags): the last job's MMAs are not issued
  int stochastic;              // the stochastic re-encoding, keyed by seed_lo, seed_hi
  uint32_t seed_lo, seed_hi;
  NF4LevelCells lcells;        // its cells (nf4_level_cells)
  int n, nk_max;               // adapters (non-zero s), the most K blocks of any of them
  int wide;                    // the 256-column form (merge_nf4_wide_plan), with its plan:
  int s_a, s_c;                //   A_p stages and code stages,
  int kbox[kMaxAd];            //   each adapter's K rows per A_p box (r rounded up to 16, at most 64),
  int boff[kMaxAd];            //   its first B_p box in a group buffer,
  int a_bytes, b_bytes;        //   one A_p stage, one group's B_p boxes
  int nk[kMaxAd];
  float s[kMaxAd];
  int* status;
  unsigned long long timeout_ns;
};
struct MergeNF4Maps {
  CUtensorMap p[kMaxAd];       // B_p [rows, r_p]: boxes of 64 K x 128 rows
  CUtensorMap q[kMaxAd];       // A_p^T [cols, r_p]: boxes of 64 K x 64 rows; wide: A_p [r_p, cols] itself,
                               // boxes of 64 columns x kbox rows
  CUtensorMap codes;           // wide: codes [rows, cols / 2] bytes, boxes of 128 B x 128 rows, 128-byte swizzle
  CUtensorMap am;              // wide: absmax [rows, cols / 64] fp32, boxes of 4 x 128 rows
};
// The wide form applies (columns a multiple of 256, shared memory for its stages) to adapters
// of these ranks: fills p's plan (kbox, nk, boff, a_bytes, b_bytes, s_a, s_c).
bool merge_nf4_wide_plan(const int* ranks, int n, long long cols, MergeNF4Params* p);
int launch_merge_nf4(const MergeNF4Maps& maps, const MergeNF4Params& p, cudaStream_t stream);

int launch_nf4_to_f32(const void* codes, const float* absmax, long long numel, const NF4Table& tab, float* U,
                      cudaStream_t stream);
int launch_nf4_requant(const float* U, long long numel, const NF4Table& tab, void* codes, float* absmax,
                       cudaStream_t stream);
// The same with the stochastic re-encoding (U's linear index is the element's logical index).
int launch_nf4_requant_stochastic(const float* U, long long numel, const NF4Table& tab, void* codes,
                                  float* absmax, uint64_t seed, cudaStream_t stream);
int launch_transpose_bf16(const void* src, long long ld_s, int R, int C, void* dst, long long ld_d,
                          cudaStream_t stream);

// ------------------------------------------------------------------ unfused chain (exact tier)
// One elementwise step of the chain on a [T, N] bf16 matrix Y (N % 8 == 0, 16-byte aligned
// rows): kChainScale: Y = bf16(Y * c); kChainAdd: Y = bf16(Y + d), d [T, N] bf16 or fp32.
// Each result is the correctly rounded value of the exact product or sum (wp_chain.cu).
enum { kChainScale = 0, kChainAdd = 1 };
struct ChainParams {
  int mode;
  long long T, N;
  uint16_t* Y; long long ldy;
  const void* d; long long ldd; int d_f32;
  float c;
};
int launch_chain(const ChainParams& q, cudaStream_t stream);

// ------------------------------------------------------------------ dense patch
int launch_dense_patch(void* param, int param_dtype, const void* payload, int payload_dtype,
                       long long n, int kind, float k, cudaStream_t stream);

// ------------------------------------------------------------------ NF4 table (host)
void nf4_codebook_host(float out[16]);

// ------------------------------------------------------------------ misc
void set_last_cuda_error(cudaError_t e);
int device_sm_count();

}  // namespace wp
