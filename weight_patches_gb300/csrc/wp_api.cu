// wp_api.cu -- the C ABI: argument checks, combined scales, tensor maps, dispatch.
//
// Every entry point validates on the host and launches nothing when it rejects a
// call.  The library never allocates device memory and never synchronises; all work
// is enqueued on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "wp_internal.h"

namespace wp {

namespace {
thread_local std::string g_last_error;

// How long a bounded device wait spins before its kernel gives up (lora_set_wait_limit), and
// the test hook that holds the fused forward's row-block flags one release short and keeps
// the one-pass 4-bit merge's last MMAs back (lora_debug_hold_flags).
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_hold_flags{0};
unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [outer, inner] matrix with row pitch ld
// (elements), 128-byte swizzled boxes of {box_inner, box_outer}; out-of-range
// elements read as zero.
// swizzle: 128 or 64 (the box's inner extent must then be 128 or 64 bytes) or 0 (none)
int make_map(CUtensorMap* m, int dtype, const void* ptr, long long inner, long long outer,
             long long ld, int box_inner, int box_outer, int swizzle = 128) {
  auto fn = encode_fn();
  if (!fn) {
    g_last_error = "cuTensorMapEncodeTiled unavailable";
    return WP_ERR_CUDA;
  }
  const int esz = dtype == WP_FP32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dtype == WP_FP32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                  : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    g_last_error = buf;
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

// 2-D byte tensor map (4-bit codes, two per byte) without swizzle: boxes of
// {box_inner bytes, box_outer rows}, rows box_inner bytes apart in shared memory.
// Byte tensor map; swizzle 32 or 64 stores each box row's 16-byte units swizzled like
// the bf16 tiles (the 4-bit codes, so that a quarter-warp's rows read different banks).
int make_map_u8(CUtensorMap* m, const void* ptr, long long inner_bytes, long long outer,
                long long ld_bytes, int box_inner, int box_outer, int swizzle = 0) {
  auto fn = encode_fn();
  if (!fn) {
    g_last_error = "cuTensorMapEncodeTiled unavailable";
    return WP_ERR_CUDA;
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner_bytes), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                  : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                  : swizzle == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                  : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled (u8) failed (%d)", static_cast<int>(r));
    g_last_error = buf;
    return WP_ERR_CUDA;
  }
  return WP_OK;
}

int make_map_bf16(CUtensorMap* m, const void* ptr, long long inner, long long outer, long long ld,
                  int box_inner, int box_outer) {
  return make_map(m, WP_BF16, ptr, inner, outer, ld, box_inner, box_outer);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A matrix of no rows needs no memory: its pointers may be null (an empty batch).
bool valid_input(const wp_mat* m, bool allow_nf4) {
  if (!m) return false;
  if (m->rows < 0 || m->cols <= 0) return false;
  if (!m->data && m->rows != 0) return false;
  if (m->dtype == WP_NF4) {
    if (!allow_nf4 || (!m->absmax && m->rows != 0)) return false;
    return true;
  }
  if (m->dtype != WP_BF16 && m->dtype != WP_FP32) return false;
  return m->ld >= m->cols;
}

bool valid_output(const wp_out* y) {
  if (!y || (!y->data && y->rows != 0)) return false;
  if (y->dtype != WP_BF16 && y->dtype != WP_FP32) return false;
  return y->rows >= 0 && y->cols > 0 && y->ld >= y->cols;
}

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

struct FwdPlan {
  bool tc = false;        // tensor-core path
  int rank32_total = 0;   // fp32 adapters' total rank (tensor-core path)
  int rank_all = 0;       // all adapters' total rank (fp32 path)
  size_t split_bytes = 0; // bf16 B pieces of the fp32 adapters (tensor-core path)
  int htilde_cols = 0;    // H~ columns, at most (tensor-core path)
  int rank_cols = 0;      // rank-item columns, at most (tensor-core path)
  size_t pack_bytes = 0;  // packed A rows of the rank item (tensor-core path)
  size_t skinny_bytes = 0;  // small-token path: packed A rows + K-split partial sums
  size_t fold_bytes = 0;  // the fp32 bias with the adapters' legacy vectors folded in
};

// Small-token path (T <= 64, bf16 X and adapters, bf16 or 4-bit W): the fp32 partial sums
// [splits, T, N + R16].  K is split so that the
// (row block, K range) units spread evenly over the SMs, with at least two K steps each.
struct SkinnyPlan {
  bool use = false;
  int Tp = 0, nbW = 0, nbA = 0, R16 = 0, splits = 1, kbps = 1, units = 0, k_blocks = 0;
  int kkb = 1;                 // 64-wide K blocks per pipeline step
  long long N = 0;
  size_t part_bytes = 0;
  // one to four tokens against a weight, K a multiple of 256: the CUDA-core kernel (wp_gemv.cu)
  bool gemv = false;
  int g_splits = 1, g_ks_len = 0, g_grid = 0;
  size_t g_smem = 0;
  // one token against a 4-bit weight, K a multiple of 2048: the plain-load kernel instead
  bool g_ld = false;
};

// The split of K for the CUDA-core small-token kernel: each block holds the fp32 X of its
// split, so a split is at most kGemvXBudget / T elements; among those, the split whose
// busiest warp streams the fewest elements (32-row groups x split length), fewer splits on a
// tie.  The grid is a multiple of the splits.
bool plan_gemv(long long T, long long K, long long N, bool nf4, SkinnyPlan* sp) {
  const int kb = static_cast<int>(K / kGemvStageK);
  const int ngW = static_cast<int>((N + 31) / 32);
  const int sms = device_sm_count();
  long long best = -1;
  for (int s_try = 1; s_try <= kGemvMaxSplits && s_try <= kb; ++s_try) {
    const int ks_len = (kb + s_try - 1) / s_try * kGemvStageK;
    if (T * ks_len > kGemvXBudget) continue;
    const int splits = static_cast<int>((K + ks_len - 1) / ks_len);
    const size_t smem = gemv_smem_bytes(static_cast<int>(T), ks_len);
    const int per_sm = gemv_blocks_per_sm(static_cast<int>(T), nf4, smem);
    if (per_sm < 1) continue;
    const int nbs = sms * per_sm / splits;
    if (nbs < 1) continue;
    const long long rounds = (ngW + nbs * kGemvWarps - 1) / (nbs * kGemvWarps);
    const long long cost = rounds * ks_len;
    if (best < 0 || cost < best) {
      best = cost;
      sp->g_splits = splits;
      sp->g_ks_len = ks_len;
      sp->g_grid = nbs * splits;
      sp->g_smem = smem;
    }
  }
  return best >= 0;
}

// It serves 4-bit weights up to 64 tokens; a bf16 weight (or none) only up to 4 tokens:
// beyond that the general path, whose tiles read a bf16 weight without dequantisation,
// measured faster on GB300 (about 22 us against 32-42 us at 16-64 tokens for the 1536-wide
// layers).
constexpr int kSkinnyMaxTBf16 = 4;

bool plan_skinny(const wp_mat* X, const wp_mat* W, const wp_adapter* ad, int n, SkinnyPlan* sp) {
  *sp = SkinnyPlan{};
  const long long T = X->rows, K = X->cols;
  if (T < 1 || T > kSkinnyMaxT || X->dtype != WP_BF16 || K < 1) return false;
  if (!(W && W->dtype == WP_NF4) && T > kSkinnyMaxTBf16) return false;
  if (W && W->dtype != WP_BF16 && W->dtype != WP_NF4) return false;
  if (!W && n < 1) return false;
  int R16 = 0;
  for (int i = 0; i < n; ++i) {
    if (ad[i].A.dtype != WP_BF16 || ad[i].B.dtype != WP_BF16) return false;
    R16 += static_cast<int>((ad[i].A.rows + 15) / 16 * 16);
  }
  if (R16 > kHCols || n > kMaxAd) return false;
  long long N = 0;
  if (W) N = W->rows;
  else for (int i = 0; i < n; ++i) N = std::max<long long>(N, ad[i].B.rows);
  sp->N = N;
  sp->R16 = R16;
  sp->Tp = static_cast<int>((T + 15) / 16 * 16);
  sp->nbW = W ? static_cast<int>((N + 127) / 128) : 0;
  sp->nbA = (R16 + 127) / 128;
  const int rows = sp->nbW + sp->nbA;
  sp->k_blocks = static_cast<int>((K + kBK - 1) / kBK);
  // a 4-bit weight goes two K blocks per step: half the hand-offs between the kernel's
  // roles per byte of weight
  sp->kkb = (W && W->dtype == WP_NF4) ? 2 : 1;
  const int grid = device_sm_count();
  double best = 1e30;
  for (int sp_try = 1; sp_try <= 8; ++sp_try) {
    if (sp_try > 1 && sp->k_blocks / sp_try < 2) break;
    const long long units = static_cast<long long>(rows) * sp_try;
    const double waste = static_cast<double>((units + grid - 1) / grid) * grid / units;
    if (waste < best - 0.02) { best = waste; sp->splits = sp_try; }
  }
  sp->kbps = (sp->k_blocks + sp->splits - 1) / sp->splits;
  sp->kbps = (sp->kbps + sp->kkb - 1) / sp->kkb * sp->kkb;
  sp->splits = (sp->k_blocks + sp->kbps - 1) / sp->kbps;
  sp->units = rows * sp->splits;
  sp->part_bytes = round256(static_cast<size_t>(sp->splits) * T * (N + R16) * 4);
  if (W && T <= kGemvMaxT && K % kGemvStageK == 0 && plan_gemv(T, K, N, W->dtype == WP_NF4, sp)) {
    sp->gemv = true;
    if (W->dtype == WP_NF4 && T == 1 && K % kGemvLdSlice == 0 && K / kGemvLdSlice <= kGemvMaxSplits) {
      // one split per 2048-element slice; two 8-warp blocks per SM over the slices
      sp->g_ld = true;
      sp->g_splits = static_cast<int>(K / kGemvLdSlice);
      sp->g_ks_len = kGemvLdSlice;
      sp->g_grid = std::max(1, 2 * grid / sp->g_splits) * sp->g_splits;
      sp->g_smem = 0;
    }
    sp->part_bytes =
        std::max(sp->part_bytes, round256(static_cast<size_t>(sp->g_splits) * T * (N + R16) * 4));
  }
  sp->use = true;
  return true;
}

// FP32 adapters on the tensor-core path travel as three bf16 pieces per factor: rank
// padded to rp (16), A pieces [3 rp, round8(K)], B pieces [out, 6 rp].
int split_rp(long long r) { return static_cast<int>((r + 15) / 16 * 16); }
size_t split_b_bytes(long long r, long long out) {
  return round256(static_cast<size_t>(out) * 6 * split_rp(r) * 2);
}

// Decide the path from the dtypes alone (the same answer lora_workspace_size gives).
int plan_fwd(const wp_mat* X, const wp_mat* W, const wp_adapter* ad, int n, FwdPlan* plan) {
  plan->tc = X->dtype == WP_BF16 && (!W || W->dtype == WP_BF16 || W->dtype == WP_NF4);
  for (int i = 0; i < n; ++i) {
    const int r = static_cast<int>(ad[i].A.rows);
    plan->rank_all += r;
    if (ad[i].A.dtype == WP_FP32) {
      plan->rank32_total += r;
      plan->split_bytes += split_b_bytes(r, ad[i].B.rows);
      plan->htilde_cols += 6 * split_rp(r);
      plan->rank_cols += 3 * split_rp(r);
    } else {
      plan->htilde_cols += static_cast<int>((r + 15) / 16 * 16);
      plan->rank_cols += static_cast<int>((r + 15) / 16 * 16);
    }
  }
  // packed A rows: one pass of rank_cols rows, or npass passes of at most kHCols rows each;
  // the passes are filled first-fit, so at most one is half empty: npass <= 2 rank_cols /
  // kHCols + 1 (and never more than the adapters)
  size_t pack_rows = static_cast<size_t>(plan->rank_cols);
  if (plan->rank_cols > kHCols)
    pack_rows = static_cast<size_t>(kHCols) * std::min(n, 2 * plan->rank_cols / kHCols + 1);
  plan->pack_bytes = round256(pack_rows * static_cast<size_t>((X->cols + 7) / 8 * 8) * 2);
  SkinnyPlan sp;
  if (plan_skinny(X, W, ad, n, &sp)) plan->skinny_bytes = sp.part_bytes;
  // legacy adapter bias vectors: an fp32 [out] vector ahead of everything else (out bounded
  // by the sum of the adapters' B rows when there is no W)
  bool legacy = false;
  long long nb = W ? W->rows : 0;
  for (int i = 0; i < n; ++i) {
    legacy = legacy || ad[i].bias_B != nullptr;
    if (!W) nb += ad[i].B.rows;
  }
  plan->fold_bytes = legacy ? round256(static_cast<size_t>(nb) * 4) : 0;
  return WP_OK;
}

// Bytes the call needs on its general path (min) and, with the small-token path's on top,
// what lora_workspace_size reports.
size_t fwd_workspace(const wp_mat* X, const FwdPlan& plan, bool min_only = false) {
  const size_t T = static_cast<size_t>(X->rows);
  if (plan.tc) {
    size_t tc = 0;
    if (plan.htilde_cols > 0) {
      const size_t m_tiles = (T + kPairM - 1) / kPairM;
      tc = round256(T * plan.rank32_total * 4) + plan.split_bytes + round256(T * plan.htilde_cols * 2) +
           round256(m_tiles * 4) + plan.pack_bytes;
    }
    return plan.fold_bytes + (min_only ? tc : std::max(tc, plan.skinny_bytes));
  }
  return plan.fold_bytes + (plan.rank_all ? round256(T * plan.rank_all * 4) : 0);
}

// The last CUDA error, recorded for lora_last_cuda_error, as a status.
int record_cuda() {
  set_last_cuda_error(cudaGetLastError());
  return WP_ERR_CUDA;
}

// Small-token path: stream W and the adapters' A rows (one after another at 16-aligned row
// offsets, each from its own tensor map) through skinny_kernel, finish in
// skinny_reduce_kernel.  Arguments are validated by the caller.  Returns
// WP_ERR_UNSUPPORTED (before any CUDA call) when the shapes or alignments do not suit it.
int skinny_impl(const wp_mat* X, const wp_mat* W, const wp_mat* bias, int G, bool grouped,
                const wp_adapter* adapters, int n_adapters, const float* s_of, const wp_out* Y,
                void* workspace, cudaStream_t stream) {
  SkinnyPlan sp;
  if (!plan_skinny(X, W, adapters, n_adapters, &sp)) return WP_ERR_UNSUPPORTED;
  const long long T = X->rows, K = X->cols, N = sp.N;
  const long long out_g = N / G;
  if (!aligned16(X->data) || X->ld % 8) return WP_ERR_UNSUPPORTED;
  if (W && (!aligned16(W->data) || W->ld % 8)) return WP_ERR_UNSUPPORTED;
  for (int i = 0; i < n_adapters; ++i)
    if (!aligned16(adapters[i].A.data) || adapters[i].A.ld % 8) return WP_ERR_UNSUPPORTED;
  const bool nf4 = W && W->dtype == WP_NF4;
  float* part = static_cast<float*>(workspace);

  SkinnyReduceParams q{};
  q.T = static_cast<int>(T); q.N = static_cast<int>(N); q.out_g = static_cast<int>(out_g);
  q.R16 = sp.R16; q.splits = sp.splits; q.has_w = W ? 1 : 0;
  q.ldp = N + sp.R16;
  q.part = part;
  q.bias = bias ? bias->data : nullptr;
  q.bias_f32 = bias && bias->dtype == WP_FP32;
  q.Y = Y->data; q.ldy = Y->ld; q.y_f32 = Y->dtype == WP_FP32;
  SkinnyParams p{};
  int toff = 0;
  for (int i = 0; i < n_adapters; ++i) {
    const wp_adapter& a = adapters[i];
    const int r = static_cast<int>(a.A.rows);
    SkinnyReduceParams::Ad& d = q.ad[q.n_ad++];
    d.group = grouped ? i : 0; d.rank = r; d.toff = toff; d.s = s_of[i];
    d.B = static_cast<const uint16_t*>(a.B.data); d.ldb = a.B.ld;
    d.vec = aligned16(a.B.data) && a.B.ld % 8 == 0;
    p.a_off[i] = toff;
    toff += (r + 15) / 16 * 16;
  }
  p.n_ad = n_adapters;
  p.a_off[n_adapters] = toff;

  if (sp.gemv && (!nf4 || aligned16(W->absmax))) {
    GemvParams g{};
    g.T = static_cast<int>(T); g.K = static_cast<int>(K); g.N = static_cast<int>(N);
    g.splits = sp.g_splits; g.ks_len = sp.g_ks_len;
    g.ngW = static_cast<int>((N + 31) / 32);
    g.R16 = sp.R16;
    g.n_ad = n_adapters;
    for (int i = 0; i < n_adapters; ++i) {
      g.a_off[i] = p.a_off[i];
      g.rank[i] = static_cast<int>(adapters[i].A.rows);
      g.A[i] = static_cast<const uint16_t*>(adapters[i].A.data);
      g.lda[i] = adapters[i].A.ld;
    }
    g.a_off[n_adapters] = toff;
    nf4_codebook_host(g.nf4_code);
    g.X = static_cast<const uint16_t*>(X->data); g.ldx = X->ld;
    g.part = part; g.ldp = q.ldp;
    g.status = tc_status_ptr();
    g.timeout_ns = wait_limit_ns();
    if (!g.status) return record_cuda();
    int rc = WP_OK;
    if (sp.g_ld) {
      rc = launch_gemv_ld(g, W->data, W->absmax, sp.g_grid, stream);
      if (rc != WP_OK) return rc;
      q.splits = sp.g_splits;
      return launch_skinny_reduce(q, stream);
    }
    GemvMaps gm;
    std::memset(&gm, 0, sizeof(gm));
    if (nf4) {
      rc = make_map_u8(&gm.wq, W->data, K / 2, N, K / 2, kGemvStageK / 2, 32, 128);
      if (rc != WP_OK) return rc;
      rc = make_map(&gm.am, WP_FP32, W->absmax, K / 64, N, K / 64, kGemvStageK / 64, 32, /*swizzle=*/0);
    } else {
      rc = make_map_bf16(&gm.w, W->data, K, N, W->ld, kBK, 32);
    }
    if (rc != WP_OK) return rc;
    rc = launch_gemv(gm, g, nf4, sp.g_grid, sp.g_smem, stream);
    if (rc != WP_OK) return rc;
    q.splits = sp.g_splits;
    return launch_skinny_reduce(q, stream);
  }

  SkinnyMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  p.T = static_cast<int>(T); p.Tp = sp.Tp; p.K = static_cast<int>(K); p.k_blocks = sp.k_blocks;
  p.N = static_cast<int>(N);              // the A rows' partial sums start at column N
  p.nbW = sp.nbW; p.nbA = sp.nbA; p.R16 = sp.R16;
  p.splits = sp.splits; p.kb_per_split = sp.kbps; p.units = sp.units; p.kkb = sp.kkb;
  p.part = part; p.ldp = q.ldp;
  p.status = tc_status_ptr();
  p.timeout_ns = wait_limit_ns();
  if (!p.status) return record_cuda();
  // barriers (3 per stage, 1 per code slot, 5 more), the TMEM address, the abort flag and
  // the per-slot copy counts
  const size_t bar_bytes = 1024;
  size_t smem = 0;
  if (nf4) {
    // stage = [kkb W tiles | kkb boxes of Tp X rows]; one K block per step: 8 stages (two
    // per dequantisation group) while the codes ring keeps at least 8 slots, else 4; two
    // K blocks per step: 4 stages, and the block scales come from global memory when a ring
    // of at least 4 slots has no room for them
    const int kkb = sp.kkb;
    p.stage_bytes = kkb * (kWTileBytesSkinny + sp.Tp * 128);
    p.am_tma = (K % 256 == 0 && aligned16(W->absmax)) ? 1 : 0;
    const size_t avail = kSmemLimit - 1024 - bar_bytes;
    if (kkb == 2 && (avail - 4 * static_cast<size_t>(p.stage_bytes)) /
                            (static_cast<size_t>(kkb) * kRawBytes + kAmBytes) < 4)
      p.am_tma = 0;
    const size_t slot = static_cast<size_t>(kkb) * kRawBytes + (p.am_tma ? kAmBytes : 0);
    p.stages = 4;
    if (kkb == 1 && (avail - 8 * static_cast<size_t>(p.stage_bytes)) / slot >= 8) p.stages = 8;
    p.code_slots = static_cast<int>(
        std::min<size_t>(kSkinnyCodeSlots, (avail - static_cast<size_t>(p.stages) * p.stage_bytes) / slot));
    if (p.code_slots < p.stages) return WP_ERR_UNSUPPORTED;
    smem = 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + static_cast<size_t>(p.code_slots) * slot +
           bar_bytes;
  } else {
    p.stage_bytes = kWTileBytesSkinny + kSkinnyXBytes;
    p.stages = std::min<int>(kMaxStages, static_cast<int>((kSmemLimit - 1024 - bar_bytes) / p.stage_bytes));
    p.code_slots = 0;
    smem = 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + bar_bytes;
  }
  if (smem > static_cast<size_t>(kSmemLimit)) return WP_ERR_UNSUPPORTED;
  int rc = make_map_bf16(&maps.x, X->data, K, T, X->ld, kBK, sp.Tp);
  if (rc != WP_OK) return rc;
  if (nf4) {
    rc = make_map_u8(&maps.wq, W->data, K / 2, N, K / 2, sp.kkb * kBK / 2, 128, sp.kkb * 32);
    if (rc != WP_OK) return rc;
    p.absmax = W->absmax;
    if (p.am_tma) {
      rc = make_map(&maps.am, WP_FP32, W->absmax, K / 64, N, K / 64, 4, 128, /*swizzle=*/0);
      if (rc != WP_OK) return rc;
    }
    nf4_codebook_host(p.nf4_code);
  } else if (W) {
    rc = make_map_bf16(&maps.w, W->data, K, N, W->ld, kBK, 128);
    if (rc != WP_OK) return rc;
  }
  for (int i = 0; i < n_adapters; ++i) {
    rc = make_map_bf16(&maps.a[i], adapters[i].A.data, K, adapters[i].A.rows, adapters[i].A.ld, kBK, 16);
    if (rc != WP_OK) return rc;
  }
  rc = launch_skinny(maps, p, smem, nf4, stream);
  if (rc != WP_OK) return rc;
  return launch_skinny_reduce(q, stream);
}

// h_out (optional): s * X A^T of the tensor-core adapters in fp32, [T, h_out_ld], adapters in
// call order.  rank_only: only the rank items run (no output tiles, Y unused and may be
// null, W must be null, the adapters' B are not read); used by the backward.
int fwd_impl(const wp_mat* X, const wp_mat* W, const wp_mat* bias, int G, bool grouped,
             const wp_adapter* adapters, int n_adapters, double request_scale, const wp_out* Y,
             void* workspace, size_t ws_bytes, cudaStream_t stream, float* h_out = nullptr,
             int h_out_ld = 0, bool rank_only = false, bool swiglu = false,
             const wp_out* eg = nullptr, bool w_mn = false) {
  if (!valid_input(X, false)) return WP_ERR_INVALID;
  if (W && !valid_input(W, true)) return WP_ERR_INVALID;
  if (rank_only ? (W || bias || !h_out || n_adapters < 1 || X->dtype != WP_BF16) : !valid_output(Y))
    return WP_ERR_INVALID;
  if (!std::isfinite(request_scale)) return WP_ERR_INVALID;
  if (n_adapters < 0 || n_adapters > kMaxAd + kMaxAd32) return WP_ERR_UNSUPPORTED;
  if (n_adapters > 0 && !adapters) return WP_ERR_INVALID;
  if (grouped && (G < 1 || G > kMaxGroups || n_adapters != G)) return WP_ERR_INVALID;
  if (!grouped) G = 1;
  // SwiGLU front half: the gate and up groups of a stacked W, h = silu(e) g out
  if (swiglu && (!W || !grouped || G != 2 || rank_only || Y->dtype != WP_BF16)) return WP_ERR_INVALID;
  if (eg && (!swiglu || !valid_output(eg) || eg->dtype != WP_BF16)) return WP_ERR_INVALID;

  // w_mn (the backward's dX pass): W is stored [in, out], i.e. the forward's W as it is
  if (w_mn && (!W || swiglu || rank_only || G != 1)) return WP_ERR_INVALID;
  const long long T = X->rows, K = X->cols;
  const long long N = W ? (w_mn ? W->cols : W->rows) : rank_only ? G * adapters[0].B.rows : Y->cols;
  if (W && (w_mn ? W->rows : W->cols) != K) return WP_ERR_SHAPE;
  if (!rank_only && (Y->rows != T || Y->cols != (swiglu ? N / 2 : N))) return WP_ERR_SHAPE;
  if (eg && (eg->rows != T || eg->cols != N)) return WP_ERR_SHAPE;
  if (N % G) return WP_ERR_SHAPE;
  const long long out_g = N / G;
  if (W && W->dtype == WP_NF4 && !w_mn && (K % 64 != 0 || W->ld != K)) return WP_ERR_SHAPE;
  if (W && W->dtype == WP_NF4 && w_mn && (N % 64 != 0 || W->ld != N)) return WP_ERR_SHAPE;
  if (bias) {
    if (!bias->data || (bias->dtype != WP_BF16 && bias->dtype != WP_FP32)) return WP_ERR_INVALID;
    if (bias->rows * bias->cols != N) return WP_ERR_SHAPE;
  }
  if (T > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL) return WP_ERR_UNSUPPORTED;

  // adapters: shapes, dtypes and combined scales
  float s_of[kMaxAd + kMaxAd32];
  for (int i = 0; i < n_adapters; ++i) {
    const wp_adapter& a = adapters[i];
    if (!valid_input(&a.A, false) || !valid_input(&a.B, false)) return WP_ERR_INVALID;
    if (a.A.dtype != a.B.dtype) return WP_ERR_DTYPE;
    const long long r = a.A.rows;
    if (r <= 0) return WP_ERR_INVALID;
    if (a.A.cols != K || a.B.cols != r || a.B.rows != (grouped ? out_g : N)) return WP_ERR_SHAPE;
    if (!std::isfinite(a.alpha) || !std::isfinite(a.strength)) return WP_ERR_INVALID;
    const double s = a.alpha / static_cast<double>(r) * a.strength * request_scale;
    if (!std::isfinite(s) || !std::isfinite(static_cast<float>(s))) return WP_ERR_INVALID;
    s_of[i] = static_cast<float>(s);
  }

  // legacy adapter bias vectors (older adapters' lora_B.bias), folded with the layer's own
  // bias into one fp32 vector that the epilogue adds instead
  BiasFoldParams fold{};
  for (int i = 0; i < n_adapters; ++i) {
    const wp_adapter& a = adapters[i];
    if (!a.bias_B) continue;
    if (a.bias_B_dtype != WP_BF16 && a.bias_B_dtype != WP_FP32) return WP_ERR_DTYPE;
    if (rank_only || s_of[i] == 0.0f) continue;
    const int g = grouped ? i : 0;
    BiasFoldParams::Vec& v = fold.ad[fold.n++];
    v.v = a.bias_B;
    v.dtype = a.bias_B_dtype;
    v.s = s_of[i];
    v.col0 = static_cast<int>(g * out_g);
    v.cols = static_cast<int>(grouped ? out_g : N);
  }

  FwdPlan plan;
  plan_fwd(X, W, adapters, n_adapters, &plan);
  const size_t need = fwd_workspace(X, plan, /*min_only=*/true);
  if (need > 0 && (!workspace || ws_bytes < need)) return WP_ERR_WORKSPACE;
  if (need > 0 && !aligned16(workspace)) return WP_ERR_ALIGN;
  wp_mat folded_bias{};
  if (fold.n > 0) {
    // the first plan.fold_bytes of the workspace (at least 4 N bytes); the paths below get
    // the rest
    fold.out = static_cast<float*>(workspace);
    fold.bias = bias ? const_cast<void*>(bias->data) : nullptr;
    fold.bias_dtype = bias ? bias->dtype : WP_FP32;
    fold.N = static_cast<int>(N);
    folded_bias = wp_mat{workspace, WP_FP32, 1, N, N, nullptr};
    workspace = static_cast<uint8_t*>(workspace) + plan.fold_bytes;
    ws_bytes -= plan.fold_bytes;
  }
  if (T == 0) return WP_OK;
  if (fold.n > 0) {
    const int frc = launch_bias_fold(fold, stream);
    if (frc != WP_OK) return frc;
    bias = &folded_bias;
  }

  // a few tokens: the weight-streaming small-token path, when the workspace holds its
  // partial sums (else the general path below serves the call); it does not store s X A^T,
  // so calls that want it back (h_out) stay on the general path
  if (!rank_only && !swiglu && !h_out && !w_mn && plan.skinny_bytes > 0 && workspace &&
      ws_bytes >= plan.skinny_bytes && aligned16(workspace)) {
    const int rc = skinny_impl(X, W, bias, G, grouped, adapters, n_adapters, s_of, Y, workspace, stream);
    if (rc != WP_ERR_UNSUPPORTED) return rc;
  }

  if (!plan.tc) {
    // ------------------------------------------------------------- exact FP32 path
    if (W && W->dtype == WP_NF4) return WP_ERR_DTYPE;
    if (swiglu) return WP_ERR_DTYPE;
    F32Params fp{};
    fp.T = static_cast<int>(T); fp.K = static_cast<int>(K); fp.N = static_cast<int>(N);
    fp.X = X->data; fp.x_dtype = X->dtype; fp.ldx = X->ld;
    fp.W = W ? W->data : nullptr; fp.w_dtype = W ? W->dtype : WP_FP32; fp.ldw = W ? W->ld : 0;
    fp.bias = bias ? bias->data : nullptr; fp.bias_dtype = bias ? bias->dtype : WP_FP32;
    fp.Y = Y->data; fp.y_dtype = Y->dtype; fp.ldy = Y->ld;
    H32Params hp{};
    hp.T = fp.T; hp.K = fp.K; hp.X = X->data; hp.x_dtype = X->dtype; hp.ldx = X->ld;
    int off = 0;
    for (int i = 0; i < n_adapters; ++i) {
      if (s_of[i] == 0.0f) continue;
      const wp_adapter& a = adapters[i];
      const int k = fp.n_ad++;
      fp.ad[k].A = a.A.data; fp.ad[k].a_dtype = a.A.dtype; fp.ad[k].lda = a.A.ld;
      fp.ad[k].B = a.B.data; fp.ad[k].b_dtype = a.B.dtype; fp.ad[k].ldb = a.B.ld;
      fp.ad[k].rank = static_cast<int>(a.A.rows); fp.ad[k].s = s_of[i];
      const int g = grouped ? i : 0;
      fp.col_begin[k] = static_cast<int>(g * out_g);
      fp.col_end[k] = static_cast<int>((g + 1) * out_g);
      hp.A[k] = a.A.data; hp.a_dtype[k] = a.A.dtype; hp.lda[k] = a.A.ld;
      hp.rank[k] = fp.ad[k].rank; hp.h_off[k] = off; hp.s[k] = s_of[i];
      off += fp.ad[k].rank;
    }
    hp.n_ad = fp.n_ad; hp.H = static_cast<float*>(workspace); hp.h_cols = off;
    int rc = WP_OK;
    if (hp.n_ad > 0) rc = launch_h32(hp, stream);
    if (rc != WP_OK) return rc;
    return launch_f32_linear(fp, static_cast<const float*>(workspace), off, stream);
  }

  // --------------------------------------------------------------- tensor-core path
  const bool nf4 = W && W->dtype == WP_NF4;
  if (!aligned16(X->data) || X->ld % 8) return WP_ERR_ALIGN;
  if (W && (!aligned16(W->data) || W->ld % 8)) return WP_ERR_ALIGN;
  if (!rank_only && (!aligned16(Y->data) || Y->ld % (Y->dtype == WP_BF16 ? 8 : 4))) return WP_ERR_ALIGN;
  if (out_g % 8) return WP_ERR_ALIGN;
  if (eg && (!aligned16(eg->data) || eg->ld % 8)) return WP_ERR_ALIGN;

  TcParams p{};
  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  p.T = static_cast<int>(T); p.K = static_cast<int>(K); p.N = static_cast<int>(N);
  p.out_g = static_cast<int>(out_g); p.G = G;
  p.nt_g = static_cast<int>((out_g + kBN - 1) / kBN);
  // a 4-bit W's tile is two 256-row halves sharing each dequantised weight tile
  p.m_shift = nf4 ? 1 : 0;
  p.r_blocks = static_cast<int>((T + kPairM - 1) / kPairM);
  p.m_tiles = static_cast<int>((T + (kPairM << p.m_shift) - 1) / (kPairM << p.m_shift));
  const long long total = static_cast<long long>(p.m_tiles) * G * p.nt_g;
  if (total > 0x7FFFFFFFLL) return WP_ERR_UNSUPPORTED;
  p.total_tiles = rank_only ? 0 : static_cast<int>(total);
  p.k_blocks = static_cast<int>((K + kBK - 1) / kBK);
  p.has_base = W ? 1 : 0;
  p.w_mn = w_mn ? 1 : 0;
  p.bias = bias ? bias->data : nullptr; p.bias_f32 = bias && bias->dtype == WP_FP32;
  p.bias_vec = bias && aligned16(bias->data) ? 1 : 0;
  if (!rank_only) { p.Y = Y->data; p.ldy = Y->ld; p.y_f32 = Y->dtype == WP_FP32; }
  p.timeout_ns = wait_limit_ns();

  // Plan the adapters (host only; every rejection happens before any CUDA call).
  H32Params hp{};
  hp.T = p.T; hp.K = p.K; hp.X = X->data; hp.x_dtype = WP_BF16; hp.ldx = X->ld;
  int h_off = 0;
  int hout_of[kMaxAd + kMaxAd32];          // column of adapter i in h_out: ranks of 0..i-1
  for (int i = 0, acc = 0; i < n_adapters; ++i) {
    hout_of[i] = acc;
    acc += static_cast<int>(adapters[i].A.rows);
  }
  p.h_out = h_out;
  p.h_out_ld = h_out_ld;
  // FP32 adapters ride on the tensor cores as bf16 pieces when every adapter's rank
  // columns (3 rp for such an adapter) fit one accumulator buffer; else the FP32
  // CUDA-core projection plus an epilogue product carry them
  bool split3 = false;
  {
    int n16 = 0, n32 = 0, width = 0;
    for (int i = 0; i < n_adapters; ++i) {
      if (s_of[i] == 0.0f) continue;
      const int r = static_cast<int>(adapters[i].A.rows);
      if (adapters[i].A.dtype == WP_FP32) { ++n32; width += 3 * split_rp(r); }
      else { ++n16; width += (r + 15) / 16 * 16; }
    }
    split3 = n32 > 0 && n16 + n32 <= kMaxAd && width <= kHCols && !h_out;
  }
  // workspace: [fp32 s X A^T | bf16 B pieces | H~ | row-block flags | packed A rows]
  const size_t h32_bytes = round256(static_cast<size_t>(T) * plan.rank32_total * 4);
  size_t split_off = h32_bytes;
  const size_t hq_off = h32_bytes + plan.split_bytes;
  const size_t flags_off = hq_off + round256(static_cast<size_t>(T) * plan.htilde_cols * 2);
  const size_t pack_off = flags_off + round256((static_cast<size_t>(T) + kPairM - 1) / kPairM * 4);
  PackParams pk{};
  pk.K = static_cast<int>(K);
  pk.ldk = static_cast<int>((K + 7) / 8 * 8);
  pk.Ap = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + pack_off);
  const void* bmap_ptr[kMaxAd]; long long bmap_cols[kMaxAd], bmap_ld[kMaxAd];
  int hcols = 0;                           // H~ columns: every adapter packed, 16-aligned
  for (int g = 0; g < G; ++g) {
    p.ad_begin[g] = p.n_ad;
    for (int i = 0; i < n_adapters; ++i) {
      const int ag = grouped ? i : 0;
      if (ag != g || s_of[i] == 0.0f) continue;
      const wp_adapter& a = adapters[i];
      const int r = static_cast<int>(a.A.rows);
      if (a.A.dtype == WP_FP32 && split3) {
        TcAdapter& d = p.ad[p.n_ad];
        PackAdapter& q = pk.ad[p.n_ad];
        const int rp = split_rp(r);
        q.A = a.A.data; q.lda = a.A.ld; q.dtype = WP_FP32; q.r = r; q.rp = rp; q.split3 = 1;
        q.B = static_cast<const float*>(a.B.data); q.ldb = a.B.ld; q.out = static_cast<int>(a.B.rows);
        q.Bs = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + split_off);
        split_off += split_b_bytes(r, a.B.rows);
        d.group = g; d.rank = 6 * rp; d.rpad16 = 6 * rp; d.pw = 3 * rp; d.split3 = 1;
        d.nchunks = (6 * rp + 63) / 64; d.s = s_of[i];
        d.hout_off = hout_of[i];
        d.toff = hcols;
        hcols += d.rpad16;
        bmap_ptr[p.n_ad] = q.Bs; bmap_cols[p.n_ad] = 6 * rp; bmap_ld[p.n_ad] = 6 * rp;
        ++p.n_ad;
        continue;
      }
      if (a.A.dtype == WP_FP32) {
        if (p.n_ad32 >= kMaxAd32) return WP_ERR_UNSUPPORTED;
        TcAdapter32& d = p.ad32[p.n_ad32++];
        d.group = g; d.rank = r; d.h_off = h_off; d.ldb = static_cast<int>(a.B.ld);
        d.B = static_cast<const float*>(a.B.data);
        const int k = hp.n_ad++;
        hp.A[k] = a.A.data; hp.a_dtype[k] = WP_FP32; hp.lda[k] = a.A.ld; hp.rank[k] = r;
        hp.h_off[k] = h_off; hp.s[k] = s_of[i];
        h_off += r;
        continue;
      }
      if (p.n_ad >= kMaxAd) return WP_ERR_UNSUPPORTED;
      if (r > kHCols) return WP_ERR_UNSUPPORTED;
      if (!rank_only && (!aligned16(a.B.data) || a.B.ld % 8)) return WP_ERR_ALIGN;
      TcAdapter& d = p.ad[p.n_ad];
      PackAdapter& q = pk.ad[p.n_ad];
      d.group = g; d.rank = r; d.rpad16 = (r + 15) / 16 * 16; d.pw = d.rpad16; d.split3 = 0;
      d.nchunks = (r + 63) / 64; d.s = s_of[i];
      d.hout_off = hout_of[i];
      d.toff = hcols;
      hcols += d.rpad16;
      q.A = a.A.data; q.lda = a.A.ld; q.dtype = WP_BF16; q.r = r; q.rp = d.pw; q.split3 = 0;
      bmap_ptr[p.n_ad] = a.B.data; bmap_cols[p.n_ad] = r; bmap_ld[p.n_ad] = a.B.ld;
      ++p.n_ad;
    }
  }
  p.ad_begin[G] = p.n_ad;
  if (swiglu) {
    // one kind of tile: 128 gate and the same 128 up columns, every adapter applied (each
    // to its own half of the tile)
    if (p.n_ad32 > 0) return WP_ERR_UNSUPPORTED;
    p.swiglu = 1;
    p.G = 1;
    p.nt_g = static_cast<int>((out_g + 127) / 128);
    p.total_tiles = p.m_tiles * p.nt_g;
    p.ad_begin[1] = p.n_ad;
    if (eg) { p.eg = static_cast<uint16_t*>(eg->data); p.ld_eg = eg->ld; }
  }
  if (p.n_ad > 0) {
    // Rank passes: the adapters (whole) go first-fit, widest first, into passes of at most
    // kHCols rank columns, one accumulator buffer each; each pass is a rank item of its own
    // per 256-row block.  Within a pass the pair's MMA has N = htot columns: each CTA
    // supplies half of every adapter's packed A rows, so both halves are equally wide, and
    // every pass is padded to the widest one (zero rows).
    int order[kMaxAd], pass_w[kMaxAd] = {};
    for (int k = 0; k < p.n_ad; ++k) order[k] = k;
    std::stable_sort(order, order + p.n_ad, [&](int a, int b) { return p.ad[a].pw > p.ad[b].pw; });
    int npass = 0;
    for (int i = 0; i < p.n_ad; ++i) {
      const int k = order[i];
      if (p.ad[k].pw > kHCols) return WP_ERR_UNSUPPORTED;
      int q = 0;
      while (q < npass && pass_w[q] + p.ad[k].pw > kHCols) ++q;
      if (q == npass) ++npass;
      p.ad[k].pass = q;
      pass_w[q] += p.ad[k].pw;
    }
    int half = 0;
    for (int q = 0; q < npass; ++q) half = std::max(half, pass_w[q] / 2);
    for (int q = 0; q < npass; ++q) {
      for (int k = 0, off = 0; k < p.n_ad; ++k) {
        if (p.ad[k].pass != q) continue;
        p.ad[k].hoff = off;                     // TMEM columns within the pass
        p.ad[k].hoff2 = half + off;
        pk.ad[k].pw = p.ad[k].pw;
        pk.ad[k].hoff = q * 2 * half + off;     // packed A rows
        pk.ad[k].hoff2 = q * 2 * half + half + off;
        off += p.ad[k].pw / 2;
      }
    }
    p.htot = 2 * half;
    p.npass = npass;
    p.flag_target = 2u * static_cast<uint32_t>(npass) + (g_hold_flags.load() ? 1u : 0u);
    pk.n_ad = p.n_ad;
    pk.half = half;
    pk.npass = npass;
    pk.flags = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + flags_off);
    pk.n_flags = p.r_blocks;
    p.hq = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + hq_off);
    p.hq_ld = hcols;
    p.flags = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + flags_off);
  }
  p.h32 = static_cast<const float*>(workspace);
  p.h32_cols = h_off;
  for (int i = 0; i < p.n_ad32; ++i) {
    TcAdapter32& d = p.ad32[i];
    d.vec4 = (d.rank % 4 == 0 && d.ldb % 4 == 0 && d.h_off % 4 == 0 && h_off % 4 == 0 &&
              aligned16(d.B) && aligned16(workspace)) ? 1 : 0;
  }
  hp.H = static_cast<float*>(workspace); hp.h_cols = h_off;

  // stage: X rows (both halves' for a 4-bit W) | W half (bf16, or the dequantised 4-bit tile)
  // [| 4-bit codes | block scales]
  p.stage_bytes = nf4 ? kMHalvesNF4 * kATileBytes + kBHalfBytes : kATileBytes + kBHalfBytes;
  const size_t fixed = 1024 + 2 * kStgBytes + 512;
  int stages = static_cast<int>((kSmemLimit - fixed) / p.stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  // 4-bit W: three stages, the rest of shared memory holds the codes ring
  if (nf4) stages = 3;
  p.stages = stages;
  p.code_slots = 0;
  if (nf4) {
    const size_t left = kSmemLimit - fixed - static_cast<size_t>(stages) * p.stage_bytes;
    p.code_slots = static_cast<int>(left / kCodeSlotBytes);
    if (p.code_slots > kMaxCodeSlots) p.code_slots = kMaxCodeSlots;
    if (p.code_slots < 2 || p.code_slots % 2) return WP_ERR_UNSUPPORTED;   // even: one group per slot
  }
  if (stages < 2) return WP_ERR_UNSUPPORTED;
  const size_t smem = fixed + static_cast<size_t>(stages) * p.stage_bytes +
                      static_cast<size_t>(p.code_slots) * kCodeSlotBytes;

  // Tensor maps (driver calls from here on).
  // Each CTA of a pair loads 128 rows of X, 128 rows of the weight tile, its share of the
  // adapters' A rows, 128 rows of H~ and 128 rows of a B tile.
  int rc = make_map_bf16(&maps.x, X->data, K, T, X->ld, kBK, kBM);
  if (rc != WP_OK) return rc;
  if (nf4 && w_mn) {
    // codes stored [K rows, N/2 bytes]; each CTA loads 64 K rows x 64 bytes (its 128 output
    // columns) per K step, in the 64-byte swizzle; block scales [K, N/64] in boxes of 64 rows
    // x 4 blocks when a row of them is a multiple of 16 bytes
    rc = make_map_u8(&maps.wq, W->data, N / 2, K, N / 2, 64, kBK, 64);
    if (rc != WP_OK) return rc;
    p.absmax = W->absmax;
    p.am_tma = (N % 256 == 0 && aligned16(W->absmax)) ? 1 : 0;
    if (p.am_tma) {
      rc = make_map(&maps.am, WP_FP32, W->absmax, N / 64, K, N / 64, 4, kBK, /*swizzle=*/0);
      if (rc != WP_OK) return rc;
    }
    nf4_codebook_host(p.nf4_code);
  } else if (nf4) {
    // codes: [N rows, K/2 bytes]; each CTA loads 128 rows x 32 bytes (64 elements) per K step
    rc = make_map_u8(&maps.wq, W->data, K / 2, N, K / 2, kBK / 2, 128, 32);
    if (rc != WP_OK) return rc;
    p.absmax = W->absmax;
    // block scales [N, K/64] by TMA when a row of them is a multiple of 16 bytes
    p.am_tma = (K % 256 == 0 && aligned16(W->absmax)) ? 1 : 0;
    if (p.am_tma) {
      rc = make_map(&maps.am, WP_FP32, W->absmax, K / 64, N, K / 64, 4, 128, /*swizzle=*/0);
      if (rc != WP_OK) return rc;
    }
    nf4_codebook_host(p.nf4_code);
  } else if (W && w_mn) {
    // W stored [K rows, N columns]: boxes of 64 output columns x 64 K rows (MN-major tiles)
    rc = make_map_bf16(&maps.w, W->data, N, K, W->ld, 64, kBK);
    if (rc != WP_OK) return rc;
  } else if (W) {
    rc = make_map_bf16(&maps.w, W->data, K, N, W->ld, kBK, 128);
    if (rc != WP_OK) return rc;
  }
  if (!rank_only) {
    rc = make_map(&maps.y, Y->dtype, Y->data, swiglu ? out_g : N, T, Y->ld, Y->dtype == WP_FP32 ? 32 : 64, kBM);
    if (rc != WP_OK) return rc;
  }
  if (p.n_ad > 0) {
    // H~ and B chunks of 64 ranks (128-byte swizzle), or of 32 when at most 32 remain
    // (64-byte swizzle, half the bytes)
    rc = make_map_bf16(&maps.hq, p.hq, p.hq_ld, T, p.hq_ld, 64, kBM);
    if (rc != WP_OK) return rc;
    rc = make_map(&maps.hq32, WP_BF16, p.hq, p.hq_ld, T, p.hq_ld, 32, kBM, 64);
    if (rc != WP_OK) return rc;
  }
  if (p.n_ad > 0) {
    if (static_cast<size_t>(p.npass) * p.htot * pk.ldk * 2 > plan.pack_bytes) return WP_ERR_WORKSPACE;
    rc = make_map_bf16(&maps.ap, pk.Ap, K, static_cast<long long>(p.npass) * p.htot, pk.ldk, kBK, p.htot / 2);
    if (rc != WP_OK) return rc;
  }
  for (int k = 0; k < p.n_ad && !rank_only; ++k) {
    rc = make_map_bf16(&maps.b[k], bmap_ptr[k], bmap_cols[k], out_g, bmap_ld[k], 64, 128);
    if (rc != WP_OK) return rc;
    rc = make_map(&maps.b32[k], WP_BF16, bmap_ptr[k], bmap_cols[k], out_g, bmap_ld[k], 32, 128, 64);
    if (rc != WP_OK) return rc;
  }

  if (hp.n_ad > 0) {
    rc = launch_h32(hp, stream);
    if (rc != WP_OK) return rc;
  }
  if (p.n_ad > 0) {
    rc = launch_rank_pack(pk, stream);
    if (rc != WP_OK) return rc;
  }
  int pairs = tc_max_pairs(smem, nf4);
  if (pairs <= 0) return WP_ERR_CUDA;
  const int work = rank_only ? p.r_blocks * std::max(1, p.npass) : p.total_tiles;
  if (pairs > work) pairs = work;
  // rank items two rounds of tiles ahead, or one when the X rows of two rounds would not
  // stay in L2 until their tiles come
  const double x_two_rounds = 2.0 * pairs / (G * p.nt_g) * (kPairM << p.m_shift) * static_cast<double>(K) * 2;
  p.rlead = x_two_rounds <= 48.0 * (1 << 20) ? 2 : 1;
  // every pair opens with its first rank item unless the X rows those items read are far
  // more than L2 holds (they would then be read from HBM a second time when their tiles come):
  // measured, 30-168 MB of them (rank-128 q/k/v, the three-patch sidecar) gained 1.5-1.8 %,
  // 350 MB (the 8960-deep down projection) lost 2.6 %; the bound is 1.5 L2 capacities
  if (p.n_ad > 0) {
    const int first_items = std::min(pairs, p.r_blocks * std::max(1, p.npass));
    const double first_x = static_cast<double>(first_items) / std::max(1, p.npass) * kPairM * static_cast<double>(K) * 2;
    p.rank_first = first_x <= 192.0 * (1 << 20) ? 1 : 0;
  }
  return launch_tc_fwd(maps, p, 2 * pairs, smem, stream, nf4);
}

// ------------------------------------------------------------------ backward
// Workspace of lora_linear_bwd, in order (each region 256-byte aligned):
//   per group: B_g^T padded to [r_g, Ntot] bf16 | per group: A_g^T
//   [in, r8_g] bf16 | s G [T, R] fp32 | H [T, R] fp32 | the bf16 pieces of H and of s G
//   [T, tokN] | token-split partial sums | the forward calls' scratch
struct BwdLayout {
  size_t bhat[kMaxGroups], at[kMaxGroups], gs, h, fwd, fwd_bytes, total;
  int r8[kMaxGroups];
  int roff[kMaxGroups];
  int R;
  // dA / dB on the tensor cores: H and s G as two bf16 pieces each (hi, lo) side by side, N
  // = 128 or 256 columns per contraction.  All groups in one contraction when their pieces
  // fit 256 columns; otherwise one contraction per group (each group's pieces fit: r <= 128).
  bool per_group;
  int tokN, R16, roff16[kMaxGroups], splits_a, splits_b;
  size_t hp, gp, tpart;
};

// Token splits of a contraction with m_tiles 256-row blocks over k_blocks 64-token steps, its
// units (row block, token range) dealt to the CTA pairs: the count whose busiest pair streams
// the fewest steps (units per pair rounded up x steps per unit; the fewest splits on a tie), at
// least 8 steps per unit.  (About one unit per SM, the earlier rule, left 2.1 units per pair on
// average where the busiest had 3.)
int tok_splits(int m_tiles, int k_blocks) {
  const int pairs = std::max(1, device_sm_count() / 2);
  const int cap = std::max(1, k_blocks / 8);
  int best_s = 1;
  long long best = -1;
  for (int s = 1; s <= cap; ++s) {
    const int per = (k_blocks + s - 1) / s;              // steps per unit
    const int used = (k_blocks + per - 1) / per;         // splits that hold steps
    const long long rounds = (static_cast<long long>(m_tiles) * used + pairs - 1) / pairs;
    const long long cost = rounds * per;
    if (best < 0 || cost < best) { best = cost; best_s = used; }
  }
  return best_s;
}

// The largest rank the backward takes per group: the group's two bf16 pieces fill at most one
// 256-column accumulator.
constexpr int kBwdMaxRank = 128;

bool bwd_layout(const wp_mat* X, const wp_mat* W, const wp_adapter* ad, int G, BwdLayout* L) {
  if (!X || !W || !ad || G < 1 || G > kMaxGroups) return false;
  const size_t T = static_cast<size_t>(X->rows), K = static_cast<size_t>(X->cols);
  const size_t Ntot = static_cast<size_t>(W->rows);
  if (Ntot % G) return false;
  const size_t og = Ntot / G;
  size_t off = 0;
  int R = 0;
  for (int g = 0; g < G; ++g) {
    const int r = static_cast<int>(ad[g].A.rows);
    if (r <= 0) return false;
    L->r8[g] = (r + 7) / 8 * 8;
    L->roff[g] = R;
    R += r;
    L->bhat[g] = off;
    off += round256(static_cast<size_t>(r) * Ntot * 2);
  }
  for (int g = 0; g < G; ++g) {
    L->at[g] = off;
    off += round256(K * L->r8[g] * 2);
  }
  L->R = R;
  L->gs = off;
  off += round256(T * R * 4);
  L->h = off;
  off += round256(T * R * 4);
  L->R16 = 0;
  int max16 = 0;
  for (int g = 0; g < G; ++g) {
    const int r16 = static_cast<int>((ad[g].A.rows + 15) / 16 * 16);
    L->roff16[g] = L->R16;
    L->R16 += r16;
    max16 = std::max(max16, r16);
  }
  L->per_group = 2 * L->R16 > 256;
  const int width = L->per_group ? max16 : L->R16;          // the widest contraction's ranks
  L->tokN = 2 * width <= 128 ? 128 : 256;
  const int kbt = static_cast<int>((T + 63) / 64);
  const size_t Mb = L->per_group ? og : Ntot;                // dB's rows per contraction
  L->splits_a = tok_splits(static_cast<int>((K + 255) / 256), kbt);
  L->splits_b = tok_splits(static_cast<int>((Mb + 255) / 256), kbt);
  L->hp = off;
  off += round256(T * L->tokN * 2);
  L->gp = off;
  off += round256(T * L->tokN * 2);
  L->tpart = off;
  off += round256(std::max(static_cast<size_t>(L->splits_a) * K, static_cast<size_t>(L->splits_b) * Mb) *
                  L->tokN * 4);
  // workspace of the forward call that computes dX: X := dY [T, Ntot], the weight W [Ntot, K]
  // as stored (read MN-major: in = Ntot, out = K), adapter g A := B_g^T padded to [r_g, Ntot]
  // (bf16), B := A_g^T [K, r_g]
  {
    const wp_mat dy{nullptr, WP_BF16, static_cast<int64_t>(T), static_cast<int64_t>(Ntot),
                    static_cast<int64_t>(Ntot), nullptr};
    const wp_mat wt{nullptr, WP_BF16, static_cast<int64_t>(K), static_cast<int64_t>(Ntot),
                    static_cast<int64_t>(Ntot), nullptr};   // the sizes the plan reads: out = K
    wp_adapter fa[kMaxGroups] = {};
    for (int g = 0; g < G; ++g) {
      const int64_t r = ad[g].A.rows;
      fa[g].A = wp_mat{nullptr, WP_BF16, r, static_cast<int64_t>(Ntot), static_cast<int64_t>(Ntot), nullptr};
      fa[g].B = wp_mat{nullptr, WP_BF16, static_cast<int64_t>(K), r, r, nullptr};
      fa[g].alpha = ad[g].alpha;
      fa[g].strength = ad[g].strength;
    }
    FwdPlan plan;
    plan_fwd(&dy, &wt, fa, G, &plan);
    // and of the rank-items-only call that computes H = X A_g^T (X [T, in], A_g as given)
    FwdPlan hplan;
    plan_fwd(X, nullptr, ad, G, &hplan);
    L->fwd = off;
    L->fwd_bytes = std::max(fwd_workspace(&dy, plan), fwd_workspace(X, hplan));
    off += L->fwd_bytes;
  }
  L->total = off;
  return true;
}

int bwd_impl(const wp_mat* X, const wp_mat* W, const wp_mat* dY, int G, const wp_adapter* ad,
             double request_scale, const wp_out* dX, const wp_out* dA, const wp_out* dB,
             void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!valid_input(X, false) || !valid_input(W, true) || !valid_input(dY, false)) return WP_ERR_INVALID;
  if (!ad || !dA || !dB || G < 1 || G > kMaxGroups) return WP_ERR_INVALID;
  if (!std::isfinite(request_scale)) return WP_ERR_INVALID;
  if (X->dtype != WP_BF16 || dY->dtype != WP_BF16) return WP_ERR_DTYPE;
  if (W->dtype != WP_BF16 && W->dtype != WP_NF4) return WP_ERR_DTYPE;
  const long long T = X->rows, K = X->cols, Ntot = W->rows;
  if (W->cols != K || dY->rows != T || dY->cols != Ntot || Ntot % G) return WP_ERR_SHAPE;
  if (W->dtype == WP_NF4 && (K % 64 || W->ld != K)) return WP_ERR_SHAPE;
  if (W->dtype == WP_NF4 && !aligned16(W->data)) return WP_ERR_ALIGN;   // 4-byte code loads
  const long long og = Ntot / G;
  if (K % 8 || og % 8 || Ntot % 8) return WP_ERR_ALIGN;
  if (!aligned16(X->data) || X->ld % 8 || !aligned16(dY->data) || dY->ld % 8) return WP_ERR_ALIGN;
  if (T > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL || Ntot > 0x7FFFFFFFLL) return WP_ERR_UNSUPPORTED;
  if (dX) {
    if (!valid_output(dX)) return WP_ERR_INVALID;
    if (dX->rows != T || dX->cols != K) return WP_ERR_SHAPE;
  }
  float s_of[kMaxGroups];
  for (int g = 0; g < G; ++g) {
    const wp_adapter& a = ad[g];
    if (!valid_input(&a.A, false) || !valid_input(&a.B, false)) return WP_ERR_INVALID;
    if (a.A.dtype != WP_BF16 || a.B.dtype != WP_BF16) return WP_ERR_DTYPE;
    const long long r = a.A.rows;
    if (r <= 0) return WP_ERR_INVALID;
    if (r > kBwdMaxRank) return WP_ERR_UNSUPPORTED;
    if (a.A.cols != K || a.B.rows != og || a.B.cols != r) return WP_ERR_SHAPE;
    if (!std::isfinite(a.alpha) || !std::isfinite(a.strength)) return WP_ERR_INVALID;
    const double s = a.alpha / static_cast<double>(r) * a.strength * request_scale;
    if (!std::isfinite(s) || !std::isfinite(static_cast<float>(s))) return WP_ERR_INVALID;
    s_of[g] = static_cast<float>(s);
    const wp_out& da = dA[g];
    const wp_out& db = dB[g];
    if (!valid_output(&da) || !valid_output(&db)) return WP_ERR_INVALID;
    if (da.dtype != WP_FP32 || db.dtype != WP_FP32) return WP_ERR_DTYPE;
    if (da.rows != r || da.cols != K || db.rows != og || db.cols != r) return WP_ERR_SHAPE;
  }
  BwdLayout L;
  if (!bwd_layout(X, W, ad, G, &L)) return WP_ERR_INVALID;
  if (!workspace || ws_bytes < L.total) return WP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return WP_ERR_ALIGN;
  if (T == 0) {
    // no tokens: dA and dB are sums over nothing
    for (int g = 0; g < G; ++g) {
      for (const wp_out* o : {&dA[g], &dB[g]}) {
        const cudaError_t e = cudaMemset2DAsync(o->data, static_cast<size_t>(o->ld) * 4, 0,
                                                static_cast<size_t>(o->cols) * 4, o->rows, stream);
        if (e != cudaSuccess) return record_cuda();
      }
    }
    return WP_OK;
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* Gs = reinterpret_cast<float*>(ws + L.gs);
  float* H = reinterpret_cast<float*>(ws + L.h);
  int rc;

  // 1. per group: B_g^T placed at the group's columns of a zero [r_g, Ntot] matrix (so
  //    dY B_hat_g^T = dY_g B_g), and A_g^T [K, r8_g]
  wp_adapter fwd_ad[kMaxGroups] = {};             // (no legacy bias vectors: dX does not have them)
  for (int g = 0; g < G; ++g) {
    const wp_adapter& a = ad[g];
    const int r = static_cast<int>(a.A.rows);
    uint16_t* bh = reinterpret_cast<uint16_t*>(ws + L.bhat[g]);
    uint16_t* at = reinterpret_cast<uint16_t*>(ws + L.at[g]);
    cudaError_t e = cudaMemsetAsync(bh, 0, static_cast<size_t>(r) * Ntot * 2, stream);
    if (e != cudaSuccess) { set_last_cuda_error(e); return WP_ERR_CUDA; }
    rc = launch_transpose_bf16(a.B.data, a.B.ld, static_cast<int>(og), r, bh + g * og, Ntot, stream);
    if (rc != WP_OK) return rc;
    rc = launch_transpose_bf16(a.A.data, a.A.ld, r, static_cast<int>(K), at, L.r8[g], stream);
    if (rc != WP_OK) return rc;
    fwd_ad[g].A = wp_mat{bh, WP_BF16, r, Ntot, Ntot, nullptr};
    fwd_ad[g].B = wp_mat{at, WP_BF16, K, r, L.r8[g], nullptr};
    fwd_ad[g].alpha = a.alpha;
    fwd_ad[g].strength = a.strength;
  }

  // 2. H = X A_g^T (fp32, for dB): rank items only, on the tensor cores (s = 1)
  {
    wp_adapter h_ad[kMaxGroups];
    for (int g = 0; g < G; ++g) {
      h_ad[g] = ad[g];
      h_ad[g].alpha = static_cast<double>(ad[g].A.rows);
      h_ad[g].strength = 1.0;
      h_ad[g].bias_B = nullptr;
    }
    rc = fwd_impl(X, nullptr, nullptr, G, G > 1, h_ad, G, 1.0, nullptr, ws + L.fwd, L.fwd_bytes,
                  stream, H, L.R, /*rank_only=*/true);
    if (rc != WP_OK) return rc;
  }

  // 3. dX = dY W + sum_g s_g (dY B_g) A_g on the fused tensor-core kernel, the weight read as
  //    stored ([Ntot, K]: MN-major tiles, a 4-bit W dequantised straight into them), which
  //    also leaves s_g dY B_g (fp32) in Gs; without dX, a rank-items-only call computes Gs
  if (dX) {
    rc = fwd_impl(dY, W, nullptr, 1, false, fwd_ad, G, request_scale, dX, ws + L.fwd, L.fwd_bytes, stream, Gs,
                  L.R, /*rank_only=*/false, /*swiglu=*/false, /*eg=*/nullptr, /*w_mn=*/true);
    if (rc != WP_OK) return rc;
  } else {
    // s_g dY B_g alone: rank items only
    rc = fwd_impl(dY, nullptr, nullptr, 1, false, fwd_ad, G, request_scale, nullptr, ws + L.fwd,
                  L.fwd_bytes, stream, Gs, L.R, /*rank_only=*/true);
    if (rc != WP_OK) return rc;
  }

  // 4. dA_g = (s_g G_g)^T X  and  dB_g = s_g dY_g^T H_g (exact zeros when s_g == 0): token
  //    contractions on the tensor cores with the fp32 H and s G as two bf16 pieces each; all
  //    groups in one contraction when their pieces fit 256 columns, else one per group
  for (int g = 0; g < G; ++g) {
    if (s_of[g] != 0.0f) continue;
    for (const wp_out* o : {&dA[g], &dB[g]}) {
      cudaError_t e = cudaMemset2DAsync(o->data, o->ld * 4, 0, o->cols * 4, o->rows, stream);
      if (e != cudaSuccess) { set_last_cuda_error(e); return WP_ERR_CUDA; }
    }
  }
  uint16_t* Hp = reinterpret_cast<uint16_t*>(ws + L.hp);
  uint16_t* Gp = reinterpret_cast<uint16_t*>(ws + L.gp);
  float* tpart = reinterpret_cast<float*>(ws + L.tpart);
  const int Ti = static_cast<int>(T);
  TokGemmParams tp{};
  tp.T = Ti; tp.k_blocks = (Ti + 63) / 64;
  tp.part = tpart;
  tp.status = tc_status_ptr();
  tp.timeout_ns = wait_limit_ns();
  if (!tp.status) return record_cuda();
  const size_t sb = 2 * 64 * 128 + static_cast<size_t>(L.tokN) / 2 * 128;
  tp.stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemLimit - 1024 - 256) / sb));
  const size_t smem = 1024 + tp.stages * sb + 256;
  const int max_pairs = tokgemm_max_pairs(smem);
  if (max_pairs <= 0) return WP_ERR_CUDA;
  // one contraction per entry of this loop: all groups at once (g0 = 0, g1 = G), or group g0
  for (int g0 = 0; g0 < G; ) {
    const int g1 = L.per_group ? g0 + 1 : G;
    bool any = false;
    for (int g = g0; g < g1; ++g) any = any || s_of[g] != 0.0f;
    if (!any) { g0 = g1; continue; }
    TokPieceMap pm{};
    pm.G = g1 - g0;
    for (int g = g0; g < g1; ++g) {
      const int k = g - g0;
      pm.roff16[k] = L.roff16[g] - L.roff16[g0];
      pm.off[k] = L.roff[g];
      pm.r[k] = static_cast<int>(ad[g].A.rows);
    }
    pm.R16 = (g1 < G ? L.roff16[g1] : L.R16) - L.roff16[g0];
    const int N = 2 * pm.R16 <= 128 ? 128 : 256;
    tp.N = N;
    rc = launch_pieces(H, L.R, Ti, N, pm, Hp, stream);
    if (rc == WP_OK) rc = launch_pieces(Gs, L.R, Ti, N, pm, Gp, stream);
    if (rc != WP_OK) return rc;
    // dB rows: every group's columns of dY at once, or group g0's alone
    const long long mb0 = L.per_group ? g0 * og : 0, Mb = L.per_group ? og : Ntot;
    for (int pass = 0; pass < 2; ++pass) {
      const bool db = pass == 0;
      TokGemmMaps tm;
      std::memset(&tm, 0, sizeof(tm));
      const long long M = db ? Mb : K;
      tp.M = static_cast<int>(M);
      tp.m_tiles = static_cast<int>((M + 255) / 256);
      tp.splits = db ? L.splits_b : L.splits_a;
      tp.kb_per_split = (tp.k_blocks + tp.splits - 1) / tp.splits;
      tp.splits = (tp.k_blocks + tp.kb_per_split - 1) / tp.kb_per_split;
      tp.units = tp.m_tiles * tp.splits;
      rc = db ? make_map_bf16(&tm.a, static_cast<const uint16_t*>(dY->data) + mb0, Mb, T, dY->ld, 64, 64)
              : make_map_bf16(&tm.a, X->data, K, T, X->ld, 64, 64);
      if (rc == WP_OK) rc = make_map_bf16(&tm.b, db ? Hp : Gp, N, T, N, 64, 64);
      if (rc != WP_OK) return rc;
      rc = launch_tokgemm(tm, tp, std::min(max_pairs, tp.units), smem, stream);
      if (rc != WP_OK) return rc;
      for (int g = g0; g < g1; ++g) {
        const int r = static_cast<int>(ad[g].A.rows);
        if (s_of[g] == 0.0f) continue;
        const int ro = L.roff16[g] - L.roff16[g0];
        rc = db ? launch_tok_finish(tpart, tp.M, N, tp.splits, pm.R16, ro, r, static_cast<int>(g * og - mb0),
                                    static_cast<int>(og), s_of[g], static_cast<float*>(dB[g].data), dB[g].ld,
                                    false, stream)
                : launch_tok_finish(tpart, tp.M, N, tp.splits, pm.R16, ro, r, 0, static_cast<int>(K), 1.0f,
                                    static_cast<float*>(dA[g].data), dA[g].ld, true, stream);
        if (rc != WP_OK) return rc;
      }
    }
    g0 = g1;
  }
  return WP_OK;
}

// ------------------------------------------------------------------ the unfused chain (exact tier)
// sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM", Motivation and
// Modifications (exact tier): base = bf16(X W^T + bias); per adapter t = bf16(X A^T),
// d = bf16(t B^T) (+ its legacy vector inside that GEMM), d = bf16(d c) for each scale c of
// (alpha/r, strength, request scale) -- a c of exactly 1.0 skipped when asked, which changes
// no bit -- and Y = bf16(Y + d), adapter after adapter; an FP32 adapter keeps its GEMMs and
// scaling in FP32 and is added once.  The GEMMs run on the fused kernel without adapters.
// Workspace, in order (each region 256-byte aligned): t [T, r_max] bf16 | d [T, N] fp32-sized
// | the scratch of the FP32 adapters' delta-only forwards.
struct ExactLayout {
  size_t t, d, fwd, fwd_bytes, total;
};

bool exact_layout(const wp_mat* X, const wp_mat* W, const wp_adapter* ad, int n, ExactLayout* L) {
  *L = ExactLayout{};
  if (!X || !W || n < 0 || (n > 0 && !ad) || X->rows < 0 || W->rows < 0) return false;
  const size_t T = static_cast<size_t>(X->rows), N = static_cast<size_t>(W->rows);
  size_t rmax = 0, fwd = 0;
  for (int i = 0; i < n; ++i) {
    rmax = std::max(rmax, static_cast<size_t>(std::max<int64_t>(ad[i].A.rows, 0)));
    if (ad[i].A.dtype == WP_FP32) {
      FwdPlan plan;
      plan_fwd(X, nullptr, &ad[i], 1, &plan);
      fwd = std::max(fwd, fwd_workspace(X, plan));
    }
  }
  size_t off = 0;
  L->t = off;
  off += round256(T * rmax * 2);
  L->d = off;
  off += n > 0 ? round256(T * N * 4) : 0;
  L->fwd = off;
  L->fwd_bytes = fwd;
  off += fwd;
  L->total = off;
  return true;
}

int exact_impl(const wp_mat* X, const wp_mat* W, const wp_mat* bias, int n_groups, const wp_adapter* ad, int n,
               double request_scale, bool skip_unit, const wp_out* Y, void* workspace, size_t ws_bytes,
               cudaStream_t stream) {
  if (!valid_input(X, false) || !W || !valid_input(W, true) || !valid_output(Y)) return WP_ERR_INVALID;
  if (X->dtype != WP_BF16 || Y->dtype != WP_BF16) return WP_ERR_DTYPE;   // the chain's tensors are bf16
  if (W->dtype != WP_BF16 && W->dtype != WP_NF4) return WP_ERR_DTYPE;
  if (n_groups < 0 || n < 0 || n > kMaxAd + kMaxAd32 || (n > 0 && !ad)) return WP_ERR_INVALID;
  if (n_groups > 0 && n != n_groups) return WP_ERR_INVALID;
  if (!std::isfinite(request_scale)) return WP_ERR_INVALID;
  const long long T = X->rows, K = X->cols, N = W->rows;
  const int G = n_groups > 0 ? n_groups : 1;
  if (W->cols != K || Y->rows != T || Y->cols != N || N % G) return WP_ERR_SHAPE;
  const long long cols = N / G;
  if (cols % 8 || Y->ld % 8 || !aligned16(Y->data)) return WP_ERR_ALIGN;
  for (int i = 0; i < n; ++i) {
    const wp_adapter& a = ad[i];
    if (!valid_input(&a.A, false) || !valid_input(&a.B, false)) return WP_ERR_INVALID;
    if (a.A.dtype != a.B.dtype) return WP_ERR_DTYPE;
    const long long r = a.A.rows;
    if (r <= 0) return WP_ERR_INVALID;
    if (a.A.cols != K || a.B.cols != r || a.B.rows != cols) return WP_ERR_SHAPE;
    if (!std::isfinite(a.alpha) || !std::isfinite(a.strength)) return WP_ERR_INVALID;
    const double sc = a.alpha / static_cast<double>(r) * a.strength * request_scale;
    if (!std::isfinite(sc) || !std::isfinite(static_cast<float>(sc))) return WP_ERR_INVALID;
    if (a.A.dtype == WP_BF16 && r % 8) return WP_ERR_ALIGN;    // t [T, r] is a GEMM output
    if (a.bias_B && a.bias_B_dtype != WP_BF16 && a.bias_B_dtype != WP_FP32) return WP_ERR_DTYPE;
  }
  ExactLayout L;
  if (!exact_layout(X, W, ad, n, &L)) return WP_ERR_INVALID;
  if (L.total > 0 && (!workspace || ws_bytes < L.total)) return WP_ERR_WORKSPACE;
  if (L.total > 0 && !aligned16(workspace)) return WP_ERR_ALIGN;
  if (T == 0) return WP_OK;
  char* ws = static_cast<char*>(workspace);
  // base = bf16(X W^T + bias), straight into Y
  int rc = fwd_impl(X, W, bias, 1, false, nullptr, 0, 1.0, Y, nullptr, 0, stream);
  if (rc != WP_OK) return rc;
  void* t = ws + L.t;
  void* d = ws + L.d;
  for (int i = 0; i < n; ++i) {
    const wp_adapter& a = ad[i];
    const int r = static_cast<int>(a.A.rows);
    const int g = n_groups > 0 ? i : 0;
    ChainParams add{};
    add.mode = kChainAdd;
    add.T = T; add.N = cols;
    add.Y = static_cast<uint16_t*>(Y->data) + g * cols; add.ldy = Y->ld;
    add.d = d; add.ldd = cols;
    if (a.A.dtype == WP_FP32) {
      // FP32 GEMMs and scaling, added once
      const wp_out dout{d, WP_FP32, T, cols, cols};
      rc = fwd_impl(X, nullptr, nullptr, 1, false, &a, 1, request_scale, &dout, ws + L.fwd, L.fwd_bytes, stream);
      if (rc != WP_OK) return rc;
      add.d_f32 = 1;
    } else {
      const wp_out tout{t, WP_BF16, T, r, r};
      rc = fwd_impl(X, &a.A, nullptr, 1, false, nullptr, 0, 1.0, &tout, nullptr, 0, stream);
      if (rc != WP_OK) return rc;
      const wp_mat tin{t, WP_BF16, T, r, r, nullptr};
      const wp_mat vb{a.bias_B, a.bias_B_dtype, 1, cols, cols, nullptr};
      const wp_out dout{d, WP_BF16, T, cols, cols};
      rc = fwd_impl(&tin, &a.B, a.bias_B ? &vb : nullptr, 1, false, nullptr, 0, 1.0, &dout, nullptr, 0, stream);
      if (rc != WP_OK) return rc;
      const float scales[3] = {static_cast<float>(a.alpha / r), static_cast<float>(a.strength),
                               static_cast<float>(request_scale)};
      for (float c : scales) {
        if (skip_unit && c == 1.0f) continue;
        ChainParams sc{};
        sc.mode = kChainScale;
        sc.T = T; sc.N = cols;
        sc.Y = static_cast<uint16_t*>(d); sc.ldy = cols;
        sc.c = c;
        rc = launch_chain(sc, stream);
        if (rc != WP_OK) return rc;
      }
      add.d_f32 = 0;
    }
    rc = launch_chain(add, stream);
    if (rc != WP_OK) return rc;
  }
  return WP_OK;
}

// ------------------------------------------------------------------ host-buffer forward
// Workspace of lora_linear_fwd_host, in order (each region 256-byte aligned): X chunks
// [2][chunk, in] | Y chunks [2][chunk, out] (fp32-sized, whatever Y's type) | the
// forward's scratch for one chunk.
constexpr long long kHostChunkRows = 2048;

struct HostLayout {
  size_t x[2], y[2], fwd, fwd_bytes, total;
  long long chunk, out;
};

bool host_layout(const wp_mat* X, const wp_mat* W, const wp_adapter* ad, int n, HostLayout* L) {
  if (!X || X->rows < 0 || X->cols <= 0) return false;
  // out features: W's rows, or for a delta-only layer (no W, one group) the adapters' B rows
  const long long out = W ? W->rows : (n > 0 && ad ? ad[0].B.rows : 0);
  if (out <= 0) return false;
  L->out = out;
  L->chunk = std::min(kHostChunkRows, std::max<long long>(X->rows, 1));
  const size_t xs = static_cast<size_t>(X->dtype == WP_FP32 ? 4 : 2);
  size_t off = 0;
  for (int b = 0; b < 2; ++b) {
    L->x[b] = off;
    off += round256(static_cast<size_t>(L->chunk) * X->cols * xs);
  }
  for (int b = 0; b < 2; ++b) {
    L->y[b] = off;
    off += round256(static_cast<size_t>(L->chunk) * out * 4);
  }
  wp_mat xc = *X;
  xc.rows = L->chunk;
  xc.ld = X->cols;
  FwdPlan plan;
  plan_fwd(&xc, W, ad, n, &plan);
  L->fwd = off;
  L->fwd_bytes = fwd_workspace(&xc, plan);
  off += L->fwd_bytes;
  L->total = off;
  return true;
}

// Library-owned streams and events of the host-buffer forward, per device.
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, cmp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done_c = nullptr, done_d = nullptr;
  cudaEvent_t x_ready[2] = {}, x_free[2] = {}, y_ready[2] = {}, y_free[2] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipe[64];

int host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return WP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    cudaStream_t* ss[3] = {&hp.h2d, &hp.cmp, &hp.d2h};
    for (cudaStream_t* sp : ss) {
      e = cudaStreamCreateWithFlags(sp, cudaStreamNonBlocking);
      if (e != cudaSuccess) { set_last_cuda_error(e); return WP_ERR_CUDA; }
    }
    cudaEvent_t* es[11] = {&hp.start, &hp.done_c, &hp.done_d, &hp.x_ready[0], &hp.x_ready[1],
                           &hp.x_free[0], &hp.x_free[1], &hp.y_ready[0], &hp.y_ready[1],
                           &hp.y_free[0], &hp.y_free[1]};
    for (cudaEvent_t* ep : es) {
      e = cudaEventCreateWithFlags(ep, cudaEventDisableTiming);
      if (e != cudaSuccess) { set_last_cuda_error(e); return WP_ERR_CUDA; }
    }
    hp.ready = true;
  }
  *out = &hp;
  return WP_OK;
}

int host_impl(const wp_mat* X, const wp_mat* W, const wp_mat* bias, int n_groups,
              const wp_adapter* adapters, int n_adapters, double request_scale, const wp_out* Y,
              void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!valid_input(X, false) || !valid_output(Y)) return WP_ERR_INVALID;
  if (n_groups < 0 || n_adapters < 0 || (n_adapters > 0 && !adapters)) return WP_ERR_INVALID;
  if (n_groups > 0 && (!W || n_adapters != n_groups)) return WP_ERR_INVALID;
  if (Y->rows != X->rows) return WP_ERR_SHAPE;
  HostLayout L;
  if (!host_layout(X, W, adapters, n_adapters, &L)) return WP_ERR_INVALID;
  if (Y->cols != L.out) return WP_ERR_SHAPE;
  if (!workspace || ws_bytes < L.total) return WP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return WP_ERR_ALIGN;
  const long long T = X->rows, K = X->cols, N = Y->cols;
  if (T == 0) return WP_OK;
  HostPipe* hp = nullptr;
  int rc = host_pipe(&hp);
  if (rc != WP_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  const size_t xs = X->dtype == WP_FP32 ? 4 : 2, ys = Y->dtype == WP_FP32 ? 4 : 2;
  auto fail = [](cudaError_t e) { set_last_cuda_error(e); return WP_ERR_CUDA; };
  cudaError_t e = cudaEventRecord(hp->start, stream);
  if (e != cudaSuccess) return fail(e);
  for (cudaStream_t s2 : {hp->h2d, hp->cmp, hp->d2h})
    if ((e = cudaStreamWaitEvent(s2, hp->start, 0)) != cudaSuccess) return fail(e);
  const long long nchunks = (T + L.chunk - 1) / L.chunk;
  for (long long i = 0; i < nchunks; ++i) {
    const int b = static_cast<int>(i & 1);
    const long long r0 = i * L.chunk, rows = std::min(L.chunk, T - r0);
    void* xd = ws + L.x[b];
    void* yd = ws + L.y[b];
    // chunk i in: after the forward of chunk i - 2 has read this X buffer
    if (i >= 2 && (e = cudaStreamWaitEvent(hp->h2d, hp->x_free[b], 0)) != cudaSuccess) return fail(e);
    e = cudaMemcpy2DAsync(xd, K * xs, static_cast<const char*>(X->data) + r0 * X->ld * xs, X->ld * xs,
                          K * xs, rows, cudaMemcpyDefault, hp->h2d);
    if (e != cudaSuccess) return fail(e);
    if ((e = cudaEventRecord(hp->x_ready[b], hp->h2d)) != cudaSuccess) return fail(e);
    // forward of chunk i: after its X landed and chunk i - 2's Y left this Y buffer
    if ((e = cudaStreamWaitEvent(hp->cmp, hp->x_ready[b], 0)) != cudaSuccess) return fail(e);
    if (i >= 2 && (e = cudaStreamWaitEvent(hp->cmp, hp->y_free[b], 0)) != cudaSuccess) return fail(e);
    const wp_mat xc{xd, X->dtype, rows, K, K, nullptr};
    const wp_out yc{yd, Y->dtype, rows, N, N};
    rc = fwd_impl(&xc, W, bias, n_groups > 0 ? n_groups : 1, n_groups > 0, adapters, n_adapters,
                  request_scale, &yc, ws + L.fwd, L.fwd_bytes, hp->cmp);
    if (rc != WP_OK) return rc;
    if ((e = cudaEventRecord(hp->x_free[b], hp->cmp)) != cudaSuccess) return fail(e);
    if ((e = cudaEventRecord(hp->y_ready[b], hp->cmp)) != cudaSuccess) return fail(e);
    // chunk i out
    if ((e = cudaStreamWaitEvent(hp->d2h, hp->y_ready[b], 0)) != cudaSuccess) return fail(e);
    e = cudaMemcpy2DAsync(static_cast<char*>(Y->data) + r0 * Y->ld * ys, Y->ld * ys, yd, N * ys, N * ys,
                          rows, cudaMemcpyDefault, hp->d2h);
    if (e != cudaSuccess) return fail(e);
    if ((e = cudaEventRecord(hp->y_free[b], hp->d2h)) != cudaSuccess) return fail(e);
  }
  if ((e = cudaEventRecord(hp->done_c, hp->cmp)) != cudaSuccess) return fail(e);
  if ((e = cudaEventRecord(hp->done_d, hp->d2h)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(stream, hp->done_c, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(stream, hp->done_d, 0)) != cudaSuccess) return fail(e);
  return WP_OK;
}

}  // namespace

void set_last_cuda_error(cudaError_t e) { g_last_error = cudaGetErrorString(e); }

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

// ------------------------------------------------------------------ merge
// piper-offload docs, "LoRA merge": W <- W + sum_p s_p B_p A_p in place, every LoRA of the
// target taken as one update and rounded (re-encoded, for a 4-bit weight) once.  Each
// adapter's product runs on the fused kernel's base path with B_p as the token operand
// [out, r] and A_p^T as the weight [in, r] (K = r), its epilogue computing s * acc + R:
//   bf16 W, one adapter:  R = W, written back to W;
//   bf16 W, several:      U = s_1 acc_1 + W (fp32), U = s_p acc_p + U, W = s_n acc_n + U;
//   4-bit W:              U = fl32(W_eff), U = s_p acc_p + U for every adapter, requantise.
// Workspace, each region 256-byte aligned: per adapter A^T [in, r8] bf16 and, when B's rows
// are not 16-byte aligned, a copy of B [out, r8]; the fp32 U [out, in] when needed.
struct MergeLayout {
  size_t at[kMaxAd], bp[kMaxAd], u, total;
  bool copy_b[kMaxAd];
  bool need_u;
  int n_eff;
};

bool merge_layout(const wp_mat* W, const wp_adapter* ad, int n, double scale, MergeLayout* L) {
  *L = MergeLayout{};
  if (!W || n < 0 || n > kMaxAd || (n > 0 && !ad)) return false;
  const long long out = W->rows, in = W->cols;
  size_t off = 0;
  for (int i = 0; i < n; ++i) {
    const long long r = ad[i].A.rows, r8 = (r + 7) / 8 * 8;
    const double s = ad[i].alpha / static_cast<double>(r > 0 ? r : 1) * ad[i].strength * scale;
    if (static_cast<float>(s) != 0.0f) ++L->n_eff;
    L->at[i] = off;
    off += round256(static_cast<size_t>(in) * r8 * 2);
    L->copy_b[i] = !aligned16(ad[i].B.data) || ad[i].B.ld % 8 != 0;
    L->bp[i] = off;
    if (L->copy_b[i]) off += round256(static_cast<size_t>(out) * r8 * 2);
  }
  // the fp32 sum buffer: several adapters on a bf16 weight, or a 4-bit weight whose adapters
  // do not all fit the one-pass merge (a rank above 256)
  bool nf4_fused = W->dtype == WP_NF4;
  for (int i = 0; i < n; ++i)
    if ((ad[i].A.rows + kBK - 1) / kBK > kMergeTileMaxK) nf4_fused = false;
  L->need_u = (W->dtype == WP_NF4 && !nf4_fused) || (W->dtype != WP_NF4 && L->n_eff > 1);
  L->u = off;
  if (L->need_u) off += round256(static_cast<size_t>(out) * in * 4);
  L->total = L->n_eff > 0 ? off : 0;
  return true;
}

// One product pass: Y = s * (P Q^T) + R, P [rows, r] and Q [cols, r] K-major bf16.
int merge_pass(const void* P, long long ldp, const void* Q, long long ldq, long long rows, long long cols, int r,
               float s, const void* R, bool r_f32, long long ldr, void* Y, bool y_f32, long long ldy,
               cudaStream_t stream) {
  const int nk = (r + kBK - 1) / kBK;
  if (nk <= kMergeTileMaxK && cols % 8 == 0 && rows <= 0x7FFFFFFFLL && cols <= 0x7FFFFFFFLL) {
    // r up to 256: a CTA per 128 x 128 output tile (merge_tile_kernel)
    MergeTileMaps mm;
    std::memset(&mm, 0, sizeof(mm));
    int rc = make_map_bf16(&mm.p, P, r, rows, ldp, kBK, 128);
    if (rc != WP_OK) return rc;
    // residual and result of one dtype: both through the copy engine, 128-column tiles;
    // otherwise each thread reads and writes its row, 256-column tiles
    // (fp32 tiles 64 columns wide: two CTAs per SM still fit their 32 KiB residual tile)
    const bool staged = r_f32 == y_f32;
    const int nt = staged ? (y_f32 ? 64 : 128) : (cols >= 256 ? 256 : 128);
    rc = make_map_bf16(&mm.q, Q, r, cols, ldq, kBK, nt);
    if (rc != WP_OK) return rc;
    if (staged) {
      const int dt = y_f32 ? WP_FP32 : WP_BF16, bx = y_f32 ? 32 : 64;
      rc = make_map(&mm.r, dt, R, cols, rows, ldr, bx, 128);
      if (rc != WP_OK) return rc;
      rc = make_map(&mm.y, dt, Y, cols, rows, ldy, bx, 128);
      if (rc != WP_OK) return rc;
    }
    MergeTileParams mp{};
    mp.rows = static_cast<int>(rows); mp.cols = static_cast<int>(cols); mp.nk = nk; mp.s = s; mp.nt = nt;
    mp.staged = staged ? 1 : 0;
    mp.R = R; mp.ldr = ldr; mp.r_f32 = r_f32 ? 1 : 0;
    mp.Y = Y; mp.ldy = ldy; mp.y_f32 = y_f32 ? 1 : 0;
    mp.status = tc_status_ptr();
    mp.timeout_ns = wait_limit_ns();
    if (!mp.status) return record_cuda();
    return launch_merge_tile(mm, mp, stream);
  }
  TcParams p{};
  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  p.T = static_cast<int>(rows); p.K = r; p.N = static_cast<int>(cols);
  p.out_g = p.N; p.G = 1;
  p.nt_g = (p.N + kBN - 1) / kBN;
  p.m_shift = 0;
  p.r_blocks = (p.T + kPairM - 1) / kPairM;
  p.m_tiles = p.r_blocks;
  p.total_tiles = p.m_tiles * p.nt_g;
  p.k_blocks = (r + kBK - 1) / kBK;
  p.has_base = 1;
  p.Y = Y; p.ldy = ldy; p.y_f32 = y_f32 ? 1 : 0;
  p.acc_scale = s; p.resid = R; p.ld_resid = ldr; p.resid_f32 = r_f32 ? 1 : 0;
  p.timeout_ns = wait_limit_ns();
  p.stage_bytes = kATileBytes + kBHalfBytes;
  const size_t fixed = 1024 + 2 * kStgBytes + 512;
  p.stages = std::min<int>(kMaxStages, static_cast<int>((kSmemLimit - fixed) / p.stage_bytes));
  const size_t smem = fixed + static_cast<size_t>(p.stages) * p.stage_bytes;
  int rc = make_map_bf16(&maps.x, P, r, rows, ldp, kBK, kBM);
  if (rc != WP_OK) return rc;
  rc = make_map_bf16(&maps.w, Q, r, cols, ldq, kBK, 128);
  if (rc != WP_OK) return rc;
  rc = make_map(&maps.y, y_f32 ? WP_FP32 : WP_BF16, Y, cols, rows, ldy, y_f32 ? 32 : 64, kBM);
  if (rc != WP_OK) return rc;
  int pairs = tc_max_pairs(smem, false);
  if (pairs <= 0) return WP_ERR_CUDA;
  if (pairs > p.total_tiles) pairs = p.total_tiles;
  p.rlead = 1;
  return launch_tc_fwd(maps, p, 2 * pairs, smem, stream, false);
}

int merge_impl(const wp_mat* W, const wp_out* bias, const wp_adapter* ad, int n, double scale, void* workspace,
               size_t ws_bytes, cudaStream_t stream, bool stochastic = false, uint64_t seed = 0) {
  if (!W || !W->data || W->rows <= 0 || W->cols <= 0) return WP_ERR_INVALID;
  if (W->dtype != WP_BF16 && W->dtype != WP_NF4) return WP_ERR_DTYPE;
  if (!std::isfinite(scale)) return WP_ERR_INVALID;
  if (n < 0 || n > kMaxAd) return WP_ERR_UNSUPPORTED;
  if (n > 0 && !ad) return WP_ERR_INVALID;
  const long long out = W->rows, in = W->cols;
  if (out > 0x7FFFFFFFLL || in > 0x7FFFFFFFLL) return WP_ERR_UNSUPPORTED;
  const bool nf4 = W->dtype == WP_NF4;
  if (nf4 ? (in % 64 != 0 || W->ld != in || !W->absmax || !aligned16(W->absmax) || !aligned16(W->data))
          : (W->ld < in || W->ld % 8 != 0 || in % 8 != 0 || !aligned16(W->data)))
    return nf4 ? WP_ERR_SHAPE : WP_ERR_ALIGN;
  if (bias) {
    if (!bias->data) return WP_ERR_INVALID;
    if (bias->dtype != WP_BF16 && bias->dtype != WP_FP32) return WP_ERR_DTYPE;
    if (bias->rows * bias->cols != out) return WP_ERR_SHAPE;
  }
  float s_of[kMaxAd];
  BiasFoldParams fold{};                           // the adapters' legacy bias vectors
  for (int i = 0; i < n; ++i) {
    const wp_adapter& a = ad[i];
    if (!a.A.data || !a.B.data) return WP_ERR_INVALID;
    if (a.A.dtype != WP_BF16 || a.B.dtype != WP_BF16) return WP_ERR_DTYPE;
    const long long r = a.A.rows;
    if (r <= 0 || r > 0x7FFFFFFFLL) return WP_ERR_INVALID;
    if (a.A.cols != in || a.B.rows != out || a.B.cols != r || a.A.ld < in || a.B.ld < r) return WP_ERR_SHAPE;
    if (!std::isfinite(a.alpha) || !std::isfinite(a.strength)) return WP_ERR_INVALID;
    const double s = a.alpha / static_cast<double>(r) * a.strength * scale;
    if (!std::isfinite(s) || !std::isfinite(static_cast<float>(s))) return WP_ERR_INVALID;
    s_of[i] = static_cast<float>(s);
    if (a.bias_B) {
      if (a.bias_B_dtype != WP_BF16 && a.bias_B_dtype != WP_FP32) return WP_ERR_DTYPE;
      if (s_of[i] == 0.0f) continue;
      // a legacy vector needs a bias to land in: refused before anything is written
      if (!bias) return WP_ERR_INVALID;
      BiasFoldParams::Vec& v = fold.ad[fold.n++];
      v.v = a.bias_B;
      v.dtype = a.bias_B_dtype;
      v.s = s_of[i];
      v.col0 = 0;
      v.cols = static_cast<int>(out);
    }
  }
  MergeLayout L;
  if (!merge_layout(W, ad, n, scale, &L)) return WP_ERR_INVALID;
  if (L.n_eff == 0) return WP_OK;                 // nothing to add: the weight stays bit-identical
  if (!workspace || ws_bytes < L.total) return WP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return WP_ERR_ALIGN;
  char* ws = static_cast<char*>(workspace);
  float* U = reinterpret_cast<float*>(ws + L.u);
  void* wdata = const_cast<void*>(W->data);        // the weight is updated in place
  NF4Table tab;
  int rc = WP_OK;
  // a 4-bit weight with every adapter's rank up to 256: one pass (merge_nf4_kernel) that
  // dequantises, adds the adapters and requantises each block in registers
  bool fused = nf4;
  for (int i = 0; i < n && fused; ++i)
    if (s_of[i] != 0.0f && (ad[i].A.rows + kBK - 1) / kBK > kMergeTileMaxK) fused = false;
  MergeNF4Maps fm;
  MergeNF4Params fp{};
  if (fused) {
    // the 256-column form when the shape, the alignment and shared memory allow it; it reads
    // each A_p where it lies
    int ranks[kMaxAd], nr = 0;
    bool ok = aligned16(W->data) && aligned16(W->absmax);
    for (int i = 0; i < n; ++i)
      if (s_of[i] != 0.0f) {
        ranks[nr++] = static_cast<int>(ad[i].A.rows);
        ok = ok && aligned16(ad[i].A.data) && ad[i].A.ld % 8 == 0;
      }
    fp.wide = ok && merge_nf4_wide_plan(ranks, nr, in, &fp);
  }
  if (nf4) nf4_codebook_host(tab.level);
  if (nf4 && !fused) {
    rc = launch_nf4_to_f32(W->data, W->absmax, out * in, tab, U, stream);
    if (rc != WP_OK) return rc;
  }
  int done = 0;
  for (int i = 0; i < n; ++i) {
    if (s_of[i] == 0.0f) continue;
    const wp_adapter& a = ad[i];
    const int r = static_cast<int>(a.A.rows);
    const long long r8 = (r + 7) / 8 * 8;
    uint16_t* at = reinterpret_cast<uint16_t*>(ws + L.at[i]);
    if (!fp.wide) {
      rc = launch_transpose_bf16(a.A.data, a.A.ld, r, static_cast<int>(in), at, r8, stream);
      if (rc != WP_OK) return rc;
    }
    const void* bp = a.B.data;
    long long ldb = a.B.ld;
    if (L.copy_b[i]) {
      bp = ws + L.bp[i];
      ldb = r8;
      if (cudaMemcpy2DAsync(ws + L.bp[i], r8 * 2, a.B.data, a.B.ld * 2, static_cast<size_t>(r) * 2, out,
                            cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return record_cuda();
    }
    ++done;
    const bool first = done == 1, last = done == L.n_eff;
    if (fused) {
      const int k = fp.n++;
      rc = make_map_bf16(&fm.p[k], bp, r, out, ldb, kBK, 128);
      if (rc != WP_OK) return rc;
      rc = fp.wide ? make_map_bf16(&fm.q[k], a.A.data, in, r, a.A.ld, 64, fp.kbox[k])
                   : make_map_bf16(&fm.q[k], at, r, in, r8, kBK, 64);
      if (rc != WP_OK) return rc;
      fp.nk[k] = (r + kBK - 1) / kBK;
      fp.nk_max = std::max(fp.nk_max, fp.nk[k]);
      fp.s[k] = s_of[i];
      continue;
    }
    if (nf4) {
      rc = merge_pass(bp, ldb, at, r8, out, in, r, s_of[i], U, true, in, U, true, in, stream);
    } else if (L.n_eff == 1) {
      rc = merge_pass(bp, ldb, at, r8, out, in, r, s_of[i], wdata, false, W->ld, wdata, false, W->ld, stream);
    } else {
      const void* R = first ? W->data : static_cast<const void*>(U);
      void* Y = last ? wdata : static_cast<void*>(U);
      rc = merge_pass(bp, ldb, at, r8, out, in, r, s_of[i], R, !first, first ? W->ld : in, Y, !last,
                      last ? W->ld : in, stream);
    }
    if (rc != WP_OK) return rc;
  }
  if (fused) {
    fp.rows = static_cast<int>(out);
    fp.cols = static_cast<int>(in);
    fp.codes = static_cast<uint8_t*>(wdata);
    fp.absmax = const_cast<float*>(W->absmax);
    fp.tab = tab;
    if (!nf4_code_cells(tab, &fp.cells) || !nf4_level_cells(tab, &fp.lcells)) return WP_ERR_UNSUPPORTED;
    fp.stochastic = stochastic ? 1 : 0;
    fp.hold = g_hold_flags.load() ? 1 : 0;
    fp.seed_lo = static_cast<uint32_t>(seed);
    fp.seed_hi = static_cast<uint32_t>(seed >> 32);
    if (fp.wide) {
      rc = make_map_u8(&fm.codes, W->data, in / 2, out, in / 2, 128, 128, 128);
      if (rc == WP_OK) rc = make_map(&fm.am, WP_FP32, W->absmax, in / 64, out, in / 64, 16, 128, /*swizzle=*/0);
      if (rc != WP_OK) return rc;
    }
    fp.status = tc_status_ptr();
    fp.timeout_ns = wait_limit_ns();
    if (!fp.status) return record_cuda();
    rc = launch_merge_nf4(fm, fp, stream);
  } else if (nf4) {
    rc = stochastic ? launch_nf4_requant_stochastic(U, out * in, tab, wdata, const_cast<float*>(W->absmax), seed, stream)
                    : launch_nf4_requant(U, out * in, tab, wdata, const_cast<float*>(W->absmax), stream);
  }
  if (rc == WP_OK && fold.n > 0) {
    // bias <- bias + sum_p s_p bias_B_p, rounded once to the bias's dtype
    fold.bias = bias->data;
    fold.bias_dtype = bias->dtype;
    fold.N = static_cast<int>(out);
    rc = launch_bias_fold(fold, stream);
  }
  return rc;
}

}  // namespace wp

using namespace wp;

extern "C" {

int lora_linear_fwd(const wp_mat* X, const wp_mat* W, const wp_mat* bias,
                    const wp_adapter* adapters, int32_t n_adapters, double request_scale,
                    const wp_out* Y, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(X, W, bias, 1, false, adapters, n_adapters, request_scale, Y, workspace,
                  workspace_bytes, static_cast<cudaStream_t>(stream));
}

int lora_linear_fwd_grouped(const wp_mat* X, const wp_mat* W_stacked, const wp_mat* bias,
                            int32_t n_groups, const wp_adapter* adapters, double request_scale,
                            const wp_out* Y, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!W_stacked) return WP_ERR_INVALID;
  return fwd_impl(X, W_stacked, bias, n_groups, true, adapters, n_groups, request_scale, Y,
                  workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int lora_merge(const wp_mat* W, const wp_out* bias, const wp_adapter* adapters, int32_t n_adapters, double scale,
               void* workspace, size_t workspace_bytes, void* stream) {
  return merge_impl(W, bias, adapters, n_adapters, scale, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream));
}

int lora_merge_seeded(const wp_mat* W, const wp_out* bias, const wp_adapter* adapters, int32_t n_adapters,
                      double scale, uint64_t rounding_seed, void* workspace, size_t workspace_bytes, void* stream) {
  return merge_impl(W, bias, adapters, n_adapters, scale, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream), true, rounding_seed);
}

int lora_swiglu_fwd(const wp_mat* X, const wp_mat* W_gate_up, const wp_mat* bias,
                    const wp_adapter* adapters, double request_scale, const wp_out* H,
                    const wp_out* EG, void* workspace, size_t workspace_bytes, void* stream) {
  if (!W_gate_up || !H) return WP_ERR_INVALID;
  return fwd_impl(X, W_gate_up, bias, 2, true, adapters, 2, request_scale, H, workspace,
                  workspace_bytes, static_cast<cudaStream_t>(stream), nullptr, 0, false, true, EG);
}

int lora_swiglu_bwd(const wp_mat* dH, const wp_mat* EG, const wp_out* dEG, const wp_out* H,
                    void* stream) {
  if (!dH || !EG || !dEG) return WP_ERR_INVALID;
  const bool none = dH->rows == 0;                 // an empty batch needs no memory
  if (!none && (!dH->data || !EG->data || !dEG->data || (H && !H->data))) return WP_ERR_INVALID;
  if (dH->dtype != WP_BF16 || EG->dtype != WP_BF16 || dEG->dtype != WP_BF16 ||
      (H && H->dtype != WP_BF16))
    return WP_ERR_DTYPE;
  const long long T = dH->rows, F = dH->cols;
  if (T < 0 || F < 0 || EG->rows != T || EG->cols != 2 * F || dEG->rows != T || dEG->cols != 2 * F ||
      (H && (H->rows != T || H->cols != F)))
    return WP_ERR_SHAPE;
  if (dH->ld < F || EG->ld < 2 * F || dEG->ld < 2 * F || (H && H->ld < F)) return WP_ERR_SHAPE;
  if (F % 8 || dH->ld % 8 || EG->ld % 8 || dEG->ld % 8 || (H && H->ld % 8) || !aligned16(dH->data) ||
      !aligned16(EG->data) || !aligned16(dEG->data) || (H && !aligned16(H->data)))
    return WP_ERR_ALIGN;
  if (T * F == 0) return WP_OK;
  SwigluBwdParams q{};
  q.T = T; q.F = F;
  q.dh = static_cast<const uint16_t*>(dH->data); q.ld_dh = dH->ld;
  q.eg = static_cast<const uint16_t*>(EG->data); q.ld_eg = EG->ld;
  q.deg = static_cast<uint16_t*>(dEG->data); q.ld_deg = dEG->ld;
  q.h = H ? static_cast<uint16_t*>(H->data) : nullptr; q.ld_h = H ? H->ld : 0;
  return launch_swiglu_bwd(q, static_cast<cudaStream_t>(stream));
}

int lora_linear_bwd(const wp_mat* X, const wp_mat* W, const wp_mat* dY, int32_t n_groups,
                    const wp_adapter* adapters, double request_scale, const wp_out* dX,
                    const wp_out* dA, const wp_out* dB, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return bwd_impl(X, W, dY, n_groups, adapters, request_scale, dX, dA, dB, workspace,
                  workspace_bytes, static_cast<cudaStream_t>(stream));
}

int lora_dense_patch(void* param, int32_t param_dtype, int64_t param_numel, const void* payload,
                     int32_t payload_dtype, int64_t payload_numel, int32_t kind, double strength,
                     void* stream) {
  if ((!param || !payload) && param_numel != 0) return WP_ERR_INVALID;
  if (kind != WP_PATCH_ADD && kind != WP_PATCH_SET) return WP_ERR_INVALID;
  if (!std::isfinite(strength)) return WP_ERR_INVALID;
  if ((param_dtype != WP_BF16 && param_dtype != WP_FP32) ||
      (payload_dtype != WP_BF16 && payload_dtype != WP_FP32))
    return WP_ERR_DTYPE;
  if (param_numel < 0 || payload_numel != param_numel) return WP_ERR_SHAPE;
  return launch_dense_patch(param, param_dtype, payload, payload_dtype, param_numel, kind,
                            static_cast<float>(strength), static_cast<cudaStream_t>(stream));
}

size_t lora_workspace_size(int32_t op, const wp_mat* X, const wp_mat* W,
                           const wp_adapter* adapters, int32_t n_adapters) {
  if (op == WP_OP_MERGE) {
    MergeLayout L;
    return merge_layout(W, adapters, n_adapters, 1.0, &L) ? L.total : 0;
  }
  if (!X || n_adapters < 0 || (n_adapters > 0 && !adapters)) return 0;
  if (op == WP_OP_FWD || op == WP_OP_FWD_GROUPED || op == WP_OP_SWIGLU_FWD) {
    FwdPlan plan;
    plan_fwd(X, W, adapters, n_adapters, &plan);
    return fwd_workspace(X, plan);
  }
  if (op == WP_OP_BWD) {
    BwdLayout L;
    return bwd_layout(X, W, adapters, n_adapters, &L) ? L.total : 0;
  }
  if (op == WP_OP_FWD_EXACT) {
    ExactLayout L;
    return exact_layout(X, W, adapters, n_adapters, &L) ? L.total : 0;
  }
  if (op == WP_OP_FWD_HOST) {
    HostLayout L;
    return host_layout(X, W, adapters, n_adapters, &L) ? L.total : 0;
  }
  return 0;
}

int lora_linear_fwd_exact(const wp_mat* X, const wp_mat* W, const wp_mat* bias, int32_t n_groups,
                          const wp_adapter* adapters, int32_t n_adapters, double request_scale,
                          int32_t skip_unit_scales, const wp_out* Y, void* workspace, size_t workspace_bytes,
                          void* stream) {
  return exact_impl(X, W, bias, n_groups, adapters, n_adapters, request_scale, skip_unit_scales != 0, Y, workspace,
                    workspace_bytes, static_cast<cudaStream_t>(stream));
}

int lora_linear_fwd_host(const wp_mat* X_host, const wp_mat* W, const wp_mat* bias,
                         int32_t n_groups, const wp_adapter* adapters, int32_t n_adapters,
                         double request_scale, const wp_out* Y_host, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return host_impl(X_host, W, bias, n_groups, adapters, n_adapters, request_scale, Y_host,
                   workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

const char* lora_status_string(int status) {
  switch (status) {
    case WP_OK: return "ok";
    case WP_ERR_INVALID: return "invalid argument";
    case WP_ERR_SHAPE: return "shape mismatch";
    case WP_ERR_DTYPE: return "unsupported dtype";
    case WP_ERR_ALIGN: return "misaligned pointer or row pitch";
    case WP_ERR_WORKSPACE: return "workspace missing or too small";
    case WP_ERR_CUDA: return "CUDA error";
    case WP_ERR_TIMEOUT: return "device wait timed out";
    case WP_ERR_UNSUPPORTED: return "unsupported size or feature";
    default: return "unknown status";
  }
}

int lora_device_status(int32_t reset) {
  const int tc = tc_fwd_status(reset);
  return tc;
}

void lora_nf4_codebook(float out[16]) { nf4_codebook_host(out); }

int lora_set_wait_limit(uint64_t timeout_ns) {
  if (timeout_ns < 1000000ull || timeout_ns > 60000000000ull) return WP_ERR_INVALID;
  g_wait_limit_ns.store(timeout_ns);
  return WP_OK;
}

int lora_debug_hold_flags(int32_t on) {
  g_hold_flags.store(on ? 1 : 0);
  return WP_OK;
}

const char* lora_last_cuda_error(void) { return g_last_error.c_str(); }

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Forward without any device allocation by anyone.
//
// Some callers cannot hand the library a workspace and cannot allocate one either: hosts
// that own every byte of device memory through their own allocator and give plug-ins no
// allocation rights, fixed-budget inference servers, and latency-critical paths where
// cudaMalloc/cudaFree (which may synchronise the device) are not acceptable.  For them the
// forward's scratch (the bf16 s * X A^T rows of the adapters with a flag per 256-row
// block, and for FP32 adapters their bf16 pieces or fp32 projection) lives in a fixed
// array in this library's own device memory instead of a workspace.
//
// The array holds kNoAllocScratchBytes per device, for as long as the library is loaded.
// Host code must not pass the array's name to a kernel (on the host it is only a stand-in
// symbol); the device address is looked up once per device with cudaGetSymbolAddress, on
// the first call made with that device current, and passed to the kernels.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array for the current device (set-up on first use).
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return WP_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return WP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      set_last_cuda_error(e);
      return WP_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return WP_OK;
}

}  // namespace

extern "C" {

int lora_linear_fwd_noalloc(const wp_mat* X, const wp_mat* W, const wp_mat* bias,
                            const wp_adapter* adapters, int32_t n_adapters, double request_scale,
                            const wp_out* Y, void* stream) {
  if (!X || n_adapters < 0 || (n_adapters > 0 && !adapters)) return WP_ERR_INVALID;
  // The general path's own need decides; the few-token routes take the call only when their
  // partial sums fit the array as well (fwd_impl checks that against the bytes it is given)
  FwdPlan plan;
  plan_fwd(X, W, adapters, n_adapters, &plan);
  const size_t need = fwd_workspace(X, plan, /*min_only=*/true);
  if (need > kNoAllocScratchBytes) {
    char buf[160];
    snprintf(buf, sizeof(buf),
             "lora_linear_fwd_noalloc: needs %zu bytes of scratch, the static array holds %zu",
             need, kNoAllocScratchBytes);
    g_last_error = buf;
    return WP_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const bool any = need > 0 || plan.skinny_bytes > 0;
  if (any) {
    const int rc = noalloc_scratch(&scratch);
    if (rc != WP_OK) return rc;
  }
  return fwd_impl(X, W, bias, 1, false, adapters, n_adapters, request_scale, Y, scratch,
                  any ? kNoAllocScratchBytes : 0, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
