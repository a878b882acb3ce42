/*
 * weight_patches.h -- C ABI of the GB300 (sm_103a) dynamic-LoRA linear library.
 *
 * Computes the dynamic, unmerged LoRA linear
 *
 *     Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T,
 *     s_p = alpha_p / rank_p * strength_p * request_scale,
 *
 * and its siblings (stacked column groups, closed-form backward, dense patches) on
 * one GPU.  Sources of the operations, cited by page title and section:
 *   - sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM",
 *     Motivation and Modifications: the combined scale multiplies the rank-wide
 *     intermediate X A^T as a runtime value, the second low-rank GEMM accumulates
 *     straight onto the base output so the [tokens, out] delta is never stored, the
 *     bias lives in the base GEMM's epilogue, stacked q/k/v (gate/up) adapters take
 *     one update per column group, an FP32 adapter keeps FP32 GEMMs and adds once;
 *   - InvokeAI sidecar-patch article, sections 三-四: several patches on one layer are
 *     summed, each weighted by its own strength;
 *   - Unsloth fast_lora walkthrough, sections 2-4: 4-bit base weights dequantised
 *     into the matmul, and the closed-form backward dX, dA, dB;
 *   - FastVideo API docs, fastvideo.models.loader.lora_patch, DenseLoRAPatch:
 *     .diff / .diff_b additive deltas summed in float32 and .set_weight replacement.
 *
 * Conventions for every entry point:
 *   - All tensors are row-major.  X [T, in], W [out, in], A [r, in], B [out, r],
 *     bias [1, out], Y [T, out].  "ld" is the row pitch in elements.
 *   - Every data pointer is a DEVICE pointer on the current CUDA device; the caller
 *     owns all memory.  The library allocates no device memory, never synchronises
 *     and launches only on the caller's stream (`stream` is a cudaStream_t; NULL is
 *     the legacy default stream).  Inputs are never written.
 *   - Return value: WP_OK (0) or a negative WP_ERR_* code.  Argument checks run on
 *     the host before anything is launched; a rejected call launches nothing.
 *   - An empty batch (a matrix of zero rows: T = 0 tokens) is legal and its pointers may
 *     be null; such a call writes nothing, except lora_linear_bwd, whose dA and dB are
 *     then sums over no tokens and are set to zero.
 *   - A kernel whose bounded wait expires records WP_ERR_TIMEOUT in a device status
 *     word instead of hanging; read it with lora_device_status() after the stream has
 *     been synchronised.  The word is sticky until reset: while it reads WP_ERR_TIMEOUT,
 *     the outputs of every call made since the last reset are undefined (a kernel that
 *     gave up leaves its outputs partly written, and a later pass of the same call may
 *     have combined stale scratch), even though each of those calls returned WP_OK.
 */
#ifndef WEIGHT_PATCHES_H
#define WEIGHT_PATCHES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* storage types */
enum {
  WP_BF16 = 0, /* bfloat16 */
  WP_FP32 = 1, /* IEEE binary32 */
  WP_NF4 = 2   /* 4-bit NormalFloat: packed codes + one fp32 absmax per 64 elements */
};

/* status codes */
enum {
  WP_OK = 0,
  WP_ERR_INVALID = -1,     /* null pointer, non-finite alpha/strength/scale, rank <= 0, bad kind */
  WP_ERR_SHAPE = -2,       /* dimensions disagree (e.g. payload numel != parameter numel) */
  WP_ERR_DTYPE = -3,       /* unsupported storage type or combination */
  WP_ERR_ALIGN = -4,       /* a pointer or row pitch breaks the 16-byte alignment rule */
  WP_ERR_WORKSPACE = -5,   /* workspace missing or smaller than lora_workspace_size() */
  WP_ERR_CUDA = -6,        /* a CUDA runtime/driver call or a launch failed */
  WP_ERR_TIMEOUT = -7,     /* a bounded device wait expired (device status word) */
  WP_ERR_UNSUPPORTED = -8  /* a size beyond the documented limits */
};

/* dense-patch kinds */
enum { WP_PATCH_ADD = 0, WP_PATCH_SET = 1 };

/* An input matrix.  For WP_NF4, `data` holds rows*cols/2 bytes (row-major; byte k of
 * the stream holds element 2k in its high nibble and element 2k+1 in its low
 * nibble), `absmax` holds rows*cols/64 fp32 scales (one per 64 consecutive
 * elements), cols % 64 == 0, and `ld` must equal `cols`. */
typedef struct wp_mat {
  const void* data;
  int32_t dtype;
  int64_t rows, cols, ld;
  const float* absmax;
} wp_mat;

/* An output matrix (WP_BF16 or WP_FP32). */
typedef struct wp_out {
  void* data;
  int32_t dtype;
  int64_t rows, cols, ld;
} wp_out;

/* One low-rank patch.  A [r, in], B [out, r] (for grouped calls, out = the group's
 * width); both WP_BF16, or both WP_FP32 for an FP32 adapter.  The combined scale
 * s = alpha / r * strength * request_scale is formed on the host in double and
 * rounded once to fp32; an adapter whose s is exactly +-0 contributes nothing.
 * bias_B: the optional vector older PEFT/Wan adapters carry beside A and B (their
 * lora_B.bias; piper-offload docs, "LoRA merge"), [out] contiguous on the device,
 * WP_BF16 or WP_FP32 (bias_B_dtype), or NULL.  The forwards add s * bias_B to the
 * adapter's output columns (also when the layer has no bias of its own); lora_merge adds
 * it to the module's bias; the backward's dX, dA and dB do not depend on it. */
typedef struct wp_adapter {
  wp_mat A;
  wp_mat B;
  double alpha;
  double strength;
  const void* bias_B;
  int32_t bias_B_dtype;
} wp_adapter;

/* Operation ids for lora_workspace_size(). */
enum { WP_OP_FWD = 0, WP_OP_FWD_GROUPED = 1, WP_OP_BWD = 2, WP_OP_FWD_HOST = 3, WP_OP_SWIGLU_FWD = 4, WP_OP_MERGE = 5,
       WP_OP_FWD_EXACT = 6 };

/*
 * lora_linear_fwd -- Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T.
 * (sglang PR "Add the dynamic LoRA delta inside the second GEMM", Modifications;
 *  InvokeAI sidecar-patch article, section 四, for the sum over patches.)
 *
 *   X        [T, in], WP_BF16 (tensor-core path) or WP_FP32 (exact FP32 path).
 *   W        [out, in], WP_BF16 or WP_NF4 with a bf16 X, WP_FP32 with an fp32 X;
 *            NULL computes the low-rank delta only.
 *   bias     [1, out] WP_BF16 or WP_FP32, or NULL; added in the epilogue.  With adapters
 *            that carry a legacy bias_B (and a non-zero s), bias + sum_p s_p bias_B_p is
 *            first formed in fp32 in the workspace (the first ceil256(4 out) bytes) and
 *            that vector is what the epilogue adds.
 *   adapters n_adapters patches (0..12); bf16 adapters on a bf16 X run on the tensor
 *            cores.  FP32 adapters on a bf16 X run there too, as three bf16 pieces per
 *            factor (every product above 2^-24 of the leading one is kept), when the
 *            call's rank columns allow; otherwise they run in FP32 on the CUDA cores.
 *            Either way their terms join the same FP32 accumulator before the single
 *            output rounding.
 *   Y        [T, out] WP_BF16 or WP_FP32, ld >= out; must not overlap the inputs.
 *   workspace device scratch of at least lora_workspace_size(WP_OP_FWD, ...) bytes
 *            (may be NULL when that size is 0).
 * Alignment (tensor-core path): every base pointer 16-byte aligned, every ld a
 * multiple of 8 elements (bf16) / 4 (fp32), in % 8 == 0, out % 8 == 0.
 * Limits (tensor-core path): at most 8 adapters on the tensor cores, each of rank <= 256.
 * A bf16 adapter counts ceil(r / 16) * 16 rank columns, an FP32 adapter as pieces
 * 3 * ceil(r / 16) * 16.  When the adapters' rank columns fit one 256-column accumulator,
 * s X A^T of all of them comes from one extra pass over X per 256 token rows; otherwise
 * the adapters (whole) are grouped into several such rank passes of at most 256 columns
 * each (e.g. three rank-128 q/k/v adapters: two passes), and FP32 adapters then take the
 * CUDA-core route (at most 4 of them), as they do whenever their pieces do not fit.
 * Few tokens (bf16 X and adapters): one to four tokens with in % 256 == 0 stream the
 * weight once on the CUDA cores; up to 64 tokens with a WP_NF4 weight (4 with bf16)
 * stream it through swapped tensor-core MMAs.  Both keep the same W_eff and the single
 * bf16 rounding of s X A^T, sum in fp32, and leave fp32 partial sums in the workspace
 * (lora_workspace_size counts them).
 */
int lora_linear_fwd(const wp_mat* X, const wp_mat* W, const wp_mat* bias,
                    const wp_adapter* adapters, int32_t n_adapters, double request_scale,
                    const wp_out* Y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * lora_linear_fwd_grouped -- stacked column groups (q/k/v, gate/up):
 *   Y[:, g*out_g:(g+1)*out_g] = X W_g^T + bias_g + s_g (X A_g^T) B_g^T,
 * with W_stacked = [W_0; ...; W_{G-1}] of shape [G*out_g, in] and one adapter per
 * group (adapters[g], B_g of shape [out_g, r_g]).
 * (sglang PR, Modifications: one update per group on column views of the output;
 *  Unsloth walkthrough, section 4, LoRA_QKV.)
 * Same dtypes, alignment and ownership as lora_linear_fwd; 1 <= n_groups <= 8,
 * out_g % 8 == 0.
 */
int lora_linear_fwd_grouped(const wp_mat* X, const wp_mat* W_stacked, const wp_mat* bias,
                            int32_t n_groups, const wp_adapter* adapters, double request_scale,
                            const wp_out* Y, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * lora_linear_fwd_host -- lora_linear_fwd (n_groups == 0) or lora_linear_fwd_grouped
 * (n_groups >= 1) with X and Y in host memory, for callers whose activations live on the
 * host.  A deployment variant with no counterpart in the pages.
 *
 * The rows are processed in chunks of 2048: the host-to-device copy of chunk i + 1, the
 * forward of chunk i and the device-to-host copy of chunk i - 1 run at the same time on
 * three streams owned by the library (created on the first call per device); the call
 * returns at once and `stream` waits for the whole operation.  X and Y should be pinned
 * (page-locked) for the copies to overlap; pageable memory works, serialised.
 *   X_host  [T, in] WP_BF16 (or WP_FP32 for the all-FP32 layer), host pointer.
 *   W, bias, adapters, request_scale: as lora_linear_fwd / lora_linear_fwd_grouped (device).
 *   Y_host  [T, out] WP_BF16 or WP_FP32, host pointer, ld >= out.
 *   workspace  device scratch of at least lora_workspace_size(WP_OP_FWD_HOST, X_host, W,
 *              adapters, n_adapters) bytes: two device chunks of X and of Y, and the
 *              forward's own scratch for one chunk.
 * Errors as lora_linear_fwd; a failure found after copies were queued still returns its
 * status, and `stream` then does not wait for the internal streams.
 */
int lora_linear_fwd_host(const wp_mat* X_host, const wp_mat* W, const wp_mat* bias,
                         int32_t n_groups, const wp_adapter* adapters, int32_t n_adapters,
                         double request_scale, const wp_out* Y_host, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * lora_merge -- bake adapters into the base weight in place (piper-offload docs, "LoRA
 * merge" and "Quantized weight support"; the PEFT merge):
 *     W <- W + sum_p s_p B_p A_p,   s_p = alpha_p / r_p * strength_p * scale,
 *     bias <- bias + sum_p s_p bias_B_p   (adapters that carry the legacy vector),
 * every adapter of the call taken as one update, accumulated in fp32 and rounded once:
 *   W WP_BF16 [out, in] (device): bf16_rne(fl32(W) + ...);
 *   W WP_NF4 (codes [out, in/2] and absmax [out*in/64], device, both rewritten): dequantised
 *     to W_eff, the update added in fp32, re-encoded with deterministic round-to-nearest: per
 *     64-element block absmax' = max |u|, code = the nearest level of u / absmax' (a value on
 *     a midpoint between two levels takes the lower code), an all-zero block keeps scale 0.
 *   adapters: bf16 A [r, in], B [out, r]; strength 0 skips one; scale -1 undoes an earlier
 *   merge of the same adapters up to the roundings.
 *   workspace: lora_workspace_size(WP_OP_MERGE, NULL, W, adapters, n) bytes (A^T copies, and
 *   an fp32 [out, in] buffer for several adapters on a bf16 W, or for a 4-bit W with a rank
 *   above 256; a 4-bit W with ranks up to 256 is dequantised, updated and requantised block by
 *   block in one pass, with the same arithmetic).
 *   bias: the module's bias [out] (WP_BF16 or WP_FP32, device, rewritten in place) or NULL.
 *   The legacy vectors are added in fp32 in call order (each term fl32(s_p * v)) and the
 *   sum rounded once to the bias's dtype; for one adapter that is the dense patch's add.
 * Errors: WP_ERR_SHAPE, WP_ERR_DTYPE (fp32 adapters), WP_ERR_ALIGN (bf16 W rows must be
 * 16-byte aligned), WP_ERR_WORKSPACE; WP_ERR_INVALID, before anything is written, when an
 * adapter with a non-zero s carries a legacy vector and bias is NULL (the merge does not
 * create a bias the module does not have).  With no non-zero adapter nothing is launched.
 */
int lora_merge(const wp_mat* W, const wp_out* bias, const wp_adapter* adapters, int32_t n_adapters,
               double scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * lora_merge_seeded -- lora_merge with the stochastic re-encoding of a 4-bit weight
 * (piper-offload docs, "LoRA merge": the default for quantised merges, so that updates smaller
 * than one quantisation step are not rounded away systematically).  The block scales are the
 * deterministic ones (absmax' = max |u|); only each code is sampled, between the two levels
 * around x = fl32(u / absmax'): x on a level keeps that level's code, otherwise the upper
 * level lo < x < hi is taken when U * w < d * 2^23 (d = fl32(x - lo), w = fl32(hi - lo)), U
 * being the element's 23-bit draw: word e % 4 of Philox4x32-10 (Salmon et al., SC 2011) of
 * counter (e / 4 as two 32-bit words, 0, 0) under key (the seed's low and high 32 bits), shifted
 * right by 9, e = row * in + column the element's logical index -- so the codes depend on the
 * seed and the data only, not on the launch.  The same seed gives the same codes.  A bf16 W has
 * no code to sample: the call is lora_merge.  Arguments, workspace and errors as lora_merge.
 */
int lora_merge_seeded(const wp_mat* W, const wp_out* bias, const wp_adapter* adapters, int32_t n_adapters,
                      double scale, uint64_t rounding_seed, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * lora_swiglu_fwd -- the front half of a SwiGLU LoRA MLP in one pass: the gate and up
 * LoRA linears and the activation,
 *     e = X W_gate^T + bias_gate + s_g (X A_g^T) B_g^T,
 *     g = X W_up^T   + bias_up   + s_u (X A_u^T) B_u^T,
 *     h = silu(e) g,   silu(e) = e / (1 + exp(-e)).
 * (Unsloth fast_lora walkthrough, section 4, LoRA_MLP forward: e and g by two LoRA
 *  matmuls, h by the SwiGLU kernel, e and g kept for the backward.)
 *   X [T, in] WP_BF16; W_gate_up [2F, in] WP_BF16 or WP_NF4, gate rows 0..F-1 then up
 *   rows F..2F-1; bias [2F] (gate then up) or NULL; adapters[0] the gate adapter
 *   (B [F, r]), adapters[1] the up adapter (strength 0 disables one); bf16 adapters, or
 *   FP32 ones small enough to ride as bf16 pieces.
 *   H [T, F] WP_BF16 output.  EG [T, 2F] WP_BF16 or NULL: receives e | g.
 * e and g are rounded to bf16 once (EG holds exactly those values, bit-equal to
 * lora_linear_fwd_grouped with n_groups = 2), h = bf16(silu(e) * g) from them, so the
 * h that lora_swiglu_bwd recomputes from EG is bit-equal to H.
 *   workspace: lora_workspace_size(WP_OP_SWIGLU_FWD, X, W_gate_up, adapters, 2) bytes.
 * Limits: as lora_linear_fwd_grouped; F % 8 == 0.  Errors as lora_linear_fwd.
 */
int lora_swiglu_fwd(const wp_mat* X, const wp_mat* W_gate_up, const wp_mat* bias,
                    const wp_adapter* adapters, double request_scale, const wp_out* H,
                    const wp_out* EG, void* workspace, size_t workspace_bytes, void* stream);

/*
 * lora_swiglu_bwd -- the SwiGLU step of the LoRA MLP backward, elementwise.  From the
 * gradient dH at h (the dX of the down projection) and the saved e | g:
 *     f = silu(e),  dg = dH f,  de = dH g sigmoid(e) (1 + e (1 - sigmoid(e))),
 * and, when H is given, h = f g again (for the down adapter's gradients).
 * (Unsloth fast_lora walkthrough, section 4, LoRA_MLP backward: one kernel gives h and
 *  the gradients at g and e.)
 *   dH [T, F], EG [T, 2F] WP_BF16 inputs; dEG [T, 2F] WP_BF16 output, de | dg (the
 *   stacked output gradient for the grouped gate/up backward); H [T, F] WP_BF16 or NULL.
 * Every product is one float32 rounding, each output one bf16 rounding.
 * Errors: WP_ERR_SHAPE, WP_ERR_DTYPE (not bf16), WP_ERR_ALIGN (16-byte bases, F and
 * row pitches multiples of 8 elements).  Outputs must not overlap the inputs.
 */
int lora_swiglu_bwd(const wp_mat* dH, const wp_mat* EG, const wp_out* dEG, const wp_out* H,
                    void* stream);

/*
 * lora_linear_bwd -- closed-form gradients of Y = X W_g^T + s_g (X A_g^T) B_g^T over
 * n_groups column groups (n_groups = 1 for a plain layer), with G_g = dY_g B_g:
 *     dX   = sum_g dY_g W_g + s_g G_g A_g          [T, in]
 *     dA_g = s_g G_g^T X                          [r_g, in]
 *     dB_g = s_g dY_g^T (X A_g^T)                 [out_g, r_g]
 * (Unsloth fast_lora walkthrough, sections 2 and 4: dX, dA, dB by hand, no
 *  autograd graph, only X kept from the forward.)
 *   X [T, in] WP_BF16; W [G*out_g, in] WP_BF16 or WP_NF4; dY [T, G*out_g] WP_BF16.
 *   dX: WP_BF16 or WP_FP32 output, or NULL to skip; dA[g], dB[g]: WP_FP32 outputs.
 *   dA/dB are overwritten (not accumulated).
 * Limits: bf16 adapters, r_g <= 128 each (any sum over the groups); in % 8 == 0 and
 * out_g % 8 == 0.
 */
int lora_linear_bwd(const wp_mat* X, const wp_mat* W, const wp_mat* dY, int32_t n_groups,
                    const wp_adapter* adapters, double request_scale, const wp_out* dX,
                    const wp_out* dA, const wp_out* dB, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * lora_dense_patch -- the dense half of an adapter, applied in place to `param`.
 * (FastVideo API docs, fastvideo.models.loader.lora_patch, DenseLoRAPatch.apply_to
 *  and replacement_for.)
 *   kind WP_PATCH_ADD (.diff / .diff_b): param = cast(fp32(param) + fp32(payload) * k)
 *   kind WP_PATCH_SET (.set_weight):     param = cast(fp32(payload) * k)
 * where k = (float)strength, the product and the sum are separate float32 roundings
 * (no fused multiply-add) and cast is round-to-nearest-even into param_dtype.
 *   param: param_numel elements of param_dtype (WP_BF16 or WP_FP32), device.
 *   payload: payload_numel elements of payload_dtype (WP_BF16 or WP_FP32), device.
 * Errors: WP_ERR_SHAPE if payload_numel != param_numel; WP_ERR_INVALID for a
 * non-finite strength or unknown kind.  param and payload must not overlap.
 */
int lora_dense_patch(void* param, int32_t param_dtype, int64_t param_numel,
                     const void* payload, int32_t payload_dtype, int64_t payload_numel,
                     int32_t kind, double strength, void* stream);

/*
 * lora_linear_fwd_exact -- the unfused dynamic-LoRA chain, the "exact" tier.
 * (sglang PR "[diffusion] Add the dynamic LoRA delta inside the second GEMM", Motivation:
 *  the chain every dynamic layer ran before the fused design; Modifications: the exact
 *  tier keeps that chain and skips multiplications by a unit scale, which leaves every bit
 *  of the output as it was.)
 *     Y = bf16(X W^T + bias)
 *     for each adapter p, in order (its column group when n_groups > 0):
 *       t = bf16(X A_p^T);  d = bf16(t B_p^T [+ bias_B,p])
 *       d = bf16(d * c) for c = fl32(alpha_p / r_p), fl32(strength_p), fl32(request_scale)
 *       Y = bf16(Y + d)
 *   An FP32 adapter keeps its two GEMMs and its scaling in FP32 (s = alpha/r * strength *
 *   request_scale formed in double) and is added once: Y = bf16(Y + fl32 delta).
 *   skip_unit_scales != 0 skips each scale multiplication whose c is exactly 1.0 (the PR's
 *   exact tier); 0 runs every one (the chain before the PR).  The two give bit-identical Y.
 *   Every elementwise step is the correctly rounded bf16 of its exact result; the GEMMs sum
 *   in fp32 on the tensor cores.  This path materialises t and d (it is the reference the
 *   fused lora_linear_fwd improves on), so it is slower by design.
 *   X [T, in] WP_BF16; W [n_groups * out_g, in] (or [out, in]) WP_BF16 or WP_NF4; bias as
 *   lora_linear_fwd; adapters: n_adapters (== n_groups when n_groups > 0); Y [T, out] WP_BF16.
 *   workspace: lora_workspace_size(WP_OP_FWD_EXACT, X, W, adapters, n_adapters) bytes.
 * Limits: bf16 adapters of rank r % 8 == 0 (t is a GEMM output); out_g % 8 == 0; the
 * alignment rules of lora_linear_fwd.  Errors as lora_linear_fwd.
 */
int lora_linear_fwd_exact(const wp_mat* X, const wp_mat* W, const wp_mat* bias, int32_t n_groups,
                          const wp_adapter* adapters, int32_t n_adapters, double request_scale,
                          int32_t skip_unit_scales, const wp_out* Y, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * lora_linear_fwd_noalloc -- lora_linear_fwd for callers that cannot provide or allocate
 * device scratch memory.  The pages have no counterpart: this is a deployment variant.
 *
 * Who needs it: code embedded in a host that owns all device memory through its own
 * allocator and gives plug-ins no allocation rights, fixed-budget inference servers, and
 * latency-critical paths where cudaMalloc/cudaFree (which may synchronise the device)
 * are not acceptable.  Such a caller still passes its inputs and output; the scratch that
 * lora_workspace_size(WP_OP_FWD, ...) reports (on the tensor-core path about T x sum of the
 * ranks rounded up to 16 x 2 bytes for the bf16 s * X A^T rows, plus the FP32 adapters'
 * share; on the all-FP32 path T x sum of the ranks floats) comes from a fixed 4 MiB array
 * inside the library, held on every device that uses it until the process exits.  The
 * call allocates nothing.
 *
 * Same arguments, dtypes, alignment rules and errors as lora_linear_fwd, minus the
 * workspace.  A call whose general path would need more than 4 MiB of scratch (the
 * minimum above, not counting the few-token routes' partial sums) is rejected with
 * WP_ERR_WORKSPACE before anything is launched (lora_last_cuda_error() says how much was
 * needed).  A call of 1 to 64 tokens takes a few-token route only when that route's fp32
 * partial sums (splits x T x (out + sum of the ranks rounded up to 16) x 4 bytes) fit the
 * array as well; otherwise it runs on the general path, with the same results within the
 * tolerances of lora_linear_fwd.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any stream
 * capture.  Every call on a device shares the one array and leaves its contents behind
 * (the call clears the few flags it needs on its stream; every other scratch element is
 * written before it is read): calls whose kernels overlap on the GPU, e.g. on two streams
 * at once, race on it and must be serialised by the caller.
 */
int lora_linear_fwd_noalloc(const wp_mat* X, const wp_mat* W, const wp_mat* bias,
                            const wp_adapter* adapters, int32_t n_adapters, double request_scale,
                            const wp_out* Y, void* stream);

/* Bytes of device workspace the given call needs (0 if none).  `op` is WP_OP_*;
 * the other arguments are those of the call (adapters: n_adapters, or n_groups). */
size_t lora_workspace_size(int32_t op, const wp_mat* X, const wp_mat* W,
                           const wp_adapter* adapters, int32_t n_adapters);

/* Human-readable text for a status code (static storage). */
const char* lora_status_string(int status);

/* Reads (and, if `reset` != 0, clears) the device status word of the current device:
 * WP_OK or WP_ERR_TIMEOUT.  Synchronous: call after the stream has finished. */
int lora_device_status(int32_t reset);

/* How long every bounded device wait of the library's kernels spins (mbarriers, the fused
 * forward's row-block flags) before the kernel records WP_ERR_TIMEOUT in the device status
 * word, drains its own copies in flight, frees its tensor memory and returns.  Applies to
 * calls made after it, process-wide.  Default 2 s; accepted range 1 ms .. 60 s, otherwise
 * WP_ERR_INVALID and the setting is unchanged.  Not in the pages: a safety bound of this
 * library's persistent kernels. */
int lora_set_wait_limit(uint64_t timeout_ns);

/* Test hook for the timeout path (not in the pages): while `on` is non-zero, the tiles of
 * every fused forward launched afterwards wait for one more release of their row-block flag
 * than any rank item gives, and every one-pass 4-bit merge (ranks up to 256) leaves the MMAs
 * of its CTAs' last jobs unissued, so those bounded waits run out (after
 * lora_set_wait_limit's limit) and the call's outputs are left undefined;
 * lora_device_status() then reads WP_ERR_TIMEOUT.  Process-wide; 0 restores normal
 * operation.  Always returns WP_OK. */
int lora_debug_hold_flags(int32_t on);

/* The library's 16 NormalFloat levels in ascending order (host memory, fp32). */
void lora_nf4_codebook(float out[16]);

/* The last CUDA error text the library saw on this host thread ("" if none). */
const char* lora_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* WEIGHT_PATCHES_H */
