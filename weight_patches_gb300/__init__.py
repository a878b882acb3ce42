"""weight_patches_gb300 -- the dynamic, unmerged LoRA linear on GB300 (sm_103a).

A thin ctypes binding over ``libweight_patches_gb300.so`` (C ABI in
``include/weight_patches.h``).  The functions here only marshal arguments: torch
tensors supply device memory and the current CUDA stream; every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the shared
library has not been built, importing it raises.

Entry points (same names as the C ABI):
    lora_linear_fwd          Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T
    lora_linear_fwd_grouped  stacked column groups, one adapter per group
    lora_linear_bwd          closed-form dX, dA, dB
    lora_linear_fwd_exact    the unfused bf16 chain (the "exact" tier), unit scales skipped or not
    lora_dense_patch         .diff / .diff_b (add) and .set_weight (replace), in place
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libweight_patches_gb300.so")

WP_BF16, WP_FP32, WP_NF4 = 0, 1, 2
WP_PATCH_ADD, WP_PATCH_SET = 0, 1
WP_OP_FWD, WP_OP_FWD_GROUPED, WP_OP_BWD, WP_OP_FWD_HOST, WP_OP_SWIGLU_FWD, WP_OP_MERGE, WP_OP_FWD_EXACT = range(7)
STATUS = {0: "WP_OK", -1: "WP_ERR_INVALID", -2: "WP_ERR_SHAPE", -3: "WP_ERR_DTYPE",
          -4: "WP_ERR_ALIGN", -5: "WP_ERR_WORKSPACE", -6: "WP_ERR_CUDA", -7: "WP_ERR_TIMEOUT",
          -8: "WP_ERR_UNSUPPORTED"}


class WpMat(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ld", ctypes.c_int64), ("absmax", ctypes.c_void_p)]


class WpOut(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ld", ctypes.c_int64)]


class WpAdapter(ctypes.Structure):
    _fields_ = [("A", WpMat), ("B", WpMat), ("alpha", ctypes.c_double),
                ("strength", ctypes.c_double), ("bias_B", ctypes.c_void_p), ("bias_B_dtype", ctypes.c_int32)]


class WeightPatchesError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = _load()
        msg = lib.lora_status_string(status).decode()
        cuda = lib.lora_last_cuda_error().decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg}){' / ' + cuda if cuda else ''}")


_LIB = None


def _load():
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()'"
            " or python weight_patches_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, D, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_size_t
    pm, po, pa = ctypes.POINTER(WpMat), ctypes.POINTER(WpOut), ctypes.POINTER(WpAdapter)
    lib.lora_linear_fwd.argtypes = [pm, pm, pm, pa, I32, D, po, P, SZ, P]
    lib.lora_linear_fwd_grouped.argtypes = [pm, pm, pm, I32, pa, D, po, P, SZ, P]
    lib.lora_linear_fwd_noalloc.argtypes = [pm, pm, pm, pa, I32, D, po, P]
    lib.lora_linear_fwd_host.argtypes = [pm, pm, pm, I32, pa, I32, D, po, P, SZ, P]
    lib.lora_linear_fwd_exact.argtypes = [pm, pm, pm, I32, pa, I32, D, I32, po, P, SZ, P]
    lib.lora_linear_bwd.argtypes = [pm, pm, pm, I32, pa, D, po, po, po, P, SZ, P]
    lib.lora_swiglu_fwd.argtypes = [pm, pm, pm, pa, D, po, po, P, SZ, P]
    lib.lora_merge.argtypes = [pm, po, pa, I32, D, P, SZ, P]
    lib.lora_merge_seeded.argtypes = [pm, po, pa, I32, D, ctypes.c_uint64, P, SZ, P]
    lib.lora_swiglu_bwd.argtypes = [pm, pm, po, po, P]
    lib.lora_dense_patch.argtypes = [P, I32, I64, P, I32, I64, I32, D, P]
    lib.lora_workspace_size.argtypes = [I32, pm, pm, pa, I32]
    lib.lora_workspace_size.restype = SZ
    lib.lora_status_string.argtypes = [ctypes.c_int]
    lib.lora_status_string.restype = ctypes.c_char_p
    lib.lora_device_status.argtypes = [I32]
    lib.lora_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.lora_debug_hold_flags.argtypes = [I32]
    lib.lora_nf4_codebook.argtypes = [ctypes.POINTER(ctypes.c_float)]
    lib.lora_nf4_codebook.restype = None
    lib.lora_last_cuda_error.restype = ctypes.c_char_p
    for name in ("lora_linear_fwd", "lora_linear_fwd_grouped", "lora_linear_bwd", "lora_dense_patch",
                 "lora_device_status", "lora_linear_fwd_noalloc", "lora_linear_fwd_host",
                 "lora_linear_fwd_exact", "lora_set_wait_limit", "lora_debug_hold_flags"):
        getattr(lib, name).restype = ctypes.c_int
    _LIB = lib
    return lib


def lib():
    """The loaded shared library (ctypes.CDLL)."""
    return _load()


# ------------------------------------------------------------------------- marshalling
@dataclass
class NF4Weight:
    """A 4-bit NormalFloat weight [rows, cols]: ``packed`` uint8 [rows, cols // 2] (element
    2k in the high nibble of byte k), ``absmax`` fp32 [rows * cols // 64]."""

    packed: torch.Tensor
    absmax: torch.Tensor
    rows: int
    cols: int


@dataclass
class Adapter:
    """One low-rank patch: A [r, in], B [out, r] (bf16, or fp32 for an FP32 adapter), and the
    optional legacy ``bias_B`` [out] (bf16 or fp32) older adapters carry as lora_B.bias: the
    forwards add s * bias_B to the patch's output columns, ``lora_merge`` adds it to the
    module's bias."""

    A: torch.Tensor
    B: torch.Tensor
    alpha: float
    strength: float = 1.0
    bias_B: Optional[torch.Tensor] = None


_DT = {torch.bfloat16: WP_BF16, torch.float32: WP_FP32}


def _mat(t) -> Optional[WpMat]:
    if t is None:
        return None
    if isinstance(t, NF4Weight):
        if not (t.packed.is_contiguous() and t.absmax.is_contiguous()):
            raise ValueError("NF4Weight tensors must be contiguous")
        return WpMat(t.packed.data_ptr(), WP_NF4, t.rows, t.cols, t.cols, t.absmax.data_ptr())
    if t.dim() == 1:
        return WpMat(t.data_ptr(), _DT[t.dtype], 1, t.shape[0], t.shape[0], None)
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D row-major tensor (stride(1) == 1)")
    return WpMat(t.data_ptr(), _DT[t.dtype], t.shape[0], t.shape[1], t.stride(0), None)


def _out(t: torch.Tensor) -> WpOut:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D row-major output tensor")
    return WpOut(t.data_ptr(), _DT[t.dtype], t.shape[0], t.shape[1], t.stride(0))


def _adapters(adapters: Sequence[Adapter]):
    arr = (WpAdapter * max(1, len(adapters)))()
    for i, a in enumerate(adapters):
        vb = getattr(a, "bias_B", None)
        if vb is not None and not vb.is_contiguous():
            raise ValueError("bias_B must be contiguous")
        arr[i] = WpAdapter(_mat(a.A), _mat(a.B), float(a.alpha), float(a.strength),
                           vb.data_ptr() if vb is not None else None,
                           _DT[vb.dtype] if vb is not None else WP_BF16)
    return arr


def _ref(m):
    return ctypes.byref(m) if m is not None else None


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(status: int, where: str):
    if status != 0:
        raise WeightPatchesError(status, where)


def _workspace(op, xm, wm, arr, n, device, workspace):
    need = _load().lora_workspace_size(op, ctypes.byref(xm), _ref(wm), arr, n)
    if need == 0:
        return None, 0
    if workspace is not None and workspace.numel() * workspace.element_size() >= need:
        return workspace, need
    return torch.empty(need, dtype=torch.uint8, device=device), need


def lora_workspace_size(op: int, X, W, adapters: Sequence[Adapter]) -> int:
    xm, wm, arr = _mat(X), _mat(W), _adapters(adapters)
    return _load().lora_workspace_size(op, _ref(xm), _ref(wm), arr, len(adapters))


def _out_features(X, W, adapters):
    if W is not None:
        return W.rows if isinstance(W, NF4Weight) else W.shape[0]
    return adapters[0].B.shape[0]


def lora_linear_fwd(X: torch.Tensor, W, bias: Optional[torch.Tensor], adapters: Sequence[Adapter],
                    request_scale: float = 1.0, out: Optional[torch.Tensor] = None,
                    out_dtype: torch.dtype = torch.bfloat16,
                    workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Y = X W^T + bias + sum_p s_p (X A_p^T) B_p^T with s_p = alpha/r * strength * request_scale."""
    if out is None:
        out = torch.empty(X.shape[0], _out_features(X, W, adapters), dtype=out_dtype, device=X.device)
    xm, wm, bm, arr, ym = _mat(X), _mat(W), _mat(bias), _adapters(adapters), _out(out)
    ws, nbytes = _workspace(WP_OP_FWD, xm, wm, arr, len(adapters), X.device, workspace)
    st = _load().lora_linear_fwd(ctypes.byref(xm), _ref(wm), _ref(bm), arr, len(adapters),
                                 float(request_scale), ctypes.byref(ym),
                                 ws.data_ptr() if ws is not None else None, nbytes, _stream(X.device))
    _check(st, "lora_linear_fwd")
    return out


def lora_linear_fwd_grouped(X: torch.Tensor, W_stacked, bias: Optional[torch.Tensor],
                            adapters: Sequence[Adapter], request_scale: float = 1.0,
                            out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.bfloat16,
                            workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Stacked column groups: group g of the output gets X W_g^T + bias_g + s_g (X A_g^T) B_g^T."""
    n = W_stacked.rows if isinstance(W_stacked, NF4Weight) else W_stacked.shape[0]
    if out is None:
        out = torch.empty(X.shape[0], n, dtype=out_dtype, device=X.device)
    xm, wm, bm, arr, ym = _mat(X), _mat(W_stacked), _mat(bias), _adapters(adapters), _out(out)
    ws, nbytes = _workspace(WP_OP_FWD_GROUPED, xm, wm, arr, len(adapters), X.device, workspace)
    st = _load().lora_linear_fwd_grouped(ctypes.byref(xm), ctypes.byref(wm), _ref(bm), len(adapters),
                                         arr, float(request_scale), ctypes.byref(ym),
                                         ws.data_ptr() if ws is not None else None, nbytes,
                                         _stream(X.device))
    _check(st, "lora_linear_fwd_grouped")
    return out


def lora_merge(W, adapters: Sequence[Adapter], scale: float = 1.0, workspace: Optional[torch.Tensor] = None,
               bias: Optional[torch.Tensor] = None, rounding_seed: Optional[int] = None):
    """Bake the adapters into W in place: W <- W + sum_p s_p B_p A_p (s_p = alpha/r * strength
    * scale), accumulated in fp32 and rounded once; a 4-bit ``NF4Weight`` is requantised,
    round to nearest, or with ``rounding_seed`` (an unsigned 64-bit integer) stochastically
    (``lora_merge_seeded``).  Adapters with a legacy ``bias_B`` also update ``bias`` in place
    (bias <- bias + sum_p s_p bias_B_p, one rounding); the call fails before writing anything
    when such an adapter meets ``bias=None``.  Returns W."""
    wm, arr = _mat(W), _adapters(adapters)
    bo = None
    if bias is not None:
        if not bias.is_contiguous():
            raise ValueError("bias must be contiguous")
        bo = WpOut(bias.data_ptr(), _DT[bias.dtype], 1, bias.numel(), bias.numel())
    device = W.packed.device if isinstance(W, NF4Weight) else W.device
    need = _load().lora_workspace_size(WP_OP_MERGE, None, ctypes.byref(wm), arr, len(adapters))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    nbytes = workspace.numel() if workspace is not None else 0
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    if rounding_seed is None:
        st = _load().lora_merge(ctypes.byref(wm), _ref(bo), arr, len(adapters), float(scale), ws_ptr, nbytes,
                                _stream(device))
        _check(st, "lora_merge")
    else:
        seed = int(rounding_seed)
        if not 0 <= seed < 1 << 64:
            raise ValueError("rounding_seed must be an unsigned 64-bit integer")
        st = _load().lora_merge_seeded(ctypes.byref(wm), _ref(bo), arr, len(adapters), float(scale), seed, ws_ptr,
                                       nbytes, _stream(device))
        _check(st, "lora_merge_seeded")
    return W


def lora_swiglu_fwd(X: torch.Tensor, W_gate_up, bias: Optional[torch.Tensor], adapters: Sequence[Adapter],
                    request_scale: float = 1.0, out: Optional[torch.Tensor] = None,
                    eg: Optional[torch.Tensor] = None, save_eg: bool = False,
                    workspace: Optional[torch.Tensor] = None):
    """SwiGLU front half: h = silu(e) g with e, g the gate and up LoRA linears of the stacked
    ``W_gate_up`` ([2F, in]; ``adapters`` = [gate, up]).  Returns h, or (h, eg) when
    ``save_eg`` or ``eg`` is given (eg = e | g, [T, 2F], what the backward needs)."""
    n2 = W_gate_up.rows if isinstance(W_gate_up, NF4Weight) else W_gate_up.shape[0]
    if out is None:
        out = torch.empty(X.shape[0], n2 // 2, dtype=torch.bfloat16, device=X.device)
    if eg is None and save_eg:
        eg = torch.empty(X.shape[0], n2, dtype=torch.bfloat16, device=X.device)
    xm, wm, bm, arr, hm = _mat(X), _mat(W_gate_up), _mat(bias), _adapters(adapters), _out(out)
    egm = _out(eg) if eg is not None else None
    ws, nbytes = _workspace(WP_OP_SWIGLU_FWD, xm, wm, arr, len(adapters), X.device, workspace)
    st = _load().lora_swiglu_fwd(ctypes.byref(xm), ctypes.byref(wm), _ref(bm), arr, float(request_scale),
                                 ctypes.byref(hm), _ref(egm), ws.data_ptr() if ws is not None else None,
                                 nbytes, _stream(X.device))
    _check(st, "lora_swiglu_fwd")
    return (out, eg) if eg is not None else out


def lora_swiglu_bwd(dH: torch.Tensor, eg: torch.Tensor, deg: Optional[torch.Tensor] = None,
                    h: Optional[torch.Tensor] = None, want_h: bool = False):
    """SwiGLU backward: from the gradient at h and the saved e | g, de | dg ([T, 2F], the
    stacked gate/up output gradient); with ``want_h`` (or ``h``) also h recomputed.
    Returns deg, or (deg, h)."""
    if deg is None:
        deg = torch.empty_like(eg)
    if h is None and want_h:
        h = torch.empty_like(dH)
    hm = _out(h) if h is not None else None
    st = _load().lora_swiglu_bwd(ctypes.byref(_mat(dH)), ctypes.byref(_mat(eg)), ctypes.byref(_out(deg)),
                                 _ref(hm), _stream(dH.device))
    _check(st, "lora_swiglu_bwd")
    return (deg, h) if h is not None else deg


def lora_linear_fwd_host(X_host: torch.Tensor, W, bias: Optional[torch.Tensor], adapters: Sequence[Adapter],
                         request_scale: float = 1.0, out: Optional[torch.Tensor] = None,
                         out_dtype: torch.dtype = torch.bfloat16, grouped: bool = False,
                         workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The forward with X and the result in host memory (pin both for the copies to overlap
    the compute): rows go through the device in chunks, copies and kernels overlapped.
    ``grouped`` selects the stacked column-group form (one adapter per group)."""
    if isinstance(W, NF4Weight):
        device, n = W.packed.device, W.rows
    elif W is not None:
        device, n = W.device, W.shape[0]
    else:
        device, n = adapters[0].A.device, adapters[0].B.shape[0]
    if out is None:
        out = torch.empty(X_host.shape[0], n, dtype=out_dtype, pin_memory=True)
    xm, wm, bm, arr, ym = _mat(X_host), _mat(W), _mat(bias), _adapters(adapters), _out(out)
    ws, nbytes = _workspace(WP_OP_FWD_HOST, xm, wm, arr, len(adapters), device, workspace)
    st = _load().lora_linear_fwd_host(ctypes.byref(xm), _ref(wm), _ref(bm), len(adapters) if grouped else 0,
                                      arr, len(adapters), float(request_scale), ctypes.byref(ym),
                                      ws.data_ptr() if ws is not None else None, nbytes, _stream(device))
    _check(st, "lora_linear_fwd_host")
    return out


def lora_linear_fwd_exact(X: torch.Tensor, W, bias: Optional[torch.Tensor], adapters: Sequence[Adapter],
                          request_scale: float = 1.0, skip_unit_scales: bool = True, grouped: bool = False,
                          out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The unfused bf16 chain (base, X A^T, then B^T, one rounded multiplication per scale, the
    add), the exact tier when ``skip_unit_scales``; ``grouped``: one adapter per column group."""
    n = W.rows if isinstance(W, NF4Weight) else W.shape[0]
    if out is None:
        out = torch.empty(X.shape[0], n, dtype=torch.bfloat16, device=X.device)
    xm, wm, bm, arr, ym = _mat(X), _mat(W), _mat(bias), _adapters(adapters), _out(out)
    ws, nbytes = _workspace(WP_OP_FWD_EXACT, xm, wm, arr, len(adapters), X.device, workspace)
    st = _load().lora_linear_fwd_exact(ctypes.byref(xm), ctypes.byref(wm), _ref(bm), len(adapters) if grouped else 0,
                                       arr, len(adapters), float(request_scale), 1 if skip_unit_scales else 0,
                                       ctypes.byref(ym), ws.data_ptr() if ws is not None else None, nbytes,
                                       _stream(X.device))
    _check(st, "lora_linear_fwd_exact")
    return out


def lora_linear_bwd(X: torch.Tensor, W, dY: torch.Tensor, adapters: Sequence[Adapter],
                    request_scale: float = 1.0, need_dX: bool = True,
                    dX_dtype: torch.dtype = torch.bfloat16, workspace: Optional[torch.Tensor] = None):
    """Closed-form (dX, [dA_g], [dB_g]) of Y = X W_g^T + s_g (X A_g^T) B_g^T over len(adapters) groups."""
    G = len(adapters)
    dX = torch.empty_like(X, dtype=dX_dtype) if need_dX else None
    dA = [torch.empty(a.A.shape, dtype=torch.float32, device=X.device) for a in adapters]
    dB = [torch.empty(a.B.shape, dtype=torch.float32, device=X.device) for a in adapters]
    xm, wm, dym, arr = _mat(X), _mat(W), _mat(dY), _adapters(adapters)
    dxo = _out(dX) if dX is not None else None
    dao = (WpOut * G)(*[_out(t) for t in dA])
    dbo = (WpOut * G)(*[_out(t) for t in dB])
    ws, nbytes = _workspace(WP_OP_BWD, xm, wm, arr, G, X.device, workspace)
    st = _load().lora_linear_bwd(ctypes.byref(xm), ctypes.byref(wm), ctypes.byref(dym), G, arr,
                                 float(request_scale), _ref(dxo), dao, dbo,
                                 ws.data_ptr() if ws is not None else None, nbytes, _stream(X.device))
    _check(st, "lora_linear_bwd")
    return dX, dA, dB


def lora_dense_patch(param: torch.Tensor, payload: torch.Tensor, kind: int, strength: float = 1.0) -> torch.Tensor:
    """Apply a dense payload to ``param`` in place (.diff/.diff_b: kind=WP_PATCH_ADD,
    .set_weight: kind=WP_PATCH_SET) and return it."""
    if not (param.is_contiguous() and payload.is_contiguous()):
        raise ValueError("dense patch tensors must be contiguous")
    st = _load().lora_dense_patch(param.data_ptr(), _DT[param.dtype], param.numel(), payload.data_ptr(),
                                  _DT[payload.dtype], payload.numel(), int(kind), float(strength),
                                  _stream(param.device))
    _check(st, "lora_dense_patch")
    return param


def lora_device_status(reset: bool = True) -> int:
    """The device status word (0, or -7 after a bounded wait expired).  Synchronises."""
    torch.cuda.synchronize()
    return _load().lora_device_status(1 if reset else 0)


def lora_set_wait_limit(timeout_ns: int) -> None:
    """How long a bounded device wait spins before its kernel gives up (default 2 s)."""
    _check(_load().lora_set_wait_limit(int(timeout_ns)), "lora_set_wait_limit")


def lora_nf4_codebook() -> list:
    buf = (ctypes.c_float * 16)()
    _load().lora_nf4_codebook(buf)
    return list(buf)


def lora_status_string(status: int) -> str:
    return _load().lora_status_string(status).decode()
