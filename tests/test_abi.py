"""The C-ABI library loads, exports every function include/*.h declares, and rejects
bad arguments on the host (no GPU needed: a rejected call launches nothing)."""
import ctypes
import glob
import math
import os
import re

import numpy as np
import pytest

import weight_patches_gb300 as wpg
from oracle import nf4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M):
            name = m.group(1)
            if name not in ("if", "for", "while", "sizeof", "return"):
                names.add(name)
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    return wpg.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "lora_linear_fwd" in names and "lora_dense_patch" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_nf4_codebook_matches_oracle_bitwise():
    got = np.array(wpg.lora_nf4_codebook(), dtype=np.float32)
    want = nf4.codebook_f32()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


FAKE = 0x10000  # a non-null, 16-byte aligned "device" address never dereferenced


def _m(rows, cols, dtype=wpg.WP_BF16, ld=None, data=FAKE):
    return wpg.WpMat(data, dtype, rows, cols, cols if ld is None else ld, None)


def _o(rows, cols, dtype=wpg.WP_BF16, ld=None):
    return wpg.WpOut(FAKE, dtype, rows, cols, cols if ld is None else ld)


def _ad(r, n_in, n_out, alpha=8.0, strength=1.0, dtype=wpg.WP_BF16):
    return wpg.WpAdapter(_m(r, n_in, dtype), _m(n_out, r, dtype), alpha, strength)


def _fwd(lib, X, W, bias, ads, Y, rs=1.0, ws=None, ws_bytes=0):
    arr = (wpg.WpAdapter * max(1, len(ads)))(*ads)
    return lib.lora_linear_fwd(ctypes.byref(X), ctypes.byref(W) if W else None,
                               ctypes.byref(bias) if bias else None, arr, len(ads), rs,
                               ctypes.byref(Y), ws, ws_bytes, None)


def test_fwd_rejections(lib):
    X, W, Y = _m(64, 128), _m(256, 128), _o(64, 256)
    assert _fwd(lib, X, W, None, [_ad(8, 128, 256)], _o(64, 255)) == -2          # Y cols
    assert _fwd(lib, X, _m(256, 127), None, [], Y) == -2                          # W cols
    assert _fwd(lib, X, W, None, [_ad(8, 128, 300)], Y) == -2                     # B rows
    assert _fwd(lib, X, W, None, [_ad(8, 120, 256)], Y) == -2                     # A cols
    assert _fwd(lib, X, W, None, [_ad(8, 128, 256, alpha=math.nan)], Y) == -1     # non-finite alpha
    assert _fwd(lib, X, W, None, [_ad(8, 128, 256, strength=math.inf)], Y) == -1
    assert _fwd(lib, X, W, None, [_ad(8, 128, 256)], Y, rs=math.nan) == -1       # request scale
    assert _fwd(lib, X, W, _m(1, 255), [], Y) == -2                               # bias numel
    bad = wpg.WpAdapter(_m(8, 128), _m(256, 8, wpg.WP_FP32), 8.0, 1.0)
    assert _fwd(lib, X, W, None, [bad], Y) == -3                                  # mixed A/B dtypes
    assert _fwd(lib, _m(64, 128, data=None), W, None, [], Y) == -1               # null X
    # fp32 adapter needs workspace (s * X A^T in fp32); none given
    assert _fwd(lib, X, W, None, [_ad(8, 128, 256, dtype=wpg.WP_FP32)], Y) == -5
    # tensor-core path alignment: row pitch not a multiple of 8 elements
    assert _fwd(lib, _m(64, 128, ld=130), W, None, [], Y) == -4
    assert _fwd(lib, X, W, None, [], _o(64, 256, ld=260)) == -4
    # bf16 adapters need workspace too (their H~ rows); none given
    assert _fwd(lib, X, W, None, [_ad(8, 128, 256)], Y) == -5
    # an adapter wider than one tensor-memory accumulator buffer, and more bf16 adapters than
    # the kernel carries (several adapters of 384 rank columns in all are served, in passes)
    assert _fwd(lib, X, W, None, [_ad(264, 128, 256)], Y, ws=FAKE, ws_bytes=1 << 30) == -8
    nine = [_ad(8, 128, 256) for _ in range(9)]
    assert _fwd(lib, X, W, None, nine, Y, ws=FAKE, ws_bytes=1 << 30) == -8


def test_grouped_rejections(lib):
    X, W = _m(64, 128), _m(3 * 256, 128)
    Y = _o(64, 3 * 256)
    arr = (wpg.WpAdapter * 2)(_ad(8, 128, 256), _ad(8, 128, 256))
    assert lib.lora_linear_fwd_grouped(ctypes.byref(X), ctypes.byref(W), None, 3, arr, 1.0,
                                       ctypes.byref(Y), None, 0, None) != 0   # adapters per group
    arr = (wpg.WpAdapter * 3)(_ad(8, 128, 256), _ad(8, 128, 256), _ad(8, 128, 200))
    assert lib.lora_linear_fwd_grouped(ctypes.byref(X), ctypes.byref(W), None, 3, arr, 1.0,
                                       ctypes.byref(Y), None, 0, None) == -2


def test_dense_patch_rejections(lib):
    assert lib.lora_dense_patch(FAKE, wpg.WP_BF16, 10, FAKE, wpg.WP_BF16, 11, 0, 1.0, None) == -2
    assert lib.lora_dense_patch(FAKE, wpg.WP_BF16, 10, FAKE, wpg.WP_BF16, 10, 0, math.nan, None) == -1
    assert lib.lora_dense_patch(FAKE, wpg.WP_BF16, 10, FAKE, wpg.WP_BF16, 10, 7, 1.0, None) == -1
    assert lib.lora_dense_patch(FAKE, wpg.WP_NF4, 10, FAKE, wpg.WP_BF16, 10, 0, 1.0, None) == -3
    assert lib.lora_dense_patch(None, wpg.WP_BF16, 10, FAKE, wpg.WP_BF16, 10, 0, 1.0, None) == -1


def test_workspace_sizes(lib):
    X, W = _m(1000, 128), _m(256, 128)
    arr = (wpg.WpAdapter * 2)(_ad(8, 128, 256), _ad(16, 128, 256, dtype=wpg.WP_FP32))
    # tensor-core path: the fp32 adapter's s * X A^T (1000 x 16 fp32, for the CUDA-core
    # route), its bf16 B pieces (256 x 6 x 16), the H~ rows of both adapters
    # (1000 x (16 + 96) bf16), one flag per 256-row block (4, padded to 256 B) and the
    # packed A rows of the rank item ((16 + 3 x 16) x 128 bf16)
    assert (lib.lora_workspace_size(0, ctypes.byref(X), ctypes.byref(W), arr, 2)
            == 64000 + 49152 + 224000 + 256 + 16384)
    assert lib.lora_workspace_size(0, ctypes.byref(X), ctypes.byref(W), arr, 1) == 32000 + 256 + 4096
    assert lib.lora_workspace_size(0, ctypes.byref(X), ctypes.byref(W), arr, 0) == 0
    Xf = _m(1000, 128, wpg.WP_FP32)
    # fp32 path: every adapter's s * X A^T, 1000 x 24 fp32, rounded up to 256 bytes
    assert lib.lora_workspace_size(0, ctypes.byref(Xf), ctypes.byref(W), arr, 2) == 96000


def test_status_strings(lib):
    for code in wpg.STATUS:
        assert wpg.lora_status_string(code)


def _ad_vec(r, n_in, n_out, vec_dtype=wpg.WP_BF16, strength=1.0):
    a = _ad(r, n_in, n_out, strength=strength)
    a.bias_B = FAKE
    a.bias_B_dtype = vec_dtype
    return a


def test_legacy_vector_rejections(lib):
    """Older adapters' bias vector: a bad dtype, a missing workspace for the folded bias, and
    (merge) a vector meeting a module without a bias, all refused on the host."""
    X, W, Y = _m(64, 128), _m(256, 128), _o(64, 256)
    assert _fwd(lib, X, W, None, [_ad_vec(8, 128, 256, vec_dtype=wpg.WP_NF4)], Y,
                ws=FAKE, ws_bytes=1 << 30) == -3
    assert _fwd(lib, X, W, None, [_ad_vec(8, 128, 256)], Y) == -5
    Wm = _m(256, 128)

    def merge(ads, bias):
        arr = (wpg.WpAdapter * max(1, len(ads)))(*ads)
        return lib.lora_merge(ctypes.byref(Wm), ctypes.byref(bias) if bias is not None else None, arr,
                              len(ads), 1.0, FAKE, 1 << 30, None)

    assert merge([_ad_vec(8, 128, 256)], None) == -1                    # no bias to add it to
    assert merge([_ad_vec(8, 128, 256)], _o(1, 255)) == -2              # bias numel != out
    assert merge([_ad_vec(8, 128, 256)], wpg.WpOut(FAKE, wpg.WP_NF4, 1, 256, 256)) == -3
    assert merge([_ad_vec(8, 128, 256, vec_dtype=7)], _o(1, 256)) == -3
    # a vector whose s is zero asks for nothing: no bias needed, nothing launched
    assert merge([_ad_vec(8, 128, 256, strength=0.0)], None) == 0


def test_workspace_reserves_the_folded_bias(lib):
    X, W = _m(1000, 128), _m(256, 128)
    plain = (wpg.WpAdapter * 1)(_ad(8, 128, 256))
    vec = (wpg.WpAdapter * 1)(_ad_vec(8, 128, 256))
    a = lib.lora_workspace_size(wpg.WP_OP_FWD, ctypes.byref(X), ctypes.byref(W), plain, 1)
    b = lib.lora_workspace_size(wpg.WP_OP_FWD, ctypes.byref(X), ctypes.byref(W), vec, 1)
    assert b - a == 256 * 4 + (-(256 * 4) % 256)                          # fp32 [out], 256-byte rounded


def test_exact_tier_rejections(lib):
    X, W, Y = _m(64, 128), _m(256, 128), _o(64, 256)
    call = lambda ads, y=Y, groups=0: lib.lora_linear_fwd_exact(
        ctypes.byref(X), ctypes.byref(W), None, groups, (wpg.WpAdapter * max(1, len(ads)))(*ads), len(ads), 1.0, 1,
        ctypes.byref(y), ctypes.c_void_p(FAKE), 1 << 30, None)
    assert call([_ad(12, 128, 256)]) == -4                     # t = X A^T needs r % 8 == 0
    assert call([_ad(8, 128, 256)], y=_o(64, 256, dtype=wpg.WP_FP32)) == -3   # the chain's Y is bf16
    assert call([_ad(8, 128, 256)], groups=2) == -1            # one adapter per group
    assert lib.lora_workspace_size(wpg.WP_OP_FWD_EXACT, ctypes.byref(X), ctypes.byref(W),
                                   (wpg.WpAdapter * 1)(_ad(8, 128, 256)), 1) >= 64 * 256 * 4
