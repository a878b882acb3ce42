"""Dense LoRA payloads (``.diff`` / ``.diff_b`` / ``.set_weight``), oracle side.

Test infrastructure only; see the package docstring.

Source: FastVideo API docs, ``fastvideo.models.loader.lora_patch``, class
``DenseLoRAPatch``:
  * ``apply_to``: the additive delta is summed in float32 whatever the operands are,
    ``param.to(float32) + delta.to(float32) * strength``, and the caller casts back to
    the parameter's dtype; a delta whose shape differs from the parameter's is an
    error;
  * ``replacement_for``: the payload replaces a parameter the base zero-initialises,
    returned as ``payload.to(float32) * strength``;
  * the constructor rejects a non-finite strength.

Reading (the page is silent on scalar precision): the Python-float strength enters a
float32 tensor op, so it is rounded to float32 first; the product and the sum are two
separate float32 roundings (no fused multiply-add); the cast back is
round-to-nearest-even.
"""
from __future__ import annotations

import math

import numpy as np

from .numerics import bf16_bits_to_f32, f32_to_bf16_bits


class PatchError(ValueError):
    pass


def _as_f32(values: np.ndarray, kind: str) -> np.ndarray:
    if kind == "bf16":
        return bf16_bits_to_f32(values)
    if kind == "fp32":
        return np.asarray(values, dtype=np.float32)
    raise PatchError(f"unsupported dtype {kind}")


def _cast_back(x32: np.ndarray, kind: str) -> np.ndarray:
    if kind == "bf16":
        return f32_to_bf16_bits(x32)
    return np.asarray(x32, dtype=np.float32)


def _check_strength(strength: float) -> np.float32:
    if not math.isfinite(strength):
        raise PatchError(f"strength must be finite, got {strength}")
    return np.float32(strength)


def apply_diff(param: np.ndarray, param_kind: str, delta: np.ndarray, delta_kind: str,
               strength: float) -> np.ndarray:
    """``.diff`` / ``.diff_b``: returns the new parameter in the parameter's storage."""
    k = _check_strength(strength)
    if np.shape(param) != np.shape(delta):
        raise PatchError(f"delta shape {np.shape(delta)} != parameter shape {np.shape(param)}")
    p32 = _as_f32(param, param_kind)
    d32 = _as_f32(delta, delta_kind)
    scaled = (d32 * k).astype(np.float32)
    total = (p32 + scaled).astype(np.float32)
    return _cast_back(total, param_kind)


def apply_set(payload: np.ndarray, payload_kind: str, param_kind: str, strength: float,
              param_shape=None) -> np.ndarray:
    """``.set_weight``: returns the replacement in the parameter's storage."""
    k = _check_strength(strength)
    if param_shape is not None and tuple(param_shape) != tuple(np.shape(payload)):
        raise PatchError(f"payload shape {np.shape(payload)} != parameter shape {tuple(param_shape)}")
    v32 = _as_f32(payload, payload_kind)
    return _cast_back((v32 * k).astype(np.float32), param_kind)
