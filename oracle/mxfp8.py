"""MXFP8 (E4M3 elements, E8M0 block scales) quantisation for the oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix: [TE-JAX] "Accelerating Dropless MoE Training in JAX with
NVIDIA Transformer Engine" ¶6 names a group-aware MXFP8 grouped GEMM for the
expert matmuls; [MoE-Eng] "LLM Infrastructure Engineering 08: MoE Training
Engineering" §13.6 asks for fine-grained (per-tile, not per-tensor) scaling
with fp32 accumulation.  The pages give no encoding, so this module follows
the published OCP Microscaling (MX) v1.0 and OCP 8-bit floating point (OFP8)
definitions, written here from those definitions:

* a block is 32 consecutive elements along the contraction dimension;
* shared scale ``X = 2^(floor(log2(amax)) - 8)``, 8 being the largest
  exponent of E4M3; stored as an E8M0 byte ``127 + log2(X)`` (clamped to
  [0, 254]); an all-zero block stores byte 0 and zero elements;
* elements ``x / X`` rounded to the nearest E4M3 value, ties to even,
  saturating at +-448 (E4M3 has no infinities; S.1111.111 is NaN).
"""
from __future__ import annotations

import numpy as np

__all__ = ["e4m3_decode", "e4m3_encode", "e8m0_scale_exponent", "mx_quantize",
           "mx_dequantize", "mx_fake_quant", "swiglu_expert_mxfp8", "moe_forward_mxfp8",
           "E4M3_MAX", "MX_BLOCK"]

E4M3_MAX = 448.0
MX_BLOCK = 32
_E4M3_BIAS = 7
_E4M3_EMAX = 8


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 byte -> float64 value (NaN for S.1111.111)."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    sub = exp == 0
    val = np.where(sub, man / 8.0 * 2.0 ** (1 - _E4M3_BIAS),
                   (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - _E4M3_BIAS))
    val = np.where((exp == 0xF) & (man == 0x7), np.nan, val)
    return sign * val


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float -> E4M3 byte, round to nearest even, saturate to +-448, NaN -> 0x7F."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    finite = np.isfinite(a)
    a_f = np.where(finite, a, 0.0)
    # exponent of the binade (subnormals share the minimum normal exponent -6)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a_f > 0, a_f, 1.0)))
    e = np.maximum(e, 1 - _E4M3_BIAS)
    q = np.exp2(e - 3)                      # spacing of values in that binade
    r = np.rint(a_f / q) * q                # np.rint rounds half to even
    r = np.minimum(r, E4M3_MAX)             # saturate (also +-inf)
    r = np.where(np.isinf(a), E4M3_MAX, r)
    # value -> code
    e2 = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    is_sub = r < 2.0 ** (1 - _E4M3_BIAS)
    man_sub = np.rint(r / 2.0 ** (1 - _E4M3_BIAS - 3))
    man_nrm = np.rint((r / np.exp2(e2) - 1.0) * 8.0)
    exp_nrm = e2 + _E4M3_BIAS
    code = np.where(is_sub, man_sub, exp_nrm * 8 + man_nrm).astype(np.int64)
    code = np.where(r == 0, 0, code)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def e8m0_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Unbiased scale exponent ``floor(log2(amax)) - 8``, clamped to the E8M0
    range [-127, 127]; an amax of zero maps to -127 (stored byte 0)."""
    a = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        fl = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    ex = fl - _E4M3_EMAX
    ex = np.where(a > 0, ex, -127)
    return np.clip(ex, -127, 127).astype(np.int64)


def mx_quantize(x: np.ndarray, axis: int = -1, group_starts=None):
    """Quantise ``x`` to MXFP8 in blocks of 32 along ``axis``.

    ``group_starts`` (optional, for the ragged token axis): block boundaries
    restart at each listed index, so a block never spans two experts' rows;
    the last block of a group may be short and its amax covers only its own
    rows (reading of "group-aware" in [TE-JAX] ¶6).

    Returns ``(codes uint8 same shape, scale_bytes uint8)`` where the scale
    array has the blocked axis replaced by its number of blocks.
    """
    x = np.moveaxis(np.asarray(x, dtype=np.float64), axis, -1)
    length = x.shape[-1]
    if group_starts is None:
        starts = list(range(0, length, MX_BLOCK))
    else:
        bounds = sorted(set(list(group_starts) + [length]))
        starts = []
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            starts.extend(range(lo, hi, MX_BLOCK))
    ends = starts[1:] + [length]
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1] + (len(starts),), dtype=np.uint8)
    for b, (lo, hi) in enumerate(zip(starts, ends)):
        blk = x[..., lo:hi]
        amax = np.abs(blk).max(axis=-1)
        ex = e8m0_scale_exponent(amax)
        scales[..., b] = (ex + 127).astype(np.uint8)
        codes[..., lo:hi] = e4m3_encode(blk / np.exp2(ex)[..., None])
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis), starts


def mx_dequantize(codes: np.ndarray, scales: np.ndarray, starts, axis: int = -1) -> np.ndarray:
    """Inverse of :func:`mx_quantize`: element value times its block's scale."""
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1)
    length = c.shape[-1]
    ends = list(starts[1:]) + [length]
    out = np.empty(c.shape, dtype=np.float64)
    vals = e4m3_decode(c)
    for b, (lo, hi) in enumerate(zip(starts, ends)):
        out[..., lo:hi] = vals[..., lo:hi] * np.exp2(s[..., b].astype(np.float64) - 127)[..., None]
    return np.moveaxis(out, -1, axis)


def mx_fake_quant(x: np.ndarray, axis: int = -1) -> np.ndarray:
    """Quantise to MXFP8 along ``axis`` and dequantise again (float64)."""
    codes, scales, starts = mx_quantize(x, axis=axis)
    return mx_dequantize(codes, scales, starts, axis=axis)


def swiglu_expert_mxfp8(x, w1, w3, w2):
    """One SwiGLU expert with MXFP8 operands (quantisation-aware reference).

    Every GEMM operand is quantised along its contraction dimension: x, w1,
    w3 along D; h and w2 along F.  The arithmetic on the dequantised values
    is fp32, as on the tensor cores.  Returns (y, a1, a3, h) with h before its
    quantisation."""
    f32 = np.float32
    xq = mx_fake_quant(x, axis=1).astype(f32)
    a1 = np.matmul(xq, mx_fake_quant(w1, axis=1).astype(f32).T)
    a3 = np.matmul(xq, mx_fake_quant(w3, axis=1).astype(f32).T)
    h = (a1 / (f32(1.0) + np.exp(-a1)) * a3).astype(f32)
    y = np.matmul(mx_fake_quant(h, axis=1).astype(f32), mx_fake_quant(w2, axis=1).astype(f32).T)
    return y, a1, a3, h


def moe_forward_mxfp8(x, idx, g, w1, w3, w2, shared=None):
    """Layer forward of the dropless MoE layer with MXFP8 expert GEMMs: the
    loop over experts of the simplified MoE layer ("LLM Infrastructure
    Engineering 08: MoE Training Engineering" §9) with every expert replaced
    by :func:`swiglu_expert_mxfp8`; gate weights and the combine stay fp32."""
    n, d = x.shape
    out = np.zeros((n, d), dtype=np.float32)
    for e in range(w1.shape[0]):
        tok, kk = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        y = swiglu_expert_mxfp8(x[tok], w1[e], w3[e], w2[e])[0]
        np.add.at(out, tok, y * g[tok, kk].astype(np.float32)[:, None])
    if shared is not None:
        out = out + swiglu_expert_mxfp8(x, shared[0], shared[1], shared[2])[0]
    return out
