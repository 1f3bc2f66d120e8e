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
           "moe_backward_mxfp8", "bf16_round", "fp8_tile_quantize", "fp8_tile_dequantize",
           "FP8_TILE", "E4M3_MAX", "MX_BLOCK"]

E4M3_MAX = 448.0
MX_BLOCK = 32
FP8_TILE = 128
_E4M3_BIAS = 7
_E4M3_EMAX = 8


def _e4m3_decode_formula(c: np.ndarray) -> np.ndarray:
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    sub = exp == 0
    val = np.where(sub, man / 8.0 * 2.0 ** (1 - _E4M3_BIAS),
                   (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - _E4M3_BIAS))
    val = np.where((exp == 0xF) & (man == 0x7), np.nan, val)
    return sign * val


_E4M3_TABLE = _e4m3_decode_formula(np.arange(256, dtype=np.int64))


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 byte -> float64 value (NaN for S.1111.111): sign, 4 exponent bits
    (bias 7), 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6).  Looked up
    in the 256-entry table of that formula."""
    return _E4M3_TABLE[np.asarray(codes).astype(np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float -> E4M3 byte, round to nearest even, saturate to +-448, NaN -> 0x7F.

    The binade exponent e = floor(log2|v|) comes from frexp (subnormals share
    the minimum normal exponent -6); |v| / 2^(e-3) rounded half to even gives
    the significand m in 8..16 (16 carries into the next binade) or, for
    subnormals, 0..8; the code is then (e + 7) * 8 + (m - 8), or m for a
    subnormal.  Values past 448 (and infinities) saturate to 448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    nan = np.isnan(v)
    inf = np.isinf(v)
    a_f = np.where(nan | inf, 0.0, a)
    _, ex = np.frexp(a_f)                    # a = f * 2^ex with f in [0.5, 1)
    e = np.maximum(ex - 1, 1 - _E4M3_BIAS)
    m = np.rint(np.ldexp(a_f, -(e - 3)))     # exact power-of-two scaling, then RNE
    carry = m >= 16
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 8, m)
    over = inf | (e > _E4M3_EMAX) | ((e == _E4M3_EMAX) & (m > 14))   # 14 -> 1.75 * 2^8 = 448
    e = np.where(over, _E4M3_EMAX, e)
    m = np.where(over, 14, m)
    code = np.where(m < 8, m, (e + _E4M3_BIAS) * 8 + (m - 8)).astype(np.int64)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(nan, 0x7F, code)
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
    if group_starts is None and length % MX_BLOCK == 0:
        # every block is a full 32 elements: the same steps on all blocks at once
        xb = x.reshape(x.shape[:-1] + (length // MX_BLOCK, MX_BLOCK))
        ex = e8m0_scale_exponent(np.abs(xb).max(axis=-1))
        codes = e4m3_encode(xb / np.exp2(ex)[..., None]).reshape(x.shape)
        scales = (ex + 127).astype(np.uint8)
        return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis), list(range(0, length, MX_BLOCK))
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
    if list(starts) == list(range(0, length, MX_BLOCK)) and length % MX_BLOCK == 0:
        vals = e4m3_decode(c).reshape(c.shape[:-1] + (length // MX_BLOCK, MX_BLOCK))
        out = vals * np.exp2(s.astype(np.float64) - 127)[..., None]
        return np.moveaxis(out.reshape(c.shape), -1, axis)
    ends = list(starts[1:]) + [length]
    out = np.empty(c.shape, dtype=np.float64)
    vals = e4m3_decode(c)
    for b, (lo, hi) in enumerate(zip(starts, ends)):
        out[..., lo:hi] = vals[..., lo:hi] * np.exp2(s[..., b].astype(np.float64) - 127)[..., None]
    return np.moveaxis(out, -1, axis)


def bf16_round(a) -> np.ndarray:
    """Round fp32 values to the nearest bfloat16 value (ties to even), kept as
    fp32: the storage precision of the layer's intermediate activations."""
    u = np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


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


def moe_forward_mxfp8(x, idx, g, w1, w3, w2, shared=None, return_saved=False, store=bf16_round):
    """Layer forward of the dropless MoE layer with MXFP8 expert GEMMs: the
    loop over experts of the simplified MoE layer ("LLM Infrastructure
    Engineering 08: MoE Training Engineering" §9) with every expert replaced
    by :func:`swiglu_expert_mxfp8`; gate weights and the combine stay fp32.

    With ``return_saved`` also returns what the backward needs, in the layout
    of the bf16 oracle's ``moe_forward``: ``experts[e] = (tok, kk, y, a1, a3,
    h)`` (rows in ascending token order) and ``shared = (y, a1, a3, h)``, as
    the layer stores them (``store``: bf16 by default, the intermediate
    precision the layer keeps; the identity keeps fp32)."""
    n, d = x.shape
    out = np.zeros((n, d), dtype=np.float32)
    saved = {"experts": {}}
    for e in range(w1.shape[0]):
        tok, kk = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        y, a1, a3, h = swiglu_expert_mxfp8(x[tok], w1[e], w3[e], w2[e])
        saved["experts"][e] = (tok, kk, store(y), store(a1), store(a3), store(h))
        np.add.at(out, tok, y * g[tok, kk].astype(np.float32)[:, None])
    if shared is not None:
        ys, a1s, a3s, hs = swiglu_expert_mxfp8(x, shared[0], shared[1], shared[2])
        saved["shared"] = (store(ys), store(a1s), store(a3s), store(hs))
        out = out + ys
    return (out, saved) if return_saved else out


def _mx_matmul(a, a_axis, b, b_axis, quant=mx_fake_quant):
    """``a @ b`` in fp32 with both operands MXFP8-quantised along the
    contraction: ``a`` along ``a_axis`` (its columns, 1, or its rows, 0, in
    which case the product is ``a^T @ b``) and ``b`` along ``b_axis``."""
    f32 = np.float32
    aq = quant(a, axis=a_axis).astype(f32)
    bq = quant(b, axis=b_axis).astype(f32)
    return np.matmul(aq.T if a_axis == 0 else aq, bq.T if b_axis == 1 else bq)


def moe_backward_mxfp8(dy, x, logits, idx, g, w_gate, w1, w3, w2, saved, gate, shared=None,
                       quant=mx_fake_quant, store=bf16_round):
    """Backward of the MXFP8 layer.

    The chain rule is that of the bf16 oracle's ``moe_backward`` (sparse
    per-expert backward, "LLM Infrastructure Engineering 08: MoE Training
    Engineering" §11.3); what changes is that every expert GEMM takes both
    operands MXFP8-quantised along its own contraction dimension (reading of
    the group-aware MXFP8 grouped GEMM of "Accelerating Dropless MoE Training
    in JAX with NVIDIA Transformer Engine" ¶6 for the backward):

    * ``dh = dYw w2``: dYw along D (its columns), w2 [D, F] along D (rows);
    * ``dx_e = da1 w1 + da3 w3``: da1, da3 along F, w1, w3 [F, D] along F;
    * ``dW2 = dYw^T h``, ``dW1 = da1^T x_e``, ``dW3 = da3^T x_e``: every
      operand along the expert's rows (tokens); the blocks start at the
      expert's first row, so no block spans two experts (group-aware).

    The SwiGLU derivative, the router gradient and the combine backward are
    fp32 as in the bf16 oracle.  The tensors the layer stores between steps
    (dYw, da1, da3) pass through ``store`` (bf16 by default) before they are
    quantised or reused, as the activations in ``saved`` did.  ``saved``
    comes from ``moe_forward_mxfp8(..., return_saved=True)``.  ``quant`` is
    the fake quantiser; with the identity for both ``quant`` and ``store``
    this is the bf16 oracle's backward.
    """
    f32 = np.float32
    n, d = x.shape
    n_exp, f, _ = w1.shape
    k = idx.shape[1]
    xx = x.astype(f32)
    dyy = dy.astype(f32)
    dx = np.zeros((n, d), dtype=f32)
    dw1 = np.zeros((n_exp, f, d), dtype=f32)
    dw3 = np.zeros((n_exp, f, d), dtype=f32)
    dw2 = np.zeros((n_exp, d, f), dtype=f32)
    dg = np.zeros((n, k), dtype=f32)

    def expert_bwd(dyw, xe, a1, a3, h, we1, we3, we2):
        dh = _mx_matmul(dyw, 1, we2, 0, quant)
        s = 1.0 / (1.0 + np.exp(-a1))
        da3 = store(dh * (a1 * s))
        da1 = store(dh * a3 * s * (1.0 + a1 * (1.0 - s)))
        gw2 = _mx_matmul(dyw, 0, h, 0, quant)
        gw1 = _mx_matmul(da1, 0, xe, 0, quant)
        gw3 = _mx_matmul(da3, 0, xe, 0, quant)
        gx = _mx_matmul(da1, 1, we1, 0, quant) + _mx_matmul(da3, 1, we3, 0, quant)
        return gw1, gw3, gw2, gx

    for e, (tok, kk, y, a1, a3, h) in saved["experts"].items():
        dg[tok, kk] = (dyy[tok] * y).sum(axis=1)
        dyw = store(dyy[tok] * g[tok, kk].astype(f32)[:, None])
        gw1, gw3, gw2, gx = expert_bwd(dyw, xx[tok], a1, a3, h, w1[e], w3[e], w2[e])
        dw1[e], dw3[e], dw2[e] = gw1, gw3, gw2
        np.add.at(dx, tok, gx)

    res = {}
    if shared is not None:
        ys, a1s, a3s, hs = saved["shared"]
        gw1, gw3, gw2, gx = expert_bwd(dyy, xx, a1s, a3s, hs, shared[0], shared[1], shared[2])
        res.update(dws1=gw1, dws3=gw3, dws2=gw2)
        dx = dx + gx

    # router: as the bf16 oracle (fp32 logits, no quantised GEMM)
    from .moe_oracle import router_logit_grad
    dl = router_logit_grad(dg, g, logits, idx, gate, f32)
    dw_gate = np.matmul(dl.T, xx)
    dx = dx + np.matmul(dl, w_gate.astype(f32))
    res.update(dx=dx, dw1=dw1, dw3=dw3, dw2=dw2, dw_gate=dw_gate, dg=dg, dlogits=dl)
    return res


# ----------------------------------------------------------------------------
# FP8 weights with per-tile scales ("LLM Infrastructure Engineering 08: MoE
# Training Engineering" §13.6: forward act(BF16) x weight(FP8) -> BF16,
# backward grad(BF16) x weight_T(FP8), per-tile scaling, FP32 accumulation)
# ----------------------------------------------------------------------------
def fp8_tile_quantize(w: np.ndarray, tile: int = FP8_TILE):
    """Quantise weight matrices [..., rows, cols] to E4M3 with one fp32 scale
    per ``tile x tile`` block (reading of "per-tile scaling": 128 x 128 blocks
    of the weight, a plain fp32 scale ``amax / 448`` so that the block
    maximum maps to the largest E4M3 value; an all-zero block gets scale 1).
    Returns (codes uint8 [..., rows, cols], scales fp32 [..., ceil(rows/t),
    ceil(cols/t)])."""
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape[-2:]
    nr, nc = -(-rows // tile), -(-cols // tile)
    scales = np.ones(w.shape[:-2] + (nr, nc), dtype=np.float32)
    codes = np.zeros(w.shape, dtype=np.uint8)
    for i in range(nr):
        for j in range(nc):
            blk = w[..., i * tile:(i + 1) * tile, j * tile:(j + 1) * tile]
            amax = np.abs(blk).max(axis=(-2, -1))
            sc = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0))
            scales[..., i, j] = sc
            codes[..., i * tile:(i + 1) * tile, j * tile:(j + 1) * tile] = e4m3_encode(
                blk.astype(np.float64) / sc.astype(np.float64)[..., None, None])
    return codes, scales


def fp8_tile_dequantize(codes: np.ndarray, scales: np.ndarray, tile: int = FP8_TILE) -> np.ndarray:
    """The bf16 operand the tensor cores take: decoded E4M3 value times its
    tile's fp32 scale (an fp32 product), rounded to bf16."""
    rows, cols = codes.shape[-2:]
    sc = np.repeat(np.repeat(scales, tile, axis=-2), tile, axis=-1)[..., :rows, :cols]
    return bf16_round((e4m3_decode(codes).astype(np.float32) * sc).astype(np.float32))
