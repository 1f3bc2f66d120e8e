"""Python binding of libmoe: one function per C entry point, same names.

Each function only marshals arguments (checks device, dtype, contiguity and
shape; passes ``data_ptr()`` and the current CUDA stream) and raises
:class:`MoEError` on a non-OK status.  All computation happens in the CUDA
kernels of libmoe.so.  :class:`MoELayer` owns the buffers of one layer and
calls the entry points in forward/backward order.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from .inputs import MoEConfig

BF16, F32, I32 = torch.bfloat16, torch.float32, torch.int32


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        lib = _lib.load()
        super().__init__(f"{fn}: {lib.moe_status_string(code).decode()} (status {code})")
        self.code = code


def _check(fn: str, code: int):
    if code != 0:
        raise MoEError(fn, code)


def _p(t: torch.Tensor | None, dtype=None, shape=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(stream)


def make_desc(cfg: MoEConfig) -> _lib.MoeDesc:
    return _lib.MoeDesc(cfg.n_tok, cfg.d_model, cfg.d_ff, cfg.n_exp, cfg.top_k,
                        1 if cfg.gate == "sigmoid" else 0, 1 if cfg.use_bias else 0,
                        cfg.n_shared, cfg.d_ff_shared if cfg.n_shared else 0,
                        {"bf16": 0, "mxfp8": 1, "fp8w": 2}[cfg.precision])


# --------------------------------------------------------------- entry points
def moe_workspace_size(desc: _lib.MoeDesc) -> tuple[int, int]:
    f, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check("moe_workspace_size", _lib.load().moe_workspace_size(ctypes.byref(desc), ctypes.byref(f), ctypes.byref(b)))
    return f.value, b.value


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check("moe_workspace_init", _lib.load().moe_workspace_init(_p(ws, name="ws"), ws.numel() * ws.element_size(),
                                                                _s(stream)))


def moe_get_device_status(ws: torch.Tensor, stream=None) -> tuple[int, int]:
    out = (ctypes.c_int32 * 2)()
    _check("moe_get_device_status", _lib.load().moe_get_device_status(_p(ws, name="ws"), out, _s(stream)))
    return out[0], out[1]


def moe_route(desc, x, w_gate, bias, logits, topk_idx, topk_w, counts, offsets, ws, stream=None):
    n, d, e, k = desc.n_tok, desc.d_model, desc.n_exp, desc.top_k
    _check("moe_route", _lib.load().moe_route(
        ctypes.byref(desc), _p(x, BF16, (n, d), "x"), _p(w_gate, BF16, (e, d), "w_gate"),
        _p(bias, F32, (e,), "bias"), _p(logits, F32, (n, e), "logits"), _p(topk_idx, I32, (n, k), "topk_idx"),
        _p(topk_w, F32, (n, k), "topk_w"), _p(counts, I32, (e,), "counts"), _p(offsets, I32, (e + 1,), "offsets"),
        _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


def moe_route_from_logits(desc, logits, bias, topk_idx, topk_w, counts, offsets, ws, stream=None):
    n, e, k = desc.n_tok, desc.n_exp, desc.top_k
    _check("moe_route_from_logits", _lib.load().moe_route_from_logits(
        ctypes.byref(desc), _p(logits, F32, (n, e), "logits"), _p(bias, F32, (e,), "bias"),
        _p(topk_idx, I32, (n, k), "topk_idx"), _p(topk_w, F32, (n, k), "topk_w"), _p(counts, I32, (e,), "counts"),
        _p(offsets, I32, (e + 1,), "offsets"), _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


def moe_route_permute(desc, x, w_gate, bias, logits, topk_idx, topk_w, counts, offsets, row_of_copy, copy_of_row,
                      x_perm, ws, stream=None):
    n, d, e, k = desc.n_tok, desc.d_model, desc.n_exp, desc.top_k
    r = n * k
    _check("moe_route_permute", _lib.load().moe_route_permute(
        ctypes.byref(desc), _p(x, BF16, (n, d), "x"), _p(w_gate, BF16, (e, d), "w_gate"),
        _p(bias, F32, (e,), "bias"), _p(logits, F32, (n, e), "logits"), _p(topk_idx, I32, (n, k), "topk_idx"),
        _p(topk_w, F32, (n, k), "topk_w"), _p(counts, I32, (e,), "counts"), _p(offsets, I32, (e + 1,), "offsets"),
        _p(row_of_copy, I32, (r,), "row_of_copy"), _p(copy_of_row, I32, (r,), "copy_of_row"),
        _p(x_perm, BF16, (r, d), "x_perm"), _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


def moe_permute(desc, x, topk_idx, offsets, row_of_copy, copy_of_row, x_perm, ws, stream=None):
    n, d, e, k = desc.n_tok, desc.d_model, desc.n_exp, desc.top_k
    r = n * k
    _check("moe_permute", _lib.load().moe_permute(
        ctypes.byref(desc), _p(x, BF16, (n, d), "x"), _p(topk_idx, I32, (n, k), "topk_idx"),
        _p(offsets, I32, (e + 1,), "offsets"), _p(row_of_copy, I32, (r,), "row_of_copy"),
        _p(copy_of_row, I32, (r,), "copy_of_row"), _p(x_perm, BF16, (r, d), "x_perm"), _p(ws, name="ws"),
        ws.numel() * ws.element_size(), _s(stream)))


def moe_permute_noalloc(desc, x, topk_idx, offsets, row_of_copy, copy_of_row, x_perm, stream=None):
    """moe_permute for callers that cannot provide a workspace (see moe.h):
    the chunk tables live in a fixed device array inside the library."""
    n, d, e, k = desc.n_tok, desc.d_model, desc.n_exp, desc.top_k
    r = n * k
    _check("moe_permute_noalloc", _lib.load().moe_permute_noalloc(
        ctypes.byref(desc), _p(x, BF16, (n, d), "x"), _p(topk_idx, I32, (n, k), "topk_idx"),
        _p(offsets, I32, (e + 1,), "offsets"), _p(row_of_copy, I32, (r,), "row_of_copy"),
        _p(copy_of_row, I32, (r,), "copy_of_row"), _p(x_perm, BF16, (r, d), "x_perm"), _s(stream)))


def moe_grouped_ffn(desc, x_perm, offsets, x, w1, w3, w2, ws1, ws3, ws2, a1, a3, h, a1s, a3s, hs, y_perm,
                    y_shared, ws, stream=None):
    n, d, f, e, k = desc.n_tok, desc.d_model, desc.d_ff, desc.n_exp, desc.top_k
    r, fs = n * k, desc.d_ff_shared
    sh = desc.n_shared
    w = _lib.MoeExpertWeights(_p(w1, BF16, (e, f, d), "w1"), _p(w3, BF16, (e, f, d), "w3"),
                              _p(w2, BF16, (e, d, f), "w2"),
                              _p(ws1, BF16, (fs, d), "ws1") if sh else None,
                              _p(ws3, BF16, (fs, d), "ws3") if sh else None,
                              _p(ws2, BF16, (d, fs), "ws2") if sh else None)
    sv = _lib.MoeFfnSaved(_p(a1, BF16, (r, f), "a1"), _p(a3, BF16, (r, f), "a3"), _p(h, BF16, (r, f), "h"),
                          _p(a1s, BF16, (n, fs), "a1s") if sh else None,
                          _p(a3s, BF16, (n, fs), "a3s") if sh else None,
                          _p(hs, BF16, (n, fs), "hs") if sh else None)
    _check("moe_grouped_ffn", _lib.load().moe_grouped_ffn(
        ctypes.byref(desc), _p(x_perm, BF16, (r, d), "x_perm"), _p(offsets, I32, (e + 1,), "offsets"),
        _p(x, BF16, (n, d), "x") if sh else None, ctypes.byref(w), ctypes.byref(sv),
        _p(y_perm, BF16, (r, d), "y_perm"), _p(y_shared, BF16, (n, d), "y_shared") if sh else None,
        _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


def moe_permute_maps(desc, topk_idx, offsets, row_of_copy, copy_of_row, ws, stream=None):
    """The permutation maps of moe_permute without copying any row."""
    n, e, k = desc.n_tok, desc.n_exp, desc.top_k
    r = n * k
    _check("moe_permute_maps", _lib.load().moe_permute_maps(
        ctypes.byref(desc), _p(topk_idx, I32, (n, k), "topk_idx"), _p(offsets, I32, (e + 1,), "offsets"),
        _p(row_of_copy, I32, (r,), "row_of_copy"), _p(copy_of_row, I32, (r,), "copy_of_row"), _p(ws, name="ws"),
        ws.numel() * ws.element_size(), _s(stream)))


def moe_grouped_ffn_gather(desc, x, copy_of_row, offsets, w1, w3, w2, ws1, ws3, ws2, a1, a3, h, a1s, a3s, hs,
                           y_perm, y_shared, ws, stream=None):
    """moe_grouped_ffn reading GEMM1's rows from x through copy_of_row (TMA gathers)."""
    n, d, f, e, k = desc.n_tok, desc.d_model, desc.d_ff, desc.n_exp, desc.top_k
    r, fs = n * k, desc.d_ff_shared
    sh = desc.n_shared
    w = _lib.MoeExpertWeights(_p(w1, BF16, (e, f, d), "w1"), _p(w3, BF16, (e, f, d), "w3"),
                              _p(w2, BF16, (e, d, f), "w2"),
                              _p(ws1, BF16, (fs, d), "ws1") if sh else None,
                              _p(ws3, BF16, (fs, d), "ws3") if sh else None,
                              _p(ws2, BF16, (d, fs), "ws2") if sh else None)
    sv = _lib.MoeFfnSaved(_p(a1, BF16, (r, f), "a1"), _p(a3, BF16, (r, f), "a3"), _p(h, BF16, (r, f), "h"),
                          _p(a1s, BF16, (n, fs), "a1s") if sh else None,
                          _p(a3s, BF16, (n, fs), "a3s") if sh else None,
                          _p(hs, BF16, (n, fs), "hs") if sh else None)
    _check("moe_grouped_ffn_gather", _lib.load().moe_grouped_ffn_gather(
        ctypes.byref(desc), _p(x, BF16, (n, d), "x"), _p(copy_of_row, I32, (r,), "copy_of_row"),
        _p(offsets, I32, (e + 1,), "offsets"), ctypes.byref(w), ctypes.byref(sv),
        _p(y_perm, BF16, (r, d), "y_perm"), _p(y_shared, BF16, (n, d), "y_shared") if sh else None,
        _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


def moe_combine(desc, y_perm, row_of_copy, topk_w, y_shared, out, stream=None):
    n, d, k = desc.n_tok, desc.d_model, desc.top_k
    r = n * k
    _check("moe_combine", _lib.load().moe_combine(
        ctypes.byref(desc), _p(y_perm, BF16, (r, d), "y_perm"), _p(row_of_copy, I32, (r,), "row_of_copy"),
        _p(topk_w, F32, (n, k), "topk_w"), _p(y_shared, BF16, (n, d), "y_shared"), _p(out, BF16, (n, d), "out"),
        _s(stream)))


def _bwd_structs(desc, state: dict, grads: dict, need_x_perm: bool = True):
    n, d, f, e, k = desc.n_tok, desc.d_model, desc.d_ff, desc.n_exp, desc.top_k
    r, fs, sh = n * k, desc.d_ff_shared, desc.n_shared
    S = state
    st = _lib.MoeFwdState(
        _p(S["x"], BF16, (n, d), "x"),
        _p(S.get("x_perm"), BF16, (r, d), "x_perm") if (need_x_perm or S.get("x_perm") is not None) else None,
        _p(S["logits"], F32, (n, e), "logits"),
        _p(S["topk_idx"], I32, (n, k), "topk_idx"), _p(S["topk_w"], F32, (n, k), "topk_w"),
        _p(S["offsets"], I32, (e + 1,), "offsets"), _p(S["row_of_copy"], I32, (r,), "row_of_copy"),
        _p(S["copy_of_row"], I32, (r,), "copy_of_row"), _p(S["a1"], BF16, (r, f), "a1"), _p(S["a3"], BF16, (r, f), "a3"),
        _p(S["h"], BF16, (r, f), "h"), _p(S["y_perm"], BF16, (r, d), "y_perm"),
        _p(S.get("a1s"), BF16, (n, fs), "a1s") if sh else None, _p(S.get("a3s"), BF16, (n, fs), "a3s") if sh else None,
        _p(S.get("hs"), BF16, (n, fs), "hs") if sh else None,
        _p(S.get("offsets_full"), I32, (e + 1,), "offsets_full"),
        _p(S.get("copy_of_row_full"), I32, (r,), "copy_of_row_full"))
    G = grads
    gr = _lib.MoeGrads(
        _p(G["dx"], BF16, (n, d), "dx"), _p(G["dw_gate"], F32, (e, d), "dw_gate"), _p(G["dw1"], F32, (e, f, d), "dw1"),
        _p(G["dw3"], F32, (e, f, d), "dw3"), _p(G["dw2"], F32, (e, d, f), "dw2"),
        _p(G.get("dws1"), F32, (fs, d), "dws1") if sh else None, _p(G.get("dws3"), F32, (fs, d), "dws3") if sh else None,
        _p(G.get("dws2"), F32, (d, fs), "dws2") if sh else None,
        _p(G.get("dg"), F32, (n, k), "dg"), _p(G.get("dlogits"), F32, (n, k), "dlogits"))
    return st, gr


def moe_backward(desc, w_gate, weights: dict, state: dict, dy, grads: dict, ws, stream=None):
    """``weights``: w1, w3, w2 (+ ws1, ws3, ws2); ``state``: the fields of
    moe_fwd_state_t; ``grads``: the fields of moe_grads_t (dg, dlogits optional)."""
    n, d, f, e = desc.n_tok, desc.d_model, desc.d_ff, desc.n_exp
    fs, sh = desc.d_ff_shared, desc.n_shared
    w = _lib.MoeExpertWeights(_p(weights["w1"], BF16, (e, f, d), "w1"), _p(weights["w3"], BF16, (e, f, d), "w3"),
                              _p(weights["w2"], BF16, (e, d, f), "w2"),
                              _p(weights.get("ws1"), BF16, (fs, d), "ws1") if sh else None,
                              _p(weights.get("ws3"), BF16, (fs, d), "ws3") if sh else None,
                              _p(weights.get("ws2"), BF16, (d, fs), "ws2") if sh else None)
    st, gr = _bwd_structs(desc, state, grads)
    _check("moe_backward", _lib.load().moe_backward(
        ctypes.byref(desc), _p(w_gate, BF16, (e, d), "w_gate"), ctypes.byref(w), ctypes.byref(st),
        _p(dy, BF16, (n, d), "dy"), ctypes.byref(gr), _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


def moe_permute_capacity(desc, x, topk_idx, offsets, capacity_factor: float, row_of_copy_full, copy_of_row_full,
                         kept_offsets, row_of_copy, copy_of_row, x_perm, n_dropped, ws, stream=None):
    n, d, e, k = desc.n_tok, desc.d_model, desc.n_exp, desc.top_k
    r = n * k
    _check("moe_permute_capacity", _lib.load().moe_permute_capacity(
        ctypes.byref(desc), _p(x, BF16, (n, d), "x"), _p(topk_idx, I32, (n, k), "topk_idx"),
        _p(offsets, I32, (e + 1,), "offsets"), ctypes.c_double(capacity_factor),
        _p(row_of_copy_full, I32, (r,), "row_of_copy_full"), _p(copy_of_row_full, I32, (r,), "copy_of_row_full"),
        _p(kept_offsets, I32, (e + 1,), "kept_offsets"), _p(row_of_copy, I32, (r,), "row_of_copy"),
        _p(copy_of_row, I32, (r,), "copy_of_row"), _p(x_perm, BF16, (r, d), "x_perm"),
        _p(n_dropped, I32, (1,), "n_dropped"), _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


def moe_aux_loss(desc, logits, counts, loss, dlogits_aux=None, ws=None, coef: float = 1.0, stream=None):
    """``loss``: fp32 device tensor of one element; ``dlogits_aux``: optional
    fp32 [N, E] receiving the loss's logit gradient."""
    n, e = desc.n_tok, desc.n_exp
    _check("moe_aux_loss", _lib.load().moe_aux_loss(
        ctypes.byref(desc), _p(logits, F32, (n, e), "logits"), _p(counts, I32, (e,), "counts"), ctypes.c_float(coef),
        _p(loss, F32, (1,), "loss"), _p(dlogits_aux, F32, (n, e), "dlogits_aux"), _p(ws, name="ws"),
        ws.numel() * ws.element_size(), _s(stream)))


def moe_monitor_stats(counts_hist, stats, stream=None):
    """``counts_hist``: int32 [H, E] device tensor (one routing histogram per
    step); ``stats``: fp32 device tensor [3] <- min load, entropy, cold experts."""
    h, e = counts_hist.shape
    _check("moe_monitor_stats", _lib.load().moe_monitor_stats(
        e, _p(counts_hist, I32, (h, e), "counts_hist"), h, _p(stats, F32, (3,), "stats"), _s(stream)))


# --------------------------------------------------------------- kernel timing
TIMING_KINDS = {"gate": 0, "ffn_fwd": 1, "dgrad": 2, "wgrad": 3}


def moe_timing_enable(capacity: int = 4096):
    """Start timing the library's grouped-GEMM launches with CUDA events
    (``capacity`` launches at most; earlier records are cleared)."""
    _check("moe_timing_enable", _lib.load().moe_timing_enable(capacity))


def moe_timing_read(kind: str) -> tuple[float, int, int]:
    """(total milliseconds, timed launches, untimed launches) of one kind of
    grouped GEMM since moe_timing_enable; waits for the recorded events."""
    ms, n, u = ctypes.c_double(), ctypes.c_int64(), ctypes.c_int64()
    _check("moe_timing_read", _lib.load().moe_timing_read(TIMING_KINDS[kind], ctypes.byref(ms), ctypes.byref(n),
                                                          ctypes.byref(u)))
    return ms.value, n.value, u.value


def moe_timing_disable():
    _check("moe_timing_disable", _lib.load().moe_timing_disable())


def moe_selftest_wait_timeout(ws, limit_ns: int, site: int, stream=None):
    """Run the library's bounded-wait self-test (see moe.h): a wait that
    nothing completes runs out after ``limit_ns`` and reports through the
    status words of ``ws``."""
    _check("moe_selftest_wait_timeout", _lib.load().moe_selftest_wait_timeout(
        _p(ws, name="ws"), ws.numel() * ws.element_size(), int(limit_ns), int(site), _s(stream)))


def moe_update_bias(desc, counts, bias, gamma: float, mode: int = 0, stream=None):
    _check("moe_update_bias", _lib.load().moe_update_bias(
        ctypes.byref(desc), _p(counts, I32, (desc.n_exp,), "counts"), _p(bias, F32, (desc.n_exp,), "bias"),
        ctypes.c_float(gamma), mode, _s(stream)))


# --------------------------------------------------------------- MXFP8 forward
U8 = torch.uint8


def mx_scale_ld(rows: int) -> int:
    """Leading dimension of an MXFP8 scale array (rows rounded up to 16)."""
    return (rows + 15) // 16 * 16


def moe_quantize_mxfp8(src, codes, scales, stream=None):
    """src bf16 [G, rows, cols] (or [rows, cols]) -> codes uint8 (same shape),
    scales uint8 [G, cols/32, ld] (or [cols/32, ld]), ld = mx_scale_ld(rows)."""
    g, rows, cols = (1,) + tuple(src.shape) if src.dim() == 2 else tuple(src.shape)
    ld = scales.shape[-1]
    _check("moe_quantize_mxfp8", _lib.load().moe_quantize_mxfp8(
        _p(src, BF16, name="src"), g, rows, cols, _p(codes, U8, tuple(src.shape), "codes"),
        _p(scales, U8, (scales.shape if src.dim() == 3 else (cols // 32, ld)), "scales"), ld, _s(stream)))


def quantize_weights_mxfp8(p: dict, stream=None) -> dict:
    """MXFP8 copies (codes, scales) of the expert weights in ``p``."""
    out = {}
    for key in ("w1", "w3", "w2", "ws1", "ws3", "ws2"):
        w = p.get(key)
        if w is None:
            continue
        codes = torch.empty(w.shape, dtype=U8, device=w.device)
        rows, cols = w.shape[-2], w.shape[-1]
        sshape = (w.shape[0], cols // 32, mx_scale_ld(rows)) if w.dim() == 3 else (cols // 32, mx_scale_ld(rows))
        scales = torch.zeros(sshape, dtype=U8, device=w.device)
        moe_quantize_mxfp8(w, codes, scales, stream)
        out[key], out[key + "_scale"] = codes, scales
    return out


def moe_quantize_mxfp8_t(src, codes, scales, stream=None):
    """src bf16 [G, rows, cols] (or [rows, cols]) quantised along rows and
    transposed: codes uint8 [G, cols, rows], scales uint8 [G, rows/32, ld]
    (ld = scales.shape[-1] >= cols, a multiple of 16)."""
    g, rows, cols = (1,) + tuple(src.shape) if src.dim() == 2 else tuple(src.shape)
    ld = scales.shape[-1]
    cshape = (cols, rows) if src.dim() == 2 else (g, cols, rows)
    sshape = (rows // 32, ld) if src.dim() == 2 else (g, rows // 32, ld)
    _check("moe_quantize_mxfp8_t", _lib.load().moe_quantize_mxfp8_t(
        _p(src, BF16, name="src"), g, rows, cols, _p(codes, U8, cshape, "codes"), _p(scales, U8, sshape, "scales"),
        ld, _s(stream)))


def quantize_weights_mxfp8_t(p: dict, stream=None) -> dict:
    """Transposed MXFP8 copies of the expert weights for the backward's data
    gradients (quantised along the other weight dimension)."""
    out = {}
    for key in ("w1", "w3", "w2", "ws1", "ws3", "ws2"):
        w = p.get(key)
        if w is None:
            continue
        rows, cols = w.shape[-2], w.shape[-1]
        lead = (w.shape[0],) if w.dim() == 3 else ()
        codes = torch.empty(lead + (cols, rows), dtype=U8, device=w.device)
        scales = torch.zeros(lead + (rows // 32, mx_scale_ld(cols)), dtype=U8, device=w.device)
        moe_quantize_mxfp8_t(w, codes, scales, stream)
        out[key], out[key + "_scale"] = codes, scales
    return out


def moe_backward_mxfp8(desc, w_gate, wt: dict, state: dict, dy, grads: dict, ws, stream=None):
    """Backward of the MXFP8 layer.  ``wt``: output of
    :func:`quantize_weights_mxfp8_t`; ``state`` as for :func:`moe_backward`
    (x_perm not needed)."""
    n, d, e, sh = desc.n_tok, desc.d_model, desc.n_exp, desc.n_shared
    w = _lib.MoeExpertWeightsMx(*[_p(wt.get(key)) if (sh or not key.startswith("ws")) else None
                                  for key in ("w1", "w1_scale", "w3", "w3_scale", "w2", "w2_scale",
                                              "ws1", "ws1_scale", "ws3", "ws3_scale", "ws2", "ws2_scale")])
    st, gr = _bwd_structs(desc, state, grads, need_x_perm=False)
    _check("moe_backward_mxfp8", _lib.load().moe_backward_mxfp8(
        ctypes.byref(desc), _p(w_gate, BF16, (e, d), "w_gate"), ctypes.byref(w), ctypes.byref(st),
        _p(dy, BF16, (n, d), "dy"), ctypes.byref(gr), _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


# --------------------------------------------------------------- FP8 weights
def quantize_weights_fp8_tile(p: dict, stream=None) -> dict:
    """E4M3 codes with one fp32 scale per 128 x 128 tile of every expert
    weight in ``p`` (keys w1, w3, w2, ws1, ws3, ws2 and *_scale)."""
    out = {}
    for key in ("w1", "w3", "w2", "ws1", "ws3", "ws2"):
        w = p.get(key)
        if w is None:
            continue
        g, rows, cols = (1,) + tuple(w.shape) if w.dim() == 2 else tuple(w.shape)
        codes = torch.empty(w.shape, dtype=U8, device=w.device)
        lead = (w.shape[0],) if w.dim() == 3 else ()
        scales = torch.empty(lead + ((rows + 127) // 128, (cols + 127) // 128), dtype=F32, device=w.device)
        _check("moe_quantize_fp8_tile", _lib.load().moe_quantize_fp8_tile(
            _p(w, BF16, name=key), g, rows, cols, _p(codes, U8, name=key + " codes"),
            _p(scales, F32, name=key + " scales"), _s(stream)))
        out[key], out[key + "_scale"] = codes, scales
    return out


def _mx_struct(desc, wq):
    sh = desc.n_shared
    return _lib.MoeExpertWeightsMx(*[_p(wq.get(key)) if (sh or not key.startswith("ws")) else None
                                     for key in ("w1", "w1_scale", "w3", "w3_scale", "w2", "w2_scale",
                                                 "ws1", "ws1_scale", "ws3", "ws3_scale", "ws2", "ws2_scale")])


def moe_grouped_ffn_fp8w(desc, x_perm, offsets, x, wq: dict, saved: dict, y_perm, y_shared, ws, stream=None):
    """``wq``: output of :func:`quantize_weights_fp8_tile`; other arguments as
    :func:`moe_grouped_ffn` (``saved``: a1, a3, h, a1s, a3s, hs)."""
    n, d, e, k = desc.n_tok, desc.d_model, desc.n_exp, desc.top_k
    r, sh = n * k, desc.n_shared
    w = _mx_struct(desc, wq)
    sv = _lib.MoeFfnSaved(*[_p(saved.get(key)) for key in ("a1", "a3", "h", "a1s", "a3s", "hs")])
    _check("moe_grouped_ffn_fp8w", _lib.load().moe_grouped_ffn_fp8w(
        ctypes.byref(desc), _p(x_perm, BF16, (r, d), "x_perm"), _p(offsets, I32, (e + 1,), "offsets"),
        _p(x, BF16, (n, d), "x"), ctypes.byref(w), ctypes.byref(sv), _p(y_perm, BF16, (r, d), "y_perm"),
        _p(y_shared, BF16, (n, d), "y_shared") if sh else None, _p(ws, name="ws"), ws.numel() * ws.element_size(),
        _s(stream)))


def moe_backward_fp8w(desc, w_gate, wq: dict, state: dict, dy, grads: dict, ws, stream=None):
    n, d, e = desc.n_tok, desc.d_model, desc.n_exp
    w = _mx_struct(desc, wq)
    st, gr = _bwd_structs(desc, state, grads)
    _check("moe_backward_fp8w", _lib.load().moe_backward_fp8w(
        ctypes.byref(desc), _p(w_gate, BF16, (e, d), "w_gate"), ctypes.byref(w), ctypes.byref(st),
        _p(dy, BF16, (n, d), "dy"), ctypes.byref(gr), _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


def moe_permute_mxfp8(desc, x, topk_idx, offsets, row_of_copy, copy_of_row, xq_perm, xs_perm, xq_tok, xs_tok, ws,
                      stream=None):
    n, d, e, k = desc.n_tok, desc.d_model, desc.n_exp, desc.top_k
    r = n * k
    _check("moe_permute_mxfp8", _lib.load().moe_permute_mxfp8(
        ctypes.byref(desc), _p(x, BF16, (n, d), "x"), _p(topk_idx, I32, (n, k), "topk_idx"),
        _p(offsets, I32, (e + 1,), "offsets"), _p(row_of_copy, I32, (r,), "row_of_copy"),
        _p(copy_of_row, I32, (r,), "copy_of_row"), _p(xq_perm, U8, (r, d), "xq_perm"),
        _p(xs_perm, U8, (d // 32, mx_scale_ld(r)), "xs_perm"), _p(xq_tok, U8, (n, d), "xq_tok"),
        _p(xs_tok, U8, (d // 32, mx_scale_ld(n)), "xs_tok"), _p(ws, name="ws"), ws.numel() * ws.element_size(),
        _s(stream)))


def moe_grouped_ffn_mxfp8(desc, xq_perm, xs_perm, offsets, xq_tok, xs_tok, wq: dict, saved: dict, y_perm, y_shared,
                          ws, stream=None):
    """``wq``: output of :func:`quantize_weights_mxfp8`; ``saved``: optional bf16
    a1, a3, h, a1s, a3s, hs for a bf16 backward (missing keys = not saved)."""
    n, d, f, e, k = desc.n_tok, desc.d_model, desc.d_ff, desc.n_exp, desc.top_k
    r, fs, sh = n * k, desc.d_ff_shared, desc.n_shared
    w = _lib.MoeExpertWeightsMx(*[_p(wq.get(key)) if (sh or not key.startswith("ws")) else None
                                  for key in ("w1", "w1_scale", "w3", "w3_scale", "w2", "w2_scale",
                                              "ws1", "ws1_scale", "ws3", "ws3_scale", "ws2", "ws2_scale")])
    sv = _lib.MoeFfnSaved(*[_p(saved.get(key)) for key in ("a1", "a3", "h", "a1s", "a3s", "hs")])
    _check("moe_grouped_ffn_mxfp8", _lib.load().moe_grouped_ffn_mxfp8(
        ctypes.byref(desc), _p(xq_perm, U8, (r, d), "xq_perm"), _p(xs_perm, U8, (d // 32, mx_scale_ld(r)), "xs_perm"),
        _p(offsets, I32, (e + 1,), "offsets"), _p(xq_tok, U8, (n, d), "xq_tok") if sh else None,
        _p(xs_tok, U8, (d // 32, mx_scale_ld(n)), "xs_tok") if sh else None, ctypes.byref(w), ctypes.byref(sv),
        _p(y_perm, BF16, (r, d), "y_perm"), _p(y_shared, BF16, (n, d), "y_shared") if sh else None,
        _p(ws, name="ws"), ws.numel() * ws.element_size(), _s(stream)))


# --------------------------------------------------------------- layer runner
class MoELayer:
    """Buffers of one layer plus the forward / backward call sequences.

    ``params``: x-independent tensors from :func:`inputs.make_layer` on the GPU
    (w_gate, w1, w3, w2, bias, and ws1, ws3, ws2 with a shared expert).
    """

    def __init__(self, cfg: MoEConfig, params: dict, train: bool = True, device="cuda", gather: bool = False,
                 fused_dispatch: bool = True):
        self.cfg = cfg
        self.desc = make_desc(cfg)
        self.p = params
        self.train = train
        n, d, f, e, k = cfg.n_tok, cfg.d_model, cfg.d_ff, cfg.n_exp, cfg.top_k
        r, fs = cfg.rows, cfg.d_ff_shared
        z = lambda *s, dt=BF16: torch.empty(s, dtype=dt, device=device)  # noqa: E731
        # gather=True (inference, bf16 experts, no capacity): GEMM1 reads its rows
        # straight from x (moe_permute_maps + moe_grouped_ffn_gather), no x_perm
        self.gather = gather and (not train) and cfg.precision == "bf16" and cfg.capacity_factor <= 0
        self.buf = {
            "logits": z(n, e, dt=F32), "topk_idx": z(n, k, dt=I32), "topk_w": z(n, k, dt=F32),
            "counts": z(e, dt=I32), "offsets": z(e + 1, dt=I32), "row_of_copy": z(r, dt=I32),
            "copy_of_row": z(r, dt=I32), "x_perm": None if self.gather else z(r, d), "h": z(r, f),
            "y_perm": z(r, d), "out": z(n, d),
            "a1": z(r, f) if train else None, "a3": z(r, f) if train else None,
        }
        if cfg.n_shared:
            self.buf.update(hs=z(n, fs), y_shared=z(n, d), a1s=z(n, fs) if train else None,
                            a3s=z(n, fs) if train else None)
        else:
            self.buf.update(hs=None, y_shared=None, a1s=None, a3s=None)
        self.w8 = cfg.precision == "fp8w"
        self.w8q = quantize_weights_fp8_tile(params) if self.w8 else None
        self.cap = cfg.capacity_factor > 0
        if self.cap:
            if cfg.precision == "mxfp8":
                raise ValueError("the capacity-factor mode runs with bf16 operands")
            # routing writes the dropless offsets here; b["offsets"] holds the kept ones
            self.buf.update(offsets_full=z(e + 1, dt=I32), row_of_copy_full=z(r, dt=I32),
                            copy_of_row_full=z(r, dt=I32), n_dropped=z(1, dt=I32))
        self.mx = cfg.precision == "mxfp8"
        # E <= 32, bf16 rows, dropless, permuted copy: routing and dispatch in
        # one launch (moe_route_permute); fused_dispatch=False keeps two calls
        self.fused_dispatch = (fused_dispatch and e <= 32 and not self.mx and not self.cap and not self.gather)
        if self.mx:
            self.wq = quantize_weights_mxfp8(params)
            self.wqt = quantize_weights_mxfp8_t(params) if train else None
            self.buf.update(xq_perm=z(r, d, dt=U8), xs_perm=torch.zeros(d // 32, mx_scale_ld(r), dtype=U8, device=device),
                            xq_tok=z(n, d, dt=U8) if cfg.n_shared else None,
                            xs_tok=(torch.zeros(d // 32, mx_scale_ld(n), dtype=U8, device=device)
                                    if cfg.n_shared else None))
        fwd_b, bwd_b = moe_workspace_size(self.desc)
        self.ws = torch.empty((bwd_b if train else fwd_b) + 256, dtype=torch.uint8, device=device)
        moe_workspace_init(self.ws)
        self.grads = None
        if train:
            self.grads = {"dx": z(n, d), "dw_gate": z(e, d, dt=F32), "dw1": z(e, f, d, dt=F32),
                          "dw3": z(e, f, d, dt=F32), "dw2": z(e, d, f, dt=F32), "dg": z(n, k, dt=F32),
                          "dlogits": z(n, k, dt=F32)}
            if cfg.n_shared:
                self.grads.update(dws1=z(fs, d, dt=F32), dws3=z(fs, d, dt=F32), dws2=z(d, fs, dt=F32))
        self.x = None

    def forward(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        b, p = self.buf, self.p
        self.x = x
        if self.fused_dispatch:
            # routing and the permuted copy of the tokens in one launch (E <= 32)
            moe_route_permute(self.desc, x, p["w_gate"], p.get("bias"), b["logits"], b["topk_idx"], b["topk_w"],
                              b["counts"], b["offsets"], b["row_of_copy"], b["copy_of_row"], b["x_perm"], self.ws,
                              stream)
            return self._ffn_combine(x, stream)
        moe_route(self.desc, x, p["w_gate"], p.get("bias"), b["logits"], b["topk_idx"], b["topk_w"], b["counts"],
                  b["offsets_full"] if self.cap else b["offsets"], self.ws, stream)
        if self.mx:
            return self._forward_mx(x, stream)
        if self.gather:
            b = self.buf
            moe_permute_maps(self.desc, b["topk_idx"], b["offsets"], b["row_of_copy"], b["copy_of_row"], self.ws,
                             stream)
            moe_grouped_ffn_gather(self.desc, x, b["copy_of_row"], b["offsets"], p["w1"], p["w3"], p["w2"],
                                   p.get("ws1"), p.get("ws3"), p.get("ws2"), None, None, b["h"], None, None,
                                   b["hs"], b["y_perm"], b["y_shared"], self.ws, stream)
            moe_combine(self.desc, b["y_perm"], b["row_of_copy"], b["topk_w"], b["y_shared"], b["out"], stream)
            return b["out"]
        self._permute(x, stream)
        return self._ffn_combine(x, stream)

    def _permute(self, x, stream=None):
        b = self.buf
        if self.cap:
            moe_permute_capacity(self.desc, x, b["topk_idx"], b["offsets_full"], self.cfg.capacity_factor,
                                 b["row_of_copy_full"], b["copy_of_row_full"], b["offsets"], b["row_of_copy"],
                                 b["copy_of_row"], b["x_perm"], b["n_dropped"], self.ws, stream)
        else:
            moe_permute(self.desc, x, b["topk_idx"], b["offsets"], b["row_of_copy"], b["copy_of_row"], b["x_perm"],
                        self.ws, stream)

    def _ffn_combine(self, x, stream=None):
        b, p = self.buf, self.p
        if self.w8:
            saved = {key: b[key] for key in ("a1", "a3", "h", "a1s", "a3s", "hs") if b.get(key) is not None}
            moe_grouped_ffn_fp8w(self.desc, b["x_perm"], b["offsets"], x, self.w8q, saved, b["y_perm"],
                                 b["y_shared"], self.ws, stream)
        else:
            moe_grouped_ffn(self.desc, b["x_perm"], b["offsets"], x, p["w1"], p["w3"], p["w2"], p.get("ws1"),
                            p.get("ws3"), p.get("ws2"), b["a1"], b["a3"], b["h"], b["a1s"], b["a3s"], b["hs"],
                            b["y_perm"], b["y_shared"], self.ws, stream)
        moe_combine(self.desc, b["y_perm"], b["row_of_copy"], b["topk_w"], b["y_shared"], b["out"], stream)
        return b["out"]

    def _forward_mx(self, x, stream=None):
        b = self.buf
        moe_permute_mxfp8(self.desc, x, b["topk_idx"], b["offsets"], b["row_of_copy"], b["copy_of_row"],
                          b["xq_perm"], b["xs_perm"], b["xq_tok"], b["xs_tok"], self.ws, stream)
        saved = ({key: b[key] for key in ("a1", "a3", "h", "a1s", "a3s", "hs") if b.get(key) is not None}
                 if self.train else {})
        moe_grouped_ffn_mxfp8(self.desc, b["xq_perm"], b["xs_perm"], b["offsets"], b["xq_tok"], b["xs_tok"], self.wq,
                              saved, b["y_perm"], b["y_shared"], self.ws, stream)
        moe_combine(self.desc, b["y_perm"], b["row_of_copy"], b["topk_w"], b["y_shared"], b["out"], stream)
        return b["out"]

    def backward(self, dy: torch.Tensor, stream=None) -> dict:
        b = self.buf
        if self.mx:
            state = {key: b[key] for key in ("logits", "topk_idx", "topk_w", "offsets", "row_of_copy",
                                             "copy_of_row", "a1", "a3", "h", "y_perm", "a1s", "a3s", "hs")}
            state["x"] = self.x
            moe_backward_mxfp8(self.desc, self.p["w_gate"], self.wqt, state, dy, self.grads, self.ws, stream)
            return self.grads
        state = {key: b[key] for key in ("x_perm", "logits", "topk_idx", "topk_w", "offsets", "row_of_copy",
                                         "copy_of_row", "a1", "a3", "h", "y_perm", "a1s", "a3s", "hs")}
        state["x"] = self.x
        if self.cap:
            state.update(offsets_full=b["offsets_full"], copy_of_row_full=b["copy_of_row_full"])
        if self.w8:
            moe_backward_fp8w(self.desc, self.p["w_gate"], self.w8q, state, dy, self.grads, self.ws, stream)
        else:
            moe_backward(self.desc, self.p["w_gate"], self.p, state, dy, self.grads, self.ws, stream)
        return self.grads

    def drop_rate(self) -> float:
        """Fraction of token copies dropped by the capacity in the last forward (0 when dropless)."""
        if not self.cap:
            return 0.0
        return int(self.buf["n_dropped"].item()) / self.cfg.rows

    def update_bias(self, gamma: float = 1e-3, mode: int = 0, stream=None):
        moe_update_bias(self.desc, self.buf["counts"], self.p["bias"], gamma, mode, stream)

    def device_status(self) -> tuple[int, int]:
        return moe_get_device_status(self.ws)
