"""Runs the CPU oracle on independent token groups in parallel processes.

The MXFP8 oracle quantises every weight matrix it touches, about a second
per DeepSeek-V3-sized expert matrix, so a full-size token sample takes
minutes on one core.  Tokens are independent in the forward and in the
input-side gradients, so the tests cut a sample into groups of tokens with
few distinct experts and hand each group to one worker of a pool of
processes started with ``spawn`` (never forked from a process that already
holds a CUDA context).  The expert weights are copied once into shared
memory as raw bfloat16 bits; each worker widens only the experts its group
uses.  The workers run the oracle's own top-level functions unchanged."""
from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np


class SharedBf16:
    """A bfloat16 array (given as its uint16 bits) in shared memory."""

    def __init__(self, bits: np.ndarray):
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        self.shm = shared_memory.SharedMemory(create=True, size=max(bits.nbytes, 1))
        np.ndarray(bits.shape, np.uint16, buffer=self.shm.buf)[...] = bits
        self.spec = (self.shm.name, bits.shape)

    def close(self):
        self.shm.close()
        self.shm.unlink()


def _widen(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _experts(spec, used) -> np.ndarray:
    name, shape = spec
    shm = shared_memory.SharedMemory(name=name)
    try:
        arr = np.ndarray(shape, np.uint16, buffer=shm.buf)
        return np.stack([_widen(arr[int(e)]) for e in used])
    finally:
        shm.close()


def run_group(job: dict) -> dict:
    """One group: the oracle's MXFP8 (or bf16) forward and backward on the
    group's tokens, experts re-indexed 0..U-1 in the order of ``used``."""
    import oracle as O
    used = job["used"]
    w1, w3, w2 = (_experts(job[k], used) for k in ("w1", "w3", "w2"))
    x, ic, g, lgc, dy, wg = job["x"], job["idx"], job["g"], job["logits"], job["dy"], job["w_gate"]
    shared = job["shared"]
    if job["mxfp8"]:
        out, saved = O.moe_forward_mxfp8(x, ic, g, w1, w3, w2, shared, return_saved=True)
        rg = O.moe_backward_mxfp8(dy, x, lgc, ic, g, wg, w1, w3, w2, saved, job["gate"], shared)
    else:
        out, saved = O.moe_forward(x, lgc, ic, g, w1, w3, w2, shared)
        rg = O.moe_backward(dy, x, lgc, ic, g, wg, w1, w3, w2, saved, job["gate"], shared)
    keep = job.get("keep", ("dx", "dg", "dlogits"))
    res = {"out": out}
    res.update({k: rg[k] for k in keep})
    return res


def _init_worker():
    # one BLAS thread per worker: the pool itself provides the parallelism
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"


def run_groups(jobs: list[dict]) -> list[dict]:
    """run_group over ``jobs`` in a spawn pool (one process per core, at most one per job)."""
    if not jobs:
        return []
    n = max(1, min(len(jobs), os.cpu_count() or 1))
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    _init_worker()          # inherited by the spawned workers when they import numpy
    try:
        with mp.get_context("spawn").Pool(n, initializer=_init_worker) as pool:
            return pool.map(run_group, jobs, chunksize=1)
    finally:
        for v, val in saved.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val


def token_groups(idx: np.ndarray, tokens, max_experts: int, max_tokens: int) -> list[np.ndarray]:
    """Cut ``tokens`` (in order) into groups whose union of experts stays
    within ``max_experts``; at most ``max_tokens`` tokens in all."""
    groups, cur, cur_e, total = [], [], set(), 0
    for t in tokens:
        if total >= max_tokens:
            break
        es = set(idx[t].tolist())
        if cur and len(cur_e | es) > max_experts:
            groups.append(np.array(cur))
            cur, cur_e = [], set()
        cur.append(int(t))
        cur_e |= es
        total += 1
    if cur:
        groups.append(np.array(cur))
    return groups


def per_token_error(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Error of every token row, ``||got_t - want_t||``, over the root mean
    square row norm of ``want``: a token whose row is wrong shows up as an
    error near 1 however many tokens the sample holds, while rows whose own
    norm is small (a dot product that cancels) are not over-weighted."""
    got = np.asarray(got, np.float64).reshape(len(got), -1)
    want = np.asarray(want, np.float64).reshape(len(want), -1)
    scale = np.sqrt(np.mean(np.sum(want * want, axis=1)))
    return np.linalg.norm(got - want, axis=1) / max(scale, 1e-30)
