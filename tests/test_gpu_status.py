"""Device-side input checks report through the status word without faulting:
an expert index outside [0, E) handed to moe_permute sets MOE_DEV_BAD_INDEX,
the copy gets no row (row_of_copy = -1) and every other copy is permuted as
usual.  The bad input is built so that the offsets stay consistent with the
valid copies, so every access of the kernels stays in bounds."""
import numpy as np
import pytest
import torch

import oracle as O
from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, make_layer

pytestmark = pytest.mark.gpu

MOE_DEV_BAD_INDEX = 2


def test_out_of_range_expert_index_is_reported_and_skipped():
    cfg = CONFIGS["tiny"]
    n, e, k, d = cfg.n_tok, cfg.n_exp, cfg.top_k, cfg.d_model
    p = make_layer(cfg, "cpu")
    x = p["x"]
    lg = O.gate_logits(x.float().numpy(), p["w_gate"].float().numpy())
    idx, _ = O.route(lg, None, k, cfg.gate)
    idx = idx.astype(np.int32)
    bad_t, bad_k = 5, 1
    idx[bad_t, bad_k] = e                                   # one index outside [0, E)
    valid = idx[(idx >= 0) & (idx < e)]
    counts = np.bincount(valid, minlength=e)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)   # ends at N*K - 1
    desc = api.make_desc(cfg)
    f, _ = api.moe_workspace_size(desc)
    ws = torch.empty(f, dtype=torch.uint8, device="cuda")
    api.moe_workspace_init(ws)
    r = n * k
    row_of_copy = torch.full((r,), 12345, dtype=torch.int32, device="cuda")
    copy_of_row = torch.full((r,), -7, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros(r, d, dtype=torch.bfloat16, device="cuda")
    api.moe_permute(desc, x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(offsets).cuda(), row_of_copy,
                    copy_of_row, x_perm, ws)
    torch.cuda.synchronize()
    bits, _ = api.moe_get_device_status(ws)
    assert bits & MOE_DEV_BAD_INDEX
    roc = row_of_copy.cpu().numpy()
    bad_c = bad_t * k + bad_k
    assert roc[bad_c] == -1
    good = np.ones(r, bool)
    good[bad_c] = False
    # the valid copies fill rows 0..R-2 exactly once, each row holding its token's x
    assert np.array_equal(np.sort(roc[good]), np.arange(r - 1))
    cor = copy_of_row.cpu().numpy()
    assert np.array_equal(cor[roc[good]], np.nonzero(good)[0])
    xp = x_perm.cpu()
    for c in np.nonzero(good)[0][::17]:
        assert torch.equal(xp[roc[c]], x[c // k])


MOE_DEV_TIMEOUT = 1
MOE_DEV_BAD_OFFSETS = 4


def test_bounded_wait_runs_out_and_reports_its_site():
    """A wait on an mbarrier that nothing arrives on, with a 50 us limit,
    ends with MOE_DEV_TIMEOUT and its site in the status words; the second
    wait (default 2 s limit) stops on the abort flag, so the kernel ends far
    sooner than 2 s, and the context stays usable for the next call."""
    import time
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    api.moe_workspace_init(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    api.moe_selftest_wait_timeout(ws, 50_000, 777)
    bits, site = api.moe_get_device_status(ws)
    elapsed = time.perf_counter() - t0
    assert bits == MOE_DEV_TIMEOUT
    assert site == 777
    assert elapsed < 1.0, elapsed
    # the context is still usable: a clean workspace reports nothing
    api.moe_workspace_init(ws)
    assert api.moe_get_device_status(ws) == (0, 0)
    test_out_of_range_expert_index_is_reported_and_skipped()


def test_offsets_inconsistent_with_indices_are_reported_and_skipped():
    """Offsets that give expert 0 three rows too many and expert 1 three too
    few: the copies of expert 1 that would land past offsets[2] get no row
    (row_of_copy = -1) and MOE_DEV_BAD_OFFSETS is raised; every other copy is
    permuted as usual.  All positions written stay inside [0, R)."""
    cfg = CONFIGS["tiny"]
    n, e, k, d = cfg.n_tok, cfg.n_exp, cfg.top_k, cfg.d_model
    p = make_layer(cfg, "cpu")
    x = p["x"]
    lg = O.gate_logits(x.float().numpy(), p["w_gate"].float().numpy())
    idx, _ = O.route(lg, None, k, cfg.gate)
    idx = idx.astype(np.int32)
    counts = O.histogram(idx, e)
    assert counts[1] >= 3
    good_off = O.exclusive_offsets(counts)
    off = good_off.copy()
    off[1] += 3                                  # expert 1 now starts 3 rows later
    desc = api.make_desc(cfg)
    f, _ = api.moe_workspace_size(desc)
    ws = torch.empty(f, dtype=torch.uint8, device="cuda")
    api.moe_workspace_init(ws)
    r = n * k
    roc = torch.full((r,), 12345, dtype=torch.int32, device="cuda")
    cor = torch.full((r,), -7, dtype=torch.int32, device="cuda")
    xp = torch.zeros(r, d, dtype=torch.bfloat16, device="cuda")
    api.moe_permute(desc, x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(off).cuda(), roc, cor, xp, ws)
    bits, _ = api.moe_get_device_status(ws)
    assert bits & MOE_DEV_BAD_OFFSETS
    ref_roc, _ = O.permutation(idx, e)
    got = roc.cpu().numpy()
    flat = idx.reshape(-1)
    # expert 1's copies: the first count-3 land 3 rows later, the last 3 are dropped
    c1 = np.nonzero(flat == 1)[0]
    assert np.array_equal(got[c1[:-3]], ref_roc[c1[:-3]] + 3)
    assert (got[c1[-3:]] == -1).all()
    others = flat != 1
    assert np.array_equal(got[others], ref_roc[others])
