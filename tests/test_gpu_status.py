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
