"""moe_permute_noalloc, the permutation entry point for callers that cannot
give the library device memory (for example a plugin called with only its
input and output buffers, or a loop under a fixed memory budget where new
allocations are not allowed).  It keeps its chunk tables in a fixed array
inside the library instead of a caller workspace.  This file is collected
last so that a run stopping at its first failure has already run every other
test; it also passes on its own in a fresh process."""
import pytest
import torch

from ragged_grouped_gemm_gb300 import api
from ragged_grouped_gemm_gb300.inputs import CONFIGS, MoEConfig, make_layer, route_bias, skewed_logits

pytestmark = pytest.mark.gpu


def _routed(cfg, mode):
    """Routing of seeded logits through the library's own router."""
    n, e, k = cfg.n_tok, cfg.n_exp, cfg.top_k
    d = api.make_desc(cfg)
    _, b = api.moe_workspace_size(d)
    ws = torch.empty(b, dtype=torch.uint8, device="cuda")
    api.moe_workspace_init(ws)
    idx = torch.empty(n, k, dtype=torch.int32, device="cuda")
    w = torch.empty(n, k, dtype=torch.float32, device="cuda")
    cnt = torch.empty(e, dtype=torch.int32, device="cuda")
    off = torch.empty(e + 1, dtype=torch.int32, device="cuda")
    bias = route_bias(cfg)
    api.moe_route_from_logits(d, skewed_logits(n, e, mode).cuda(), None if bias is None else bias.cuda(),
                              idx, w, cnt, off, ws)
    return d, ws, idx, off


def test_noalloc_permute_matches_workspace_permute_on_two_calls_in_a_row():
    for name, mode in (("dsv3", "zipf"), ("small_fine", "half0")):
        cfg = CONFIGS[name]
        n, dm, k = cfg.n_tok, cfg.d_model, cfg.top_k
        r = n * k
        d, ws, idx, off = _routed(cfg, mode)
        x = make_layer(cfg.replace(d_ff=64, n_exp=1, top_k=1, use_bias=False, n_shared=0), "cpu")["x"].cuda()
        outs = []
        for fn in ("ws", "noalloc"):
            roc = torch.full((r,), -1, dtype=torch.int32, device="cuda")
            cor = torch.full((r,), -1, dtype=torch.int32, device="cuda")
            xp = torch.zeros(r, dm, dtype=torch.bfloat16, device="cuda")
            if fn == "ws":
                api.moe_permute(d, x, idx, off, roc, cor, xp, ws)
            else:
                api.moe_permute_noalloc(d, x, idx, off, roc, cor, xp)
            torch.cuda.synchronize()
            outs.append((roc.cpu(), cor.cpu(), xp.cpu().view(torch.int16)))
        # integer maps and copied rows: identical bit for bit
        for a, b in zip(*outs):
            assert torch.equal(a, b)


def _buffers(cfg):
    n, dm, k = cfg.n_tok, cfg.d_model, cfg.top_k
    r = n * k
    x = make_layer(cfg.replace(d_ff=64, n_exp=1, top_k=1, use_bias=False, n_shared=0), "cpu")["x"].cuda()
    roc = torch.full((r,), -1, dtype=torch.int32, device="cuda")
    cor = torch.full((r,), -1, dtype=torch.int32, device="cuda")
    xp = torch.zeros(r, dm, dtype=torch.bfloat16, device="cuda")
    return x, roc, cor, xp


# 1024 experts, top-2, 64-wide rows: ceil(n_tok / 128) * 1024 chunk-table
# entries, i.e. exactly the 65536 the built-in array holds at n_tok = 8192
LIMIT_CFG = MoEConfig("noalloc_limit", 8192, 64, 64, 1024, 2)


def test_noalloc_permute_at_its_largest_accepted_size():
    """ceil(8192/128) * 1024 = 65536 entries per chunk table, the most the
    array holds: the call runs and matches moe_permute bit for bit."""
    cfg = LIMIT_CFG
    d, ws, idx, off = _routed(cfg, "uniform")
    outs = []
    for fn in ("ws", "noalloc"):
        x, roc, cor, xp = _buffers(cfg)
        if fn == "ws":
            api.moe_permute(d, x, idx, off, roc, cor, xp, ws)
        else:
            api.moe_permute_noalloc(d, x, idx, off, roc, cor, xp)
        torch.cuda.synchronize()
        outs.append((roc.cpu(), cor.cpu(), xp.cpu().view(torch.int16)))
    assert api.moe_get_device_status(ws)[0] == 0
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_noalloc_permute_rejects_sizes_beyond_its_array():
    """One more token (65 chunks of 128 tokens * 1024 experts = 66560 entries
    per table) is beyond the array: MOE_ERR_WORKSPACE, returned before anything
    is enqueued.  The buffers are real and sized for the call, and the outputs
    are left as they were."""
    cfg = LIMIT_CFG.replace(n_tok=LIMIT_CFG.n_tok + 1)
    d, ws, idx, off = _routed(cfg, "uniform")
    x, roc, cor, xp = _buffers(cfg)
    with pytest.raises(api.MoEError) as err:
        api.moe_permute_noalloc(d, x, idx, off, roc, cor, xp)
    assert err.value.code == 3     # MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((roc == -1).all()) and bool((cor == -1).all())
