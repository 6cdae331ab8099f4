"""pe_draft_forward_noalloc: the drafter pass for callers that cannot allocate device memory.

Such callers (a plugin whose host framework owns every device allocation, a serving
loop that must never call cudaMalloc) cannot hand the library a workspace; this entry
point uses a fixed scratch array owned by the library instead.  Its results must match
the workspace-based pe_draft_forward, call after call, even though the array keeps the
previous call's contents.  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import speculative_decoding_step_gb300 as pe
from pe_workload import Config, config

from gpu_harness import LOGIT_TOL, run_stages, setup

pytestmark = pytest.mark.gpu

CASES = {
    "bf16-small": Config("noalloc-bf16", B=3, K=4, n_layers=1, d=256, n_q=8, n_kv=2, head_dim=64, ffn=384,
                         vocab=1000, dtype="bf16", prefix="uniform", prefix_args=(1, 300), accepted="uniform",
                         seed=21),
    "f32-tiny": config(0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_forward_twice(name):
    cfg_np = CASES[name]
    c = setup(cfg_np)
    assert pe.workspace_bytes(c.cfg) <= pe.NOALLOC_SCRATCH_BYTES
    assert run_stages(c) == 0                       # workspace path: reference results
    want_logits = c.rd.logits.clone()
    want_drafts = c.rd.draft_tokens.clone()
    tol = LOGIT_TOL[cfg_np.dtype]
    for _ in range(2):                              # two calls in a row share the scratch array
        for l in range(cfg_np.n_layers):            # same cache contents as the reference call saw
            c.kv.k_cache[l].copy_(c.k_before[l])
            c.kv.v_cache[l].copy_(c.v_before[l])
        drafts = torch.full_like(want_drafts, -1)
        logits = torch.full_like(want_logits, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pe.draft_forward_noalloc(c.cfg, c.weights, c.kv, c.Rd["block_table"], c.rd.x0, c.rd.meta, drafts, err,
                                 logits)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(drafts, want_drafts)
        diff = (logits - want_logits).abs().max().item()
        assert np.isfinite(diff) and diff <= tol


def test_noalloc_rejects_configs_beyond_its_scratch():
    cfg = pe.Config.make(64, 8, 2880, 64, 8, 64, 7680, 201088, 2, 1100, "bf16")
    assert pe.workspace_bytes(cfg) > pe.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    w = pe.DeviceWeights(dummy, dummy, dummy, [dummy, dummy], [dummy, dummy], [dummy, dummy], [dummy, dummy],
                         [dummy, dummy], [dummy, dummy], dummy, dummy)
    kv = pe.DeviceKV([dummy, dummy], [dummy, dummy])
    meta = {k: dummy for k in ("positions", "slot_mapping", "row_list", "n_valid", "draft_rows")}
    with pytest.raises(pe.PeError) as e:
        pe.draft_forward_noalloc(cfg, w, kv, dummy, dummy, meta, dummy, dummy)
    assert e.value.status == 2                      # PE_ERR_SHAPE, nothing launched
