"""Failure detection on the GPU without faulting it: a bounded pipeline wait that runs out.

The test shortens the wait limit to 1 ms and has the next tensor-core GEMM launch (the fc
contraction of the drafter pass) leave one pipeline stage of its first CTA unarmed.  Its MMA
role's wait on that stage runs out: the kernel must record PE_DEV_TIMEOUT in the error word,
unwind (abort flag, copies and MMAs in flight waited for, tensor memory freed) and return,
and the stream must stay usable: the next round, with the default limit, passes parity.
"""

import time

import pytest
import torch

import speculative_decoding_step_gb300 as pe
from pe_workload import Config

from gpu_harness import check_kv_writes, check_logits, oracle_round, run_stages, setup

pytestmark = pytest.mark.gpu

CFG = Config("expiry-bf16", B=3, K=4, n_layers=1, d=256, n_q=8, n_kv=2, head_dim=64, ffn=384, vocab=1000,
             dtype="bf16", prefix="uniform", prefix_args=(1, 300), accepted="uniform", seed=31)


@pytest.mark.parametrize("stage", [0, 1])
def test_wait_expiry_unwinds_and_next_round_passes(stage):
    c = setup(CFG)
    assert run_stages(c) == 0                     # warm: every kernel has run once
    for l in range(CFG.n_layers):
        c.kv.k_cache[l].copy_(c.k_before[l])
        c.kv.v_cache[l].copy_(c.v_before[l])
    pe.set_wait_limit_ns(1_000_000)
    try:
        pe.skip_pipeline_stage_for_test(stage)
        t0 = time.perf_counter()
        err = run_stages(c)                       # synchronises: the kernels returned
        elapsed = time.perf_counter() - t0
    finally:
        pe.skip_pipeline_stage_for_test(-1)
        pe.set_wait_limit_ns(0)
    assert err == pe.PE_DEV_TIMEOUT
    assert elapsed < 1.0                          # a few waits of 1 ms, not the default second
    # the same stream, the next round, default limit: parity with the oracle
    for l in range(CFG.n_layers):
        c.kv.k_cache[l].copy_(c.k_before[l])
        c.kv.v_cache[l].copy_(c.v_before[l])
    c.rd.err.zero_()
    assert run_stages(c) == 0
    ref = oracle_round(c, want_kv=True)
    check_logits(c, ref)
    check_kv_writes(c, ref)
    torch.cuda.synchronize()
