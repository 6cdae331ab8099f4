"""The DFlash-style KV injection (pe_inject_kv) on the GPU against the oracle, through the C ABI.

Every cache entry at an injected slot (an accepted or bonus position of the previous verify
batch) holds the oracle's post-RoPE k / v of the projected verifier state, to the storage
tolerance of the cache; every other entry is bit-identical to its value before the call.
"""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_step_gb300 as pe
from pe_workload import Config, config, f32_to_bf16, make_round
from pe_workload.device import to_torch

from gpu_harness import KV_TOL, setup, to_np_storage

pytestmark = pytest.mark.gpu


def _small(**kw) -> Config:
    base = dict(name="inject", B=3, K=4, n_layers=1, d=256, n_q=8, n_kv=2, head_dim=64, ffn=384, vocab=1000,
                dtype="bf16", prefix="uniform", prefix_args=(1, 300), accepted="uniform", seed=41)
    base.update(kw)
    return Config(**base)


CASES = {
    "bf16-hd64": (_small(), None),
    "bf16-hd128-L2": (_small(B=2, K=8, n_q=16, n_kv=2, head_dim=128, d=512, n_layers=2, seed=42), None),
    "bf16-all-rejected": (_small(B=4, K=5, seed=43), 0),
    "bf16-all-accepted": (_small(B=4, K=5, seed=44), "K"),
    "f32-c0": (config(0), None),
    # the Qwen3-Coder-30B-shaped drafter at B = 8: a split-K projection over 2048 features
    "bf16-qwen3-coder-30b-B8-K7": (config(1), None),
    # many rows: the projection and the k | v GEMM run on CTA pairs
    "bf16-pairs": (_small(B=40, K=8, d=320, ffn=448, seed=45), None),
}


@pytest.mark.parametrize("name", list(CASES))
def test_inject_kv_against_oracle(name):
    cfg_np, acc = CASES[name]
    rnd = make_round(cfg_np)
    if acc is not None:
        rnd.num_accepted[:] = cfg_np.K if acc == "K" else acc
    c = setup(cfg_np, rnd=rnd)
    rng = np.random.default_rng(7)
    w32 = (rng.standard_normal((cfg_np.d, cfg_np.d)) * 0.02).astype(np.float32)
    w_inj = f32_to_bf16(w32) if cfg_np.dtype == "bf16" else w32
    ws = pe.alloc_workspace(c.cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    R = c.Rd
    pe.inject_kv(c.cfg, c.weights, to_torch(w_inj), c.kv, R["block_table"], R["prev_pos"], R["num_accepted"],
                 R["target_hidden"], ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.inject_kv(cfg_np, c.w_np, w_inj, rnd.target_hidden, rnd.prev_pos, rnd.num_accepted,
                           rnd.block_table)
    assert len(ref["slots"]) == int((rnd.num_accepted + 1).sum())
    kvd = cfg_np.n_kv * cfg_np.head_dim
    slots = ref["slots"]
    for l in range(cfg_np.n_layers):
        for nm, dev, before, want in (("k", c.kv.k_cache[l], c.k_before[l], ref["new_k"][l]),
                                      ("v", c.kv.v_cache[l], c.v_before[l], ref["new_v"][l])):
            a_bits = to_np_storage(dev).reshape(-1, kvd)
            b_bits = to_np_storage(before).reshape(-1, kvd)
            got = oracle.widen(a_bits[slots])
            diff = np.abs(got - want) / np.maximum(1.0, np.abs(want))
            assert diff.max() <= KV_TOL[cfg_np.dtype], f"{nm} cache layer {l}: rel diff {diff.max():.3g}"
            untouched = np.ones(a_bits.shape[0], dtype=bool)
            untouched[slots] = False
            assert np.array_equal(a_bits[untouched], b_bits[untouched]), f"{nm} cache layer {l}: stray write"


def test_inject_kv_device_check_bad_accepted_count():
    """An accepted count above K is flagged on the device and nothing of that sequence is
    written; the other sequences are injected as usual."""
    cfg_np = _small(seed=46)
    rnd = make_round(cfg_np)
    rnd.num_accepted[1] = cfg_np.K + 2
    c = setup(cfg_np, rnd=rnd)
    w_inj = f32_to_bf16((np.random.default_rng(8).standard_normal((cfg_np.d, cfg_np.d)) * 0.02).astype(np.float32))
    ws = pe.alloc_workspace(c.cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    R = c.Rd
    pe.inject_kv(c.cfg, c.weights, to_torch(w_inj), c.kv, R["block_table"], R["prev_pos"], R["num_accepted"],
                 R["target_hidden"], ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == pe.PE_DEV_BAD_ACCEPTED
    kvd = cfg_np.n_kv * cfg_np.head_dim
    bad = rnd.block_table[1]
    pages = bad[bad >= 0]
    a_bits = to_np_storage(c.kv.k_cache[0]).reshape(rnd.num_pages, -1)
    b_bits = to_np_storage(c.k_before[0]).reshape(rnd.num_pages, -1)
    assert np.array_equal(a_bits[pages], b_bits[pages])
    assert kvd > 0
