"""Host-side logic of the benchmark: the round's algorithmic cost model (the roofline
denominators), the whole-job rate and the recorded-traffic lookup.  No GPU."""

import dataclasses
import json
import os

import numpy as np

import bench
from pe_workload import Config, config, make_round


def _tiny():
    return Config(name="cost-tiny", B=2, K=2, n_layers=1, d=8, n_q=2, n_kv=1, head_dim=4, ffn=16, vocab=10,
                  dtype="bf16", prefix="fixed", prefix_args=(5,), accepted="fixed", accepted_args=(1,), seed=0)


def test_round_cost_tiny_by_hand():
    """B = 2 sequences, K = 2, a = 1 each, prefix 5, d = 8, two q heads and one kv head of
    width 4, ffn 16, vocabulary 10, bf16.  Every count written out term by term."""
    cfg = _tiny()
    rnd = make_round(cfg, with_cache=False)
    rnd = dataclasses.replace(rnd, num_accepted=np.array([1, 1], np.int32), prefix_len=np.array([5, 5], np.int32))
    c = bench.round_cost(cfg, rnd)
    n_valid = 2 * (1 + 2)                    # a + K rows per sequence
    assert c["n_valid"] == n_valid
    qkv = (2 + 2 * 1) * 4 * 8                # (n_q + 2 n_kv) hd x d
    o = 8 * 2 * 4
    mlp = 2 * 16 * 8 + 8 * 16
    layer = qkv + o + mlp
    weights = (8 * 16 + layer + 2 * 8 + 8 + 10 * 8) * 2   # fc, layer, its two gains, final gain, LM head
    assert c["weights_bytes"] == weights
    kv_read = 1 * 2 * (5 + 3) * 1 * 4 * 2 * 2  # layers x seqs x (prefix + rows) x n_kv x hd x (K and V) x 2 B
    kv_write = n_valid * 1 * 4 * 2 * 2
    rows = n_valid * 8 * 2 * 2
    meta = 2 * 3 * 4 * 4 + 2 * 4 * 32
    assert c["kv_read_bytes"] == kv_read
    assert c["bytes"] == weights + kv_read + kv_write + rows + meta
    assert c["lm_bytes"] == 10 * 8 * 2
    # positions 5, 6, 7 per sequence: causal ranges 6, 7, 8
    ctx = 2 * (6 + 7 + 8)
    flops = 2 * n_valid * (8 * 16 + layer) + 2 * 2 * 2 * 10 * 8 + 4 * 2 * 4 * ctx
    assert c["flops"] == flops and c["lm_flops"] == 2 * 2 * 2 * 10 * 8 and c["attn_flops"] == 4 * 2 * 4 * ctx


def test_round_cost_single_sequence_workload():
    """The GPT-OSS-20B-shaped drafter at B = 1: LM head 201088 x 2880 bf16 (1158.3 MB), all
    weights once (1377.3 MB: fc 2880 x 5760, QKV 5120 x 2880, o 2880 x 4096, gate/up
    15360 x 2880, down 2880 x 7680, three gains, the LM head), the 3891-position prefix of
    eight kv heads of width 64 read once."""
    cfg = config(2)
    rnd = make_round(cfg, with_cache=False)
    c = bench.round_cost(cfg, rnd)
    assert c["lm_bytes"] == 201088 * 2880 * 2
    mats = 2880 * 5760 + 5120 * 2880 + 2880 * 4096 + 15360 * 2880 + 2880 * 7680
    assert c["weights_bytes"] == (mats + 3 * 2880 + 201088 * 2880) * 2
    rows = int(rnd.num_accepted[0]) + 7
    assert c["kv_read_bytes"] == (3891 + rows) * 8 * 64 * 2 * 2
    assert 1.38e9 < c["bytes"] < 1.39e9


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(1, 8, 7, 0.2) == 8 * 7 / 0.2e-3
    assert bench.whole_job_rate(4, 8, 7, 0.2) == 4 * bench.whole_job_rate(1, 8, 7, 0.2)


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    """A recorded capture is reported only while the kernel source still has the hash it was
    taken with; unknown workloads and kernels report none."""
    root = tmp_path
    (root / "profiles").mkdir()
    (root / "k.cu").write_text("kernel v1\n")
    import hashlib
    sha = hashlib.sha256(b"kernel v1\n").hexdigest()
    rec = {"lm_head_argmax": {"w": {"source": "k.cu", "source_sha256": sha, "dram_bytes_per_launch": 123}}}
    (root / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.recorded_traffic("lm_head_argmax", "w") == 123
    assert bench.recorded_traffic("lm_head_argmax", "other") is None
    assert bench.recorded_traffic("attention", "w") is None
    (root / "k.cu").write_text("kernel v2\n")
    assert bench.recorded_traffic("lm_head_argmax", "w") is None


def test_stage_names_match_trace_points():
    """One name per stage: pe_step's first launch spans trace points 0..3, every later stage one
    interval between consecutive points, the last ending at the final point (8 + 7 L points)."""
    for L in (1, 2, 4):
        pts = bench.stage_points(L)
        assert len(bench.stage_names(L)) == len(pts)
        assert pts[0] == (0, 3) and pts[-1][1] == 8 + 7 * L - 1
        assert all(a[1] == b[0] for a, b in zip(pts, pts[1:]))


def test_stage_costs_split_the_round_cost():
    """The per-stage bytes and flops add up to the round's (verification's few bytes of drafts
    and target tokens aside), on every workload and for two layers."""
    for cfg in [config(i) for i in range(4)] + [_tiny()]:
        rnd = make_round(cfg, with_cache=False)
        for L in sorted({cfg.n_layers, 2}):
            c = dataclasses.replace(cfg, n_layers=L)
            st = bench.stage_costs(c, rnd)
            assert list(st) == bench.stage_names(L)
            total = bench.round_cost(c, rnd)
            b = sum(v[0] for k, v in st.items() if k != "verify")
            f = sum(v[1] for v in st.values())
            assert b == total["bytes"], (cfg.name, L)
            assert f == total["flops"], (cfg.name, L)


def test_both_arms_describe_the_workload_identically():
    """The reference arm and the GPU arm print the same config object for one workload."""
    cfg = _tiny()
    rnd = make_round(cfg)
    a, b = bench.config_dict(cfg, rnd, 1), bench.config_dict(cfg, make_round(cfg), 1)
    assert a == b and a["workload"] == cfg.name and a["n_valid_rows"] == int(rnd.num_accepted.sum()) + cfg.B * cfg.K
