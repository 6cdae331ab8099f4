"""Pins of the CPU oracle to facts fixed by the P-EAGLE pages and by mathematics.

Nothing here uses the CUDA path.  Each test names the passage or the closed form
it checks.  A plausible slip in the oracle (a dropped term, a wrong sign or index,
a transposed operand, an off-by-one causal bound, a wrong GQA head mapping)
fails at least one of them.
"""

import itertools
import math
import os

import numpy as np
import pytest

import oracle
from pe_workload import Config, config, make_round, make_weights, f32_to_bf16, bf16_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tiny(**kw) -> Config:
    base = dict(name="pin", B=2, K=3, n_layers=1, d=64, n_q=4, n_kv=2, head_dim=16, ffn=96, vocab=101,
                dtype="f32", prefix="uniform", prefix_args=(5, 40), accepted="uniform", seed=11)
    base.update(kw)
    return Config(**base)


# ----------------------------------------------------------------------------- R1: batch rebuild

def _read_r1_golden(path):
    rows, extra = [], {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        parts = line.split()
        if parts[0].isdigit():
            rows.append([int(p) for p in parts])
        else:
            extra[parts[0]] = [int(p) for p in parts[1:]]
    return np.array(rows), extra


def test_r1_hand_written_table():
    """The pages' batch rebuild on one sequence (K=4, a=2), checked field by field."""
    table, extra = _read_r1_golden(os.path.join(GOLDEN, "r1_B1_K4_a2.txt"))
    prev_tokens = np.array([[10, 11, 12, 13, 14]])
    prev_pos = np.array([[128, 129, 130, 131, 132]])
    bt = np.array([[0, 1, 2, 3, 4, 5, 6, 7, 9, 8]])
    m = oracle.prepare_batch(4, 4096, prev_tokens, prev_pos, [2], [99], bt)
    assert (m["input_ids"] == table[:, 1]).all()
    assert (m["positions"] == table[:, 2]).all()
    assert (m["slot_mapping"] == table[:, 3]).all()
    assert (m["is_rejected"] == table[:, 4]).all()
    assert (m["is_mask"] == table[:, 5]).all()
    assert (m["hidden_map"] == table[:, 6]).all()
    assert list(m["row_list"]) == extra["row_list"]
    assert m["n_valid"] == extra["n_valid"][0]
    assert list(m["draft_rows"]) == extra["draft_rows"]


def test_r1_k1_has_no_mask_rows():
    """K=1: only the NTP row exists (no MASK slot), so single-step EAGLE drafting remains."""
    for a in (0, 1):
        m = oracle.prepare_batch(1, 50, [[3, 4]], [[7, 8]], [a], [9], [[0]])
        assert m["is_mask"].sum() == 0
        assert m["n_valid"] == a + 1
        ntp = a  # row a is the NTP row
        assert m["input_ids"][ntp] == 9 and m["positions"][ntp] == 7 + a
        assert list(m["draft_rows"]) == [a]


@pytest.mark.parametrize("K", range(1, 9))
def test_r1_invariants_every_a(K):
    """For every accepted count a in 0..K: a+K valid rows; slot -1 exactly on rejected rows;
    valid slots distinct; MASK positions contiguous after the NTP position; the MASK id on MASK
    rows only; the hidden map follows the shift-by-one rule; K drafts per sequence."""
    B, V, P = 3, 1000, 37
    rng = np.random.default_rng(K)
    for a in range(K + 1):
        prev_tokens = rng.integers(0, V, size=(B, K + 1))
        prev_pos = P + np.arange(K + 1)[None, :].repeat(B, 0) + 100 * np.arange(B)[:, None]
        nacc = np.full(B, a)
        bonus = rng.integers(0, V, size=B)
        npages = (prev_pos[:, 0].max() + 2 * K) // 16 + 1
        bt = rng.permutation(B * npages).reshape(B, npages)
        m = oracle.prepare_batch(K, V, prev_tokens, prev_pos, nacc, bonus, bt)
        S = 2 * K
        assert m["n_valid"] == B * (a + K)
        assert ((m["slot_mapping"] == -1) == (m["is_rejected"] == 1)).all()
        valid_slots = m["slot_mapping"][m["row_list"]]
        assert len(set(valid_slots.tolist())) == len(valid_slots)
        assert ((m["input_ids"] == V) == (m["is_mask"] == 1)).all()
        assert (m["hidden_map"][m["is_mask"] == 1] == -1).all()
        for b in range(B):
            rows = np.arange(b * S, (b + 1) * S)
            pos = m["positions"][rows]
            ntp_pos = prev_pos[b][a]
            assert list(pos[K + 1:]) == [ntp_pos + j for j in range(1, K)]
            for r in range(a):                  # token at p+1 with the hidden state at p
                assert m["input_ids"][rows[r]] == prev_tokens[b][r + 1]
                assert m["hidden_map"][rows[r]] == b * (K + 1) + r
                assert pos[r] == prev_pos[b][r]
            assert m["input_ids"][rows[a]] == bonus[b]
            # valid positions of a sequence: P..P+a+K-1, each once
            vpos = sorted(pos[m["is_rejected"][rows] == 0].tolist())
            assert vpos == list(range(prev_pos[b][0], prev_pos[b][0] + a + K))
        assert len(m["draft_rows"]) == B * K
        assert (np.diff(m["row_list"]) > 0).all()


def test_r1_rejected_positions_overlap_mask_positions():
    """The rejected rows' copied positions P+a+1..P+K coincide with MASK positions; slot -1 is
    what keeps them from writing over the MASK rows' cache entries."""
    K, a = 5, 1
    m = oracle.prepare_batch(K, 10, [[1] * (K + 1)], [[20 + j for j in range(K + 1)]], [a], [2], [[0, 1, 2]])
    rej = set(m["positions"][m["is_rejected"] == 1].tolist())
    mask = set(m["positions"][m["is_mask"] == 1].tolist())
    assert rej <= mask | {20 + K}
    assert (m["slot_mapping"][m["is_rejected"] == 1] == -1).all()


# ----------------------------------------------------------------------------- R2: input rows

def test_r2_rows_and_mask_identity():
    """NTP row = emb(new) with h_context; MASK rows = emb(mask) with h_shared -- bit-identical
    across every sequence; context rows = emb(token at p+1) with h(p)."""
    cfg = _tiny(B=3, K=4, dtype="bf16")
    w = make_weights(cfg)
    rnd = make_round(cfg, with_cache=False)
    m = oracle.prepare_batch(cfg.K, cfg.vocab, rnd.prev_tokens, rnd.prev_pos, rnd.num_accepted, rnd.bonus,
                             rnd.block_table)
    x0 = oracle.scatter_hidden(w.emb, w.h_shared, rnd.target_hidden, m["input_ids"], m["is_mask"], m["hidden_map"])
    d = cfg.d
    mask_rows = np.nonzero(m["is_mask"])[0]
    assert len(mask_rows) == cfg.B * (cfg.K - 1)
    for r in mask_rows:
        assert (x0[r] == x0[mask_rows[0]]).all()
        assert (x0[r, :d] == w.emb[cfg.vocab]).all() and (x0[r, d:] == w.h_shared).all()
    S = 2 * cfg.K
    for b in range(cfg.B):
        a = int(rnd.num_accepted[b])
        ntp = b * S + a
        assert (x0[ntp, :d] == w.emb[rnd.bonus[b]]).all()
        assert (x0[ntp, d:] == rnd.target_hidden[b * (cfg.K + 1) + a]).all()
        for r in range(a):
            assert (x0[b * S + r, :d] == w.emb[rnd.prev_tokens[b][r + 1]]).all()
            assert (x0[b * S + r, d:] == rnd.target_hidden[b * (cfg.K + 1) + r]).all()


# ----------------------------------------------------------------------------- R3: single ops

def test_widen_and_bf16_rounding():
    assert oracle.widen(np.array([0x3F80, 0xC000, 0x0000], np.uint16)).tolist() == [1.0, -2.0, 0.0]
    # round to nearest even at the 8th fraction bit
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -9], np.float32)
    assert bf16_to_f32(f32_to_bf16(x)).tolist() == [1.0, 1.0 + 2 ** -6, -1.0]


def test_linear_matches_blas():
    """Y = X W^T (nn.Linear, no bias) against numpy's BLAS product, for both storages."""
    rng = np.random.default_rng(0)
    X = rng.standard_normal((7, 33))
    W32 = rng.standard_normal((19, 33)).astype(np.float32)
    np.testing.assert_allclose(oracle.linear(X, W32), X @ W32.astype(np.float64).T, rtol=1e-12, atol=1e-12)
    Wb = f32_to_bf16(W32)
    np.testing.assert_allclose(oracle.linear(X, Wb), X @ bf16_to_f32(Wb).astype(np.float64).T, rtol=1e-12, atol=1e-12)
    # orientation: a one-hot input picks a column of W
    e = np.zeros((1, 33)); e[0, 5] = 1.0
    assert np.array_equal(oracle.linear(e, W32)[0], W32[:, 5].astype(np.float64))


def test_rmsnorm_closed_form():
    g = np.ones(2, np.float32)
    y = oracle.rmsnorm(np.array([3.0, 4.0]), g, 0.0)[0]
    np.testing.assert_allclose(y, np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15)
    y = oracle.rmsnorm(np.array([3.0, 4.0]), np.array([2.0, 0.5], np.float32), 0.5)[0]
    np.testing.assert_allclose(y, np.array([6.0, 2.0]) / math.sqrt(13.0), rtol=1e-15)
    # zero row: eps keeps it finite and zero
    assert (oracle.rmsnorm(np.zeros(4), np.ones(4, np.float32), 1e-6) == 0).all()
    # unit gains: the output has root-mean-square 1 (eps = 0)
    x = np.random.default_rng(1).standard_normal(100) * 7
    y = oracle.rmsnorm(x, np.ones(100, np.float32), 0.0)[0]
    assert abs(math.sqrt((y ** 2).mean()) - 1.0) < 1e-14


def test_rope_rotate_half():
    """Rotate-half RoPE: pair (i, i+hd/2), angle p * theta^(-2i/hd)."""
    hd = 8
    e0 = np.zeros(hd); e0[0] = 1.0
    v = oracle.rope(e0, 1, 10000.0)
    expect = np.zeros(hd); expect[0] = math.cos(1.0); expect[hd // 2] = math.sin(1.0)
    np.testing.assert_allclose(v, expect, atol=1e-15)
    # second-half unit vector rotates the other way: (x1, x2) = (0, 1) -> (-sin, cos)
    e4 = np.zeros(hd); e4[hd // 2 + 1] = 1.0
    ang = 3 * 10000.0 ** (-2.0 / hd)
    v = oracle.rope(e4, 3, 10000.0)
    assert abs(v[1] + math.sin(ang)) < 1e-15 and abs(v[hd // 2 + 1] - math.cos(ang)) < 1e-15
    # position 0 is the identity; rotations preserve length; scores depend on p - p' only
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    assert np.array_equal(oracle.rope(q, 0, 10000.0), q)
    assert abs(np.linalg.norm(oracle.rope(q, 1234, 10000.0)) - np.linalg.norm(q)) < 1e-12
    s1 = oracle.rope(q, 50, 100.0) @ oracle.rope(k, 20, 100.0)
    s2 = oracle.rope(q, 530, 100.0) @ oracle.rope(k, 500, 100.0)
    assert abs(s1 - s2) < 1e-10


def test_silu_closed_form():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12 and abs(oracle.silu(-40.0)) < 1e-15


def test_attend_closed_forms():
    rng = np.random.default_rng(3)
    hd = 4
    q = rng.standard_normal(hd)
    K1, V1 = rng.standard_normal((1, hd)), rng.standard_normal((1, hd))
    # a single position: the output is its value row
    np.testing.assert_allclose(oracle.attend(q, K1, V1, 0.5), V1[0], rtol=1e-15)
    # scores 0 and ln 3 -> weights 1/4, 3/4 (scale applied to q.k)
    q = np.array([1.0, 0, 0, 0])
    K2 = np.array([[0.0, 0, 0, 0], [2 * math.log(3.0), 0, 0, 0]])
    V2 = np.array([[4.0, 0, 0, 0], [8.0, 0, 0, 0]])
    np.testing.assert_allclose(oracle.attend(q, K2, V2, 0.5), [7.0, 0, 0, 0], rtol=1e-14)


# ----------------------------------------------------------------------------- R3: whole pass

def _structured_forward(position_list, group_map_check=True):
    """fc = 0 -> x = 0 -> q = k = 0 (uniform attention); rows write nothing (slot -1), so each
    head averages the cache's values over positions 0..p.  Cache value of kv head g at position t
    is (+t if g == 0 else -t); W_o copies element 0 of q-head h into feature h; the MLP adds 0."""
    cfg = _tiny(B=1, K=2, n_q=4, n_kv=2, head_dim=8, d=16, ffn=8, vocab=5)
    d, hd = cfg.d, cfg.head_dim
    z = lambda *s: np.zeros(s, np.float32)
    wo = z(d, cfg.n_q * hd)
    for h in range(cfg.n_q):
        wo[h, h * hd] = 1.0
    w = type("W", (), {})()
    w.fc, w.norm_final, w.lm_head = z(d, 2 * d), np.ones(d, np.float32), z(cfg.vocab, d)
    w.norm_attn, w.norm_mlp = [np.ones(d, np.float32)], [np.ones(d, np.float32)]
    w.wqkv, w.wo = [z(cfg.qkv_out, d)], [wo]
    w.w_gate_up, w.w_down = [z(2 * cfg.ffn, d)], [z(d, cfg.ffn)]
    npos = max(position_list) + 1
    pages = (npos + 15) // 16
    bt = np.arange(pages, dtype=np.int32)[None, :]
    kc = z(pages, 16, cfg.n_kv, hd)
    vc = z(pages, 16, cfg.n_kv, hd)
    for t in range(pages * 16):
        vc[t // 16, t % 16, 0, :] = t
        vc[t // 16, t % 16, 1, :] = -t
    n = len(position_list)
    res = oracle.draft_forward(cfg, w, np.zeros((n, 2 * d)), position_list, [-1] * n, [0] * n, bt, [kc], [vc],
                               [0], want_x=True)
    return res["x"]


def test_forward_gqa_mapping_and_causal_bound():
    """q head h reads kv head h // (n_q/n_kv); a row at position p attends to positions 0..p."""
    x = _structured_forward([0, 5, 30])
    for r, p in enumerate([0, 5, 30]):
        mean = p / 2.0                          # mean of 0..p inclusive
        np.testing.assert_allclose(x[r, :4], [mean, mean, -mean, -mean], rtol=1e-14, atol=1e-14)
        assert (x[r, 4:] == 0).all()


def closed_form_pass_checks() -> dict:
    """One row through the whole drafter pass with weights chosen so that every step has a
    closed form (the drafter of "N transformer layers and an LM head", P-EAGLE: Parallel
    Speculative Decoding in vLLM, step 2 "Parallel Drafting"; the layer is fc 2d -> d, then
    pre-norm GQA attention with rotate-half RoPE over the paged cache, a pre-norm SwiGLU MLP,
    a final norm and the LM head).  Returns check name -> (got, want) in float64.

    d = 32, one q head and one kv head of hd = 8, F = 4, vocab = d, RoPE base 10^4 (pair i
    turns by p * 10^(-i/2) radians: 1 rad per position for i = 0, 0.1 rad for i = 1).
    The row sits at position p = 1 of a sequence whose cache holds position 0.

    * fc = [I | 0] and X0 = [s e0 ; 0]: x = s e0; the attention RMSNorm (gains 1) gives
      y1 = r e0 with r = s / sqrt(s^2 / d + eps).
    * W_qkv reads y1[0] into q = alpha r e0 (q block), k = beta r e1 (k block), v = gamma r e0
      (v block): the three blocks in the order q | k | v.
    * k and q turn by their own position (k: pair 1 by 0.1 rad; q: pair 0 by 1 rad); v does
      not turn.
    * Scores: the cached key at position 0 is kappa e0, so s0 = alpha r kappa cos(1) / sqrt(hd);
      q and k lie in different rotation planes, so s1 = 0.  The output is
      w0 * mu e6 (cached value) + w1 * gamma r e0 (the row's own value, written before the
      attention reads the cache), w0 = 1 / (1 + exp(-s0)).
    * W_o copies the head output into x[8..15]; the MLP RMSNorm gives y2; W_gate row f reads
      a_f y2[0], W_up row f reads b_f y2[0]; u_f = silu(gate_f) * up_f; W_down copies u into
      x[16..19].
    * The final norm (gains 1) of x, then the LM head = I: the logits are that normalised x.
    """
    d, hd, F, eps, theta, p = 32, 8, 4, 1e-6, 10000.0, 1
    s, alpha, beta, gamma, kappa, mu = 3.0, 1.5, 0.75, 1.25, 2.0, 5.0  # exact in float32 storage
    a = np.array([1.0, -0.5, 2.0, 0.375])
    b = np.array([0.625, 1.5, -1.0, 2.5])
    cfg = _tiny(B=1, K=1, d=d, n_q=1, n_kv=1, head_dim=hd, ffn=F, vocab=d, rope_theta=theta)
    z = lambda *sh: np.zeros(sh, np.float32)
    fc = z(d, 2 * d)
    fc[np.arange(d), np.arange(d)] = 1.0
    wqkv = z(3 * hd, d)
    wqkv[0, 0], wqkv[hd + 1, 0], wqkv[2 * hd + 0, 0] = alpha, beta, gamma
    wo = z(d, hd)
    wo[8 + np.arange(hd), np.arange(hd)] = 1.0
    wgu = z(2 * F, d)
    wgu[np.arange(F), 0] = a
    wgu[F + np.arange(F), 0] = b
    wdown = z(d, F)
    wdown[16 + np.arange(F), np.arange(F)] = 1.0
    w = type("W", (), {})()
    w.fc, w.norm_final, w.lm_head = fc, np.ones(d, np.float32), np.eye(d, dtype=np.float32)
    w.norm_attn, w.norm_mlp, w.wqkv, w.wo = [np.ones(d, np.float32)], [np.ones(d, np.float32)], [wqkv], [wo]
    w.w_gate_up, w.w_down = [wgu], [wdown]
    kc = np.full((1, 16, 1, hd), 100.0, np.float32)   # every slot but position 0's: stale garbage
    vc = np.full((1, 16, 1, hd), -100.0, np.float32)
    kc[0, 0, 0, :] = 0.0
    kc[0, 0, 0, 0] = kappa
    vc[0, 0, 0, :] = 0.0
    vc[0, 0, 0, 6] = mu
    x0 = np.zeros((1, 2 * d))
    x0[0, 0] = s
    res = oracle.draft_forward(cfg, w, x0, [p], [p], [0], np.zeros((1, 1), np.int32), [kc], [vc], [0],
                               want_kv=True, want_x=True)
    r = s / math.sqrt(s * s / d + eps)
    k_want = np.zeros(hd)
    ang_k = p * theta ** (-2.0 * 1 / hd)
    k_want[1], k_want[1 + hd // 2] = beta * r * math.cos(ang_k), beta * r * math.sin(ang_k)
    v_want = np.zeros(hd)
    v_want[0] = gamma * r
    s0 = alpha * r * math.cos(p * 1.0) * kappa / math.sqrt(hd)
    w0 = 1.0 / (1.0 + math.exp(-s0))
    o = np.zeros(hd)
    o[6] = w0 * mu
    o[0] = (1.0 - w0) * gamma * r
    x1 = np.zeros(d)
    x1[0] = s
    x1[8:16] = o
    y2 = x1 / math.sqrt((x1 ** 2).mean() + eps)
    g, up = a * y2[0], b * y2[0]
    u = g / (1.0 + np.exp(-g)) * up
    x2 = x1.copy()
    x2[16:20] = u
    logits = x2 / math.sqrt((x2 ** 2).mean() + eps)
    return {"k_block_rope": (res["new_k"][0, 0], k_want), "v_block_unrotated": (res["new_v"][0, 0], v_want),
            "attention_q_rope": (res["x"][0, 8:16], o), "swiglu_roles": (res["x"][0, 16:20], u),
            "residual_stream": (res["x"][0], x2), "final_norm_lm_head": (res["logits"][0], logits)}


def closed_form_failures(checks: dict, rtol=1e-12) -> list:
    return [k for k, (got, want) in checks.items()
            if not np.allclose(got, want, rtol=rtol, atol=rtol * max(1.0, float(np.abs(want).max())))]


def test_forward_closed_form_every_step():
    """Every step of the drafter pass against its closed form (q | k | v order, RoPE of q and k
    at the row's own position, v not rotated, the row's write read by its own attention, the
    SwiGLU gate and up roles, the residual adds, the final norm and LM head).  A planted
    mistake in any of them fails this test (tests/test_oracle_mutants.py)."""
    assert closed_form_failures(closed_form_pass_checks()) == []


def _c0_like():
    return _tiny(B=3, K=4, n_layers=1, d=64, n_q=4, n_kv=2, head_dim=16, ffn=96, vocab=211)


def test_forward_rejected_rows_change_nothing():
    """Rows with slot -1 write no cache entry: running the pass over all padded rows (rejected ones
    included, with any input) gives bit-identical draft logits to running it over valid rows."""
    cfg = _c0_like()
    w, rnd = make_weights(cfg), make_round(cfg)
    res = oracle.run_round(cfg, w, rnd, n_threads=2)
    meta, x0 = res["meta"], res["x0"].copy()
    n_all = cfg.rows
    rows_all = np.arange(n_all)
    rej = np.nonzero(meta["is_rejected"])[0]
    assert len(rej) > 0
    x0[rej] = np.random.default_rng(9).standard_normal((len(rej), 2 * cfg.d)).astype(np.float32)
    pos, sl, sq = oracle.round_rows(cfg, meta, rows_all)
    dr_padded = meta["row_list"][meta["draft_rows"]]
    out = oracle.draft_forward(cfg, w, x0, pos, sl, sq, rnd.block_table, rnd.k_cache, rnd.v_cache, dr_padded)
    assert np.array_equal(out["logits"], res["logits"])


def test_forward_page_permutation_invariance():
    """The same logical cache under a different physical page assignment gives bit-identical logits."""
    cfg = _c0_like()
    w, rnd = make_weights(cfg), make_round(cfg)
    base = oracle.run_round(cfg, w, rnd, n_threads=2)["logits"]
    perm = np.random.default_rng(5).permutation(rnd.num_pages)    # physical page p moves to perm[p]
    kc = [np.empty_like(k) for k in rnd.k_cache]
    vc = [np.empty_like(v) for v in rnd.v_cache]
    for l in range(cfg.n_layers):
        kc[l][perm] = rnd.k_cache[l]
        vc[l][perm] = rnd.v_cache[l]
    bt = np.where(rnd.block_table >= 0, perm[np.maximum(rnd.block_table, 0)], -1).astype(np.int32)
    rnd.k_cache, rnd.v_cache, rnd.block_table = kc, vc, bt
    assert np.array_equal(oracle.run_round(cfg, w, rnd, n_threads=2)["logits"], base)


def test_forward_identity_layer_and_mask_rows():
    """With W_o = 0 and W_down = 0 a layer adds nothing, so logits equal the zero-layer pass
    lm(rms(fc(X0))); in that pass all MASK rows (identical inputs) give identical logits."""
    cfg = _c0_like()
    w, rnd = make_weights(cfg), make_round(cfg)
    w.wo = [np.zeros_like(x) for x in w.wo]
    w.w_down = [np.zeros_like(x) for x in w.w_down]
    one = oracle.run_round(cfg, w, rnd, n_threads=2)
    cfg0 = cfg.replace(n_layers=0)
    zero = oracle.run_round(cfg0, w, rnd, n_threads=2)
    assert np.array_equal(one["logits"], zero["logits"])
    lg = zero["logits"].reshape(cfg.B, cfg.K, -1)
    for b in range(cfg.B):
        for k in range(1, cfg.K):
            assert np.array_equal(lg[b, k], lg[0, 1])


def test_forward_sequences_independent():
    """Sequences share nothing but weights: a pass over one sequence alone equals its rows of the
    full-batch pass (bit-exact)."""
    cfg = _c0_like()
    w, rnd = make_weights(cfg), make_round(cfg)
    full = oracle.run_round(cfg, w, rnd, n_threads=2)["logits"].reshape(cfg.B, cfg.K, -1)
    for b in range(cfg.B):
        one = oracle.run_round(cfg, w, rnd, n_threads=1, seqs=[b])["logits"]
        assert np.array_equal(one, full[b])


def test_forward_k1_single_step():
    """K=1: the batch has no MASK rows; the single draft is the argmax of the NTP row's logits."""
    cfg = _c0_like().replace(K=1)
    w, rnd = make_weights(cfg), make_round(cfg)
    res = oracle.run_round(cfg, w, rnd, n_threads=2)
    assert res["meta"]["is_mask"].sum() == 0
    assert res["drafts"].shape == (cfg.B, 1)
    assert (res["drafts"][:, 0] == np.argmax(res["logits"], axis=1)).all()


def test_forward_block_causal():
    """Attention reads the cache after this round's writes and only up to the row's own position:
    dropping a sequence's MASK rows leaves its NTP row's logits bit-identical, while the last MASK
    row's logits depend on the NTP row's write (it sees the context rows, the NTP row and the
    MASK rows before it)."""
    cfg = _c0_like().replace(B=1)
    w, rnd = make_weights(cfg), make_round(cfg)
    res = oracle.run_round(cfg, w, rnd, n_threads=2)
    meta, x0 = res["meta"], res["x0"]
    rows = res["rows"]
    a = int(rnd.num_accepted[0])
    ntp = a                                           # compacted index of the NTP row
    no_mask = rows[: a + 1]                           # context rows + NTP row only
    pos, sl, sq = oracle.round_rows(cfg, meta, no_mask)
    out = oracle.draft_forward(cfg, w, x0[no_mask], pos, sl, sq, rnd.block_table, rnd.k_cache,
                               rnd.v_cache, [ntp])
    assert np.array_equal(out["logits"][0], res["logits"][0])
    # perturb the NTP row's input: every MASK row's logits move
    x0b = x0.copy()
    x0b[rows[ntp]] = x0[rows[0]] if a > 0 else x0[rows[-1]] * 0
    pos, sl, sq = oracle.round_rows(cfg, meta, rows)
    out = oracle.draft_forward(cfg, w, x0b[rows], pos, sl, sq, rnd.block_table, rnd.k_cache, rnd.v_cache,
                               meta["draft_rows"])
    for k in range(1, cfg.K):
        assert not np.array_equal(out["logits"][k], res["logits"][k])


# ----------------------------------------------------------------------------- R4: verify

@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_verify_brute_force(K):
    """All draft/target pairs over vocab {0,1,2}, packed 3 sequences per batch, against the
    longest-matching-prefix definition: a = max{j : draft[i] == target[i] for all i < j}."""
    drafts = list(itertools.product(range(3), repeat=K))
    targets = list(itertools.product(range(3), repeat=K + 1))
    pairs = [(d, t) for d in drafts for t in targets]
    for i in range(0, len(pairs), 3):
        chunk = pairs[i:i + 3]
        D = np.array([p[0] for p in chunk])
        T = np.array([p[1] for p in chunk])
        a, bonus = oracle.verify(D, T)
        for j, (d, t) in enumerate(chunk):
            best = max(jj for jj in range(K + 1) if all(d[x] == t[x] for x in range(jj)))
            assert a[j] == best and bonus[j] == t[best]


# ----------------------------------------------------------------------------- the next verify batch

def test_next_verify_batch_hand_example():
    """Sequence at P = 100 with K = 3: a = 2 accepted, so the NTP row sat at 102 and the
    bonus token belongs at 103; the drafts follow at 104..106.  a = 0: bonus at 101."""
    prev_pos = np.array([[100, 101, 102, 103], [40, 41, 42, 43]])
    drafts = np.array([[5, 6, 8], [9, 10, 11]])
    tok, pos = oracle.next_verify_batch(prev_pos, [2, 0], [7, 3], drafts)
    assert tok.tolist() == [[7, 5, 6, 8], [3, 9, 10, 11]]
    assert pos.tolist() == [[103, 104, 105, 106], [41, 42, 43, 44]]


@pytest.mark.parametrize("K", [1, 2, 5, 8])
def test_next_verify_batch_consistent_with_rebuild(K):
    """Against the rebuild's positions (a row at position p carries the token at p + 1 and
    predicts the one at p + 2): the bonus token, carried by the NTP row, lands one position
    after it; draft t_k, predicted by the k-th draft row, lands two positions after that row;
    and the next rebuild's copy slots continue without a gap."""
    rng = np.random.default_rng(K)
    B, V = 6, 50
    P = rng.integers(0, 200, size=B)
    prev_pos = P[:, None] + np.arange(K + 1)[None, :]
    prev_tokens = rng.integers(0, V, size=(B, K + 1))
    acc = np.array([b % (K + 1) for b in range(B)])
    bonus = rng.integers(0, V, size=B)
    bt = np.arange(B * 40).reshape(B, 40)
    meta = oracle.prepare_batch(K, V, prev_tokens, prev_pos, acc, bonus, bt)
    drafts = rng.integers(0, V, size=(B, K))
    tok, pos = oracle.next_verify_batch(prev_pos, acc, bonus, drafts)
    dr = meta["row_list"][meta["draft_rows"]].reshape(B, K)
    for b in range(B):
        ntp = dr[b][0]
        assert tok[b][0] == meta["input_ids"][ntp] == bonus[b]
        assert pos[b][0] == meta["positions"][ntp] + 1
        for k in range(K):
            assert tok[b][k + 1] == drafts[b][k]
            assert pos[b][k + 1] == meta["positions"][dr[b][k]] + 2
    # the next round: its accepted rows and NTP row sit at consecutive positions from pos[b][0]
    acc2 = np.array([(b * 3) % (K + 1) for b in range(B)])
    meta2 = oracle.prepare_batch(K, V, tok, pos, acc2, bonus, bt)
    for b in range(B):
        rows = [b * 2 * K + r for r in range(acc2[b] + 1)]
        assert [meta2["positions"][r] for r in rows] == list(range(pos[b][0], pos[b][0] + acc2[b] + 1))


# ----------------------------------------------------------------------------- R5: sampled drafting + verification

def test_inverse_cdf_hand_cases():
    """Weights [1, 2, 3, 4] (total 10): the draw changes index where u * 10 reaches the
    running sums 1, 3, 6 (a boundary itself goes to the next index); zero weights are
    skipped."""
    w = [1.0, 2.0, 3.0, 4.0]
    cases = {0.0: 0, 0.05: 0, 0.0999: 0, 0.1: 1, 0.29: 1, 0.3: 2, 0.59: 2, 0.6: 3, 0.999999: 3}
    for u, v in cases.items():
        assert oracle.inverse_cdf(w, u) == v, u
    assert [oracle.inverse_cdf([0, 0, 5, 0, 5, 0], u) for u in (0.0, 0.49, 0.5, 0.99)] == [2, 2, 4, 4]


@pytest.mark.parametrize("T", [1.0, 0.5, 2.0])
def test_sample_drafts_frequencies_and_normaliser(T):
    """Logits log(1), log(2), log(3): q is proportional to [1, 2, 3]^(1/T).  Uniforms on an
    even midpoint grid land on each token in proportion to its probability (exactly, up to
    one grid step), and lse is the log of the sum of exp(logits / T)."""
    lg = np.log(np.array([1.0, 2.0, 3.0]))
    q_closed = np.array([1.0, 2.0, 3.0]) ** (1 / T)
    q_closed /= q_closed.sum()
    N = 30000
    u = ((np.arange(N) + 0.5) / N).reshape(N, 1)
    drafts, lse = oracle.sample_drafts(np.tile(lg, (N, 1)), u, T)
    freq = np.bincount(drafts.reshape(-1), minlength=3) / N
    assert np.abs(freq - q_closed).max() <= 1.0 / N + 1e-12
    assert np.allclose(lse, math.log(np.sum(np.array([1.0, 2.0, 3.0]) ** (1 / T))), atol=1e-12)


def test_verify_sampled_closed_forms():
    """q == p: every draft is accepted (u * q < p for u < 1) and the bonus is drawn from
    p_K.  A one-hot target at token y: a draft equal to y is accepted, any other draft is
    rejected, and the residual max(0, p - q) is concentrated on y, so the bonus is y."""
    rng = np.random.default_rng(5)
    B, K, V = 6, 3, 7
    lg = rng.normal(0, 1.5, size=(B * K, V))
    q = np.array([oracle.drafter_distribution(r, 1.0)[0] for r in lg]).reshape(B, K, V)
    pK = rng.dirichlet(np.ones(V), size=B)
    P = np.concatenate([q, pK[:, None, :]], axis=1)
    drafts = rng.integers(0, V, size=(B, K))
    u_res = rng.random(B)
    a, bonus = oracle.verify_sampled(drafts, lg, 1.0, P, rng.random((B, K)) * 0.999999, u_res)
    assert (a == K).all()
    assert [int(x) for x in bonus] == [oracle.inverse_cdf(pK[b], u_res[b]) for b in range(B)]
    y = 4
    P1 = np.zeros((B, K + 1, V))
    P1[:, :, y] = 1.0
    drafts = np.full((B, K), y)
    drafts[:, 1] = [0, 1, 2, 3, 5, 6]  # the second draft is never y
    a, bonus = oracle.verify_sampled(drafts, lg, 1.0, P1, rng.random((B, K)), rng.random(B))
    assert (a == 1).all() and (bonus == y).all()


def test_verify_sampled_preserves_target_distribution():
    """The defining property of the scheme: whatever the drafter proposes, the token emitted
    at a position (the accepted draft, else the bonus) follows the target's distribution
    there.  Monte Carlo over 40000 sequences with V = 4, K = 2 and q far from p: the first
    emitted token follows p_0, and among sequences that accepted the first draft, the second
    follows p_1 (5-sigma bounds)."""
    rng = np.random.default_rng(11)
    B, K, V = 40000, 2, 4
    lg_rows = np.log(np.array([[0.55, 0.25, 0.15, 0.05], [0.1, 0.2, 0.3, 0.4]]))
    lg = np.tile(lg_rows, (B, 1))
    p = np.array([[0.1, 0.2, 0.3, 0.4], [0.4, 0.4, 0.1, 0.1], [0.25, 0.25, 0.25, 0.25]])
    P = np.broadcast_to(p, (B, K + 1, V))
    drafts, _ = oracle.sample_drafts(lg, rng.random((B, K)), 1.0)
    a, bonus = oracle.verify_sampled(drafts, lg, 1.0, P, rng.random((B, K)), rng.random(B))
    first = np.where(a >= 1, drafts[:, 0], bonus)
    f0 = np.bincount(first, minlength=V) / B
    assert np.abs(f0 - p[0]).max() <= 5 * np.sqrt(p[0] * (1 - p[0]) / B).max()
    sel = a >= 1
    second = np.where(a[sel] >= 2, drafts[sel, 1], bonus[sel])
    n = int(sel.sum())
    f1 = np.bincount(second, minlength=V) / n
    assert np.abs(f1 - p[1]).max() <= 5 * np.sqrt(p[1] * (1 - p[1]) / n).max()
    # acceptance rate of the first draft: sum_v min(p_0, q_0)
    assert abs(sel.mean() - np.minimum(p[0], np.exp(lg_rows[0])).sum()) <= 5 * 0.0025


# ----------------------------------------------------------------------------- R6: DFlash-style KV injection

def test_inject_kv_closed_form_and_rejected_positions():
    """The verifier's hidden state h of an accepted (or bonus) position goes through
    x = W_inj h, the attention RMSNorm, the k and v blocks of W_qkv, and RoPE on k at the
    position: with W_inj = I, h = s e0 and one-hot k / v rows the entries have closed forms
    (k pair 1 turned by 0.1 rad per position at RoPE base 10^4; v unrotated).  Positions after
    the accepted count are not written."""
    d, hd, s_, beta, gamma = 32, 8, 3.0, 0.75, 1.25
    cfg = _tiny(B=2, K=3, d=d, n_q=1, n_kv=1, head_dim=hd, ffn=8, vocab=d)
    wqkv = np.zeros((3 * hd, d), np.float32)
    wqkv[hd + 1, 0], wqkv[2 * hd, 0] = beta, gamma
    w = type("W", (), {})()
    w.norm_attn, w.wqkv = [np.ones(d, np.float32)], [wqkv]
    H = np.zeros((2 * (cfg.K + 1), d), np.float32)
    H[:, 0] = s_
    prev_pos = np.array([[10, 11, 12, 13], [40, 41, 42, 43]])
    bt = np.arange(2 * 4, dtype=np.int32).reshape(2, 4)
    res = oracle.inject_kv(cfg, w, np.eye(d, dtype=np.float32), H, prev_pos, [2, 0], bt)
    assert res["rows"].tolist() == [0, 1, 2, 4]          # (b=0, j=0..2), (b=1, j=0)
    assert res["slots"].tolist() == [16 * 0 + 10, 11, 12, 16 * 6 + 40 % 16]
    r = s_ / math.sqrt(s_ * s_ / d + cfg.rms_eps)
    for i, p in enumerate(res["positions"]):
        ang = p * 10000.0 ** (-2.0 / hd)
        k = np.zeros(hd)
        k[1], k[1 + hd // 2] = beta * r * math.cos(ang), beta * r * math.sin(ang)
        np.testing.assert_allclose(res["new_k"][0, i], k, rtol=1e-12, atol=1e-12)
        v = np.zeros(hd)
        v[0] = gamma * r
        np.testing.assert_allclose(res["new_v"][0, i], v, rtol=1e-12, atol=1e-12)


def test_inject_kv_matches_the_drafter_layer_on_projected_rows():
    """A drafter row whose fc output is W_inj h (fc = [0 | W_inj], so emb drops out) writes, in
    the first layer, exactly the k and v that injection writes for h at the same position."""
    cfg = _c0_like().replace(B=2, K=3, n_layers=2)
    w, rnd = make_weights(cfg), make_round(cfg)
    d = cfg.d
    rng = np.random.default_rng(4)
    w_inj = (rng.standard_normal((d, d)) * 0.05).astype(np.float32)
    inj = oracle.inject_kv(cfg, w, w_inj, rnd.target_hidden, rnd.prev_pos, rnd.num_accepted, rnd.block_table)
    w.fc = np.concatenate([np.zeros((d, d), np.float32), w_inj], axis=1)
    x0 = np.concatenate([np.zeros((len(inj["rows"]), d)), oracle.widen(rnd.target_hidden)[inj["rows"]]], axis=1)
    seqs = inj["rows"] // (cfg.K + 1)
    out = oracle.draft_forward(cfg, w, x0, inj["positions"], inj["slots"], seqs, rnd.block_table, rnd.k_cache,
                               rnd.v_cache, [0], want_kv=True)
    np.testing.assert_allclose(out["new_k"][0], inj["new_k"][0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out["new_v"][0], inj["new_v"][0], rtol=1e-10, atol=1e-12)
