"""Non-greedy drafting and rejection-sampling verification on the GPU against the oracle.

The draws are integers decided by floating point: the GPU sums the weights in fp32 in a
fixed blocked order, the oracle in fp64 in index order.  A draw therefore equals the
oracle's except where the uniform lies within the fp32 error of a cumulative-sum boundary;
there the GPU's token is checked to be a valid draw: the oracle's normalised cumulative
sums around it bracket the uniform to within that error.  Error bound for the sums: 16
sequential additions within a lane, 5 tree levels within a 512-entry step, about V/16384
steps per lane of the drawing warp and 32 lane totals, each addition off by at most 2^-24
of the running total, plus a few ulp per exponential (base 2, hardware approximation):
below 2e-5 of the total for V <= 2^18; the checks use 5e-5.
"""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_step_gb300 as pe
from pe_workload import Config

from gpu_harness import LOGIT_TOL, run_stages, setup

pytestmark = pytest.mark.gpu

CDF_EPS = 5e-5


def _cfg(B, K, V):
    return pe.Config.make(B, K, 64, 1, 1, 64, 64, V, 1, 1, "f32")


def _seeded(B, K, V, seed, scale=3.0):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0.0, scale, size=(B * K, V)).astype(np.float32)
    return rng, logits


def _in_band(w, x, u, eps):
    """x is a valid inverse-CDF draw of u from weights w, to within eps of the total."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    c = c / c[-1]
    lo = c[x - 1] if x > 0 else 0.0
    return w[x] > 0 and lo - eps <= u < c[x] + eps


def _gpu_sample(cfg, logits, u, T):
    B, K = u.shape
    lg = torch.from_numpy(logits).cuda()
    ud = torch.from_numpy(u.astype(np.float32)).cuda()
    drafts = torch.empty((B, K), dtype=torch.int32, device="cuda")
    lse = torch.empty(B * K, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pe.alloc_workspace(cfg)
    pe.sample_drafts(cfg, lg, ud, T, ws, drafts, lse, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return lg, drafts, lse


@pytest.mark.parametrize("B,K,V,T", [(16, 8, 1000, 1.0), (5, 3, 4099, 0.7), (8, 7, 151936, 1.0), (1, 7, 201088, 1.3)])
def test_sample_drafts_against_oracle(B, K, V, T):
    rng, logits = _seeded(B, K, V, seed=V + B)
    u = rng.random((B, K)).astype(np.float32).astype(np.float64)
    cfg = _cfg(B, K, V)
    _, drafts, lse = _gpu_sample(cfg, logits, u, T)
    g = drafts.cpu().numpy()
    want, want_lse = oracle.sample_drafts(logits, u, T)
    assert np.abs(lse.cpu().numpy().reshape(B, K) - want_lse).max() <= 1e-4 * max(1.0, np.abs(want_lse).max())
    mismatch = np.argwhere(g != want)
    assert len(mismatch) <= max(1, (B * K) // 10)
    for b, k in mismatch:
        q, _ = oracle.drafter_distribution(logits[b * K + k], T)
        assert _in_band(q, int(g[b, k]), u[b, k], CDF_EPS), (b, k)


def test_sample_drafts_frequencies():
    """Many rows of the same logits with uniforms on an even grid: the GPU's draws land on
    each token in proportion to its probability (up to one grid step and the sum error)."""
    V, N = 6, 4096
    lg_row = np.log(np.array([1.0, 2.0, 3.0, 0.5, 0.25, 4.0])).astype(np.float32)
    q = np.exp(lg_row.astype(np.float64))
    q /= q.sum()
    B, K = N // 8, 8
    u = ((np.arange(N) + 0.5) / N).reshape(B, K)
    _, drafts, _ = _gpu_sample(_cfg(B, K, V), np.tile(lg_row, (N, 1)), u, 1.0)
    freq = np.bincount(drafts.cpu().numpy().reshape(-1), minlength=V) / N
    assert np.abs(freq - q).max() <= 1.0 / N + CDF_EPS


@pytest.mark.parametrize("V", [2048, 4099])
def test_sample_drafts_masked_logits(V):
    """-inf logits are masked entries: probability 0, never drawn, no error.  Rows with a whole
    512-entry step masked, a partial step masked, all but three entries masked, and none."""
    B, K = 2, 2
    rng, logits = _seeded(B, K, V, seed=V)
    logits[0, 512:1024] = -np.inf                   # a whole step
    logits[1, 100:300] = -np.inf                    # part of a step
    keep = [7, 1500, V - 1]
    row2 = np.full(V, -np.inf, np.float32)
    row2[keep] = logits[2, keep]
    logits[2] = row2                                # every step but three entries masked
    u = rng.random((B, K)).astype(np.float32).astype(np.float64)
    _, drafts, lse = _gpu_sample(_cfg(B, K, V), logits, u, 1.0)
    g = drafts.cpu().numpy().reshape(-1)
    want, want_lse = oracle.sample_drafts(logits, u, 1.0)
    gl = lse.cpu().numpy()
    assert np.isfinite(gl).all()
    assert np.abs(gl - want_lse.reshape(-1)).max() <= 1e-4 * max(1.0, np.abs(want_lse).max())
    for r in range(B * K):
        assert np.isfinite(logits[r, g[r]]), r
        if g[r] != want.reshape(-1)[r]:
            q, _ = oracle.drafter_distribution(logits[r], 1.0)
            assert _in_band(q, int(g[r]), u.reshape(-1)[r], CDF_EPS), r
    assert g[2] in keep


@pytest.mark.parametrize("where", ["full-step-nan", "full-step-posinf", "last-step-nan", "none"])
def test_sample_drafts_nonfinite_logit_is_flagged(where):
    """A NaN or +inf logit, in a step inside the row (the statistics' fast path) or in the
    ragged last step, leaves that row without a distribution and sets PE_DEV_NONFINITE; the
    error word stays clear without one."""
    B, K, V = 2, 2, 4099
    rng, logits = _seeded(B, K, V, seed=23)
    if where == "full-step-nan":
        logits[1, 1500] = np.nan
    elif where == "full-step-posinf":
        logits[2, 700] = np.inf
    elif where == "last-step-nan":
        logits[3, V - 2] = np.nan
    u = rng.random((B, K))
    cfg = _cfg(B, K, V)
    lg = torch.from_numpy(logits).cuda()
    drafts = torch.empty((B, K), dtype=torch.int32, device="cuda")
    lse = torch.empty(B * K, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pe.sample_drafts(cfg, lg, torch.from_numpy(u.astype(np.float32)).cuda(), 1.0, pe.alloc_workspace(cfg), drafts,
                     lse, err)
    torch.cuda.synchronize()
    assert int(err.item()) == (0 if where == "none" else pe.PE_DEV_NONFINITE)
    gl = lse.cpu().numpy()
    bad_row = {"full-step-nan": 1, "full-step-posinf": 2, "last-step-nan": 3}.get(where)
    for r in range(B * K):
        assert np.isfinite(gl[r]) == (r != bad_row), r


def test_sample_drafts_fully_masked_row_is_flagged():
    """A row whose every logit is -inf has no distribution: token 0, lse NaN, PE_DEV_NONFINITE;
    the other rows draw normally."""
    B, K, V = 1, 2, 1000
    rng, logits = _seeded(B, K, V, seed=5)
    logits[1] = -np.inf
    u = rng.random((B, K))
    cfg = _cfg(B, K, V)
    lg = torch.from_numpy(logits).cuda()
    drafts = torch.empty((B, K), dtype=torch.int32, device="cuda")
    lse = torch.empty(B * K, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pe.sample_drafts(cfg, lg, torch.from_numpy(u.astype(np.float32)).cuda(), 1.0, pe.alloc_workspace(cfg), drafts,
                     lse, err)
    torch.cuda.synchronize()
    assert int(err.item()) == pe.PE_DEV_NONFINITE
    g, gl = drafts.cpu().numpy().reshape(-1), lse.cpu().numpy()
    assert g[1] == 0 and np.isnan(gl[1])
    q, want_lse = oracle.drafter_distribution(logits[0], 1.0)
    assert abs(gl[0] - want_lse) <= 1e-4 * max(1.0, abs(want_lse))
    assert q[g[0]] > 0


def _targets(rng, drafts, B, K, V, boost=3.0):
    """Seeded target distributions: normalised exp of N(0, 2) draws, with the draft token
    raised at about 60 % of positions so that drafts get accepted."""
    z = rng.normal(0.0, 2.0, size=(B, K + 1, V))
    up = rng.random((B, K)) < 0.6
    for b in range(B):
        for k in range(K):
            if up[b, k]:
                z[b, k, drafts[b, k]] += boost + z[b, k].max()
    p = np.exp(z - z.max(axis=2, keepdims=True))
    return (p / p.sum(axis=2, keepdims=True)).astype(np.float32)


@pytest.mark.parametrize("B,K,V,T", [(32, 4, 1000, 1.0), (8, 7, 151936, 0.8)])
def test_verify_sampled_against_oracle(B, K, V, T):
    rng, logits = _seeded(B, K, V, seed=3 * V + K, scale=2.0)
    # drafts: the row's most likely token half of the time, else a uniform token
    am = logits.reshape(B, K, V).argmax(axis=2)
    drafts = np.where(rng.random((B, K)) < 0.5, am, rng.integers(0, V, size=(B, K))).astype(np.int32)
    P = _targets(rng, drafts, B, K, V)
    u_acc = rng.random((B, K)).astype(np.float32)
    u_res = rng.random(B).astype(np.float32)
    cfg = _cfg(B, K, V)
    lg, _, lse = _gpu_sample(cfg, logits, rng.random((B, K)), T)  # lse of these logits
    d = torch.from_numpy(drafts).cuda()
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bonus = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pe.verify_sampled(cfg, d, lg, lse, T, torch.from_numpy(P).cuda(), torch.from_numpy(u_acc).cuda(),
                      torch.from_numpy(u_res).cuda(), pe.alloc_workspace(cfg), acc, bonus, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ga, gb = acc.cpu().numpy(), bonus.cpu().numpy()
    Pd = P.astype(np.float64)
    wa, wb = oracle.verify_sampled(drafts, logits, T, Pd, u_acc.astype(np.float64), u_res.astype(np.float64))
    assert 0 < int(wa.sum()) < B * K  # some drafts accepted, some rejected
    n_checked = 0
    for b in range(B):
        # accept decisions within the fp32 error of their threshold are left out
        close = False
        for k in range(min(int(wa[b]) + 1, K)):
            q, _ = oracle.drafter_distribution(logits[b * K + k], T)
            x = drafts[b, k]
            if abs(u_acc[b, k] * q[x] - Pd[b, k, x]) <= 1e-5 * max(Pd[b, k, x], q[x]):
                close = True
        if close:
            continue
        n_checked += 1
        assert ga[b] == wa[b], b
        if gb[b] != wb[b]:
            a = int(wa[b])
            if a < K:
                q, _ = oracle.drafter_distribution(logits[b * K + a], T)
                w = np.maximum(0.0, Pd[b, a] - q)
                w = w if w.sum() > 0 else Pd[b, a]
            else:
                w = Pd[b, K]
            assert _in_band(w, int(gb[b]), u_res[b], CDF_EPS), b
    assert n_checked >= B - 2


def test_pipeline_forward_sample_verify_f32():
    """The drafter's own logits (f32 config): forward with logits, draw the drafts, verify
    by rejection sampling.  Drafts against the oracle's draws from its fp64 logits, to
    within the band the logit tolerance allows; where every draft and accept decision is
    clear of its boundary, accepted counts are equal."""
    cfg_np = Config(name="small-f32-L2", B=3, K=4, n_layers=2, d=256, n_q=8, n_kv=2, head_dim=64, ffn=384,
                    vocab=1000, dtype="f32", prefix="uniform", prefix_args=(1, 300), accepted="uniform", seed=11)
    c = setup(cfg_np)
    assert run_stages(c) == 0
    B, K, V = cfg_np.B, cfg_np.K, cfg_np.vocab
    T = 1.0
    rng = np.random.default_rng(21)
    u_d = rng.random((B, K)).astype(np.float32)
    c.rd.sample(torch.from_numpy(u_d).cuda(), T)
    torch.cuda.synchronize()
    assert int(c.rd.err.item()) == 0
    g = c.rd.draft_tokens.cpu().numpy()
    ref = oracle.run_round(cfg_np, c.w_np, c.r_np)
    want, _ = oracle.sample_drafts(ref["logits"], u_d.astype(np.float64), T)
    eps = 4 * LOGIT_TOL[cfg_np.dtype] / T
    for b in range(B):
        for k in range(K):
            if g[b, k] != want[b, k]:
                q, _ = oracle.drafter_distribution(ref["logits"][b * K + k], T)
                assert _in_band(q, int(g[b, k]), u_d[b, k], eps), (b, k)
    P = _targets(rng, want, B, K, V)
    u_acc = rng.random((B, K)).astype(np.float32)
    u_res = rng.random(B).astype(np.float32)
    c.rd.verify_sampled(torch.from_numpy(P).cuda(), torch.from_numpy(u_acc).cuda(), torch.from_numpy(u_res).cuda(), T)
    torch.cuda.synchronize()
    assert int(c.rd.err.item()) == 0
    ga = c.rd.out["num_accepted"].cpu().numpy()
    wa, _ = oracle.verify_sampled(want, ref["logits"], T, P.astype(np.float64), u_acc.astype(np.float64),
                                  u_res.astype(np.float64))
    for b in range(B):
        if not np.array_equal(g[b], want[b]):
            continue
        clear = True
        for k in range(K):
            q, _ = oracle.drafter_distribution(ref["logits"][b * K + k], T)
            x = want[b, k]
            if abs(u_acc[b, k] * q[x] - P[b, k, x]) <= eps * max(P[b, k, x], q[x]):
                clear = False
        if clear:
            assert ga[b] == wa[b], b
