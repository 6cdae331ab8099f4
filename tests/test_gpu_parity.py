"""CUDA path against the CPU oracle, element by element, through the C ABI.

Integer work (batch metadata, compaction, verification) is bit-exact; the input
rows are a copy, so bit-exact too; logits are within 1e-3 (fp32) / 5e-2 (bf16)
and draft tokens equal wherever the oracle's top-1/top-2 gap exceeds 0.1.
"""

import dataclasses
import itertools

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_step_gb300 as pe
from pe_workload import (Config, bf16_to_f32, config, f32_to_bf16, loop_round_draws, make_round, make_targets,
                         make_weights, sweep_config)
from pe_workload.device import to_torch

from gpu_harness import (GAP, KV_TOL, LOGIT_TOL, check_kv_writes, check_logits, meta_np, oracle_round, run_stages,
                         setup, to_np_storage)

pytestmark = pytest.mark.gpu


def _small(**kw) -> Config:
    base = dict(name="small-bf16", B=3, K=4, n_layers=1, d=256, n_q=8, n_kv=2, head_dim=64, ffn=384,
                vocab=1000, dtype="bf16", prefix="uniform", prefix_args=(1, 300), accepted="uniform", seed=7)
    base.update(kw)
    return Config(**base)


SMALL = {
    "bf16-hd64": _small(),
    "bf16-hd128-K8-G8": _small(B=2, K=8, n_q=16, n_kv=2, head_dim=128, d=512, ffn=640, vocab=777, seed=8),
    "bf16-K1": _small(B=5, K=1, seed=9),
    "bf16-L2-long": _small(B=2, K=7, n_layers=2, prefix_args=(900, 2100), vocab=3001, seed=10),
    # more vocabulary tiles (161, the last one ragged) than SMs with a short last wave:
    # the LM head cuts tiles at CTA range boundaries and sums the two pieces
    "bf16-lm-balanced": _small(B=4, K=8, vocab=160 * 128 + 37, seed=12),
    # odd numbers of 64-wide k atoms in every contraction (d 320 = 5, 2d = 10, ffn 448 = 7,
    # n_q*hd 512 = 8): two-atom pipeline stages end on a half stage whose second atom is
    # past K and zero-filled
    "bf16-odd-atoms": _small(B=3, K=5, d=320, ffn=448, seed=13),
    # a deeper drafter: four layers, each its own weights and KV cache
    "bf16-L4": _small(B=2, K=6, n_layers=4, prefix_args=(100, 700), seed=14),
    # more than 256 rows and an LM head of 160 rows: every GEMM runs on CTA pairs (M = 256
    # over two SMs); three weight tiles (an odd count: the last pair's second tile is past
    # the end), split K in fc / o-proj / down, and a ragged nine-tile vocabulary
    "bf16-pairs": _small(B=20, K=8, d=320, ffn=448, vocab=1037, seed=15),
    # contractions short enough that no GEMM splits K (every epilogue writes final values and
    # every RMSNorm reads the residual as it is), on single CTAs over two layers, and on CTA
    # pairs
    "bf16-fold": _small(B=6, K=8, d=192, n_q=4, n_kv=2, ffn=384, vocab=1037, n_layers=2, seed=16),
    "bf16-fold-pairs": _small(B=20, K=8, d=192, n_q=4, n_kv=2, ffn=384, vocab=1037, seed=17),
    # 128 (sequence, kv head) pairs with several chunks each: the chunk merge that packs
    # several query vectors into a warp
    "bf16-many-pairs": _small(B=64, K=2, n_q=4, n_kv=2, d=128, ffn=128, vocab=500, prefix_args=(300, 900),
                              seed=18),
    # LM heads on CTA pairs over more units than pairs (161 vocabulary tiles, the last
    # ragged: 81 units of two), with one token tile of 160 rows and with two of 160
    "bf16-pairs-many-units": _small(B=20, K=8, d=320, ffn=448, vocab=160 * 128 + 37, seed=19),
    "bf16-pairs-many-units-2t": _small(B=40, K=8, d=320, ffn=448, vocab=160 * 128 + 37, seed=20),
    "f32-c0": config(0),
    "f32-L2": _small(dtype="f32", n_layers=2, seed=11),
}


# ----------------------------------------------------------------------------- stage (a)

def _prep_compare(cfg_np, rnd):
    R = {k: torch.from_numpy(np.ascontiguousarray(getattr(rnd, k), dtype=np.int32)).cuda()
         for k in ("prev_tokens", "prev_pos", "num_accepted", "bonus", "block_table")}
    cfg = pe.Config.make(cfg_np.B, cfg_np.K, cfg_np.d, cfg_np.n_q, cfg_np.n_kv, cfg_np.head_dim, cfg_np.ffn,
                         cfg_np.vocab, cfg_np.n_layers, rnd.block_table.shape[1], cfg_np.dtype)
    meta = pe.alloc_batch(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pe.prepare_batch(cfg, R["prev_tokens"], R["prev_pos"], R["num_accepted"], R["bonus"], R["block_table"],
                     rnd.num_pages, meta, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.prepare_batch(cfg_np.K, cfg_np.vocab, rnd.prev_tokens, rnd.prev_pos, rnd.num_accepted, rnd.bonus,
                               rnd.block_table, cfg_np.page_size)
    got = {k: v.cpu().numpy() for k, v in meta.items()}
    n = ref["n_valid"]
    assert int(got["n_valid"][0]) == n
    for k in ("input_ids", "positions", "slot_mapping", "is_rejected", "is_mask", "hidden_map"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["row_list"][:n], ref["row_list"])
    assert (got["row_list"][n:] == -1).all()
    assert np.array_equal(got["draft_rows"], ref["draft_rows"])


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_prepare_batch_bit_exact_configs(idx):
    cfg_np = config(idx)
    _prep_compare(cfg_np, make_round(cfg_np, with_cache=False))


@pytest.mark.parametrize("K,a_mode", [(1, "all0"), (1, "allK"), (8, "all0"), (8, "allK"), (5, "mixed")])
def test_prepare_batch_bit_exact_edges(K, a_mode):
    cfg_np = sweep_config(37, K)
    rnd = make_round(cfg_np, with_cache=False)
    if a_mode == "all0":
        rnd.num_accepted[:] = 0
    elif a_mode == "allK":
        rnd.num_accepted[:] = K
    _prep_compare(cfg_np, rnd)


def test_prepare_batch_large_batch_multi_chunk():
    """B*2K > 1024: the single-CTA rebuild scans several chunks with a carry."""
    cfg_np = sweep_config(100, 8)   # 1600 padded rows
    _prep_compare(cfg_np, make_round(cfg_np, with_cache=False))


# ----------------------------------------------------------------------------- stage (e)

def test_verify_brute_force_and_random():
    rows_d, rows_t = [], []
    K = 3
    for d in itertools.product(range(3), repeat=K):
        for t in itertools.product(range(3), repeat=K + 1):
            rows_d.append(d)
            rows_t.append(t)
    rng = np.random.default_rng(0)
    for _ in range(500):
        d = rng.integers(0, 4, K)
        rows_d.append(tuple(d))
        rows_t.append(tuple(rng.integers(0, 4, K + 1)))
    D = np.array(rows_d, np.int32)
    T = np.array(rows_t, np.int32)
    cfg = pe.Config.make(len(D), K, 256, 4, 4, 64, 256, 16, 1, 4, "bf16")
    acc = torch.empty(len(D), dtype=torch.int32, device="cuda")
    bon = torch.empty_like(acc)
    pe.verify(cfg, torch.from_numpy(D).cuda(), torch.from_numpy(T).cuda(), acc, bon)
    torch.cuda.synchronize()
    ra, rb = oracle.verify(D, T)
    assert np.array_equal(acc.cpu().numpy(), ra)
    assert np.array_equal(bon.cpu().numpy(), rb)


# ----------------------------------------------------------------------------- stage (b)

@pytest.mark.parametrize("name", ["f32-c0", "bf16-hd64", "bf16-K1"])
def test_scatter_bit_exact(name):
    c = setup(SMALL[name])
    R = c.Rd
    c.rd.prepare(R["prev_tokens"], R["prev_pos"], R["num_accepted"], R["bonus"])
    c.rd.scatter(R["target_hidden"])
    torch.cuda.synchronize()
    assert int(c.rd.err.item()) == 0
    m = oracle.prepare_batch(c.cfg_np.K, c.cfg_np.vocab, c.r_np.prev_tokens, c.r_np.prev_pos,
                             c.r_np.num_accepted, c.r_np.bonus, c.r_np.block_table)
    x0 = oracle.scatter_hidden(c.w_np.emb, c.w_np.h_shared, c.r_np.target_hidden, m["input_ids"], m["is_mask"],
                               m["hidden_map"])
    got = to_np_storage(c.rd.x0)[: m["n_valid"]]
    assert np.array_equal(got, x0[m["row_list"]])


def test_scatter_bit_exact_full_size_c3():
    cfg_np = config(3)
    c = setup(cfg_np)
    R = c.Rd
    c.rd.prepare(R["prev_tokens"], R["prev_pos"], R["num_accepted"], R["bonus"])
    c.rd.scatter(R["target_hidden"])
    torch.cuda.synchronize()
    assert int(c.rd.err.item()) == 0
    m = oracle.prepare_batch(cfg_np.K, cfg_np.vocab, c.r_np.prev_tokens, c.r_np.prev_pos, c.r_np.num_accepted,
                             c.r_np.bonus, c.r_np.block_table)
    x0 = oracle.scatter_hidden(c.w_np.emb, c.w_np.h_shared, c.r_np.target_hidden, m["input_ids"], m["is_mask"],
                               m["hidden_map"])
    assert np.array_equal(to_np_storage(c.rd.x0)[: m["n_valid"]], x0[m["row_list"]])


# ----------------------------------------------------------------------------- stages (c)+(d)

@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small_full_oracle(name):
    """Every sequence, every draft logit, and every cache entry, against the oracle."""
    c = setup(SMALL[name])
    assert run_stages(c) == 0
    ref = oracle_round(c, want_kv=True)
    check_logits(c, ref)
    check_kv_writes(c, ref)


def _ramped_keys(cfg_np, rnd, octaves_per_block: float):
    """The round with its cached prefix keys scaled by 2^(octaves_per_block * p / 64) at
    position p: each 64-position block's scores run far above the last one's, so the
    attention's reference maximum moves (and O is rescaled in TMEM) block after block."""
    out = []
    for kc in rnd.k_cache:
        kf = bf16_to_f32(kc) if cfg_np.dtype == "bf16" else np.array(kc, dtype=np.float32)
        kf = kf.copy()
        for b in range(cfg_np.B):
            for p in range(int(rnd.prefix_len[b])):
                page = int(rnd.block_table[b][p // cfg_np.page_size])
                kf[page, p % cfg_np.page_size] *= np.float32(2.0 ** (octaves_per_block * p / 64.0))
        out.append(f32_to_bf16(kf) if cfg_np.dtype == "bf16" else kf)
    return dataclasses.replace(rnd, k_cache=out)


@pytest.mark.parametrize("name,octaves", [("bf16-hd64", 1.0), ("bf16-hd64", 1.25), ("bf16-hd128-K8-G8", 1.0)])
def test_attention_lazy_rescale(name, octaves):
    """Scores that keep growing along the prefix (keys ramped by up to 2^5.9, the block
    maximum roughly doubling from block to block): in the later blocks the running maximum
    outgrows the reference by more than 2^8, so the lazy O rescale (which waits for the
    previous block's PV product) runs: an instrumented copy of the kernel counted 9-28
    warp-wide rescales per case, and none in the same rounds without the ramp (the other
    parity cases never reach this path).  Every logit and cache entry against the oracle.  (Steeper ramps make the scores so large that the bf16
    rounding of q, which the fp64 oracle does not share, moves the softmax weights by more
    than the logit tolerance: a precision limit, not a fault of the path.)"""
    cfg_np = dataclasses.replace(SMALL[name], prefix_args=(250, 300))
    rnd = _ramped_keys(cfg_np, make_round(cfg_np), octaves)
    c = setup(cfg_np, rnd=rnd)
    assert run_stages(c) == 0
    ref = oracle_round(c, want_kv=True)
    check_logits(c, ref)
    check_kv_writes(c, ref)


@pytest.mark.parametrize("idx,seqs", [(1, None), (2, None), (3, "sample")])
def test_forward_full_size(idx, seqs):
    """The benchmark workloads at their full sizes; at B=64 the oracle checks a sample of
    sequences (independent of one another): the shortest, the longest, and two fully rejected
    ones where present."""
    cfg_np = config(idx)
    c = setup(cfg_np)
    assert run_stages(c) == 0
    if seqs == "sample":
        P, a = c.r_np.prefix_len, c.r_np.num_accepted
        seqs = sorted({int(np.argmin(P)), int(np.argmax(P))} | set(np.nonzero(a == 0)[0][:2].tolist())
                      | {int(np.argmax(a))})
    ref = oracle_round(c, seqs=seqs, want_kv=False)
    check_logits(c, ref, seqs)


def test_forward_sweep_corners():
    """K x B sweep drafter (2 layers): corners B=1, K=1 and B=64, K=8 (sampled)."""
    for B, K in ((1, 1), (64, 8)):
        cfg_np = sweep_config(B, K)
        c = setup(cfg_np)
        assert run_stages(c) == 0
        seqs = None if B == 1 else [0, int(np.argmax(c.r_np.prefix_len))]
        check_logits(c, oracle_round(c, seqs=seqs), seqs)


# ----------------------------------------------------------------------------- invariants on the GPU path

def test_deterministic_and_page_permutation_invariant():
    cfg_np = SMALL["bf16-L2-long"]
    c = setup(cfg_np)
    assert run_stages(c) == 0
    lg1, d1 = c.rd.logits.clone(), c.rd.draft_tokens.clone()
    # same inputs again (fresh cache copy): bit-identical
    for l in range(cfg_np.n_layers):
        c.kv.k_cache[l].copy_(c.k_before[l])
        c.kv.v_cache[l].copy_(c.v_before[l])
    assert run_stages(c) == 0
    assert torch.equal(lg1, c.rd.logits) and torch.equal(d1, c.rd.draft_tokens)
    # the same logical cache on permuted physical pages
    rnd = c.r_np
    perm = np.random.default_rng(1).permutation(rnd.num_pages)
    for l in range(cfg_np.n_layers):
        rnd.k_cache[l] = rnd.k_cache[l].copy()
        rnd.v_cache[l] = rnd.v_cache[l].copy()
        k2, v2 = np.empty_like(rnd.k_cache[l]), np.empty_like(rnd.v_cache[l])
        k2[perm], v2[perm] = rnd.k_cache[l], rnd.v_cache[l]
        rnd.k_cache[l], rnd.v_cache[l] = k2, v2
    rnd.block_table = np.where(rnd.block_table >= 0, perm[np.maximum(rnd.block_table, 0)], -1).astype(np.int32)
    c2 = setup(cfg_np, weights=c.w_np, rnd=rnd)
    assert run_stages(c2) == 0
    assert torch.equal(lg1, c2.rd.logits) and torch.equal(d1, c2.rd.draft_tokens)


@pytest.mark.parametrize("path", ["stages", "step"])
def test_context_positions_decreasing(path):
    """Rows whose positions do not increase along the verify batch: the context rows of
    sequence b sit at P + 2(K - r), the NTP row above them all, so the sequence's smallest
    position this round is its last context row's (neither its first row's nor the NTP
    row's).  The attention loads the cache pages wholly below that position before the
    kernel writing the round's k / v has finished; logits, drafts and every cache entry match
    the oracle."""
    cfg_np = SMALL["bf16-L2-long"]
    K = cfg_np.K
    rnd = make_round(cfg_np, extra_positions=K + 2)
    P, a = rnd.prefix_len, rnd.num_accepted
    pp = np.empty_like(rnd.prev_pos)
    for b in range(cfg_np.B):
        for r in range(K + 1):
            pp[b, r] = P[b] + 2 * (K - r) if r < a[b] else P[b] + 2 * K + 1 + (r - a[b])
    rnd.prev_pos = pp.astype(np.int32)
    assert (a > 1).any()  # some sequence has its smallest position at a context row past the first
    c = setup(cfg_np, rnd=rnd)
    if path == "stages":
        assert run_stages(c) == 0
    else:
        drafts_target = np.zeros((cfg_np.B, K), dtype=np.int32)
        R = c.Rd
        c.rd.step(R["prev_tokens"], R["prev_pos"], R["num_accepted"], R["bonus"], R["target_hidden"],
                  torch.from_numpy(drafts_target).cuda(), logits=True)
        torch.cuda.synchronize()
        assert int(c.rd.err.item()) == 0
    ref = oracle_round(c, want_kv=True)
    check_logits(c, ref)
    check_kv_writes(c, ref)


@pytest.mark.parametrize("idx", [1, 2])
def test_repeat_runs_bit_identical_full_size(idx):
    """The full-size workloads run repeatedly give bit-identical logits and drafts: a
    synchronisation race between the pipelines' warps (a stage or accumulator read before
    its producer finished) shows up as run-to-run differences."""
    cfg_np = config(idx)
    c = setup(cfg_np)
    assert run_stages(c) == 0
    lg1, d1 = c.rd.logits.clone(), c.rd.draft_tokens.clone()
    for _ in range(6):
        for l in range(cfg_np.n_layers):
            c.kv.k_cache[l].copy_(c.k_before[l])
            c.kv.v_cache[l].copy_(c.v_before[l])
        assert run_stages(c) == 0
        assert torch.equal(d1, c.rd.draft_tokens)
        assert torch.equal(lg1, c.rd.logits)


def test_step_equals_stages_and_next_batch():
    cfg_np = SMALL["bf16-hd64"]
    c = setup(cfg_np)
    assert run_stages(c) == 0
    drafts = c.rd.draft_tokens.cpu().numpy()
    target = make_targets(drafts, c.r_np.target_u, c.r_np.target_r)
    # fresh cache, then the whole round in one call
    for l in range(cfg_np.n_layers):
        c.kv.k_cache[l].copy_(c.k_before[l])
        c.kv.v_cache[l].copy_(c.v_before[l])
    lg_stages = c.rd.logits.clone()
    R = c.Rd
    c.rd.step(R["prev_tokens"], R["prev_pos"], R["num_accepted"], R["bonus"], R["target_hidden"],
              torch.from_numpy(target).cuda(), logits=True)
    torch.cuda.synchronize()
    assert int(c.rd.err.item()) == 0
    assert torch.equal(c.rd.logits, lg_stages)
    assert np.array_equal(c.rd.draft_tokens.cpu().numpy(), drafts)
    ra, rb = oracle.verify(drafts, target)
    assert np.array_equal(c.rd.out["num_accepted"].cpu().numpy(), ra)
    assert np.array_equal(c.rd.out["bonus"].cpu().numpy(), rb)
    nt = c.rd.out["next_prev_tokens"].cpu().numpy()
    npos = c.rd.out["next_prev_pos"].cpu().numpy()
    for b in range(cfg_np.B):
        a = int(c.r_np.num_accepted[b])
        assert nt[b, 0] == c.r_np.bonus[b] and np.array_equal(nt[b, 1:], drafts[b])
        assert np.array_equal(npos[b], c.r_np.prev_pos[b][a] + 1 + np.arange(cfg_np.K + 1))


# ----------------------------------------------------------------------------- the timed path at full size

def _sampled_seqs(r_np):
    """Sequences the oracle checks at B > 8: the shortest and longest prefix, two fully rejected
    ones where present, and the one with the most accepted drafts."""
    if len(r_np.prefix_len) <= 8:
        return list(range(len(r_np.prefix_len)))
    P, a = r_np.prefix_len, r_np.num_accepted
    return sorted({int(np.argmin(P)), int(np.argmax(P)), int(np.argmax(a))} | set(np.nonzero(a == 0)[0][:2].tolist()))


@pytest.mark.parametrize("which", ["c1", "c2", "c3", "sweep-B64-K8"])
def test_step_graph_full_size(which):
    """The path the benchmark times: pe_step without debug logits, captured once in a CUDA graph
    and replayed, at full size.  Drafts agree with the oracle on the checked sequences (exactly
    where the oracle's top-1/top-2 gap is clear, otherwise the picked token's oracle logit is
    within twice the tolerance of the top one); accepted counts, bonus tokens and the next
    verify batch are bit-exact for every sequence; the KV entries the checked sequences write
    match the oracle's post-RoPE k / v, and no other cache entry changes; two more replays give
    bit-identical drafts and outputs."""
    cfg_np = {"c1": config(1), "c2": config(2), "c3": config(3), "sweep-B64-K8": sweep_config(64, 8)}[which]
    c = setup(cfg_np)
    B, K, L = cfg_np.B, cfg_np.K, cfg_np.n_layers
    R = c.Rd
    target = torch.zeros((B, K + 1), dtype=torch.int32, device="cuda")
    step = lambda: c.rd.step(R["prev_tokens"], R["prev_pos"], R["num_accepted"], R["bonus"], R["target_hidden"],
                             target)
    step()                                  # launch attributes are set on each kernel's first use
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    torch.cuda.synchronize()
    assert int(c.rd.err.item()) == 0
    drafts = c.rd.draft_tokens.cpu().numpy()
    tgt = make_targets(drafts, c.r_np.target_u, c.r_np.target_r)
    target.copy_(torch.from_numpy(tgt))
    outs = []
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert int(c.rd.err.item()) == 0
        outs.append({k: v.cpu().numpy().copy() for k, v in c.rd.out.items()})
    for k in outs[0]:
        assert np.array_equal(outs[0][k], outs[1][k]), k
    out = outs[0]
    assert np.array_equal(out["draft_tokens"], drafts)
    # verification and the next verify batch, for every sequence, on the GPU's own drafts
    acc, bon = oracle.verify(drafts, tgt)
    assert np.array_equal(out["num_accepted"], acc) and np.array_equal(out["bonus"], bon)
    nt, npos = oracle.next_verify_batch(c.r_np.prev_pos, c.r_np.num_accepted, c.r_np.bonus, drafts)
    assert np.array_equal(out["next_prev_tokens"], nt) and np.array_equal(out["next_prev_pos"], npos)
    # drafts of the checked sequences against the oracle
    seqs = _sampled_seqs(c.r_np)
    ref = oracle_round(c, seqs=seqs, want_kv=True)
    tol = LOGIT_TOL[cfg_np.dtype]
    lg = ref["logits"].reshape(len(seqs), K, -1)
    got = drafts[seqs]
    picked = np.take_along_axis(lg, got[..., None].astype(np.int64), axis=2)[..., 0]
    assert (picked >= lg.max(axis=2) - 2 * tol).all()
    sure = (oracle.top2_gap(ref["logits"]) > GAP).reshape(len(seqs), K)
    assert sure.any()
    assert np.array_equal(got[sure], ref["drafts"][sure])
    # cache: the checked sequences' entries, then no entry outside the round's slots changed
    meta = ref["meta"]
    kvd = cfg_np.n_kv * cfg_np.head_dim
    slots_all = torch.from_numpy(meta["slot_mapping"][meta["row_list"]]).cuda()
    slots_chk = meta["slot_mapping"][ref["rows"]]
    for l in range(L):
        for nm, dev, before, new in (("k", c.kv.k_cache[l], c.k_before[l], ref["new_k"][l]),
                                     ("v", c.kv.v_cache[l], c.v_before[l], ref["new_v"][l])):
            a2, b2 = dev.view(-1, kvd), before.view(-1, kvd)
            changed = (a2 != b2).any(dim=1)
            changed[slots_all] = False
            assert int(changed.sum().item()) == 0, f"{nm} cache layer {l}: stray write"
            gotv = a2[torch.from_numpy(slots_chk).cuda()].float().cpu().numpy().astype(np.float64)
            diff = np.abs(gotv - new) / np.maximum(1.0, np.abs(new))
            assert diff.max() <= KV_TOL[cfg_np.dtype], f"{nm} cache layer {l}: rel diff {diff.max():.3g}"


# ----------------------------------------------------------------------------- rounds back to back

@pytest.mark.parametrize("name", ["f32-L2", "bf16-hd64", "bf16-L2-long"])
def test_multi_round_loop_in_place_graph(name):
    """Rounds back to back with the round state updated in place: round 0 through a direct
    pe_step call, then replays of one captured CUDA graph, the caller refilling the target's
    hidden states and tokens in between.  The oracle runs every round from the same state:
    the drafts agree (exactly where the oracle's top-1/top-2 gap is clear, otherwise the
    picked token's oracle logit is within twice the logit tolerance of the top one); accepted
    counts, bonus tokens and the next verify batch are bit-exact; and after the last round the
    caches hold the oracle's writes of every round, a later round's write winning where a
    position was written twice (a MASK row's speculative entry overwritten by the next round's
    accepted row at that position)."""
    n_rounds = 4
    cfg_np = SMALL[name]
    B, K, L = cfg_np.B, cfg_np.K, cfg_np.n_layers
    kvd = cfg_np.n_kv * cfg_np.head_dim
    rnd = make_round(cfg_np, extra_positions=n_rounds * (K + 1))
    c = setup(cfg_np, rnd=rnd)
    storage = (lambda x: f32_to_bf16(x)) if cfg_np.dtype == "bf16" else (lambda x: x.astype(np.float32))
    ok, ov = [x.copy() for x in rnd.k_cache], [x.copy() for x in rnd.v_cache]
    written = np.zeros(ok[0].shape[0] * ok[0].shape[1], dtype=bool)
    st = dict(prev_tokens=rnd.prev_tokens.copy(), prev_pos=rnd.prev_pos.copy(),
              num_accepted=rnd.num_accepted.copy(), bonus=rnd.bonus.copy())
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    state = {k: i32(v) for k, v in st.items()}
    th = c.Rd["target_hidden"].clone()
    tt = torch.zeros((B, K + 1), dtype=torch.int32, device="cuda")
    tol = LOGIT_TOL[cfg_np.dtype]
    graph, total_accepted = None, 0
    for r in range(n_rounds):
        hidden, u, tr = (rnd.target_hidden, rnd.target_u, rnd.target_r) if r == 0 else loop_round_draws(cfg_np, r)
        ref = oracle.run_round(cfg_np, c.w_np, dataclasses.replace(rnd, target_hidden=hidden, k_cache=ok,
                                                                    v_cache=ov, **st), want_kv=True)
        target = make_targets(ref["drafts"], u, tr)
        th.copy_(to_torch(hidden))
        tt.copy_(i32(target))
        if r == 0:
            c.rd.step_inplace(state, th, tt)
        else:
            if graph is None:
                graph = c.rd.capture_loop(state, th, tt)
            graph.replay()
        torch.cuda.synchronize()
        assert int(c.rd.err.item()) == 0, f"round {r}"
        drafts = c.rd.draft_tokens.cpu().numpy()
        lg = ref["logits"].reshape(B, K, -1)
        picked = np.take_along_axis(lg, drafts[..., None].astype(np.int64), axis=2)[..., 0]
        assert (picked >= lg.max(axis=2) - 2 * tol).all(), f"round {r}"
        sure = (oracle.top2_gap(ref["logits"]) > GAP).reshape(B, K)
        assert np.array_equal(drafts[sure], ref["drafts"][sure]), f"round {r}"
        acc, bon = oracle.verify(drafts, target)
        nt, npos = oracle.next_verify_batch(st["prev_pos"], st["num_accepted"], st["bonus"], drafts)
        got = {k: v.cpu().numpy() for k, v in state.items()}
        assert np.array_equal(got["num_accepted"], acc) and np.array_equal(got["bonus"], bon), f"round {r}"
        assert np.array_equal(got["prev_tokens"], nt) and np.array_equal(got["prev_pos"], npos), f"round {r}"
        slots = ref["meta"]["slot_mapping"][ref["rows"]]
        for l in range(L):
            ok[l].reshape(-1, kvd)[slots] = storage(ref["new_k"][l])
            ov[l].reshape(-1, kvd)[slots] = storage(ref["new_v"][l])
        written[slots] = True
        st = dict(prev_tokens=nt, prev_pos=npos, num_accepted=acc, bonus=bon)
        total_accepted += int(acc.sum())
    assert total_accepted > 0  # the loop went past the first verify batch
    for l in range(L):
        for nm, dev, want in (("k", c.kv.k_cache[l], ok[l]), ("v", c.kv.v_cache[l], ov[l])):
            g_bits = to_np_storage(dev).reshape(-1, kvd)
            w_bits = want.reshape(-1, kvd)
            assert np.array_equal(g_bits[~written], w_bits[~written]), f"{nm} cache layer {l}: stray write"
            g, w = oracle.widen(g_bits[written]), oracle.widen(w_bits[written])
            diff = np.abs(g - w) / np.maximum(1.0, np.abs(w))
            assert diff.max() <= KV_TOL[cfg_np.dtype], f"{nm} cache layer {l}: rel diff {diff.max():.3g}"


# ----------------------------------------------------------------------------- device-side checks

def test_device_check_bad_accepted_count():
    """An accepted count above K is flagged on the device; the rows stay in bounds."""
    cfg_np = SMALL["bf16-hd64"]
    rnd = make_round(cfg_np)
    rnd.num_accepted[1] = cfg_np.K + 3
    c = setup(cfg_np, rnd=rnd)
    assert run_stages(c) == pe.PE_DEV_BAD_ACCEPTED


def test_device_check_bad_page():
    """A block-table entry outside the page pool is flagged and no cache access uses it."""
    cfg_np = SMALL["bf16-hd64"]
    rnd = make_round(cfg_np)
    rnd.block_table[0, 0] = rnd.num_pages + 5
    c = setup(cfg_np, rnd=rnd)
    assert run_stages(c) == pe.PE_DEV_BAD_PAGE
