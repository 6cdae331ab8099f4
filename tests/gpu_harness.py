"""Shared set-up for the GPU parity tests: seeded inputs on the device, the C-ABI calls, and
the oracle on the same inputs.  Nothing here computes what the method computes."""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import speculative_decoding_step_gb300 as pe
from pe_workload import Config, make_round, make_weights
from pe_workload.device import round_to_device, weights_to_device

LOGIT_TOL = {"f32": 1e-3, "bf16": 5e-2}
KV_TOL = {"f32": 1e-4, "bf16": 3e-2}  # relative to max(1, |value|); bf16 storage of k and v
GAP = 0.1


@dataclasses.dataclass
class Case:
    cfg_np: Config
    w_np: object
    r_np: object
    W: dict
    Rd: dict
    cfg: pe.Config
    weights: pe.DeviceWeights
    kv: pe.DeviceKV
    rd: pe.Round
    k_before: list
    v_before: list


def abi_config(cfg_np: Config, max_pages: int) -> pe.Config:
    return pe.Config.make(cfg_np.B, cfg_np.K, cfg_np.d, cfg_np.n_q, cfg_np.n_kv, cfg_np.head_dim, cfg_np.ffn,
                          cfg_np.vocab, cfg_np.n_layers, max_pages, cfg_np.dtype, rms_eps=cfg_np.rms_eps,
                          rope_theta=cfg_np.rope_theta)


def setup(cfg_np: Config, seed=None, weights=None, rnd=None) -> Case:
    w_np = weights if weights is not None else make_weights(cfg_np, seed)
    r_np = rnd if rnd is not None else make_round(cfg_np, seed)
    W, Rd = weights_to_device(w_np), round_to_device(r_np)
    cfg = abi_config(cfg_np, r_np.block_table.shape[1])
    dw = pe.DeviceWeights(**W)
    kv = pe.DeviceKV(Rd["k_cache"], Rd["v_cache"])
    rd = pe.Round(cfg, dw, kv, Rd["block_table"])
    return Case(cfg_np, w_np, r_np, W, Rd, cfg, dw, kv, rd, [k.clone() for k in Rd["k_cache"]],
                [v.clone() for v in Rd["v_cache"]])


def run_stages(c: Case, logits=True):
    R = c.Rd
    c.rd.prepare(R["prev_tokens"], R["prev_pos"], R["num_accepted"], R["bonus"])
    c.rd.scatter(R["target_hidden"])
    c.rd.forward(logits=logits)
    torch.cuda.synchronize()
    return int(c.rd.err.item())


def meta_np(c: Case) -> dict:
    return {k: v.cpu().numpy() for k, v in c.rd.meta.items()}


def to_np_storage(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> numpy in the workload's storage convention (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_round(c: Case, seqs=None, want_kv=False, n_threads=0):
    return oracle.run_round(c.cfg_np, c.w_np, c.r_np, n_threads=n_threads, seqs=seqs, want_kv=want_kv)


def check_logits(c: Case, ref: dict, seqs=None):
    """GPU debug logits and draft tokens of the given sequences against the oracle."""
    K = c.cfg_np.K
    seqs = list(range(c.cfg_np.B)) if seqs is None else list(seqs)
    rows = np.concatenate([np.arange(b * K, (b + 1) * K) for b in seqs])
    lg = c.rd.logits.cpu().numpy()[rows].astype(np.float64)
    err = np.abs(lg - ref["logits"]).max()
    tol = LOGIT_TOL[c.cfg_np.dtype]
    assert err <= tol, f"max |logit diff| {err:.3g} > {tol}"
    drafts = c.rd.draft_tokens.cpu().numpy().reshape(-1)[rows]
    sure = oracle.top2_gap(ref["logits"]) > GAP
    assert np.array_equal(drafts[sure], ref["drafts"].reshape(-1)[sure])
    # the argmax epilogue picks exactly the argmax of the logits it computed
    assert np.array_equal(drafts, np.argmax(c.rd.logits.cpu().numpy()[rows], axis=1))
    return err


def check_kv_writes(c: Case, ref: dict):
    """Cache entries at the valid rows' slots hold the oracle's post-RoPE k / v (storage rounding
    tolerance); every other entry is bit-identical to its value before the round."""
    cfg = c.cfg_np
    rows = ref["rows"]
    slots = ref["meta"]["slot_mapping"][rows]
    tol = KV_TOL[cfg.dtype]
    for l in range(cfg.n_layers):
        for name, after, before, new in (("k", c.kv.k_cache[l], c.k_before[l], ref["new_k"]),
                                         ("v", c.kv.v_cache[l], c.v_before[l], ref["new_v"])):
            a = oracle.widen(to_np_storage(after)).reshape(-1, cfg.n_kv * cfg.head_dim)
            b = to_np_storage(before).reshape(-1, cfg.n_kv * cfg.head_dim)
            got = a[slots]
            want = new[l]
            diff = np.abs(got - want) / np.maximum(1.0, np.abs(want))
            assert diff.max() <= tol, f"{name} cache layer {l}: rel diff {diff.max():.3g}"
            untouched = np.ones(a.shape[0], dtype=bool)
            untouched[slots] = False
            a_bits = to_np_storage(after).reshape(-1, cfg.n_kv * cfg.head_dim)
            assert np.array_equal(a_bits[untouched], b[untouched]), f"{name} cache layer {l}: stray write"
