"""Seeded synthetic workloads for one P-EAGLE parallel-drafting round.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It holds the five workload configurations and seeded generators of their
inputs: drafter weights, target hidden states, the previous round's verify
batch (tokens, positions, accepted count, bonus token), the paged KV prefix
and the block table.  It performs none of the method's arithmetic: only
random draws, rounding of stored values to bf16, and array layout.

Storage conventions (nn.Linear layout, ``[out][in]``):

* bf16 tensors are numpy ``uint16`` arrays holding the bf16 bit pattern;
  fp32 tensors are ``float32`` arrays.
* ``emb`` has ``vocab + 1`` rows; row ``vocab`` is the learned mask
  embedding emb(mask), so the MASK token id is ``vocab``.
* ``wqkv`` rows are the q heads, then the k heads, then the v heads, each
  head ``head_dim`` consecutive rows.
* ``w_gate_up`` rows are the ``ffn`` gate rows followed by the ``ffn`` up rows.
* The KV cache of each layer is ``[num_pages][page_size][n_kv][head_dim]``,
  K and V separate.

Value distributions follow the workload statements on the P-EAGLE pages'
benchmarks (GPT-OSS-20B and Qwen3-Coder-30B shaped drafters): linear and
embedding weights (emb(mask) and h_shared included) ~ N(0, 0.02), norm gains 1,
target hidden states ~ N(0, 1), token ids uniform over the vocabulary.
Prefix lengths for the high-concurrency workloads follow a lognormal with the
UltraChat sequence-length statistics (median 3891, p90 10800 tokens) quoted on
the pages, capped at 16384.  No public dataset item is reproduced.
"""

from __future__ import annotations

import dataclasses
import math
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "Config", "config", "sweep_config", "Weights", "RoundInputs",
    "make_weights", "make_round", "make_targets", "loop_round_draws", "bf16_to_f32", "f32_to_bf16",
    "LOGNORMAL_MEDIAN", "LOGNORMAL_SIGMA", "PREFIX_CAP",
]

# Sequence-length statistics of the pages' long-sequence discussion
# (GPT-OSS-120B on UltraChat: median 3891, p90 10800 tokens).
LOGNORMAL_MEDIAN = 3891.0
LOGNORMAL_SIGMA = math.log(10800.0 / 3891.0) / 1.2815515655446004  # z_0.90
PREFIX_CAP = 16384

_CHUNK = 1 << 22  # elements per independent random stream (fixed: results do not depend on threads)


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    B: int
    K: int
    n_layers: int
    d: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    dtype: str                 # "f32" or "bf16"
    prefix: str                # "fixed", "uniform", "lognormal"
    prefix_args: tuple
    accepted: str              # "fixed", "uniform", "uniform_20pct_zero"
    accepted_args: tuple = ()
    page_size: int = 16
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    seed: int = 0

    @property
    def rows(self) -> int:
        """Padded drafter rows: 2K per sequence (K+1 copy slots, K-1 MASK slots)."""
        return self.B * 2 * self.K

    @property
    def qkv_out(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


_GPT_OSS_20B_DRAFTER = dict(d=2880, n_q=64, n_kv=8, head_dim=64, ffn=7680, vocab=201088)


def config(i: int) -> Config:
    """The five workloads (index 0..3; index 4 is the K x B sweep, see sweep_config)."""
    if i == 0:
        return Config("tiny-f32-B1-K4", B=1, K=4, n_layers=1, d=256, n_q=4, n_kv=4, head_dim=64,
                      ffn=1024, vocab=4096, dtype="f32", prefix="fixed", prefix_args=(128,),
                      accepted="fixed", accepted_args=(2,), seed=0)
    if i == 1:
        return Config("qwen3-coder-30b-drafter-B8-K7", B=8, K=7, n_layers=1, d=2048, n_q=32,
                      n_kv=4, head_dim=128, ffn=6144, vocab=151936, dtype="bf16",
                      prefix="uniform", prefix_args=(512, 4096), accepted="uniform", seed=1)
    if i == 2:
        return Config("gpt-oss-20b-drafter-B1-K7", B=1, K=7, n_layers=1, dtype="bf16",
                      prefix="fixed", prefix_args=(3891,), accepted="uniform", seed=2,
                      **_GPT_OSS_20B_DRAFTER)
    if i == 3:
        return Config("gpt-oss-20b-drafter-B64-K7", B=64, K=7, n_layers=1, dtype="bf16",
                      prefix="lognormal", prefix_args=(LOGNORMAL_MEDIAN, LOGNORMAL_SIGMA, PREFIX_CAP),
                      accepted="uniform_20pct_zero", seed=3, **_GPT_OSS_20B_DRAFTER)
    if i == 4:
        return sweep_config(64, 7)
    raise ValueError(f"no workload {i}")


def sweep_config(B: int, K: int) -> Config:
    """The K x B sweep workload: the GPT-OSS-20B-shaped drafter with 2 layers."""
    return Config(f"gpt-oss-20b-drafter-L2-B{B}-K{K}", B=B, K=K, n_layers=2, dtype="bf16",
                  prefix="lognormal", prefix_args=(LOGNORMAL_MEDIAN, LOGNORMAL_SIGMA, PREFIX_CAP),
                  accepted="uniform", seed=4, **_GPT_OSS_20B_DRAFTER)


# ----------------------------------------------------------------------------- bf16 storage

def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u >> 16) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= 16
    return r.astype(np.uint16)


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- random draws

def _stream(seed: int, name: str, chunk: int) -> np.random.Generator:
    key = zlib.crc32(name.encode())
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(key, chunk))))


def _pool() -> ThreadPoolExecutor:
    return ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))


def _normal(seed: int, name: str, shape, std: float, dtype: str) -> np.ndarray:
    """N(0, std^2) draws stored in ``dtype``; chunked independent streams, filled in parallel."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        v = _stream(seed, name, c).standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[lo:hi] = f32_to_bf16(v) if dtype == "bf16" else v

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        fill(0) if n else None
    else:
        with _pool() as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def _ones(shape, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return np.full(shape, 0x3F80, dtype=np.uint16)
    return np.ones(shape, dtype=np.float32)


# ----------------------------------------------------------------------------- weights

@dataclasses.dataclass
class Weights:
    emb: np.ndarray            # [(V+1)][d]; row V = emb(mask)
    h_shared: np.ndarray       # [d]
    fc: np.ndarray             # [d][2d]
    norm_attn: list            # L x [d]
    wqkv: list                 # L x [(n_q+2n_kv)*hd][d]
    wo: list                   # L x [d][n_q*hd]
    norm_mlp: list             # L x [d]
    w_gate_up: list            # L x [2F][d]
    w_down: list               # L x [d][F]
    norm_final: np.ndarray     # [d]
    lm_head: np.ndarray        # [V][d]


def make_weights(cfg: Config, seed: int | None = None) -> Weights:
    s = cfg.seed if seed is None else seed
    dt, d = cfg.dtype, cfg.d
    std = 0.02
    L = cfg.n_layers
    return Weights(
        emb=_normal(s, "emb", (cfg.vocab + 1, d), std, dt),
        h_shared=_normal(s, "h_shared", (d,), std, dt),
        fc=_normal(s, "fc", (d, 2 * d), std, dt),
        norm_attn=[_ones((d,), dt) for _ in range(L)],
        wqkv=[_normal(s, f"wqkv{l}", (cfg.qkv_out, d), std, dt) for l in range(L)],
        wo=[_normal(s, f"wo{l}", (d, cfg.n_q * cfg.head_dim), std, dt) for l in range(L)],
        norm_mlp=[_ones((d,), dt) for _ in range(L)],
        w_gate_up=[_normal(s, f"wgu{l}", (2 * cfg.ffn, d), std, dt) for l in range(L)],
        w_down=[_normal(s, f"wdown{l}", (d, cfg.ffn), std, dt) for l in range(L)],
        norm_final=_ones((d,), dt),
        lm_head=_normal(s, "lm_head", (cfg.vocab, d), std, dt),
    )


# ----------------------------------------------------------------------------- one round's inputs

@dataclasses.dataclass
class RoundInputs:
    prev_tokens: np.ndarray    # [B][K+1] int32: previous verify batch [last, d1..dK]
    prev_pos: np.ndarray       # [B][K+1] int32: its positions P_b + j
    num_accepted: np.ndarray   # [B] int32: a_b in [0, K]
    bonus: np.ndarray          # [B] int32: target token at the first mismatch
    block_table: np.ndarray    # [B][max_pages] int32 physical page ids (-1 = unused)
    num_pages: int
    prefix_len: np.ndarray     # [B] int32: P_b (cache holds positions 0..P_b-1)
    target_hidden: np.ndarray  # [B*(K+1)][d]: target hidden state of each verify position
    k_cache: list              # L x [num_pages][page][n_kv][hd]
    v_cache: list
    target_u: np.ndarray       # [B][K] uniform draws for the synthetic target tokens
    target_r: np.ndarray       # [B][K+1] uniform token draws for the synthetic target tokens


def _prefix_lengths(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    if cfg.prefix == "fixed":
        return np.full(cfg.B, cfg.prefix_args[0], dtype=np.int32)
    if cfg.prefix == "uniform":
        lo, hi = cfg.prefix_args
        return rng.integers(lo, hi + 1, size=cfg.B).astype(np.int32)
    if cfg.prefix == "lognormal":
        med, sigma, cap = cfg.prefix_args
        v = np.exp(rng.normal(math.log(med), sigma, size=cfg.B))
        return np.clip(np.rint(v), 1, cap).astype(np.int32)
    raise ValueError(cfg.prefix)


def _accepted(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    if cfg.accepted == "fixed":
        return np.full(cfg.B, cfg.accepted_args[0], dtype=np.int32)
    if cfg.accepted == "uniform":
        return rng.integers(0, cfg.K + 1, size=cfg.B).astype(np.int32)
    if cfg.accepted == "uniform_20pct_zero":
        # exactly round(0.2*B) sequences fully rejected, the rest uniform in 1..K
        a = rng.integers(1, cfg.K + 1, size=cfg.B).astype(np.int32)
        zero = rng.permutation(cfg.B)[: int(round(0.2 * cfg.B))]
        a[zero] = 0
        return a
    raise ValueError(cfg.accepted)


def make_round(cfg: Config, seed: int | None = None, with_cache: bool = True,
               extra_positions: int = 0) -> RoundInputs:
    """Inputs of one drafting round.  The KV prefix is N(0,1) on every cache slot.
    ``extra_positions`` gives every sequence pages for that many more positions (rounds run
    back to back grow the prefix by up to K + 1 positions each)."""
    s = cfg.seed if seed is None else seed
    rng = _stream(s, "round-metadata", 0)
    B, K, ps = cfg.B, cfg.K, cfg.page_size
    P = _prefix_lengths(cfg, rng)
    a = _accepted(cfg, rng)
    prev_tokens = rng.integers(0, cfg.vocab, size=(B, K + 1)).astype(np.int32)
    prev_pos = (P[:, None] + np.arange(K + 1, dtype=np.int32)[None, :]).astype(np.int32)
    bonus = rng.integers(0, cfg.vocab, size=B).astype(np.int32)
    pages_per_seq = (P + 2 * K + extra_positions + ps - 1) // ps
    num_pages = int(pages_per_seq.sum())
    perm = rng.permutation(num_pages).astype(np.int32)
    max_pages = int(pages_per_seq.max())
    block_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(pages_per_seq[b])
        block_table[b, :n] = perm[off:off + n]
        off += n
    target_u = rng.random(size=(B, K))
    target_r = rng.integers(0, cfg.vocab, size=(B, K + 1)).astype(np.int32)
    hidden = _normal(s, "target_hidden", (B * (K + 1), cfg.d), 1.0, cfg.dtype)
    kshape = (num_pages, ps, cfg.n_kv, cfg.head_dim)
    if with_cache:
        kc = [_normal(s, f"kcache{l}", kshape, 1.0, cfg.dtype) for l in range(cfg.n_layers)]
        vc = [_normal(s, f"vcache{l}", kshape, 1.0, cfg.dtype) for l in range(cfg.n_layers)]
    else:
        kc, vc = [], []
    return RoundInputs(prev_tokens=prev_tokens, prev_pos=prev_pos, num_accepted=a, bonus=bonus,
                       block_table=block_table, num_pages=num_pages, prefix_len=P,
                       target_hidden=hidden, k_cache=kc, v_cache=vc,
                       target_u=target_u, target_r=target_r)


def loop_round_draws(cfg: Config, r: int, seed: int | None = None):
    """Fresh inputs of round r >= 1 of rounds run back to back: the target hidden states of
    the new verify batch ~ N(0, 1) and the target-token draws (uniforms and uniform tokens)
    that ``make_targets`` turns into that batch's target tokens."""
    s = cfg.seed if seed is None else seed
    rng = _stream(s, f"loop-round{r}", 0)
    target_u = rng.random(size=(cfg.B, cfg.K))
    target_r = rng.integers(0, cfg.vocab, size=(cfg.B, cfg.K + 1)).astype(np.int32)
    hidden = _normal(s, f"target_hidden/round{r}", (cfg.B * (cfg.K + 1), cfg.d), 1.0, cfg.dtype)
    return hidden, target_u, target_r


def make_targets(drafts: np.ndarray, u: np.ndarray, r: np.ndarray, p_match: float = 0.6) -> np.ndarray:
    """Synthetic target tokens for a verify batch: each of the first K equals the draft with
    probability p_match, else a uniform token; the last one is uniform."""
    drafts = np.asarray(drafts, dtype=np.int32)
    B, K = drafts.shape
    t = r.astype(np.int32).copy()
    t[:, :K] = np.where(u < p_match, drafts, r[:, :K])
    return t
