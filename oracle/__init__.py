"""CPU oracle for one P-EAGLE parallel-drafting round.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  It shares no code
with the CUDA path (``speculative_decoding_step_gb300``) and never imports it.

Sources (the three P-EAGLE web pages; cited by title and section):

* P-EAGLE: Parallel Speculative Decoding in vLLM (agentlenshq), "P-EAGLE
  architecture and mechanism", step 2 "Parallel Drafting" -- how the input of
  every draft position is built; "vLLM implementation details" -- the fused
  batch-metadata kernel, the hidden-state copy kernel, PADDING_SLOT_ID = -1.
* vLLM Speculators: parallel drafting for speculative decoding (agentlenshq),
  closing paragraph of "Production integration in vLLM" -- verification keeps
  the target's output distribution; its greedy form is the longest matching
  prefix plus the target's token at the first mismatch.

Functions (each a plain restatement; pure Python loops where sizes are small):

* ``prepare_batch``  (R1) batch rebuild: tokens, positions, slot mapping,
  rejected / MASK masks, hidden-state map, compacted valid rows, draft rows.
* ``scatter_hidden`` (R2) drafter input rows concat(emb(token), hidden).
* ``draft_forward``  (R3) drafter pass + LM head, fp64, in ``pe_oracle.c``.
* ``verify``         (R4) greedy verification.
* ``next_verify_batch`` the verify batch the target checks after a round (the
  next round's previous batch): the bonus token, then the K drafts.
* ``inject_kv`` (R6) the DFlash-style variant: the verifier's hidden states
  projected into the drafter's KV cache (vLLM Speculators: parallel drafting
  for speculative decoding, "DFlash").
* ``inverse_cdf``, ``drafter_distribution``, ``sample_drafts``,
  ``verify_sampled`` (R5) non-greedy drafting and verification by rejection
  sampling (speculative sampling): drafts drawn from the drafter's
  temperature softmax, each accepted with probability min(1, p/q), the first
  rejected one replaced by a draw from the normalised residual max(0, p - q),
  a bonus drawn from the target when every draft is accepted.  The pages
  state only that verification uses rejection sampling to keep the target's
  output distribution; the steps are the standard speculative-sampling
  scheme that does so.

Parity status: the pages print no numeric example, so every function is
pinned by closed forms, brute force and invariants in the tests rather than by
printed values ("parity unpinned" by the pages themselves).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libpe_oracle.so")
_lib = None

PADDING_SLOT_ID = -1
PAD_TOKEN = 0


# ----------------------------------------------------------------------------- build / load

SOURCE = os.path.join(_HERE, "pe_oracle.c")


def compile_source(src: str, out: str) -> str:
    """Compile a C oracle source to a shared library with gcc (IEEE semantics, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", "-pthread", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C part of the oracle (``pe_oracle.c``) in-tree."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("d", ctypes.c_int32), ("n_q", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("storage", ctypes.c_int32), ("rms_eps", ctypes.c_double),
                ("rope_theta", ctypes.c_double), ("n_threads", ctypes.c_int32)]


class _W(ctypes.Structure):
    _fields_ = [("fc", ctypes.c_void_p), ("norm_final", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("norm_attn", ctypes.POINTER(ctypes.c_void_p)), ("wqkv", ctypes.POINTER(ctypes.c_void_p)),
                ("wo", ctypes.POINTER(ctypes.c_void_p)), ("norm_mlp", ctypes.POINTER(ctypes.c_void_p)),
                ("w_gate_up", ctypes.POINTER(ctypes.c_void_p)), ("w_down", ctypes.POINTER(ctypes.c_void_p))]


def load_library(path: str):
    """Load a compiled copy of ``pe_oracle.c`` and declare its functions' signatures."""
    L = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    L.oc_linear.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, dp]
    L.oc_rmsnorm.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_double, dp]
    L.oc_rope.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_double]
    L.oc_silu.argtypes = [ctypes.c_double]
    L.oc_silu.restype = ctypes.c_double
    L.oc_attend.argtypes = [dp, dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_double, dp]
    L.oc_forward.restype = ctypes.c_int
    L.oc_threads_used.restype = ctypes.c_int
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _dptr(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _storage(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    raise TypeError(f"storage dtype {a.dtype}")


def widen(a: np.ndarray) -> np.ndarray:
    """Exact float64 value of a float32 or bf16 (uint16 bit pattern) array."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ----------------------------------------------------------------------------- single ops (exported for pin tests)

def linear(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    X = np.ascontiguousarray(X, dtype=np.float64)
    W = np.ascontiguousarray(W)
    n, k = X.shape
    Y = np.zeros((n, W.shape[0]), dtype=np.float64)
    lib().oc_linear(_dptr(X), n, k, W.ctypes.data, W.shape[0], _storage(W), _dptr(Y))
    return Y


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    g = np.ascontiguousarray(g)
    y = np.zeros_like(x)
    lib().oc_rmsnorm(_dptr(x), x.shape[0], x.shape[1], g.ctypes.data, _storage(g), eps, _dptr(y))
    return y


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64)
    lib().oc_rope(_dptr(v), v.shape[0], int(pos), float(theta))
    return v


def silu(x: float) -> float:
    return lib().oc_silu(float(x))


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    out = np.zeros(q.shape[0], dtype=np.float64)
    lib().oc_attend(_dptr(q), _dptr(K), _dptr(V), K.shape[0], q.shape[0], scale, _dptr(out))
    return out


# ----------------------------------------------------------------------------- R1: batch rebuild

def prepare_batch(K: int, vocab: int, prev_tokens, prev_pos, num_accepted, bonus, block_table,
                  page_size: int = 16) -> dict:
    """Rebuild the drafter batch from the previous verify batch in one pass.

    The previous verify batch of sequence b is [last, d_1..d_K] at positions
    P..P+K; a_b drafts were accepted and the target produced ``bonus``.  Each
    sequence gets 2K rows: K+1 copy slots in verify order, then K-1 MASK
    slots.  Copy slot r:

    * r < a  : accepted context row -- token at position P+r+1 paired with the
      target hidden state of position P+r (shifted by one);
    * r == a : the next-token-prediction row -- the bonus token with the
      hidden state that produced it (h_context);
    * r > a  : rejected -- PAD token, PADDING_SLOT_ID, excluded from the pass.

    MASK slot m = 1..K-1 (row K+m): the MASK token id (= vocab), position
    P+a+m, hidden state h_shared (hidden_map -1).  Drafts t_1..t_K come from
    the NTP row and then the MASK rows in order.
    """
    prev_tokens = np.asarray(prev_tokens, dtype=np.int64)
    prev_pos = np.asarray(prev_pos, dtype=np.int64)
    B = prev_tokens.shape[0]
    S = 2 * K
    MASK_ID = vocab
    n = B * S
    out = dict(
        input_ids=np.zeros(n, np.int32), positions=np.zeros(n, np.int32),
        slot_mapping=np.full(n, PADDING_SLOT_ID, np.int64), is_rejected=np.zeros(n, np.uint8),
        is_mask=np.zeros(n, np.uint8), hidden_map=np.full(n, -1, np.int32),
    )

    def slot(b, p):
        return int(block_table[b][p // page_size]) * page_size + p % page_size

    for b in range(B):
        a = int(num_accepted[b])
        for r in range(S):
            row = b * S + r
            if r < a:                       # accepted context row
                tok, pos, hm, sl, rej, msk = prev_tokens[b][r + 1], prev_pos[b][r], b * (K + 1) + r, None, 0, 0
            elif r == a:                    # NTP row: bonus token with h_context
                tok, pos, hm, sl, rej, msk = bonus[b], prev_pos[b][a], b * (K + 1) + a, None, 0, 0
            elif r <= K:                    # rejected draft position: no cache write
                tok, pos, hm, sl, rej, msk = PAD_TOKEN, prev_pos[b][r], b * (K + 1) + r, PADDING_SLOT_ID, 1, 0
            else:                           # MASK row m = r - K
                m = r - K
                tok, pos, hm, sl, rej, msk = MASK_ID, prev_pos[b][a] + m, -1, None, 0, 1
            out["input_ids"][row] = tok
            out["positions"][row] = pos
            out["hidden_map"][row] = hm
            out["slot_mapping"][row] = slot(b, int(pos)) if sl is None else sl
            out["is_rejected"][row] = rej
            out["is_mask"][row] = msk
    valid = [row for row in range(n) if not out["is_rejected"][row]]
    out["row_list"] = np.array(valid, dtype=np.int32)
    out["n_valid"] = len(valid)
    compact = {row: i for i, row in enumerate(valid)}
    draft = []
    for b in range(B):
        a = int(num_accepted[b])
        draft.append(compact[b * S + a])
        for m in range(1, K):
            draft.append(compact[b * S + K + m])
    out["draft_rows"] = np.array(draft, dtype=np.int32)
    return out


# ----------------------------------------------------------------------------- R2: input rows

def scatter_hidden(emb, h_shared, target_hidden, input_ids, is_mask, hidden_map) -> np.ndarray:
    """Drafter input of every padded row: concat(emb[token], hidden) with the embedding first;
    the hidden part is h_shared on MASK rows and the mapped target hidden state elsewhere.
    Returned in the storage dtype (a pure copy)."""
    n = len(input_ids)
    d = emb.shape[1]
    x0 = np.zeros((n, 2 * d), dtype=emb.dtype)
    for row in range(n):
        x0[row, :d] = emb[input_ids[row]]
        x0[row, d:] = h_shared if is_mask[row] else target_hidden[hidden_map[row]]
    return x0


# ----------------------------------------------------------------------------- R3: drafter pass

def draft_forward(cfg, weights, x0_rows, positions, slots, seqs, block_table, k_cache, v_cache,
                  draft_rows, n_threads: int = 0, want_kv: bool = False, want_x: bool = False) -> dict:
    """Run the fp64 drafter pass over the given rows (see ``pe_oracle.c``).

    ``x0_rows`` [n][2d] (storage dtype or float64), ``positions``/``slots``/``seqs`` per row,
    ``draft_rows`` indices into these rows.  Returns logits [n_draft][V] (float64) and,
    on request, the post-RoPE k/v of every row and the final residual stream.
    """
    L = lib()
    x0 = widen(np.asarray(x0_rows)) if np.asarray(x0_rows).dtype != np.float64 else np.ascontiguousarray(x0_rows)
    x0 = np.ascontiguousarray(x0)
    n = x0.shape[0]
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    c = _Cfg(n_rows=n, d=cfg.d, n_q=cfg.n_q, n_kv=cfg.n_kv, head_dim=cfg.head_dim, ffn=cfg.ffn,
             vocab=cfg.vocab, n_layers=cfg.n_layers, page_size=cfg.page_size, max_pages=bt.shape[1],
             storage=_storage(weights.lm_head), rms_eps=cfg.rms_eps, rope_theta=cfg.rope_theta,
             n_threads=n_threads)
    Lc = cfg.n_layers
    arr = lambda xs: (ctypes.c_void_p * max(Lc, 1))(*[np.ascontiguousarray(x).ctypes.data for x in list(xs)[:Lc]])
    keep = [weights.norm_attn, weights.wqkv, weights.wo, weights.norm_mlp, weights.w_gate_up, weights.w_down]
    for group in keep:
        for x in group:
            assert x.flags.c_contiguous
    w = _W(fc=weights.fc.ctypes.data, norm_final=weights.norm_final.ctypes.data,
           lm_head=weights.lm_head.ctypes.data, norm_attn=arr(weights.norm_attn), wqkv=arr(weights.wqkv),
           wo=arr(weights.wo), norm_mlp=arr(weights.norm_mlp), w_gate_up=arr(weights.w_gate_up),
           w_down=arr(weights.w_down))
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    sq = np.ascontiguousarray(seqs, dtype=np.int32)
    dr = np.ascontiguousarray(draft_rows, dtype=np.int32)
    for kc in list(k_cache) + list(v_cache):
        assert kc.flags.c_contiguous
    kp = (ctypes.c_void_p * max(Lc, 1))(*[x.ctypes.data for x in list(k_cache)[:Lc]])
    vp = (ctypes.c_void_p * max(Lc, 1))(*[x.ctypes.data for x in list(v_cache)[:Lc]])
    logits = np.zeros((len(dr), cfg.vocab), dtype=np.float64)
    kvd = cfg.n_kv * cfg.head_dim
    nk = np.zeros((Lc, n, kvd)) if want_kv else None
    nv = np.zeros((Lc, n, kvd)) if want_kv else None
    xo = np.zeros((n, cfg.d)) if want_x else None
    P = lambda a: a.ctypes.data if a is not None else None
    rc = L.oc_forward(ctypes.byref(c), ctypes.byref(w), ctypes.c_void_p(x0.ctypes.data),
                      ctypes.c_void_p(pos.ctypes.data), ctypes.c_void_p(sl.ctypes.data),
                      ctypes.c_void_p(sq.ctypes.data), ctypes.c_void_p(bt.ctypes.data), kp, vp,
                      ctypes.c_int32(len(dr)), ctypes.c_void_p(dr.ctypes.data),
                      ctypes.c_void_p(logits.ctypes.data), ctypes.c_void_p(P(nk)), ctypes.c_void_p(P(nv)),
                      ctypes.c_void_p(P(xo)))
    if rc != 0:
        raise ValueError("oracle: a row's causal range leaves its block table")
    return dict(logits=logits, new_k=nk, new_v=nv, x=xo)


def threads_used() -> int:
    return int(lib().oc_threads_used())


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Index of the largest logit per row; the lowest index wins a tie."""
    return np.argmax(logits, axis=-1).astype(np.int32)


def top2_gap(logits: np.ndarray) -> np.ndarray:
    part = np.partition(logits, -2, axis=-1)
    return part[..., -1] - part[..., -2]


# ----------------------------------------------------------------------------- R4: verify

def verify(draft_tokens, target_tokens) -> tuple[np.ndarray, np.ndarray]:
    """Greedy verification: a = the length of the longest prefix of drafts equal to the target's
    tokens; bonus = the target's token at the first mismatch (target[a], the K+1-th when all match)."""
    draft_tokens = np.asarray(draft_tokens)
    target_tokens = np.asarray(target_tokens)
    B, K = draft_tokens.shape
    acc = np.zeros(B, np.int32)
    bon = np.zeros(B, np.int32)
    for b in range(B):
        a = 0
        while a < K and draft_tokens[b][a] == target_tokens[b][a]:
            a += 1
        acc[b] = a
        bon[b] = target_tokens[b][a]
    return acc, bon


def next_verify_batch(prev_pos, num_accepted, bonus, drafts) -> tuple[np.ndarray, np.ndarray]:
    """The verify batch after a round: sequence b's NTP row sat at position prev_pos[b][a]
    (a = its accepted count) and carried the bonus token, which belongs one position further
    on; the target then checks [bonus, t_1..t_K] at consecutive positions from there.  This
    batch is what the next round's rebuild copies token ids and positions from (P-EAGLE
    pages, "vLLM implementation details", fused batch-metadata kernel)."""
    drafts = np.asarray(drafts, dtype=np.int32)
    B, K = drafts.shape
    tokens = np.zeros((B, K + 1), np.int32)
    positions = np.zeros((B, K + 1), np.int32)
    for b in range(B):
        p0 = int(prev_pos[b][int(num_accepted[b])]) + 1
        tokens[b][0] = bonus[b]
        for k in range(K):
            tokens[b][k + 1] = drafts[b][k]
        for j in range(K + 1):
            positions[b][j] = p0 + j
    return tokens, positions


# ----------------------------------------------------------------------------- R6: DFlash-style KV injection
# vLLM Speculators: parallel drafting for speculative decoding, "DFlash": the verifier's
# hidden states are projected and injected straight into the drafter's KV cache, so the
# drafter attends to the verifier's state without extra input rows.  The page gives that
# one sentence; the reading here: the projected state x = W_inj h stands where a row's
# residual stream would, so each layer turns it into k and v exactly as it does for its
# own rows (attention RMSNorm, the k and v blocks of W_qkv, RoPE on k at the position),
# and writes them at the position's cache slot.

def inject_kv(cfg, weights, w_inj, target_hidden, prev_pos, num_accepted, block_table, page_size: int = 16) -> dict:
    """KV entries injected from the verifier's hidden states of the previous verify batch.

    Sequence b, verify element j <= num_accepted[b] (the accepted drafts' positions and the
    bonus token's position; rejected ones are not written): h = target_hidden[b*(K+1) + j],
    p = prev_pos[b][j], x = W_inj h (W_inj [d][d], no bias); per layer l:
    y = rms(x) * g_attn[l], k = RoPE(W_k[l] y, p), v = W_v[l] y.
    Returns slots [n] (int64, the written cache slots in (b, j) order) and new_k / new_v
    [L][n][n_kv * head_dim] (float64, post-RoPE k)."""
    K = cfg.K
    B = len(num_accepted)
    hd, nq, nkv = cfg.head_dim, cfg.n_q, cfg.n_kv
    H = widen(np.asarray(target_hidden))
    rows, slots, pos = [], [], []
    for b in range(B):
        for j in range(int(num_accepted[b]) + 1):
            p = int(prev_pos[b][j])
            rows.append(b * (K + 1) + j)
            pos.append(p)
            slots.append(int(block_table[b][p // page_size]) * page_size + p % page_size)
    X = linear(H[rows], np.asarray(w_inj))
    L = cfg.n_layers
    new_k = np.zeros((L, len(rows), nkv * hd))
    new_v = np.zeros((L, len(rows), nkv * hd))
    for l in range(L):
        Y = rmsnorm(X, weights.norm_attn[l], cfg.rms_eps)
        wkv = np.asarray(weights.wqkv[l])[nq * hd:]            # the k heads, then the v heads
        KV = linear(Y, wkv)
        for i in range(len(rows)):
            for g in range(nkv):
                new_k[l, i, g * hd:(g + 1) * hd] = rope(KV[i, g * hd:(g + 1) * hd], pos[i], cfg.rope_theta)
            new_v[l, i] = KV[i, nkv * hd:]
    return dict(slots=np.array(slots, dtype=np.int64), rows=np.array(rows, dtype=np.int32), new_k=new_k,
                new_v=new_v, positions=np.array(pos, dtype=np.int32))


# ----------------------------------------------------------------------------- R5: sampled drafting and verification
# vLLM Speculators: parallel drafting for speculative decoding, closing paragraph of
# "Production integration in vLLM": verification by rejection sampling keeps the target
# model's output distribution.  Every random number is an input (one uniform in [0, 1)
# per draw), so both sides draw the same sample.

def inverse_cdf(w, u: float) -> int:
    """One draw from the non-negative weights ``w`` (not all zero) with the uniform ``u``:
    the smallest index whose running sum of weights exceeds u times the total.  A
    zero-weight index is never drawn."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    v = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(v, len(c) - 1)


def drafter_distribution(logits_row, temperature: float) -> tuple[np.ndarray, float]:
    """The drafter's distribution q = softmax(logits / temperature) and its natural-log
    normaliser lse (q[v] = exp(logits[v] / temperature - lse))."""
    z = np.asarray(logits_row, dtype=np.float64) / temperature
    m = z.max()
    e = np.exp(z - m)
    tot = e.sum()
    return e / tot, float(m + np.log(tot))


def sample_drafts(logits, u_draft, temperature: float) -> tuple[np.ndarray, np.ndarray]:
    """Non-greedy drafting: draft row (b, k) (logits row b*K + k) draws its token from its own
    q with the uniform u_draft[b][k].  Returns the drafts [B][K] and each row's lse [B][K]."""
    u_draft = np.asarray(u_draft, dtype=np.float64)
    B, K = u_draft.shape
    lg = np.asarray(logits).reshape(B * K, -1)
    drafts = np.zeros((B, K), np.int32)
    lse = np.zeros((B, K))
    for b in range(B):
        for k in range(K):
            q, lse[b][k] = drafter_distribution(lg[b * K + k], temperature)
            drafts[b][k] = inverse_cdf(q, u_draft[b][k])
    return drafts, lse


def verify_sampled(drafts, logits, temperature: float, target_probs, u_accept, u_resample):
    """Rejection-sampling verification of sequence b's drafts t_1..t_K (``drafts[b]``).

    target_probs[b][k] is the target's distribution p_k for the position of draft k
    (after the verify batch's element k; p_K follows the last draft), q_k the drafter's
    distribution of draft row k.  For k = 0, 1, ...: draft x = drafts[b][k] is accepted
    when u_accept[b][k] * q_k(x) < p_k(x) (probability min(1, p_k(x) / q_k(x))).  At the
    first rejection the accepted count is k and the bonus token is drawn with
    u_resample[b] from max(0, p_k - q_k) (from p_k itself if that residual is all zero);
    when all K are accepted the bonus is drawn from p_K.  Returns (accepted, bonus)."""
    drafts = np.asarray(drafts)
    B, K = drafts.shape
    lg = np.asarray(logits).reshape(B * K, -1)
    P = np.asarray(target_probs, dtype=np.float64)
    acc = np.zeros(B, np.int32)
    bonus = np.zeros(B, np.int32)
    for b in range(B):
        a = K
        for k in range(K):
            q, _ = drafter_distribution(lg[b * K + k], temperature)
            x = int(drafts[b][k])
            if not (u_accept[b][k] * q[x] < P[b][k][x]):
                a = k
                break
        acc[b] = a
        if a < K:
            q, _ = drafter_distribution(lg[b * K + a], temperature)
            res = np.maximum(0.0, P[b][a] - q)
            bonus[b] = inverse_cdf(res if res.sum() > 0 else P[b][a], u_resample[b])
        else:
            bonus[b] = inverse_cdf(P[b][K], u_resample[b])
    return acc, bonus


# ----------------------------------------------------------------------------- composition

def round_rows(cfg, meta: dict, rows=None):
    """Per-row positions / slots / sequence ids for the compacted valid rows (or the given rows)."""
    rows = meta["row_list"] if rows is None else np.asarray(rows)
    S = 2 * cfg.K
    return (meta["positions"][rows], meta["slot_mapping"][rows], (rows // S).astype(np.int32))


def run_round(cfg, weights, rnd, n_threads: int = 0, seqs=None, want_kv=False) -> dict:
    """R1 -> R2 -> R3 -> draft tokens for one round.  ``seqs`` restricts the pass to a subset of
    sequences (they are independent: separate rows, pages and verification)."""
    meta = prepare_batch(cfg.K, cfg.vocab, rnd.prev_tokens, rnd.prev_pos, rnd.num_accepted, rnd.bonus,
                         rnd.block_table, cfg.page_size)
    w = weights
    x0 = scatter_hidden(w.emb, w.h_shared, rnd.target_hidden, meta["input_ids"], meta["is_mask"],
                        meta["hidden_map"])
    S = 2 * cfg.K
    rows = meta["row_list"]
    if seqs is not None:
        keep = np.isin(rows // S, np.asarray(seqs))
        rows = rows[keep]
    pos, sl, sq = round_rows(cfg, meta, rows)
    # draft rows of the kept sequences, in (b, k) order, as indices into `rows`
    idx = {int(r): i for i, r in enumerate(rows)}
    seq_list = range(cfg.B) if seqs is None else list(seqs)
    draft_padded = []
    for b in seq_list:
        a = int(rnd.num_accepted[b])
        draft_padded.append(b * S + a)
        draft_padded += [b * S + cfg.K + m for m in range(1, cfg.K)]
    dr = np.array([idx[r] for r in draft_padded], dtype=np.int32)
    res = draft_forward(cfg, w, x0[rows], pos, sl, sq, rnd.block_table, rnd.k_cache, rnd.v_cache, dr,
                        n_threads=n_threads, want_kv=want_kv)
    res["meta"] = meta
    res["rows"] = rows
    res["x0"] = x0
    res["drafts"] = argmax_lowest(res["logits"]).reshape(len(seq_list), cfg.K)
    return res
