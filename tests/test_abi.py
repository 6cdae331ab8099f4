"""The C-ABI library loads, exports every symbol include/pe.h declares, and validates
arguments on the host (no GPU needed: nothing here launches a kernel)."""

import ctypes
import os
import re

import pytest

import speculative_decoding_step_gb300 as pe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pe_[a-z_]+)\s*\(", src)))


def test_header_declares_the_five_stage_calls():
    names = _declared_functions()
    for n in ["pe_prepare_batch", "pe_scatter_hidden", "pe_draft_forward", "pe_verify", "pe_step"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    L = pe.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name
    assert set(_declared_functions()) == set(pe.EXPORTED_SYMBOLS)


def _cfg(**kw):
    base = dict(B=8, K=7, d=2048, n_q=32, n_kv=4, head_dim=128, ffn=6144, vocab=151936, n_layers=1,
                max_pages_per_seq=257, dtype="bf16")
    base.update(kw)
    return pe.Config.make(**base)


def test_config_validation_codes():
    assert pe.check_config(_cfg()) == pe.PE_OK
    assert pe.check_config(_cfg(B=0)) == 2
    assert pe.check_config(_cfg(n_q=30, n_kv=4)) == 2          # n_kv must divide n_q
    assert pe.check_config(_cfg(head_dim=96)) == 3
    assert pe.check_config(_cfg(page_size=32)) == 3
    assert pe.check_config(_cfg(K=9, n_q=64, n_kv=8)) == 3     # 2K * (n_q/n_kv) > 128 query rows
    assert pe.check_config(_cfg(d=2052)) == 3                  # bf16 rows must be 16-byte multiples
    assert pe.check_config(_cfg(dtype="f32", d=2050)) == 3     # fp32 rows too
    assert pe.check_config(_cfg(dtype="f32", d=2048)) == pe.PE_OK
    assert pe.check_config(_cfg(d=2080)) == 3                  # bf16 contractions tile in 64-wide k atoms
    assert pe.check_config(_cfg(ffn=6176)) == 3
    assert pe.check_config(_cfg(dtype="f32", d=2080, ffn=6176)) == pe.PE_OK
    assert pe.check_config(_cfg(d=10240)) == pe.PE_OK
    assert pe.check_config(_cfg(d=10304)) == 3                 # input rows staged in shared memory
    assert pe.check_config(_cfg(dtype="f32", d=5184)) == 3
    assert pe.status_str(0) == "ok"


def test_workspace_bytes_grow_with_batch():
    small = pe.workspace_bytes(_cfg(B=1))
    big = pe.workspace_bytes(_cfg(B=64, K=7, n_q=64, n_kv=8))
    assert 0 < small < big
    assert pe.workspace_bytes(_cfg(B=0)) == 0
    assert pe.trace_points(_cfg(n_layers=2)) == 8 + 14


def test_null_pointers_rejected_before_launch():
    L = pe.lib()
    cfg = _cfg()
    null = ctypes.c_void_p(None)
    st = L.pe_prepare_batch(ctypes.byref(cfg), null, null, null, null, null, 10, *([null] * 11))
    assert st == 1
    st = L.pe_verify(ctypes.byref(cfg), null, null, null, null, null)
    assert st == 1
    assert L.pe_set_trace_events(None, -1) == 1


def test_sampling_calls_validate_before_launch():
    """The non-greedy drafting and verification calls reject null pointers and a temperature
    that is not positive and finite, before anything is launched."""
    L = pe.lib()
    cfg = _cfg()
    null = ctypes.c_void_p(None)
    some = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    st = L.pe_sample_drafts(ctypes.byref(cfg), null, null, ctypes.c_float(1.0), null, 0, null, null, null, null)
    assert st == 1
    for T in (0.0, -1.0, float("inf"), float("nan")):
        st = L.pe_sample_drafts(ctypes.byref(cfg), some, some, ctypes.c_float(T), some, 1 << 30, some, some, some,
                                null)
        assert st == 1, T
        st = L.pe_verify_sampled(ctypes.byref(cfg), some, some, some, ctypes.c_float(T), some, some, some, some,
                                 1 << 30, some, some, some, null)
        assert st == 1, T
    st = L.pe_verify_sampled(ctypes.byref(cfg), null, null, null, ctypes.c_float(1.0), null, null, null, null, 0,
                             null, null, null, null)
    assert st == 1


def test_step_rejects_overlapping_outputs_before_launch():
    """pe_step: a state output may be exactly its paired input (rounds back to back in
    place); any other overlap of an output with an input or another output is rejected
    before anything is launched.  Every call here stops at a host check (the workspace size
    is zero): the pointers are placeholders that are never dereferenced."""
    L = pe.lib()
    cfg = _cfg(B=2, K=3)
    B, K = 2, 3
    base = 1 << 40
    nxt = iter(range(base, base + (1 << 36), 1 << 20))  # disjoint 1 MiB-spaced placeholders
    P = lambda: next(nxt)
    layer = (ctypes.c_void_p * cfg.n_layers)(*[P() for _ in range(cfg.n_layers)])
    w = pe._Weights(P(), P(), P(), layer, layer, layer, layer, layer, layer, P(), P())
    kv = pe._KV(layer, layer, 4)
    ins = dict(block_table=P(), prev_tokens=P(), prev_pos=P(), num_accepted=P(), bonus=P(), target_hidden=P(),
               target_tokens=P())
    outs = dict(draft_tokens=P(), num_accepted_out=P(), bonus_out=P(), next_prev_tokens=P(), next_prev_pos=P())
    ws, err = P(), P()

    def call(ws=ws, ws_bytes=0, err=err, **over):
        a = {**ins, **outs, **over}
        v = lambda k: ctypes.c_void_p(a[k])
        return L.pe_step(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(kv), v("block_table"), v("prev_tokens"),
                         v("prev_pos"), v("num_accepted"), v("bonus"), v("target_hidden"), v("target_tokens"),
                         ctypes.c_void_p(ws), ctypes.c_size_t(ws_bytes), v("draft_tokens"), v("num_accepted_out"),
                         v("bonus_out"), v("next_prev_tokens"), v("next_prev_pos"), ctypes.c_void_p(None),
                         ctypes.c_void_p(err), ctypes.c_void_p(None))

    # control: disjoint buffers, and the state updated exactly in place, pass every argument
    # check and stop at the (deliberately empty) workspace: PE_ERR_SHAPE, still no launch
    assert call() == 2
    assert call(next_prev_tokens=ins["prev_tokens"], next_prev_pos=ins["prev_pos"],
                num_accepted_out=ins["num_accepted"], bonus_out=ins["bonus"]) == 2
    # a state output shifted by one element into its paired input
    assert call(next_prev_tokens=ins["prev_tokens"] + 4) == 1
    # a state output equal to another input than its pair
    assert call(next_prev_pos=ins["prev_tokens"]) == 1
    assert call(bonus_out=ins["num_accepted"]) == 1
    # the drafts written over the target tokens, or over another output
    assert call(draft_tokens=ins["target_tokens"]) == 1
    assert call(draft_tokens=outs["next_prev_tokens"] + 4 * (K + 1) * B - 4) == 1
    # a block table running into the next verify batch
    assert call(next_prev_pos=ins["block_table"] + 4) == 1
    # the error word inside an output or an input
    assert call(err=outs["draft_tokens"] + 4) == 1
    assert call(err=ins["target_tokens"]) == 1
    # a workspace (of sufficient size) that runs into an input or holds the error word: only the
    # rejected calls get a usable size, so no call here reaches a launch
    need = pe.workspace_bytes(cfg)
    assert need > 0
    assert call(ws=ins["target_hidden"] - 256, ws_bytes=need) == 1
    assert call(ws=err - 4096 // 256 * 256, ws_bytes=need) == 1


def test_wait_limit_and_stage_hook_host_checks():
    """The wait limit and the wait-expiry test hook are host settings: no launch, no GPU."""
    L = pe.lib()
    assert L.pe_test_skip_pipeline_stage(-2) == 1
    assert L.pe_test_skip_pipeline_stage(-1) == 0
    assert L.pe_set_wait_limit_ns(1000) == 0
    assert L.pe_set_wait_limit_ns(0) == 0


def test_inject_kv_host_checks():
    """pe_inject_kv rejects null or misaligned pointers and a short workspace before any launch
    (placeholder pointers, never dereferenced)."""
    L = pe.lib()
    cfg = _cfg(B=2, K=3)
    P = iter(range(1 << 40, (1 << 40) + (1 << 30), 1 << 20))
    layer = (ctypes.c_void_p * cfg.n_layers)(*[next(P) for _ in range(cfg.n_layers)])
    w = pe._Weights(next(P), next(P), next(P), layer, layer, layer, layer, layer, layer, next(P), next(P))
    kv = pe._KV(layer, layer, 4)
    v = lambda: ctypes.c_void_p(next(P))

    def call(w_inj=None, ws_bytes=0, hidden=None):
        return L.pe_inject_kv(ctypes.byref(cfg), ctypes.byref(w), w_inj if w_inj is not None else v(),
                              ctypes.byref(kv), v(), v(), v(), hidden if hidden is not None else v(), v(),
                              ctypes.c_size_t(ws_bytes), v(), ctypes.c_void_p(None))

    assert call(w_inj=ctypes.c_void_p(None)) == 1          # null projection
    assert call(hidden=ctypes.c_void_p((1 << 41) + 8)) == 1  # misaligned hidden states
    assert call(ws_bytes=16) == 2                          # workspace too short: PE_ERR_SHAPE
