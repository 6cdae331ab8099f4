"""P-EAGLE parallel-drafting round on one GB300: Python binding of the C ABI.

Thin ctypes marshalling over ``libpe.so`` (``include/pe.h``): every entry point
takes torch CUDA tensors (PyTorch supplies device memory and streams only) and
passes their device pointers and sizes to the library.  All computation runs in
the library's CUDA kernels.  Loading fails loudly when the library has not been
built; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB, build

__all__ = [
    "PeError", "Config", "DeviceWeights", "DeviceKV", "lib", "build", "check_config", "workspace_bytes",
    "prepare_batch", "scatter_hidden", "draft_forward", "verify", "step", "status_str",
    "PE_OK", "PE_DEV_BAD_TOKEN", "PE_DEV_BAD_ACCEPTED", "PE_DEV_BAD_PAGE", "PE_DEV_BAD_POSITION",
    "PE_DEV_NONFINITE", "PE_DEV_BAD_ROW", "PE_DEV_TIMEOUT", "EXPORTED_SYMBOLS",
]

PE_OK = 0
PE_F32, PE_BF16 = 0, 1
PE_DEV_BAD_TOKEN = 0x0105
PE_DEV_BAD_ACCEPTED = 0x0205
PE_DEV_BAD_PAGE = 0x0305
PE_DEV_BAD_POSITION = 0x0405
PE_DEV_NONFINITE = 0x0505
PE_DEV_BAD_ROW = 0x0605
PE_DEV_TIMEOUT = 0x0106

EXPORTED_SYMBOLS = ["pe_prepare_batch", "pe_scatter_hidden", "pe_draft_forward", "pe_verify", "pe_step",
                    "pe_sample_drafts", "pe_verify_sampled",
                    "pe_workspace_bytes", "pe_check_config", "pe_status_str", "pe_set_trace_events",
                    "pe_trace_points", "pe_kernel_launches", "pe_draft_forward_noalloc", "pe_set_wait_limit_ns",
                    "pe_test_skip_pipeline_stage", "pe_inject_kv"]

# Size of the library-owned scratch used by pe_draft_forward_noalloc (PE_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 48 << 20


class PeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({status_str(status)})")
        self.status = status


class Config(ctypes.Structure):
    """pe_config (host struct)."""
    _fields_ = [("B", ctypes.c_int32), ("K", ctypes.c_int32), ("d", ctypes.c_int32), ("n_q", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("dtype", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float)]

    @classmethod
    def make(cls, B, K, d, n_q, n_kv, head_dim, ffn, vocab, n_layers, max_pages_per_seq, dtype="bf16",
             page_size=16, rms_eps=1e-6, rope_theta=1e4) -> "Config":
        return cls(B, K, d, n_q, n_kv, head_dim, ffn, vocab, n_layers, page_size, max_pages_per_seq,
                   PE_BF16 if dtype == "bf16" else PE_F32, rms_eps, rope_theta)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == PE_BF16 else torch.float32


class _Weights(ctypes.Structure):
    _fields_ = [("emb", ctypes.c_void_p), ("h_shared", ctypes.c_void_p), ("fc", ctypes.c_void_p),
                ("norm_attn", ctypes.POINTER(ctypes.c_void_p)), ("wqkv", ctypes.POINTER(ctypes.c_void_p)),
                ("wo", ctypes.POINTER(ctypes.c_void_p)), ("norm_mlp", ctypes.POINTER(ctypes.c_void_p)),
                ("w_gate_up", ctypes.POINTER(ctypes.c_void_p)), ("w_down", ctypes.POINTER(ctypes.c_void_p)),
                ("norm_final", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


class _KV(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.POINTER(ctypes.c_void_p)), ("v_cache", ctypes.POINTER(ctypes.c_void_p)),
                ("num_pages", ctypes.c_int32)]


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _arr(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


class DeviceWeights:
    """Drafter weights resident on the device (tensors in nn.Linear layout) + the pe_weights struct."""

    def __init__(self, emb, h_shared, fc, norm_attn, wqkv, wo, norm_mlp, w_gate_up, w_down, norm_final, lm_head):
        self.tensors = dict(emb=emb, h_shared=h_shared, fc=fc, norm_attn=list(norm_attn), wqkv=list(wqkv),
                            wo=list(wo), norm_mlp=list(norm_mlp), w_gate_up=list(w_gate_up),
                            w_down=list(w_down), norm_final=norm_final, lm_head=lm_head)
        self._arrays = [_arr(list(x)) for x in (norm_attn, wqkv, wo, norm_mlp, w_gate_up, w_down)]
        a = self._arrays
        self.struct = _Weights(emb.data_ptr(), h_shared.data_ptr(), fc.data_ptr(), a[0], a[1], a[2], a[3], a[4],
                               a[5], norm_final.data_ptr(), lm_head.data_ptr())


class DeviceKV:
    """Paged KV cache per layer ([num_pages][page][n_kv][hd] K and V) + the pe_kv struct."""

    def __init__(self, k_cache, v_cache):
        self.k_cache, self.v_cache = list(k_cache), list(v_cache)
        self._k, self._v = _arr(self.k_cache), _arr(self.v_cache)
        self.struct = _KV(self._k, self._v, self.k_cache[0].shape[0])


_lib = None


def lib():
    """Load libpe.so (building it first if needed).  Raises if it cannot be loaded."""
    global _lib
    if _lib is None:
        path = os.environ.get("PE_LIB")  # an alternative build of the same C ABI
        if path is None:
            if not os.path.exists(LIB):
                build()
            path = LIB
        L = ctypes.CDLL(path)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        cp = ctypes.POINTER(Config)
        for name in EXPORTED_SYMBOLS:
            getattr(L, name)
        L.pe_sample_drafts.argtypes = [cp, vp, vp, ctypes.c_float, vp, ctypes.c_size_t, vp, vp, vp, vp]
        L.pe_verify_sampled.argtypes = [cp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, ctypes.c_size_t, vp, vp, vp,
                                        vp]
        L.pe_status_str.restype = ctypes.c_char_p
        L.pe_status_str.argtypes = [ctypes.c_int]
        L.pe_workspace_bytes.restype = ctypes.c_size_t
        L.pe_workspace_bytes.argtypes = [cp]
        L.pe_check_config.argtypes = [cp]
        L.pe_prepare_batch.argtypes = [cp, vp, vp, vp, vp, vp, i32] + [vp] * 11
        L.pe_scatter_hidden.argtypes = [cp, ctypes.POINTER(_Weights)] + [vp] * 9
        L.pe_draft_forward.argtypes = ([cp, ctypes.POINTER(_Weights), ctypes.POINTER(_KV)] + [vp] * 7 +
                                       [vp, ctypes.c_size_t, vp, vp, vp, vp])
        L.pe_draft_forward_noalloc.argtypes = ([cp, ctypes.POINTER(_Weights), ctypes.POINTER(_KV)] + [vp] * 7 +
                                               [vp, vp, vp, vp])
        L.pe_verify.argtypes = [cp, vp, vp, vp, vp, vp]
        L.pe_step.argtypes = ([cp, ctypes.POINTER(_Weights), ctypes.POINTER(_KV)] + [vp] * 7 +
                              [vp, ctypes.c_size_t] + [vp] * 8)
        L.pe_set_trace_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
        L.pe_trace_points.argtypes = [cp]
        L.pe_kernel_launches.restype = ctypes.c_uint64
        L.pe_kernel_launches.argtypes = []
        L.pe_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.pe_inject_kv.argtypes = [cp, ctypes.POINTER(_Weights), vp, ctypes.POINTER(_KV), vp, vp, vp, vp, vp,
                                   ctypes.c_size_t, vp, vp]
        L.pe_test_skip_pipeline_stage.argtypes = [i32]
        for name in EXPORTED_SYMBOLS:
            if name not in ("pe_status_str", "pe_workspace_bytes", "pe_kernel_launches"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().pe_status_str(int(status)).decode()


def _check(status: int, what: str):
    if status != PE_OK:
        raise PeError(status, what)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def set_trace_events(events) -> None:
    """Record these torch.cuda.Event objects at the stage boundaries of pe_draft_forward / pe_step
    (see pe.h); pass [] to stop tracing."""
    handles = [ctypes.c_void_p(e.cuda_event) for e in events]
    arr = (ctypes.c_void_p * max(1, len(handles)))(*handles)
    _check(lib().pe_set_trace_events(arr, len(handles)), "pe_set_trace_events")


def trace_points(cfg: Config) -> int:
    return int(lib().pe_trace_points(ctypes.byref(cfg)))


def kernel_launches() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().pe_kernel_launches())


def set_wait_limit_ns(ns: int) -> None:
    """Limit of every bounded pipeline wait in kernels launched from now on (0: the default, 1 s)."""
    _check(lib().pe_set_wait_limit_ns(int(ns)), "pe_set_wait_limit_ns")


def skip_pipeline_stage_for_test(stage: int) -> None:
    """Failure-detection test hook: the next tensor-core GEMM launch leaves this pipeline stage of
    its first CTA unarmed, so a wait on it runs out (-1 clears it)."""
    _check(lib().pe_test_skip_pipeline_stage(int(stage)), "pe_test_skip_pipeline_stage")


def check_config(cfg: Config) -> int:
    return int(lib().pe_check_config(ctypes.byref(cfg)))


def workspace_bytes(cfg: Config) -> int:
    return int(lib().pe_workspace_bytes(ctypes.byref(cfg)))


def prepare_batch(cfg, prev_tokens, prev_pos, num_accepted, bonus, block_table, num_pages, out: dict, err,
                  stream=None):
    """Stage (a).  ``out`` holds input_ids, positions, slot_mapping, is_rejected, is_mask, hidden_map,
    row_list, n_valid, draft_rows (device tensors)."""
    st = lib().pe_prepare_batch(ctypes.byref(cfg), _ptr(prev_tokens), _ptr(prev_pos), _ptr(num_accepted),
                                _ptr(bonus), _ptr(block_table), int(num_pages), _ptr(out["input_ids"]),
                                _ptr(out["positions"]), _ptr(out["slot_mapping"]), _ptr(out["is_rejected"]),
                                _ptr(out["is_mask"]), _ptr(out["hidden_map"]), _ptr(out["row_list"]),
                                _ptr(out["n_valid"]), _ptr(out["draft_rows"]), _ptr(err), _stream(stream))
    _check(st, "pe_prepare_batch")


def scatter_hidden(cfg, weights: DeviceWeights, target_hidden, meta: dict, x0, err, stream=None):
    """Stage (b): x0[i] = concat(emb[token], hidden) for the compacted valid rows."""
    st = lib().pe_scatter_hidden(ctypes.byref(cfg), ctypes.byref(weights.struct), _ptr(target_hidden),
                                 _ptr(meta["input_ids"]), _ptr(meta["is_mask"]), _ptr(meta["hidden_map"]),
                                 _ptr(meta["row_list"]), _ptr(meta["n_valid"]), _ptr(x0), _ptr(err),
                                 _stream(stream))
    _check(st, "pe_scatter_hidden")


def draft_forward(cfg, weights: DeviceWeights, kv: DeviceKV, block_table, x0, meta: dict, workspace,
                  draft_tokens, err, logits_dbg=None, stream=None):
    """Stages (c)+(d): drafter pass over the valid rows, LM head + argmax -> draft_tokens [B][K]."""
    st = lib().pe_draft_forward(ctypes.byref(cfg), ctypes.byref(weights.struct), ctypes.byref(kv.struct),
                                _ptr(block_table), _ptr(x0), _ptr(meta["positions"]), _ptr(meta["slot_mapping"]),
                                _ptr(meta["row_list"]), _ptr(meta["n_valid"]), _ptr(meta["draft_rows"]),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _ptr(draft_tokens), _ptr(logits_dbg), _ptr(err), _stream(stream))
    _check(st, "pe_draft_forward")


def draft_forward_noalloc(cfg, weights: DeviceWeights, kv: DeviceKV, block_table, x0, meta: dict, draft_tokens,
                          err, logits_dbg=None, stream=None):
    """draft_forward without a workspace: the library's own fixed scratch array is used, for callers
    that cannot allocate device memory.  Calls that overlap on the GPU race on that array."""
    st = lib().pe_draft_forward_noalloc(ctypes.byref(cfg), ctypes.byref(weights.struct), ctypes.byref(kv.struct),
                                        _ptr(block_table), _ptr(x0), _ptr(meta["positions"]),
                                        _ptr(meta["slot_mapping"]), _ptr(meta["row_list"]), _ptr(meta["n_valid"]),
                                        _ptr(meta["draft_rows"]), _ptr(draft_tokens), _ptr(logits_dbg), _ptr(err),
                                        _stream(stream))
    _check(st, "pe_draft_forward_noalloc")


def verify(cfg, draft_tokens, target_tokens, num_accepted_out, bonus_out, stream=None):
    """Stage (e): greedy verification."""
    st = lib().pe_verify(ctypes.byref(cfg), _ptr(draft_tokens), _ptr(target_tokens), _ptr(num_accepted_out),
                         _ptr(bonus_out), _stream(stream))
    _check(st, "pe_verify")


def sample_drafts(cfg, logits, u_draft, temperature, workspace, draft_tokens, lse, err, stream=None):
    """Non-greedy drafting: draft tokens drawn from softmax(logits / temperature)."""
    st = lib().pe_sample_drafts(ctypes.byref(cfg), _ptr(logits), _ptr(u_draft), ctypes.c_float(temperature),
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(draft_tokens),
                                _ptr(lse), _ptr(err), _stream(stream))
    _check(st, "pe_sample_drafts")


def verify_sampled(cfg, draft_tokens, logits, lse, temperature, target_probs, u_accept, u_resample, workspace,
                   num_accepted_out, bonus_out, err, stream=None):
    """Verification by rejection sampling against the target's distributions."""
    st = lib().pe_verify_sampled(ctypes.byref(cfg), _ptr(draft_tokens), _ptr(logits), _ptr(lse),
                                 ctypes.c_float(temperature), _ptr(target_probs), _ptr(u_accept), _ptr(u_resample),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _ptr(num_accepted_out), _ptr(bonus_out), _ptr(err), _stream(stream))
    _check(st, "pe_verify_sampled")


def inject_kv(cfg, weights: DeviceWeights, w_inj, kv: DeviceKV, block_table, prev_pos, num_accepted, target_hidden,
              workspace, err, stream=None):
    """DFlash-style KV injection: the verifier's hidden states of the previous verify batch,
    projected by w_inj [d][d], written as k / v into every layer's cache at the accepted
    positions (see pe.h)."""
    st = lib().pe_inject_kv(ctypes.byref(cfg), ctypes.byref(weights.struct), _ptr(w_inj), ctypes.byref(kv.struct),
                            _ptr(block_table), _ptr(prev_pos), _ptr(num_accepted), _ptr(target_hidden),
                            _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err),
                            _stream(stream))
    _check(st, "pe_inject_kv")


def step(cfg, weights: DeviceWeights, kv: DeviceKV, block_table, prev_tokens, prev_pos, num_accepted, bonus,
         target_hidden, target_tokens, workspace, out: dict, err, logits_dbg=None, stream=None):
    """One whole round.  ``out`` holds draft_tokens, num_accepted, bonus, next_prev_tokens, next_prev_pos."""
    st = lib().pe_step(ctypes.byref(cfg), ctypes.byref(weights.struct), ctypes.byref(kv.struct),
                       _ptr(block_table), _ptr(prev_tokens), _ptr(prev_pos), _ptr(num_accepted), _ptr(bonus),
                       _ptr(target_hidden), _ptr(target_tokens), _ptr(workspace),
                       workspace.numel() * workspace.element_size(), _ptr(out["draft_tokens"]),
                       _ptr(out["num_accepted"]), _ptr(out["bonus"]), _ptr(out["next_prev_tokens"]),
                       _ptr(out["next_prev_pos"]), _ptr(logits_dbg), _ptr(err), _stream(stream))
    _check(st, "pe_step")


# ----------------------------------------------------------------------------- buffer helpers

def alloc_batch(cfg: Config, device="cuda") -> dict:
    """Device buffers for pe_prepare_batch's outputs."""
    R, T = cfg.B * 2 * cfg.K, cfg.B * cfg.K
    i32 = dict(dtype=torch.int32, device=device)
    return dict(input_ids=torch.empty(R, **i32), positions=torch.empty(R, **i32),
                slot_mapping=torch.empty(R, dtype=torch.int64, device=device),
                is_rejected=torch.empty(R, dtype=torch.uint8, device=device),
                is_mask=torch.empty(R, dtype=torch.uint8, device=device), hidden_map=torch.empty(R, **i32),
                row_list=torch.empty(R, **i32), n_valid=torch.empty(1, **i32), draft_rows=torch.empty(T, **i32))


def alloc_workspace(cfg: Config, device="cuda") -> torch.Tensor:
    n = workspace_bytes(cfg)
    if n == 0:
        raise PeError(check_config(cfg), "pe_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


class Round:
    """Device buffers for one drafter batch plus calls of the five entry points in order.

    ``weights`` / ``kv`` are DeviceWeights / DeviceKV; ``block_table`` an int32 CUDA tensor.
    Buffers are allocated once here with torch; the library itself allocates nothing.
    """

    def __init__(self, cfg: Config, weights: DeviceWeights, kv: DeviceKV, block_table, device="cuda"):
        self.cfg, self.weights, self.kv, self.block_table = cfg, weights, kv, block_table
        R, T = cfg.B * 2 * cfg.K, cfg.B * cfg.K
        self.meta = alloc_batch(cfg, device)
        self.x0 = torch.empty((R, 2 * cfg.d), dtype=cfg.torch_dtype, device=device)
        self.workspace = alloc_workspace(cfg, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.draft_tokens = torch.empty((cfg.B, cfg.K), **i32)
        self.out = dict(draft_tokens=self.draft_tokens, num_accepted=torch.empty(cfg.B, **i32),
                        bonus=torch.empty(cfg.B, **i32), next_prev_tokens=torch.empty((cfg.B, cfg.K + 1), **i32),
                        next_prev_pos=torch.empty((cfg.B, cfg.K + 1), **i32))
        self.logits = None
        self.lse = None

    def _logits(self, want: bool):
        if not want:
            return None
        if self.logits is None:
            self.logits = torch.empty((self.cfg.B * self.cfg.K, self.cfg.vocab), dtype=torch.float32,
                                      device=self.x0.device)
        return self.logits

    def prepare(self, prev_tokens, prev_pos, num_accepted, bonus, stream=None):
        prepare_batch(self.cfg, prev_tokens, prev_pos, num_accepted, bonus, self.block_table,
                      self.kv.struct.num_pages, self.meta, self.err, stream)

    def scatter(self, target_hidden, stream=None):
        scatter_hidden(self.cfg, self.weights, target_hidden, self.meta, self.x0, self.err, stream)

    def forward(self, logits: bool = False, stream=None):
        draft_forward(self.cfg, self.weights, self.kv, self.block_table, self.x0, self.meta, self.workspace,
                      self.draft_tokens, self.err, self._logits(logits), stream)

    def verify(self, target_tokens, stream=None):
        verify(self.cfg, self.draft_tokens, target_tokens, self.out["num_accepted"], self.out["bonus"], stream)

    def step(self, prev_tokens, prev_pos, num_accepted, bonus, target_hidden, target_tokens, logits=False,
             stream=None):
        step(self.cfg, self.weights, self.kv, self.block_table, prev_tokens, prev_pos, num_accepted, bonus,
             target_hidden, target_tokens, self.workspace, self.out, self.err, self._logits(logits), stream)

    def sample(self, u_draft, temperature: float = 1.0, stream=None):
        """Non-greedy drafting from the logits of the last ``forward(logits=True)``: overwrites
        draft_tokens with draws from softmax(logits / temperature) and fills ``lse``."""
        if self.logits is None:
            raise RuntimeError("sample() needs the logits of forward(logits=True)")
        if self.lse is None:
            self.lse = torch.empty(self.cfg.B * self.cfg.K, dtype=torch.float32, device=self.x0.device)
        sample_drafts(self.cfg, self.logits, u_draft, temperature, self.workspace, self.draft_tokens, self.lse,
                      self.err, stream)

    def verify_sampled(self, target_probs, u_accept, u_resample, temperature: float = 1.0, stream=None):
        """Rejection-sampling verification of the drafts of the last ``sample``."""
        verify_sampled(self.cfg, self.draft_tokens, self.logits, self.lse, temperature, target_probs, u_accept,
                       u_resample, self.workspace, self.out["num_accepted"], self.out["bonus"], self.err, stream)

    def step_inplace(self, state: dict, target_hidden, target_tokens, stream=None):
        """One round whose next verify batch, accepted counts and bonus tokens overwrite ``state``
        (prev_tokens, prev_pos, num_accepted, bonus): the same call, or a CUDA graph of it, is
        the next round once the caller has refilled ``target_hidden`` and ``target_tokens``."""
        out = dict(draft_tokens=self.draft_tokens, num_accepted=state["num_accepted"], bonus=state["bonus"],
                   next_prev_tokens=state["prev_tokens"], next_prev_pos=state["prev_pos"])
        step(self.cfg, self.weights, self.kv, self.block_table, state["prev_tokens"], state["prev_pos"],
             state["num_accepted"], state["bonus"], target_hidden, target_tokens, self.workspace, out, self.err,
             None, stream)

    def capture_loop(self, state: dict, target_hidden, target_tokens) -> torch.cuda.CUDAGraph:
        """CUDA graph of ``step_inplace`` on these buffers; every replay runs the next round.
        Run one round directly first (launch attributes are set on a kernel's first use)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step_inplace(state, target_hidden, target_tokens)
        return g
