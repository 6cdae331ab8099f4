"""Upload seeded workload arrays (numpy) to torch CUDA tensors.  Layout only, no arithmetic."""

from __future__ import annotations

import numpy as np
import torch


def to_torch(a: np.ndarray, device="cuda") -> torch.Tensor:
    """float32 arrays stay float32; uint16 arrays hold bf16 bit patterns and become bfloat16."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def weights_to_device(w, device="cuda") -> dict:
    t = lambda a: to_torch(a, device)
    return dict(emb=t(w.emb), h_shared=t(w.h_shared), fc=t(w.fc), norm_attn=[t(x) for x in w.norm_attn],
                wqkv=[t(x) for x in w.wqkv], wo=[t(x) for x in w.wo], norm_mlp=[t(x) for x in w.norm_mlp],
                w_gate_up=[t(x) for x in w.w_gate_up], w_down=[t(x) for x in w.w_down],
                norm_final=t(w.norm_final), lm_head=t(w.lm_head))


def round_to_device(rnd, device="cuda") -> dict:
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    return dict(prev_tokens=i32(rnd.prev_tokens), prev_pos=i32(rnd.prev_pos), num_accepted=i32(rnd.num_accepted),
                bonus=i32(rnd.bonus), block_table=i32(rnd.block_table), target_hidden=to_torch(rnd.target_hidden, device),
                k_cache=[to_torch(x, device) for x in rnd.k_cache], v_cache=[to_torch(x, device) for x in rnd.v_cache])
