"""Device-side marshalling of a synthetic workload for the libgdn.so entry points.

Copies a `workloads.Workload` into torch device tensors laid out as include/gdn.h asks
(activations in bf16 or f32, f32 weights and states, slot pools, WY pointer tables) and
calls the binding.  No compute happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import gdn
from .workloads import LayerShape, Workload


def dims_of(shape: LayerShape) -> gdn.gdn_dims:
    return gdn.make_dims(shape.n_k_heads, shape.n_v_heads, shape.d_k, shape.d_v, shape.d_conv,
                         shape.q_scale, shape.l2_eps, shape.norm_eps, shape.norm_gate)


def act_dtype(wl: Workload) -> torch.dtype:
    return torch.bfloat16 if wl.bf16 else torch.float32


def weights_to(wl: Workload, device) -> gdn.Weights:
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(device) for k, v in wl.weights.items()}
    return gdn.Weights(t["conv_w"], t["A_log"], t["dt_bias"], t["norm_w"])


def tokens_to(tok: dict, dtype: torch.dtype, device) -> gdn.Inputs:
    t = {k: torch.from_numpy(np.ascontiguousarray(tok[k])).to(device=device, dtype=dtype)
         for k in ("qkv", "z", "a", "b")}
    return gdn.Inputs(t["qkv"], t["z"], t["a"], t["b"])


def states_to(wl: Workload, device, slot_perm=None, n_slots=None):
    """Slot pools holding each sequence's initial state at slot slot_perm[i]."""
    n = wl.n
    perm = np.arange(n, dtype=np.int32) if slot_perm is None else np.asarray(slot_perm, np.int32)
    n_slots = n if n_slots is None else n_slots
    sh = wl.shape
    h_pool = torch.zeros((n_slots, sh.n_v_heads, sh.d_k, sh.d_v), dtype=torch.float32,
                         device=device)
    conv_pool = torch.zeros((n_slots, sh.conv_dim, sh.d_conv), dtype=act_dtype(wl),
                            device=device)
    idx = torch.from_numpy(perm.astype(np.int64)).to(device)
    h_pool[idx] = torch.from_numpy(wl.H0).to(device)
    conv_pool[idx] = torch.from_numpy(wl.conv0).to(device=device, dtype=act_dtype(wl))
    slots = torch.from_numpy(perm).to(device)
    return h_pool, conv_pool, slots


def wy_tables_to(ks, h_ptrs, inter_ptrs, device) -> torch.Tensor:
    host = gdn.gdn_wy_tables_fill(ks, h_ptrs, inter_ptrs)
    return torch.from_numpy(host.view(np.int64)).to(device)
