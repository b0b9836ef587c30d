"""GPU test of gdn_prefill_chunked_noalloc, the prefill entry point for callers that cannot
allocate device memory when they prefill (an engine that reserved almost all of HBM for its
own pools, or a plug-in whose host runtime owns every allocation).  It must give the same
results as gdn_prefill_chunked given a workspace, call after call, while the library's
shared scratch keeps whatever the previous call left in it.  Under CUDA's lazy module loading
the scratch is reserved by the first call on a device (a call with n = 0 does only that), so a
caller makes that call before it reserves the rest of the device's memory; a later call must
then reserve nothing.

This file is collected last on purpose, so a run that stops at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _prefill(w: wl.Workload, noalloc: bool):
    """One prefill of workload w from its initial states, through one of the two entry
    points.  Returns y, core output, final h states and conv states (host arrays)."""
    d = torch.device("cuda")
    sh = w.shape
    dims = dev.dims_of(sh)
    h_pool, conv_pool, slots = dev.states_to(w, d)
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
    hp = torch.tensor([h_pool.data_ptr() + i * hsz for i in range(w.n)], dtype=torch.int64,
                      device=d)
    cu = torch.from_numpy(w.cu_seqlens).to(d)
    T, max_len = int(w.lens.sum()), int(w.lens.max())
    y = torch.empty((T, sh.n_v_heads * sh.d_v), dtype=dev.act_dtype(w), device=d)
    core = torch.empty((T, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    weights, inputs = dev.weights_to(w, d), dev.tokens_to(w.tokens, dev.act_dtype(w), d)
    if noalloc:
        gdn.gdn_prefill_chunked_noalloc(dims, weights, inputs, w.n, cu, T, max_len, hp,
                                        conv_pool, w.n, slots, y, core, status)
    else:
        nbytes = gdn.gdn_prefill_workspace_bytes(dims, w.n, T, max_len)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=d)
        gdn.gdn_prefill_chunked(dims, weights, inputs, w.n, cu, T, max_len, hp, conv_pool, w.n,
                                slots, y, core, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, gdn.status_string(int(status.item()))
    return (y.float().cpu().numpy(), core.cpu().numpy(), h_pool.cpu().numpy(),
            conv_pool.float().cpu().numpy())


def _same(ref, got):
    """Both entry points run the same deterministic kernels on the same inputs, so every
    output must agree bit for bit: a stale byte of scratch left by an earlier call that
    reached a result would show here."""
    for r, g in zip(ref, got):
        np.testing.assert_array_equal(g, r)


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    first = wl.varlen_prefill([100, 7, 129], seed=21)      # ragged chunks, 3 sequences
    second = wl.varlen_prefill([500, 64], seed=22)         # longer, more scratch than the first
    for w in (first, second):
        ref = _prefill(w, noalloc=False)
        got = _prefill(w, noalloc=True)
        _same(ref, got)


def test_noalloc_refuses_a_problem_larger_than_its_scratch():
    w = wl.varlen_prefill([64], seed=23)
    dims = dev.dims_of(w.shape)
    too_many = 8192  # 130 chunk slots of about 2.8 MiB each: more than the 64 MiB scratch
    assert gdn.gdn_prefill_workspace_bytes(dims, 1, too_many, too_many) > gdn.NOALLOC_SCRATCH_BYTES
    d = torch.device("cuda")
    h_pool, conv_pool, slots = dev.states_to(w, d)
    hp = torch.tensor([h_pool.data_ptr()], dtype=torch.int64, device=d)
    cu = torch.tensor([0, too_many], dtype=torch.int32, device=d)
    qkv = torch.zeros((too_many, w.shape.conv_dim), dtype=torch.bfloat16, device=d)
    z = torch.zeros((too_many, w.shape.z_dim), dtype=torch.bfloat16, device=d)
    ab = torch.zeros((too_many, w.shape.n_v_heads), dtype=torch.bfloat16, device=d)
    y = torch.empty_like(z)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_chunked_noalloc(dims, dev.weights_to(w, d), gdn.Inputs(qkv, z, ab, ab), 1,
                                        cu, too_many, too_many, hp, conv_pool, 1, slots, y, None,
                                        status)
    assert e.value.status == 9  # GDN_ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert int(status.item()) == 0  # nothing ran


_SETUP_ORDER = r"""
import json, sys, torch
sys.path.insert(0, sys.argv[1])
from gated_deltanet_layer_conv1d_gb300 import device as dev, gdn, workloads as wl
d = torch.device("cuda")
w = wl.varlen_prefill([100, 7], seed=24)
sh = w.shape
dims, weights = dev.dims_of(sh), dev.weights_to(w, d)
inputs = dev.tokens_to(w.tokens, torch.bfloat16, d)
h_pool, conv_pool, slots = dev.states_to(w, d)
hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
hp = torch.tensor([h_pool.data_ptr() + i * hsz for i in range(w.n)], dtype=torch.int64, device=d)
cu = torch.from_numpy(w.cu_seqlens).to(d)
T, L = int(w.lens.sum()), int(w.lens.max())
y = torch.empty((T, sh.z_dim), dtype=torch.bfloat16, device=d)
status = torch.zeros(1, dtype=torch.int32, device=d)
# every kernel module the prefill uses is loaded by one call with a caller workspace
ws = torch.empty(gdn.gdn_prefill_workspace_bytes(dims, w.n, T, L), dtype=torch.uint8, device=d)
gdn.gdn_prefill_chunked(dims, weights, inputs, w.n, cu, T, L, hp, conv_pool, w.n, slots, y,
                        None, ws, status)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
gdn.gdn_prefill_chunked_noalloc(dims, weights, inputs, 0, None, 0, 0, None, None, 0, None,
                                None)                                    # the set-up call
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
gdn.gdn_prefill_chunked_noalloc(dims, weights, inputs, w.n, cu, T, L, hp, conv_pool, w.n,
                                slots, y, None, status)
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
print(json.dumps({"setup": free0 - free1, "call": free1 - free2, "status": int(status.item())}))
"""


def test_noalloc_setup_call_reserves_the_scratch_and_later_calls_reserve_nothing():
    """In a fresh process: after the set-up call (n = 0), a real call changes the device's
    free memory by less than the scratch's size, whatever CUDA_MODULE_LOADING says."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _SETUP_ORDER, root], capture_output=True,
                       text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stdout + r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    assert got["status"] == 0, gdn.status_string(got["status"])
    assert got["call"] < gdn.NOALLOC_SCRATCH_BYTES // 2, got
    if os.environ.get("CUDA_MODULE_LOADING", "LAZY").upper() == "LAZY":
        # the set-up call is where the scratch was reserved
        assert got["setup"] >= gdn.NOALLOC_SCRATCH_BYTES // 2, got
