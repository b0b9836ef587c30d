"""GPU parity of the f32 prefill option (gdn_dims.prefill_precision = GDN_PREFILL_F32) on the
tensor-core path's own workloads -- bf16 activations at d = 128 -- held to the f32 class of the
decode and verify paths: state and core output 1e-4, y 2e-3, conv states bit-exact, with the
row and element bounds of gpu_common.  The long prefill (1 x 8192 tokens, chunk 64 on the
tensor-core path) and the mixed-serving step's 32 prefills are the two workloads whose state
the tensor-core form holds only to 1e-3."""
import dataclasses

import numpy as np
import pytest
import torch

from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import (assert_core_close, assert_state_close, assert_y_close, oracle_seqs,
                              require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_f32(w: wl.Workload):
    d = torch.device("cuda")
    sh = w.shape
    dims = dev.dims_of(sh)
    dims.prefill_precision = gdn.GDN_PREFILL_F32
    h_pool, conv_pool, slots = dev.states_to(w, d)
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
    hp = torch.tensor([h_pool.data_ptr() + i * hsz for i in range(w.n)], dtype=torch.int64,
                      device=d)
    cu = torch.from_numpy(w.cu_seqlens).to(d)
    T, L = int(w.lens.sum()), int(w.lens.max())
    assert gdn.gdn_prefill_workspace_bytes(dims, w.n, T, L) == 0  # the sequential form needs none
    y = torch.empty((T, sh.z_dim), dtype=torch.bfloat16, device=d)
    core = torch.empty((T, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    gdn.gdn_prefill_chunked(dims, dev.weights_to(w, d), dev.tokens_to(w.tokens, torch.bfloat16, d),
                            w.n, cu, T, L, hp, conv_pool, w.n, slots, y, core, None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, gdn.status_string(int(status.item()))
    res = oracle_seqs(w, w.tokens, [int(x) for x in w.lens])
    o_orc = np.concatenate([x.o for x in res])
    assert_y_close(y, np.concatenate([x.y for x in res]), "f32 prefill y", o_orc=o_orc)
    assert_core_close(core, o_orc, "f32 prefill core o")
    H = h_pool.cpu().numpy()
    conv = conv_pool.float().cpu().numpy()
    for i, x in enumerate(res):
        assert_state_close(H[i], x.H, f"f32 prefill state seq {i}")
        np.testing.assert_array_equal(conv[i], x.conv_state)


def test_f32_prefill_long_8192():
    run_f32(wl.long_prefill(8192))


def test_f32_prefill_mixed_serving_prefills():
    pre, _ = wl.mixed_serving()
    run_f32(pre)


def test_f32_prefill_ragged_and_sigmoid_gate():
    w = wl.varlen_prefill([100, 7, 0, 129, 64, 1], seed=98)
    run_f32(w)
    w = wl.varlen_prefill([70, 33], seed=99)
    w.shape = dataclasses.replace(w.shape, norm_gate=gdn.GDN_NORM_GATE_SIGMOID)
    run_f32(w)


def test_prefill_precision_is_validated():
    w = wl.varlen_prefill([5], seed=100)
    dims = dev.dims_of(w.shape)
    dims.prefill_precision = 2
    assert gdn.gdn_prefill_workspace_bytes(dims, 1, 5, 5) == 0  # invalid dims
