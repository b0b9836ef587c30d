"""GPU parity of the sigmoid-gated norm (the gdn_norm_sigmoid models; layer_struct.rs, the
gated_rms_norm_f32_strided_k field): gdn_dims.norm_gate = GDN_NORM_GATE_SIGMOID through
every entry point that ends in the gated norm -- decode (norm warp), verify (per-token norm
warps), the tensor-core prefill in both spine forms (whole rows, and column slices with
the norm in the launch's spare CTAs), the token-sequential prefill -- and the
stand-alone gdn_gated_rmsnorm_sigmoid.  Same tolerances as the SiLU-gated tests."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import assert_y_close, require_gpu
from tests.test_decode_gpu import check_against_oracle, run_decode
from tests.test_prefill_gpu import check_prefill, run_prefill
from tests.test_verify_gpu import check, run_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def sigmoid_gated(w: wl.Workload) -> wl.Workload:
    w.shape = dataclasses.replace(w.shape, norm_gate=gdn.GDN_NORM_GATE_SIGMOID)
    return w


@pytest.mark.parametrize("shape,n,bf16", [(wl.TINY, 5, False), (wl.FULL, 37, True)])
def test_decode_sigmoid_gate(shape, n, bf16):
    w = sigmoid_gated(wl.batched_decode(n=n, steps=3, shape=shape, seed=51, bf16=bf16))
    ys, cores, H, conv, _ = run_decode(w)
    check_against_oracle(w, ys, cores, H, conv)


def test_verify_sigmoid_gate():
    w = sigmoid_gated(wl.ragged_verify(n=24, seed=52))
    r = run_verify(w)
    assert r["status"] == 0
    check(w, r, [0, 11])


@pytest.mark.parametrize("lens", [[100, 7, 129, 64, 1, 128],  # 192 (seq, head) units: whole rows
                                  [300]])                      # 32 units: sliced spine
def test_tensor_core_prefill_sigmoid_gate(lens):
    w = sigmoid_gated(wl.varlen_prefill(lens, seed=53))
    check_prefill(w, run_prefill(w))


def test_sequential_prefill_sigmoid_gate():
    w = sigmoid_gated(wl.varlen_prefill([70, 5, 64], shape=wl.TINY, seed=54))
    check_prefill(w, run_prefill(w))


@pytest.mark.parametrize("shape,bf16", [(wl.TINY, False), (wl.FULL, True)])
def test_gated_rmsnorm_sigmoid(shape, bf16):
    rng = np.random.default_rng(55)
    T, Hv, dv = 33, shape.n_v_heads, shape.d_v
    o = rng.standard_normal((T, Hv, dv)).astype(np.float32)
    z = rng.standard_normal((T, Hv * dv)).astype(np.float32)
    if bf16:
        z = wl.round_bf16(z)
    w = (1 + 0.1 * rng.standard_normal(dv)).astype(np.float32)
    d = torch.device("cuda")
    dt = torch.bfloat16 if bf16 else torch.float32
    y = torch.empty((T, Hv * dv), dtype=dt, device=d)
    gdn.gdn_gated_rmsnorm(torch.from_numpy(o).to(d), torch.from_numpy(z).to(d, dt),
                          torch.from_numpy(w).to(d), 1e-6, y, sigmoid=True)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(o, z, w, float(np.float32(1e-6)), gate=1)
    assert_y_close(y, ref, "sigmoid-gated rmsnorm")
