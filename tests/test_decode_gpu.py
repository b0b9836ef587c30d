"""GPU parity of gdn_decode_batched against the fp64 oracle (batched single-token decode,
trait_layer.rs TransformerLayer::decode_batched / decode_multi_seq)."""
import numpy as np
import pytest
import torch

from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import (assert_core_close, assert_state_close, assert_y_close,
                              oracle_seqs, require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _stack_steps(w: wl.Workload):
    """Per-sequence token rows (sequence-major) from the per-step rows."""
    steps = [w.tokens] + w.steps
    n = w.n
    return {k: np.stack([s[k] for s in steps], axis=1).reshape(n * len(steps), -1)
            for k in ("qkv", "z", "a", "b")}


def run_decode(w: wl.Workload, slot_perm=None, n_slots=None, canary=False):
    """All decode steps of w on the GPU.  Returns (ys [steps][n][Hv*dv], cores, H [n],
    conv [n], pools)."""
    d = torch.device("cuda")
    dims = dev.dims_of(w.shape)
    weights = dev.weights_to(w, d)
    h_pool, conv_pool, slots = dev.states_to(w, d, slot_perm, n_slots)
    if canary:  # slots no sequence uses must come back untouched
        used = set(int(s) for s in slots.cpu())
        for s in range(h_pool.shape[0]):
            if s not in used:
                h_pool[s].fill_(7.25)
                conv_pool[s].fill_(-3.5)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    n = w.n
    sh = w.shape
    ys, cores = [], []
    for tok in [w.tokens] + w.steps:
        inp = dev.tokens_to(tok, dev.act_dtype(w), d)
        y = torch.empty((n, sh.n_v_heads * sh.d_v), dtype=dev.act_dtype(w), device=d)
        core = torch.empty((n, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=d)
        gdn.gdn_decode_batched(dims, weights, inp, n, h_pool, conv_pool, h_pool.shape[0], slots,
                               y, core, status)
        ys.append(y)
        cores.append(core)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, gdn.status_string(int(status.item()))
    sl = slots.long()
    return ys, cores, h_pool[sl].cpu().numpy(), conv_pool[sl].float().cpu().numpy(), (
        h_pool, conv_pool, slots)


def check_against_oracle(w, ys, cores, H, conv):
    steps = 1 + len(w.steps)
    res = oracle_seqs(w, _stack_steps(w), [steps] * w.n)
    y_orc = np.stack([r.y for r in res], axis=0)       # [n][steps][Hv*dv]
    o_orc = np.stack([r.o for r in res], axis=0)       # [n][steps][Hv][dv]
    for s in range(steps):
        assert_y_close(ys[s], y_orc[:, s], f"y step {s}", o_orc=o_orc[:, s])
        assert_core_close(cores[s], o_orc[:, s], f"core o step {s}")
    for i, r in enumerate(res):
        assert_state_close(H[i], r.H, f"state seq {i}")
        np.testing.assert_array_equal(conv[i], r.conv_state)  # bit-exact rotation


def test_decode_tiny_f32():
    w = wl.batched_decode(n=5, steps=8, shape=wl.TINY, seed=1, bf16=False)
    ys, cores, H, conv, _ = run_decode(w)
    check_against_oracle(w, ys, cores, H, conv)


def test_decode_tiny_bf16_permuted_slots():
    w = wl.batched_decode(n=7, steps=4, shape=wl.TINY, seed=2)
    perm = np.array([5, 0, 9, 2, 7, 11, 3], np.int32)
    ys, cores, H, conv, (h_pool, conv_pool, _) = run_decode(w, perm, n_slots=12, canary=True)
    check_against_oracle(w, ys, cores, H, conv)
    for s in set(range(12)) - set(perm.tolist()):
        assert (h_pool[s] == 7.25).all() and (conv_pool[s] == -3.5).all()


def test_decode_full_128_one_step_permuted_slots():
    w = wl.batched_decode(n=128, steps=1)
    perm = w.extra["slot_perm"]
    ys, cores, H, conv, (h_pool, conv_pool, _) = run_decode(w, perm, n_slots=136, canary=True)
    check_against_oracle(w, ys, cores, H, conv)
    for s in range(128, 136):
        assert (h_pool[s] == 7.25).all() and (conv_pool[s] == -3.5).all()


def test_decode_full_128_64_steps():
    """The state after 64 decode steps stays within 1e-4 of the oracle."""
    w = wl.batched_decode(n=128, steps=64, seed=3)
    ys, cores, H, conv, _ = run_decode(w)
    check_against_oracle(w, ys, cores, H, conv)


def test_decode_single_sequence_and_partial_batch():
    for n in (1, 37):
        w = wl.batched_decode(n=n, steps=2, seed=10 + n)
        ys, cores, H, conv, _ = run_decode(w)
        check_against_oracle(w, ys, cores, H, conv)


def test_decode_bad_slot_sets_status_and_skips():
    w = wl.batched_decode(n=3, steps=1, shape=wl.TINY, seed=4)
    d = torch.device("cuda")
    h_pool, conv_pool, slots = dev.states_to(w, d)
    before = h_pool.clone()
    slots[1] = 99  # outside [0, n_slots)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    y = torch.zeros((3, 32), dtype=torch.bfloat16, device=d)
    gdn.gdn_decode_batched(dev.dims_of(w.shape), dev.weights_to(w, d),
                           dev.tokens_to(w.tokens, torch.bfloat16, d), 3, h_pool, conv_pool, 3,
                           slots, y, None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 17  # GDN_ERR_BAD_SLOT
    assert (h_pool[1] == before[1]).all()  # slot 1 belonged to the skipped sequence
    assert not torch.equal(h_pool[0], before[0])  # the others ran
