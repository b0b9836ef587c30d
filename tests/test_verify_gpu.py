"""GPU parity of gdn_verify_multi (ragged speculative verify through the WY pointer
tables of transformer_layer.rs, VERIFY_WY_TABLE_SEQS; trait_layer.rs
TransformerLayer::decode_verify_multi) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import (assert_core_close, assert_state_close, assert_y_close,
                              oracle_seqs, require_gpu)

pytestmark = pytest.mark.gpu

CANARY = 1.5e30


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_verify(w: wl.Workload, slot_perm=None, conv_inter=True, spoil=None):
    """Runs one ragged verify on the GPU.  Intermediates live in one buffer
    [n][15][Hv][dk][dv] prefilled with a canary; final states in a slot pool."""
    d = torch.device("cuda")
    n, sh = w.n, w.shape
    ks = [int(k) for k in w.lens]
    h_pool, conv_pool, slots = dev.states_to(w, d, slot_perm)
    inter = torch.full((n, 15, sh.n_v_heads, sh.d_k, sh.d_v), CANARY, dtype=torch.float32,
                       device=d)
    ci = None
    if conv_inter:
        ci = torch.full((n, 15, sh.conv_dim, sh.d_conv), -7.0, dtype=dev.act_dtype(w), device=d)
    sl = slots.long().cpu().numpy()
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
    h_ptrs = [h_pool.data_ptr() + int(sl[i]) * hsz for i in range(n)]
    inter_ptrs = [[inter[i, t].data_ptr() for t in range(15)] for i in range(n)]
    tables = dev.wy_tables_to(ks, h_ptrs, inter_ptrs, d)
    if spoil is not None:
        tables.view(16, 128)[spoil] = 0
    tables_before = tables.clone()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    rows = sum(ks)
    y = torch.empty((rows, sh.n_v_heads * sh.d_v), dtype=dev.act_dtype(w), device=d)
    core = torch.empty((rows, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=d)
    gdn.gdn_verify_multi(dev.dims_of(sh), dev.weights_to(w, d),
                         dev.tokens_to(w.tokens, dev.act_dtype(w), d), n, ks, tables, conv_pool,
                         h_pool.shape[0], slots, ci, y, core, status)
    torch.cuda.synchronize()
    assert torch.equal(tables, tables_before), "the kernel must never write the tables"
    return dict(status=int(status.item()), y=y, core=core, H=h_pool[slots.long()].cpu().numpy(),
                conv=conv_pool[slots.long()].float().cpu().numpy(), inter=inter, ci=ci, ks=ks)


def check(w, r, snap_seqs):
    ks = r["ks"]
    off = np.concatenate([[0], np.cumsum(ks)])
    res = oracle_seqs(w, w.tokens, ks)
    y_orc = np.concatenate([x.y for x in res])
    o_orc = np.concatenate([x.o for x in res])
    assert_y_close(r["y"], y_orc, "verify y", o_orc=o_orc)
    assert_core_close(r["core"], o_orc, "verify core o")
    for i, x in enumerate(res):
        assert_state_close(r["H"][i], x.H, f"final state seq {i}")
        np.testing.assert_array_equal(r["conv"][i], x.conv_state)
    # intermediates: intermediate t = state after t+1 tokens; slots t >= k-1 untouched
    snaps = oracle_seqs(w, w.tokens, ks, idx=snap_seqs, snapshots=True)
    for i, x in zip(snap_seqs, snaps):
        k = ks[i]
        got = r["inter"][i].cpu().numpy()
        for t in range(k - 1):
            assert_state_close(got[t], x.H_snap[t], f"seq {i} intermediate {t}")
        assert (got[k - 1:] == CANARY).all(), f"seq {i}: wrote beyond its k"
        if r["ci"] is not None:
            ci = r["ci"][i].float().cpu().numpy()
            for t in range(k - 1):
                np.testing.assert_array_equal(ci[t], x.conv_snap[t])
            assert (ci[k - 1:] == -7.0).all()
    # the outputs of sequence i are its rows off[i] .. off[i+1]
    assert r["y"].shape[0] == off[-1]


def test_verify_tiny_f32_all_k():
    w = wl.ragged_verify(n=15, shape=wl.TINY, seed=5, bf16=False)
    w.lens[:] = np.arange(2, 17)  # every k once
    w.tokens = wl.make_tokens(np.random.default_rng(6), wl.TINY, int(w.lens.sum()), bf16=False)
    r = run_verify(w)
    assert r["status"] == 0
    check(w, r, range(15))


def test_verify_full_128_ragged():
    w = wl.ragged_verify(n=128)
    r = run_verify(w, slot_perm=w.extra["slot_perm"])
    assert r["status"] == 0
    ks = w.lens
    # snapshots for a sample that covers k = 2 and k = 16 and a few in between
    sample = sorted({int(np.argmax(ks)), int(np.argmin(ks))} | set(range(0, 128, 17)))
    check(w, r, sample)


def test_verify_all_k16_and_all_k2():
    for k in (16, 2):
        w = wl.ragged_verify(n=9, k_lo=k, k_hi=k, seed=20 + k)
        r = run_verify(w, conv_inter=False)
        assert r["status"] == 0
        check(w, r, range(9))


def test_verify_null_entry_sets_status_and_skips_that_sequence():
    w = wl.ragged_verify(n=4, shape=wl.TINY, seed=7)
    w.lens[:] = [3, 5, 2, 4]
    w.tokens = wl.make_tokens(np.random.default_rng(8), wl.TINY, 14, bf16=True)
    r = run_verify(w, spoil=(2, 1))  # intermediate 1 of sequence 1 (k = 5) missing
    assert r["status"] == 16  # GDN_ERR_BAD_TABLE_ENTRY
    assert (r["inter"][1].cpu().numpy() == CANARY).all()
    np.testing.assert_array_equal(r["H"][1], w.H0[1])  # untouched
    res = oracle_seqs(w, w.tokens, [int(k) for k in w.lens])
    for i in (0, 2, 3):
        assert_state_close(r["H"][i], res[i].H, f"seq {i}")
