"""GPU parity of gdn_fold_accepted (trait_layer.rs, LayerWriteOnAccept::gdn_fold_accepted;
layer_struct.rs, gdn_wy4_fold_k): after a ragged verify and a fold with m_i accepted
drafts, sequence i holds exactly the state and conv state of m_i sequential decode steps."""
import numpy as np
import pytest
import torch

from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import assert_state_close, oracle_seqs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def verify_then_fold(w: wl.Workload, accepted, slot_perm=None):
    """Runs the verify (with conv intermediates) and the fold.  Returns the folded states
    and conv states per sequence, the verify's intermediates and the status word."""
    d = torch.device("cuda")
    n, sh = w.n, w.shape
    ks = [int(k) for k in w.lens]
    h_pool, conv_pool, slots = dev.states_to(w, d, slot_perm)
    inter = torch.zeros((n, 15, sh.n_v_heads, sh.d_k, sh.d_v), dtype=torch.float32, device=d)
    ci = torch.zeros((n, 15, sh.conv_dim, sh.d_conv), dtype=dev.act_dtype(w), device=d)
    sl = slots.long().cpu().numpy()
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
    tables = dev.wy_tables_to(ks, [h_pool.data_ptr() + int(sl[i]) * hsz for i in range(n)],
                              [[inter[i, t].data_ptr() for t in range(15)] for i in range(n)], d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    rows = sum(ks)
    y = torch.empty((rows, sh.n_v_heads * sh.d_v), dtype=dev.act_dtype(w), device=d)
    dims = dev.dims_of(sh)
    gdn.gdn_verify_multi(dims, dev.weights_to(w, d), dev.tokens_to(w.tokens, dev.act_dtype(w), d),
                         n, ks, tables, conv_pool, h_pool.shape[0], slots, ci, y, None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    after_k = (h_pool[slots.long()].cpu().numpy(), conv_pool[slots.long()].float().cpu().numpy())
    acc = torch.tensor(np.asarray(accepted, np.int32), device=d)
    code = gdn.GDN_DTYPE_BF16 if w.bf16 else gdn.GDN_DTYPE_F32
    gdn.gdn_fold_accepted(dims, n, ks, acc, tables, conv_pool, h_pool.shape[0], slots, ci, code,
                          status)
    torch.cuda.synchronize()
    return dict(status=int(status.item()), H=h_pool[slots.long()].cpu().numpy(),
                conv=conv_pool[slots.long()].float().cpu().numpy(), inter=inter.cpu().numpy(),
                after_k=after_k, ks=ks)


def prefix_rows(w: wl.Workload, ks, m):
    """The first m_i token rows of every sequence (rows are sequence-major)."""
    off = np.concatenate([[0], np.cumsum(ks)])
    idx = np.concatenate([np.arange(off[i], off[i] + m[i]) for i in range(len(ks))])
    return {key: v[idx] for key, v in w.tokens.items()}


def check_fold(w, r, m):
    ks = r["ks"]
    res = oracle_seqs(w, prefix_rows(w, ks, m), m)
    for i, x in enumerate(res):
        if m[i] < ks[i]:
            # the copy is exact: the folded state is the verify's intermediate m - 1
            np.testing.assert_array_equal(r["H"][i], r["inter"][i, m[i] - 1])
        else:
            np.testing.assert_array_equal(r["H"][i], r["after_k"][0][i])
            np.testing.assert_array_equal(r["conv"][i], r["after_k"][1][i])
        assert_state_close(r["H"][i], x.H, f"folded state seq {i} (m={m[i]}, k={ks[i]})")
        np.testing.assert_array_equal(r["conv"][i], x.conv_state)


def test_fold_full_128_ragged():
    w = wl.ragged_verify(n=128, seed=31)
    rng = np.random.default_rng(32)
    m = np.array([rng.integers(1, k + 1) for k in w.lens], np.int32)
    m[:3] = 1                 # roll back to the first draft
    m[3:6] = w.lens[3:6]      # everything accepted: nothing moves
    r = verify_then_fold(w, m, slot_perm=w.extra["slot_perm"])
    assert r["status"] == 0
    check_fold(w, r, m)


def test_fold_tiny_f32_every_m():
    w = wl.ragged_verify(n=15, shape=wl.TINY, seed=33, bf16=False)
    w.lens[:] = 16
    w.tokens = wl.make_tokens(np.random.default_rng(34), wl.TINY, int(w.lens.sum()), bf16=False)
    m = np.arange(1, 16, dtype=np.int32)  # m = 1 .. 15 of k = 16
    r = verify_then_fold(w, m)
    assert r["status"] == 0
    check_fold(w, r, m)


def test_fold_refuses_a_count_outside_1_to_k():
    w = wl.ragged_verify(n=3, shape=wl.TINY, seed=35)
    w.lens[:] = [4, 4, 4]
    w.tokens = wl.make_tokens(np.random.default_rng(36), wl.TINY, 12, bf16=True)
    r = verify_then_fold(w, [0, 2, 5])
    assert r["status"] == 20  # GDN_ERR_BAD_ACCEPTED
    # the two bad sequences keep the state after all k tokens; the good one is folded
    for i in (0, 2):
        np.testing.assert_array_equal(r["H"][i], r["after_k"][0][i])
        np.testing.assert_array_equal(r["conv"][i], r["after_k"][1][i])
    np.testing.assert_array_equal(r["H"][1], r["inter"][1, 1])
