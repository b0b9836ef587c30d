"""GPU parity of the write-on-accept verify and its deferred fold (trait_layer.rs,
LayerWriteOnAccept: gdn_woa_stash_seq_floats, gdn_woa_bind; layer_struct.rs, the
gdn_wy4_woa_k / gdn_wy4_fold_k / gdn_wy4_clear_k handles).

gdn_verify_woa must give the outputs of the verify while leaving every state as it was;
gdn_woa_fold then moves each sequence to the state and conv state after its m accepted
drafts, which the oracle's token loop over the first m rows defines; gdn_woa_clear disarms
the stash, after which a fold changes nothing."""
import numpy as np
import pytest
import torch

from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import (assert_core_close, assert_state_close, assert_y_close,
                              oracle_seqs, require_gpu)
from tests.test_fold_gpu import prefix_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_woa(w: wl.Workload, slot_perm=None):
    d = torch.device("cuda")
    n, sh = w.n, w.shape
    ks = [int(k) for k in w.lens]
    h_pool, conv_pool, slots = dev.states_to(w, d, slot_perm)
    sl = slots.long().cpu().numpy()
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
    # only table 0 is read: the intermediate tables stay zero
    tables = dev.wy_tables_to(ks, [h_pool.data_ptr() + int(sl[i]) * hsz for i in range(n)],
                              [[0] * 15 for _ in range(n)], d)
    dims = dev.dims_of(sh)
    words = gdn.gdn_woa_stash_seq_floats(dims, gdn.GDN_DTYPE_BF16 if w.bf16 else gdn.GDN_DTYPE_F32)
    assert words > 0
    stash = torch.full((n + 1, words), float("nan"), dtype=torch.float32, device=d)
    flag = torch.zeros(1, dtype=torch.int32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    rows = sum(ks)
    y = torch.empty((rows, sh.n_v_heads * sh.d_v), dtype=dev.act_dtype(w), device=d)
    core = torch.empty((rows, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=d)
    h_before, c_before = h_pool.clone(), conv_pool.clone()
    gdn.gdn_verify_woa(dims, dev.weights_to(w, d), dev.tokens_to(w.tokens, dev.act_dtype(w), d),
                       n, ks, tables, conv_pool, h_pool.shape[0], slots, stash, n + 1, flag, y,
                       core, status)
    torch.cuda.synchronize()
    return dict(status=int(status.item()), y=y, core=core, h_pool=h_pool, conv_pool=conv_pool,
                slots=slots, tables=tables, stash=stash, flag=flag, ks=ks, dims=dims,
                h_before=h_before, c_before=c_before)


def fold(w, r, m):
    d = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=d)
    acc = torch.tensor(np.asarray(m, np.int32), device=d)
    gdn.gdn_woa_fold(r["dims"], w.n, acc, r["tables"], r["conv_pool"], r["h_pool"].shape[0],
                     r["slots"], r["stash"], r["flag"],
                     gdn.GDN_DTYPE_BF16 if w.bf16 else gdn.GDN_DTYPE_F32, status)
    torch.cuda.synchronize()
    return int(status.item())


def check_verify_outputs(w, r):
    assert r["status"] == 0, gdn.status_string(r["status"])
    assert int(r["flag"].item()) == 1, "the verify engages the stash"
    # no state moved
    assert torch.equal(r["h_pool"], r["h_before"])
    assert torch.equal(r["conv_pool"], r["c_before"])
    res = oracle_seqs(w, w.tokens, r["ks"])
    o_orc = np.concatenate([x.o for x in res])
    assert_y_close(r["y"], np.concatenate([x.y for x in res]), "woa verify y", o_orc=o_orc)
    assert_core_close(r["core"], o_orc, "woa verify core o")
    # the stash of sequence i starts with k_i
    k_read = r["stash"][:w.n, 0].view(torch.int32).cpu().numpy()
    np.testing.assert_array_equal(k_read, r["ks"])


def check_fold(w, r, m):
    ks = r["ks"]
    res = oracle_seqs(w, prefix_rows(w, ks, m), m)
    sl = r["slots"].long()
    H = r["h_pool"][sl].cpu().numpy()
    conv = r["conv_pool"][sl].float().cpu().numpy()
    for i, x in enumerate(res):
        assert_state_close(H[i], x.H, f"folded state seq {i} (m={m[i]}, k={ks[i]})")
        np.testing.assert_array_equal(conv[i], x.conv_state)


@pytest.mark.parametrize("bf16", [True, False])
def test_woa_verify_fold_clear_tiny(bf16):
    w = wl.ragged_verify(n=15, shape=wl.TINY, seed=91, bf16=bf16)
    w.lens[:] = np.arange(2, 17)
    w.tokens = wl.make_tokens(np.random.default_rng(92), wl.TINY, int(w.lens.sum()), bf16=bf16)
    r = run_woa(w, slot_perm=np.random.default_rng(93).permutation(15))
    check_verify_outputs(w, r)
    m = np.array([1 + (i * 7) % k for i, k in enumerate(w.lens)], np.int32)
    m[0], m[-1] = w.lens[0], 1  # everything accepted; only the first draft
    assert fold(w, r, m) == 0
    check_fold(w, r, m)
    # disarmed: a second fold is a no-op
    after = (r["h_pool"].clone(), r["conv_pool"].clone())
    gdn.gdn_woa_clear(r["flag"])
    torch.cuda.synchronize()
    assert int(r["flag"].item()) == 0
    assert fold(w, r, m) == 0
    assert torch.equal(r["h_pool"], after[0]) and torch.equal(r["conv_pool"], after[1])


def test_woa_full_128_ragged_matches_the_copy_fold():
    """128 sequences, k ~ U{2..16}: the deferred fold lands where the oracle's token loop does
    after m tokens, and within the f32 tolerance of the copy-form fold after gdn_verify_multi."""
    w = wl.ragged_verify(n=128, seed=94)
    rng = np.random.default_rng(95)
    m = np.array([rng.integers(1, k + 1) for k in w.lens], np.int32)
    r = run_woa(w, slot_perm=w.extra["slot_perm"])
    check_verify_outputs(w, r)
    assert fold(w, r, m) == 0
    check_fold(w, r, m)
    # the copy form on the same inputs
    from tests.test_fold_gpu import verify_then_fold
    c = verify_then_fold(w, m, slot_perm=w.extra["slot_perm"])
    assert c["status"] == 0
    H = r["h_pool"][r["slots"].long()].cpu().numpy()
    for i in range(w.n):
        assert_state_close(H[i], c["H"][i], f"woa vs copy fold seq {i}")
    np.testing.assert_array_equal(r["conv_pool"][r["slots"].long()].float().cpu().numpy(), c["conv"])


def test_woa_fold_refuses_a_count_outside_1_to_k():
    w = wl.ragged_verify(n=3, shape=wl.TINY, seed=96)
    w.lens[:] = [4, 4, 4]
    w.tokens = wl.make_tokens(np.random.default_rng(97), wl.TINY, 12, bf16=True)
    r = run_woa(w)
    check_verify_outputs(w, r)
    assert fold(w, r, [0, 2, 5]) == 20  # GDN_ERR_BAD_ACCEPTED
    sl = r["slots"].long()
    for i in (0, 2):  # the bad sequences keep their states
        assert torch.equal(r["h_pool"][sl[i]], r["h_before"][sl[i]])
        assert torch.equal(r["conv_pool"][sl[i]], r["c_before"][sl[i]])
    res = oracle_seqs(w, prefix_rows(w, r["ks"], [4, 2, 4]), [4, 2, 4], idx=[1])
    assert_state_close(r["h_pool"][sl[1]].cpu().numpy(), res[0].H, "seq 1 (m=2)")
