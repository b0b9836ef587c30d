"""GPU parity of the half-width h-state pools (layer_struct.rs: the FP16 h-state variants
gdn_f16_norm_k, gdn_wyn_f16_table_k and the width converters ssm_h_f16_to_f32_k /
ssm_h_f32_to_f16_k): gdn_decode_batched_h16, gdn_verify_multi_h16, the fold on fp16 states
and gdn_state_convert, against the fp64 oracle with binary16 state storage.

Tolerance: the kernels update in f32 and round each stored state to fp16; the oracle
updates in fp64 and rounds the same way, so now and then one element lands one fp16 step
(2^-10 relative) apart and the difference is carried forward.  States and the f32 core
output are held to 1e-3 relative; bf16 outputs keep the 2e-3 of every bf16 output; conv
states stay bit-exact.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import (assert_core_close, assert_state_close, assert_y_close, odims,
                              require_gpu)

pytestmark = pytest.mark.gpu

H16_TOL = 1e-3
H16_ULP = 2.0 ** -10  # spacing of binary16 relative to the value (at most)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def oracle_h16(w, token_rows, lens, H0, snapshots=False, idx=None):
    """The oracle with binary16 state storage over the sequences in idx (default: all)."""
    dims = dataclasses.replace(odims(w.shape), h_fp16=True)
    off = np.concatenate([[0], np.cumsum(lens)])
    idx = range(len(lens)) if idx is None else idx
    seqs = [dict(qkv=token_rows["qkv"][off[i]:off[i + 1]], z=token_rows["z"][off[i]:off[i + 1]],
                 a=token_rows["a"][off[i]:off[i + 1]], b=token_rows["b"][off[i]:off[i + 1]],
                 conv_state=w.conv0[i], H=H0[i]) for i in idx]
    return oracle.mixer_batch(dims, w.weights, seqs, snapshots=snapshots)


def run_decode_h16(w, slot_perm=None):
    d = torch.device("cuda")
    sh = w.shape
    act = dev.act_dtype(w)
    h_pool, conv_pool, slots = dev.states_to(w, d, slot_perm)
    h16 = h_pool.half()
    sl = slots.long()
    H0 = h16[sl].double().cpu().numpy()
    dims, weights = dev.dims_of(sh), dev.weights_to(w, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    ys, cores = [], []
    for tok in [w.tokens] + w.steps:
        y = torch.empty((w.n, sh.n_v_heads * sh.d_v), dtype=act, device=d)
        core = torch.empty((w.n, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=d)
        gdn.gdn_decode_batched_h16(dims, weights, dev.tokens_to(tok, act, d), w.n, h16,
                                   conv_pool, h16.shape[0], slots, y, core, status)
        ys.append(y)
        cores.append(core)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ys, cores, h16, conv_pool, sl, H0


def test_decode_h16_tiny_f32_activations():
    w = wl.batched_decode(n=5, steps=8, shape=wl.TINY, seed=1, bf16=False)
    ys, cores, h16, conv_pool, sl, H0 = run_decode_h16(w)
    steps = [w.tokens] + w.steps
    rows = {k: np.stack([s[k] for s in steps], axis=1).reshape(w.n * len(steps), -1)
            for k in ("qkv", "z", "a", "b")}
    res = oracle_h16(w, rows, [len(steps)] * w.n, H0)
    for s in range(len(steps)):
        assert_y_close(ys[s], np.stack([r.y for r in res])[:, s], f"y step {s}", tol=H16_TOL,
                       o_orc=np.stack([r.o for r in res])[:, s])
    H = h16[sl].double().cpu().numpy()
    for i, r in enumerate(res):
        assert_state_close(H[i], r.H, f"fp16 state seq {i}", H16_TOL, H16_ULP)
        np.testing.assert_array_equal(conv_pool[sl][i].cpu().numpy(), r.conv_state)


@pytest.mark.parametrize("G", [1, 3, 4])
def test_decode_h16_head_groupings(G):
    """fp16-pool decode takes an item's value heads two at a time: G = 3 mixes a pair and a
    single head, G = 4 two pairs, G = 1 only the single-head path."""
    shape = wl.LayerShape(2, 2 * G, 16, 16, 4, q_scale=16 ** -0.5)
    w = wl.batched_decode(n=6, steps=5, shape=shape, seed=20 + G)
    ys, cores, h16, conv_pool, sl, H0 = run_decode_h16(w, w.extra["slot_perm"])
    steps = [w.tokens] + w.steps
    rows = {k: np.stack([s[k] for s in steps], axis=1).reshape(w.n * len(steps), -1)
            for k in ("qkv", "z", "a", "b")}
    res = oracle_h16(w, rows, [len(steps)] * w.n, H0)
    y_orc = np.stack([r.y for r in res])
    for s in range(len(steps)):
        assert_y_close(ys[s], y_orc[:, s], f"G={G} y step {s}",
                       o_orc=np.stack([r.o for r in res])[:, s])
    H = h16[sl].double().cpu().numpy()
    for i, r in enumerate(res):
        assert_state_close(H[i], r.H, f"G={G} fp16 state seq {i}", H16_TOL, H16_ULP)


def test_decode_h16_128_sequences_64_steps():
    w = wl.batched_decode(n=128, steps=64, seed=3)
    ys, cores, h16, conv_pool, sl, H0 = run_decode_h16(w, w.extra["slot_perm"])
    steps = [w.tokens] + w.steps
    rows = {k: np.stack([s[k] for s in steps], axis=1).reshape(w.n * len(steps), -1)
            for k in ("qkv", "z", "a", "b")}
    res = oracle_h16(w, rows, [len(steps)] * w.n, H0)
    y_orc = np.stack([r.y for r in res])
    o_orc = np.stack([r.o for r in res])
    for s in range(len(steps)):
        assert_y_close(ys[s], y_orc[:, s], f"y step {s}", o_orc=o_orc[:, s])
        assert_core_close(cores[s], o_orc[:, s], f"core step {s}", H16_TOL)
    H = h16[sl].double().cpu().numpy()
    conv = conv_pool[sl].float().cpu().numpy()
    for i, r in enumerate(res):
        assert_state_close(H[i], r.H, f"fp16 state seq {i}", H16_TOL, H16_ULP)
        np.testing.assert_array_equal(conv[i], r.conv_state)


def _verify_h16(w):
    d = torch.device("cuda")
    n, sh = w.n, w.shape
    ks = [int(k) for k in w.lens]
    h_pool, conv_pool, slots = dev.states_to(w, d)
    h16 = h_pool.half()
    H0 = h16[slots.long()].double().cpu().numpy()
    inter = torch.zeros((n, 15, sh.n_v_heads, sh.d_k, sh.d_v), dtype=torch.float16, device=d)
    ci = torch.zeros((n, 15, sh.conv_dim, sh.d_conv), dtype=torch.bfloat16, device=d)
    sl = slots.long().cpu().numpy()
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 2
    tables = dev.wy_tables_to(ks, [h16.data_ptr() + int(sl[i]) * hsz for i in range(n)],
                              [[inter[i, t].data_ptr() for t in range(15)] for i in range(n)], d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    y = torch.empty((sum(ks), sh.n_v_heads * sh.d_v), dtype=torch.bfloat16, device=d)
    core = torch.empty((sum(ks), sh.n_v_heads, sh.d_v), dtype=torch.float32, device=d)
    gdn.gdn_verify_multi_h16(dev.dims_of(sh), dev.weights_to(w, d),
                             dev.tokens_to(w.tokens, torch.bfloat16, d), n, ks, tables, conv_pool,
                             h16.shape[0], slots, ci, y, core, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dict(ks=ks, H0=H0, h16=h16, slots=slots, inter=inter, ci=ci, y=y, core=core,
                tables=tables, conv_pool=conv_pool, status=status)


def test_verify_h16_128_ragged_with_intermediates():
    w = wl.ragged_verify(n=128, seed=41)
    r = _verify_h16(w)
    ks = r["ks"]
    res = oracle_h16(w, w.tokens, ks, r["H0"])
    assert_y_close(r["y"], np.concatenate([x.y for x in res]), "verify y",
                   o_orc=np.concatenate([x.o for x in res]))
    assert_core_close(r["core"], np.concatenate([x.o for x in res]), "verify core", H16_TOL)
    H = r["h16"][r["slots"].long()].double().cpu().numpy()
    conv = r["conv_pool"][r["slots"].long()].float().cpu().numpy()
    for i, x in enumerate(res):
        assert_state_close(H[i], x.H, f"final fp16 state seq {i}", H16_TOL, H16_ULP)
        np.testing.assert_array_equal(conv[i], x.conv_state)
    sample = sorted({int(np.argmax(ks)), int(np.argmin(ks))} | set(range(0, 128, 21)))
    snaps = oracle_h16(w, w.tokens, ks, r["H0"], snapshots=True, idx=sample)
    for i, x in zip(sample, snaps):
        got = r["inter"][i].double().cpu().numpy()
        for t in range(ks[i] - 1):
            assert_state_close(got[t], x.H_snap[t], f"seq {i} intermediate {t}", H16_TOL, H16_ULP)


def test_fold_on_fp16_states():
    w = wl.ragged_verify(n=16, seed=42)
    r = _verify_h16(w)
    ks = r["ks"]
    rng = np.random.default_rng(43)
    m = np.array([rng.integers(1, k + 1) for k in ks], np.int32)
    after_k = r["h16"][r["slots"].long()].clone()
    acc = torch.tensor(m, device="cuda")
    gdn.gdn_fold_accepted(dev.dims_of(w.shape), w.n, ks, acc, r["tables"], r["conv_pool"],
                          r["h16"].shape[0], r["slots"], r["ci"], gdn.GDN_DTYPE_BF16,
                          r["status"], h_dtype=gdn.GDN_DTYPE_F16)
    torch.cuda.synchronize()
    assert int(r["status"].item()) == 0
    H = r["h16"][r["slots"].long()]
    for i in range(w.n):
        expect = r["inter"][i, m[i] - 1] if m[i] < ks[i] else after_k[i]
        assert torch.equal(H[i], expect), i
        conv = r["conv_pool"][r["slots"][i].long()]
        if m[i] < ks[i]:
            assert torch.equal(conv, r["ci"][i, m[i] - 1]), i


@pytest.mark.parametrize("count", [8, 1_000_003])
def test_state_convert_round_trip(count):
    d = torch.device("cuda")
    x = torch.randn(count + 8, dtype=torch.float32, device=d)[:count] * 3.0
    x[: min(4, count)] = torch.tensor([65519.0, 65520.0, 1e-8, -0.0][: min(4, count)], device=d)
    h = torch.empty(count + 8, dtype=torch.float16, device=d)[:count]
    gdn.gdn_state_convert(x, gdn.GDN_DTYPE_F32, h, gdn.GDN_DTYPE_F16, count)
    back = torch.empty(count, dtype=torch.float32, device=d)
    gdn.gdn_state_convert(h, gdn.GDN_DTYPE_F16, back, gdn.GDN_DTYPE_F32, count)
    torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int16), x.half().view(torch.int16))
    assert torch.equal(back, h.float())
