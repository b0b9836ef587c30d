"""GPU parity of gdn_prefill_chunked, gdn_conv_step and gdn_gated_rmsnorm against the
fp64 oracle (trait_layer.rs LayerSplitPrefill::prefill_gdn_full_batched_fla_varlen,
prefill_phase1_conv1d_one / prefill_phase1_l2_batched; layer_struct.rs
gated_rms_norm_f32_k)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import (assert_core_close, assert_state_close, assert_y_close, odims,
                              oracle_seqs, require_gpu, ELEM_FACTOR, F32_TOL, STATE_TOL,
                              TC_CORE_TOL, TC_ELEM_FACTOR, TC_STATE_TOL)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_prefill(w: wl.Workload, slot_perm=None, with_core=True):
    d = torch.device("cuda")
    sh = w.shape
    dims = dev.dims_of(sh)
    h_pool, conv_pool, slots = dev.states_to(w, d, slot_perm)
    sl = slots.long().cpu().numpy()
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
    hp = torch.tensor([h_pool.data_ptr() + int(s) * hsz for s in sl], dtype=torch.int64, device=d)
    cu = torch.from_numpy(w.cu_seqlens).to(d)
    T = int(w.lens.sum())
    ws_bytes = gdn.gdn_prefill_workspace_bytes(dims, w.n, T, int(w.lens.max()))
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=d) if ws_bytes else None
    y = torch.empty((T, sh.n_v_heads * sh.d_v), dtype=dev.act_dtype(w), device=d)
    core = (torch.empty((T, sh.n_v_heads, sh.d_v), dtype=torch.float32, device=d)
            if with_core else None)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    gdn.gdn_prefill_chunked(dims, dev.weights_to(w, d), dev.tokens_to(w.tokens, dev.act_dtype(w), d),
                            w.n, cu, T, int(w.lens.max()), hp, conv_pool, h_pool.shape[0], slots,
                            y, core, ws, status)
    torch.cuda.synchronize()
    return dict(status=int(status.item()), y=y, core=core, h_pool=h_pool, conv_pool=conv_pool,
                slots=slots)


def tensor_core_path(w) -> bool:
    """d = 128 with bf16 activations takes the tcgen05 chunked prefill."""
    return w.shape.d_k == 128 and w.bf16


def check_prefill(w, r):
    assert r["status"] == 0, gdn.status_string(r["status"])
    tc = tensor_core_path(w)
    res = oracle_seqs(w, w.tokens, [int(x) for x in w.lens])
    errs = {"y": assert_y_close(r["y"], np.concatenate([x.y for x in res]), "prefill y",
                                o_orc=np.concatenate([x.o for x in res]))}
    if r["core"] is not None:
        errs["core"] = assert_core_close(r["core"], np.concatenate([x.o for x in res]),
                                         "prefill core o", TC_CORE_TOL if tc else F32_TOL,
                                         TC_ELEM_FACTOR if tc else ELEM_FACTOR)
    sl = r["slots"].long()
    H = r["h_pool"][sl].cpu().numpy()
    conv = r["conv_pool"][sl].float().cpu().numpy()
    errs["state"] = 0.0
    for i, x in enumerate(res):
        errs["state"] = max(errs["state"], assert_state_close(
            H[i], x.H, f"state seq {i}", TC_STATE_TOL if tc else STATE_TOL,
            elem_factor=TC_ELEM_FACTOR if tc else ELEM_FACTOR))
        np.testing.assert_array_equal(conv[i], x.conv_state)
    print(f"{w.name}: rel errors {errs}")
    return res


def test_tiny_prefill_then_decode_f32():
    """64-token prefill from zero state, then 8 decode steps, f32 throughout."""
    for q_one in (False, True):
        w = wl.tiny_check(q_scale_one=q_one)
        r = run_prefill(w)
        check_prefill(w, r)
        d = torch.device("cuda")
        dims = dev.dims_of(w.shape)
        weights = dev.weights_to(w, d)
        status = torch.zeros(1, dtype=torch.int32, device=d)
        ys = []
        for tok in w.steps:
            y = torch.empty((1, 32), dtype=torch.float32, device=d)
            gdn.gdn_decode_batched(dims, weights, dev.tokens_to(tok, torch.float32, d), 1,
                                   r["h_pool"], r["conv_pool"], 1, r["slots"], y, None, status)
            ys.append(y)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        all_tok = {k: np.concatenate([w.tokens[k]] + [s[k] for s in w.steps]) for k in w.tokens}
        res = oracle_seqs(w, all_tok, [72])[0]
        assert_y_close(torch.cat(ys), res.y[64:], "decode y after prefill", o_orc=res.o[64:])
        assert_state_close(r["h_pool"][0].cpu().numpy(), res.H, "state after 72 tokens")
        np.testing.assert_array_equal(r["conv_pool"][0].cpu().numpy(), res.conv_state)


def test_varlen_prefill_tiny_bf16():
    w = wl.varlen_prefill([1, 5, 70, 3, 64, 65], shape=wl.TINY, seed=9)
    check_prefill(w, run_prefill(w, slot_perm=[3, 0, 5, 1, 2, 4]))


def test_varlen_prefill_full_small():
    """Tensor-core path: ragged last chunks, a sequence shorter than one chunk, exact
    multiples of 64, and non-zero initial states."""
    w = wl.varlen_prefill([100, 7, 129, 64, 1, 128], seed=11)
    assert tensor_core_path(w)
    check_prefill(w, run_prefill(w, slot_perm=[2, 5, 0, 1, 4, 3]))


def test_prefill_without_core_output():
    """No f32 core output requested: two sequences take the column-sliced spine, which
    hands O to the norm in fp16; y and the states still match."""
    w = wl.varlen_prefill([300, 77], seed=18)
    assert tensor_core_path(w)
    check_prefill(w, run_prefill(w, with_core=False))


@pytest.mark.parametrize("with_core", [True, False])
def test_prefill_sliced_spine_empty_and_ragged(with_core):
    """Column-sliced spine: an empty sequence (its chains leave at once) beside one with a
    3-token last chunk, and a single-token sequence on its own (its norm in the spare CTAs
    of the spine's launch)."""
    for lens, seed in (([0, 131], 19), ([1], 20)):
        w = wl.varlen_prefill(lens, seed=seed)
        assert tensor_core_path(w) and w.n * w.shape.n_v_heads * 2 <= 152
        r = run_prefill(w, with_core=with_core)
        check_prefill(w, r)
        if lens[0] == 0:
            np.testing.assert_array_equal(r["h_pool"][0].cpu().numpy(), w.H0[0])


@pytest.mark.parametrize("n,with_core", [(9, False), (9, True), (16, False)])
def test_prefill_sliced_spine_norm_ctas(n, with_core):
    """d = 128 with 4 value heads.  9 sequences: 36 (sequence, head) units whose two column
    slices take 72 SMs; the 80 left run the norm, up to four 8-row parts of a chunk each,
    over sequences of every length class (empty, one token, one chunk, ragged).  16
    sequences leave fewer than two spare SMs per head, and the norm runs as its own kernel
    after the chains."""
    shape = wl.LayerShape(1, 4, 128, 128, 4, q_scale=128 ** -0.5)
    rng = np.random.default_rng(21 + n)
    lens = rng.integers(1, 160, size=n)
    lens[:4] = [64, 0, 129, 1]
    w = wl.varlen_prefill(lens, shape=shape, seed=21 + n)
    assert tensor_core_path(w)
    check_prefill(w, run_prefill(w, with_core=with_core))


def test_prefill_norm_ctas_bad_seqlens_sets_status():
    """Tensor-core path with norm CTAs beside the chains (4 value heads, 2 sequences): a
    decreasing cu_seqlens is reported on the status word, and the norm CTAs, which skip
    what the chains skip, wait on nothing."""
    shape = wl.LayerShape(1, 4, 128, 128, 4, q_scale=128 ** -0.5)
    w = wl.varlen_prefill([9, 2], shape=shape, seed=25)
    assert tensor_core_path(w)
    d = torch.device("cuda")
    dims = dev.dims_of(shape)
    h_pool, conv_pool, slots = dev.states_to(w, d)
    hsz = shape.n_v_heads * shape.d_k * shape.d_v * 4
    hp = torch.tensor([h_pool.data_ptr() + i * hsz for i in range(2)], dtype=torch.int64, device=d)
    cu = torch.from_numpy(np.array([0, 9, 7], np.int32)).to(d)  # decreasing: invalid
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(dims, 2, 11, 9), dtype=torch.uint8, device=d)
    y = torch.zeros((11, shape.n_v_heads * shape.d_v), dtype=torch.bfloat16, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    gdn.gdn_prefill_chunked(dims, dev.weights_to(w, d), dev.tokens_to(w.tokens, torch.bfloat16, d),
                            2, cu, 11, 9, hp, conv_pool, 2, slots, y, None, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 18  # GDN_ERR_BAD_SEQLENS


def test_prefill_norm_ctas_in_cuda_graph():
    """The cooperative two-slice spine (one sequence, norm CTAs beside the chains) captured
    in a CUDA graph and replayed gives y and the state bit for bit as an eager call does."""
    w = wl.varlen_prefill([200], seed=27)
    assert tensor_core_path(w)
    d = torch.device("cuda")
    sh = w.shape
    dims = dev.dims_of(sh)
    T = int(w.lens.sum())
    cu = torch.from_numpy(w.cu_seqlens).to(d)
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(dims, 1, T, T), dtype=torch.uint8, device=d)
    weights = dev.weights_to(w, d)
    tokens = dev.tokens_to(w.tokens, torch.bfloat16, d)
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
    outs = []
    for graph in (False, True):
        h_pool, conv_pool, slots = dev.states_to(w, d)
        hp = torch.tensor([h_pool.data_ptr() + int(slots[0]) * hsz], dtype=torch.int64, device=d)
        y = torch.empty((T, sh.n_v_heads * sh.d_v), dtype=torch.bfloat16, device=d)
        status = torch.zeros(1, dtype=torch.int32, device=d)

        def call(st):
            gdn.gdn_prefill_chunked(dims, weights, tokens, 1, cu, T, T, hp, conv_pool, 1, slots,
                                    y, None, ws, status, st)

        if graph:
            side = torch.cuda.Stream(d)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                call(side)
            g.replay()
        else:
            call(torch.cuda.current_stream(d))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append((y.clone(), h_pool[slots.long()].clone()))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])


def test_varlen_prefill_full_f32_sequential():
    """d = 128 with f32 activations runs the token-sequential kernel (f32 class)."""
    rng = np.random.default_rng(15)
    w = wl.varlen_prefill([70, 5, 64], seed=15)
    w.bf16 = False
    w.tokens = wl.make_tokens(rng, wl.FULL, 139, bf16=False)
    w.conv0 = rng.standard_normal(w.conv0.shape).astype(np.float32) * np.float32(0.3)
    check_prefill(w, run_prefill(w))


def test_prefill_many_short_sequences():
    """520 sequences of 0..4 tokens on the tensor-core path: more sequences than the
    spine orders by length (512), so its units go in call order; empty sequences keep
    their states."""
    rng = np.random.default_rng(17)
    lens = rng.integers(0, 5, size=520)
    lens[:3] = [0, 4, 1]
    w = wl.varlen_prefill(lens, seed=17)
    assert tensor_core_path(w)
    r = run_prefill(w)
    check_prefill(w, r)
    for i in np.flatnonzero(lens == 0)[:5]:
        np.testing.assert_array_equal(r["h_pool"][i].cpu().numpy(), w.H0[i])


def test_prefill_zero_length_sequence_keeps_state():
    w = wl.varlen_prefill([65, 0, 3], seed=16)
    r = run_prefill(w)
    check_prefill(w, r)
    np.testing.assert_array_equal(r["h_pool"][1].cpu().numpy(), w.H0[1])


@pytest.mark.slow
def test_long_prefill_8192():
    w = wl.long_prefill(8192)
    check_prefill(w, run_prefill(w))


def test_prefill_bad_seqlens_sets_status():
    w = wl.varlen_prefill([5, 6], shape=wl.TINY, seed=12)
    w_cu = w.cu_seqlens.copy()
    d = torch.device("cuda")
    sh = w.shape
    h_pool, conv_pool, slots = dev.states_to(w, d)
    hp = torch.tensor([h_pool[i].data_ptr() for i in range(2)], dtype=torch.int64, device=d)
    cu = torch.from_numpy(np.array([0, 9, 7], np.int32)).to(d)  # decreasing: invalid
    y = torch.zeros((11, 32), dtype=torch.bfloat16, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    gdn.gdn_prefill_chunked(dev.dims_of(sh), dev.weights_to(w, d),
                            dev.tokens_to(w.tokens, torch.bfloat16, d), 2, cu, 11, 9, hp,
                            conv_pool, 2, slots, y, None, None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 18  # GDN_ERR_BAD_SEQLENS
    assert w_cu[-1] == 11


@pytest.mark.parametrize("shape,lens,bf16", [(wl.TINY, [3, 1, 9], False),
                                             (wl.FULL, [5, 70, 2], True)])
def test_conv_step(shape, lens, bf16):
    rng = np.random.default_rng(13)
    w = wl.varlen_prefill(lens, shape=shape, seed=13)
    if not bf16:
        w.bf16 = False
        w.tokens = wl.make_tokens(rng, shape, int(sum(lens)), bf16=False)
        w.conv0 = rng.standard_normal(w.conv0.shape).astype(np.float32)
    d = torch.device("cuda")
    _, conv_pool, slots = dev.states_to(w, d)
    cu = torch.from_numpy(w.cu_seqlens).to(d)
    T = int(sum(lens))
    out = torch.empty((T, shape.conv_dim), dtype=torch.float32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    gdn.gdn_conv_step(dev.dims_of(shape), dev.weights_to(w, d),
                      dev.tokens_to(w.tokens, dev.act_dtype(w), d), len(lens), cu, T, conv_pool,
                      len(lens), slots, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    od = odims(shape)
    got = out.cpu().numpy()
    off = w.cu_seqlens
    for i in range(len(lens)):
        xc, st, _ = oracle.conv(w.weights["conv_w"], w.conv0[i], w.tokens["qkv"][off[i]:off[i + 1]])
        qn, kn, v = oracle.l2norm_split(od, xc)
        g = got[off[i]:off[i + 1]]
        Hk, dk = shape.n_k_heads, shape.d_k
        np.testing.assert_allclose(g[:, :Hk * dk], qn.reshape(len(qn), -1), rtol=2e-5, atol=2e-6)
        np.testing.assert_allclose(g[:, Hk * dk:2 * Hk * dk], kn.reshape(len(kn), -1), rtol=2e-5,
                                   atol=2e-6)
        np.testing.assert_allclose(g[:, 2 * Hk * dk:], v.reshape(len(v), -1), rtol=2e-5,
                                   atol=2e-5)
        np.testing.assert_array_equal(conv_pool[i].float().cpu().numpy(), st)


@pytest.mark.parametrize("shape,bf16", [(wl.TINY, False), (wl.FULL, True)])
def test_gated_rmsnorm(shape, bf16):
    rng = np.random.default_rng(14)
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
                          torch.from_numpy(w).to(d), 1e-6, y)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(o, z, w, float(np.float32(1e-6)))
    assert_y_close(y, ref, "gated rmsnorm")


def test_mixed_serving_step_two_streams():
    """32 varlen prefills (U{512..4096}) on one stream next to a 96-sequence ragged verify on
    another, as one serving step; sampled sequences are compared with the oracle."""
    pre, ver = wl.mixed_serving()
    d = torch.device("cuda")
    dims, weights = dev.dims_of(pre.shape), dev.weights_to(pre, d)
    ph, pc, ps = dev.states_to(pre, d)
    hsz = 32 * 128 * 128 * 4
    php = torch.tensor([ph.data_ptr() + i * hsz for i in range(pre.n)], dtype=torch.int64, device=d)
    cu = torch.from_numpy(pre.cu_seqlens).to(d)
    T, Lmax = int(pre.lens.sum()), int(pre.lens.max())
    py = torch.empty((T, 4096), dtype=torch.bfloat16, device=d)
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(dims, pre.n, T, Lmax), dtype=torch.uint8,
                     device=d)
    ks = [int(k) for k in ver.lens]
    vh, vc, vs = dev.states_to(ver, d)
    inter = torch.zeros((ver.n, 15, 32, 128, 128), dtype=torch.float32, device=d)
    tables = dev.wy_tables_to(ks, [vh.data_ptr() + i * hsz for i in range(ver.n)],
                              [[inter[i, t].data_ptr() for t in range(15)] for i in range(ver.n)], d)
    vy = torch.empty((sum(ks), 4096), dtype=torch.bfloat16, device=d)
    status = torch.zeros(2, dtype=torch.int32, device=d)
    s_pre, s_ver = torch.cuda.Stream(d), torch.cuda.Stream(d)
    pin = dev.tokens_to(pre.tokens, torch.bfloat16, d)
    vin = dev.tokens_to(ver.tokens, torch.bfloat16, d)
    torch.cuda.synchronize()  # every input is on the device before either side stream starts
    gdn.gdn_prefill_chunked(dims, weights, pin, pre.n, cu, T, Lmax, php, pc, pre.n, ps, py, None,
                            ws, status[0:1], s_pre)
    gdn.gdn_verify_multi(dims, weights, vin, ver.n, ks, tables, vc, ver.n, vs, None, vy, None,
                         status[1:2], s_ver)
    torch.cuda.synchronize()
    assert int(status.abs().sum().item()) == 0
    # prefill: the four shortest sequences and the two longest (which run next to the
    # verify for most of the step), in full
    off = pre.cu_seqlens
    order = np.argsort(pre.lens, kind="stable")
    idx = [int(i) for i in order[:4]] + [int(i) for i in order[-2:]]
    res = oracle_seqs(pre, pre.tokens, [int(x) for x in pre.lens], idx=idx)
    H = ph.cpu().numpy()
    for i, x in zip(idx, res):
        assert_y_close(py[off[i]:off[i + 1]], x.y, f"prefill y seq {i}", o_orc=x.o)
        assert_state_close(H[i], x.H, f"prefill state seq {i}", TC_STATE_TOL,
                           elem_factor=TC_ELEM_FACTOR)
        np.testing.assert_array_equal(pc[i].float().cpu().numpy(), x.conv_state)
    # verify: every sequence's outputs and final state, intermediates of a sample
    resv = oracle_seqs(ver, ver.tokens, ks)
    assert_y_close(vy, np.concatenate([x.y for x in resv]), "verify y",
                   o_orc=np.concatenate([x.o for x in resv]))
    Hv = vh.cpu().numpy()
    for i, x in enumerate(resv):
        assert_state_close(Hv[i], x.H, f"verify state seq {i}")
