"""Host-side tests of the C ABI (no GPU): the library loads, exports every symbol the
header declares, refuses bad arguments before touching CUDA, and fills the WY pointer
tables in the layout of transformer_layer.rs (VERIFY_WY_TABLE_SEQS and friends)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    from gated_deltanet_layer_conv1d_gb300 import _build
    _build.build()
    from gated_deltanet_layer_conv1d_gb300 import gdn
    return gdn


def _header():
    with open(os.path.join(ROOT, "include", "gdn.h")) as f:
        return f.read()


def test_exports_every_declared_symbol(g):
    declared = re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", _header())
    assert set(declared) == set(g.EXPORTS)
    L = ctypes.CDLL(g.LIB_PATH)
    for name in declared:
        assert hasattr(L, name), name


def test_header_constants_match_the_table_layout():
    h = _header()
    val = lambda k: re.search(rf"#define {k} (\d+)", h).group(1)
    assert int(val("GDN_VERIFY_WY_TABLE_SEQS")) == 128
    assert int(val("GDN_VERIFY_WY_TABLES_PER_LAYER")) == 16
    assert "GDN_VERIFY_WY_TABLE_STRIDE_BYTES (GDN_VERIFY_WY_TABLE_SEQS * 8)" in h
    assert ("(GDN_VERIFY_WY_TABLES_PER_LAYER * GDN_VERIFY_WY_TABLE_STRIDE_BYTES)" in h)
    # the widest verify arm (k = 16) is admitted, and a batch of 16 fits one table
    assert 2 <= 16 <= int(val("GDN_VERIFY_WY_TABLES_PER_LAYER"))
    assert int(val("GDN_VERIFY_WY_TABLE_SEQS")) >= 16


def test_binding_constants(g):
    assert g.VERIFY_WY_TABLE_STRIDE_BYTES == 1024
    assert g.VERIFY_WY_LAYER_STRIDE_BYTES == 16384


def test_wy_tables_fill_layout(g):
    ks = [2, 16, 5, 9]
    n = len(ks)
    h = [0x1000 * (i + 1) for i in range(n)]
    inter = [[0x100000 * (i + 1) + 0x40 * t for t in range(15)] for i in range(n)]
    tab = g.gdn_wy_tables_fill(ks, h, inter)
    assert tab.shape == (16, 128) and tab.nbytes == 16384
    for i, k in enumerate(ks):
        assert tab[0, i] == h[i]
        for t in range(15):
            expect = inter[i][t] if t < k - 1 else 0
            assert tab[t + 1, i] == expect, (i, t)
    assert (tab[:, n:] == 0).all()  # entries of absent sequences stay zero


@pytest.mark.parametrize("bad_k", [0, 1, 17])
def test_wy_tables_fill_refuses_bad_k(g, bad_k):
    with pytest.raises(g.GdnError) as e:
        g.gdn_wy_tables_fill([4, bad_k], [16, 32], [[0] * 15, [0] * 15])
    assert e.value.status == 5  # GDN_ERR_BAD_K


def test_wy_tables_fill_refuses_too_many(g):
    with pytest.raises(g.GdnError) as e:
        g.gdn_wy_tables_fill([2] * 129, [16] * 129, [[0] * 15] * 129)
    assert e.value.status == 6


def _dims(g, **kw):
    base = dict(n_k_heads=16, n_v_heads=32, d_k=128, d_v=128, d_conv=4, q_scale=0.088,
                l2_eps=1e-6, norm_eps=1e-6)
    base.update(kw)
    return g.make_dims(**base)


class _FakeT:
    """Stands in for a device tensor: only its address and strides are read on the host."""

    def __init__(self, ptr, shape=(1, 1), dtype=None):
        import torch
        self._p, self.shape = ptr, shape
        self.dtype = dtype or torch.bfloat16

    def data_ptr(self):
        return self._p

    def dim(self):
        return 2

    def stride(self, i):
        return (self.shape[1], 1)[i]


def _inputs(g, conv_dim=8192, z=4096, ab=32, base=0x10000):
    return g.Inputs(_FakeT(base, (1, conv_dim)), _FakeT(base, (1, z)), _FakeT(base, (1, ab)),
                    _FakeT(base, (1, ab)))


def _weights(g, base=0x10000):
    return g.Weights(_FakeT(base), _FakeT(base), _FakeT(base), _FakeT(base))


def _decode(g, dims, n=4, inputs=None, h_pool=0x20000, conv_pool=0x30000, slots=0x40000,
            y=0x50000, status=0x60000, n_slots=8):
    return g.gdn_decode_batched(dims, _weights(g), inputs or _inputs(g), n, h_pool, conv_pool,
                                n_slots, slots, y, None, status, stream=0)


@pytest.mark.parametrize("kw,code", [
    (dict(d_k=64, d_v=64), 2), (dict(d_k=128, d_v=16), 2), (dict(d_conv=3), 2),
    (dict(n_v_heads=80), 2),           # G = 5 > 4
    (dict(n_v_heads=24), 2),           # not a multiple of n_k_heads
    (dict(n_k_heads=0), 1), (dict(norm_eps=-1.0), 1), (dict(q_scale=float("nan")), 1),
    (dict(norm_gate=2), 1), (dict(norm_gate=-1), 1)])
def test_decode_refuses_bad_dims(g, kw, code):
    with pytest.raises(g.GdnError) as e:
        _decode(g, _dims(g, **kw))
    assert e.value.status == code


def test_decode_refuses_bad_arguments(g):
    d = _dims(g)
    for kwargs, code in [(dict(n=129), 6), (dict(n=-1), 1), (dict(h_pool=None), 3),
                         (dict(h_pool=0x20004), 4), (dict(status=None), 3),
                         (dict(slots=None), 3), (dict(n_slots=0), 1), (dict(y=0x50008), 4),
                         (dict(inputs=_inputs(g, conv_dim=8000)), 1),
                         (dict(inputs=_inputs(g, conv_dim=8196)), 4),
                         (dict(inputs=_inputs(g, base=0x10008)), 4)]:
        with pytest.raises(g.GdnError) as e:
            _decode(g, d, **kwargs)
        assert e.value.status == code, kwargs


def test_decode_zero_sequences_is_a_noop(g):
    _decode(g, _dims(g), n=0)  # returns OK without touching CUDA


def test_verify_refuses_bad_k_and_counts(g):
    d = _dims(g)
    w, i = _weights(g), _inputs(g)
    for ks, code in [([2, 1], 5), ([17], 5), ([0], 5), ([2] * 129, 6)]:
        with pytest.raises(g.GdnError) as e:
            g.gdn_verify_multi(d, w, i, len(ks), ks, 0x70000, 0x30000, 8, 0x40000, None,
                               0x50000, None, 0x60000, stream=0)
        assert e.value.status == code, ks
    with pytest.raises(g.GdnError) as e:  # NULL tables
        g.gdn_verify_multi(d, w, i, 2, [2, 3], None, 0x30000, 8, 0x40000, None, 0x50000, None,
                           0x60000, stream=0)
    assert e.value.status == 3


def test_prefill_refuses_bad_chunk_and_workspace(g):
    d = _dims(g)
    w, i = _weights(g), _inputs(g)
    with pytest.raises(g.GdnError) as e:
        g.gdn_prefill_chunked(d, w, i, 1, 0x80000, 64, 64, 0x90000, 0x30000, 4, 0x40000,
                              0x50000, status=0x60000, stream=0, chunk=32)
    assert e.value.status == 1
    assert g.gdn_prefill_workspace_bytes(d, 1, 64, 64, chunk=32) == 0


@pytest.mark.parametrize("name", ["gdn_gated_rmsnorm", "gdn_gated_rmsnorm_sigmoid"])
def test_gated_rmsnorm_refuses_bad_args(g, name):
    st = getattr(g.lib(), name)
    assert st(0x1000, 0x1000, 4096, 0x1000, ctypes.c_float(1e-6), 4, 32, 64, 1, 0x1000, 0) == 2
    assert st(0x1000, 0x1000, 4096, 0x1000, ctypes.c_float(-1.0), 4, 32, 128, 1, 0x1000, 0) == 1
    assert st(0x1004, 0x1000, 4096, 0x1000, ctypes.c_float(1e-6), 4, 32, 128, 1, 0x1000, 0) == 4
    assert st(None, 0x1000, 4096, 0x1000, ctypes.c_float(1e-6), 4, 32, 128, 1, 0x1000, 0) == 3


def test_fold_refuses_bad_arguments(g):
    d = _dims(g)

    def fold(n=2, ks=(3, 5), accepted=0xA0000, tables=0x70000, conv_pool=0x30000, n_slots=8,
             slots=0x40000, conv_inter=0xB0000, dtype=1, status=0x60000, h_dtype=0):
        g.gdn_fold_accepted(d, n, list(ks), accepted, tables, conv_pool, n_slots, slots,
                            conv_inter, dtype, status, stream=0, h_dtype=h_dtype)

    for kwargs, code in [(dict(n=0, ks=()), 1), (dict(n=129, ks=[2] * 129), 6),
                         (dict(ks=(3, 17)), 5), (dict(ks=(1, 4)), 5), (dict(dtype=7), 1),
                         (dict(h_dtype=1), 1), (dict(dtype=2), 1),
                         (dict(accepted=None), 3), (dict(tables=None), 3),
                         (dict(conv_inter=None), 3), (dict(status=None), 3),
                         (dict(slots=None), 3), (dict(n_slots=0), 1),
                         (dict(accepted=0xA0002), 4), (dict(conv_inter=0xB0008), 4),
                         (dict(tables=0x70004), 4)]:
        with pytest.raises(g.GdnError) as e:
            fold(**kwargs)
        assert e.value.status == code, kwargs
    with pytest.raises(g.GdnError) as e:
        g.gdn_fold_accepted(_dims(g, d_k=64, d_v=64), 2, [3, 5], 0xA0000, 0x70000, 0x30000, 8,
                            0x40000, 0xB0000, 1, 0x60000, stream=0)
    assert e.value.status == 2


def test_h16_entry_points_validate_like_the_f32_ones(g):
    d = _dims(g)
    for kwargs, code in [(dict(n=129), 6), (dict(h_pool=None), 3), (dict(h_pool=0x20004), 4)]:
        args = dict(n=4, h_pool=0x20000)
        args.update(kwargs)
        with pytest.raises(g.GdnError) as e:
            g.gdn_decode_batched_h16(d, _weights(g), _inputs(g), args["n"], args["h_pool"],
                                     0x30000, 8, 0x40000, 0x50000, None, 0x60000, stream=0)
        assert e.value.status == code, kwargs
    with pytest.raises(g.GdnError) as e:
        g.gdn_verify_multi_h16(d, _weights(g), _inputs(g), 2, [2, 17], 0x70000, 0x30000, 8,
                               0x40000, None, 0x50000, None, 0x60000, stream=0)
    assert e.value.status == 5


def test_state_convert_refuses_bad_arguments(g):
    for args, code in [((0x1000, 0, 0x2000, 0, 8), 1), ((0x1000, 2, 0x2000, 2, 8), 1),
                       ((0x1000, 1, 0x2000, 2, 8), 1), ((0x1000, 0, 0x2000, 2, -1), 1),
                       ((None, 0, 0x2000, 2, 8), 3), ((0x1008, 0, 0x2000, 2, 8), 4)]:
        with pytest.raises(g.GdnError) as e:
            g.gdn_state_convert(*args, stream=0)
        assert e.value.status == code, args
    g.gdn_state_convert(0x1000, 0, 0x2000, 2, 0, stream=0)  # nothing to do


def test_status_strings(g):
    for code in (0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 17, 18, 19, 20):
        s = g.status_string(code)
        assert s and s != "unknown status"
    assert g.status_string(12345) == "unknown status"


def test_proj_gemm_refuses_bad_arguments(g):
    f = g.lib().gdn_proj_gemm
    ok = dict(A=0x10000, lda=64, B=0x20000, ldb=64, C=0x30000, ldc=64, M=4, N=64, K=64,
              status=0x40000)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["A"], a["lda"], a["B"], a["ldb"], a["C"], a["ldc"], a["M"], a["N"], a["K"],
                 a["status"], None)

    for kw, code in [(dict(M=-1), 1), (dict(N=4), 1), (dict(K=0), 1), (dict(N=60), 1),
                     (dict(K=12), 1), (dict(lda=32), 1), (dict(ldc=32), 1), (dict(A=None), 3),
                     (dict(status=None), 3), (dict(B=0x20008), 4), (dict(C=0x30002), 4),
                     (dict(lda=68), 4)]:
        assert call(**kw) == code, kw
    assert call(M=0) == 0  # nothing to do: no launch
    assert call(M=0, A=None, C=None) == 0  # an empty tensor's address may be NULL


def test_in_proj_width(g):
    assert g.gdn_in_proj_width(_dims(g)) == 8192 + 4096 + 64
    assert g.gdn_in_proj_width(_dims(g, d_conv=3)) == 0
    # H_k = 1, H_v = 2, d = 16: 64 + 32 + 4 = 100 columns, padded to 104 (16-byte rows)
    assert g.gdn_in_proj_width(_dims(g, n_k_heads=1, n_v_heads=2, d_k=16, d_v=16)) == 104


def test_selftest_wait_refuses_bad_arguments(g):
    f = g.lib().gdn_selftest_wait
    assert f(0, 0x60000, None) == 1
    assert f(2_000_000_000, 0x60000, None) == 1
    assert f(1000, None, None) == 3
    assert f(1000, 0x60002, None) == 4
