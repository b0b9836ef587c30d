"""GPU parity of the bf16 projections around the mixer (layer_struct.rs, Qwen3SsmLayer: the
sequential [Q | K | V | Z] QKVZ projection, the b / a inputs of ba_gates_k, out_proj; the
dense_gemm fields): gdn_proj_gemm at small ragged sizes and at the full in_proj / out_proj
sizes, and one layer chain in_proj -> prefill -> decode -> out_proj against the oracle
chain.  The shapes cover the launch forms the host picks on a GB300: whole-K persistent
tiles 64 wide (the small calls), 128 wide (in_proj at 128 tokens) and 256 wide (2048 x 2048,
the 8000 / 8192-token calls), and K split over a cluster -- 64-wide tiles in 8
(64 x 200 x 1024, ragged M and N) and in 4 (out_proj at 128 tokens), 128-wide in 3
(300 x 2048 x 4096, three row blocks), 256-wide in 3 (100 x 9856 x 6144: a wide, deep
call of few rows, ragged M and a half-filled last tile) -- and the SM-pair kernel (256 x 256 tiles on two
SMs) for every 256-wide call of two row blocks or more: 2048 x 2048, the 8000 / 8192-token
calls, in_proj in the layer chain (259 rows) and 4000 x 1000 x 520 (ragged M, N and K).

Tolerance (element by element, from the arithmetic): the kernel accumulates bf16 products
in f32 and rounds the sum to bf16 once, so |c - c_exact| <= 2^-8 |c_exact| (the final
rounding, half a bf16 ulp) + K 2^-23 sum_k |x_k w_k| (f32 accumulation, a generous bound),
and the two bf16 roundings of nearly equal sums can differ by one ulp: the test allows
2^-7 |c_exact| + K 2^-23 sum_k |x_k w_k|.  In the layer chain the mixer's y keeps the 2e-3
relative L2 of every bf16 output, and out_proj's output is held to the bound its test
derives from y's measured error.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_conv1d_gb300 import device as dev
from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import (ELEM_FACTOR, ROW_FACTOR, TC_ELEM_FACTOR, TC_STATE_TOL,
                              assert_state_close, assert_y_close, check_rows, odims,
                              require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def bf16_dev(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to("cuda", torch.bfloat16)


def assert_gemm_close(c_gpu: torch.Tensor, x, w, rows=None, what="gemm"):
    """Element-wise bound above on the given rows (default all)."""
    xs = x if rows is None else x[rows]
    exact = oracle.proj(xs, w)
    mag = oracle.proj(np.abs(xs), np.abs(w))
    got = c_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    K = x.shape[1]
    bound = 2.0 ** -7 * np.abs(exact) + K * 2.0 ** -23 * mag
    err = np.abs(got - exact)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of bound, first {bad[0]}: "
                           f"{got[tuple(bad[0])]} vs {exact[tuple(bad[0])]}")


def run_gemm(x, w):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, b = bf16_dev(x), bf16_dev(w)
    c = torch.full((x.shape[0], w.shape[0]), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_proj_gemm(a, b, c, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return c


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (100, 200, 72), (129, 136, 8), (64, 200, 1024),
                                   (300, 2048, 4096), (2048, 2048, 2048), (4000, 1000, 520),
                                   (100, 9856, 6144)])
def test_gemm_small_and_ragged(M, N, K):
    rng = np.random.default_rng(M * 7 + N)
    x = wl.round_bf16(rng.standard_normal((M, K)).astype(np.float32))
    w = wl.round_bf16((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    assert_gemm_close(run_gemm(x, w), x, w, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(200, 12352, 2048), (2048, 2048, 2048), (100, 200, 72)])
def test_gemm_strided_operands(M, N, K):
    """A read from a wider buffer (lda > K) and C written into one (ldc > N), on the pair
    kernel with a single 256-row block (the odd CTA's rows partly past M), on the pair
    kernel with full blocks, and on the one-SM kernel."""
    rng = np.random.default_rng(M + K)
    x = wl.round_bf16(rng.standard_normal((M, K)).astype(np.float32))
    w = wl.round_bf16((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a_big = torch.zeros((M, K + 24), dtype=torch.bfloat16, device="cuda")
    a_big[:, 8:8 + K] = bf16_dev(x)
    c_big = torch.full((M, N + 40), 7.0, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_proj_gemm(a_big[:, 8:8 + K], bf16_dev(w), c_big[:, 16:16 + N], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_gemm_close(c_big[:, 16:16 + N], x, w, what=f"strided {M}x{N}x{K}")
    # columns outside the view are untouched
    assert (c_big[:, :16] == 7.0).all() and (c_big[:, 16 + N:] == 7.0).all()


@pytest.mark.parametrize("T", [128, 8000])
def test_in_proj_full_width(T):
    """in_proj of the 16/32-head layer: N = 12352 outputs, K = 2048; T = 8000 compares a
    sample of rows (every 64 x 12352 block boundary region and the ragged tail)."""
    P = wl.projections(T, seed=71 + T)
    dims = dev.dims_of(wl.FULL)
    width = gdn.gdn_in_proj_width(dims)
    assert width == wl.in_proj_width(wl.FULL) == 12352
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((T, width), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_in_proj(dims, bf16_dev(P.hidden), bf16_dev(P.w_in), out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = None
    if T > 1024:
        rng = np.random.default_rng(72)
        rows = np.unique(np.concatenate([rng.integers(0, T, 96), np.arange(T - 70, T),
                                         [0, 127, 128, 4095, 4096]]))
    assert_gemm_close(out, P.hidden, P.w_in, rows, f"in_proj T={T}")


@pytest.mark.parametrize("T", [128, 8192])
def test_out_proj(T):
    P = wl.projections(T, seed=73 + T)
    dims = dev.dims_of(wl.FULL)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((T, wl.HIDDEN), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_out_proj(dims, bf16_dev(P.y), bf16_dev(P.w_out), out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = None
    if T > 1024:
        rows = np.unique(np.concatenate([np.random.default_rng(74).integers(0, T, 96),
                                         np.arange(T - 40, T)]))
    assert_gemm_close(out, P.y, P.w_out, rows, f"out_proj T={T}")


def test_zero_rows_is_a_no_op():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_proj_gemm(a, b, c, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_layer_chain_in_proj_prefill_decode_out_proj():
    """hidden -> in_proj -> prefill of two sequences (the in_proj rows read in place as
    qkv, z, b, a) -> one decode step each -> out_proj, against the oracle chain (bf16
    activations between the steps, as the layer stores them)."""
    lens = [200, 57]
    T = sum(lens)
    sh = wl.FULL
    base = wl.varlen_prefill(lens, seed=75)  # weights and initial states of the mixer
    P = wl.projections(T + 2, seed=76)      # T prefill rows, then one decode row per sequence
    d = torch.device("cuda")
    dims = dev.dims_of(sh)
    width = gdn.gdn_in_proj_width(dims)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    w_in, w_out = bf16_dev(P.w_in), bf16_dev(P.w_out)
    weights = dev.weights_to(base, d)
    h_pool, conv_pool, slots = dev.states_to(base, d)

    rows = torch.empty((T + 2, width), dtype=torch.bfloat16, device=d)
    gdn.gdn_in_proj(dims, bf16_dev(P.hidden), w_in, rows, status)
    y = torch.empty((T + 2, sh.z_dim), dtype=torch.bfloat16, device=d)
    hsz = sh.n_v_heads * sh.d_k * sh.d_v * 4
    hp = torch.tensor([h_pool.data_ptr() + i * hsz for i in range(2)], dtype=torch.int64, device=d)
    cu = torch.tensor([0, lens[0], T], dtype=torch.int32, device=d)
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(dims, 2, T, max(lens)), dtype=torch.uint8,
                     device=d)
    gdn.gdn_prefill_chunked(dims, weights, gdn.in_proj_inputs(dims, rows[:T]), 2, cu, T,
                            max(lens), hp, conv_pool, 2, slots, y[:T], None, ws, status)
    gdn.gdn_decode_batched(dims, weights, gdn.in_proj_inputs(dims, rows[T:]), 2, h_pool,
                           conv_pool, 2, slots, y[T:], None, status)
    out = torch.empty((T + 2, wl.HIDDEN), dtype=torch.bfloat16, device=d)
    gdn.gdn_out_proj(dims, y, w_out, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    od = odims(sh)
    orows = wl.round_bf16(oracle.proj(P.hidden, P.w_in).astype(np.float32))
    sp = oracle.split_in_proj(od, orows)
    # The GPU's in_proj rows equal the oracle's bf16-rounded rows except where the f32 sum and
    # the exact one round to different bf16 values (one step apart, or more where the sum
    # cancels: the f32 accumulation error is relative to sum |x w|), and that is rare.
    got_rows = rows.float().cpu().numpy()[:, :orows.shape[1]]
    ne = got_rows != orows
    acc = np.abs(P.hidden.astype(np.float64)) @ np.abs(P.w_in.astype(np.float64)).T
    step = np.abs(orows) * 2.0 ** -7 + P.hidden.shape[1] * 2.0 ** -23 * acc[:, :orows.shape[1]]
    assert (np.abs(got_rows - orows)[ne] <= step[ne]).all()
    assert ne.mean() < 1e-2, ne.mean()
    y_orc = np.empty((T + 2, sh.z_dim))
    o_orc = np.empty((T + 2, sh.n_v_heads, sh.d_v))
    off = [0, lens[0], T]
    seqs = []
    for i in range(2):
        idx = np.r_[off[i]:off[i + 1], T + i]  # the sequence's prefill rows, then its decode row
        seqs.append({k: sp[k][idx] for k in ("qkv", "z", "a", "b")} |
                    dict(conv_state=base.conv0[i], H=base.H0[i]))
    res = oracle.mixer_batch(od, base.weights, seqs)
    for i, r in enumerate(res):
        y_orc[off[i]:off[i + 1]] = r.y[:-1]
        y_orc[T + i] = r.y[-1]
        o_orc[off[i]:off[i + 1]] = r.o[:-1]
        o_orc[T + i] = r.o[-1]
        # The mixer's inputs are the GPU's in_proj rows, a few elements of which round to
        # the neighbouring bf16 value of the oracle's (their f32 sums straddle a rounding
        # boundary); a state row that such a b or a gate logit feeds carries that input
        # difference, so rows and elements here get four times the common factors.
        assert_state_close(h_pool[i].cpu().numpy(), r.H, f"state seq {i}", TC_STATE_TOL,
                           row_factor=4 * ROW_FACTOR, elem_factor=4 * TC_ELEM_FACTOR)
    # (the same input differences reach y: four times the common row and element factors)
    e_y = assert_y_close(y, y_orc, "mixer y in the chain", o_orc=o_orc,
                         row_factor=4 * ROW_FACTOR, elem_factor=4 * ELEM_FACTOR)
    # out = bf16(y W^T): the error of y (measured against bf16(y_oracle), the oracle's own
    # stored y) passes through W_out about unchanged in relative L2 (25 % slack for a random
    # W), and the final bf16 rounding adds at most 2^-9 relative per element.
    out_orc = oracle.proj(wl.round_bf16(y_orc.astype(np.float32)), P.w_out)
    # Each out row mixes the 32 head rows of its token's y, so its floor carries theirs:
    # ||out_t|| * sqrt(sum_h max(||y_th||, floor_th)^2) / ||y_t||, with the y floors of
    # assert_y_close (a y row of a tiny core-output row may carry a larger relative error).
    yr = wl.round_bf16(y_orc.astype(np.float32)).astype(np.float64).reshape(T + 2, -1, sh.d_v)
    yn = np.linalg.norm(yr, axis=2)
    on = np.linalg.norm(o_orc, axis=2)
    yfl = np.maximum(yn, yn * np.median(on) / np.where(on > 0, on, np.inf))
    out_floor = (np.linalg.norm(out_orc, axis=1) * np.linalg.norm(yfl, axis=1) /
                 np.linalg.norm(yn, axis=1))
    e = check_rows(out.float().cpu().numpy(), out_orc, wl.HIDDEN, 1.25 * e_y + 2.0 ** -9,
                   f"out_proj in the chain (y {e_y:.3e})", 2.0 ** -7, out_floor)[0]
