"""Helpers shared by the GPU parity tests: build/load, oracle runs, comparisons.

Every comparison of a floating-point result with the oracle checks three things:
  1. the whole tensor: ||x - ref||_2 / ||ref||_2 <= tol (the relative error the targets
     state: 2e-3 on bf16 outputs, 1e-4 on f32 outputs and on the f32 state);
  2. every row -- one (token, value head) row of d_v values of y and of the core output o,
     one (value head, d_k index) row of d_v values of a state:
        ||x_row - ref_row|| <= ROW_FACTOR * tol * max(||ref_row||, s_row),
     so a wrong head, token or state row cannot hide in the tensor norm;
  3. every element: |x - ref| <= ulp(ref) + ELEM_FACTOR * tol * max(rms(ref_row), s_row/sqrt(d)),
     where ulp is the spacing of the output format at ref (2^-7 |ref| for bf16, 2^-22 |ref|
     for f32): two values that differ by e round to bf16 values at most e + one spacing apart.
     One element that is wrong by its row's rms fails this at any tolerance used here.
The floor s_row is the typical row norm (the median over the tensor's rows).  Rounding errors
of a sum are relative to the size of its terms, not of its result: a row that comes out
hundreds of times smaller than its neighbours (o_t = S_t q_t with q_t nearly orthogonal to
what S_t holds, or a state row i after a reset with k_i ~ 0) carries the same absolute error
as they do, which is a large relative one.  The floor keeps such rows to the absolute error a
typical row is allowed; a row that is wrong carries an error of the typical size and fails
all the same.  For y, which the gated norm rescales row by row, the floor of a row is
||y_row|| * median(||o||) / ||o_row||: the error its core-output row o_row may carry, seen
through the same rescaling (y_row / ||y_row|| depends on o_row only through its direction).

Tolerances (written here once, used by every parity test):
  * bf16 outputs y: compared against bf16(y_oracle) (round to nearest even), tol 2e-3;
  * f32 outputs (core o, f32 y): tol 1e-4;
  * f32 state: tol 1e-4 (the tensor check is per sequence, or per intermediate state);
  * conv state, slot indexing, table memory: bit-exact.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_layer_conv1d_gb300 import workloads as wl

Y_BF16_TOL = 2e-3
F32_TOL = 1e-4
STATE_TOL = 1e-4
# The tensor-core chunked prefill multiplies fp16 operands (q, k, v, T, W, Delta, P and an
# fp16 copy of the state), each rounded to 2^-11 relative; the oracle's own operand-rounding
# emulation puts the resulting f32 state and core-output error near 4e-4, so they are held
# to 1e-3 instead of the 1e-4 of the f32 paths.
TC_STATE_TOL = 1e-3
TC_CORE_TOL = 1e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_layer_conv1d_gb300 import _build
    _build.build()
    oracle.build()


# Row and element factors of the comparisons (see the module docstring).  A row's error is
# the same rounding noise as the tensor's measured on d_v = 128 values instead of millions, so
# it spreads more: 4x the tensor tolerance leaves room for that spread and still fails a row
# that is wrong by a few tenths of a percent at the f32 tolerance.
ROW_FACTOR = 4.0
ELEM_FACTOR = 8.0
# The tensor-core prefill rounds its operands to fp16 (2^-11 relative), among them q, k, v and
# a copy of the state at each chunk start whose rows can be ten times larger than the result's
# (an initial state of variance 0.1 decays to rows of norm ~0.1-0.4 within a chunk).  Its
# per-element errors are heavier-tailed than the f32 paths': a plain numpy restatement of that
# rounding reproduces the measured core outputs digit for digit and puts the worst element at
# 1.2-1.4 times the 8 * tol bound, so the tensor-core path's element bound takes twice the
# factor (its tensor and row bounds are the common ones).
TC_ELEM_FACTOR = 16.0


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def check_rows(x, ref, d: int, tol: float, what: str, ulp_rel: float = 2.0 ** -22,
               floor=None, row_factor: float = ROW_FACTOR, elem_factor: float = ELEM_FACTOR):
    """The three checks of the module docstring on x against ref, rows of d values along the
    last axis.  floor: per-row norm floor (default: the median row norm of ref).  Returns
    (tensor error, worst row error / its bound, worst element error / its bound)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape, f"{what}: shape {x.shape} != {ref.shape}"
    assert np.isfinite(x).all(), f"{what}: non-finite values"
    e = rel_l2(x, ref)
    assert e <= tol, f"{what}: rel L2 {e:.3e} > {tol:.0e}"
    if x.size == 0:
        return e, 0.0, 0.0
    xr = x.reshape(-1, d)
    rr = ref.reshape(-1, d)
    diff = xr - rr
    rn = np.linalg.norm(rr, axis=1)
    dn = np.linalg.norm(diff, axis=1)
    floor = (np.full(len(rr), np.median(rn)) if floor is None
             else np.broadcast_to(np.asarray(floor, np.float64), rn.shape))
    scale = np.maximum(rn, floor)
    # a row whose reference is exactly zero (and has no floor) must come out exactly zero
    zero = scale == 0
    assert not (zero & (dn > 0)).any(), f"{what}: a zero reference row is not zero"
    row_err = np.where(zero, 0.0, dn / np.where(zero, 1.0, scale))
    worst = int(np.argmax(row_err))
    row_bound = row_factor * tol
    assert row_err[worst] <= row_bound, (
        f"{what}: row {worst} (of {len(rr)}, rows of {d}) error {dn[worst]:.3e} = "
        f"{row_err[worst]:.3e} x max(norm {rn[worst]:.3e}, floor {floor[worst]:.3e}) > "
        f"{row_bound:.1e}")
    rms = scale / np.sqrt(d)
    bound = ulp_rel * np.abs(rr) + elem_factor * tol * rms[:, None]
    ratio = np.abs(diff) / np.where(bound > 0, bound, 1.0)
    ratio[(bound == 0) & (diff == 0)] = 0.0
    ratio[(bound == 0) & (diff != 0)] = np.inf
    wi = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    log = os.environ.get("GDN_PARITY_LOG")
    if log:  # margins of every comparison, one line each: tensor error, row and element ratios
        with open(log, "a") as f:
            f.write(f"{os.environ.get('PYTEST_CURRENT_TEST', '').split(' ')[0]}\t{what}\t"
                    f"{e:.3e}\t{e / tol:.3f}\t{row_err[worst] / row_bound:.3f}\t"
                    f"{ratio[wi]:.3f}\n")
    assert ratio[wi] <= 1.0, (
        f"{what}: element (row {wi[0]}, col {wi[1]}) = {xr[wi]:.6e} vs {rr[wi]:.6e}: "
        f"|diff| {abs(diff[wi]):.3e} > bound {bound[wi]:.3e} (row scale {rms[wi[0]]:.3e})")
    return e, float(row_err[worst] / row_bound), float(ratio[wi])


def _d_of(cols: int) -> int:
    """Head width of a [rows][H_v * d_v] output: 128 where it divides the row, else 16."""
    return 128 if cols % 128 == 0 else 16


def assert_y_close(y_gpu: torch.Tensor, y_orc: np.ndarray, what="y", tol=None, d=None,
                   o_orc=None, row_factor=ROW_FACTOR, elem_factor=ELEM_FACTOR):
    """y (bf16 or f32 rows [T][H_v * d_v]) against the oracle's y; per tensor, per
    (token, head) row and per element.  o_orc: the oracle's core output of the same rows
    ([T][H_v][d_v]), which sets each row's floor (module docstring); without it the floor is
    the median row norm of y.  Returns the tensor error."""
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    if y_gpu.dtype == torch.bfloat16:
        ref = wl.round_bf16(np.asarray(y_orc, np.float32)).astype(np.float64)
        tol = Y_BF16_TOL if tol is None else tol
        ulp = 2.0 ** -7
    else:
        ref = np.asarray(y_orc, np.float64)
        tol = F32_TOL if tol is None else tol
        ulp = 2.0 ** -22
    d = _d_of(ref.shape[-1]) if d is None else d
    ref = ref.reshape(y.shape)
    floor = None
    if o_orc is not None:
        on = np.linalg.norm(np.asarray(o_orc, np.float64).reshape(-1, d), axis=1)
        yn = np.linalg.norm(ref.reshape(-1, d), axis=1)
        floor = yn * np.median(on) / np.where(on > 0, on, np.inf)
    return check_rows(y, ref, d, tol, what, ulp, floor, row_factor, elem_factor)[0]


def assert_core_close(core_gpu, o_orc, what="core o", tol=F32_TOL, elem_factor=ELEM_FACTOR):
    """The f32 core output o [T][H_v][d_v] against the oracle's; per tensor, per
    (token, head) row and per element.  Returns the tensor error."""
    o = core_gpu.cpu().numpy() if isinstance(core_gpu, torch.Tensor) else core_gpu
    ref = np.asarray(o_orc, np.float64)
    return check_rows(o, ref.reshape(np.shape(o)), ref.shape[-1], tol, what,
                      elem_factor=elem_factor)[0]


def assert_state_close(H_gpu, H_orc, what="state", tol=STATE_TOL, ulp_rel=2.0 ** -22,
                       row_factor=ROW_FACTOR, elem_factor=ELEM_FACTOR):
    """One sequence's state [H_v][d_k][d_v] (or any stack of them) against the oracle's;
    relative Frobenius error of the whole, per (head, d_k index) row of d_v values, and per
    element.  ulp_rel: relative spacing of the stored format (2^-10 for fp16 state pools).
    Returns the tensor error."""
    H = np.asarray(H_gpu, np.float64)
    ref = np.asarray(H_orc, np.float64)
    return check_rows(H, ref, ref.shape[-1], tol, what, ulp_rel, row_factor=row_factor,
                      elem_factor=elem_factor)[0]


def odims(shape: wl.LayerShape) -> oracle.Dims:
    return oracle.Dims(shape.n_k_heads, shape.n_v_heads, shape.d_k, shape.d_v, shape.d_conv,
                       float(np.float32(shape.q_scale)), float(np.float32(shape.l2_eps)),
                       float(np.float32(shape.norm_eps)), norm_gate=shape.norm_gate)


def oracle_seqs(w: wl.Workload, token_rows: dict, lens, H0=None, conv0=None, idx=None,
                snapshots=False):
    """Runs the oracle over sequences whose token rows are sequence-major in token_rows."""
    H0 = w.H0 if H0 is None else H0
    conv0 = w.conv0 if conv0 is None else conv0
    off = np.concatenate([[0], np.cumsum(lens)])
    idx = range(len(lens)) if idx is None else idx
    seqs = []
    for i in idx:
        sl = slice(int(off[i]), int(off[i + 1]))
        seqs.append(dict(qkv=token_rows["qkv"][sl], z=token_rows["z"][sl], a=token_rows["a"][sl],
                         b=token_rows["b"][sl], conv_state=conv0[i], H=H0[i]))
    return oracle.mixer_batch(odims(w.shape), w.weights, seqs, snapshots=snapshots)
