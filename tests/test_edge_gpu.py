"""GPU parity at the edges of the gates and of the output gate, for decode, verify and both
prefill paths, against the fp64 oracle under the per-tensor, per-row and per-element bounds of
gpu_common.  Gate logits of +-30 drive each gate to its limit (workloads.set_extreme):

  * reset (a = +30): the decay's softplus takes its x > 20 branch and alpha is ~0 -- the old
    state is forgotten (alpha = 0 resets the state, a special case the oracle pins);
  * hold (a = b = -30): alpha = 1 and beta = 0 to f32 precision -- the state must come out as
    it went in (beta = 0, alpha = 1 leaves the state unchanged), checked here against the
    initial state itself to 1e-6 as well as against the oracle;
  * write (b = +30) and reset + write: beta = 1, the delta rule's full-strength write;
  * |z| = 30 in the gated norm: SiLU(30) = 30 and SiLU(-30) ~ -3e-12 in one row;
  * in the chunked prefill, a reset in the middle of a chunk makes the cumulative log decay
    drop by 16 .. 117 (log2 units) inside the chunk, so e^(g_r - g_s) underflows to zero for
    every pair that straddles it.
"""
import numpy as np
import pytest

from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import require_gpu, rel_l2
from tests.test_decode_gpu import check_against_oracle, run_decode
from tests.test_prefill_gpu import check_prefill, run_prefill
from tests.test_verify_gpu import check, run_verify

pytestmark = pytest.mark.gpu

HOLD_TOL = 1e-6  # the state under beta = 0, alpha = 1, against the initial state itself


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _rows(off, i, positions):
    return [int(off[i]) + p for p in positions]


def test_decode_extreme_gates():
    """Eight sequences, six steps: one pattern per sequence (reset every step, hold every
    step, write every step, reset + write at step 2, |z| = 30 every step, hold and reset in
    turn), two untouched."""
    steps = 6
    w = wl.batched_decode(n=8, steps=steps, seed=61)
    all_steps = [w.tokens] + w.steps
    for s, tok in enumerate(all_steps):
        wl.set_extreme(tok, [0], "reset")
        wl.set_extreme(tok, [1], "hold")
        wl.set_extreme(tok, [2], "write")
        if s == 2:
            wl.set_extreme(tok, [3], "reset_write")
        wl.set_extreme(tok, [4], "zbig")
        wl.set_extreme(tok, [5], "hold" if s % 2 == 0 else "reset")
    ys, cores, H, conv, _ = run_decode(w)
    check_against_oracle(w, ys, cores, H, conv)
    e = rel_l2(H[1], w.H0[1])
    assert e <= HOLD_TOL, f"hold: state moved by {e:.3e}"


def test_decode_extreme_gates_tiny_f32():
    w = wl.batched_decode(n=5, steps=8, shape=wl.TINY, seed=62, bf16=False)
    for s, tok in enumerate([w.tokens] + w.steps):
        for i, kind in enumerate(wl.EXTREME):
            if (s + i) % 2 == 0:
                wl.set_extreme(tok, [i], kind)
    ys, cores, H, conv, _ = run_decode(w)
    check_against_oracle(w, ys, cores, H, conv)


@pytest.mark.parametrize("k", [2, 16])
def test_verify_extreme_gates(k):
    """Six sequences of k drafts: every intermediate state and every output row against the
    oracle, with the patterns at the first, a middle and the last draft."""
    w = wl.ragged_verify(n=6, k_lo=k, k_hi=k, seed=63 + k)
    off = np.concatenate([[0], np.cumsum(w.lens)])
    mid = k // 2
    wl.set_extreme(w.tokens, _rows(off, 0, [mid]), "reset")
    wl.set_extreme(w.tokens, _rows(off, 1, range(k)), "hold")
    wl.set_extreme(w.tokens, _rows(off, 2, range(k)), "write")
    wl.set_extreme(w.tokens, _rows(off, 3, [0, k - 1]), "reset_write")
    wl.set_extreme(w.tokens, _rows(off, 4, range(k)), "zbig")
    wl.set_extreme(w.tokens, _rows(off, 5, [k - 1]), "reset")
    r = run_verify(w)
    assert r["status"] == 0
    check(w, r, range(6))
    e = rel_l2(r["H"][1], w.H0[1])
    assert e <= HOLD_TOL, f"hold: final state moved by {e:.3e}"
    inter = r["inter"][1].cpu().numpy()
    for t in range(k - 1):
        e = rel_l2(inter[t], w.H0[1])
        assert e <= HOLD_TOL, f"hold: intermediate {t} moved by {e:.3e}"


def _extreme_prefill(lens, seed, shape=wl.FULL):
    """Varlen prefill whose sequences take the patterns: 0 hold throughout; 1 resets at
    tokens 40 and 100 (inside chunks 0 and 1); 2 resets at every token; 3 writes with
    beta = 1 throughout; 4 |z| = 30 throughout; 5 a random mix of every pattern and plain
    tokens."""
    w = wl.varlen_prefill(lens, shape=shape, seed=seed)
    off = w.cu_seqlens
    L = w.lens
    wl.set_extreme(w.tokens, _rows(off, 0, range(L[0])), "hold")
    wl.set_extreme(w.tokens, _rows(off, 1, [p for p in (40, 100) if p < L[1]]), "reset")
    wl.set_extreme(w.tokens, _rows(off, 2, range(L[2])), "reset")
    wl.set_extreme(w.tokens, _rows(off, 3, range(L[3])), "write")
    wl.set_extreme(w.tokens, _rows(off, 4, range(L[4])), "zbig")
    rng = np.random.default_rng(seed + 1)
    kinds = ("normal",) + wl.EXTREME
    for p in range(L[5]):
        wl.set_extreme(w.tokens, _rows(off, 5, [p]), kinds[int(rng.integers(len(kinds)))])
    return w


def test_tensor_core_prefill_extreme_gates():
    """Six sequences on the tensor-core chunked path (whole-row spine with the fused norm)."""
    w = _extreme_prefill([200, 130, 64, 100, 77, 150], seed=65)
    r = run_prefill(w)
    check_prefill(w, r)
    H1 = r["h_pool"][r["slots"].long()][0].cpu().numpy()
    e = rel_l2(H1, w.H0[0])
    assert e <= HOLD_TOL, f"hold: state moved by {e:.3e}"


def test_tensor_core_prefill_extreme_gates_sliced_spine():
    """One sequence (the column-sliced spine and the separate norm kernel): a reset inside
    every fourth chunk, |z| = 30 on a run of tokens, beta = 1 on another, holds elsewhere."""
    w = wl.varlen_prefill([1000], seed=67)
    for c in range(0, 16, 4):
        wl.set_extreme(w.tokens, [64 * c + 37], "reset")
    wl.set_extreme(w.tokens, range(300, 360), "zbig")
    wl.set_extreme(w.tokens, range(500, 580), "write")
    wl.set_extreme(w.tokens, range(700, 900), "hold")
    check_prefill(w, run_prefill(w, with_core=False))


def test_sequential_prefill_extreme_gates_tiny_f32():
    """The token-sequential path (d = 16, f32 activations)."""
    w = _extreme_prefill([70, 130, 9, 64, 5, 90], seed=69, shape=wl.TINY)
    w.bf16 = False
    rng = np.random.default_rng(70)
    tok = wl.make_tokens(rng, wl.TINY, int(w.lens.sum()), bf16=False)
    for key in ("qkv",):
        w.tokens[key] = tok[key]  # f32 values for the raw stream; the gate patterns stay
    r = run_prefill(w)
    check_prefill(w, r)
    H1 = r["h_pool"][r["slots"].long()][0].cpu().numpy()
    assert rel_l2(H1, w.H0[0]) <= HOLD_TOL
