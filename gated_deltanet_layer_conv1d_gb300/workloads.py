"""Seeded synthetic workloads for the GDN mixer (data only: no step of the method here).

Both the CUDA path's tests/benchmark and the fp64 oracle take their inputs from this
module, so the two see identical values.  Values are drawn in float32 from numpy's
PCG64 with a fixed seed and a fixed draw order, then rounded to the nearest bfloat16
(ties to even) wherever a tensor is stored as bf16; the returned arrays are float32
holding exactly those values.

Distributions (N(m, s2) names the mean and the VARIANCE):
  raw QKV, Z, gate logits a and b ............ N(0, 1)
  conv weights [conv_dim][d_conv] ............ N(0, 1/4), float32
  A_log [H_v] ................................ U(-1, 1), float32
  dt_bias [H_v] .............................. 0
  gated-RMSNorm weight [d_v] ................. 1 + N(0, 0.02), float32
  initial recurrent state (where not zero) ... N(0, 0.1), float32
  initial conv state (where not zero) ........ N(0, 0.1), stored like the activations
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED = 0


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(x.shape)


@dataclass(frozen=True)
class LayerShape:
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    d_conv: int
    q_scale: float
    l2_eps: float = 1e-6
    norm_eps: float = 1e-6
    norm_gate: int = 0  # 0: SiLU(z) gate, 1: sigmoid(z) gate

    @property
    def conv_dim(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    @property
    def z_dim(self) -> int:
        return self.n_v_heads * self.d_v


TINY = LayerShape(1, 2, 16, 16, 4, q_scale=16 ** -0.5)
TINY_UNSCALED = LayerShape(1, 2, 16, 16, 4, q_scale=1.0)
FULL = LayerShape(16, 32, 128, 128, 4, q_scale=128 ** -0.5)


def _normal(rng, shape, var=1.0):
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(np.sqrt(var))).astype(
        np.float32)


def make_weights(rng: np.random.Generator, shape: LayerShape) -> dict:
    """Layer parameters, always float32: conv_w, A_log, dt_bias, norm_w."""
    conv_w = _normal(rng, (shape.conv_dim, shape.d_conv), 0.25)
    A_log = rng.uniform(-1.0, 1.0, size=shape.n_v_heads).astype(np.float32)
    dt_bias = np.zeros(shape.n_v_heads, dtype=np.float32)
    norm_w = (1.0 + _normal(rng, (shape.d_v,), 0.02)).astype(np.float32)
    return {"conv_w": conv_w, "A_log": A_log, "dt_bias": dt_bias, "norm_w": norm_w}


def make_tokens(rng: np.random.Generator, shape: LayerShape, T: int, bf16: bool) -> dict:
    """T rows of raw activations: qkv [T][conv_dim], z [T][H_v*d_v], a, b [T][H_v]."""
    rnd = round_bf16 if bf16 else (lambda x: x)
    qkv = rnd(_normal(rng, (T, shape.conv_dim)))
    z = rnd(_normal(rng, (T, shape.z_dim)))
    a = rnd(_normal(rng, (T, shape.n_v_heads)))
    b = rnd(_normal(rng, (T, shape.n_v_heads)))
    return {"qkv": qkv, "z": z, "a": a, "b": b}


def make_states(rng: np.random.Generator, shape: LayerShape, n: int, bf16: bool,
                zero: bool = False):
    """Initial states: H [n][H_v][d_k][d_v] float32, conv [n][conv_dim][d_conv]."""
    hs = (n, shape.n_v_heads, shape.d_k, shape.d_v)
    cs = (n, shape.conv_dim, shape.d_conv)
    if zero:
        return np.zeros(hs, np.float32), np.zeros(cs, np.float32)
    H = _normal(rng, hs, 0.1)
    conv = _normal(rng, cs, 0.1)
    return H, (round_bf16(conv) if bf16 else conv)


@dataclass
class Workload:
    """One synthetic workload.  Token rows are sequence-major and contiguous."""
    name: str
    shape: LayerShape
    bf16: bool
    weights: dict
    H0: np.ndarray                 # [n][H_v][d_k][d_v]
    conv0: np.ndarray              # [n][conv_dim][d_conv]
    lens: np.ndarray               # [n] tokens per sequence in one call
    tokens: dict                   # rows of all sequences, sequence-major
    steps: list = field(default_factory=list)   # extra calls (decode steps), each a tokens dict
    extra: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.lens.shape[0])

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lens)]).astype(np.int32)


# Residual width of the layer around the mixer (a reading: the pages fix the head counts and
# dims, 16 key heads and 32 value heads of 128, not the hidden size; 2048 is the width such
# a layer has in the Qwen3-Next family).
HIDDEN = 2048


def in_proj_width(shape: LayerShape) -> int:
    """One in_proj output row [Q | K | V | Z | b | a], padded to a multiple of 8 columns
    (16-byte rows); the padding's weight rows are zero."""
    return (shape.conv_dim + shape.z_dim + 2 * shape.n_v_heads + 7) // 8 * 8


@dataclass
class Projections:
    """Synthetic projection operands, all bf16 values held in float32 arrays."""
    hidden: np.ndarray  # [T][H] ~ N(0, 1)
    w_in: np.ndarray    # [in_proj_width][H] ~ N(0, 1/H): in_proj outputs ~ N(0, 1)
    w_out: np.ndarray   # [H][H_v d_v] ~ N(0, 1/(H_v d_v))
    y: np.ndarray       # [T][H_v d_v] ~ N(0, 1): a stand-in mixer output for out_proj alone


def projections(T: int, shape: LayerShape = FULL, hidden: int = HIDDEN,
                seed: int = SEED) -> Projections:
    rng = np.random.default_rng(seed)
    x = round_bf16(_normal(rng, (T, hidden)))
    w_in = round_bf16(_normal(rng, (in_proj_width(shape), hidden), 1.0 / hidden))
    w_in[shape.conv_dim + shape.z_dim + 2 * shape.n_v_heads:] = 0.0
    w_out = round_bf16(_normal(rng, (hidden, shape.z_dim), 1.0 / shape.z_dim))
    y = round_bf16(_normal(rng, (T, shape.z_dim)))
    return Projections(x, w_in, w_out, y)


def tiny_check(q_scale_one: bool = False, prefill_tokens: int = 64, decode_steps: int = 8,
               seed: int = SEED) -> Workload:
    """One sequence, H_k = 1, H_v = 2, d_k = d_v = 16, width 4, float32 throughout:
    a 64-token prefill from zero state, then 8 single-token decode steps."""
    shape = TINY_UNSCALED if q_scale_one else TINY
    rng = np.random.default_rng(seed)
    w = make_weights(rng, shape)
    H0, conv0 = make_states(rng, shape, 1, bf16=False, zero=True)
    pre = make_tokens(rng, shape, prefill_tokens, bf16=False)
    steps = [make_tokens(rng, shape, 1, bf16=False) for _ in range(decode_steps)]
    return Workload("tiny_check", shape, False, w, H0, conv0,
                    np.array([prefill_tokens], np.int32), pre, steps)


def batched_decode(n: int = 128, steps: int = 1, shape: LayerShape = FULL,
                   seed: int = SEED, bf16: bool = True) -> Workload:
    """n sequences x 1 token per step; f32 state and conv state ~N(0, 0.1); bf16 (or f32)
    activations and conv state.  `tokens` is step 0, `steps` the following steps."""
    rng = np.random.default_rng(seed)
    w = make_weights(rng, shape)
    H0, conv0 = make_states(rng, shape, n, bf16=bf16)
    all_steps = [make_tokens(rng, shape, n, bf16=bf16) for _ in range(steps)]
    perm = rng.permutation(n).astype(np.int32)
    return Workload(f"batched_decode_{n}seq", shape, bf16, w, H0, conv0,
                    np.ones(n, np.int32), all_steps[0], all_steps[1:],
                    extra={"slot_perm": perm})


def ragged_verify(n: int = 128, k_lo: int = 2, k_hi: int = 16, shape: LayerShape = FULL,
                  seed: int = SEED, bf16: bool = True) -> Workload:
    """n sequences with k_i ~ U{k_lo..k_hi} draft tokens each; states ~N(0, 0.1)."""
    rng = np.random.default_rng(seed)
    w = make_weights(rng, shape)
    ks = rng.integers(k_lo, k_hi + 1, size=n).astype(np.int32)
    H0, conv0 = make_states(rng, shape, n, bf16=bf16)
    tok = make_tokens(rng, shape, int(ks.sum()), bf16=bf16)
    perm = rng.permutation(n).astype(np.int32)
    return Workload(f"ragged_verify_{n}seq", shape, bf16, w, H0, conv0, ks, tok,
                    extra={"slot_perm": perm})


def long_prefill(T: int = 8192, shape: LayerShape = FULL, seed: int = SEED) -> Workload:
    """One sequence of T tokens from zero state; bf16 activations."""
    rng = np.random.default_rng(seed)
    w = make_weights(rng, shape)
    H0, conv0 = make_states(rng, shape, 1, bf16=True, zero=True)
    tok = make_tokens(rng, shape, T, bf16=True)
    return Workload(f"long_prefill_{T}tok", shape, True, w, H0, conv0,
                    np.array([T], np.int32), tok)


def varlen_prefill(lens, shape: LayerShape = FULL, seed: int = SEED,
                   zero_state: bool = False) -> Workload:
    """Several sequences of the given lengths, one prefill call; states ~N(0, 0.1)."""
    rng = np.random.default_rng(seed)
    w = make_weights(rng, shape)
    lens = np.asarray(lens, np.int32)
    H0, conv0 = make_states(rng, shape, len(lens), bf16=True, zero=zero_state)
    tok = make_tokens(rng, shape, int(lens.sum()), bf16=True)
    return Workload(f"varlen_prefill_{len(lens)}seq", shape, True, w, H0, conv0, lens, tok)


def mixed_serving(n_prefill: int = 32, n_verify: int = 96, len_lo: int = 512,
                  len_hi: int = 4096, shape: LayerShape = FULL, seed: int = SEED):
    """32 sequences prefilling U{512..4096} tokens next to 96 sequences verifying
    k ~ U{2..16} drafts; one shared weight set, states ~N(0, 0.1).
    Returns (prefill Workload, verify Workload)."""
    rng = np.random.default_rng(seed)
    w = make_weights(rng, shape)
    lens = rng.integers(len_lo, len_hi + 1, size=n_prefill).astype(np.int32)
    ks = rng.integers(2, 17, size=n_verify).astype(np.int32)
    Hp, cp = make_states(rng, shape, n_prefill, bf16=True)
    Hv_, cv = make_states(rng, shape, n_verify, bf16=True)
    tp = make_tokens(rng, shape, int(lens.sum()), bf16=True)
    tv = make_tokens(rng, shape, int(ks.sum()), bf16=True)
    pre = Workload("mixed_prefill", shape, True, w, Hp, cp, lens, tp)
    ver = Workload("mixed_verify", shape, True, w, Hv_, cv, ks, tv,
                   extra={"slot_perm": np.arange(n_verify, dtype=np.int32)})
    return pre, ver


# Extreme gate and gate-input rows for the edge cases of the method: logits of +-30 are exact
# in bf16 and drive each gate to its limit (the decay gate's softplus(a + dt_bias) is 30, past
# the point where softplus(x) = x to f32 precision).
#   "reset"       a = +30            decay alpha = exp(-exp(A_log) * 30) ~ 1e-5 .. 1e-35
#   "hold"        a = -30, b = -30   alpha = 1 and beta = 0 to f32 precision: state unchanged
#   "write"       b = +30            beta = 1 to f32 precision
#   "reset_write" a = +30, b = +30   the state becomes the one rank-1 write
#   "zbig"        z = +-30           the output gate at both ends (SiLU(30) = 30, SiLU(-30) ~ 0)
EXTREME = ("reset", "hold", "write", "reset_write", "zbig")


def set_extreme(tokens: dict, rows, kind: str) -> None:
    """Overwrites the given token rows of a tokens dict (in place) with one extreme pattern."""
    rows = np.atleast_1d(np.asarray(rows, np.int64))
    if rows.size == 0 or kind == "normal":
        return
    if kind in ("reset", "reset_write"):
        tokens["a"][rows] = 30.0
    if kind == "hold":
        tokens["a"][rows] = -30.0
        tokens["b"][rows] = -30.0
    if kind in ("write", "reset_write"):
        tokens["b"][rows] = 30.0
    if kind == "zbig":
        z = tokens["z"][rows]
        tokens["z"][rows] = np.where(z >= 0, np.float32(30.0), np.float32(-30.0))
    if kind not in EXTREME:
        raise ValueError(kind)
