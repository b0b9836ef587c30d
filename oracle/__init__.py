"""fp64 CPU oracle of the Gated DeltaNet token mixer (ctypes wrapper over gdn_oracle.cpp).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only users.  The oracle shares no code with the
CUDA library and never calls it; the CUDA library never imports this package.

All arrays are numpy float64, C-contiguous.  Shapes follow gdn_oracle.cpp:
raw QKV rows are ``[Q | K | V]`` (layer_struct.rs, Qwen3SsmLayer doc on the QKVZ
layout), the state of a value head is stored ``[d_k][d_v]`` (= S transposed;
layer_struct.rs, h_state_bytes = nv * kd * vd), the conv state ``[conv_dim][d_conv]``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_STAMP = os.path.join(_HERE, "liboracle.so.stamp")

_lib = None


def _src_hash() -> str:
    with open(_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def build(force: bool = False) -> str:
    """Compile gdn_oracle.cpp into liboracle.so next to it (g++, fp64, OpenMP)."""
    h = _src_hash()
    if not force and os.path.exists(_LIB) and os.path.exists(_STAMP):
        with open(_STAMP) as f:
            if f.read().strip() == h:
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-adds, so x86 and Arm hosts agree bit for bit.
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    with open(_STAMP, "w") as f:
        f.write(h)
    return _LIB


class OrcDims(ctypes.Structure):
    _fields_ = [
        ("n_k_heads", ctypes.c_int32),
        ("n_v_heads", ctypes.c_int32),
        ("d_k", ctypes.c_int32),
        ("d_v", ctypes.c_int32),
        ("d_conv", ctypes.c_int32),
        ("q_scale", ctypes.c_double),
        ("l2_eps", ctypes.c_double),
        ("norm_eps", ctypes.c_double),
        ("h_fp16", ctypes.c_int32),
        ("norm_gate", ctypes.c_int32),
    ]


@dataclass(frozen=True)
class Dims:
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    d_conv: int
    q_scale: float
    l2_eps: float
    norm_eps: float
    h_fp16: bool = False  # store the state as binary16 after every token
    norm_gate: int = 0    # 0: y gated by SiLU(z); 1: gated by sigmoid(z)

    @property
    def conv_dim(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    def c(self) -> OrcDims:
        return OrcDims(self.n_k_heads, self.n_v_heads, self.d_k, self.d_v, self.d_conv,
                       self.q_scale, self.l2_eps, self.norm_eps, int(self.h_fp16),
                       int(self.norm_gate))


_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.c_int32
_PD = ctypes.POINTER(_D)


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.orc_softplus.restype = ctypes.c_double
        L.orc_softplus.argtypes = [ctypes.c_double]
        L.orc_round_fp16.argtypes = [ctypes.c_double]
        L.orc_round_fp16.restype = ctypes.c_double
        L.orc_gates.argtypes = [_I32, _I32, _D, _D, _D, _D, _D, _D]
        L.orc_conv.argtypes = [_I32, _I32, _I32, _D, _D, _D, _D, _D]
        L.orc_l2norm_split.argtypes = [ctypes.POINTER(OrcDims), _I32, _D, _D, _D, _D]
        L.orc_delta_step.argtypes = [_I32, _I32, _D, _D, _D, _D, ctypes.c_double,
                                     ctypes.c_double, _D]
        L.orc_recurrence.argtypes = [ctypes.POINTER(OrcDims), _I32, _D, _D, _D, _D, _D, _D,
                                     _D, _D]
        L.orc_gated_rmsnorm.argtypes = [_I32, _I32, _I32, _D, _D, _D, ctypes.c_double, _I32,
                                        _D]
        L.orc_mixer.argtypes = [ctypes.POINTER(OrcDims), _I32] + [_D] * 14
        L.orc_chunked.argtypes = [ctypes.POINTER(OrcDims), _I32, _I32, _D, _D, _D, _D, _D,
                                  _D, _D, _I32]
        L.orc_mixer_batch.argtypes = ([ctypes.POINTER(OrcDims), _I32,
                                       ctypes.POINTER(ctypes.c_int32)] + [_PD] * 4 +
                                      [_D] * 4 + [_PD] * 6)
        L.orc_max_threads.restype = _I32
        L.orc_set_threads.argtypes = [_I32]
        _lib = L
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(x):
    if x is None:
        return None
    assert x.dtype == np.float64 and x.flags.c_contiguous
    return x.ctypes.data_as(_D)


def max_threads() -> int:
    return int(lib().orc_max_threads())


def set_threads(n: int) -> None:
    """Threads mixer_batch uses from now on (OpenMP over sequences)."""
    lib().orc_set_threads(int(n))


def round_fp16(x: float) -> float:
    """The oracle's binary16 rounding (nearest, ties to even) of one value."""
    return float(lib().orc_round_fp16(float(x)))


def softplus(x: float) -> float:
    return float(lib().orc_softplus(float(x)))


def gates(a, b, A_log, dt_bias):
    """a1: alpha, beta of shape [T][H_v] from logits a, b [T][H_v]."""
    a, b, A_log, dt_bias = map(_f64, (a, b, A_log, dt_bias))
    T, Hv = a.shape
    alpha = np.empty((T, Hv))
    beta = np.empty((T, Hv))
    lib().orc_gates(T, Hv, _p(a), _p(b), _p(A_log), _p(dt_bias), _p(alpha), _p(beta))
    return alpha, beta


def conv(w, state, x, snapshots: bool = False):
    """a2: conv + SiLU.  Returns (out [T][C], new state [C][W], snaps [T][C][W] or None)."""
    w, x = _f64(w), _f64(x)
    st = _f64(state).copy()
    T, C = x.shape
    W = w.shape[1]
    out = np.empty((T, C))
    snap = np.empty((T, C, W)) if snapshots else None
    lib().orc_conv(T, C, W, _p(w), _p(st), _p(x), _p(out), _p(snap))
    return out, st, snap


def l2norm_split(dims: Dims, xc):
    """a3: (qn [T][H_k][d_k], kn [T][H_k][d_k], v [T][H_v][d_v]) from conv outputs."""
    xc = _f64(xc)
    T = xc.shape[0]
    qn = np.empty((T, dims.n_k_heads, dims.d_k))
    kn = np.empty((T, dims.n_k_heads, dims.d_k))
    v = np.empty((T, dims.n_v_heads, dims.d_v))
    d = dims.c()
    lib().orc_l2norm_split(ctypes.byref(d), T, _p(xc), _p(qn), _p(kn), _p(v))
    return qn, kn, v


def delta_step(H, q, k, v, alpha: float, beta: float):
    """a4 for one head and one token on H = S^T [d_k][d_v].  Returns (H_new, o)."""
    Hn = _f64(H).copy()
    q, k, v = map(_f64, (q, k, v))
    dk, dv = Hn.shape
    o = np.empty(dv)
    lib().orc_delta_step(dk, dv, _p(Hn), _p(q), _p(k), _p(v), float(alpha), float(beta), _p(o))
    return Hn, o


def recurrence(dims: Dims, qn, kn, v, alpha, beta, H, snapshots: bool = False):
    """a4 over T tokens, all heads.  Returns (H_new, o [T][H_v][d_v], snaps or None)."""
    qn, kn, v, alpha, beta = map(_f64, (qn, kn, v, alpha, beta))
    Hn = _f64(H).copy()
    T = qn.shape[0]
    o = np.empty((T, dims.n_v_heads, dims.d_v))
    snap = np.empty((T,) + Hn.shape) if snapshots else None
    d = dims.c()
    lib().orc_recurrence(ctypes.byref(d), T, _p(qn), _p(kn), _p(v), _p(alpha), _p(beta),
                         _p(Hn), _p(o), _p(snap))
    return Hn, o, snap


def gated_rmsnorm(o, z, w, eps: float, gate: int = 0):
    """a7: o [T][H_v][d_v], z [T][H_v*d_v], w [d_v] -> y [T][H_v*d_v]; gate 0 multiplies by
    SiLU(z), gate 1 by sigmoid(z)."""
    o, z, w = map(_f64, (o, z, w))
    T, Hv, dv = o.shape
    y = np.empty((T, Hv * dv))
    lib().orc_gated_rmsnorm(T, Hv, dv, _p(o), _p(z), _p(w), float(eps), int(gate), _p(y))
    return y


@dataclass
class MixerResult:
    y: np.ndarray            # [T][H_v*d_v]
    o: np.ndarray            # [T][H_v][d_v]
    H: np.ndarray            # [H_v][d_k][d_v], state after the last token
    conv_state: np.ndarray   # [conv_dim][d_conv]
    H_snap: np.ndarray | None = None      # [T][H_v][d_k][d_v]
    conv_snap: np.ndarray | None = None   # [T][conv_dim][d_conv]


def mixer(dims: Dims, weights: dict, qkv, z, a, b, conv_state, H,
          snapshots: bool = False) -> MixerResult:
    """The whole mixer (a2, a3, a1, a4, a7) for T tokens of one sequence.

    weights: dict with conv_w [conv_dim][d_conv], A_log [H_v], dt_bias [H_v], norm_w [d_v].
    """
    qkv, z, a, b = map(_f64, (qkv, z, a, b))
    cw, Al, dtb, nw = (_f64(weights[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w"))
    cs = _f64(conv_state).copy()
    Hn = _f64(H).copy()
    T = qkv.shape[0]
    y = np.empty((T, dims.n_v_heads * dims.d_v))
    o = np.empty((T, dims.n_v_heads, dims.d_v))
    hs = np.empty((T,) + Hn.shape) if snapshots else None
    csn = np.empty((T,) + cs.shape) if snapshots else None
    d = dims.c()
    lib().orc_mixer(ctypes.byref(d), T, _p(qkv), _p(z), _p(a), _p(b), _p(cw), _p(Al), _p(dtb),
                    _p(nw), _p(cs), _p(Hn), _p(y), _p(o), _p(hs), _p(csn))
    return MixerResult(y, o, Hn, cs, hs, csn)


def mixer_batch(dims: Dims, weights: dict, seqs: list[dict], snapshots: bool = False):
    """Independent sequences in parallel (one OpenMP thread per sequence).

    seqs[i]: dict with qkv [T_i][conv_dim], z, a, b, conv_state, H.  Returns a list of
    MixerResult.
    """
    n = len(seqs)
    cw, Al, dtb, nw = (_f64(weights[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w"))
    keep = []
    Ts = (ctypes.c_int32 * n)()
    arrs = {k: (_D * n)() for k in ("qkv", "z", "a", "b", "cs", "H", "y", "o", "hs", "csn")}
    results = []
    for i, s in enumerate(seqs):
        qkv, z, a, b = (_f64(s[k]) for k in ("qkv", "z", "a", "b"))
        cs = _f64(s["conv_state"]).copy()
        Hn = _f64(s["H"]).copy()
        T = qkv.shape[0]
        Ts[i] = T
        y = np.empty((T, dims.n_v_heads * dims.d_v))
        o = np.empty((T, dims.n_v_heads, dims.d_v))
        hs = np.empty((T,) + Hn.shape) if snapshots else None
        csn = np.empty((T,) + cs.shape) if snapshots else None
        keep += [qkv, z, a, b]
        for k, arr in (("qkv", qkv), ("z", z), ("a", a), ("b", b), ("cs", cs), ("H", Hn),
                       ("y", y), ("o", o), ("hs", hs), ("csn", csn)):
            arrs[k][i] = _p(arr) if arr is not None else None
        results.append(MixerResult(y, o, Hn, cs, hs, csn))
    d = dims.c()
    lib().orc_mixer_batch(ctypes.byref(d), n, Ts, arrs["qkv"], arrs["z"], arrs["a"],
                          arrs["b"], _p(cw), _p(Al), _p(dtb), _p(nw), arrs["cs"], arrs["H"],
                          arrs["y"], arrs["o"], arrs["hs"] if snapshots else None,
                          arrs["csn"] if snapshots else None)
    del keep
    return results


# ------------------------------------------------------------------ projections
# layer_struct.rs, Qwen3SsmLayer: the sequential [Q | K | V | Z] QKVZ projection, the b / a
# gate inputs of ba_gates_k, and out_proj; the dense_gemm fields are the layer's bf16 GEMMs.
# Plain fp64 products; numpy's matmul is the one step.

def proj(x, w) -> np.ndarray:
    """x [M][K] times w [N][K] transposed, in fp64: [M][N]."""
    return _f64(x) @ _f64(w).T


def in_proj_width(dims: Dims) -> int:
    """One in_proj output row: [Q | K | V | Z | b | a]."""
    return dims.conv_dim + dims.n_v_heads * dims.d_v + 2 * dims.n_v_heads


def split_in_proj(dims: Dims, rows) -> dict:
    """The mixer's inputs as column ranges of in_proj output rows [T][width]:
    qkv [T][conv_dim], z [T][H_v d_v], b [T][H_v], a [T][H_v] (that order in the row);
    columns past them (row padding) are not inputs."""
    rows = _f64(rows)
    cd, vd, hv = dims.conv_dim, dims.n_v_heads * dims.d_v, dims.n_v_heads
    assert rows.shape[1] >= cd + vd + 2 * hv
    return {"qkv": rows[:, :cd], "z": rows[:, cd:cd + vd], "b": rows[:, cd + vd:cd + vd + hv],
            "a": rows[:, cd + vd + hv:cd + vd + 2 * hv]}


def chunked(dims: Dims, chunk: int, qn, kn, v, alpha, beta, H, round_operands: bool = False):
    """The chunked (WY / UT-transform) form of a4.  Returns (H_new, o [T][H_v][d_v])."""
    qn, kn, v, alpha, beta = map(_f64, (qn, kn, v, alpha, beta))
    Hn = _f64(H).copy()
    T = qn.shape[0]
    o = np.empty((T, dims.n_v_heads, dims.d_v))
    d = dims.c()
    lib().orc_chunked(ctypes.byref(d), T, int(chunk), _p(qn), _p(kn), _p(v), _p(alpha),
                      _p(beta), _p(Hn), _p(o), 1 if round_operands else 0)
    return Hn, o


# ------------------------------------------------------------------ write-on-accept
# trait_layer.rs, LayerWriteOnAccept (gdn_woa_stash_seq_floats, gdn_woa_bind); layer_struct.rs,
# the gdn_wy4_woa_k / gdn_wy4_fold_k handles.  The pages name a verify that leaves the state
# alone and stashes what a later fold needs; the reading taken: each token's update of the
# delta rule is rank one, S_t = alpha_t S_{t-1} + delta_t k_hat_t^T with
# delta_t = beta_t (v_t - alpha_t S_{t-1} k_hat_t), so the stash holds (alpha_t, k_hat_t,
# delta_t) per token and the fold replays the accepted ones.

def woa_factors(dims: Dims, weights: dict, qkv, a, b, conv_state, H):
    """Per-token factors of the k draft rows of one sequence, from the recurrence itself:
    alpha [k][H_v], k_hat [k][H_k][d_k], delta [k][H_v][d_v] (H stored [H_v][d_k][d_v])."""
    qkv, a, b = map(_f64, (qkv, a, b))
    xc, _, _ = conv(weights["conv_w"], conv_state, qkv)
    qn, kn, v = l2norm_split(dims, xc)
    alpha, beta = gates(a, b, weights["A_log"], weights["dt_bias"])
    G = dims.n_v_heads // dims.n_k_heads
    Hs = _f64(H).copy()
    T = qkv.shape[0]
    delta = np.empty((T, dims.n_v_heads, dims.d_v))
    for t in range(T):
        for h in range(dims.n_v_heads):
            k = kn[t, h // G]
            u = Hs[h].T @ k                      # S_{t-1} k_hat (S = H^T)
            d = beta[t, h] * (v[t, h] - alpha[t, h] * u)
            Hs[h] = alpha[t, h] * Hs[h] + np.outer(k, d)
            delta[t, h] = d
    return alpha, kn, delta


def woa_fold(dims: Dims, H, alpha, k_hat, delta, m: int):
    """The deferred fold: H [H_v][d_k][d_v] after replaying tokens 0 .. m-1."""
    Hn = _f64(H).copy()
    G = dims.n_v_heads // dims.n_k_heads
    for t in range(m):
        for h in range(dims.n_v_heads):
            Hn[h] = alpha[t, h] * Hn[h] + np.outer(k_hat[t, h // G], delta[t, h])
    return Hn
