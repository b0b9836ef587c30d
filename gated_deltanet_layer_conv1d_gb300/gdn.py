"""Thin ctypes binding of libgdn.so (include/gdn.h): argument marshalling only.

Every function here has the name of the C entry point it calls and takes torch tensors
(device memory owned by the caller) where the C call takes device pointers.  All compute
runs in the CUDA kernels of libgdn.so; there is no fallback: if the library is missing
or fails to load, every call raises.  A nonzero status from the C call raises GdnError.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK = 0
GDN_DTYPE_F32 = 0
GDN_DTYPE_BF16 = 1
GDN_DTYPE_F16 = 2  # h-state pools only
GDN_NORM_GATE_SILU = 0
GDN_NORM_GATE_SIGMOID = 1
GDN_PREFILL_TENSOR_FP16 = 0
GDN_PREFILL_F32 = 1
MAX_SEQS = 128
VERIFY_WY_TABLE_SEQS = 128
VERIFY_WY_TABLES_PER_LAYER = 16
VERIFY_WY_TABLE_STRIDE_BYTES = VERIFY_WY_TABLE_SEQS * 8
VERIFY_WY_LAYER_STRIDE_BYTES = VERIFY_WY_TABLES_PER_LAYER * VERIFY_WY_TABLE_STRIDE_BYTES
PREFILL_CHUNK = 64

# Symbols include/gdn.h declares.
EXPORTS = ("gdn_decode_batched", "gdn_verify_multi", "gdn_conv_step", "gdn_prefill_chunked",
           "gdn_prefill_workspace_bytes", "gdn_gated_rmsnorm", "gdn_wy_tables_fill",
           "gdn_status_string", "gdn_version", "gdn_prefill_chunked_noalloc",
           "gdn_fold_accepted", "gdn_decode_batched_h16", "gdn_verify_multi_h16",
           "gdn_gated_rmsnorm_sigmoid", "gdn_proj_gemm", "gdn_in_proj_width", "gdn_in_proj",
           "gdn_out_proj", "gdn_selftest_wait",
           "gdn_state_convert", "gdn_woa_stash_seq_floats", "gdn_verify_woa", "gdn_woa_fold",
           "gdn_woa_clear")
NOALLOC_SCRATCH_BYTES = 64 << 20


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: status {status} ({status_string(status)})")


class gdn_dims(ctypes.Structure):
    _fields_ = [("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("d_conv", ctypes.c_int32),
                ("q_scale", ctypes.c_float), ("l2_eps", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("norm_gate", ctypes.c_int32),
                ("prefill_precision", ctypes.c_int32)]


class gdn_weights(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("norm_w", ctypes.c_void_p)]


class gdn_inputs(ctypes.Structure):
    _fields_ = [("qkv", ctypes.c_void_p), ("qkv_stride", ctypes.c_int64),
                ("z", ctypes.c_void_p), ("z_stride", ctypes.c_int64),
                ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("ab_stride", ctypes.c_int64),
                ("dtype", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libgdn.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libgdn.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        D, W, IN = (ctypes.POINTER(gdn_dims), ctypes.POINTER(gdn_weights),
                    ctypes.POINTER(gdn_inputs))
        L.gdn_decode_batched.argtypes = [D, W, IN, I32, P, P, I32, P, P, P, P, P]
        L.gdn_verify_multi.argtypes = [D, W, IN, I32, P, P, P, I32, P, P, P, P, P, P]
        L.gdn_conv_step.argtypes = [D, W, IN, I32, P, I32, P, I32, P, P, P, P]
        L.gdn_fold_accepted.argtypes = [D, I32, P, P, P, P, I32, P, P, I32, I32, P, P]
        L.gdn_woa_stash_seq_floats.argtypes = [D, I32]
        L.gdn_woa_stash_seq_floats.restype = SZ
        L.gdn_verify_woa.argtypes = [D, W, IN, I32, P, P, P, I32, P, P, I32, P, P, P, P, P]
        L.gdn_woa_fold.argtypes = [D, I32, P, P, P, I32, P, P, P, I32, P, P]
        L.gdn_woa_clear.argtypes = [P, P]
        L.gdn_decode_batched_h16.argtypes = L.gdn_decode_batched.argtypes
        L.gdn_verify_multi_h16.argtypes = L.gdn_verify_multi.argtypes
        L.gdn_state_convert.argtypes = [P, I32, P, I32, I64, P]
        L.gdn_prefill_chunked.argtypes = [D, W, IN, I32, P, I32, I32, I32, P, P, I32, P, P, P,
                                          P, SZ, P, P]
        L.gdn_prefill_chunked_noalloc.argtypes = [D, W, IN, I32, P, I32, I32, I32, P, P, I32, P,
                                                  P, P, P, P]
        L.gdn_prefill_workspace_bytes.argtypes = [D, I32, I32, I32, I32]
        L.gdn_prefill_workspace_bytes.restype = SZ
        L.gdn_gated_rmsnorm.argtypes = [P, P, I64, P, ctypes.c_float, I32, I32, I32, I32, P, P]
        L.gdn_gated_rmsnorm_sigmoid.argtypes = L.gdn_gated_rmsnorm.argtypes
        L.gdn_wy_tables_fill.argtypes = [P, I32, P, P, P]
        L.gdn_proj_gemm.argtypes = [P, I64, P, I64, P, I64, I32, I32, I32, P, P]
        L.gdn_in_proj_width.argtypes = [D]
        L.gdn_in_proj_width.restype = I32
        L.gdn_in_proj.argtypes = [D, I32, P, I64, I32, P, P, P, P]
        L.gdn_out_proj.argtypes = [D, I32, P, I32, P, P, I64, P, P]
        L.gdn_selftest_wait.argtypes = [I64, P, P]
        L.gdn_status_string.argtypes = [I32]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_version.restype = I32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != GDN_OK:
        raise GdnError(fn, status)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_DTYPE_BF16
    if t.dtype == torch.float32:
        return GDN_DTYPE_F32
    raise TypeError(f"unsupported activation dtype {t.dtype}")


@dataclass
class Weights:
    conv_w: torch.Tensor   # [conv_dim][d_conv] f32
    A_log: torch.Tensor    # [H_v] f32
    dt_bias: torch.Tensor  # [H_v] f32
    norm_w: torch.Tensor   # [d_v] f32

    def c(self) -> gdn_weights:
        return gdn_weights(_ptr(self.conv_w), _ptr(self.A_log), _ptr(self.dt_bias),
                           _ptr(self.norm_w))


@dataclass
class Inputs:
    qkv: torch.Tensor  # [T][>= conv_dim]
    z: torch.Tensor    # [T][>= H_v*d_v]
    a: torch.Tensor    # [T][>= H_v]
    b: torch.Tensor    # [T][>= H_v]

    def c(self) -> gdn_inputs:
        for t in (self.qkv, self.z, self.a, self.b):
            assert t.dim() == 2 and t.stride(1) == 1, "rows must be contiguous"
        assert self.a.stride(0) == self.b.stride(0)
        return gdn_inputs(_ptr(self.qkv), self.qkv.stride(0), _ptr(self.z), self.z.stride(0),
                          _ptr(self.a), _ptr(self.b), self.a.stride(0), _dtype_code(self.qkv))


def make_dims(n_k_heads, n_v_heads, d_k, d_v, d_conv, q_scale, l2_eps, norm_eps,
              norm_gate=GDN_NORM_GATE_SILU, prefill_precision=0) -> gdn_dims:
    return gdn_dims(n_k_heads, n_v_heads, d_k, d_v, d_conv, q_scale, l2_eps, norm_eps, norm_gate,
                    prefill_precision)


def gdn_decode_batched(dims: gdn_dims, weights: Weights, inputs: Inputs, n: int, h_pool,
                       conv_pool, n_slots: int, slots, y, core_out=None, status=None,
                       stream=None):
    w, i = weights.c(), inputs.c()
    _check("gdn_decode_batched", lib().gdn_decode_batched(
        ctypes.byref(dims), ctypes.byref(w), ctypes.byref(i), n, _ptr(h_pool), _ptr(conv_pool),
        n_slots, _ptr(slots), _ptr(y), _ptr(core_out), _ptr(status), _stream(stream)))


def gdn_verify_multi(dims: gdn_dims, weights: Weights, inputs: Inputs, n: int, ks_host,
                     wy_tables, conv_pool, n_slots: int, slots, conv_inter, y, core_out=None,
                     status=None, stream=None):
    ks = (ctypes.c_int32 * len(ks_host))(*[int(k) for k in ks_host])
    w, i = weights.c(), inputs.c()
    _check("gdn_verify_multi", lib().gdn_verify_multi(
        ctypes.byref(dims), ctypes.byref(w), ctypes.byref(i), n, ctypes.cast(ks, ctypes.c_void_p),
        _ptr(wy_tables), _ptr(conv_pool), n_slots, _ptr(slots), _ptr(conv_inter), _ptr(y),
        _ptr(core_out), _ptr(status), _stream(stream)))


def gdn_fold_accepted(dims: gdn_dims, n: int, ks_host, accepted, wy_tables, conv_pool,
                      n_slots: int, slots, conv_inter, dtype: int, status=None, stream=None,
                      h_dtype: int = GDN_DTYPE_F32):
    ks = (ctypes.c_int32 * len(ks_host))(*[int(k) for k in ks_host])
    _check("gdn_fold_accepted", lib().gdn_fold_accepted(
        ctypes.byref(dims), n, ctypes.cast(ks, ctypes.c_void_p), _ptr(accepted), _ptr(wy_tables),
        _ptr(conv_pool), n_slots, _ptr(slots), _ptr(conv_inter), int(dtype), int(h_dtype),
        _ptr(status), _stream(stream)))


def gdn_woa_stash_seq_floats(dims: gdn_dims, dtype: int) -> int:
    """4-byte words of write-on-accept stash per sequence."""
    return int(lib().gdn_woa_stash_seq_floats(ctypes.byref(dims), int(dtype)))


def gdn_verify_woa(dims: gdn_dims, weights: Weights, inputs: Inputs, n: int, ks_host,
                   wy_tables, conv_pool, n_slots: int, slots, stash, stash_seqs: int, flag, y,
                   core_out=None, status=None, stream=None):
    """gdn_verify_multi that leaves the states alone and stashes each token's update."""
    ks = (ctypes.c_int32 * len(ks_host))(*[int(k) for k in ks_host])
    w, i = weights.c(), inputs.c()
    _check("gdn_verify_woa", lib().gdn_verify_woa(
        ctypes.byref(dims), ctypes.byref(w), ctypes.byref(i), n, ctypes.cast(ks, ctypes.c_void_p),
        _ptr(wy_tables), _ptr(conv_pool), n_slots, _ptr(slots), _ptr(stash), int(stash_seqs),
        _ptr(flag), _ptr(y), _ptr(core_out), _ptr(status), _stream(stream)))


def gdn_woa_fold(dims: gdn_dims, n: int, accepted, wy_tables, conv_pool, n_slots: int, slots,
                 stash, flag, dtype: int, status=None, stream=None):
    _check("gdn_woa_fold", lib().gdn_woa_fold(
        ctypes.byref(dims), n, _ptr(accepted), _ptr(wy_tables), _ptr(conv_pool), n_slots,
        _ptr(slots), _ptr(stash), _ptr(flag), int(dtype), _ptr(status), _stream(stream)))


def gdn_woa_clear(flag, stream=None):
    _check("gdn_woa_clear", lib().gdn_woa_clear(_ptr(flag), _stream(stream)))


def gdn_decode_batched_h16(dims: gdn_dims, weights: Weights, inputs: Inputs, n: int, h_pool,
                           conv_pool, n_slots: int, slots, y, core_out=None, status=None,
                           stream=None):
    w, i = weights.c(), inputs.c()
    _check("gdn_decode_batched_h16", lib().gdn_decode_batched_h16(
        ctypes.byref(dims), ctypes.byref(w), ctypes.byref(i), n, _ptr(h_pool), _ptr(conv_pool),
        n_slots, _ptr(slots), _ptr(y), _ptr(core_out), _ptr(status), _stream(stream)))


def gdn_verify_multi_h16(dims: gdn_dims, weights: Weights, inputs: Inputs, n: int, ks_host,
                         wy_tables, conv_pool, n_slots: int, slots, conv_inter, y,
                         core_out=None, status=None, stream=None):
    ks = (ctypes.c_int32 * len(ks_host))(*[int(k) for k in ks_host])
    w, i = weights.c(), inputs.c()
    _check("gdn_verify_multi_h16", lib().gdn_verify_multi_h16(
        ctypes.byref(dims), ctypes.byref(w), ctypes.byref(i), n, ctypes.cast(ks, ctypes.c_void_p),
        _ptr(wy_tables), _ptr(conv_pool), n_slots, _ptr(slots), _ptr(conv_inter), _ptr(y),
        _ptr(core_out), _ptr(status), _stream(stream)))


def gdn_state_convert(src, src_dtype: int, dst, dst_dtype: int, count: int, stream=None):
    _check("gdn_state_convert", lib().gdn_state_convert(
        _ptr(src), int(src_dtype), _ptr(dst), int(dst_dtype), int(count), _stream(stream)))


def gdn_conv_step(dims: gdn_dims, weights: Weights, inputs: Inputs, n: int, cu_seqlens,
                  total_tokens: int, conv_pool, n_slots: int, slots, qkv_out, status=None,
                  stream=None):
    w, i = weights.c(), inputs.c()
    _check("gdn_conv_step", lib().gdn_conv_step(
        ctypes.byref(dims), ctypes.byref(w), ctypes.byref(i), n, _ptr(cu_seqlens), total_tokens,
        _ptr(conv_pool), n_slots, _ptr(slots), _ptr(qkv_out), _ptr(status), _stream(stream)))


def gdn_prefill_workspace_bytes(dims: gdn_dims, n: int, total_tokens: int, max_seqlen: int,
                                chunk: int = PREFILL_CHUNK) -> int:
    return int(lib().gdn_prefill_workspace_bytes(ctypes.byref(dims), n, total_tokens,
                                                 max_seqlen, chunk))


def gdn_prefill_chunked(dims: gdn_dims, weights: Weights, inputs: Inputs, n: int, cu_seqlens,
                        total_tokens: int, max_seqlen: int, h_state_ptrs, conv_pool,
                        n_slots: int, slots, y, core_out=None, workspace=None, status=None,
                        stream=None, chunk: int = PREFILL_CHUNK):
    w, i = weights.c(), inputs.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("gdn_prefill_chunked", lib().gdn_prefill_chunked(
        ctypes.byref(dims), ctypes.byref(w), ctypes.byref(i), n, _ptr(cu_seqlens), total_tokens,
        max_seqlen, chunk, _ptr(h_state_ptrs), _ptr(conv_pool), n_slots, _ptr(slots), _ptr(y),
        _ptr(core_out), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)))


def gdn_prefill_chunked_noalloc(dims: gdn_dims, weights: Weights, inputs: Inputs, n: int,
                                cu_seqlens, total_tokens: int, max_seqlen: int, h_state_ptrs,
                                conv_pool, n_slots: int, slots, y, core_out=None, status=None,
                                stream=None, chunk: int = PREFILL_CHUNK):
    """gdn_prefill_chunked without a workspace argument, for callers that cannot allocate
    device memory when they prefill: the library's own fixed scratch (NOALLOC_SCRATCH_BYTES
    per GPU) stands in for it.  Calls that overlap on the GPU race on that scratch."""
    w, i = weights.c(), inputs.c()
    _check("gdn_prefill_chunked_noalloc", lib().gdn_prefill_chunked_noalloc(
        ctypes.byref(dims), ctypes.byref(w), ctypes.byref(i), n, _ptr(cu_seqlens), total_tokens,
        max_seqlen, chunk, _ptr(h_state_ptrs), _ptr(conv_pool), n_slots, _ptr(slots), _ptr(y),
        _ptr(core_out), _ptr(status), _stream(stream)))


def gdn_gated_rmsnorm(o, z, w, eps: float, y, stream=None, sigmoid=False):
    T, Hv, dv = o.shape
    name = "gdn_gated_rmsnorm_sigmoid" if sigmoid else "gdn_gated_rmsnorm"
    _check(name, getattr(lib(), name)(
        _ptr(o), _ptr(z), z.stride(0), _ptr(w), float(eps), T, Hv, dv, _dtype_code(z), _ptr(y),
        _stream(stream)))


def _bf16_rows(t, name):
    assert t.dtype == torch.bfloat16 and t.dim() == 2 and t.stride(1) == 1, \
        f"{name}: bf16 rows with contiguous columns"


def gdn_proj_gemm(a, b, c, status, stream=None):
    """c[M][N] = a[M][K] b[N][K]^T (bf16 in and out, f32 accumulation)."""
    for t, nm in ((a, "a"), (b, "b"), (c, "c")):
        _bf16_rows(t, nm)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == K and c.shape == (M, N)
    _check("gdn_proj_gemm", lib().gdn_proj_gemm(
        _ptr(a), a.stride(0), _ptr(b), b.stride(0), _ptr(c), c.stride(0), M, N, K, _ptr(status),
        _stream(stream)))


def gdn_in_proj_width(dims: gdn_dims) -> int:
    return int(lib().gdn_in_proj_width(ctypes.byref(dims)))


def gdn_in_proj(dims: gdn_dims, hidden, w_in, out, status, stream=None):
    """out[T][width] = rows [Q | K | V | Z | b | a] of hidden[T][H] w_in[width][H]^T."""
    _bf16_rows(hidden, "hidden")
    T, H = hidden.shape
    width = gdn_in_proj_width(dims)
    assert w_in.shape == (width, H) and w_in.is_contiguous() and w_in.dtype == torch.bfloat16
    assert out.shape == (T, width) and out.is_contiguous() and out.dtype == torch.bfloat16
    _check("gdn_in_proj", lib().gdn_in_proj(
        ctypes.byref(dims), H, _ptr(hidden), hidden.stride(0), T, _ptr(w_in), _ptr(out),
        _ptr(status), _stream(stream)))


def in_proj_inputs(dims: gdn_dims, out) -> "Inputs":
    """The mixer's inputs as column ranges of an in_proj output [T][width]."""
    cd = 2 * dims.n_k_heads * dims.d_k + dims.n_v_heads * dims.d_v
    vd, hv = dims.n_v_heads * dims.d_v, dims.n_v_heads
    return Inputs(out[:, :cd], out[:, cd:cd + vd], out[:, cd + vd + hv:cd + vd + 2 * hv],
                  out[:, cd + vd:cd + vd + hv])


def gdn_out_proj(dims: gdn_dims, y, w_out, out, status, stream=None):
    """out[T][H] = y[T][H_v d_v] w_out[H][H_v d_v]^T."""
    _bf16_rows(y, "y")
    _bf16_rows(out, "out")
    T = y.shape[0]
    H = w_out.shape[0]
    assert y.is_contiguous() and w_out.is_contiguous() and w_out.dtype == torch.bfloat16
    assert w_out.shape[1] == y.shape[1] and out.shape == (T, H)
    _check("gdn_out_proj", lib().gdn_out_proj(
        ctypes.byref(dims), H, _ptr(y), T, _ptr(w_out), _ptr(out), out.stride(0), _ptr(status),
        _stream(stream)))


def gdn_selftest_wait(budget_ns: int, status, stream=None):
    """One bounded wait that nothing completes: sets status to GDN_ERR_TIMEOUT (19)."""
    _check("gdn_selftest_wait", lib().gdn_selftest_wait(int(budget_ns), _ptr(status),
                                                        _stream(stream)))


def gdn_wy_tables_fill(ks, h_ptrs, inter_ptrs):
    """Returns the host table block (numpy uint64 [16][128]) the C helper filled."""
    import numpy as np
    n = len(ks)
    tables = np.zeros((VERIFY_WY_TABLES_PER_LAYER, VERIFY_WY_TABLE_SEQS), np.uint64)
    ks_a = np.ascontiguousarray(np.asarray(ks, np.int32))
    hp = np.ascontiguousarray(np.asarray(h_ptrs, np.uint64))
    ip = np.ascontiguousarray(np.asarray(inter_ptrs, np.uint64).reshape(n, 15) if n else
                              np.zeros((0, 15), np.uint64))
    _check("gdn_wy_tables_fill", lib().gdn_wy_tables_fill(
        tables.ctypes.data, n, ks_a.ctypes.data, hp.ctypes.data, ip.ctypes.data))
    return tables


def gdn_version() -> int:
    return int(lib().gdn_version())
