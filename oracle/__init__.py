"""Oracle for the state-cached causal short convolution (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library
under ``state_cached_causal_gb300/`` and never imports it.

The arithmetic lives in ``cconv_oracle.c`` (plain C loops, fp32 accumulation,
no fused multiply-add). This module compiles it with gcc on first use and
marshals numpy arrays into its C entry points. Every array is host memory;
bf16 data travels as raw ``uint16`` bits.

Pages the functions follow (each function's docstring names its passage):
  * "vllm.model_executor.models.zaya" -- ZayaCCA, _mix_with_state
  * "vllm.model_executor.layers.mamba.ops.cpu.gdn_attention" -- the
    causal_conv1d prefill/decode calls and the _spec_forward rolling buffer
  * "Qwen4ExpPLELayer" -- the dilated depthwise conv and its spec/decode/prefill
    dispatch
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cconv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``cconv_oracle.c`` into ``liboracle.so`` (gcc, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.oracle_cconv_fwd_varlen.argtypes = [
        P, I64, P, P, P, I64, I64, I64, I32, I32, I32, P, P, P, I32, I32, I32, I32,
        I32, I32, P, I64]
    lib.oracle_cconv_fwd_varlen.restype = ctypes.c_int
    lib.oracle_cconv_update.argtypes = [
        P, I64, P, I64, I64, I64, I32, I32, I32, P, P, P, I32, I32, P, P, I32, I32,
        I32, I32, I32, P, I64]
    lib.oracle_cconv_update.restype = ctypes.c_int
    lib.oracle_cca_qk_conv.argtypes = [
        P, I64, P, P, P, P, I32, I32, I32, P, I64, P, I32, P, I64, I64, I64,
        I32, I32, I32, P, I64, P, P, P, I32, I32, I32, P, I64, P, I64]
    lib.oracle_cca_qk_conv.restype = ctypes.c_int
    lib.oracle_cconv_fwd_varlen_fused.argtypes = [
        P, I64, P, P, P, I64, I64, I64, I32, I32, I32, P, P, P, I32, I32, I32, I32,
        I32, I32, P, I32, P, I64, P, I64]
    lib.oracle_cconv_fwd_varlen_fused.restype = ctypes.c_int
    lib.oracle_cconv_update_fused.argtypes = [
        P, I64, P, I64, I64, I64, I32, I32, I32, P, P, P, I32, I32, P, P, I32, I32,
        I32, I32, I32, P, I32, P, I64, P, I64]
    lib.oracle_cconv_update_fused.restype = ctypes.c_int
    lib.oracle_cconv_checkpoint_export.argtypes = [
        P, I64, P, I64, I64, I64, I32, I32, I32, P, P, P, I32, P, I32, P, I32, I32, I32,
        I32, I32]
    lib.oracle_cconv_checkpoint_export.restype = ctypes.c_int
    lib.oracle_cca_project_epilogue.argtypes = [
        P, I64, P, I64, P, I64, P, I64, I32, I32, I32, I32, I32, P, I64]
    lib.oracle_cca_project_epilogue.restype = ctypes.c_int
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


# ---- helpers ---------------------------------------------------------------

def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle arrays are float32 or uint16 (bf16 bits), got {a.dtype}")


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a


def _rows(a: np.ndarray) -> int:
    """Row stride (elements) of a 2-D array whose rows are contiguous."""
    if a.ndim == 2 and a.size == 0:
        return a.shape[1]
    assert a.ndim == 2 and a.strides[1] == a.itemsize, "rows must be contiguous"
    return a.strides[0] // a.itemsize


def _pool_strides(pool: np.ndarray):
    assert pool.ndim == 3
    e = pool.itemsize
    return tuple(s // e for s in pool.strides)


def _pool_base(pool: np.ndarray):
    return ctypes.c_void_p(pool.__array_interface__["data"][0])


def bf16_to_f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


# ---- the three operations ---------------------------------------------------

def cconv_fwd_varlen(x, w, bias, pool, state_idx, cu_seqlens, has_init, width, dilation,
                     act, out):
    """Varlen prefill/decode conv with state, in place on ``pool`` and ``out``.

    Follows the prefill and decode conv calls of "gdn_attention"
    (_spec_aware_nonspec: causal conv over each sequence of the packed stream,
    state in the first (width-1) columns) and the "Qwen4ExpPLELayer"
    dilated conv (state_len = (width-1)*dilation).

    x, out: [T, C] (rows contiguous); w: [C, width]; bias: [C] or None;
    pool: [slots, C, cap] view (any strides); state_idx: int32 [B];
    cu_seqlens: int32 [B+1]; has_init: uint8 [B] or None (all true).
    """
    lib = _load()
    dt = _dtype_code(x)
    w = _c(w)
    bias = _c(bias)
    state_idx = _c(state_idx, np.int32)
    cu_seqlens = _c(cu_seqlens, np.int32)
    has_init = _c(has_init, np.uint8)
    ss, sc, scol = _pool_strides(pool)
    B = int(state_idx.shape[0])
    rc = lib.oracle_cconv_fwd_varlen(
        _ptr(x), _rows(x), _ptr(w), _ptr(bias), _pool_base(pool), ss, sc, scol,
        pool.shape[0], pool.shape[2], _dtype_code(pool),
        _ptr(state_idx), _ptr(cu_seqlens), _ptr(has_init),
        B, x.shape[1], width, dilation, act, dt, _ptr(out), _rows(out))
    if rc != 0:
        raise ValueError(f"oracle_cconv_fwd_varlen rejected its arguments ({rc})")


def cconv_update(x, pool, w, bias, state_idx, n_spec, num_accepted, has_init, width,
                 dilation, act, out):
    """Decode (n_spec == 0) or speculative decode (n_spec > 0), in place.

    Follows "gdn_attention" _spec_aware_nonspec (decode branch, first
    width-1 columns) and _spec_forward (rolling buffer: prior window at
    num_accepted-1, keep B[off+1 : off+1+cap-q], append the q new tokens), with
    the dilation of "Qwen4ExpPLELayer".

    x, out: [B*q, C]; num_accepted: int32 [B] (n_spec > 0) or None.
    """
    lib = _load()
    dt = _dtype_code(x)
    w = _c(w)
    bias = _c(bias)
    state_idx = _c(state_idx, np.int32)
    num_accepted = _c(num_accepted, np.int32)
    has_init = _c(has_init, np.uint8)
    ss, sc, scol = _pool_strides(pool)
    B = int(state_idx.shape[0])
    rc = lib.oracle_cconv_update(
        _ptr(x), _rows(x), _pool_base(pool), ss, sc, scol, pool.shape[0], pool.shape[2],
        _dtype_code(pool),
        _ptr(w), _ptr(bias), _ptr(state_idx), B, n_spec, _ptr(num_accepted),
        _ptr(has_init), x.shape[1], width, dilation, act, dt, _ptr(out), _rows(out))
    if rc != 0:
        raise ValueError(f"oracle_cconv_update rejected its arguments ({rc})")


def cconv_fwd_varlen_fused(x, w, bias, pool, state_idx, cu_seqlens, has_init, width,
                           dilation, act, residual, outer=None, token_indices=None):
    """cconv_fwd_varlen with the fused residual epilogue of "Qwen4ExpPLELayer"
    _short_conv, in place on ``pool`` and ``residual``.

    Logical row i (cu_seqlens index logical rows) is physical row
    p = token_indices[i] (identity when None) of x, residual and outer;
    residual[p] = round(residual[p] + act(conv)[i] + outer[p]) in fp32.
    """
    lib = _load()
    dt = _dtype_code(x)
    w, bias = _c(w), _c(bias)
    state_idx = _c(state_idx, np.int32)
    cu_seqlens = _c(cu_seqlens, np.int32)
    has_init = _c(has_init, np.uint8)
    token_indices = _c(token_indices, np.int32)
    ss, sc, scol = _pool_strides(pool)
    B = int(state_idx.shape[0])
    rc = lib.oracle_cconv_fwd_varlen_fused(
        _ptr(x), _rows(x), _ptr(w), _ptr(bias), _pool_base(pool), ss, sc, scol,
        pool.shape[0], pool.shape[2], _dtype_code(pool),
        _ptr(state_idx), _ptr(cu_seqlens), _ptr(has_init),
        B, x.shape[1], width, dilation, act, dt, _ptr(token_indices), x.shape[0],
        _ptr(residual), _rows(residual), _ptr(outer), _rows(outer) if outer is not None else 0)
    if rc != 0:
        raise ValueError(f"oracle_cconv_fwd_varlen_fused rejected its arguments ({rc})")


def cconv_update_fused(x, pool, w, bias, state_idx, n_spec, num_accepted, has_init, width,
                       dilation, act, residual, outer=None, token_indices=None):
    """cconv_update with the fused residual epilogue and logical row order of
    "Qwen4ExpPLELayer" (_short_conv, _short_conv_dilated_dispatch); request s
    owns logical rows [s*q, s*q + q)."""
    lib = _load()
    dt = _dtype_code(x)
    w, bias = _c(w), _c(bias)
    state_idx = _c(state_idx, np.int32)
    num_accepted = _c(num_accepted, np.int32)
    has_init = _c(has_init, np.uint8)
    token_indices = _c(token_indices, np.int32)
    ss, sc, scol = _pool_strides(pool)
    B = int(state_idx.shape[0])
    rc = lib.oracle_cconv_update_fused(
        _ptr(x), _rows(x), _pool_base(pool), ss, sc, scol, pool.shape[0], pool.shape[2],
        _dtype_code(pool),
        _ptr(w), _ptr(bias), _ptr(state_idx), B, n_spec, _ptr(num_accepted),
        _ptr(has_init), x.shape[1], width, dilation, act, dt, _ptr(token_indices),
        x.shape[0], _ptr(residual), _rows(residual), _ptr(outer),
        _rows(outer) if outer is not None else 0)
    if rc != 0:
        raise ValueError(f"oracle_cconv_update_fused rejected its arguments ({rc})")


def cconv_checkpoint_export(x, pool, ck_seq, ck_off, ck_slot, cu_seqlens, width, dilation,
                            token_indices=None):
    """Prefill checkpoint export of "Qwen4ExpPLELayer" (the conv window ending at a
    checkpoint is a copy of its last (width-1)*dilation inputs), in place on ``pool``.

    Checkpoint k: request ck_seq[k], token offset ck_off[k] in [S, L], slot ck_slot[k].
    """
    lib = _load()
    dt = _dtype_code(x)
    ck_seq, ck_off, ck_slot = (np.ascontiguousarray(np.asarray(a, dtype=np.int32))
                               for a in (ck_seq, ck_off, ck_slot))
    cu_seqlens = _c(cu_seqlens, np.int32)
    token_indices = _c(token_indices, np.int32)
    ss, sc, scol = _pool_strides(pool)
    rc = lib.oracle_cconv_checkpoint_export(
        _ptr(x), _rows(x), _pool_base(pool), ss, sc, scol, pool.shape[0], pool.shape[2],
        _dtype_code(pool),
        _ptr(ck_seq), _ptr(ck_off), _ptr(ck_slot), int(ck_seq.shape[0]), _ptr(cu_seqlens),
        int(cu_seqlens.shape[0]) - 1, _ptr(token_indices), x.shape[0], x.shape[1], width,
        dilation, dt)
    if rc != 0:
        raise ValueError(f"oracle_cconv_checkpoint_export rejected its arguments ({rc})")


def cca_qk_conv(qk, w_dw, b_dw, w_gr, b_gr, groups, t0, t1, delayed, delayed_init, pool,
                delayed_state, state_idx, cu_seqlens, has_init, out_qk, out_delayed_prev):
    """Zaya CCA two-stage q/k conv + delayed-v shift with state, in place.

    Follows "vllm.model_executor.models.zaya" ZayaCCA._mix_with_state and the
    two nn.Conv1d modules of ZayaCCA.__init__ (depthwise, then grouped, both
    with bias; the depthwise output is stored in the module dtype).

    qk, out_qk: [T, Cqk]; w_dw: [Cqk, t0]; w_gr: [Cqk, Cqk/groups, t1];
    delayed, out_delayed_prev: [T, Dv]; delayed_init: [Dv];
    pool: [slots, Cqk, cap] view; delayed_state: [slots, Dv].
    """
    lib = _load()
    dt = _dtype_code(qk)
    ss, sc, scol = _pool_strides(pool)
    B = int(np.asarray(state_idx).shape[0])
    state_idx = _c(state_idx, np.int32)
    cu_seqlens = _c(cu_seqlens, np.int32)
    has_init = _c(has_init, np.uint8)
    w_dw, b_dw, w_gr, b_gr = _c(w_dw), _c(b_dw), _c(w_gr), _c(b_gr)
    delayed_init = _c(delayed_init)
    rc = lib.oracle_cca_qk_conv(
        _ptr(qk), _rows(qk), _ptr(w_dw), _ptr(b_dw), _ptr(w_gr), _ptr(b_gr), groups, t0,
        t1, _ptr(delayed), _rows(delayed), _ptr(delayed_init), delayed.shape[1],
        _pool_base(pool), ss, sc, scol, pool.shape[0], pool.shape[2], _dtype_code(pool),
        _ptr(delayed_state),
        _rows(delayed_state), _ptr(state_idx), _ptr(cu_seqlens), _ptr(has_init), B,
        qk.shape[1], dt, _ptr(out_qk), _rows(out_qk), _ptr(out_delayed_prev),
        _rows(out_delayed_prev))
    if rc != 0:
        raise ValueError(f"oracle_cca_qk_conv rejected its arguments ({rc})")


def oracle_f32_to_bf16_scalar(v: float) -> int:
    return int(_load().oracle_f32_to_bf16(ctypes.c_float(v)))


def cca_project_epilogue(qk, conv, v_current, delayed_prev, num_q_heads, num_kv_heads, out):
    """The q/k residual mix and value assembly of "vllm.model_executor.models.zaya"
    ZayaCCA.project after the conv: out = [conv_q + q_res | conv_k + k_res |
    v_current | delayed_prev] per token (head_dim = qk channels / heads)."""
    lib = _load()
    dt = _dtype_code(qk)
    hd = qk.shape[1] // (num_q_heads + num_kv_heads)
    rc = lib.oracle_cca_project_epilogue(
        _ptr(qk), _rows(qk), _ptr(conv), _rows(conv), _ptr(v_current), _rows(v_current),
        _ptr(delayed_prev), _rows(delayed_prev), qk.shape[0], num_q_heads, num_kv_heads, hd, dt,
        _ptr(out), _rows(out))
    if rc != 0:
        raise ValueError(f"oracle_cca_project_epilogue rejected its arguments ({rc})")

