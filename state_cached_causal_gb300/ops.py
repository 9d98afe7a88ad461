"""ctypes binding of libcconv.so (declared in include/cconv.h).

Argument marshalling only: each function takes torch CUDA tensors, checks
their dtypes and shapes, and passes raw device pointers, element strides and
the current CUDA stream to the C entry point of the same name. Every step of
the computation runs in the library's kernels; there is no other path. A
missing library raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcconv.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_LAUNCH, ERR_TOO_LARGE = 0, -1, -2, -3, -4
DTYPE_F32, DTYPE_BF16 = 0, 1
ACT_NONE, ACT_SILU = 0, 1
DERR_SLOT_RANGE, DERR_CU_SEQLENS, DERR_NUM_ACCEPTED, DERR_TIMEOUT = 1, 2, 4, 8
DERR_ROW_INDEX, DERR_CHECKPOINT = 16, 32

_lock = threading.Lock()
_lib = None


class Epilogue(ctypes.Structure):
    """cconv_epilogue_t: residual rows updated in place, optional outer residual,
    optional logical -> physical row map."""
    _fields_ = [("residual", ctypes.c_void_p), ("residual_row_stride", ctypes.c_int64),
                ("outer_residual", ctypes.c_void_p), ("outer_row_stride", ctypes.c_int64),
                ("token_indices", ctypes.c_void_p), ("num_rows", ctypes.c_int32)]


class Pool(ctypes.Structure):
    """cconv_pool_t: [slot, channel, column] view of a conv-state pool."""
    _fields_ = [("p", ctypes.c_void_p), ("s_slot", ctypes.c_int64),
                ("s_chan", ctypes.c_int64), ("s_col", ctypes.c_int64),
                ("num_slots", ctypes.c_int32), ("cap", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class CConvError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn}: status {status} ({status_string(status)})")
        self.status = status


def load():
    """Load libcconv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "state_cached_causal_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.cconv_fwd_varlen.argtypes = [P, I64, P, P, Pool, P, P, P, I32, I32, I32, I32, I32,
                                         I32, I32, P, I64, P, P]
        lib.cconv_fwd_varlen.restype = ctypes.c_int
        lib.cconv_update.argtypes = [P, I64, Pool, P, P, P, I32, I32, P, P, I32, I32, I32, I32,
                                     I32, P, I64, P, P]
        lib.cconv_update.restype = ctypes.c_int
        lib.cconv_fwd_varlen_fused.argtypes = [P, I64, P, P, Pool, P, P, P, I32, I32, I32, I32,
                                               I32, I32, I32, Epilogue, P, P]
        lib.cconv_fwd_varlen_fused.restype = ctypes.c_int
        lib.cconv_update_fused.argtypes = [P, I64, Pool, P, P, P, I32, I32, P, P, I32, I32, I32,
                                           I32, I32, Epilogue, P, P]
        lib.cconv_update_fused.restype = ctypes.c_int
        lib.cconv_checkpoint_export.argtypes = [P, I64, Pool, P, P, P, I32, P, I32, I32, P, I32,
                                                I32, I32, I32, I32, P, P]
        lib.cconv_checkpoint_export.restype = ctypes.c_int
        lib.cca_qk_conv.argtypes = [P, I64, P, P, P, P, I32, I32, I32, P, I64, P, I32, Pool, P,
                                    I64, P, P, P, I32, I32, I32, I32, P, I64, P, I64, P, P]
        lib.cca_qk_conv.restype = ctypes.c_int
        lib.cca_qk_conv_noalloc.argtypes = lib.cca_qk_conv.argtypes
        lib.cca_qk_conv_noalloc.restype = ctypes.c_int
        lib.cca_qk_conv_fused.argtypes = [P, I64, P, P, P, P, I32, I32, I32, I32, P, I64, P, I32,
                                          P, I64, Pool, P, I64, P, P, P, I32, I32, I32, I32, P,
                                          I64, P, P]
        lib.cca_qk_conv_fused.restype = ctypes.c_int
        lib.cconv_status_string.argtypes = [ctypes.c_int]
        lib.cconv_status_string.restype = ctypes.c_char_p
        lib.cconv_abi_version.argtypes = []
        lib.cconv_abi_version.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().cconv_status_string(int(status)).decode()


def abi_version() -> int:
    return int(load().cconv_abi_version())


# ---- marshalling helpers ---------------------------------------------------

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libcconv must live on the GPU")
    return ctypes.c_void_p(t.data_ptr())


def _rows(t: torch.Tensor) -> int:
    if t.dim() != 2 or (t.shape[0] > 1 and t.stride(1) != 1):
        raise ValueError("expected a 2-D tensor with contiguous rows")
    return int(t.stride(0)) if t.shape[0] > 0 else int(t.shape[1])


def _pool(view: torch.Tensor) -> Pool:
    if view.dim() != 3:
        raise ValueError("pool view must be [slot, channel, column]")
    s = view.stride()
    return Pool(ctypes.c_void_p(view.data_ptr()), s[0], s[1], s[2], view.shape[0],
                view.shape[2], _dtype_code(view))


def _same_state_dtype(conv_state, delayed_state):
    if delayed_state.dtype != conv_state.dtype:
        raise TypeError("delayed_state must have the conv-state pool's dtype")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _i32(t, name):
    if t is not None and t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return t


def _u8(t, name):
    if t is not None and t.dtype not in (torch.uint8, torch.bool):
        raise TypeError(f"{name} must be uint8/bool")
    return t


def _check(fn, status):
    if status != OK:
        raise CConvError(fn, status)


# ---- entry points ----------------------------------------------------------

def cconv_fwd_varlen(x, w, bias, conv_states, state_idx, cu_seqlens, has_init, width,
                     dilation, act, out, dev_err=None, stream=None, num_tokens=None):
    """Varlen causal depthwise conv with state (see cconv_fwd_varlen in cconv.h).

    x, out: [T, C]; w: [C, width]; bias: [C] or None; conv_states: [slot, C, cap]
    view (fp32 or bf16, whatever x's dtype); state_idx/cu_seqlens: int32;
    has_init: uint8/bool or None.
    """
    _i32(state_idx, "state_idx")
    _i32(cu_seqlens, "cu_seqlens")
    _u8(has_init, "has_init")
    T = int(x.shape[0]) if num_tokens is None else int(num_tokens)
    rc = load().cconv_fwd_varlen(
        _ptr(x), _rows(x), _ptr(w), _ptr(bias), _pool(conv_states), _ptr(state_idx),
        _ptr(cu_seqlens), _ptr(has_init), int(state_idx.shape[0]), T, int(x.shape[1]),
        int(width), int(dilation), int(act), _dtype_code(x), _ptr(out), _rows(out),
        _ptr(dev_err), _stream(stream))
    _check("cconv_fwd_varlen", rc)


def cconv_update(x, conv_states, w, bias, state_idx, n_spec, num_accepted, has_init, width,
                 dilation, act, out, dev_err=None, stream=None):
    """Decode / speculative decode against the pool (see cconv_update in cconv.h).

    x, out: [B*(1+n_spec), C]; num_accepted: int32 [B] when n_spec > 0.
    """
    _i32(state_idx, "state_idx")
    _i32(num_accepted, "num_accepted")
    _u8(has_init, "has_init")
    rc = load().cconv_update(
        _ptr(x), _rows(x), _pool(conv_states), _ptr(w), _ptr(bias), _ptr(state_idx),
        int(state_idx.shape[0]), int(n_spec), _ptr(num_accepted), _ptr(has_init),
        int(x.shape[1]), int(width), int(dilation), int(act), _dtype_code(x), _ptr(out),
        _rows(out), _ptr(dev_err), _stream(stream))
    _check("cconv_update", rc)


def _epilogue(residual, outer, token_indices, x):
    _i32(token_indices, "token_indices")
    return Epilogue(_ptr(residual), _rows(residual), _ptr(outer),
                    _rows(outer) if outer is not None else 0, _ptr(token_indices),
                    int(x.shape[0]))


def cconv_fwd_varlen_fused(x, w, bias, conv_states, state_idx, cu_seqlens, has_init, width,
                           dilation, act, residual, outer=None, token_indices=None,
                           dev_err=None, stream=None, num_tokens=None):
    """cconv_fwd_varlen with the fused residual epilogue (see cconv_fwd_varlen_fused
    in cconv.h): residual[p] += act(conv)[i] (+ outer[p]), p = token_indices[i].

    x, residual, outer: [R, C] physical rows; num_tokens: logical rows (default
    len(token_indices), else R).
    """
    _i32(state_idx, "state_idx")
    _i32(cu_seqlens, "cu_seqlens")
    _u8(has_init, "has_init")
    if num_tokens is None:
        num_tokens = int(token_indices.shape[0]) if token_indices is not None else int(x.shape[0])
    rc = load().cconv_fwd_varlen_fused(
        _ptr(x), _rows(x), _ptr(w), _ptr(bias), _pool(conv_states), _ptr(state_idx),
        _ptr(cu_seqlens), _ptr(has_init), int(state_idx.shape[0]), int(num_tokens),
        int(x.shape[1]), int(width), int(dilation), int(act), _dtype_code(x),
        _epilogue(residual, outer, token_indices, x), _ptr(dev_err), _stream(stream))
    _check("cconv_fwd_varlen_fused", rc)


def cconv_update_fused(x, conv_states, w, bias, state_idx, n_spec, num_accepted, has_init,
                       width, dilation, act, residual, outer=None, token_indices=None,
                       dev_err=None, stream=None):
    """cconv_update with the fused residual epilogue (see cconv_update_fused in
    cconv.h); request s owns logical rows [s*q, s*q + q)."""
    _i32(state_idx, "state_idx")
    _i32(num_accepted, "num_accepted")
    _u8(has_init, "has_init")
    rc = load().cconv_update_fused(
        _ptr(x), _rows(x), _pool(conv_states), _ptr(w), _ptr(bias), _ptr(state_idx),
        int(state_idx.shape[0]), int(n_spec), _ptr(num_accepted), _ptr(has_init),
        int(x.shape[1]), int(width), int(dilation), int(act), _dtype_code(x),
        _epilogue(residual, outer, token_indices, x), _ptr(dev_err), _stream(stream))
    _check("cconv_update_fused", rc)


def cconv_checkpoint_export(x, conv_states, ckpt_seq, ckpt_offset, ckpt_slot, cu_seqlens,
                            width, dilation, token_indices=None, num_tokens=None,
                            dev_err=None, stream=None):
    """Prefill checkpoint export (see cconv_checkpoint_export in cconv.h): the conv
    window ending at ckpt_offset[k] of request ckpt_seq[k] into slot ckpt_slot[k].

    x: [R, C] physical rows; ckpt_*: int32 [K]; cu_seqlens: int32 [B+1] over
    num_tokens logical rows (default len(token_indices), else R).
    """
    for t, n in ((ckpt_seq, "ckpt_seq"), (ckpt_offset, "ckpt_offset"), (ckpt_slot, "ckpt_slot"),
                 (cu_seqlens, "cu_seqlens"), (token_indices, "token_indices")):
        _i32(t, n)
    if num_tokens is None:
        num_tokens = int(token_indices.shape[0]) if token_indices is not None else int(x.shape[0])
    rc = load().cconv_checkpoint_export(
        _ptr(x), _rows(x), _pool(conv_states), _ptr(ckpt_seq), _ptr(ckpt_offset),
        _ptr(ckpt_slot), int(ckpt_seq.shape[0]), _ptr(cu_seqlens), int(cu_seqlens.shape[0]) - 1,
        int(num_tokens), _ptr(token_indices), int(x.shape[0]), int(x.shape[1]), int(width),
        int(dilation), _dtype_code(x), _ptr(dev_err), _stream(stream))
    _check("cconv_checkpoint_export", rc)


def cca_qk_conv(qk, w_dw, b_dw, w_gr, b_gr, groups, t0, t1, delayed, delayed_init,
                conv_state, delayed_state, state_idx, cu_seqlens, has_init, out_qk,
                out_delayed_prev, dev_err=None, stream=None, num_tokens=None):
    """Zaya CCA two-stage q/k conv + delayed-v shift (see cca_qk_conv in cconv.h)."""
    _cca_call("cca_qk_conv", qk, w_dw, b_dw, w_gr, b_gr, groups, t0, t1, delayed,
              delayed_init, conv_state, delayed_state, state_idx, cu_seqlens, has_init, out_qk,
              out_delayed_prev, dev_err, stream, num_tokens)


def cca_qk_conv_noalloc(qk, w_dw, b_dw, w_gr, b_gr, groups, t0, t1, delayed, delayed_init,
                        conv_state, delayed_state, state_idx, cu_seqlens, has_init, out_qk,
                        out_delayed_prev, dev_err=None, stream=None, num_tokens=None):
    """cca_qk_conv whose kernel scratch lives in a fixed array inside the library,
    for callers that must not allocate (see cca_qk_conv_noalloc in cconv.h). Calls
    whose kernels overlap on the GPU share that scratch and race."""
    _cca_call("cca_qk_conv_noalloc", qk, w_dw, b_dw, w_gr, b_gr, groups, t0, t1, delayed,
              delayed_init, conv_state, delayed_state, state_idx, cu_seqlens, has_init, out_qk,
              out_delayed_prev, dev_err, stream, num_tokens)


def _cca_call(fn, qk, w_dw, b_dw, w_gr, b_gr, groups, t0, t1, delayed, delayed_init,
              conv_state, delayed_state, state_idx, cu_seqlens, has_init, out_qk,
              out_delayed_prev, dev_err, stream, num_tokens):
    _same_state_dtype(conv_state, delayed_state)
    _i32(state_idx, "state_idx")
    _i32(cu_seqlens, "cu_seqlens")
    _u8(has_init, "has_init")
    T = int(qk.shape[0]) if num_tokens is None else int(num_tokens)
    rc = getattr(load(), fn)(
        _ptr(qk), _rows(qk), _ptr(w_dw), _ptr(b_dw), _ptr(w_gr), _ptr(b_gr), int(groups),
        int(t0), int(t1), _ptr(delayed), _rows(delayed), _ptr(delayed_init),
        int(delayed.shape[1]), _pool(conv_state), _ptr(delayed_state), _rows(delayed_state),
        _ptr(state_idx), _ptr(cu_seqlens), _ptr(has_init), int(state_idx.shape[0]), T,
        int(qk.shape[1]), _dtype_code(qk), _ptr(out_qk), _rows(out_qk),
        _ptr(out_delayed_prev), _rows(out_delayed_prev), _ptr(dev_err), _stream(stream))
    _check(fn, rc)


def cca_qk_conv_fused(qk, w_dw, b_dw, w_gr, b_gr, groups, num_q_heads, t0, t1, delayed,
                      delayed_init, v_current, conv_state, delayed_state, state_idx, cu_seqlens,
                      has_init, out, dev_err=None, stream=None, num_tokens=None):
    """cca_qk_conv with ZayaCCA.project's residual mix and value assembly (see
    cca_qk_conv_fused in cconv.h); out: [T, Cqk + 2*Dv] = [query | key | value]."""
    _same_state_dtype(conv_state, delayed_state)
    _i32(state_idx, "state_idx")
    _i32(cu_seqlens, "cu_seqlens")
    _u8(has_init, "has_init")
    T = int(qk.shape[0]) if num_tokens is None else int(num_tokens)
    rc = load().cca_qk_conv_fused(
        _ptr(qk), _rows(qk), _ptr(w_dw), _ptr(b_dw), _ptr(w_gr), _ptr(b_gr), int(groups),
        int(num_q_heads), int(t0), int(t1), _ptr(delayed), _rows(delayed), _ptr(delayed_init),
        int(delayed.shape[1]), _ptr(v_current), _rows(v_current), _pool(conv_state),
        _ptr(delayed_state), _rows(delayed_state), _ptr(state_idx), _ptr(cu_seqlens),
        _ptr(has_init), int(state_idx.shape[0]), T, int(qk.shape[1]), _dtype_code(qk),
        _ptr(out), _rows(out), _ptr(dev_err), _stream(stream))
    _check("cca_qk_conv_fused", rc)

