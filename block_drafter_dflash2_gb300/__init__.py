"""Python binding of libdflash2 (the DFlash2 draft tail on one GB300).

Argument marshalling only: every step runs in the CUDA library through its C ABI
(``include/dflash2.h``). Tensors are passed as device pointers; torch tensors are
accepted for convenience (``data_ptr()``), as are plain integers. The library is
loaded from this package directory; if it has not been built, importing the
entry points raises ``ImportError`` (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash2.so")

OK = 0
ERR_INVALID_ARGUMENT = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE_TOO_SMALL = 3
ERR_CUDA = 4
ERR_DEVICE = 5

BF16 = 0
FP32 = 1

CONV_TAPS_SOFTMAX = 0
CONV_TAPS_RAW = 1 << 0
WALK_VITERBI = 0
WALK_GREEDY = 1 << 1
FIRST_SLOT_1 = 1 << 2  # row 0 of each block is the anchor's position; slots are rows 1..block-1
SCORE_LOGITS = 1 << 3  # whole-tail calls: the walk's score on raw logits (log-softmax score + sum of lse)

DEVERR_ANCHOR_RANGE = 1 << 0
DEVERR_CANDIDATE_RANGE = 1 << 1
DEVERR_WAIT_TIMEOUT = 1 << 2


class Shape(ctypes.Structure):
    """dflash2_shape_t."""
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("block", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("vocab", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("rank", ctypes.c_int32),
        ("conv_group_size", ctypes.c_int32),
        ("conv_kernel_size", ctypes.c_int32),
        ("conv_layers", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
    ]

    @classmethod
    def make(cls, batch, block, hidden, vocab, top_k, rank, conv_layers, dtype="bf16",
             conv_group_size=16, conv_kernel_size=2, raw_taps=False, greedy=False,
             first_slot=0, score_logits=False) -> "Shape":
        flags = (CONV_TAPS_RAW if raw_taps else 0) | (WALK_GREEDY if greedy else 0) | \
            (FIRST_SLOT_1 if first_slot else 0) | (SCORE_LOGITS if score_logits else 0)
        dt = {"bf16": BF16, "f32": FP32, BF16: BF16, FP32: FP32}[dtype]
        return cls(batch, block, hidden, vocab, top_k, rank, conv_group_size, conv_kernel_size,
                   conv_layers, dt, flags)


class DFlash2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None


def load(path: str = LIB_PATH):
    """Load libdflash2.so and declare its signatures. Raises ImportError if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libdflash2.so is not built at {path}; run block_drafter_dflash2_gb300._build.build()")
    lib = ctypes.CDLL(path)
    vp, sz, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
    st = ctypes.c_int
    sp = ctypes.POINTER(Shape)
    lib.dflash2_workspace_size.argtypes = [sp]
    lib.dflash2_workspace_size.restype = sz
    lib.dflash2_conv.argtypes = [sp, vp, vp, vp, vp, sz, vp]
    lib.dflash2_conv.restype = st
    lib.dflash2_select_topk.argtypes = [sp, vp, vp, i32p, vp, vp, vp, sz, vp]
    lib.dflash2_select_topk.restype = st
    lib.dflash2_select_topk_noalloc.argtypes = [sp, vp, vp, i32p, vp, vp, vp]
    lib.dflash2_select_topk_noalloc.restype = st
    lib.dflash2_lmhead_partials.argtypes = [sp, vp, vp, vp, sz, vp]
    lib.dflash2_lmhead_partials.restype = st
    lib.dflash2_merge_partials.argtypes = [sp, i32p, vp, vp, vp, sz, vp]
    lib.dflash2_merge_partials.restype = st
    lib.dflash2_viterbi.argtypes = [sp, i32p, i32p, vp, vp, vp, i32p, i32p, vp, vp, sz, vp]
    lib.dflash2_viterbi.restype = st
    lib.dflash2_draft_tail.argtypes = [sp, vp, vp, vp, vp, vp, i32p, i32p, i32p, vp, i32p, vp, vp, vp, sz, vp]
    lib.dflash2_draft_tail.restype = st
    lib.dflash2_select_topk_gated.argtypes = [sp, vp, vp, vp, i32p, vp, vp, vp, vp, sz, vp]
    lib.dflash2_select_topk_gated.restype = st
    lib.dflash2_viterbi_gated.argtypes = [sp, i32p, i32p, vp, vp, vp, vp, i32p, i32p, vp, vp, sz, vp]
    lib.dflash2_viterbi_gated.restype = st
    lib.dflash2_draft_tail_gated.argtypes = [sp, vp, vp, vp, vp, vp, vp, i32p, i32p, i32p, vp, i32p, vp, vp, vp,
                                             vp, sz, vp]
    lib.dflash2_draft_tail_gated.restype = st
    f32 = ctypes.c_float
    lib.dflash2_sample_walk.argtypes = [sp, i32p, i32p, vp, vp, vp, vp, f32, vp, i32p, i32p, vp, vp, sz, vp]
    lib.dflash2_sample_walk.restype = st
    lib.dflash2_draft_tail_sampled.argtypes = [sp, vp, vp, vp, vp, vp, vp, i32p, f32, vp, i32p, i32p, vp, i32p, vp,
                                               vp, vp, vp, sz, vp]
    lib.dflash2_draft_tail_sampled.restype = st
    lib.dflash2_read_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.dflash2_read_device_error.restype = st
    lib.dflash2_status_string.argtypes = [st]
    lib.dflash2_status_string.restype = ctypes.c_char_p
    lib.dflash2_version.argtypes = []
    lib.dflash2_version.restype = ctypes.c_int32
    _lib = lib
    return lib


def _ptr(x):
    """Device pointer of a torch tensor (must be CUDA and contiguous), an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("tensor arguments must live on the GPU")
        if not x.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a device pointer")


def _ws(ws):
    if hasattr(ws, "data_ptr"):
        return _ptr(ws), ws.numel() * ws.element_size()
    ptr, nbytes = ws
    return ptr, nbytes


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != OK:
        raise DFlash2Error(status, where)


def status_string(status: int) -> str:
    return load().dflash2_status_string(status).decode()


def version() -> int:
    return load().dflash2_version()


def workspace_size(shape: Shape) -> int:
    return int(load().dflash2_workspace_size(ctypes.byref(shape)))


def conv(shape: Shape, x, conv_w, y, ws, stream=None):
    """dflash2_conv: all conv layers on x [B,T,H] -> y [B,T,H]."""
    wp, wn = _ws(ws)
    _check(load().dflash2_conv(ctypes.byref(shape), _ptr(x), _ptr(conv_w), _ptr(y), wp, wn, _stream(stream)),
           "dflash2_conv")


def select_topk(shape: Shape, rows, lm_head, cand_ids, cand_lp, lse, ws, stream=None):
    """dflash2_select_topk: rows [M,H] x lm_head [V,H] -> top-K ids / log-probs, lse."""
    wp, wn = _ws(ws)
    _check(load().dflash2_select_topk(ctypes.byref(shape), _ptr(rows), _ptr(lm_head), _ptr(cand_ids),
                                      _ptr(cand_lp), _ptr(lse), wp, wn, _stream(stream)), "dflash2_select_topk")


def select_topk_noalloc(shape: Shape, rows, lm_head, cand_ids, cand_lp, lse, stream=None):
    """dflash2_select_topk_noalloc: the same selection with the library's own fixed device
    scratch instead of a workspace, for callers that cannot allocate device memory. Calls
    share that scratch, so calls that may overlap on the GPU must be serialised."""
    _check(load().dflash2_select_topk_noalloc(ctypes.byref(shape), _ptr(rows), _ptr(lm_head), _ptr(cand_ids),
                                              _ptr(cand_lp), _ptr(lse), _stream(stream)),
           "dflash2_select_topk_noalloc")


def lmhead_partials(shape: Shape, rows, lm_head, ws, stream=None):
    """dflash2_lmhead_partials: contraction + fused per-partition top-16 / (max, sum) into ws."""
    wp, wn = _ws(ws)
    _check(load().dflash2_lmhead_partials(ctypes.byref(shape), _ptr(rows), _ptr(lm_head), wp, wn, _stream(stream)),
           "dflash2_lmhead_partials")


def merge_partials(shape: Shape, cand_ids, cand_lp, lse, ws, stream=None):
    """dflash2_merge_partials: the workspace's partials -> top-K ids, log-probs, lse."""
    wp, wn = _ws(ws)
    _check(load().dflash2_merge_partials(ctypes.byref(shape), _ptr(cand_ids), _ptr(cand_lp), _ptr(lse), wp, wn,
                                         _stream(stream)), "dflash2_merge_partials")


def viterbi(shape: Shape, anchor, cand_ids, cand_lp, U, V, path_ids, path_idx, score, ws, stream=None):
    """dflash2_viterbi: transitions through U/V and the walk from the anchor."""
    wp, wn = _ws(ws)
    _check(load().dflash2_viterbi(ctypes.byref(shape), _ptr(anchor), _ptr(cand_ids), _ptr(cand_lp), _ptr(U),
                                  _ptr(V), _ptr(path_ids), _ptr(path_idx), _ptr(score), wp, wn,
                                  _stream(stream)), "dflash2_viterbi")


def draft_tail(shape: Shape, hidden, lm_head, U, V, conv_w, anchor, path_ids, path_idx, score, ws,
               cand_ids=None, cand_lp=None, lse=None, stream=None):
    """dflash2_draft_tail: conv -> LM-head top-K + lse -> transitions + walk, one call."""
    wp, wn = _ws(ws)
    _check(load().dflash2_draft_tail(ctypes.byref(shape), _ptr(hidden), _ptr(lm_head), _ptr(U), _ptr(V),
                                     _ptr(conv_w), _ptr(anchor), _ptr(path_ids), _ptr(path_idx), _ptr(score),
                                     _ptr(cand_ids), _ptr(cand_lp), _ptr(lse), wp, wn, _stream(stream)),
           "dflash2_draft_tail")


def select_topk_gated(shape: Shape, rows, lm_head, gate_w, cand_ids, cand_lp, lse, gate, ws, stream=None):
    """dflash2_select_topk_gated: select_topk plus the context gate rows . gate_w [R,H] -> gate [M,R]."""
    wp, wn = _ws(ws)
    _check(load().dflash2_select_topk_gated(ctypes.byref(shape), _ptr(rows), _ptr(lm_head), _ptr(gate_w),
                                            _ptr(cand_ids), _ptr(cand_lp), _ptr(lse), _ptr(gate), wp, wn,
                                            _stream(stream)), "dflash2_select_topk_gated")


def viterbi_gated(shape: Shape, anchor, cand_ids, cand_lp, U, V, gate, path_ids, path_idx, score, ws, stream=None):
    """dflash2_viterbi_gated: transitions U (.) gate_t against V, and the walk from the anchor."""
    wp, wn = _ws(ws)
    _check(load().dflash2_viterbi_gated(ctypes.byref(shape), _ptr(anchor), _ptr(cand_ids), _ptr(cand_lp), _ptr(U),
                                        _ptr(V), _ptr(gate), _ptr(path_ids), _ptr(path_idx), _ptr(score), wp, wn,
                                        _stream(stream)), "dflash2_viterbi_gated")


def draft_tail_gated(shape: Shape, hidden, lm_head, U, V, conv_w, gate_w, anchor, path_ids, path_idx, score, ws,
                     cand_ids=None, cand_lp=None, lse=None, gate=None, stream=None):
    """dflash2_draft_tail_gated: the whole tail with the context gate (gate [B,T,R] optional out)."""
    wp, wn = _ws(ws)
    _check(load().dflash2_draft_tail_gated(ctypes.byref(shape), _ptr(hidden), _ptr(lm_head), _ptr(U), _ptr(V),
                                           _ptr(conv_w), _ptr(gate_w), _ptr(anchor), _ptr(path_ids),
                                           _ptr(path_idx), _ptr(score), _ptr(cand_ids), _ptr(cand_lp), _ptr(lse),
                                           _ptr(gate), wp, wn, _stream(stream)), "dflash2_draft_tail_gated")


def sample_walk(shape: Shape, anchor, cand_ids, cand_lp, U, V, temperature, uniforms, path_ids, path_idx, score,
                ws, gate=None, stream=None):
    """dflash2_sample_walk: a path drawn at temperature > 0 with the caller's uniforms [B,T];
    score receives log P(path)."""
    wp, wn = _ws(ws)
    _check(load().dflash2_sample_walk(ctypes.byref(shape), _ptr(anchor), _ptr(cand_ids), _ptr(cand_lp), _ptr(U),
                                      _ptr(V), _ptr(gate), ctypes.c_float(temperature), _ptr(uniforms),
                                      _ptr(path_ids), _ptr(path_idx), _ptr(score), wp, wn, _stream(stream)),
           "dflash2_sample_walk")


def draft_tail_sampled(shape: Shape, hidden, lm_head, U, V, conv_w, anchor, temperature, uniforms, path_ids,
                       path_idx, score, ws, gate_w=None, cand_ids=None, cand_lp=None, lse=None, gate=None,
                       stream=None):
    """dflash2_draft_tail_sampled: the whole tail, the walk drawing a path at temperature > 0."""
    wp, wn = _ws(ws)
    _check(load().dflash2_draft_tail_sampled(ctypes.byref(shape), _ptr(hidden), _ptr(lm_head), _ptr(U), _ptr(V),
                                             _ptr(conv_w), _ptr(gate_w), _ptr(anchor), ctypes.c_float(temperature),
                                             _ptr(uniforms), _ptr(path_ids), _ptr(path_idx), _ptr(score),
                                             _ptr(cand_ids), _ptr(cand_lp), _ptr(lse), _ptr(gate), wp, wn,
                                             _stream(stream)), "dflash2_draft_tail_sampled")


def read_device_error(ws, stream=None) -> int:
    """Synchronise the stream, return and clear the workspace's device error word."""
    wp, _ = _ws(ws)
    code = ctypes.c_int32(0)
    _check(load().dflash2_read_device_error(wp, _stream(stream), ctypes.byref(code)), "dflash2_read_device_error")
    return int(code.value)
