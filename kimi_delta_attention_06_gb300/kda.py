"""Thin ctypes binding of the KDA C ABI (include/kda.h).

The functions named like the C entry points (``kda_chunk_prefill``,
``kda_chunk_prefill_ex``, ``kda_chunk_prefill_noalloc``, ``kda_decode_step``,
``kda_prepare_inputs``, ``kda_output_norm``, ``kda_decode_multi``, ``kda_ckpt_count``,
``kda_device_status``, ``kda_status_string``, ``kda_chunk_size``) only marshal
arguments: torch
tensors become raw device pointers, the current torch stream becomes the
``stream`` argument, and a negative status raises ``KdaError``.  ``prefill``
and ``decode_step`` additionally allocate the output tensors with torch.

There is no fallback: if ``libkda.so`` is missing or cannot be loaded the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libkda.so")
_lock = threading.Lock()
_lib = None

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_CUDA = -3
KDA_ERR_TIMEOUT = -4
KDA_ERR_RANGE = -5
KDA_OUT_BF16 = 0
KDA_OUT_F32 = 1
KDA_NOALLOC_MAX_SEQ_HEADS = 32
KDA_MAX_SEGMENTS = 64
KDA_DECAY_CHANNEL = 0
KDA_DECAY_HEAD = 1
KDA_DECAY_NONE = 2

_vp = ctypes.c_void_p
_i = ctypes.c_int


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {kda_status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libkda.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"KDA CUDA library not built: {_LIB_PATH} is missing "
                                   "(run kimi_delta_attention_06_gb300.build.build())")
            lib = ctypes.CDLL(_LIB_PATH)
            for name in ("kda_chunk_prefill", "kda_chunk_prefill_noalloc"):
                fn = getattr(lib, name)
                fn.restype = _i
                fn.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp, _vp, _i, _vp]
            lib.kda_chunk_prefill_ex.restype = _i
            lib.kda_chunk_prefill_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i,
                                                 _vp, _vp, _i, _i, _vp, _vp, _vp, ctypes.c_float, _vp]
            lib.kda_chunk_prefill_segmented.restype = _i
            lib.kda_chunk_prefill_segmented.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _i,
                                                        _vp, _vp, _i, _i, _i, _i, _vp, ctypes.c_float, _vp]
            lib.kda_chunk_prefill_segmented_ex.restype = _i
            lib.kda_chunk_prefill_segmented_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                                                           _i, _vp, _vp, _i, _i, _vp, _i, _vp, ctypes.c_float, _vp]
            lib.kda_segment_plan.restype = _i
            lib.kda_segment_plan.argtypes = [_i, _i, _i, _i, _vp, _vp, _i]
            lib.kda_prefill_clusters_at_once.restype = _i
            lib.kda_prefill_clusters_at_once.argtypes = []
            lib.kda_decode_step.restype = _i
            lib.kda_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]
            lib.kda_decode_multi.restype = _i
            lib.kda_decode_multi.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _i,
                                             _i, _i, _i, _i, _i, _i, _vp]
            lib.kda_prepare_inputs.restype = _i
            lib.kda_prepare_inputs.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                               _vp, _vp, _vp, _vp, _vp, _vp]
            lib.kda_output_norm.restype = _i
            lib.kda_output_norm.argtypes = [_vp, _i, _vp, ctypes.c_float, _vp, _i, _i, _i, _vp]
            lib.kda_ckpt_count.restype = ctypes.c_int64
            lib.kda_ckpt_count.argtypes = [_vp, _i, _i]
            lib.kda_ckpt_count_ex.restype = ctypes.c_int64
            lib.kda_ckpt_count_ex.argtypes = [_vp, _vp, _i, _i]
            lib.kda_device_status.restype = _i
            lib.kda_device_status.argtypes = [_vp]
            lib.kda_status_string.restype = ctypes.c_char_p
            lib.kda_status_string.argtypes = [_i]
            lib.kda_chunk_size.restype = _i
            lib.kda_chunk_size.argtypes = []
            lib.kda_debug_expire_wait.restype = _i
            lib.kda_debug_expire_wait.argtypes = [ctypes.c_ulonglong, _vp]
            _lib = lib
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("KDA tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, what: str):
    if rc != KDA_OK:
        raise KdaError(rc, what)


def _bits16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.bfloat16:
        raise TypeError(f"expected a bfloat16 tensor, got {t.dtype}")
    return t


# --- the C entry points, one to one --------------------------------------------------

def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def kda_chunk_size() -> int:
    return int(load().kda_chunk_size())


def kda_ckpt_count(cu_seqlens_host: torch.Tensor, ckpt_stride: int) -> int:
    cu = cu_seqlens_host.to(device="cpu", dtype=torch.int32).contiguous()
    n = load().kda_ckpt_count(ctypes.c_void_p(cu.data_ptr()), cu.numel() - 1, int(ckpt_stride))
    if n < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "kda_ckpt_count")
    return int(n)


def kda_ckpt_count_ex(cu_seqlens_host: torch.Tensor, start_pos_host, ckpt_stride: int) -> int:
    cu = cu_seqlens_host.to(device="cpu", dtype=torch.int32).contiguous()
    sp = None if start_pos_host is None else start_pos_host.to(device="cpu", dtype=torch.int32).contiguous()
    n = load().kda_ckpt_count_ex(ctypes.c_void_p(cu.data_ptr()), None if sp is None else ctypes.c_void_p(sp.data_ptr()),
                                 cu.numel() - 1, int(ckpt_stride))
    if n < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "kda_ckpt_count_ex")
    return int(n)


def _call_prefill(name, q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host, num_seqs,
                  total_tokens, H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride, stream):
    cu_host = cu_seqlens_host.to(device="cpu", dtype=torch.int32).contiguous()
    rc = getattr(load(), name)(
        _ptr(_bits16(q)), _ptr(_bits16(k)), _ptr(_bits16(v)), _ptr(log_alpha), _ptr(_bits16(beta)),
        _ptr(init_state), _ptr(cu_seqlens), ctypes.c_void_p(cu_host.data_ptr()),
        int(num_seqs), int(total_tokens), int(H), int(Dk), int(Dv),
        _ptr(out), int(out_dtype), _ptr(final_state), _ptr(ckpt_states), int(ckpt_stride),
        _stream(stream))
    _check(rc, name)


def kda_chunk_prefill(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host,
                      num_seqs: int, total_tokens: int, H: int, Dk: int, Dv: int,
                      out, out_dtype: int, final_state, ckpt_states, ckpt_stride: int, stream=None):
    _call_prefill("kda_chunk_prefill", q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host,
                  num_seqs, total_tokens, H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride, stream)


def kda_chunk_prefill_ex(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host,
                         num_seqs: int, total_tokens: int, H: int, Dk: int, Dv: int,
                         out, out_dtype: int, final_state, ckpt_states, ckpt_stride: int, decay: int,
                         start_pos=None, start_pos_host=None, out_norm_gamma=None, out_norm_eps: float = 1e-6,
                         stream=None):
    sp_host = None if start_pos_host is None else start_pos_host.to(device="cpu", dtype=torch.int32).contiguous()
    cu_host = cu_seqlens_host.to(device="cpu", dtype=torch.int32).contiguous()
    rc = load().kda_chunk_prefill_ex(
        _ptr(_bits16(q)), _ptr(_bits16(k)), _ptr(_bits16(v)), _ptr(log_alpha), _ptr(_bits16(beta)),
        _ptr(init_state), _ptr(cu_seqlens), ctypes.c_void_p(cu_host.data_ptr()),
        int(num_seqs), int(total_tokens), int(H), int(Dk), int(Dv),
        _ptr(out), int(out_dtype), _ptr(final_state), _ptr(ckpt_states), int(ckpt_stride), int(decay),
        _ptr(start_pos), None if sp_host is None else ctypes.c_void_p(sp_host.data_ptr()),
        _ptr(out_norm_gamma), float(out_norm_eps), _stream(stream))
    _check(rc, "kda_chunk_prefill_ex")


def kda_chunk_prefill_segmented(q, k, v, log_alpha, beta, init_state, total_tokens: int, H: int, Dk: int, Dv: int,
                                out, out_dtype: int, final_state, ckpt_states, ckpt_stride: int, decay: int,
                                start_pos: int, segments: int, out_norm_gamma=None, out_norm_eps: float = 1e-6,
                                stream=None):
    rc = load().kda_chunk_prefill_segmented(
        _ptr(_bits16(q)), _ptr(_bits16(k)), _ptr(_bits16(v)), _ptr(log_alpha), _ptr(_bits16(beta)),
        _ptr(init_state), int(total_tokens), int(H), int(Dk), int(Dv),
        _ptr(out), int(out_dtype), _ptr(final_state), _ptr(ckpt_states), int(ckpt_stride), int(decay),
        int(start_pos), int(segments), _ptr(out_norm_gamma), float(out_norm_eps), _stream(stream))
    _check(rc, "kda_chunk_prefill_segmented")


def kda_chunk_prefill_segmented_ex(q, k, v, log_alpha, beta, init_state, cu_seqlens_host, num_seqs: int,
                                   total_tokens: int, H: int, Dk: int, Dv: int, out, out_dtype: int, final_state,
                                   ckpt_states, ckpt_stride: int, decay: int, start_pos_host, segments: int,
                                   out_norm_gamma=None, out_norm_eps: float = 1e-6, stream=None):
    cu_host = cu_seqlens_host.to(device="cpu", dtype=torch.int32).contiguous()
    sp_host = None if start_pos_host is None else \
        torch.as_tensor(start_pos_host).to(device="cpu", dtype=torch.int32).contiguous()
    rc = load().kda_chunk_prefill_segmented_ex(
        _ptr(_bits16(q)), _ptr(_bits16(k)), _ptr(_bits16(v)), _ptr(log_alpha), _ptr(_bits16(beta)),
        _ptr(init_state), ctypes.c_void_p(cu_host.data_ptr()), int(num_seqs), int(total_tokens), int(H), int(Dk),
        int(Dv), _ptr(out), int(out_dtype), _ptr(final_state), _ptr(ckpt_states), int(ckpt_stride), int(decay),
        None if sp_host is None else ctypes.c_void_p(sp_host.data_ptr()), int(segments), _ptr(out_norm_gamma),
        float(out_norm_eps), _stream(stream))
    _check(rc, "kda_chunk_prefill_segmented_ex")


def kda_segment_plan(total_tokens: int, start_pos: int, segments: int, ckpt_stride: int = 0):
    """(bounds, ckpt_slots) of kda_chunk_prefill_segmented's plan: the segment bounds in tokens
    from the prompt's start, and for each of the prompt's checkpoints the slot it comes from,
    counted over run A's slots then run F's (empty when there are no checkpoints or one plain
    prefill runs)."""
    bounds = (ctypes.c_int32 * (KDA_MAX_SEGMENTS + 1))()
    cap = 1 << 16
    slots = (ctypes.c_int32 * cap)()
    P = load().kda_segment_plan(int(total_tokens), int(start_pos), int(segments), int(ckpt_stride),
                                ctypes.cast(bounds, ctypes.c_void_p), ctypes.cast(slots, ctypes.c_void_p), cap)
    _check(min(P, 0), "kda_segment_plan")
    n = kda_ckpt_count_ex(torch.tensor([0, int(total_tokens)], dtype=torch.int32),
                          torch.tensor([int(start_pos)], dtype=torch.int32), ckpt_stride) \
        if ckpt_stride > 0 and P >= 3 else 0
    return [int(x) for x in bounds[:P + 1]], [int(x) for x in slots[:n]]


def kda_prefill_clusters_at_once() -> int:
    n = load().kda_prefill_clusters_at_once()
    _check(min(n, 0), "kda_prefill_clusters_at_once")
    return int(n)


def segments_for(H: int, clusters_at_once: Optional[int] = None, num_seqs: int = 1) -> int:
    """Segments for kda_chunk_prefill_segmented(_ex): clusters_at_once // H + 1, at most 32, so
    that each run (P - 1 segments of a single sequence per head) fills the device in one wave.
    0 (a plain prefill) when that is below 3, or when the call's (sequence, head) pairs
    already fill the device (num_seqs * H >= clusters_at_once): splitting then only adds work.
    Beyond 32 segments the serial chain of segment states and the per-segment fixed costs
    grow while the runs shrink, and short segments are less likely to let their transitions
    be dropped."""
    n = kda_prefill_clusters_at_once() if clusters_at_once is None else int(clusters_at_once)
    H, num_seqs = max(1, int(H)), max(1, int(num_seqs))
    if num_seqs * H >= n:
        return 0
    p = min(n // H + 1, 32)
    return p if p >= 3 else 0


def kda_chunk_prefill_noalloc(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host,
                              num_seqs: int, total_tokens: int, H: int, Dk: int, Dv: int,
                              out, out_dtype: int, final_state, ckpt_states, ckpt_stride: int, stream=None):
    _call_prefill("kda_chunk_prefill_noalloc", q, k, v, log_alpha, beta, init_state, cu_seqlens,
                  cu_seqlens_host, num_seqs, total_tokens, H, Dk, Dv, out, out_dtype, final_state, ckpt_states,
                  ckpt_stride, stream)


def kda_decode_step(q, k, v, log_alpha, beta, state, out, out_dtype: int,
                    N: int, H: int, Dk: int, Dv: int, stream=None):
    rc = load().kda_decode_step(_ptr(_bits16(q)), _ptr(_bits16(k)), _ptr(_bits16(v)), _ptr(log_alpha),
                                _ptr(_bits16(beta)), _ptr(state), _ptr(out), int(out_dtype),
                                int(N), int(H), int(Dk), int(Dv), _stream(stream))
    _check(rc, "kda_decode_step")


def kda_decode_multi(q, k, v, log_alpha, beta, state_pool, num_slots: int, state_slots, num_tokens,
                     commit: int, out, out_dtype: int, N: int, K: int, H: int, Dk: int, Dv: int,
                     decay: int = KDA_DECAY_CHANNEL, stream=None):
    rc = load().kda_decode_multi(_ptr(_bits16(q)), _ptr(_bits16(k)), _ptr(_bits16(v)), _ptr(log_alpha),
                                 _ptr(_bits16(beta)), _ptr(state_pool), int(num_slots), _ptr(state_slots),
                                 _ptr(num_tokens), int(commit), _ptr(out), int(out_dtype),
                                 int(N), int(K), int(H), int(Dk), int(Dv), int(decay), _stream(stream))
    _check(rc, "kda_decode_multi")


def kda_prepare_inputs(xq, xk, xv, conv_w, conv_state, a_raw, b_raw, cu_seqlens, cu_seqlens_host,
                       num_seqs: int, total_tokens: int, H: int, D: int, conv_act: int,
                       q, k, v, log_alpha, beta, stream=None):
    cu_host = cu_seqlens_host.to(device="cpu", dtype=torch.int32).contiguous()
    rc = load().kda_prepare_inputs(_ptr(_bits16(xq)), _ptr(_bits16(xk)), _ptr(_bits16(xv)), _ptr(conv_w),
                                   _ptr(None if conv_state is None else _bits16(conv_state)), _ptr(a_raw),
                                   _ptr(_bits16(b_raw)), _ptr(cu_seqlens), ctypes.c_void_p(cu_host.data_ptr()),
                                   int(num_seqs), int(total_tokens), int(H), int(D), int(conv_act),
                                   _ptr(_bits16(q)), _ptr(_bits16(k)), _ptr(_bits16(v)), _ptr(log_alpha),
                                   _ptr(_bits16(beta)), _stream(stream))
    _check(rc, "kda_prepare_inputs")


def kda_output_norm(o, o_dtype: int, gamma, eps: float, y, total_tokens: int, H: int, Dv: int, stream=None):
    rc = load().kda_output_norm(_ptr(o), int(o_dtype), _ptr(gamma), float(eps), _ptr(_bits16(y)),
                                int(total_tokens), int(H), int(Dv), _stream(stream))
    _check(rc, "kda_output_norm")


def kda_debug_expire_wait(limit_ns: int, stream=None):
    _check(load().kda_debug_expire_wait(int(limit_ns), _stream(stream)), "kda_debug_expire_wait")


def kda_device_status(stream=None) -> int:
    return int(load().kda_device_status(_stream(stream)))


# --- conveniences: allocate outputs, then call the entry point ----------------------------

def prefill(q, k, v, log_alpha, beta, cu_seqlens_host, init_state=None, ckpt_stride: int = 0,
            out_dtype=torch.bfloat16, want_final: bool = True, cu_seqlens=None, stream=None,
            decay: int = KDA_DECAY_CHANNEL, start_pos_host=None, norm_gamma=None, norm_eps: float = 1e-6,
            segments: int = 0):
    """Allocate outputs and run kda_chunk_prefill (kda_chunk_prefill_ex for another decay
    layout, for start positions or with the output norm fused in: norm_gamma [H, Dv];
    kda_chunk_prefill_segmented(_ex) when segments > 0).
    Returns (out, final_state, ckpt_states)."""
    T, H, Dk = q.shape
    Dv = v.shape[2]
    cu_host = cu_seqlens_host.to(device="cpu", dtype=torch.int32).contiguous()
    N = cu_host.numel() - 1
    dev = q.device
    if cu_seqlens is None:
        cu_seqlens = cu_host.to(dev, non_blocking=False)
    out = torch.empty(T, H, Dv, device=dev, dtype=out_dtype)
    fin = torch.empty(N, H, Dk, Dv, device=dev, dtype=torch.float32) if want_final else None
    nck = kda_ckpt_count_ex(cu_host, start_pos_host, ckpt_stride) if ckpt_stride > 0 else 0
    ck = torch.empty(nck, H, Dk, Dv, device=dev, dtype=torch.float32) if ckpt_stride > 0 else None
    odt = KDA_OUT_F32 if out_dtype == torch.float32 else KDA_OUT_BF16
    if segments > 0 and N == 1:
        sp0 = 0 if start_pos_host is None else int(torch.as_tensor(start_pos_host).reshape(-1)[0])
        kda_chunk_prefill_segmented(q, k, v, log_alpha, beta, init_state, T, H, Dk, Dv, out, odt, fin,
                                    ck if nck > 0 else None, ckpt_stride, decay, sp0, segments, norm_gamma,
                                    norm_eps, stream)
    elif segments > 0:
        kda_chunk_prefill_segmented_ex(q, k, v, log_alpha, beta, init_state, cu_host, N, T, H, Dk, Dv, out, odt,
                                       fin, ck if nck > 0 else None, ckpt_stride, decay, start_pos_host, segments,
                                       norm_gamma, norm_eps, stream)
    elif decay == KDA_DECAY_CHANNEL and start_pos_host is None and norm_gamma is None:
        kda_chunk_prefill(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_host, N, T, H, Dk, Dv,
                          out, odt, fin, ck if nck > 0 else None, ckpt_stride, stream)
    else:
        sp = None if start_pos_host is None else start_pos_host.to(device="cpu", dtype=torch.int32).contiguous()
        kda_chunk_prefill_ex(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_host, N, T, H, Dk, Dv,
                             out, odt, fin, ck if nck > 0 else None, ckpt_stride, decay,
                             None if sp is None else sp.to(dev), sp, norm_gamma, norm_eps, stream)
    return out, fin, ck


def decode_step(q, k, v, log_alpha, beta, state, out_dtype=torch.bfloat16, stream=None):
    """Run kda_decode_step in place on ``state``; returns the output tensor."""
    N, H, Dk = q.shape
    Dv = v.shape[2]
    out = torch.empty(N, H, Dv, device=q.device, dtype=out_dtype)
    kda_decode_step(q, k, v, log_alpha, beta, state, out,
                    KDA_OUT_F32 if out_dtype == torch.float32 else KDA_OUT_BF16, N, H, Dk, Dv, stream)
    return out
