"""Torch-facing binding of libkda.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks shapes and dtypes, derives the kda_params_t record from the tensors,
passes raw device pointers and the current CUDA stream, and turns a non-OK
status into an exception (the argument checks mirror the chunked DeltaNet
launcher of "From Attention to Learned Memory", sec. 4).
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import KdaError, KdaParams

_QKV_DTYPES = {torch.float32: _lib.KDA_DTYPE_F32, torch.bfloat16: _lib.KDA_DTYPE_BF16}
_INDEX_DTYPES = (torch.int32, getattr(torch, "uint32", torch.int32))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _row_stride(x: torch.Tensor, name: str) -> int:
    # [T, H, D] with the last two dims dense; the token stride may be wider
    # (a column block of a packed buffer)
    if x.dim() != 3 or x.stride(2) != 1 or x.stride(1) != x.shape[2]:
        raise ValueError(f"{name} must be [T, H, D] with dense (H, D) rows")
    return int(x.stride(0)) if x.shape[0] > 1 else int(x.shape[1] * x.shape[2])


def _on(dev, fn, *args):
    """Calls a library entry point with `dev` current: the library finds its per-device
    error word and scratch on the current device, and the stream passed belongs to `dev`."""
    with torch.cuda.device(dev):
        return fn(*args)


def _check_cuda(*ts):
    dev = None
    for t in ts:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on the same device")
    return dev


def make_params(*, num_seqs, num_k_heads, num_v_heads, d, num_slots, total_tokens=0, chunk=64,
                qkv_dtype=torch.bfloat16, state_dtype=torch.float32, per_channel=True,
                scale=0.0, l2norm=True, checked=False, cuda_cores=False, compact=False,
                delta_rule=True, q_row_stride=0,
                k_row_stride=0, v_row_stride=0) -> KdaParams:
    return KdaParams(num_seqs=num_seqs, num_k_heads=num_k_heads, num_v_heads=num_v_heads, d_k=d,
                     d_v=d, num_slots=num_slots, total_tokens=total_tokens, chunk=chunk,
                     qkv_dtype=_QKV_DTYPES[qkv_dtype], state_dtype=_QKV_DTYPES[state_dtype],
                     decay_kind=(_lib.KDA_DECAY_PER_CHANNEL if per_channel
                                 else _lib.KDA_DECAY_SCALAR),
                     scale=float(scale), l2norm_qk=int(bool(l2norm)),
                     flags=((_lib.KDA_FLAG_CHECKED if checked else 0)
                            | (_lib.KDA_FLAG_CUDA_CORES if cuda_cores else 0)
                            | (_lib.KDA_FLAG_COMPACT if compact else 0)
                            | (0 if delta_rule else _lib.KDA_FLAG_NO_DELTA)),
                     q_row_stride=q_row_stride,
                     k_row_stride=k_row_stride, v_row_stride=v_row_stride)


def workspace_size(params: KdaParams) -> int:
    n = ctypes.c_size_t(0)
    st = _lib.load().kda_prefill_workspace_size(ctypes.byref(params), ctypes.byref(n))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_prefill_workspace_size")
    return int(n.value)


def uses_tensor_cores(params: KdaParams) -> bool:
    """Whether kda_prefill_fwd runs these parameters on the tensor-core path."""
    r = _lib.load().kda_prefill_uses_tensor_cores(ctypes.byref(params))
    if r < 0:
        raise KdaError(_lib.KDA_ERR_INVALID_ARG, "kda_prefill_uses_tensor_cores")
    return bool(r)


def _prefill_params(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool, chunk,
                    scale, l2norm, checked, cuda_cores=False, compact=False, delta_rule=True):
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3:
        raise ValueError("q, k must be [T, HK, D] and v [T, HV, D]")
    T, HK, D = q.shape
    HV = v.shape[1]
    if v.shape[0] != T or v.shape[2] != D:
        raise ValueError("v must be [T, HV, D] with the same T and D as q")
    if q.dtype not in _QKV_DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype: float32 or bfloat16")
    if beta.dtype != torch.float32 or tuple(beta.shape) != (T, HV) or not beta.is_contiguous():
        raise ValueError("beta must be contiguous float32 [T, HV]")
    if log_decay.dtype != torch.float32 or not log_decay.is_contiguous():
        raise ValueError("log_decay must be contiguous float32")
    if tuple(log_decay.shape) == (T, HV):
        per_channel = False
    elif tuple(log_decay.shape) == (T, HV, D):
        per_channel = True
    else:
        raise ValueError("log_decay must be [T, HV] (scalar) or [T, HV, D] (per channel)")
    if input_row_offsets.dtype not in _INDEX_DTYPES or slot_idx.dtype not in _INDEX_DTYPES:
        raise ValueError("input_row_offsets and slot_idx must be int32/uint32")
    if not input_row_offsets.is_contiguous() or not slot_idx.is_contiguous():
        raise ValueError("input_row_offsets and slot_idx must be contiguous")
    B = input_row_offsets.numel() - 1
    if B < 0 or slot_idx.numel() != B:
        raise ValueError("input_row_offsets must have B+1 entries and slot_idx B")
    if (state_pool.dim() != 4 or state_pool.shape[1] != HV or state_pool.shape[2] != D
            or state_pool.shape[3] != D or state_pool.dtype not in _QKV_DTYPES
            or not state_pool.is_contiguous()):
        raise ValueError("state_pool must be contiguous [num_slots, HV, D, D] float32/bfloat16")
    return make_params(num_seqs=B, num_k_heads=HK, num_v_heads=HV, d=D,
                       num_slots=state_pool.shape[0], total_tokens=T, chunk=chunk,
                       qkv_dtype=q.dtype, state_dtype=state_pool.dtype, per_channel=per_channel,
                       scale=scale, l2norm=l2norm, checked=checked, cuda_cores=cuda_cores,
                       compact=compact, delta_rule=delta_rule, q_row_stride=_row_stride(q, "q"),
                       k_row_stride=_row_stride(k, "k"),
                       v_row_stride=_row_stride(v, "v"))


def prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
            log_decay: torch.Tensor, input_row_offsets: torch.Tensor, slot_idx: torch.Tensor,
            state_pool: torch.Tensor, *, chunk: int = 64, scale: float = 0.0,
            l2norm: bool = True, checked: bool = False, cuda_cores: bool = False,
            compact: bool = False, delta_rule: bool = True, out: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Chunkwise gated-delta-rule prefill (kda_prefill_fwd).  Returns o [T, HV, D] fp32.

    The pool slots named by slot_idx are updated in place with each sequence's final state.
    `cuda_cores=True` asks for the fp32 CUDA-core path where the tensor-core path applies;
    `compact=True` runs the tensor-core path as a single kernel with a small workspace;
    `delta_rule=False` selects the additive write (KDA_FLAG_NO_DELTA: gated linear attention).
    """
    dev = _check_cuda(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool)
    p = _prefill_params(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool, chunk,
                        scale, l2norm, checked, cuda_cores, compact, delta_rule)
    T, HV, D = v.shape
    if out is None:
        out = torch.empty((T, HV, D), dtype=torch.float32, device=dev)
    elif out.dtype != torch.float32 or tuple(out.shape) != (T, HV, D) or not out.is_contiguous():
        raise ValueError("out must be contiguous float32 [T, HV, D]")
    need = workspace_size(p)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    st = _on(dev, _lib.load().kda_prefill_fwd, 
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_decay),
        _ptr(input_row_offsets), _ptr(slot_idx), _ptr(state_pool), _ptr(out), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_prefill_fwd")
    return out


def no_alloc_form(params: KdaParams) -> str:
    """Which form kda_prefill_fwd_no_alloc runs for these parameters: "two_kernel" or
    "compact" (tensor cores), "cuda_cores", or "rejected" (invalid or too large for the
    library's scratch)."""
    r = _lib.load().kda_prefill_no_alloc_form(ctypes.byref(params))
    return {0: "two_kernel", 1: "compact", 2: "cuda_cores"}.get(r, "rejected")


def prefill_no_alloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                     log_decay: torch.Tensor, input_row_offsets: torch.Tensor,
                     slot_idx: torch.Tensor, state_pool: torch.Tensor, *, chunk: int = 64,
                     scale: float = 0.0, l2norm: bool = True, checked: bool = False,
                     cuda_cores: bool = False, delta_rule: bool = True, out: torch.Tensor,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """kda_prefill_fwd_no_alloc: the prefill with the library's built-in scratch array.

    For callers that must not allocate device memory: `out` (fp32 [T, HV, D]) is
    required and nothing is allocated here or in the library.  Problems needing more
    than KDA_NO_ALLOC_SCRATCH_BYTES of scratch raise KdaError(KDA_ERR_WORKSPACE); when the
    tensor-core path's chunk records do not fit, the single-kernel form runs instead
    (`no_alloc_form` tells which).
    Calls that overlap on the GPU share the scratch and race; keep them on one stream.
    """
    dev = _check_cuda(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool, out)
    p = _prefill_params(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool, chunk,
                        scale, l2norm, checked, cuda_cores, delta_rule=delta_rule)
    T, HV, D = v.shape
    if out.dtype != torch.float32 or tuple(out.shape) != (T, HV, D) or not out.is_contiguous():
        raise ValueError("out must be contiguous float32 [T, HV, D]")
    st = _on(dev, _lib.load().kda_prefill_fwd_no_alloc, 
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_decay),
        _ptr(input_row_offsets), _ptr(slot_idx), _ptr(state_pool), _ptr(out),
        _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_prefill_fwd_no_alloc")
    return out



def prefill_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                log_decay: torch.Tensor, input_row_offsets: torch.Tensor, slot_idx: torch.Tensor,
                state_pool: torch.Tensor, d_o: torch.Tensor, d_state: Optional[torch.Tensor] = None,
                *, chunk: int = 64, scale: float = 0.0, l2norm: bool = True,
                delta_rule: bool = True, checked: bool = False, compact: bool = False,
                d_state0: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None):
    """Backward of `prefill` (kda_prefill_bwd).  `state_pool` holds the INITIAL states (the
    pool before the forward call) and is only read; `d_o` [T, HV, D] and `d_state` (pool-shaped
    fp32, or None for zero) are the loss's gradients w.r.t. o and the final states.
    `compact` (KDA_FLAG_COMPACT; bf16 q/k/v, d = 128, chunk 64) bounds the workspace: windows of
    chunk positions with a checkpointed state per window, at the cost of rerunning the forward
    recurrence and one stream synchronisation.
    Returns (dq, dk [T, HK, D], dv [T, HV, D], dbeta [T, HV], dlog_decay (shape of log_decay),
    d_state0 (pool-shaped fp32: the touched slots' gradients, zero elsewhere unless given))."""
    dev = _check_cuda(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool, d_o)
    p = _prefill_params(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool, chunk,
                        scale, l2norm, checked, compact=compact, delta_rule=delta_rule)
    T, HK, D = q.shape
    HV = v.shape[1]
    if d_o.dtype != torch.float32 or tuple(d_o.shape) != (T, HV, D) or not d_o.is_contiguous():
        raise ValueError("d_o must be contiguous float32 [T, HV, D]")
    pool_shape = tuple(state_pool.shape)
    for name, t in (("d_state", d_state), ("d_state0", d_state0)):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != pool_shape
                              or not t.is_contiguous()):
            raise ValueError(f"{name} must be contiguous float32 shaped like state_pool")
    if d_state is not None:
        _check_cuda(d_state)
    if d_state0 is None:
        d_state0 = torch.zeros(pool_shape, dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dq = torch.empty((T, HK, D), **f32)
    dk = torch.empty((T, HK, D), **f32)
    dv = torch.empty((T, HV, D), **f32)
    dbeta = torch.empty((T, HV), **f32)
    dlog_decay = torch.empty(tuple(log_decay.shape), **f32)
    n = ctypes.c_size_t(0)
    st = _lib.load().kda_prefill_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_prefill_bwd_workspace_size")
    workspace = _workspace(int(n.value), workspace, dev)
    st = _on(dev, _lib.load().kda_prefill_bwd, 
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_decay),
        _ptr(input_row_offsets), _ptr(slot_idx), _ptr(state_pool), _ptr(d_o), _ptr(d_state),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dlog_decay), _ptr(d_state0),
        _ptr(workspace), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
        _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_prefill_bwd")
    return dq, dk, dv, dbeta, dlog_decay, d_state0


def conv_gates(x: torch.Tensor, conv_weight: torch.Tensor, a: torch.Tensor, b: torch.Tensor, *,
               num_k_heads: int, num_v_heads: int, d: int, conv_bias: Optional[torch.Tensor] = None,
               A_log: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
               input_row_offsets: Optional[torch.Tensor] = None,
               slot_idx: Optional[torch.Tensor] = None, conv_state: Optional[torch.Tensor] = None,
               num_seqs: Optional[int] = None, stream: Optional[torch.cuda.Stream] = None):
    """The front end before the recurrence (kda_conv_gates_fwd): causal depthwise convolution
    + SiLU over the packed [Q | K | V] projection x [T, conv_dim], and the gates.  `a` is
    [T, HV] (scalar decay) or [T, HV, d] (per channel), `b` [T, HV].  Without
    `input_row_offsets` every row is its own sequence (the decode form).  Returns
    (y [T, conv_dim] in x's dtype, log_decay shaped like a, beta [T, HV]); `conv_state`
    [num_slots, conv_dim, width - 1] (x's dtype) is updated in place."""
    dev = _check_cuda(x, conv_weight, a, b)
    if x.dim() != 2 or x.dtype not in _QKV_DTYPES or not x.is_contiguous():
        raise ValueError("x must be contiguous [T, conv_dim] float32/bfloat16")
    T, CD = x.shape
    if CD != (2 * num_k_heads + num_v_heads) * d:
        raise ValueError("x's width must be 2 * HK * d + HV * d")
    if conv_weight.dtype != torch.float32 or conv_weight.dim() != 2 or conv_weight.shape[0] != CD \
            or not conv_weight.is_contiguous():
        raise ValueError("conv_weight must be contiguous float32 [conv_dim, width]")
    width = conv_weight.shape[1]
    if tuple(a.shape) == (T, num_v_heads):
        per_channel = False
    elif tuple(a.shape) == (T, num_v_heads, d):
        per_channel = True
    else:
        raise ValueError("a must be [T, HV] or [T, HV, d]")
    for name, t in (("a", a), ("b", b), ("conv_bias", conv_bias), ("A_log", A_log),
                    ("dt_bias", dt_bias)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be contiguous float32")
    if tuple(b.shape) != (T, num_v_heads):
        raise ValueError("b must be [T, HV]")
    if input_row_offsets is None:
        B = T
    else:
        if input_row_offsets.dtype not in _INDEX_DTYPES or not input_row_offsets.is_contiguous():
            raise ValueError("input_row_offsets must be contiguous int32/uint32")
        B = input_row_offsets.numel() - 1
    if num_seqs is not None and num_seqs != B:
        raise ValueError("num_seqs does not match input_row_offsets")
    num_slots = 1
    if conv_state is not None:
        if (conv_state.dtype != x.dtype or conv_state.dim() != 3 or conv_state.shape[1] != CD
                or conv_state.shape[2] != width - 1 or not conv_state.is_contiguous()):
            raise ValueError("conv_state must be contiguous [num_slots, conv_dim, width - 1] in x's dtype")
        if slot_idx is None or slot_idx.numel() != B or slot_idx.dtype not in _INDEX_DTYPES:
            raise ValueError("conv_state needs slot_idx [B] int32/uint32")
        num_slots = conv_state.shape[0]
    p = make_params(num_seqs=B, num_k_heads=num_k_heads, num_v_heads=num_v_heads, d=d,
                    num_slots=num_slots, total_tokens=T, qkv_dtype=x.dtype,
                    per_channel=per_channel)
    y = torch.empty_like(x)
    log_decay = torch.empty(tuple(a.shape), dtype=torch.float32, device=dev)
    beta = torch.empty((T, num_v_heads), dtype=torch.float32, device=dev)
    st = _on(dev, _lib.load().kda_conv_gates_fwd, 
        ctypes.byref(p), int(width), _ptr(x), _ptr(conv_weight), _ptr(conv_bias), _ptr(a), _ptr(b),
        _ptr(A_log), _ptr(dt_bias), _ptr(input_row_offsets), _ptr(slot_idx), _ptr(conv_state),
        _ptr(y), _ptr(log_decay), _ptr(beta), _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_conv_gates_fwd")
    return y, log_decay, beta

def decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                log_decay: torch.Tensor, slot_idx: torch.Tensor, state_pool: torch.Tensor, *,
                scale: float = 0.0, l2norm: bool = True, delta_rule: bool = True,
                out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """One recurrent decode step (kda_decode_step) for B sequences.  Returns o [B, HV, D] fp32.
    `delta_rule=False` selects the additive write (KDA_FLAG_NO_DELTA)."""
    dev = _check_cuda(q, k, v, beta, log_decay, slot_idx, state_pool)
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[0] != q.shape[0]:
        raise ValueError("q, k must be [B, HK, D] and v [B, HV, D]")
    B, HK, D = q.shape
    HV = v.shape[1]
    if q.dtype not in _QKV_DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype: float32 or bfloat16")
    if beta.dtype != torch.float32 or tuple(beta.shape) != (B, HV) or not beta.is_contiguous():
        raise ValueError("beta must be contiguous float32 [B, HV]")
    if tuple(log_decay.shape) == (B, HV):
        per_channel = False
    elif tuple(log_decay.shape) == (B, HV, D):
        per_channel = True
    else:
        raise ValueError("log_decay must be [B, HV] or [B, HV, D]")
    if log_decay.dtype != torch.float32 or not log_decay.is_contiguous():
        raise ValueError("log_decay must be contiguous float32")
    if slot_idx.dtype not in _INDEX_DTYPES or slot_idx.numel() != B or not slot_idx.is_contiguous():
        raise ValueError("slot_idx must be contiguous int32/uint32 [B]")
    if (state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (HV, D, D)
            or state_pool.dtype not in _QKV_DTYPES or not state_pool.is_contiguous()):
        raise ValueError("state_pool must be contiguous [num_slots, HV, D, D]")
    p = make_params(num_seqs=B, num_k_heads=HK, num_v_heads=HV, d=D,
                    num_slots=state_pool.shape[0], qkv_dtype=q.dtype,
                    state_dtype=state_pool.dtype, per_channel=per_channel, scale=scale,
                    l2norm=l2norm, delta_rule=delta_rule, q_row_stride=_row_stride(q, "q"),
                    k_row_stride=_row_stride(k, "k"), v_row_stride=_row_stride(v, "v"))
    if out is None:
        out = torch.empty((B, HV, D), dtype=torch.float32, device=dev)
    st = _on(dev, _lib.load().kda_decode_step, ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                     _ptr(log_decay), _ptr(slot_idx), _ptr(state_pool), _ptr(out),
                                     _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_decode_step")
    return out


def get_device_error(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronises the stream and returns (and clears) the device error code (0 = none)."""
    code = ctypes.c_int32(0)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = _on(s.device, _lib.load().kda_get_device_error, ctypes.c_void_p(s.cuda_stream),
             ctypes.byref(code))
    if st not in (_lib.KDA_OK, _lib.KDA_ERR_DEVICE):
        raise KdaError(st, "kda_get_device_error")
    return int(code.value)


def set_stage_events(events) -> None:
    """Register torch.cuda.Event objects (enable_timing=True) that later library calls
    record on their stream: events[0] before the first kernel, events[i] after kernel i
    (kda_set_stage_events).  An empty list clears the registration."""
    events = list(events)
    if len(events) > 8:
        raise ValueError("at most 8 stage events")
    for e in events:
        e.record()                      # torch creates CUDA events lazily; make them exist
    handles = (ctypes.c_void_p * max(len(events), 1))(*[e.cuda_event for e in events])
    st = _lib.load().kda_set_stage_events(handles if events else None, len(events))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_set_stage_events")


def ring_record_elems(params: KdaParams) -> int:
    n = _lib.load().kda_ring_record_elems(ctypes.byref(params))
    if n < 0:
        raise KdaError(_lib.KDA_ERR_INVALID_ARG, "kda_ring_record_elems")
    return n


def _window_params(q, k, v, beta, log_decay, slot_idx, state_pool, window, scale, l2norm,
                   delta_rule=True):
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[0] != q.shape[0]:
        raise ValueError("q, k must be [B*window, HK, D] and v [B*window, HV, D]")
    BW, HK, D = q.shape
    HV = v.shape[1]
    if window < 1 or BW % window != 0:
        raise ValueError("the token dimension must be B * window")
    B = BW // window
    if q.dtype not in _QKV_DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype: float32 or bfloat16")
    if beta.dtype != torch.float32 or tuple(beta.shape) != (BW, HV) or not beta.is_contiguous():
        raise ValueError("beta must be contiguous float32 [B*window, HV]")
    if tuple(log_decay.shape) == (BW, HV):
        per_channel = False
    elif tuple(log_decay.shape) == (BW, HV, D):
        per_channel = True
    else:
        raise ValueError("log_decay must be [B*window, HV] or [B*window, HV, D]")
    if log_decay.dtype != torch.float32 or not log_decay.is_contiguous():
        raise ValueError("log_decay must be contiguous float32")
    if slot_idx.dtype not in _INDEX_DTYPES or slot_idx.numel() != B or not slot_idx.is_contiguous():
        raise ValueError("slot_idx must be contiguous int32/uint32 [B]")
    if (state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (HV, D, D)
            or state_pool.dtype not in _QKV_DTYPES or not state_pool.is_contiguous()):
        raise ValueError("state_pool must be contiguous [num_slots, HV, D, D]")
    return make_params(num_seqs=B, num_k_heads=HK, num_v_heads=HV, d=D,
                       num_slots=state_pool.shape[0], qkv_dtype=q.dtype,
                       state_dtype=state_pool.dtype, per_channel=per_channel, scale=scale,
                       l2norm=l2norm, delta_rule=delta_rule, q_row_stride=_row_stride(q, "q"),
                       k_row_stride=_row_stride(k, "k"), v_row_stride=_row_stride(v, "v"))


def verify_window(q, k, v, beta, log_decay, slot_idx, state_pool, *, window: int,
                  scale: float = 0.0, l2norm: bool = True, delta_rule: bool = True, out=None,
                  ring=None, stream=None):
    """kda_verify_window: `window` draft tokens per sequence from its pool slot, pool untouched.

    Token t of sequence b is row b*window + t.  Returns (o [B*window, HV, D] fp32,
    ring [B, window, HV, R] fp32) where R = ring_record_elems.
    """
    dev = _check_cuda(q, k, v, beta, log_decay, slot_idx, state_pool)
    p = _window_params(q, k, v, beta, log_decay, slot_idx, state_pool, window, scale, l2norm,
                       delta_rule)
    BW, HV, D = v.shape
    rec = ring_record_elems(p)
    if out is None:
        out = torch.empty((BW, HV, D), dtype=torch.float32, device=dev)
    if ring is None:
        ring = torch.empty((BW // window, window, HV, rec), dtype=torch.float32, device=dev)
    elif (ring.dtype != torch.float32 or not ring.is_contiguous()
          or ring.numel() != BW * HV * rec):
        raise ValueError("ring must be contiguous float32 [B, window, HV, R]")
    st = _on(dev, _lib.load().kda_verify_window, ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                       _ptr(log_decay), _ptr(slot_idx), int(window),
                                       _ptr(state_pool), _ptr(out), _ptr(ring),
                                       _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_verify_window")
    return out, ring


def fold_accepted(ring, accepted, slot_idx, state_pool, *, window: int, num_k_heads: int = 1,
                  per_channel: bool = True, stream=None):
    """kda_fold_accepted: apply the first accepted[b] ring records of each sequence to its slot."""
    dev = _check_cuda(ring, accepted, slot_idx, state_pool)
    B = slot_idx.numel()
    HV, D = state_pool.shape[1], state_pool.shape[2]
    if accepted.dtype not in _INDEX_DTYPES or accepted.numel() != B or not accepted.is_contiguous():
        raise ValueError("accepted must be contiguous int32/uint32 [B]")
    p = make_params(num_seqs=B, num_k_heads=num_k_heads, num_v_heads=HV, d=D,
                    num_slots=state_pool.shape[0], state_dtype=state_pool.dtype,
                    per_channel=per_channel)
    rec = ring_record_elems(p)
    if ring.dtype != torch.float32 or not ring.is_contiguous() or ring.numel() != B * window * HV * rec:
        raise ValueError("ring does not match [B, window, HV, R]")
    st = _on(dev, _lib.load().kda_fold_accepted, ctypes.byref(p), _ptr(ring), int(window), _ptr(accepted),
                                       _ptr(slot_idx), _ptr(state_pool),
                                       _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_fold_accepted")
    return state_pool


# ----------------------------------------------------------------------------- Gated DeltaProduct

def _gdp_params(q, k, v, beta, log_decay, num_seqs, slot_idx, state_pool, chunk, scale, l2norm,
                checked, cuda_cores, decode):
    if q.dim() != 3 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q must be [T, HK, D], k [T, n_h, HK, D], v [T, n_h, HV, D]")
    T, HK, D = q.shape
    n_h, HV = k.shape[1], v.shape[2]
    if tuple(k.shape) != (T, n_h, HK, D) or tuple(v.shape) != (T, n_h, HV, D):
        raise ValueError("k must be [T, n_h, HK, D] and v [T, n_h, HV, D]")
    if q.dtype not in _QKV_DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype: float32 or bfloat16")
    if not (k.is_contiguous() and v.is_contiguous()):
        raise ValueError("k and v must be contiguous")
    if beta.dtype != torch.float32 or tuple(beta.shape) != (T, n_h, HV) or not beta.is_contiguous():
        raise ValueError("beta must be contiguous float32 [T, n_h, HV]")
    if log_decay.dtype != torch.float32 or not log_decay.is_contiguous():
        raise ValueError("log_decay must be contiguous float32")
    if tuple(log_decay.shape) == (T, HV):
        per_channel = False
    elif tuple(log_decay.shape) == (T, HV, D):
        per_channel = True
    else:
        raise ValueError("log_decay must be [T, HV] (scalar) or [T, HV, D] (per channel)")
    if slot_idx.dtype not in _INDEX_DTYPES or not slot_idx.is_contiguous() or slot_idx.numel() != num_seqs:
        raise ValueError("slot_idx must be contiguous int32/uint32 with one entry per sequence")
    if (state_pool.dim() != 4 or state_pool.shape[1] != HV or state_pool.shape[2] != D
            or state_pool.shape[3] != D or state_pool.dtype not in _QKV_DTYPES
            or not state_pool.is_contiguous()):
        raise ValueError("state_pool must be contiguous [num_slots, HV, D, D] float32/bfloat16")
    p = make_params(num_seqs=num_seqs, num_k_heads=HK, num_v_heads=HV, d=D,
                    num_slots=state_pool.shape[0], total_tokens=T, chunk=chunk,
                    qkv_dtype=q.dtype, state_dtype=state_pool.dtype, per_channel=per_channel,
                    scale=scale, l2norm=l2norm, checked=checked, cuda_cores=cuda_cores,
                    q_row_stride=_row_stride(q, "q"))
    n = ctypes.c_size_t(0)
    st = _lib.load().kda_gdp_workspace_size(ctypes.byref(p), n_h, int(decode), ctypes.byref(n))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_gdp_workspace_size")
    return p, n_h, int(n.value)


def _workspace(need, workspace, dev):
    if workspace is None:
        return torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace needs {need} bytes")
    return workspace


def gdp_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                log_decay: torch.Tensor, input_row_offsets: torch.Tensor, slot_idx: torch.Tensor,
                state_pool: torch.Tensor, *, chunk: int = 64, scale: float = 0.0,
                l2norm: bool = True, checked: bool = False, cuda_cores: bool = False,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Gated DeltaProduct prefill (kda_gdp_prefill_fwd): n_h = k.shape[1] transitions per
    token.  q [T, HK, D]; k [T, n_h, HK, D]; v [T, n_h, HV, D]; beta [T, n_h, HV];
    log_decay [T, HV] or [T, HV, D].  Returns o [T, HV, D] fp32; the pool slots are updated
    in place."""
    dev = _check_cuda(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool)
    if input_row_offsets.dtype not in _INDEX_DTYPES or not input_row_offsets.is_contiguous():
        raise ValueError("input_row_offsets must be contiguous int32/uint32")
    p, n_h, need = _gdp_params(q, k, v, beta, log_decay, input_row_offsets.numel() - 1, slot_idx,
                               state_pool, chunk, scale, l2norm, checked, cuda_cores, False)
    T, HV, D = q.shape[0], v.shape[2], q.shape[2]
    if out is None:
        out = torch.empty((T, HV, D), dtype=torch.float32, device=dev)
    elif out.dtype != torch.float32 or tuple(out.shape) != (T, HV, D) or not out.is_contiguous():
        raise ValueError("out must be contiguous float32 [T, HV, D]")
    workspace = _workspace(need, workspace, dev)
    st = _on(dev, _lib.load().kda_gdp_prefill_fwd, 
        ctypes.byref(p), n_h, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_decay),
        _ptr(input_row_offsets), _ptr(slot_idx), _ptr(state_pool), _ptr(out), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_gdp_prefill_fwd")
    return out


def gdp_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                    log_decay: torch.Tensor, slot_idx: torch.Tensor, state_pool: torch.Tensor, *,
                    chunk: int = 0, scale: float = 0.0, l2norm: bool = True,
                    out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """One Gated DeltaProduct decode step (kda_gdp_decode_step): one token of n_h transitions
    per sequence; arrays as gdp_prefill with T = B.  Returns o [B, HV, D] fp32."""
    dev = _check_cuda(q, k, v, beta, log_decay, slot_idx, state_pool)
    p, n_h, need = _gdp_params(q, k, v, beta, log_decay, q.shape[0], slot_idx, state_pool, chunk,
                               scale, l2norm, False, False, True)
    B, HV, D = q.shape[0], v.shape[2], q.shape[2]
    if out is None:
        out = torch.empty((B, HV, D), dtype=torch.float32, device=dev)
    elif out.dtype != torch.float32 or tuple(out.shape) != (B, HV, D) or not out.is_contiguous():
        raise ValueError("out must be contiguous float32 [B, HV, D]")
    workspace = _workspace(need, workspace, dev)
    st = _on(dev, _lib.load().kda_gdp_decode_step, 
        ctypes.byref(p), n_h, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_decay),
        _ptr(slot_idx), _ptr(state_pool), _ptr(out), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_handle(stream, dev))
    if st != _lib.KDA_OK:
        raise KdaError(st, "kda_gdp_decode_step")
    return out
