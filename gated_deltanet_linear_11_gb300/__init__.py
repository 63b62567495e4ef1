"""GB300-native (sm_103a) Gated DeltaNet layer hot path.

Thin Python binding over the C ABI of ``libgdn.so`` (declared in ``include/gdn.h``).
PyTorch supplies device memory and the current CUDA stream; every step of the layer runs
in this package's CUDA kernels.  The functions keep the C entry points' names:

* :func:`gdn_conv1d_fwd`       -- prefill conv1d + SiLU over packed sequences
* :func:`gdn_conv1d_update`    -- decode conv step on a pool of conv states
* :func:`gdn_chunk_prefill`    -- chunked gated delta rule over packed sequences
* :func:`gdn_recurrent_decode` -- one-token gated delta rule step on a state pool
* :func:`gdn_fused_decode`     -- conv update + gates from raw logits + recurrent step,
  one call

plus :func:`gdn_layer_prefill` / :func:`gdn_layer_decode`, which chain the conv and the
scan over the packed q||k||v channels (q, k, v are strided views of the conv output;
nothing is copied).

There is no CPU fallback: without the built library every call raises.

Two environment variables serve debugging and callers' failure tests, read at each call:

* ``GDN_DEBUG=1`` adds ``GDN_CHECK_INPUTS`` to every call that takes flags. Before
  launching anything (it waits for the stream), the library copies the gate inputs to the
  host and fails with ``GDN_ERR_NONFINITE`` (11) on a NaN or an infinity. It also fails
  with ``GDN_ERR_SEQLENS`` (5) if a prefill's device ``cu_seqlens`` differs from its host
  copy.
* ``GDN_FORCE_ERROR="gdn_chunk_prefill=7,gdn_fused_decode=10"`` makes each named entry
  raise :class:`GdnError` with that status code at once, without calling the library:
  host-side fault injection for code that handles this package's errors.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _lib
from ._lib import (GDN_CHECK_INPUTS, GDN_LAYER_FUSED_VCONV, GDN_PREFILL_SIMT,  # noqa: F401
                   GDN_PREFILL_TILES2, GDN_PREFILL_TILES3, GDN_QK_L2NORM, GdnError)

__all__ = ["gdn_conv1d_fwd", "gdn_conv1d_update", "gdn_chunk_prefill",
           "gdn_chunk_prefill_noalloc", "gdn_chunk_prefill_cp",
           "gdn_chunk_prefill_cp_workspace_size", "gdn_chunk_prefill_cp_range_hint",
           "gdn_recurrent_decode", "gdn_fused_decode", "gdn_chunk_prefill_workspace_size",
           "gdn_layer_prefill", "gdn_layer_decode", "GdnError", "load"]

_DT = {torch.bfloat16: _lib.GDN_BF16, torch.float32: _lib.GDN_F32}


def load():
    """Load the CUDA library (raises when it is not built)."""
    return _lib.load()


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _desc(t):
    if t.dtype not in _DT:
        raise TypeError("activations must be bf16 or fp32, got %s" % t.dtype)
    if t.dim() not in (3, 4):
        raise ValueError("activations must be [T,H,D] or [1,T,H,D]")
    d = _lib.GdnTensor()
    d.ptr = t.data_ptr()
    d.ndim = t.dim()
    d.dtype = _DT[t.dtype]
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _debug_flags():
    """GDN_CHECK_INPUTS when GDN_DEBUG is set (to anything but "" or "0")."""
    return GDN_CHECK_INPUTS if os.environ.get("GDN_DEBUG", "") not in ("", "0") else 0


def _forced(name):
    """Raise the status GDN_FORCE_ERROR assigns to entry `name`, if any."""
    spec = os.environ.get("GDN_FORCE_ERROR", "")
    for item in filter(None, (x.strip() for x in spec.split(","))):
        entry, sep, code = item.partition("=")
        if not sep or not code.strip().lstrip("-").isdigit():
            raise ValueError("GDN_FORCE_ERROR items are name=code, got %r" % item)
        if entry.strip() == name:
            raise GdnError(int(code), name + " (GDN_FORCE_ERROR)")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensor must live on a CUDA device")


def _seqlens(cu_seqlens, cu_seqlens_host):
    """Device and host int32 copies of the offsets (a host copy avoids a sync)."""
    if cu_seqlens_host is None:
        cu_seqlens_host = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
    else:
        cu_seqlens_host = cu_seqlens_host.to(torch.int32).contiguous()
    if not cu_seqlens.is_cuda:
        cu_seqlens = cu_seqlens.to(torch.int32).cuda()
    cu_seqlens = cu_seqlens.to(torch.int32).contiguous()
    return cu_seqlens, cu_seqlens_host


def gdn_conv1d_fwd(x, w, bias, cu_seqlens, conv_state_in=None, conv_state_out=None,
                   y=None, cu_seqlens_host=None):
    """y = silu(conv1d(cat(conv_state, x_seq))) per sequence; returns (y, conv_state_out).

    x [T, C] bf16; w [C, 4] (or [C, 1, 4]) bf16; bias [C] or None; cu_seqlens [N+1] int32;
    conv_state_in [N, 3, C] or None (zeros); conv_state_out may be conv_state_in.
    """
    _forced("gdn_conv1d_fwd")
    lib = _lib.load()
    _need_cuda(x, w, bias, conv_state_in, conv_state_out, y)
    T, C = x.shape
    w = w.reshape(C, 4).contiguous()
    cu, cu_h = _seqlens(cu_seqlens, cu_seqlens_host)
    N = cu_h.numel() - 1
    if y is None:
        y = torch.empty_like(x)
    if conv_state_out is None:
        conv_state_out = torch.empty((N, 3, C), dtype=x.dtype, device=x.device)
    rc = lib.gdn_conv1d_fwd(_vp(x), T, C, _vp(w), _vp(bias), _vp(cu),
                            ctypes.c_void_p(cu_h.data_ptr()), N, _vp(conv_state_in),
                            _vp(conv_state_out), _vp(y), _stream())
    _lib.check(rc, "gdn_conv1d_fwd")
    return y, conv_state_out


def gdn_conv1d_update(x, w, bias, conv_state, state_idx=None, y=None, status=None):
    """One-token conv step; conv_state [P, 3, C] is shifted in place.  Returns y [N, C]."""
    _forced("gdn_conv1d_update")
    lib = _lib.load()
    _need_cuda(x, w, bias, conv_state, state_idx, y, status)
    N, C = x.shape
    w = w.reshape(C, 4).contiguous()
    if y is None:
        y = torch.empty_like(x)
    rc = lib.gdn_conv1d_update(_vp(x), N, C, _vp(w), _vp(bias), _vp(conv_state),
                               conv_state.shape[0], _vp(state_idx), _vp(y), _vp(status),
                               _stream())
    _lib.check(rc, "gdn_conv1d_update")
    return y


def gdn_chunk_prefill_workspace_size(N, T, Hk, Hv, dk, dv, chunk=64, simt=False):
    lib = _lib.load()
    return int(lib.gdn_chunk_prefill_workspace_size(N, T, Hk, Hv, dk, dv, chunk,
                                                    GDN_PREFILL_SIMT if simt else 0))


def _tile_flag(tiles):
    if tiles is None:
        return 0
    if tiles not in (2, 3):
        raise ValueError("tiles must be 2, 3 or None")
    return GDN_PREFILL_TILES2 if tiles == 2 else GDN_PREFILL_TILES3


def gdn_chunk_prefill(q, k, v, g, beta, cu_seqlens, chunk=64, scale=1.0, l2norm=False,
                      initial_state=None, output_final_state=True, o=None,
                      final_state=None, simt=False, cu_seqlens_host=None, workspace=None,
                      status=None, tiles=None):
    """Chunked gated delta rule over packed sequences.  Returns (o, final_state).

    q, k [T, Hk, dk]; v [T, Hv, dv] (token-major views; head-first is rejected);
    g, beta [T, Hv] fp32; cu_seqlens [N+1]; initial_state [N, Hv, dk, dv] fp32 or None.
    tiles: None (chosen from N and the SM count), 2 or 3 dv tiles per head in the
    tensor-core state pass; the bits are the same under every choice.
    """
    _forced("gdn_chunk_prefill")
    lib = _lib.load()
    _need_cuda(q, k, v, g, beta, initial_state, o, final_state, workspace, status)
    cu, cu_h = _seqlens(cu_seqlens, cu_seqlens_host)
    N = cu_h.numel() - 1
    T, Hk, dk = q.shape[-3:]
    Hv, dv = v.shape[-2:]
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=q.device)
    flags = ((GDN_QK_L2NORM if l2norm else 0) | (GDN_PREFILL_SIMT if simt else 0) |
             _tile_flag(tiles) | _debug_flags())
    ws_bytes = int(lib.gdn_chunk_prefill_workspace_size(N, T, Hk, Hv, dk, dv, chunk, flags))
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    g = g.contiguous()
    beta = beta.contiguous()
    dq, dk_, dv_, do = _desc(q), _desc(k), _desc(v), _desc(o)
    rc = lib.gdn_chunk_prefill(
        ctypes.byref(dq), ctypes.byref(dk_), ctypes.byref(dv_), _vp(g), _vp(beta), _vp(cu),
        ctypes.c_void_p(cu_h.data_ptr()), N, chunk, float(scale), flags,
        _vp(initial_state), ctypes.byref(do), _vp(final_state), _vp(workspace),
        ws_bytes, _vp(status), _stream())
    _lib.check(rc, "gdn_chunk_prefill")
    return o, final_state


def gdn_chunk_prefill_cp_workspace_size(cu_seqlens_host, T, Hk, Hv, dk, dv, range_chunks,
                                        chunk=64):
    """Workspace bytes of gdn_chunk_prefill_cp (0 for a shape it does not take)."""
    lib = _lib.load()
    cu_h = cu_seqlens_host.to(torch.int32).contiguous()
    return int(lib.gdn_chunk_prefill_cp_workspace_size(
        ctypes.c_void_p(cu_h.data_ptr()), cu_h.numel() - 1, T, Hk, Hv, dk, dv, chunk,
        range_chunks))


def gdn_chunk_prefill_cp_range_hint(seq_len, Hv, sm_count=None):
    """range_chunks for one sequence of ``seq_len`` tokens over ``Hv`` v-heads alone on
    the current device (or on one with ``sm_count`` SMs), or 0 when the plain scan is
    expected to be as fast (C entries gdn_chunk_prefill_cp_range_hint and
    gdn_chunk_prefill_cp_range_hint_for; depends on the sequence's own length only)."""
    lib = _lib.load()
    if sm_count is None:
        return int(lib.gdn_chunk_prefill_cp_range_hint(int(seq_len), int(Hv)))
    return int(lib.gdn_chunk_prefill_cp_range_hint_for(int(seq_len), int(Hv), int(sm_count)))


def gdn_chunk_prefill_cp(q, k, v, g, beta, cu_seqlens, range_chunks, chunk=64, scale=1.0,
                         l2norm=False, initial_state=None, output_final_state=True, o=None,
                         final_state=None, cu_seqlens_host=None, workspace=None, status=None,
                         tiles=None):
    """gdn_chunk_prefill with every sequence split into ranges of ``range_chunks`` chunks
    run side by side (the context-parallel scan; tensor-core path only).  Returns
    (o, final_state)."""
    _forced("gdn_chunk_prefill_cp")
    lib = _lib.load()
    _need_cuda(q, k, v, g, beta, initial_state, o, final_state, workspace, status)
    cu, cu_h = _seqlens(cu_seqlens, cu_seqlens_host)
    N = cu_h.numel() - 1
    T, Hk, dk = q.shape[-3:]
    Hv, dv = v.shape[-2:]
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=q.device)
    flags = (GDN_QK_L2NORM if l2norm else 0) | _tile_flag(tiles) | _debug_flags()
    ws_bytes = int(lib.gdn_chunk_prefill_cp_workspace_size(
        ctypes.c_void_p(cu_h.data_ptr()), N, T, Hk, Hv, dk, dv, chunk, range_chunks))
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    dq, dk_, dv_, do = _desc(q), _desc(k), _desc(v), _desc(o)
    rc = lib.gdn_chunk_prefill_cp(
        ctypes.byref(dq), ctypes.byref(dk_), ctypes.byref(dv_), _vp(g.contiguous()),
        _vp(beta.contiguous()), _vp(cu), ctypes.c_void_p(cu_h.data_ptr()), N, chunk,
        float(scale), flags, int(range_chunks), _vp(initial_state), ctypes.byref(do),
        _vp(final_state), _vp(workspace), ws_bytes, _vp(status), _stream())
    _lib.check(rc, "gdn_chunk_prefill_cp")
    return o, final_state


def gdn_chunk_prefill_noalloc(q, k, v, g, beta, cu_seqlens, chunk=64, scale=1.0,
                              l2norm=False, initial_state=None, output_final_state=True,
                              o=None, final_state=None, simt=False, cu_seqlens_host=None,
                              status=None):
    """gdn_chunk_prefill for callers that cannot allocate device scratch: the library
    uses its own fixed 128 MiB device array instead of a workspace.  Output tensors are
    still the caller's; pass ``o``/``final_state`` (and the device ``cu_seqlens``, ``g`` and
    ``beta`` as contiguous tensors) to avoid any allocation on the Python side as well.
    Returns (o, final_state)."""
    _forced("gdn_chunk_prefill_noalloc")
    lib = _lib.load()
    _need_cuda(q, k, v, g, beta, initial_state, o, final_state, status)
    cu, cu_h = _seqlens(cu_seqlens, cu_seqlens_host)
    N = cu_h.numel() - 1
    T, Hk, dk = q.shape[-3:]
    Hv, dv = v.shape[-2:]
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=q.device)
    flags = ((GDN_QK_L2NORM if l2norm else 0) | (GDN_PREFILL_SIMT if simt else 0) |
             _debug_flags())
    dq, dk_, dv_, do = _desc(q), _desc(k), _desc(v), _desc(o)
    rc = lib.gdn_chunk_prefill_noalloc(
        ctypes.byref(dq), ctypes.byref(dk_), ctypes.byref(dv_), _vp(g.contiguous()),
        _vp(beta.contiguous()), _vp(cu), ctypes.c_void_p(cu_h.data_ptr()), N, chunk,
        float(scale), flags, _vp(initial_state), ctypes.byref(do), _vp(final_state),
        _vp(status), _stream())
    _lib.check(rc, "gdn_chunk_prefill_noalloc")
    return o, final_state


def gdn_recurrent_decode(q, k, v, g, beta, state, state_idx=None, scale=1.0, l2norm=False,
                         o=None, status=None):
    """One token per sequence; state [P, Hv, dk, dv] fp32 updated in place.  Returns o."""
    _forced("gdn_recurrent_decode")
    lib = _lib.load()
    _need_cuda(q, k, v, g, beta, state, state_idx, o, status)
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    dq, dk_, dv_, do = _desc(q), _desc(k), _desc(v), _desc(o)
    rc = lib.gdn_recurrent_decode(
        ctypes.byref(dq), ctypes.byref(dk_), ctypes.byref(dv_), _vp(g.contiguous()),
        _vp(beta.contiguous()), _vp(state), state.shape[0], _vp(state_idx), float(scale),
        (GDN_QK_L2NORM if l2norm else 0) | _debug_flags(), ctypes.byref(do), _vp(status),
        _stream())
    _lib.check(rc, "gdn_recurrent_decode")
    return o


def gdn_fused_decode(x_qkv, conv_w, conv_bias, a_raw, b_raw, conv_state, state, Hk, Hv, dk,
                     dv, state_idx=None, scale=1.0, l2norm=True, o=None, status=None):
    """The whole one-token decode step in one call: conv update (conv_state shifted in
    place), q/k/v split, optional q/k L2 norm, beta = sigmoid(b_raw), g = -softplus(a_raw),
    recurrent step (state updated in place).  x_qkv [N, C] bf16; a_raw, b_raw [N, Hv] fp32.
    Returns o [N, Hv, dv] bf16."""
    _forced("gdn_fused_decode")
    lib = _lib.load()
    _need_cuda(x_qkv, conv_w, conv_bias, a_raw, b_raw, conv_state, state, state_idx, o, status)
    N = x_qkv.shape[0]
    if o is None:
        o = torch.empty((N, Hv, dv), dtype=torch.bfloat16, device=x_qkv.device)
    for t in (x_qkv, conv_w, conv_state, state, o):
        if not t.is_contiguous():
            raise ValueError("gdn_fused_decode takes contiguous tensors")
    rc = lib.gdn_fused_decode(
        _vp(x_qkv), N, Hk, Hv, dk, dv, _vp(conv_w), _vp(conv_bias), _vp(conv_state),
        _vp(a_raw.contiguous()), _vp(b_raw.contiguous()), _vp(state), state.shape[0],
        _vp(state_idx), float(scale), (GDN_QK_L2NORM if l2norm else 0) | _debug_flags(),
        _vp(o), _vp(status), _stream())
    _lib.check(rc, "gdn_fused_decode")
    return o


def split_qkv(y, Hk, Hv, dk, dv):
    """Strided [T, H, D] views of the packed q||k||v conv output (no copy)."""
    T = y.shape[0]
    q = y[:, : Hk * dk].unflatten(1, (Hk, dk))
    k = y[:, Hk * dk: 2 * Hk * dk].unflatten(1, (Hk, dk))
    v = y[:, 2 * Hk * dk: 2 * Hk * dk + Hv * dv].unflatten(1, (Hv, dv))
    assert q.shape[0] == T
    return q, k, v


def gdn_layer_prefill(x_qkv, conv_w, conv_bias, g, beta, cu_seqlens, Hk, Hv, dk, dv,
                      conv_state_in=None, conv_state_out=None, initial_state=None,
                      final_state=None, scale=1.0, chunk=64, l2norm=True, y=None, o=None,
                      cu_seqlens_host=None, workspace=None, status=None, side_stream=None,
                      fused_vconv=False, tiles=None):
    """conv1d + SiLU over packed q||k||v, then the chunked scan with in-kernel q/k L2 norm,
    in one call of the C entry gdn_layer_prefill.  With ``side_stream`` (a second
    torch.cuda.Stream) the v channels' conv runs on it, overlapping the chunk preparation;
    without one everything runs on the current stream.  ``fused_vconv`` instead convolves
    the v channels inside the scan's state pass (GDN_LAYER_FUSED_VCONV).  Every path gives
    the bits of the two calls in sequence (y included, when passed).

    Returns (o [T, Hv, dv], final_state [N, Hv, dk, dv], conv_state_out [N, 3, C]).
    """
    _forced("gdn_layer_prefill")
    if chunk != 64:
        raise ValueError("gdn_layer_prefill runs the 64-token chunk scan")
    lib = _lib.load()
    _need_cuda(x_qkv, conv_w, conv_bias, g, beta, conv_state_in, conv_state_out,
               initial_state, final_state, y, o, workspace, status)
    T, C = x_qkv.shape
    if C != 2 * Hk * dk + Hv * dv:
        raise ValueError("x_qkv has %d channels, not 2*Hk*dk + Hv*dv" % C)
    conv_w = conv_w.reshape(C, 4).contiguous()
    cu, cu_h = _seqlens(cu_seqlens, cu_seqlens_host)
    N = cu_h.numel() - 1
    dev = x_qkv.device
    if y is None:
        y = torch.empty_like(x_qkv)
    if conv_state_out is None:
        conv_state_out = torch.empty((N, 3, C), dtype=x_qkv.dtype, device=dev)
    if o is None:
        o = torch.empty((T, Hv, dv), dtype=torch.bfloat16, device=dev)
    if final_state is None:
        final_state = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=dev)
    flags = (GDN_QK_L2NORM if l2norm else 0) | (GDN_LAYER_FUSED_VCONV if fused_vconv else 0)
    flags |= _tile_flag(tiles) | _debug_flags()
    ws_bytes = int(lib.gdn_chunk_prefill_workspace_size(N, T, Hk, Hv, dk, dv, 64, flags))
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    for t in (x_qkv, y, o):
        if not t.is_contiguous():
            raise ValueError("gdn_layer_prefill takes contiguous x_qkv, y and o")
    rc = lib.gdn_layer_prefill(
        _vp(x_qkv), T, Hk, Hv, dk, dv, _vp(conv_w), _vp(conv_bias), _vp(cu),
        ctypes.c_void_p(cu_h.data_ptr()), N, _vp(conv_state_in), _vp(conv_state_out), _vp(y),
        _vp(g.contiguous()), _vp(beta.contiguous()), float(scale), flags, _vp(initial_state),
        _vp(o), _vp(final_state), _vp(workspace), ws_bytes, _vp(status),
        None if side_stream is None else ctypes.c_void_p(side_stream.cuda_stream), _stream())
    _lib.check(rc, "gdn_layer_prefill")
    return o, final_state, conv_state_out


def gdn_layer_decode(x_qkv, conv_w, conv_bias, g, beta, conv_state, state, Hk, Hv, dk, dv,
                     state_idx=None, scale=1.0, l2norm=True, y=None, o=None, status=None):
    """One-token layer step: conv update, then the recurrent step (states in place)."""
    y = gdn_conv1d_update(x_qkv, conv_w, conv_bias, conv_state, state_idx, y, status)
    q, k, v = split_qkv(y, Hk, Hv, dk, dv)
    return gdn_recurrent_decode(q, k, v, g, beta, state, state_idx, scale, l2norm, o,
                                status)


def gdn_selftest_bounded_wait(status=None):
    """The failure path of the kernels' bounded waits, without a GPU fault: one CTA waits
    on an mbarrier phase that nothing completes, gives up after about 2 s and writes
    GDN_ERR_TIMEOUT to the status word.  Returns the status tensor (int32 [1])."""
    lib = _lib.load()
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _need_cuda(status)
    _lib.check(lib.gdn_selftest_bounded_wait(_vp(status), _stream()),
               "gdn_selftest_bounded_wait")
    return status
