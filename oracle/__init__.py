"""fp64 CPU oracle for the Gated DeltaNet layer hot path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may use this package; the product library never does.  It shares no
code with the CUDA path.

Two independent forms of the same operator live here:

* ``gdn_oracle.c`` -- the literal token-by-token recurrence and the literal conv1d, in
  C, fp64, threaded over (sequence, v-head).  Wrapped by :func:`gated_delta_rule`,
  :func:`conv1d_varlen` and the decode helpers below.
* ``chunked.py`` -- the chunked WY/UT form of the same recurrence in numpy fp64, used
  to pin the chunk algebra against the token form.

Sources (page title, section):

* "Qwen3.5-27B GPTQ Garbage Inference -- Root Cause Analysis", "Why abliteration failed
  on Qwen3.5", item 3: the GatedDeltaNet recurrence S = exp(g) S + beta dv (x) k.
* "[Feature] Add batch invariance support to GDN_ATTN backend - #45819", Birol's comment,
  "1. Recurrent state in fp32" (state shape (batch, v_heads, k_head_dim, v_head_dim),
  fp32) and "3. The chunked delta-rule scan itself" (conv-state carry, initial_state,
  use_qk_l2norm_in_kernel, chunk multiple of 64).

Readings where the pages are silent (each one is listed with its reason in the design
notes): decay before the delta correction; o_t taken after the update; an explicit
output ``scale`` (1.0 = the literal formula); v-head h uses k-head h // (Hv // Hk);
L2-norm epsilon 1e-6 inside the square root.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .chunked import chunked_gated_delta_rule  # noqa: F401  (re-export)

L2NORM_EPS = 1e-6

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so`` (plain gcc, -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        lib.oracle_conv1d_varlen.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp,
                                             ctypes.c_int, ip, dp, dp, dp]
        lib.oracle_conv1d_varlen.restype = ctypes.c_int
        lib.oracle_gated_delta_rule.argtypes = [
            ctypes.c_int, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            dp, dp, dp, dp, dp, ctypes.c_double, ctypes.c_int, ctypes.c_double, dp, dp,
            dp, ctypes.c_int]
        lib.oracle_gated_delta_rule.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> exact upcast of the stored values
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _dp(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


# ------------------------------------------------------------------------- conv1d

def conv1d_varlen(x, w, bias, cu_seqlens, state_in=None):
    """Causal depthwise conv1d (width 4) + SiLU over packed sequences.

    x: [T, C]; w: [C, 4]; bias: [C] or None; cu_seqlens: [N+1];
    state_in: [N, 3, C] (the three conv inputs that precede each sequence) or None for
    zeros.  Returns (y [T, C], state_out [N, 3, C]) in float64.
    """
    x = _f64(x)
    w = _f64(w).reshape(-1, 4)
    bias = _f64(bias)
    cu = _i32(cu_seqlens)
    T, C = x.shape
    N = cu.shape[0] - 1
    s_in = _f64(state_in)
    if s_in is not None:
        s_in = s_in.reshape(N, 3, C)
    y = np.zeros((T, C), np.float64)
    s_out = np.zeros((N, 3, C), np.float64)
    rc = _load().oracle_conv1d_varlen(T, C, _dp(x), _dp(w), _dp(bias), N,
                                      cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                      _dp(s_in), _dp(y), _dp(s_out))
    if rc:
        raise ValueError("oracle_conv1d_varlen failed with code %d" % rc)
    return y, s_out


def conv1d_update(x, w, bias, conv_state_pool, state_idx=None):
    """One-token conv step per sequence on a pool of conv states.

    x: [N, C]; conv_state_pool: [P, 3, C]; state_idx: [N] (None = identity).
    Returns (y [N, C], new_pool [P, 3, C]).  Same definition as conv1d_varlen with one
    token per sequence.
    """
    x = _f64(x)
    N, C = x.shape
    pool = _f64(conv_state_pool).copy()
    idx = np.arange(N) if state_idx is None else _i32(state_idx).astype(np.int64)
    cu = np.arange(N + 1, dtype=np.int32)
    y, s_out = conv1d_varlen(x, w, bias, cu, pool[idx])
    pool[idx] = s_out
    return y, pool


# ---------------------------------------------------------------- gated delta rule

def gated_delta_rule(q, k, v, g, beta, cu_seqlens, scale=1.0, l2norm=False,
                     initial_state=None, nthreads=None):
    """Token-by-token gated delta rule in fp64.

    q, k: [T, Hk, dk]; v: [T, Hv, dv]; g, beta: [T, Hv]; cu_seqlens: [N+1];
    initial_state: [N, Hv, dk, dv] or None (zeros).
    Returns (o [T, Hv, dv], final_state [N, Hv, dk, dv]).
    """
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    cu = _i32(cu_seqlens)
    T, Hk, dk = q.shape
    _, Hv, dv = v.shape
    N = cu.shape[0] - 1
    if cu[-1] != T:
        raise ValueError("cu_seqlens[-1] must equal T")
    h0 = _f64(initial_state)
    if h0 is not None:
        h0 = h0.reshape(N, Hv, dk, dv)
    o = np.zeros((T, Hv, dv), np.float64)
    hT = np.zeros((N, Hv, dk, dv), np.float64)
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = _load().oracle_gated_delta_rule(
        N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), Hk, Hv, dk, dv,
        _dp(q), _dp(k), _dp(v), _dp(g.reshape(T, Hv)), _dp(beta.reshape(T, Hv)),
        float(scale), int(bool(l2norm)), L2NORM_EPS, _dp(h0), _dp(o), _dp(hT), nt)
    if rc:
        raise ValueError("oracle_gated_delta_rule failed with code %d" % rc)
    return o, hT


def recurrent_decode(q, k, v, g, beta, state_pool, state_idx=None, scale=1.0,
                     l2norm=False, nthreads=None):
    """One token per sequence on a pool of recurrent states.

    q, k: [N, Hk, dk]; v: [N, Hv, dv]; g, beta: [N, Hv]; state_pool: [P, Hv, dk, dv];
    state_idx: [N] (None = identity).  Returns (o [N, Hv, dv], new_pool).
    """
    q = _f64(q)
    N = q.shape[0]
    pool = _f64(state_pool).copy()
    idx = np.arange(N) if state_idx is None else _i32(state_idx).astype(np.int64)
    cu = np.arange(N + 1, dtype=np.int32)
    o, hT = gated_delta_rule(q, k, v, g, beta, cu, scale=scale, l2norm=l2norm,
                             initial_state=pool[idx], nthreads=nthreads)
    pool[idx] = hT
    return o, pool


def l2_normalise(x, eps=L2NORM_EPS):
    """x / sqrt(sum x^2 + eps) over the last axis, fp64."""
    x = _f64(x)
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


# ------------------------------------------------------------------- layer helpers

def round_to_bf16(a):
    """Round fp64 values to bf16 (via fp32, round-to-nearest-even) and return fp64.

    The conv output that feeds the scan is an activation in the model's compute dtype,
    bf16 ("[Feature] Add batch invariance support to GDN_ATTN backend - #45819", Birol's
    comment, part 1: conv state in compute dtype)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float64)).float().to(
        torch.bfloat16).double().numpy()


def split_qkv(y, Hk, Hv, dk, dv):
    T = y.shape[0]
    q = y[:, :Hk * dk].reshape(T, Hk, dk)
    k = y[:, Hk * dk:2 * Hk * dk].reshape(T, Hk, dk)
    v = y[:, 2 * Hk * dk:2 * Hk * dk + Hv * dv].reshape(T, Hv, dv)
    return q, k, v


def layer_prefill(x, w, bias, g, beta, cu_seqlens, Hk, Hv, dk, dv, conv_state=None,
                  initial_state=None, scale=1.0, l2norm=True, v_heads=None, nthreads=None):
    """conv1d+SiLU over packed q||k||v (bf16 activations), then the gated delta rule.

    v_heads: optional list of v-heads to evaluate (the others are skipped); the result
    arrays then hold those heads in that order.  Returns (o, final_state, conv_state_out).
    """
    y, s_out = conv1d_varlen(x, w, bias, cu_seqlens, conv_state)
    q, k, v = split_qkv(round_to_bf16(y), Hk, Hv, dk, dv)
    g = _f64(g)
    beta = _f64(beta)
    h0 = _f64(initial_state)
    if v_heads is None:
        o, hT = gated_delta_rule(q, k, v, g, beta, cu_seqlens, scale, l2norm, h0, nthreads)
        return o, hT, s_out
    G = Hv // Hk
    outs, states = [], []
    for hv in v_heads:
        hk = hv // G
        o, hT = gated_delta_rule(q[:, hk:hk + 1], k[:, hk:hk + 1], v[:, hv:hv + 1],
                                 g[:, hv:hv + 1], beta[:, hv:hv + 1], cu_seqlens, scale,
                                 l2norm, None if h0 is None else h0[:, hv:hv + 1], nthreads)
        outs.append(o)
        states.append(hT)
    return np.concatenate(outs, 1), np.concatenate(states, 1), s_out


# ----------------------------------------------------------------- fused decode step

def sigmoid(x):
    """1 / (1 + e^{-x}) in fp64, evaluated on the side that cannot overflow."""
    x = _f64(x)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def softplus(x):
    """log(1 + e^x) in fp64: max(x, 0) + log1p(e^{-|x|})."""
    x = _f64(x)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def gates_from_logits(a_raw, b_raw):
    """The fused decode entry's gates ("[Feature] Add batch invariance support to GDN_ATTN
    backend - #45819" names fused_sigmoid_gating_delta_rule_update and gives no formula;
    the plainest reading): beta = sigmoid(b_raw), g = -softplus(a_raw).  Returns (g, beta)."""
    return -softplus(a_raw), sigmoid(b_raw)


def fused_decode(x, w, bias, a_raw, b_raw, conv_state_pool, state_pool, Hk, Hv, dk, dv,
                 state_idx=None, scale=1.0, l2norm=True, nthreads=None):
    """One decode step from raw inputs: conv update (the output taken as the bf16
    activation the conv stores), q/k/v split, gates from logits, recurrent step.
    Returns (o [N, Hv, dv], new conv pool, new state pool)."""
    y, conv_pool = conv1d_update(x, w, bias, conv_state_pool, state_idx)
    q, k, v = split_qkv(round_to_bf16(y), Hk, Hv, dk, dv)
    g, beta = gates_from_logits(a_raw, b_raw)
    o, pool = recurrent_decode(q, k, v, g, beta, state_pool, state_idx, scale, l2norm,
                               nthreads)
    return o, conv_pool, pool
