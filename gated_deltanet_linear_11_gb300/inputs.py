"""Seeded synthetic inputs for the GDN layer workloads.

This module only draws random numbers and lays them out; it holds none of the layer's
arithmetic and imports nothing else from this package, so both the CUDA path's tests and
the fp64 oracle's tests consume exactly the same values.  Every tensor is returned on the
CPU; bf16 tensors are rounded once (round-to-nearest-even by torch) from fp32 draws and
the oracle reads those stored bf16 values upcast exactly.

Shapes follow the pages: token-major [T, H, D] activations ("Fix [Bug]: Qwen3.5 ... FLA
linear attention tensor format mismatch", Root Cause: head_first=False expects
[B, T, H, ...]); packed varlen offsets cu_seqlens; fp32 recurrent state
[N, Hv, dk, dv] and a three-row conv state per sequence ("[Feature] Add batch invariance
support to GDN_ATTN backend - #45819", Birol's comment, parts 1 and 3).  Qwen3.5-27B
head counts: 48 GDN v-heads with dv = 128 (out_proj [5120, 6144] in "Qwen3.5-27B GPTQ
Garbage Inference -- Root Cause Analysis", Architecture Background) and 16 q/k heads.

Distributions: q, k ~ N(0,1) then L2-normalised per head (where pre-normalised), v ~ N(0,1),
beta = sigmoid(N(0,1)), g = -softplus(N(0,1) + shift), initial states ~ N(0, 0.02^2),
conv weights ~ U(-0.5, 0.5), conv states ~ N(0,1).
"""
from __future__ import annotations

import numpy as np
import torch

DTYPE_BF16 = torch.bfloat16


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _t(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dtype)


def _unit(a):
    return a / np.sqrt((a.astype(np.float64) ** 2).sum(-1, keepdims=True)).astype(np.float32)


def _softplus(x):
    return np.logaddexp(0.0, x)


def gates(rng, T, Hv, g_shift=0.0):
    """beta = sigmoid(N(0,1)), g = -softplus(N(0,1) + g_shift); both fp32 [T, Hv]."""
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, Hv))))
    g = -_softplus(rng.standard_normal((T, Hv)) + g_shift)
    return _t(g, torch.float32), _t(beta, torch.float32)


def scan_inputs(seed, lens, Hk, Hv, dk, dv, dtype=DTYPE_BF16, g_shift=2.0,
                normalise_qk=True, init_state_std=None):
    """Packed varlen q/k/v/g/beta (+ optional initial state) for the scan.

    lens: list of sequence lengths.  Returns a dict with q, k [T,Hk,dk], v [T,Hv,dv],
    g, beta [T,Hv] fp32, cu_seqlens int32 [N+1], initial_state fp32 [N,Hv,dk,dv] or None.
    """
    rng = _rng(seed)
    lens = [int(x) for x in lens]
    T = int(sum(lens))
    q = rng.standard_normal((T, Hk, dk)).astype(np.float32)
    k = rng.standard_normal((T, Hk, dk)).astype(np.float32)
    if normalise_qk:
        q, k = _unit(q), _unit(k)
    v = rng.standard_normal((T, Hv, dv)).astype(np.float32)
    g, beta = gates(rng, T, Hv, g_shift)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    h0 = None
    if init_state_std:
        h0 = _t(rng.standard_normal((len(lens), Hv, dk, dv)) * init_state_std,
                torch.float32)
    return dict(q=_t(q, dtype), k=_t(k, dtype), v=_t(v, dtype), g=g, beta=beta,
                cu_seqlens=torch.from_numpy(cu), initial_state=h0)


def conv_inputs(seed, lens, C, with_state=False, with_bias=False, dtype=DTYPE_BF16):
    """Packed conv input x [T, C], weights [C, 4], bias [C] or None, conv state [N,3,C]."""
    rng = _rng(seed)
    lens = [int(x) for x in lens]
    T = int(sum(lens))
    x = rng.standard_normal((T, C))
    w = rng.uniform(-0.5, 0.5, (C, 4))
    b = rng.uniform(-0.5, 0.5, (C,)) if with_bias else None
    st = rng.standard_normal((len(lens), 3, C)) if with_state else None
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    return dict(x=_t(x, dtype), w=_t(w, dtype), bias=None if b is None else _t(b, dtype),
                conv_state=None if st is None else _t(st, dtype),
                cu_seqlens=torch.from_numpy(cu))


# ------------------------------------------------------------------ named workloads

def tiny(seed=1):
    """Tiny gated delta rule in fp32: one sequence T=64, 2 heads, dk=dv=16, chunk 16."""
    d = scan_inputs(seed, [64], 2, 2, 16, 16, dtype=torch.float32, g_shift=0.0)
    d["chunk"] = 16
    return d


QWEN35_27B = dict(Hk=16, Hv=48, dk=128, dv=128)
QWEN35_4B = dict(Hk=16, Hv=32, dk=128, dv=128)


def conv_channels(Hk, Hv, dk, dv):
    """Packed q||k||v conv channel count (10240 for the 27B head shapes)."""
    return Hk * dk * 2 + Hv * dv


def layer_27b(seed=2, T=4096):
    """Qwen3.5-27B-shaped GDN layer prefill: conv over packed q||k||v, then the scan."""
    s = QWEN35_27B
    C = conv_channels(**s)
    conv = conv_inputs(seed, [T], C)
    rng = _rng(seed + 100)
    g, beta = gates(rng, T, s["Hv"], 2.0)
    return dict(conv=conv, g=g, beta=beta, **s)


def varlen_lengths(seed=3, n=8, lo=1, hi=8192):
    return [int(x) for x in _rng(seed).integers(lo, hi + 1, n)]


def varlen_27b(seed=3, n=8, hi=8192):
    s = QWEN35_27B
    lens = varlen_lengths(seed, n, 1, hi)
    d = scan_inputs(seed, lens, s["Hk"], s["Hv"], s["dk"], s["dv"], init_state_std=0.02)
    d["conv"] = conv_inputs(seed + 100, lens, conv_channels(**s), with_state=True)
    d["lens"] = lens
    return d


def decode_27b(seed=4, N=256, pool=None):
    """Decode step: N sequences, one token each, fp32 state pool [P, Hv, dk, dv]."""
    s = QWEN35_27B
    d = scan_inputs(seed, [1] * N, s["Hk"], s["Hv"], s["dk"], s["dv"])
    rng = _rng(seed + 200)
    P = N if pool is None else int(pool)
    d["state_pool"] = _t(rng.standard_normal((P, s["Hv"], s["dk"], s["dv"])) * 0.02,
                         torch.float32)
    d["state_idx"] = torch.from_numpy(rng.permutation(P)[:N].astype(np.int32))
    d["conv"] = conv_inputs(seed + 300, [1] * N, conv_channels(**s), with_state=True)
    return d


def mix_lengths(seed=5, n_each=20, lo=12, hi=32768):
    rng = _rng(seed)
    fresh = [int(x) for x in rng.integers(lo, hi + 1, n_each)]
    return fresh, [2048] * n_each, [1] * n_each


def fused_decode_inputs(seed=6, N=256, pool=None, Hk=16, Hv=48, d=128, with_bias=False):
    """Raw inputs of one decode step for the fused entry: x_qkv [N, C] bf16 (q|k|v before
    the conv), conv weights [C, 4] (and bias), conv state pool [P, 3, C] bf16, gate logits
    a_raw = N(0,1) + 2 and b_raw = N(0,1) [N, Hv] fp32 (their -softplus and sigmoid follow
    the g and beta distributions of the decode workload), fp32 state pool
    [P, Hv, d, d] ~ N(0, 0.02), and state_idx: N distinct slots of P in random order."""
    rng = _rng(seed)
    P = N if pool is None else int(pool)
    C = conv_channels(Hk, Hv, d, d)
    x = rng.standard_normal((N, C))
    w = rng.uniform(-0.5, 0.5, (C, 4))
    b = rng.uniform(-0.5, 0.5, (C,)) if with_bias else None
    cs = rng.standard_normal((P, 3, C))
    a_raw = rng.standard_normal((N, Hv)) + 2.0
    b_raw = rng.standard_normal((N, Hv))
    st = rng.standard_normal((P, Hv, d, d)).astype(np.float32) * np.float32(0.02)
    idx = rng.permutation(P)[:N].astype(np.int32)
    return dict(x=_t(x, DTYPE_BF16), w=_t(w, DTYPE_BF16),
                bias=None if b is None else _t(b, DTYPE_BF16), conv_state=_t(cs, DTYPE_BF16),
                a_raw=_t(a_raw, torch.float32), b_raw=_t(b_raw, torch.float32),
                state_pool=torch.from_numpy(st), state_idx=torch.from_numpy(idx),
                Hk=Hk, Hv=Hv, d=d)
