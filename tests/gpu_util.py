"""Shared helpers for the GPU parity tests: tolerances and comparisons.

Tolerances (floating point, written here once and used by every parity test):

* bf16 outputs o, y:  max |gpu - oracle| <= OUT_ATOL = 2e-2.
* fp32 states:        ||gpu - oracle||_F / max(||oracle||_F, 1e-30) <= STATE_RTOL = 1e-3,
                      per (sequence, v-head).
* fp32 activations (small CUDA-core path): the same two bounds tightened to
  OUT_ATOL_F32 = 1e-4 and STATE_RTOL_F32 = 1e-5 (fp32 arithmetic throughout).
* Copies (conv tails) and batch-invariance checks: bit-exact.
"""
import numpy as np
import torch

OUT_ATOL = 2e-2
STATE_RTOL = 1e-3
OUT_ATOL_F32 = 1e-4
STATE_RTOL_F32 = 1e-5


def np64(t):
    return t.detach().float().cpu().double().numpy() if t.dtype == torch.bfloat16 \
        else t.detach().cpu().double().numpy()


def assert_out_close(gpu, ref, atol=OUT_ATOL, what="o"):
    g = np64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    err = np.abs(g - ref)
    assert np.isfinite(g).all(), "%s has non-finite values" % what
    mx = float(err.max()) if err.size else 0.0
    assert mx <= atol, "%s max abs err %.3e > %.1e (at %s)" % (
        what, mx, atol, np.unravel_index(err.argmax(), err.shape))
    return mx


def assert_state_close(gpu, ref, rtol=STATE_RTOL, what="state"):
    g = np64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    assert np.isfinite(g).all(), "%s has non-finite values" % what
    g = g.reshape(-1, g.shape[-2] * g.shape[-1])
    r = ref.reshape(-1, ref.shape[-2] * ref.shape[-1])
    num = np.linalg.norm(g - r, axis=1)
    den = np.maximum(np.linalg.norm(r, axis=1), 1e-30)
    rel = num / den
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= rtol, "%s rel err %.3e > %.1e (unit %d)" % (what, worst, rtol,
                                                                 int(rel.argmax()))
    return worst


def bits(t):
    return t.detach().contiguous().view(-1).view(torch.uint8)


def assert_bits_equal(a, b, what):
    assert a.shape == b.shape and a.dtype == b.dtype, "%s: shape/dtype differ" % what
    assert torch.equal(bits(a), bits(b)), "%s differs bitwise" % what
