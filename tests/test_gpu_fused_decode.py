"""gdn_fused_decode on the GPU: conv update + gates from raw logits + recurrent step in one
launch, against the fp64 oracle, against the two-launch path, and alone against batched.

Sizes: the 27B head shapes (Hk=16, Hv=48, d=128, 10240 conv channels) with a small
sequence count so the oracle finishes in seconds, plus the 4B head shapes (Hv=32).
Tolerances are the parity ones of tests/gpu_util.py; conv pools and batch comparisons
are bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_11_gb300 import inputs
from gpu_util import assert_bits_equal, assert_out_close, assert_state_close, np64

pytestmark = pytest.mark.gpu

gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def run_fused(d, idx=None, l2norm=True, scale=1.0, status=None, state=None, conv=None):
    state = d["state_pool"].cuda() if state is None else state
    conv = d["conv_state"].cuda() if conv is None else conv
    o = gdn.gdn_fused_decode(d["x"].cuda(), d["w"].cuda(),
                             None if d["bias"] is None else d["bias"].cuda(),
                             d["a_raw"].cuda(), d["b_raw"].cuda(), conv, state, d["Hk"],
                             d["Hv"], d["d"], d["d"],
                             state_idx=None if idx is None else idx.cuda(), scale=scale,
                             l2norm=l2norm, status=status)
    return o, conv, state


@pytest.mark.parametrize("shape,with_bias,l2norm", [("27b", False, True),
                                                      ("27b", True, False),
                                                      ("4b", False, True)])
def test_fused_decode_parity(shape, with_bias, l2norm):
    s = inputs.QWEN35_27B if shape == "27b" else inputs.QWEN35_4B
    d = inputs.fused_decode_inputs(61, N=6, pool=9, Hk=s["Hk"], Hv=s["Hv"], d=s["dk"],
                                   with_bias=with_bias)
    idx = d["state_idx"]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, conv, state = run_fused(d, idx, l2norm=l2norm, scale=0.8, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, conv_ref, pool_ref = oracle.fused_decode(
        d["x"], d["w"], d["bias"], d["a_raw"], d["b_raw"], d["conv_state"], d["state_pool"],
        s["Hk"], s["Hv"], s["dk"], s["dv"], state_idx=idx, scale=0.8, l2norm=l2norm)
    assert_out_close(o, o_ref)
    assert_state_close(state, pool_ref)
    # the conv pool only shifts stored bf16 values: exact
    assert np.array_equal(np64(conv), conv_ref)


def test_fused_matches_two_launch_path():
    """Same conv bits as gdn_conv1d_update; outputs and states within the parity bounds of
    gdn_conv1d_update + gdn_recurrent_decode fed the gates computed in fp32 by torch."""
    s = inputs.QWEN35_27B
    d = inputs.fused_decode_inputs(62, N=8, pool=8, Hk=s["Hk"], Hv=s["Hv"], d=s["dk"])
    idx = d["state_idx"].cuda()
    o, conv, state = run_fused(d, d["state_idx"])
    conv2 = d["conv_state"].cuda()
    state2 = d["state_pool"].cuda()
    g = -torch.nn.functional.softplus(d["a_raw"].cuda())
    beta = torch.sigmoid(d["b_raw"].cuda())
    o2 = gdn.gdn_layer_decode(d["x"].cuda(), d["w"].cuda(), None, g, beta, conv2, state2,
                              s["Hk"], s["Hv"], s["dk"], s["dv"], state_idx=idx)
    torch.cuda.synchronize()
    assert_bits_equal(conv, conv2, "conv pool")
    assert_out_close(o, np64(o2), what="o fused vs two-launch")
    assert_state_close(state, np64(state2), what="state fused vs two-launch")


def test_fused_decode_batch_invariance_bits():
    """Each sequence's o, state tile and conv state are bit-identical alone and batched."""
    s = inputs.QWEN35_27B
    d = inputs.fused_decode_inputs(63, N=5, pool=7, Hk=s["Hk"], Hv=s["Hv"], d=s["dk"])
    idx = d["state_idx"]
    o, conv, state = run_fused(d, idx)
    for n in range(5):
        one = dict(d)
        for key in ("x", "a_raw", "b_raw"):
            one[key] = d[key][n:n + 1]
        o1, conv1, state1 = run_fused(one, idx[n:n + 1])
        sl = int(idx[n])
        assert_bits_equal(o[n:n + 1], o1, "o[%d]" % n)
        assert_bits_equal(state[sl], state1[sl], "state[%d]" % n)
        assert_bits_equal(conv[sl], conv1[sl], "conv[%d]" % n)


def test_fused_decode_bad_index_reports_and_skips():
    s = inputs.QWEN35_4B
    d = inputs.fused_decode_inputs(64, N=3, pool=3, Hk=s["Hk"], Hv=s["Hv"], d=s["dk"])
    idx = torch.tensor([0, 7, 2], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = d["state_pool"].clone()
    o, conv, state = run_fused(d, idx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 10  # GDN_ERR_INDEX
    # slot 1 belongs to no valid token: untouched
    assert torch.equal(state[1].cpu(), before[1])
    assert torch.equal(conv[1].cpu(), d["conv_state"][1])
