"""Failure paths on the GPU, without a fault.

Every mbarrier wait of the tensor-core kernels gives up after 2 s, records
GDN_ERR_TIMEOUT in the caller's status word and lets the CTA return.  The self-test entry
runs that path on a barrier phase that nothing completes; the context must stay usable
afterwards.  The debug checks of the inputs (GDN_CHECK_INPUTS, set by GDN_DEBUG) must
reject a NaN or an infinity among the gates, and device offsets that differ from the
host copy, before anything is launched.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_11_gb300 import inputs
from gpu_util import assert_out_close, assert_state_close

pytestmark = pytest.mark.gpu

gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")
GDN_ERR_TIMEOUT = 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    gdn.gdn_selftest_bounded_wait(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == GDN_ERR_TIMEOUT
    assert 1.5 < waited < 60.0, waited

    # the next call on the same context runs normally and leaves its status clean
    x = inputs.scan_inputs(51, [70, 130], 2, 4, 128, 128, init_state_std=0.02)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, hT = gdn.gdn_chunk_prefill(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(),
                                  x["g"].cuda(), x["beta"].cuda(), x["cu_seqlens"].cuda(),
                                  initial_state=x["initial_state"].cuda(),
                                  cu_seqlens_host=x["cu_seqlens"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, h_ref = oracle.gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                           x["cu_seqlens"],
                                           initial_state=x["initial_state"])
    assert_out_close(o, o_ref)
    assert_state_close(hT, h_ref)


# ------------------------------------------------------- GDN_CHECK_INPUTS (debug mode)

GDN_ERR_NONFINITE = 11
GDN_ERR_SEQLENS = 5


def _same(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def test_check_finite_prefill(monkeypatch):
    """With GDN_DEBUG set, a NaN in g or an infinity in beta fails the call with
    GDN_ERR_NONFINITE, and a device cu_seqlens that differs from the host copy with
    GDN_ERR_SEQLENS, before anything is launched (o and the final state keep their
    sentinels); finite gates give the bits of the unchecked call."""
    x = inputs.scan_inputs(53, [70, 130], 2, 4, 128, 128, init_state_std=0.02)
    xg = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    cu_h = x["cu_seqlens"]

    def run(g, beta, o, hT, cp=False):
        if cp:
            return gdn.gdn_chunk_prefill_cp(xg["q"], xg["k"], xg["v"], g, beta,
                                            xg["cu_seqlens"], 1, o=o, final_state=hT,
                                            initial_state=xg["initial_state"],
                                            cu_seqlens_host=cu_h)
        return gdn.gdn_chunk_prefill(xg["q"], xg["k"], xg["v"], g, beta, xg["cu_seqlens"],
                                     o=o, final_state=hT, initial_state=xg["initial_state"],
                                     cu_seqlens_host=cu_h)

    def fresh():
        return (torch.full(xg["v"].shape, 3.0, dtype=torch.bfloat16, device="cuda"),
                torch.full((2, 4, 128, 128), 7.0, device="cuda"))

    monkeypatch.delenv("GDN_DEBUG", raising=False)
    o_ref, h_ref = run(xg["g"], xg["beta"], *fresh())
    monkeypatch.setenv("GDN_DEBUG", "1")
    o1, h1 = run(xg["g"], xg["beta"], *fresh())
    torch.cuda.synchronize()
    assert _same(o1, o_ref) and _same(h1, h_ref)
    g_bad = xg["g"].clone()
    g_bad[150, 3] = float("nan")
    beta_bad = xg["beta"].clone()
    beta_bad[5, 0] = float("inf")
    # a device cu_seqlens that disagrees with the host copy is refused before any launch
    # (the call below runs only with the check on: no kernel ever sees these offsets)
    cu_bad = xg["cu_seqlens"].clone()
    cu_bad[1] += 64
    o, hT = fresh()
    o0, h0 = o.clone(), hT.clone()
    assert gdn._debug_flags() == gdn.GDN_CHECK_INPUTS
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_prefill(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"], cu_bad, o=o,
                              final_state=hT, initial_state=xg["initial_state"],
                              cu_seqlens_host=cu_h)
    assert e.value.code == GDN_ERR_SEQLENS
    torch.cuda.synchronize()
    assert _same(o, o0) and _same(hT, h0)
    for g, beta, cp in ((g_bad, xg["beta"], False), (xg["g"], beta_bad, False),
                        (g_bad, xg["beta"], True)):
        o, hT = fresh()
        o0, h0 = o.clone(), hT.clone()
        with pytest.raises(gdn.GdnError) as e:
            run(g, beta, o, hT, cp=cp)
        assert e.value.code == GDN_ERR_NONFINITE
        torch.cuda.synchronize()
        assert _same(o, o0) and _same(hT, h0)


def test_check_finite_layer_and_decode(monkeypatch):
    """The layer entry checks before its conv launches (y keeps its sentinel); the decode
    entries check their gates (g and beta; the fused step's logits) and leave the state
    and conv pools as they were."""
    monkeypatch.setenv("GDN_DEBUG", "1")
    Hk, Hv, d = 2, 4, 128
    C = inputs.conv_channels(Hk, Hv, d, d)
    cv = inputs.conv_inputs(54, [90, 40], C)
    T = 130
    g, beta = inputs.gates(np.random.default_rng(55), T, Hv, 2.0)
    g[17, 1] = float("nan")
    y = torch.full((T, C), 5.0, dtype=torch.bfloat16, device="cuda")
    y0 = y.clone()
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_layer_prefill(cv["x"].cuda(), cv["w"].cuda(), None, g.cuda(), beta.cuda(),
                              cv["cu_seqlens"].cuda(), Hk, Hv, d, d, y=y,
                              cu_seqlens_host=cv["cu_seqlens"])
    assert e.value.code == GDN_ERR_NONFINITE
    torch.cuda.synchronize()
    assert _same(y, y0)

    x = inputs.scan_inputs(56, [1] * 3, Hk, Hv, d, d)
    pool = (torch.randn(3, Hv, d, d, generator=torch.Generator().manual_seed(5)) * 0.02).cuda()
    pool0 = pool.clone()
    gd = x["g"].clone()
    gd[2, 3] = float("-inf")
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_recurrent_decode(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gd.cuda(),
                                 x["beta"].cuda(), pool)
    assert e.value.code == GDN_ERR_NONFINITE
    torch.cuda.synchronize()
    assert _same(pool, pool0)

    fd = inputs.fused_decode_inputs(seed=57, N=4, Hk=Hk, Hv=Hv, d=d)
    a_raw = fd["a_raw"].clone()
    a_raw[1, 2] = float("nan")
    state, conv = fd["state_pool"].cuda(), fd["conv_state"].cuda()
    state0, conv0 = state.clone(), conv.clone()
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_fused_decode(fd["x"].cuda(), fd["w"].cuda(), None, a_raw.cuda(),
                             fd["b_raw"].cuda(), conv, state, Hk, Hv, d, d,
                             state_idx=fd["state_idx"].cuda())
    assert e.value.code == GDN_ERR_NONFINITE
    torch.cuda.synchronize()
    assert _same(state, state0) and _same(conv, conv0)
