"""The bounded waits' failure path, on the GPU and without a fault.

Every mbarrier wait of the tensor-core kernels gives up after 2 s, records
GDN_ERR_TIMEOUT in the caller's status word and lets the CTA return.  The self-test entry
runs that path on a barrier phase that nothing completes; the context must stay usable
afterwards.
"""
import time

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
