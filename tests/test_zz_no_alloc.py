"""gdn_chunk_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Such callers (an engine whose allocator owns all device memory, a loop that must not
allocate, a host program without a device allocator) cannot hand the library a
workspace; this entry point uses the library's own fixed device array instead.  The test
calls it through the C ABI twice in a row, with different inputs, and checks each result
against the workspace-taking gdn_chunk_prefill within the parity tolerances.  It sits in
a file that pytest collects last and passes both alone and after the other tests.
"""
import pytest
import torch

from gated_deltanet_linear_11_gb300 import _lib as gdn_lib
from gated_deltanet_linear_11_gb300 import inputs
from gpu_util import assert_out_close, assert_state_close, np64

pytestmark = pytest.mark.gpu

gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def both_paths(x, l2norm):
    xg = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    args = (xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"], xg["cu_seqlens"])
    ref_o, ref_h = gdn.gdn_chunk_prefill(*args, l2norm=l2norm,
                                         initial_state=xg["initial_state"],
                                         cu_seqlens_host=x["cu_seqlens"])
    o = torch.empty_like(ref_o)
    h = torch.empty_like(ref_h)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_chunk_prefill_noalloc(*args, l2norm=l2norm, initial_state=xg["initial_state"],
                                  o=o, final_state=h, cu_seqlens_host=x["cu_seqlens"],
                                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return (o, h), (ref_o, ref_h)


def test_noalloc_matches_workspace_entry_point_twice():
    first = inputs.scan_inputs(71, [1, 63, 64, 65, 300], 2, 6, 128, 128,
                               init_state_std=0.02)
    second = inputs.scan_inputs(72, [200, 9], 2, 6, 128, 128, normalise_qk=False,
                                init_state_std=0.02)
    for x, l2 in ((first, False), (second, True)):
        (o, h), (ro, rh) = both_paths(x, l2)
        assert_out_close(o, np64(ro), what="noalloc o")
        assert_state_close(h, np64(rh), what="noalloc state")


def test_noalloc_rejects_requests_beyond_its_scratch():
    # the workspace of this call exceeds the library's fixed scratch array
    T, Hk, Hv = 70000, 1, 8
    x = inputs.scan_inputs(73, [T], Hk, Hv, 128, 128)
    xg = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    need = gdn.gdn_chunk_prefill_workspace_size(1, T, Hk, Hv, 128, 128)
    assert need > gdn_lib.NOALLOC_SCRATCH_BYTES
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_prefill_noalloc(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"],
                                      xg["cu_seqlens"], cu_seqlens_host=x["cu_seqlens"])
    assert e.value.code == 9  # GDN_ERR_WORKSPACE
