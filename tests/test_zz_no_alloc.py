"""gdn_chunk_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Such callers (an engine whose allocator owns all device memory, a loop that must not
allocate, a host program without a device allocator) cannot hand the library a
workspace; this entry point uses the library's own fixed device array instead.  The tests
call it through the C ABI: two calls in a row with different inputs must give exactly the
bits of the workspace-taking gdn_chunk_prefill (the same kernels run on the same inputs),
one of them is also checked against the fp64 oracle, and the call must make no device
allocation through the caller's allocator.  fp32 activations run on the CUDA-core kernel,
which needs no scratch, so a size far beyond the array still runs; a bf16 call of that size
is rejected.  The file is collected last and passes both alone and after the other tests.
"""
import gc

import pytest
import torch

import oracle
from gated_deltanet_linear_11_gb300 import _lib as gdn_lib
from gated_deltanet_linear_11_gb300 import inputs
from gpu_util import assert_bits_equal, assert_out_close, assert_state_close

pytestmark = pytest.mark.gpu

gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def on_gpu(x):
    out = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out["cu_seqlens"] = out["cu_seqlens"].to(torch.int32).contiguous()
    return out


def both_paths(x, l2norm):
    """The workspace entry, then the allocation-free one into preallocated outputs;
    returns their results and the number of allocation requests torch's allocator served
    during the second call."""
    xg = on_gpu(x)
    args = (xg["q"], xg["k"], xg["v"], xg["g"].contiguous(), xg["beta"].contiguous(),
            xg["cu_seqlens"])
    ref_o, ref_h = gdn.gdn_chunk_prefill(*args, l2norm=l2norm,
                                         initial_state=xg["initial_state"],
                                         cu_seqlens_host=x["cu_seqlens"])
    o = torch.full_like(ref_o, float("nan"))
    h = torch.full_like(ref_h, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu_host = x["cu_seqlens"].to(torch.int32).contiguous()
    gc.collect()
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats()["allocation.all.allocated"]
    gdn.gdn_chunk_prefill_noalloc(*args, l2norm=l2norm, initial_state=xg["initial_state"],
                                  o=o, final_state=h, cu_seqlens_host=cu_host,
                                  status=status)
    torch.cuda.synchronize()
    grown = torch.cuda.memory_stats()["allocation.all.allocated"] - before
    assert int(status.item()) == 0
    return (o, h), (ref_o, ref_h), grown


def test_noalloc_matches_workspace_entry_point_twice():
    first = inputs.scan_inputs(71, [1, 63, 64, 65, 300], 2, 6, 128, 128,
                               init_state_std=0.02)
    second = inputs.scan_inputs(72, [200, 9], 2, 6, 128, 128, normalise_qk=False,
                                init_state_std=0.02)
    for i, (x, l2) in enumerate(((first, False), (second, True))):
        (o, h), (ro, rh), grown = both_paths(x, l2)
        assert grown == 0, "the allocation-free call made %d device allocations" % grown
        assert_bits_equal(o, ro, "noalloc o (call %d)" % i)
        assert_bits_equal(h, rh, "noalloc state (call %d)" % i)
        if i == 1:
            o_ref, h_ref = oracle.gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                                   x["cu_seqlens"], l2norm=l2,
                                                   initial_state=x["initial_state"])
            assert_out_close(o, o_ref, what="noalloc o vs oracle")
            assert_state_close(h, h_ref, what="noalloc state vs oracle")


def test_noalloc_fp32_needs_no_scratch_at_any_size():
    """fp32 activations take the CUDA-core kernel, which uses no scratch: a size whose
    tensor-core workspace would be several times the array runs, bit-equal to the
    workspace entry on the same kernel."""
    T, Hk, Hv = 70000, 1, 8
    x = inputs.scan_inputs(74, [T], Hk, Hv, 128, 128, dtype=torch.float32)
    assert gdn.gdn_chunk_prefill_workspace_size(1, T, Hk, Hv, 128, 128) > \
        gdn_lib.NOALLOC_SCRATCH_BYTES
    (o, h), (ro, rh), grown = both_paths(x, False)
    assert grown == 0
    assert_bits_equal(o, ro, "noalloc fp32 o")
    assert_bits_equal(h, rh, "noalloc fp32 state")


def test_noalloc_rejects_requests_beyond_its_scratch():
    # the workspace of this bf16 call exceeds the library's fixed scratch array
    T, Hk, Hv = 70000, 1, 8
    x = inputs.scan_inputs(73, [T], Hk, Hv, 128, 128)
    xg = on_gpu(x)
    need = gdn.gdn_chunk_prefill_workspace_size(1, T, Hk, Hv, 128, 128)
    assert need > gdn_lib.NOALLOC_SCRATCH_BYTES
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_prefill_noalloc(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"],
                                      xg["cu_seqlens"], cu_seqlens_host=x["cu_seqlens"])
    assert e.value.code == 9  # GDN_ERR_WORKSPACE
