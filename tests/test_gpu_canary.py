"""Guard bands: the kernels write exactly their outputs.

Every output buffer is placed inside a larger allocation filled with a sentinel bit
pattern; after the call the bytes before and after the output (and, for the state, the
neighbouring sequence slots) must still hold the sentinel.  The packed batches end in
partial chunks, so the last, partial chunk of every sequence is exercised at the end of
the buffer, where a row written past the sequence's end would land in the guard band.
"""
import pytest
import torch

from gated_deltanet_linear_11_gb300 import inputs

pytestmark = pytest.mark.gpu

gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")

SENTINEL_BF16 = 0x7FA5     # a NaN payload no kernel produces
SENTINEL_F32 = 0x7FA5A5A5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def guarded(shape, dtype, pad_rows):
    """A [pad + rows + pad, ...] buffer of sentinels and the [rows, ...] view inside it."""
    full = torch.empty((shape[0] + 2 * pad_rows,) + tuple(shape[1:]), dtype=dtype, device="cuda")
    bits = full.view(torch.int16 if dtype == torch.bfloat16 else torch.int32)
    bits.fill_(SENTINEL_BF16 if dtype == torch.bfloat16 else SENTINEL_F32)
    return full, full[pad_rows:pad_rows + shape[0]]


def assert_guards_intact(full, pad_rows, rows, what):
    bits = full.view(torch.int16 if full.dtype == torch.bfloat16 else torch.int32)
    want = SENTINEL_BF16 if full.dtype == torch.bfloat16 else SENTINEL_F32
    head, tail = bits[:pad_rows], bits[pad_rows + rows:]
    assert bool((head == want).all()), "%s: guard band before the output was written" % what
    assert bool((tail == want).all()), "%s: guard band after the output was written" % what
    inner = bits[pad_rows:pad_rows + rows]
    assert not bool((inner == want).all(dim=tuple(range(1, inner.dim()))).any()), \
        "%s: an output row was never written" % what


@pytest.mark.parametrize("simt", [False, True])
def test_prefill_writes_only_its_outputs(simt):
    lens = [70, 1, 129, 63, 5]          # every sequence ends in a partial chunk
    x = inputs.scan_inputs(61, lens, 2, 6, 128, 128, init_state_std=0.02)
    xg = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    T, N = sum(lens), len(lens)
    pad = 64
    o_full, o = guarded((T, 6, 128), torch.bfloat16, pad)
    h_full, h = guarded((N, 6, 128, 128), torch.float32, 2)
    gdn.gdn_chunk_prefill(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"], xg["cu_seqlens"],
                          initial_state=xg["initial_state"], o=o, final_state=h, simt=simt,
                          cu_seqlens_host=x["cu_seqlens"])
    torch.cuda.synchronize()
    assert_guards_intact(o_full, pad, T, "o")
    assert_guards_intact(h_full, 2, N, "final state")


@pytest.mark.parametrize("fused_vconv", [False, True])
def test_layer_prefill_writes_only_its_outputs(fused_vconv):
    s = dict(Hk=2, Hv=6, dk=128, dv=128)
    C = inputs.conv_channels(**s)
    lens = [100, 1, 67]
    cv = inputs.conv_inputs(62, lens, C, with_state=True)
    x = inputs.scan_inputs(63, lens, 2, 6, 128, 128, init_state_std=0.02)
    T, N = sum(lens), len(lens)
    pad = 64
    y_full, y = guarded((T, C), torch.bfloat16, pad)
    o_full, o = guarded((T, 6, 128), torch.bfloat16, pad)
    h_full, h = guarded((N, 6, 128, 128), torch.float32, 2)
    cs_full, cs = guarded((N, 3, C), torch.bfloat16, 2)
    gdn.gdn_layer_prefill(cv["x"].cuda(), cv["w"].cuda(), None, x["g"].cuda(),
                          x["beta"].cuda(), cv["cu_seqlens"].cuda(), s["Hk"], s["Hv"], 128,
                          128, conv_state_in=cv["conv_state"].cuda(), conv_state_out=cs,
                          initial_state=x["initial_state"].cuda(), final_state=h, y=y, o=o,
                          cu_seqlens_host=cv["cu_seqlens"], fused_vconv=fused_vconv)
    torch.cuda.synchronize()
    assert_guards_intact(y_full, pad, T, "conv output y")
    assert_guards_intact(o_full, pad, T, "o")
    assert_guards_intact(h_full, 2, N, "final state")
    assert_guards_intact(cs_full, 2, N, "conv state")


def test_decode_writes_only_its_outputs():
    N, P, Hk, Hv = 4, 8, 2, 6
    x = inputs.scan_inputs(64, [1] * N, Hk, Hv, 128, 128)
    xg = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    pool = (torch.randn(P, Hv, 128, 128, generator=torch.Generator().manual_seed(9)) * 0.02).cuda()
    idx = torch.tensor([5, 1, 6, 2], dtype=torch.int32, device="cuda")
    untouched = [0, 3, 4, 7]
    before = pool[untouched].clone()
    o_full, o = guarded((N, Hv, 128), torch.bfloat16, 4)
    gdn.gdn_recurrent_decode(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"], pool, idx, o=o)
    torch.cuda.synchronize()
    assert_guards_intact(o_full, 4, N, "decode o")
    assert torch.equal(pool[untouched], before), "decode wrote a pool slot outside state_idx"
