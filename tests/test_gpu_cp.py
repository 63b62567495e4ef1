"""GPU: the context-parallel scan (gdn_chunk_prefill_cp) through the C ABI.

Each sequence is split into ranges of ``range_chunks`` 64-token chunks.  A range's end
state is an affine map of its start state, so the ranges run side by side and their
start states are composed in order (the pin of that algebra is
test_range_end_state_is_affine_in_start_state).  The results must meet the oracle's
tolerances, equal gdn_chunk_prefill bit for bit when a sequence is a single range, and be
the same bits alone and in any batch for a given range length.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_11_gb300 import inputs
from gpu_util import assert_bits_equal, assert_out_close, assert_state_close

pytestmark = pytest.mark.gpu

gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def run_cp(x, range_chunks, l2norm=False, tiles=None):
    xg = cuda(x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, hT = gdn.gdn_chunk_prefill_cp(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"],
                                     xg["cu_seqlens"], range_chunks, l2norm=l2norm,
                                     initial_state=xg["initial_state"],
                                     cu_seqlens_host=x["cu_seqlens"], status=status,
                                     tiles=tiles)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o, hT


def run_plain(x, l2norm=False):
    xg = cuda(x)
    return gdn.gdn_chunk_prefill(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"],
                                 xg["cu_seqlens"], l2norm=l2norm,
                                 initial_state=xg["initial_state"],
                                 cu_seqlens_host=x["cu_seqlens"])


@pytest.mark.parametrize("range_chunks,l2norm", [(1, False), (2, True), (3, False)])
def test_cp_matches_oracle(range_chunks, l2norm):
    """Packed ragged sequences with initial states: from one range (short ones, empty
    ones) to eleven (700 tokens at one chunk per range), partial last chunks included."""
    lens = [700, 64, 1, 0, 300, 129, 200]
    x = inputs.scan_inputs(101, lens, 2, 6, 128, 128, normalise_qk=not l2norm,
                           init_state_std=0.02)
    o, hT = run_cp(x, range_chunks, l2norm=l2norm)
    o_ref, h_ref = oracle.gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                           x["cu_seqlens"], l2norm=l2norm,
                                           initial_state=x["initial_state"])
    assert_out_close(o, o_ref, what="cp o")
    assert_state_close(hT, h_ref, what="cp final state")


def test_cp_weak_decay_long_sequence():
    """A slowly decaying state carried through many composed ranges (g_shift -3: the
    state remembers far back, so errors in the composed maps would show)."""
    x = inputs.scan_inputs(102, [1536], 1, 3, 128, 128, g_shift=-3.0, init_state_std=0.02)
    o, hT = run_cp(x, 4)
    o_ref, h_ref = oracle.gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                           x["cu_seqlens"], initial_state=x["initial_state"])
    assert_out_close(o, o_ref, what="cp o")
    assert_state_close(hT, h_ref, what="cp final state")


def test_cp_single_range_equals_plain_scan_bits():
    """When every sequence fits one range the context-parallel scan runs exactly the
    plain scan's arithmetic."""
    lens = [130, 1, 64, 300, 17]
    x = inputs.scan_inputs(103, lens, 2, 4, 128, 128, init_state_std=0.02)
    o1, h1 = run_cp(x, 64)
    o2, h2 = run_plain(x)
    assert_bits_equal(o1, o2, "o, one range vs plain scan")
    assert_bits_equal(h1, h2, "final state, one range vs plain scan")


def test_cp_batch_invariance_and_tilings():
    """Each sequence's bits are the same alone and inside a batch (ranges depend only on
    its own length), and under either dv tiling."""
    lens = [500, 77, 256, 1, 190]
    x = inputs.scan_inputs(104, lens, 2, 6, 128, 128, init_state_std=0.02)
    o_b, h_b = run_cp(x, 2)
    o_t, h_t = run_cp(x, 2, tiles=2)
    assert_bits_equal(o_b, o_t, "o, cp under both tilings")
    assert_bits_equal(h_b, h_t, "final state, cp under both tilings")
    cu = x["cu_seqlens"].tolist()
    for n in (0, 2, 4):
        a, b = cu[n], cu[n + 1]
        xs = dict(x)
        for key in ("q", "k", "v", "g", "beta"):
            xs[key] = x[key][a:b].clone()
        xs["cu_seqlens"] = torch.tensor([0, b - a], dtype=torch.int32)
        xs["initial_state"] = x["initial_state"][n:n + 1].clone()
        o1, h1 = run_cp(xs, 2)
        assert_bits_equal(o1, o_b[a:b], "o of sequence %d alone vs in the batch" % n)
        assert_bits_equal(h1, h_b[n:n + 1], "state of sequence %d alone vs in the batch" % n)


def test_cp_range_hint():
    """The range hint follows the wave arithmetic of the two passes: a single-chunk
    sequence cannot be split, the 27B layer's 4096 tokens over 48 v-heads already fill
    the SMs (when there are fewer than 3 * 48 * 2 of them), one 32768-token sequence over
    6 v-heads is split, and the hint depends on the sequence alone (the same answer
    whenever asked)."""
    hint = gdn.gdn_chunk_prefill_cp_range_hint
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert hint(64, 6) == 0
    if sms < 3 * 48 * 2:
        assert hint(4096, 48) == 0
    r = hint(32768, 6)
    assert 0 < r < 512
    assert hint(32768, 6) == r
    assert hint(32768, 6, sm_count=sms) == r     # the device's own SM count


def test_cp_27b_shapes_sampled_heads():
    """27B head shapes (Hk = 16, Hv = 48), one 4096-token sequence from a random state,
    in ranges of 16 chunks; the oracle runs three sampled v-heads of different k-heads."""
    x = inputs.scan_inputs(105, [4096], 16, 48, 128, 128, normalise_qk=False,
                           init_state_std=0.02)
    o, hT = run_cp(x, 16, l2norm=True)
    heads = [0, 22, 47]
    G = 3
    for hv in heads:
        hk = hv // G
        o_ref, h_ref = oracle.gated_delta_rule(
            x["q"][:, hk:hk + 1], x["k"][:, hk:hk + 1], x["v"][:, hv:hv + 1],
            x["g"][:, hv:hv + 1], x["beta"][:, hv:hv + 1], x["cu_seqlens"], l2norm=True,
            initial_state=x["initial_state"][:, hv:hv + 1])
        assert_out_close(o[:, hv:hv + 1], o_ref, what="cp o head %d" % hv)
        assert_state_close(hT[:, hv:hv + 1], h_ref, what="cp state head %d" % hv)


def test_cp_graph_replay_matches_eager():
    """gdn_chunk_prefill_cp captured once in a CUDA graph (its table, prep, two state and
    composition launches, no host synchronisation) and replayed on new inputs gives the
    eager call's bits."""
    lens = [700, 0, 190]
    xs = [inputs.scan_inputs(110 + i, lens, 2, 6, 128, 128, init_state_std=0.02)
          for i in range(3)]
    cu_h = xs[0]["cu_seqlens"]
    T, N = int(cu_h[-1]), len(lens)
    ws = torch.empty(max(gdn.gdn_chunk_prefill_cp_workspace_size(cu_h, T, 2, 6, 128, 128, 2),
                         256), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    static = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in xs[0].items()}
    o = torch.empty((T, 6, 128), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty((N, 6, 128, 128), dtype=torch.float32, device="cuda")

    def call():
        gdn.gdn_chunk_prefill_cp(static["q"], static["k"], static["v"], static["g"],
                                 static["beta"], static["cu_seqlens"], 2,
                                 initial_state=static["initial_state"], o=o, final_state=hT,
                                 cu_seqlens_host=cu_h, workspace=ws, status=status)

    eager = []
    for x in xs:
        for key in ("q", "k", "v", "g", "beta", "initial_state"):
            static[key].copy_(x[key])
        call()
        eager.append((o.clone(), hT.clone()))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for i, x in enumerate(xs):
        for key in ("q", "k", "v", "g", "beta", "initial_state"):
            static[key].copy_(x[key])
        graph.replay()
        torch.cuda.synchronize()
        assert_bits_equal(o, eager[i][0], "cp graph replay %d o" % i)
        assert_bits_equal(hT, eager[i][1], "cp graph replay %d final state" % i)
    assert int(status.item()) == 0
