"""The decode step (conv update + recurrent step) captured in a CUDA graph and replayed.

The decode entry points take device-side state indices and need no host round trip, so
a serving loop can capture one step and replay it ("[Feature] Add batch invariance
support to GDN_ATTN backend - #45819", the commit that replaces .item()-based slicing by
tensor-indexed ssm_state_indices to avoid graph breaks).  Replays must give the same
bits as the same steps run eagerly.
"""
import pytest
import torch

from gated_deltanet_linear_11_gb300 import inputs
from gpu_util import assert_bits_equal

pytestmark = pytest.mark.gpu

gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def test_decode_step_graph_replay_matches_eager():
    s = inputs.QWEN35_27B
    N, P = 8, 12
    d = inputs.decode_27b(seed=11, N=N, pool=P)
    cv = d["conv"]
    cs0 = torch.randn(P, 3, cv["x"].shape[1], generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    w = cv["w"].cuda()
    idx = d["state_idx"].cuda()
    xs = [torch.randn(cv["x"].shape, generator=torch.Generator().manual_seed(40 + i)).to(torch.bfloat16).cuda()
          for i in range(3)]
    g, b = d["g"].cuda(), d["beta"].cuda()

    def run_eager():
        pool, cs = d["state_pool"].cuda(), cs0.cuda()
        outs = []
        for x in xs:
            outs.append(gdn.gdn_layer_decode(x, w, None, g, b, cs, pool, s["Hk"], s["Hv"],
                                             128, 128, state_idx=idx).clone())
        return outs, pool, cs

    o_e, pool_e, cs_e = run_eager()

    pool, cs = d["state_pool"].cuda(), cs0.cuda()
    x_static = torch.empty_like(xs[0])
    y = torch.empty_like(xs[0])
    o = torch.empty((N, s["Hv"], 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up outside the graph on the capture stream
        x_static.copy_(xs[0])
        pool_w, cs_w = pool.clone(), cs.clone()
        gdn.gdn_layer_decode(x_static, w, None, g, b, cs_w, pool_w, s["Hk"], s["Hv"], 128,
                             128, state_idx=idx, y=y, o=o, status=status)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.gdn_layer_decode(x_static, w, None, g, b, cs, pool, s["Hk"], s["Hv"], 128, 128,
                             state_idx=idx, y=y, o=o, status=status)
    outs = []
    for x in xs:
        x_static.copy_(x)
        graph.replay()
        outs.append(o.clone())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(3):
        assert_bits_equal(outs[i], o_e[i], "graph step %d output" % i)
    assert_bits_equal(pool, pool_e, "graph state pool")
    assert_bits_equal(cs, cs_e, "graph conv state")


def test_fused_decode_graph_replay_matches_eager():
    """gdn_fused_decode (two kernels per call) captured once and replayed on new tokens."""
    s = inputs.QWEN35_4B
    N, P = 6, 9
    d = inputs.fused_decode_inputs(12, N=N, pool=P, Hk=s["Hk"], Hv=s["Hv"], d=s["dk"])
    w = d["w"].cuda()
    idx = d["state_idx"].cuda()
    a, b = d["a_raw"].cuda(), d["b_raw"].cuda()
    xs = [torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(50 + i)).to(torch.bfloat16).cuda()
          for i in range(3)]

    def step(x, cs, pool, o=None, status=None):
        return gdn.gdn_fused_decode(x, w, None, a, b, cs, pool, s["Hk"], s["Hv"], 128, 128,
                                    state_idx=idx, o=o, status=status)

    pool_e, cs_e = d["state_pool"].cuda(), d["conv_state"].cuda()
    o_e = [step(x, cs_e, pool_e).clone() for x in xs]

    pool, cs = d["state_pool"].cuda(), d["conv_state"].cuda()
    x_static = torch.empty_like(xs[0])
    o = torch.empty((N, s["Hv"], 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up outside the graph on the capture stream
        x_static.copy_(xs[0])
        step(x_static, cs.clone(), pool.clone(), o=o, status=status)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(x_static, cs, pool, o=o, status=status)
    outs = []
    for x in xs:
        x_static.copy_(x)
        graph.replay()
        outs.append(o.clone())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(3):
        assert_bits_equal(outs[i], o_e[i], "fused graph step %d output" % i)
    assert_bits_equal(pool, pool_e, "fused graph state pool")
    assert_bits_equal(cs, cs_e, "fused graph conv state")
