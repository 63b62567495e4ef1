"""Decode steps and the prefill layer entry captured in CUDA graphs and replayed.

The decode entry points take device-side state indices and need no host round trip, so
a serving loop can capture one step and replay it ("[Feature] Add batch invariance
support to GDN_ATTN backend - #45819", the commit that replaces .item()-based slicing by
tensor-indexed ssm_state_indices to avoid graph breaks).  The prefill layer entry runs
part of its work on a second stream that forks from and joins the calling stream, so it
captures as one graph as well.  Replays must give the same bits as the same calls run
eagerly.
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


@pytest.mark.parametrize("use_side", [True, False, "fused"])
def test_layer_prefill_graph_replay_matches_eager(use_side):
    """gdn_layer_prefill captured once in a CUDA graph (with a side stream, that stream
    forks from and joins the capturing stream; without one, one stream; with the v conv
    fused into the state pass) and replayed on new inputs gives the eager call's bits."""
    s = dict(Hk=2, Hv=4, dk=128, dv=128)
    C = inputs.conv_channels(**s)
    lens = [150, 0, 183]
    cv = inputs.conv_inputs(91, lens, C, with_state=True, with_bias=True)
    sc = inputs.scan_inputs(92, lens, s["Hk"], s["Hv"], 128, 128, init_state_std=0.02)
    w, bias = cv["w"].cuda(), cv["bias"].cuda()
    g, beta = sc["g"].cuda(), sc["beta"].cuda()
    cu_h = cv["cu_seqlens"]
    cu = cu_h.cuda()
    cs_in, h0 = cv["conv_state"].cuda(), sc["initial_state"].cuda()
    xs = [inputs.conv_inputs(93 + i, lens, C)["x"].cuda() for i in range(3)]
    T, N = int(cu_h[-1]), len(lens)

    def outputs():
        return (torch.empty((T, s["Hv"], 128), dtype=torch.bfloat16, device="cuda"),
                torch.empty((N, s["Hv"], 128, 128), dtype=torch.float32, device="cuda"),
                torch.empty((N, 3, C), dtype=torch.bfloat16, device="cuda"),
                torch.empty((T, C), dtype=torch.bfloat16, device="cuda"))

    ws_bytes = gdn.gdn_chunk_prefill_workspace_size(N, T, s["Hk"], s["Hv"], 128, 128, 64)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    v_stream = torch.cuda.Stream() if use_side is True else None

    def call(x, out):
        o, hT, cs_out, y = out
        gdn.gdn_layer_prefill(x, w, bias, g, beta, cu, s["Hk"], s["Hv"], 128, 128,
                              conv_state_in=cs_in, conv_state_out=cs_out, initial_state=h0,
                              final_state=hT, scale=0.5, y=y, o=o, cu_seqlens_host=cu_h,
                              workspace=ws, status=status, side_stream=v_stream,
                              fused_vconv=use_side == "fused")

    eager = []
    for x in xs:
        out = outputs()
        call(x, out)
        eager.append([t.clone() for t in out])

    x_static = torch.empty_like(xs[0])
    out = outputs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up outside the graph on the capture stream
        x_static.copy_(xs[0])
        call(x_static, out)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(x_static, out)
    names = ("o", "final state", "conv state", "conv output")
    for i, x in enumerate(xs):
        x_static.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        for got, want, name in zip(out, eager[i], names):
            assert_bits_equal(got, want, "graph replay %d %s" % (i, name))
    assert int(status.item()) == 0
