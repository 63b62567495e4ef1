"""GPU parity: every entry point of libgdn.so against the fp64 oracle, through the C ABI.

Sizes are small enough for the oracle to finish in seconds but span several chunks,
several conv tiles and ragged tails.  Tolerances live in tests/gpu_util.py.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_11_gb300 import inputs
from gpu_util import (OUT_ATOL_F32, STATE_RTOL_F32, assert_bits_equal, assert_out_close,
                      assert_state_close, np64)

pytestmark = pytest.mark.gpu

gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.load()


def cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


# ----------------------------------------------------------------------------- conv

@pytest.mark.parametrize("with_state,with_bias", [(False, False), (True, True)])
def test_conv1d_fwd_parity(with_state, with_bias):
    lens = [1, 2, 3, 15, 16, 17, 100]
    C = 1024 + 8 * 3
    d = inputs.conv_inputs(21, lens, C, with_state=with_state, with_bias=with_bias)
    x, w, b, st, cu = (d["x"].cuda(), d["w"].cuda(),
                       None if d["bias"] is None else d["bias"].cuda(),
                       None if d["conv_state"] is None else d["conv_state"].cuda(),
                       d["cu_seqlens"])
    y, s_out = gdn.gdn_conv1d_fwd(x, w, b, cu.cuda(), st, None, cu_seqlens_host=cu)
    yr, sr = oracle.conv1d_varlen(d["x"], d["w"], d["bias"], cu, d["conv_state"])
    assert_out_close(y, yr, what="conv y")
    # tails are copies of inputs: bit-exact
    np.testing.assert_array_equal(np64(s_out), sr)


def test_conv1d_fwd_in_place_state_and_empty_sequence():
    lens = [0, 5, 0, 40]
    C = 256
    d = inputs.conv_inputs(22, lens, C, with_state=True)
    st = d["conv_state"].cuda()
    cu = d["cu_seqlens"]
    y, s_out = gdn.gdn_conv1d_fwd(d["x"].cuda(), d["w"].cuda(), None, cu.cuda(), st, st,
                                  cu_seqlens_host=cu)
    assert s_out.data_ptr() == st.data_ptr()
    yr, sr = oracle.conv1d_varlen(d["x"], d["w"], None, cu, d["conv_state"])
    assert_out_close(y, yr, what="conv y")
    np.testing.assert_array_equal(np64(st), sr)


def test_conv_silu_over_the_bf16_range():
    """The conv's SiLU against the fp64 definition z / (1 + e^-z) on every finite bf16
    value with |z| <= 120: a conv whose only tap is the newest input (w = [0, 0, 0, 1],
    no bias) outputs silu(x) rounded to bf16, which must be within one bf16 unit in the
    last place of the exactly rounded value, or within 1e-30 where that value is tiny
    (below z = -87 the exponential overflows and the kernel returns a signed zero)."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    z = vals[np.isfinite(vals) & (np.abs(vals) <= 120.0)]
    C = 1024
    T = -(-z.size // C)
    x = np.zeros(T * C, dtype=np.float32)
    x[:z.size] = z
    xt = torch.from_numpy(x.reshape(T, C)).to(torch.bfloat16)
    assert np.array_equal(xt.float().numpy().ravel()[:z.size], z)   # exact bf16 values
    w = torch.zeros(C, 4, dtype=torch.bfloat16)
    w[:, 3] = 1.0
    cu = torch.tensor([0, T], dtype=torch.int32)
    y, _ = gdn.gdn_conv1d_fwd(xt.cuda(), w.cuda(), None, cu.cuda(), cu_seqlens_host=cu)
    got = y.float().cpu().numpy().ravel()[:z.size].astype(np.float64)
    zd = z.astype(np.float64)
    with np.errstate(over="ignore"):
        exact = zd / (1.0 + np.exp(-zd))
    ref = torch.from_numpy(exact).to(torch.bfloat16).double().numpy()   # round to nearest
    r32 = ref.astype(np.float32)
    ulp = 65536.0 * np.maximum(np.abs(np.nextafter(r32, np.float32(np.inf)) - ref),
                               np.abs(np.nextafter(r32, np.float32(-np.inf)) - ref))
    err = np.abs(got - ref)
    bad = ~((err <= ulp) | (err <= 1e-30))
    assert not bad.any(), (z[bad][:8], got[bad][:8], ref[bad][:8])


def test_conv1d_update_matches_oracle_and_prefill_bits():
    N, P, C = 12, 20, 1024
    d = inputs.conv_inputs(23, [1] * N, C, with_state=True, with_bias=True)
    pool = torch.randn(P, 3, C, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    idx = torch.randperm(P, generator=torch.Generator().manual_seed(6))[:N].to(torch.int32)
    pool_gpu = pool.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = gdn.gdn_conv1d_update(d["x"].cuda(), d["w"].cuda(), d["bias"].cuda(), pool_gpu,
                              idx.cuda(), status=status)
    yr, pr = oracle.conv1d_update(d["x"], d["w"], d["bias"], pool, idx)
    assert int(status.item()) == 0
    assert_out_close(y, yr, what="conv update y")
    np.testing.assert_array_equal(np64(pool_gpu), pr)
    # The decode step is the prefill conv for one token: same bits.
    cu = torch.arange(N + 1, dtype=torch.int32)
    y2, _ = gdn.gdn_conv1d_fwd(d["x"].cuda(), d["w"].cuda(), d["bias"].cuda(), cu.cuda(),
                               pool[idx.long()].contiguous().cuda(), None, cu_seqlens_host=cu)
    assert_bits_equal(y, y2, "conv update vs prefill conv")


def test_conv1d_update_bad_index_reports_status():
    N, P, C = 4, 4, 64
    x = torch.randn(N, C, device="cuda").to(torch.bfloat16)
    w = torch.rand(C, 4, device="cuda").to(torch.bfloat16)
    pool = torch.zeros(P, 3, C, device="cuda", dtype=torch.bfloat16)
    idx = torch.tensor([0, 1, 7, 2], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_conv1d_update(x, w, None, pool, idx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 10  # GDN_ERR_INDEX; the other sequences still ran
    assert pool[[0, 1, 2], 2].abs().sum().item() > 0


# --------------------------------------------------------------------------- decode

@pytest.mark.parametrize("l2norm", [False, True])
def test_recurrent_decode_parity(l2norm):
    N, P, Hk, Hv, d = 8, 11, 2, 6, 128
    x = inputs.scan_inputs(31, [1] * N, Hk, Hv, d, d, normalise_qk=not l2norm)
    pool = (torch.randn(P, Hv, d, d, generator=torch.Generator().manual_seed(3)) * 0.02)
    idx = torch.tensor([3, 0, 10, 5, 7, 1, 9, 2], dtype=torch.int32)
    pool_gpu = pool.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.gdn_recurrent_decode(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(),
                                 x["g"].cuda(), x["beta"].cuda(), pool_gpu, idx.cuda(),
                                 scale=0.75, l2norm=l2norm, status=status)
    o_ref, pool_ref = oracle.recurrent_decode(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                              pool, idx, scale=0.75, l2norm=l2norm)
    assert int(status.item()) == 0
    assert_out_close(o, o_ref)
    assert_state_close(pool_gpu, pool_ref)


def test_recurrent_decode_fp32_tight():
    N, Hk, Hv, d = 3, 1, 2, 128
    x = inputs.scan_inputs(32, [1] * N, Hk, Hv, d, d, dtype=torch.float32)
    pool = torch.randn(N, Hv, d, d, generator=torch.Generator().manual_seed(4)) * 0.02
    pool_gpu = pool.cuda()
    o = gdn.gdn_recurrent_decode(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(),
                                 x["g"].cuda(), x["beta"].cuda(), pool_gpu)
    o_ref, pool_ref = oracle.recurrent_decode(x["q"], x["k"], x["v"], x["g"], x["beta"], pool)
    assert_out_close(o, o_ref, atol=OUT_ATOL_F32)
    assert_state_close(pool_gpu, pool_ref, rtol=STATE_RTOL_F32)


# --------------------------------------------------------------------- chunk prefill

def run_prefill(x, chunk=64, l2norm=False, simt=False, scale=1.0):
    xg = cuda(x)
    o, hT = gdn.gdn_chunk_prefill(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"],
                                  xg["cu_seqlens"], chunk=chunk, scale=scale, l2norm=l2norm,
                                  initial_state=xg["initial_state"], simt=simt,
                                  cu_seqlens_host=x["cu_seqlens"])
    return o, hT


def ref_prefill(x, l2norm=False, scale=1.0):
    return oracle.gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                   x["cu_seqlens"], scale=scale, l2norm=l2norm,
                                   initial_state=x["initial_state"])


def test_tiny_fp32_config():
    """B=1, T=64, 2 heads, dk=dv=16, chunk 16, fp32."""
    x = inputs.tiny()
    o, hT = run_prefill(x, chunk=16)
    o_ref, h_ref = ref_prefill(x)
    assert_out_close(o, o_ref, atol=OUT_ATOL_F32)
    assert_state_close(hT, h_ref, rtol=STATE_RTOL_F32)


@pytest.mark.parametrize("d,chunk", [(16, 16), (32, 32), (64, 64), (128, 16)])
def test_simt_fp32_shapes(d, chunk):
    x = inputs.scan_inputs(41, [1, chunk - 1, chunk, chunk + 1, 3 * chunk + 5], 2, 4, d, d,
                           dtype=torch.float32, g_shift=0.0, init_state_std=0.05)
    o, hT = run_prefill(x, chunk=chunk, simt=True, scale=0.5)
    o_ref, h_ref = ref_prefill(x, scale=0.5)
    assert_out_close(o, o_ref, atol=OUT_ATOL_F32)
    assert_state_close(hT, h_ref, rtol=STATE_RTOL_F32)


@pytest.mark.parametrize("simt", [True, False])
@pytest.mark.parametrize("l2norm", [False, True])
def test_prefill_bf16_d128_parity(simt, l2norm):
    lens = [1, 63, 64, 65, 200, 7]
    x = inputs.scan_inputs(42, lens, 2, 6, 128, 128, normalise_qk=not l2norm,
                           init_state_std=0.02)
    o, hT = run_prefill(x, chunk=64, l2norm=l2norm, simt=simt)
    o_ref, h_ref = ref_prefill(x, l2norm=l2norm)
    assert_out_close(o, o_ref)
    assert_state_close(hT, h_ref)


@pytest.mark.parametrize("nseq", [6, 9])
def test_prefill_tc_scale_parity(nseq):
    """Tensor-core scan with scale != 1 against the oracle: the scale enters both output
    paths (full chunks leave by tensor store, a sequence's partial last chunk by plain
    stores).  On a 152-SM GB300, 6 sequences x 6 v-heads run the state pass in three dv
    tiles (48 + 48 + 32 columns), 9 sequences in two (3 * Hv * N > 152)."""
    lens = [64, 130, 1, 192, 77, 5, 128, 63, 200][:nseq]
    x = inputs.scan_inputs(49, lens, 2, 6, 128, 128, init_state_std=0.02)
    o, hT = run_prefill(x, scale=0.6)
    o_ref, h_ref = ref_prefill(x, scale=0.6)
    assert_out_close(o, o_ref)
    assert_state_close(hT, h_ref)


@pytest.mark.parametrize("simt", [True, False])
def test_prefill_empty_sequences_keep_their_state(simt):
    """Zero-length sequences inside a packed batch: their final state is their initial
    state, bit for bit, and the neighbours match the oracle."""
    lens = [0, 70, 0, 1, 0]
    x = inputs.scan_inputs(47, lens, 2, 6, 128, 128, init_state_std=0.02)
    o, hT = run_prefill(x, simt=simt)
    o_ref, h_ref = ref_prefill(x)
    assert_out_close(o, o_ref)
    assert_state_close(hT, h_ref)
    for n in (0, 2, 4):
        assert torch.equal(hT[n].cpu(), x["initial_state"][n])


@pytest.mark.parametrize("simt", [True, False])
def test_prefill_no_tokens_at_all(simt):
    """T = 0 with N = 2 sequences: nothing to scan; final states equal initial states."""
    x = inputs.scan_inputs(48, [0, 0], 2, 6, 128, 128, init_state_std=0.02)
    o, hT = run_prefill(x, simt=simt)
    assert o.shape[0] == 0
    assert torch.equal(hT.cpu(), x["initial_state"])


@pytest.mark.parametrize("case", ["beta0", "forget", "nodecay"])
def test_prefill_degenerate_gates(case):
    """The method's degenerate gates through the tensor-core path, against the oracle:
    beta = 0 (nothing is written, the state only decays: o_t = e^{gamma_t} q_t . S0),
    g = -30 at every token (the state forgets all but the newest write, so
    o_t = beta_t (k_t . q_t) v_t, with decays that underflow to exact zeros), and g = 0
    (no decay: the plain delta rule)."""
    lens = [130, 64, 1, 77]
    x = inputs.scan_inputs(61, lens, 2, 6, 128, 128, g_shift=-3.0, init_state_std=0.05)
    if case == "beta0":
        x["beta"] = torch.zeros_like(x["beta"])
    elif case == "forget":
        x["g"] = torch.full_like(x["g"], -30.0)
    else:
        x["g"] = torch.zeros_like(x["g"])
    o, hT = run_prefill(x)
    o_ref, h_ref = ref_prefill(x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all()
    assert_out_close(o, o_ref)
    assert_state_close(hT, h_ref)


def test_prefill_65535_sequences():
    """The most sequences one call takes (N = 65535, the state pass's grid limit), almost
    all empty: every empty sequence ends with its (zero) initial state exactly, and the
    40 non-empty ones, spread over the batch, match the oracle."""
    N = 65535
    rng = np.random.default_rng(62)
    lens = np.zeros(N, np.int64)
    busy = np.sort(rng.choice(N, 40, replace=False))
    lens[busy] = rng.integers(1, 140, 40)
    x = inputs.scan_inputs(62, lens.tolist(), 1, 1, 128, 128)
    o, hT = run_prefill(x)
    torch.cuda.synchronize()
    empty = torch.ones(N, dtype=torch.bool, device="cuda")
    empty[torch.from_numpy(busy).cuda()] = False
    assert int(torch.count_nonzero(hT[empty])) == 0
    # the oracle on the non-empty sequences alone: their tokens are the whole packed
    # batch, in the same order
    xb = dict(x)
    xb["cu_seqlens"] = torch.from_numpy(np.concatenate([[0], np.cumsum(lens[busy])]).astype(np.int32))
    o_ref, h_ref = ref_prefill(xb)
    assert_out_close(o, o_ref)
    assert_state_close(hT[torch.from_numpy(busy).cuda()], h_ref)


@pytest.mark.parametrize("simt", [True, False])
def test_prefill_weak_decay_long(simt):
    """g = -softplus(N(0,1) - 3): long memory, errors carried across many chunks."""
    x = inputs.scan_inputs(43, [777], 1, 3, 128, 128, g_shift=-3.0, init_state_std=0.02)
    o, hT = run_prefill(x, simt=simt)
    o_ref, h_ref = ref_prefill(x)
    assert_out_close(o, o_ref)
    assert_state_close(hT, h_ref)


@pytest.mark.parametrize("simt,lens", [(True, [130, 1, 64, 300, 17]),
                                       (False, [130, 1, 64, 300, 17]),
                                       # enough sequences that the batch runs the state
                                       # kernel with two dv tiles per head and each
                                       # sequence alone with three
                                       (False, [130, 1, 64, 300, 17, 65, 2, 200, 64, 9,
                                                128, 3, 70, 33])])
def test_prefill_batch_invariance_bits(simt, lens):
    x = inputs.scan_inputs(44, lens, 2, 4, 128, 128, init_state_std=0.02)
    o, hT = run_prefill(x, simt=simt)
    cu = x["cu_seqlens"]
    for n, L in enumerate(lens):
        s0, s1 = int(cu[n]), int(cu[n + 1])
        solo = {k: x[k][s0:s1] for k in ("q", "k", "v", "g", "beta")}
        solo["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int32)
        solo["initial_state"] = x["initial_state"][n:n + 1]
        o1, h1 = run_prefill(solo, simt=simt)
        assert_bits_equal(o[s0:s1], o1, "o of sequence %d" % n)
        assert_bits_equal(hT[n:n + 1], h1, "state of sequence %d" % n)


@pytest.mark.parametrize("N", [2, 256, 257])
def test_prefill_sequence_order_changes_no_bits(N):
    """The state pass takes up to 256 sequences longest first (a grid-order table built on
    the host) and more in batch order.  Either way every sequence's o and final state are
    the bits of the same sequence run alone, and reversing the batch changes nothing."""
    rng = np.random.default_rng(N)
    lens = [int(x) for x in rng.integers(1, 140, size=N)]
    lens[N // 2] = 400                      # the longest sits mid-batch
    lens[-1] = 260
    x = inputs.scan_inputs(47, lens, 2, 4, 128, 128, init_state_std=0.02)
    o, hT = run_prefill(x)
    cu = x["cu_seqlens"].numpy()
    rev = {}
    order = list(range(N))[::-1]
    for key in ("q", "k", "v", "g", "beta"):
        rev[key] = torch.cat([x[key][cu[n]:cu[n + 1]] for n in order])
    rev["cu_seqlens"] = torch.tensor(np.concatenate([[0], np.cumsum([lens[n] for n in order])]),
                                     dtype=torch.int32)
    rev["initial_state"] = x["initial_state"][order]
    o_r, h_r = run_prefill(rev)
    cu_r = rev["cu_seqlens"].numpy()
    for j, n in enumerate(order):
        assert_bits_equal(o_r[cu_r[j]:cu_r[j + 1]], o[cu[n]:cu[n + 1]], "o of sequence %d reversed" % n)
        assert_bits_equal(h_r[j:j + 1], hT[n:n + 1], "state of sequence %d reversed" % n)
    for n in sorted({0, 1, N // 2, N - 1} | set(int(i) for i in rng.integers(0, N, size=6))):
        s0, s1 = int(cu[n]), int(cu[n + 1])
        solo = {k: x[k][s0:s1] for k in ("q", "k", "v", "g", "beta")}
        solo["cu_seqlens"] = torch.tensor([0, lens[n]], dtype=torch.int32)
        solo["initial_state"] = x["initial_state"][n:n + 1]
        o1, h1 = run_prefill(solo)
        assert_bits_equal(o[s0:s1], o1, "o of sequence %d" % n)
        assert_bits_equal(hT[n:n + 1], h1, "state of sequence %d" % n)


@pytest.mark.parametrize("simt", [True, False])
def test_prefill_continuation_split_on_chunk_multiple_is_exact(simt):
    T, tau = 333, 128
    x = inputs.scan_inputs(45, [T], 2, 4, 128, 128, init_state_std=0.02)
    o, hT = run_prefill(x, simt=simt)
    a = {k: x[k][:tau] for k in ("q", "k", "v", "g", "beta")}
    a["cu_seqlens"] = torch.tensor([0, tau], dtype=torch.int32)
    a["initial_state"] = x["initial_state"]
    o1, h1 = run_prefill(a, simt=simt)
    b = {k: x[k][tau:] for k in ("q", "k", "v", "g", "beta")}
    b["cu_seqlens"] = torch.tensor([0, T - tau], dtype=torch.int32)
    b["initial_state"] = h1.cpu()
    o2, h2 = run_prefill(b, simt=simt)
    assert_bits_equal(torch.cat([o1, o2]), o, "continued o")
    assert_bits_equal(h2, hT, "continued state")


def test_prefill_rejects_head_first():
    x = cuda(inputs.scan_inputs(46, [12], 16, 32, 128, 128))
    hf = x["q"].transpose(0, 1).contiguous().transpose(0, 1)   # [T,H,D] view of [H,T,D]
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_prefill(hf, x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"])
    assert e.value.code == 3
    # a genuine 12-token prompt with 16/32 heads (T < H) is accepted
    o, _ = gdn.gdn_chunk_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"])
    assert torch.isfinite(o.float()).all()


def test_layer_prefill_27b_heads_sampled():
    """Conv over the packed 10240 q||k||v channels, then the scan with in-kernel L2 norm,
    at the 27B head shapes on a shorter packed batch; every v-head checked."""
    s = inputs.QWEN35_27B
    lens = [300, 65]
    C = inputs.conv_channels(**s)
    cv = inputs.conv_inputs(47, lens, C, with_state=True)
    rng = np.random.default_rng(48)
    T = sum(lens)
    g, beta = inputs.gates(rng, T, s["Hv"], 2.0)
    h0 = torch.randn(len(lens), s["Hv"], 128, 128, generator=torch.Generator().manual_seed(1)) * 0.02
    cu = cv["cu_seqlens"]
    o, hT, st = gdn.gdn_layer_prefill(cv["x"].cuda(), cv["w"].cuda(), None, g.cuda(),
                                      beta.cuda(), cu.cuda(), s["Hk"], s["Hv"], 128, 128,
                                      conv_state_in=cv["conv_state"].cuda(),
                                      initial_state=h0.cuda(), cu_seqlens_host=cu)
    heads = list(range(0, 48, 5)) + [47]
    o_ref, h_ref, st_ref = oracle.layer_prefill(cv["x"], cv["w"], None, g, beta, cu,
                                                s["Hk"], s["Hv"], 128, 128,
                                                conv_state=cv["conv_state"],
                                                initial_state=h0, v_heads=heads)
    assert_out_close(o[:, heads], o_ref)
    assert_state_close(hT[:, heads], h_ref)
    np.testing.assert_array_equal(np64(st), st_ref)


@pytest.mark.parametrize("l2norm,mode", [(True, "fused"), (False, "fused"), (True, "fused3"),
                                         (True, "side"), (False, "side"), (True, "separate")])
def test_layer_prefill_entry_equals_two_calls_bits(l2norm, mode):
    """gdn_layer_prefill gives exactly the bits of gdn_conv1d_fwd followed by
    gdn_chunk_prefill, for y, o, the final states and the conv states, on every path: the
    conv with the v channels on a caller's side stream overlapping the chunk preparation,
    everything on the current stream, and the v channels' conv fused into the state pass
    ("fused3" under the 48 + 48 + 32 column tiling).  The batch has an empty sequence and
    ones shorter than the conv window."""
    s = dict(Hk=2, Hv=6, dk=128, dv=128)
    C = inputs.conv_channels(**s)
    lens = [70, 1, 0, 129, 64, 2]
    cv = inputs.conv_inputs(81, lens, C, with_state=True, with_bias=True)
    x = inputs.scan_inputs(82, lens, s["Hk"], s["Hv"], 128, 128, init_state_std=0.02)
    args = [cv["x"].cuda(), cv["w"].cuda(), cv["bias"].cuda(), x["g"].cuda(),
            x["beta"].cuda(), cv["cu_seqlens"].cuda()]
    y1 = torch.empty_like(args[0])
    o1, h1, st1 = gdn.gdn_layer_prefill(*args, s["Hk"], s["Hv"], 128, 128,
                                        conv_state_in=cv["conv_state"].cuda(),
                                        initial_state=x["initial_state"].cuda(), l2norm=l2norm,
                                        scale=0.7, cu_seqlens_host=cv["cu_seqlens"], y=y1,
                                        fused_vconv=mode in ("fused", "fused3"),
                                        side_stream=torch.cuda.Stream() if mode == "side" else None,
                                        tiles=3 if mode == "fused3" else None)
    y, st2 = gdn.gdn_conv1d_fwd(args[0], args[1], args[2], args[5], cv["conv_state"].cuda(),
                                cu_seqlens_host=cv["cu_seqlens"])
    q, k, v = gdn.split_qkv(y, s["Hk"], s["Hv"], 128, 128)
    o2, h2 = gdn.gdn_chunk_prefill(q, k, v, args[3], args[4], args[5], l2norm=l2norm,
                                   scale=0.7, initial_state=x["initial_state"].cuda(),
                                   cu_seqlens_host=cv["cu_seqlens"])
    torch.cuda.synchronize()
    assert_bits_equal(y1, y, "conv output y")
    assert_bits_equal(o1, o2, "o")
    assert_bits_equal(h1, h2, "final state")
    assert_bits_equal(st1, st2, "conv state")


def test_layer_prefill_fused_conv_without_conv_state():
    """The fused v conv of fresh sequences (no conv state: zeros before each sequence,
    including one sequence's first chunk that follows another's tokens in the packed
    rows) against the oracle layer, every v-head."""
    s = dict(Hk=2, Hv=6, dk=128, dv=128)
    C = inputs.conv_channels(**s)
    lens = [130, 3, 64, 65]
    cv = inputs.conv_inputs(83, lens, C, with_state=False, with_bias=True)
    rng = np.random.default_rng(84)
    T = sum(lens)
    g, beta = inputs.gates(rng, T, s["Hv"], 2.0)
    cu = cv["cu_seqlens"]
    y = torch.empty_like(cv["x"]).cuda()
    o, hT, st = gdn.gdn_layer_prefill(cv["x"].cuda(), cv["w"].cuda(), cv["bias"].cuda(),
                                      g.cuda(), beta.cuda(), cu.cuda(), s["Hk"], s["Hv"], 128,
                                      128, y=y, cu_seqlens_host=cu, fused_vconv=True)
    o_ref, h_ref, st_ref = oracle.layer_prefill(cv["x"], cv["w"], cv["bias"], g, beta, cu,
                                                s["Hk"], s["Hv"], 128, 128)
    assert_out_close(o, o_ref)
    assert_state_close(hT, h_ref)
    np.testing.assert_array_equal(np64(st), st_ref)
    y_ref, _ = oracle.conv1d_varlen(cv["x"], cv["w"], cv["bias"], cu)
    assert_out_close(y, y_ref, what="conv output y")


@pytest.mark.parametrize("l2norm", [False, True])
def test_prefill_dv_tilings_give_identical_bits(l2norm):
    """The state pass groups each head's 128 dv columns into two tiles of 64 or three of
    48 + 48 + 32 (chosen from N and the SM count).  The same batch run under both tilings,
    forced by flag, gives the same bits for o and the final states, and the oracle
    agrees with both."""
    lens = [130, 1, 64, 300, 17, 65]
    x = inputs.scan_inputs(51, lens, 2, 6, 128, 128, normalise_qk=not l2norm,
                           init_state_std=0.02)
    xg = cuda(x)
    outs = []
    for tiles in (2, 3):
        o, hT = gdn.gdn_chunk_prefill(xg["q"], xg["k"], xg["v"], xg["g"], xg["beta"],
                                      xg["cu_seqlens"], l2norm=l2norm,
                                      initial_state=xg["initial_state"],
                                      cu_seqlens_host=x["cu_seqlens"], tiles=tiles)
        outs.append((o, hT))
    assert_bits_equal(outs[0][0], outs[1][0], "o, two vs three dv tiles")
    assert_bits_equal(outs[0][1], outs[1][1], "final state, two vs three dv tiles")
    o_ref, h_ref = ref_prefill(x, l2norm=l2norm)
    assert_out_close(outs[0][0], o_ref)
    assert_state_close(outs[0][1], h_ref)
