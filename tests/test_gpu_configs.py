"""GPU parity and batch invariance at the full sizes of the named workloads.

* 27B varlen layer: 8 packed sequences (lengths U[1, 8192], ~32k tokens) with random
  initial states and conv states; conv + scan on the GPU; the oracle recomputes a
  sample of v-heads over every sequence.
* 27B decode: 256 sequences on a [256, 48, 128, 128] fp32 pool with a permuted index;
  the oracle recomputes a sample of sequences (all heads); every slot is checked to be
  written once.
* 4B batch-invariance mix: 20 fresh prefills (U[12, 32768]), 20 chunked-prefill
  continuations of 2048 tokens on random states, 20 single-token decodes; every
  sequence's outputs and states must be bit-identical to running it alone, and a
  seeded subset of 6 (2 of each kind) is checked against the oracle on sampled heads.

Tolerances: tests/gpu_util.py.
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


def test_varlen_27b_layer_full_size_sampled_heads():
    s = inputs.QWEN35_27B
    d = inputs.varlen_27b(seed=3)
    cv = d["conv"]
    cu = d["cu_seqlens"]
    T = int(cu[-1])
    assert len(d["lens"]) == 8 and T == sum(d["lens"])
    o, hT, st = gdn.gdn_layer_prefill(cv["x"].cuda(), cv["w"].cuda(), None, d["g"].cuda(),
                                      d["beta"].cuda(), cu.cuda(), s["Hk"], s["Hv"], 128, 128,
                                      conv_state_in=cv["conv_state"].cuda(),
                                      initial_state=d["initial_state"].cuda(),
                                      cu_seqlens_host=cu)
    torch.cuda.synchronize()
    heads = [0, 23, 47]
    o_ref, h_ref, st_ref = oracle.layer_prefill(cv["x"], cv["w"], None, d["g"], d["beta"], cu,
                                                s["Hk"], s["Hv"], 128, 128,
                                                conv_state=cv["conv_state"],
                                                initial_state=d["initial_state"],
                                                v_heads=heads)
    assert_out_close(o[:, heads], o_ref)
    assert_state_close(hT[:, heads], h_ref)
    np.testing.assert_array_equal(np64(st), st_ref)


def test_decode_27b_full_pool_sampled_sequences():
    s = inputs.QWEN35_27B
    d = inputs.decode_27b(seed=4, N=256)
    pool0 = d["state_pool"]
    pool = pool0.cuda()
    idx = d["state_idx"]
    cv = d["conv"]
    cstate = cv["conv_state"].cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    w = cv["w"].cuda()
    o = gdn.gdn_layer_decode(cv["x"].cuda(), w, None, d["g"].cuda(), d["beta"].cuda(), cstate,
                             pool, s["Hk"], s["Hv"], 128, 128, state_idx=idx.cuda(),
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # conv update: every sequence, against the oracle
    y_ref, cs_ref = oracle.conv1d_update(cv["x"], cv["w"], None, cv["conv_state"], idx)
    np.testing.assert_array_equal(np64(cstate), cs_ref)
    # scan: a sample of sequences, every head, on the bf16 conv outputs the oracle makes
    sample = [0, 1, 77, 128, 200, 255]
    yb = oracle.round_to_bf16(y_ref[sample])
    q, k, v = oracle.split_qkv(yb, s["Hk"], s["Hv"], 128, 128)
    sidx = idx[sample].numpy()
    o_ref, h_ref = oracle.recurrent_decode(q, k, v, d["g"][sample], d["beta"][sample],
                                           pool0[sidx], None, l2norm=True)
    assert_out_close(o[sample], o_ref)
    assert_state_close(pool[torch.from_numpy(sidx).long()], h_ref)
    # the permutation covers the pool: every slot changed exactly once
    changed = (pool.cpu() != pool0).flatten(1).any(1)
    assert bool(changed.all())


def _mix_batch(seed=5):
    s = inputs.QWEN35_4B
    fresh, cont, dec = inputs.mix_lengths(seed)
    lens = fresh + cont
    x = inputs.scan_inputs(seed, lens, s["Hk"], s["Hv"], 128, 128, init_state_std=0.02)
    x["initial_state"][: len(fresh)] = 0.0          # fresh prefills start from zero
    d = inputs.scan_inputs(seed + 1, [1] * len(dec), s["Hk"], s["Hv"], 128, 128)
    pool = torch.randn(len(dec), s["Hv"], 128, 128,
                       generator=torch.Generator().manual_seed(seed)) * 0.02
    return s, fresh, cont, x, d, pool


def test_mix_4b_batch_invariance_bits_and_oracle_subset():
    s, fresh, cont, x, d, pool = _mix_batch()
    cu = x["cu_seqlens"]
    N = len(fresh) + len(cont)
    xg = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    # the whole prefill batch in one call, in a shuffled order of sequences
    perm = np.random.default_rng(9).permutation(N)
    cu_np = cu.numpy().astype(np.int64)
    tok_p = np.concatenate([np.arange(cu_np[i], cu_np[i + 1]) for i in perm])
    cu_p = np.zeros(N + 1, np.int32)
    cu_p[1:] = np.cumsum([int(cu[i + 1] - cu[i]) for i in perm])
    tp = torch.from_numpy(tok_p).cuda()
    o_b, h_b = gdn.gdn_chunk_prefill(xg["q"][tp], xg["k"][tp], xg["v"][tp], xg["g"][tp],
                                     xg["beta"][tp], torch.from_numpy(cu_p).cuda(),
                                     initial_state=xg["initial_state"][torch.from_numpy(perm).cuda()],
                                     cu_seqlens_host=torch.from_numpy(cu_p))
    for j, i in enumerate(perm):
        a, b = int(cu[i]), int(cu[i + 1])
        o1, h1 = gdn.gdn_chunk_prefill(xg["q"][a:b], xg["k"][a:b], xg["v"][a:b],
                                       xg["g"][a:b], xg["beta"][a:b],
                                       torch.tensor([0, b - a], dtype=torch.int32).cuda(),
                                       initial_state=xg["initial_state"][i:i + 1],
                                       cu_seqlens_host=torch.tensor([0, b - a], dtype=torch.int32))
        pa, pb = int(cu_p[j]), int(cu_p[j + 1])
        assert_bits_equal(o_b[pa:pb], o1, "prefill o of sequence %d" % i)
        assert_bits_equal(h_b[j:j + 1], h1, "prefill state of sequence %d" % i)
    # decodes: the batch of 20 against 20 single-sequence calls
    dg = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    pool_b = pool.cuda()
    o_d = gdn.gdn_recurrent_decode(dg["q"], dg["k"], dg["v"], dg["g"], dg["beta"], pool_b)
    for n in range(pool.shape[0]):
        p1 = pool[n:n + 1].cuda()
        o1 = gdn.gdn_recurrent_decode(dg["q"][n:n + 1], dg["k"][n:n + 1], dg["v"][n:n + 1],
                                      dg["g"][n:n + 1], dg["beta"][n:n + 1], p1)
        assert_bits_equal(o_d[n:n + 1], o1, "decode o of sequence %d" % n)
        assert_bits_equal(pool_b[n:n + 1], p1, "decode state of sequence %d" % n)
    # oracle on a seeded subset: 2 fresh, 2 continuations (sampled heads), 2 decodes
    rng = np.random.default_rng(10)
    pick = list(rng.choice(len(fresh), 2, replace=False)) + \
        list(len(fresh) + rng.choice(len(cont), 2, replace=False))
    heads, kheads = [0, 31], [0, 31 // (s["Hv"] // s["Hk"])]
    for i in pick:
        a, b = int(cu[i]), int(cu[i + 1])
        j = int(np.where(perm == i)[0][0])
        pa, pb = int(cu_p[j]), int(cu_p[j + 1])
        o_r, h_r = oracle.gated_delta_rule(
            x["q"][a:b][:, kheads], x["k"][a:b][:, kheads], x["v"][a:b][:, heads],
            x["g"][a:b][:, heads], x["beta"][a:b][:, heads], [0, b - a],
            initial_state=x["initial_state"][i:i + 1][:, heads])
        assert_out_close(o_b[pa:pb][:, heads], o_r, what="mix o of sequence %d" % i)
        assert_state_close(h_b[j:j + 1][:, heads], h_r, what="mix state of sequence %d" % i)
    o_r, pool_r = oracle.recurrent_decode(d["q"][:2], d["k"][:2], d["v"][:2], d["g"][:2],
                                          d["beta"][:2], pool[:2])
    assert_out_close(o_d[:2], o_r, what="mix decode o")
    assert_state_close(pool_b[:2], pool_r, what="mix decode state")
