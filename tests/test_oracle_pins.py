"""Pins for the fp64 oracle, checked against what the pages and the mathematics fix.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a wrong sign,
a transposed state, decay and delta swapped, output read before the update, a wrong
GQA head map, an off-by-one conv tap) fails at least one of them.  No GPU is needed.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle.chunked import chunked_gated_delta_rule

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(seed, lens, Hk, Hv, dk, dv, unit_k=False, g_scale=1.0, with_h0=True):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    q = rng.standard_normal((T, Hk, dk))
    k = rng.standard_normal((T, Hk, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, dv))
    g = -np.logaddexp(0, rng.standard_normal((T, Hv))) * g_scale
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, Hv))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    h0 = rng.standard_normal((len(lens), Hv, dk, dv)) * 0.3 if with_h0 else None
    return q, k, v, g, beta, cu, h0


def brute_force(q, k, v, g, beta, cu, h0, scale, l2norm):
    """Dense matrix form S_t = e^g S (I - b k k^T) + b v k^T, o_t = scale S_t q_t."""
    T, Hk, dk = q.shape
    _, Hv, dv = v.shape
    G = Hv // Hk
    N = len(cu) - 1
    o = np.zeros((T, Hv, dv))
    hT = np.zeros((N, Hv, dk, dv))
    for n in range(N):
        for hv in range(Hv):
            S = np.zeros((dv, dk)) if h0 is None else h0[n, hv].T.copy()
            for t in range(cu[n], cu[n + 1]):
                kk = k[t, hv // G].copy()
                qq = q[t, hv // G].copy()
                if l2norm:
                    kk /= np.sqrt(kk @ kk + oracle.L2NORM_EPS)
                    qq /= np.sqrt(qq @ qq + oracle.L2NORM_EPS)
                P = np.eye(dk) - beta[t, hv] * np.outer(kk, kk)
                S = np.exp(g[t, hv]) * S @ P + beta[t, hv] * np.outer(v[t, hv], kk)
                o[t, hv] = scale * S @ qq
            hT[n, hv] = S.T
    return o, hT


@pytest.mark.parametrize("l2norm", [False, True])
def test_bruteforce_dense_matrix_form(l2norm):
    case = rand_case(0, [5, 1, 9], 2, 4, 6, 3)
    o, hT = oracle.gated_delta_rule(*case[:6], scale=0.7, l2norm=l2norm,
                                    initial_state=case[6], nthreads=3)
    ob, hb = brute_force(*case, scale=0.7, l2norm=l2norm)
    np.testing.assert_allclose(o, ob, atol=1e-12, rtol=0)
    np.testing.assert_allclose(hT, hb, atol=1e-12, rtol=0)


def test_empty_sequences_in_a_packed_batch():
    """Zero-length sequences between others: each keeps its initial state and its conv
    state exactly, and the neighbours equal the dense brute force, whose loop over an
    empty range does nothing; the chunked form agrees."""
    lens = [0, 5, 0, 9, 0]
    case = rand_case(12, lens, 1, 2, 6, 4)
    o, hT = oracle.gated_delta_rule(*case[:6], scale=0.9, initial_state=case[6])
    ob, hb = brute_force(*case, scale=0.9, l2norm=False)
    np.testing.assert_allclose(o, ob, atol=1e-12, rtol=0)
    np.testing.assert_allclose(hT, hb, atol=1e-12, rtol=0)
    for n in (0, 2, 4):
        np.testing.assert_array_equal(hT[n], case[6][n])
    oc, hc = chunked_gated_delta_rule(*case[:6], chunk=16, scale=0.9,
                                      initial_state=case[6])
    np.testing.assert_allclose(oc, o, atol=1e-10, rtol=0)
    np.testing.assert_allclose(hc, hT, atol=1e-10, rtol=0)
    rng = np.random.default_rng(13)
    C = 6
    x = rng.standard_normal((sum(lens), C))
    w = rng.uniform(-0.5, 0.5, (C, 4))
    s0 = rng.standard_normal((len(lens), 3, C))
    _, s1 = oracle.conv1d_varlen(x, w, None, case[5], s0)
    for n in (0, 2, 4):
        np.testing.assert_array_equal(s1[n], s0[n])


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_example.json")) as f:
        ex = json.load(f)
    o, hT = oracle.gated_delta_rule(
        np.array(ex["q"]), np.array(ex["k"]), np.array(ex["v"]), np.array(ex["g"]),
        np.array(ex["beta"]), np.array(ex["cu_seqlens"]),
        initial_state=np.array(ex["initial_state"]))
    np.testing.assert_allclose(o, np.array(ex["expected_o"]), atol=1e-14)
    np.testing.assert_allclose(hT, np.array(ex["expected_final_state"]), atol=1e-14)


def test_beta_zero_closed_form():
    q, k, v, g, beta, cu, h0 = rand_case(1, [7, 4], 1, 2, 5, 4)
    beta[:] = 0.0
    o, hT = oracle.gated_delta_rule(q, k, v, g, beta, cu, initial_state=h0)
    for n in range(2):
        for hv in range(2):
            G = np.cumsum(g[cu[n]:cu[n + 1], hv])
            for i, t in enumerate(range(cu[n], cu[n + 1])):
                expect = np.exp(G[i]) * (h0[n, hv].T @ q[t, 0])
                np.testing.assert_allclose(o[t, hv], expect, atol=1e-13)
            np.testing.assert_allclose(hT[n, hv], np.exp(G[-1]) * h0[n, hv], atol=1e-13)


def test_store_then_retrieve_orthonormal_keys():
    dk, dv, m = 8, 5, 6
    rng = np.random.default_rng(2)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm[:, :m].T                                # m orthonormal keys
    vals = rng.standard_normal((m, dv))
    v_new = rng.standard_normal(dv)
    # writes of (k_i, v_i), then the overwrite of key 2 with v_new, then m reads
    T = m + 1 + m
    q = rng.standard_normal((T, 1, dk))
    k = np.zeros((T, 1, dk))
    v = np.zeros((T, 1, dv))
    beta = np.zeros((T, 1))
    k[:m, 0] = keys
    v[:m, 0] = vals
    beta[:m] = 1.0
    k[m, 0], v[m, 0], beta[m] = keys[2], v_new, 1.0
    q[m + 1:, 0] = keys
    g = np.zeros((T, 1))
    o, hT = oracle.gated_delta_rule(q, k, v, g, beta, [0, T])
    expect = vals.copy()
    expect[2] = v_new                                  # delta rule replaces, not adds
    np.testing.assert_allclose(o[m + 1:, 0], expect, atol=1e-12)
    # the state is exactly sum_i v_i k_i^T in [dk][dv] layout
    np.testing.assert_allclose(hT[0, 0], keys.T @ expect, atol=1e-12)


def test_forget_all_limit():
    q, k, v, g, beta, cu, h0 = rand_case(3, [6], 1, 1, 4, 3)
    g[:] = -1.0e4                                      # exp(g) == 0.0 in fp64
    o, hT = oracle.gated_delta_rule(q, k, v, g, beta, cu, scale=1.3, initial_state=h0)
    for t in range(6):
        expect = 1.3 * beta[t, 0] * (k[t, 0] @ q[t, 0]) * v[t, 0]
        np.testing.assert_allclose(o[t, 0], expect, atol=1e-13)
    np.testing.assert_allclose(hT[0, 0], beta[5, 0] * np.outer(k[5, 0], v[5, 0]),
                               atol=1e-13)


@pytest.mark.parametrize("chunk", [16, 64])
@pytest.mark.parametrize("l2norm", [False, True])
def test_chunked_equals_recurrent(chunk, l2norm):
    lens = [1, 16, 37, 64, 130]
    q, k, v, g, beta, cu, h0 = rand_case(4, lens, 2, 4, 16, 8)
    o, hT = oracle.gated_delta_rule(q, k, v, g, beta, cu, scale=0.5, l2norm=l2norm,
                                    initial_state=h0)
    oc, hc = chunked_gated_delta_rule(q, k, v, g, beta, cu, chunk=chunk, scale=0.5,
                                      l2norm=l2norm, initial_state=h0)
    np.testing.assert_allclose(oc, o, atol=1e-10, rtol=0)
    np.testing.assert_allclose(hc, hT, atol=1e-10, rtol=0)


def test_chunked_strong_decay_no_overflow():
    """g ~ -softplus(N(0,1)+2) over 64 tokens: gamma reaches ~-136, exp(-gamma) would
    overflow; only exp(gamma_r - gamma_s) with s <= r may be formed."""
    q, k, v, g, beta, cu, h0 = rand_case(5, [64, 200], 1, 1, 16, 16, unit_k=True)
    g = -np.logaddexp(0, np.random.default_rng(9).standard_normal(g.shape) + 2.0) * 3
    o, hT = oracle.gated_delta_rule(q, k, v, g, beta, cu, initial_state=h0)
    oc, hc = chunked_gated_delta_rule(q, k, v, g, beta, cu, chunk=64, initial_state=h0)
    assert np.isfinite(oc).all() and np.isfinite(hc).all()
    np.testing.assert_allclose(oc, o, atol=1e-10)
    np.testing.assert_allclose(hc, hT, atol=1e-10)


def test_gqa_head_map_contiguous_groups():
    q, k, v, g, beta, cu, h0 = rand_case(6, [9], 2, 6, 4, 3)
    o, hT = oracle.gated_delta_rule(q, k, v, g, beta, cu, initial_state=h0)
    for hv in range(6):
        hk = hv // 3
        o1, h1 = oracle.gated_delta_rule(q[:, hk:hk + 1], k[:, hk:hk + 1],
                                         v[:, hv:hv + 1], g[:, hv:hv + 1],
                                         beta[:, hv:hv + 1], cu,
                                         initial_state=h0[:, hv:hv + 1])
        np.testing.assert_array_equal(o[:, hv:hv + 1], o1)
        np.testing.assert_array_equal(hT[:, hv:hv + 1], h1)


def test_split_and_carry_invariance():
    """Running [0,T) equals [0,tau) then [tau,T) with recurrent state and conv tail
    carried (the chunked-prefill continuation of the batch-invariance PR, part 3(a))."""
    rng = np.random.default_rng(7)
    T, C, tau = 23, 10, 9
    x = rng.standard_normal((T, C))
    w = rng.uniform(-0.5, 0.5, (C, 4))
    b = rng.uniform(-0.5, 0.5, C)
    s0 = rng.standard_normal((1, 3, C))
    y, s_full = oracle.conv1d_varlen(x, w, b, [0, T], s0)
    y1, s_mid = oracle.conv1d_varlen(x[:tau], w, b, [0, tau], s0)
    y2, s_end = oracle.conv1d_varlen(x[tau:], w, b, [0, T - tau], s_mid)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, atol=1e-14)
    np.testing.assert_allclose(s_end, s_full, atol=0)
    q, k, v, g, beta, cu, h0 = rand_case(8, [T], 1, 2, 5, 4)
    o, hT = oracle.gated_delta_rule(q, k, v, g, beta, cu, initial_state=h0)
    o1, hm = oracle.gated_delta_rule(q[:tau], k[:tau], v[:tau], g[:tau], beta[:tau],
                                     [0, tau], initial_state=h0)
    o2, he = oracle.gated_delta_rule(q[tau:], k[tau:], v[tau:], g[tau:], beta[tau:],
                                     [0, T - tau], initial_state=hm)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, atol=1e-12)
    np.testing.assert_allclose(he, hT, atol=1e-12)


def test_range_end_state_is_affine_in_start_state():
    """The context-parallel scan's composition: each token's update
    h <- e^g (I - beta k k^T) h + beta k v^T is affine in the [dk][dv] state, so a range's
    end state is P h_start + R, with P the end state from the identity with V = 0 and R
    the end state from zero; two ranges compose as P2 (P1 S + R1) + R2.  Checked on the
    recurrence itself (the batch-invariance PR's use_cp commit names the variant)."""
    dk = dv = 6
    q, k, v, g, beta, cu, h0 = rand_case(31, [17, 11], 1, 2, dk, dv, unit_k=True)
    N, Hv = 2, 2
    eye = np.broadcast_to(np.eye(dk), (N, Hv, dk, dk)).copy()
    _, P = oracle.gated_delta_rule(q, k, np.zeros_like(v), g, beta, cu, initial_state=eye)
    _, R = oracle.gated_delta_rule(q, k, v, g, beta, cu, initial_state=np.zeros_like(h0))
    _, hT = oracle.gated_delta_rule(q, k, v, g, beta, cu, initial_state=h0)
    np.testing.assert_allclose(hT, np.einsum("nhik,nhkj->nhij", P, h0) + R, atol=1e-12)
    # two ranges of the first sequence, [0, 7) and [7, 17), composed
    tau = 7
    sl = lambda a, lo, hi: a[lo:hi]  # noqa: E731
    parts = []
    for lo, hi in ((0, tau), (tau, 17)):
        args = [sl(a, lo, hi) for a in (q, k, v, g, beta)]
        _, Pr = oracle.gated_delta_rule(args[0], args[1], np.zeros_like(args[2]), args[3],
                                        args[4], [0, hi - lo], initial_state=eye[:1])
        _, Rr = oracle.gated_delta_rule(*args, [0, hi - lo],
                                        initial_state=np.zeros_like(h0[:1]))
        parts.append((Pr, Rr))
    S = h0[:1]
    for Pr, Rr in parts:
        S = np.einsum("nhik,nhkj->nhij", Pr, S) + Rr
    np.testing.assert_allclose(S, hT[:1], atol=1e-12)


def test_contraction_bound():
    """Unit k, beta in (0,1], g <= 0: ||I - beta k k^T||_2 = 1, so
    ||S_t||_2 <= e^{g_t} ||S_{t-1}||_2 + beta_t ||v_t||."""
    q, k, v, g, beta, cu, h0 = rand_case(9, [40], 1, 1, 6, 5, unit_k=True)
    h = h0
    for t in range(40):
        _, hn = oracle.gated_delta_rule(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                        beta[t:t + 1], [0, 1], initial_state=h)
        lhs = np.linalg.norm(hn[0, 0], 2)
        rhs = np.exp(g[t, 0]) * np.linalg.norm(h[0, 0], 2) + beta[t, 0] * np.linalg.norm(v[t, 0])
        assert lhs <= rhs + 1e-12
        h = hn


def test_conv_matches_torch_conv1d_fp64():
    rng = np.random.default_rng(10)
    lens = [1, 2, 3, 17]
    C = 12
    T = sum(lens)
    x = rng.standard_normal((T, C))
    w = rng.uniform(-0.5, 0.5, (C, 4))
    b = rng.uniform(-0.5, 0.5, C)
    st = rng.standard_normal((len(lens), 3, C))
    cu = np.concatenate([[0], np.cumsum(lens)])
    y, s_out = oracle.conv1d_varlen(x, w, b, cu, st)
    for n, L in enumerate(lens):
        seg = np.concatenate([st[n], x[cu[n]:cu[n + 1]]])          # [L+3, C]
        inp = torch.from_numpy(seg.T[None])                        # [1, C, L+3]
        ref = F.conv1d(inp, torch.from_numpy(w[:, None, :]), torch.from_numpy(b),
                       padding=0, groups=C)
        ref = F.silu(ref[..., -L:])[0].T.numpy()
        np.testing.assert_allclose(y[cu[n]:cu[n + 1]], ref, atol=1e-13)
        np.testing.assert_array_equal(s_out[n], seg[-3:])


def test_conv_tap_closed_forms():
    rng = np.random.default_rng(11)
    T, C = 7, 3
    x = rng.standard_normal((T, C))
    st = rng.standard_normal((1, 3, C))
    w = np.zeros((C, 4))
    w[:, 3] = 1.0                                       # current token only
    y, _ = oracle.conv1d_varlen(x, w, None, [0, T], st)
    np.testing.assert_allclose(y, x / (1 + np.exp(-x)), atol=1e-15)
    w = np.zeros((C, 4))
    w[:, 0] = 1.0                                       # token t-3 (state for t<3)
    y, _ = oracle.conv1d_varlen(x, w, None, [0, T], st)
    prev = np.concatenate([st[0], x])[:T]
    np.testing.assert_allclose(y, prev / (1 + np.exp(-prev)), atol=1e-15)
    y, _ = oracle.conv1d_varlen(x, w, None, [0, T], None)  # fresh: zeros in front
    prev = np.concatenate([np.zeros((3, C)), x])[:T]
    np.testing.assert_allclose(y, prev / (1 + np.exp(-prev)), atol=1e-15)


def test_decode_helpers_match_one_token_sequences():
    rng = np.random.default_rng(12)
    N, P, Hk, Hv, dk, dv = 4, 6, 1, 2, 4, 3
    q, k, v, g, beta, cu, _ = rand_case(13, [1] * N, Hk, Hv, dk, dv)
    pool = rng.standard_normal((P, Hv, dk, dv))
    idx = np.array([5, 0, 3, 2], np.int32)
    o, newpool = oracle.recurrent_decode(q, k, v, g, beta, pool, idx, scale=0.9)
    for n in range(N):
        o1, h1 = oracle.gated_delta_rule(q[n:n + 1], k[n:n + 1], v[n:n + 1], g[n:n + 1],
                                         beta[n:n + 1], [0, 1], scale=0.9,
                                         initial_state=pool[idx[n]][None])
        np.testing.assert_array_equal(o[n], o1[0])
        np.testing.assert_array_equal(newpool[idx[n]], h1[0])
    untouched = [p for p in range(P) if p not in idx]
    np.testing.assert_array_equal(newpool[untouched], pool[untouched])
    C = 5
    x = rng.standard_normal((N, C))
    w = rng.uniform(-0.5, 0.5, (C, 4))
    cpool = rng.standard_normal((P, 3, C))
    y, cnew = oracle.conv1d_update(x, w, None, cpool, idx)
    for n in range(N):
        s = cpool[idx[n]]
        z = (w * np.concatenate([s, x[n:n + 1]]).T).sum(1)
        np.testing.assert_allclose(y[n], z / (1 + np.exp(-z)), atol=1e-14)
        np.testing.assert_array_equal(cnew[idx[n]], np.concatenate([s[1:], x[n:n + 1]]))


def test_thread_count_does_not_change_result():
    case = rand_case(14, [33, 2, 70], 2, 4, 8, 8)
    a = oracle.gated_delta_rule(*case[:6], initial_state=case[6], nthreads=1)
    b = oracle.gated_delta_rule(*case[:6], initial_state=case[6], nthreads=5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------------- fused decode gates

def test_gate_functions_closed_forms():
    """sigmoid and softplus against values the mathematics fixes: sigmoid(0) = 1/2 with
    slope 1/4, sigmoid(x) + sigmoid(-x) = 1; softplus(0) = ln 2 with slope 1/2,
    softplus(x) - softplus(-x) = x, softplus(x) -> x for large x and e^x for very
    negative x; and e^{-softplus(a)} = sigmoid(-a).  A wrong sign, a missing log or a
    scaled argument fails one of these."""
    x = np.linspace(-30.0, 30.0, 121)
    s = oracle.sigmoid(x)
    assert abs(oracle.sigmoid(np.array([0.0]))[0] - 0.5) < 1e-15
    h = 1e-6
    slope = (oracle.sigmoid(np.array([h]))[0] - oracle.sigmoid(np.array([-h]))[0]) / (2 * h)
    assert abs(slope - 0.25) < 1e-9
    np.testing.assert_allclose(s + oracle.sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    assert np.all(np.diff(s) > 0)
    sp = oracle.softplus(x)
    assert abs(oracle.softplus(np.array([0.0]))[0] - np.log(2.0)) < 1e-15
    slope = (oracle.softplus(np.array([h]))[0] - oracle.softplus(np.array([-h]))[0]) / (2 * h)
    assert abs(slope - 0.5) < 1e-9
    np.testing.assert_allclose(sp - oracle.softplus(-x), x, rtol=0, atol=1e-12)
    assert abs(oracle.softplus(np.array([50.0]))[0] - 50.0) < 1e-20
    assert abs(oracle.softplus(np.array([-50.0]))[0] / np.exp(-50.0) - 1.0) < 1e-12
    np.testing.assert_allclose(np.exp(-sp), oracle.sigmoid(-x), rtol=1e-13, atol=0)
    g, beta = oracle.gates_from_logits(np.array([[0.0, 3.0]]), np.array([[0.0, -3.0]]))
    np.testing.assert_allclose(g, -np.log1p(np.exp([[0.0, 3.0]])), rtol=1e-15)
    np.testing.assert_allclose(beta, [[0.5, 1.0 / (1.0 + np.exp(3.0))]], rtol=1e-15)


def test_fused_decode_equals_one_token_layer_prefill():
    """The fused decode oracle from raw logits equals, per sequence, the prefill-layer
    oracle (conv over [conv state ; x] + token recurrence, an independent code path) run
    on a one-token sequence from the same conv state and recurrent state, with the gates
    of the logits.  Catches a slip in the channel split, the pool indexing or the gates."""
    rng = np.random.default_rng(41)
    N, P, Hk, Hv, d = 3, 5, 2, 4, 8
    C = 2 * Hk * d + Hv * d
    x = rng.standard_normal((N, C))
    w = rng.uniform(-0.5, 0.5, (C, 4))
    bias = rng.uniform(-0.5, 0.5, (C,))
    conv_pool = rng.standard_normal((P, 3, C))
    pool = rng.standard_normal((P, Hv, d, d)) * 0.3
    a_raw = rng.standard_normal((N, Hv)) + 1.0
    b_raw = rng.standard_normal((N, Hv))
    idx = np.array([4, 0, 2], np.int32)
    o, conv_new, pool_new = oracle.fused_decode(x, w, bias, a_raw, b_raw, conv_pool, pool,
                                                Hk, Hv, d, d, state_idx=idx, scale=0.5,
                                                l2norm=True)
    g, beta = oracle.gates_from_logits(a_raw, b_raw)
    for n in range(N):
        s = idx[n]
        o1, h1, c1 = oracle.layer_prefill(x[n:n + 1], w, bias, g[n:n + 1], beta[n:n + 1],
                                          np.array([0, 1], np.int32), Hk, Hv, d, d,
                                          conv_state=conv_pool[s:s + 1],
                                          initial_state=pool[s:s + 1], scale=0.5,
                                          l2norm=True)
        np.testing.assert_allclose(o[n], o1[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(pool_new[s], h1[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(conv_new[s], c1[0])
    untouched = [s for s in range(P) if s not in set(idx.tolist())]
    np.testing.assert_array_equal(pool_new[untouched], pool[untouched])
    np.testing.assert_array_equal(conv_new[untouched], conv_pool[untouched])


# ------------------------------------------------------------- layer helpers

def test_split_qkv_channel_order_hand_example():
    """The packed conv output is q || k || v along channels, head by head, as the
    hand-built fixture lays out from the batch-invariance PR's mixed_qkv split; the same
    split through torch.split + view (an independent route) agrees on a larger case."""
    with open(os.path.join(GOLDEN, "qkv_channel_split.json")) as f:
        ex = json.load(f)
    q, k, v = oracle.split_qkv(np.array(ex["y"], np.float64), ex["Hk"], ex["Hv"], ex["dk"],
                               ex["dv"])
    np.testing.assert_array_equal(q, np.array(ex["expected_q"]))
    np.testing.assert_array_equal(k, np.array(ex["expected_k"]))
    np.testing.assert_array_equal(v, np.array(ex["expected_v"]))
    Hk, Hv, dk, dv, T = 2, 6, 4, 3, 5
    y = np.arange(T * (2 * Hk * dk + Hv * dv), dtype=np.float64).reshape(T, -1)
    qt, kt, vt = torch.split(torch.from_numpy(y), [Hk * dk, Hk * dk, Hv * dv], dim=-1)
    q, k, v = oracle.split_qkv(y, Hk, Hv, dk, dv)
    np.testing.assert_array_equal(q, qt.reshape(T, Hk, dk).numpy())
    np.testing.assert_array_equal(k, kt.reshape(T, Hk, dk).numpy())
    np.testing.assert_array_equal(v, vt.reshape(T, Hv, dv).numpy())


def _bf16_rne_bits(x32):
    """Round-to-nearest-even of fp32 bit patterns to bf16 by integer arithmetic on the
    bits (add 0x7FFF plus the lowest kept bit, then clear the 16 dropped bits)."""
    u = x32.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def test_round_to_bf16_nearest_even():
    """Hand-picked ties and near-ties (every input exact in fp32): a tie goes to the even
    8-bit mantissa, anything past the tie rounds away; fp64 inputs are first rounded to
    fp32 (the GPU conv's accumulation type), then to bf16.  A random sample agrees bit
    for bit with the integer form of round-to-nearest-even."""
    e = 2.0 ** -8
    cases = [(1.0, 1.0), (1 + e, 1.0), (1 + 3 * e, 1 + 4 * e), (1 + e + 2.0 ** -23, 1 + 2 * e),
             (1 + e - 2.0 ** -23, 1.0), (-(1 + 3 * e), -(1 + 4 * e)), (3.0, 3.0),
             (2.0 ** -130, 2.0 ** -130), (0.0, 0.0), (1 + e + 2.0 ** -30, 1.0)]
    got = oracle.round_to_bf16(np.array([c[0] for c in cases]))
    np.testing.assert_array_equal(got, np.array([c[1] for c in cases]))
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    np.testing.assert_array_equal(oracle.round_to_bf16(x.astype(np.float64)), _bf16_rne_bits(x))


def test_layer_prefill_v_heads_subset_equals_full_call():
    """The v_heads branch of the layer oracle (one call per requested v-head with its own
    k-head) returns exactly the matching heads of the call over all heads, in the order
    asked for, including heads of different k-head groups."""
    rng = np.random.default_rng(31)
    Hk, Hv, d = 2, 6, 4
    lens = [5, 0, 9]
    C = 2 * Hk * d + Hv * d
    T = sum(lens)
    x = rng.standard_normal((T, C))
    w = rng.uniform(-0.5, 0.5, (C, 4))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    g = -np.logaddexp(0, rng.standard_normal((T, Hv)))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, Hv))))
    cs = rng.standard_normal((len(lens), 3, C))
    h0 = rng.standard_normal((len(lens), Hv, d, d)) * 0.3
    full = oracle.layer_prefill(x, w, None, g, beta, cu, Hk, Hv, d, d, conv_state=cs,
                                initial_state=h0, scale=0.8)
    heads = [5, 0, 3, 1, 4]   # k-heads 1, 0, 1, 0, 1 under contiguous groups
    sub = oracle.layer_prefill(x, w, None, g, beta, cu, Hk, Hv, d, d, conv_state=cs,
                               initial_state=h0, scale=0.8, v_heads=heads)
    np.testing.assert_array_equal(sub[0], full[0][:, heads])
    np.testing.assert_array_equal(sub[1], full[1][:, heads])
    np.testing.assert_array_equal(sub[2], full[2])
