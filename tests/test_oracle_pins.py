"""Pins of the CPU oracle against facts that do not come from the oracle itself:
brute-force enumeration on tiny inputs, invariants of the layout, special
cases that reduce to a library routine, exact algebraic identities in fp64, a
hand-worked layout, and the memory closed forms the torchtitan issue prints.
Each planted-mistake test feeds the oracle a deliberately wrong input and
checks that the corresponding pin rejects it."""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import synth
from tests.common import assert_ulp, gw_tolerance_ok, ulp_dist

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# brute-force selection


def brute_topk(keys, K, eligible=None):
    """The K-subset whose keys, sorted descending, are lexicographically
    largest; among equal key vectors the one with the smaller indices.  Returned
    in descending key order, equal keys by ascending index."""
    cands = [e for e in range(len(keys)) if eligible is None or eligible[e]]
    best = None
    for sub in itertools.combinations(cands, K):
        order = sorted(sub, key=lambda e: (-keys[e], e))
        score = ([keys[e] for e in order], [-e for e in order])
        if best is None or score > best[0]:
            best = (score, order)
    return best[1]


def tie_heavy_logits(rng, T, E):
    return rng.integers(-2, 3, size=(T, E)).astype(np.float32) * np.float32(0.5)


@pytest.mark.parametrize("E,K", [(4, 1), (4, 2), (6, 3), (8, 2), (8, 3)])
@pytest.mark.parametrize("ties", [False, True])
def test_softmax_topk_matches_bruteforce(E, K, ties):
    rng = np.random.default_rng(100 + E * 10 + K)
    T = 64
    logits = tie_heavy_logits(rng, T, E) if ties else rng.standard_normal((T, E)).astype(np.float32)
    idx, w = oracle.route_softmax(logits, K)
    for t in range(T):
        assert list(idx[t]) == brute_topk(list(logits[t]), K), t


def test_softmax_all_equal_row_selects_lowest_indices():
    for K in (1, 2, 4, 8):
        logits = np.full((3, 16), 0.75, np.float32)
        idx, w = oracle.route_softmax(logits, K)
        assert (idx == np.arange(K)).all()
        assert (w == np.float32(1.0 / K)).all()


def test_softmax_weights_invariants():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((200, 32)).astype(np.float32) * 2
    K = 6
    idx, w = oracle.route_softmax(logits, K)
    s = w.astype(np.float64).sum(1)
    assert np.abs(s - 1).max() <= K * 2.0 ** -24 * 1.01
    # ratio of two renormalised weights = exp(logit difference)
    sel = np.take_along_axis(logits, idx, 1).astype(np.float64)
    ratio = w[:, 1:].astype(np.float64) / w[:, :1]
    assert np.allclose(ratio, np.exp(sel[:, 1:] - sel[:, :1]), rtol=3e-7, atol=0)
    assert (np.diff(sel, axis=1) <= 0).all()


def test_softmax_full_selection_is_scipy_softmax():
    """With K = E every expert is kept, and the renormalised weights are the
    full softmax (library routine), in the selected order."""
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((100, 8)).astype(np.float32) * 3
    idx, w = oracle.route_softmax(logits, 8)
    ref = np.take_along_axis(scipy.special.softmax(logits.astype(np.float64), axis=1), idx, 1)
    assert_ulp(w, ref.astype(np.float32), 1, "softmax K=E")


def test_softmax_no_renorm_is_scipy_softmax_of_all():
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((100, 16)).astype(np.float32)
    idx, w = oracle.route_softmax(logits, 4, renorm=False)
    ref = np.take_along_axis(scipy.special.softmax(logits.astype(np.float64), axis=1), idx, 1)
    assert_ulp(w, ref.astype(np.float32), 1, "softmax renorm=0")
    idx2, w2 = oracle.route_softmax(logits, 4, renorm=True, route_scale=2.5)
    _, w1 = oracle.route_softmax(logits, 4, renorm=True)
    assert_ulp(w2, (w1.astype(np.float64) * 2.5).astype(np.float32), 1, "route_scale")


def test_softmax_planted_wrong_weights_fail_ratio_pin():
    rng = np.random.default_rng(10)
    logits = rng.standard_normal((50, 16)).astype(np.float32)
    idx, w = oracle.route_softmax(logits, 4)
    sel = np.take_along_axis(logits, idx, 1).astype(np.float64)
    wrong = np.roll(w, 1, axis=1)  # misaligned scores
    ratio = wrong[:, 1:].astype(np.float64) / wrong[:, :1]
    assert not np.allclose(ratio, np.exp(sel[:, 1:] - sel[:, :1]), rtol=3e-7, atol=0)


# ----------------------------------------------------------------------------
# group-limited sigmoid routing


def py_keys(logits_row, bias):
    return [1.0 / (1.0 + math.exp(-float(l))) + (float(bias[e]) if bias is not None else 0.0)
            for e, l in enumerate(logits_row)]


def brute_grouped(keys, G, tg, gk, K):
    E = len(keys)
    gsz = E // G
    gscore = [sum(sorted(keys[g * gsz:(g + 1) * gsz], reverse=True)[:gk]) for g in range(G)]
    kept = set(brute_topk(gscore, tg))
    elig = [e // gsz in kept for e in range(E)]
    return brute_topk(keys, K, elig)


@pytest.mark.parametrize("G,tg,gk,K", [(4, 2, 1, 3), (4, 2, 2, 3), (2, 1, 2, 2), (4, 3, 2, 4), (8, 4, 1, 3)])
@pytest.mark.parametrize("ties", [False, True])
def test_sigmoid_grouped_matches_bruteforce(G, tg, gk, K, ties):
    rng = np.random.default_rng(G * 100 + tg * 10 + gk + K)
    T, E = 48, 8
    if ties:
        logits = tie_heavy_logits(rng, T, E)
        bias = (rng.integers(-1, 2, size=E) * 0.25).astype(np.float32)
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
        bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    idx, w = oracle.route_sigmoid_grouped(logits, bias, K, G, tg, gk)
    for t in range(T):
        assert list(idx[t]) == brute_grouped(py_keys(logits[t], bias), G, tg, gk, K), t


def test_sigmoid_one_group_no_bias_selects_like_softmax():
    """sigmoid is strictly increasing, so without bias and groups the selected
    experts and their order equal the softmax (logit) selection."""
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((300, 64)).astype(np.float32)
    i1, _ = oracle.route_softmax(logits, 8)
    i2, w2 = oracle.route_sigmoid_grouped(logits, None, 8, 1, 1, 1)
    assert (i1 == i2).all()
    s = scipy.special.expit(np.take_along_axis(logits, i2, 1).astype(np.float64))
    assert_ulp(w2, (s / s.sum(1, keepdims=True)).astype(np.float32), 1, "sigmoid renorm")
    _, w3 = oracle.route_sigmoid_grouped(logits, None, 8, 1, 1, 1, renorm=False)
    assert_ulp(w3, s.astype(np.float32), 1, "sigmoid no renorm")


def test_sigmoid_bias_moves_selection_not_weights():
    rng = np.random.default_rng(12)
    T, E, K = 100, 32, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = np.zeros(E, np.float32)
    bias[5] = 10.0  # expert 5 always selected first
    idx, w = oracle.route_sigmoid_grouped(logits, bias, K, 1, 1, 1)
    assert (idx[:, 0] == 5).all()
    s = scipy.special.expit(np.take_along_axis(logits, idx, 1).astype(np.float64))
    assert_ulp(w, (s / s.sum(1, keepdims=True)).astype(np.float32), 1, "unbiased weights")


def test_sigmoid_group_limit_confines_experts():
    wl = synth.WORKLOADS[3].with_tokens(512)
    logits = synth.router_logits(wl)
    bias = synth.selection_bias(wl)
    idx, w = oracle.route_sigmoid_grouped(logits, bias, 8, 8, 4, 2)
    groups = idx // 32
    assert all(len(set(r)) <= 4 for r in groups)
    assert (np.sort(idx, 1)[:, 1:] != np.sort(idx, 1)[:, :-1]).all()


# ----------------------------------------------------------------------------
# layout


def test_layout_hand_worked_example():
    # T=4, E=4, K=2, R=2 (ranks {0,1} and {2,3}); worked by hand from the
    # definitions of the expert-grouped receive and rank-major send layouts.
    idx = np.array([[2, 0], [1, 0], [3, 2], [0, 3]], np.int32)
    L = oracle.layout(idx, 4, 2)
    assert L.cnt_e.tolist() == [3, 1, 2, 2]
    assert L.off_e.tolist() == [0, 3, 4, 6, 8]
    assert L.pos.tolist() == [[4, 0], [3, 1], [6, 5], [2, 7]]
    assert L.recv_token.tolist() == [0, 1, 3, 1, 0, 2, 2, 3]
    assert L.recv_k.tolist() == [1, 1, 0, 0, 0, 1, 0, 1]
    assert L.cnt_send_r.tolist() == [3, 3]
    assert L.off_send_r.tolist() == [0, 3, 6]
    assert L.S == 6
    assert L.send_token.tolist() == [0, 1, 3, 0, 2, 3, -1, -1]
    assert L.send_row_of.tolist() == [[3, 0], [1, 1], [4, 4], [2, 5]]
    assert L.recv_send_row.tolist() == [0, 1, 2, 1, 3, 4, 4, 5]
    assert L.cnt_recv_r.tolist() == [4, 4]
    assert L.off_recv_r.tolist() == [0, 4, 8]
    assert L.dropped == 0


def random_idx(rng, T, E, K):
    return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


def sort_based_layout(idx, E, R):
    """The layout re-derived by stable sorting (expert, token, k) and
    (rank, token) pairs instead of running counters."""
    T, K = idx.shape
    epr = E // R
    flat_e = idx.reshape(-1).astype(np.int64)
    order = np.argsort(flat_e, kind="stable")  # flat index = t*K+k: token-then-k order
    recv_token = (order // K).astype(np.int32)
    recv_k = (order % K).astype(np.int32)
    pos = np.empty(T * K, np.int32)
    pos[order] = np.arange(T * K)
    pairs = sorted({(int(e) // epr, t) for t in range(T) for e in idx[t]})
    send_token = [t for _, t in pairs]
    row = {p: i for i, p in enumerate(pairs)}
    send_row_of = np.array([[row[(int(e) // epr, t)] for e in idx[t]] for t in range(T)],
                           np.int32).reshape(T, K)
    return recv_token, recv_k, pos.reshape(T, K), send_token, send_row_of


@pytest.mark.parametrize("T,E,K,R", [(50, 8, 3, 4), (64, 8, 2, 2), (33, 16, 4, 8), (20, 8, 3, 1),
                                     (20, 8, 3, 8), (1, 4, 2, 2), (0, 4, 2, 2)])
def test_layout_matches_sort_based_definition(T, E, K, R):
    rng = np.random.default_rng(T * 1000 + E * 10 + K + R)
    idx = random_idx(rng, T, E, K) if T else np.zeros((0, K), np.int32)
    L = oracle.layout(idx, E, R)
    rt, rk, pos, st, sro = sort_based_layout(idx, E, R)
    assert (L.recv_token == rt).all() and (L.recv_k == rk).all() and (L.pos == pos).all()
    assert L.send_token[:L.S].tolist() == st and (L.send_token[L.S:] == -1).all()
    assert (L.send_row_of == sro).all()
    # invariants
    assert L.cnt_e.sum() == T * K and L.off_e[-1] == T * K
    assert sorted(L.pos.reshape(-1).tolist()) == list(range(T * K))  # bijection
    for e in range(E):
        seg = L.recv_token[L.off_e[e]:L.off_e[e + 1]]
        assert (np.diff(seg) > 0).all()
        assert (idx[seg] == e).any(1).all()
    assert L.S == L.cnt_send_r.sum() <= T * min(K, R)
    assert (L.recv_send_row == L.send_row_of.reshape(-1)[np.argsort(L.pos.reshape(-1))]).all()
    epr = E // R
    for r in range(R):
        assert L.cnt_recv_r[r] == L.cnt_e[r * epr:(r + 1) * epr].sum()
        assert L.off_recv_r[r] == L.off_e[r * epr]
    if R == 1:
        assert L.S == T
    if R == E:
        assert L.S == T * K


def test_layout_zero_load_expert_and_skew():
    wl = synth.WORKLOADS[2].with_tokens(2048)
    idx, _ = oracle.route_softmax(synth.router_logits(wl), wl.K)
    L = oracle.layout(idx, wl.E, wl.R)
    zero = np.flatnonzero(L.cnt_e == 0)
    assert zero.tolist() == [wl.E - 1]
    assert L.off_e[wl.E - 1] == L.off_e[wl.E]
    mean = wl.T * wl.K / wl.E
    assert L.cnt_e.max() > 5 * mean


def test_layout_drops_invalid_entries():
    idx = np.array([[0, 0, 3], [9, 1, -1], [2, 3, 1]], np.int32)
    L = oracle.layout(idx, 4, 2)
    assert L.dropped == 3
    assert L.pos[0, 1] == -1 and L.pos[1, 0] == -1 and L.pos[1, 2] == -1
    assert L.cnt_e.tolist() == [1, 2, 1, 2]
    assert L.off_e[-1] == 6
    assert (L.recv_token[6:] == -1).all()
    assert L.send_row_of[1, 0] == -1
    valid = L.pos[L.pos >= 0]
    assert sorted(valid.tolist()) == list(range(6))


def test_layout_planted_duplicate_breaks_bijection_pin():
    """If the layout forgot to drop a repeated expert, two entries would share
    a row; the bijection pin is what rejects that."""
    idx = np.array([[1, 1], [0, 1]], np.int32)
    L = oracle.layout(idx, 2, 1)
    assert sorted(L.pos[L.pos >= 0].tolist()) == list(range(L.off_e[-1]))
    planted = L.pos.copy()
    planted[0, 1] = planted[0, 0]
    assert sorted(planted.reshape(-1).tolist()) != list(range(4))


# ----------------------------------------------------------------------------
# dispatch / combine and their backward


def small_case(seed, T=40, H=24, E=8, K=4, R=4, dtype=np.float32):
    rng = np.random.default_rng(seed)
    idx = random_idx(rng, T, E, K)
    L = oracle.layout(idx, E, R)
    w = rng.random((T, K)).astype(np.float32)
    x = rng.standard_normal((T, H)).astype(np.float32)
    y = rng.standard_normal((T * K, H)).astype(np.float32)
    g = rng.standard_normal((T, H)).astype(np.float32)
    if dtype == np.uint16:
        x, y, g = synth.to_bf16_bits(x), synth.to_bf16_bits(y), synth.to_bf16_bits(g)
    return idx, L, w, x, y, g


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_dispatch_is_gather_by_recv_token(dtype):
    idx, L, w, x, y, g = small_case(1, dtype=dtype)
    recv, recv_w, send = oracle.dispatch(x, L, w, with_send=True)
    assert (recv == x[L.recv_token]).all()
    assert (recv_w == w[L.recv_token, L.recv_k]).all()
    assert (send[:L.S] == x[L.send_token[:L.S]]).all()


@pytest.mark.parametrize("K,dtype", [(2, np.float32), (2, np.uint16), (8, np.uint16), (8, np.float32)])
def test_identity_experts_unit_weights_give_x_times_K(K, dtype):
    """dispatch then combine with identity experts and unit weights is x*K.
    Exact for bf16 rows (the partial sums k*x need at most 8+3 significant bits,
    which fp32 holds) and for K=2; for fp32 rows with K=8 the partial sums 3x,
    5x, 6x, 7x may round, so there it holds within the fp32 summation bound."""
    idx, L, w, x, y, g = small_case(2, T=64, H=32, E=16, K=K, R=4, dtype=dtype)
    recv, _, _ = oracle.dispatch(x, L)
    out_plain = oracle.combine(recv, L)
    out_unit = oracle.combine(recv, L, np.ones_like(w))
    xf = x if dtype == np.float32 else oracle.bf16_to_f32(x)
    ref = (xf * np.float32(K)).astype(np.float32)
    if dtype == np.uint16:
        ref = synth.to_bf16_bits(ref)
    if dtype == np.float32 and K == 8:
        for out in (out_plain, out_unit):
            assert (np.abs(out.astype(np.float64) - ref) <= K * K * 2.0 ** -24 * np.abs(ref)).all()
        return
    assert (out_plain == ref).all() and (out_unit == ref).all()


def test_renormalised_identity_combine_returns_x():
    wl = synth.WORKLOADS[0]
    inp = synth.make_inputs(wl, want=("logits", "x"))
    idx, w = oracle.route_softmax(inp["logits"], wl.K)
    L = oracle.layout(idx, wl.E, wl.R)
    recv, _, _ = oracle.dispatch(inp["x"], L)
    out = oracle.combine(recv, L, w)
    # sum_k w_k x = x (1 + O(K eps)) for weights summing to 1 within K ulp
    err = np.abs(out.astype(np.float64) - inp["x"])
    assert (err <= 4 * wl.K * 2.0 ** -24 * np.abs(inp["x"]) + 1e-30).all()


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_combine_within_rounding_of_exact_sum(dtype):
    idx, L, w, x, y, g = small_case(3, T=64, H=40, E=8, K=6, R=2, dtype=dtype)
    out = oracle.combine(y, L, w)
    yf = y if dtype == np.float32 else oracle.bf16_to_f32(y)
    exact = oracle.combine_f64(yf, L, w)
    absmag = oracle.combine_f64(np.abs(yf), L, np.abs(w))
    fp32_bound = 6 * 2.0 ** -24 * absmag * 1.01
    if dtype == np.float32:
        assert (np.abs(out - exact) <= fp32_bound).all()
    else:
        o = oracle.bf16_to_f32(out).astype(np.float64)
        half_ulp = np.abs(o) * 2.0 ** -8
        assert (np.abs(o - exact) <= fp32_bound + half_ulp + 1e-300).all()


def test_k1_combine_is_scaled_permutation():
    idx, L, w, x, y, g = small_case(4, T=50, H=16, E=8, K=1, R=2)
    out = oracle.combine(y, L, w)
    ref = (w[:, :1] * y[L.pos[:, 0]]).astype(np.float32)  # fp32 product, correctly rounded
    assert (out == ref).all()


def adjoint_residuals(L, x, y, w):
    """<dispatch(x), y> - <x, combine_unit(y)> and the same for weights, fp64."""
    H = x.shape[1]
    d = oracle.dispatch_f64(x, L)
    r1 = np.vdot(d, y) - np.vdot(x, oracle.combine_f64(y, L))
    # <combine_w(y), g> = <y, W^T g> where (W^T g)[pos[t,k]] = w[t,k] g[t]
    g = x
    wtg = np.zeros_like(y)
    for t in range(L.T):
        for k in range(L.K):
            wtg[L.pos[t, k]] = w[t, k] * g[t]
    r2 = np.vdot(oracle.combine_f64(y, L, w), g) - np.vdot(y, wtg)
    scale = np.abs(x).sum() * np.abs(y).max() * L.K + 1.0
    return abs(r1) / scale, abs(r2) / scale


def test_adjoint_identities_fp64():
    rng = np.random.default_rng(5)
    idx, L, w, x, y, g = small_case(5, T=30, H=12, E=8, K=3, R=4)
    x = rng.standard_normal(x.shape)
    y = rng.standard_normal(y.shape)
    r1, r2 = adjoint_residuals(L, x, y, w.astype(np.float64))
    assert r1 < 1e-13 and r2 < 1e-13


def test_combine_bwd_adjoint_and_score_gradient():
    idx, L, w, x, y, g = small_case(6, T=30, H=20, E=8, K=3, R=4)
    gy, gw = oracle.combine_bwd(g, y, L, w)
    out64 = oracle.combine_f64(y, L, w)
    lhs = np.vdot(out64, g.astype(np.float64))
    rhs = np.vdot(y.astype(np.float64), gy.astype(np.float64))
    assert abs(lhs - rhs) <= 1e-6 * (np.abs(out64).sum() * np.abs(g).max())
    # d<combine_w(y), g>/dw by central differences (exactly linear in w)
    for (t, k) in [(0, 0), (3, 2), (17, 1), (29, 0)]:
        eps = 0.5
        wp = w.astype(np.float64).copy()
        wm = wp.copy()
        wp[t, k] += eps
        wm[t, k] -= eps
        fd = (np.vdot(oracle.combine_f64(y, L, wp), g) - np.vdot(oracle.combine_f64(y, L, wm), g)) / (2 * eps)
        assert abs(fd - gw[t, k]) <= 1e-9 * (1 + abs(fd))
    # and as a dot of gathered rows (numpy einsum)
    ref = np.einsum("th,tkh->tk", g.astype(np.float64), y.astype(np.float64)[L.pos])
    assert np.allclose(gw, ref, rtol=1e-12, atol=1e-12)


def test_combine_bwd_plain_sum_copies_g():
    idx, L, w, x, y, g = small_case(7, dtype=np.uint16)
    gy, gw = oracle.combine_bwd(g, y, L, None)
    assert gw is None
    assert (gy == g[L.recv_token]).all()


def test_dispatch_bwd_adjoint():
    idx, L, w, x, y, g = small_case(8, T=30, H=20, E=8, K=3, R=4)
    recv, _, _ = oracle.dispatch(x, L)
    gx = oracle.dispatch_bwd(y, L)
    lhs = np.vdot(recv.astype(np.float64), y.astype(np.float64))
    rhs = np.vdot(x.astype(np.float64), gx.astype(np.float64))
    assert abs(lhs - rhs) <= 1e-6 * np.abs(recv).sum() * np.abs(y).max()


@pytest.mark.parametrize("mutation", ["rolled", "doubled", "dropped"])
def test_planted_score_mistakes_fail_adjoint_pin(mutation):
    rng = np.random.default_rng(9)
    idx, L, w, x, y, g = small_case(9, T=30, H=12, E=8, K=3, R=4)
    x = rng.standard_normal(x.shape)
    y = rng.standard_normal(y.shape)
    w64 = w.astype(np.float64)
    bad = {"rolled": np.roll(w64, 1, axis=0), "doubled": 2 * w64,
           "dropped": np.where(np.arange(3) == 1, 0.0, w64)}[mutation]
    # the weighted combine with the mutated scores against the adjoint built from the true ones
    wtg = np.zeros_like(y)
    for t in range(L.T):
        for k in range(L.K):
            wtg[L.pos[t, k]] = w64[t, k] * x[t]
    r = abs(np.vdot(oracle.combine_f64(y, L, bad), x) - np.vdot(y, wtg))
    assert r > 1e-3 * np.abs(np.vdot(y, wtg))


def test_gw_tolerance_rejects_rolled_rows_and_two_ulp_is_caught():
    idx, L, w, x, y, g = small_case(10, T=30, H=64, E=8, K=3, R=4)
    gy, gw = oracle.combine_bwd(g, y, L, w)
    gn = np.linalg.norm(g.astype(np.float64), axis=1)[:, None] * np.ones((30, 3))
    yn = np.linalg.norm(y.astype(np.float64), axis=1)[L.pos]
    assert gw_tolerance_ok(gw, gw, gn, yn).all()
    assert not gw_tolerance_ok(np.roll(gw, 1, axis=0), gw, gn, yn).all()
    out = oracle.combine(synth.to_bf16_bits(y), L, w)
    bumped = out.copy()
    bumped[3, 5] = np.uint16(int(bumped[3, 5]) + 2)
    assert ulp_dist(bumped, out).max() == 2


# ----------------------------------------------------------------------------
# absorption of router scores into the W2 input


def absorbed_vs_post_combine(h, w2, L, w, mutate=None):
    """fp32-scale comparison of the two orders of the same linear map:
    post  = combine_w(h @ W2_e)        (scores applied after W2)
    abs   = combine_plain(scale_rows(h, recv_w) @ W2_e)."""
    recv_w = w[L.recv_token, L.recv_k]
    if mutate == "rolled":
        recv_w = np.roll(recv_w, 1)
    elif mutate == "doubled":
        recv_w = 2 * recv_w
    elif mutate == "dropped":
        recv_w = recv_w.copy()
        recv_w[::3] = 0
    E = w2.shape[0]
    expert_of_row = np.repeat(np.arange(E), L.cnt_e)
    hs = oracle.scale_rows(h, recv_w)
    y_abs = np.einsum("ri,rio->ro", hs.astype(np.float64), w2[expert_of_row])
    y_post = np.einsum("ri,rio->ro", h.astype(np.float64), w2[expert_of_row])
    out_abs = oracle.combine_f64(y_abs, L)
    out_post = oracle.combine_f64(y_post, L, w.astype(np.float64))
    return out_abs, out_post


@pytest.mark.parametrize("mutate", [None, "rolled", "doubled", "dropped"])
def test_absorbed_equals_post_combine(mutate):
    rng = np.random.default_rng(11)
    T, E, K, R, I, D = 40, 8, 3, 4, 16, 12
    idx = random_idx(rng, T, E, K)
    L = oracle.layout(idx, E, R)
    w = rng.random((T, K)).astype(np.float32)
    h = rng.standard_normal((T * K, I)).astype(np.float32)
    w2 = rng.standard_normal((E, I, D))
    a, p = absorbed_vs_post_combine(h, w2, L, w, mutate)
    ok = np.allclose(a, p, rtol=1e-5, atol=1e-5 * np.abs(p).max())
    assert ok == (mutate is None)


def test_scale_rows_bwd_gradient_matches_post_combine_gradient():
    """Absorbed: d/dw of <combine_plain((w*h) W2), g> = <ghs, h> with ghs = g W2^T;
    post-combine: <g, h W2>.  Both are the same number."""
    rng = np.random.default_rng(12)
    T, E, K, R, I, D = 30, 8, 3, 2, 10, 14
    idx = random_idx(rng, T, E, K)
    L = oracle.layout(idx, E, R)
    w = rng.random((T, K)).astype(np.float32)
    h = rng.standard_normal((T * K, I)).astype(np.float32)
    g = rng.standard_normal((T, D)).astype(np.float32)
    w2 = rng.standard_normal((E, I, D)).astype(np.float32)
    expert_of_row = np.repeat(np.arange(E), L.cnt_e)
    gy, _ = oracle.combine_bwd(g, np.zeros((T * K, D), np.float32), L, None)
    ghs = np.einsum("ro,rio->ri", gy.astype(np.float64), w2[expert_of_row].astype(np.float64)).astype(np.float32)
    recv_w = w[L.recv_token, L.recv_k]
    gh, gw_abs = oracle.scale_rows_bwd(ghs, h, recv_w, L)
    y = np.einsum("ri,rio->ro", h.astype(np.float64), w2[expert_of_row]).astype(np.float32)
    _, gw_post = oracle.combine_bwd(g, y, L, w)
    assert np.allclose(gw_abs, gw_post, rtol=1e-4, atol=1e-4)
    assert (gh == (recv_w[:, None] * ghs).astype(np.float32)).all()


# ----------------------------------------------------------------------------
# memory closed forms printed on the torchtitan issue


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v, _unit = line.split()
            vals[k] = float(v)
    return vals


def test_memory_closed_forms_from_layout():
    g = read_golden("memory_closed_forms.txt")
    T, K, D, layers = int(g["T"]), int(g["top_k"]), int(g["D"]), int(g["layers"])
    rng = np.random.default_rng(13)
    logits = rng.standard_normal((T, 256)).astype(np.float32)
    idx, _ = oracle.route_sigmoid_grouped(logits, None, K, 8, 4, 2)
    L = oracle.layout(idx, 256, 64)
    MiB, GiB = 2.0 ** 20, 2.0 ** 30
    recv_rows = int(L.off_e[-1])
    assert recv_rows * D * 2 / MiB == g["w2_out_per_layer"]
    assert T * D * 2 / MiB == g["combine_out_per_layer"]
    assert round(T * D * 2 * layers / GiB, 2) == g["combine_out_all_layers"]
    assert round(recv_rows * D * 2 * layers / GiB, 1) == g["w2_out_all_layers"]
    # the page adds its two rounded figures: 25.4 + 3.17 (the exact sum is 28.55)
    total = round(recv_rows * D * 2 * layers / GiB, 1) + round(T * D * 2 * layers / GiB, 2)
    assert round(total, 1) == g["total_per_gpu"]


# ----------------------------------------------------------------------------
# input generator properties


def test_generator_is_deterministic_and_chunk_stable():
    a = synth.normal_f32(0, "x", (3, synth.CHUNK + 5), threads=1)
    b = synth.normal_f32(0, "x", (3, synth.CHUNK + 5), threads=4)
    assert (a == b).all()
    c = synth.normal_f32(1, "x", (3, 10))
    assert not (c == a[:, :10]).all()


def test_bf16_rounding_of_generator_matches_oracle_rounding():
    rng = np.random.default_rng(14)
    a = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([0.0, -0.0, np.inf, -np.inf, 1.00390625, 1.01171875, 3.4e38],
                                 np.float32)])
    assert (synth.to_bf16_bits(a) == oracle.f32_to_bf16(a)).all()
    assert (oracle.bf16_to_f32(synth.to_bf16_bits(np.float32([1.00390625]))) == np.float32(1.0)).all()


# ----------------------------------------------------------------------------
# router backward to the logits


def weights_fp64(logits_row, sel, score_fn, renorm, scale):
    """Routing weights of a fixed selection as a function of the logits, from
    library routines (scipy softmax / expit), for numerical differentiation."""
    l = np.asarray(logits_row, np.float64)
    if score_fn == "softmax":
        p = scipy.special.softmax(l[sel]) if renorm else scipy.special.softmax(l)[sel]
        return scale * p
    s = scipy.special.expit(l[sel])
    return scale * (s / s.sum() if renorm else s)


@pytest.mark.parametrize("score_fn", ["softmax", "sigmoid"])
@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("scale", [1.0, 2.5])
def test_route_bwd_matches_central_differences(score_fn, renorm, scale):
    rng = np.random.default_rng(31)
    T, E, K = 12, 16, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if score_fn == "softmax":
        idx, _ = oracle.route_softmax(logits, K, renorm, scale)
    else:
        idx, _ = oracle.route_sigmoid_grouped(logits, None, K, 1, 1, 1, renorm, scale)
    gw = rng.standard_normal((T, K))
    g = oracle.route_bwd(logits, idx, gw, score_fn, renorm, scale)
    eps = 1e-6
    for t in range(T):
        for e in range(E):
            lp = logits[t].astype(np.float64).copy()
            lm = lp.copy()
            lp[e] += eps
            lm[e] -= eps
            fd = (np.dot(gw[t], weights_fp64(lp, idx[t], score_fn, renorm, scale)) -
                  np.dot(gw[t], weights_fp64(lm, idx[t], score_fn, renorm, scale))) / (2 * eps)
            assert abs(fd - g[t, e]) <= 1e-7 * (1 + abs(fd)), (t, e, fd, g[t, e])


def test_route_bwd_invariants():
    rng = np.random.default_rng(32)
    logits = rng.standard_normal((50, 32)).astype(np.float32)
    idx, w = oracle.route_softmax(logits, 6)
    gw = rng.standard_normal((50, 6))
    g = oracle.route_bwd(logits, idx, gw)
    # softmax is shift invariant: the gradient sums to zero over the logits
    assert np.abs(g.sum(1)).max() < 1e-12
    # only the selected logits move a renormalised softmax
    mask = np.zeros_like(g, bool)
    np.put_along_axis(mask, idx, True, 1)
    assert (g[~mask] == 0).all()
    # a gradient proportional to the weights (uniform rescaling) changes nothing
    g2 = oracle.route_bwd(logits, idx, np.ones_like(gw))
    assert np.abs(g2).max() < 1e-15


# ----------------------------------------------------------------------------
# staged (wire-faithful) dispatch and combine


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_dispatch_through_send_rows_equals_direct_dispatch(dtype):
    idx, L, w, x, y, g = small_case(40, T=64, H=24, E=16, K=4, R=4, dtype=dtype)
    recv, _, send = oracle.dispatch(x, L, w, with_send=True)
    assert (oracle.expand(send, L) == recv).all()
    # each token travels once per destination rank
    assert L.S == sum(len({int(e) // (L.E // L.R) for e in row}) for row in idx)


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_staged_combine_with_one_rank_is_the_combine(dtype):
    """R = 1: one send row per token holding all K entries, so stage 1 is the
    combine itself and stage 2 adds it to zero."""
    idx, L, w, x, y, g = small_case(41, T=50, H=24, E=8, K=4, R=1, dtype=dtype)
    staged = oracle.combine_reduce(oracle.combine_partial(y, L, w), L)
    assert (staged == oracle.combine(y, L, w)).all()


def test_staged_combine_identity_experts_give_x_times_K_in_bf16():
    idx, L, w, x, y, g = small_case(42, T=64, H=32, E=16, K=8, R=4, dtype=np.uint16)
    recv, _, send = oracle.dispatch(x, L, with_send=True)
    out = oracle.combine_reduce(oracle.combine_partial(oracle.expand(send, L), L), L)
    ref = synth.to_bf16_bits(oracle.bf16_to_f32(x) * np.float32(8))
    assert (out == ref).all()


def test_staged_combine_within_rounding_of_exact_sum():
    idx, L, w, x, y, g = small_case(43, T=64, H=40, E=16, K=6, R=4)
    staged = oracle.combine_reduce(oracle.combine_partial(y, L, w), L)
    exact = oracle.combine_f64(y, L, w)
    absmag = oracle.combine_f64(np.abs(y), L, np.abs(w))
    # stage 1 rounds each partial once and stage 2 adds at most min(K,R) of them
    bound = (6 + 4 + 4) * 2.0 ** -24 * absmag * 1.01
    assert (np.abs(staged - exact) <= bound).all()


# ----------------------------------------------------------------------------
# padded (capacity-aligned) receive layout


@pytest.mark.parametrize("align", [1, 4, 7, 128])
def test_padded_layout_shifts_segments_to_aligned_starts(align):
    rng = np.random.default_rng(50 + align)
    T, E, K, R = 90, 16, 4, 4
    idx = random_idx(rng, T, E, K)
    L0 = oracle.layout(idx, E, R)
    L = oracle.layout(idx, E, R, align)
    assert (L.cnt_e == L0.cnt_e).all()
    assert (L.off_e % align == 0).all()
    assert (np.diff(L.off_e) == -(-L0.cnt_e // align) * align).all()
    # same rank inside each segment, only the segment start moves
    e_of = idx
    assert ((L.pos - L.off_e[e_of]) == (L0.pos - L0.off_e[e_of])).all()
    for e in range(E):
        seg = slice(L.off_e[e], L.off_e[e + 1])
        n = L.cnt_e[e]
        assert (L.recv_token[seg][:n] == L0.recv_token[L0.off_e[e]:L0.off_e[e + 1]]).all()
        assert (L.recv_token[seg][n:] == -1).all() and (L.recv_k[seg][n:] == -1).all()
    assert L.recv_rows == T * K + E * (align - 1)
    assert (L.send_token == L0.send_token).all() and (L.send_row_of == L0.send_row_of).all()


def test_padded_layout_leaves_row_results_unchanged():
    idx, L0, w, x, y0, g = small_case(51, T=60, H=24, E=8, K=3, R=2, dtype=np.uint16)
    L = oracle.layout(idx, 8, 2, 16)
    recv0, rw0, _ = oracle.dispatch(x, L0, w)
    recv, rw, _ = oracle.dispatch(x, L, w)
    # the same rows, moved to the padded positions; pad rows stay zero
    assert (recv[L.pos.reshape(-1)] == recv0[L0.pos.reshape(-1)]).all()
    pad = np.ones(L.recv_rows, bool)
    pad[L.pos.reshape(-1)] = False
    assert (recv[pad] == 0).all() and (rw[pad] == 0).all()
    y = np.zeros((L.recv_rows, y0.shape[1]), np.uint16)
    y[L.pos.reshape(-1)] = y0[L0.pos.reshape(-1)]
    assert (oracle.combine(y, L, w) == oracle.combine(y0, L0, w)).all()
    assert (oracle.dispatch_bwd(y, L) == oracle.dispatch_bwd(y0, L0)).all()
