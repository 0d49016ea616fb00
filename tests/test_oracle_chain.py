"""Pins for the chain-verification part of the CPU oracle.

Each test checks the oracle against something the pages or mathematics fix,
never against a retyped copy of its own formula:
  * eq. (3) / eq. (4) of the DART notes §2.3 as identities,
  * chi-square agreement of emitted tokens with q (losslessness),
  * E[A] = sum_i prod_{j<=i} a_j (DART notes §2.2 eq. (2)) and its constant-a
    closed form a(1-a^d)/(1-a), by Monte Carlo and by exact enumeration,
  * special cases (p = q, disjoint supports, T -> 0 reduces to argmax),
  * scipy's softmax as an independent reference for the temperature softmax.
"""
import itertools

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
import synth


def _probs(seed, stream, shape, scale=1.0):
    return scipy.special.softmax(scale * synth.normal(seed, stream, shape), axis=-1)


def _draw(p, seed, stream):
    """Draft tokens x ~ p via the synthetic drafter (Gumbel-max on log p)."""
    with np.errstate(divide="ignore"):
        return synth.gumbel_max_tokens(np.log(p), 1.0, seed, stream)


def _chisq_ok(samples, expected, V, n):
    counts = np.bincount(samples, minlength=V).astype(np.float64)
    support = expected > 0
    assert counts[~support].sum() == 0, "mass emitted where q = 0"
    stat, pval = scipy.stats.chisquare(counts[support], n * expected[support])
    return pval


# --------------------------------------------------------------------------- basics
def test_softmax_matches_scipy_and_temperature():
    x = 3.0 * synth.normal(11, 1, (5, 97))
    for T in (0.25, 1.0, 2.0):
        np.testing.assert_allclose(oracle.softmax_t(x, T), scipy.special.softmax(x / T, axis=-1), rtol=1e-13, atol=1e-15)
    with pytest.raises(ValueError):
        oracle.softmax_t(x, 0.0)


def test_inverse_cdf_brackets_and_exact_steps():
    w = np.array([0.0, 1.0, 0.0, 3.0])
    # C = [0, 1, 1, 4]: u in [0, 1/4) -> token 1, u in [1/4, 1) -> token 3
    for u, tok in [(0.0, 1), (0.2499, 1), (0.25, 3), (0.9999, 3)]:
        t, lo, hi = oracle.inverse_cdf(w, np.array(u))
        assert t == tok
        assert lo <= u < hi
    t, lo, hi = oracle.inverse_cdf(np.zeros(4), np.array(0.5))
    assert t == -1


# --------------------------------------------------------------------------- eq. (3), (4)
@pytest.mark.parametrize("V", [2, 8, 64, 1000])
def test_eq3_eq4_identities(V):
    q = _probs(12, 1, (20, V), 2.0)
    p = _probs(12, 2, (20, V), 2.0)
    r, R = oracle.residual(q, p)
    mins = np.minimum(p, q)
    # eq. (3): R = 1 - sum min(p, q)
    np.testing.assert_allclose(R, 1.0 - mins.sum(-1), atol=1e-12)
    # eq. (4): min(p, q) + R r = q elementwise
    np.testing.assert_allclose(mins + R[:, None] * r, q, atol=1e-12)
    # residual is a distribution
    np.testing.assert_allclose(r.sum(-1), 1.0, atol=1e-12)
    assert (r >= 0).all()
    # c* = 1 - 1/2 ||p - q||_1 equals sum min(p, q) = 1 - R
    np.testing.assert_allclose(oracle.tv_accept_probs(q, p), 1.0 - R, atol=1e-12)


def test_no_residual_when_R_zero():
    q = _probs(13, 1, (3, 16))
    r, R = oracle.residual(q, q)
    assert (R == 0).all() and np.isnan(r).all()


# --------------------------------------------------------------------------- c*
def test_tv_accept_closed_forms():
    q = _probs(14, 1, (4, 33))
    np.testing.assert_allclose(oracle.tv_accept_probs(q, q), 1.0, atol=1e-15)
    a = np.array([[0.5, 0.5, 0.0, 0.0]])
    b = np.array([[0.0, 0.0, 0.25, 0.75]])
    assert oracle.tv_accept_probs(a, b)[0] == 0.0
    for x, y in [(0.3, 0.7), (0.9, 0.1), (0.5, 0.5)]:
        c = oracle.tv_accept_probs(np.array([x, 1 - x]), np.array([y, 1 - y]))
        assert abs(c - (1.0 - abs(x - y))) < 1e-15


# --------------------------------------------------------------------------- losslessness
PAIRS = ["random", "disjoint", "equal", "partial"]


def _pair(kind, V):
    if kind == "random":
        return _probs(15, 1, (V,), 1.5), _probs(15, 2, (V,), 1.5)
    if kind == "disjoint":
        q = np.zeros(V); q[: V // 2] = _probs(15, 3, (V // 2,))
        p = np.zeros(V); p[V // 2:] = _probs(15, 4, (V - V // 2,))
        return q, p
    if kind == "equal":
        q = _probs(15, 5, (V,), 1.5)
        return q, q.copy()
    q = _probs(15, 6, (V,), 2.0)
    p = _probs(15, 7, (V,), 2.0)
    q[::3] = 0.0; q /= q.sum()
    p[1::4] = 0.0; p /= p.sum()
    return q, p


def _emitted_block(kind, V, m, seed):
    """One block of the gamma = 1 trials: the first committed token of each."""
    q0, p0 = _pair(kind, V)
    q1 = _probs(16, 1, (V,))
    q = np.broadcast_to(np.stack([q0, q1]), (m, 2, V))
    p = np.broadcast_to(p0[None, None], (m, 1, V))
    x = _draw(p, seed, 1)
    u = synth.uniform_u24(seed, 2, (m, 2, 2))
    res = oracle.verify_chain_probs(q, p, x, u)
    emitted = np.where(res.accepted >= 1, x[:, 0], res.token)
    return emitted, bool((res.accepted == 1).all()), bool((res.accepted == 0).all())


@pytest.mark.parametrize("V", [8, 64])
@pytest.mark.parametrize("kind", PAIRS)
def test_first_emitted_token_is_distributed_as_q(V, kind, pool):
    """gamma = 1: the first committed token (x_0 if accepted, else the residual
    draw) must follow q exactly (DART notes §2.3 eq. (4))."""
    n = 1_000_000
    q0, _ = _pair(kind, V)
    block = 200_000
    futs = [pool.submit(_emitted_block, kind, V, min(block, n - s), 1000 + s // block) for s in range(0, n, block)]
    parts = [f.result() for f in futs]
    emitted = np.concatenate([e for e, _, _ in parts])
    if kind == "equal":
        assert all(all_acc for _, all_acc, _ in parts)
    if kind == "disjoint":
        assert all(all_rej for _, _, all_rej in parts)
    assert _chisq_ok(emitted, q0, V, n) > 1e-3


def _bonus_block(q0, u):
    m, V = u.shape[0], q0.shape[0]
    q = np.broadcast_to(q0[None, None], (m, 1, V))
    res = oracle.verify_chain_probs(q, np.zeros((m, 0, V)), np.zeros((m, 0), dtype=np.int64), u)
    return res.accepted, res.token


@pytest.mark.parametrize("V", [8, 64])
def test_bonus_token_is_distributed_as_q(V, pool):
    from conftest import split_rows
    n = 1_000_000
    q0 = _probs(17, 1, (V,), 1.5)
    u = synth.uniform_u24(17, 2, (n, 1, 2))
    futs = [pool.submit(_bonus_block, q0, u[a:b]) for a, b in split_rows(n, 8)]
    parts = [f.result() for f in futs]
    accepted = np.concatenate([a for a, _ in parts])
    token = np.concatenate([t for _, t in parts])
    assert (accepted == 0).all()
    assert _chisq_ok(token, q0, V, n) > 1e-3


def test_disjoint_supports_residual_is_q():
    V = 8
    q, p = _pair("disjoint", V)
    r, R = oracle.residual(q, p)
    assert abs(R - 1.0) < 1e-15
    np.testing.assert_allclose(r, q, atol=1e-15)


def test_zero_residual_mass_falls_back_to_q():
    """Reading R4: a rejection with sum [q-p]_+ == 0 (only reachable through
    rounding or unnormalised rows) draws the correction token from q."""
    q = np.array([[[0.5, 0.5], [0.5, 0.5]]])
    p = np.array([[[0.6, 0.6]]])                    # p >= q everywhere: no residual
    x = np.array([[0]])
    u = np.array([[[0.9, 0.75], [0.0, 0.0]]])       # 0.9 >= 0.5/0.6: reject
    res = oracle.verify_chain_probs(q, p, x, u)
    assert res.accepted[0] == 0 and res.resid_mass[0, 0] == 0.0
    assert res.token[0] == 1                          # inverse CDF of q at 0.75


# --------------------------------------------------------------------------- eq. (2)
def _position_pairs(seed, gamma, V, c_target=None):
    qs, ps = [], []
    for k in range(gamma):
        q = _probs(seed, 2 * k + 1, (V,), 1.5)
        p = _probs(seed, 2 * k + 2, (V,), 1.5)
        if c_target is not None:
            # blend p towards q so that c* = 1 - ||p - q||_1 / 2 equals c_target
            c0 = oracle.tv_accept_probs(q, p)
            lam = (1.0 - c_target) / (1.0 - c0)
            p = q + lam * (p - q)
        qs.append(q)
        ps.append(p)
    return np.array(qs), np.array(ps)


def _expected_A_exact(qs, ps):
    """Enumerate every draft sequence x and use the oracle's accept
    thresholds: E[A] = sum_x P(x) sum_i prod_{k<i} thr_k(x_k)."""
    gamma, V = ps.shape
    seqs = np.array(list(itertools.product(range(V), repeat=gamma)))
    n = len(seqs)
    q = np.broadcast_to(np.concatenate([qs, qs[-1:]])[None], (n, gamma + 1, V))
    p = np.broadcast_to(ps[None], (n, gamma, V))
    u = np.zeros((n, gamma + 1, 2))
    thr = oracle.verify_chain_probs(q, p, seqs, u).thr
    px = np.prod(ps[np.arange(gamma)[None, :], seqs], axis=1)
    surv = np.cumprod(thr, axis=1)
    return float((px[:, None] * surv).sum())


def _accepted_block(qs, ps, x, u):
    m = x.shape[0]
    gamma, V = ps.shape
    q = np.broadcast_to(np.concatenate([qs, qs[-1:]])[None], (m, gamma + 1, V))
    p = np.broadcast_to(ps[None], (m, gamma, V))
    return oracle.verify_chain_probs(q, p, x, u).accepted


def _expected_A_mc(qs, ps, n, seed, pool):
    from conftest import split_rows
    gamma, V = ps.shape
    p = np.broadcast_to(ps[None], (n, gamma, V))
    x = _draw(p, seed, 1)
    u = synth.uniform_u24(seed, 2, (n, gamma + 1, 2))
    futs = [pool.submit(_accepted_block, qs, ps, x[a:b], u[a:b]) for a, b in split_rows(n, 8)]
    A = np.concatenate([f.result() for f in futs])
    return A.mean(), A.std() / np.sqrt(n)


def test_expected_accept_length_eq2(pool):
    gamma, V = 3, 3
    qs, ps = _position_pairs(18, gamma, V)
    c = oracle.tv_accept_probs(qs, ps)
    eq2 = float(np.cumprod(c).sum())            # sum_i prod_{j<=i} a_j with a_j = c*_j
    assert abs(_expected_A_exact(qs, ps) - eq2) < 1e-12
    mean, se = _expected_A_mc(qs, ps, 1_000_000, 19, pool)
    assert abs(mean - eq2) < 5 * se


def test_expected_accept_length_constant_a_closed_form(pool):
    gamma, V, a = 3, 3, 0.7
    qs, ps = _position_pairs(20, gamma, V, c_target=a)
    np.testing.assert_allclose(oracle.tv_accept_probs(qs, ps), a, atol=1e-12)
    closed = a * (1 - a ** gamma) / (1 - a)
    assert abs(_expected_A_exact(qs, ps) - closed) < 1e-12
    mean, se = _expected_A_mc(qs, ps, 1_000_000, 21, pool)
    assert abs(mean - closed) < 5 * se


# --------------------------------------------------------------------------- greedy
def test_greedy_chain_hand_example():
    V, gamma = 5, 3
    t = np.full((1, gamma + 1, V), -1.0)
    g = [2, 4, 0, 1]
    for k, gk in enumerate(g):
        t[0, k, gk] = 1.0
    t[0, 0, 3] = 1.0          # tie with token 2 at position 0: the argmax stays 2 (lowest id)
    t[0, 0, 2] = 1.0
    t[0, 0, 3] = 0.5
    cases = [([2, 4, 3], 2, 0), ([2, 4, 0], 3, 1), ([1, 4, 0], 0, 2), ([2, 0, 0], 1, 4)]
    for x, A, tok in cases:
        acc, token, _, gg = oracle.verify_chain_greedy(t, np.array([x]))
        assert (gg[0] == g).all()
        assert acc[0] == A and token[0] == tok
    tie = np.array([[[1.0, 3.0, 3.0, 0.0]]])
    acc, token, _, gg = oracle.verify_chain_greedy(tie, np.zeros((1, 0), dtype=np.int64))
    assert gg[0, 0] == 1 and token[0] == 1


def test_greedy_lengths_and_cstar():
    V, gamma = 6, 4
    t = synth.normal(22, 1, (3, gamma + 1, V))
    d = synth.normal(22, 2, (3, gamma, V))
    g = np.argmax(t, -1)
    x = g[:, :gamma].copy()
    ell = np.array([0, 2, 4])
    acc, token, cst, _ = oracle.verify_chain_greedy(t, x, ell, d)
    assert (acc == ell).all()
    assert (token == g[np.arange(3), ell]).all()
    assert np.isnan(cst[0]).all() and np.isnan(cst[1, 2:]).all() and not np.isnan(cst[2]).any()


def _cstar_case():
    """Hand case for c* at T = 0 (reading R7): 2 requests, gamma = 4, V = 5.
    Each row is -1 except the entries listed; argmaxes are read off by eye."""
    R, gamma, V = 2, 4, 5
    t = np.full((R, gamma + 1, V), -1.0)
    d = np.full((R, gamma, V), -1.0)
    # request 0: target argmaxes 2, 4, 1, 3, 0 for rows 0..4
    for k, g in enumerate([2, 4, 1, 3, 0]):
        t[0, k, g] = 2.0
    # draft argmaxes 2 (agrees), 3 (disagrees; equals target row 3's argmax, so
    # comparing draft row k with target row k+1 would score it), tie {1, 3} with
    # target 1 (agrees: lowest id), 0 (disagrees; equals target row 4's argmax)
    d[0, 0, 2] = 1.5
    d[0, 1, 3] = 0.5
    d[0, 2, 1] = 0.7
    d[0, 2, 3] = 0.7
    d[0, 3, 0] = 3.0
    # request 1: target argmaxes 0, 0, 3, 3, 2; draft: tie {1, 3} with target 3
    # (disagrees: the draft's argmax is 1), 0 (agrees), 3 (agrees), 4 (disagrees)
    for k, g in enumerate([0, 0, 3, 3, 2]):
        t[1, k, g] = 1.0
    t[1, 2, 4] = 0.5
    d[1, 0, 1] = 2.0
    d[1, 0, 3] = 2.0
    d[1, 1, 0] = 0.1
    d[1, 2, 3] = 5.0
    d[1, 3, 4] = 1.0
    want = np.array([[1.0, 0.0, 1.0, 0.0], [0.0, 1.0, 1.0, 0.0]])
    return t, d, want


def test_cstar_at_T0_hand_case():
    """c* at T = 0 is the indicator that the draft's and the target's argmaxes
    at the same position agree, ties to the lowest id (reading R7).  Literal
    expected values; a slip to target row k+1, or a reduction over the
    position axis, changes at least one entry."""
    t, d, want = _cstar_case()
    got = oracle.tv_accept(t, d, 0.0)
    assert got.shape == want.shape and (got == want).all()
    x = np.zeros((2, 4), dtype=np.int64)
    ell = np.array([4, 3])
    _, _, cst, _ = oracle.verify_chain_greedy(t, x, ell, d)
    assert (cst[0] == want[0]).all()
    assert (cst[1, :3] == want[1, :3]).all() and np.isnan(cst[1, 3])


def test_cstar_at_T0_is_the_small_T_limit():
    """Away from ties, c*(T) = sum_v min(p_T, q_T) tends to the argmax
    indicator as T -> 0+ (the limit reading R7 takes): with logit gaps >= 0.5,
    T = 1e-3 already puts less than e^-400 of each row's mass off its argmax."""
    t, d, want = _cstar_case()
    lim = oracle.tv_accept_probs(scipy.special.softmax(t[:, :4] / 1e-3, axis=-1),
                                 scipy.special.softmax(d / 1e-3, axis=-1))
    no_tie = np.ones_like(want, dtype=bool)
    no_tie[0, 2] = no_tie[1, 0] = False            # draft ties: the limit there is 1/2 and 0
    np.testing.assert_allclose(lim[no_tie], want[no_tie], atol=1e-12)
    np.testing.assert_allclose(lim[~no_tie], [0.5, 0.0], atol=1e-12)
    # and a random case with distinct maxima, through the oracle's T = 0 branch
    tr = synth.normal(25, 1, (5, 4, 9))
    dr = synth.normal(25, 2, (5, 3, 9))
    dr[::2] = tr[::2, :3] + 0.01 * dr[::2]         # half the requests agree at most positions
    gap_ok = (np.diff(np.sort(tr, -1)[..., -2:], axis=-1)[..., 0] > 0.05)[:, :3] & \
             (np.diff(np.sort(dr, -1)[..., -2:], axis=-1)[..., 0] > 0.05)
    small = oracle.tv_accept(tr, dr, 1e-4)
    exact = oracle.tv_accept(tr, dr, 0.0)
    assert gap_ok.sum() >= 8 and 0 < exact[gap_ok].sum() < gap_ok.sum()
    np.testing.assert_allclose(small[gap_ok], exact[gap_ok], atol=1e-9)


def test_T_to_zero_reduces_to_argmax():
    """q replaced by one-hot(argmax target) gives the greedy result for any p
    with full support (SD survey §1.3)."""
    R, gamma, V = 200, 4, 7
    t = synth.normal(23, 1, (R, gamma + 1, V))
    g = np.argmax(t, -1)
    q = np.zeros((R, gamma + 1, V))
    np.put_along_axis(q, g[..., None], 1.0, -1)
    p = _probs(23, 2, (R, gamma, V))
    # half the draft tokens copy the target argmax so that accepted prefixes vary
    rnd = synth.randint(23, 3, (R, gamma), V)
    coin = synth.uniform_u24(23, 4, (R, gamma)) < 0.7
    x = np.where(coin, g[:, :gamma], rnd)
    u = synth.uniform_u24(23, 5, (R, gamma + 1, 2))
    res = oracle.verify_chain_probs(q, p, x, u)
    acc, token, _, _ = oracle.verify_chain_greedy(t, x)
    assert (res.accepted == acc).all() and (res.token == token).all()


def test_logits_path_matches_probability_path_and_lengths():
    c = synth.chain_tiny(seed=1, R=3, gamma=4, V=50)
    ell = np.array([4, 0, 2], dtype=np.int32)
    res = oracle.verify_chain(c.target.f64, c.draft.f64, c.tokens, c.uniforms, 1.0, ell)
    q = scipy.special.softmax(c.target.f64, axis=-1)
    p = scipy.special.softmax(c.draft.f64, axis=-1)
    ref = oracle.verify_chain_probs(q, p, c.tokens, c.uniforms, ell)
    assert (res.accepted == ref.accepted).all() and (res.token == ref.token).all()
    np.testing.assert_allclose(res.c_star, ref.c_star, atol=1e-12)
    assert (res.accepted <= ell).all()
    assert np.isnan(res.c_star[1]).all() and np.isnan(res.c_star[2, 2:]).all()
    # the emitted token of a fully accepted request is its bonus draw from q_{l_r}
    for r in range(3):
        if res.accepted[r] == ell[r]:
            assert res.sample_at[r, ell[r]] == res.token[r]


def test_bonus_after_full_acceptance_uses_the_next_target_row():
    """gamma = 1 with p = q: x_0 is always accepted and the bonus must follow q_1
    (the target row after the last draft token), not q_0."""
    V, n = 8, 1_000_000
    q0 = _probs(24, 1, (V,), 1.5)
    q1 = _probs(24, 2, (V,), 1.5)
    q = np.broadcast_to(np.stack([q0, q1])[None], (n, 2, V))
    p = np.broadcast_to(q0[None, None], (n, 1, V))
    x = _draw(p, 24, 3)
    u = synth.uniform_u24(24, 4, (n, 2, 2))
    res = oracle.verify_chain_probs(q, p, x, u)
    assert (res.accepted == 1).all()
    assert _chisq_ok(res.token, q1, V, n) > 1e-3
