"""Pins for the greedy throughput scheduler in the CPU oracle (DSpark guide,
scheduler section): brute force over every length vector when Theta is unimodal,
the early stop at the first local maximum when it is not, the two SPS limits
with closed-form answers, ties, the batch cap, and the fixed-point reading."""
import itertools

import numpy as np
import pytest

import oracle
import synth


def _theta(a, ell, sps):
    R = a.shape[0]
    tau = sum(1.0 + a[r, :ell[r]].sum() for r in range(R))
    B = sum(1 + ell[r] for r in range(R))
    return tau * sps[B - 1]


def test_survival_products_are_left_to_right_products():
    c = np.array([[0.5, 0.5, 1.0, 0.25]], dtype=np.float32)
    a = oracle.survival_products(c)
    assert list(a[0]) == [0.5, 0.25, 0.25, 0.0625]
    c = synth.confidences(51, 10, 7)
    a = oracle.survival_products(c)
    assert (np.diff(a, axis=1) <= 0).all()       # non-increasing in j


def test_constant_sps_takes_everything():
    c = synth.confidences(52, 6, 5)
    res = oracle.schedule(c, np.full(64, 7.0))
    assert (res.lengths == 5).all() and res.n_included == 30


def test_inverse_square_sps_takes_nothing():
    # tau <= B, so Theta_n / Theta_{n-1} <= B / (B + 1) < 1 for SPS = B^-2
    c = synth.confidences(53, 6, 5, mean=4.0)
    sps = 1.0 / np.arange(1, 65, dtype=np.float64) ** 2
    res = oracle.schedule(c, sps)
    assert (res.lengths == 0).all() and res.n_included == 0
    assert res.theta_best == 6 * sps[5]


@pytest.mark.parametrize("seed", range(8))
def test_greedy_equals_brute_force_when_unimodal(seed):
    R, gamma = 3, 3
    c = synth.confidences(60 + seed, R, gamma, mean=1.0, sd=1.5)
    B = np.arange(1, 13, dtype=np.float64)
    sps = 100.0 / (1.0 + 0.15 * B + 0.01 * B * B)
    a = oracle.survival_products(c)
    best = max(_theta(a, ell, sps) for ell in itertools.product(range(gamma + 1), repeat=R))
    res = oracle.schedule(c, sps)
    assert abs(res.theta_best - best) <= 1e-9 * best
    assert abs(_theta(a, res.lengths, sps) - best) <= 1e-9 * best


def test_non_unimodal_stops_at_first_local_maximum():
    """Theta dips and then rises past its first peak: the early-stop rule keeps the
    first peak (the DSpark guide's break on Theta <= Theta_best), not the global one."""
    R, gamma = 2, 3
    c = np.full((R, gamma), 0.9, dtype=np.float32)
    sps = np.array([10.0, 10.0, 10.0, 7.0, 9.0, 9.0, 9.0, 9.0])  # SPS(B) for B = 1..8
    res = oracle.schedule(c, sps)
    a = oracle.survival_products(c)
    # B = 2 -> 3 rises (tau 2 -> 2.9, SPS 10); B = 4 drops (SPS 7): stop with one entry
    assert res.n_included == 1 and list(res.lengths) == [1, 0]
    glob = max(_theta(a, ell, sps) for ell in itertools.product(range(gamma + 1), repeat=R))
    assert res.theta_best < glob


def test_ties_go_to_lower_request_then_lower_position():
    c = np.array([[1.0, 0.5], [1.0, 1.0]], dtype=np.float32)
    # a = [[1, .5], [1, 1]]: pool order (1,r0,j0) (1,r1,j0) (1,r1,j1) (.5,r0,j1)
    sps = np.full(8, 1.0)
    res = oracle.schedule(c, sps, B_max=3)
    assert list(res.lengths) == [1, 0]
    res = oracle.schedule(c, sps, B_max=5)
    assert list(res.lengths) == [1, 2]


def test_batch_cap():
    c = synth.confidences(54, 4, 7)
    res = oracle.schedule(c, np.full(64, 1.0), B_max=6)
    assert res.lengths.sum() == 2 and res.n_included == 2
    with pytest.raises(ValueError):
        oracle.schedule(c, np.full(64, 1.0), B_max=3)


def test_equal_theta_stops():
    # an entry with a = 0 adds to B but not to tau; with constant SPS, Theta stays equal -> stop
    c = np.array([[1.0, 0.0, 1.0]], dtype=np.float32)
    res = oracle.schedule(c, np.full(8, 2.0))
    assert list(res.lengths) == [1]


def test_fixed_point_reading_matches_real_arithmetic_on_random_cases():
    """Reading R6 quantises a to 2^-48; away from exact ties it chooses what a
    float64 evaluation of the same greedy loop chooses."""
    for seed in range(5):
        c = synth.confidences(70 + seed, 40, 7)
        sps = synth.sps_table(512)
        res = oracle.schedule(c, sps)
        a = oracle.survival_products(c)
        order = sorted(((a[r, j], r, j) for r in range(40) for j in range(7)), key=lambda e: (-e[0], e[1], e[2]))
        tau, B, best, n = 40.0, 40, 40.0 * sps[39], 0
        for av, r, j in order:
            th = (tau + av) * sps[B]
            if th <= best:
                break
            tau, B, best, n = tau + av, B + 1, th, n + 1
        assert n == res.n_included
        assert abs(best - res.theta_best) <= 1e-12 * best


# --------------------------------------------------------------------------- asynchronous form
def _brute_best(a, sps, B_max):
    """max over every length vector of tau * SPS(B) (plain float64 sums), with
    the smallest B among the maxima."""
    R, gamma = a.shape
    best = None
    for ell in itertools.product(range(gamma + 1), repeat=R):
        B = R + sum(ell)
        if B > B_max:
            continue
        th = _theta(a, ell, sps)
        if best is None or th > best[0] * (1 + 1e-12) or (abs(th - best[0]) <= 1e-12 * best[0] and B < best[1]):
            best = (th, B)
    return best


@pytest.mark.parametrize("seed", range(6))
def test_global_search_equals_brute_force_over_all_lengths(seed):
    """With stale = current confidences the global search is the optimum over
    every length vector: the top-n entries maximise tau for each batch size
    because a_{r,j} does not increase with j (DSpark guide, scheduler)."""
    rng = np.random.default_rng(900 + seed)
    R, gamma = 3, 3
    c = rng.uniform(0.05, 1.0, size=(R, gamma)).astype(np.float32)
    sps = rng.uniform(0.2, 1.0, size=R * gamma + R).astype(np.float64)     # arbitrary, not unimodal
    res = oracle.schedule_global(c, sps)
    a = oracle.survival_products(c)
    th, B = _brute_best(a, sps, len(sps))
    assert res.theta_best == pytest.approx(th, rel=1e-12)
    assert R + res.n_included == B
    assert _theta(a, res.lengths, sps) == pytest.approx(th, rel=1e-12)


def test_global_search_never_below_the_early_stop():
    for seed in range(8):
        c = synth.confidences(700 + seed, 16, 5)
        sps = synth.sps_table(128)
        g = oracle.schedule_global(c, sps)
        e = oracle.schedule(c, sps)
        assert g.theta_best >= e.theta_best
        # the smooth decreasing table keeps Theta unimodal here: the two agree
        assert (g.lengths == e.lengths).all()


def test_saw_tooth_table_global_search_passes_the_cliff():
    """SPS falls from 10 to 4 at B = 2 and then stays flat: the early stop halts
    at n = 0 (Theta_1 = 1.9 * 4 < 10), the global search takes all three entries
    (Theta_3 = (1 + 0.9 + 0.81 + 0.729) * 4 = 13.756)."""
    c = np.array([[0.9, 0.9, 0.9]], dtype=np.float64)
    sps = np.array([10.0, 4.0, 4.0, 4.0])
    assert oracle.schedule(c, sps).lengths.tolist() == [0]
    g = oracle.schedule_global(c, sps)
    assert g.lengths.tolist() == [3] and g.n_included == 3
    assert g.theta_best == pytest.approx(3.439 * 4.0, rel=1e-12)


def test_stale_confidences_set_K_current_ones_pick_the_entries():
    """K = 1 from the stale pool (Theta: 2 * 1 = 2, 2.9 * 0.8 = 2.32, 3.0 * 0.7 = 2.1);
    the one entry taken is the current pool's top, request 1."""
    stale = np.array([[0.9], [0.1]])
    cur = np.array([[0.1], [0.9]])
    sps = np.array([5.0, 1.0, 0.8, 0.7])
    g = oracle.schedule_global(cur, sps, conf_stale=stale)
    assert g.n_included == 1
    assert g.lengths.tolist() == [0, 1]
    assert g.theta_best == pytest.approx(2.9 * 0.8, rel=1e-12)


def test_global_ties_take_the_smallest_n_and_respect_the_cap():
    c = np.array([[0.5, 0.0, 0.0]])
    sps = np.full(8, 2.0)                      # Theta_1 = Theta_2 = Theta_3 = 3.0
    g = oracle.schedule_global(c, sps)
    assert g.n_included == 1 and g.lengths.tolist() == [1]
    c = synth.confidences(55, 4, 3)
    g = oracle.schedule_global(c, np.full(64, 1.0), B_max=5)     # R + n <= 5
    assert g.n_included == 1 and g.lengths.sum() == 1


# --------------------------------------------------------------------------- threshold pruning
def test_prune_threshold_hand_cases():
    c = np.array([[0.9, 0.9, 0.5, 1.0], [0.4, 1.0, 1.0, 1.0], [0.5, 1.0, 1.0, 0.5]])
    # s = [0.9, 0.81, 0.405, 0.405], [0.4, 0.4, 0.4, 0.4], [0.5, 0.5, 0.5, 0.25]
    assert oracle.prune_threshold(c, 0.5).tolist() == [2, 0, 3]     # s >= threshold is kept
    assert oracle.prune_threshold(c, 0.0).tolist() == [4, 4, 4]
    assert oracle.prune_threshold(c, 1.5).tolist() == [0, 0, 0]


def test_prune_threshold_is_the_survival_count_and_monotone():
    c = synth.confidences(56, 32, 7)
    s = oracle.survival_products(c)
    prev = None
    for th in np.linspace(0.0, 1.0, 21):
        ell = oracle.prune_threshold(c, th)
        assert (ell == (s >= th).sum(axis=1)).all()   # s does not increase, so the kept set is a prefix
        if prev is not None:
            assert (ell <= prev).all()
        prev = ell


# --------------------------------------------------------------------------- confidence head
def test_confidence_head_zero_weights_give_the_sigmoid_of_the_bias():
    rng = np.random.default_rng(3)
    h = rng.normal(size=(2, 3, 8))
    W1 = rng.normal(size=(10, 4))
    c = oracle.confidence_head(h, W1, np.zeros(12), 0.7, np.array([1, 2]), np.array([[3, 4, 5], [6, 7, 8]]))
    np.testing.assert_allclose(c, 1.0 / (1.0 + np.exp(-0.7)), rtol=0, atol=0)


def test_confidence_head_hand_case_and_the_previous_token():
    """One-hot features: h_k = e_k, W1[v] = v * e_0 (rank 2), w = [1, 2, 3 | 0.5, 0],
    b = -1: z_k = w_h[k] + 0.5 * x_{k-1} - 1 with x_0 the anchor."""
    H, r = 3, 2
    h = np.eye(3)[None]                               # [1, 3, 3]: h_k = e_k
    W1 = np.zeros((10, r)); W1[:, 0] = np.arange(10)
    w = np.array([1.0, 2.0, 3.0, 0.5, 0.0])
    c = oracle.confidence_head(h, W1, w, -1.0, np.array([4]), np.array([[6, 2, 9]]))
    z = np.array([1.0 + 0.5 * 4 - 1.0, 2.0 + 0.5 * 6 - 1.0, 3.0 + 0.5 * 2 - 1.0])     # the last draft token is unused
    expect = [1.0 / (1.0 + np.exp(-x)) for x in z]
    np.testing.assert_allclose(c[0], expect, rtol=1e-15)
    assert 0.0 < c.min() and c.max() < 1.0


def test_confidence_head_matches_scipy_expit_and_flips_with_the_sign():
    import scipy.special
    rng = np.random.default_rng(4)
    R, gamma, H, r, V = 5, 4, 16, 8, 30
    h, W1, w = rng.normal(size=(R, gamma, H)), rng.normal(size=(V, r)), rng.normal(size=H + r)
    a, x = rng.integers(0, V, R), rng.integers(0, V, (R, gamma))
    c = oracle.confidence_head(h, W1, w, 0.3, a, x)
    prev = np.concatenate([a[:, None], x[:, :gamma - 1]], axis=1)
    z = np.einsum("rkh,h->rk", h, w[:H]) + np.einsum("rki,i->rk", W1[prev], w[H:]) + 0.3
    np.testing.assert_allclose(c, scipy.special.expit(z), rtol=1e-13)
    np.testing.assert_allclose(oracle.confidence_head(h, W1, -w, -0.3, a, x), 1.0 - c, atol=1e-14)
