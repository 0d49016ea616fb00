"""Pins for the greedy-tree and Markov-head parts of the CPU oracle.

Tree: brute force over root-to-node paths (a path-based restatement, not the
oracle's incremental walk), the fan-out-1 tree equals the greedy chain, and the
all-wrong tree.  Markov head: W1 = 0 gives U exactly, an explicit V x V matrix
B = W1 W2 built by loops, chi-square of the sampled pair (x_1, x_2) against
p_1(x_1) p_2(x_2 | x_1), and the pages' two-position worked example.
"""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- tree
def _brute_force_tree(target, parents, tokens):
    """Walk every root-to-node path; a node is on an accepted path iff every
    edge on the path carries the argmax of the row above it."""
    g = np.argmax(target, -1)
    N1 = len(parents)
    best, best_path = 0, []
    for i in range(N1):
        path = []
        j = i
        while j != 0:
            path.append(j)
            j = parents[j]
        path.reverse()
        ok = all(tokens[n] == g[parents[n]] for n in path)
        if ok and (len(path) > len(best_path) or (len(path) == len(best_path) and i < best)):
            best, best_path = i, path
    return best_path, g[best]


@pytest.mark.parametrize("seed", range(6))
def test_tree_matches_brute_force(seed):
    V, N, max_depth = 3, 12, 5
    for r in range(20):
        u = synth.uniform_u24(seed, 100 + r, (N,))
        parents, depths = synth.random_tree(u, N, max_depth, 3)
        target = synth.normal(seed, 200 + r, (N + 1, V))
        g = np.argmax(target, -1)
        coin = synth.uniform_u24(seed, 300 + r, (N + 1,)) < 0.6
        rnd = synth.randint(seed, 400 + r, (N + 1,), V)
        tokens = np.where(coin, g[np.maximum(parents, 0)], rnd)
        tokens[0] = 0
        res = oracle.verify_tree_greedy(target[None], parents[None], tokens[None], max_depth)
        path, tok = _brute_force_tree(target, parents, tokens)
        assert res.path_len[0] == len(path)
        assert list(res.path_nodes[0, :len(path)]) == path
        assert (res.path_nodes[0, len(path):] == -1).all()
        assert res.token[0] == tok
        assert depths.max() <= max_depth


def test_fan_out_one_tree_is_the_greedy_chain():
    R, gamma, V = 30, 6, 5
    t = synth.normal(31, 1, (R, gamma + 1, V))
    g = np.argmax(t, -1)
    rnd = synth.randint(31, 2, (R, gamma), V)
    coin = synth.uniform_u24(31, 3, (R, gamma)) < 0.8
    x = np.where(coin, g[:, :gamma], rnd)
    acc, token, _, _ = oracle.verify_chain_greedy(t, x)
    parents = np.tile(np.arange(-1, gamma), (R, 1))
    tokens = np.concatenate([np.zeros((R, 1), dtype=np.int64), x], 1)
    res = oracle.verify_tree_greedy(t, parents, tokens, gamma)
    assert (res.path_len == acc).all() and (res.token == token).all()
    for r in range(R):
        assert list(res.path_nodes[r, :acc[r]]) == list(range(1, acc[r] + 1))


def test_all_wrong_tree():
    V, N = 6, 9
    u = synth.uniform_u24(32, 1, (N,))
    parents, _ = synth.random_tree(u, N, 4, 3)
    t = synth.normal(32, 2, (N + 1, V))
    g = np.argmax(t, -1)
    tokens = (g[np.maximum(parents, 0)] + 1) % V
    res = oracle.verify_tree_greedy(t[None], parents[None], tokens[None], 4)
    assert res.path_len[0] == 0 and res.token[0] == g[0] and (res.path_nodes[0] == -1).all()


def test_tree_sibling_tie_prefers_lowest_index():
    # root with two children carrying the same (correct) token: both accepted at depth 1
    t = np.array([[0.0, 5.0, 1.0], [9.0, 0.0, 0.0], [0.0, 0.0, 9.0]])
    parents = np.array([-1, 0, 0])
    tokens = np.array([0, 1, 1])
    res = oracle.verify_tree_greedy(t[None], parents[None], tokens[None], 2)
    assert res.path_len[0] == 1 and res.path_nodes[0, 0] == 1 and res.token[0] == 0


def test_tree_rejects_bad_parents():
    with pytest.raises(ValueError):
        oracle.verify_tree_greedy(np.zeros((1, 3, 2)), np.array([[-1, 2, 0]]), np.zeros((1, 3)), 3)


# --------------------------------------------------------------------------- Markov head
def test_markov_zero_factor_gives_base_logits():
    m = synth.markov(seed=41, R=3, gamma=4, V=37, rank=8)
    U, W2 = m.U.f64, m.W2.f64
    toks, logits, _, _ = oracle.markov_draft(U, np.zeros((37, 8)), W2, m.anchor, m.uniforms, 1.0)
    assert np.array_equal(logits, U)
    # with B = 0 each position is an independent draw from softmax(U_k)
    for k in range(4):
        t, _, _ = oracle.inverse_cdf(scipy.special.softmax(U[:, k], axis=-1), m.uniforms[:, k])
        assert (t == toks[:, k]).all()


def _explicit_B(W1, W2):
    V, rank = W1.shape
    B = np.zeros((V, V))
    for a in range(V):
        for v in range(V):
            s = 0.0
            for j in range(rank):
                s += W1[a, j] * W2[j, v]
            B[a, v] = s
    return B


def test_markov_matches_explicit_transition_matrix():
    V, rank, gamma = 7, 3, 5
    m = synth.markov(seed=42, R=4, gamma=gamma, V=V, rank=rank, w_scale=0.8)
    W1, W2, U = m.W1.f64, m.W2.f64, m.U.f64
    B = _explicit_B(W1, W2)
    for T in (1.0, 0.5, 0.0):
        toks, logits, _, _ = oracle.markov_draft(U, W1, W2, m.anchor, m.uniforms, T)
        prev = m.anchor.astype(np.int64)
        for k in range(gamma):
            np.testing.assert_allclose(logits[:, k], U[:, k] + B[prev], atol=1e-12)
            if T == 0.0:
                assert (toks[:, k] == np.argmax(U[:, k] + B[prev], -1)).all()
            prev = toks[:, k]


def _markov_block(U, W1, W2, anchor, u):
    m, V = u.shape[0], U.shape[-1]
    toks, _, _, _ = oracle.markov_draft(np.broadcast_to(U[None], (m, 2, V)), W1, W2, np.full(m, anchor), u, 1.0)
    return toks


def test_markov_pair_chi_square(pool):
    """(x_1, x_2) sampled by the head follows p_1(x_1) p_2(x_2 | x_1) over V^2 cells."""
    V, rank, n = 8, 4, 1_000_000
    m = synth.markov(seed=43, R=1, gamma=2, V=V, rank=rank, w_scale=1.0, u_scale=1.0)
    W1, W2, U = m.W1.f64, m.W2.f64, m.U.f64[0]
    anchor = 3
    B = _explicit_B(W1, W2)
    p1 = scipy.special.softmax(U[0] + B[anchor])
    p2 = scipy.special.softmax(U[1][None, :] + B, axis=-1)       # row = x_1
    expected = (p1[:, None] * p2).ravel()
    from conftest import split_rows
    u = synth.uniform_u24(43, 50, (n, 2))
    futs = [pool.submit(_markov_block, U, W1, W2, anchor, u[a:b]) for a, b in split_rows(n, 8)]
    toks = np.concatenate([f.result() for f in futs])
    counts = np.bincount(toks[:, 0] * V + toks[:, 1], minlength=V * V)
    assert scipy.stats.chisquare(counts, n * expected).pvalue > 1e-3


def test_markov_two_position_worked_example():
    """The pages' red-apple / blue-berry toy: a rank-2 transition bias restores the
    two-point joint that the product of marginals spreads over four pairs."""
    gold = json.load(open(os.path.join(GOLDEN, "two_position_joint.json")))
    vocab = gold["vocab"]
    ix = {w: i for i, w in enumerate(vocab)}
    NEG = -1e4
    U = np.array([[0.0, 0.0, NEG, NEG],       # position 1: red / blue
                  [NEG, NEG, 0.0, 0.0]])      # position 2: apple / berry
    W1 = np.zeros((4, 2)); W1[ix["red"], 0] = 1.0; W1[ix["blue"], 1] = 1.0
    W2 = np.zeros((2, 4))
    W2[0, ix["apple"]], W2[0, ix["berry"]] = 30.0, -30.0
    W2[1, ix["apple"]], W2[1, ix["berry"]] = -30.0, 30.0
    anchor = ix["apple"]                       # a token whose W1 row is zero

    def joint(W1_):
        L1, _, _, _ = oracle.markov_step(U[None, 0], W1_, W2, np.array([anchor]), np.array([0.0]), 1.0)
        p1 = oracle.softmax_t(L1, 1.0)[0]
        out = {}
        for a in ("red", "blue"):
            L2, _, _, _ = oracle.markov_step(U[None, 1], W1_, W2, np.array([ix[a]]), np.array([0.0]), 1.0)
            p2 = oracle.softmax_t(L2, 1.0)[0]
            for b in ("apple", "berry"):
                out[f"{a} {b}"] = p1[ix[a]] * p2[ix[b]]
        return out

    with_head = joint(W1)
    for pair, val in gold["joint"].items():
        assert abs(with_head[pair] - val) < 1e-20 if val == 0.0 else abs(with_head[pair] - val) < 1e-12
    off = sum(v for k, v in with_head.items() if gold["joint"][k] == 0.0)
    assert off < 1e-20
    independent = joint(np.zeros_like(W1))
    for pair, val in gold["product_of_marginals"].items():
        assert abs(independent[pair] - val) < 1e-12
    off = sum(v for k, v in independent.items() if gold["joint"][k] == 0.0)
    assert abs(off - gold["product_mass_off_support"]) < 1e-12


# --------------------------------------------------------------------------- DART tree construction
def _delta(p, i, v, eps=1e-10):
    """eq. (10) with g = 1, restated for the pins."""
    return (0.9 ** i * np.log(p[i - 1, v] + eps) + 0.5 * np.log(1.0 + eps)) / (i + 1) ** 0.7


def test_dart_tree_without_pruning_is_the_brute_force_selection():
    """w large enough that no path is dropped: T is every path over the per-offset
    top-k, and the tree is the theta largest bottleneck keys (ties: shallower),
    computed here by enumerating the paths."""
    rng = np.random.default_rng(61)
    d, V, k, theta = 3, 9, 3, 10
    x = rng.normal(size=(1, d, V)) * 2.0
    t = oracle.dart_tree(x, 1.0, k=k, w=k ** d, theta=theta)
    p = scipy.special.softmax(x[0], axis=-1)
    tops = [list(np.argsort(-p[i], kind="stable")[:k]) for i in range(d)]
    paths = []                                               # (key, depth, tokens)
    for depth in range(1, d + 1):
        for combo in itertools.product(*tops[:depth]):
            s, key = 0.0, np.inf
            for i, v in enumerate(combo, start=1):
                s += _delta(p, i, v)
                key = min(key, s)
            paths.append((key, depth, combo))
    assert t.n_expanded[0] == len(paths) == k + k ** 2 + k ** 3
    best = sorted(paths, key=lambda e: (-e[0], e[1]))[:theta]
    # rebuild each selected node's token path from the linearised tree
    got = []
    for i in range(1, t.n_nodes[0]):
        toks, j = [], i
        while j > 0:
            toks.append(int(t.tokens[0, j]))
            j = int(t.parents[0, j])
        got.append(tuple(reversed(toks)))
    assert sorted(got) == sorted(tuple(int(v) for v in c) for _, _, c in best)
    np.testing.assert_allclose(sorted(t.key[0, 1:], reverse=True), [b[0] for b in best], rtol=1e-12)


def test_dart_tree_masked_vocabulary_is_the_brute_force_selection():
    """Two finite logits per offset and k = 3: each offset's third pick is the
    lowest-id token of probability 0, scored with ln(0 + eps).  No path is
    dropped (w = k^d), so the tree is again the theta largest bottleneck keys
    over every path, enumerated here."""
    rng = np.random.default_rng(64)
    d, V, k, theta = 3, 9, 3, 12
    x = np.full((1, d, V), -np.inf)
    for i in range(d):
        ids = rng.choice(V, size=2, replace=False)
        x[0, i, ids] = rng.normal(size=2) * 2.0
    t = oracle.dart_tree(x, 1.0, k=k, w=k ** d, theta=theta)
    p = scipy.special.softmax(x[0], axis=-1)
    assert (p > 0).sum() == 2 * d
    tops = [list(np.argsort(-p[i], kind="stable")[:k]) for i in range(d)]
    paths = []
    for depth in range(1, d + 1):
        for combo in itertools.product(*tops[:depth]):
            s_, key = 0.0, np.inf
            for i, v in enumerate(combo, start=1):
                s_ += _delta(p, i, v)
                key = min(key, s_)
            paths.append((key, depth, combo))
    best = sorted(paths, key=lambda e: (-e[0], e[1]))
    assert (best[theta - 1][0], best[theta - 1][1]) != (best[theta][0], best[theta][1])   # no tie at the cut
    got = []
    for i in range(1, t.n_nodes[0]):
        toks, j = [], i
        while j > 0:
            toks.append(int(t.tokens[0, j]))
            j = int(t.parents[0, j])
        got.append(tuple(reversed(toks)))
    assert sorted(got) == sorted(tuple(int(v) for v in c) for _, _, c in best[:theta])
    for i in range(d):                                    # the masked pick is the lowest zero-probability id
        assert tops[i][2] == int(np.flatnonzero(p[i] == 0)[0])


def test_dart_tree_beam_of_one_is_the_argmax_chain_with_its_siblings():
    rng = np.random.default_rng(62)
    d, V, k = 4, 20, 3
    x = rng.normal(size=(1, d, V)) * 3.0
    t = oracle.dart_tree(x, 1.0, k=k, w=1, theta=d * k)
    assert t.n_expanded[0] == k * d and t.n_nodes[0] == d * k + 1
    # along the chain the parent of every depth-(i+1) node is the depth-i argmax
    g = np.argmax(x[0], axis=-1)
    for i in range(1, t.n_nodes[0]):
        dep = t.depth[0, i]
        par = t.parents[0, i]
        if dep > 1:
            assert t.depth[0, par] == dep - 1 and t.tokens[0, par] == g[dep - 2]


def test_dart_tree_expansion_bound_closure_and_key_order():
    """eq. (9): |T| = k + (d-1) w k once each level has w paths; parents precede
    children; keys never increase along a path; depth <= d."""
    x = 3.0 * synth.normal(63, 1, (2, 8, 500))
    t = oracle.dart_tree(x, 1.0, k=25, w=20, theta=59)
    assert (t.n_expanded == 25 + 7 * 20 * 25).all()          # 3525, the notes' bound met with equality
    assert (t.n_nodes == 60).all()
    for r in range(2):
        for i in range(1, 60):
            par = t.parents[r, i]
            assert 0 <= par < i
            assert t.depth[r, i] == t.depth[r, par] + 1 or par == 0 and t.depth[r, i] == 1
            assert t.key[r, i] <= t.key[r, par]
        assert t.depth[r].max() <= 8
