"""CPU oracle for lossless draft verification (TEST INFRASTRUCTURE).

This file is test infrastructure, not product code.  Only the tests, the smoke
check in ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import or run it.  The CUDA library never calls it and shares
no code with it.

It is a plain, slow, float64 restatement of what the verification path computes,
written from these pages:

* [DART notes]  "DART：把草稿并行生成之后，还要补上哪些依赖？" (DART reading notes,
  zhongzhuzhou.org, 2026-10-14): §2.2 eq. (2) expected accepted length; §2.3
  eq. (3)-(4) single-token speculative sampling (accept with min(1, q/p),
  rejection mass R, residual r = [q-p]_+ / R); §2.3 last paragraph and
  Algorithm 3 steps 9-10 (greedy verification of a candidate tree at T = 0).
* [DSpark guide] the DSpark paper guide (personal-site-bgy.pages.dev/ai-notes/dspark-paper-guide):
  the verification rule (accept x_k with min(1, p^t_k(x_k)/p^d_k(x_k)), strict
  left-to-right prefix survival, bonus token), the Markov head
  p_k(v | x0, x<k) = softmax(U_k(v) + B(x_{k-1}, v)), B = W1 W2, the analytic
  acceptance c*_k = 1 - 1/2 ||p^d_k - p^t_k||_1, and the greedy throughput
  scheduler (pool sorted by a_{r,j}, Theta = tau * SPS(B), break when Theta stops
  rising).
* [SD survey]  "投机解码综述" (zhifeiding.github.io, 2026-11-02): §1.2 the
  accept-and-correct step, §1.3 greedy verification = position-wise argmax,
  §2.1 tau = N + 1.

Notation follows the DART notes: q = target distribution, p = draft
distribution.  Probabilities are float64; bf16/float32 logits are widened to
float64 exactly by the caller.

Readings taken where the pages are silent, ambiguous or garbled:
  R1  temperature: q = softmax(target / T), p = softmax(draft / T); T = 0 means
      greedy (argmax) verification.
  R2  accept iff u < min(1, q(x)/p(x)) with u in [0, 1); p(x) = 0 accepts.
  R3  sampling from a weight vector w is by inverse CDF over ascending token
      id: y = min{v : C(v) > u * S}, C the running sum of w in index order and
      S = C(V-1).
  R4  if a rejection happens with S = sum [q-p]_+ == 0 (possible only through
      rounding), the correction token is drawn from q (no residual exists when
      R = 0, DART notes §2.3).
  R5  argmax ties resolve to the lowest token id; tree ties (two accepted
      nodes at the same depth) resolve to the lowest linear index.
  R6  the scheduler accumulates tau in fixed point with quantum 2**-48
      (a_{r,j} truncated), so that the sum is exact and independent of order;
      Theta_n = float(tau_n) * SPS(B_n) in float64.
  R7  c* at T = 0 is the T -> 0+ limit: 1 if the draft and target argmaxes
      agree, else 0.
  R13 the asynchronous scheduler's global search takes, among equal Theta_n,
      the smallest n (verifying fewer tokens for the same throughput), and
      counts n = 0 (bonus positions only) as a candidate.
  R14 the confidence head's linear projection is one weight vector w over the
      concatenation [h_k; W1[x_{k-1}]] plus a scalar bias; x_0 is the anchor.
  R15 DART's tree construction without the n-gram index uses g == 1 in eq. (10),
      depth i = 1..d for the future offsets (the notes leave the numbering
      open), eps = 1e-10, and generation order (path rank, then token rank) to
      break equal scores.
  R16 node selection: key = min(own score, parent's key); the theta largest keys,
      then the smaller depth, then generation order; ancestor-closed by
      construction (the notes ask for closure but give no rule).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "softmax_t", "inverse_cdf", "residual", "ChainResult", "verify_chain_probs", "verify_chain",
    "verify_chain_greedy", "tv_accept", "tv_accept_probs", "TreeResult", "verify_tree_greedy",
    "markov_step", "markov_draft", "ScheduleResult", "schedule", "survival_products", "schedule_global",
    "prune_threshold", "confidence_head", "DartTree", "dart_tree",
]


# --------------------------------------------------------------------------- basics
def softmax_t(logits: np.ndarray, temperature: float) -> np.ndarray:
    """softmax(logits / T) over the last axis in float64 (reading R1), with the
    row maximum subtracted before exponentiation."""
    if not temperature > 0.0:
        raise ValueError("softmax_t needs T > 0; T = 0 is the greedy path")
    z = np.asarray(logits, dtype=np.float64) / temperature
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def inverse_cdf(w: np.ndarray, u: np.ndarray):
    """Draw one index per row of the non-negative weights `w` [..., V] with the
    uniform `u` [...] (reading R3).

    Returns (token, c_lo, c_hi): token = min{v : C(v) > u*S}, and the two CDF
    values C(token-1)/S and C(token)/S that bracket u (a decision threshold for
    parity accounting).  Rows with S == 0 return token -1.
    """
    w = np.asarray(w, dtype=np.float64)
    C = np.cumsum(w, axis=-1)
    S = C[..., -1]
    target = np.asarray(u, dtype=np.float64) * S
    above = C > target[..., None]
    tok = np.argmax(above, axis=-1)
    ok = S > 0.0
    tok = np.where(ok, tok, -1)
    safe = np.where(ok, S, 1.0)
    hi = np.take_along_axis(C, np.maximum(tok, 0)[..., None], -1)[..., 0] / safe
    prev = np.where(tok > 0, np.take_along_axis(C, np.maximum(tok - 1, 0)[..., None], -1)[..., 0], 0.0)
    lo = prev / safe
    return tok.astype(np.int64), lo, hi


def residual(q: np.ndarray, p: np.ndarray):
    """Rejection mass and residual distribution (DART notes §2.3, eq. (3)):
    R = sum_v [q(v) - p(v)]_+ and r(v) = [q(v) - p(v)]_+ / R over the last axis.
    Returns (r, R); rows with R == 0 get r = NaN (no residual exists)."""
    pos = np.maximum(np.asarray(q, np.float64) - np.asarray(p, np.float64), 0.0)
    mass = pos.sum(axis=-1)
    with np.errstate(invalid="ignore", divide="ignore"):
        r = pos / mass[..., None]
    return r, mass


# --------------------------------------------------------------------------- chain
@dataclass
class ChainResult:
    accepted: np.ndarray        # int64 [R]  A_r: accepted draft tokens
    token: np.ndarray           # int64 [R]  correction (residual) or bonus token
    c_star: np.ndarray          # float64 [R, gamma], NaN where k >= l_r
    thr: np.ndarray             # float64 [R, gamma] accept threshold min(1, q/p), NaN where k >= l_r
    sample_at: np.ndarray       # int64 [R, gamma+1]  token emitted if the chain stopped at k
    lo_at: np.ndarray           # float64 [R, gamma+1]  CDF value below that token
    hi_at: np.ndarray           # float64 [R, gamma+1]  CDF value at that token
    resid_mass: np.ndarray      # float64 [R, gamma+1] S = sum [q-p]_+ at k (bonus column: 1)


def _lengths(lengths, R, gamma):
    if lengths is None:
        return np.full(R, gamma, dtype=np.int64)
    ell = np.asarray(lengths, dtype=np.int64)
    if ell.shape != (R,) or (ell < 0).any() or (ell > gamma).any():
        raise ValueError("lengths must be [R] with 0 <= l_r <= gamma")
    return ell


def verify_chain_probs(q: np.ndarray, p: np.ndarray, x: np.ndarray, u: np.ndarray, lengths=None) -> ChainResult:
    """Chain speculative sampling on probability rows.

    q [R, gamma+1, V] target distributions (row gamma' = l_r is the bonus row),
    p [R, gamma, V] draft distributions, x [R, gamma] draft tokens,
    u [R, gamma+1, 2] uniforms (u[...,0] accept test, u[...,1] correction/bonus draw).

    Per request (DART notes §2.3 eq. (3)-(4); DSpark guide, verification rule;
    SD survey §1.2 step 3):
      1. for k = 0 .. l_r-1 left to right, accept x_k iff u[k,0] < min(1, q_k(x_k)/p_k(x_k));
         the first rejection at k ends the chain: A = k (prefix survival);
      2. no rejection: A = l_r and the bonus token is drawn from q_{l_r};
      3. rejection at A: the correction token is drawn from the residual
         r = [q_A - p_A]_+ / R, R = sum_v [q_A(v) - p_A(v)]_+ (eq. (3)).
    c*_k = 1 - 1/2 sum_v |p_k(v) - q_k(v)| (DSpark guide, analytic acceptance).
    """
    q = np.asarray(q, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    x = np.asarray(x, dtype=np.int64)
    u = np.asarray(u, dtype=np.float64)
    R, gamma = x.shape
    V = q.shape[-1]
    assert q.shape == (R, gamma + 1, V) and p.shape == (R, gamma, V) and u.shape == (R, gamma + 1, 2)
    ell = _lengths(lengths, R, gamma)
    rows = np.arange(R)

    thr = np.full((R, gamma), np.nan)
    c_star = np.full((R, gamma), np.nan)
    sample_at = np.full((R, gamma + 1), -1, dtype=np.int64)
    lo_at = np.full((R, gamma + 1), np.nan)
    hi_at = np.full((R, gamma + 1), np.nan)
    resid_mass = np.full((R, gamma + 1), np.nan)

    for k in range(gamma + 1):
        live = k < ell            # position k is a draft position of request r
        bonus = k == ell          # position k is request r's bonus position
        if k < gamma:
            qk, pk = q[:, k], p[:, k]
            qx = qk[rows, x[:, k]]
            px = pk[rows, x[:, k]]
            ratio = np.divide(qx, px, out=np.full(R, np.inf), where=px > 0.0)
            thr[:, k] = np.where(live, np.minimum(1.0, ratio), np.nan)
            c_star[:, k] = np.where(live, 1.0 - 0.5 * np.abs(pk - qk).sum(axis=-1), np.nan)
            resid, S = residual(qk, pk)
            w = np.where((S > 0.0)[:, None], resid, qk)          # reading R4
            t, lo, hi = inverse_cdf(w, u[:, k, 1])
            sample_at[:, k] = np.where(live, t, sample_at[:, k])
            lo_at[:, k] = np.where(live, lo, lo_at[:, k])
            hi_at[:, k] = np.where(live, hi, hi_at[:, k])
            resid_mass[:, k] = np.where(live, S, resid_mass[:, k])
        t, lo, hi = inverse_cdf(q[:, k], u[:, k, 1])
        sample_at[:, k] = np.where(bonus, t, sample_at[:, k])
        lo_at[:, k] = np.where(bonus, lo, lo_at[:, k])
        hi_at[:, k] = np.where(bonus, hi, hi_at[:, k])
        resid_mass[:, k] = np.where(bonus, 1.0, resid_mass[:, k])

    accepted = ell.copy()
    for r in range(R):
        for k in range(ell[r]):
            if not (u[r, k, 0] < thr[r, k]):
                accepted[r] = k
                break
    token = sample_at[rows, accepted]
    return ChainResult(accepted, token, c_star, thr, sample_at, lo_at, hi_at, resid_mass)


def verify_chain_greedy(target: np.ndarray, draft_tokens: np.ndarray, lengths=None, draft=None):
    """Greedy (T = 0) chain verification (SD survey §1.3: verification reduces
    to a position-wise argmax comparison; correction/bonus = target argmax).

    g_k = argmax_v target[r, k, v] (lowest id on ties, reading R5);
    A = first k < l_r with x_k != g_k, else l_r; token = g_A.
    c*_k (reading R7) = [argmax draft_k == g_k] when `draft` is given.
    Returns (accepted [R], token [R], c_star [R, gamma] or None, g [R, gamma+1]).
    """
    target = np.asarray(target, dtype=np.float64)
    x = np.asarray(draft_tokens, dtype=np.int64)
    R, gamma = x.shape
    ell = _lengths(lengths, R, gamma)
    g = np.argmax(target, axis=-1)                 # first maximum = lowest id
    accepted = ell.copy()
    for r in range(R):
        for k in range(ell[r]):
            if x[r, k] != g[r, k]:
                accepted[r] = k
                break
    token = g[np.arange(R), accepted]
    c_star = None
    if draft is not None:
        gd = np.argmax(np.asarray(draft, dtype=np.float64), axis=-1)
        c_star = np.where(np.arange(gamma)[None, :] < ell[:, None], (gd == g[:, :gamma]).astype(np.float64), np.nan)
    return accepted, token, c_star, g


def verify_chain(target: np.ndarray, draft: np.ndarray, draft_tokens: np.ndarray, uniforms: np.ndarray,
                 temperature: float, lengths=None, block: int = 4):
    """Logit-level chain verification: T > 0 is speculative sampling on
    q = softmax(target/T), p = softmax(draft/T); T = 0 is the greedy path.

    `target` [R, gamma+1, V] and `draft` [R, gamma, V] are float64 logits.  Requests
    are processed `block` at a time to bound memory.  Returns a ChainResult
    (T > 0) or the tuple of verify_chain_greedy (T = 0)."""
    if temperature == 0.0:
        return verify_chain_greedy(target, draft_tokens, lengths, draft)
    R = target.shape[0]
    parts = []
    ell_all = None if lengths is None else np.asarray(lengths)
    for s in range(0, R, block):
        e = min(R, s + block)
        q = softmax_t(target[s:e], temperature)
        p = softmax_t(draft[s:e], temperature)
        parts.append(verify_chain_probs(q, p, draft_tokens[s:e], uniforms[s:e],
                                        None if ell_all is None else ell_all[s:e]))
    return ChainResult(*[np.concatenate([getattr(pt, f) for pt in parts]) for f in ChainResult.__dataclass_fields__])


# --------------------------------------------------------------------------- c*
def tv_accept_probs(q: np.ndarray, p: np.ndarray) -> np.ndarray:
    """c* = 1 - 1/2 ||p - q||_1 over the last axis (DSpark guide, analytic acceptance)."""
    return 1.0 - 0.5 * np.abs(np.asarray(p, np.float64) - np.asarray(q, np.float64)).sum(axis=-1)


def tv_accept(target: np.ndarray, draft: np.ndarray, temperature: float, block: int = 4) -> np.ndarray:
    """c*_{r,k} for k < gamma from target [R, P >= gamma, V] and draft [R, gamma, V]
    float64 logits; T = 0 gives the argmax-agreement indicator (reading R7)."""
    R, gamma, V = draft.shape
    if temperature == 0.0:
        return (np.argmax(draft, -1) == np.argmax(target[:, :gamma], -1)).astype(np.float64)
    out = np.empty((R, gamma))
    for s in range(0, R, block):
        e = min(R, s + block)
        out[s:e] = tv_accept_probs(softmax_t(target[s:e, :gamma], temperature), softmax_t(draft[s:e], temperature))
    return out


# --------------------------------------------------------------------------- tree
@dataclass
class TreeResult:
    path_len: np.ndarray        # int64 [R] accepted non-root nodes
    path_nodes: np.ndarray      # int64 [R, max_depth] root->leaf node ids, -1 padded
    token: np.ndarray           # int64 [R] target argmax at the deepest accepted node
    accepted: np.ndarray        # bool [R, N+1] per-node acceptance
    g: np.ndarray               # int64 [R, N+1] row argmax


def verify_tree_greedy(target: np.ndarray, parents: np.ndarray, tokens: np.ndarray, max_depth: int) -> TreeResult:
    """Greedy verification of a linearised candidate tree (DART notes §2.3 last
    paragraph: at T = 0 check the target argmax along candidate paths; Algorithm 3
    steps 9-10: ancestors are present and the accepted path is committed with the
    correction token; SD survey §2.3: the tree is linearised and verified in one
    forward).

    target [R, N+1, V] float64 logits, row i = the target distribution after node i
    (row 0 = after the root, i.e. the committed prefix).  parents [R, N+1] with
    parents[:, 0] = -1 and 0 <= parents[i] < i.  tokens[:, i] = the token of node i.

      g_i = argmax row i (lowest id);  node 0 accepted;  node i accepted iff its
      parent is accepted and tokens[i] == g_{parent(i)};  i* = accepted node of
      maximum depth, lowest index on ties (reading R5);  path = ancestors of i*
      below the root, root-to-leaf;  token = g_{i*}.
    """
    target = np.asarray(target, dtype=np.float64)
    parents = np.asarray(parents, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    R, N1 = parents.shape
    g = np.argmax(target, axis=-1)
    path_len = np.zeros(R, dtype=np.int64)
    path_nodes = np.full((R, max_depth), -1, dtype=np.int64)
    token = np.zeros(R, dtype=np.int64)
    accepted = np.zeros((R, N1), dtype=bool)
    for r in range(R):
        depth = np.zeros(N1, dtype=np.int64)
        accepted[r, 0] = True
        for i in range(1, N1):
            par = parents[r, i]
            if not (0 <= par < i):
                raise ValueError("parents must satisfy 0 <= parents[i] < i")
            depth[i] = depth[par] + 1
            if depth[i] > max_depth:
                raise ValueError("tree deeper than max_depth")
            accepted[r, i] = accepted[r, par] and tokens[r, i] == g[r, par]
        best = 0
        for i in range(1, N1):
            if accepted[r, i] and depth[i] > depth[best]:
                best = i
        path = []
        i = best
        while i != 0:
            path.append(i)
            i = parents[r, i]
        path.reverse()
        path_len[r] = len(path)
        path_nodes[r, :len(path)] = path
        token[r] = g[r, best]
    return TreeResult(path_len, path_nodes, token, accepted, g)


# --------------------------------------------------------------------------- Markov head
def markov_step(U_k: np.ndarray, W1: np.ndarray, W2: np.ndarray, x_prev: np.ndarray, u: np.ndarray,
                temperature: float):
    """One serial step of the DSpark Markov head (DSpark guide, Markov head:
    p_k(v | x0, x<k) = softmax(U_k(v) + B(x_{k-1}, v)), B = W1 W2 with W1 [V, r]
    used as a row lookup and W2 [r, V] as the projection).

    U_k [R, V], W1 [V, r], W2 [r, V] float64; x_prev [R] token ids; u [R].
    L = U_k + W1[x_prev] @ W2 (raw logits); x = inverse-CDF draw from
    softmax(L / T) (T = 0: argmax, lowest id).  Returns (L, x, lo, hi)."""
    x_prev = np.asarray(x_prev, dtype=np.int64)
    L = np.asarray(U_k, np.float64) + np.asarray(W1, np.float64)[x_prev] @ np.asarray(W2, np.float64)
    if temperature == 0.0:
        x = np.argmax(L, axis=-1)
        return L, x, np.full(x.shape, np.nan), np.full(x.shape, np.nan)
    x, lo, hi = inverse_cdf(softmax_t(L, temperature), u)
    return L, x, lo, hi


def markov_draft(U: np.ndarray, W1: np.ndarray, W2: np.ndarray, anchor: np.ndarray, uniforms: np.ndarray,
                 temperature: float):
    """Semi-autoregressive drafting with the Markov head (DSpark guide): x_0 is
    the anchor; for k = 1..gamma, x_k is drawn from p_k(. | x_{k-1}) with the
    uniform uniforms[:, k-1].  U [R, gamma, V] are the parallel base logits.
    Returns (tokens [R, gamma], logits [R, gamma, V], lo [R, gamma], hi [R, gamma])."""
    R, gamma, V = U.shape
    toks = np.zeros((R, gamma), dtype=np.int64)
    logits = np.zeros((R, gamma, V))
    lo = np.zeros((R, gamma))
    hi = np.zeros((R, gamma))
    x = np.asarray(anchor, dtype=np.int64)
    for k in range(gamma):
        L, x, l_, h_ = markov_step(U[:, k], W1, W2, x, uniforms[:, k], temperature)
        toks[:, k], logits[:, k], lo[:, k], hi[:, k] = x, L, l_, h_
    return toks, logits, lo, hi


# --------------------------------------------------------------------------- scheduler
QUANTUM_BITS = 48


def survival_products(conf: np.ndarray) -> np.ndarray:
    """a_{r,j} = prod_{i <= j} c_{r,i}, float64, multiplied left to right
    (DSpark guide, scheduler: survival probability of prefix position j)."""
    conf = np.asarray(conf)
    R, gamma = conf.shape
    a = np.empty((R, gamma), dtype=np.float64)
    for r in range(R):
        prod = 1.0
        for j in range(gamma):
            prod = prod * float(conf[r, j])
            a[r, j] = prod
    return a


@dataclass
class ScheduleResult:
    lengths: np.ndarray         # int64 [R] l_r
    theta_best: float           # best Theta (tau in token units * SPS)
    n_included: int             # pool entries included


def schedule(conf: np.ndarray, sps: np.ndarray, B_max: int | None = None) -> ScheduleResult:
    """Greedy throughput scheduler (DSpark guide, scheduler section):
    a_{r,j} = prod_{i<=j} c_{r,i}; B = sum_r (1 + l_r); tau = sum_r (1 + sum_{j<=l_r} a_{r,j});
    Theta = tau * SPS(B).  All (r, j) go into one pool sorted by a descending
    (ties: r, then j ascending); entries are taken from the top, updating B and
    tau, and the loop breaks as soon as Theta <= Theta_best (early stop), which
    keeps every truncation independent of later tokens.  The lengths at
    Theta_best are returned.  sps[B-1] = SPS(B); B may not exceed B_max
    (default len(sps)).  tau is kept in fixed point (reading R6)."""
    conf = np.asarray(conf)
    sps = np.asarray(sps, dtype=np.float64)
    R, gamma = conf.shape
    if B_max is None:
        B_max = len(sps)
    if B_max < R or B_max > len(sps):
        raise ValueError("need R <= B_max <= len(sps)")
    a = survival_products(conf)
    pool = sorted(((a[r, j], r, j) for r in range(R) for j in range(gamma)),
                  key=lambda e: (-e[0], e[1], e[2]))
    Q = 1 << QUANTUM_BITS
    tau = R * Q                  # every request verifies its bonus position: tau = sum_r 1
    B = R
    theta_best = float(tau) * sps[B - 1]
    ell = np.zeros(R, dtype=np.int64)
    n = 0
    for a_rj, r, j in pool:
        if B + 1 > B_max:
            break
        tau_next = tau + int(math.floor(a_rj * Q))
        theta = float(tau_next) * sps[B]          # SPS(B + 1)
        if theta <= theta_best:
            break
        tau, B, theta_best = tau_next, B + 1, theta
        if j != ell[r]:
            raise AssertionError("pool order broke prefix closure")
        ell[r] += 1
        n += 1
    return ScheduleResult(ell, theta_best / Q, n)


def schedule_global(conf: np.ndarray, sps: np.ndarray, B_max: int | None = None,
                    conf_stale: np.ndarray | None = None) -> ScheduleResult:
    """The asynchronous form of the scheduler (DSpark guide, production
    deployment): the early stop is removed and the number of pool entries K is
    the one that maximises Theta_n = tau_n * SPS(R + n) over every
    n = 0 .. min(R * gamma, B_max - R), searched globally; on equal Theta the
    smallest n (reading R13).  K is computed from `conf_stale`, confidence-head
    outputs two steps old (default: `conf`), which keeps the truncation
    independent of the tokens being verified; the entries verified are then the
    top K of the pool ordered by the current survival products (dynamic top-K).
    tau, the pool order and Theta_n are those of `schedule` (reading R6).
    Returns the lengths from the current pool, Theta_K of the stale pool (in
    token units) and K."""
    conf = np.asarray(conf)
    stale = conf if conf_stale is None else np.asarray(conf_stale)
    sps = np.asarray(sps, dtype=np.float64)
    R, gamma = conf.shape
    if stale.shape != conf.shape:
        raise ValueError("conf_stale must have the shape of conf")
    if B_max is None:
        B_max = len(sps)
    if B_max < R or B_max > len(sps):
        raise ValueError("need R <= B_max <= len(sps)")
    Q = 1 << QUANTUM_BITS

    def pool(c):
        a = survival_products(c)
        return sorted(((a[r, j], r, j) for r in range(R) for j in range(gamma)),
                      key=lambda e: (-e[0], e[1], e[2]))

    tau = R * Q
    best_n, best_theta = 0, float(tau) * sps[R - 1]
    for n, (a_rj, _, _) in enumerate(pool(stale), start=1):
        if R + n > B_max:
            break
        tau += int(math.floor(a_rj * Q))
        theta = float(tau) * sps[R + n - 1]
        if theta > best_theta:
            best_n, best_theta = n, theta
    ell = np.zeros(R, dtype=np.int64)
    for _, r, j in pool(conf)[:best_n]:
        if j != ell[r]:
            raise AssertionError("pool order broke prefix closure")
        ell[r] += 1
    return ScheduleResult(ell, best_theta / Q, best_n)


def confidence_head(h: np.ndarray, W1: np.ndarray, w: np.ndarray, b: float, anchor: np.ndarray,
                    draft_tokens: np.ndarray) -> np.ndarray:
    """DSpark's confidence head (DSpark guide, confidence head: a light linear
    projection plus a sigmoid over the backbone hidden state h_k and the Markov
    embedding W1[x_{k-1}], giving the conditional survival probability c_k):
    c_{r,k} = 1 / (1 + exp(-(w[:H] . h[r,k] + w[H:] . W1[x_{r,k-1}] + b))) in float64,
    with x_{r,0} = anchor[r] and x_{r,k-1} = draft_tokens[r, k-2] for k >= 2
    (reading R14).  h [R, gamma, H], W1 [V, r], w [H + r]; returns [R, gamma]."""
    h = np.asarray(h, np.float64)
    W1 = np.asarray(W1, np.float64)
    w = np.asarray(w, np.float64)
    R, gamma, H = h.shape
    prev = np.concatenate([np.asarray(anchor, np.int64)[:, None],
                           np.asarray(draft_tokens, np.int64)[:, :gamma - 1]], axis=1)      # x_{k-1}
    z = h @ w[:H] + W1[prev] @ w[H:] + float(b)
    return 1.0 / (1.0 + np.exp(-z))


@dataclass
class DartTree:
    parents: np.ndarray         # int64 [R, theta+1]; parents[:, 0] = -1; -1 padding past n_nodes
    tokens: np.ndarray          # int64 [R, theta+1]; tokens[:, 0] = the root placeholder 0
    n_nodes: np.ndarray         # int64 [R]: 1 + selected nodes
    depth: np.ndarray           # int64 [R, theta+1]
    key: np.ndarray             # float64 [R, theta+1]: selection key of each node (root: +inf)
    n_expanded: np.ndarray      # int64 [R]: nodes generated (|T|, DART notes eq. (9))


def dart_tree(draft_logits: np.ndarray, temperature: float = 1.0, k: int = 25, w: int = 20, theta: int = 59,
              eps: float = 1e-10) -> DartTree:
    """DART's candidate-tree construction without the n-gram term (DART notes
    §5.2 and Algorithm 3 steps 1-8, with g == 1; reading R15):

      p_i = softmax(draft_logits[:, i-1] / T) for the future offsets i = 1..d;
      active paths C = {root, score 0}; for i = 1..d: K_i = the top-k tokens of
      p_i (lower id first on equal p); every path in C (in its order) is extended
      by every token of K_i (in K_i's order) with
        s_new = s_parent + (0.9^i log(p_i(v) + eps) + 0.5 log(1 + eps)) / (i + 1)^0.7   (eq. 10);
      all extensions enter the node set T; the w best (score descending, then
      generation order) become C.
    Node selection (reading R16): key(node) = min(s_node, key(parent)), root key
    +inf; the theta nodes with the largest key (then smaller depth, then
    generation order) are taken.  Keys never increase along a path and ties go to
    the shallower node, so the selection contains every selected node's parents.
    Linearisation: depth-first preorder from the root, children in selection
    order; row 0 is the root (the committed prefix)."""
    x = np.asarray(draft_logits, dtype=np.float64)
    R, d, V = x.shape
    out_par = np.full((R, theta + 1), -1, dtype=np.int64)
    out_tok = np.zeros((R, theta + 1), dtype=np.int64)
    out_dep = np.zeros((R, theta + 1), dtype=np.int64)
    out_key = np.full((R, theta + 1), -np.inf)
    n_nodes = np.zeros(R, dtype=np.int64)
    n_exp = np.zeros(R, dtype=np.int64)
    for r in range(R):
        p = softmax_t(x[r], temperature)                  # [d, V]
        # nodes: (score, key, depth, parent node id, token); node id = generation order
        nodes = []
        active = [(-1, 0.0, math.inf)]                    # (node id, score, key); -1 = root
        for i in range(1, d + 1):
            order = sorted(range(V), key=lambda v: (-p[i - 1, v], v))[:k]
            scale = (i + 1) ** 0.7
            ext = []
            for (pid, ps, pk) in active:
                for v in order:
                    s = ps + (0.9 ** i * math.log(p[i - 1, v] + eps) + 0.5 * math.log(1.0 + eps)) / scale
                    nid = len(nodes)
                    nodes.append((s, min(s, pk), i, pid, v))
                    ext.append((nid, s, min(s, pk)))
            ext.sort(key=lambda e: (-e[1], e[0]))
            active = ext[:w]
        sel = sorted(range(len(nodes)), key=lambda n: (-nodes[n][1], nodes[n][2], n))[:theta]
        chosen = set(sel)
        rank = {n: j for j, n in enumerate(sel)}
        children = {}
        for n in sel:
            par = nodes[n][3]
            if par != -1 and par not in chosen:
                raise AssertionError("selection is not ancestor-closed")
            children.setdefault(par, []).append(n)
        for ch in children.values():
            ch.sort(key=lambda n: rank[n])
        # depth-first preorder
        row = {-1: 0}
        out_par[r, 0] = -1
        out_key[r, 0] = math.inf
        stack = list(reversed(children.get(-1, [])))
        nxt = 1
        while stack:
            n = stack.pop()
            row[n] = nxt
            out_par[r, nxt] = row[nodes[n][3]]
            out_tok[r, nxt] = nodes[n][4]
            out_dep[r, nxt] = nodes[n][2]
            out_key[r, nxt] = nodes[n][1]
            nxt += 1
            stack.extend(reversed(children.get(n, [])))
        n_nodes[r] = nxt
        n_exp[r] = len(nodes)
    return DartTree(out_par, out_tok, n_nodes, out_dep, out_key, n_exp)


def prune_threshold(conf: np.ndarray, threshold: float) -> np.ndarray:
    """Confidence-threshold suffix pruning (SD survey §6.1): with the prefix
    survival s_{r,i} = prod_{j<=i} c_{r,j} (float64, left to right), the draft of
    request r is cut before its first position with s_{r,i} < threshold, so
    l_r = #{i : s_{r,i} >= threshold} (s does not increase along i)."""
    s = survival_products(conf)
    keep = s >= float(threshold)
    ell = np.zeros(s.shape[0], dtype=np.int64)
    for r in range(s.shape[0]):
        i = 0
        while i < s.shape[1] and keep[r, i]:
            i += 1
        ell[r] = i
    return ell
