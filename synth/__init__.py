"""Seeded synthetic inputs for lossless draft verification.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It holds no arithmetic of the verification method itself: it only
draws random numbers and shapes them into logits, token ids, trees, uniforms and
confidence tables with the sizes and value distributions of the workloads the
pages describe (synthetic stand-ins; no dataset, prompt or trained weight is
used).

Random source: PCG-XSH-RR 64/32 ("pcg32"), written from M. O'Neill's published
description (64-bit LCG state, multiplier 6364136223846793005, odd increment
selecting the stream; output = rotate_right(((s >> 18) ^ s) >> 27, s >> 59)).
A tensor is filled by `LANES` pcg32 generators in lock-step: element
`j*LANES + i` is the j-th draw of lane i, lane i seeded with
initseq = (stream << 20) + i and initstate = SplitMix64 of (seed, stream, i)
(Steele, Lea and Flood's published mixer), so that lanes do not start on an
arithmetic progression.  Everything is integer arithmetic, so the draws are
identical on every machine.

Uniforms for the method are u = (x >> 8) * 2**-24: exactly representable in
float32 and float64, in [0, 1).  Gaussians come from Box-Muller on two such
draws.  bf16 tensors are carried as uint16 bit patterns (round-to-nearest-even
from float64).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

LANES = 1 << 20
_BLOCKS = 16                     # lane blocks filled by worker threads (result does not depend on it)
_MULT = np.uint64(6364136223846793005)
_TWO_M24 = 2.0 ** -24
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)


def splitmix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output mixing (Steele, Lea and Flood, 2014) applied to uint64 z."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def _pool():
    return ThreadPoolExecutor(max_workers=min(_BLOCKS, os.cpu_count() or 1))


# --------------------------------------------------------------------------- pcg32
class Pcg32Lanes:
    """`lanes` pcg32 generators advanced together (vectorised with numpy)."""

    def __init__(self, seed: int, stream: int, lanes: int = LANES):
        with np.errstate(over="ignore"):
            seq = (np.uint64(stream) << np.uint64(20)) + np.arange(lanes, dtype=np.uint64)
            self.inc = (seq << np.uint64(1)) | np.uint64(1)
            # per-lane initstate from SplitMix64 so that lane states are not an
            # arithmetic progression in the lane index (which makes the lanes'
            # same-step outputs a lattice)
            base = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ (np.uint64(stream) * np.uint64(0xD1B54A32D192ED03))
            initstate = splitmix64(base + (np.arange(lanes, dtype=np.uint64) + np.uint64(1)) * _GOLDEN)
            self.state = np.zeros(lanes, dtype=np.uint64)
            self.state = self._step(self.state, self.inc)[0]
            self.state = self.state + initstate
            self.state = self._step(self.state, self.inc)[0]

    @staticmethod
    def _step(state, inc):
        """Advance `state`; return (new_state, output of the old state)."""
        with np.errstate(over="ignore"):
            new = state * _MULT + inc
        xorshifted = (((state >> np.uint64(18)) ^ state) >> np.uint64(27)).astype(np.uint32)
        rot = (state >> np.uint64(59)).astype(np.uint32)
        left = (np.uint32(32) - rot) & np.uint32(31)
        return new, (xorshifted >> rot) | (xorshifted << left)

    def _next(self) -> np.ndarray:
        self.state, out = self._step(self.state, self.inc)
        return out

    def draws(self, n: int) -> np.ndarray:
        """n uint32 draws; element j*lanes+i is the j-th draw of lane i."""
        lanes = self.state.shape[0]
        steps = (n + lanes - 1) // lanes
        out = np.empty((steps, lanes), dtype=np.uint32)
        bounds = np.linspace(0, lanes, _BLOCKS + 1).astype(np.int64)

        def fill(b):
            lo, hi = bounds[b], bounds[b + 1]
            st, inc = self.state[lo:hi].copy(), self.inc[lo:hi]
            for s in range(steps):
                st, out[s, lo:hi] = self._step(st, inc)
            return st

        with _pool() as ex:
            states = list(ex.map(fill, range(_BLOCKS)))
        self.state = np.concatenate(states)
        return out.reshape(-1)[:n]


def uniform_u24(seed: int, stream: int, shape) -> np.ndarray:
    """Uniforms k * 2**-24 in [0, 1) as float64 (exact in float32 too)."""
    n = int(np.prod(shape))
    x = Pcg32Lanes(seed, stream).draws(n)
    return ((x >> np.uint32(8)).astype(np.float64) * _TWO_M24).reshape(shape)


def uniform_f32(seed: int, stream: int, shape) -> np.ndarray:
    return uniform_u24(seed, stream, shape).astype(np.float32)


def normal(seed: int, stream: int, shape) -> np.ndarray:
    """Standard normals (float64) by Box-Muller on pcg32 uniforms."""
    n = int(np.prod(shape))
    half = (n + 1) // 2
    u = uniform_u24(seed, stream, (2 * half,))
    z = np.empty(2 * half, dtype=np.float64)
    bounds = np.linspace(0, half, _BLOCKS + 1).astype(np.int64)

    def part(b):
        lo, hi = bounds[b], bounds[b + 1]
        r = np.sqrt(-2.0 * np.log(1.0 - u[lo:hi]))       # 1 - u in (0, 1]
        th = (2.0 * math.pi) * u[half + lo:half + hi]
        z[lo:hi] = r * np.cos(th)
        z[half + lo:half + hi] = r * np.sin(th)

    with _pool() as ex:
        list(ex.map(part, range(_BLOCKS)))
    return z[:n].reshape(shape)


def randint(seed: int, stream: int, shape, high: int) -> np.ndarray:
    """Integers in [0, high) (multiply-shift on 32-bit draws)."""
    n = int(np.prod(shape))
    x = Pcg32Lanes(seed, stream).draws(n).astype(np.uint64)
    return ((x * np.uint64(high)) >> np.uint64(32)).astype(np.int64).reshape(shape)


# --------------------------------------------------------------------------- bf16
def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 -> bf16 (nearest-even), returned as uint16 bit patterns."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)  # float64->float32 is RNE
    b = f.view(np.uint32).astype(np.uint64)
    # round float32 -> bf16 to nearest even; the double rounding f64->f32->bf16
    # only matters on exact float32 ties, which do not occur for these draws.
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    b = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- helpers
def gumbel_max_tokens(logits: np.ndarray, temperature: float, seed: int, stream: int) -> np.ndarray:
    """Draw one token per row of `logits` (float64 [..., V]) from softmax(logits/T)
    with the Gumbel-max trick; T == 0 returns the row argmax.  This is how the
    synthetic drafter proposes tokens; it is not part of the verifier."""
    if temperature == 0.0:
        return np.argmax(logits, axis=-1).astype(np.int32)
    V = logits.shape[-1]
    flat = logits.reshape(-1, V)
    u = uniform_u24(seed, stream, flat.shape)
    out = np.empty(flat.shape[0], dtype=np.int32)
    bounds = np.linspace(0, flat.shape[0], _BLOCKS + 1).astype(np.int64)

    def part(b):
        lo, hi = bounds[b], bounds[b + 1]
        g = -np.log(-np.log(u[lo:hi] + 0.5 * _TWO_M24))  # u + 2^-25 in (0, 1)
        out[lo:hi] = np.argmax(flat[lo:hi] / temperature + g, axis=-1)

    with _pool() as ex:
        list(ex.map(part, range(_BLOCKS)))
    return out.reshape(logits.shape[:-1])


@dataclass
class Logits:
    """A logit tensor in the form it is handed to both sides."""
    dtype: str                  # "bf16" or "f32"
    raw: np.ndarray             # uint16 bits (bf16) or float32 values

    @property
    def f64(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f64(self.raw)
        return self.raw.astype(np.float64)

    @property
    def shape(self):
        return self.raw.shape


def make_logits(x64: np.ndarray, dtype: str) -> Logits:
    if dtype == "bf16":
        return Logits("bf16", f64_to_bf16_bits(x64))
    if dtype == "f32":
        return Logits("f32", x64.astype(np.float32))
    raise ValueError(dtype)


# --------------------------------------------------------------------------- workloads
@dataclass
class ChainCase:
    target: Logits              # [R, gamma+1, V]
    draft: Logits               # [R, gamma, V]
    tokens: np.ndarray          # int32 [R, gamma]
    uniforms: np.ndarray        # float32 [R, gamma+1, 2]
    temperature: float
    lengths: np.ndarray | None = None   # int32 [R] or None (= gamma)
    meta: dict = field(default_factory=dict)

    @property
    def R(self):
        return self.tokens.shape[0]

    @property
    def gamma(self):
        return self.tokens.shape[1]

    @property
    def V(self):
        return self.target.shape[-1]


def chain_tiny(seed: int = 1, temperature: float = 1.0, R: int = 1, gamma: int = 4, V: int = 1024,
               dtype: str = "f32") -> ChainCase:
    """Tiny chain: target ~ N(0, 2^2); draft = target[:, :gamma] + N(0, 0.5^2)."""
    t = 2.0 * normal(seed, 1, (R, gamma + 1, V))
    d = t[:, :gamma] + 0.5 * normal(seed, 2, (R, gamma, V))
    target, draft = make_logits(t, dtype), make_logits(d, dtype)
    tok = gumbel_max_tokens(draft.f64, temperature, seed, 3)
    u = uniform_f32(seed, 4, (R, gamma + 1, 2))
    return ChainCase(target, draft, tok, u, temperature, None, {"name": "tiny chain"})


def chain_long_vocab(seed: int = 2, temperature: float = 1.0, R: int = 1, gamma: int = 7,
                     V: int = 151936, dtype: str = "bf16") -> ChainCase:
    """One planted +8 peak per target position over N(0, 3^2); draft = target + N(0, 1)."""
    t = 3.0 * normal(seed, 1, (R, gamma + 1, V))
    peak = randint(seed, 5, (R, gamma + 1), V)
    np.put_along_axis(t, peak[..., None], np.take_along_axis(t, peak[..., None], -1) + 8.0, -1)
    d = t[:, :gamma] + normal(seed, 2, (R, gamma, V))
    target, draft = make_logits(t, dtype), make_logits(d, dtype)
    tok = gumbel_max_tokens(draft.f64, temperature, seed, 3)
    u = uniform_f32(seed, 4, (R, gamma + 1, 2))
    return ChainCase(target, draft, tok, u, temperature, None, {"name": "long-vocab chain"})


def chain_batched(seed: int = 3, temperature: float = 1.0, R: int = 64, gamma: int = 7,
                  V: int = 151936, dtype: str = "bf16", ragged_lengths: bool = False) -> ChainCase:
    """Batched chain: per-request scale s_r ~ U(1,4), target = s_r N(0,1);
    draft noise sigma_r ~ U(0.3, 2.0), draft = target[:, :gamma] + sigma_r N(0,1)."""
    s = 1.0 + 3.0 * uniform_u24(seed, 6, (R, 1, 1))
    sig = 0.3 + 1.7 * uniform_u24(seed, 7, (R, 1, 1))
    t = s * normal(seed, 1, (R, gamma + 1, V))
    d = t[:, :gamma] + sig * normal(seed, 2, (R, gamma, V))
    target, draft = make_logits(t, dtype), make_logits(d, dtype)
    tok = gumbel_max_tokens(draft.f64, temperature if temperature > 0 else 1.0, seed, 3)
    u = uniform_f32(seed, 4, (R, gamma + 1, 2))
    lengths = None
    if ragged_lengths:
        lengths = randint(seed, 8, (R,), gamma + 1).astype(np.int32)
    return ChainCase(target, draft, tok, u, temperature, lengths,
                     {"name": "batched chain", "scale": s.ravel(), "sigma": sig.ravel()})


@dataclass
class TreeCase:
    target: Logits              # [R, N+1, V]
    parents: np.ndarray         # int32 [R, N+1], parents[:, 0] = -1
    tokens: np.ndarray          # int32 [R, N+1], tokens[:, 0] unused (0)
    max_depth: int


def random_tree(rng_u: np.ndarray, n_nodes: int, max_depth: int, max_children: int):
    """Branching process: repeatedly attach a child to a uniformly chosen node of
    depth < max_depth with < max_children children, until n_nodes non-root nodes
    exist; then relabel in depth-first preorder (children in creation order).
    rng_u supplies the uniforms.  Returns (parents, depth) in preorder."""
    par = [-1]
    depth = [0]
    kids = [[]]
    it = 0
    while len(par) < n_nodes + 1:
        open_nodes = [i for i in range(len(par)) if depth[i] < max_depth and len(kids[i]) < max_children]
        j = open_nodes[int(rng_u[it] * len(open_nodes))]
        it += 1
        kids[j].append(len(par))
        par.append(j)
        depth.append(depth[j] + 1)
        kids.append([])
    order = []
    stack = [0]
    while stack:
        i = stack.pop()
        order.append(i)
        stack.extend(reversed(kids[i]))
    new = {old: n for n, old in enumerate(order)}
    parents = np.array([-1] + [new[par[old]] for old in order[1:]], dtype=np.int32)
    depths = np.array([depth[old] for old in order], dtype=np.int32)
    return parents, depths


def tree_greedy(seed: int = 4, R: int = 16, N: int = 60, max_depth: int = 8, V: int = 151936,
                dtype: str = "bf16", p_follow: float = 0.5) -> TreeCase:
    """Greedy-tree workload: target [R, N+1, V] ~ N(0, 3^2); node tokens copy the
    parent's row argmax with probability p_follow, else uniform in [0, V)."""
    t = 3.0 * normal(seed, 1, (R, N + 1, V))
    target = make_logits(t, dtype)
    tf = target.f64
    row_argmax = np.argmax(tf, axis=-1)      # planting only: half the tokens follow it
    u_tree = uniform_u24(seed, 9, (R, N))
    coin = uniform_u24(seed, 10, (R, N + 1))
    rnd = randint(seed, 11, (R, N + 1), V)
    parents = np.zeros((R, N + 1), dtype=np.int32)
    tokens = np.zeros((R, N + 1), dtype=np.int32)
    for r in range(R):
        p, _ = random_tree(u_tree[r], N, max_depth, 4)
        parents[r] = p
        for i in range(1, N + 1):
            tokens[r, i] = row_argmax[r, p[i]] if coin[r, i] < p_follow else rnd[r, i]
    return TreeCase(target, parents, tokens, max_depth)


@dataclass
class MarkovCase:
    U: Logits                   # bf16 [R, gamma, V]
    W1: Logits                  # bf16 [V, rank]
    W2: Logits                  # bf16 [rank, V]
    anchor: np.ndarray          # int32 [R]
    uniforms: np.ndarray        # float32 [R, gamma]
    temperature: float


def markov(seed: int = 2, R: int = 1, gamma: int = 7, V: int = 151936, rank: int = 256,
           temperature: float = 1.0, u_scale: float = 3.0, w_scale: float = 0.02) -> MarkovCase:
    """Markov draft head inputs: U ~ N(0, u_scale^2), W1, W2 ~ N(0, w_scale^2), bf16."""
    U = make_logits(u_scale * normal(seed, 21, (R, gamma, V)), "bf16")
    W1 = make_logits(w_scale * normal(seed, 22, (V, rank)), "bf16")
    W2 = make_logits(w_scale * normal(seed, 23, (rank, V)), "bf16")
    anchor = randint(seed, 24, (R,), V).astype(np.int32)
    u = uniform_f32(seed, 25, (R, gamma))
    return MarkovCase(U, W1, W2, anchor, u, temperature)


def dspark_target(seed: int, U: Logits) -> Logits:
    """Target logits for verifying Markov drafts: rows k < gamma are U_k + sigma_r N(0,1)
    with sigma_r ~ U(0.3, 2.0), the bonus row is N(0, 3^2); bf16 [R, gamma + 1, V]."""
    R, gamma, V = U.raw.shape
    sig = 0.3 + 1.7 * uniform_u24(seed, 41, (R, 1, 1))
    t = np.empty((R, gamma + 1, V), dtype=np.float64)
    t[:, :gamma] = U.f64 + sig * normal(seed, 42, (R, gamma, V))
    t[:, gamma] = 3.0 * normal(seed, 43, (R, V))
    return make_logits(t, "bf16")


def confidences(seed: int = 5, R: int = 512, gamma: int = 7, mean: float = 1.5, sd: float = 1.0) -> np.ndarray:
    """c = sigmoid(N(mean, sd^2)) as float32 [R, gamma] (synthetic confidence-head output)."""
    z = mean + sd * normal(seed, 31, (R, gamma))
    return (1.0 / (1.0 + np.exp(-z))).astype(np.float32)


def sps_table(B_max: int = 4096) -> np.ndarray:
    """Synthetic smooth decreasing steps-per-second curve SPS(B), B = 1..B_max (float64)."""
    B = np.arange(1, B_max + 1, dtype=np.float64)
    return 1000.0 / (10.0 + 0.004 * B + 1e-6 * B * B)
