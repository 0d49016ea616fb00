"""Helpers that compare CUDA outputs with the CPU oracle.

Decision rule (the contract of the verification path): integer results from
exact comparisons (argmax, tree paths, scheduler lengths) must be identical.
Decisions that floating point takes (an accept test u < min(1, q/p), an
inverse-CDF draw) must agree with the oracle except where the uniform lies
within TOL = 1e-5 of the decision threshold; such cases are counted.
Probabilities and c* must agree within 1e-5 absolute.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle

TOL = 1e-5

# (test name, counts) of every parity check that counted flagged cases; the
# session's terminal summary prints them (tests/conftest.py), so they show in
# the tail of a quiet run.
REPORT: list = []


def report(name: str, **counts) -> None:
    """Record one test's exact / flagged counts for the end-of-run summary."""
    REPORT.append((name, counts))


def to_torch(x, device, kind=None):
    import torch
    from synth import Logits
    if isinstance(x, Logits):
        if x.dtype == "bf16":
            return torch.from_numpy(x.raw.view(np.int16).copy()).view(torch.bfloat16).to(device)
        return torch.from_numpy(x.raw.copy()).to(device)
    arr = np.ascontiguousarray(x)
    if kind is not None:
        arr = arr.astype(kind)
    return torch.from_numpy(arr).to(device)


@dataclass
class ChainCheck:
    n: int = 0
    exact: int = 0
    flagged_accept: int = 0
    flagged_sample: int = 0
    mismatched: int = 0


def _weights(q_row, p_row, resid):
    if resid:
        w, S = oracle.residual(q_row, p_row)
        if not S > 0:
            return q_row
        return w
    return q_row


def check_chain(A_gpu, y_gpu, res: oracle.ChainResult, q_rows, p_rows, u, ell, tol=TOL) -> ChainCheck:
    """Validate each request's GPU trajectory against the oracle.

    q_rows(r, k) / p_rows(r, k) return float64 probability rows.  For the GPU's
    accepted length A: every accept decision k < A must be an oracle accept or
    flagged, the decision at A (if A < l_r) an oracle reject or flagged; the
    GPU token must be a token the oracle's CDF at A brackets around u (within
    tol).  Returns counts; raises AssertionError on an unexplained mismatch."""
    st = ChainCheck()
    R = len(A_gpu)
    for r in range(R):
        st.n += 1
        A, y, L = int(A_gpu[r]), int(y_gpu[r]), int(ell[r])
        assert 0 <= A <= L, f"request {r}: accepted {A} outside [0, {L}]"
        flagged = False
        for k in range(A + (1 if A < L else 0)):
            thr = res.thr[r, k]
            u0 = float(u[r, k, 0])
            gpu_accept = k < A
            if gpu_accept != (u0 < thr):
                assert abs(u0 - thr) < tol, f"request {r} position {k}: accept decision differs (u={u0}, thr={thr})"
                flagged = True
                st.flagged_accept += 1
        u1 = float(u[r, A, 1])
        if A == res.accepted[r] and y == res.token[r]:
            if not flagged:
                st.exact += 1
            continue
        w = _weights(q_rows(r, A), p_rows(r, A) if A < L else None, A < L)
        C = np.cumsum(w)
        S = C[-1]
        assert 0 <= y < len(w) and w[y] > 0, f"request {r}: token {y} has no mass"
        lo = (C[y - 1] if y > 0 else 0.0) / S
        hi = C[y] / S
        if not (lo - tol <= u1 < hi + tol):
            st.mismatched += 1
            raise AssertionError(f"request {r}: token {y} (CDF [{lo}, {hi})) does not bracket u={u1}")
        if not flagged and y != res.sample_at[r, A]:
            st.flagged_sample += 1
    return st
