"""Vocabulary-sharded verification on two gloo ranks (CPU): each rank holds a
contiguous slice of every row's V logits, reduces its slice, exchanges the
partials with all_gather / all_reduce, and combines them with the library's
host functions (specv_shard_*).  The combined results must equal the oracle's
on the unsharded rows: the softmax normalisers, c*, the accept thresholds, the
correction or bonus token, the greedy argmax (with a tie planted across the
shard boundary) and one Markov step.  The per-slice reductions are plain numpy
here, standing in for a kernel run on each rank's slice; the test needs no GPU.
"""
import ctypes
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LOG2E = 1.4426950408889634
V, R, GAMMA, SPLIT = 64, 3, 4, 40          # shard 0: ids [0, 40), shard 1: [40, 64)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _gather(dist, torch, x):
    t = torch.from_numpy(np.ascontiguousarray(x))
    out = [torch.zeros_like(t) for _ in range(dist.get_world_size())]
    dist.all_gather(out, t)
    return np.stack([o.numpy() for o in out])


def _allsum(dist, torch, x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    dist.all_reduce(t)
    return t.numpy()


def _normalisers(specv, dist, torch, x, c2):
    """(M_c2, Z) per row of the sharded logits x [rows, V_s] (float64 values)."""
    with np.errstate(invalid="ignore"):
        m = x.max(axis=-1) * c2
        z = np.exp2(x * c2 - m[:, None]).sum(axis=-1)
    part = np.stack([m, z], axis=-1).astype(np.float32)                     # [rows, 2]
    allp = np.ascontiguousarray(_gather(dist, torch, part))                 # [S, rows, 2]
    out = np.zeros((x.shape[0], 2), np.float32)
    assert specv.specv_shard_combine_normalisers(_ptr(allp), allp.shape[0], x.shape[0], _ptr(out)) == 0
    return out


def _pick(specv, dist, torch, mass_local, u):
    allm = np.ascontiguousarray(_gather(dist, torch, mass_local.astype(np.float64)))     # [S, rows]
    rows = mass_local.shape[0]
    shard = np.zeros(rows, np.int32)
    target = np.zeros(rows, np.float64)
    uu = np.ascontiguousarray(u, dtype=np.float32)
    assert specv.specv_shard_pick(_ptr(allm), allm.shape[0], rows, _ptr(uu), _ptr(shard), _ptr(target)) == 0
    return shard, target


def _draw_in_slice(w, target):
    """min{v : C(v) > target} over the slice's weights, else the last positive one."""
    c = np.cumsum(w)
    hit = np.nonzero((c > target) & (w > 0))[0]
    return int(hit[0]) if hit.size else int(np.nonzero(w > 0)[0][-1])


def _rank_body(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import lossless_draft_verification_gb300 as specv
    import synth
    specv.load()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = (0, SPLIT) if rank == 0 else (SPLIT, V)
    case = synth.chain_tiny(seed=11, R=R, gamma=GAMMA, V=V)
    T = 1.0
    c2 = LOG2E / T
    tg = case.target.f64[..., lo:hi]                   # [R, G+1, V_s]
    dr = case.draft.f64[..., lo:hi]                    # [R, G, V_s]
    res = {}
    # 1. normalisers of every target and draft row, and the probabilities of this slice
    nq = _normalisers(specv, dist, torch, tg.reshape(-1, hi - lo), c2).reshape(R, GAMMA + 1, 2)
    npd = _normalisers(specv, dist, torch, dr.reshape(-1, hi - lo), c2).reshape(R, GAMMA, 2)
    q = np.exp2(tg * c2 - nq[..., :1].astype(np.float64)) / nq[..., 1:].astype(np.float64)
    p = np.exp2(dr * c2 - npd[..., :1].astype(np.float64)) / npd[..., 1:].astype(np.float64)
    res["q"] = q                                       # this rank's slice (widths differ)
    # 2. c* = sum_v min(q, p): an all-reduce sum of the slices' sums
    res["c_star"] = _allsum(dist, torch, np.minimum(q[:, :GAMMA], p).sum(-1))
    # 3. accept thresholds: the shard owning x_k contributes q(x)/p(x)
    x = case.tokens.astype(np.int64)
    own = (x >= lo) & (x < hi)
    ratio = np.zeros((R, GAMMA))
    rr, kk = np.nonzero(own)
    ratio[rr, kk] = q[rr, kk, x[rr, kk] - lo] / p[rr, kk, x[rr, kk] - lo]
    thr = np.minimum(1.0, _allsum(dist, torch, ratio))
    res["thr"] = thr
    # 4. first rejection, then the residual (or bonus) draw across the shards
    u = case.uniforms.astype(np.float64)
    A = np.full(R, GAMMA)
    for r in range(R):
        rej = np.nonzero(~(u[r, :GAMMA, 0] < thr[r]))[0]
        if rej.size:
            A[r] = rej[0]
    w = np.zeros((R, hi - lo))
    for r in range(R):
        if A[r] < GAMMA:
            resid = np.maximum(q[r, A[r]] - p[r, A[r]], 0.0)
            total = _allsum(dist, torch, np.array([resid.sum()]))[0]
            w[r] = resid if total > 0.0 else q[r, A[r]]
        else:
            _allsum(dist, torch, np.array([0.0]))               # keep the collectives in step
            w[r] = q[r, GAMMA]
    shard, target = _pick(specv, dist, torch, w.sum(-1), u[np.arange(R), A, 1])
    tok = np.zeros(R, np.int64)
    for r in range(R):
        if shard[r] == rank:
            tok[r] = lo + _draw_in_slice(w[r], target[r])
    res["A"], res["token"] = A, _allsum(dist, torch, tok.astype(np.float64)).astype(np.int64)
    # 5. greedy argmax with a tie planted across the boundary (ids 5 and 50)
    g = case.target.f64.copy()
    g[0, 0, 5] = g[0, 0, 50] = g[0, 0].max() + 1.0
    gs = g[..., lo:hi].reshape(-1, hi - lo)
    val = gs.max(-1).astype(np.float32)
    idx = (gs.argmax(-1) + lo).astype(np.int32)
    allv, alli = _gather(dist, torch, val), _gather(dist, torch, idx)
    am = np.zeros(gs.shape[0], np.int32)
    assert specv.specv_shard_argmax_combine(_ptr(np.ascontiguousarray(allv)), _ptr(np.ascontiguousarray(alli)),
                                            world, gs.shape[0], _ptr(am)) == 0
    res["argmax"] = am
    # 6. one Markov step: W2 column-sharded, W1 replicated
    m = synth.markov(seed=12, R=R, gamma=1, V=V, rank=4, w_scale=1.0, u_scale=1.0)
    anchor, um = m.anchor.astype(np.int64), m.uniforms[:, 0].astype(np.float64)
    L = m.U.f64[:, 0, lo:hi] + m.W1.f64[anchor] @ m.W2.f64[:, lo:hi]
    nm = _normalisers(specv, dist, torch, L, c2)
    pm = np.exp2(L * c2 - nm[:, :1].astype(np.float64)) / nm[:, 1:].astype(np.float64)
    shard, target = _pick(specv, dist, torch, pm.sum(-1), um)
    mt = np.zeros(R, np.int64)
    for r in range(R):
        if shard[r] == rank:
            mt[r] = lo + _draw_in_slice(pm[r], target[r])
    res["markov"] = _allsum(dist, torch, mt.astype(np.float64)).astype(np.int64)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, res))


def _rank_main(rank, world, port, out):
    try:
        _rank_body(rank, world, port, out)
    except BaseException:
        import traceback
        out.put((rank, {"error": traceback.format_exc()}))
        raise


@pytest.fixture(scope="module")
def sharded():
    import torch.multiprocessing as mp
    from lossless_draft_verification_gb300 import build
    build.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=180) for _ in procs)
    for rank, res in results.items():
        assert "error" not in res, f"rank {rank}:\n{res['error']}"
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return results


def _oracle_case():
    import oracle
    import synth
    case = synth.chain_tiny(seed=11, R=R, gamma=GAMMA, V=V)
    return oracle, synth, case


def test_sharded_normalisers_give_the_full_softmax(sharded):
    oracle, _, case = _oracle_case()
    q_full = oracle.softmax_t(case.target.f64, 1.0)
    q = np.concatenate([sharded[0]["q"], sharded[1]["q"]], axis=-1)     # slices back in id order
    np.testing.assert_allclose(q, q_full, rtol=2e-6, atol=1e-9)


def test_sharded_c_star_and_thresholds(sharded):
    oracle, _, case = _oracle_case()
    ref = oracle.verify_chain(case.target.f64, case.draft.f64, case.tokens, case.uniforms, 1.0)
    for rank in (0, 1):
        np.testing.assert_allclose(sharded[rank]["c_star"], ref.c_star, atol=1e-6)
        np.testing.assert_allclose(sharded[rank]["thr"], ref.thr, rtol=1e-5)


def test_sharded_draw_matches_the_unsharded_inverse_cdf(sharded):
    oracle, _, case = _oracle_case()
    ref = oracle.verify_chain(case.target.f64, case.draft.f64, case.tokens, case.uniforms, 1.0)
    for rank in (0, 1):
        assert (sharded[rank]["A"] == ref.accepted).all()
        assert (sharded[rank]["token"] == ref.token).all()


def test_sharded_argmax_keeps_the_lower_id_on_a_cross_shard_tie(sharded):
    _, _, case = _oracle_case()
    g = case.target.f64.copy()
    g[0, 0, 5] = g[0, 0, 50] = g[0, 0].max() + 1.0
    ref = g.reshape(-1, V).argmax(-1)
    for rank in (0, 1):
        am = sharded[rank]["argmax"]
        assert am[0] == 5
        assert (am == ref).all()


def test_sharded_markov_step(sharded):
    import oracle
    import synth
    m = synth.markov(seed=12, R=R, gamma=1, V=V, rank=4, w_scale=1.0, u_scale=1.0)
    _, x, _, _ = oracle.markov_step(m.U.f64[:, 0], m.W1.f64, m.W2.f64, m.anchor, m.uniforms[:, 0], 1.0)
    for rank in (0, 1):
        assert (sharded[rank]["markov"] == x).all()


def test_shard_pick_rules():
    """Hand cases: the first shard whose cumulative mass passes u*S, the target
    inside it, the last shard with mass when rounding leaves none, -1 for none."""
    import lossless_draft_verification_gb300 as specv
    specv.load()
    mass = np.ascontiguousarray(np.array([[0.25, 0.0, 0.3], [0.0, 0.0, 0.0], [0.75, 0.0, 0.7]]))   # [S=3, rows=3]
    u = np.array([0.5, 0.9, 0.25], np.float32)
    shard = np.zeros(3, np.int32)
    target = np.zeros(3)
    assert specv.specv_shard_pick(_ptr(mass), 3, 3, _ptr(u), _ptr(shard), _ptr(target)) == 0
    assert shard.tolist() == [2, -1, 0]
    np.testing.assert_allclose(target, [0.25, 0.0, 0.25])
    bad = np.ascontiguousarray(-mass)
    assert specv.specv_shard_pick(_ptr(bad), 3, 3, _ptr(u), _ptr(shard), _ptr(target)) == specv.SPECV_ERR_INVALID_ARG
