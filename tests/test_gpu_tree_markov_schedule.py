"""CUDA vs oracle parity for specv_verify_tree_greedy, specv_markov_draft and
specv_schedule.  Tree paths and scheduler lengths are bit-exact; Markov logits
agree within a float32-accumulation bound and sampled tokens follow the
flagged-threshold rule, checked step by step with the GPU's own previous token
as the conditioning input."""
import numpy as np
import pytest

import oracle
import synth
from parity import TOL, check_chain, report, to_torch

pytestmark = pytest.mark.gpu


# --------------------------------------------------------------------------- tree
def _run_tree(lib, case):
    import torch
    dev = torch.device("cuda")
    plen, nodes, tok = lib.verify_tree_greedy(to_torch(case.target, dev), to_torch(case.parents, dev, np.int32),
                                              to_torch(case.tokens, dev, np.int32), case.max_depth)
    return plen.cpu().numpy(), nodes.cpu().numpy(), tok.cpu().numpy()


def _check_tree(lib, case):
    plen, nodes, tok = _run_tree(lib, case)
    ref = oracle.verify_tree_greedy(case.target.f64, case.parents, case.tokens, case.max_depth)
    assert (plen == ref.path_len).all()
    assert (nodes == ref.path_nodes).all()
    assert (tok == ref.token).all()
    return ref


@pytest.mark.parametrize("dtype,V", [("bf16", 4096), ("f32", 999), ("bf16", 33001)])
def test_tree_small(lib, dtype, V):
    case = synth.tree_greedy(seed=201, R=6, N=25, max_depth=6, V=V, dtype=dtype, p_follow=0.8)
    ref = _check_tree(lib, case)
    assert ref.path_len.max() >= 2


def test_tree_degenerate(lib):
    # a root-only tree and a single chain
    case = synth.tree_greedy(seed=202, R=3, N=0, max_depth=1, V=100, dtype="f32")
    _check_tree(lib, case)
    case = synth.tree_greedy(seed=203, R=4, N=8, max_depth=8, V=300, dtype="f32", p_follow=0.9)
    case.parents[:] = np.arange(-1, 8)
    _check_tree(lib, case)


def test_tree_bad_parent_sets_error(lib):
    import torch
    case = synth.tree_greedy(seed=204, R=3, N=10, max_depth=5, V=256, dtype="f32")
    case.parents[1, 4] = 7                       # a child before its parent
    dev = torch.device("cuda")
    nbytes = lib.specv_verify_tree_greedy_workspace_size(3, 10, 256, lib.SPECV_F32)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    plen, nodes, tok = lib.verify_tree_greedy(to_torch(case.target, dev), to_torch(case.parents, dev, np.int32),
                                              to_torch(case.tokens, dev, np.int32), 5, workspace=ws)
    plen = plen.cpu().numpy()
    assert plen[1] == -1 and plen[0] >= 0 and plen[2] >= 0
    assert lib.read_device_error(ws) == lib.SPECV_ERR_DEVICE_DATA


def test_tree_maximum_sizes(lib):
    """1024 nodes (SPECV_MAX_TREE_NODES) and max_depth 64 (SPECV_MAX_TREE_DEPTH);
    a 64-deep chain accepted to its end."""
    case = synth.tree_greedy(seed=205, R=2, N=1023, max_depth=64, V=512, dtype="f32", p_follow=0.9)
    _check_tree(lib, case)
    chain = synth.tree_greedy(seed=206, R=2, N=64, max_depth=64, V=300, dtype="f32", p_follow=1.0)
    chain.parents[:] = np.arange(-1, 64)
    g = np.argmax(chain.target.f64, axis=-1)
    chain.tokens[:, 1:] = g[:, :64]
    ref = _check_tree(lib, chain)
    assert (ref.path_len == 64).all()


def test_tree_full_size(lib):
    """R=16 trees of 60 nodes + root, depth <= 8, V=151936 bf16."""
    case = synth.tree_greedy(seed=4)
    ref = _check_tree(lib, case)
    print(f"\ntree full size: mean accepted path {ref.path_len.mean():.2f}, max {ref.path_len.max()}")


# --------------------------------------------------------------------------- Markov head
def _markov_check(lib, m, T, logits_dtype="f32"):
    import torch
    dev = torch.device("cuda")
    U, W1, W2 = to_torch(m.U, dev), to_torch(m.W1, dev), to_torch(m.W2, dev)
    anchor = to_torch(m.anchor, dev, np.int32)
    u = to_torch(m.uniforms, dev, np.float32)
    ldt = torch.bfloat16 if logits_dtype == "bf16" else torch.float32
    toks, logits = lib.markov_draft(U, W1, W2, anchor, u, T, True, ldt)
    toks = toks.cpu().numpy()
    W164, W264 = m.W1.f64, m.W2.f64
    R, gamma, V = m.U.shape
    prev = m.anchor.astype(np.int64)
    flagged = 0
    for k in range(gamma):
        # one step at a time keeps the host copies to one [R, V] slice
        L_k = logits[:, k].float().cpu().numpy().astype(np.float64)
        U_k = synth.bf16_bits_to_f64(m.U.raw[:, k])
        Lref, _, _, _ = oracle.markov_step(U_k, W164, W264, prev, m.uniforms[:, k], max(T, 1.0))
        # float32 sum of `rank` exact bf16 products: |error| <= rank * 2^-24 * sum |products|
        # (recursive-summation bound), one rounding of U + bias, and the bf16 output rounding
        rank = W164.shape[1]
        acc_bound = rank * 2.0 ** -24 * (np.abs(W164[prev]) @ np.abs(W264))
        bound = 1e-6 * (1.0 + np.abs(Lref)) + acc_bound + (np.abs(Lref) * 2.0 ** -8 if logits_dtype == "bf16" else 0.0)
        assert (np.abs(L_k - Lref) <= bound).all(), f"step {k}: logits differ"
        for r in range(R):
            y = int(toks[r, k])
            Lr = L_k[r] if logits_dtype == "bf16" else Lref[r]
            if T == 0.0:
                g = int(np.argmax(Lref[r]))
                if y != g:
                    srt = np.sort(Lref[r])
                    assert Lref[r, y] >= srt[-1] - 2e-6 * (1 + abs(srt[-1])), "argmax differs beyond a near tie"
                    flagged += 1
                continue
            pr = oracle.softmax_t(Lr, T)
            C = np.cumsum(pr)
            S = C[-1]
            uu = float(m.uniforms[r, k])
            lo = (C[y - 1] if y > 0 else 0.0) / S
            hi = C[y] / S
            assert pr[y] > 0 and lo - TOL <= uu < hi + TOL, f"step {k} request {r}: token {y} outside CDF bracket"
            t_or, _, _ = oracle.inverse_cdf(pr, np.array(uu))
            if int(t_or) != y:
                flagged += 1
        prev = toks[:, k].astype(np.int64)
    return toks, flagged


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_markov_small(lib, T):
    m = synth.markov(seed=301, R=37, gamma=4, V=1000, rank=64, temperature=T, w_scale=0.5)
    _, flagged = _markov_check(lib, m, T)
    assert flagged <= 3


def test_markov_bf16_logits_and_rank256(lib):
    m = synth.markov(seed=302, R=5, gamma=3, V=5000, rank=256, temperature=1.0, w_scale=0.3)
    _markov_check(lib, m, 1.0, "bf16")


@pytest.mark.parametrize("V,rank", [(1001, 64), (4096, 320), (2000, 48)])
def test_markov_shapes_outside_the_tensor_core_form(lib, V, rank):
    """V not a multiple of 8, rank above 256 or not a multiple of 64: the
    CUDA-core contraction serves these shapes."""
    m = synth.markov(seed=303, R=9, gamma=3, V=V, rank=rank, temperature=1.0, w_scale=0.3)
    _, flagged = _markov_check(lib, m, 1.0)
    assert flagged <= 2


def test_markov_tensor_core_partial_blocks(lib):
    """R = 300 (one full and one partial 128-request block in the second group
    of 256), V = 70000 (last vocabulary tile partial): every row checked."""
    m = synth.markov(seed=304, R=300, gamma=2, V=70000, rank=256, temperature=1.0)
    _, flagged = _markov_check(lib, m, 1.0)
    # every draw is inside its CDF bracket (checked above); a draw that differs from the
    # oracle's lies within 1e-5 of a boundary, and CDF steps here average 1.4e-5
    assert flagged <= 3 + 600 // 50
    m0 = synth.markov(seed=305, R=130, gamma=2, V=4104, rank=128, temperature=0.0)
    _markov_check(lib, m0, 0.0)


def test_markov_long_vocab_single_request(lib):
    """R=1, gamma=7, V=151936, rank 256, W ~ N(0, 0.02^2), T=1 and T=0."""
    for T in (1.0, 0.0):
        m = synth.markov(seed=2, temperature=T)
        _markov_check(lib, m, T)


def test_markov_large_batch_every_row(lib):
    """R=512, gamma=7, V=129280, rank 256: the full DSpark drafting shape.  All
    512 rows are checked at each of the 7 steps, teacher-forced on the GPU's own
    previous tokens: logits within the float32 accumulation bound, every token
    inside its CDF bracket, and draws that differ from the oracle's counted
    (CDF steps here average 7.7e-6, so a uniform lands within 1e-5 of a boundary
    often; a differing draw is allowed only there)."""
    m = synth.markov(seed=5, R=512, gamma=7, V=129280)
    _, flagged = _markov_check(lib, m, 1.0)
    n = 512 * 7
    report("markov R=512 gamma=7 V=129280 T=1 (every row)", draws=n, differing_from_oracle_within_tol=flagged)
    assert flagged <= 3 + n // 100                  # measured on GB300: 17 of 3584


def _markov_tokens_only_check(lib, m, T):
    """Drafting with no logits kept: the tensor-core epilogue writes only tile
    partials and the sampler recomputes the 64 logits of the tile it draws
    from.  Every token must lie in the oracle's CDF bracket (within 1e-5) for
    the oracle's logits conditioned on the GPU's own previous token; tokens
    that differ from the logits-kept call are counted."""
    import torch
    dev = torch.device("cuda")
    args = (to_torch(m.U, dev), to_torch(m.W1, dev), to_torch(m.W2, dev), to_torch(m.anchor, dev, np.int32),
            to_torch(m.uniforms, dev, np.float32), T)
    toks, none = lib.markov_draft(*args, False)
    assert none is None
    toks = toks.cpu().numpy()
    kept, _ = lib.markov_draft(*args, True)
    kept = kept.cpu().numpy()
    W164, W264 = m.W1.f64, m.W2.f64
    R, gamma, V = m.U.shape
    prev = m.anchor.astype(np.int64)
    differ = 0
    for k in range(gamma):
        U_k = synth.bf16_bits_to_f64(m.U.raw[:, k])
        Lref, _, _, _ = oracle.markov_step(U_k, W164, W264, prev, m.uniforms[:, k], max(T, 1.0))
        for r in range(R):
            y = int(toks[r, k])
            if T == 0.0:
                srt = np.sort(Lref[r])
                assert Lref[r, y] >= srt[-1] - 2e-6 * (1 + abs(srt[-1])), "argmax differs beyond a near tie"
                continue
            pr = oracle.softmax_t(Lref[r], T)
            C = np.cumsum(pr)
            uu = float(m.uniforms[r, k])
            lo = (C[y - 1] if y > 0 else 0.0) / C[-1]
            hi = C[y] / C[-1]
            assert pr[y] > 0 and lo - TOL <= uu < hi + TOL, f"step {k} request {r}: token {y} outside CDF bracket"
        prev = toks[:, k].astype(np.int64)
    differ = int((toks != kept).sum())
    return toks, differ


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_markov_tokens_only(lib, T):
    """Tensor-core shapes with no logits kept: R = 300 (a partial request
    block), V = 70000 (a partial last tile), rank 256."""
    m = synth.markov(seed=306, R=300, gamma=3, V=70000, rank=256, temperature=T)
    _, differ = _markov_tokens_only_check(lib, m, T)
    assert differ <= 3 + 900 // 50


@pytest.mark.parametrize("R,V,rank,T", [(130, 4104, 128, 1.0), (130, 4104, 128, 0.0), (257, 1000, 64, 1.0)])
def test_markov_tokens_only_pair_shapes(lib, R, V, rank, T):
    """CTA-pair drafting (more than one 128-request block, no logits kept) at
    ragged shapes: a second block of 2 rows (R = 130) or an empty fourth block
    (R = 257), a last 256-column tile that is almost all past V (one CTA's half
    entirely), rank 128 and 64, T = 1 and T = 0."""
    m = synth.markov(seed=309, R=R, gamma=3, V=V, rank=rank, temperature=T, w_scale=0.3)
    _, differ = _markov_tokens_only_check(lib, m, T)
    assert differ <= 3 + R * 3 // 50


def test_markov_tokens_only_dspark_shape(lib):
    """R=512, gamma=7, V=129280, rank 256 with no logits kept (the drafting step
    of a DSpark round whose verification recomputes the draft logits)."""
    m = synth.markov(seed=5, R=512, gamma=7, V=129280)
    _, differ = _markov_tokens_only_check(lib, m, 1.0)
    report("markov R=512 gamma=7 V=129280 tokens only", draws=512 * 7, differing_from_logits_kept_call=differ)
    assert differ <= 3 + 3584 // 100


def _recompute_case(lib, m, lengths, T=1.0):
    """Draft with no kept logits (bf16 draw precision), then recompute the
    verified rows.  Returns (tokens, recomputed bf16 logits as float64 [R, gamma, V]
    with NaN in rows that must stay unwritten, the sentinel-filled tensor)."""
    import torch
    dev = torch.device("cuda")
    U, W1, W2 = to_torch(m.U, dev), to_torch(m.W1, dev), to_torch(m.W2, dev)
    anchor = to_torch(m.anchor, dev, np.int32)
    toks, _ = lib.markov_draft(U, W1, W2, anchor, to_torch(m.uniforms, dev, np.float32), T, False, torch.bfloat16)
    R, G, V = m.U.shape
    out = torch.full((R, G, V), 7.0, dtype=torch.bfloat16, device=dev)   # sentinel for rows not written
    lib.markov_recompute_logits(U, W1, W2, anchor, toks, to_torch(lengths, dev, np.int32), out=out)
    return toks.cpu().numpy(), out


def _check_recomputed_rows(m, toks, out, lengths, T=1.0):
    """Every listed row within the float32-accumulation + bf16-rounding bound of
    the oracle's L (conditioned on the GPU's tokens); every other row untouched;
    each drafted token inside the CDF bracket of its recomputed row (the draw
    used those logits)."""
    import torch
    R, G, V = m.U.shape
    W164, W264 = m.W1.f64, m.W2.f64
    rank = W164.shape[1]
    for k in range(G):
        prev = (m.anchor if k == 0 else toks[:, k - 1]).astype(np.int64)
        Lk = out[:, k].float().cpu().numpy().astype(np.float64)
        live = k < lengths
        assert (Lk[~live] == 7.0).all(), f"position {k}: a row past its length was written"
        if not live.any():
            continue
        U_k = synth.bf16_bits_to_f64(m.U.raw[live, k])
        Lref, _, _, _ = oracle.markov_step(U_k, W164, W264, prev[live], m.uniforms[live, k], 1.0)
        bound = 1e-6 * (1 + np.abs(Lref)) + rank * 2.0 ** -24 * (np.abs(W164[prev[live]]) @ np.abs(W264)) \
            + np.abs(Lref) * 2.0 ** -8
        assert (np.abs(Lk[live] - Lref) <= bound).all(), f"position {k}: recomputed logits differ"
        for i, r in enumerate(np.nonzero(live)[0]):
            pr = oracle.softmax_t(Lk[r], T)
            C = np.cumsum(pr)
            y, uu = int(toks[r, k]), float(m.uniforms[r, k])
            lo = (C[y - 1] if y > 0 else 0.0) / C[-1]
            assert pr[y] > 0 and lo - TOL <= uu < C[y] / C[-1] + TOL, f"({r}, {k}): token outside the recomputed CDF"


def test_markov_recompute_logits_ragged_lengths(lib):
    """Verified rows only (ragged lengths, l_r = 0 and l_r = gamma included),
    R = 300 (a partial 128-row block of listed rows), V = 70000 (a partial last
    256-column tile)."""
    m = synth.markov(seed=307, R=300, gamma=4, V=70000, rank=256)
    lengths = (synth.uniform_u24(307, 9, (300,)) * 5).astype(np.int32)
    lengths[:3] = [0, 4, 1]
    toks, out = _recompute_case(lib, m, lengths)
    _check_recomputed_rows(m, toks, out, lengths)


def test_markov_recompute_logits_equal_the_kept_logits(lib):
    """The recomputed rows against the logits specv_markov_draft keeps when asked
    (bf16), on the same tokens: the float32 sums may differ only in their
    order-dependent last bits, so the bf16 values agree except at rounding ties
    of those bits (counted)."""
    import torch
    dev = torch.device("cuda")
    m = synth.markov(seed=308, R=256, gamma=3, V=129280, rank=256)
    lengths = np.full(256, 3, dtype=np.int32)
    toks, out = _recompute_case(lib, m, lengths)
    kept_toks, kept = lib.markov_draft(to_torch(m.U, dev), to_torch(m.W1, dev), to_torch(m.W2, dev),
                                       to_torch(m.anchor, dev, np.int32), to_torch(m.uniforms, dev, np.float32), 1.0,
                                       True, torch.bfloat16)
    same_tok = (kept_toks.cpu().numpy() == toks)
    rows = torch.from_numpy(np.nonzero(same_tok.all(1))[0]).to(dev)
    a = out[rows].view(torch.int16)
    b = kept[rows].view(torch.int16)
    differ = int((a != b).sum().item())
    total = a.numel()
    report("markov recompute vs kept bf16 logits R=256 gamma=3 V=129280", elements=total, differing_bf16=differ,
           requests_with_equal_tokens=int(rows.numel()))
    assert differ <= total // 1000


def test_dspark_round_with_recomputed_draft_logits(lib):
    """The DSpark round without kept draft logits: tokens-only drafting (bf16
    draw precision) -> scheduler -> the verified rows' draft logits recomputed
    -> chain verification.  The recomputed rows are checked against the oracle's
    logits and the verification against oracle.verify_chain on them, request by
    request (flagged-threshold rule, c* within 1e-5)."""
    import torch
    dev = torch.device("cuda")
    R, G, V = 512, 7, 129280
    m = synth.markov(seed=5, R=R, gamma=G, V=V)
    tgt = synth.dspark_target(5, m.U)
    conf = synth.confidences(5, R, G)
    sps = synth.sps_table(4096)
    lengths, _ = lib.schedule(to_torch(conf, dev, np.float32), to_torch(sps, dev, np.float64))
    ell = lengths.cpu().numpy()
    assert (ell == oracle.schedule(conf, sps).lengths).all()
    toks, out = _recompute_case(lib, m, ell)
    _check_recomputed_rows(m, toks, out, ell)
    u_np = synth.uniform_f32(5, 44, (R, G + 1, 2))
    A, y, c = lib.verify_chain(to_torch(tgt, dev), out, to_torch(toks, dev, np.int32), to_torch(u_np, dev, np.float32),
                               1.0, lengths)
    A, y, c = A.cpu().numpy(), y.cpu().numpy(), c.cpu().numpy()
    d_bits = out.view(torch.int16).cpu().numpy().view(np.uint16)
    tot = dict(requests=0, exact=0, flagged_accept=0, flagged_sample=0)
    worst = 0.0
    for r in range(R):
        L = int(ell[r])
        t64 = synth.bf16_bits_to_f64(tgt.raw[r:r + 1, :L + 1])
        d64 = synth.bf16_bits_to_f64(d_bits[r:r + 1, :L])
        u = u_np[r:r + 1, :L + 1]
        res = oracle.verify_chain(t64, d64, toks[r:r + 1, :L].astype(np.int64), u, 1.0)
        st = check_chain(A[r:r + 1], y[r:r + 1], res, lambda _r, kk: oracle.softmax_t(t64[0, kk], 1.0),
                         lambda _r, kk: oracle.softmax_t(d64[0, kk], 1.0), u, np.array([L]))
        for key in ("exact", "flagged_accept", "flagged_sample"):
            tot[key] += getattr(st, key)
        tot["requests"] += 1
        if L:
            diff = np.abs(c[r, :L] - res.c_star[0])
            worst = max(worst, float(diff.max()))
            assert (diff <= TOL).all()
    report("dspark round with recomputed draft logits R=512 gamma=7 V=129280", sum_l=int(ell.sum()),
           max_abs_cstar_diff=worst, **tot)
    assert tot["exact"] >= R - 16


# --------------------------------------------------------------------------- scheduler
def _run_sched(lib, conf, sps, B_max=None):
    import torch
    dev = torch.device("cuda")
    lengths, theta = lib.schedule(to_torch(conf, dev, np.float32), to_torch(sps, dev, np.float64), B_max)
    return lengths.cpu().numpy(), float(theta.cpu().numpy()[0])


@pytest.mark.parametrize("R,gamma", [(1, 1), (3, 3), (40, 7), (512, 7), (1000, 8), (8192, 1)])
def test_schedule_matches_oracle(lib, R, gamma):
    conf = synth.confidences(400 + R, R, gamma)
    sps = synth.sps_table(max(4096, R * (gamma + 1)))
    ell, theta = _run_sched(lib, conf, sps)
    ref = oracle.schedule(conf, sps)
    assert (ell == ref.lengths).all()
    assert theta == ref.theta_best


def test_schedule_special_tables(lib):
    conf = synth.confidences(410, 64, 7)
    ell, _ = _run_sched(lib, conf, np.full(4096, 5.0))
    assert (ell == 7).all()
    ell, _ = _run_sched(lib, conf, 1.0 / np.arange(1, 4097, dtype=np.float64) ** 2)
    assert (ell == 0).all()
    sps = np.array([10.0, 10.0, 10.0, 7.0, 9.0, 9.0, 9.0, 9.0])
    c = np.full((2, 3), 0.9, dtype=np.float32)
    ell, _ = _run_sched(lib, c, sps)
    assert list(ell) == list(oracle.schedule(c, sps).lengths) == [1, 0]
    # ties and the batch cap
    c = np.array([[1.0, 0.5], [1.0, 1.0]], dtype=np.float32)
    for bmax in (3, 4, 5, 6):
        ell, _ = _run_sched(lib, c, np.full(8, 1.0), bmax)
        assert list(ell) == list(oracle.schedule(c, np.full(8, 1.0), bmax).lengths)


def test_schedule_bad_confidence(lib):
    import torch
    conf = synth.confidences(411, 8, 3)
    conf[3, 1] = 1.5
    dev = torch.device("cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    lengths, _ = lib.schedule(to_torch(conf, dev, np.float32), to_torch(synth.sps_table(64), dev, np.float64),
                              workspace=ws)
    assert (lengths.cpu().numpy() == -1).all()
    assert lib.read_device_error(ws) == lib.SPECV_ERR_DEVICE_DATA


def _run_global(lib, conf, sps, stale=None, B_max=None):
    import torch
    dev = torch.device("cuda")
    R, gamma = conf.shape
    c = to_torch(conf, dev, np.float32)
    cs = to_torch(stale, dev, np.float32) if stale is not None else None
    t = to_torch(sps, dev, np.float64)
    ell = torch.empty(R, dtype=torch.int32, device=dev)
    theta = torch.empty(1, dtype=torch.float64, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    st = lib.specv_schedule_global(c.data_ptr(), cs.data_ptr() if cs is not None else None, t.data_ptr(), R, gamma,
                                   B_max or len(sps), ell.data_ptr(), theta.data_ptr(), ws.data_ptr(), 256,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return ell.cpu().numpy(), float(theta.cpu().numpy()[0]), ws


@pytest.mark.parametrize("R,gamma", [(1, 1), (3, 3), (40, 7), (512, 7), (1000, 8), (8192, 1)])
def test_schedule_global_matches_oracle(lib, R, gamma):
    conf = synth.confidences(420 + R, R, gamma)
    stale = synth.confidences(430 + R, R, gamma)
    rng = np.random.default_rng(R)
    sps = synth.sps_table(max(4096, R * (gamma + 1))) * rng.uniform(0.9, 1.1, max(4096, R * (gamma + 1)))  # saw-tooth
    for st in (None, stale):
        ell, theta, _ = _run_global(lib, conf, sps, st)
        ref = oracle.schedule_global(conf, sps, conf_stale=st)
        assert (ell == ref.lengths).all()
        assert theta == ref.theta_best


def test_schedule_global_hand_cases(lib):
    ell, theta, _ = _run_global(lib, np.array([[0.9, 0.9, 0.9]]), np.array([10.0, 4.0, 4.0, 4.0]))
    assert list(ell) == [3]                                           # past the cliff
    ell, _, _ = _run_global(lib, np.array([[0.1], [0.9]]), np.array([5.0, 1.0, 0.8, 0.7]),
                            stale=np.array([[0.9], [0.1]]))
    assert list(ell) == [0, 1]                                        # K from stale, entry from current
    ell, _, _ = _run_global(lib, np.array([[0.5, 0.0, 0.0]]), np.full(8, 2.0))
    assert list(ell) == [1]                                           # ties: the smallest n
    c = synth.confidences(57, 4, 3)
    ell, _, _ = _run_global(lib, c, np.full(64, 1.0), B_max=5)
    assert ell.sum() == 1                                             # batch cap
    c[2, 1] = -0.5
    ell, _, ws = _run_global(lib, c, np.full(64, 1.0))
    assert (ell == -1).all()
    assert lib.read_device_error(ws) == lib.SPECV_ERR_DEVICE_DATA


@pytest.mark.parametrize("R,gamma", [(1, 1), (64, 7), (5000, 8)])
def test_prune_threshold_matches_oracle(lib, R, gamma):
    import torch
    dev = torch.device("cuda")
    conf = synth.confidences(440 + R, R, gamma)
    c = to_torch(conf, dev, np.float32)
    ell = torch.empty(R, dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    s = oracle.survival_products(conf)
    for th in (0.0, 0.3, 0.5, float(s[0, 0]), 0.95, 2.0):              # s[0, 0] exactly: kept (s >= threshold)
        st = lib.specv_prune_threshold(c.data_ptr(), R, gamma, th, ell.data_ptr(), ws.data_ptr(), 256,
                                       torch.cuda.current_stream().cuda_stream)
        assert st == 0
        assert (ell.cpu().numpy() == oracle.prune_threshold(conf, th)).all()
    bad = conf.copy()
    bad[0, 0] = float("nan")
    cb = to_torch(bad, dev, np.float32)
    assert lib.specv_prune_threshold(cb.data_ptr(), R, gamma, 0.5, ell.data_ptr(), ws.data_ptr(), 256,
                                     torch.cuda.current_stream().cuda_stream) == 0
    got = ell.cpu().numpy()
    assert got[0] == -1 and (got[1:] == oracle.prune_threshold(conf, 0.5)[1:]).all()
    assert lib.read_device_error(ws) == lib.SPECV_ERR_DEVICE_DATA


# --------------------------------------------------------------------------- DART candidate tree
def _run_dart(lib, logits, dtype, T, k, w, theta):
    import torch
    dev = torch.device("cuda")
    R, d, V = logits.shape
    if dtype == "bf16":
        x = torch.from_numpy(np.ascontiguousarray(logits.raw.view(np.int16))).to(dev)
        dt = lib.SPECV_BF16
    else:
        x = torch.from_numpy(np.ascontiguousarray(logits.raw)).to(dev)
        dt = lib.SPECV_F32
    par = torch.empty(R, theta + 1, dtype=torch.int32, device=dev)
    tok = torch.empty(R, theta + 1, dtype=torch.int32, device=dev)
    nn = torch.empty(R, dtype=torch.int32, device=dev)
    nb = lib.specv_dart_tree_workspace_size(R, d, V, k, w, theta, dt)
    assert nb > 0
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    st = lib.specv_dart_tree(x.data_ptr(), dt, R, d, V, T, k, w, theta, par.data_ptr(), tok.data_ptr(), nn.data_ptr(),
                             ws.data_ptr(), nb, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return par.cpu().numpy(), tok.cpu().numpy(), nn.cpu().numpy()


@pytest.mark.parametrize("R,d,V,k,w,theta,dtype,T", [
    (3, 8, 151936, 25, 20, 59, "bf16", 1.0),       # the notes' (d, k, w, theta)
    (4, 8, 2048, 25, 20, 59, "f32", 1.0),
    (2, 3, 512, 4, 2, 11, "bf16", 0.7),
    (1, 1, 64, 5, 3, 3, "f32", 1.0),
    (2, 5, 1024, 32, 32, 200, "bf16", 1.0),
    (1, 4, 1024, 16, 8, 300, "f32", 1.0),
    (1, 4, 1024, 32, 8, 600, "bf16", 1.0),         # theta > 512: the selection's list merge
])
def test_dart_tree_matches_oracle(lib, R, d, V, k, w, theta, dtype, T):
    logits = synth.make_logits(3.0 * synth.normal(70 + d + k, 1, (R, d, V)), dtype)
    par, tok, nn = _run_dart(lib, logits, dtype, T, k, w, theta)
    ref = oracle.dart_tree(logits.f64, T, k=k, w=w, theta=theta)
    assert (nn == ref.n_nodes).all()
    assert (par == ref.parents).all()
    assert (tok == ref.tokens).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_dart_tree_heavy_ties(lib, dtype):
    """Integer logits in 0..3: hundreds of values tie at every tile's bound, so
    the tiles take the repeated-maximum path; equal logits go lower id first.
    Whole depths of equal scores send the beam and the selection to their list
    merges."""
    R, d, V = 2, 3, 151936
    raw = np.floor(synth.uniform_f32(81, 1, (R, d, V)) * 4.0).astype(np.float64)
    raw[1, 2, :] = 1.0                                   # one constant row
    logits = synth.make_logits(raw, dtype)
    par, tok, nn = _run_dart(lib, logits, dtype, 1.0, 25, 20, 59)
    ref = oracle.dart_tree(logits.f64, 1.0, k=25, w=20, theta=59)
    assert (nn == ref.n_nodes).all()
    assert (par == ref.parents).all()
    assert (tok == ref.tokens).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_dart_tree_masked_vocabulary(lib, dtype):
    """Fewer finite logits than k: the rest of the top-k are -inf logits
    (p = 0), lowest id first, each scored with ln(0 + eps)."""
    R, d, V, k = 2, 4, 4096, 25
    raw = np.full((R, d, V), -np.inf)
    g = synth.normal(82, 1, (R, d, 10))
    ids = (synth.uniform_u24(82, 2, (R, d, 10)) * V).astype(np.int64)
    for r in range(R):
        for i in range(d):
            raw[r, i, ids[r, i]] = 2.0 * g[r, i]
    logits = synth.make_logits(raw, dtype)
    par, tok, nn = _run_dart(lib, logits, dtype, 1.0, k, 6, 40)
    ref = oracle.dart_tree(logits.f64, 1.0, k=k, w=6, theta=40)
    assert (nn == ref.n_nodes).all()
    assert (par == ref.parents).all()
    assert (tok == ref.tokens).all()


def test_dart_tree_feeds_the_tree_verifier(lib):
    """The constructed tree goes straight into specv_verify_tree_greedy."""
    import torch
    dev = torch.device("cuda")
    R, d, V = 2, 8, 4096
    logits = synth.make_logits(3.0 * synth.normal(77, 1, (R, d, V)), "bf16")
    par, tok, nn = _run_dart(lib, logits, "bf16", 1.0, 25, 20, 59)
    target = synth.make_logits(3.0 * synth.normal(78, 1, (R, 60, V)), "bf16")
    ref = oracle.verify_tree_greedy(target.f64, par.astype(np.int64), tok.astype(np.int64), 8)
    path_len, path, token = lib.verify_tree_greedy(
        torch.from_numpy(np.ascontiguousarray(target.raw.view(np.int16))).to(dev).view(torch.bfloat16),
        to_torch(par, dev, np.int32), to_torch(tok, dev, np.int32), 8)
    assert (path_len.cpu().numpy() == ref.path_len).all()
    assert (token.cpu().numpy() == ref.token).all()


# --------------------------------------------------------------------------- confidence head
def _conf_case(seed, R, gamma, H, V, rank):
    h = synth.make_logits(synth.normal(seed, 1, (R, gamma, H)), "bf16")
    W1 = synth.make_logits(0.5 * synth.normal(seed, 2, (V, rank)), "bf16")
    w = (synth.normal(seed, 3, (H + rank,)) / np.sqrt(H + rank)).astype(np.float32)
    anchor = (synth.uniform_u24(seed, 4, (R,)) * V).astype(np.int64)
    toks = (synth.uniform_u24(seed, 5, (R, gamma)) * V).astype(np.int64)
    return h, W1, w, anchor, toks


def _run_conf(lib, h, W1, w, b, anchor, toks, R, gamma, H, V, rank):
    import torch
    dev = torch.device("cuda")
    ht = torch.from_numpy(np.ascontiguousarray(h.raw.view(np.int16))).to(dev)
    W1t = torch.from_numpy(np.ascontiguousarray(W1.raw.view(np.int16))).to(dev)
    wt = to_torch(w, dev, np.float32)
    at, tt = to_torch(anchor, dev, np.int32), to_torch(toks, dev, np.int32)
    out = torch.empty(R, gamma, dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    st = lib.specv_confidence_head(ht.data_ptr(), W1t.data_ptr(), wt.data_ptr(), b, at.data_ptr(), tt.data_ptr(), R,
                                   gamma, H, V, rank, out.data_ptr(), ws.data_ptr(), 256,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), ws


@pytest.mark.parametrize("R,gamma,H,V,rank", [(512, 7, 4096, 129280, 256), (3, 4, 100, 50, 12), (1, 1, 8, 9, 8)])
def test_confidence_head_matches_oracle(lib, R, gamma, H, V, rank):
    """float32 accumulation of H + rank exact products: |dz| <= (H + rank) 2^-24
    sum |w_i x_i|, and the sigmoid's slope is at most 1/4."""
    h, W1, w, anchor, toks = _conf_case(80 + H, R, gamma, H, V, rank)
    c, _ = _run_conf(lib, h, W1, w, 0.5, anchor, toks, R, gamma, H, V, rank)
    ref = oracle.confidence_head(h.f64, W1.f64, w, 0.5, anchor, toks)
    prev = np.concatenate([anchor[:, None], toks[:, :gamma - 1]], axis=1)
    mag = np.abs(h.f64) @ np.abs(w[:H].astype(np.float64)) + np.abs(W1.f64[prev]) @ np.abs(w[H:].astype(np.float64))
    bound = 1e-6 + (H + rank) * 2.0 ** -24 * mag / 4
    assert (np.abs(c - ref) <= bound).all()
    assert (c > 0).all() and (c < 1).all()


def test_confidence_head_bad_token(lib):
    R, gamma, H, V, rank = 4, 3, 64, 20, 8
    h, W1, w, anchor, toks = _conf_case(90, R, gamma, H, V, rank)
    anchor[2] = V                       # out of range: position 0 of request 2
    toks[1, 0] = -1                     # conditions position 1 of request 1
    c, ws = _run_conf(lib, h, W1, w, 0.0, anchor, toks, R, gamma, H, V, rank)
    assert np.isnan(c[2, 0]) and np.isnan(c[1, 1])
    ok = ~np.isnan(c)
    assert ok.sum() == R * gamma - 2
    assert lib.read_device_error(ws) == lib.SPECV_ERR_DEVICE_DATA


# --------------------------------------------------------------------------- the DSpark round
def test_dspark_round_full_size(lib):
    """Markov drafting (R=512, gamma=7, V=129280, bf16 logits) -> scheduler -> chain
    verification with the scheduled lengths, all on the device.  The scheduler's
    lengths are checked bit-exact against the oracle (its inputs are synthetic).
    The verification is checked against the oracle on the GPU's own drafts: the
    bf16 draft logits and tokens it wrote, with the scheduled l_r, go through
    oracle.verify_chain request by request (only the l_r + 1 live target rows and
    l_r draft rows of each), and A_r, the emitted token and every c*_{r,k} must
    agree under the flagged-threshold rule and the 1e-5 tolerance."""
    import torch
    dev = torch.device("cuda")
    R, G, V = 512, 7, 129280
    m = synth.markov(seed=5, R=R, gamma=G, V=V)
    tgt = synth.dspark_target(5, m.U)
    U, W1, W2, target = (to_torch(x, dev) for x in (m.U, m.W1, m.W2, tgt))
    toks, dlog = lib.markov_draft(U, W1, W2, to_torch(m.anchor, dev, np.int32), to_torch(m.uniforms, dev, np.float32),
                                  1.0, True, torch.bfloat16)
    conf = synth.confidences(5, R, G)
    sps = synth.sps_table(4096)
    lengths, _ = lib.schedule(to_torch(conf, dev, np.float32), to_torch(sps, dev, np.float64))
    ell = lengths.cpu().numpy()
    assert (ell == oracle.schedule(conf, sps).lengths).all()
    u_np = synth.uniform_f32(5, 44, (R, G + 1, 2))
    A, y, c = lib.verify_chain(target, dlog, toks, to_torch(u_np, dev, np.float32), 1.0, lengths)
    A, y, c = A.cpu().numpy(), y.cpu().numpy(), c.cpu().numpy()
    t = toks.cpu().numpy()
    d_bits = dlog.view(torch.int16).cpu().numpy().view(np.uint16)
    del dlog
    assert ((t >= 0) & (t < V)).all()
    k = np.arange(G)[None, :]
    live = k < ell[:, None]
    assert np.isnan(c[~live]).all()
    tot = dict(requests=0, exact=0, flagged_accept=0, flagged_sample=0)
    worst = 0.0
    for r in range(R):
        L = int(ell[r])
        t64 = synth.bf16_bits_to_f64(tgt.raw[r:r + 1, :L + 1])
        d64 = synth.bf16_bits_to_f64(d_bits[r:r + 1, :L])
        x = t[r:r + 1, :L].astype(np.int64)
        u = u_np[r:r + 1, :L + 1]
        res = oracle.verify_chain(t64, d64, x, u, 1.0)
        st = check_chain(A[r:r + 1], y[r:r + 1], res, lambda _r, kk: oracle.softmax_t(t64[0, kk], 1.0),
                         lambda _r, kk: oracle.softmax_t(d64[0, kk], 1.0), u, np.array([L]))
        for key in ("exact", "flagged_accept", "flagged_sample"):
            tot[key] += getattr(st, key)
        tot["requests"] += 1
        if L:
            diff = np.abs(c[r, :L] - res.c_star[0])
            worst = max(worst, float(diff.max()))
            assert (diff <= TOL).all(), f"request {r}: c* differs by {diff.max()}"
    report("dspark round R=512 gamma=7 V=129280 T=1 (verify of the GPU's drafts)", sum_l=int(ell.sum()),
           max_abs_cstar_diff=worst, **tot)
    assert tot["exact"] >= R - 16
