"""CUDA vs oracle parity for specv_verify_chain and specv_tv_accept.

Sizes span several warp tiles, a cluster of CTAs and ragged tails; the last
tests run the batched workload at full size (R=64, gamma=7, V=151936 bf16) in
the launch configuration the benchmark times."""
import numpy as np
import pytest

import oracle
import synth
from parity import TOL, check_chain, report, to_torch

pytestmark = pytest.mark.gpu


def _run_chain(lib, case, want_c_star=True):
    import torch
    dev = torch.device("cuda")
    target = to_torch(case.target, dev)
    draft = to_torch(case.draft, dev)
    tok = to_torch(case.tokens, dev, np.int32)
    u = to_torch(case.uniforms, dev, np.float32)
    lengths = None if case.lengths is None else to_torch(case.lengths, dev, np.int32)
    A, y, c = lib.verify_chain(target, draft, tok, u, case.temperature, lengths, want_c_star)
    torch.cuda.synchronize()
    return A.cpu().numpy(), y.cpu().numpy(), None if c is None else c.cpu().numpy()


def _check_sampling(lib, case, name=None):
    A, y, c = _run_chain(lib, case)
    t64, d64 = case.target.f64, case.draft.f64
    T = case.temperature
    res = oracle.verify_chain(t64, d64, case.tokens, case.uniforms, T, case.lengths)
    ell = case.lengths if case.lengths is not None else np.full(case.R, case.gamma)
    st = check_chain(A, y, res, lambda r, k: oracle.softmax_t(t64[r, k], T),
                     lambda r, k: oracle.softmax_t(d64[r, k], T), case.uniforms, ell)
    ok = ~np.isnan(res.c_star)
    assert (np.isnan(c) == ~ok).all(), "c* NaN pattern differs"
    assert np.abs(c[ok] - res.c_star[ok]).max(initial=0.0) <= TOL
    if name is not None:
        report(name, requests=st.n, exact=st.exact, flagged_accept=st.flagged_accept,
               flagged_sample=st.flagged_sample, max_abs_cstar_diff=float(np.abs(c[ok] - res.c_star[ok]).max(initial=0.0)))
    return st, A, y, res


def _check_greedy(lib, case):
    A, y, c = _run_chain(lib, case)
    acc, tok, cst, _ = oracle.verify_chain_greedy(case.target.f64, case.tokens, case.lengths, case.draft.f64)
    assert (A == acc).all() and (y == tok).all()
    ok = ~np.isnan(cst)
    assert (np.isnan(c) == ~ok).all() and (c[ok] == cst[ok]).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1024, 1000, 4099, 50000])
def test_chain_sampling_small(lib, dtype, V):
    case = synth.chain_batched(seed=101, R=12, gamma=5, V=V, dtype=dtype, ragged_lengths=True)
    st, A, _, res = _check_sampling(lib, case)
    assert st.exact >= st.n - 2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1024, 1001, 70000])
def test_chain_greedy_small(lib, dtype, V):
    case = synth.chain_batched(seed=102, R=10, gamma=6, V=V, dtype=dtype, temperature=0.0, ragged_lengths=True)
    # make some drafts agree with the target argmax so accepted prefixes vary
    g = np.argmax(case.target.f64, -1)
    coin = synth.uniform_u24(102, 40, case.tokens.shape) < 0.7
    case.tokens = np.where(coin, g[:, :case.gamma], case.tokens).astype(np.int32)
    _check_greedy(lib, case)


@pytest.mark.parametrize("ragged,chunks", [(True, 3), (False, 4)])
def test_host_inputs_chunked_equal_device_call(lib, ragged, chunks):
    """Pinned host inputs through verify_chain with `chunks` request groups
    (copies on two streams overlapping the previous group's kernels, the three
    outputs returned by one transfer) give exactly the device call's outputs."""
    import torch
    case = synth.chain_batched(seed=110, R=10, gamma=4, V=5000, dtype="bf16", ragged_lengths=ragged)
    A, y, c = _run_chain(lib, case)
    host = lambda a, dt=None: (torch.from_numpy(np.ascontiguousarray(a.raw.view(np.int16))).view(torch.bfloat16)
                               if dt is None else torch.from_numpy(np.ascontiguousarray(a.astype(dt)))).pin_memory()
    h_len = None if case.lengths is None else host(case.lengths, np.int32)
    for _ in range(2):                            # the second call reuses the cached copy streams
        Ah, yh, ch = lib.verify_chain(host(case.target), host(case.draft), host(case.tokens, np.int32),
                                      host(case.uniforms, np.float32), case.temperature, h_len, True, chunks=chunks)
        assert Ah.device.type == "cpu" and ch.shape == (10, 4)
        np.testing.assert_array_equal(Ah.numpy(), A)
        np.testing.assert_array_equal(yh.numpy(), y)
        np.testing.assert_array_equal(ch.numpy().view(np.int32), c.view(np.int32))   # bitwise, NaN pattern included


def test_tiny_chain_config(lib):
    """R=1, gamma=4, V=1024 float32 at T=1 and T=0."""
    for T in (1.0, 0.0):
        case = synth.chain_tiny(seed=1, temperature=T)
        if T > 0:
            _check_sampling(lib, case)
        else:
            _check_greedy(lib, case)


@pytest.mark.parametrize("T", [0.5, 1.0, 2.5])
def test_temperatures(lib, T):
    case = synth.chain_batched(seed=103, R=8, gamma=4, V=3000, dtype="bf16", temperature=T)
    _check_sampling(lib, case)


def test_equal_distributions_accept_everything(lib):
    case = synth.chain_batched(seed=104, R=6, gamma=5, V=2048, dtype="bf16")
    case.draft.raw[:] = case.target.raw[:, :case.gamma]
    A, y, c = _run_chain(lib, case)
    assert (A == case.gamma).all()
    np.testing.assert_allclose(c, 1.0, atol=TOL)
    _check_sampling(lib, case)


def test_disjoint_support_rejects_and_draws_from_q(lib):
    V, R, gamma = 512, 16, 3
    case = synth.chain_batched(seed=105, R=R, gamma=gamma, V=V, dtype="f32")
    t = case.target.raw
    d = case.draft.raw
    t[:, :, V // 2:] = -np.inf            # q lives on the lower half
    d[:, :, : V // 2] = -np.inf           # p lives on the upper half
    case.tokens = synth.gumbel_max_tokens(case.draft.f64, 1.0, 105, 9)
    A, y, c = _run_chain(lib, case)
    assert (A == 0).all() and (y < V // 2).all()
    np.testing.assert_allclose(c, 0.0, atol=TOL)
    _check_sampling(lib, case)


def test_bonus_only_and_degenerate_sizes(lib):
    # gamma = 0: only the bonus draw
    case = synth.chain_batched(seed=106, R=5, gamma=0, V=777, dtype="f32")
    _check_sampling(lib, case)
    # V = 1: every token is 0
    case = synth.chain_batched(seed=107, R=3, gamma=2, V=1, dtype="f32")
    case.tokens[:] = 0
    A, y, c = _run_chain(lib, case)
    assert (A == 2).all() and (y == 0).all()
    np.testing.assert_allclose(c, 1.0, atol=TOL)


def test_bad_token_sets_device_error(lib):
    import torch
    case = synth.chain_batched(seed=108, R=4, gamma=3, V=640, dtype="bf16")
    case.tokens[2, 1] = 640               # out of range
    dev = torch.device("cuda")
    target, draft = to_torch(case.target, dev), to_torch(case.draft, dev)
    tok, u = to_torch(case.tokens, dev, np.int32), to_torch(case.uniforms, dev, np.float32)
    nbytes = lib.specv_verify_chain_workspace_size(4, 3, 640, lib.SPECV_BF16)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    A, y, _ = lib.verify_chain(target, draft, tok, u, 1.0, None, False, workspace=ws)
    A, y = A.cpu().numpy(), y.cpu().numpy()
    assert lib.read_device_error(ws) == lib.SPECV_ERR_DEVICE_DATA
    ok = [0, 1, 3]
    if A[2] != -1:
        # the bad token sits after an earlier rejection only if A[2] < 1
        assert A[2] == 0
    assert (A[ok] >= 0).all()
    # a clean call clears the word
    case.tokens[2, 1] = 0
    lib.verify_chain(target, draft, to_torch(case.tokens, dev, np.int32), u, 1.0, None, False, workspace=ws)
    assert lib.read_device_error(ws) == lib.SPECV_OK


def test_tv_accept_matches_oracle(lib):
    import torch
    dev = torch.device("cuda")
    for dtype, V in (("bf16", 151936), ("f32", 3001)):
        case = synth.chain_batched(seed=109, R=3, gamma=4, V=V, dtype=dtype)
        target, draft = to_torch(case.target, dev), to_torch(case.draft, dev)
        for T in (1.0, 0.7):
            c = lib.tv_accept(target, draft, T).cpu().numpy()
            ref = oracle.tv_accept(case.target.f64, case.draft.f64, T)
            assert np.abs(c - ref).max() <= TOL
        c0 = lib.tv_accept(target, draft, 0.0).cpu().numpy()
        assert (c0 == oracle.tv_accept(case.target.f64, case.draft.f64, 0.0)).all()


def test_long_vocab_single_request(lib):
    """R=1, gamma=7, V=151936 bf16, one planted +8 peak per position, T=1 and T=0."""
    case = synth.chain_long_vocab(seed=2)
    _check_sampling(lib, case, "chain R=1 gamma=7 V=151936 T=1")
    g = synth.chain_long_vocab(seed=2, temperature=0.0)
    _check_greedy(lib, g)


def test_batched_full_size(lib):
    """The benchmarked workload: R=64, gamma=7, V=151936 bf16, T=1, every request
    and every c*_{r,k} checked against the oracle."""
    case = synth.chain_batched(seed=3)
    st, A, y, res = _check_sampling(lib, case, "chain R=64 gamma=7 V=151936 T=1 (benchmarked workload)")
    assert st.exact >= st.n - 8


def test_full_vocab_ragged_lengths(lib):
    """V=151936 bf16 (the pipelined ten-slot tiling) with ragged l_r in [0, gamma]:
    skipped positions, early bonus rows and l_r = 0 requests, T=1 and T=0."""
    case = synth.chain_batched(seed=111, R=16, gamma=7, ragged_lengths=True)
    assert (case.lengths == 0).any() or (case.lengths < 7).any()
    st, A, y, res = _check_sampling(lib, case, "chain R=16 ragged lengths V=151936 T=1")
    assert st.exact >= st.n - 2
    g = synth.chain_batched(seed=112, R=12, gamma=7, temperature=0.0, ragged_lengths=True)
    _check_greedy(lib, g)


def test_max_gamma_full_vocab(lib):
    """gamma = SPECV_MAX_GAMMA = 32 at V=151936 bf16: 33 positions per request."""
    case = synth.chain_batched(seed=113, R=3, gamma=32)
    st, A, y, res = _check_sampling(lib, case, "chain R=3 gamma=32 V=151936 T=1")
    assert st.exact >= st.n - 1
