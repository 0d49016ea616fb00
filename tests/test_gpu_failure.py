"""Failure detection without a GPU fault: a bounded device-side wait that is
made to run out reports SPECV_ERR_TIMEOUT through the workspace error word,
the kernel returns, and the context stays usable for the next call.

The wait is the poll-limited mbarrier wait the Markov kernel uses for its
copies; here it waits on a barrier that nothing arrives at (no copy targets
it), so it ends after its poll budget, never by a trap."""
import time

import numpy as np
import pytest

import oracle
import synth
from parity import to_torch


def test_selftest_arguments_are_checked_on_the_host():
    import lossless_draft_verification_gb300 as specv
    from lossless_draft_verification_gb300 import build
    build.build()
    specv.load()
    E = specv.SPECV_ERR_INVALID_ARG
    fake = 1 << 20                                   # never dereferenced
    assert specv.specv_selftest_bounded_wait(0, 0, fake, 256, None) == E
    assert specv.specv_selftest_bounded_wait(65537, 0, fake, 256, None) == E
    assert specv.specv_selftest_bounded_wait(16, 0, None, 256, None) == E
    assert specv.specv_selftest_bounded_wait(16, 0, fake, 255, None) == E
    assert specv.specv_selftest_bounded_wait(16, 0, fake + 8, 256, None) == E


@pytest.mark.gpu
def test_bounded_wait_times_out_and_the_context_survives(lib):
    import torch
    dev = torch.device("cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    sp = torch.cuda.current_stream().cuda_stream
    # control: the barrier's phase completes, the wait succeeds
    assert lib.specv_selftest_bounded_wait(64, 1, ws.data_ptr(), 256, sp) == lib.SPECV_OK
    assert lib.read_device_error(ws) == lib.SPECV_OK
    # nothing arrives: the wait gives up after its polls and says so
    t0 = time.perf_counter()
    assert lib.specv_selftest_bounded_wait(1024, 0, ws.data_ptr(), 256, sp) == lib.SPECV_OK
    assert lib.read_device_error(ws) == lib.SPECV_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # the context is intact: a verification call right after is correct
    case = synth.chain_tiny(seed=1, R=3, gamma=4, V=1024)
    A, y, c = lib.verify_chain(to_torch(case.target, dev), to_torch(case.draft, dev),
                               to_torch(case.tokens, dev, np.int32), to_torch(case.uniforms, dev), 1.0)
    res = oracle.verify_chain(case.target.f64, case.draft.f64, case.tokens, case.uniforms, 1.0)
    assert (A.cpu().numpy() == res.accepted).all() and (y.cpu().numpy() == res.token).all()
    assert np.abs(c.cpu().numpy() - res.c_star).max() <= 1e-5
    # and the word is rewritten by the next successful wait
    assert lib.specv_selftest_bounded_wait(64, 1, ws.data_ptr(), 256, sp) == lib.SPECV_OK
    assert lib.read_device_error(ws) == lib.SPECV_OK
