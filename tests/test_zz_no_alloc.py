"""specv_verify_chain_noalloc against specv_verify_chain, both through the C ABI.

The allocation-free call runs the same kernels on a built-in scratch buffer,
so its outputs must equal the workspace call's bit for bit.  Each case runs
the allocation-free call twice in a row (the second on a buffer the first has
dirtied) and once more after a different problem.  This file sorts last so
that the GPU run also covers a process in which every other entry point has
already run."""
import numpy as np
import pytest

import synth
from parity import to_torch


def _args(lib, case, dev):
    import torch
    t = to_torch(case.target, dev)
    d = to_torch(case.draft, dev)
    x = to_torch(case.tokens, dev, np.int32)
    u = to_torch(case.uniforms, dev, np.float32)
    ln = None if case.lengths is None else to_torch(case.lengths, dev, np.int32)
    R, P, V = t.shape
    code = lib.SPECV_BF16 if t.dtype == torch.bfloat16 else lib.SPECV_F32
    return t, d, x, u, ln, R, P - 1, V, code


def _outputs(R, gamma, dev):
    import torch
    return (torch.full((R,), -7, dtype=torch.int32, device=dev), torch.full((R,), -7, dtype=torch.int32, device=dev),
            torch.full((R, gamma), 7.0, dtype=torch.float32, device=dev))


def _p(x):
    return None if x is None else x.data_ptr()


def _with_workspace(lib, case, T, dev):
    import torch
    t, d, x, u, ln, R, gamma, V, code = _args(lib, case, dev)
    acc, tok, cst = _outputs(R, gamma, dev)
    nbytes = lib.specv_verify_chain_workspace_size(R, gamma, V, code)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = lib.specv_verify_chain(_p(t), _p(d), code, _p(x), _p(ln), _p(u) if T > 0 else None, R, gamma, V, T,
                                _p(acc), _p(tok), _p(cst), _p(ws), nbytes, torch.cuda.current_stream().cuda_stream)
    assert st == lib.SPECV_OK, lib.status_string(st)
    return acc, tok, cst


def _no_alloc(lib, case, T, dev):
    import torch
    t, d, x, u, ln, R, gamma, V, code = _args(lib, case, dev)
    acc, tok, cst = _outputs(R, gamma, dev)
    st = lib.specv_verify_chain_noalloc(_p(t), _p(d), code, _p(x), _p(ln), _p(u) if T > 0 else None, R, gamma, V, T,
                                        _p(acc), _p(tok), _p(cst), torch.cuda.current_stream().cuda_stream)
    assert st == lib.SPECV_OK, lib.status_string(st)
    return acc, tok, cst


def _same(a, b):
    import torch
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))   # bitwise, NaN included


@pytest.mark.gpu
def test_noalloc_matches_workspace_call(lib):
    import torch
    dev = torch.device("cuda")
    big = synth.chain_batched(seed=31, R=12, gamma=7, V=151936, dtype="bf16", ragged_lengths=True)
    small = synth.chain_tiny(seed=32, R=5, gamma=4, V=3001, dtype="f32")
    for case, T in ((big, 1.0), (small, 0.0), (small, 1.0), (big, 0.0)):
        ref = _with_workspace(lib, case, T, dev)
        first = _no_alloc(lib, case, T, dev)
        second = _no_alloc(lib, case, T, dev)
        torch.cuda.synchronize()
        _same(first, ref)
        _same(second, ref)
        assert (ref[0] >= 0).all() and (ref[1] >= 0).all()
    # after a different problem has used the buffer
    again = _no_alloc(lib, big, 1.0, dev)
    _same(again, _with_workspace(lib, big, 1.0, dev))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """Decided on the host before any CUDA call, so it needs no GPU."""
    import lossless_draft_verification_gb300 as specv
    specv.load()
    fake = 1 << 20                                   # never dereferenced
    need = specv.specv_verify_chain_workspace_size(2048, 7, 151936, specv.SPECV_BF16)
    assert need > 16 << 20
    st = specv.specv_verify_chain_noalloc(fake, fake, specv.SPECV_BF16, fake, None, fake, 2048, 7, 151936, 1.0, fake,
                                          fake, None, None)
    assert st == specv.SPECV_ERR_SCRATCH_LIMIT
    assert "scratch" in specv.status_string(st)
    assert specv.specv_verify_chain_workspace_size(1024, 7, 151936, specv.SPECV_BF16) <= 16 << 20
    # an invalid shape is an argument error, an empty batch a no-op
    assert specv.specv_verify_chain_noalloc(fake, fake, specv.SPECV_BF16, fake, None, fake, 4, 40, 100, 1.0, fake,
                                            fake, None, None) == specv.SPECV_ERR_INVALID_ARG
    assert specv.specv_verify_chain_noalloc(None, None, specv.SPECV_BF16, None, None, None, 0, 7, 100, 1.0, None,
                                            None, None, None) == specv.SPECV_OK
