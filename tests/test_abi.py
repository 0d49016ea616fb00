"""Host-side checks of the C-ABI library that need no GPU: it builds, loads,
exports every symbol include/specv.h declares, and rejects invalid arguments
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cdll():
    from lossless_draft_verification_gb300 import build as b
    path = b.build()
    lib = ctypes.CDLL(path)
    return lib


def _declared():
    src = open(os.path.join(ROOT, "include", "specv.h")).read()
    return sorted(set(re.findall(r"SPECV_API\s+[\w\s\*]+?\b(specv_\w+)\s*\(", src)))


def test_header_declares_the_five_entry_points():
    names = _declared()
    for n in ("specv_verify_chain", "specv_verify_tree_greedy", "specv_markov_draft", "specv_tv_accept",
              "specv_schedule"):
        assert n in names


def test_every_declared_symbol_is_exported(cdll):
    import lossless_draft_verification_gb300 as specv
    for name in _declared():
        assert hasattr(cdll, name), name
        assert name in specv.EXPORTED, f"binding lacks {name}"
        assert callable(getattr(specv, name))


def test_version_and_status_strings():
    import lossless_draft_verification_gb300 as specv
    specv.load()
    assert specv.specv_abi_version() == 1
    for s in range(6):
        assert specv.status_string(s)


def test_workspace_sizes_are_host_only():
    import lossless_draft_verification_gb300 as specv
    n = specv.specv_verify_chain_workspace_size(64, 7, 151936, specv.SPECV_BF16)
    assert 256 < n < 64 << 20
    assert specv.specv_verify_chain_workspace_size(-1, 7, 10, specv.SPECV_BF16) == 0
    assert specv.specv_verify_chain_workspace_size(1, 33, 10, specv.SPECV_BF16) == 0
    assert specv.specv_verify_chain_workspace_size(1, 1, 10, 7) == 0
    assert specv.specv_verify_tree_greedy_workspace_size(16, 60, 151936, specv.SPECV_BF16) > 256
    assert specv.specv_markov_draft_workspace_size(512, 7, 129280, 256) > 512 * 129280 * 4
    assert specv.specv_schedule_workspace_size(512, 7) == 256
    assert specv.specv_schedule_workspace_size(8192, 2) == 0


def test_invalid_arguments_rejected_before_launch():
    """Each call below fails host validation, so it never reaches the CUDA runtime."""
    import lossless_draft_verification_gb300 as specv
    E = specv.SPECV_ERR_INVALID_ARG
    fake = 1 << 20                          # never dereferenced
    # negative R, gamma too large, bad dtype, negative or tiny temperature
    assert specv.specv_verify_chain(fake, fake, 1, fake, None, fake, -1, 3, 10, 1.0, fake, fake, None, fake, 1 << 20, None) == E
    assert specv.specv_verify_chain(fake, fake, 1, fake, None, fake, 2, 40, 10, 1.0, fake, fake, None, fake, 1 << 20, None) == E
    assert specv.specv_verify_chain(fake, fake, 9, fake, None, fake, 2, 3, 10, 1.0, fake, fake, None, fake, 1 << 20, None) == E
    assert specv.specv_verify_chain(fake, fake, 1, fake, None, fake, 2, 3, 10, -1.0, fake, fake, None, fake, 1 << 20, None) == E
    assert specv.specv_verify_chain(fake, fake, 1, fake, None, fake, 2, 3, 10, 1e-9, fake, fake, None, fake, 1 << 20, None) == E
    # missing uniforms at T > 0, missing draft, misaligned workspace, short workspace
    assert specv.specv_verify_chain(fake, fake, 1, fake, None, None, 2, 3, 10, 1.0, fake, fake, None, fake, 1 << 20, None) == E
    assert specv.specv_verify_chain(fake, None, 1, fake, None, fake, 2, 3, 10, 1.0, fake, fake, None, fake, 1 << 20, None) == E
    assert specv.specv_verify_chain(fake, fake, 1, fake, None, fake, 2, 3, 10, 1.0, fake, fake, None, fake + 4, 1 << 20, None) == E
    assert specv.specv_verify_chain(fake, fake, 1, fake, None, fake, 2, 3, 10, 1.0, fake, fake, None, fake, 16, None) == E
    # R == 0 is a no-op
    assert specv.specv_verify_chain(None, None, 1, None, None, None, 0, 3, 10, 1.0, None, None, None, None, 0, None) == 0
    assert specv.specv_tv_accept(fake, fake, 1, 2, 3, 2, 10, 1.0, fake, fake, 1 << 20, None) == E
    assert specv.specv_verify_tree_greedy(fake, 1, fake, fake, 2, 5, 10, 0, fake, fake, fake, fake, 1 << 20, None) == E
    assert specv.specv_verify_tree_greedy(fake, 1, fake, fake, 2, 2000, 10, 4, fake, fake, fake, fake, 1 << 20, None) == E
    assert specv.specv_markov_draft(fake, fake, fake, fake, fake, 2, 3, 10, 20, 1.0, fake, None, 0, fake, 1 << 30, None) == E
    assert specv.specv_schedule(fake, fake, 5, 3, 4, fake, None, fake, 256, None) == E   # R > B_max
    assert specv.specv_schedule(fake, fake, 5000, 3, 8192, fake, None, fake, 256, None) == E
