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


def test_next_rows_reject_invalid_arguments_before_launch():
    """The scheduler's global form, the pruning, the confidence head and the
    DART tree validate on the host: every call below returns before any CUDA
    call (R == 0 is a no-op)."""
    import lossless_draft_verification_gb300 as specv
    E, U = specv.SPECV_ERR_INVALID_ARG, specv.SPECV_ERR_UNSUPPORTED
    fake = 1 << 20                          # 256-byte aligned, never dereferenced
    # global-search scheduler: R > B_max, missing SPS table, short workspace
    assert specv.specv_schedule_global(fake, fake, fake, 5, 3, 4, fake, None, fake, 256, None) == E
    assert specv.specv_schedule_global(fake, fake, None, 2, 3, 8, fake, None, fake, 256, None) == E
    assert specv.specv_schedule_global(fake, fake, fake, 2, 3, 8, fake, None, fake, 16, None) == E
    assert specv.specv_schedule_global(None, None, None, 0, 3, 8, None, None, None, 0, None) == 0
    # pruning: NaN threshold, misaligned confidences, R == 0
    assert specv.specv_prune_threshold(fake, 2, 3, float("nan"), fake, fake, 256, None) == E
    assert specv.specv_prune_threshold(fake + 2, 2, 3, 0.5, fake, fake, 256, None) == E
    assert specv.specv_prune_threshold(None, 0, 3, 0.5, None, None, 0, None) == 0
    # confidence head: NaN bias, negative gamma, missing anchor, short workspace
    ch = specv.specv_confidence_head
    assert ch(fake, fake, fake, float("nan"), fake, fake, 2, 3, 64, 100, 16, fake, fake, 256, None) == E
    assert ch(fake, fake, fake, 0.5, fake, fake, 2, -1, 64, 100, 16, fake, fake, 256, None) == E
    assert ch(fake, fake, fake, 0.5, None, fake, 2, 3, 64, 100, 16, fake, fake, 256, None) == E
    assert ch(fake, fake, fake, 0.5, fake, fake, 2, 3, 64, 100, 16, fake, fake, 8, None) == E
    assert ch(None, None, None, 0.5, None, None, 0, 3, 64, 100, 16, None, None, 0, None) == 0
    assert specv.specv_confidence_head_workspace_size(512, 7) == 256
    # DART tree: ranges of d, k, w, theta, dtype and T; unaligned rows and
    # shapes past the tile or shared-memory limits are unsupported
    ws = specv.specv_dart_tree_workspace_size
    BF, F32 = specv.SPECV_BF16, specv.SPECV_F32
    assert ws(16, 8, 151936, 25, 20, 59, BF) > 16 * 8 * 60 * 25 * 8
    assert ws(16, 9, 151936, 25, 20, 59, BF) == 0          # d > 8
    assert ws(16, 8, 151936, 33, 20, 59, BF) == 0          # k > 32
    assert ws(16, 8, 20, 25, 20, 59, BF) == 0              # k > V
    assert ws(16, 8, 151936, 25, 20, 1024, BF) == 0        # theta > 1023
    assert ws(16, 8, 151936, 32, 32, 59, BF) == 0          # 7200 nodes: over 200 KB of shared memory
    assert ws(16, 8, 128 * 2560 + 8, 25, 20, 59, BF) == 0  # more than 128 warp tiles per row
    assert ws(16, 8, 151936, 25, 20, 59, 7) == 0           # dtype
    dt = specv.specv_dart_tree
    args = lambda x, dtype, V, T, k, w, th, nb: (x, dtype, 2, 3, V, T, k, w, th, fake, fake, fake, fake, nb, None)
    nb = ws(2, 3, 4096, 4, 2, 11, BF)
    assert nb > 0
    assert dt(*args(fake, BF, 4096, 1.0, 0, 2, 11, nb)) == E                 # k < 1
    assert dt(fake, BF, 2, 0, 4096, 1.0, 4, 2, 11, fake, fake, fake, fake, nb, None) == E   # d < 1
    assert dt(*args(fake, BF, 4096, 0.0, 4, 2, 11, nb)) == E                 # T <= 0
    assert dt(*args(fake, BF, 4096, float("nan"), 4, 2, 11, nb)) == E
    assert dt(*args(fake, BF, 4096, 1.0, 4, 0, 11, nb)) == E                 # w < 1
    assert dt(*args(fake, BF, 4096, 1.0, 4, 2, 0, nb)) == E                  # theta < 1
    assert dt(*args(fake + 8, BF, 4096, 1.0, 4, 2, 11, nb)) == U             # rows not 16-byte aligned
    assert dt(*args(fake, BF, 4100, 1.0, 4, 2, 11, nb)) == U                 # V not a multiple of 8 (bf16)
    assert dt(*args(fake, F32, 4098, 1.0, 4, 2, 11, nb)) == U                # V not a multiple of 4 (float32)
    assert dt(*args(fake, BF, 4096, 1.0, 4, 2, 11, nb - 256)) == E           # short workspace
    assert dt(None, BF, 0, 3, 4096, 1.0, 4, 2, 11, None, None, None, None, 0, None) == 0


def test_tensor_helpers_check_shapes_before_any_device_call():
    """The helpers of the newer entry points reject mismatched tensors (and the
    DART helper unsupported shapes) before they touch a stream or a device."""
    import torch
    import lossless_draft_verification_gb300 as specv
    conf = torch.zeros(4, 7, dtype=torch.float32)
    sps = torch.ones(64, dtype=torch.float64)
    with pytest.raises(ValueError):
        specv.schedule_global(conf, sps, conf_stale=torch.zeros(4, 6, dtype=torch.float32))
    with pytest.raises(TypeError):
        specv.schedule_global(conf, sps.float())
    with pytest.raises(TypeError):
        specv.prune_threshold(conf.double(), 0.5)
    h = torch.zeros(4, 7, 64, dtype=torch.bfloat16)
    W1 = torch.zeros(100, 16, dtype=torch.bfloat16)
    anchor = torch.zeros(4, dtype=torch.int32)
    toks = torch.zeros(4, 7, dtype=torch.int32)
    with pytest.raises(ValueError):
        specv.confidence_head(h, W1, torch.zeros(64, dtype=torch.float32), 0.5, anchor, toks)    # w is H + rank long
    with pytest.raises(TypeError):
        specv.confidence_head(h.float(), W1, torch.zeros(80, dtype=torch.float32), 0.5, anchor, toks)
    with pytest.raises(TypeError):
        specv.dart_tree(torch.zeros(2, 3, 64, dtype=torch.float16))
    with pytest.raises(specv.SpecvError):
        specv.dart_tree(torch.zeros(2, 9, 4096, dtype=torch.bfloat16))                     # d > 8
    assert callable(specv.dart_tree) and "dart_tree" in specv.__all__
