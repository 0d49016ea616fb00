import os
import sys

# numpy asks the kernel for transparent huge pages on large arrays; where THP
# defragmentation compacts memory on each fault, the oracle's large temporaries
# then spend most of their time in the kernel.  Set before numpy is imported
# (here and in the spawned workers, which inherit the environment).
os.environ.setdefault("NUMPY_MADVISE_HUGEPAGE", "0")

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_terminal_summary(terminalreporter):
    """Print the flagged-threshold counts the parity tests recorded: decisions
    the GPU took differently from the oracle because the uniform lay within
    1e-5 of the threshold (allowed, but counted and reported)."""
    parity = sys.modules.get("parity")
    if parity is None or not getattr(parity, "REPORT", None):
        return
    terminalreporter.write_sep("-", "parity: exact and flagged-threshold counts")
    for name, counts in parity.REPORT:
        terminalreporter.write_line(f"{name}: " + ", ".join(f"{k} {v}" for k, v in counts.items()))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library through its Python binding; the binding raises if the
    shared object is missing, so GPU tests never run on a fallback."""
    import lossless_draft_verification_gb300 as specv
    from lossless_draft_verification_gb300 import build
    build.build()
    specv.load()
    return specv


@pytest.fixture(scope="session")
def pool():
    """Worker processes for the oracle's long Monte Carlo pins.  Their trials
    are split into independent blocks of rows whose random numbers are the
    same as in a single call, so spreading them over the host cores changes
    no sample.  Spawned, never forked, so no parent state is inherited."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    n = max(1, min(8, os.cpu_count() or 1))
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"              # one thread per worker: no oversubscription
    # glibc keeps freed blocks in the heap instead of unmapping them, so the
    # oracle's repeated large temporaries reuse pages instead of faulting anew
    os.environ["MALLOC_MMAP_MAX_"] = "0"
    os.environ["MALLOC_TRIM_THRESHOLD_"] = str(1 << 34)
    with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
        yield ex


def split_rows(n, parts):
    """[start, stop) bounds of `parts` near-equal blocks of n rows."""
    step = -(-n // parts)
    return [(s, min(n, s + step)) for s in range(0, n, step)]
