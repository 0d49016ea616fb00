"""CPU oracle (test infrastructure only).

Plain float64 restatement of the verification path, used by the tests, the
smoke check and the CPU baseline of the benchmark.  The CUDA library neither
imports nor links anything here.
"""
from .specv_oracle import *  # noqa: F401,F403
from .specv_oracle import __all__  # noqa: F401
