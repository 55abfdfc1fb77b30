"""CPU oracle for the quantized decode linear layer.

TEST INFRASTRUCTURE ONLY: a plain, slow, fp64 restatement of what the layer computes,
used to check the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the library itself never does, and the
oracle never imports the library.  See ``oracle/qlinear_oracle.py`` for the functions and
the readings taken where the source pages are silent.
"""
from . import formats, qlinear_oracle  # noqa: F401
from .formats import *  # noqa: F401,F403
from .qlinear_oracle import *  # noqa: F401,F403
