"""Oracle for gated delta-rule linear attention with the bounded decay g = -5*sigmoid(a).

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import anything from this package. The product
library never imports, links or runs it, and it never imports the product.

Contents
--------
``recurrence``  the oracle proper: the plain fp64 token-by-token recurrence, in C
                (``kda_oracle.c``) with a ctypes loader.
``chunked``     an fp64 NumPy restatement of the 16-token chunked algebra, used only
                to pin that the chunked form equals the recurrence.
``brute``       an fp64 NumPy unrolled transition-matrix form, used only on tiny
                inputs to pin the recurrence.
``backward``    the gradients of the recurrence (its vector-Jacobian product), by
                PyTorch reverse-mode differentiation of a plain fp64 token loop;
                pinned to central finite differences of ``recurrence``.

``projection``  the gate projection a = x W^T + b (one fp64 matrix product).

``recurrence.decode_step`` is the recurrence on one-token sequences (a decode step).
"""
from .recurrence import build, kda_forward, oracle_library_path  # noqa: F401
