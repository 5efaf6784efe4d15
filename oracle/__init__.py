"""Plain CPU oracle for the truly sparse linear layer.

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package; the library in
``sparse_linear_layer_gb300`` never does.  See ``snk_oracle.c`` for what each
function computes and which passage of the pages it follows.
"""
from .oracle import *  # noqa: F401,F403
