"""FP64 CPU oracle for the AttnRes read operator (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this package.  It shares no code with the CUDA library.  See
``attnres_oracle.c`` for the definition it follows.
"""
from .oracle import attnres_oracle, build_oracle, oracle_library_path  # noqa: F401
from .multi import attnres_multi_oracle, attnres_selected_oracle  # noqa: F401,E402
from .partial import attnres_partial_oracle  # noqa: F401,E402
