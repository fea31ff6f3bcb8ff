"""Plain float64 CPU oracle for exact attention and Flash-Decoding.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library and
its Python binding never import it, and it never imports them.

The arithmetic lives in ``fa_oracle.c`` (plain C, float64, OpenMP over query
rows); this module only compiles it with gcc, loads it with ctypes and
marshals numpy/torch arrays.  Every function cites the passage it follows in
the C source.
"""
from .oracle import (  # noqa: F401
    build,
    library_path,
    softmax_naive,
    softmax_safe,
    online_softmax_trace,
    block_state,
    state_merge,
    lse_reduce,
    attend_scores,
    sdpa_rows,
    sdpa_forward,
    decode,
    decode_paged,
    sdpa_forward_f64,
    sdpa_backward,
    e4m3_to_f64,
    sdpa_forward_e4m3,
    max_threads,
)
