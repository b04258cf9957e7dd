"""CPU oracle for the mixed-iteration paged attention step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code with the CUDA path (no kernels, headers, helpers or
constant tables) and imports nothing from the product package.

Modules
-------
attention
    NumPy fp64 definition of the step: gather a request's logical K/V through
    its block table, build the visibility mask explicitly, softmax, weighted
    sum; plus the KV-append scatter on raw bit patterns.
brute
    The same attention written as pure-Python loops with ``math.exp`` for
    tiny inputs; it cross-checks ``attention``.
rope
    The rotary embedding fused into the KV append (rotate-half pairs at the
    token's position, the fp64 angle table) and the fused append itself.
fp8
    The e4m3 codec from the format's definition, per-row quantization with
    fp32 scales, the fp8 append; attention over an fp8 cache is ``attention``
    on the dequantized values.

Every function is pinned by ``tests/test_oracle.py`` (worked example,
special cases reducing to library routines, closed forms, invariants and
brute force). No function is unpinned.
"""

from . import attention, brute, fp8, rope  # noqa: F401
