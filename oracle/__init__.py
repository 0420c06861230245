"""CPU fp64 oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``paged_kv_decode_bind_gb300``) never imports it and shares no
code with it; both sides take their inputs from ``pkv_inputs``.

Every function is pinned by ``tests/test_oracle.py`` against closed forms,
invariants, hand-derived worked examples (``tests/golden/``) and a library
routine (``torch.nn.functional.scaled_dot_product_attention`` in float64),
none of which the oracle itself calls.  The one part with no such pin is
agreement with the engine's own ``attn_paged_decode`` kernel, whose code and
outputs the pages do not give: for that comparison, parity unpinned.
"""
from .ref import *  # noqa: F401,F403
