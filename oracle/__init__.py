"""Plain fp64 CPU oracle for gated causal softmax attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this package: only the
tests, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use
it.  It shares no code with the CUDA path.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py`` against
library routines (fp64 ``scaled_dot_product_attention``, ``torch.autograd``,
``torch.float8_e4m3fn`` / ``torch.bfloat16`` conversions), closed forms, finite
differences, invariants and hand-derived fixtures (``tests/golden/``), and on random small
cases in ``tests/test_oracle_properties.py``.  No function is "parity unpinned".
"""
from .formats import bf16_round, e4m3_decode  # noqa: F401
from .attention import (  # noqa: F401
    gate_cumsum,
    prefill_forward,
    prefill_backward,
    decode_paged,
    decode_partials,
    decode_combine,
    decode_paged_splitk,
    gather_kv,
    rel_rms,
)
