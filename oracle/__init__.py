"""Float64 CPU oracle for paged MLA decode: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the library never does.
"""
from .mla_oracle import (attend, decode_bf16, decode_e4m3, dequantize,  # noqa: F401
                         gather_request, lse_merge, mla_decode, mla_decode_inputs,
                         unabsorbed_attention)
