"""fp64 CPU oracle for single-token decode attention over a KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The CUDA library never calls it, and it shares no code with the
CUDA path: the only common module is ``kvgen`` (seeded random inputs, no
attention arithmetic).

Every function is the plain definition from the source pages, in numpy float64
on values widened exactly from bf16.  See ``oracle/attention.py`` for the
citations.  Parity pins (tests that tie each function to something other than
itself) live in ``tests/test_oracle_pins.py``.
"""
from .attention import (  # noqa: F401
    attend, gqa_decode, mla_decode_absorbed, mla_absorb_q, mla_project_out, mla_decode_nonabsorbed,
    combine_splits, split_partials, rope_rotate, rope_matrix,
    append_rope_mla, append_rope_gqa, bf16_to_f64, f64_to_bf16_bits,
    bf16_bits_to_f64, gather_tokens, gather_slots, window_slots,
    e4m3_bits_to_f64, f64_to_e4m3_bits, dequant_e4m3, gqa_decode_fp8, E4M3_MAX,
    dequant_mla_e4m3, mla_decode_absorbed_fp8,
    mla_prefill_expand, mla_prefill,
)
from . import closed_forms  # noqa: F401
