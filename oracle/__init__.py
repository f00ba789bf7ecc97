"""float64 CPU oracle for exact scaled-dot-product attention and paged decode.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the product library never does, and
this package imports nothing from the product package.

The arithmetic lives in ``oracle.c`` (plain C, float64, three-pass safe
softmax per output row); this module only compiles it with gcc and marshals
numpy / torch CPU arrays into it.

Parity status of each function (the pins live in tests/test_oracle_pins.py):
  attention      pinned (worked example, closed forms, tiled-vs-naive, mpmath)
  attention_bwd  pinned (central finite differences of attention, softmax
                 shift invariance, constant-value and probability-sum identities)
  paged_decode   pinned (equal to attention on the gathered keys; table invariance)
  paged_attention pinned (grouped heads equal multi-head attention on a cache
                 whose KV heads are repeated; prefill chunks equal dense
                 bottom-right causal attention on the gathered keys; one
                 token per request equals paged_decode; closed forms)
  varlen_attention pinned (equal to dense bottom-right causal attention per
                 request; it is paged_attention on one-row pages)
  decode_elems   pinned (bf16 / e4m3fn codes against torch's conversions)
"""
from .oracle import (  # noqa: F401
    OracleError,
    attention,
    attention_bwd,
    build,
    decode_elems,
    default_threads,
    paged_attention,
    paged_decode,
    varlen_attention,
)
