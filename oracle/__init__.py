"""CPU oracle of the CLO decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls anything here.
"""
from .clo_oracle import (  # noqa: F401
    OracleCLO,
    load_oracle,
    kv_bytes_per_token,
    kv_roundtrip,
    kv_record_bytes,
    hash_codes,
    cosine,
    scores,
    topk,
    attention,
    exact_sign,
    topk_count,
    DEC_HIT,
    DEC_MISS,
    DEC_PERSIST,
)
