"""Quantised host pool (kv_bits 4 and 2) against the CPU oracle (needs a GPU).

The pool stores b-bit asymmetric codes with an fp32 (scale, min) per 64-channel
group; the fetch dequantises into the bf16 cache slots and the resident fill into
the persistent heads' HBM copies.  The oracle applies the same quantisation to the
appended rows, so the lock-step checks stay bit-exact for codes, selections,
decisions, gathered rows and host bytes (k x record bytes per missed unit), and
outputs within 2e-3 max abs / 1e-3 relative L2."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as orc  # noqa: E402
from clo_harness import LockStep, Spec  # noqa: E402

pytestmark = pytest.mark.gpu


def test_int4_pool_fixed_tau():
    spec = Spec(L=2, B=2, Hq=8, Hkv=2, d=128, ntok=[9000, 6000], seed=51, tau=0.85, kv_bits=4)
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        for t in range(5):
            ls.step(per_layer=(t == 3))
        assert sum(r["miss"] for r in ls.log) > 0 and sum(r["hit"] for r in ls.log) > 0
        assert orc.kv_record_bytes(128, 4) == 128
    finally:
        ls.close()


def test_int2_pool_warmup_and_persistent_heads():
    spec = Spec(L=2, B=2, Hq=4, Hkv=2, d=64, ntok=[5000, 4000], seed=53, tau=None, warmup_steps=3, n_persist=1,
                kv_bits=2)
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        for _ in range(6):
            ls.step()
        assert all(r["persist"] == 4 for r in ls.log[3:])
    finally:
        ls.close()


def test_int4_pool_host_buffers():
    spec = Spec(L=1, B=1, Hq=4, Hkv=1, d=128, ntok=[3000], seed=55, tau=0.9, kv_bits=4)
    ls = LockStep(spec)
    try:
        for _ in range(3):
            ls.step(io_on_device=False)
    finally:
        ls.close()
