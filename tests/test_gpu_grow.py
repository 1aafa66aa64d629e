"""Streaming growth (clo_append_step) against the CPU oracle (needs a GPU).

Each step first appends one token to every (layer, sequence) on the device (record,
key code, length, top-k count), then decodes over the grown context.  The lock-step
checks stay bit-exact (all key codes including the new ones, selections with the
growing k, decisions, gathered rows, host bytes) and outputs within 2e-3 / 1e-3."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from clo_harness import LockStep, Spec  # noqa: E402

pytestmark = pytest.mark.gpu


def test_growing_context_crosses_k_and_chunk_boundaries():
    # 8190 -> 8196 tokens: k = ceil(0.1 N) goes 819 -> 820, and the context crosses the
    # 8192-token selection chunk; host and device sources alternate
    spec = Spec(L=2, B=2, Hq=8, Hkv=2, d=128, ntok=[8190, 5000], seed=71, tau=0.85, max_tokens=8200)
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        for t in range(6):
            ls.append_step(src_is_device=(t % 2 == 0))
            ls.step()
        ls.check_key_codes()
        assert ls.lib.k_of(0) == 820 and ls.orc.k_of(0) == 820
    finally:
        ls.close()


def test_growing_context_quantised_pool_with_persistent_heads():
    spec = Spec(L=2, B=2, Hq=4, Hkv=2, d=64, ntok=[3000, 2000], seed=73, tau=None, warmup_steps=3, n_persist=1,
                kv_bits=4, max_tokens=3100)
    ls = LockStep(spec)
    try:
        for _ in range(7):
            ls.append_step()
            ls.step()
        ls.check_key_codes()
        assert all(r["persist"] == 4 for r in ls.log[3:])
    finally:
        ls.close()


def test_append_step_at_capacity_is_refused():
    from host_offloaded_kv_gb300 import clo

    spec = Spec(L=1, B=1, Hq=2, Hkv=1, d=64, ntok=[100], seed=75, tau=0.9, max_tokens=101)
    ls = LockStep(spec)
    try:
        ls.append_step()
        ls.step()
        K = torch.zeros((1, 1, 1, 64), dtype=torch.int16, device="cuda")
        with pytest.raises(clo.CLOError) as e:
            ls.lib.append_step(K, K)
        assert e.value.status == 6
    finally:
        ls.close()
