"""Parity at the benchmark's full size (needs a GPU and ~40 GB of host memory).

Llama3-8B-shaped stack, 32 layers, batch 8, 32/8 heads, head_dim 128, 32K-token
context per sequence in pinned host memory, top-k 10 %, thresholds from 16 warm-up
steps, 4 persistent heads per layer -- the workload bench.py times, in the same
launch configuration.  The oracle follows every unit's reuse decision and host
bytes, and checks 16 sampled units (all kv heads of two (layer, sequence) pairs,
so persistent and non-persistent heads both appear) bit-exactly: key and query
codes, selections, gathered rows; attention outputs within 2e-3 / 1e-3."""
import os

import pytest

torch = pytest.importorskip("torch")

from clo_harness import LockStep, Spec  # noqa: E402

pytestmark = pytest.mark.gpu


def _host_gib():
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) / 2**20
    return 0.0


@pytest.mark.skipif(_host_gib() < 45, reason="needs ~45 GiB of free host memory for the 32 GiB pinned pool")
def test_llama32k_full_size_sampled_parity():
    from host_offloaded_kv_gb300.synth import get_workload

    w = get_workload("llama32k")
    sample = [(0, 0, h) for h in range(w.n_kv_heads)] + [(w.n_layers - 1, w.batch - 1, h) for h in range(w.n_kv_heads)]
    spec = Spec(L=w.n_layers, B=w.batch, Hq=w.n_q_heads, Hkv=w.n_kv_heads, d=w.head_dim,
                ntok=[w.n_tokens] * w.batch, seed=w.seed, topk=w.topk, topk_ratio=w.topk_ratio, tau=None,
                warmup_steps=w.warmup_steps, tau_offset=w.tau_offset, n_persist=w.n_persist,
                rho=(w.rho_lo, w.rho_hi), hh_ratio=w.hh_ratio, sample=sample)
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        for _ in range(w.warmup_steps + 4):
            ls.step()
        post = ls.log[w.warmup_steps:]
        assert all(r["persist"] == w.n_layers * w.batch * w.n_persist for r in post)
        assert sum(r["hit"] for r in post) > 0 and sum(r["miss"] for r in post) > 0
        # the sampled pairs hold both persistent and reused/missed heads
        kinds = {int(ls.orc.persist[l, h]) for (l, b, h) in sample}
        assert kinds == {0, 1}
    finally:
        ls.close()
