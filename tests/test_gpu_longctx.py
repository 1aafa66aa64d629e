"""Lock-step parity at the per-unit sizes of the long-context and miss-heavy workloads
(needs a GPU and about 20 GiB of free host memory).

Each case keeps the full per-unit shape of its workload -- context length, top-k,
GQA group, persistent heads, query similarity -- with fewer layers and sequences,
which the kernels treat alike.  Every unit is compared with the oracle every step:
key and query codes, selections, gathered rows and host bytes bit for bit, reuse
decisions outside the 1e-4 band, attention outputs within 2e-3 / 1e-3.

* Qwen2.5-14B-shaped, 512K tokens (the synthesis page's motivating long context,
  section 3.4 attack 7): 40/8 heads (G = 5), k = 52429, 6 persistent heads per layer
  after warm-up; selection in 32 chunks of 16384 tokens, 52 attention splits and 205
  fetch chunks per unit, max_tokens at its cap.
* Llama3-8B-shaped at 128K tokens: k = 13108, thresholds from warm-up, no persistent
  heads.
* Miss-heavy batch (the abstract's batch up to 64): Llama3-8B shapes at 32K tokens,
  tau = 0.8 fixed and low query similarity (rho ~ U[0.2, 0.7]), so nearly every unit
  misses and the fetch carries every selection.
"""
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


needs_host = pytest.mark.skipif(_host_gib() < 24, reason="needs ~24 GiB of free host memory")


def _run(spec, steps):
    """Runs the lock-step case; returns its log and the library's k of sequence 0."""
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        for _ in range(steps):
            ls.step()
        return ls.log, ls.lib.k_of(0)
    finally:
        ls.close()


@needs_host
def test_qwen512k_unit_shape_parity():
    W = 4
    spec = Spec(L=2, B=1, Hq=40, Hkv=8, d=128, ntok=[524288], seed=3, tau=None, warmup_steps=W, n_persist=6,
                rho=(0.7, 0.98))
    log, k = _run(spec, W + 3)
    assert k == 52429
    post = log[W:]
    assert all(r["persist"] == 2 * 6 for r in post)
    assert all(r["hit"] + r["miss"] == 2 * 2 for r in post)


@needs_host
def test_llama128k_unit_shape_parity():
    W = 4
    spec = Spec(L=1, B=2, Hq=32, Hkv=8, d=128, ntok=[131072, 131072], seed=2, tau=None, warmup_steps=W,
                n_persist=0, rho=(0.6, 0.98))
    log, k = _run(spec, W + 3)
    assert k == 13108
    post = log[W:]
    assert sum(r["hit"] for r in post) > 0 and sum(r["miss"] for r in post) > 0


@needs_host
def test_stress_unit_shape_parity_mostly_misses():
    spec = Spec(L=2, B=4, Hq=32, Hkv=8, d=128, ntok=[32768] * 4, seed=4, tau=0.8, rho=(0.2, 0.7))
    log, k = _run(spec, 4)
    units = 2 * 4 * 8
    assert k == 3277
    later = log[1:]
    assert sum(r["miss"] for r in later) >= 0.9 * units * len(later)
