"""Online adaptive thresholds (adaptive_tau) against the CPU oracle (needs a GPU).

After warm-up (or from fixed starting thresholds) every step folds the batch-mean
adjacent-step cosine of each (layer, kv head) into s_hat and sets tau = s_hat -
offset for the next step.  The lock-step harness compares the device thresholds
with the oracle's after every step (1e-5) besides the usual bit-exact codes,
selections, decisions and gathered rows."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from clo_harness import LockStep, Spec  # noqa: E402

pytestmark = pytest.mark.gpu


def test_adaptive_tau_after_warmup_with_persistent_heads():
    spec = Spec(L=2, B=3, Hq=8, Hkv=4, d=128, ntok=[5000, 7000, 4000], seed=43, tau=None, warmup_steps=3,
                n_persist=1, adaptive_tau=True, tau_ema=0.25, rho=(0.5, 0.99))
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        taus = []
        for t in range(9):
            ls.step(per_layer=(t == 5))
            if t >= 2:
                taus.append(ls.lib.tau().copy())
        assert not np.allclose(taus[0], taus[-1])     # the thresholds moved
        assert sum(r["hit"] for r in ls.log[3:]) > 0 and sum(r["miss"] for r in ls.log[3:]) > 0
    finally:
        ls.close()


def test_adaptive_tau_from_fixed_thresholds():
    spec = Spec(L=1, B=2, Hq=4, Hkv=2, d=64, ntok=[3000, 3000], seed=45, tau=0.2, adaptive_tau=True,
                tau_ema=0.5, rho=(0.9, 0.99))
    ls = LockStep(spec)
    try:
        for _ in range(6):
            ls.step()
        assert np.all(ls.lib.tau() > 0.5)   # tracks the live similarity (rho >= 0.9)
    finally:
        ls.close()
