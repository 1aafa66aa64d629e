"""Layer-by-layer decode (clo_decode_layer) against the CPU oracle (needs a GPU).

A model that runs layer by layer only has layer l+1's query after layer l; the
library then takes one call per layer.  Calls over all layers must compute exactly
what one whole-step call computes, so the same lock-step checks apply: bit-exact
codes, selections, decisions, gathered rows and host bytes; outputs within 2e-3
max abs / 1e-3 relative L2."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from clo_harness import LockStep, Spec  # noqa: E402

pytestmark = pytest.mark.gpu


def test_layer_by_layer_warmup_persistent_and_mixed_steps():
    # 3 layers, warm-up thresholds, 1 persistent head per layer, G = 4, 2 selection chunks;
    # steps alternate between per-layer calls and whole-step calls
    spec = Spec(L=3, B=2, Hq=8, Hkv=2, d=128, ntok=[12000, 9000], seed=31, tau=None, warmup_steps=3, n_persist=1)
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        for t in range(8):
            ls.step(per_layer=(t % 3 != 1))
        assert all(r["persist"] == 6 for r in ls.log[3:])
        assert sum(r["hit"] for r in ls.log[3:]) > 0
    finally:
        ls.close()


def test_layer_by_layer_host_buffers():
    spec = Spec(L=2, B=2, Hq=4, Hkv=2, d=64, ntok=[3000, 2500], seed=33, tau=0.85)
    ls = LockStep(spec)
    try:
        for _ in range(4):
            ls.step(per_layer=True, io_on_device=False)
    finally:
        ls.close()


def test_layer_order_is_enforced():
    from host_offloaded_kv_gb300 import clo

    spec = Spec(L=2, B=1, Hq=2, Hkv=1, d=64, ntok=[500], seed=35, tau=0.9)
    ls = LockStep(spec)
    try:
        q = torch.from_numpy(ls.qs.next().view(np.int16)).cuda()
        out = torch.empty((2, 1, 2, 64), dtype=torch.float32, device="cuda")
        with pytest.raises(clo.CLOError) as e:
            ls.lib.decode_layer(1, q[1], out[1])                 # layer 1 before layer 0
        assert e.value.status == 5
        ls.lib.decode_layer(0, q[0], out[0])
        with pytest.raises(clo.CLOError) as e:
            ls.lib.decode_step(q, out)                           # a layer-by-layer step is open
        assert e.value.status == 5
        K = np.zeros((1, 1, 64), dtype=np.uint16)
        with pytest.raises(clo.CLOError) as e:
            ls.lib.append_kv(0, 0, K, K, src_is_device=False)    # appends wait for the step's end
        assert e.value.status == 5
        with pytest.raises(clo.CLOError) as e:
            ls.lib.decode_layer(2, q[1], out[1])                 # out of range
        assert e.value.status == 1
        ls.lib.decode_layer(1, q[1], out[1])
        ls.lib.sync()
        assert ls.lib.stats()["steps"] == 1
    finally:
        ls.close()
