"""Failure detection without a GPU fault: a ready flag that nothing sets makes the
bounded device-side wait give up, the step reports CLO_ERR_TIMEOUT, and the context
stays usable; host-side argument and state errors come back as status codes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from clo_harness import LockStep, Spec  # noqa: E402

pytestmark = pytest.mark.gpu


def test_dropped_ready_flag_times_out_then_recovers():
    from host_offloaded_kv_gb300 import clo

    # tau = 2: every unit misses, so every attention split of layer 1 waits on a fetch flag
    spec = Spec(L=2, B=2, Hq=4, Hkv=2, d=64, ntok=[2000, 2000], seed=31, tau=2.0)
    ls = LockStep(spec)
    try:
        ls.step()  # a normal step first
        ls.lib.set(clo.CLO_SET_WAIT_TIMEOUT_NS, 20_000_000)  # 20 ms
        ls.lib.set(clo.CLO_SET_DROP_FLAG_LAYER, 1)           # the fetch of layer 1 never signals
        q = ls.qs.next()
        qd = torch.from_numpy(q.view(np.int16)).cuda()
        out = torch.empty((2, 2, 4, 64), dtype=torch.float32, device="cuda")
        ls.lib.decode_step(qd, out)          # enqueues and returns
        with pytest.raises(clo.CLOError) as e:
            ls.lib.sync()
        assert e.value.status == clo.CLO_ERR_TIMEOUT
        st = ls.lib.stats()                  # the latch was cleared when reported
        assert st["timeouts"] >= 4           # 2 seqs x 2 heads x 1 split of layer 1
        ls.orc.step(q)                       # keep the oracle in lock-step (all units missed)
        ls.lib.set(clo.CLO_SET_DROP_FLAG_LAYER, -1)
        ls.lib.set(clo.CLO_SET_WAIT_TIMEOUT_NS, 2_000_000_000)
        for _ in range(2):
            ls.step()                        # full parity again
    finally:
        ls.close()


def test_host_side_errors_are_status_codes():
    from host_offloaded_kv_gb300 import clo
    from host_offloaded_kv_gb300.clo import CLOContext, CLOError
    from host_offloaded_kv_gb300.synth import Synth

    syn = Synth(3)
    L, B, Hq, Hkv, d = 2, 2, 4, 2, 64
    R = syn.hash_matrices(L, Hkv, d)
    lib = CLOContext(n_layers=L, batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, max_tokens=100, hash_R=R,
                     tau=np.full(L * Hkv, 0.8, dtype=np.float32))
    try:
        q = torch.zeros((L, B, Hq, d), dtype=torch.int16, device="cuda")
        out = torch.empty((L, B, Hq, d), dtype=torch.float32, device="cuda")
        with pytest.raises(CLOError) as e:
            lib.decode_step(q, out)  # nothing appended yet
        assert e.value.status == clo.CLO_ERR_STATE
        K, V = syn.layer_seq_kv(0, 0, Hkv, 0, 80, d)
        lib.append_kv(0, 0, K, V, src_is_device=False)
        with pytest.raises(CLOError) as e:
            lib.append_kv(0, 0, K, V, src_is_device=False)  # 160 > max_tokens 100
        assert e.value.status == clo.CLO_ERR_CAPACITY
        with pytest.raises(CLOError) as e:
            lib.decode_step(q, out)  # layer 1 / seq 1 empty: ragged
        assert e.value.status == clo.CLO_ERR_STATE
        with pytest.raises(CLOError) as e:
            clo.clo_append_kv(lib.ctx, 5, 0, K, V, 80, False)
        assert e.value.status == clo.CLO_ERR_INVALID
        with pytest.raises(CLOError) as e:
            clo.clo_debug_get(lib.ctx, 99, 0, 0, 0, np.empty(4, dtype=np.uint8))
        assert e.value.status == clo.CLO_ERR_INVALID
        with pytest.raises(CLOError) as e:
            lib.set(77, 1)
        assert e.value.status == clo.CLO_ERR_INVALID
        # the context is still usable: fill it and decode
        for l in range(L):
            for b in range(B):
                if (l, b) != (0, 0):
                    lib.append_kv(l, b, *syn.layer_seq_kv(l, b, Hkv, 0, 80, d), src_is_device=False)
        q = torch.from_numpy(syn.query_stream(L, B, Hq, d, 0.6, 0.9).next().view(np.int16)).cuda()
        lib.decode_step(q, out)
        lib.sync()
        assert torch.isfinite(out).all()
    finally:
        lib.close()
