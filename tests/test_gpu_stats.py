"""The per-step byte history (timing mode) agrees with the per-step counters of
clo_stats: every step's host-link and algorithmic HBM bytes, whole steps and
layer-by-layer steps alike (needs a GPU)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def test_step_byte_history_matches_per_step_counters():
    from host_offloaded_kv_gb300.clo import CLOContext
    from host_offloaded_kv_gb300.synth import Synth

    L, B, Hq, Hkv, d, N = 2, 2, 8, 2, 64, 3000
    syn = Synth(31)
    lib = CLOContext(n_layers=L, batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, max_tokens=N,
                     hash_R=syn.hash_matrices(L, Hkv, d), tau=np.full(L * Hkv, 0.85, dtype=np.float32), timing=True)
    try:
        for l in range(L):
            for b in range(B):
                K, V = syn.layer_seq_kv(l, b, Hkv, 0, N, d)
                lib.append_kv(l, b, K, V, src_is_device=False)
        qs = syn.query_stream(L, B, Hq, d, 0.6, 0.98)
        want = []
        for step in range(6):
            q = torch.from_numpy(qs.next().view(np.int16)).cuda()
            out = torch.empty((L, B, Hq, d), dtype=torch.float32, device="cuda")
            if step % 2:
                for l in range(L):
                    lib.decode_layer(l, q[l], out[l])
            else:
                lib.decode_step(q, out)
            st = lib.stats()
            want.append((st["last_host_bytes"], st["last_hbm_bytes_alg"]))
        got = lib.step_bytes(1, 6)
        assert got.tolist() == [list(w) for w in want[1:]]
        assert any(h > 0 for h, _ in want) and all(m > 0 for _, m in want)
    finally:
        lib.close()
