"""The allocation-free attention entry point, checked against the decode step.

clo_sparse_attention_noalloc is for callers that may not allocate device memory:
serving engines or plugin hosts that plan all device memory up front and give a
kernel only its inputs and outputs, and latency-critical loops that cannot take
the stalls an allocation can cause.  It keeps its scratch in a fixed device
array inside the library.  Here it is given the rows the library's decode step
selected and fetched, and must reproduce that step's attention outputs, on two
calls in a row (the second call reuses the scratch the first one left behind).
This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ATOL, RTOL_L2 = 2e-3, 1e-3


def test_noalloc_attention_matches_decode_step_on_two_calls():
    from host_offloaded_kv_gb300.clo import CLO_ERR_INVALID, CLOContext, CLOError, clo_sparse_attention_noalloc
    from host_offloaded_kv_gb300.synth import Synth

    L, B, Hq, Hkv, d, N = 2, 2, 8, 2, 128, 3000
    G = Hq // Hkv
    U = L * B * Hkv
    syn = Synth(21)
    R = syn.hash_matrices(L, Hkv, d)
    # tau = 2: every unit misses, so each step's cache slots hold exactly the rows it attended to
    lib = CLOContext(n_layers=L, batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, max_tokens=N, hash_R=R,
                     tau=np.full(L * Hkv, 2.0, dtype=np.float32))
    try:
        for l in range(L):
            for b in range(B):
                K, V = syn.layer_seq_kv(l, b, Hkv, 0, N, d)
                lib.append_kv(l, b, K, V, src_is_device=False)
        qs = syn.query_stream(L, B, Hq, d, 0.6, 0.98)
        k = lib.k_of(0)
        for call in range(2):
            q = qs.next()
            qd = torch.from_numpy(q.view(np.int16)).cuda()
            ref = torch.empty((L, B, Hq, d), dtype=torch.float32, device="cuda")
            lib.decode_step(qd, ref)
            lib.sync()
            rows = np.stack([lib.slot_rows(l, b, h) for l in range(L) for b in range(B) for h in range(Hkv)])
            rows_d = torch.from_numpy(rows.view(np.int16)).cuda()
            qg = qd.view(U, G, d).contiguous()
            out = torch.full((U, G, d), float("nan"), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            clo_sparse_attention_noalloc(qg, rows_d, out, U, G, d, k, None)
            torch.cuda.synchronize()
            want = ref.cpu().numpy().reshape(U, G, d).astype(np.float64)
            got = out.cpu().numpy().astype(np.float64)
            for u in range(U):
                err = np.abs(got[u] - want[u]).max()
                rel = np.linalg.norm(got[u] - want[u]) / np.linalg.norm(want[u])
                assert err <= ATOL and rel <= RTOL_L2, f"call {call} group {u}: max abs {err:.3g}, rel {rel:.3g}"
        # sizes beyond the fixed scratch are refused with a clear error
        with pytest.raises(CLOError) as e:
            clo_sparse_attention_noalloc(qg, rows_d, out, 5000, G, d, k, None)
        assert e.value.status == CLO_ERR_INVALID and "scratch" in str(e.value)
        with pytest.raises(CLOError) as e:
            clo_sparse_attention_noalloc(qg, rows_d, out, 4096, 8, 128, 1 << 20, None)
        assert e.value.status == CLO_ERR_INVALID
    finally:
        lib.close()
