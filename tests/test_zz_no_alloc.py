"""The allocation-free attention entry point, checked against the decode step and
against the CPU oracle's fp64 attention.

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
        # sizes beyond the fixed scratch are refused with a clear error by the library
        # itself (raw addresses skip the wrapper's own size checks; nothing is launched)
        with pytest.raises(CLOError) as e:
            clo_sparse_attention_noalloc(qg.data_ptr(), rows_d.data_ptr(), out.data_ptr(), 5000, G, d, k, None)
        assert e.value.status == CLO_ERR_INVALID and "scratch" in str(e.value)
        with pytest.raises(CLOError) as e:
            clo_sparse_attention_noalloc(qg.data_ptr(), rows_d.data_ptr(), out.data_ptr(), 4096, 8, 128, 1 << 20,
                                         None)
        assert e.value.status == CLO_ERR_INVALID
        # the wrapper refuses tensors smaller than the sizes it is given
        with pytest.raises(ValueError):
            clo_sparse_attention_noalloc(qg, rows_d, out, 5000, G, d, k, None)
    finally:
        lib.close()


@pytest.mark.parametrize("d,G,k", [(64, 4, 300), (64, 8, 100), (128, 8, 1000), (128, 1, 1)])
def test_noalloc_attention_matches_the_oracle_on_two_calls(d, G, k):
    # head_dim 64 (two row groups per CTA), the largest group of 8, a single split (k < 256)
    # and a single row; every group's output against fp64 softmax attention over its rows,
    # on two calls in a row with different rows (the second reuses the scratch)
    import oracle as orc
    from host_offloaded_kv_gb300.clo import clo_sparse_attention_noalloc
    from host_offloaded_kv_gb300.synth import Synth

    n = 7
    syn = Synth(90 + d + G + k)
    for call in range(2):
        q = syn.normal_bf16(2 * call, n * G * d).reshape(n, G, d)
        rows = syn.normal_bf16(2 * call + 1, n * k * 2 * d).reshape(n, k, 2, d)
        qd = torch.from_numpy(q.view(np.int16)).cuda()
        rd = torch.from_numpy(rows.view(np.int16)).cuda()
        out = torch.full((n, G, d), float("nan"), dtype=torch.float32, device="cuda")
        clo_sparse_attention_noalloc(qd, rd, out, n, G, d, k, None)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        for g in range(n):
            want = orc.attention(q[g], rows[g, :, 0, :], rows[g, :, 1, :])
            err = np.abs(got[g] - want).max()
            rel = np.linalg.norm(got[g] - want) / np.linalg.norm(want)
            assert err <= ATOL and rel <= RTOL_L2, f"call {call} group {g}: max abs {err:.3g}, rel {rel:.3g}"
