"""One small decode step of the CLO hot path on cuda:0, checked against the CPU
oracle (used by the package smoke entry point)."""
from __future__ import annotations

import numpy as np


def run_smoke() -> None:
    import torch

    import oracle as orc  # test infrastructure: only the smoke check and tests use it
    from host_offloaded_kv_gb300.clo import CLOContext
    from host_offloaded_kv_gb300.synth import Synth

    assert torch.cuda.is_available(), "smoke needs a GPU"
    L, B, Hq, Hkv, d, N, k = 1, 1, 8, 2, 64, 4096, 410
    syn = Synth(0)
    R = syn.hash_matrices(L, Hkv, d)
    tau = np.full(L * Hkv, 0.8, dtype=np.float32)
    lib = CLOContext(n_layers=L, batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, max_tokens=N, hash_R=R,
                     topk=k, tau=tau)
    ref = orc.OracleCLO(L, B, Hq, Hkv, d, R, topk=k, tau=tau, ntok=[N])
    K, V = syn.layer_seq_kv(0, 0, Hkv, 0, N, d)
    lib.append_kv(0, 0, K, V, src_is_device=False)
    for h in range(Hkv):
        ref.set_unit_kv(0, 0, h, np.ascontiguousarray(K[:, h]), np.ascontiguousarray(V[:, h]))
    qs = syn.query_stream(L, B, Hq, d, 0.6, 0.98)
    for _ in range(2):
        q = qs.next()
        qd = torch.from_numpy(q.view(np.int16)).cuda()
        out = torch.empty((L, B, Hq, d), dtype=torch.float32, device="cuda")
        lib.decode_step(qd, out)
        lib.sync()
        dec = lib.decisions()
        res = ref.step(q, device_decision=dec)
        o = out.cpu().numpy()
        for h in range(Hkv):
            assert np.array_equal(lib.idx(0, 0, h), res.idx[(0, 0, h)]), "selection differs from the oracle"
            err = np.abs(o[0, 0, h * 4:(h + 1) * 4] - res.out[(0, 0, h)]).max()
            assert err <= 2e-3, f"attention output differs from the oracle by {err}"
    lib.close()
    print("smoke ok")
