"""Lock-step harness: the CUDA library and the CPU oracle on the same seeded inputs.

Both sides take their inputs from the seeded generator (``synth``); the oracle
never sees anything computed by the library except the reuse decisions of units
whose cosine lies within 1e-4 of their threshold (and an ambiguous persistent
choice), which it adopts so the two stay in lock-step.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import oracle as orc
from host_offloaded_kv_gb300.clo import CLOContext
from host_offloaded_kv_gb300.synth import Synth, bf16_to_float

ATOL = 2e-3      # max abs error of attention outputs
RTOL_L2 = 1e-3   # relative L2 error of attention outputs


@dataclass
class Spec:
    L: int
    B: int
    Hq: int
    Hkv: int
    d: int
    ntok: list            # tokens per sequence
    seed: int = 0
    topk: int = 0
    topk_ratio: float = 0.1
    tau: float | None = 0.8   # fixed tau for all heads, or None -> warm-up
    persist_mask: np.ndarray | None = None
    warmup_steps: int = 16
    tau_offset: float = 0.05
    n_persist: int = 0
    rho: tuple = (0.6, 0.98)
    hh_ratio: float = 0.01
    max_tokens: int | None = None
    sample: list | None = None   # units (l, b, h) given to the oracle; None = all
    kv_override: dict = field(default_factory=dict)  # (l, b) -> (K, V) replacing generated data
    adaptive_tau: bool = False
    tau_ema: float = 0.0625
    kv_bits: int = 16


class LockStep:
    def __init__(self, spec: Spec, torch_device="cuda"):
        import torch

        self.torch = torch
        self.spec = s = spec
        self.G = s.Hq // s.Hkv
        self.syn = Synth(s.seed, s.hh_ratio)
        self.R = self.syn.hash_matrices(s.L, s.Hkv, s.d)
        LH = s.L * s.Hkv
        tau = None if s.tau is None else np.full(LH, s.tau, dtype=np.float32)
        maxtok = s.max_tokens or max(s.ntok)
        self.lib = CLOContext(n_layers=s.L, batch=s.B, n_q_heads=s.Hq, n_kv_heads=s.Hkv, head_dim=s.d,
                              max_tokens=maxtok, hash_R=self.R, topk=s.topk, topk_ratio=s.topk_ratio, tau=tau,
                              persist_mask=s.persist_mask, warmup_steps=s.warmup_steps, tau_offset=s.tau_offset,
                              n_persist=s.n_persist, adaptive_tau=s.adaptive_tau, tau_ema=s.tau_ema,
                              kv_bits=s.kv_bits)
        self.orc = orc.OracleCLO(s.L, s.B, s.Hq, s.Hkv, s.d, self.R, topk=s.topk, topk_ratio=s.topk_ratio,
                                 tau=tau, persist_mask=s.persist_mask, warmup_steps=s.warmup_steps,
                                 tau_offset=s.tau_offset, n_persist=s.n_persist, ntok=s.ntok,
                                 adaptive_tau=s.adaptive_tau, tau_ema=s.tau_ema, kv_bits=s.kv_bits)
        units = s.sample if s.sample is not None else [
            (l, b, h) for l in range(s.L) for b in range(s.B) for h in range(s.Hkv)]
        self.units = list(units)
        self.kv = {}
        want = set(self.units)
        for l in range(s.L):
            for b in range(s.B):
                if (l, b) in s.kv_override:
                    K, V = s.kv_override[(l, b)]
                else:
                    K, V = self.syn.layer_seq_kv(l, b, s.Hkv, 0, s.ntok[b], s.d)
                self.lib.append_kv(l, b, K, V, src_is_device=False)
                for h in range(s.Hkv):
                    if (l, b, h) in want:
                        Kh, Vh = np.ascontiguousarray(K[:, h, :]), np.ascontiguousarray(V[:, h, :])
                        self.kv[(l, b, h)] = (Kh, Vh)
                        self.orc.set_unit_kv(l, b, h, Kh, Vh)
        self.qs = self.syn.query_stream(s.L, s.B, s.Hq, s.d, *s.rho)
        self.prev_idx = {}
        self.t = 0
        self.log = []

    # ------------------------------------------------------------------------------
    def check_key_codes(self):
        for u in self.units:
            got = self.lib.key_codes(*u)
            want = self.orc.kcodes[u]
            assert np.array_equal(got, want), f"key codes differ for unit {u}"

    def append_step(self, src_is_device=True):
        """One new token for every (layer, sequence), from the seeded generator at each
        sequence's current length; the library appends it on the device, the oracle on
        its own copy."""
        s = self.spec
        Knew = np.empty((s.L, s.B, s.Hkv, s.d), dtype=np.uint16)
        Vnew = np.empty_like(Knew)
        for l in range(s.L):
            for b in range(s.B):
                K, V = self.syn.layer_seq_kv(l, b, s.Hkv, int(self.orc.ntok[b]), 1, s.d)
                Knew[l, b], Vnew[l, b] = K[0], V[0]
        if src_is_device:
            kd = self.torch.from_numpy(Knew.view(np.int16)).cuda()
            vd = self.torch.from_numpy(Vnew.view(np.int16)).cuda()
            self.lib.append_step(kd, vd)
            self.lib.sync()
        else:
            self.lib.append_step(Knew, Vnew, src_is_device=False)
        self.orc.append_tokens(Knew, Vnew)
        for l in range(s.L):
            for b in range(s.B):
                for h in range(s.Hkv):
                    if (l, b, h) in self.kv:
                        Kh, Vh = self.kv[(l, b, h)]
                        self.kv[(l, b, h)] = (np.concatenate([Kh, Knew[l, b, h][None]]),
                                              np.concatenate([Vh, Vnew[l, b, h][None]]))

    def step(self, q=None, check=True, io_on_device=True, per_layer=False):
        """One decode step through clo_decode_step, or (per_layer) through one
        clo_decode_layer call per layer; the oracle takes the whole step."""
        torch = self.torch
        s = self.spec
        if q is None:
            q = self.qs.next()
        if io_on_device:
            qd = torch.from_numpy(q.view(np.int16)).cuda()
            outd = torch.empty((s.L, s.B, s.Hq, s.d), dtype=torch.float32, device="cuda")
            if per_layer:
                for l in range(s.L):
                    self.lib.decode_layer(l, qd[l], outd[l])
            else:
                self.lib.decode_step(qd, outd)
            self.lib.sync()
            out = outd.cpu().numpy()
        else:
            out = np.empty((s.L, s.B, s.Hq, s.d), dtype=np.float32)
            if per_layer:
                for l in range(s.L):
                    self.lib.decode_layer(l, np.ascontiguousarray(q[l]), out[l], io_on_device=False)
            else:
                self.lib.decode_step(q, out, io_on_device=False)
        dec = self.lib.decisions()
        stats = self.lib.stats()
        dev_persist = self.lib.persist()
        res = self.orc.step(q, device_decision=dec, device_persist=dev_persist)
        self.t += 1
        rec = {"step": res.step, "excused": int(res.excused.sum()), "hit": int((res.decision == 0).sum()),
               "miss": int((res.decision == 1).sum()), "persist": int((res.decision == 2).sum())}
        self.log.append(rec)
        if not check:
            return res, out, dec, stats
        assert np.array_equal(dec.astype(np.int8), res.decision), (
            f"step {res.step}: decisions differ at {np.argwhere(dec.astype(np.int8) != res.decision)[:5]}")
        assert stats["last_host_bytes"] == res.host_bytes, (stats["last_host_bytes"], res.host_bytes)
        if s.adaptive_tau and self.orc.tau is not None:   # thresholds after this step's update
            np.testing.assert_allclose(self.lib.tau(), self.orc.tau, atol=1e-5, rtol=0)
        G, d = self.G, s.d
        qr = q.reshape(s.L, s.B, s.Hkv, G, d)
        for u in self.units:
            l, b, h = u
            du = int(res.decision[u])
            idx_lib = self.lib.idx(*u)
            assert np.array_equal(idx_lib, res.idx[u]), f"step {res.step} unit {u}: selection differs"
            if du != orc.DEC_HIT:
                qc_lib = self.lib.query_codes(*u)
                qc_orc = orc.hash_codes(qr[l, b, h], self.R[l, h])
                assert np.array_equal(qc_lib, qc_orc), f"step {res.step} unit {u}: query codes differ"
            else:
                assert np.array_equal(idx_lib, self.prev_idx[u]), f"unit {u}: hit changed the selection"
            if du == orc.DEC_MISS:
                K, V = self.orc.kv[u]   # the rows as the pool stores them (dequantised if quantised)
                rows = self.lib.slot_rows(*u)
                assert np.array_equal(rows[:, 0, :], K[res.idx[u]]), f"unit {u}: gathered K rows differ"
                assert np.array_equal(rows[:, 1, :], V[res.idx[u]]), f"unit {u}: gathered V rows differ"
            self.prev_idx[u] = idx_lib
            got = out[l, b, h * G:(h + 1) * G].astype(np.float64)
            want = res.out[u]
            err = np.abs(got - want).max()
            rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
            assert err <= ATOL and rel <= RTOL_L2, f"step {res.step} unit {u}: max abs {err:.3g}, rel L2 {rel:.3g}"
        return res, out, dec, stats

    def close(self):
        self.lib.close()
