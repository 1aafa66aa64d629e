"""CPU oracle of the CLO decode step -- TEST INFRASTRUCTURE ONLY.

Plain restatement of the decode step of CLO, the CPU-light KV-cache offloading
system, on the CPU, in fp64, one unit (layer, sequence, kv head) at a time.
The arithmetic primitives (hash sign, cosine, scores, top-k sort, softmax
attention) are in ``clo_oracle.c``; this file holds the per-step state machine.

Sources (page title, section):
  [SYN] "CLO (2511.14510) - L3 Per-Paper Synthesis"
  [KVO] "KV Cache Offloading 完全拆解" (KV-cache offloading survey blog)
  [ABS] CLO abstract (arXiv 2511.14510v1, paper-check page)

Per decode step t and unit (l, b, h), with G = Hq / Hkv query heads per group:
  1. reuse test ([SYN] 2.1 item 2, [ABS] feature (1)): cosine of the group's
     concatenated query with the query cached at the unit's last refresh;
     hit iff cos >= tau[l, h].  The first step, and every warm-up step, misses.
  2. persistent heads ([ABS] feature (2), [SYN] 3.3 attack 6): always reselect,
     read rows from their GPU-resident copy, fetch no host bytes.
  3. miss / persistent: hash-code scores of all N cached tokens, top-k with
     k = ceil(ratio * N) ([SYN] 2.2: top-k = 10 %), ties to the lowest index,
     selection kept in ascending index order.
  4. miss (non-persistent): the selected K/V rows are fetched from host memory
     ([ABS] features (2)-(3)): 4*d bytes per row.
  5. sparse softmax attention over the selected rows (fp64).
Warm-up (when no thresholds are given): the first W steps all miss and collect
cos(q_t, q_{t-1}); s_hat[l, h] is its mean over the batch and the W-1 adjacent
pairs, tau = s_hat - offset, and the n_persist heads with the lowest s_hat in each
layer become persistent ([SYN] 3.3 attack 6: s_hat_i, D_i, N_persist from
profiling; D_i read as 1 - s_hat_i).
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle_clo.so")

DEC_HIT, DEC_MISS, DEC_PERSIST = 0, 1, 2
EXCUSE_BAND = 1e-4  # decisions with |cos - tau| below this may follow the device's

_lib = None
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def load_oracle():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} missing: run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    lib.orc_bf16.restype = ctypes.c_double
    lib.orc_bf16.argtypes = [ctypes.c_uint16]
    lib.orc_kv_bytes_per_token.restype = _i64
    lib.orc_kv_bytes_per_token.argtypes = [_i64, _i64, _i64, _i64]
    lib.orc_exact_sign.restype = _int
    lib.orc_exact_sign.argtypes = [_p, _int]
    lib.orc_hash_codes.restype = None
    lib.orc_hash_codes.argtypes = [_p, _i64, _int, _p, _p]
    lib.orc_cosine.restype = ctypes.c_double
    lib.orc_cosine.argtypes = [_p, _p, _i64]
    lib.orc_scores.restype = None
    lib.orc_scores.argtypes = [_p, _int, _p, _i64, _p]
    lib.orc_topk.restype = _int
    lib.orc_topk.argtypes = [_p, _i64, _i64, _p]
    lib.orc_attention.restype = None
    lib.orc_attention.argtypes = [_p, _int, _int, _p, _p, _i64, _p]
    lib.orc_num_threads.restype = _int
    lib.orc_num_threads.argtypes = []
    lib.orc_kv_roundtrip.restype = None
    lib.orc_kv_roundtrip.argtypes = [_p, _i64, _int, _p]
    lib.orc_kv_record_bytes.restype = _i64
    lib.orc_kv_record_bytes.argtypes = [_i64, _int]
    _lib = lib
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- primitives
def kv_bytes_per_token(n_kv: int, d_head: int, elem_bytes: int, n_layers: int) -> int:
    """2 * n_kv * d_head * bytes * L  ([KVO] "KV Cache 到底有多大")."""
    return int(load_oracle().orc_kv_bytes_per_token(n_kv, d_head, elem_bytes, n_layers))


def exact_sign(p) -> int:
    p = _c(p, np.float64)
    return int(load_oracle().orc_exact_sign(p.ctypes.data, p.size))


def hash_codes(X: np.ndarray, R: np.ndarray) -> np.ndarray:
    """X bf16 [n][d], R bf16 [d][128] -> uint64 [n][2] sign codes."""
    X = _c(X, np.uint16)
    R = _c(R, np.uint16)
    n, d = X.shape
    assert R.shape == (d, 128)
    out = np.zeros((n, 2), dtype=np.uint64)
    load_oracle().orc_hash_codes(X.ctypes.data, n, d, R.ctypes.data, out.ctypes.data)
    return out


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a = _c(a, np.uint16).reshape(-1)
    b = _c(b, np.uint16).reshape(-1)
    assert a.size == b.size
    return float(load_oracle().orc_cosine(a.ctypes.data, b.ctypes.data, a.size))


def kv_roundtrip(x: np.ndarray, bits: int) -> np.ndarray:
    """bf16 values (last axis a multiple of 64) -> their values after the host pool's
    b-bit quantisation and the GPU's dequantisation (identity for bits 16)."""
    x = _c(x, np.uint16)
    if bits >= 16:
        return x.copy()
    assert x.shape[-1] % 64 == 0
    y = np.empty_like(x)
    load_oracle().orc_kv_roundtrip(x.ctypes.data, x.size, int(bits), y.ctypes.data)
    return y


def kv_record_bytes(d: int, bits: int) -> int:
    """Host-pool bytes of one token's K|V record of one kv head."""
    return int(load_oracle().orc_kv_record_bytes(int(d), int(bits)))


def scores(qcodes: np.ndarray, kcodes: np.ndarray) -> np.ndarray:
    """qcodes uint64 [G][2], kcodes uint64 [N][2] -> int32 [N]."""
    qcodes = _c(qcodes, np.uint64)
    kcodes = _c(kcodes, np.uint64)
    N = kcodes.shape[0]
    out = np.empty(N, dtype=np.int32)
    load_oracle().orc_scores(qcodes.ctypes.data, qcodes.shape[0], kcodes.ctypes.data, N, out.ctypes.data)
    return out


def topk(sc: np.ndarray, k: int) -> np.ndarray:
    sc = _c(sc, np.int32)
    idx = np.empty(k, dtype=np.int32)
    rc = load_oracle().orc_topk(sc.ctypes.data, sc.size, k, idx.ctypes.data)
    if rc != 0:
        raise ValueError(f"orc_topk failed ({rc}) for N={sc.size}, k={k}")
    return idx


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """q bf16 [G][d], K/V bf16 [k][d] -> float64 [G][d]."""
    q = _c(q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    G, d = q.shape
    k = K.shape[0]
    out = np.empty((G, d), dtype=np.float64)
    load_oracle().orc_attention(q.ctypes.data, G, d, K.ctypes.data, V.ctypes.data, k, out.ctypes.data)
    return out


def topk_count(N: int, topk_fixed: int, ratio: float) -> int:
    """k for a context of N tokens: the fixed k (clamped to N) or ceil(ratio * N)
    evaluated as one IEEE double product, clamped to [1, N]."""
    if N <= 0:
        return 0
    if topk_fixed > 0:
        return min(int(topk_fixed), N)
    k = int(math.ceil(float(ratio) * float(N)))
    return max(1, min(k, N))


# --------------------------------------------------------------------------- state machine
@dataclass
class StepResult:
    step: int
    decision: np.ndarray                 # int8 [L][B][Hkv]
    cos: np.ndarray                      # float64 [L][B][Hkv] (nan where not evaluated)
    excused: np.ndarray                  # bool [L][B][Hkv]: decision taken from the device
    host_bytes: int                      # bytes fetched from host this step
    out: dict = field(default_factory=dict)   # (l,b,h) -> float64 [G][d]
    idx: dict = field(default_factory=dict)   # (l,b,h) -> int32 [k]  (selection used this step)


class OracleCLO:
    """Decode-step oracle.  Units whose K/V were given with ``set_unit_kv`` get
    selections and attention outputs; decisions and host-byte counts cover all
    units (they need only the queries)."""

    def __init__(self, L, B, Hq, Hkv, d, R, *, topk=0, topk_ratio=0.1, tau=None, persist_mask=None,
                 warmup_steps=16, tau_offset=0.05, n_persist=0, ntok=None, adaptive_tau=False, tau_ema=0.0625,
                 kv_bits=16):
        load_oracle()
        assert Hq % Hkv == 0
        self.L, self.B, self.Hq, self.Hkv, self.d = L, B, Hq, Hkv, d
        self.G = Hq // Hkv
        self.R = _c(R, np.uint16).reshape(L, Hkv, d, 128)
        self.topk_fixed, self.ratio = int(topk), float(topk_ratio)
        self.kv_bits = int(kv_bits)
        self.record_bytes = kv_record_bytes(d, self.kv_bits)
        self.ntok = np.zeros(B, dtype=np.int64) if ntok is None else np.asarray(ntok, dtype=np.int64).copy()
        self.kv = {}
        self.kcodes = {}
        self.qcache = np.zeros((L, B, Hkv, self.G * d), dtype=np.uint16)
        self.qvalid = np.zeros((L, B, Hkv), dtype=bool)
        self.sel = {}
        self.t = 0
        self.warmup = tau is None
        self.W = int(warmup_steps)
        self.tau_offset = float(tau_offset)
        self.n_persist = int(n_persist)
        if self.warmup:
            if self.W < 2:
                raise ValueError("warm-up needs at least 2 steps")
            self.tau = None
            self.persist = np.zeros((L, Hkv), dtype=bool)
        else:
            self.tau = np.asarray(tau, dtype=np.float64).reshape(L, Hkv).copy()
            self.persist = (np.zeros((L, Hkv), dtype=bool) if persist_mask is None
                            else np.asarray(persist_mask, dtype=bool).reshape(L, Hkv).copy())
        self.shat_sum = np.zeros((L, Hkv), dtype=np.float64)
        self.shat = None
        self.persist_ambiguous = False
        # online adaptive thresholds ("CLO (2511.14510) - L3 Per-Paper Synthesis",
        # section 5.3): s_hat follows the live adjacent-step cosines after warm-up
        self.adaptive = bool(adaptive_tau)
        self.ema = float(tau_ema)
        self.qprev = np.zeros((L, B, Hkv, self.G * d), dtype=np.uint16)
        self.qprev_valid = np.zeros((L, B, Hkv), dtype=bool)
        if self.adaptive and not self.warmup:
            self.shat = self.tau + self.tau_offset

    # context -------------------------------------------------------------------
    def set_unit_kv(self, l, b, h, K, V):
        K = _c(K, np.uint16)
        V = _c(V, np.uint16)
        assert K.shape == V.shape and K.shape[1] == self.d
        # codes from the keys as given; attention sees the rows as stored in the pool
        self.kcodes[(l, b, h)] = hash_codes(K, self.R[l, h])
        self.kv[(l, b, h)] = (kv_roundtrip(K, self.kv_bits), kv_roundtrip(V, self.kv_bits))
        self.ntok[b] = K.shape[0]

    def append_tokens(self, Knew, Vnew):
        """Streaming growth ("CLO (2511.14510) - L3 Per-Paper Synthesis", section 5.7:
        incremental offloading): one new token per (layer, sequence), bf16
        [L][B][Hkv][d]; its key code joins the unit's codes and every length grows by 1."""
        Knew = _c(Knew, np.uint16).reshape(self.L, self.B, self.Hkv, self.d)
        Vnew = _c(Vnew, np.uint16).reshape(self.L, self.B, self.Hkv, self.d)
        for (l, b, h), (K, V) in list(self.kv.items()):
            kr, vr = Knew[l, b, h][None, :], Vnew[l, b, h][None, :]
            self.kcodes[(l, b, h)] = np.concatenate([self.kcodes[(l, b, h)], hash_codes(kr, self.R[l, h])])
            self.kv[(l, b, h)] = (np.concatenate([K, kv_roundtrip(kr, self.kv_bits)]),
                                  np.concatenate([V, kv_roundtrip(vr, self.kv_bits)]))
        self.ntok += 1

    def k_of(self, b: int) -> int:
        return topk_count(int(self.ntok[b]), self.topk_fixed, self.ratio)

    # one step --------------------------------------------------------------------
    def step(self, q: np.ndarray, device_decision=None, device_persist=None) -> StepResult:
        """q: bf16 [L][B][Hq][d].  device_decision (int [L][B][Hkv]) is consulted only
        for units whose cosine lies within EXCUSE_BAND of tau; device_persist only when
        the oracle's own persistent choice is ambiguous within EXCUSE_BAND."""
        L, B, Hkv, G, d = self.L, self.B, self.Hkv, self.G, self.d
        q = _c(q, np.uint16).reshape(L, B, Hkv, G * d)
        dec = np.zeros((L, B, Hkv), dtype=np.int8)
        cosv = np.full((L, B, Hkv), np.nan)
        excused = np.zeros((L, B, Hkv), dtype=bool)
        in_warmup = self.warmup and self.t < self.W
        for l in range(L):
            for b in range(B):
                for h in range(Hkv):
                    if self.qvalid[l, b, h]:
                        cosv[l, b, h] = cosine(q[l, b, h], self.qcache[l, b, h])
                    if in_warmup:
                        dec[l, b, h] = DEC_MISS
                        if self.t >= 1:
                            self.shat_sum[l, h] += cosv[l, b, h]
                    elif self.persist[l, h]:
                        dec[l, b, h] = DEC_PERSIST
                    elif not self.qvalid[l, b, h]:
                        dec[l, b, h] = DEC_MISS
                    else:
                        c, tau = cosv[l, b, h], self.tau[l, h]
                        dec[l, b, h] = DEC_HIT if c >= tau else DEC_MISS
                        if device_decision is not None and abs(c - tau) < EXCUSE_BAND:
                            dd = int(np.asarray(device_decision)[l, b, h])
                            if dd in (DEC_HIT, DEC_MISS):
                                dec[l, b, h] = dd
                                excused[l, b, h] = True
                    if dec[l, b, h] == DEC_MISS:
                        self.qcache[l, b, h] = q[l, b, h]
                        self.qvalid[l, b, h] = True
        res = StepResult(self.t, dec, cosv, excused, 0)
        host = 0
        for l in range(L):
            for b in range(B):
                for h in range(Hkv):
                    if dec[l, b, h] == DEC_MISS:
                        host += self.k_of(b) * self.record_bytes
        res.host_bytes = host
        qr = q.reshape(L, B, Hkv, G, d)
        for (l, b, h), (K, V) in self.kv.items():
            u = (l, b, h)
            if dec[u] != DEC_HIT:
                qc = hash_codes(qr[l, b, h], self.R[l, h])
                sc = scores(qc, self.kcodes[u])
                self.sel[u] = topk(sc, self.k_of(b))
            idx = self.sel[u]
            res.idx[u] = idx
            res.out[u] = attention(qr[l, b, h], K[idx], V[idx])
        if self.adaptive:
            if not in_warmup:
                self._adapt_tau(q)
            self.qprev[...] = q
            self.qprev_valid[...] = True
        if in_warmup and self.t == self.W - 1:
            self._finish_warmup(device_persist)
        self.t += 1
        return res

    def _adapt_tau(self, q):
        """s_hat[l, h] <- (1 - a) s_hat + a * mean_b cos(q_t, q_{t-1}), tau = s_hat - offset;
        the new tau applies from the next step."""
        for l in range(self.L):
            for h in range(self.Hkv):
                vals = [cosine(q[l, b, h], self.qprev[l, b, h]) for b in range(self.B) if self.qprev_valid[l, b, h]]
                if vals:
                    m = sum(vals) / len(vals)
                    self.shat[l, h] = (1.0 - self.ema) * self.shat[l, h] + self.ema * m
                    self.tau[l, h] = self.shat[l, h] - self.tau_offset

    def _finish_warmup(self, device_persist=None):
        npairs = self.B * (self.W - 1)
        self.shat = self.shat_sum / npairs
        self.tau = self.shat - self.tau_offset
        P = self.n_persist
        persist = np.zeros((self.L, self.Hkv), dtype=bool)
        self.persist_ambiguous = False
        for l in range(self.L):
            order = sorted(range(self.Hkv), key=lambda h: (self.shat[l, h], h))
            chosen = order[:P]
            persist[l, chosen] = True
            if 0 < P < self.Hkv:
                gap = self.shat[l, order[P]] - self.shat[l, order[P - 1]]
                if gap < EXCUSE_BAND:
                    self.persist_ambiguous = True
        if self.persist_ambiguous and device_persist is not None:
            dp = np.asarray(device_persist, dtype=bool).reshape(self.L, self.Hkv)
            ok = True
            for l in range(self.L):
                if dp[l].sum() != P:
                    ok = False
                    break
                if P and (self.shat[l, dp[l]].max() > self.shat[l, ~dp[l]].min() + EXCUSE_BAND):
                    ok = False
                    break
            if ok:
                persist = dp.copy()
        self.persist = persist
