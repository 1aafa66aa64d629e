"""ctypes wrapper around the seeded input generator (``libclo_synth.so``)."""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libclo_synth.so")

_u64 = ctypes.c_uint64
_i64 = ctypes.c_int64
_int = ctypes.c_int
_dbl = ctypes.c_double
_p = ctypes.c_void_p

_lib = None


def load_synth():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')"
        )
    lib = ctypes.CDLL(LIB_PATH)
    lib.synth_u64.restype = _u64
    lib.synth_u64.argtypes = [_u64, _u64, _u64]
    lib.synth_normal.restype = _dbl
    lib.synth_normal.argtypes = [_u64, _u64, _u64]
    lib.synth_bf16_from_double.restype = ctypes.c_uint16
    lib.synth_bf16_from_double.argtypes = [_dbl]
    lib.synth_bf16_to_double.restype = _dbl
    lib.synth_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.synth_head_direction.restype = None
    lib.synth_head_direction.argtypes = [_u64, _int, _int, _int, _p]
    lib.synth_is_heavy.restype = _int
    lib.synth_is_heavy.argtypes = [_u64, _int, _int, _int, _i64, _dbl]
    lib.synth_unit_kv.restype = None
    lib.synth_unit_kv.argtypes = [_u64, _int, _int, _int, _i64, _i64, _int, _dbl, _p, _p, _i64]
    lib.synth_layer_seq_kv.restype = None
    lib.synth_layer_seq_kv.argtypes = [_u64, _int, _int, _int, _i64, _i64, _int, _dbl, _p, _p]
    lib.synth_hash_matrix.restype = None
    lib.synth_hash_matrix.argtypes = [_u64, _int, _int, _int, _p]
    lib.synth_query_rho.restype = None
    lib.synth_query_rho.argtypes = [_u64, _int, _int, _int, _dbl, _dbl, _p]
    lib.synth_query_step.restype = None
    lib.synth_query_step.argtypes = [_u64, _int, _int, _int, _int, _i64, _p, _p, _p]
    lib.synth_normal_bf16.restype = None
    lib.synth_normal_bf16.argtypes = [_u64, _u64, _i64, _p]
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def bf16_to_float(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def float_to_bf16(x) -> np.ndarray:
    """float64/float32 -> bf16 bit patterns, one round-to-nearest-even from the input value."""
    lib = load_synth()
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in = x.reshape(-1)
    flat_out = out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.synth_bf16_from_double(float(flat_in[i]))
    return out


class Synth:
    """Generator bound to one workload seed."""

    def __init__(self, seed: int, hh_ratio: float = 0.01):
        self.lib = load_synth()
        self.seed = int(seed)
        self.hh_ratio = float(hh_ratio)

    # keys / values ---------------------------------------------------------
    def unit_kv(self, l: int, b: int, h: int, t0: int, n: int, d: int):
        """K, V of one (layer, seq, kv head) for tokens [t0, t0+n): uint16 [n][d] each."""
        K = np.empty((n, d), dtype=np.uint16)
        V = np.empty((n, d), dtype=np.uint16)
        self.lib.synth_unit_kv(self.seed, l, b, h, t0, n, d, self.hh_ratio, _ptr(K), _ptr(V), d)
        return K, V

    def layer_seq_kv(self, l: int, b: int, Hkv: int, t0: int, n: int, d: int, K=None, V=None):
        """K, V of all kv heads of (layer, seq): uint16 [n][Hkv][d] each (append layout)."""
        if K is None:
            K = np.empty((n, Hkv, d), dtype=np.uint16)
        if V is None:
            V = np.empty((n, Hkv, d), dtype=np.uint16)
        self.lib.synth_layer_seq_kv(self.seed, l, b, Hkv, t0, n, d, self.hh_ratio, _ptr(K), _ptr(V))
        return K, V

    def is_heavy(self, l: int, b: int, h: int, t: int) -> bool:
        return bool(self.lib.synth_is_heavy(self.seed, l, b, h, t, self.hh_ratio))

    def head_direction(self, l: int, h: int, d: int) -> np.ndarray:
        u = np.empty(d, dtype=np.float64)
        self.lib.synth_head_direction(self.seed, l, h, d, _ptr(u))
        return u

    # hash projection -------------------------------------------------------
    def hash_matrix(self, l: int, h: int, d: int) -> np.ndarray:
        R = np.empty((d, 128), dtype=np.uint16)
        self.lib.synth_hash_matrix(self.seed, l, h, d, _ptr(R))
        return R

    def hash_matrices(self, L: int, Hkv: int, d: int) -> np.ndarray:
        R = np.empty((L, Hkv, d, 128), dtype=np.uint16)
        for l in range(L):
            for h in range(Hkv):
                self.lib.synth_hash_matrix(self.seed, l, h, d, _ptr(R[l, h]))
        return R

    # queries -----------------------------------------------------------------
    def query_stream(self, L: int, B: int, Hq: int, d: int, rho_lo: float, rho_hi: float):
        return QueryStream(self, L, B, Hq, d, rho_lo, rho_hi)

    def normal_bf16(self, stream: int, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.uint16)
        self.lib.synth_normal_bf16(self.seed, stream, n, _ptr(out))
        return out


class QueryStream:
    """AR(1) queries, one bf16 [L][B][Hq][d] array per decode step."""

    def __init__(self, syn: Synth, L, B, Hq, d, rho_lo, rho_hi):
        self.syn = syn
        self.shape = (L, B, Hq, d)
        self.rho = np.empty(L * B * Hq, dtype=np.float64)
        syn.lib.synth_query_rho(syn.seed, L, B, Hq, rho_lo, rho_hi, _ptr(self.rho))
        self.state = np.zeros(L * B * Hq * d, dtype=np.float64)
        self.t = 0

    def next(self, out: np.ndarray | None = None) -> np.ndarray:
        L, B, Hq, d = self.shape
        if out is None:
            out = np.empty(self.shape, dtype=np.uint16)
        self.syn.lib.synth_query_step(
            self.syn.seed, L, B, Hq, d, self.t, _ptr(self.rho), _ptr(self.state), _ptr(out)
        )
        self.t += 1
        return out
