"""Python binding of the CLO C ABI (``include/clo.h``): argument marshalling only.

The functions carry the C names; every step of the decode path runs in the CUDA
library ``_lib/libclo.so``.  There is no fallback: if the library is missing or
fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libclo.so")

CLO_OK, CLO_ERR_INVALID, CLO_ERR_OOM, CLO_ERR_CUDA, CLO_ERR_TIMEOUT, CLO_ERR_STATE, CLO_ERR_CAPACITY, \
    CLO_ERR_DEVICE = range(8)
CLO_DEC_HIT, CLO_DEC_MISS, CLO_DEC_PERSIST = 0, 1, 2
(CLO_DBG_KEY_CODES, CLO_DBG_QUERY_CODES, CLO_DBG_IDX, CLO_DBG_DECISION, CLO_DBG_SLOT_ROWS, CLO_DBG_TAU,
 CLO_DBG_PERSIST, CLO_DBG_SHAT, CLO_DBG_COS, CLO_DBG_TIMELINE, CLO_DBG_TOPK, CLO_DBG_POOL_NODE,
 CLO_DBG_STEP_BYTES) = range(1, 14)
STEP_HIST = 4096
CLO_SET_DROP_FLAG_LAYER, CLO_SET_WAIT_TIMEOUT_NS = 1, 2

_STATUS_NAMES = {0: "CLO_OK", 1: "CLO_ERR_INVALID", 2: "CLO_ERR_OOM", 3: "CLO_ERR_CUDA", 4: "CLO_ERR_TIMEOUT",
                 5: "CLO_ERR_STATE", 6: "CLO_ERR_CAPACITY", 7: "CLO_ERR_DEVICE"}

EXPORTED = ["clo_config_default", "clo_init", "clo_destroy", "clo_append_kv", "clo_append_step", "clo_decode_step",
            "clo_decode_layer",
            "clo_sync", "clo_stats", "clo_last_error", "clo_debug_get", "clo_set", "clo_sparse_attention_noalloc"]


class CLOError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class clo_config(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("max_tokens", ctypes.c_int64),
        ("topk", ctypes.c_int64),
        ("topk_ratio", ctypes.c_double),
        ("hash_R", ctypes.c_void_p),
        ("tau", ctypes.c_void_p),
        ("persist_mask", ctypes.c_void_p),
        ("warmup_steps", ctypes.c_int32),
        ("tau_offset", ctypes.c_float),
        ("n_persist", ctypes.c_int32),
        ("wait_timeout_ns", ctypes.c_int64),
        ("timing", ctypes.c_int32),
        ("debug_drop_flag_layer", ctypes.c_int32),
        ("stream", ctypes.c_void_p),
        ("adaptive_tau", ctypes.c_int32),
        ("tau_ema", ctypes.c_double),
        ("kv_bits", ctypes.c_int32),
    ]


class clo_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "steps", "units_hit", "units_miss", "units_persist", "host_bytes", "hbm_bytes_alg", "timeouts",
        "last_hit", "last_miss", "last_persist", "last_host_bytes", "last_hbm_bytes_alg")] + \
        [("warmup_done", ctypes.c_int32), ("timed_steps", ctypes.c_int32)] + \
        [(n, ctypes.c_float) for n in ("last_ms_decide", "last_ms_fused", "last_ms_total")] + \
        [(n, ctypes.c_double) for n in ("sum_ms_decide", "sum_ms_fused", "sum_ms_total")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libclo.so (raises if it is missing: the package has no CPU path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.clo_config_default.restype = None
    lib.clo_config_default.argtypes = [ctypes.POINTER(clo_config)]
    lib.clo_init.restype = ctypes.c_int
    lib.clo_init.argtypes = [ctypes.POINTER(clo_config), ctypes.POINTER(vp)]
    lib.clo_destroy.restype = ctypes.c_int
    lib.clo_destroy.argtypes = [vp]
    lib.clo_append_kv.restype = ctypes.c_int
    lib.clo_append_kv.argtypes = [vp, i32, i32, vp, vp, i64, i32]
    lib.clo_decode_step.restype = ctypes.c_int
    lib.clo_decode_step.argtypes = [vp, vp, vp, i32]
    lib.clo_append_step.restype = ctypes.c_int
    lib.clo_append_step.argtypes = [vp, vp, vp, i32]
    lib.clo_decode_layer.restype = ctypes.c_int
    lib.clo_decode_layer.argtypes = [vp, i32, vp, vp, i32]
    lib.clo_sync.restype = ctypes.c_int
    lib.clo_sync.argtypes = [vp]
    lib.clo_stats.restype = ctypes.c_int
    lib.clo_stats.argtypes = [vp, ctypes.POINTER(clo_stats_t)]
    lib.clo_last_error.restype = ctypes.c_char_p
    lib.clo_last_error.argtypes = []
    lib.clo_debug_get.restype = ctypes.c_int
    lib.clo_debug_get.argtypes = [vp, i32, i32, i32, i32, vp, i64]
    lib.clo_set.restype = ctypes.c_int
    lib.clo_set.argtypes = [vp, i32, i64]
    lib.clo_sparse_attention_noalloc.restype = ctypes.c_int
    lib.clo_sparse_attention_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i64, vp]
    _lib = lib
    return lib


def clo_last_error() -> str:
    return load_library().clo_last_error().decode(errors="replace")


def _check(status: int, where: str):
    if status != CLO_OK:
        raise CLOError(status, where, clo_last_error())


def _ptr(x):
    """(pointer, on_device) of a numpy array or torch tensor (must be contiguous)."""
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return x.ctypes.data, False
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return x.data_ptr(), x.device.type == "cuda"
    if isinstance(x, int):
        return x, None
    raise TypeError(f"unsupported buffer type {type(x)}")


# ----------------------------------------------------------------------------- C names
def clo_config_default() -> clo_config:
    cfg = clo_config()
    load_library().clo_config_default(ctypes.byref(cfg))
    return cfg


def clo_init(cfg: clo_config) -> ctypes.c_void_p:
    ctx = ctypes.c_void_p()
    _check(load_library().clo_init(ctypes.byref(cfg), ctypes.byref(ctx)), "clo_init")
    return ctx


def clo_destroy(ctx) -> None:
    _check(load_library().clo_destroy(ctx), "clo_destroy")


def clo_append_kv(ctx, layer: int, seq: int, k, v, n_tokens: int, src_is_device: bool | None = None) -> None:
    kp, kdev = _ptr(k)
    vp_, vdev = _ptr(v)
    dev = kdev if src_is_device is None else bool(src_is_device)
    _check(load_library().clo_append_kv(ctx, layer, seq, kp, vp_, int(n_tokens), int(bool(dev))), "clo_append_kv")


def clo_append_step(ctx, k, v, src_is_device: bool | None = None) -> None:
    kp, kdev = _ptr(k)
    vp_, vdev = _ptr(v)
    dev = kdev if src_is_device is None else bool(src_is_device)
    _check(load_library().clo_append_step(ctx, kp, vp_, int(bool(dev))), "clo_append_step")


def clo_decode_step(ctx, q, out, io_on_device: bool | None = None) -> None:
    qp, qdev = _ptr(q)
    op, odev = _ptr(out)
    dev = qdev if io_on_device is None else bool(io_on_device)
    _check(load_library().clo_decode_step(ctx, qp, op, int(bool(dev))), "clo_decode_step")


def clo_decode_layer(ctx, layer: int, q, out, io_on_device: bool | None = None) -> None:
    qp, qdev = _ptr(q)
    op, odev = _ptr(out)
    dev = qdev if io_on_device is None else bool(io_on_device)
    _check(load_library().clo_decode_layer(ctx, int(layer), qp, op, int(bool(dev))), "clo_decode_layer")


def clo_sync(ctx) -> None:
    _check(load_library().clo_sync(ctx), "clo_sync")


def clo_stats(ctx) -> dict:
    st = clo_stats_t()
    _check(load_library().clo_stats(ctx, ctypes.byref(st)), "clo_stats")
    return st.as_dict()


def clo_debug_get(ctx, what: int, layer: int, seq: int, kvh: int, dst: np.ndarray) -> np.ndarray:
    p, _ = _ptr(dst)
    _check(load_library().clo_debug_get(ctx, what, layer, seq, kvh, p, dst.nbytes), "clo_debug_get")
    return dst


def clo_set(ctx, key: int, value: int) -> None:
    _check(load_library().clo_set(ctx, key, int(value)), "clo_set")


def clo_sparse_attention_noalloc(q, rows, out, n_groups: int, group_size: int, head_dim: int, k: int,
                                 stream=None) -> None:
    """Allocation-free sparse attention (device buffers; see include/clo.h).

    q: bf16 (int16/uint16 bit patterns) [n_groups][group_size][head_dim], rows: bf16
    [n_groups][>= k][2][head_dim], out: fp32 [n_groups][group_size][head_dim]; all
    three CUDA tensors on the current device.  Plain integers are passed through as raw
    device addresses (the caller vouches for them)."""
    import torch

    G, D, n = int(group_size), int(head_dim), int(n_groups)
    want = {"q": (q, n * G * D, (torch.int16, torch.uint16, torch.bfloat16)),
            "rows": (rows, n * int(k) * 2 * D, (torch.int16, torch.uint16, torch.bfloat16)),
            "out": (out, n * G * D, (torch.float32,))}
    for name, (t, numel, dtypes) in want.items():
        if isinstance(t, int):
            continue
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device.index != torch.cuda.current_device():
            raise ValueError(f"{name} is on {t.device}, not on the current device")
        if t.dtype not in dtypes:
            raise ValueError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
        if (t.numel() < numel) if name == "rows" else (t.numel() != numel):
            raise ValueError(f"{name} holds {t.numel()} elements; expected {numel}")
    qp, _ = _ptr(q)
    rp, _ = _ptr(rows)
    op, _ = _ptr(out)
    _check(load_library().clo_sparse_attention_noalloc(qp, rp, op, int(n_groups), int(group_size), int(head_dim),
                                                       int(k), stream), "clo_sparse_attention_noalloc")


# ----------------------------------------------------------------------------- convenience
class CLOContext:
    """Owns one library context; keeps the shapes needed to size debug read-backs."""

    def __init__(self, *, n_layers, batch, n_q_heads, n_kv_heads, head_dim, max_tokens, hash_R, topk=0,
                 topk_ratio=0.1, tau=None, persist_mask=None, warmup_steps=16, tau_offset=0.05, n_persist=0,
                 wait_timeout_ns=2_000_000_000, timing=False, stream=None, adaptive_tau=False, tau_ema=0.0625,
                 kv_bits=16):
        self.L, self.B, self.Hq, self.Hkv, self.d = n_layers, batch, n_q_heads, n_kv_heads, head_dim
        self.G = n_q_heads // n_kv_heads
        self.topk, self.topk_ratio = int(topk), float(topk_ratio)
        self._R = np.ascontiguousarray(hash_R, dtype=np.uint16)
        self._tau = None if tau is None else np.ascontiguousarray(tau, dtype=np.float32)
        self._pm = None if persist_mask is None else np.ascontiguousarray(persist_mask, dtype=np.uint8)
        cfg = clo_config_default()
        cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim = (
            n_layers, batch, n_q_heads, n_kv_heads, head_dim)
        cfg.max_tokens = int(max_tokens)
        cfg.topk = int(topk)
        cfg.topk_ratio = float(topk_ratio)
        cfg.hash_R = self._R.ctypes.data
        cfg.tau = None if self._tau is None else self._tau.ctypes.data
        cfg.persist_mask = None if self._pm is None else self._pm.ctypes.data
        cfg.warmup_steps = int(warmup_steps)
        cfg.tau_offset = float(tau_offset)
        cfg.n_persist = int(n_persist)
        cfg.wait_timeout_ns = int(wait_timeout_ns)
        cfg.timing = int(bool(timing))
        cfg.debug_drop_flag_layer = -1
        cfg.stream = stream
        cfg.adaptive_tau = int(bool(adaptive_tau))
        cfg.tau_ema = float(tau_ema)
        cfg.kv_bits = int(kv_bits)
        self.kv_bits = int(kv_bits)
        self.cfg = cfg
        self.ctx = clo_init(cfg)
        self.ntok = np.zeros((n_layers, batch), dtype=np.int64)

    def close(self):
        if self.ctx is not None:
            clo_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def step_bytes(self, first: int, last: int) -> np.ndarray:
        """Host-link and algorithmic HBM bytes of each step in [first, last) (timing mode):
        int64 [last - first][2], from the library's cumulative per-step history."""
        if last - first + 1 > STEP_HIST or first < 1:
            raise ValueError("the history keeps the last 4096 steps and needs the step before the first")
        h = clo_debug_get(self.ctx, CLO_DBG_STEP_BYTES, 0, 0, 0, np.empty((STEP_HIST, 2), dtype=np.uint64))
        cum = np.array([h[s % STEP_HIST] for s in range(first - 1, last)], dtype=np.int64)
        return np.diff(cum, axis=0)

    def pool_node(self) -> int:
        """NUMA node of the pinned pool's pages, or -1 when the pool was not placed."""
        return int(clo_debug_get(self.ctx, CLO_DBG_POOL_NODE, 0, 0, 0, np.empty(1, dtype=np.int32))[0])

    def k_of(self, b: int, layer: int = 0) -> int:
        """The library's top-k count of (layer, sequence b) at its current length."""
        k = clo_debug_get(self.ctx, CLO_DBG_TOPK, 0, 0, 0, np.empty((self.L, self.B), dtype=np.int32))
        return int(k[layer, b])

    def append_kv(self, layer, seq, k, v, src_is_device=None):
        n = k.shape[0]
        clo_append_kv(self.ctx, layer, seq, k, v, n, src_is_device)
        self.ntok[layer, seq] += n

    def append_step(self, k, v, src_is_device=None):
        """One new token for every (layer, sequence): k, v bf16 [L][B][Hkv][d]."""
        clo_append_step(self.ctx, k, v, src_is_device)
        self.ntok += 1

    def decode_step(self, q, out, io_on_device=None):
        clo_decode_step(self.ctx, q, out, io_on_device)

    def decode_layer(self, layer, q, out, io_on_device=None):
        """One layer of a step: q bf16 [B][Hq][d], out fp32 [B][Hq][d]; layers in order."""
        clo_decode_layer(self.ctx, layer, q, out, io_on_device)

    def sync(self):
        clo_sync(self.ctx)

    def stats(self):
        return clo_stats(self.ctx)

    def set(self, key, value):
        clo_set(self.ctx, key, value)

    # debug read-backs ----------------------------------------------------------
    def key_codes(self, l, b, h):
        return clo_debug_get(self.ctx, CLO_DBG_KEY_CODES, l, b, h,
                             np.empty((int(self.ntok[l, b]), 2), dtype=np.uint64))

    def query_codes(self, l, b, h):
        return clo_debug_get(self.ctx, CLO_DBG_QUERY_CODES, l, b, h, np.empty((self.G, 2), dtype=np.uint64))

    def idx(self, l, b, h):
        return clo_debug_get(self.ctx, CLO_DBG_IDX, l, b, h, np.empty(self.k_of(b, l), dtype=np.int32))

    def slot_rows(self, l, b, h):
        return clo_debug_get(self.ctx, CLO_DBG_SLOT_ROWS, l, b, h,
                             np.empty((self.k_of(b, l), 2, self.d), dtype=np.uint16))

    def decisions(self):
        return clo_debug_get(self.ctx, CLO_DBG_DECISION, 0, 0, 0,
                             np.empty((self.L, self.B, self.Hkv), dtype=np.uint8))

    def cosines(self):
        return clo_debug_get(self.ctx, CLO_DBG_COS, 0, 0, 0, np.empty((self.L, self.B, self.Hkv), dtype=np.float32))

    def tau(self):
        return clo_debug_get(self.ctx, CLO_DBG_TAU, 0, 0, 0, np.empty((self.L, self.Hkv), dtype=np.float32))

    def persist(self):
        return clo_debug_get(self.ctx, CLO_DBG_PERSIST, 0, 0, 0, np.empty((self.L, self.Hkv), dtype=np.uint8))

    def shat(self):
        return clo_debug_get(self.ctx, CLO_DBG_SHAT, 0, 0, 0, np.empty((self.L, self.Hkv), dtype=np.float64))

    def timeline(self):
        """Stamps of the last step's fused kernel (timing mode), in us from its start."""
        t = clo_debug_get(self.ctx, CLO_DBG_TIMELINE, 0, 0, 0, np.empty(16, dtype=np.uint64)).astype(np.int64)
        if t[0] == 0:
            return None
        rel = lambda v: None if v == 0 else round((int(v) - int(t[0])) / 1e3, 1)  # noqa: E731
        return {"sel_missed_done_us": rel(t[1]), "sel_persistent_done_us": rel(t[2]),
                "first_fetch_us": rel(t[3]), "fetch_done_us": rel(t[4]), "first_attention_us": rel(t[5]),
                "attention_done_us": rel(t[6]), "fetch_wait_sum_us": round(int(t[7]) / 1e3, 1),
                "attention_wait_sum_us": round(int(t[8]) / 1e3, 1),
                "selection_chunk_mean_us": round(int(t[9]) / 1e3 / max(1, int(t[10])), 2),
                "selection_chunks": int(t[10]),
                "attention_split_mean_us": round(int(t[11]) / 1e3 / max(1, int(t[12])), 2),
                "attention_splits": int(t[12]), "decide_start_us": rel(t[13]), "decide_end_us": rel(t[14]),
                "attention_split_run_mean_us": round(int(t[15]) / 1e3 / max(1, int(t[12])), 2)}
