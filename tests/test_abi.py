"""The C-ABI library loads and exports every entry point include/clo.h declares
(no compute call: runs without a GPU)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "clo.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CLO_API\s+[\w\s\*]+?\b(clo_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def libpath():
    import __graft_entry__ as ge

    ge.build()
    from host_offloaded_kv_gb300 import clo

    return clo.LIB_PATH


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("clo_init", "clo_append_kv", "clo_decode_step", "clo_stats", "clo_destroy", "clo_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    for n in _declared():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (clo_\w+)", out))
    assert set(_declared()) <= exported
    # nothing but the C ABI is exported
    assert all(s.startswith("clo_") for s in exported)


def test_binding_names_match_header(libpath):
    from host_offloaded_kv_gb300 import clo

    assert set(clo.EXPORTED) == set(_declared())
    for n in clo.EXPORTED:
        assert callable(getattr(clo, n))


def test_config_default_and_invalid_config_without_gpu(libpath):
    from host_offloaded_kv_gb300 import clo

    cfg = clo.clo_config_default()
    assert abs(cfg.topk_ratio - 0.1) < 1e-15 and cfg.warmup_steps == 16 and cfg.debug_drop_flag_layer == -1
    # invalid shapes are rejected before any CUDA call
    cfg.n_layers = 0
    with pytest.raises(clo.CLOError) as e:
        clo.clo_init(cfg)
    assert e.value.status == clo.CLO_ERR_INVALID
    assert "shapes" in clo.clo_last_error()


_R = np.zeros((1, 1, 64, 128), dtype=np.uint16)


def _valid_shapes(clo):
    cfg = clo.clo_config_default()
    cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.max_tokens = 1, 1, 4, 1, 64, 128
    cfg.hash_R = _R.ctypes.data
    return cfg


@pytest.mark.parametrize("field,value,text", [("kv_bits", 3, "kv_bits"), ("kv_bits", 8, "kv_bits"),
                                              ("tau_ema", 0.0, "tau_ema"), ("tau_ema", 1.5, "tau_ema")])
def test_invalid_extension_settings_without_gpu(libpath, field, value, text):
    from host_offloaded_kv_gb300 import clo

    cfg = _valid_shapes(clo)
    assert cfg.kv_bits == 0 and abs(cfg.tau_ema - 0.0625) < 1e-15 and cfg.adaptive_tau == 0
    cfg.adaptive_tau = 1
    setattr(cfg, field, value)
    with pytest.raises(clo.CLOError) as e:
        clo.clo_init(cfg)
    assert e.value.status == clo.CLO_ERR_INVALID
    assert text in clo.clo_last_error()


def test_struct_layout_matches_header(libpath):
    from host_offloaded_kv_gb300 import clo

    # the C struct sizes as compiled by the host compiler (probe through a tiny C file)
    src = "#include <stdio.h>\n#include \"clo.h\"\nint main(){printf(\"%zu %zu\", sizeof(clo_config), sizeof(clo_stats_t));}\n"
    tmp = os.path.join(ROOT, "host_offloaded_kv_gb300", "_lib", "layout_probe.c")
    exe = tmp[:-2]
    with open(tmp, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), tmp, "-o", exe], check=True)
    sizes = subprocess.run([exe], capture_output=True, text=True).stdout.split()
    assert int(sizes[0]) == ctypes.sizeof(clo.clo_config)
    assert int(sizes[1]) == ctypes.sizeof(clo.clo_stats_t)


@pytest.mark.parametrize("q,rows,out", [(0x10000, 0x10008, 0x20000), (0x10001, 0x10000, 0x20000),
                                        (0x10000, 0x10000, 0x20002)])
def test_noalloc_refuses_misaligned_pointers_without_gpu(libpath, q, rows, out):
    # rows are read with 16-byte copies, q as bf16, out as fp32: a misaligned pointer is
    # refused before any CUDA call (the addresses are never dereferenced)
    from host_offloaded_kv_gb300 import clo

    lib = clo.load_library()
    st = lib.clo_sparse_attention_noalloc(q, rows, out, 4, 4, 128, 300, None)
    assert st == clo.CLO_ERR_INVALID
    assert "aligned" in clo.clo_last_error()


def test_noalloc_python_wrapper_refuses_host_buffers(libpath):
    from host_offloaded_kv_gb300 import clo

    torch = pytest.importorskip("torch")
    q = torch.zeros((2, 4, 64), dtype=torch.int16)
    rows = torch.zeros((2, 10, 2, 64), dtype=torch.int16)
    out = torch.zeros((2, 4, 64), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        clo.clo_sparse_attention_noalloc(q, rows, out, 2, 4, 64, 10)
    with pytest.raises(ValueError, match="CUDA tensor"):
        clo.clo_sparse_attention_noalloc(q.numpy(), rows, out, 2, 4, 64, 10)
