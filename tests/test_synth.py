"""The seeded input generator: determinism, rounding and the stated distributions."""
import math
from fractions import Fraction

import numpy as np

from host_offloaded_kv_gb300.synth import Synth, bf16_to_float, float_to_bf16, get_workload


def _rne_bf16_exact(x: float) -> int:
    """Round a double to bf16 (nearest, ties to even) with exact rational arithmetic."""
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    sign = 0x8000 if x < 0 else 0
    a = Fraction(abs(x))
    e = math.floor(math.log2(abs(x)))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                       # subnormals share the smallest exponent
    ulp = Fraction(2) ** (e - 7)
    m = a / ulp
    f = math.floor(m)
    r = m - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    v = float(f * ulp)
    bits = int(np.array([v], dtype=np.float32).view(np.uint32)[0] >> 16)
    return sign | bits


def test_bf16_rounding_single_step():
    rng = np.random.default_rng(0)
    xs = list(rng.standard_normal(400) * np.exp2(rng.integers(-20, 20, 400)))
    # values on and near bf16 midpoints, where double rounding through float would go wrong
    xs += [1.0 + 2.0**-8, 1.0 + 2.0**-8 + 2.0**-40, 1.0 + 3 * 2.0**-8, -(1.0 + 2.0**-8 - 2.0**-45), 1e-40, 3.0e38]
    got = float_to_bf16(np.array(xs))
    for x, g in zip(xs, got):
        assert int(g) == _rne_bf16_exact(float(x)), x


def test_generator_is_counter_based_and_deterministic():
    s1, s2 = Synth(3), Synth(3)
    K1, V1 = s1.unit_kv(2, 1, 3, 100, 50, 64)
    K2, V2 = s2.unit_kv(2, 1, 3, 100, 50, 64)
    assert np.array_equal(K1, K2) and np.array_equal(V1, V2)
    # a sub-range regenerates the same rows
    K3, _ = s1.unit_kv(2, 1, 3, 120, 10, 64)
    assert np.array_equal(K3, K1[20:30])
    # the [n][Hkv][d] layout holds the same per-head rows
    Kall, Vall = s1.layer_seq_kv(2, 1, 4, 100, 50, 64)
    assert np.array_equal(Kall[:, 3, :], K1) and np.array_equal(Vall[:, 3, :], V1)
    assert not np.array_equal(Synth(4).unit_kv(2, 1, 3, 100, 50, 64)[0], K1)


def test_kv_distribution_and_heavy_hitters():
    syn = Synth(1)
    n, d = 20000, 64
    K, V = syn.unit_kv(0, 0, 0, 0, n, d)
    v = bf16_to_float(V).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    heavy = np.array([syn.is_heavy(0, 0, 0, t) for t in range(n)])
    assert 0.008 < heavy.mean() < 0.012           # 1 % heavy hitters
    u = syn.head_direction(0, 0, d)
    assert abs(np.linalg.norm(u) - 1.0) < 1e-12
    k = bf16_to_float(K).astype(np.float64)
    proj = k @ u
    assert abs(proj[heavy].mean() - 4.0) < 0.2    # heavy keys carry 4 * u
    assert abs(proj[~heavy].mean()) < 0.05


def test_query_ar1_similarity():
    syn = Synth(2)
    L, B, Hq, d = 1, 2, 8, 128
    qs = syn.query_stream(L, B, Hq, d, 0.9, 0.9)
    q0 = bf16_to_float(qs.next()).astype(np.float64).reshape(-1, d)
    q1 = bf16_to_float(qs.next()).astype(np.float64).reshape(-1, d)
    cos = (q0 * q1).sum(1) / np.linalg.norm(q0, axis=1) / np.linalg.norm(q1, axis=1)
    assert abs(cos.mean() - 0.9) < 0.03
    assert np.all((qs.rho >= 0.9) & (qs.rho <= 0.9))
    rho = syn.query_stream(4, 4, 8, 16, 0.6, 0.98).rho
    assert rho.min() >= 0.6 and rho.max() <= 0.98 and rho.std() > 0.05


def test_workload_shapes():
    w = get_workload("llama32k")
    assert (w.n_layers, w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_tokens) == (32, 8, 32, 8, 128, 32768)
    assert w.n_persist == 4 and w.tau_fixed is None and w.warmup_steps == 16
    t = get_workload("tiny")
    assert t.topk == 410 and t.tau_fixed == 0.8 and t.group == 4
    assert get_workload("qwen512k").group == 5
