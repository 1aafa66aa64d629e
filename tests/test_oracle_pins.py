"""Pins of the CPU oracle against facts fixed outside the oracle itself:
worked values printed on the pages, closed forms, brute force on tiny inputs
with exact rational arithmetic, library routines, and special cases whose result
is known in advance.  A plausible slip in the oracle (a dropped term, a wrong sign
or index, ties broken the wrong way, a transposed operand) fails one of these."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc
from host_offloaded_kv_gb300.synth import Synth, bf16_to_float, float_to_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- KV size
def test_kv_size_worked_values():
    cases = json.load(open(os.path.join(GOLDEN, "kv_size_worked_values.json")))["cases"]
    for c in cases:
        per_tok = orc.kv_bytes_per_token(c["n_kv"], c["d_head"], c["elem_bytes"], c["n_layers"])
        if "bytes_per_token" in c:
            assert per_tok == c["bytes_per_token"], c["cite"]
        if "tokens" in c:
            total = per_tok * c["tokens"] * c.get("batch", 1)
            if "exact_gib" in c:
                assert total == int(c["exact_gib"] * 2**30), c["cite"]
            else:
                assert abs(total / 2**30 - c["approx_gib"]) <= c["approx_tol_gib"], c["cite"]


def test_kv_size_of_workload_pools():
    # the host pools of the named workloads follow the same closed form
    assert orc.kv_bytes_per_token(8, 128, 2, 32) * 32768 * 8 == 32 * 2**30      # Llama3-8B 32K x 8
    assert orc.kv_bytes_per_token(8, 128, 2, 32) * 131072 * 16 == 256 * 2**30   # 128K x 16
    assert orc.kv_bytes_per_token(8, 128, 2, 48) * 524288 == 96 * 2**30         # Qwen2.5-14B 512K
    assert orc.kv_bytes_per_token(2, 64, 2, 1) * 4096 == 2 * 2**20              # tiny


# --------------------------------------------------------------------------- exact sign
def test_exact_sign_against_fractions():
    rng = np.random.default_rng(1)
    for trial in range(300):
        n = int(rng.integers(1, 40))
        base = rng.standard_normal(n) * np.exp2(rng.integers(-60, 60, size=n))
        # plant exact cancellations
        p = list(base)
        for _ in range(int(rng.integers(0, 4))):
            a = float(rng.standard_normal() * 2.0 ** int(rng.integers(-30, 80)))
            p += [a, -a]
        rng.shuffle(p)
        exact = sum(Fraction(x) for x in p)
        want = (exact > 0) - (exact < 0)
        assert orc.exact_sign(np.array(p)) == want


def test_exact_sign_beats_naive_summation():
    p = np.array([2.0**100, 1.0, -(2.0**100)])
    assert sum(p) == 0.0            # naive left-to-right fp64 loses the 1
    assert orc.exact_sign(p) == 1
    assert orc.exact_sign(np.array([2.0**100, -(2.0**100)])) == 0
    assert orc.exact_sign(np.array([-1e-300, 1e300, -1e300])) == -1


# --------------------------------------------------------------------------- hash codes
def _bits_exact(x_u16, R_u16):
    x = [Fraction(float(v)) for v in bf16_to_float(x_u16)]
    Rf = bf16_to_float(R_u16.reshape(-1)).reshape(R_u16.shape)
    code = [0, 0]
    for j in range(128):
        s = sum(x[i] * Fraction(float(Rf[i, j])) for i in range(len(x)))
        if s > 0:
            code[j >> 6] |= 1 << (j & 63)
    return code


@pytest.mark.parametrize("d", [8, 16, 64])
def test_hash_brute_force_exact(d):
    syn = Synth(11)
    R = syn.hash_matrix(0, 0, d)
    X = syn.normal_bf16(99, 12 * d).reshape(12, d)
    codes = orc.hash_codes(X, R)
    for t in range(X.shape[0]):
        want = _bits_exact(X[t], R)
        assert [int(codes[t, 0]), int(codes[t, 1])] == want


def test_hash_cancellation_needs_exact_sum():
    # x . r_j = 2^100 + 1 - 2^100 = 1 exactly; fp64 left-to-right gives 0
    d = 4
    x = float_to_bf16([2.0**100, 1.0, -(2.0**100), 0.0])
    R = np.zeros((d, 128), dtype=np.uint16)
    one = int(float_to_bf16([1.0])[0])
    R[:3, 5] = one
    R[0, 6] = one
    R[2, 6] = one      # column 6: 2^100 - 2^100 = 0 exactly -> bit 0
    code = orc.hash_codes(x[None, :], R)[0]
    assert (int(code[0]) >> 5) & 1 == 1
    assert (int(code[0]) >> 6) & 1 == 0


def test_hash_identity_projection_gives_signs():
    # R[:, j] = e_j for j < d: bit j is sign(x_j) > 0; other columns all zero -> 0
    d = 64
    syn = Synth(5)
    x = syn.normal_bf16(3, d)
    R = np.zeros((d, 128), dtype=np.uint16)
    one = int(float_to_bf16([1.0])[0])
    for j in range(d):
        R[j, j] = one
    code = orc.hash_codes(x[None, :], R)[0]
    xf = bf16_to_float(x)
    for j in range(128):
        bit = (int(code[j >> 6]) >> (j & 63)) & 1
        assert bit == (1 if (j < d and xf[j] > 0) else 0)


def test_hash_negation_and_scaling():
    d = 128
    syn = Synth(6)
    R = syn.hash_matrix(1, 1, d)
    X = syn.normal_bf16(8, 16 * d).reshape(16, d)
    neg = X ^ np.uint16(0x8000)            # flips the sign of every element
    c = orc.hash_codes(X, R)
    cn = orc.hash_codes(neg, R)
    # no exact zero sums with generic data: every bit flips
    assert np.all(c ^ cn == np.uint64(0xFFFFFFFFFFFFFFFF))
    # multiplying by 2^4 (exponent +4 on every nonzero element) changes no sign
    Xf = bf16_to_float(X).astype(np.float64) * 16.0
    c16 = orc.hash_codes(float_to_bf16(Xf), R)
    assert np.array_equal(c, c16)
    # zero vector -> all bits 0
    z = orc.hash_codes(np.zeros((1, d), dtype=np.uint16), R)
    assert int(z[0, 0]) == 0 and int(z[0, 1]) == 0


# --------------------------------------------------------------------------- cosine
def test_cosine_special_cases_and_scipy():
    from scipy.spatial.distance import cosine as scipy_cosine_distance

    syn = Synth(7)
    a = syn.normal_bf16(1, 512)
    b = syn.normal_bf16(2, 512)
    assert orc.cosine(a, a) == pytest.approx(1.0, abs=1e-15)
    assert orc.cosine(a, a ^ np.uint16(0x8000)) == pytest.approx(-1.0, abs=1e-15)
    e1 = np.zeros(8, dtype=np.uint16)
    e2 = np.zeros(8, dtype=np.uint16)
    e1[0] = float_to_bf16([3.0])[0]
    e2[1] = float_to_bf16([-2.0])[0]
    assert orc.cosine(e1, e2) == 0.0
    assert orc.cosine(np.zeros(8, dtype=np.uint16), e1) == 0.0
    want = 1.0 - scipy_cosine_distance(bf16_to_float(a).astype(np.float64), bf16_to_float(b).astype(np.float64))
    assert orc.cosine(a, b) == pytest.approx(want, abs=1e-12)


# --------------------------------------------------------------------------- scores
def test_scores_closed_form_and_extremes():
    rng = np.random.default_rng(3)
    G, N = 4, 200
    q = rng.integers(0, 2**63, size=(G, 2), dtype=np.uint64) * np.uint64(2) + rng.integers(0, 2, size=(G, 2), dtype=np.uint64)
    k = rng.integers(0, 2**63, size=(N, 2), dtype=np.uint64) * np.uint64(2) + rng.integers(0, 2, size=(N, 2), dtype=np.uint64)
    s = orc.scores(q, k)
    qb = np.unpackbits(q.view(np.uint8).reshape(G, 16), axis=1)
    kb = np.unpackbits(k.view(np.uint8).reshape(N, 16), axis=1)
    ham = (qb[None, :, :] != kb[:, None, :]).sum(axis=2)      # [N][G]
    assert np.array_equal(s, G * 128 - ham.sum(axis=1))
    same = orc.scores(q, np.repeat(q[:1], 3, axis=0))
    assert int(same[0]) == 128 + int(orc.scores(q[1:], q[:1])[0])  # head 0 matches fully
    assert int(orc.scores(q[:1], q[:1])[0]) == 128
    assert int(orc.scores(q[:1], ~q[:1])[0]) == 0


# --------------------------------------------------------------------------- top-k
def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(4)
    for _ in range(100):
        N = int(rng.integers(1, 300))
        k = int(rng.integers(1, N + 1))
        sc = rng.integers(0, 6, size=N).astype(np.int32)     # many ties
        want = sorted(sorted(range(N), key=lambda t: (-int(sc[t]), t))[:k])
        got = orc.topk(sc, k)
        assert got.tolist() == want


def test_topk_special_cases():
    N = 1000
    ties = np.zeros(N, dtype=np.int32)
    assert orc.topk(ties, 410).tolist() == list(range(410))
    sc = np.arange(N, dtype=np.int32)[::-1].copy()
    assert orc.topk(sc, N).tolist() == list(range(N))
    sc = np.zeros(N, dtype=np.int32)
    sc[777] = 5
    sc[123] = 5
    assert orc.topk(sc, 1).tolist() == [123]
    got = orc.topk(np.random.default_rng(0).integers(0, 512, size=N).astype(np.int32), 100)
    assert len(got) == 100 and np.all(np.diff(got) > 0)


def test_topk_count_rule():
    assert orc.topk_count(4096, 410, 0.1) == 410
    assert orc.topk_count(4096, 0, 0.1) == 410
    assert orc.topk_count(32768, 0, 0.1) == 3277
    assert orc.topk_count(131072, 0, 0.1) == 13108
    assert orc.topk_count(524288, 0, 0.1) == 52429
    assert orc.topk_count(5, 410, 0.1) == 5
    assert orc.topk_count(3, 0, 0.1) == 1


# --------------------------------------------------------------------------- attention
def test_attention_full_selection_equals_dense_sdpa():
    import torch

    syn = Synth(9)
    G, d, k = 4, 64, 37
    q = syn.normal_bf16(1, G * d).reshape(G, d)
    K = syn.normal_bf16(2, k * d).reshape(k, d)
    V = syn.normal_bf16(3, k * d).reshape(k, d)
    got = orc.attention(q, K, V)
    qt = torch.from_numpy(bf16_to_float(q).astype(np.float64)).view(1, 1, G, d)
    Kt = torch.from_numpy(bf16_to_float(K).astype(np.float64)).view(1, 1, k, d)
    Vt = torch.from_numpy(bf16_to_float(V).astype(np.float64)).view(1, 1, k, d)
    want = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)[0, 0].numpy()
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def test_attention_special_cases():
    syn = Synth(10)
    G, d = 3, 32
    q = syn.normal_bf16(1, G * d).reshape(G, d)
    V = syn.normal_bf16(2, 5 * d).reshape(5, d)
    K = syn.normal_bf16(3, 5 * d).reshape(5, d)
    one = orc.attention(q, K[:1], V[:1])
    assert np.array_equal(one, np.repeat(bf16_to_float(V[:1]).astype(np.float64), G, axis=0))
    same_keys = np.repeat(K[:1], 5, axis=0)
    mean = orc.attention(q, same_keys, V)
    assert np.allclose(mean, np.repeat(bf16_to_float(V).astype(np.float64).mean(0, keepdims=True), G, 0), atol=1e-14)
    # one key aligned with a huge query dominates: output is that row's value
    qh = np.zeros((1, d), dtype=np.uint16)
    qh[0, 0] = float_to_bf16([1000.0])[0]
    Kh = np.zeros((5, d), dtype=np.uint16)
    Kh[3, 0] = float_to_bf16([1.0])[0]
    out = orc.attention(qh, Kh, V)
    assert np.allclose(out[0], bf16_to_float(V[3]), atol=1e-12)
    assert np.array_equal(orc.attention(q, K[:0], V[:0]), np.zeros((G, d)))


# --------------------------------------------------------------------------- state machine
def _small(tau=None, n_persist=0, persist_mask=None, seed=21, rho=(0.6, 0.98), W=4, L=2, B=2, N=64):
    Hq, Hkv, d = 4, 2, 16
    syn = Synth(seed)
    R = syn.hash_matrices(L, Hkv, d)
    o = orc.OracleCLO(L, B, Hq, Hkv, d, R, topk_ratio=0.1, tau=tau, persist_mask=persist_mask,
                      warmup_steps=W, tau_offset=0.05, n_persist=n_persist)
    kv = {}
    for l in range(L):
        for b in range(B):
            for h in range(Hkv):
                K, V = syn.unit_kv(l, b, h, 0, N, d)
                kv[(l, b, h)] = (K, V)
                o.set_unit_kv(l, b, h, K, V)
    qs = syn.query_stream(L, B, Hq, d, *rho)
    return o, qs, kv, (L, B, Hq, Hkv, d, N)


def test_state_tau_minus_one_reuses_forever():
    L, Hkv = 2, 2
    o, qs, kv, (L, B, Hq, Hkv, d, N) = _small(tau=np.full(L * Hkv, -1.0))
    r0 = o.step(qs.next())
    assert np.all(r0.decision == orc.DEC_MISS)
    k = orc.topk_count(N, 0, 0.1)
    assert r0.host_bytes == L * B * Hkv * k * 4 * d
    first = dict(r0.idx)
    for _ in range(5):
        r = o.step(qs.next())
        assert np.all(r.decision == orc.DEC_HIT)
        assert r.host_bytes == 0                 # reused heads fetch nothing
        for u in first:
            assert np.array_equal(r.idx[u], first[u])   # previous selection reused


def test_state_tau_two_never_reuses():
    L, Hkv = 2, 2
    o, qs, kv, (L, B, Hq, Hkv, d, N) = _small(tau=np.full(L * Hkv, 2.0))
    k = orc.topk_count(N, 0, 0.1)
    for _ in range(4):
        q = qs.next()
        r = o.step(q)
        assert np.all(r.decision == orc.DEC_MISS)
        assert r.host_bytes == L * B * Hkv * k * 4 * d
        qr = q.reshape(L, B, Hkv, Hq // Hkv, d)
        for (l, b, h), (K, V) in kv.items():
            # fresh selection = top-k of the current scores; output = attention over it
            sc = orc.scores(orc.hash_codes(qr[l, b, h], o.R[l, h]), orc.hash_codes(K, o.R[l, h]))
            idx = orc.topk(sc, k)
            assert np.array_equal(r.idx[(l, b, h)], idx)
            assert np.allclose(r.out[(l, b, h)], orc.attention(qr[l, b, h], K[idx], V[idx]))
            assert len(idx) == k and np.all(np.diff(idx) > 0)


def test_state_identical_queries_hit_after_first_step():
    L, Hkv = 2, 2
    o, qs, kv, (L, B, Hq, Hkv, d, N) = _small(tau=np.full(L * Hkv, 0.999))
    q = qs.next()
    assert np.all(o.step(q).decision == orc.DEC_MISS)
    r = o.step(q.copy())
    assert np.all(r.decision == orc.DEC_HIT)
    assert np.allclose(r.cos, 1.0, atol=1e-15)


def test_state_persistent_heads_always_reselect():
    L, Hkv = 2, 2
    mask = np.zeros((L, Hkv), dtype=bool)
    mask[:, 1] = True
    o, qs, kv, (L, B, Hq, Hkv, d, N) = _small(tau=np.full(L * Hkv, -1.0), persist_mask=mask)
    k = orc.topk_count(N, 0, 0.1)
    for step in range(3):
        q = qs.next()
        r = o.step(q)
        assert np.all(r.decision[:, :, 1] == orc.DEC_PERSIST)
        want_miss = orc.DEC_MISS if step == 0 else orc.DEC_HIT
        assert np.all(r.decision[:, :, 0] == want_miss)
        # persistent units never fetch host bytes
        assert r.host_bytes == (L * B * k * 4 * d if step == 0 else 0)
        qr = q.reshape(L, B, Hkv, Hq // Hkv, d)
        for l in range(L):
            for b in range(B):
                K, V = kv[(l, b, 1)]
                sc = orc.scores(orc.hash_codes(qr[l, b, 1], o.R[l, 1]), orc.hash_codes(K, o.R[l, 1]))
                assert np.array_equal(r.idx[(l, b, 1)], orc.topk(sc, k))


def test_state_warmup_profile_and_persistent_choice():
    # queries built so that head 0 of every layer repeats exactly (s_hat = 1) and head 1
    # alternates sign (s_hat = -1): head 1 is the hardest to reuse -> persistent.
    L, B, Hq, Hkv, d, W = 2, 2, 4, 2, 16, 4
    syn = Synth(30)
    R = syn.hash_matrices(L, Hkv, d)
    o = orc.OracleCLO(L, B, Hq, Hkv, d, R, topk_ratio=0.1, tau=None, warmup_steps=W, tau_offset=0.05,
                      n_persist=1)
    for l in range(L):
        for b in range(B):
            for h in range(Hkv):
                o.set_unit_kv(l, b, h, *syn.unit_kv(l, b, h, 0, 64, d))
    base = syn.normal_bf16(5, L * B * Hq * d).reshape(L, B, Hq, d)
    for t in range(W):
        q = base.copy()
        if t % 2 == 1:
            q[:, :, 2:, :] ^= np.uint16(0x8000)   # heads of kv group 1 flip sign
        r = o.step(q)
        assert np.all(r.decision == orc.DEC_MISS)
    assert np.allclose(o.shat[:, 0], 1.0) and np.allclose(o.shat[:, 1], -1.0)
    assert np.allclose(o.tau, o.shat - 0.05)
    assert o.persist.tolist() == [[False, True], [False, True]]
    r = o.step(base.copy())
    assert np.all(r.decision[:, :, 1] == orc.DEC_PERSIST)
    assert np.all(r.decision[:, :, 0] == orc.DEC_HIT)       # cos 1 >= 0.95


def test_state_excused_band_follows_device():
    L, Hkv = 2, 2
    o, qs, kv, (L, B, Hq, Hkv, d, N) = _small(tau=np.full(L * Hkv, 2.0))
    q0 = qs.next()
    o.step(q0)
    q1 = qs.next()
    c = orc.cosine(q1.reshape(L, B, Hkv, -1)[0, 0, 0], q0.reshape(L, B, Hkv, -1)[0, 0, 0])
    o.tau[0, 0] = c + 5e-5                  # inside the band: device decision adopted
    dev = np.full((L, B, Hkv), orc.DEC_MISS, dtype=np.int8)
    dev[0, 0, 0] = orc.DEC_HIT
    r = o.step(q1, device_decision=dev)
    assert r.excused[0, 0, 0] and r.decision[0, 0, 0] == orc.DEC_HIT
    assert r.excused.sum() == 1


def _adaptive_small(tau0, ema):
    L, B, Hq, Hkv, d = 1, 2, 4, 2, 16
    syn = Synth(41)
    R = syn.hash_matrices(L, Hkv, d)
    o = orc.OracleCLO(L, B, Hq, Hkv, d, R, topk_ratio=0.1, tau=np.full(L * Hkv, tau0, dtype=np.float32),
                      tau_offset=0.05, adaptive_tau=True, tau_ema=ema)
    return o, syn.normal_bf16(0, L * B * Hq * d).reshape(L, B, Hq, d)


def test_adaptive_tau_closed_form_geometric_decay():
    # sequence 0 repeats its query (cos 1), sequence 1 flips its sign each step
    # (cos -1): the batch mean is 0, so s_hat_n = s_hat_0 (1 - a)^n after the first step
    a = 0.25
    o, q = _adaptive_small(0.3, a)
    s0 = float(np.float32(0.3)) + 0.05
    assert np.allclose(o.shat, s0, rtol=0, atol=1e-15)
    for t in range(6):
        qt = q.copy()
        if t % 2:
            qt[:, 1] ^= 0x8000
        tau_before = o.tau.copy()
        o.step(qt)
        n = max(0, t)            # no previous query at step 0: no update
        want = s0 * (1 - a) ** n
        assert np.allclose(o.shat, want, rtol=0, atol=1e-12), (t, o.shat, want)
        assert np.allclose(o.tau, want - 0.05, rtol=0, atol=1e-12)
        if t == 0:
            assert np.array_equal(o.tau, tau_before)


def test_adaptive_tau_closed_form_converges_to_one():
    # both sequences repeat their queries: m = 1, s_hat_n = 1 - (1 - a)^n (1 - s_hat_0)
    a = 0.5
    o, q = _adaptive_small(0.1, a)
    s0 = float(np.float32(0.1)) + 0.05
    for t in range(5):
        o.step(q)
        want = 1.0 - (1 - a) ** t * (1.0 - s0)
        assert np.allclose(o.shat, want, rtol=0, atol=1e-12)
    # with tau near 1 - 0.05 every reused head now hits (cos = 1 >= tau)
    r = o.step(q)
    assert np.all(r.decision == orc.DEC_HIT)


# ---- quantised host KV -----------------------------------------------------------------
def test_kv_record_bytes_worked_values():
    # host-pool bytes of one token's K|V record of one kv head (what a fetch moves over
    # the link): the codes of 2 d values at b bits, the groups' (scale, min) pairs being
    # kept in GPU memory; d = 128: 2*128*4/8 = 128 B at 4 bits, 64 B at 2 bits; bf16:
    # 2 rows * 128 values * 2 B = 512 B
    assert orc.kv_record_bytes(128, 4) == 128
    assert orc.kv_record_bytes(128, 2) == 64
    assert orc.kv_record_bytes(64, 4) == 64
    assert orc.kv_record_bytes(64, 2) == 32
    assert orc.kv_record_bytes(128, 16) == 512


@pytest.mark.parametrize("bits", [4, 2])
def test_kv_quant_grid_values_roundtrip_exactly(bits):
    # values on the quantisation grid (offset and power-of-two step exact in fp32) come back unchanged
    rng = np.random.default_rng(3)
    levels = (1 << bits) - 1
    for step in (2.0 ** -3, 0.5, 4.0):
        base = float(rng.integers(-8, 8)) * step
        codes = rng.integers(0, levels + 1, size=(5, 64))
        codes[:, 0], codes[:, 1] = 0, levels            # the group spans the whole grid
        x = float_to_bf16(base + codes * step)
        assert np.array_equal(bf16_to_float(x), base + codes * step)
        assert np.array_equal(orc.kv_roundtrip(x, bits), x)


def test_kv_quant_constant_group_is_exact():
    x = np.full((3, 128), 0x3fc0, dtype=np.uint16)     # 1.5 everywhere: scale 0
    for bits in (4, 2):
        assert np.array_equal(orc.kv_roundtrip(x, bits), x)


@pytest.mark.parametrize("bits", [4, 2])
def test_kv_quant_picks_the_nearest_level(bits):
    # brute force over the 2^b levels of each group: the dequantised value is the level
    # nearest to x (up to the rounding of the division), and the group minimum is exact
    rng = np.random.default_rng(5 + bits)
    x = float_to_bf16(rng.standard_normal((40, 64)) * rng.uniform(0.1, 5.0, size=(40, 1)))
    y = bf16_to_float(orc.kv_roundtrip(x, bits)).astype(np.float64)
    xf = bf16_to_float(x).astype(np.float64)
    levels = (1 << bits) - 1
    for g in range(x.shape[0]):
        mn, mx = xf[g].min(), xf[g].max()
        scale = float(np.float32(np.float32(mx - mn) / np.float32(levels)))
        grid = mn + np.arange(levels + 1) * scale
        for i in range(64):
            dist = np.abs(xf[g, i] - grid)
            q = int(np.argmin(np.abs(y[g, i] - grid)))   # level the value came from
            assert dist[q] <= dist.min() + 1e-6 * scale
            assert abs(y[g, i] - grid[q]) <= abs(grid[q]) * 2.0 ** -8 + 1e-30
        assert y[g][np.argmin(xf[g])] == mn


def test_append_tokens_equals_prefill_of_the_longer_context():
    # streaming growth: appending tokens one step at a time gives the same unit state (codes,
    # rows, length, top-k count) as offloading the longer context at once
    L, B, Hq, Hkv, d, N, extra = 1, 2, 4, 2, 64, 300, 5
    syn = Synth(81)
    R = syn.hash_matrices(L, Hkv, d)
    grow = orc.OracleCLO(L, B, Hq, Hkv, d, R, tau=np.full(L * Hkv, 0.9), ntok=[N] * B, kv_bits=4)
    full = orc.OracleCLO(L, B, Hq, Hkv, d, R, tau=np.full(L * Hkv, 0.9), ntok=[N + extra] * B, kv_bits=4)
    rows = {}
    for b in range(B):
        K, V = syn.layer_seq_kv(0, b, Hkv, 0, N + extra, d)
        rows[b] = (K, V)
        for h in range(Hkv):
            grow.set_unit_kv(0, b, h, np.ascontiguousarray(K[:N, h]), np.ascontiguousarray(V[:N, h]))
            full.set_unit_kv(0, b, h, np.ascontiguousarray(K[:, h]), np.ascontiguousarray(V[:, h]))
    for i in range(extra):
        Knew = np.stack([rows[b][0][N + i] for b in range(B)])[None]
        Vnew = np.stack([rows[b][1][N + i] for b in range(B)])[None]
        grow.append_tokens(Knew, Vnew)
    assert np.array_equal(grow.ntok, full.ntok)
    for b in range(B):
        assert grow.k_of(b) == full.k_of(b) == math.ceil(0.1 * (N + extra))
        for h in range(Hkv):
            assert np.array_equal(grow.kcodes[(0, b, h)], full.kcodes[(0, b, h)])
            assert np.array_equal(grow.kv[(0, b, h)][0], full.kv[(0, b, h)][0])
            assert np.array_equal(grow.kv[(0, b, h)][1], full.kv[(0, b, h)][1])


# --------------------------------------------------------------------------- cached query
def _plane_query(theta_deg, d):
    """bf16 query of unit norm at angle theta in the plane of the first two axes."""
    x = np.zeros(d)
    x[0], x[1] = math.cos(math.radians(theta_deg)), math.sin(math.radians(theta_deg))
    return float_to_bf16(x)


def test_state_cached_query_is_the_last_refresh_not_the_previous_step():
    # Reuse test of "CLO (2511.14510) - L3 Per-Paper Synthesis" section 2.1 item 2 read
    # as: compare with the query cached at the unit's last refresh (a miss), so slow
    # drift still triggers a refresh.  Queries turn by 20, 20, 15, 15 degrees per step
    # against tau = 0.9 (cos 20 = 0.940, cos 30 = 0.866, cos 40 = 0.766): every step is
    # within tau of the previous one, so a cache refreshed on hits would hit at every step
    # after the first.
    d = 16
    syn = Synth(71)
    R = syn.hash_matrices(1, 1, d)
    o = orc.OracleCLO(1, 1, 1, 1, d, R, topk_ratio=0.1, tau=np.array([0.9]))
    K, V = syn.unit_kv(0, 0, 0, 0, 200, d)
    o.set_unit_kv(0, 0, 0, K, V)
    k = orc.topk_count(200, 0, 0.1)
    plan = [(0, orc.DEC_MISS, None), (20, orc.DEC_HIT, 0), (40, orc.DEC_MISS, 0), (55, orc.DEC_HIT, 40),
            (70, orc.DEC_MISS, 40), (80, orc.DEC_HIT, 70)]
    for theta, want, ref in plan:
        q = _plane_query(theta, d).reshape(1, 1, 1, d)
        r = o.step(q)
        assert r.decision[0, 0, 0] == want, (theta, r.cos[0, 0, 0])
        if ref is None:
            assert np.isnan(r.cos[0, 0, 0])
        else:
            # the cosine is taken against the query of the last refresh
            assert abs(r.cos[0, 0, 0] - math.cos(math.radians(theta - ref))) < 0.01
        assert r.host_bytes == (k * 4 * d if want == orc.DEC_MISS else 0)
        if want == orc.DEC_MISS:
            refresh_q, refresh_idx = q.copy(), r.idx[(0, 0, 0)].copy()
            sc = orc.scores(orc.hash_codes(q.reshape(1, d), R[0, 0]), orc.hash_codes(K, R[0, 0]))
            assert np.array_equal(refresh_idx, orc.topk(sc, k))
        else:
            assert np.array_equal(r.idx[(0, 0, 0)], refresh_idx)   # the refresh's selection
        assert np.array_equal(o.qcache[0, 0, 0], refresh_q.reshape(-1))


def test_state_persistent_unit_keeps_no_cached_query():
    # persistent heads always reselect ([ABS] feature (2)); they never refresh the cached
    # query, so head 1 stays without one while head 0 refreshes only on its misses
    d, L, B, Hkv = 16, 1, 1, 2
    syn = Synth(72)
    R = syn.hash_matrices(L, Hkv, d)
    mask = np.array([[False, True]])
    o = orc.OracleCLO(L, B, 2, Hkv, d, R, topk_ratio=0.1, tau=np.full(2, 0.9), persist_mask=mask)
    for h in range(Hkv):
        o.set_unit_kv(0, 0, h, *syn.unit_kv(0, 0, h, 0, 100, d))
    for theta in (0, 20, 40, 55):
        q = np.stack([_plane_query(theta, d), _plane_query(theta + 90, d)]).reshape(1, 1, 2, d)
        r = o.step(q)
        assert r.decision[0, 0, 1] == orc.DEC_PERSIST
        assert not o.qvalid[0, 0, 1] and not o.qcache[0, 0, 1].any()
    assert r.decision[0, 0, 0] == orc.DEC_HIT
    assert np.array_equal(o.qcache[0, 0, 0], _plane_query(40, d))


def test_state_warmup_then_persistent_cache_frozen():
    # after warm-up (all misses) the persistent head keeps the cached query of the last
    # warm-up step: later steps neither compare against nor overwrite it
    L, B, Hq, Hkv, d, W = 1, 1, 2, 2, 16, 3
    syn = Synth(73)
    R = syn.hash_matrices(L, Hkv, d)
    o = orc.OracleCLO(L, B, Hq, Hkv, d, R, topk_ratio=0.1, tau=None, warmup_steps=W, tau_offset=0.05,
                      n_persist=1)
    for h in range(Hkv):
        o.set_unit_kv(0, 0, h, *syn.unit_kv(0, 0, h, 0, 100, d))
    # head 0 repeats (s_hat 1), head 1 turns 90 degrees each step (s_hat 0): head 1 persistent
    for t in range(W):
        q = np.stack([_plane_query(0, d), _plane_query(90 * t, d)]).reshape(1, 1, 2, d)
        o.step(q)
    assert o.persist.tolist() == [[False, True]]
    frozen = o.qcache[0, 0, 1].copy()
    assert np.array_equal(frozen, _plane_query(90 * (W - 1), d))
    for t in range(3):
        q = np.stack([_plane_query(0, d), _plane_query(45 * t + 10, d)]).reshape(1, 1, 2, d)
        r = o.step(q)
        assert r.decision[0, 0, 1] == orc.DEC_PERSIST and r.decision[0, 0, 0] == orc.DEC_HIT
        assert np.array_equal(o.qcache[0, 0, 1], frozen)
