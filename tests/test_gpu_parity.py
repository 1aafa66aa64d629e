"""CUDA library vs CPU oracle, element by element, on seeded inputs (needs a GPU).

Bit-exact: key and query hash codes, top-k index sets, reuse decisions (except
|cos - tau| < 1e-4), gathered rows, host byte counts.  Attention outputs: max abs
error 2e-3 and relative L2 error 1e-3."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from clo_harness import LockStep, Spec  # noqa: E402

pytestmark = pytest.mark.gpu


def _run(spec, steps, io_on_device=True):
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        for _ in range(steps):
            ls.step(io_on_device=io_on_device)
        return ls.log
    finally:
        ls.close()


def test_tiny_workload_full_parity():
    # 1 layer, batch 1, 8/2 heads, d 64, 4096 tokens, k 410, tau 0.8, 16 steps, seed 0
    log = _run(Spec(L=1, B=1, Hq=8, Hkv=2, d=64, ntok=[4096], seed=0, topk=410, tau=0.8), 16)
    assert sum(r["hit"] for r in log) > 0 and sum(r["miss"] for r in log) > 0


def test_warmup_profiling_and_persistent_heads():
    # warm-up thresholds, 1 persistent head per layer; G = 2, d = 128, several tiles
    spec = Spec(L=2, B=2, Hq=8, Hkv=4, d=128, ntok=[6000, 6000], seed=5, tau=None, warmup_steps=4, n_persist=1)
    log = _run(spec, 9)
    assert all(r["persist"] == 4 for r in log[4:])
    assert sum(r["hit"] for r in log[4:]) > 0


def test_ragged_sequences_and_multi_chunk_selection():
    # three sequences of different lengths: 5, 3 and 1 selection chunks of 8192 tokens,
    # ragged last chunks, empty chunks for the shorter sequences; G = 5
    spec = Spec(L=1, B=3, Hq=10, Hkv=2, d=128, ntok=[40000, 17000, 3001], seed=7, tau=0.8, rho=(0.7, 0.98))
    _run(spec, 4)


def test_host_buffer_io_matches_device_io():
    spec = Spec(L=1, B=2, Hq=4, Hkv=2, d=64, ntok=[3000, 2500], seed=9, tau=0.85)
    _run(spec, 5, io_on_device=False)


def test_topk_equals_context_is_dense_attention():
    # k = N: every token selected; attention is plain softmax attention
    spec = Spec(L=1, B=1, Hq=4, Hkv=1, d=64, ntok=[700], seed=11, topk=700, tau=2.0)
    _run(spec, 2)


def test_single_token_context():
    spec = Spec(L=2, B=2, Hq=2, Hkv=1, d=64, ntok=[1, 1], seed=12, tau=0.5)
    _run(spec, 3)


@pytest.mark.parametrize("N,topk", [(5000, 0), (20000, 10000)])
def test_all_scores_tied_selects_lowest_indices(N, topk):
    # all-zero keys: every key code is 0 and every score ties -> selection {0..k-1}; with
    # N = 20000 and k = 10000 the tie quota fills chunk 0 and part of chunk 1
    L, B, Hkv, d = 1, 1, 2, 64
    K = np.zeros((N, Hkv, d), dtype=np.uint16)
    V = np.zeros((N, Hkv, d), dtype=np.uint16)
    V[:, :, :] = np.arange(N, dtype=np.uint16)[:, None, None] & 0x3fff   # distinct finite values
    spec = Spec(L=L, B=B, Hq=4, Hkv=Hkv, d=d, ntok=[N], seed=13, tau=2.0, topk=topk, kv_override={(0, 0): (K, V)})
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        ls.step()
        k = ls.lib.k_of(0)
        assert ls.lib.idx(0, 0, 0).tolist() == list(range(k))
    finally:
        ls.close()


def test_hash_cancellations_take_the_exact_tiers():
    # keys built from the projection's own columns: token t uses column j = t % 128 and
    # x = (R[1, j], -R[0, j], c, 0, ...), whose dot with column j is exactly c * R[2, j]:
    # c = 0 (exact zero: bit 0), c = 2^-18 (too small for the fp32 chain's bound, settled
    # by the compensated sum) or c = 2^-40 (below that bound too: settled by the exact
    # fixed-point tier).  Codes must match the oracle bit for bit.
    from host_offloaded_kv_gb300.synth import Synth

    L, B, Hkv, d, N, seed = 1, 1, 1, 64, 768, 21
    R = Synth(seed, 0.01).hash_matrices(L, Hkv, d)[0, 0]   # bf16 bits [d][128]
    K = np.zeros((N, Hkv, d), dtype=np.uint16)
    tiny = {0: 0, 1: 0x3680, 2: 0x2B80}                      # bf16 bits of 0, 2^-18, 2^-40
    for t in range(N):
        j = t % 128
        K[t, 0, 0] = R[1, j]
        K[t, 0, 1] = R[0, j] ^ 0x8000
        K[t, 0, 2] = tiny[(t // 128) % 3]
    V = np.zeros((N, Hkv, d), dtype=np.uint16)
    V[:, :, :] = (np.arange(N, dtype=np.uint16)[:, None, None] % 977 + 0x3c00) & 0x7fff
    spec = Spec(L=L, B=B, Hq=2, Hkv=Hkv, d=d, ntok=[N], seed=seed, tau=2.0, kv_override={(0, 0): (K, V)})
    ls = LockStep(spec)
    try:
        ls.check_key_codes()
        codes = ls.lib.key_codes(0, 0, 0)
        bits = np.unpackbits(codes.view(np.uint8), bitorder="little").reshape(N, 128)
        zero_rows = [t for t in range(N) if (t // 128) % 3 == 0]
        assert not bits[zero_rows, np.array(zero_rows) % 128].any()  # exact zeros give bit 0
        ls.step()
    finally:
        ls.close()


def test_whole_unit_selection_many_units():
    # 2 layers x 38 sequences x 8 kv heads = 608 units: enough for persistent units to be
    # selected whole by one compute group each, while missed units use chunks (the smaller
    # cases above cover chunks only); ragged lengths, G = 4, two persistent heads per layer
    ntok = [3000 - 37 * b for b in range(38)]
    pm = np.zeros((2, 8), dtype=np.uint8)
    pm[:, [0, 5]] = 1
    spec = Spec(L=2, B=38, Hq=32, Hkv=8, d=64, ntok=ntok, seed=61, tau=0.9, rho=(0.8, 0.99), persist_mask=pm)
    log = _run(spec, 3)
    assert all(r["persist"] == 2 * 38 * 2 for r in log) and sum(r["miss"] for r in log) > 0


@pytest.mark.parametrize("G", [3, 6, 7, 8])
def test_group_sizes_chunked_selection(G):
    # the bit-plane scorer at every plane count (G = 3: 2 planes, 6 and 7: 3, 8: 4, with
    # scores up to 1024) through chunked selection: ragged lengths, one persistent head
    pm = np.array([[1, 0]], dtype=np.uint8)
    spec = Spec(L=1, B=2, Hq=2 * G, Hkv=2, d=64, ntok=[9001, 4099], seed=80 + G, tau=0.85, rho=(0.7, 0.98),
                persist_mask=pm)
    log = _run(spec, 4)
    assert sum(r["miss"] for r in log) > 0


def test_whole_unit_selection_largest_group():
    # G = 8 (64/8 heads), 2 layers x 38 sequences x 8 kv heads = 608 units: the persistent
    # units are selected whole, with scores spanning 0 .. 1024; ragged lengths
    ntok = [2500 - 29 * b for b in range(38)]
    pm = np.zeros((2, 8), dtype=np.uint8)
    pm[:, [2, 7]] = 1
    spec = Spec(L=2, B=38, Hq=64, Hkv=8, d=64, ntok=ntok, seed=88, tau=0.9, rho=(0.8, 0.99), persist_mask=pm)
    log = _run(spec, 2)
    assert all(r["persist"] == 2 * 38 * 2 for r in log)


def test_cached_query_is_the_last_refresh():
    # queries turning 20, 20, 15, 15, 10 degrees per step against tau = 0.9: the reuse test
    # compares with the query of the unit's last refresh, so it misses at 40 and 70 degrees
    # although every step is within tau of the previous one; head 1 is persistent
    import math

    from host_offloaded_kv_gb300.synth import float_to_bf16

    d = 64
    pm = np.array([[0, 1]], dtype=np.uint8)
    spec = Spec(L=1, B=1, Hq=2, Hkv=2, d=d, ntok=[3000], seed=74, tau=0.9, persist_mask=pm)
    ls = LockStep(spec)
    try:
        want = []
        for theta in (0, 20, 40, 55, 70, 80):
            q = np.zeros((1, 1, 2, d))
            for h, a in ((0, theta), (1, theta + 90)):
                q[0, 0, h, 0], q[0, 0, h, 1] = math.cos(math.radians(a)), math.sin(math.radians(a))
            res, _, dec, _ = ls.step(q=float_to_bf16(q))
            want.append(int(dec[0, 0, 0]))
            assert dec[0, 0, 1] == 2
        assert want == [1, 0, 1, 0, 1, 0]
    finally:
        ls.close()
