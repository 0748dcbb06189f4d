"""Host-side planning of a pass, checked without a GPU through the C ABI.

tee_plan_attention: the attention work items (global layers: one per text
and 128-query tile, consecutive texts spanning at most 128 tokens sharing one;
window layers: one per 128-row tile of the packed sequence) with the key range
the tile's queries may see, compared with a
brute force over every query row of the tile (whole text on global layers,
|i - j| <= window inside the text otherwise).  tee_plan_gemm: the tensor-core
GEMM's tile shapes for the projections of the 310m shape, pinned to values
worked out by hand from the column-wave rule, plus invariants over a grid of
shapes.
"""
import ctypes
import os
import shutil

import numpy as np
import pytest

from text_embedding_encoder_gb300 import binding


@pytest.fixture(scope="module")
def built_lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no CUDA toolkit")
    from text_embedding_encoder_gb300 import build
    return binding.load(build.build())


def _plan_attention(lib, cu, window, is_global, max_items=None):
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    n = len(cu) - 1
    count = lib.tee_plan_attention(cu.ctypes.data, n, window, int(is_global), None, 0)
    if count < 0:
        return count, None
    cap = count if max_items is None else max_items
    out = np.zeros((max(cap, 1), 4), dtype=np.int32)
    rc = lib.tee_plan_attention(cu.ctypes.data, n, window, int(is_global), out.ctypes.data, cap)
    return rc, out[:max(rc, 0)]


def _visible(cu, window, is_global):
    """Dense mask [T, T]: query i may see key j (same text, and |i - j| <= window
    unless the layer is global)."""
    T = int(cu[-1])
    text = np.searchsorted(cu, np.arange(T), side="right") - 1
    same = text[:, None] == text[None, :]
    if is_global:
        return same
    idx = np.arange(T)
    return same & (np.abs(idx[:, None] - idx[None, :]) <= window)


def _brute_force_items(cu, window, is_global):
    """Global layers: every (text, 128-query tile); window layers: every 128-row
    tile of the packed sequence.  Each with the smallest key interval holding
    every key that some query row of the tile may attend to."""
    vis = _visible(cu, window, is_global)
    items = []

    def add(q0, ql):
        cols = np.nonzero(vis[q0:q0 + ql].any(axis=0))[0]
        items.append((q0, ql, int(cols.min()), int(cols.max()) + 1))

    if is_global:
        n = len(cu) - 1
        j = 0
        while j < n:
            s0, s1 = int(cu[j]), int(cu[j + 1])
            if s1 - s0 <= 128:
                # consecutive texts of <= 128 tokens share a tile while their span fits
                k = j + 1
                while k < n and int(cu[k + 1]) - s0 <= 128:
                    k += 1
                add(s0, int(cu[k]) - s0)
                j = k
            else:
                for q0 in range(s0, s1, 128):
                    add(q0, min(128, s1 - q0))
                j += 1
        items = sorted(items, key=lambda it: -it[1] * (it[3] - it[2]))   # most work first, stable
    else:
        T = int(cu[-1])
        for q0 in range(0, T, 128):
            add(q0, min(128, T - q0))
    return items


@pytest.mark.parametrize("lengths", [[1], [2, 1, 3], [127, 128, 129], [65, 66, 130, 257], [300, 8, 1000, 64],
                                     [129] * 5])
@pytest.mark.parametrize("window", [0, 1, 64, 200])
@pytest.mark.parametrize("is_global", [False, True])
def test_attention_items_match_brute_force(built_lib, lengths, window, is_global):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    rc, got = _plan_attention(built_lib, cu, window, is_global)
    want = _brute_force_items(cu, window, is_global)
    assert rc == len(want)
    assert [tuple(int(v) for v in it) for it in got] == want


def test_attention_items_random_packings(built_lib):
    rng = np.random.default_rng(5)
    for _ in range(20):
        lengths = rng.integers(1, 400, size=int(rng.integers(1, 9)))
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        for is_global in (False, True):
            rc, got = _plan_attention(built_lib, cu, 64, is_global)
            assert [tuple(int(v) for v in it) for it in got] == _brute_force_items(cu, 64, is_global)


def test_attention_plan_rejects_bad_input(built_lib):
    for cu in ([1, 5], [0, 5, 5], [0, 7, 3]):
        rc, _ = _plan_attention(built_lib, cu, 64, False)
        assert rc == binding.TEE_EINVAL, cu
    rc, _ = _plan_attention(built_lib, [0, 5], -1, False)
    assert rc == binding.TEE_EINVAL
    assert built_lib.tee_plan_attention(None, 1, 64, 0, None, 0) == binding.TEE_EINVAL
    cu = np.array([0, 300], dtype=np.int32)
    assert built_lib.tee_plan_attention(cu.ctypes.data, 0, 64, 0, None, 0) == binding.TEE_EINVAL
    rc, _ = _plan_attention(built_lib, cu, 64, False, max_items=2)   # 3 tiles of 128 queries
    assert rc == binding.TEE_ETOOLONG
    assert built_lib.tee_last_error(None).decode() != ""


def _schedule(lib, items, n_heads, grid):
    items = np.ascontiguousarray(np.asarray(items, dtype=np.int32).reshape(-1, 4))
    n = len(items)
    slots = np.full((max(n * n_heads, 1), 4), -7, dtype=np.int32)
    off = np.full(grid + 1, -7, dtype=np.int32)
    rc = lib.tee_plan_attention_schedule(items.ctypes.data if n else None, n, n_heads, grid, slots.ctypes.data,
                                         off.ctypes.data)
    return rc, slots[:max(rc, 0)], off


def _brute_force_schedule(items, n_heads, grid):
    """The rule restated: units (item, head) in order of decreasing work
    (2 * key tiles + 1, ties in unit order), each to the CTA with the least work
    so far (ties to the lower index, found by a linear scan); per CTA in the
    order taken."""
    work = [2 * ((it[3] - it[2] + 127) // 128) + 1 for it in items]
    units = sorted(range(len(items) * n_heads), key=lambda u: -work[u // n_heads])
    load = [0] * grid
    taken = [[] for _ in range(grid)]
    for u in units:
        c = min(range(grid), key=lambda k: (load[k], k))
        load[c] += work[u // n_heads]
        it = items[u // n_heads]
        taken[c].append((it[0], it[1] | (u % n_heads) << 16, it[2], it[3]))
    return taken, load


def _cta_lists(slots, off):
    return [[tuple(int(v) for v in s) for s in slots[off[c]:off[c + 1]]] for c in range(len(off) - 1)]


@pytest.mark.parametrize("lengths,n_heads,grid", [([300, 8, 1000, 64], 12, 5), ([129] * 5, 3, 7), ([1], 12, 152),
                                                  ([2, 1, 3], 1, 1), ([700, 40, 40, 900, 5], 12, 152)])
@pytest.mark.parametrize("is_global", [False, True])
def test_attention_schedule_matches_brute_force(built_lib, lengths, n_heads, grid, is_global):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    _, items = _plan_attention(built_lib, cu, 64, is_global)
    rc, slots, off = _schedule(built_lib, items, n_heads, grid)
    assert rc == len(items) * n_heads
    want, _ = _brute_force_schedule([tuple(int(v) for v in it) for it in items], n_heads, grid)
    assert off[0] == 0 and off[-1] == rc and np.all(np.diff(off) >= 0)
    assert _cta_lists(slots, off) == want


def test_attention_schedule_balances_the_sweep_batch(built_lib):
    """Every (item, head) unit exactly once, fields intact; on the global layers
    of a 32768-token sweep batch the busiest of 152 CTAs holds at most one unit's
    work more than the mean, where round robin over the unit order was ~10%
    over it."""
    from text_embedding_encoder_gb300 import synth
    _, cu = synth.sweep_batch(32768, 0, 1000)
    n_heads, grid = 12, 152
    for is_global in (True, False):
        _, items = _plan_attention(built_lib, np.asarray(cu, dtype=np.int32), 64, is_global)
        rc, slots, off = _schedule(built_lib, items, n_heads, grid)
        assert rc == len(items) * n_heads
        heads = slots[:, 1] >> 16
        fields = np.stack([slots[:, 0], slots[:, 1] & 0xFFFF, slots[:, 2], slots[:, 3]], axis=1)
        got = sorted((tuple(int(v) for v in f), int(h)) for f, h in zip(fields, heads))
        want = sorted((tuple(int(v) for v in it), h) for it in items for h in range(n_heads))
        assert got == want
        work = 2 * ((slots[:, 3] - slots[:, 2] + 127) // 128) + 1
        load = np.array([work[off[c]:off[c + 1]].sum() for c in range(grid)])
        assert load.max() <= load.mean() + work.max()
        if is_global:
            rr = np.repeat(2 * ((items[:, 3] - items[:, 2] + 127) // 128) + 1, n_heads)
            rr_load = np.array([rr[c::grid].sum() for c in range(grid)])
            assert load.max() < rr_load.max()


def test_attention_schedule_rejects_bad_input(built_lib):
    items = np.array([[0, 5, 0, 5]], dtype=np.int32)
    out = np.zeros((16, 4), dtype=np.int32)
    off = np.zeros(2000, dtype=np.int32)
    f = built_lib.tee_plan_attention_schedule
    assert f(items.ctypes.data, 1, 0, 4, out.ctypes.data, off.ctypes.data) == binding.TEE_EINVAL
    assert f(items.ctypes.data, 1, 12, 0, out.ctypes.data, off.ctypes.data) == binding.TEE_EINVAL
    assert f(items.ctypes.data, 1, 12, 1025, out.ctypes.data, off.ctypes.data) == binding.TEE_EINVAL
    assert f(None, 1, 12, 4, out.ctypes.data, off.ctypes.data) == binding.TEE_EINVAL
    assert f(items.ctypes.data, 1, 12, 4, None, off.ctypes.data) == binding.TEE_EINVAL
    bad = np.array([[0, 70000, 0, 5]], dtype=np.int32)
    assert f(bad.ctypes.data, 1, 12, 4, out.ctypes.data, off.ctypes.data) == binding.TEE_EINVAL
    assert built_lib.tee_last_error(None).decode() != ""


def _plan_gemm(lib, M, N, K, epi, sms=152):
    bn, pair = ctypes.c_int(-1), ctypes.c_int(-1)
    rc = lib.tee_plan_gemm(M, N, K, epi, sms, ctypes.byref(bn), ctypes.byref(pair))
    return rc, bn.value, pair.value


# epilogues: 0 bf16 store, 1 fp32 residual add, 2 QKV + RoPE, 3 GeGLU
H, I = 768, 3072


@pytest.mark.parametrize("M,N,K,epi,want", [
    # QKV and Wi: CTA pairs on 256-column tiles from two row tiles on
    (32768, 3 * H, H, 2, (256, 1)), (2048, 3 * H, H, 2, (256, 1)), (100, 3 * H, H, 2, (256, 0)),
    (32768, 2 * I, H, 3, (256, 1)), (129, 2 * I, H, 3, (256, 1)),
    # attention out-projection (short K, single CTAs): 32768 rows: 192 columns
    # take 7 waves x 192 = 1344 column-waves against 11 x 128 = 1408; 24000
    # rows: 5 x 192 = 960 < 8 x 128 = 1024; 2048 rows: 1 wave either way, so
    # 128; 8192 / 16384 / 65536 rows: ties (384, 768, 2688), so 128
    (32768, H, H, 1, (192, 0)), (24000, H, H, 1, (192, 0)), (2048, H, H, 1, (128, 0)),
    (8192, H, H, 1, (128, 0)), (16384, H, H, 1, (128, 0)), (65536, H, H, 1, (128, 0)),
    # FFN out-projection (long K): cost = waves x width x {single 128: 1.05,
    # pairs 256: 0.87, pairs 192: 1.0}; 32768 rows: 1478.4 / 1336.3 / 1344;
    # 8192: 403.2 / 445.4 / 384; 2048: 134.4 / 222.7 / 192; 20000: 940.8 / 890.9 / 960
    (32768, H, I, 1, (256, 1)), (8192, H, I, 1, (192, 1)), (2048, H, I, 1, (128, 0)), (20000, H, I, 1, (256, 1)),
    # N = 384 (128 and 192 divide it, 256 does not); 9728 rows = 76 row tiles:
    # 152 tiles of 192 columns fill one wave, 228 of 128 columns two
    (1000, 384, 192, 0, (128, 1)), (1000, 384, 192, 1, (128, 0)), (9728, 384, 192, 1, (192, 0)),
    (100, 384, 192, 1, (128, 0)),
])
def test_gemm_tile_choices(built_lib, M, N, K, epi, want):
    rc, bn, pair = _plan_gemm(built_lib, M, N, K, epi)
    assert rc == binding.TEE_OK
    assert (bn, pair) == want


def test_gemm_tile_invariants(built_lib):
    for M in (1, 127, 128, 255, 256, 1051, 4096, 30000, 65536):
        for N in (128, 256, 384, 768, 2304, 6144):
            for K in (64, 768, 1024, 1088, 3072):
                for epi in range(4):
                    if epi == 3 and N % 256:
                        continue
                    rc, bn, pair = _plan_gemm(built_lib, M, N, K, epi)
                    assert rc == binding.TEE_OK
                    assert bn in (128, 192, 256) and N % bn == 0
                    assert pair in (0, 1)
                    if pair:
                        assert (M + 127) // 128 >= 2
                    if epi != 1:
                        assert bn != 192
                    if epi == 3:
                        assert bn == 256


def test_gemm_plan_rejects_bad_shapes(built_lib):
    for args in ((0, 768, 768, 0), (64, 100, 768, 0), (64, 768, 100, 0), (64, 384, 768, 3), (64, 768, 768, 4)):
        rc, _, _ = _plan_gemm(built_lib, *args)
        assert rc == binding.TEE_EINVAL, args
    rc, _, _ = _plan_gemm(built_lib, 64, 768, 768, 0, sms=1)
    assert rc == binding.TEE_EINVAL
