"""CPU tests of the C ABI: the library loads, exports every function the
header declares, rejects bad arguments with the documented codes (host-only
validation, nothing launched), and its decision model reproduces the worked
numbers of the CS336 Lecture 05 notes."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

from complexity_matmul_tcgen05_gb300 import fgemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "cs336_quantization_examples.json")


@pytest.fixture(scope="module")
def L():
    from complexity_matmul_tcgen05_gb300 import build
    build.build()
    return fgemm.lib()


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fgemm_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_function(L):
    names = _declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n


def test_create_without_device_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    h = ctypes.c_void_p()
    assert L.fgemm_create(ctypes.byref(h)) == fgemm.ERR_NO_DEVICE
    assert h.value is None
    assert L.fgemm_destroy(None) == fgemm.OK


def test_status_strings(L):
    for s in range(8):
        assert fgemm.status_string(s).startswith("FGEMM_")


def _v(M, N, K, A=16, lda=None, B=16, ldb=None, C=16, ldc=None, dtype=fgemm.BF16,
       epi=None, algo="auto", tile=0, tile_m=0):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    n_out = N // 2 if (epi is not None and epi.kind == 3) else N
    ldc = n_out if ldc is None else ldc
    return fgemm.validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, epi, algo, tile, tile_m)


def test_validation_codes(L):
    ok = fgemm.OK
    assert _v(256, 256, 256) == ok
    assert _v(0, 256, 256, A=0, B=0, C=0) == ok                    # empty: nothing to do
    assert _v(8, 16, 0, A=0, B=0) == ok                            # K = 0: C = epi(bias)
    assert _v(8, 16, 64, A=0) == fgemm.ERR_INVALID_ARG             # NULL A
    assert _v(8, 16, 64, lda=32) == fgemm.ERR_INVALID_ARG          # lda < K
    assert _v(8, 16, 64, ldb=8) == fgemm.ERR_INVALID_ARG           # ldb < N
    assert _v(8, 16, 64, ldc=8) == fgemm.ERR_INVALID_ARG           # ldc < N
    assert _v(-1, 16, 64) == fgemm.ERR_INVALID_ARG
    assert _v(8, 16, 64, A=18) == fgemm.ERR_ALIGNMENT              # A not 16-byte aligned
    assert _v(8, 16, 64, C=24) == fgemm.ERR_ALIGNMENT
    assert _v(8, 16, 60, lda=60) == fgemm.ERR_ALIGNMENT            # 120-byte rows
    assert _v(8, 16, 64, dtype=7) == fgemm.ERR_INVALID_ARG
    assert _v(8, 16, 64, algo="classical", tile=96) == fgemm.ERR_INVALID_ARG
    sb = fgemm.make_epilogue("scale_bias", 1.0, None)
    assert _v(8, 16, 64, epi=sb) == fgemm.ERR_INVALID_ARG          # SCALE_BIAS without bias
    sw = fgemm.make_epilogue("swiglu", 1.0, None)
    assert _v(8, 24, 64, epi=sw) == fgemm.ERR_ALIGNMENT            # up half at column 12
    assert _v(8, 32, 64, epi=sw) == ok
    assert _v(8, 32, 64, epi=sw, algo="classical", tile=64) == fgemm.ERR_UNSUPPORTED
    # Strassen legality: 2^d blocks of whole 128 x tile_n x 64 tiles
    assert _v(256, 256, 128, algo="strassen1", tile=128) == ok
    assert _v(256, 256, 128, algo="strassen1", tile=256) == fgemm.ERR_UNSUPPORTED
    assert _v(384, 256, 128, algo="strassen1") == fgemm.ERR_UNSUPPORTED
    assert _v(256, 256, 96, lda=96, algo="strassen1") == fgemm.ERR_UNSUPPORTED
    assert _v(512, 512, 256, algo="strassen2", tile=128) == ok
    assert _v(256, 512, 256, algo="strassen2") == fgemm.ERR_UNSUPPORTED
    # CTA-pair tiles: 256 x {128, 256}, classical and one or two Strassen levels
    assert _v(512, 512, 256, tile_m=256, tile=128) == ok
    assert _v(512, 512, 256, tile_m=256, tile=64) == fgemm.ERR_UNSUPPORTED
    assert _v(512, 512, 256, algo="strassen1", tile_m=256) == ok
    assert _v(256, 512, 256, algo="strassen1", tile_m=256) == fgemm.ERR_UNSUPPORTED  # 2 x 256 rows
    assert _v(1024, 1024, 512, algo="strassen2", tile_m=256) == ok   # 4 x 256 rows, 4 x 256 columns
    assert _v(512, 1024, 512, algo="strassen2", tile_m=256) == fgemm.ERR_UNSUPPORTED
    assert _v(1024, 1024, 128, algo="strassen2", tile_m=256) == fgemm.ERR_UNSUPPORTED  # K / 4 < 64
    assert _v(4 * 8 * 65536, 1024, 1024, algo="strassen2", tile_m=256) == fgemm.ERR_UNSUPPORTED  # pre-pass grid
    assert _v(1024, 2048, 512, algo="strassen2", tile_m=256,
              epi=fgemm.make_epilogue("swiglu", 1.0, None)) == fgemm.ERR_UNSUPPORTED
    assert _v(512, 512, 256, tile_m=192) == fgemm.ERR_INVALID_ARG
    assert _v(100, 512, 256, tile_m=256) == ok                     # ragged rows are fine


def test_swiglu_odd_n_rejected(L):
    sw = fgemm.make_epilogue("swiglu", 1.0, None)
    assert fgemm.validate(8, 31, 64, 16, 64, 16, 32, 16, 16, fgemm.BF16, sw, "auto", 0) == \
        fgemm.ERR_INVALID_ARG


# ------------------------------------------------ decision model geometry

def _model(L, sms=152, peak=2250.0, bw=7900.0):
    m = fgemm.DeviceModel()
    L.fgemm_model_default(ctypes.byref(m), sms, peak, bw)
    return m


def test_tile_quantization_page_example(L):
    g = json.load(open(GOLDEN))["tile_quantization"]
    T = g["tile"]
    for n, tiles in g["cases"]:
        assert L.fgemm_model_tiles(n, T, T, T) == tiles          # one dimension
        assert L.fgemm_model_tiles(n, n, T, T) == tiles * tiles  # square


def test_wave_quantization_page_example(L):
    g = json.load(open(GOLDEN))["wave_quantization"]
    for c in g["cases"]:
        tiles = L.fgemm_model_tiles(c["n"], c["n"], g["tile_m"], g["tile_n"])
        assert tiles == c["tiles"] == c["tiles_m"] * c["tiles_n"]
        tail = ctypes.c_double()
        waves = L.fgemm_model_waves(tiles, g["sms"], ctypes.byref(tail))
        assert waves == c["waves"]
        if "tail_tiles" in c:
            assert abs(tail.value - c["tail_tiles"] / g["sms"]) < 1e-12
            assert abs(tail.value - c["tail_utilization"]) < 1e-4


def test_tiled_reads_page_formula(L):
    g = json.load(open(GOLDEN))["tiled_reads"]
    for c in g["cases"]:
        n, t = c["n"], c["t"]
        assert L.fgemm_model_tiled_reads(n, n, n, t, t) == 2 * n ** 3 / t
        # the untiled limit (T = 1) reads 2 N^3 elements
        assert L.fgemm_model_tiled_reads(n, n, n, 1, 1) == 2 * n ** 3


def test_roofline_page_examples(L):
    g = json.load(open(GOLDEN))["roofline"]
    for c in g["cases"]:
        got = L.fgemm_model_roofline(c["flops"], c["bytes"], c["peak_flops"], c["bw"])
        assert abs(got - c["perf"]) <= 1e-9 * c["perf"]
    r = json.load(open(GOLDEN))["relu_bytes_per_flop"]
    # ReLU: 1 FLOP per element, read + write of the element
    for bytes_per_elem, key in ((4, "fp32"), (2, "fp16")):
        perf = L.fgemm_model_roofline(1.0, 2.0 * bytes_per_elem, 1e30, 1.0)
        assert abs(1.0 / perf - r[key]) < 1e-12


def _predict(L, m, M, N, K, algo, tile, epi=0, tile_m=128):
    us = ctypes.c_double()
    s = L.fgemm_model_predict(ctypes.byref(m), M, N, K, epi, fgemm.ALGOS[algo], tile_m, tile,
                              ctypes.byref(us))
    return s, us.value


def test_model_wave_sawtooth_and_monotonicity(L):
    m = _model(L)
    # one more tile than the SM count costs a whole extra wave
    s1, t1 = _predict(L, m, 128 * 152, 256, 4096, "classical", 256)
    s2, t2 = _predict(L, m, 128 * 153, 256, 4096, "classical", 256)
    assert s1 == s2 == fgemm.OK
    assert t2 > 1.8 * (t1 - m.launch_us)
    # more K never predicts less time
    prev = 0
    for K in (512, 1024, 2048, 4096):
        _, t = _predict(L, m, 4096, 4096, K, "classical", 256)
        assert t >= prev
        prev = t


def test_model_strassen_tradeoffs(L):
    m = _model(L)
    # illegal shapes are reported, never predicted
    assert _predict(L, m, 384, 256, 128, "strassen1", 128)[0] == fgemm.ERR_UNSUPPORTED
    # with equal efficiencies and ample L2 bandwidth the 7/8 work wins at
    # large compute-bound sizes
    m.l2_gbs = 1e9
    m.eff_strassen[0][1] = m.eff_classical[2]
    _, tc = _predict(L, m, 16384, 16384, 16384, "classical", 256)
    _, ts = _predict(L, m, 16384, 16384, 16384, "strassen1", 256)
    assert ts < tc
    # and loses when its mainloop is much slower
    m.eff_strassen[0][1] = 0.5 * m.eff_classical[2]
    m.eff_strassen[0][0] = 0.5 * m.eff_classical[1]
    _, ts = _predict(L, m, 16384, 16384, 16384, "strassen1", 256)
    assert ts > tc
    a = ctypes.c_int()
    tm, tn, us = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
    assert L.fgemm_model_plan(ctypes.byref(m), 16384, 16384, 16384, 0, ctypes.byref(a),
                              ctypes.byref(tm), ctypes.byref(tn), ctypes.byref(us)) == fgemm.OK
    assert fgemm.ALGO_NAMES[a.value] == "classical"


def test_model_operand_traffic_term(L):
    # with scarce L2 bandwidth, narrow tiles (which re-read A more often,
    # tiled reads ~ (128 + tile_n) / (128 * tile_n)) predict more time
    m = _model(L)
    m.l2_gbs = 2000.0
    _, t64 = _predict(L, m, 8192, 8192, 8192, "classical", 64)
    _, t256 = _predict(L, m, 8192, 8192, 8192, "classical", 256)
    assert t64 > 1.5 * t256
    # and Strassen's extra source terms (24 vs 16 per 2x2 block) cost more
    m.eff_strassen[0][1] = m.eff_classical[2]
    _, tc = _predict(L, m, 16384, 16384, 16384, "classical", 256)
    _, ts = _predict(L, m, 16384, 16384, 16384, "strassen1", 256)
    assert ts > tc


def test_model_plan_small_shapes_stay_classical(L):
    m = _model(L)
    a = ctypes.c_int()
    tm, tn, us = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
    for (M, N, K) in [(16, 2048, 2048), (128, 4096, 4096), (256, 256, 256), (1000, 1000, 1000)]:
        assert L.fgemm_model_plan(ctypes.byref(m), M, N, K, 0, ctypes.byref(a), ctypes.byref(tm),
                                  ctypes.byref(tn), ctypes.byref(us)) == fgemm.OK
        assert fgemm.ALGO_NAMES[a.value] == "classical"
        assert tm.value in (16, 32, 64, 128, 256) and tn.value in (64, 128, 256)
        assert tm.value >= 128 or M <= tm.value   # the small-M tiles only where M fits


def test_model_pair_tiles_fix_wave_quantization(L):
    # 4096^2 output: 512 tiles of 128x256 on 152 SMs is 3.37 waves (the last
    # runs 56 SMs); 512 pair tiles of 256x128 on 76 pairs is 6.74 waves.
    m = _model(L)
    m.eff_classical[2] = m.eff_pair[0] = 0.8
    _, t_single = _predict(L, m, 4096, 4096, 4096, "classical", 256)
    _, t_pair = _predict(L, m, 4096, 4096, 4096, "classical", 128, tile_m=256)
    assert t_pair < t_single
    tail = ctypes.c_double()
    assert L.fgemm_model_waves(L.fgemm_model_tiles(4096, 4096, 128, 256), 152, ctypes.byref(tail)) == 4
    assert L.fgemm_model_waves(L.fgemm_model_tiles(4096, 4096, 256, 128), 76, ctypes.byref(tail)) == 7


# ----------------------------------------------------------- K-split schedule

def _split(L, tiles, clusters, kb, mode=2, m=None):
    pieces = ctypes.c_int32()
    r = L.fgemm_model_split_tail(None if m is None else ctypes.byref(m), tiles, clusters, kb, 256,
                                 mode, ctypes.byref(pieces))
    return r, pieces.value


@pytest.mark.parametrize("tiles,clusters,kb", [
    (256, 76, 64),    # 4096^2 in 256x256 pair tiles on 76 pairs, K = 4096: R = 28, S = 2
    (1024, 76, 128),  # 8192^3: R = 36, S = 2
    (77, 76, 76),     # one tail tile: S capped at 4
    (96, 76, 64),     # R = 20: S = 3
    (64, 76, 32),     # R = 64 > 76/2: no split
    (10, 76, 1),      # one K block: a piece needs at least one
    (5, 3, 7),        # R = 2 > 3/2: no split
    (13, 4, 3),       # R = 1, S = min(4, 3) = 3
    (200, 7, 9),      # R = 4 > 7/2: no split
])
def test_split_schedule_covers_every_k_block_once(L, tiles, clusters, kb):
    split, pieces = _split(L, tiles, clusters, kb)
    rem = tiles % clusters
    if rem == 0 or 2 * rem > clusters or min(clusters // rem, kb, 4) < 2:
        assert (split, pieces) == (0, 1)
    else:
        assert split == rem and pieces == min(clusters // rem, kb, 4)
        assert split * pieces <= clusters
    sched = [fgemm.split_work_items(tiles, split, pieces, clusters, kb, c) for c in range(clusters)]
    seen = {}
    for c, items in enumerate(sched):
        for n, (unit, k0, k1, piece, npieces) in enumerate(items):
            assert 0 <= unit < tiles and 0 <= k0 < k1 <= kb
            if unit >= split:
                assert (k0, k1, piece, npieces) == (0, kb, 0, 1)
                assert (unit - split) % clusters == c
            else:  # a piece: the pair's first item, pair = tile * S + piece
                assert n == 0 and npieces == pieces and c == unit * pieces + piece
            for k in range(k0, k1):
                assert (unit, k) not in seen, (unit, k)
                seen[(unit, k)] = piece
    assert len(seen) == tiles * kb
    # the pieces of a split tile are numbered 0.. in K order
    for t in range(split):
        order = [seen[(t, k)] for k in range(kb)]
        assert order == sorted(order) and order[0] == 0 and order[-1] == pieces - 1
    # every pair runs the same whole tiles count; the split adds at most one
    # piece of ceil(kb / S) K blocks
    work = [sum(k1 - k0 for (_, k0, k1, _, _) in items) for items in sched]
    whole = (tiles - split) // clusters * kb
    assert all(whole <= w <= whole + (kb + pieces - 1) // pieces for w in work) if split else True


def test_split_rule(L):
    m = _model(L)
    # 4096^3 + bias: 256 pair tiles on 76 pairs, the last wave 28/76 busy
    assert _split(L, 256, 76, 64, 1, m) == (28, 2)
    assert _split(L, 256, 76, 64, 0, m) == (0, 1)
    # full waves: nothing to split
    assert _split(L, 152, 76, 64, 2) == (0, 1)
    # a short K makes the saved time smaller than the split's cost
    assert _split(L, 256, 76, 2, 1, m) == (0, 1)
    m.split_fix_us = 1e9
    assert _split(L, 256, 76, 64, 1, m) == (0, 1)
    # invalid cluster counts are never split
    assert _split(L, 256, 1, 64, 2) == (0, 1)
    assert _split(L, 1000, 300, 64, 2) == (0, 1)


def test_model_split_removes_the_pair_sawtooth(L):
    # 77 pair tiles on 76 pairs: whole waves cost two tile times; split, the
    # one extra tile runs as 4 pieces on 4 pairs: 1 + 1/4 tile times
    m = _model(L)
    m.hbm_gbs = 1e9  # compute-bound: the sawtooth is in the compute term
    _, t76 = _predict(L, m, 256 * 76, 256, 8192, "classical", 256, tile_m=256)
    _, t77 = _predict(L, m, 256 * 77, 256, 8192, "classical", 256, tile_m=256)
    fixed = m.launch_us + m.tile_fill_us   # once per launch
    t_tile = t76 - fixed
    assert abs(t77 - (fixed + 1.25 * t_tile + 3 * m.split_fix_us)) < 1e-6 * t77
    m.split_fix_us = 1e9  # split never pays: back to the whole-wave sawtooth
    _, t77w = _predict(L, m, 256 * 77, 256, 8192, "classical", 256, tile_m=256)
    assert abs(t77w - (fixed + 2 * t_tile)) < 1e-6 * t77w
    assert t77 < 0.8 * t77w


def test_winograd_legality_and_model(L):
    # one level on single-CTA tiles of 128 x {128, 256} and on CTA pairs of
    # 256 x {128, 256} (whole tiles in every block), never 64 wide
    ep = fgemm.make_epilogue("none")
    ok = lambda M, N, K, tm, tn: fgemm.validate(M, N, K, 16, K, 16, N, 16, N, fgemm.BF16, ep,
                                                "winograd1", tn, tm)
    assert ok(512, 512, 256, 128, 128) == fgemm.OK
    assert ok(512, 1024, 256, 128, 256) == fgemm.OK
    assert ok(512, 512, 256, 256, 256) == fgemm.OK                 # one pair tile per block
    assert ok(512, 768, 256, 256, 256) == fgemm.ERR_UNSUPPORTED    # 384-column blocks
    assert ok(768, 512, 256, 256, 128) == fgemm.ERR_UNSUPPORTED    # 384-row blocks
    assert ok(512, 512, 256, 128, 64) == fgemm.ERR_UNSUPPORTED
    assert ok(384, 512, 256, 128, 128) == fgemm.ERR_UNSUPPORTED   # 192-row blocks
    m = _model(L)
    s, tw = _predict(L, m, 16384, 16384, 16384, "winograd1", 256)
    assert s == fgemm.OK and tw > 0
    s, twp = _predict(L, m, 16384, 16384, 16384, "winograd1", 256, tile_m=256)
    assert s == fgemm.OK and twp > 0
    # with the Strassen mainloop rate, the extra source terms (14 + 14 vs
    # 12 + 12) make it predict no faster than Strassen-1
    m.eff_winograd[1] = m.eff_strassen[0][1]
    _, ts = _predict(L, m, 16384, 16384, 16384, "strassen1", 256)
    _, tw = _predict(L, m, 16384, 16384, 16384, "winograd1", 256)
    assert tw >= ts


# ------------------------------------------------------- small-M stream-K

@pytest.mark.parametrize("tiles,kb,ctas", [
    (128, 256, 152),   # 16 x 16384 x 16384: 128 column tiles, K = 16384
    (16, 32, 152),     # 16 x 2048 x 2048
    (64, 128, 152),    # 16 x 8192 x 8192
    (1, 1, 1),
    (3, 5, 7),         # fewer iterations per CTA than one tile
    (200, 3, 152),     # more tiles than CTAs, short K
    (1, 400, 152),     # one tile over every CTA
    # the grids fgemm_small_m_grid picks on 152 SMs
    (128, 256, 128),   # 16 x 16384^2: one whole tile per CTA
    (64, 128, 128),    # 16 x 8192^2: half a tile per CTA
    (96, 192, 144),    # 16 x 12288^2: 2/3 of a tile per CTA
    (32, 256, 128),    # 16 x 4096 x 16384: a quarter tile per CTA
    (224, 64, 128),    # 16 x 28672 x 4096: 1.75 tiles per CTA
])
def test_stream_k_schedule_covers_and_slots_are_unique(L, tiles, kb, ctas):
    ctas = min(ctas, tiles * kb)
    seen = {}
    slots = {}
    counters = {}
    per_cta = []
    for c in range(ctas):
        items = fgemm.stream_k_work_items(tiles, kb, ctas, c)
        per_cta.append(sum(k1 - k0 for (_, k0, k1, _, _, _) in items))
        for n, (unit, k0, k1, piece, npieces, slot) in enumerate(items):
            assert 0 <= unit < tiles and 0 <= k0 < k1 <= kb
            for k in range(k0, k1):
                assert (unit, k) not in seen
                seen[(unit, k)] = (c, piece, npieces)
            if npieces == 1:
                assert (k0, k1) == (0, kb)
                continue
            # only a CTA's first and last items are pieces of a shared tile
            assert n == 0 or n == len(items) - 1
            assert 0 <= slot < 2 * ctas and slot // 2 == c
            assert slot not in slots, "two pieces share a partial slot"
            slots[slot] = (unit, piece)
            if piece == 0:
                assert unit not in counters
                counters[unit] = slot
    assert len(seen) == tiles * kb
    assert max(per_cta) - min(per_cta) <= 1   # equal shares
    for t in range(tiles):
        pieces = [seen[(t, k)][1] for k in range(kb)]
        assert pieces == sorted(pieces) and pieces[0] == 0
        n = seen[(t, 0)][2]
        assert pieces[-1] == n - 1
        if n > 1:
            assert t in counters


def test_small_m_legality_and_model(L):
    ep = fgemm.make_epilogue("none")
    ok = lambda M, N, K, tm, tn, epi=ep: fgemm.validate(M, N, K, 16, K, 16, N, 16, N, fgemm.BF16, epi,
                                                        "classical", tn, tm)
    assert ok(16, 4096, 4096, 16, 128) == fgemm.OK
    assert ok(7, 1000, 520, 16, 128) == fgemm.OK
    assert ok(17, 4096, 4096, 16, 128) == fgemm.ERR_UNSUPPORTED      # M > tile_m
    assert ok(16, 4096, 4096, 16, 256) == fgemm.ERR_UNSUPPORTED      # 128-column tiles only
    assert ok(64, 4096, 4096, 64, 128, fgemm.make_epilogue("swiglu")) == fgemm.ERR_UNSUPPORTED
    assert fgemm.validate(16, 4096, 4096, 16, 4096, 16, 4096, 16, 4096, fgemm.BF16, ep,
                          "strassen1", 128, 16) == fgemm.ERR_UNSUPPORTED
    m = _model(L)
    # 16 x 16384 x 16384 streams 512 MiB of B on 128 CTAs of one whole tile
    # each (every share starts at K offset 0): the aligned rate, plus the
    # fixed cost and the launch
    _, t_small = _predict(L, m, 16, 16384, 16384, "classical", 128, tile_m=16)
    b = 2.0 * (16 * 16384 + 16384 * 16384 + 16 * 16384)
    stream_us = b / (m.hbm_gbs * 1e3 * m.small_m_aligned_eff)
    assert abs(t_small - (stream_us + m.small_m_fix_us + m.launch_us)) < 1e-6 * t_small
    # 16 x 20480 x 8128: 160 tiles of 127 K blocks; of 114..152 CTAs only 127
    # divides the 20320 iterations, and its shares start at 127 offsets, so
    # every SM streams at the misaligned rate
    assert fgemm.small_m_grid(160, 127, 152) == (152, 152)
    _, t_mis = _predict(L, m, 16, 20480, 8128, "classical", 128, tile_m=16)
    b = 2.0 * (16 * 8128 + 8128 * 20480 + 16 * 20480)
    stream_us = b / (m.hbm_gbs * 1e3 * m.small_m_stream_eff)
    assert abs(t_mis - (stream_us + m.small_m_fix_us + m.launch_us)) < 1e-6 * t_mis
    # and AUTO takes the small-M form for 16 x 16384^2
    a = ctypes.c_int()
    tm, tn, us = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
    assert L.fgemm_model_plan(ctypes.byref(m), 16, 16384, 16384, 0, ctypes.byref(a), ctypes.byref(tm),
                              ctypes.byref(tn), ctypes.byref(us)) == fgemm.OK
    assert (fgemm.ALGO_NAMES[a.value], tm.value, tn.value) == ("classical", 16, 128)
    # 16 x 8192 x 8192 as 128 x 64 tiles keeps 128 of 152 SMs streaming: the
    # small-M form, on every SM, predicts less
    _, t_small = _predict(L, m, 16, 8192, 8192, "classical", 128, tile_m=16)
    _, t_wide = _predict(L, m, 16, 8192, 8192, "classical", 64, tile_m=128)
    assert t_small < t_wide


@pytest.mark.parametrize("tiles,kb,sms,want", [
    (128, 256, 152, (128, 1)),   # 16 x 16384^2: one whole tile per CTA
    (64, 128, 152, (128, 2)),    # 16 x 8192^2: half a tile per CTA, shares start at 0 or 64
    (96, 192, 152, (144, 3)),    # 16 x 12288^2: 2/3 of a tile, shares start at 0, 128, 64
    (32, 256, 152, (128, 4)),    # 16 x 4096 x 16384: a quarter tile
    (128, 64, 152, (128, 1)),    # 16 x 16384 x 4096
    (16, 32, 152, (64, 4)),      # 16 x 2048^2: 512 iterations, at most 64 CTAs of 8 blocks
    (1, 1, 152, (1, 1)),         # one block
])
def test_small_m_grid_picks(tiles, kb, sms, want):
    assert fgemm.small_m_grid(tiles, kb, sms) == want


def test_small_m_grid_invariants():
    rng = np.random.default_rng(7)
    for _ in range(400):
        tiles = int(rng.integers(1, 400))
        kb = int(rng.integers(1, 600))
        sms = int(rng.choice([8, 76, 132, 148, 152]))
        ctas, phases = fgemm.small_m_grid(tiles, kb, sms)
        iters = tiles * kb
        most = max(1, min(sms, -(-iters // 8)))
        assert 1 <= ctas <= most
        if phases <= 4:
            assert iters % ctas == 0 and ctas >= -(-most * 3 // 4)
            share = iters // ctas
            starts = {(i * share) % kb for i in range(ctas)}   # brute force
            assert phases == len(starts)
            # no grid in range with fewer phases (ties go to the larger grid)
            for c in range(-(-most * 3 // 4), most + 1):
                if iters % c == 0:
                    other = len({(i * (iters // c)) % kb for i in range(c)})
                    assert other > phases or (other == phases and c <= ctas)
        else:
            assert ctas == most and phases == most
    assert fgemm.small_m_grid(0, 4, 152) == (0, 0)


# ------------------------------------------------- calibration files (host)

def _flat(m):
    """Every number of a device model, by field name."""
    out = {}
    for name, ct in fgemm.DeviceModel._fields_:
        v = getattr(m, name)
        if hasattr(v, "__len__"):
            flat = np.array([list(x) if hasattr(x, "__len__") else x for x in v], dtype=float).ravel()
            for i, x in enumerate(flat):
                out[f"{name}[{i}]"] = float(x)
        else:
            out[name] = float(v)
    return out


def test_model_json_round_trip(L, tmp_path):
    m = _model(L)
    m.eff_pair[1] = 0.777
    m.launch_us = 3.25
    m.small_m_fix_us = 5.5
    m.eff_strassen[1][0] = 0.0123
    path = str(tmp_path / "calib.json").encode()
    assert L.fgemm_model_save_json(ctypes.byref(m), path) == fgemm.OK
    d = json.load(open(path))                     # valid JSON, one key per field
    assert d["eff_pair_256"] == 0.777 and d["launch_us"] == 3.25 and d["num_sms"] == 152
    assert d["eff_strassen2_128"] == 0.0123 and d["small_m_fix_us"] == 5.5
    m2 = _model(L, sms=100, peak=1.0, bw=1.0)     # everything different before the load
    assert L.fgemm_model_load_json(path, ctypes.byref(m2)) == fgemm.OK
    a, b = _flat(m), _flat(m2)
    for k in a:
        if k != "reserved":
            assert abs(a[k] - b[k]) <= 1e-8 * max(1.0, abs(a[k])), k


def test_model_json_measured_peaks_change_only_the_denominators(L, tmp_path):
    # a file of measured peaks (the format the driver's peak measurement
    # writes): the peak and bandwidth become the denominators, the efficiencies
    # are rescaled, and every predicted time stays the same
    m = _model(L)
    shapes = [(16384, 16384, 16384, "classical", 256, 256), (4096, 4096, 4096, "classical", 128, 128),
              (16, 16384, 16384, "classical", 16, 128), (8192, 8192, 8192, "strassen1", 256, 256),
              (8192, 8192, 8192, "strassen2", 128, 256)]
    before = [_predict(L, m, M, N, K, a, tn, tile_m=tm)[1] for (M, N, K, a, tm, tn) in shapes]
    path = tmp_path / "peaks.json"
    path.write_text(json.dumps({"hbm_gbs": 6000.0, "bf16_tflops": 1700.0,
                                "bf16_tflops_sustained": 1600.0, "gpu_name": "NVIDIA GB300"}))
    assert L.fgemm_model_load_json(str(path).encode(), ctypes.byref(m)) == fgemm.OK
    assert m.peak_tflops == 1700.0 and m.hbm_gbs == 6000.0
    after = [_predict(L, m, M, N, K, a, tn, tile_m=tm)[1] for (M, N, K, a, tm, tn) in shapes]
    for b, a in zip(before, after):
        assert abs(a - b) <= 1e-9 * b


def test_model_json_rejects_bad_files_and_keeps_the_model(L, tmp_path):
    m = _model(L)
    ref = _flat(m)
    cases = {"garbage.json": "this is not a calibration", "negative.json": '{"peak_tflops": -5}',
             "zero_bw.json": '{"hbm_gbs": 0}', "neg_launch.json": '{"launch_us": -1.0}',
             "empty.json": "{}"}
    for name, text in cases.items():
        p = tmp_path / name
        p.write_text(text)
        assert L.fgemm_model_load_json(str(p).encode(), ctypes.byref(m)) == fgemm.ERR_CALIBRATION, name
        assert _flat(m) == ref, name
    assert L.fgemm_model_load_json(str(tmp_path / "missing.json").encode(), ctypes.byref(m)) == \
        fgemm.ERR_CALIBRATION
    assert L.fgemm_model_load_json(None, ctypes.byref(m)) == fgemm.ERR_INVALID_ARG
    assert _flat(m) == ref


def test_model_in_kernel_formation_term(L):
    """One Winograd level on CTA pairs: with at least 16 waves of its two
    sum-free products the model charges the in-kernel formation (its drag,
    and what outlasts the first three products) instead of the pre-pass;
    Strassen's scheme, which has no sum-free product, keeps the pre-pass."""
    m = _model(L)
    m.eff_strassen_pair[1] = m.eff_pair[1] * 7.0 / 8.0  # products at the classical rate

    def parts(n, algo):
        s, t = _predict(L, m, n, n, n, algo, 256, tile_m=256)
        assert s == fgemm.OK
        return t

    def with_formation(n, eff, drag):
        m.form_in_kernel_eff, m.form_in_kernel_drag = eff, drag
        return parts(n, "winograd1")

    base_eff, base_drag = m.form_in_kernel_eff, m.form_in_kernel_drag
    # 16384^3: 1024 positions on 76 pairs, 13 whole waves: 26 >= 16 -> in-kernel.
    # A free, infinitely fast formation leaves the product time alone...
    t_free = with_formation(16384, 1e9, 0.0)
    # ...drag is charged on the formation's duration...
    t_drag = with_formation(16384, 1e9 / 16384.0, 0.1)
    assert t_drag > t_free
    # ...and a slow formation shows once it outlasts three products' waves
    t_slow = with_formation(16384, 0.01, 0.0)
    assert t_slow > t_free + 1000.0
    m.form_in_kernel_eff, m.form_in_kernel_drag = base_eff, base_drag
    # Strassen at the same size: B's sums in the kernel (its M2 and M5 read
    # none), A's by a pre-pass half the full one; so even a free in-kernel
    # formation leaves the half pre-pass, and a slow one shows
    m.form_in_kernel_eff, m.form_in_kernel_drag = 1e9, 0.0
    ts_free = parts(16384, "strassen1")
    tw_free = parts(16384, "winograd1")
    assert ts_free > tw_free + 50.0   # the A-side pre-pass (1.15 GB at 16384^3)
    m.form_in_kernel_eff = 0.01
    assert parts(16384, "strassen1") > ts_free + 1000.0
    m.form_in_kernel_eff, m.form_in_kernel_drag = base_eff, base_drag
    # 8192^3: 3 whole waves (6 < 16): the pre-pass, whatever the in-kernel rate
    tw = parts(8192, "winograd1")
    m.form_in_kernel_eff = 1e-3
    assert parts(8192, "winograd1") == tw


def test_model_plan_margin_for_low_complexity_forms(L):
    """AUTO takes a low-complexity form only when it beats the best classical
    prediction by lcma_margin."""
    m = _model(L)
    a = ctypes.c_int()
    tm, tn, us = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()

    def pick():
        assert L.fgemm_model_plan(ctypes.byref(m), 32768, 32768, 32768, 0, ctypes.byref(a),
                                  ctypes.byref(tm), ctypes.byref(tn), ctypes.byref(us)) == fgemm.OK
        return fgemm.ALGO_NAMES[a.value], us.value

    _, tc = _predict(L, m, 32768, 32768, 32768, "classical", 256, tile_m=256)
    # Winograd's pair products 5 % faster per MAC than the classical kernel's
    m.eff_strassen_pair[1] = m.eff_pair[1] * 1.05
    _, tw = _predict(L, m, 32768, 32768, 32768, "winograd1", 256, tile_m=256)
    gain = 1.0 - tw / tc
    assert gain > 0.03
    m.lcma_margin = gain + 0.01          # not enough: classical stays
    algo, t = pick()
    assert algo == "classical" and abs(t - tc) < 1e-6 * tc
    m.lcma_margin = gain - 0.01          # enough: the low-complexity form, its own prediction
    algo, t = pick()
    assert algo in ("winograd1", "strassen1") and t <= tw * (1 + 1e-9)


def test_model_operand_dram_term_and_the_large_cube_picks(L):
    """The operand panels' DRAM re-reads: no cost while a wave's panels fit
    the L2 (8192^3), a cost beyond it (24576^3); with it the defaults pick one
    Winograd level on CTA pairs from 20480^3 up (measured 4-5 % ahead from there
    on in long runs) and keep the classical kernel at 12288^3 (12 % behind) and
    16384^3 (2 % ahead, within the margin)."""
    m = _model(L)

    def classical(n):
        return _predict(L, m, n, n, n, "classical", 256, tile_m=256)[1]

    def pick(n):
        a = ctypes.c_int()
        tm, tn, us = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
        assert L.fgemm_model_plan(ctypes.byref(m), n, n, n, 0, ctypes.byref(a), ctypes.byref(tm),
                                  ctypes.byref(tn), ctypes.byref(us)) == fgemm.OK
        return fgemm.ALGO_NAMES[a.value], tm.value, tn.value

    with_term = [classical(n) for n in (8192, 24576)]
    assert pick(12288) == ("classical", 256, 256)
    assert pick(16384) == ("classical", 256, 256)
    assert pick(20480) == ("winograd1", 256, 256)
    assert pick(24576) == ("winograd1", 256, 256)
    assert pick(32768) == ("winograd1", 256, 256)
    exposed = m.dram_exposed
    m.dram_exposed = 0.0
    without = [classical(n) for n in (8192, 24576)]
    assert with_term[0] == without[0]                 # 8192^3: the panels fit
    assert with_term[1] > without[1] * 1.05           # 24576^3: about 1.4 ms of 17
    assert pick(24576)[0] == "classical"              # and without it AUTO stays classical
    m.dram_exposed = exposed


def test_model_two_levels_on_pairs_fold_term_and_picks(L):
    """Two Strassen levels on CTA pairs: each product unit's fold (about
    three fp32 output-block reductions) overlaps its MMAs only in part, so a
    unit costs the longer of the two plus a share of the shorter: the
    prediction grows with the fold time and is at least the fold time per
    unit; with fewer positions than pairs each pair runs one position whole.
    AUTO takes the form on none of the cubes or sweep shapes (it is slower
    than the classical kernel up to 32768^3 and than one Winograd level)."""
    m = _model(L, peak=0.0, bw=0.0)
    n = 16384
    s, base = _predict(L, m, n, n, n, "strassen2", 256, tile_m=256)
    assert s == fgemm.OK
    m.fold2_unit_us = 60.0
    _, slower = _predict(L, m, n, n, n, "strassen2", 256, tile_m=256)
    assert slower > base
    units_per_pair = 3 * 49 + -(-(28 * 49) // 76)  # 256 positions: 3 whole waves + 28 positions as units
    assert slower >= units_per_pair * 60.0
    m.fold2_unit_us = 30.0
    # 4096 x 16384: 64 positions on 76 pairs -> 49 units per pair, no tail
    _, t64 = _predict(L, m, 4096, 16384, 16384, "strassen2", 256, tile_m=256)
    _, t76 = _predict(L, m, 4096, 19456, 16384, "strassen2", 256, tile_m=256)
    assert abs(t64 - t76) < 0.05 * t76
    assert _predict(L, m, 4096, 4096, 4096, "strassen2", 256, epi=3, tile_m=256)[0] == fgemm.ERR_UNSUPPORTED

    def pick(M, N, K):
        a = ctypes.c_int()
        tm, tn, us = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
        assert L.fgemm_model_plan(ctypes.byref(m), M, N, K, 0, ctypes.byref(a), ctypes.byref(tm),
                                  ctypes.byref(tn), ctypes.byref(us)) == fgemm.OK
        return fgemm.ALGO_NAMES[a.value], tm.value

    shapes = [(c, c, c) for c in (4096, 8192, 16384, 24576, 32768, 49152)] + \
        [(M, k, k) for M in (16, 128, 1024, 8192) for k in (2048, 4096, 8192, 16384)]
    for shape in shapes:
        assert pick(*shape)[0] != "strassen2", shape


def test_lcma_pair_clusters(L):
    """Pairs of a Strassen-like launch on CTA pairs: one level every pair that
    has work; two levels one pair per position below the pair count, every
    pair while the partial wave's units stay within 24 per pair, else the
    most pairs (down to half) that divide the positions into whole waves."""
    f = L.fgemm_lcma_pair_clusters
    assert f(0, 1, 76) == 0 and f(10, 2, 0) == 0
    assert f(1, 1, 76) == 7 and f(64, 1, 76) == 76 and f(1024, 1, 76) == 76
    assert f(64, 2, 76) == 64                      # fewer positions than pairs
    assert f(76, 2, 76) == 76 and f(152, 2, 76) == 76
    assert f(256, 2, 76) == 76                     # 28 positions left: 19 units per pair
    assert f(80, 2, 76) == 76                      # 4 positions left: 3 units per pair
    assert f(128, 2, 76) == 64                     # 52 left would be 34 units per pair: 2 waves of 64
    assert f(1024, 2, 76) == 76                    # 36 left: 24 units per pair
    assert f(200, 2, 76) == 50                     # 48 left would be 31 per pair: 4 waves of 50
    assert f(151, 2, 76) == 76                     # 75 left, and no pair count from 38 to 76 divides 151
