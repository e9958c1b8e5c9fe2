"""Host-side checks of the C-ABI library that need no GPU: it builds for
sm_103a, loads, exports every entry point the header declares, validates
arguments before touching a device, and plans tiles as documented."""

import ctypes
import os
import re

import numpy as np
import pytest

from half_precision_dense_gb300 import binding
from half_precision_dense_gb300 import build as hbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hgemm.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    hbuild.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \t\*]*?\b(hgemm_?\w*)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["hgemm", "hgemm_ex", "hgemm_host", "hgemm_plan", "hgemm_tile_coord",
              "hgemm_get_device_status", "hgemm_set_timeout_ns", "hgemm_status_string",
              "hgemm_last_error", "hgemm_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_is_sm103a_only():
    # Every kernel is compiled for sm_103a and nothing else.
    assert hbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version_and_strings(lib):
    assert binding.version() == 200
    for s, frag in [(0, "OK"), (1, "INVALID_ARG"), (2, "UNSUPPORTED_DEVICE"), (5, "TIMEOUT")]:
        assert frag in binding.status_string(s)


@pytest.mark.parametrize("args", [
    (1, 1, 1, -1, 4, 4, 1),     # negative M
    (1, 1, 1, 4, 4, 1 << 31, 1),  # K too large
    (1, 1, 1, 4, 4, 4, 7),      # unknown dtype
    (0, 16, 32, 4, 4, 4, 1),    # null A
    (16, 16, 0, 4, 4, 4, 0),    # null C
    (3, 16, 32, 4, 4, 4, 1),    # odd address
])
def test_invalid_arguments_rejected_without_device(lib, args):
    a, b, c, M, N, K, dt = args
    st = lib.hgemm(a, b, c, M, N, K, dt, None)
    assert st == 1, binding.STATUS_NAMES.get(st)


def test_fp8_blockscaled_arguments_rejected_without_device(lib):
    f = lib.hgemm_fp8_blockscaled
    A, B, C, sa, sb = 1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20
    assert f(A, B, C, sa, sb, 64, 64, 64, 16, 3, None) == 1        # block 16
    assert f(A, B, C, sa, sb, 64, 64, 64, 32, 1, None) == 1        # bf16 is not fp8
    assert f(A, B, C, None, sb, 64, 64, 64, 32, 3, None) == 1      # no a_scale
    assert f(A, B, C, sa, None, 64, 64, 64, 64, 4, None) == 1      # no b_scale
    assert f(A, B, C, sa + 2, sb, 64, 64, 64, 32, 3, None) == 1    # misaligned a_scale
    bad_cfg = binding.Config(block_n=256)._c()
    assert lib.hgemm_fp8_blockscaled_ex(A, B, C, sa, sb, 64, 64, 64, 32, 3, ctypes.byref(bad_cfg), None) == 1
    # empty shapes need no scales
    assert f(None, None, C, None, None, 0, 64, 64, 32, 3, None) == 0
    import torch
    if not torch.cuda.is_available():
        # a well-formed call without a GB300 fails loudly (no CPU fallback)
        assert f(A, B, C, sa, sb, 64, 64, 64, 32, 3, None) == 2


def test_overlap_rejected(lib):
    base = 1 << 20
    # C = [base, base + 2*4*4) overlaps A = [base + 16, ...)
    assert lib.hgemm(base + 16, base + 4096, base, 4, 4, 4, 1, None) == 1


def test_empty_shapes_are_noops(lib):
    assert lib.hgemm(None, None, None, 0, 5, 3, 1, None) == 0
    assert lib.hgemm(None, None, None, 5, 0, 3, 0, None) == 0


def test_no_cpu_fallback(lib):
    # A well-formed call on a machine without a GB300 must fail loudly.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = lib.hgemm(1 << 20, 2 << 20, 3 << 20, 64, 64, 64, 1, None)
    assert st == 2


def test_tile_coord_is_a_bijection(lib):
    for tiles_m, tiles_n, group in [(16, 16, 8), (7, 5, 3), (1, 32, 8), (64, 56, 8), (5, 9, 16)]:
        seen = set()
        for t in range(tiles_m * tiles_n):
            tm, tn = binding.tile_coord(t, tiles_m, tiles_n, group)
            assert 0 <= tm < tiles_m and 0 <= tn < tiles_n
            seen.add((tm, tn))
        assert len(seen) == tiles_m * tiles_n


def test_plan_fills_the_machine_at_4096(lib):
    # 152 SMs: 256-wide pair tiles give 256 tiles, 4 waves on 64 of the 76
    # pairs; 224-wide ones give 16 x 19 = 304 tiles, 4 whole waves on all 76
    # (and a 224-wide pair stage runs at 0.97 of a 256-wide one per flop)
    p = binding.plan(4096, 4096, 4096, "bf16", sm_count=152)
    assert (p["cta_group"], p["block_n"], p["grid_ctas"], p["num_tiles"]) == (2, 224, 152, 304)
    assert p["num_tiles"] % (p["grid_ctas"] // p["cta_group"]) == 0 and p["sk_tiles"] == 0


def test_tile_coord_groups_rows_first(lib):
    # inside a group the row index varies fastest
    coords = [binding.tile_coord(t, 16, 4, 8) for t in range(10)]
    assert coords[:8] == [(r, 0) for r in range(8)]
    assert coords[8:10] == [(0, 1), (1, 1)]


def test_plan_shapes(lib):
    p = binding.plan(4096, 4096, 4096, "bf16", sm_count=148)
    assert p["cta_group"] in (1, 2) and p["block_n"] in (64, 128, 224, 256)
    assert p["tiles_m"] * p["block_m"] >= 4096 and p["tiles_n"] * p["block_n"] >= 4096
    assert p["grid_ctas"] % p["cta_group"] == 0 and p["grid_ctas"] <= 148
    assert p["tmem_cols"] >= 2 * p["block_n"] and p["tmem_cols"] & (p["tmem_cols"] - 1) == 0
    assert p["smem_bytes"] <= 232448 and p["stages"] >= 2
    # aligned C: rows written back from the staging box by 16-byte stores
    assert p["repack_a"] == 0 and p["repack_b"] == 0 and p["store_mode"] == 4
    t = binding.plan(1000, 4095, 4104, "bf16", sm_count=152)
    # an unaligned 16-bit C: realigned 16-byte stores with element stores at
    # the ragged ends; B copied (8190-byte rows), and A too: its 8208-byte rows
    # are an odd multiple of 16 bytes, which slows its loads on 224-wide pair
    # tiles, and N is large
    assert (t["cta_group"], t["block_n"]) == (2, 224)
    assert t["repack_b"] == 1 and t["repack_a"] == 1 and t["store_mode"] == 5
    # that A copy only on 224-wide tiles, where N repays it, only for A, only
    # for odd multiples of 16 bytes
    p = binding.plan(4096, 4096, 4104, "bf16", sm_count=152)
    assert p["block_n"] == 224 and p["repack_a"] == 1
    p = binding.plan(4096, 4096, 4104, "bf16", binding.Config(cta_group=2, block_n=256), sm_count=152)
    assert p["repack_a"] == 0
    assert binding.plan(2048, 2048, 2056, "bf16", sm_count=152)["repack_a"] == 0
    assert binding.plan(4096, 4096, 4112, "bf16", sm_count=152)["repack_a"] == 0
    assert binding.plan(4096, 4104, 4096, "bf16", sm_count=152)["repack_b"] == 0
    forced = binding.plan(512, 512, 512, "f16",
                          binding.Config(cta_group=1, block_n=64, max_clusters=3), sm_count=148)
    assert (forced["cta_group"], forced["block_n"], forced["grid_ctas"]) == (1, 64, 3)
    with pytest.raises(binding.HgemmError):
        binding.plan(512, 512, 512, "f16", binding.Config(cta_group=2, block_n=64), sm_count=148)


def test_plan_stream_k(lib):
    # 4096^3 on 152 SMs with pair tiles: 256 tiles, 76 clusters, 3.37 waves.
    # Two data-parallel waves (152 tiles), then the last 104 tiles' 6656 K
    # blocks in 76 equal ranges of 87 or 88 blocks.
    p = binding.plan(4096, 4096, 4096, "bf16", binding.Config(cta_group=2, block_n=256, stream_k=2),
                     sm_count=152)
    assert (p["num_tiles"], p["dp_tiles"], p["sk_tiles"]) == (256, 152, 104)
    assert (p["sk_blocks"], p["sk_extra"], p["grid_ctas"], p["num_kb"]) == (87, 44, 152, 64)
    assert p["workspace_bytes"] >= 152 * 4 * 32 * 256 * 4
    # stream_k = 1, and the planner's own choice for pair tiles: whole waves
    # only, spread evenly (4 waves of 64 clusters)
    for mode in (1, 0):
        off = binding.plan(4096, 4096, 4096, "bf16",
                           binding.Config(cta_group=2, block_n=256, stream_k=mode), sm_count=152)
        assert (off["sk_tiles"], off["dp_tiles"], off["grid_ctas"], off["workspace_bytes"]) == (0, 256, 128, 0)
    # a single tile row on a long K loop: 128-wide one-CTA tiles, each K loop
    # split over a cluster of two (the planner never picks stream-K)
    sk = binding.plan(128, 8192, 8192, "bf16", sm_count=152)
    assert (sk["cta_group"], sk["block_n"], sk["sk_tiles"], sk["grid_ctas"], sk["split_k"]) == (1, 128, 0, 128, 2)
    # 64 K blocks: still split (32 per CTA); a shorter K loop: the narrowest
    # one-CTA tiles that keep every tile in one wave, whole
    sk = binding.plan(128, 8192, 4096, "bf16", sm_count=152)
    assert (sk["cta_group"], sk["block_n"], sk["sk_tiles"], sk["grid_ctas"], sk["split_k"]) == (1, 128, 0, 128, 2)
    sk = binding.plan(128, 8192, 2048, "bf16", sm_count=152)
    assert (sk["cta_group"], sk["block_n"], sk["sk_tiles"], sk["grid_ctas"], sk["split_k"]) == (1, 64, 0, 128, 1)
    wide = binding.plan(128, 16384, 8192, "bf16", sm_count=152)
    assert (wide["cta_group"], wide["block_n"], wide["sk_tiles"]) == (1, 128, 0)
    # whole waves leave nothing to share; one K block leaves nothing to cut
    even = binding.plan(128 * 76, 256, 4096, "bf16", binding.Config(cta_group=1, block_n=256), sm_count=76)
    assert even["sk_tiles"] == 0 and even["grid_ctas"] == 76
    short = binding.plan(4096, 4096, 64, "bf16", binding.Config(cta_group=2, block_n=256), sm_count=152)
    assert short["sk_tiles"] == 0
    # mode 4: three whole waves of 76, then only the 28 leftover tiles' 1792
    # K blocks, 23 or 24 per cluster
    left = binding.plan(4096, 4096, 4096, "bf16", binding.Config(cta_group=2, block_n=256, stream_k=4),
                        sm_count=152)
    assert (left["dp_tiles"], left["sk_tiles"], left["sk_blocks"], left["sk_extra"]) == (228, 28, 23, 44)
    assert left["grid_ctas"] == 152
    # mode 3 shares every tile
    every = binding.plan(1024, 1024, 1024, "f16",
                         binding.Config(cta_group=1, block_n=128, stream_k=3), sm_count=20)
    assert every["sk_tiles"] == every["num_tiles"] and every["dp_tiles"] == 0


def _check_schedule(p):
    clusters = p["grid_ctas"] // (p["cta_group"] * p["split_k"])
    kb = p["num_kb"]
    seen = {}
    units_of = {}
    for c in range(clusters):
        units = binding.work_units(p, c)
        units_of[c] = units
        for i, (tile, kb0, kb1, kind) in enumerate(units):
            assert 0 <= tile < p["num_tiles"] and 0 <= kb0 < kb1 <= kb
            for k in range(kb0, kb1):
                assert (tile, k) not in seen, "K block computed twice"
                seen[(tile, k)] = (c, i, kind)
            if tile < p["dp_tiles"]:
                assert (kb0, kb1, kind) == (0, kb, 0) and tile % clusters == c
            if kind == 0:
                assert (kb0, kb1) == (0, kb)
            if kind == 1:
                assert kb0 == 0 and kb1 < kb and i == len(units) - 1  # owner: last unit, holds block 0
            if kind == 2:
                assert kb0 > 0
                ndp = sum(1 for u in units if u[0] < p["dp_tiles"])
                assert i == ndp  # a non-owning part is the first stream-K unit: it never waits
    assert len(seen) == p["num_tiles"] * kb, "some K block never computed"
    for tile in range(p["num_tiles"]):
        holders = sorted({seen[(tile, k)][0] for k in range(kb)})
        kinds = {seen[(tile, k)][2] for k in range(kb)}
        if len(holders) == 1:
            assert kinds == {0}
        else:
            owner = seen[(tile, 0)][0]
            assert seen[(tile, 0)][2] == 1 and owner == holders[0]
            # every partner of the owner is a later cluster, in one contiguous run
            assert holders == list(range(owner, owner + len(holders)))
            for c in holders[1:]:
                assert all(seen[(tile, k)][2] == 2 for k in range(kb) if seen[(tile, k)][0] == c)


@pytest.mark.parametrize("shape,cfg,sms", [
    ((4096, 4096, 4096), dict(cta_group=2, block_n=256), 152),
    ((8192, 8192, 8192), dict(), 152),
    ((128, 8192, 8192), dict(), 152),
    ((1000, 4095, 4104), dict(), 152),
    ((1024, 1280, 704), dict(cta_group=1, block_n=128, max_clusters=3, stream_k=2), 152),
    ((1024, 1280, 704), dict(cta_group=2, block_n=224, max_clusters=5, stream_k=3), 152),
    ((300, 700, 130), dict(cta_group=1, block_n=64, stream_k=3), 152),
    ((777, 999, 4444), dict(stream_k=2), 37),
    ((4096, 4096, 4096), dict(cta_group=2, block_n=256, stream_k=4), 152),
    ((1024, 1280, 704), dict(cta_group=1, block_n=128, max_clusters=7, stream_k=4), 152),
    ((128, 8192, 8192), dict(split_k=4), 152),
    ((300, 1000, 704), dict(block_n=128, split_k=2), 152),
])
def test_schedule_covers_every_block_once_without_wait_cycles(lib, shape, cfg, sms):
    p = binding.plan(*shape, "bf16", binding.Config(**cfg), sm_count=sms)
    _check_schedule(p)


def test_plan_split_k_clusters(lib):
    # split_k: a cluster of 2, 4 or 8 single CTAs per tile, one tile per cluster
    p = binding.plan(128, 8192, 8192, "bf16", binding.Config(split_k=4), sm_count=152)
    assert (p["cta_group"], p["block_m"], p["block_n"], p["split_k"], p["multicast"]) == (1, 128, 256, 4, 1)
    assert (p["tiles_m"], p["tiles_n"], p["num_tiles"], p["grid_ctas"]) == (1, 32, 32, 128)
    assert (p["sk_tiles"], p["workspace_bytes"]) == (0, 0)   # partial sums stay on chip
    q = binding.plan(200, 1000, 300, "f16", binding.Config(block_n=128, split_k=2), sm_count=152)
    assert (q["tiles_m"], q["tiles_n"], q["grid_ctas"]) == (2, 8, 32)
    for c in range(q["grid_ctas"] // 2):
        assert binding.work_units(q, c) == [(c, 0, 5, 0)]   # the whole K range; the CTAs share it
    # the combinations that are not built, and too many tiles for one cluster each
    for cfg, dt, shape in [(dict(split_k=3), "bf16", (128, 1024, 1024)),
                           (dict(block_n=128, split_k=8), "bf16", (128, 1024, 1024)),
                           (dict(block_n=64, split_k=2), "bf16", (128, 1024, 1024)),
                           (dict(cta_group=2, block_n=256, split_k=2), "bf16", (128, 1024, 1024)),
                           (dict(split_k=2), "tf32", (128, 1024, 1024)),
                           (dict(split_k=2, stream_k=3), "bf16", (128, 1024, 1024)),
                           (dict(split_k=2), "bf16", (4096, 4096, 4096))]:
        with pytest.raises(binding.HgemmError):
            binding.plan(*shape, dt, binding.Config(**cfg), sm_count=152)


@pytest.mark.parametrize("shape,dtype,split", [
    ((128, 4096, 14336), "bf16", 4),    # 32 tiles x 4 CTAs, 56 K blocks each
    ((128, 2048, 8192), "f16", 4),
    ((1024, 1024, 8192), "bf16", 2),    # 64 tiles: a split of 4 would need 256 SMs
    ((128, 8192, 4096), "bf16", 2),     # 64 K blocks, 32 per CTA
    ((128, 4096, 4096), "bf16", 4),     # 32 tiles x 4 CTAs, 16 K blocks each
    ((128, 8192, 2048), "bf16", 1),     # 32 K blocks: too short a loop to split
    ((8192, 8192, 8192), "bf16", 1),    # enough tiles already
    ((128, 4096, 14336), "tf32", 1),    # 16-bit kinds only
    ((128, 4096, 14336), "e4m3", 1),
])
def test_plan_auto_split(lib, shape, dtype, split):
    p = binding.plan(*shape, dtype, sm_count=152)
    assert p["split_k"] == split
    if split > 1:
        assert (p["cta_group"], p["block_n"]) == (1, 128)
        assert p["grid_ctas"] == p["num_tiles"] * split <= 152
    # a forced shape keeps whole tiles unless the split is asked for
    assert binding.plan(*shape, dtype, binding.Config(cta_group=1, block_n=128), sm_count=152)["split_k"] == 1


@pytest.mark.parametrize("n", [0, 1, 3, 7, 8, 63, 64, 127, 128, 224, 1001])
@pytest.mark.parametrize("parts", [2, 4, 8])
def test_split_share_partitions_the_k_range(lib, n, parts):
    # the K split's shares (the kernel's own function): contiguous, in rank
    # order, covering [kb0, kb1) exactly, sizes equal to within one block;
    # with fewer blocks than CTAs some shares are empty (those CTAs add zeros)
    kb0 = 5
    shares = [binding.split_share(kb0, kb0 + n, r, parts) for r in range(parts)]
    assert shares[0][0] == kb0 and shares[-1][1] == kb0 + n
    for (lo, hi), (lo2, _) in zip(shares, shares[1:]):
        assert lo <= hi == lo2
    sizes = [hi - lo for lo, hi in shares]
    assert max(sizes) - min(sizes) <= 1 and sum(sizes) == n
    # out-of-range ranks and sizes leave the outputs untouched
    assert binding.split_share(0, 10, parts, parts) == (-1, -1)
    assert binding.split_share(0, 10, 0, 0) == (-1, -1)
    assert binding.split_share(10, 0, 0, parts) == (-1, -1)


@pytest.mark.parametrize("shape,store_mode,tile", [
    ((4096, 4096, 64), 1, (1, 256)),      # one K block per tile: the epilogue sets the pace
    ((8192, 8192, 64), 1, (1, 256)),      # single CTAs beat pairs on short K loops
    ((8192, 8192, 256), 1, (2, 256)),     # 16-warp pair tiles
    ((16384, 16384, 64), 1, (1, 256)),
    ((8192, 8192, 512), 1, (2, 256)),
    ((4096, 4096, 512), 1, (2, 224)),     # 8 blocks: still TMA stores
    ((4096, 4096, 576), 4, (2, 224)),     # 9 blocks: row stores
    ((4096, 4096, 4096), 4, (2, 224)),
])
def test_plan_short_k_uses_tma_stores(lib, shape, store_mode, tile):
    p = binding.plan(*shape, "bf16", sm_count=152)
    assert p["store_mode"] == store_mode and (p["cta_group"], p["block_n"]) == tile
    # an unaligned 16-bit C takes the realigned stores; a forced mode is kept
    assert binding.plan(shape[0], shape[1] + 1, shape[2], "bf16", sm_count=152)["store_mode"] == 5
    assert binding.plan(*shape, "bf16", binding.Config(store_mode=3), sm_count=152)["store_mode"] == 3


@pytest.mark.parametrize("shape,dtype,epi", [
    ((4096, 4096, 64), "bf16", 16),       # single 256-wide tiles, one K block
    ((8192, 8192, 256), "f16", 16),
    ((16384, 16384, 64), "bf16", 16),
    ((8192, 8192, 512), "bf16", 16),      # pair tiles
    ((4096, 4096, 4096), "bf16", 16),     # a long K loop
    ((128, 8192, 8192), "bf16", 8),       # a K split
    ((1024, 1024, 1024), "bf16", 8),      # 64-wide tiles
    ((4096, 4096, 64), "tf32", 8),        # fp32 C
    ((4096, 4096, 128), "fp8_e4m3", 16),  # fp8 writes a bf16 C
    ((4096, 4096, 4096), "fp8_e5m2", 16),
    ((128, 8192, 8192), "fp8_e4m3", 8),   # 64-wide tiles
])
def test_plan_epilogue_warps(lib, shape, dtype, epi):
    assert binding.plan(*shape, dtype, sm_count=152)["epi_warps"] == epi


def test_plan_epilogue_warps_forced(lib):
    one = binding.Config(cta_group=1, block_n=256)
    assert binding.plan(4096, 4096, 4096, "bf16", binding.Config(cta_group=1, block_n=256, epi_warps=16),
                        sm_count=152)["epi_warps"] == 16
    assert binding.plan(4096, 4096, 64, "bf16", binding.Config(epi_warps=8), sm_count=152)["epi_warps"] == 8
    assert binding.plan(4096, 4096, 64, "bf16", one, sm_count=152)["epi_warps"] == 16
    assert binding.plan(4096, 4096, 64, "bf16", binding.Config(cta_group=2, block_n=224, epi_warps=16),
                        sm_count=152)["epi_warps"] == 16
    for bad in (binding.Config(cta_group=2, block_n=128, epi_warps=16),      # 128-wide pair tiles
                binding.Config(cta_group=1, block_n=128, epi_warps=16),      # 128-wide tiles
                binding.Config(cta_group=1, block_n=256, epi_warps=12),      # not 8 or 16
                binding.Config(cta_group=1, block_n=256, stream_k=3, epi_warps=16)):
        with pytest.raises(binding.HgemmError):
            binding.plan(4096, 4096, 64, "bf16", bad, sm_count=152)
    with pytest.raises(binding.HgemmError):
        binding.plan(4096, 4096, 64, "tf32", binding.Config(cta_group=1, block_n=256, epi_warps=16), sm_count=152)
    assert binding.plan(4096, 4096, 64, "fp8_e4m3", binding.Config(cta_group=2, block_n=224, epi_warps=16),
                        sm_count=152)["epi_warps"] == 16
    with pytest.raises(binding.HgemmError):
        binding.plan(128, 8192, 8192, "bf16", binding.Config(cta_group=1, block_n=256, split_k=2, epi_warps=16),
                     sm_count=152)
    # stream-K leaves the planner's default at 8
    assert binding.plan(4096, 4096, 64, "bf16", binding.Config(cta_group=1, block_n=256, stream_k=3),
                        sm_count=152)["epi_warps"] == 8


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32", "fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("sms", [152, 148, 132, 64])
def test_every_planned_kernel_is_compiled(lib, dtype, sms):
    """The planner refuses a configuration whose kernel instance is not
    compiled; none of its own choices may be refused, over shapes from one
    tile to the projection GEMMs (skinny, short K, ragged, long K)."""
    dims = [1, 100, 128, 129, 1000, 2048, 4095, 4096, 8192, 16384]
    ks = [1, 64, 100, 512, 4096, 4104, 14336]
    for M in dims:
        for N in dims[::2]:
            for K in ks:
                p = binding.plan(M, N, K, dtype, sm_count=sms)
                assert p["epi_warps"] in (8, 16)


def test_plan_refuses_a_kernel_that_is_not_compiled(lib):
    # 16 epilogue warps exist for fp8's 224-wide pair tile but not for a
    # 128-wide one; the K split exists for 128- and 256-wide single tiles only
    binding.plan(4096, 4096, 4096, "fp8_e4m3", binding.Config(cta_group=2, block_n=224, epi_warps=16), sm_count=152)
    with pytest.raises(binding.HgemmError):
        binding.plan(4096, 4096, 4096, "fp8_e4m3", binding.Config(cta_group=2, block_n=128, epi_warps=16),
                     sm_count=152)
    with pytest.raises(binding.HgemmError):
        binding.plan(128, 4096, 4096, "bf16", binding.Config(cta_group=1, block_n=64, split_k=2), sm_count=152)


def test_plan_skinny_prefers_narrow_tiles(lib):
    p = binding.plan(128, 8192, 8192, "bf16", sm_count=148)
    assert p["block_m"] == 128  # one tile row: no half-empty CTA pairs


# --- the epilogue's shared-memory staging layout, modelled on the CPU -------

def bank_of(byte_addr):
    return (byte_addr // 4) % 32


def test_page_swizzle_c_example_is_conflict_free():
    """The page's SWIZZLE_C worked example: warp 0's 32 lanes write 4 bytes each
    to 32 distinct banks of the 128-wide half-precision tile."""
    rows = {}
    for ln in open(os.path.join(GOLDEN, "swizzle_c_warp0.txt"), encoding="utf-8"):
        if ln.strip() and not ln.startswith("#"):
            k, *vals = ln.split()
            rows[k] = [int(v) for v in vals]
    banks = []
    for r, c in zip(rows["row"], rows["col"]):
        sc = c ^ ((r & 7) << 3)
        banks.append(bank_of((r * 128 + sc) * 2))
    assert sorted(banks) == list(range(32))
    unswizzled = {bank_of((r * 128 + c) * 2) for r, c in zip(rows["row"], rows["col"])}
    assert len(unswizzled) < 32  # the 8-way conflict the page describes


def test_epilogue_staging_layout_is_conflict_free_and_tma_compatible():
    """Our staging box: lane l owns row l (128 B); its 16-byte chunk j goes to
    chunk j ^ (l % 8). Each 8-lane phase of a 16-byte store then covers all 32
    banks once, and the layout is exactly the TMA 128-byte swizzle (chunk bits
    4-6 of the address XOR row bits 7-9)."""
    for j in range(8):
        for phase in range(4):
            lanes = range(8 * phase, 8 * phase + 8)
            banks = []
            for l in lanes:
                addr = l * 128 + ((j ^ (l & 7)) << 4)
                banks.extend(bank_of(addr + 4 * w) for w in range(4))
            assert sorted(banks) == list(range(32))
    for l in range(32):
        for j in range(8):
            addr = l * 128 + ((j ^ (l & 7)) << 4)
            logical = l * 128 + j * 16
            tma = logical ^ (((logical >> 7) & 7) << 4)
            assert addr == tma


@pytest.mark.parametrize("ew,chunk_cols", [(8, 64), (16, 32)])
@pytest.mark.parametrize("bn", [64, 128, 224, 256])
def test_epilogue_chunks_cover_each_tile_column_once(ew, chunk_cols, bn):
    """The epilogue's work split, as the kernel computes it: warp w takes TMEM
    lane quarter w % 4 and chunks w // 4, w // 4 + ew // 4, ... of chunk_cols
    columns (a 32-column last chunk when 64-column chunks do not divide the
    tile). Every (quarter, column) of the tile is written by exactly one
    warp, and each warp's last chunk is the one that hands the accumulator
    back."""
    if ew == 16 and bn < 224:
        return  # 16 warps serve the 224- and 256-wide tiles only
    nch = (bn + chunk_cols - 1) // chunk_cols
    groups = ew // 4
    owner = {}
    for w in range(ew):
        quarter, colhalf = w & 3, w >> 2
        mine = list(range(colhalf, nch, groups))
        for c in mine:
            last = c + groups >= nch
            assert last == (c == mine[-1])
            half = chunk_cols == 32 or (bn % 64 != 0 and c == nch - 1)
            width = 32 if half else 64
            for col in range(chunk_cols * c, chunk_cols * c + width):
                if col < bn:
                    assert (quarter, col) not in owner
                    owner[(quarter, col)] = w
    assert len(owner) == 4 * bn


def test_epilogue_32_column_box_is_conflict_free_and_tma_compatible():
    """The 32-column staging box (16 epilogue warps, and the last chunk of a
    224-wide tile): lane l owns row l (64 B); its 16-byte chunk j goes to
    chunk j ^ ((l / 2) % 4). Each 8-lane phase of a 16-byte store covers all
    32 banks once; the layout is the TMA 64-byte swizzle (chunk bits 4-5 of
    the address XOR bits 7-8); and sixteen 2 KB boxes fill the same 32 KB as
    eight 4 KB ones."""
    for j in range(4):
        for phase in range(4):
            banks = []
            for l in range(8 * phase, 8 * phase + 8):
                addr = l * 64 + ((j ^ ((l >> 1) & 3)) << 4)
                banks.extend(bank_of(addr + 4 * w) for w in range(4))
            assert sorted(banks) == list(range(32))
    for l in range(32):
        for j in range(4):
            addr = l * 64 + ((j ^ ((l >> 1) & 3)) << 4)
            logical = l * 64 + j * 16
            assert addr == logical ^ (((logical >> 7) & 3) << 4)
    assert 16 * 32 * 32 * 2 == 8 * 32 * 64 * 2


def test_plan_tf32(lib):
    # fp32 operands: 32 K values per 128-byte stage row, same tiles and ring
    p = binding.plan(4096, 4096, 4096, "tf32", sm_count=152)
    assert (p["cta_group"], p["block_n"], p["block_k"], p["num_kb"]) == (2, 224, 32, 128)
    assert p["stages"] == binding.plan(4096, 4096, 4096, "bf16", binding.Config(2, 256), sm_count=152)["stages"]
    # K = 1001 floats is not a 16-byte pitch: A is repacked; N = 1024 is
    assert binding.plan(64, 1024, 1001, "tf32", sm_count=152)["repack_a"] == 1
    # B is read in place (MN-major), unless its pitch is not 16-byte aligned
    tp = binding.plan(64, 1024, 1001, "tf32", sm_count=152)
    assert tp["repack_b"] == 0
    assert binding.plan(4096, 4096, 4096, "tf32", sm_count=152)["workspace_bytes"] == 0
    assert binding.plan(64, 1022, 1024, "tf32", sm_count=152)["repack_b"] == 1
    assert binding.plan(64, 1024, 1000, "tf32", sm_count=152)["repack_a"] == 0
    # no operand multicast is built: the field is reserved (0 or 1), for every dtype
    for dt in ("bf16", "f16", "tf32", "e4m3"):
        with pytest.raises(binding.HgemmError):
            binding.plan(1024, 1024, 1024, dt, binding.Config(cta_group=2, block_n=256, multicast=2), sm_count=152)
        assert binding.plan(1024, 1024, 1024, dt, binding.Config(multicast=1), sm_count=152)["multicast"] == 1
    # an unknown dtype code is refused by the library itself
    out = binding._Plan()
    assert lib.hgemm_plan(64, 64, 64, 5, None, 152, ctypes.byref(out)) == 1


def test_plan_fp8(lib):
    # 8-bit operands: 128 K values per 128-byte stage row; B read in place
    for code in (binding.HGEMM_E4M3, binding.HGEMM_E5M2):
        p = binding.plan(4096, 4096, 4096, code, sm_count=152)
        # the 256-wide pair tile (the 224-wide one, which fills 8-bit B atoms
        # badly, only when a config asks for it)
        assert (p["cta_group"], p["block_n"], p["block_k"], p["num_kb"]) == (2, 256, 128, 32)
        # B is read MN-major from the caller's matrix: no copy, no workspace
        assert p["repack_b"] == 0 and p["workspace_bytes"] == 0
    # N = 1000 bytes is not a 16-byte pitch: B is repacked
    assert binding.plan(64, 1000, 1024, "e4m3", sm_count=152)["repack_b"] == 1
    # K = 1000 bytes is not a 16-byte pitch (A repacked); 1008 is
    assert binding.plan(64, 1024, 1000, "e4m3", sm_count=152)["repack_a"] == 1
    assert binding.plan(64, 1024, 1008, "e4m3", sm_count=152)["repack_a"] == 0
    # C is bf16: N = 1004 gives a 2008-byte pitch, not a multiple of 16 -> realigned stores
    assert binding.plan(64, 1004, 1024, "e5m2", sm_count=152)["store_mode"] == 5
    # fp32 C (tf32) with an unaligned pitch keeps plain stores; mode 5 is for 16-bit C only
    assert binding.plan(64, 1001, 1024, "tf32", sm_count=152)["store_mode"] == 2
    with pytest.raises(binding.HgemmError):
        binding.plan(64, 1024, 1024, "tf32", binding.Config(store_mode=5), sm_count=152)
    # on an unaligned 16-bit C only the element and realigned modes are accepted
    for mode in (1, 3, 4):
        with pytest.raises(binding.HgemmError):
            binding.plan(64, 1001, 1024, "bf16", binding.Config(store_mode=mode), sm_count=152)
    assert binding.plan(64, 1001, 1024, "bf16", binding.Config(store_mode=2), sm_count=152)["store_mode"] == 2
    # every dtype takes the 224-wide pair tile (its last chunk is 32 columns)
    for dt in ("tf32", "e4m3", "e5m2", "bf16", "f16"):
        assert binding.plan(1024, 1024, 1024, dt, binding.Config(cta_group=2, block_n=224),
                            sm_count=152)["block_n"] == 224
    with pytest.raises(binding.HgemmError):
        binding.plan(1024, 1024, 1024, "tf32", binding.Config(cta_group=1, block_n=224), sm_count=152)
    # the fp8 entry point refuses other dtypes
    assert lib.hgemm_fp8(None, None, None, None, None, 0, 0, 0, 1, None) == 1


# --- the K split's reduction layout, modelled on the CPU ---------------------

SPLIT_SHAPES = [(128, 2), (128, 4), (256, 2), (256, 4), (256, 8)]


def _split_slot(q, r, col, bn, parts):
    """Owner CTA and byte offset in its ring of sender q's partial sum for tile
    row r, columns col..col+3 (the kernel's push): owner col // S, block q of
    128 rows x S floats, 16-byte unit u of row r at unit u ^ (r % 8)."""
    s = bn // parts
    u = (col % s) // 4
    return col // s, q * 128 * s * 4 + r * s * 4 + ((u ^ (r & 7)) << 4)


def _repack_model(src, src_addr, rows, row_bytes, dst_pitch, batch=8):
    """The operand copy (repack_rows_kernel) on the CPU, as the kernel issues
    it: a warp per pass of kPassSegs = 32 * batch 16-byte segments of a row;
    lane l loads the aligned source blocks t0 + 32q + l (t <= nseg, nothing
    at or past the end of the source), lane 31 also block t0 + kPassSegs,
    and each segment t < nseg is bytes [off, off + 16) of block t followed by
    block t + 1, taken from the next lane, the next batch's lane 0, or lane
    31's extra block. src_addr is the device address of src[0]."""
    pass_segs = 32 * batch
    end = src_addr + rows * row_bytes
    nseg = (row_bytes + 15) // 16
    passes = (row_bytes + 16 * pass_segs - 1) // (16 * pass_segs)
    dst = bytearray(rows * dst_pitch)
    loads = []
    def block(addr):
        if addr >= end:
            return bytes(16)
        loads.append(addr)
        # bytes outside the source (before its start or past its end, inside
        # the same aligned block) are not the copy's: model them as 0
        return bytes(src[a - src_addr] if 0 <= a - src_addr < len(src) else 0 for a in range(addr, addr + 16))
    for r in range(rows):
        row = src_addr + r * row_bytes
        off = row & 15
        base = row - off
        for ps in range(passes):
            t0 = ps * pass_segs
            v = [[block(base + 16 * (t0 + 32 * q + l)) if t0 + 32 * q + l <= nseg else bytes(16) for l in range(32)]
                 for q in range(batch)]
            tx = t0 + pass_segs
            x = block(base + 16 * tx) if off != 0 and tx <= nseg else bytes(16)
            for q in range(batch):
                for l in range(32):
                    t = t0 + 32 * q + l
                    if t >= nseg:
                        continue
                    if off == 0:
                        seg = v[q][l]
                    else:
                        hi = v[q][l + 1] if l < 31 else (v[q + 1][0] if q + 1 < batch else x)
                        seg = (v[q][l] + hi)[off:off + 16]
                    dst[r * dst_pitch + 16 * t: r * dst_pitch + 16 * t + 16] = seg
    return dst, loads


@pytest.mark.parametrize("row_bytes", [1, 2, 15, 16, 17, 100, 4095, 4096, 4097, 8190, 8208])
def test_operand_copy_model_reproduces_every_row(row_bytes):
    """The operand copy on the CPU, for every misalignment of the source and
    rows whose pitch drifts across 16-byte boundaries (one and several passes
    per row): each row of the destination starts with the source row, and no
    load touches a 16-byte block at or past the source's end."""
    rows = 5
    pitch = -(-row_bytes // 128) * 128
    rng = np.random.default_rng(row_bytes)
    src = rng.integers(0, 256, rows * row_bytes + 32, dtype=np.uint8).tobytes()
    for mis in range(16):
        addr = 4096 + mis
        body = src[:rows * row_bytes]
        dst, loads = _repack_model(body, addr, rows, row_bytes, pitch)
        for r in range(rows):
            assert dst[r * pitch:r * pitch + row_bytes] == body[r * row_bytes:(r + 1) * row_bytes], (mis, r)
        end = addr + rows * row_bytes
        assert all(a % 16 == 0 and addr - (addr & 15) <= a < end for a in loads)

@pytest.mark.parametrize("cpieces", [1, 2, 3, 4, 5, 8, 16, 31, 32, 33, 64])
@pytest.mark.parametrize("warps", [1, 3, 8])
def test_im2col_lane_split_writes_each_piece_once(cpieces, warps):
    """The vector im2col's work split on the CPU: a warp takes `group`
    (row, tap) segments at once when a tap has fewer than 32 16-byte pieces
    (lane = segment within the group, piece), else one segment with its lanes
    striding over the pieces; the padding columns are one more segment per
    row. Every piece of every segment is written exactly once, by any number
    of warps in the grid."""
    rows, taps, pad_pieces = 7, 9, 3
    segs = taps + 1
    total = rows * segs
    group = 1 if cpieces >= 32 else 32 // cpieces
    step = 32 if cpieces >= 32 else cpieces
    seen = {}
    for wid in range(warps):
        for lane in range(32):
            sub = 0 if cpieces >= 32 else lane // cpieces
            sl = lane if cpieces >= 32 else lane - sub * cpieces
            g0 = wid * group
            while g0 < total:
                g = g0 + sub
                if sub < group and g < total:
                    m, seg = divmod(g, segs)
                    n_pieces = pad_pieces if seg == taps else cpieces
                    for j in range(sl, n_pieces, step):
                        seen[(m, seg, j)] = seen.get((m, seg, j), 0) + 1
                g0 += warps * group
    want = {(m, seg, j) for m in range(rows) for seg in range(segs)
            for j in range(pad_pieces if seg == taps else cpieces)}
    assert set(seen) == want
    assert all(v == 1 for v in seen.values())

def _realigned_store_model(half, o, nvalid, rows=32):
    """The realigned stores of a staged chunk (store mode 5), as the kernel
    issues them: one 16-byte box chunk g of row rr per piece, the aligned
    16-byte segment that ends in it shifted into place from chunks g - 1 and
    g, and element stores for a row's head and tail. Returns per row the
    element writes {element: [values]} and the vector stores' byte offsets
    from the row start (the row starts o bytes past a 16-byte boundary)."""
    nseg = 4 if half else 8
    nel = 8 * nseg
    val = lambda rr, e: (rr << 8) | e
    def box_bytes(rr):
        sw = ((rr >> 1) & 3) if half else (rr & 7)
        b = bytearray(64 if half else 128)
        for e in range(nel):
            a = (((e >> 3) ^ sw) << 4) + ((e & 7) << 1)
            b[a:a + 2] = val(rr, e).to_bytes(2, "little")
        return b, sw
    writes = {rr: {} for rr in range(rows)}
    vec = {rr: [] for rr in range(rows)}
    for piece in range(32 * nseg):
        rr, g = piece // nseg, piece % nseg
        if rr >= rows:
            continue
        brow, sw = box_bytes(rr)
        chunk = lambda j: bytes(brow[((j ^ sw) << 4):((j ^ sw) << 4) + 16])
        elems = lambda sixteen: [int.from_bytes(sixteen[2 * i:2 * i + 2], "little") for i in range(8)]
        def put(e0, sixteen):
            vals = elems(sixteen)
            if e0 + 8 <= nvalid:
                vec[rr].append(o + 2 * e0)
                for i in range(8):
                    writes[rr].setdefault(e0 + i, []).append(vals[i])
            else:
                for e in range(e0, min(nvalid, e0 + 8)):
                    writes[rr].setdefault(e, []).append(vals[e - e0])
        if o == 0:
            put(8 * g, chunk(g))
            continue
        half_o = o >> 1
        if g > 0:
            put(8 * g - half_o, (chunk(g - 1) + chunk(g))[16 - o:32 - o])
        for k in range(g, 8, nseg):
            e = k if k < 8 - half_o else nel - 8 + k
            if e < nvalid:
                ue = e
                a = (((ue >> 3) ^ sw) << 4) + ((ue & 7) << 1)
                writes[rr].setdefault(e, []).append(int.from_bytes(brow[a:a + 2], "little"))
    return writes, vec, val, nel


@pytest.mark.parametrize("half", [False, True])
@pytest.mark.parametrize("o", [0, 2, 4, 6, 8, 10, 12, 14])
def test_realigned_stores_write_each_element_once(half, o):
    """Store mode 5 on the CPU: for every even misalignment of the row start
    and every number of columns left in C, each element of the chunk inside C
    is written exactly once with its own value, nothing past C's last column
    is written, and every 16-byte store is aligned."""
    nel = 32 if half else 64
    for nvalid in list(range(1, nel + 1)) + [nel + 5]:
        writes, vec, val, _ = _realigned_store_model(half, o, nvalid)
        for rr in range(32):
            want = set(range(min(nel, nvalid)))
            assert set(writes[rr]) == want, (o, nvalid, rr)
            for e, vs in writes[rr].items():
                assert vs == [val(rr, e)], (o, nvalid, rr, e, vs)
            assert all(off % 16 == 0 for off in vec[rr]), (o, nvalid, rr)

@pytest.mark.parametrize("bn,parts", SPLIT_SHAPES)
def test_split_reduction_layout_covers_each_owner_block_once(bn, parts):
    s = bn // parts
    slots = {}
    for q in range(parts):
        for r in range(128):
            for col in range(0, bn, 4):
                owner, off = _split_slot(q, r, col, bn, parts)
                assert 0 <= off < parts * 128 * s * 4 and off % 16 == 0
                assert (owner, off) not in slots, "two partial sums in one slot"
                slots[(owner, off)] = (q, r, col)
    # every owner's region (parts blocks of 128 x S floats) is filled exactly
    for owner in range(parts):
        offs = sorted(off for (o, off) in slots if o == owner)
        assert offs == list(range(0, parts * 128 * s * 4, 16))
        # an owner receives only its own columns
        assert all(slots[(owner, off)][2] // s == owner for off in offs)
    # the region fits the ring of the split's tile (7 stages of 32 KiB for
    # 128-wide tiles, 4 of 48 KiB for 256-wide ones)
    ring = 7 * 32768 if bn == 128 else 4 * 49152
    assert parts * 128 * s * 4 <= ring


@pytest.mark.parametrize("bn,parts", SPLIT_SHAPES)
def test_split_reduction_layout_is_bank_conflict_free(bn, parts):
    s = bn // parts
    # pushes: lane l of a warp holds tile row r0 + l and stores one 16-byte
    # unit of the same columns; each 8-lane phase must cover the 32 banks once
    for r0 in (0, 32, 64, 96):
        for col in range(0, bn, 4):
            for phase in range(4):
                banks = []
                for l in range(8 * phase, 8 * phase + 8):
                    _, off = _split_slot(0, r0 + l, col, bn, parts)
                    banks.extend(bank_of(off + 4 * w) for w in range(4))
                assert sorted(banks) == list(range(32))
    # reads: thread f takes unit f % (S/4) of row f // (S/4) of each block;
    # eight consecutive threads must cover the 32 banks once
    units = s // 4
    for f0 in range(0, 128 * units, 8):
        banks = []
        for f in range(f0, f0 + 8):
            rr, u = f // units, f % units
            off = rr * s * 4 + ((u ^ (rr & 7)) << 4)
            banks.extend(bank_of(off + 4 * w) for w in range(4))
        assert sorted(banks) == list(range(32))
