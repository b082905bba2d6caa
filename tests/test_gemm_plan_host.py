"""Host-side checks of the prefill GEMM's launch plans (no GPU), through qlinear_gemm_plan.

For every shape, type, SM count and cluster capacity below, the plan must be one the kernels
can run, and the split form's work assignment, restated here from the kernels' mapping, must
cover every (row tile, superblock) of the layer exactly once:
* a head (cluster rank r < k) takes superblocks [0, L) of row tile cid k + r;
* the tail (rank k) takes [L, nsb) of the cluster's k tiles, tile after tile;
* weight stages of S superblocks never span two row tiles, and every stage is released by the
  dequantiser warps that read it (4 warps when S = 1, all 8 otherwise);
* the tail's k accumulators sit below the TMEM operand ring, its staging area below its
  receive area, and the receive area below the barriers;
* the clusters fit the SMs and the resident-cluster capacity given.
"""
import pytest

import gguf_weight_only_gb300 as ql
from gguf_weight_only_gb300 import build as qbuild

ROWS = 128
CAPS_GB300 = [76, 46, 36, 28, 23, 15, 15]   # resident clusters of 2..8 CTAs measured on GB300 (152 SMs)
TYPES = (12, 13, 14, 23, 270)
SHAPES = [(1, 4096), (129, 512), (300, 5120), (640, 4096), (1000, 4096), (4096, 4096), (4096, 12288), (5120, 17408),
          (9728, 4096), (10240, 2048), (12288, 4096), (17408, 5120), (200, 768), (256, 256)]
MS = (9, 16, 32, 48, 64, 100, 128, 200, 256, 300, 512)


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return ql.lib()


def split_assignment(plan, N, K):
    """(row tile, superblock) -> CTA, per the kernels' mapping; also checks the per-CTA rules."""
    k, L, tail, S = plan["k"], plan["L"], plan["tail"], plan["S"]
    nsb, T = K // 256, (N + ROWS - 1) // ROWS
    cover = {}
    for bx in range(plan["grid_x"]):
        crank = bx % (k + 1)
        is_tail = crank == k
        tile_c = bx // (k + 1) * k
        kk = min(k, T - tile_c)
        nv = kk * tail if is_tail else (L if crank < kk else 0)
        assert nv % S == 0
        tile_of = (lambda v: tile_c + v // tail) if is_tail else (lambda v: tile_c + crank)
        sb_of = (lambda v: L + v % tail) if is_tail else (lambda v: v)
        releases = {}
        for v in range(nv):
            si, j = v // S, v % S
            first = si * S
            assert tile_of(v) == tile_of(first) and sb_of(v) - j == sb_of(first)   # stage inside one tile
            key = (tile_of(v), sb_of(v))
            assert key not in cover, key
            cover[key] = bx
            if v + 2 >= nv or (v + 2) // S != si:   # the warps of parity v % 2 release stage si
                releases[si] = releases.get(si, 0) + 4
        for si, n in releases.items():
            assert n == (4 if S == 1 else 8), (bx, si, n)
    return cover


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("sms,caps", [(152, CAPS_GB300), (148, [74, 44, 36, 28, 22, 14, 14]), (132, [66, 40, 32, 24, 20, 12, 12]),
                                      (152, None)])
def test_plans_are_runnable_and_cover_the_layer(lib, t, sms, caps):
    for N, K in SHAPES:
        for M in MS:
            plan = ql.gemm_plan(t, N, K, M, sms, caps)
            nsb, T = K // 256, (N + ROWS - 1) // ROWS
            n, k = plan["n_tile"], plan["k"]
            assert n % 16 == 0 and 32 <= n <= 256
            assert plan["smem"] <= 227 * 1024
            assert plan["a_col"] + plan["a_slots"] * 128 <= 512 and plan["a_slots"] >= 2
            assert plan["xk"] in (1, 2, 4) and plan["xk"] * n * 128 <= 64 * 1024   # one x stage
            if k == 0:
                assert plan["grid_x"] == T and plan["grid_y"] == (M + n - 1) // n and plan["cluster"] == 1
                assert plan["recv_off"] <= plan["bar_off"]
                continue
            # the split form
            assert caps is not None, "no split without resident clusters"
            assert 1 <= k <= 2 and M <= n and T % k == 0
            assert plan["cluster"] == k + 1 and plan["grid_y"] == 1
            assert plan["grid_x"] == T // k * (k + 1) <= sms
            assert T // k <= caps[k - 1]
            L, tail, S = plan["L"], plan["tail"], plan["S"]
            assert L >= 1 and tail >= 1 and L + tail == nsb and L % S == 0 and tail % S == 0
            assert max(L, k * tail) < nsb - 1   # saves more than a superblock per CTA
            assert k * n <= plan["a_col"]
            part = ROWS * (n + 4) * 4
            assert k * part <= plan["recv_off"] and plan["recv_off"] % 16 == 0
            assert plan["recv_off"] + part <= plan["bar_off"]
            cover = split_assignment(plan, N, K)
            assert len(cover) == T * nsb


def test_split_needs_few_row_tiles(lib):
    caps = CAPS_GB300
    # pairs where they fit (T <= 76), two heads per tail where 40 clusters of three do (T = 80),
    # none where neither does (T = 96: 48 clusters of three exceed the 46 resident)
    assert ql.gemm_plan(12, 4096, 12288, 32, 152, caps)["k"] == 1
    assert ql.gemm_plan(12, 10240, 4096, 32, 152, caps)["k"] == 2
    assert ql.gemm_plan(12, 12288, 4096, 32, 152, caps)["k"] == 0
    # several token tiles are replaced by one tile of all M tokens when the split pays
    p = ql.gemm_plan(12, 4096, 12288, 128, 152, caps)
    assert p["k"] == 1 and p["n_tile"] == 128
    # M above 256 never splits
    assert ql.gemm_plan(12, 1024, 4096, 300, 152, caps)["k"] == 0


def test_plan_arguments_checked(lib):
    with pytest.raises(ql.QLinearError):
        ql.gemm_plan(7, 128, 256, 32, 152)
    with pytest.raises(ql.QLinearError):
        ql.gemm_plan(12, 128, 300, 32, 152)
    with pytest.raises(ql.QLinearError):
        ql.gemm_plan(12, 128, 256, 32, 0)
