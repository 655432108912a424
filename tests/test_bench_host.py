"""Host-side accounting of bench.py (no GPU): useful flops, executed tensor
flops under the library's default tiling, and the kernel named for each phase.

Executed flops are counted by hand here from the tile grids: 128 x 256 tiles
(one CTA) or 256 x 256 tiles (a 2-SM pair), upper tiles only for the
symmetric products, the spare half pair of an odd tile-row count included.
"""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
import workloads  # noqa: E402


def test_useful_flops_closed_form():
    # k (4 m^2 n + 2 m^3) per matrix, the rows > cols tensor viewed transposed
    fl = bench.flops_by_kind([(6144, 2048)], 5)
    m, n = 2048, 6144
    assert sum(fl.values()) == 5 * (4 * m * m * n + 2 * m ** 3)


def test_executed_flops_even_tile_rows():
    # m = 2048: 16 tile rows -> 8 pairs; 8 column tiles of 256; upper pair tiles
    # 8 + 7 + ... + 1 = 36 of 64 for the symmetric products
    ex = bench.executed_flops_by_kind([(2048, 2048)], 1)
    full = 2 * 2048 * 2048 * 2048
    assert ex["gram"] == full * 36 // 64
    assert ex["a2b"] == full * 36 // 64
    assert ex["bx"] == full


def test_executed_flops_odd_tile_rows():
    # m = 1408: 11 tile rows (odd) -> Gram and A*A on 6 pairs with a spare
    # half: 6 + 5 + ... + 1 = 21 pair tiles = 42 CTA tiles of 128 x 256;
    # B*X on single CTAs: 11 x 8 tiles, exactly m x n
    m, n = 1408, 2048
    ex = bench.executed_flops_by_kind([(m, n)], 1)
    assert ex["gram"] == 2 * 128 * 256 * n * 42
    assert ex["a2b"] == 2 * 128 * 256 * m * 42
    assert ex["bx"] == 2 * m * m * n
    assert bench.gemm_kernel_for("gram", 0, [(m, n)])[0] == "ns_gemm2sm_kernel<gram>"
    assert bench.gemm_kernel_for("a2b", 0, [(m, n)])[0] == "ns_gemm2sm_kernel<a2b>"
    assert bench.gemm_kernel_for("bx", 0, [(m, n)])[0] == "ns_gemm_kernel<bx>"
    # forced single CTAs: A*A rows r take 6 - floor(r / 2) tiles -> 41 tiles
    ex1 = bench.executed_flops_by_kind([(m, n)], 1, 1)
    assert ex1["a2b"] == 2 * 128 * 256 * m * 41
    assert bench.gemm_kernel_for("a2b", 0, [(2048, 8192)])[0] == "ns_gemm2sm_kernel<a2b>"


def test_executed_never_below_useful_for_full_tiles():
    # B*X runs whole tiles over the padded operands: executed >= useful, with
    # equality when m is a multiple of 128 and n a multiple of 256
    for m, rho, _ in workloads.sweep_points():
        shape = (m, rho * m)
        fl = bench.flops_by_kind([shape], 5)
        ex = bench.executed_flops_by_kind([shape], 5)
        assert ex["bx"] == fl["bx"]
    for shape in [(1000, 3000), (130, 130)]:
        fl = bench.flops_by_kind([shape], 5)
        ex = bench.executed_flops_by_kind([shape], 5)
        assert ex["bx"] > fl["bx"]


def test_small_matrices_count_as_one_kind():
    # m <= 128 and n <= 512: the whole iteration is one kernel; it computes the
    # padded 128-row products, exactly the useful flops at m = 128, n % 64 == 0
    fl = bench.flops_by_kind([(128, 256)], 5)
    ex = bench.executed_flops_by_kind([(128, 256)], 5)
    assert fl["gram"] == fl["a2b"] == fl["bx"] == 0
    assert fl["small"] == ex["small"] == 5 * (4 * 128 * 128 * 256 + 2 * 128 ** 3)
    fl = bench.flops_by_kind([(200, 72)], 5)
    ex = bench.executed_flops_by_kind([(200, 72)], 5)
    assert ex["small"] > fl["small"] > 0
    assert bench.flops_by_kind([(128, 256)], 5, small_path=False)["small"] == 0
    assert bench.gemm_kernel_for("small", 0, [(128, 256)])[0] == "ns_small_kernel"


def test_reference_arm_splits_the_workload_once():
    # the reference arm's timed steps together run every matrix exactly once
    w = bench.get_workload("gpt")
    for k in (1, 3, 20, 95, 96, 200):
        groups = bench.split_by_flops(w, k)
        assert len(groups) == min(k, len(w.shapes))
        assert [i for g in groups for i in g] == list(range(len(w.shapes)))


def test_blas_threads_reported():
    n = bench.blas_threads()
    assert n is None or n >= 1
