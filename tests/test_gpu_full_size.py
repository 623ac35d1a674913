"""Parity at the benchmark's configuration, on every output element.

The three N = 8192 products run through the same entry points, knobs and
launch configuration the benchmark times (CTA pairs on 256 x 256 tiles, the
persistent work list, the operand conversion of the integer routes), on the
benchmark's seeded inputs:
  INT8, INT4   all 67 M outputs bit-exact against the oracle;
  FP16         whole blocks: the first 256-row panel and the block spanned by
               the last wave's tiles, each under the element-wise bound
               |C - Cref| <= 1e-3 * sum_k |a_ik b_kj| + 1e-6 and the relative
               Frobenius bound 1e-4;
and FP16 at N = 2048 and N = 4096 in full, the sizes whose short last wave is
split in two K halves added into C by TMA reductions (the split tiles'
results included).  Sizes follow the square N = 512 ... 8192 workloads of
"Hand-Written PTX Tensor-Core GEMM Kernels: A Multi-Precision Study on NVIDIA
L4" (section III-B).
"""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16, check_f16_rows, f16_dev, int_dev

pytestmark = pytest.mark.gpu

N_BENCH = 8192
GROUP_M = 8  # raster group of the default launch (knob "group_m")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    ptc.lib()
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


def tile_coords(t, tiles_m, tiles_n, group_m=GROUP_M):
    """Grouped raster order of the persistent scheduler: tile t -> (m, n)."""
    per_group = group_m * tiles_n
    g = t // per_group
    first_m = g * group_m
    gsz = min(tiles_m - first_m, group_m)
    r = t - g * per_group
    return first_m + r % gsz, r // gsz


def last_wave_block(n, tile=256):
    """Rows and columns spanned by the tiles of the last launch's last wave."""
    grid, cluster, _, _ = ptc.ptc_last_launch()
    assert cluster == 2, "CTA pairs at this size"
    clusters = grid // cluster
    tm = tn = n // tile
    tiles = tm * tn
    tail = tiles % clusters or clusters
    coords = [tile_coords(t, tm, tn) for t in range(tiles - tail, tiles)]
    ms = [m for m, _ in coords]
    ns = [c for _, c in coords]
    return (min(ms) * tile, (max(ms) + 1) * tile, min(ns) * tile, (max(ns) + 1) * tile), tail, clusters


def test_int8_8192_every_element():
    A, Bt = datagen.s8_operands(N_BENCH)
    C = ptc.matmul_s8(int_dev(A), int_dev(Bt))
    torch.cuda.synchronize()
    assert ptc.ptc_last_conversion() == 1 and ptc.ptc_last_launch()[1] == 2
    got = C.cpu().numpy()
    del C
    ref = oracle.wrap_s32(oracle.gemm_s8(A, Bt))
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} INT8 mismatches, first at {bad[:4].tolist()}"


def test_int4_8192_every_element():
    A, Bt = datagen.s4_operands(N_BENCH)
    C = ptc.matmul_s4(int_dev(A), int_dev(Bt), N_BENCH)
    torch.cuda.synchronize()
    assert ptc.ptc_last_conversion() == 1 and ptc.ptc_last_launch()[1] == 2
    got = C.cpu().numpy()
    del C
    ref = oracle.wrap_s32(oracle.gemm_s4(A, Bt, N_BENCH))
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} INT4 mismatches, first at {bad[:4].tolist()}"


def test_fp16_8192_first_panel_and_last_wave():
    A, B = datagen.f16_operands(N_BENCH, "normal")
    C = ptc.matmul_f16(f16_dev(A), f16_dev(B))
    torch.cuda.synchronize()
    (r0, r1, c0, c1), tail, clusters = last_wave_block(N_BENCH)
    got = C.cpu().numpy()
    del C
    assert np.all(np.isfinite(got))
    check_f16_rows(got[0:256], A, B, 0, 256)
    check_f16_rows(got[r0:r1, c0:c1], A, B, r0, r1, c0, c1)
    assert (r1 - r0) * (c1 - c0) >= tail * 256 * 256


@pytest.mark.parametrize("n", [2048, 4096])
def test_fp16_full_with_split_tail(n):
    A, B = datagen.f16_operands(n, "normal")
    C = ptc.matmul_f16(f16_dev(A), f16_dev(B))
    torch.cuda.synchronize()
    _, tail, clusters = last_wave_block(n)
    got = C.cpu().numpy()
    del C
    if n == 4096:
        # the last wave fills at most half the clusters: its tiles were split
        assert 0 < tail and 2 * tail <= clusters
    check_f16(got, A, B)


@pytest.mark.parametrize("n", [2048, 4096])
def test_int8_full_with_split_tail(n):
    A, Bt = datagen.s8_operands(n)
    C = ptc.matmul_s8(int_dev(A), int_dev(Bt))
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), oracle.wrap_s32(oracle.gemm_s8(A, Bt)))
