"""The automatic launch-shape choice, on the CPU (ptc_plan_shape: host
arithmetic over the shape model, with a GB300's 152 SMs and cluster
capacities of 76 / 36 / 15 clusters of 2 / 4 / 8 one-CTA tiles).  The choices
pinned here are the ones measured fastest at each size (CUDA-graph replays of
every shape, the tuning script's launch mode); a change to the model that
moves one of them has to be re-measured."""
import pytest

import precision_tensor_core_gb300 as ptc

F16, S8, S4 = 0, 1, 2


KNOBS = (("cta_pair", 0), ("tile_n", 0), ("ksplit", 0), ("in_ring", 1))


@pytest.fixture(autouse=True)
def default_knobs():
    for k, v in KNOBS:
        ptc.ptc_set_tuning(k, v)
    yield
    for k, v in KNOBS:
        ptc.ptc_set_tuning(k, v)


@pytest.mark.parametrize("n,prec,shape", [
    (512, F16, (1, 64, 4)), (512, S8, (1, 64, 4)), (512, S4, (1, 64, 4)),
    (1024, F16, (1, 128, 2)), (1024, S8, (1, 128, 2)), (1024, S4, (1, 64, 1)),
    (1536, F16, (1, 128, 1)), (1536, S8, (1, 128, 1)), (1536, S4, (1, 128, 1)),
    (2048, F16, (2, 256, 1)), (2048, S8, (1, 256, 1)), (2048, S4, (1, 256, 1)),
    (4096, F16, (2, 256, 1)), (4096, S8, (2, 256, 1)), (4096, S4, (2, 256, 1)),
    (8192, F16, (2, 256, 1)), (8192, S8, (2, 256, 1)), (8192, S4, (2, 256, 1)),
])
def test_square_sizes(n, prec, shape):
    assert ptc.ptc_plan_shape(n, n, n, prec) == shape


def test_long_k_over_few_tiles_splits_k():
    # 4 tiles of 128 x 256 with 256 K blocks: clusters of 8 share each tile's K
    assert ptc.ptc_plan_shape(512, 512, 16384, F16) == (1, 256, 8)
    # one tile row of 2048 columns, 32 K blocks: 64-wide tiles in clusters of 4
    assert ptc.ptc_plan_shape(128, 2048, 2048, F16) == (1, 64, 4)


def test_k_split_needs_room_and_blocks():
    # a single K block never splits
    assert ptc.ptc_plan_shape(512, 512, 64, F16)[2] == 1
    # without cluster capacity no K-split shape is chosen
    for n in (512, 1024):
        assert ptc.ptc_plan_shape(n, n, n, F16, caps=(0, 0, 0))[2] == 1
    # more SMs: the same products, a different balance
    assert ptc.ptc_plan_shape(2048, 2048, 2048, F16, sms=304, caps=(152, 72, 30))[1] in (64, 128, 256)


def test_knobs_force_the_shape():
    ptc.ptc_set_tuning("cta_pair", 2)
    assert ptc.ptc_plan_shape(512, 512, 512, F16) == (2, 256, 1)
    ptc.ptc_set_tuning("cta_pair", 1)
    assert ptc.ptc_plan_shape(8192, 8192, 8192, F16) == (1, 256, 1)
    assert ptc.ptc_plan_shape(512, 512, 4096, F16)[1] == 256
    ptc.ptc_set_tuning("cta_pair", 0)
    ptc.ptc_set_tuning("tile_n", 128)
    assert ptc.ptc_plan_shape(512, 512, 512, S8) == (1, 128, 1)
    ptc.ptc_set_tuning("ksplit", 4)
    assert ptc.ptc_plan_shape(512, 512, 512, S8) == (1, 128, 4)
    ptc.ptc_set_tuning("tile_n", 0)
    ptc.ptc_set_tuning("ksplit", 1)
    assert ptc.ptc_plan_shape(512, 512, 512, F16)[2] == 1


def test_invalid_arguments():
    with pytest.raises(ptc.PtcError):
        ptc.ptc_plan_shape(0, 512, 512, F16)
    with pytest.raises(ptc.PtcError):
        ptc.ptc_plan_shape(512, 512, 512, 3)
    with pytest.raises(ptc.PtcError):
        ptc.ptc_plan_shape(512, 512, 512, F16, sms=0)


@pytest.mark.parametrize("n,prec,ring", [
    (512, S8, True), (512, S4, True), (1024, S8, True), (1024, S4, False),
    (1536, S8, False), (1536, S4, False), (2048, S8, False), (2048, S4, False),
    (4096, S8, False), (8192, S4, False), (512, F16, False), (8192, F16, False),
])
def test_in_ring_choice_at_square_sizes(n, prec, ring):
    """In-ring operand conversion where the launch-shape sweep of both paths
    measured it faster (INT8 at N = 512 and 1024, INT4 at N = 512: 6.3 us
    against 7.7 / 7.2 us with the separate pass at N = 512), the pass elsewhere
    (its fixed cost is repaid once a CTA converts more than a few K blocks)."""
    assert ptc.ptc_plan_shape(n, n, n, prec, with_ring=True)[3] is ring


def test_in_ring_rules():
    # odd K of packed s4 (a stray high nibble per row): never in ring
    assert ptc.ptc_plan_shape(512, 512, 511, S4, with_ring=True)[3] is False
    # a long K over few tiles: many K blocks per CTA, the pass
    assert ptc.ptc_plan_shape(512, 512, 16384, S8, with_ring=True)[3] is False
    # forced narrow tiles with more tiles than SMs: several units per CTA, the pass
    ptc.ptc_set_tuning("tile_n", 64)
    assert ptc.ptc_plan_shape(2048, 2048, 256, S8, with_ring=True)[3] is False
    # the knob: 0 never, 2 on every one-CTA shape (not on CTA pairs)
    ptc.ptc_set_tuning("in_ring", 2)
    assert ptc.ptc_plan_shape(2048, 2048, 256, S8, with_ring=True)[3] is True
    ptc.ptc_set_tuning("tile_n", 0)
    assert ptc.ptc_plan_shape(8192, 8192, 8192, S8, with_ring=True)[3] is False
    ptc.ptc_set_tuning("in_ring", 0)
    assert ptc.ptc_plan_shape(512, 512, 512, S8, with_ring=True)[3] is False
    assert ptc.ptc_plan_shape(512, 512, 512, S8) == (1, 64, 4)


def test_plan_invariants_over_random_shapes():
    """Every plan is launchable and consistent, over 3000 seeded shapes (sizes
    log-uniform, so small products are as common as large ones) and all
    three precisions: CTA pairs are 256-wide and never split or convert in
    ring; narrow tiles fit one wave; a K-split fits the cluster capacity and
    leaves every CTA a K block; in-ring conversion only for integer one-CTA
    single-wave launches (packed s4: even K); products with one wave or more
    of 128 x 256 tiles run on CTA pairs; with the knob at 0 nothing converts
    in ring, at 2 every one-CTA integer plan does."""
    import numpy as np
    rng = np.random.default_rng(2024)
    sms, caps = 152, (76, 36, 15)
    cap_of = {2: caps[0], 4: caps[1], 8: caps[2]}
    def log_uniform(hi):  # small products as often as large ones
        return max(1, int(np.exp(rng.uniform(0.0, np.log(hi)))))

    for _ in range(3000):
        M, N, K = log_uniform(20000), log_uniform(20000), log_uniform(70000)
        prec = int(rng.integers(0, 3))
        ctas, bn, ks, ring = ptc.ptc_plan_shape(M, N, K, prec, with_ring=True)
        num_kb = (K + (127 if prec == S4 else 63)) // (128 if prec == S4 else 64)
        tiles = ((M + 127) // 128) * ((N + bn - 1) // bn)
        t256 = ((M + 127) // 128) * ((N + 255) // 256)
        assert ctas in (1, 2) and bn in (64, 128, 256) and ks in (1, 2, 4, 8)
        if ctas == 2:
            assert bn == 256 and ks == 1 and not ring
        if t256 >= sms:
            assert ctas == 2
        if bn != 256:
            assert ks in (1, 2, 4) and tiles <= sms
        if ks > 1:
            assert ctas == 1 and num_kb >= ks and tiles <= cap_of[ks]
        if ring:
            assert prec != F16 and ctas == 1 and tiles * ks <= sms
            assert prec != S4 or K % 2 == 0
    for value, expect in ((0, False), (2, True)):
        ptc.ptc_set_tuning("in_ring", value)
        for _ in range(300):
            M, N = int(rng.integers(1, 3000)), int(rng.integers(1, 3000))
            K = 2 * int(rng.integers(1, 8000))
            prec = int(rng.integers(1, 3))
            ctas, _, _, ring = ptc.ptc_plan_shape(M, N, K, prec, with_ring=True)
            assert ring is (expect and ctas == 1)
    ptc.ptc_set_tuning("in_ring", 1)
