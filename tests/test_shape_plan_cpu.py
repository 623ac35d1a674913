"""The automatic launch-shape choice, on the CPU (ptc_plan_shape: host
arithmetic over the shape model, with a GB300's 152 SMs and cluster
capacities of 76 / 36 / 15 clusters of 2 / 4 / 8 one-CTA tiles).  The choices
pinned here are the ones measured fastest at each size (CUDA-graph replays of
every shape, the tuning script's launch mode); a change to the model that
moves one of them has to be re-measured."""
import pytest

import precision_tensor_core_gb300 as ptc

F16, S8, S4 = 0, 1, 2


@pytest.fixture(autouse=True)
def default_knobs():
    for k, v in (("cta_pair", 0), ("tile_n", 0), ("ksplit", 0)):
        ptc.ptc_set_tuning(k, v)
    yield
    for k, v in (("cta_pair", 0), ("tile_n", 0), ("ksplit", 0)):
        ptc.ptc_set_tuning(k, v)


@pytest.mark.parametrize("n,prec,shape", [
    (512, F16, (1, 64, 4)), (512, S8, (1, 64, 4)), (512, S4, (1, 64, 1)),
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
