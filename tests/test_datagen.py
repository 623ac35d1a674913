"""The seeded input generators: published SplitMix64 vectors, value ranges,
determinism and storage formats."""
import os

import numpy as np

import datagen


def test_splitmix64_published_vectors(golden_dir):
    with open(os.path.join(golden_dir, "splitmix64_vectors.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            seed, outs = int(line[0]), [int(h, 16) for h in line[1:]]
            got = datagen.splitmix64_stream(seed, len(outs))
            assert [int(x) for x in got] == outs


def test_stream_offsets_consistent():
    full = datagen.splitmix64_stream(77, 100)
    part = datagen.splitmix64_stream(77, 30, start=50)
    assert np.array_equal(full[50:80], part)
    chunked = datagen.splitmix64_stream(77, 100, chunk=7)
    assert np.array_equal(full, chunked)


def test_ranges_and_determinism():
    a = datagen.uniform_s8(1, 64, 64)
    assert a.dtype == np.int8 and a.min() == -128 and a.max() == 127
    assert np.array_equal(a, datagen.uniform_s8(1, 64, 64))
    v = datagen.uniform_s4_values(2, 64, 64)
    assert v.min() == -8 and v.max() == 7
    u = datagen.uniform_f16(3, 128, 128).view(np.float16).astype(np.float64)
    assert u.min() >= -1 and u.max() <= 1 and abs(u.mean()) < 0.02
    n = datagen.normal_f16(4, 256, 256, 1.0).view(np.float16).astype(np.float64)
    assert abs(n.mean()) < 0.02 and abs(n.std() - 1) < 0.02


def test_operand_shapes_and_seeds():
    A, B = datagen.f16_operands(32, "uniform", m=16, k=48)
    assert A.shape == (16, 48) and B.shape == (48, 32) and A.dtype == np.uint16
    A8, B8 = datagen.s8_operands(32, m=16, k=48)
    assert A8.shape == (16, 48) and B8.shape == (32, 48)
    A4, B4 = datagen.s4_operands(32, m=16, k=48)
    assert A4.shape == (16, 24) and B4.shape == (32, 24) and A4.dtype == np.uint8
    assert datagen.config_seed("s8", 2048) == 1_000_003 * 2048 + 1
    assert datagen.operand_seed(10, "A") == 10 ^ 0xA
    # A and B of one config come from different sub-streams
    assert not np.array_equal(A8[:, :16], B8[:16, :16])


def test_normal_scaling():
    A, B = datagen.f16_operands(1024, "normal", m=64)
    a = A.view(np.float16).astype(np.float64)
    assert abs(a.std() * np.sqrt(1024) - 1) < 0.05
