"""Concurrent calls on several streams: each call's split-tail workspace is
its own (stream-ordered allocations from the library pool), so products
computed concurrently equal the same products computed one at a time, bit
for bit (the kernels are deterministic), and match the oracle."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import precision_tensor_core_gb300 as ptc
from tests.gpu_util import DEV, check_f16_sampled, f16_dev, int_dev, sample_coords

pytestmark = pytest.mark.gpu

# 2560 x 2048 is 80 tiles of 256 x 256 on 76 CTA pairs: a 4-tile last wave,
# split in K (4160 values = 65 K blocks, above the split threshold of 64).
M, N, K = 2560, 2048, 4160
STREAMS = 4


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(DEV)
    yield
    assert ptc.gemm_poll_device_error() == ptc.PTC_OK


def _concurrent(run, inputs):
    streams = [torch.cuda.Stream() for _ in inputs]
    torch.cuda.synchronize()
    outs = []
    for s, x in zip(streams, inputs):
        with torch.cuda.stream(s):
            outs.append(run(*x))
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


def test_concurrent_fp16_split_tails():
    host = [datagen.f16_operands(N, "normal", seed=100 + i, m=M, k=K) for i in range(STREAMS)]
    dev = [(f16_dev(A), f16_dev(B)) for A, B in host]
    together = _concurrent(lambda A, B: ptc.matmul_f16(A, B, sync=False), dev)
    for (A, B), (Ad, Bd), C in zip(host, dev, together):
        alone = ptc.matmul_f16(Ad, Bd).cpu().numpy()
        assert np.array_equal(C.view(np.uint32), alone.view(np.uint32))
        check_f16_sampled(C, A, B, n=400)


def test_concurrent_int8_split_tails():
    host = [datagen.s8_operands(N, seed=200 + i, m=M, k=K) for i in range(STREAMS)]
    dev = [(int_dev(A), int_dev(Bt)) for A, Bt in host]
    together = _concurrent(lambda A, Bt: ptc.matmul_s8(A, Bt, sync=False), dev)
    for (A, Bt), (Ad, Bd), C in zip(host, dev, together):
        alone = ptc.matmul_s8(Ad, Bd).cpu().numpy()
        assert np.array_equal(C, alone)
        ii, jj = sample_coords(M, N, 2000)
        assert np.array_equal(C[ii, jj], oracle.wrap_s32(oracle.gemm_s8_at(A, Bt, ii, jj)))
