"""The CUDA input filler equals the numpy generator bit for bit."""
import numpy as np
import pytest
import torch

from weight_streaming_q4_gb300 import build, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def test_device_philox_known_answers():
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    synth.device_philox(out.data_ptr(), 0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344, 0xa4093822, 0x299f31d0)
    got = out.cpu().numpy().view(np.uint32)
    assert [int(v) for v in got] == [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1]


@pytest.mark.parametrize("block0,n", [(0, 1), (0, 4097), (123456789, 5000), ((1 << 33) + 7, 300)])
def test_device_q4_blocks_match_numpy(block0, n):
    dst = torch.zeros(n * 18 + 16, dtype=torch.uint8, device="cuda")
    synth.device_fill_q4(dst.data_ptr(), n, seed=11, tid=synth.tensor_id(5, 3), block0=block0)
    got = dst.cpu().numpy()[: n * 18]
    ref = synth.q4_blocks(np.arange(block0, block0 + n, dtype=np.uint64), 11, synth.tensor_id(5, 3)).reshape(-1)
    assert np.array_equal(got, ref)


def test_device_normals_match_numpy():
    n = 70001
    dst = torch.zeros(n, dtype=torch.int16, device="cuda")
    synth.device_fill_normal_f16(dst.data_ptr(), n, seed=3, tid=synth.X_TID, start=17)
    got = dst.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, synth.normal_f16(n, 3, synth.X_TID, start=17))
