"""The seeded input generator (-m "not gpu")."""
import numpy as np

from weight_streaming_q4_gb300 import synth


def test_philox_known_answers():
    # known-answer vectors published with the Philox4x32-10 definition
    kat = [((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
           ((0xffffffff,) * 4, (0xffffffff,) * 2, (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
           ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
            (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1))]
    for ctr, key, out in kat:
        got = synth.philox4x32_10(*ctr, *key)
        assert tuple(int(v) for v in got) == out


def test_distributions():
    b = synth.q4_blocks(np.arange(200000), 0, 1)
    d = b[:, :2].copy().view(np.uint16).view(np.float16).astype(np.float64).ravel()
    assert np.all(d >= 0)
    assert abs(d.mean() - 0.02 * np.sqrt(2 / np.pi)) < 2e-4
    codes = np.concatenate([b[:, 2:] & 15, b[:, 2:] >> 4]).ravel()
    counts = np.bincount(codes, minlength=16)
    assert counts.size == 16 and np.all(np.abs(counts / counts.mean() - 1) < 0.02)
    x = synth.activations(1, 200000, 0).view(np.float16).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01 and np.abs(x).max() <= 6


def test_rows_match_matrix_and_seeds_differ():
    m = synth.q4_matrix(10, 256, 5, synth.tensor_id(3, 4)).reshape(10, -1)
    r = synth.q4_rows([7, 2], 256, 5, synth.tensor_id(3, 4))
    assert np.array_equal(r, m[[7, 2]])
    other = synth.q4_matrix(10, 256, 5, synth.tensor_id(3, 5)).reshape(10, -1)
    assert not np.array_equal(m, other)


def test_layer_block_layout():
    offs, total = synth.layer_offsets(256, 256, 128, 768)
    dims = synth.layer_dims(256, 256, 128, 768)
    blk = synth.layer_block(2, 256, 256, 128, 768, seed=3)
    assert blk.size == total
    for p, (n, k) in enumerate(dims):
        assert offs[p] % 16 == 0
        m = synth.q4_matrix(n, k, 3, synth.tensor_id(2, p))
        assert np.array_equal(blk[offs[p]:offs[p] + m.size], m)
