"""The seeded generator: determinism, counter addressing and distribution."""
import numpy as np

import synth


def test_counter_addressing_and_determinism():
    a = synth.uniform_bits(7, 0, 100)
    b = synth.uniform_bits(7, 40, 60)
    np.testing.assert_array_equal(a[40:], b)
    np.testing.assert_array_equal(synth.normal_f64(3, 1001), synth.normal_f64(3, 1001))
    assert not np.array_equal(synth.normal_f64(3, 64), synth.normal_f64(4, 64))


def test_splitmix64_reference_values():
    # SplitMix64 with state seeded to 0: first outputs of the published
    # generator (Steele, Lea, Flood 2014; java.util.SplittableRandom).
    # Our stream key is mix64(seed); feed key 0 by inverting nothing: check
    # the finaliser directly on the published first state increments.
    z = np.array([0x9E3779B97F4A7C15], dtype=np.uint64)
    out = synth._mix64(z)[0]
    assert int(out) == 0xE220A8397B1DCDAF


def test_normal_moments_and_bf16_rounding():
    x = synth.normal_f64(11, 400000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    bits = synth.f64_to_bf16_bits(np.array([1.0, -2.5, 1.00390625, 1.01171875, 3.0e38]))
    np.testing.assert_array_equal(bits, [0x3F80, 0xC020, 0x3F80, 0x3F82, 0x7F62])
    back = synth.bf16_bits_to_f64(bits)
    assert back[0] == 1.0 and back[1] == -2.5


def test_workload_shapes_and_outliers():
    w = synth.make_workload(1)
    assert w.q.shape == (4096, 1, 64) and w.k.shape == (4096, 1, 64)
    assert len(w.outliers) == 8
    k = synth.bf16_bits_to_f64(w.k)
    norms = np.linalg.norm(k[:, 0], axis=-1)
    others = np.delete(norms, w.outliers)
    assert norms[w.outliers].mean() > 6 * others.mean()
    w3 = synth.make_workload(3, L=1024)
    assert w3.q.shape == (1024, 16, 128) and w3.k.shape == (1024, 2, 128) and w3.do is not None


def test_row_chunked_generation_is_bit_identical():
    # odd row length, chunk boundaries in the middle of Box-Muller pairs of
    # the flat stream are impossible (even row offsets), odd tensor end
    for shape, rpc in [((7, 3, 5), 1), ((9, 2, 8), 4), ((64, 16, 128), None)]:
        n = int(np.prod(shape))
        ref = synth.f64_to_bf16_bits(synth.normal_f64(21, n)).reshape(shape)
        np.testing.assert_array_equal(synth.normal_bf16_rows(21, shape, rows_per_chunk=rpc), ref)
    # a per-row transform sees the right rows
    shape = (10, 2, 3)
    x = synth.normal_f64(5, 60).reshape(shape)
    x[3] *= 4.0
    ref = synth.f64_to_bf16_bits(x)

    def tf(blk, r0):
        rows = np.arange(r0, r0 + blk.shape[0])
        blk[rows == 3] *= 4.0
        return blk
    np.testing.assert_array_equal(synth.normal_bf16_rows(5, shape, tf, rows_per_chunk=2), ref)
