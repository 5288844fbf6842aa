"""The seeded generator: published splitmix64 values, determinism, distributions."""
import numpy as np

import hcmix_inputs as hi


def test_splitmix64_published_first_values():
    # SplitMix64 seeded with 0 (state advanced by the golden gamma before mixing)
    z = hi.splitmix64(0, 0, 3)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_x_prefix_stable_and_thread_independent():
    a = hi.make_x(40, K=1024, threads=1, row_block=5)
    b = hi.make_x(70, K=1024, threads=4, row_block=16)
    assert np.array_equal(a, b[:40])


def test_distributions():
    x = hi.bf16_bits_to_f32(hi.make_x(64)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    W = hi.make_w()
    assert abs(W.std() * np.sqrt(W.shape[1]) - 1) < 0.01
    s = hi.make_scale()
    assert s.shape == (3,) and np.all((s >= 0.5) & (s < 1.5))
    b = hi.make_base()
    assert b.shape == (24,) and np.all(np.abs(b) < 0.5)


def test_outliers():
    ch = hi.outlier_channels(20480)
    assert len(ch) == 205 and len(np.unique(ch)) == 205
    xo = hi.bf16_bits_to_f32(hi.make_x(4, outliers=True)).astype(np.float64)
    xn = hi.bf16_bits_to_f32(hi.make_x(4)).astype(np.float64)
    mask = np.zeros(20480, bool); mask[ch] = True
    assert np.array_equal(xo[:, ~mask], xn[:, ~mask])
    assert np.allclose(xo[:, mask], 20 * xn[:, mask], rtol=2 ** -7)


def test_bf16_rounding_is_nearest_even_once():
    # 1 + 2**-8 is a tie between 1 and 1 + 2**-7: even -> 1
    # 1 + 2**-8 + 2**-30 is above the tie -> 1 + 2**-7 (a detour via fp32 would
    # drop the 2**-30 and round to 1)
    v = np.array([1 + 2 ** -8, 1 + 2 ** -8 + 2 ** -30, 1 + 3 * 2 ** -8])
    got = hi.bf16_bits_to_f32(hi.bf16_bits_from_f64(v)).astype(np.float64)
    assert list(got) == [1.0, 1 + 2 ** -7, 1 + 2 ** -6]
