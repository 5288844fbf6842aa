"""Why the oracle's chunk dot is the exact dot rounded once (design reading c2).

An fp32 running sum inside each 64-wide chunk (one plausible hardware order)
and the correctly rounded chunk dot differ by ~1 ulp per chunk; the 80 fp32
slice additions then amplify that into differences that reach the stated mix
tolerance (max(2e-6 |o|, 1e-6)) at the headline size.  A GPU whose chunk dots
are not the oracle's would therefore fail parity by chance, which is why the
CUDA kernels reproduce the correctly rounded chunk dot instead.
"""
import numpy as np
import pytest

import hcmix_inputs as hi
import oracle


@pytest.mark.slow
def test_other_inchunk_order_reaches_the_tolerance():
    x = hi.make_x(2048)
    W = hi.make_w()
    a, _ = oracle.stats(x, W, threads=8)
    b = oracle.stats_seq_f32(x, W)
    d = np.abs(a.astype(np.float64) - b)
    thr = np.maximum(2e-6 * np.abs(a), 1e-6)
    assert (d / thr).max() > 0.5
    # yet both are close to the fp64 value: the difference is rounding, not error
    m64, _ = oracle.stats_f64(x[:64], W)
    assert np.abs(a[:64] - m64).max() < 3e-6 and np.abs(b[:64] - m64).max() < 3e-6
