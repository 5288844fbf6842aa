"""Hand-built inputs with closed-form results, shared by the oracle pins and
the GPU parity tests (input construction only; no method arithmetic beyond
the closed forms the pins compare against)."""
import numpy as np

import hcmix_inputs as hi


def rms_pin_inputs(case: str):
    """Inputs on which r = 1/sqrt(sq * (1/K) + rms_eps) is an exact power of two
    while sq/K and rms_eps are of one size, so moving rms_eps outside the root,
    dropping the 1/K factor or adding eps after the reciprocal changes r by a
    large factor.  Returns (x bf16 bits, W, rms_eps, r, c) with mix * r = c
    exactly (c_j = (2j - 23) / 16, dyadic)."""
    K = 1024
    c = (2.0 * np.arange(24) - 23.0) / 16.0
    W = (np.random.default_rng(31).standard_normal((24, K)) * 0.01).astype(np.float32)
    if case == "one_hot":
        # one x = 1 at column 77: sq = 1, sq/K = 2^-10; eps = 3 * 2^-10 gives
        # sq/K + eps = 2^-8 and r = 16; mix_j = W[j, 77] = c_j / 16
        x = np.zeros((1, K))
        x[0, 77] = 1.0
        W[:, 77] = (c / 16.0).astype(np.float32)
        return hi.bf16_bits_from_f64(x), W, 3.0 * 2.0 ** -10, 16.0, c
    # x = 1 everywhere: sq = K, sq/K = 1; eps = 3 gives r = 1/2; W[j, :] = 2 c_j / K
    # makes every partial sum exact and mix_j = 2 c_j
    x = np.ones((1, K))
    W = np.repeat((2.0 * c / K)[:, None], K, axis=1).astype(np.float32)
    return hi.bf16_bits_from_f64(x), W, 3.0, 0.5, c


def rms_pin_closed_form(c, scale, base, iters=20):
    """pre, post, comb in fp64 from the exact products mix_j * r = c_j."""
    g = np.array([0] * 4 + [1] * 4 + [2] * 16)
    logit = c * scale.astype(np.float64)[g] + base.astype(np.float64)
    C = np.exp(logit[8:]).reshape(4, 4)
    for _ in range(iters):
        C = C / C.sum(1, keepdims=True)
        C = C / C.sum(0, keepdims=True)
    return 1 / (1 + np.exp(-logit[:4])), 2 / (1 + np.exp(-logit[4:8])), C
