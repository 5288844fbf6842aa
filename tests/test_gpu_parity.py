"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Tolerances of the library's parity contract: mix within max(2e-6 |o|, 1e-6);
pre, post and comb within 1e-5 absolute.  sq is compared bit for bit: the kernels evaluate the
page's fixed tree on exact squares with the same round-to-nearest adds.
"""
import os

import numpy as np
import pytest
import torch

import hcmix_inputs as hi
import oracle
from hyper_connection_mix_gb300 import binding
from pin_inputs import rms_pin_closed_form, rms_pin_inputs

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1
PATHS = ("simt", "tc", "simt_fullk", "tc_staged")


def dev_x(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def path_available(path):
    x = torch.zeros(1, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(24, 256, dtype=torch.float32, device="cuda")
    try:
        binding.hc_mix_stats(x, W, path=path)
        return True
    except binding.HcMixError as e:
        if e.status == 3:
            return False
        raise


@pytest.fixture(scope="module", params=PATHS)
def path(request):
    if not path_available(request.param):
        pytest.fail(f"kernel path {request.param} is not available in this library")
    return request.param


def run(x, W, sc, bs, path, iters=20, rms_eps=1e-6, hc_eps=0.0, x_dev=None):
    xt = dev_x(x) if x_dev is None else x_dev
    out = binding.hc_mix_fused(xt, dev(W), dev(sc), dev(bs), iters, rms_eps, hc_eps,
                               want_stats=True, path=path)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def assert_mix_close(g, o, what=""):
    thr = np.maximum(2e-6 * np.abs(o.astype(np.float64)), 1e-6)
    d = np.abs(g.astype(np.float64) - o)
    bad = d > thr
    assert not bad.any(), (f"{what} mix: {bad.sum()} of {bad.size} outside tolerance, "
                           f"max ratio {(d / thr).max():.3f}")
    return float((d / thr).max())


def assert_epilogue_close(got, want, what=""):
    for name, g, o in zip(("pre", "post", "comb"), got, want):
        err = float(np.max(np.abs(g.astype(np.float64) - o))) if g.size else 0.0
        assert err <= 1e-5, f"{what} {name}: max abs error {err}"


def check_all(x, W, sc, bs, path, what, **kw):
    want = oracle.fused(x, W, sc, bs, threads=THREADS, **kw)
    got = run(x, W, sc, bs, path, **kw)
    assert_epilogue_close(got[:3], want[:3], what)
    r = assert_mix_close(got[3], want[3], what)
    assert np.array_equal(got[4], want[4]), f"{what} sq not bit-identical"
    return r


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8])
@pytest.mark.parametrize("K", [256, 512, 768, 1024])
def test_tiny(path, M, K):
    x = hi.make_x(M, K=K)
    check_all(x, hi.make_w(K=K), hi.make_scale(), hi.make_base(), path, f"M={M} K={K}")


@pytest.mark.parametrize("M", [33, 100, 129, 255, 300])
def test_ragged_rows_several_tiles(path, M):
    K = 2048
    check_all(hi.make_x(M, K=K), hi.make_w(K=K), hi.make_scale(), hi.make_base(), path,
              f"M={M}")


@pytest.mark.parametrize("M,K", [(1, 40960), (3, 9472), (9, 2560), (127, 5120), (129, 768),
                                 (513, 20480), (1000, 1280), (2049, 2048), (6, 122880)])
def test_irregular_shapes(path, M, K):
    """Shapes off the workloads' grid: tile counts just above and below a
    multiple of 128 rows, slice counts that split unevenly over the CTAs
    (37, 5, 3 slices), more units than CTAs, and few rows with many slices,
    where each CTA refills its W slots."""
    check_all(hi.make_x(M, K=K, seed=M + K), hi.make_w(K=K), hi.make_scale(), hi.make_base(),
              path, f"M={M} K={K}")


def test_config_m16(path):
    check_all(hi.make_x(16), hi.make_w(), hi.make_scale(), hi.make_base(), path, "M=16")


def test_config_m512_outliers(path):
    check_all(hi.make_x(512, outliers=True), hi.make_w(), hi.make_scale(), hi.make_base(), path,
              "M=512 outliers")


def test_config_decode_sweep(path):
    x = hi.make_x(256)
    W, sc, bs = hi.make_w(), hi.make_scale(), hi.make_base()
    for M in (1, 4, 16, 64, 128, 256):
        check_all(np.ascontiguousarray(x[:M]), W, sc, bs, path, f"sweep M={M}")


def test_config_m4096_full(path):
    ratio = check_all(hi.make_x(4096), hi.make_w(), hi.make_scale(), hi.make_base(), path,
                      "M=4096")
    print(f"M=4096 {path}: max mix error / tolerance = {ratio:.3f}")


@pytest.mark.parametrize("case", ["one_hot", "all_ones"])
def test_rms_eps_placement_inputs(path, case):
    """Inputs on which r = 1/sqrt(sq/K + rms_eps) is an exact power of two with
    sq/K and rms_eps of one size: the kernels agree with the oracle and with
    the closed form, which a misplaced eps or a dropped 1/K would miss by far."""
    x, W, eps, r, c = rms_pin_inputs(case)
    scale = np.array([1.0, 2.0, 3.0], np.float32)
    base = (np.arange(24) * 0.03 - 0.2).astype(np.float32)
    check_all(x, W, scale, base, path, f"rms {case}", rms_eps=eps)
    got = run(x, W, scale, base, path, rms_eps=eps)
    assert np.array_equal(got[3][0].astype(np.float64) * r, c)
    p, q, C = rms_pin_closed_form(c, scale, base)
    assert np.max(np.abs(got[0][0] - p)) <= 1e-6
    assert np.max(np.abs(got[1][0] - q)) <= 1e-6
    assert np.max(np.abs(got[2][0] - C)) <= 1e-5


@pytest.mark.parametrize("M", [5, 130])
def test_long_k_more_slices_than_slots(path, M):
    """K = 131072 (512 slices): with 152 CTAs each CTA covers three or more
    slices, so the tensor-core kernel refills its two W slots while it runs."""
    K = 131072
    check_all(hi.make_x(M, K=K), hi.make_w(K=K), hi.make_scale(), hi.make_base(), path,
              f"M={M} K={K}")


def test_integer_inputs_bit_exact(path):
    """x in {-4..4}, W in {-8..8}: every partial sum is an integer < 2**24, so
    every correct evaluation order gives the exact integer product."""
    rng = np.random.default_rng(5)
    K = 2048
    xi = rng.integers(-4, 5, size=(130, K))
    wi = rng.integers(-8, 9, size=(24, K))
    got = run(hi.bf16_bits_from_f64(xi), wi.astype(np.float32), hi.make_scale(),
              hi.make_base(), path)
    assert np.array_equal(got[3].astype(np.int64), xi @ wi.T)
    assert np.array_equal(got[4].astype(np.int64), (xi * xi).sum(1))


def test_one_hot_rows_select_columns(path):
    K = 1024
    W = (np.random.default_rng(3).standard_normal((24, K)) * 0.01).astype(np.float32)
    cols = [0, 1, 63, 64, 255, 256, 511, 1023]
    x = np.zeros((len(cols), K))
    for r, k in enumerate(cols):
        x[r, k] = 1.0
    got = run(hi.bf16_bits_from_f64(x), W, hi.make_scale(), hi.make_base(), path)
    for r, k in enumerate(cols):
        assert np.array_equal(got[3][r], W[:, k])


def test_strided_inputs(path):
    K, M = 1024, 70
    rng = np.random.default_rng(8)
    xs = hi.bf16_bits_from_f64(rng.standard_normal((M, K + 64)))
    Wf = (rng.standard_normal((24, K + 32)) * 0.03).astype(np.float32)
    sc, bs = hi.make_scale(), hi.make_base()
    want = oracle.fused(np.ascontiguousarray(xs[:, :K]), np.ascontiguousarray(Wf[:, :K]), sc, bs)
    xt = dev_x(xs)[:, :K]
    Wt = dev(Wf)[:, :K]
    out = binding.hc_mix_fused(xt, Wt, dev(sc), dev(bs), want_stats=True, path=path)
    torch.cuda.synchronize()
    got = [o.cpu().numpy() for o in out]
    assert_epilogue_close(got[:3], want[:3], "strided")
    assert_mix_close(got[3], want[3], "strided")
    assert np.array_equal(got[4], want[4])


def test_deterministic_repeat(path):
    x, W, sc, bs = hi.make_x(300), hi.make_w(), hi.make_scale(), hi.make_base()
    xt = dev_x(x)
    a = run(x, W, sc, bs, path, x_dev=xt)
    b = run(x, W, sc, bs, path, x_dev=xt)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_stats_and_sinkhorn_entry_points_agree_with_fused(path):
    x, W, sc, bs = hi.make_x(77), hi.make_w(), hi.make_scale(), hi.make_base()
    xt, Wt, sct, bst = dev_x(x), dev(W), dev(sc), dev(bs)
    pre, post, comb, mix, sq = binding.hc_mix_fused(xt, Wt, sct, bst, want_stats=True, path=path)
    mix2, sq2 = binding.hc_mix_stats(xt, Wt, path=path)
    pre2, post2, comb2 = binding.hc_mix_sinkhorn(mix2, sq2, x.shape[1], sct, bst)
    torch.cuda.synchronize()
    for a, b in ((mix, mix2), (sq, sq2), (pre, pre2), (post, post2), (comb, comb2)):
        assert torch.equal(a, b)


def test_zero_weights_and_zero_rows(path):
    K = 512
    x = hi.make_x(9, K=K)
    x[3] = 0
    got = run(x, np.zeros((24, K), np.float32), hi.make_scale(), np.zeros(24, np.float32), path)
    assert np.all(got[0] == 0.5) and np.all(got[1] == 1.0) and np.all(got[2] == 0.25)
    assert got[4][3] == 0


def test_sinkhorn_iteration_counts(path):
    x, W, sc, bs = hi.make_x(20, K=1024), hi.make_w(K=1024), hi.make_scale(), hi.make_base()
    for iters in (0, 1, 3, 50):
        check_all(x, W, sc, bs, path, f"iters={iters}", iters=iters)
    check_all(x, W, sc, bs, path, "hc_eps", hc_eps=0.01)


def test_sinkhorn_row_below_the_normal_range(path):
    """A comb row whose exponentials are subnormal (logits near -89.8 with x = 0,
    so logit = hc_base): its sums fall below the normal range, where a
    reciprocal overflows; the epilogue then divides by the sums, as the oracle
    does, and the results stay within the tolerance."""
    K = 1024
    x = np.zeros((12, K), np.uint16)
    bs = hi.make_base()
    bs[8:12] = np.float32(-89.8)
    bs[12:16] = np.float32(-89.3)
    got = run(x, hi.make_w(K=K), hi.make_scale(), bs, path)
    assert all(np.isfinite(g).all() for g in got[:3])
    check_all(x, hi.make_w(K=K), hi.make_scale(), bs, path, "subnormal comb row")


def test_sinkhorn_sums_near_the_top_of_the_range(path):
    """Comb rows whose exponentials are near the top of the fp32 range (logits of
    86.2 to 87, x = 0 so logit = hc_base): their sums lie between 2^126, where an
    approximate reciprocal flushes to zero, and the largest finite float, so the
    oracle's results are finite; the epilogue notices the zero scale and
    divides by the sums instead, and the results match the oracle."""
    K = 1024
    x = np.zeros((12, K), np.uint16)
    bs = hi.make_base()
    bs[8:12] = np.float32(87.0)
    bs[12:16] = np.float32(86.5)
    bs[16:20] = np.float32(86.2)
    bs[20:24] = np.float32(86.8)
    got = run(x, hi.make_w(K=K), hi.make_scale(), bs, path)
    assert all(np.isfinite(g).all() for g in got[:3])
    check_all(x, hi.make_w(K=K), hi.make_scale(), bs, path, "comb sums near the top")


def test_nonfinite_inputs_propagate(path):
    """A NaN or an infinity in a row of x carries into that row's outputs (each
    output non-finite where the oracle's is), the other rows are unaffected,
    and the call ends cleanly."""
    K = 1024
    x, W, sc, bs = hi.make_x(20, K=K), hi.make_w(K=K), hi.make_scale(), hi.make_base()
    bf16_nan, bf16_inf = np.uint16(0x7FC0), np.uint16(0x7F80)
    x[3, 100] = bf16_nan
    x[11, 7] = bf16_inf
    want = oracle.fused(x, W, sc, bs, threads=THREADS)
    ws = binding.alloc_workspace(20, K)
    out = binding.hc_mix_fused(dev_x(x), dev(W), dev(sc), dev(bs), want_stats=True, workspace=ws,
                               path=path)
    torch.cuda.synchronize()
    got = [o.cpu().numpy() for o in out]
    bad = [3, 11]
    good = [r for r in range(20) if r not in bad]
    for name, g, o in zip(("pre", "post", "comb", "mix", "sq"), got, want):
        for r in bad:
            assert not np.all(np.isfinite(o[r])), f"the oracle's {name} of row {r} is finite"
            assert not np.any(np.isfinite(g[r]) & ~np.isfinite(o[r])), \
                f"{name} row {r}: finite where the oracle is not"
    assert_epilogue_close([g[good] for g in got[:3]], [o[good] for o in want[:3]], "finite rows")
    assert_mix_close(got[3][good], want[3][good], "finite rows")
    assert np.array_equal(got[4][good], want[4][good]), "finite rows: sq"
    assert binding.hc_mix_device_status(ws) == 0


def test_empty_batch_is_a_no_op(path):
    x = torch.zeros(0, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(24, 256, dtype=torch.float32, device="cuda")
    s = torch.ones(3, device="cuda"); b = torch.zeros(24, device="cuda")
    out = binding.hc_mix_fused(x, W, s, b, path=path)
    assert all(o.shape[0] == 0 for o in out)


def test_device_status_clean_after_runs(path):
    x, W = hi.make_x(200), hi.make_w()
    ws = binding.alloc_workspace(200, x.shape[1])
    binding.hc_mix_fused(dev_x(x), dev(W), dev(hi.make_scale()), dev(hi.make_base()),
                         workspace=ws, path=path)
    assert binding.hc_mix_device_status(ws) == 0


@pytest.mark.parametrize("M,K", [(1, 512), (3, 512), (8, 768), (130, 1024)])
def test_workspace_needs_only_its_header_zeroed(path, M, K):
    """The workspace contract asks only for its 256-byte header to be zeroed:
    with every other byte set to 0xFF (a NaN pattern in every fp32 slot), the
    fused call still gives the oracle's results and no device error, for a
    single row group (the tail run by the last CTA to arrive) and for several
    groups with a ragged last tile."""
    x, W, sc, bs = hi.make_x(M, K=K), hi.make_w(K=K), hi.make_scale(), hi.make_base()
    want = oracle.fused(x, W, sc, bs, threads=THREADS)
    ws = binding.alloc_workspace(M, K)
    ws[binding.HEADER_BYTES:].fill_(0xFF)
    out = binding.hc_mix_fused(dev_x(x), dev(W), dev(sc), dev(bs), want_stats=True, workspace=ws,
                               path=path)
    torch.cuda.synchronize()
    got = [o.cpu().numpy() for o in out]
    assert_epilogue_close(got[:3], want[:3], f"M={M}")
    assert_mix_close(got[3], want[3], f"M={M}")
    assert np.array_equal(got[4], want[4]), f"M={M}: sq"
    assert binding.hc_mix_device_status(ws) == 0


def test_small_batches_reuse_one_workspace(path):
    """Decode-sized calls that share one workspace give the oracle's results
    every time, with and without the statistics, and leave no device error."""
    K = 2048
    W, sc, bs = hi.make_w(K=K), hi.make_scale(), hi.make_base()
    for M in (1, 5, 16):
        x = hi.make_x(M, K=K)
        want = oracle.fused(x, W, sc, bs, threads=THREADS)
        xt, Wt, sct, bst = dev_x(x), dev(W), dev(sc), dev(bs)
        ws = binding.alloc_workspace(M, K)
        for rep in range(4):
            out = binding.hc_mix_fused(xt, Wt, sct, bst, want_stats=rep % 2 == 1, workspace=ws,
                                       path=path)
            torch.cuda.synchronize()
            got = [o.cpu().numpy() for o in out]
            assert_epilogue_close(got[:3], want[:3], f"M={M} call {rep}")
            if rep % 2 == 1:
                assert_mix_close(got[3], want[3], f"M={M} call {rep}")
                assert np.array_equal(got[4], want[4]), f"M={M} call {rep}: sq"
        assert binding.hc_mix_device_status(ws) == 0


def test_paths_agree_on_overlapping_sizes():
    if not (path_available("simt") and path_available("tc")):
        pytest.fail("both kernel paths must be available")
    x, W, sc, bs = hi.make_x(256), hi.make_w(), hi.make_scale(), hi.make_base()
    a = run(x, W, sc, bs, "simt")
    b = run(x, W, sc, bs, "tc")
    assert np.array_equal(a[4], b[4])
    assert_mix_close(b[3], a[3].astype(np.float64), "simt vs tc")
    for u, v in zip(a[:3], b[:3]):
        assert np.max(np.abs(u - v)) <= 1e-5


@pytest.mark.parametrize("M,K", [(37, 2048), (300, 20480)])
def test_fullk_bit_identical_to_split_k(M, K):
    """The page's fused design (one CTA walks all of K with a running total)
    and the stock split-K layout (per-slice totals, then the ordered reduce)
    add the same values in the same order, so every output is bit-identical."""
    for p in ("simt", "simt_fullk"):
        if not path_available(p):
            pytest.fail(f"kernel path {p} is not available in this library")
    x, W = hi.make_x(M, K=K, outliers=True), hi.make_w(K=K)
    sc, bs = hi.make_scale(), hi.make_base()
    a = run(x, W, sc, bs, "simt")
    b = run(x, W, sc, bs, "simt_fullk")
    for name, u, v in zip(("pre", "post", "comb", "mix", "sq"), a, b):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32)), f"{name} differs"


@pytest.mark.parametrize("case", ["m4096", "m512_outliers", "decode"])
def test_fused_tail_bit_identical_to_separate_reduce(case):
    """The tensor-core path's in-kernel tail (grid barrier, slice-ordered reduce
    and epilogue in the contraction kernel) against the same contraction
    followed by the separate reduce kernel: the same values are added in the
    same order, so every output bit agrees."""
    for p in ("tc", "tc_staged"):
        if not path_available(p):
            pytest.fail(f"kernel path {p} is not available in this library")
    W, sc, bs = hi.make_w(), hi.make_scale(), hi.make_base()
    if case == "decode":
        xs = [np.ascontiguousarray(hi.make_x(256)[:M]) for M in (1, 4, 16, 64, 128, 256)]
    else:
        xs = [hi.make_x(4096)] if case == "m4096" else [hi.make_x(512, outliers=True)]
    for x in xs:
        xt = dev_x(x)
        a = run(x, W, sc, bs, "tc", x_dev=xt)
        b = run(x, W, sc, bs, "tc_staged", x_dev=xt)
        for name, u, v in zip(("pre", "post", "comb", "mix", "sq"), a, b):
            assert np.array_equal(u.view(np.uint32), v.view(np.uint32)), \
                f"{case} M={x.shape[0]}: {name} differs"


# ---- tf32x3 mode: the page's chunk arithmetic (big = tf32 RNA of W, small =
# W - big, dot(x, small) then dot(x, big) per chunk as tf32 MMAs).  The tensor
# core rounds inside every chunk dot, so the mode is held to a bound derived
# from that arithmetic rather than to the exact path's tolerance: per chunk,
# 16 accumulations at fp32 precision (16 * 2^-23) plus the tf32 truncation of
# the small part (2^-21) stay below 2^-19 + 2^-21 of sum |x| |W|, and 2^-18
# leaves room for the slice and total additions that follow.

def tf32x3_bound(x, W):
    xf = hi.bf16_bits_to_f32(x).astype(np.float64)
    return 2.0 ** -18 * (np.abs(xf) @ np.abs(W.astype(np.float64)).T)


@pytest.fixture(scope="module")
def tf32x3():
    if not path_available("tc_tf32x3"):
        pytest.fail("kernel path tc_tf32x3 is not available in this library")
    return "tc_tf32x3"


@pytest.mark.parametrize("case", ["m7_k256", "ragged300_k2048", "m16", "m512_outliers", "m4096"])
def test_tf32x3_within_bound(tf32x3, case):
    M, K, outl = {"m7_k256": (7, 256, False), "ragged300_k2048": (300, 2048, False),
                  "m16": (16, 20480, False), "m512_outliers": (512, 20480, True),
                  "m4096": (4096, 20480, False)}[case]
    x, W = hi.make_x(M, K=K, outliers=outl), hi.make_w(K=K)
    sc, bs = hi.make_scale(), hi.make_base()
    want_mix, want_sq = oracle.stats(x, W, threads=THREADS)
    got = run(x, W, sc, bs, tf32x3)
    d = np.abs(got[3].astype(np.float64) - want_mix)
    bound = tf32x3_bound(x, W)
    assert (d <= bound).all(), f"{case}: {(d > bound).sum()} outputs beyond 2^-18 sum|x||W|"
    assert np.array_equal(got[4], want_sq), f"{case}: sq not bit-identical"
    # the epilogue of this path's own statistics
    want_ep = oracle.epilogue(got[3], got[4], K, sc, bs, threads=THREADS)
    assert_epilogue_close(got[:3], want_ep, case)
    print(f"tf32x3 {case}: max |mix error| / bound = {(d / bound).max():.4f}")


def test_tf32x3_exact_on_grid_inputs(tf32x3):
    """x in {-2..2}, W = a + b 2^-12 with a, b in {-5..5}: W splits into a big
    part and a small part that tf32 holds exactly, every product and every
    partial sum the MMAs, the slices and the total form is a multiple of
    2^-12 below 2^10, so the result is the exact sum.  A dropped small part,
    a wrong sign, column or chunk shows up as a wrong bit pattern."""
    rng = np.random.default_rng(11)
    M, K = 130, 1024
    xi = rng.integers(-2, 3, size=(M, K)).astype(np.float64)
    W64 = rng.integers(-5, 6, size=(24, K)) + rng.integers(-5, 6, size=(24, K)) * 2.0 ** -12
    W = W64.astype(np.float32)
    assert np.array_equal(W.astype(np.float64), W64)
    # every partial sum the path forms stays below 2^10 on the 2^-12 grid
    prods = xi[:, None, :] * W64[None, :, :]
    chunk = prods.reshape(M, 24, K // 64, 64)
    assert (np.abs(chunk).sum(axis=3) < 2 ** 10).all()
    cd = chunk.sum(axis=3)  # chunk dots, exact
    slices = cd.reshape(M, 24, K // 256, 4)
    assert (np.abs(np.cumsum(slices, axis=3)) < 2 ** 10).all()
    assert (np.abs(np.cumsum(slices.sum(axis=3), axis=2)) < 2 ** 10).all()
    exact = prods.sum(axis=2)
    got = run(hi.bf16_bits_from_f64(xi), W, hi.make_scale(), hi.make_base(), tf32x3)
    assert np.array_equal(got[3].astype(np.float64), exact), "tf32x3 grid inputs not exact"


def test_tf32x3_strided_and_decode_sizes(tf32x3):
    """Row pitches wider than K (x and W views of wider buffers) and the
    decode sizes, held to the same bound; the run is repeatable bit for bit."""
    K, M = 1024, 70
    rng = np.random.default_rng(8)
    xs = hi.bf16_bits_from_f64(rng.standard_normal((M, K + 64)))
    Wf = (rng.standard_normal((24, K + 32)) * 0.03).astype(np.float32)
    x, W = np.ascontiguousarray(xs[:, :K]), np.ascontiguousarray(Wf[:, :K])
    want_mix, want_sq = oracle.stats(x, W)
    out = binding.hc_mix_stats(dev_x(xs)[:, :K], dev(Wf)[:, :K], path=tf32x3)
    torch.cuda.synchronize()
    mix, sq = (o.cpu().numpy() for o in out)
    assert (np.abs(mix.astype(np.float64) - want_mix) <= tf32x3_bound(x, W)).all()
    assert np.array_equal(sq, want_sq)
    xd, Wd = hi.make_x(256), hi.make_w()
    for Md in (1, 4, 64, 256):
        xm = np.ascontiguousarray(xd[:Md])
        want_mix, want_sq = oracle.stats(xm, Wd, threads=THREADS)
        a = [o.cpu().numpy() for o in binding.hc_mix_stats(dev_x(xm), dev(Wd), path=tf32x3)]
        b = [o.cpu().numpy() for o in binding.hc_mix_stats(dev_x(xm), dev(Wd), path=tf32x3)]
        assert (np.abs(a[0].astype(np.float64) - want_mix) <= tf32x3_bound(xm, Wd)).all(), Md
        assert np.array_equal(a[1], want_sq), Md
        assert all(np.array_equal(u, v) for u, v in zip(a, b)), f"M={Md} not repeatable"


def test_tf32x3_is_not_auto():
    assert binding.hc_mix_auto_path(4096) != "tc_tf32x3"
    assert binding.hc_mix_auto_path(1) != "tc_tf32x3"


@pytest.mark.parametrize("M,K", [(1, 20480), (130, 20480), (4096, 20480), (130, 131072)])
def test_fused_packed_matches_fused(M, K):
    """W packed once gives the tensor-core path's results bit for bit, and a
    repacked buffer follows a new W."""
    if not path_available("tc"):
        pytest.fail("kernel path tc is not available in this library")
    x = dev_x(hi.make_x(M, K=K, outliers=True))
    sc, bs = dev(hi.make_scale()), dev(hi.make_base())
    packed = None
    for seed in (1, 7):
        W = dev(hi.make_w(K=K, seed=seed))
        packed = binding.pack_w(W, packed=packed)
        a = binding.hc_mix_fused(x, W, sc, bs, want_stats=True, path="tc")
        b = binding.hc_mix_fused_packed(x, packed, sc, bs, want_stats=True)
        torch.cuda.synchronize()
        for name, u, v in zip(("pre", "post", "comb", "mix", "sq"), a, b):
            assert torch.equal(u.view(torch.int32), v.view(torch.int32)), f"seed {seed}: {name}"


def test_stack86_m16384_sampled():
    """The 43-layer stack: 86 calls at M=16384 with distinct W / scale / base,
    captured once in a CUDA graph as the benchmark runs it.  Sampled rows of every
    call are checked element by element; every row is checked for the
    properties that hold at any size."""
    M, K, calls = 16384, 20480, 86
    x = hi.make_x(M)
    xt = dev_x(x)
    params = []
    for i in range(calls):
        sw, ss, sb = hi.layer_seeds(i)
        params.append((hi.make_w(seed=sw), hi.make_scale(seed=ss), hi.make_base(seed=sb)))
    dparams = [(dev(W), dev(s), dev(b)) for W, s, b in params]
    ws = binding.alloc_workspace(M, K)
    outs = [(torch.empty(M, 4, device="cuda"), torch.empty(M, 4, device="cuda"),
             torch.empty(M, 4, 4, device="cuda"), torch.empty(M, 24, device="cuda"),
             torch.empty(M, device="cuda")) for _ in range(calls)]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        binding.hc_mix_fused(xt, *dparams[0], out=outs[0], workspace=ws)  # warm-up
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(calls):
                binding.hc_mix_fused(xt, *dparams[i], out=outs[i], workspace=ws)
        g.replay()
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, M, 331), [M - 1]]))
    xs = np.ascontiguousarray(x[rows])
    for i in range(calls):
        W, s, b = params[i]
        want = oracle.fused(xs, W, s, b, threads=THREADS)
        got = [o.cpu().numpy() for o in outs[i]]
        assert_epilogue_close([got[0][rows], got[1][rows], got[2][rows]], want[:3], f"call {i}")
        assert_mix_close(got[3][rows], want[3], f"call {i}")
        assert np.array_equal(got[4][rows], want[4])
        pre, post, comb = got[:3]
        assert np.all((pre > 0) & (pre < 1)) and np.all((post > 0) & (post < 2))
        assert np.all(comb > 0)
        assert np.max(np.abs(comb.sum(1) - 1)) < 1e-5
    assert binding.hc_mix_device_status(ws) == 0


@pytest.mark.gpu
def test_self_check_paths_agree():
    """The first-call self-check: both contraction kernels agree on seeded and
    integer-valued inputs."""
    if not (path_available("simt") and path_available("tc")):
        pytest.skip("both paths needed")
    rep = binding.self_check()
    assert rep["ok"], rep
    assert rep["integer_exact"]
    assert rep["max_ratio"] <= 1.0
