"""The C ABI's own entry points, called through ctypes with raw device pointers.

hc_mix_stats and hc_mix_fused take the library's AUTO choice of kernel (the
calls a user makes); the binding's tests mostly go through the `_ex` forms with
an explicit path, so these are checked here on their own against the CPU
oracle.  A long replay of the same calls from a CUDA graph checks that every
bounded wait inside the kernels completes (the device error word stays 0) and
that the results do not change from one replay to the next.
"""
import os

import numpy as np
import pytest
import torch

import hcmix_inputs as hi
import oracle
from hyper_connection_mix_gb300 import binding

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1
ITERS, RMS_EPS, HC_EPS = 20, 1e-6, 0.0


def dev_x(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_mix_close(g, o, what):
    thr = np.maximum(2e-6 * np.abs(o.astype(np.float64)), 1e-6)
    d = np.abs(g.astype(np.float64) - o)
    assert (d <= thr).all(), f"{what}: mix max ratio {(d / thr).max():.3f}"


def inputs(M):
    x = hi.make_x(M)
    return x, hi.make_w(), hi.make_scale(), hi.make_base()


def c_fused(L, xt, Wt, sct, bst, outs, ws, stream):
    M, K = xt.shape
    pre, post, comb, mix, sq = outs
    return L.hc_mix_fused(xt.data_ptr(), xt.stride(0), Wt.data_ptr(), Wt.stride(0), M, K, 24, 4,
                          sct.data_ptr(), bst.data_ptr(), ITERS, RMS_EPS, HC_EPS,
                          pre.data_ptr(), post.data_ptr(), comb.data_ptr(),
                          None if mix is None else mix.data_ptr(),
                          None if sq is None else sq.data_ptr(),
                          ws.data_ptr(), ws.numel(), stream)


def outputs(M, stats=True):
    f = lambda *s: torch.empty(*s, device="cuda")
    return (f(M, 4), f(M, 4), f(M, 4, 4), f(M, 24) if stats else None, f(M) if stats else None)


@pytest.mark.parametrize("M", [1, 4096])
def test_hc_mix_fused_entry_point(M):
    L = binding.lib()
    x, W, sc, bs = inputs(M)
    want = oracle.fused(x, W, sc, bs, ITERS, RMS_EPS, HC_EPS, threads=THREADS)
    xt, Wt, sct, bst = dev_x(x), dev(W), dev(sc), dev(bs)
    ws = binding.alloc_workspace(M, x.shape[1])
    outs = outputs(M)
    stream = torch.cuda.current_stream().cuda_stream
    assert c_fused(L, xt, Wt, sct, bst, outs, ws, stream) == 0
    torch.cuda.synchronize()
    got = [o.cpu().numpy() for o in outs]
    for name, g, o in zip(("pre", "post", "comb"), got[:3], want[:3]):
        assert np.max(np.abs(g.astype(np.float64) - o)) <= 1e-5, f"M={M} {name}"
    assert_mix_close(got[3], want[3], f"M={M}")
    assert np.array_equal(got[4], want[4]), f"M={M} sq"
    # without the optional statistics
    outs2 = outputs(M, stats=False)
    assert c_fused(L, xt, Wt, sct, bst, outs2, ws, stream) == 0
    torch.cuda.synchronize()
    for a, b in zip(outs[:3], outs2[:3]):
        assert torch.equal(a, b)
    assert L.hc_mix_device_status(ws.data_ptr(), stream) == 0


@pytest.mark.parametrize("M", [1, 4096])
def test_hc_mix_stats_and_sinkhorn_entry_points(M):
    L = binding.lib()
    x, W, sc, bs = inputs(M)
    want = oracle.fused(x, W, sc, bs, ITERS, RMS_EPS, HC_EPS, threads=THREADS)
    xt, Wt, sct, bst = dev_x(x), dev(W), dev(sc), dev(bs)
    K = x.shape[1]
    ws = binding.alloc_workspace(M, K)
    mix, sq = torch.empty(M, 24, device="cuda"), torch.empty(M, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = L.hc_mix_stats(xt.data_ptr(), xt.stride(0), Wt.data_ptr(), Wt.stride(0), M, K, 24,
                        mix.data_ptr(), sq.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert st == 0
    pre, post, comb = outputs(M, stats=False)[:3]
    st = L.hc_mix_sinkhorn(mix.data_ptr(), sq.data_ptr(), M, K, 24, 4, sct.data_ptr(),
                           bst.data_ptr(), ITERS, RMS_EPS, HC_EPS, pre.data_ptr(),
                           post.data_ptr(), comb.data_ptr(), stream)
    assert st == 0
    torch.cuda.synchronize()
    assert_mix_close(mix.cpu().numpy(), want[3], f"M={M}")
    assert np.array_equal(sq.cpu().numpy(), want[4]), f"M={M} sq"
    for name, g, o in zip(("pre", "post", "comb"), (pre, post, comb), want[:3]):
        assert np.max(np.abs(g.cpu().numpy().astype(np.float64) - o)) <= 1e-5, f"M={M} {name}"


@pytest.mark.parametrize("M", [1, 4096])
def test_long_graph_replay_is_clean_and_repeatable(M):
    """200 back-to-back hc_mix_fused calls replayed from CUDA graphs: no
    bounded wait runs out (device error word 0) and every replay writes the
    same bits."""
    L = binding.lib()
    x, W, sc, bs = inputs(M)
    xt, Wt, sct, bst = dev_x(x), dev(W), dev(sc), dev(bs)
    ws = binding.alloc_workspace(M, x.shape[1])
    outs = outputs(M)
    stream = torch.cuda.Stream()
    s = stream.cuda_stream
    with torch.cuda.stream(stream):
        assert c_fused(L, xt, Wt, sct, bst, outs, ws, s) == 0
        torch.cuda.synchronize()
        first = [o.clone() for o in outs]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(10):
                assert c_fused(L, xt, Wt, sct, bst, outs, ws, s) == 0
        for _ in range(20):
            g.replay()
    torch.cuda.synchronize()
    assert L.hc_mix_device_status(ws.data_ptr(), s) == 0
    for a, b in zip(first, outs):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
