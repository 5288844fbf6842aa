"""hc_mix_fused_noalloc: the entry point for callers that cannot give the library
any device memory (an engine that reserved its whole memory budget up front and
forbids later cudaMalloc, or a plug-in whose host framework owns every device
allocation).  It keeps its scratch in a fixed 2 MiB device array inside the
library instead of a caller workspace.

Checked through the C ABI against hc_mix_fused's default path (which uses a
caller workspace) on two calls in a row.  Both run the same kernel with the
same arithmetic in the same order, so every output must be bit-identical; a
scratch-layout slip would show up as a changed bit before it shows up as a
tolerance failure.  This file is collected last; it must pass alone in a fresh
process and after the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

import hcmix_inputs as hi
from hyper_connection_mix_gb300 import binding

pytestmark = pytest.mark.gpu


def _dev_x(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _noalloc(L, x, W, sc, bs, outs, stream):
    M, K = x.shape
    pre, post, comb, mix, sq = outs
    return L.hc_mix_fused_noalloc(x.data_ptr(), x.stride(0), W.data_ptr(), W.stride(0), M, K, 24,
                                  4, sc.data_ptr(), bs.data_ptr(), 20, 1e-6, 0.0,
                                  pre.data_ptr(), post.data_ptr(), comb.data_ptr(),
                                  mix.data_ptr(), sq.data_ptr(), stream)


def _outs(M):
    return (torch.empty(M, 4, device="cuda"), torch.empty(M, 4, device="cuda"),
            torch.empty(M, 4, 4, device="cuda"), torch.empty(M, 24, device="cuda"),
            torch.empty(M, device="cuda"))


@pytest.mark.parametrize("M,K", [(256, 20480), (37, 20480), (129, 1024), (1, 20480), (4, 1024)])
def test_noalloc_matches_workspace_entry_point_twice(M, K):
    L = binding.lib()
    stream = torch.cuda.current_stream().cuda_stream
    x = hi.make_x(M, K=K)
    W, sc, bs = hi.make_w(K=K), hi.make_scale(), hi.make_base()
    xt = _dev_x(x)
    Wt, sct, bst = (torch.from_numpy(a).cuda() for a in (W, sc, bs))
    ref = binding.hc_mix_fused(xt, Wt, sct, bst, want_stats=True, path="auto")
    for call in range(2):
        # a different input between the two calls: the second call must not see
        # anything the first one left in the shared scratch
        outs = _outs(M)
        assert _noalloc(L, xt, Wt, sct, bst, outs, stream) == 0
        torch.cuda.synchronize()
        for name, a, b in zip(("pre", "post", "comb", "mix", "sq"), outs, ref):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"call {call}: {name}"
        other = _dev_x(hi.make_x(M, K=K, seed=7))
        assert _noalloc(L, other, Wt, sct, bst, _outs(M), stream) == 0
    assert L.hc_mix_noalloc_device_status(stream) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = binding.lib()
    M, K = 257, 20480
    xt = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    Wt = torch.zeros(24, K, device="cuda")
    sc, bs = torch.ones(3, device="cuda"), torch.zeros(24, device="cuda")
    st = _noalloc(L, xt, Wt, sc, bs, _outs(M), torch.cuda.current_stream().cuda_stream)
    assert binding.STATUS[st] == "HCMIX_ERR_WORKSPACE"
