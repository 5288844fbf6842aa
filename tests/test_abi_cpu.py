"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/hcmix.h declares, sizes its workspace, and rejects bad
arguments before launching anything."""
import ctypes
import os
import re

import pytest

from hyper_connection_mix_gb300 import binding
from hyper_connection_mix_gb300 import build as hbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    hbuild.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "hcmix.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hc_mix_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    assert sorted(binding.EXPORTS) == names
    for n in names:
        assert hasattr(L, n), n


def test_workspace_bytes(L):
    K = 20480
    n = binding.workspace_bytes(4096, K)
    parts = 80 * 25 * 4096 * 4
    assert n == 256 + parts  # header (error word, grid-barrier words) + partials
    assert binding.workspace_bytes(1, K) == 256 + 80 * 25 * 128 * 4
    assert binding.workspace_bytes(0, K) == 256
    assert binding.workspace_bytes(16, 20481) == 0     # K not a multiple of 256
    assert binding.workspace_bytes(16, K, mix=16) == 0  # mix != 24
    assert binding.workspace_bytes(-1, K) == 0


def test_path_enum_matches_binding():
    """The binding's path names carry the values hcmix_path declares."""
    src = open(os.path.join(ROOT, "include", "hcmix.h")).read()
    body = re.search(r"typedef enum \{([^}]*)\} hcmix_path;", src).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    declared = {m.group(1).lower(): int(m.group(2))
                for m in re.finditer(r"HCMIX_PATH_(\w+)\s*=\s*(\d+)", body)}
    assert declared == binding.PATHS


def test_packed_w_validation(L):
    """The pack-once entry points reject bad arguments before launching."""
    K = 20480
    assert binding.lib().hc_mix_packed_w_bytes(K, 24) == 4 * 24 * K * 2
    assert binding.lib().hc_mix_packed_w_bytes(K, 16) == 0
    assert binding.lib().hc_mix_packed_w_bytes(1000, 24) == 0
    n = 4 * 24 * K * 2
    pack = L.hc_mix_pack_w
    assert pack(None, K, K, 24, 0x100000, n, None) == 1
    assert pack(0x20000, K - 4, K, 24, 0x100000, n, None) == 1   # stride < K
    assert pack(0x20004, K, K, 24, 0x100000, n, None) == 2       # W misaligned
    assert pack(0x20000, K, K, 24, 0x100080, n, None) == 2       # packed not 256-byte aligned
    assert pack(0x20000, K, K, 24, 0x100000, n - 1, None) == 4   # packed too small
    assert pack(0x20000, K, 1000, 24, 0x100000, n, None) == 3
    fp = L.hc_mix_fused_packed
    P = 0x10000
    args = dict(x=P, xs=K, pw=0x200000, pb=n, M=8, K=K, mix=24, hc=4, sc=P, bs=P, it=20,
                re=1e-6, he=0.0, pre=P, post=P, comb=P, mo=None, so=None, wk=0x800000,
                wkb=1 << 30)

    def call(**kw):
        a = dict(args, **kw)
        return fp(a["x"], a["xs"], a["pw"], a["pb"], a["M"], a["K"], a["mix"], a["hc"], a["sc"],
                  a["bs"], a["it"], a["re"], a["he"], a["pre"], a["post"], a["comb"], a["mo"],
                  a["so"], a["wk"], a["wkb"], None)
    assert call(pw=None) == 1
    assert call(pw=0x200080) == 2
    assert call(pb=n - 1) == 4
    assert call(wkb=1024) == 4
    assert call(x=0x10002) == 2
    assert call(hc=3) == 3
    assert call(it=-1) == 1
    assert call(M=0, x=None, pw=None, wk=None) == 0


def test_status_strings(L):
    for code, name in binding.STATUS.items():
        assert binding.hc_mix_status_string(code).startswith(name)


def _stats(L, x=0x10000, xs=1024, W=0x20000, ws=1024, M=8, K=1024, mix=24, mo=0x30000,
           so=0x40000, wk=0x100000, wkb=1 << 30, path=0):
    return L.hc_mix_stats_ex(x, xs, W, ws, M, K, mix, mo, so, wk, wkb, None, path)


def test_host_validation_rejects_before_launch(L):
    # every case fails validation, so nothing is launched and no GPU is touched
    assert _stats(L, M=-1) == 1
    assert _stats(L, K=1000) == 3
    assert _stats(L, K=0) == 1
    assert _stats(L, mix=16) == 3
    assert _stats(L, K=1 << 25, xs=1 << 25, ws=1 << 25) == 3
    assert _stats(L, xs=512) == 1            # stride < K
    assert _stats(L, x=0x10002) == 2         # x not 16-byte aligned
    assert _stats(L, xs=1028) == 2           # row pitch not 16 bytes
    assert _stats(L, W=0x20004) == 2
    assert _stats(L, ws=1026) == 2
    assert _stats(L, wk=0x100080) == 2       # workspace not 256-byte aligned
    assert _stats(L, wkb=1024) == 4          # workspace too small
    assert _stats(L, x=None) == 1
    assert _stats(L, path=7) == 1
    assert _stats(L, path=6) == 1            # one past the last declared path
    assert _stats(L, path=-1) == 1
    assert _stats(L, mo=None) == 1
    assert _stats(L, M=0, x=None, W=None, wk=None) == 0  # empty: nothing to do


def test_fused_and_sinkhorn_validation(L):
    P = 0x10000
    base = dict(x=P, xs=1024, W=P, ws=1024, M=4, K=1024, mix=24, hc=4, sc=P, bs=P, it=20,
                pre=P, post=P, comb=P, wk=0x100000, wkb=1 << 30)

    def fused(**kw):
        a = dict(base, **kw)
        return L.hc_mix_fused_ex(a["x"], a["xs"], a["W"], a["ws"], a["M"], a["K"], a["mix"],
                                 a["hc"], a["sc"], a["bs"], a["it"], 1e-6, 0.0, a["pre"],
                                 a["post"], a["comb"], None, None, a["wk"], a["wkb"], None, 0)
    assert fused(hc=3) == 3
    assert fused(it=-1) == 1
    assert fused(sc=None) == 1
    assert fused(comb=None) == 1
    assert fused(M=0, x=None) == 0
    assert fused(M=0, x=None, pre=None, post=None, comb=None) == 0  # empty outputs
    s = L.hc_mix_sinkhorn
    assert s(P, P, 4, 1024, 24, 4, P, P, -1, 1e-6, 0.0, P, P, P, None) == 1
    assert s(P, P, 4, 1024, 16, 4, P, P, 20, 1e-6, 0.0, P, P, P, None) == 3
    assert s(P, P, -4, 1024, 24, 4, P, P, 20, 1e-6, 0.0, P, P, P, None) == 1
    assert s(None, P, 4, 1024, 24, 4, P, P, 20, 1e-6, 0.0, P, P, P, None) == 1
    assert s(None, None, 0, 1024, 24, 4, P, P, 20, 1e-6, 0.0, P, P, P, None) == 0
    assert s(None, None, 0, 1024, 24, 4, None, None, 20, 1e-6, 0.0, None, None, None, None) == 0
    nf = L.hc_mix_fused_noalloc
    assert nf(None, 256, None, 256, 0, 256, 24, 4, None, None, 20, 1e-6, 0.0,
              None, None, None, None, None, None) == 0
    assert nf(P, 1024, P, 1024, 257, 20480, 24, 4, P, P, 20, 1e-6, 0.0,
              P, P, P, None, None, None) == 1        # stride < K
    assert nf(P, 20480, P, 20480, 257, 20480, 24, 4, P, P, 20, 1e-6, 0.0,
              P, P, P, None, None, None) == 4        # beyond the fixed scratch


def test_device_status_rejects_bad_workspace(L):
    assert L.hc_mix_device_status(None, None) == 1
    assert L.hc_mix_device_status(0x100080, None) == 1


def test_self_check_dispatch(monkeypatch):
    """AUTO keeps to the CUDA-core kernel on a device whose self-check failed,
    only when HCMIX_SELF_CHECK=1; forced paths are never changed."""
    import torch
    d = torch.device("cuda", 0)
    monkeypatch.delenv("HCMIX_SELF_CHECK", raising=False)
    assert binding._auto("auto", d) == "auto"
    monkeypatch.setenv("HCMIX_SELF_CHECK", "1")
    monkeypatch.setitem(binding._self_checked, 0, {"ok": False})
    assert binding._auto("auto", d) == "simt"
    assert binding._auto("tc", d) == "tc"
    monkeypatch.setitem(binding._self_checked, 0, {"ok": True})
    assert binding._auto("auto", d) == "auto"
