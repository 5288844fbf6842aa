"""Thin ctypes binding to libhcmix.so, with the C ABI's names.

Argument marshalling only: shapes and dtypes of torch tensors are turned into
pointers, strides and sizes, the current CUDA stream is passed through, and a
non-OK status raises HcMixError.  Every step of the computation runs in the
library's CUDA kernels; if the library has not been built this module raises
instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libhcmix.so")

MIX = 24
HC = 4

STATUS = {0: "HCMIX_OK", 1: "HCMIX_ERR_INVALID_ARG", 2: "HCMIX_ERR_ALIGNMENT",
          3: "HCMIX_ERR_UNSUPPORTED", 4: "HCMIX_ERR_WORKSPACE", 5: "HCMIX_ERR_CUDA",
          6: "HCMIX_ERR_DEVICE"}
PATHS = {"auto": 0, "simt": 1, "tc": 2, "simt_fullk": 3, "tc_tf32x3": 4, "tc_staged": 5}

# every symbol include/hcmix.h declares
EXPORTS = ("hc_mix_workspace_bytes", "hc_mix_stats", "hc_mix_sinkhorn", "hc_mix_fused",
           "hc_mix_stats_ex", "hc_mix_fused_ex", "hc_mix_contract_ex", "hc_mix_auto_path",
           "hc_mix_device_status", "hc_mix_status_string", "hc_mix_fused_noalloc",
           "hc_mix_noalloc_device_status", "hc_mix_packed_w_bytes", "hc_mix_pack_w",
           "hc_mix_fused_packed")


class HcMixError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load libhcmix.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libhcmix.so not found at {LIB_PATH}; "
                                   "build it with __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I, F, S = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                               ctypes.c_size_t)
            L.hc_mix_workspace_bytes.restype = S
            L.hc_mix_workspace_bytes.argtypes = [I64, I64, I]
            stats_args = [P, I64, P, I64, I64, I64, I, P, P, P, S, P]
            L.hc_mix_stats.restype = I
            L.hc_mix_stats.argtypes = stats_args
            L.hc_mix_stats_ex.restype = I
            L.hc_mix_stats_ex.argtypes = stats_args + [I]
            L.hc_mix_sinkhorn.restype = I
            L.hc_mix_sinkhorn.argtypes = [P, P, I64, I64, I, I, P, P, I, F, F, P, P, P, P]
            fused_args = [P, I64, P, I64, I64, I64, I, I, P, P, I, F, F, P, P, P, P, P, P, S, P]
            L.hc_mix_fused.restype = I
            L.hc_mix_fused.argtypes = fused_args
            L.hc_mix_fused_ex.restype = I
            L.hc_mix_fused_ex.argtypes = fused_args + [I]
            L.hc_mix_contract_ex.restype = I
            L.hc_mix_contract_ex.argtypes = [P, I64, P, I64, I64, I64, I, P, S, P, I]
            L.hc_mix_fused_noalloc.restype = I
            L.hc_mix_fused_noalloc.argtypes = [P, I64, P, I64, I64, I64, I, I, P, P, I, F, F,
                                               P, P, P, P, P, P]
            L.hc_mix_noalloc_device_status.restype = I
            L.hc_mix_noalloc_device_status.argtypes = [P]
            L.hc_mix_packed_w_bytes.restype = S
            L.hc_mix_packed_w_bytes.argtypes = [I64, I]
            L.hc_mix_pack_w.restype = I
            L.hc_mix_pack_w.argtypes = [P, I64, I64, I, P, S, P]
            L.hc_mix_fused_packed.restype = I
            L.hc_mix_fused_packed.argtypes = [P, I64, P, S, I64, I64, I, I, P, P, I, F, F,
                                              P, P, P, P, P, P, S, P]
            L.hc_mix_auto_path.restype = I
            L.hc_mix_auto_path.argtypes = [I64]
            L.hc_mix_device_status.restype = I
            L.hc_mix_device_status.argtypes = [P, P]
            L.hc_mix_status_string.restype = ctypes.c_char_p
            L.hc_mix_status_string.argtypes = [I]
            _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise HcMixError(status, where)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace_bytes(M: int, K: int, mix: int = MIX) -> int:
    return int(lib().hc_mix_workspace_bytes(M, K, mix))


HEADER_BYTES = 256  # the workspace's device error word and grid-barrier counter


def alloc_workspace(M: int, K: int, device=None) -> torch.Tensor:
    """Workspace (uint8) sized for M rows, its header zeroed (the rest is
    written before it is read); torch's allocator aligns it to 512 B."""
    n = workspace_bytes(M, K)
    if n == 0:
        raise HcMixError(3, "workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    ws[:HEADER_BYTES].zero_()
    return ws


def _check_x(x: torch.Tensor) -> None:
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1):
        raise ValueError("x must be a 2-D CUDA bf16 tensor with unit inner stride")


def _check_w(W: torch.Tensor) -> None:
    if not (W.is_cuda and W.dtype == torch.float32 and W.dim() == 2 and W.stride(1) == 1):
        raise ValueError("W must be a 2-D CUDA fp32 tensor with unit inner stride")


def _f32(like: torch.Tensor, *shape) -> torch.Tensor:
    """An uninitialised fp32 tensor of `shape` on `like`'s device."""
    return like.new_empty(shape, dtype=torch.float32)


def _hc_outputs(like: torch.Tensor, M: int):
    """Output buffers (pre[M, 4], post[M, 4], comb[M, 4, 4]) on `like`'s device."""
    return (_f32(like, M, HC), _f32(like, M, HC), _f32(like, M, HC, HC))


def hc_mix_stats(x: torch.Tensor, W: torch.Tensor, mix_out=None, sq_out=None, workspace=None,
                 stream=None, path: str = "auto"):
    """(mix[M, 24], sq[M]) fp32 on x's device."""
    _check_x(x); _check_w(W)
    M, K = x.shape
    mix_out = _f32(x, M, W.shape[0]) if mix_out is None else mix_out
    sq_out = _f32(x, M) if sq_out is None else sq_out
    workspace = alloc_workspace(M, K, x.device) if workspace is None else workspace
    st = lib().hc_mix_stats_ex(_ptr(x), x.stride(0), _ptr(W), W.stride(0), M, K, W.shape[0],
                               _ptr(mix_out), _ptr(sq_out), _ptr(workspace), workspace.numel(),
                               _stream(stream), PATHS[_auto(path, x.device)])
    _check(st, "hc_mix_stats")
    return mix_out, sq_out


def hc_mix_sinkhorn(mix: torch.Tensor, sq: torch.Tensor, K: int, hc_scale: torch.Tensor,
                    hc_base: torch.Tensor, sinkhorn_iters: int = 20, rms_eps: float = 1e-6,
                    hc_eps: float = 0.0, out=None, stream=None):
    """(pre[M, 4], post[M, 4], comb[M, 4, 4]) from mix[M, 24] and sq[M]."""
    M = mix.shape[0]
    pre, post, comb = out if out is not None else _hc_outputs(mix, M)
    st = lib().hc_mix_sinkhorn(_ptr(mix), _ptr(sq), M, K, mix.shape[1], HC, _ptr(hc_scale),
                               _ptr(hc_base), sinkhorn_iters, rms_eps, hc_eps, _ptr(pre),
                               _ptr(post), _ptr(comb), _stream(stream))
    _check(st, "hc_mix_sinkhorn")
    return pre, post, comb


def hc_mix_fused(x: torch.Tensor, W: torch.Tensor, hc_scale: torch.Tensor,
                 hc_base: torch.Tensor, sinkhorn_iters: int = 20, rms_eps: float = 1e-6,
                 hc_eps: float = 0.0, want_stats: bool = False, out=None, workspace=None,
                 stream=None, path: str = "auto"):
    """(pre, post, comb) or, with want_stats, (pre, post, comb, mix, sq)."""
    _check_x(x); _check_w(W)
    M, K = x.shape
    dev = x.device
    if out is None:
        out = _hc_outputs(x, M)
        if want_stats:
            out += (_f32(x, M, W.shape[0]), _f32(x, M))
    pre, post, comb = out[:3]
    mix_out, sq_out = (out[3], out[4]) if len(out) == 5 else (None, None)
    workspace = alloc_workspace(M, K, dev) if workspace is None else workspace
    st = lib().hc_mix_fused_ex(_ptr(x), x.stride(0), _ptr(W), W.stride(0), M, K, W.shape[0], HC,
                               _ptr(hc_scale), _ptr(hc_base), sinkhorn_iters, rms_eps, hc_eps,
                               _ptr(pre), _ptr(post), _ptr(comb), _ptr(mix_out), _ptr(sq_out),
                               _ptr(workspace), workspace.numel(), _stream(stream),
                               PATHS[_auto(path, x.device)])
    _check(st, "hc_mix_fused")
    return out


def hc_mix_contract(x: torch.Tensor, W: torch.Tensor, workspace: torch.Tensor, stream=None,
                    path: str = "auto") -> None:
    """The contraction phase alone, into `workspace` (timing and profiling)."""
    _check_x(x); _check_w(W)
    M, K = x.shape
    st = lib().hc_mix_contract_ex(_ptr(x), x.stride(0), _ptr(W), W.stride(0), M, K, W.shape[0],
                                  _ptr(workspace), workspace.numel(), _stream(stream),
                                  PATHS[_auto(path, x.device)])
    _check(st, "hc_mix_contract")


def pack_w(W: torch.Tensor, packed=None, stream=None) -> torch.Tensor:
    """W[24, K] packed once into the tensor-core operand format (uint8 on W's
    device, 256-byte aligned) for hc_mix_fused_packed."""
    _check_w(W)
    K = W.shape[1]
    n = int(lib().hc_mix_packed_w_bytes(K, W.shape[0]))
    if n == 0:
        raise HcMixError(3, "hc_mix_packed_w_bytes")
    packed = torch.empty(n, dtype=torch.uint8, device=W.device) if packed is None else packed
    st = lib().hc_mix_pack_w(_ptr(W), W.stride(0), K, W.shape[0], _ptr(packed), packed.numel(),
                             _stream(stream))
    _check(st, "hc_mix_pack_w")
    return packed


def hc_mix_fused_packed(x: torch.Tensor, packed: torch.Tensor, hc_scale: torch.Tensor,
                        hc_base: torch.Tensor, sinkhorn_iters: int = 20, rms_eps: float = 1e-6,
                        hc_eps: float = 0.0, want_stats: bool = False, out=None, workspace=None,
                        stream=None):
    """hc_mix_fused on a W packed by pack_w (tensor-core path, exact limbs)."""
    _check_x(x)
    M, K = x.shape
    dev = x.device
    pre, post, comb = out if out is not None else _hc_outputs(x, M)
    mix_out = _f32(x, M, MIX) if want_stats else None
    sq_out = _f32(x, M) if want_stats else None
    workspace = alloc_workspace(M, K, dev) if workspace is None else workspace
    st = lib().hc_mix_fused_packed(_ptr(x), x.stride(0), _ptr(packed), packed.numel(), M, K, MIX,
                                   HC, _ptr(hc_scale), _ptr(hc_base), sinkhorn_iters, rms_eps,
                                   hc_eps, _ptr(pre), _ptr(post), _ptr(comb), _ptr(mix_out),
                                   _ptr(sq_out), _ptr(workspace), workspace.numel(),
                                   _stream(stream))
    _check(st, "hc_mix_fused_packed")
    return (pre, post, comb, mix_out, sq_out) if want_stats else (pre, post, comb)


def hc_mix_auto_path(M: int) -> str:
    return {v: k for k, v in PATHS.items()}[int(lib().hc_mix_auto_path(M))]


# ---------------------------------------------------------------- self-check

_self_checked: dict = {}


def self_check(device=None, M: int = 200, K: int = 1024) -> dict:
    """Runs both contraction kernels on small seeded inputs and compares them.

    Two independent GPU implementations (the tcgen05 tensor-core kernel and
    the CUDA-core split-K kernel) must agree on mix and sq within the path's
    tolerance (|a - b| <= max(2e-6 |b|, 1e-6)); on integer-valued inputs, where
    every partial sum is an integer below 2^24 and so every correct evaluation
    order gives the same bits, they must agree bit for bit, and one-hot rows
    must return the selected column of W exactly.  No arithmetic of the path
    runs here: the binding only compares the kernels' outputs.  Returns
    {"ok": bool, "max_ratio": worst |a - b| / tolerance, "integer_exact": bool}.
    Synchronises the device; not for use during CUDA-graph capture.
    """
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(12345)
    x = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    x[:, ::97] *= 20  # a few outlier channels
    W = torch.randn(MIX, K, generator=g, device=dev) * K ** -0.5
    mt, st = hc_mix_stats(x, W, path="tc")
    ms, ss = hc_mix_stats(x, W, path="simt")
    ratio = 0.0
    for a, b in ((mt, ms), (st, ss)):
        tol = torch.clamp(2e-6 * b.abs(), min=1e-6)
        ratio = max(ratio, float(((a - b).abs() / tol).max()))
    xi = torch.randint(-4, 5, (M, K), generator=g, device=dev).to(torch.bfloat16)
    wi = torch.randint(-8, 9, (MIX, K), generator=g, device=dev).float()
    mi_t, sq_t = hc_mix_stats(xi, wi, path="tc")
    mi_s, sq_s = hc_mix_stats(xi, wi, path="simt")
    ok_int = bool(torch.equal(mi_t, mi_s)) and bool(torch.equal(sq_t, sq_s))
    # one-hot rows: row r has a single 1 at column cols[r], so mix[r] = W[:, cols[r]]
    cols = torch.randint(0, K, (M,), generator=g, device=dev)
    onehot = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
    onehot[torch.arange(M, device=dev), cols] = 1
    for path in ("tc", "simt"):
        mo, _ = hc_mix_stats(onehot, W, path=path)
        ok_int = ok_int and bool(torch.equal(mo, W[:, cols].T))
    torch.cuda.synchronize(dev)
    return {"ok": ratio <= 1.0 and ok_int, "max_ratio": ratio, "integer_exact": ok_int}


def _auto(path: str, device: torch.device) -> str:
    """With HCMIX_SELF_CHECK=1, the first AUTO call on a device runs self_check
    and keeps to the CUDA-core kernel if the tensor-core kernel disagrees."""
    if path != "auto" or os.environ.get("HCMIX_SELF_CHECK") != "1":
        return path
    idx = device.index if device.index is not None else torch.cuda.current_device()
    if idx not in _self_checked:
        if torch.cuda.is_current_stream_capturing():
            return path
        _self_checked[idx] = self_check(torch.device("cuda", idx))
    return "auto" if _self_checked[idx]["ok"] else "simt"


def hc_mix_device_status(workspace: torch.Tensor, stream=None) -> int:
    return int(lib().hc_mix_device_status(_ptr(workspace), _stream(stream)))


def hc_mix_status_string(status: int) -> str:
    return lib().hc_mix_status_string(status).decode()
