"""Algorithmic traffic and work of the mix-statistics path (host-side model).

Per call at M rows and K columns:
  * bytes: x read once (M*K*2, bf16) plus W read once (mix*K*4, fp32); the
    96 B/row of outputs are excluded (under 0.25 % at the page's shapes);
  * flops: 2*mix*K per row for the contraction plus 2*K per row for the sum of
    squares.
The page's own figures (168 MB of activations and a 63 MB partial round trip
for the split-K stock path at 4096 rows; hc_fused page docstring) follow from
the same shapes.
"""
MIX = 24
HC = 4
SLICE = 256
CHUNK = 64


def activation_bytes(M: int, K: int) -> int:
    return M * K * 2


def weight_bytes(K: int, mix: int = MIX) -> int:
    return mix * K * 4


def algorithmic_bytes(M: int, K: int, mix: int = MIX) -> int:
    return activation_bytes(M, K) + weight_bytes(K, mix)


def output_bytes(M: int, hc: int = HC) -> int:
    return M * (2 * hc + hc * hc) * 4


def algorithmic_flops(M: int, K: int, mix: int = MIX) -> int:
    return M * (2 * mix * K + 2 * K)


def stock_partial_round_trip_bytes(M: int, num_slices: int, mix: int = MIX) -> int:
    """fp32 [num_slices, M, mix] partials written once and read once."""
    return num_slices * M * mix * 4 * 2
