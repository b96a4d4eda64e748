"""Work accounting for roofline fractions (no data, only counts).

Algorithmic work of the GMA forward per head of N rows counts what the method
itself must move and compute -- one read of each input, one write of the
output, two flops per multiply-add -- with the responsibilities kept on chip:

  bytes  = e_in * N * (2 d + dv) + e_out * N * dv + 4 * (2 K d + K)
  flops  = 8 N K d            log-densities of Qx and Kx as [X, X^2] (N x 2d) . (2d x K)
         + 4 N K (dv + 1)     write Gamma^K^T [V | 1] and read Gamma^Q [Vt | Z]

This relates to the paper's routing cost (section 3.4, Eq. 12),
2 N K d_r + 2 N K d_v + 4 N K + N d_v operations counted one per
multiply-add with no separate x^2 term: here each multiply-add is two flops
and the diagonal log-density needs both x and x^2 terms.  Causal work is
counted the same (the recurrence); chunking adds executed work that is not
credited.

``chain_cost`` is the matrix-chain count of Appendix B (Eq. 43-44), pinned by
the paper's worked example in tests/golden.
"""
from __future__ import annotations

ELEM = {"f32": 4, "bf16": 2}


def chain_cost(m: int, n: int, p: int, q: int) -> tuple[int, int]:
    """Scalar multiplications of (AB)C and A(BC) for A m x n, B n x p, C p x q (Eq. 43, 44)."""
    return m * n * p + m * p * q, n * p * q + m * n * q


def routing_cost(N: int, K: int, dr: int, dv: int) -> int:
    """Eq. 12: approximate routing operation count per head."""
    return 2 * N * K * dr + 2 * N * K * dv + 4 * N * K + N * dv


def routing_storage(N: int, K: int, dv: int) -> int:
    """Section 3.4: routing-specific activation entries per head, 2NK + K dv + K + N dv."""
    return 2 * N * K + K * dv + K + N * dv


def algorithmic_bytes(G, N, d, K, dv, in_dtype="bf16", out_dtype="bf16", H=None) -> int:
    e_in, e_out = ELEM[in_dtype], ELEM[out_dtype]
    params = 4 * (2 * K * d + K) * (H if H is not None else G)
    return G * (e_in * N * (2 * d + dv) + e_out * N * dv) + params


def algorithmic_flops(G, N, d, K, dv) -> int:
    return G * (8 * N * K * d + 4 * N * K * (dv + 1))


def kernel_work(name: str, G, N, d, K, dv, in_dtype="bf16", out_dtype="bf16", H=None):
    """(bound, algorithmic amount per launch, unit) of one kernel of the launch plan.

    Amounts are the kernel's share of the algorithmic work above: bytes for
    HBM-bound kernels, flops for tensor- or ALU-bound ones.
    """
    e_in, e_out = ELEM[in_dtype], ELEM[out_dtype]
    rows = G * N
    if name.startswith("simt_gamma"):
        # direct-form log-density: sub, mul, fma per (row, component, dim) = 4 flops
        return "alu", 4 * rows * K * d, "flop"
    if name in ("simt_write", "simt_read"):
        return "alu", 2 * rows * K * (dv + 1), "flop"
    if name == "simt_causal_chunk":
        return "alu", 4 * rows * K * (dv + 1), "flop"
    if name == "tc_write":
        return "hbm", rows * (e_in * (d + dv)), "byte"
    if name == "tc_read":
        return "hbm", rows * (e_in * d + e_out * dv), "byte"
    if name in ("tc_causal", "tc_causal_seg"):
        # every routing row and value in once, every output row out once
        return "hbm", rows * (e_in * (2 * d + dv) + e_out * dv), "byte"
    if name == "tc_causal_slices":
        # the component-sliced scan does all of the path's contractions
        return "tensor", algorithmic_flops(G, N, d, K, dv), "flop"
    if name == "tc_rowstats":
        return "hbm", rows * e_in * 2 * d, "byte"
    if name == "tc_combine":
        # executed (not algorithmic) traffic: the bf16 partial numerators and fp32
        # partial denominators of every component slice in, the output out
        ns = max(1, K // 64)
        return "hbm", rows * (ns * (2 * dv + 4) + e_out * dv), "byte"
    return None, 0, None
