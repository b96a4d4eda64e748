"""Pins of the work accounting against the paper's printed numbers.

"Gaussian Mixture Attention" (Huang & Raza, 2026), Appendix B: the worked example of
the matrix-chain cost (Eq. 43-44), stored with its citation in
tests/golden/appendix_b_chain_cost.txt, and the GMA identification of Eq. 45-48
(A = Gamma^Q [N x K], B = Gamma^K^T [K x N], C = V [N x dv]).
"""
import os

from gaussian_mixture_latent_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "appendix_b_chain_cost.txt")


def read_golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def test_chain_cost_matches_the_printed_example():
    g = read_golden()
    left, right = accounting.chain_cost(g["m"], g["n"], g["p"], g["q"])
    assert left == g["cost_AB_then_C"]
    assert right == g["cost_A_then_BC"]
    assert left // right == g["ratio"] and left % right == 0


def test_gma_parenthesisation_costs_two_n_k_dv():
    # Eq. 48: Gamma^Q ((Gamma^K)^T V) costs N K dv + N K dv; the explicit affinity (Eq. 45)
    # costs N^2 K + N^2 dv
    for N, K, dv in ((8192, 64, 64), (131072, 256, 128), (7, 3, 5)):
        left, right = accounting.chain_cost(N, K, N, dv)
        assert right == 2 * N * K * dv
        assert left == N * K * N + N * N * dv
