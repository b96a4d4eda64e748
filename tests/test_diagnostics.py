"""Parity of the responsibility diagnostics (CUDA path, through the C ABI) with
the fp64 oracle: "Gaussian Mixture Attention", section 5.4, Eqs. 24-29.

p is compared normwise (max |p_gpu - p_ref| / max p_ref), each scalar
statistic relatively, with the bf16-input tolerance 2e-2.  The argmax z is an
integer decided in floating point: where the oracle's top two head-averaged
responsibilities are further apart than the tolerance the GPU must pick the
same component; everywhere its pick must be within the tolerance of the
oracle's maximum (a near tie may go either way).
"""
import numpy as np
import pytest

from gaussian_mixture_latent_gb300 import inputs
from tests._util import TOL, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ZTOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_gpu(x, var_floor, B=None):
    import gaussian_mixture_latent_gb300 as gma
    Q = to_device(x["Qx"] if B is None else x["Qx"][:B])
    p, stats, z = gma.gma_diagnostics(Q, to_device(x["mu"]), to_device(x["rho"]), to_device(x["alpha"]),
                                      var_floor=var_floor)
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    return p.double().cpu().numpy(), stats.double().cpu().numpy(), z.cpu().numpy()


def oracle_gbar(Qx, mu, rho, alpha, var_floor):
    import oracle
    B, H, N, _ = Qx.shape
    K = mu.shape[1]
    g = np.zeros((B, N, K))
    for b in range(B):
        for h in range(H):
            g[b] += oracle.responsibilities(Qx[b, h], mu[h], rho[h], alpha[h], var_floor)
    return g / H


def check(w, x, got, B=None):
    import oracle
    Q = inputs.widen(x["Qx"] if B is None else x["Qx"][:B], w.dtype)
    p_ref, hu, ht, rm, z_ref = oracle.diagnostics(Q, x["mu"], x["rho"], x["alpha"], w.var_floor)
    p, stats, z = got
    assert np.abs(p - p_ref).max() / p_ref.max() <= TOL[w.dtype], (p, p_ref)
    for name, a, r in zip(("H_usage", "H_token", "R_max"), stats, (hu, ht, rm)):
        assert abs(a - r) <= TOL[w.dtype] * abs(r), f"{w.name} {name}: {a} vs {r}"
    gbar = oracle_gbar(Q, x["mu"], x["rho"], x["alpha"], w.var_floor)
    top2 = np.sort(gbar, axis=2)[:, :, -2:]
    clear = top2[:, :, 1] - top2[:, :, 0] > ZTOL
    assert np.array_equal(z[clear], z_ref[clear])
    picked = np.take_along_axis(gbar, z[:, :, None].astype(np.int64), axis=2)[:, :, 0]
    assert (picked >= gbar.max(axis=2) - ZTOL).all()
    assert clear.mean() > 0.1                     # the exact comparison is not vacuous
    return p_ref


SMALL = [
    # name, B, H, N, K, mu_std, mix_frac
    ("k64_ragged", 2, 3, 333, 64, 1.0, 0.0),
    ("k128_paper_heads", 1, 8, 1000, 128, 1.0, 0.0),
    ("single_head", 3, 1, 129, 64, 1.0, 0.0),
    ("peaked_k128", 2, 4, 500, 128, 1.0, 0.3),
    ("separated_k64", 1, 2, 300, 64, 2.0, 0.0),
    ("many_tiles_k64", 2, 6, 2000, 64, 1.0, 0.1),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_diagnostics_parity_small(case):
    name, B, H, N, K, mu_std, mix = case
    w = inputs.Workload(name, B=B, H=H, N=N, d=64, K=K, dv=64, dtype="bf16", causal=False, mu_std=mu_std,
                        mix_frac=mix, seed=5)
    x = inputs.gen_all(w)
    check(w, x, run_gpu(x, w.var_floor))


def test_diagnostics_full_size_matches_the_oracle():
    # the 96-head N = 8192 workload, every batch entry against the oracle, plus the
    # one-sequence call's per-token results equal to the full call's
    w = inputs.WORKLOADS["causal_bf16_n8192"]
    x = inputs.gen_all(w)
    full = run_gpu(x, w.var_floor)
    check(w, x, full)
    p, stats, z = full
    K = w.K
    assert abs(p.sum() - 1.0) < 1e-3
    assert 0.0 <= stats[1] <= stats[0] <= 1.0 + 1e-6
    assert 1.0 / K - 1e-6 <= stats[2] <= 1.0
    assert z.min() >= 0 and z.max() < K
    one = run_gpu(x, w.var_floor, B=1)
    assert np.array_equal(z[0], one[2][0])


def test_diagnostics_unsupported_and_empty():
    import gaussian_mixture_latent_gb300 as gma
    for K, dtype in ((256, "bf16"), (64, "f32")):
        w = inputs.Workload("u", B=1, H=2, N=100, d=64, K=K, dv=64, dtype=dtype, causal=False)
        x = inputs.gen_all(w)
        with pytest.raises(gma.GmaError) as e:
            run_gpu(x, w.var_floor)
        assert e.value.code == 2
    w = inputs.Workload("e", B=1, H=2, N=0, d=64, K=64, dv=64, dtype="bf16", causal=False)
    x = inputs.gen_all(w)
    p, stats, z = gma.gma_diagnostics(to_device(x["Qx"]), to_device(x["mu"]), to_device(x["rho"]),
                                      to_device(x["alpha"]))
    assert z.shape == (1, 0)
