"""Parity of cross-attention GMA (CUDA path, through the C ABI) with the fp64
oracle: "Gaussian Mixture Attention", sections 3.1 and 6 -- the queries of one
sequence read the latent memory (Eq. 5-8) of a context sequence of another length.

Metric as for the forward: per head max |O_gpu - O_ref| / max |O_ref|, bf16
tolerance 2e-2.
"""
import numpy as np
import pytest

from gaussian_mixture_latent_gb300 import inputs
from tests._util import TOL, to_device, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def make(B, H, Nq, Nkv, K, seed=4):
    q = inputs.gen_all(inputs.Workload("q", B=B, H=H, N=Nq, d=64, K=K, dv=64, dtype="bf16", causal=False,
                                       seed=seed))
    c = inputs.gen_all(inputs.Workload("c", B=B, H=H, N=Nkv, d=64, K=K, dv=64, dtype="bf16", causal=False,
                                       seed=seed + 1000))
    return dict(Qx=q["Qx"], Ky=c["Kx"], Vy=c["V"], mu=q["mu"], rho=q["rho"], alpha=q["alpha"])


def run_gpu(x, eps=1e-6):
    import gaussian_mixture_latent_gb300 as gma
    out = gma.gma_forward_cross(to_device(x["Qx"]), to_device(x["Ky"]), to_device(x["Vy"]), to_device(x["mu"]),
                                to_device(x["rho"]), to_device(x["alpha"]), eps=eps)
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    return to_f64(out)


def check(x, got, heads, rows=None, eps=1e-6):
    import oracle
    B, H = x["Qx"].shape[:2]
    worst = 0.0
    for g in heads:
        b, h = divmod(g, H)
        Q = inputs.widen(x["Qx"][b, h], "bf16")
        ref = oracle.cross_head(Q if rows is None else Q[rows], inputs.widen(x["Ky"][b, h], "bf16"),
                                inputs.widen(x["Vy"][b, h], "bf16"), x["mu"][h], x["rho"][h], x["alpha"][h],
                                1e-4, eps)
        o = got[b, h] if rows is None else got[b, h][rows]
        err = np.abs(o - ref).max() / np.abs(ref).max()
        worst = max(worst, err)
    assert np.isfinite(got).all()
    assert worst <= TOL["bf16"], worst
    return worst


CASES = [
    # name, B, H, Nq, Nkv, K
    ("short_queries_long_context", 2, 3, 333, 1000, 64),
    ("long_queries_short_context_k128", 1, 2, 1000, 200, 128),
    ("one_tile_each", 1, 4, 128, 128, 64),
    ("single_query", 2, 2, 1, 5000, 64),
    ("single_key", 1, 2, 4097, 1, 64),
    ("many_heads", 4, 16, 300, 700, 64),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_cross_parity(case):
    name, B, H, Nq, Nkv, K = case
    x = make(B, H, Nq, Nkv, K)
    check(x, run_gpu(x), list(range(B * H)))


def test_cross_with_the_sequence_itself_equals_the_bidirectional_forward():
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("self", B=2, H=3, N=900, d=64, K=64, dv=64, dtype="bf16", causal=False)
    x = inputs.gen_all(w)
    Q, Kx, V = to_device(x["Qx"]), to_device(x["Kx"]), to_device(x["V"])
    par = [to_device(x[k]) for k in ("mu", "rho", "alpha")]
    a = gma.gma_forward(Q, Kx, V, *par, eps=w.eps, causal=False)
    b = gma.gma_forward_cross(Q, Kx, V, *par, eps=w.eps)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_cross_large_context_sampled():
    # 8192 queries reading a 65536-row context, 16 heads: sampled heads and query rows
    x = make(2, 8, 8192, 65536, 64, seed=9)
    got = run_gpu(x)
    rows = np.random.default_rng(0).choice(8192, 512, replace=False)
    check(x, got, [0, 13], rows=rows)


def test_cross_errors():
    import gaussian_mixture_latent_gb300 as gma
    x = make(1, 2, 100, 50, 64)
    with pytest.raises(gma.GmaError) as e:
        gma.gma_forward_cross(to_device(x["Qx"]), to_device(x["Ky"][:, :, :0]), to_device(x["Vy"][:, :, :0]),
                              to_device(x["mu"]), to_device(x["rho"]), to_device(x["alpha"]))
    assert e.value.code == 1
