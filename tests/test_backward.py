"""Parity of the backward pass (CUDA path, through the C ABI) with the fp64 oracle:
"Gaussian Mixture Attention", section 4.1 (Eqs. 17-20, through Eqs. 14-15 and the
memory products of Eqs. 5-8).

Both sides read the same inputs (bf16 inputs widened exactly), so the difference is
the kernel's fp32 arithmetic: per head and per tensor, max |g_gpu - g_ref| / max |g_ref|.
The parameter gradients are summed over the batch (the parameters are shared by every
batch entry), on the oracle side head by head.

Tolerance, from the arithmetic: a score is a 128-term fp32 sum of magnitude up to ~100
(the log-determinant and Mahalanobis terms at d = 64), so its absolute error is
~sqrt(n) u |s| ~ 1e-4 typically and n u sum|terms| ~ 1.5e-3 at worst; the
responsibilities and every gradient inherit that relative error.  A routing gradient
can be far smaller than its head's others when its exact value cancels (one row: the
key gradient is O(eps)), so the row gradients are measured against at least 1e-2 of
the head's largest routing gradient.
"""
import numpy as np
import pytest

from gaussian_mixture_latent_gb300 import inputs
from tests._util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_BWD = 1e-3
NAMES = ("Qx", "Kx", "V", "mu", "omega", "alpha")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def gen_dO(shape, dtype, seed):
    """Upstream gradient dL/dO: standard normal from its own seeded stream, in the input dtype."""
    z = inputs.normal(inputs.stream_key(seed, "dO"), 0, int(np.prod(shape))).reshape(shape).astype(np.float32)
    return inputs.f32_to_bf16_bits(z) if dtype == "bf16" else z


def make(B, H, N, dtype, seed):
    w = inputs.Workload("bwd", B=B, H=H, N=N, d=64, K=64, dv=64, dtype=dtype, causal=False, seed=seed)
    x = inputs.gen_all(w)
    x["dO"] = gen_dO((B, H, N, 64), dtype, seed)
    return w, x


def run_gpu(w, x):
    import gaussian_mixture_latent_gb300 as gma
    g = gma.gma_backward(*(to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")), eps=w.eps,
                         var_floor=w.var_floor)
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    return [t.double().cpu().numpy() for t in g]


def oracle_grads(w, x, b, h):
    import oracle
    wid = lambda a: inputs.widen(a, w.dtype)
    return oracle.backward_head(wid(x["Qx"][b, h]), wid(x["Kx"][b, h]), wid(x["V"][b, h]), x["mu"][h],
                                x["rho"][h], x["alpha"][h], w.var_floor, w.eps, False, wid(x["dO"][b, h]))


def rel(a, b, floor=0.0):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), floor, 1e-30))


def check(w, x, got, heads=None, param_heads=None):
    """Row gradients on `heads` ((b, h) pairs), parameter gradients on `param_heads`."""
    B, H = w.B, w.H
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    param_heads = param_heads if param_heads is not None else list(range(H))
    cache = {}

    def og(b, h):
        if (b, h) not in cache:
            cache[(b, h)] = oracle_grads(w, x, b, h)
        return cache[(b, h)]

    worst = {}
    for b, h in heads:
        ref = og(b, h)
        floor = 1e-2 * max(np.abs(ref["Qx"]).max(), np.abs(ref["Kx"]).max())
        for i, n in enumerate(("Qx", "Kx", "V")):
            worst[n] = max(worst.get(n, 0.0), rel(got[i][b, h], ref[n], floor if n != "V" else 0.0))
    for h in param_heads:
        for i, n in ((3, "mu"), (4, "omega"), (5, "alpha")):
            ref = sum(og(b, h)[n] for b in range(B))
            worst[n] = max(worst.get(n, 0.0), rel(got[i][h], ref))
    print(w.name, w.dtype, {k: f"{v:.2e}" for k, v in worst.items()})
    for g in got:
        assert np.isfinite(g).all()
    assert max(worst.values()) <= TOL_BWD, worst
    return worst


CASES = [
    # B, H, N, dtype
    (1, 1, 1, "f32"),
    (2, 3, 63, "f32"),
    (1, 2, 65, "bf16"),
    (2, 2, 200, "bf16"),
    (1, 4, 1000, "f32"),
    (3, 2, 777, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}N{c[2]}_{c[3]}" for c in CASES])
def test_backward_parity(case):
    B, H, N, dtype = case
    w, x = make(B, H, N, dtype, seed=N)
    check(w, x, run_gpu(w, x))


def test_backward_is_deterministic():
    w, x = make(2, 3, 500, "bf16", seed=3)
    a, b = run_gpu(w, x), run_gpu(w, x)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_backward_full_size_sampled():
    # the 96-head N = 8192 workload: row gradients of two heads, parameter gradients of one
    # head set (all eight batch entries through the oracle)
    w = inputs.WORKLOADS["causal_bf16_n8192"]
    x = inputs.gen_all(w)
    x["dO"] = gen_dO((w.B, w.H, w.N, w.dv), "bf16", 8)
    got = run_gpu(w, x)
    check(w, x, got, heads=[(0, 0), (7, 11)], param_heads=[5])


def test_backward_unsupported_and_empty():
    import gaussian_mixture_latent_gb300 as gma
    w, x = make(1, 2, 100, "bf16", seed=1)
    args = [to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")]
    with pytest.raises(gma.GmaError) as e:
        gma.gma_backward(*args, causal=True)
    assert e.value.code == 2
    w2 = inputs.Workload("k128", B=1, H=2, N=100, d=64, K=128, dv=64, dtype="bf16", causal=False)
    x2 = inputs.gen_all(w2)
    x2["dO"] = x2["V"]
    with pytest.raises(gma.GmaError) as e:
        gma.gma_backward(*(to_device(x2[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")))
    assert e.value.code == 2
    empty = [a[:, :, :0].contiguous() if a.dim() == 4 else a for a in args]
    g = gma.gma_backward(*empty)
    torch.cuda.synchronize()
    assert all(float(t.abs().max()) == 0.0 for t in g[3:])
