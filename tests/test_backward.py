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

The bidirectional backward of bf16 inputs runs on the tensor cores with bf16 operands
(the responsibilities, a | b, ds, x^2 and [lambda | lambda mu], each rounded to 8
significant bits, relative error <= 2^-9 ~ 2e-3; the two memory operands as two bf16
terms; fp32 accumulation).  A gradient passes through up to five such roundings in
sequence, and the softmax Jacobian of peaked responsibilities amplifies them (a rounding
emulation of these operands against the oracle gives up to ~1e-2 over several seeds),
so it is held to the bf16 bound, 2e-2, that the pages fix for bf16 inputs with fp32
accumulation.  fp32 inputs and the causal backward
run on the CUDA cores in fp32 and keep the 1e-3 bound, and so do heads of one 128-row
tile (the single-row head, whose exact routing gradient is O(eps) because O = v for any
responsibilities, is among them: bf16 operands could not resolve that cancellation).
"""
import numpy as np
import pytest

from gaussian_mixture_latent_gb300 import inputs
from tests._util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_BWD = 1e-3
TOL_BWD_TC = 2e-2        # bidirectional, bf16 inputs: tensor-core operands


def tol_for(w):
    # the tensor-core passes take bidirectional bf16 heads of more than one 128-row tile at
    # d = dv = K = 64; every other shape runs in fp32 on the CUDA cores
    tc = w.dtype == "bf16" and not w.causal and w.N > 128 and w.d == w.K == w.dv == 64
    return TOL_BWD_TC if tc else TOL_BWD
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


def make(B, H, N, dtype, seed, causal=False, eps=1e-6):
    w = inputs.Workload("bwd", B=B, H=H, N=N, d=64, K=64, dv=64, dtype=dtype, causal=causal, seed=seed, eps=eps)
    x = inputs.gen_all(w)
    x["dO"] = gen_dO((B, H, N, 64), dtype, seed)
    return w, x


def make_shape(B, H, N, d, K, dv, dtype, seed, causal=False, eps=1e-6):
    w = inputs.Workload("bwd_gen", B=B, H=H, N=N, d=d, K=K, dv=dv, dtype=dtype, causal=causal, seed=seed, eps=eps)
    x = inputs.gen_all(w)
    x["dO"] = gen_dO((B, H, N, dv), dtype, seed)
    return w, x


def run_gpu(w, x, chunk=0):
    import gaussian_mixture_latent_gb300 as gma
    g = gma.gma_backward(*(to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")), eps=w.eps,
                         var_floor=w.var_floor, causal=w.causal, chunk=chunk)
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    return [t.double().cpu().numpy() for t in g]


def oracle_grads(w, x, b, h):
    import oracle
    wid = lambda a: inputs.widen(a, w.dtype)
    return oracle.backward_head(wid(x["Qx"][b, h]), wid(x["Kx"][b, h]), wid(x["V"][b, h]), x["mu"][h],
                                x["rho"][h], x["alpha"][h], w.var_floor, w.eps, w.causal, wid(x["dO"][b, h]))


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
    assert max(worst.values()) <= tol_for(w), worst
    return worst


CASES = [
    # B, H, N, dtype, causal, eps
    (1, 1, 1, "f32", False, 1e-6),
    (2, 3, 63, "f32", False, 1e-6),
    (1, 2, 65, "bf16", False, 1e-6),
    (2, 2, 200, "bf16", False, 1e-6),
    (1, 4, 1000, "f32", False, 1e-6),
    (3, 2, 777, "bf16", False, 1e-6),
    (1, 2, 130, "bf16", False, 0.0),
    (2, 3, 9000, "bf16", False, 1e-6),     # persistent CTAs cross head boundaries; ragged last tile
    (1, 1, 1, "bf16", False, 1e-6),       # one tile: the fp32 CUDA-core passes
    (1, 2, 129, "bf16", False, 1e-6),     # two tiles, the second of one row: the tensor-core passes
    (1, 1, 1, "f32", True, 1e-6),
    (2, 3, 63, "f32", True, 1e-6),
    (1, 2, 65, "bf16", True, 1e-6),
    (2, 2, 300, "bf16", True, 1e-6),
    (1, 3, 1500, "f32", True, 1e-6),
    (1, 2, 130, "bf16", True, 0.0),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}N{c[2]}_{c[3]}_{'causal' if c[4] else 'bidir'}"
                                             f"{'_eps0' if c[5] == 0 else ''}" for c in CASES])
def test_backward_parity(case):
    B, H, N, dtype, causal, eps = case
    w, x = make(B, H, N, dtype, seed=N, causal=causal, eps=eps)
    check(w, x, run_gpu(w, x))


GENERAL = [
    # the general CUDA-core path (every shape but d = dv = K = 64): B, H, N, d, K, dv, dtype, causal, chunk
    (1, 2, 256, 16, 8, 32, "f32", False, 0),       # the small fp32 workload's shape
    (1, 2, 256, 16, 8, 32, "f32", True, 0),
    (2, 2, 333, 64, 128, 64, "bf16", False, 0),    # K = 128
    (2, 2, 333, 64, 128, 64, "bf16", True, 0),
    (1, 2, 300, 64, 256, 128, "bf16", True, 0),    # K = 256, dv = 128 (the long causal workload's shape)
    (1, 2, 300, 64, 256, 128, "bf16", False, 0),
    (1, 3, 257, 5, 7, 9, "f32", True, 0),          # odd sizes, ragged ranges and chunks
    (1, 3, 257, 5, 7, 9, "f32", False, 0),
    # one row: with eps = 1e-6 O = v for any responsibilities, the exact routing gradients are
    # O(eps) and fp32 cannot resolve their cancellation (the paths at d = dv = K = 64 met the
    # same); with eps = 0.5 they are O(1)
    (1, 1, 1, 24, 40, 48, "bf16", False, 0, 0.5),
    (1, 1, 1, 24, 40, 48, "bf16", True, 0, 0.5),
    (2, 2, 300, 64, 64, 64, "bf16", True, 16),     # d = dv = K = 64 with a chunk of 16: the general path
    (1, 2, 700, 32, 96, 48, "f32", True, 5),       # a chunk that does not divide the ranges
    (4, 24, 200, 64, 128, 64, "bf16", False, 0),   # many head rows, several ranges each
]


@pytest.mark.parametrize("case", GENERAL, ids=[f"B{c[0]}H{c[1]}N{c[2]}d{c[3]}K{c[4]}dv{c[5]}_{c[6]}_"
                                               f"{'causal' if c[7] else 'bidir'}{'_C%d' % c[8] if c[8] else ''}"
                                               for c in GENERAL])
def test_backward_general_shapes(case):
    B, H, N, d, K, dv, dtype, causal, chunk = case[:9]
    eps = case[9] if len(case) > 9 else 1e-6
    w, x = make_shape(B, H, N, d, K, dv, dtype, seed=N + K, causal=causal, eps=eps)
    got = run_gpu(w, x, chunk=chunk)
    heads = [(b, h) for b in range(B) for h in range(H)][:8]
    check(w, x, got, heads=heads, param_heads=list(range(min(H, 4))))


def test_general_backward_causality_and_determinism():
    # dO nonzero at row t only (K = 128): the exact gradient of every other query row and of
    # every key and value row after t is zero, and the general path gives exact zeros
    # there; a second call is bitwise equal
    w, x = make_shape(1, 2, 300, 64, 128, 64, "bf16", seed=4, causal=True)
    t = 141
    dO = np.zeros_like(x["dO"])
    dO[:, :, t] = x["dO"][:, :, t]
    x["dO"] = dO
    g1 = run_gpu(w, x)
    dQ, dK, dV = g1[:3]
    rows = np.arange(300) != t
    assert np.abs(dQ[:, :, rows]).max() == 0.0 and np.abs(dQ[:, :, t]).max() > 0
    assert np.abs(dK[:, :, t + 1:]).max() == 0.0 and np.abs(dV[:, :, t + 1:]).max() == 0.0
    assert np.abs(dK[:, :, :t + 1]).max() > 0 and np.abs(dV[:, :, :t + 1]).max() > 0
    for u, v in zip(g1, run_gpu(w, x)):
        assert np.array_equal(u, v)


def test_causal_backward_reaches_only_the_prefix():
    # dO nonzero at row t only: the exact gradient of every other query row, and of every key
    # and value row after t, is zero, and the kernels produce exact zeros there
    w, x = make(1, 2, 300, "bf16", seed=5, causal=True)
    t = 137
    dO = np.zeros_like(x["dO"])
    dO[:, :, t] = x["dO"][:, :, t]
    x["dO"] = dO
    dQ, dK, dV = run_gpu(w, x)[:3]
    rows = np.arange(300) != t
    assert np.abs(dQ[:, :, rows]).max() == 0.0 and np.abs(dQ[:, :, t]).max() > 0
    assert np.abs(dK[:, :, t + 1:]).max() == 0.0 and np.abs(dV[:, :, t + 1:]).max() == 0.0
    assert np.abs(dK[:, :, :t + 1]).max() > 0 and np.abs(dV[:, :, :t + 1]).max() > 0


def test_backward_is_deterministic():
    w, x = make(2, 3, 500, "bf16", seed=3)
    a, b = run_gpu(w, x), run_gpu(w, x)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_backward_full_size_sampled():
    # the 96-head N = 8192 workload (bidirectional): row gradients of two heads, parameter
    # gradients of one head set (all eight batch entries through the oracle)
    w = inputs.WORKLOADS["causal_bf16_n8192"].replace(causal=False)
    x = inputs.gen_all(w)
    x["dO"] = gen_dO((w.B, w.H, w.N, w.dv), "bf16", 8)
    got = run_gpu(w, x)
    check(w, x, got, heads=[(0, 0), (7, 11)], param_heads=[5])


def test_backward_unsupported_and_empty():
    import gaussian_mixture_latent_gb300 as gma
    w, x = make(1, 2, 100, "bf16", seed=1)
    args = [to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")]
    # a causal state of K (dv + 1) = 256 x 257 floats does not fit a CTA's shared memory
    w2 = inputs.Workload("k256", B=1, H=2, N=100, d=64, K=256, dv=256, dtype="bf16", causal=True)
    x2 = inputs.gen_all(w2)
    x2["dO"] = x2["V"]
    with pytest.raises(gma.GmaError) as e:
        gma.gma_backward(*(to_device(x2[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")), causal=True)
    assert e.value.code == 2
    empty = [a[:, :, :0].contiguous() if a.dim() == 4 else a for a in args]
    g = gma.gma_backward(*empty)
    torch.cuda.synchronize()
    assert all(float(t.abs().max()) == 0.0 for t in g[3:])


@pytest.mark.parametrize("dtype,bound", [("f32", 1e-4), ("bf16", 2e-3)])
def test_backward_identities_of_the_gpu_gradients(dtype, bound):
    # properties the exact gradients satisfy at any size, on the GPU's gradients of a
    # 6-head N = 3000 problem: a common shift of every routing vector and every mean leaves
    # each score unchanged, so sum_i dQx_i + sum_i dKx_i + sum_k dmu_k = 0 for every head
    # set and dimension; O is homogeneous of degree one in V (Eq. 7-8), so
    # sum dV * V = sum dO * O (Euler); and sum_k dalpha_k = 0 (Eq. 15).  fp32 inputs take
    # the fp32 CUDA-core passes (bound 1e-4 of the sum of magnitudes); bf16 inputs the
    # tensor-core passes, whose bf16 operand roundings (2^-9 each, independent from term to
    # term) leave the sums at a small multiple of 2^-9 of the sum of magnitudes: bound 2e-3
    import oracle
    w, x = make(2, 3, 3000, dtype, seed=12)
    dQ, dK, dV, dmu, drho, dal = run_gpu(w, x)
    shift = dQ.sum(axis=(0, 2)) + dK.sum(axis=(0, 2)) + dmu.sum(axis=1)           # [H, d]
    scale = np.abs(dQ).sum(axis=(0, 2)) + np.abs(dK).sum(axis=(0, 2)) + np.abs(dmu).sum(axis=1)
    assert (np.abs(shift) <= bound * scale).all(), np.abs(shift / scale).max()
    O = oracle.forward(*(inputs.widen(x[n], w.dtype) for n in ("Qx", "Kx", "V")), x["mu"], x["rho"], x["alpha"],
                       w.var_floor, w.eps, False, threads=4)
    V, dO = inputs.widen(x["V"], w.dtype), inputs.widen(x["dO"], w.dtype)
    for b in range(w.B):
        for h in range(w.H):
            lhs, rhs = float((dV[b, h] * V[b, h]).sum()), float((dO[b, h] * O[b, h]).sum())
            assert abs(lhs - rhs) <= bound * np.abs(dO[b, h] * O[b, h]).sum(), (b, h, lhs, rhs)
    assert (np.abs(dal.sum(axis=1)) <= bound * np.abs(dal).sum(axis=1)).all()


def test_causal_backward_full_size_sampled():
    # the same workload as a causal backward: row gradients of one head, parameter gradients
    # of one head set
    w = inputs.WORKLOADS["causal_bf16_n8192"]
    x = inputs.gen_all(w)
    x["dO"] = gen_dO((w.B, w.H, w.N, w.dv), "bf16", 9)
    got = run_gpu(w, x)
    check(w, x, got, heads=[(3, 4)], param_heads=[4])
