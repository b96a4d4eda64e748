"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Metric (per head, then max over the heads checked): max |O_gpu - O_ref| / max |O_ref|.
Tolerance: 1e-4 for float32 inputs, 2e-2 for bf16 inputs with fp32 accumulation.
Elementwise relative error is not used: output entries are averages of
zero-mean values and cross zero.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from gaussian_mixture_latent_gb300 import inputs
from tests._util import TOL, head_rel_err, oracle_head, to_device, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, len(os.sched_getaffinity(0))))


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_gpu(w, x, **kw):
    import gaussian_mixture_latent_gb300 as gma
    out = gma.gma_forward(to_device(x["Qx"]), to_device(x["Kx"]), to_device(x["V"]),
                          to_device(x["mu"]), to_device(x["rho"]), to_device(x["alpha"]),
                          eps=kw.get("eps", w.eps), causal=w.causal, var_floor=w.var_floor,
                          chunk=kw.get("chunk", 0))
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    return out


def check_heads(w, x, out, heads, tol=None):
    tol = tol or TOL[w.dtype]
    got = to_f64(out).reshape(w.G, w.N, w.dv)
    with ThreadPoolExecutor(THREADS) as ex:
        refs = list(ex.map(lambda g: oracle_head(w, x, g), heads))
    errs = [head_rel_err(got[g], r) for g, r in zip(heads, refs)]
    assert np.isfinite(got).all()
    worst = max(errs)
    assert worst <= tol, f"{w.name}: max relative error {worst:.3e} > {tol} (heads {heads})"
    return worst


SMALL = [
    # name, B, H, N, d, K, dv, dtype, causal
    ("tiny_f32", 1, 1, 1, 3, 4, 2, "f32", False),
    ("ragged_f32", 2, 2, 333, 16, 8, 32, "f32", False),
    ("ragged_f32_causal", 2, 2, 333, 16, 8, 32, "f32", True),
    ("odd_shapes_f32", 1, 3, 257, 5, 7, 9, "f32", True),
    ("k1_f32", 1, 2, 100, 8, 1, 16, "f32", False),
    ("bf16_tiles", 2, 2, 1000, 64, 64, 64, "bf16", False),
    ("bf16_tiles_causal", 2, 2, 1000, 64, 64, 64, "bf16", True),
    ("bf16_k128", 1, 2, 777, 64, 128, 64, "bf16", False),
    ("bf16_k256_dv128", 1, 2, 640, 64, 256, 128, "bf16", True),
    ("bf16_odd", 1, 1, 515, 24, 40, 48, "bf16", True),
    # many short heads per persistent CTA: head switches, parameter-buffer reuse
    ("bf16_many_heads", 8, 64, 200, 64, 64, 64, "bf16", False),
    ("bf16_many_heads_k128", 4, 32, 300, 64, 128, 64, "bf16", False),
    ("bf16_many_heads_causal", 4, 48, 300, 64, 64, 64, "bf16", True),
    # segment-parallel causal scan (fewer heads than SMs): ranges that start inside a head
    # (prefix pass), cross into the next head, and long prefix chains
    ("bf16_seg_cross_heads", 2, 4, 1100, 64, 64, 64, "bf16", True),
    ("bf16_seg_long_chain", 1, 3, 5000, 64, 64, 64, "bf16", True),
    ("bf16_seg_one_head", 1, 1, 9000, 64, 64, 64, "bf16", True),
    # component-sliced causal path: K > 64 or dv > 64
    ("bf16_k128_causal", 2, 3, 700, 64, 128, 64, "bf16", True),
    ("bf16_k192_causal_ragged", 1, 2, 301, 64, 192, 64, "bf16", True),
    ("bf16_k64_dv128_causal", 1, 2, 333, 64, 64, 128, "bf16", True),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_parity_small(case):
    name, B, H, N, d, K, dv, dtype, causal = case
    w = inputs.Workload(name, B=B, H=H, N=N, d=d, K=K, dv=dv, dtype=dtype, causal=causal, seed=3)
    x = inputs.gen_all(w)
    out = run_gpu(w, x)
    check_heads(w, x, out, list(range(w.G)))


def test_parity_large_eps_and_zero_eps():
    w = inputs.Workload("eps", B=1, H=2, N=300, d=16, K=8, dv=32, dtype="f32", causal=True, eps=0.5)
    x = inputs.gen_all(w)
    check_heads(w, x, run_gpu(w, x), [0, 1])
    w0 = w.replace(eps=0.0, causal=False)
    check_heads(w0, x, run_gpu(w0, x), [0, 1])


FULL = ["bidir_f32_n256", "bidir_bf16_n4096", "causal_bf16_n8192", "bidir_bf16_n65536",
        "causal_bf16_n131072"]


@pytest.mark.parametrize("name", FULL)
def test_parity_full_size(name):
    # every head of every workload against the oracle, in the launch configuration the
    # benchmark times: persistent CTAs cross head boundaries at positions that differ
    # from head to head, so no head is left to a finiteness check
    w = inputs.WORKLOADS[name]
    x = inputs.gen_all(w)
    out = run_gpu(w, x)
    heads = list(range(w.G))
    err = check_heads(w, x, out, heads)
    print(f"{name}: max relative error {err:.3e} over all {len(heads)} heads")


@pytest.mark.parametrize("K,dv", [(64, 64), (256, 128)], ids=["direct", "sliced"])
def test_causal_prefix_is_exact_and_future_rows_do_not_leak(K, dv):
    # Section 5.3 of the paper checks a maximum prefix error of exactly zero.
    # Future routing rows become NaN; future values become large finite values
    # (a masked tensor-core tile multiplies them by an exact 0, and 0 * NaN is
    # NaN in IEEE arithmetic, so NaN values are not part of this check).
    w = inputs.Workload("causal_leak", B=1, H=2, N=1100, d=64, K=K, dv=dv, dtype="bf16", causal=True)
    x = inputs.gen_all(w)
    base = to_f64(run_gpu(w, x))
    cut = 517
    y = {k: v.copy() for k, v in x.items()}
    nan_bf16 = np.uint16(0x7FC0)
    y["Qx"][:, :, cut:] = nan_bf16
    y["Kx"][:, :, cut:] = nan_bf16
    big = inputs.f32_to_bf16_bits(np.float32(300.0) * inputs.bf16_bits_to_f32(y["V"][:, :, cut:]))
    y["V"][:, :, cut:] = big
    pert = to_f64(run_gpu(w, y))
    assert np.array_equal(base[:, :, :cut], pert[:, :, :cut])


def test_bitwise_deterministic():
    w = inputs.Workload("det", B=2, H=2, N=2000, d=64, K=64, dv=64, dtype="bf16", causal=False)
    x = inputs.gen_all(w)
    a, b = to_f64(run_gpu(w, x)), to_f64(run_gpu(w, x))
    assert np.array_equal(a, b)
    wc = w.replace(causal=True)
    a, b = to_f64(run_gpu(wc, x)), to_f64(run_gpu(wc, x))
    assert np.array_equal(a, b)


def test_empty_sequence_is_a_no_op():
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("empty", B=1, H=2, N=0, d=16, K=8, dv=32, dtype="f32", causal=False)
    x = inputs.gen_all(w)
    out = gma.gma_forward(to_device(x["Qx"]), to_device(x["Kx"]), to_device(x["V"]),
                          to_device(x["mu"]), to_device(x["rho"]), to_device(x["alpha"]))
    assert out.shape == (1, 2, 0, 32)


def test_misaligned_and_short_workspace_are_rejected():
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("err", B=1, H=1, N=64, d=16, K=8, dv=32, dtype="f32", causal=False)
    x = inputs.gen_all(w)
    Q = to_device(x["Qx"])
    flat = torch.empty(Q.numel() + 1, dtype=torch.float32, device="cuda")
    Qmis = flat[1:].view(Q.shape)            # 4-byte offset: not 16-byte aligned
    with pytest.raises(gma.GmaError) as e:
        gma.gma_forward(Qmis, to_device(x["Kx"]), to_device(x["V"]), to_device(x["mu"]),
                        to_device(x["rho"]), to_device(x["alpha"]))
    assert e.value.code == 1
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(gma.GmaError) as e:
        gma.gma_forward(Q, to_device(x["Kx"]), to_device(x["V"]), to_device(x["mu"]),
                        to_device(x["rho"]), to_device(x["alpha"]), workspace=small)
    assert e.value.code == 3


def test_responsibilities_export_matches_oracle():
    import gaussian_mixture_latent_gb300 as gma
    import oracle
    for dtype, tol in (("f32", 1e-5), ("bf16", 2e-2)):
        w = inputs.Workload("resp", B=1, H=2, N=300, d=64, K=64, dv=8, dtype=dtype, causal=False)
        x = inputs.gen_all(w)
        gam = gma.gma_responsibilities(to_device(x["Kx"]), to_device(x["mu"]), to_device(x["rho"]),
                                       to_device(x["alpha"]), var_floor=w.var_floor)
        got = to_f64(gam)
        for h in range(2):
            ref = oracle.responsibilities(inputs.widen(x["Kx"][0, h], dtype), x["mu"][h],
                                          x["rho"][h], x["alpha"][h], w.var_floor)
            assert np.abs(got[0, h] - ref).max() <= tol
            np.testing.assert_allclose(got[0, h].sum(1), 1.0, atol=1e-5)


def test_back_to_back_forwards_do_not_interfere():
    # Kernels of one forward start while the previous kernel drains (programmatic
    # dependent launch); consecutive forwards on different inputs, in both
    # directions and with shared workspace, must each equal a forward run alone.
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("b2b", B=2, H=4, N=1500, d=64, K=64, dv=64, dtype="bf16", causal=False)
    sets = [inputs.gen_all(w.replace(seed=s)) for s in (11, 12)]
    dev = [{k: to_device(v) for k, v in x.items()} for x in sets]

    def fwd(x, causal):
        return gma.gma_forward(x["Qx"], x["Kx"], x["V"], x["mu"], x["rho"], x["alpha"], eps=w.eps,
                               causal=causal, var_floor=w.var_floor)

    alone = {}
    for i in range(2):
        for causal in (False, True):
            alone[i, causal] = to_f64(fwd(dev[i], causal))
            torch.cuda.synchronize()
    outs = [(i % 2, causal, fwd(dev[i % 2], causal)) for i in range(6) for causal in (False, True)]
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    for i, causal, o in outs:
        assert np.array_equal(to_f64(o), alone[i, causal])


@pytest.mark.parametrize("chunk", [1, 7, 64, 100])
def test_cuda_core_causal_honours_the_chunk(chunk):
    # the float32 path scans in chunks of the requested length; every length gives the
    # oracle's result (the chunk changes only the rounding) and a ragged final chunk
    w = inputs.Workload("chunk_f32", B=1, H=2, N=301, d=16, K=8, dv=32, dtype="f32", causal=True, seed=9)
    x = inputs.gen_all(w)
    check_heads(w, x, run_gpu(w, x, chunk=chunk), [0, 1])


def test_tensor_core_causal_chunk_128_equals_default_and_others_are_refused():
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("chunk_tc", B=1, H=2, N=700, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=9)
    x = inputs.gen_all(w)
    a, b = to_f64(run_gpu(w, x, chunk=0)), to_f64(run_gpu(w, x, chunk=128))
    assert np.array_equal(a, b)
    for bad in (64, 256):
        with pytest.raises(gma.GmaError) as e:
            run_gpu(w, x, chunk=bad)
        assert e.value.code == 2
