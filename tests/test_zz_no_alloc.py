"""gma_forward_noalloc: the forward for callers that cannot allocate device memory.

Callers whose device memory belongs to another memory manager (a framework's
caching allocator, a server that hands each model a fixed budget), or that run
latency-sensitive loops where cudaMalloc's device-wide synchronisation is not
acceptable, cannot provide a workspace.  This entry point runs the same
forward on a fixed scratch array compiled into the library.  The test calls it
through the C ABI on two different problems in a row, then on the first one
again, and requires each output to equal gma_forward's bit for bit (the same
kernels with fixed-order reductions, so any difference would be scratch left
over from an earlier call); one output is also checked against the fp64
oracle.  It also checks that a problem too large for the scratch array is
refused without touching `out`.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

from gaussian_mixture_latent_gb300 import inputs
from tests._util import TOL, head_rel_err, oracle_head, to_device, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_mixture_latent_gb300 as gma
    lib = gma._load()
    vp = ctypes.c_void_p
    lib.gma_forward_noalloc.argtypes = [ctypes.POINTER(gma.gma_desc), vp, vp, vp, vp, vp, vp,
                                        ctypes.c_float, ctypes.c_int, vp, vp]
    lib.gma_forward_noalloc.restype = ctypes.c_int
    return lib


def _problem(w):
    x = inputs.gen_all(w)
    return {k: to_device(v) for k, v in x.items()}


def _noalloc(lib, w, t, out):
    import gaussian_mixture_latent_gb300 as gma
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, w.dv, tdt, tdt, w.var_floor, 0)
    return lib.gma_forward_noalloc(ctypes.byref(desc), t["Qx"].data_ptr(), t["Kx"].data_ptr(),
                                   t["V"].data_ptr(), t["mu"].data_ptr(), t["rho"].data_ptr(),
                                   t["alpha"].data_ptr(), w.eps, int(w.causal), out.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_gma_forward_on_two_calls_in_a_row(lib):
    import gaussian_mixture_latent_gb300 as gma
    wa = inputs.Workload("noalloc_a", B=1, H=2, N=1000, d=64, K=64, dv=64, dtype="bf16", causal=False)
    wb = inputs.Workload("noalloc_b", B=2, H=1, N=777, d=16, K=8, dv=32, dtype="f32", causal=True, seed=5)
    ta, tb = _problem(wa), _problem(wb)
    outs = []
    # a, b, then a again: the shared scratch array must carry nothing from one call to the next
    for w, t in ((wa, ta), (wb, tb), (wa, ta)):
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        out = torch.full((w.B, w.H, w.N, w.dv), float("nan"), dtype=tdt, device="cuda")
        assert _noalloc(lib, w, t, out) == 0
        outs.append(out)
    torch.cuda.synchronize()
    for (w, t), out in zip(((wa, ta), (wb, tb), (wa, ta)), outs):
        ref = gma.gma_forward(t["Qx"], t["Kx"], t["V"], t["mu"], t["rho"], t["alpha"], eps=w.eps,
                              causal=w.causal, var_floor=w.var_floor)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(out).all())
        assert torch.equal(out, ref), w.name
    # and against the oracle, for the bidirectional bf16 problem
    x = inputs.gen_all(wa)
    got = to_f64(outs[0])
    err = max(head_rel_err(got[0, h], oracle_head(wa, x, h)) for h in range(wa.H))
    assert err <= TOL[wa.dtype], err


def test_noalloc_refuses_problems_larger_than_its_scratch(lib):
    # float32 inputs take the CUDA-core path, whose workspace holds both
    # responsibility matrices: 64 heads x 4096 rows x 64 components x 8 bytes.
    w = inputs.Workload("noalloc_big", B=8, H=8, N=4096, d=64, K=64, dv=64, dtype="f32", causal=False)
    import gaussian_mixture_latent_gb300 as gma
    tdt = torch.float32
    desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, w.dv, tdt, tdt, w.var_floor, 0)
    need = gma.gma_workspace_size(desc, False)
    limit = 32 << 20
    assert need > limit
    t = {"Qx": torch.zeros((w.B, w.H, w.N, w.d), dtype=tdt, device="cuda"),
         "V": torch.zeros((w.B, w.H, w.N, w.dv), dtype=tdt, device="cuda"),
         "mu": torch.zeros((w.H, w.K, w.d), device="cuda"),
         "alpha": torch.zeros((w.H, w.K), device="cuda")}
    t["Kx"], t["rho"] = t["Qx"], t["mu"]
    out = torch.full((w.B, w.H, w.N, w.dv), 7.0, dtype=tdt, device="cuda")
    assert _noalloc(lib, w, t, out) == 3          # GMA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
