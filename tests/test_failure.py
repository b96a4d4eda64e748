"""The device-side failure path: a bounded wait that runs out posts GMA_ERR_TIMEOUT to
the workspace's status word and leaves the CUDA context usable.  The failure is made by
a wait on a barrier that nothing arrives at; no fault, trap or hang is involved."""
import time

import numpy as np
import pytest

from gaussian_mixture_latent_gb300 import inputs
from tests._util import TOL, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_a_wait_that_runs_out_posts_a_timeout_and_the_context_stays_usable():
    import gaussian_mixture_latent_gb300 as gma
    import oracle
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert gma.gma_get_status(ws) == 0
    t0 = time.perf_counter()
    gma.gma_selftest_timeout(ws)
    status = gma.gma_get_status(ws)
    dt = time.perf_counter() - t0
    assert status == 5, gma.gma_status_string(status)
    assert 0.2 < dt < 30.0, dt                      # the wait's bound, about one second
    assert gma.gma_get_status(ws) == 0              # read and cleared
    # a forward afterwards runs and is right
    w = inputs.Workload("after", B=1, H=2, N=300, d=64, K=64, dv=64, dtype="bf16", causal=True)
    x = inputs.gen_all(w)
    out = gma.gma_forward(*(to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha")), eps=w.eps,
                          causal=True, var_floor=w.var_floor)
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    ref = oracle.forward(*(inputs.widen(x[n], "bf16") for n in ("Qx", "Kx", "V")), x["mu"], x["rho"], x["alpha"],
                         w.var_floor, w.eps, True)
    got = out.float().cpu().numpy().astype(np.float64)
    for h in range(w.H):
        assert np.abs(got[0, h] - ref[0, h]).max() / np.abs(ref[0, h]).max() <= TOL["bf16"]


def test_check_status_raises_on_a_posted_device_error():
    # a device error already posted to a workspace's status word is raised by the next
    # call made with check_status=True on that workspace, and the word is cleared
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("chk", B=1, H=1, N=200, d=64, K=64, dv=64, dtype="bf16", causal=False)
    x = inputs.gen_all(w)
    args = [to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha")]
    desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, w.dv, torch.bfloat16, torch.bfloat16, w.var_floor, 0)
    ws = torch.zeros(gma.gma_workspace_size(desc, False), dtype=torch.uint8, device="cuda")
    gma.gma_forward(*args, eps=w.eps, workspace=ws, check_status=True)      # clean: no error
    gma.gma_selftest_timeout(ws)
    with pytest.raises(gma.GmaError) as e:
        gma.gma_forward(*args, eps=w.eps, workspace=ws, check_status=True)
    assert e.value.code == 5
    gma.gma_forward(*args, eps=w.eps, workspace=ws, check_status=True)      # cleared by the read
