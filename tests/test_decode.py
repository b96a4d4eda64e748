"""Parity of the causal decode with a carried state (CUDA path, through the C
ABI) with the fp64 oracle: "Gaussian Mixture Attention", section 3.5, Eq. 6b /
8b as a recurrence.

The oracle's causal forward of the whole sequence gives the expected outputs
of the decoded positions, and its prefix memory [Vt | Z] after the first n0
positions is the state the decode starts from; the state the decode leaves
must equal the memory after the last position.  Metric per head as for the
forward (max |err| / max |ref|), tolerance 1e-4 (fp32) / 2e-2 (bf16).
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


def oracle_split(w, x, n0):
    """Per head: outputs of positions n0.. (full causal forward), the memory after n0 positions
    and after all of them, as [K, dv + 1]."""
    import oracle
    outs, s0, s1 = [], [], []
    for g in range(w.G):
        b, h = divmod(g, w.H)
        Q, Kx, V = (inputs.widen(x[n][b, h], w.dtype) for n in ("Qx", "Kx", "V"))
        par = (x["mu"][h], x["rho"][h], x["alpha"][h], w.var_floor, w.eps, True)
        o, Vt, Z = oracle.forward_head(Q, Kx, V, *par, return_memory=True)
        outs.append(o[n0:])
        s1.append(np.concatenate([Vt, Z[:, None]], axis=1))
        if n0 > 0:
            _, Vt0, Z0 = oracle.forward_head(Q[:n0], Kx[:n0], V[:n0], *par, return_memory=True)
            s0.append(np.concatenate([Vt0, Z0[:, None]], axis=1))
        else:
            s0.append(np.zeros((w.K, w.dv + 1)))
    shape = (w.B, w.H)
    return (np.stack(outs).reshape(shape + outs[0].shape), np.stack(s0).reshape(shape + s0[0].shape),
            np.stack(s1).reshape(shape + s1[0].shape))


def decode(w, x, n0, state, step=None):
    import gaussian_mixture_latent_gb300 as gma
    d = {n: to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha")}
    outs = []
    stop = w.N
    step = step or (stop - n0)
    for a in range(n0, stop, step):
        sl = slice(a, min(stop, a + step))
        outs.append(gma.gma_decode(d["Qx"][:, :, sl].contiguous(), d["Kx"][:, :, sl].contiguous(),
                                   d["V"][:, :, sl].contiguous(), d["mu"], d["rho"], d["alpha"], state,
                                   eps=w.eps, var_floor=w.var_floor))
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    return torch.cat(outs, dim=2)


def rel(a, b):
    return max(np.abs(a[i, j] - b[i, j]).max() / np.abs(b[i, j]).max() for i in range(a.shape[0])
               for j in range(a.shape[1]))


CASES = [
    # name, B, H, N, d, K, dv, dtype, n0
    ("f32_small", 2, 2, 120, 16, 8, 32, "f32", 57),
    ("f32_from_empty", 1, 3, 80, 8, 5, 7, "f32", 0),
    ("bf16_d64_k64", 2, 3, 200, 64, 64, 64, "bf16", 150),
    ("bf16_k256_dv128", 1, 2, 90, 64, 256, 128, "bf16", 60),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_continues_the_causal_sequence(case):
    name, B, H, N, d, K, dv, dtype, n0 = case
    w = inputs.Workload(name, B=B, H=H, N=N, d=d, K=K, dv=dv, dtype=dtype, causal=True, seed=8)
    x = inputs.gen_all(w)
    o_ref, s0, s1 = oracle_split(w, x, n0)
    state = torch.from_numpy(s0.astype(np.float32)).cuda()
    got = to_f64(decode(w, x, n0, state))
    assert rel(got, o_ref) <= TOL[dtype]
    assert rel(state.double().cpu().numpy(), s1) <= TOL[dtype]


def test_decode_token_by_token_equals_one_call():
    w = inputs.Workload("tok", B=2, H=2, N=40, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=2)
    x = inputs.gen_all(w)
    _, s0, _ = oracle_split(w, x, 10)
    st_a = torch.from_numpy(s0.astype(np.float32)).cuda()
    st_b = st_a.clone()
    a = decode(w, x, 10, st_a)
    b = decode(w, x, 10, st_b, step=1)
    assert torch.equal(a, b) and torch.equal(st_a, st_b)


def test_decode_rejects_a_state_too_large_for_one_cta():
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("big", B=1, H=1, N=4, d=64, K=256, dv=256, dtype="bf16", causal=True)
    x = inputs.gen_all(w)
    state = torch.zeros((1, 1, 256, 257), dtype=torch.float32, device="cuda")
    with pytest.raises(gma.GmaError) as e:
        gma.gma_decode(*(to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha")), state)
    assert e.value.code == 2
