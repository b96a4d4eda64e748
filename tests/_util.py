"""Helpers shared by the tests: device transfer, the parity metric, oracle runs."""
import numpy as np

from gaussian_mixture_latent_gb300 import inputs

TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_device(a, dev="cuda"):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def to_f64(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def head_rel_err(got, ref):
    """Normwise relative error of one head: max|got - ref| / max|ref| (0 when ref is all zero)."""
    den = np.abs(ref).max()
    num = np.abs(got - ref).max()
    return num / den if den > 0 else num


def oracle_head(w, x, g, threads=1):
    import oracle
    h = g % w.H
    b = g // w.H
    return oracle.forward_head(inputs.widen(x["Qx"][b, h], w.dtype), inputs.widen(x["Kx"][b, h], w.dtype),
                               inputs.widen(x["V"][b, h], w.dtype), x["mu"][h], x["rho"][h],
                               x["alpha"][h], w.var_floor, w.eps, w.causal)
