"""Operand-precision study: emulated rounding of the tensor-core operands against the fp64
oracle ("Gaussian Mixture Attention", Huang & Raza, 2026; the forward of Eq. 3b, 5-8, 16 and
the backward of section 4.1).  A script, not a test: ``python tests/precision_study.py``.

Every product is evaluated in float64 from operands rounded to the stated precision (so the
accumulation is at least as accurate as the kernels' fp32); the error is normwise per head,
max |x - x_ref| / max |x_ref|, the worst over the sampled heads.

Forward: the log-density operands ([x, x^2/256] and W) are varied; Gamma, V and the memory
[Vt | Z] are bf16 operands in every variant and the output is rounded to bf16, as in the
tensor-core kernels.  Backward: the score operands, the memory and read products (Gamma, V,
[Vt | Z]) and the gradient products (a, b, ds, R, lambda) are varied separately; then the
tensor-core backward as built, with its memory operands in one or two bf16 terms.
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
from gaussian_mixture_latent_gb300 import inputs  # noqa: E402

BF16, FP16, TF32 = 7, 10, 10     # explicit mantissa bits


def rnd(x, bits):
    """Round to nearest (even on ties) keeping `bits` explicit mantissa bits; None = exact."""
    if bits is None:
        return np.asarray(x, dtype=np.float64)
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    s = 2.0 ** (bits + 1)
    return np.ldexp(np.round(m * s) / s, e)


def params(mu, om, al, vf):
    mu, om, al = (np.asarray(t, dtype=np.float64) for t in (mu, om, al))
    var = np.logaddexp(0.0, om) + vf
    lam = 1.0 / var
    logpi = al - (al.max() + np.log(np.exp(al - al.max()).sum()))
    c = logpi - 0.5 * np.log(var).sum(1) - 0.5 * (lam * mu * mu).sum(1)
    return mu, om, lam, logpi, c


def gamma(X, lam, mu, c, sbits, centre=False):
    """Eq. 16 expanded, s = c + [x, x^2] . W, from operands with `sbits` mantissa bits; the
    quadratic coefficients optionally centred over k (a row shift the softmax cancels)."""
    wq = -0.5 * lam
    shift = wq.mean(0) if centre else 0.0
    s = c + rnd(X, sbits) @ rnd(lam * mu, sbits).T + rnd(X * X / 256, sbits) @ rnd(256 * (wq - shift), sbits).T
    s = s - s.max(1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(1, keepdims=True)


def forward_bidir(Q, K, V, mu, om, al, vf, eps, sbits, centre):
    mu, om, lam, logpi, c = params(mu, om, al, vf)
    gq, gk = gamma(Q, lam, mu, c, sbits, centre), gamma(K, lam, mu, c, sbits, centre)
    M = rnd(gk, BF16).T @ np.column_stack([V, np.ones(len(V))])
    num = rnd(gq, BF16) @ rnd(M, BF16)
    return rnd(num[:, :-1] / (num[:, -1:] + eps), BF16)


def backward(Q, K, V, mu, om, al, vf, eps, dO, mbits, sbits, gbits):
    mu, om, lam, logpi, c = params(mu, om, al, vf)
    r, rg = (lambda x: rnd(x, mbits)), (lambda x: rnd(x, gbits))
    gq, gk = gamma(Q, lam, mu, c, sbits), gamma(K, lam, mu, c, sbits)
    VV = np.column_stack([V, np.ones(len(V))])
    M = r(gk).T @ r(VV)
    num = r(gq) @ r(M)
    den = num[:, -1] + eps
    O = num[:, :-1] / den[:, None]
    a, b = dO / den[:, None], -(dO * O).sum(1) / den
    AB = np.column_stack([a, b])
    g_q = rg(AB) @ rg(M).T
    ds_q = gq * (g_q - (gq * g_q).sum(1, keepdims=True))
    R = rg(gq).T @ rg(AB)
    g_k = rg(VV) @ rg(R).T
    dV = rg(gk) @ rg(R[:, :-1])
    ds_k = gk * (g_k - (gk * g_k).sum(1, keepdims=True))
    dx = lambda ds, X: rg(ds) @ rg(lam * mu) - X * (rg(ds) @ rg(lam))
    P1 = rg(ds_q).T @ rg(Q) + rg(ds_k).T @ rg(K)
    P2 = rg(ds_q).T @ rg(Q * Q) + rg(ds_k).T @ rg(K * K)
    P0 = ds_q.sum(0) + ds_k.sum(0)
    dvar = 0.5 * (lam ** 2 * (P2 - 2 * mu * P1 + mu ** 2 * P0[:, None]) - lam * P0[:, None])
    return {"Qx": dx(ds_q, Q), "Kx": dx(ds_k, K), "V": dV, "mu": lam * (P1 - mu * P0[:, None]),
            "omega": dvar / (1 + np.exp(-om)), "alpha": P0 - np.exp(logpi) * P0.sum()}


def backward_tc(Q, K, V, mu, om, al, vf, eps, dO, two_term):
    """The tensor-core backward as built: normalised Gamma, a | b, ds, x^2 and [lambda | lambda mu]
    rounded to bf16; the memories [Vt | Z] and [R | r] as one bf16 term or (two_term) as
    hi + lo; den = Gamma Z + eps sum Gamma; exact scores (the log-density error is the
    forward's)."""
    mu, om, lam, logpi, c = params(mu, om, al, vf)
    b16 = lambda t: rnd(t, BF16)
    mem = (lambda t: b16(t) + b16(t - b16(t))) if two_term else b16
    gq, gk = b16(gamma(Q, lam, mu, c, None)), b16(gamma(K, lam, mu, c, None))
    Vt, Z = mem(gk.T @ V), mem(gk.sum(0))
    num = gq @ Vt
    den = gq @ Z + eps * gq.sum(1)
    a, b = b16(dO / den[:, None]), b16(-(dO * num).sum(1) / den ** 2)
    g_q = a @ Vt.T + b[:, None] * Z[None]
    ds_q = b16(gq * (g_q - (gq * g_q).sum(1, keepdims=True)))
    R, r = mem(gq.T @ a), mem(gq.T @ b)
    g_k = V @ R.T + r[None]
    ds_k = b16(gk * (g_k - (gk * g_k).sum(1, keepdims=True)))
    dx = lambda ds, X: ds @ b16(lam * mu) - X * (ds @ b16(lam))
    P1 = ds_q.T @ Q + ds_k.T @ K
    P2 = ds_q.T @ b16(Q * Q) + ds_k.T @ b16(K * K)
    P0 = ds_q.sum(0) + ds_k.sum(0)
    dvar = 0.5 * (lam ** 2 * (P2 - 2 * mu * P1 + mu ** 2 * P0[:, None]) - lam * P0[:, None])
    return {"Qx": dx(ds_q, Q), "Kx": dx(ds_k, K), "V": gk @ R, "mu": lam * (P1 - mu * P0[:, None]),
            "omega": dvar / (1 + np.exp(-om)), "alpha": P0 - np.exp(logpi) * P0.sum()}


def err(a, b):
    return float(np.abs(a - b).max() / np.abs(b).max())


def head(x, n, h):
    return inputs.widen(x[n][0, h], "bf16")


def forward_study():
    cases = [("bidir_bf16_n4096", 2, 4096), ("bidir_bf16_n65536", 1, 16384)]
    variants = [("exact log-density operands", None, False), ("bf16 [x, x^2], bf16 W", BF16, False),
                ("fp16 [x, x^2/256], fp16 W", FP16, False), ("fp16, quadratic coefficients centred", FP16, True)]
    print("forward, bidirectional (Gamma, V, memory bf16; output bf16)")
    for name, H, N in cases:
        w = inputs.WORKLOADS[name].replace(B=1, H=H, N=N)
        x = inputs.gen_all(w)
        refs = [oracle.forward_head(head(x, "Qx", h), head(x, "Kx", h), head(x, "V", h), x["mu"][h], x["rho"][h],
                                    x["alpha"][h], w.var_floor, w.eps, False) for h in range(H)]
        for vname, sb, centre in variants:
            e = max(err(forward_bidir(head(x, "Qx", h), head(x, "Kx", h), head(x, "V", h), x["mu"][h], x["rho"][h],
                                      x["alpha"][h], w.var_floor, w.eps, sb, centre), refs[h]) for h in range(H))
            print(f"  {name:20s} N={N:6d} K={w.K:3d}  {vname:40s} {e:.1e}")


def backward_study():
    w = inputs.WORKLOADS["causal_bf16_n8192"].replace(B=1, H=3, N=2048, causal=False)
    x = inputs.gen_all(w)
    z = inputs.normal(inputs.stream_key(0, "dO"), 0, w.H * w.N * w.dv).reshape(w.H, w.N, w.dv)
    dO = inputs.bf16_bits_to_f64(inputs.f32_to_bf16_bits(z.astype(np.float32)))
    variants = [("exact", None, None, None), ("tf32 everywhere", TF32, TF32, TF32),
                ("bf16 everywhere", BF16, BF16, BF16), ("scores fp16, rest bf16", BF16, FP16, BF16),
                ("scores fp16, memory bf16, gradients tf32", BF16, FP16, TF32),
                ("scores fp32, memory bf16, gradients bf16", BF16, None, BF16)]
    print("backward, bidirectional, N=2048 K=64 (worst over the six gradients and three heads)")
    refs = [oracle.backward_head(head(x, "Qx", h), head(x, "Kx", h), head(x, "V", h), x["mu"][h], x["rho"][h],
                                 x["alpha"][h], w.var_floor, w.eps, False, dO[h]) for h in range(w.H)]
    for vname, mb, sb, gb in variants:
        worst = 0.0
        for h in range(w.H):
            got = backward(head(x, "Qx", h), head(x, "Kx", h), head(x, "V", h), x["mu"][h], x["rho"][h],
                           x["alpha"][h], w.var_floor, w.eps, dO[h], mb, sb, gb)
            worst = max(worst, max(err(got[n], refs[h][n]) for n in refs[h]))
        print(f"  {vname:45s} {worst:.1e}")


def backward_kernel_study():
    """The tensor-core backward's operand precisions on small heads (peaked responsibilities,
    where the softmax Jacobian cancels most), with the parity test's metric: row gradients
    against at least 1e-2 of the head's largest routing gradient, parameter gradients summed
    over the batch."""
    cases = [(3, 2, 777, 777), (2, 2, 200, 200), (2, 2, 200, 11), (1, 4, 300, 5), (2, 2, 1000, 7), (1, 3, 130, 3)]
    worst = {False: 0.0, True: 0.0}
    for B, H, N, seed in cases:
        w = inputs.Workload("bwd", B=B, H=H, N=N, d=64, K=64, dv=64, dtype="bf16", causal=False, seed=seed)
        x = inputs.gen_all(w)
        z = inputs.normal(inputs.stream_key(seed, "dO"), 0, B * H * N * 64).reshape(B, H, N, 64)
        dO = inputs.bf16_bits_to_f64(inputs.f32_to_bf16_bits(z.astype(np.float32)))
        for h in range(H):
            refs = [oracle.backward_head(*(inputs.widen(x[n][b, h], "bf16") for n in ("Qx", "Kx", "V")), x["mu"][h],
                                         x["rho"][h], x["alpha"][h], w.var_floor, w.eps, False, dO[b, h])
                    for b in range(B)]
            for two in (False, True):
                gots = [backward_tc(*(inputs.widen(x[n][b, h], "bf16") for n in ("Qx", "Kx", "V")), x["mu"][h],
                                    x["rho"][h], x["alpha"][h], w.var_floor, w.eps, dO[b, h], two) for b in range(B)]
                for b in range(B):
                    floor = 1e-2 * max(np.abs(refs[b]["Qx"]).max(), np.abs(refs[b]["Kx"]).max())
                    for n in ("Qx", "Kx", "V"):
                        den = max(np.abs(refs[b][n]).max(), floor if n != "V" else 0.0)
                        worst[two] = max(worst[two], float(np.abs(gots[b][n] - refs[b][n]).max() / den))
                for n in ("mu", "omega", "alpha"):
                    worst[two] = max(worst[two], err(sum(g[n] for g in gots), sum(r[n] for r in refs)))
    print("backward as built on the tensor cores, six small workloads (worst over gradients and heads)")
    print(f"  memories [Vt | Z], [R | r] as one bf16 term       {worst[False]:.1e}")
    print(f"  memories as two bf16 terms (the kernel)           {worst[True]:.1e}")


if __name__ == "__main__":
    forward_study()
    backward_study()
    backward_kernel_study()
