"""Plain fp64 CPU oracle for the Gaussian Mixture Attention forward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path
(``gaussian_mixture_latent_gb300`` and its CUDA library) never does.

The arithmetic lives in ``gma_oracle.c`` (double precision, written from the
equations of "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
Probabilistic Latent Routing", section 3 -- Eqs. 3, 3b, 5-8, 6b, 8b, 14-16, and the
input projections of Eq. 4 -- and, for the backward pass, section 4.1 -- Eqs. 17-20).
This module only marshals numpy arrays into it.

Every function here is pinned by ``tests/test_oracle.py`` against things the
paper and the mathematics fix (a textbook density routine, the explicit N x N
affinity, closed forms and invariants); see that file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gma_oracle.c")
_SO = os.path.join(_HERE, "libgma_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        cc = os.environ.get("CC", "gcc")
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call([cc, "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i, d = ctypes.c_int, ctypes.c_double
        lib.gma_oracle_scores.argtypes = [i, i, i, _dp, _dp, _dp, _dp, d, _dp]
        lib.gma_oracle_responsibilities.argtypes = [i, i, i, _dp, _dp, _dp, _dp, d, _dp]
        lib.gma_oracle_forward_head.argtypes = [i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, d, d,
                                                i, _dp, _dp, _dp]
        lib.gma_oracle_forward.argtypes = [i, i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, d, d,
                                           i, _dp, i]
        lib.gma_oracle_diagnostics.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, d, _dp, _dp,
                                               ctypes.POINTER(ctypes.c_int)]
        lib.gma_oracle_cross_head.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, d, d, _dp]
        lib.gma_oracle_backward_head.argtypes = [i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, d, d, i, _dp,
                                                 _dp, _dp, _dp, _dp, _dp, _dp]
        lib.gma_oracle_project.argtypes = [i, i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
        for fn in (lib.gma_oracle_scores, lib.gma_oracle_responsibilities,
                   lib.gma_oracle_forward_head, lib.gma_oracle_forward, lib.gma_oracle_diagnostics,
                   lib.gma_oracle_cross_head, lib.gma_oracle_backward_head, lib.gma_oracle_project):
            fn.restype = ctypes.c_int
        _lib = lib
    return _lib


def _c(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def scores(X, mu, omega, alpha, var_floor: float) -> np.ndarray:
    """Eq. (16) log-density scores s [N, K] for the rows of X [N, d]."""
    X, mu, omega, alpha = _c(X), _c(mu), _c(omega), _c(alpha)
    N, d = X.shape
    K = mu.shape[0]
    out = np.empty((N, K), dtype=np.float64)
    _check(_load().gma_oracle_scores(N, d, K, _p(X), _p(mu), _p(omega), _p(alpha),
                                     float(var_floor), _p(out)), "scores")
    return out


def responsibilities(X, mu, omega, alpha, var_floor: float) -> np.ndarray:
    """Eq. (3)/(3b) responsibilities Gamma [N, K] for the rows of X [N, d]."""
    X, mu, omega, alpha = _c(X), _c(mu), _c(omega), _c(alpha)
    N, d = X.shape
    K = mu.shape[0]
    out = np.empty((N, K), dtype=np.float64)
    _check(_load().gma_oracle_responsibilities(N, d, K, _p(X), _p(mu), _p(omega), _p(alpha),
                                               float(var_floor), _p(out)), "responsibilities")
    return out


def forward_head(Qx, Kx, V, mu, omega, alpha, var_floor: float, eps: float, causal: bool,
                 return_memory: bool = False):
    """One head: O [N, dv] (Eq. 7-8, or 8b when causal).  With ``return_memory`` also
    the latent memory Vt [K, dv] and normaliser Z [K] (Eq. 5-6; for the causal
    variant the prefix memory after the last position)."""
    Qx, Kx, V, mu, omega, alpha = map(_c, (Qx, Kx, V, mu, omega, alpha))
    N, d = Qx.shape
    K = mu.shape[0]
    dv = V.shape[1]
    out = np.empty((N, dv), dtype=np.float64)
    Vt = np.empty((K, dv), dtype=np.float64)
    Z = np.empty((K,), dtype=np.float64)
    _check(_load().gma_oracle_forward_head(N, d, K, dv, _p(Qx), _p(Kx), _p(V), _p(mu), _p(omega),
                                           _p(alpha), float(var_floor), float(eps), int(causal),
                                           _p(out), _p(Vt), _p(Z)), "forward_head")
    return (out, Vt, Z) if return_memory else out


def forward(Qx, Kx, V, mu, omega, alpha, var_floor: float, eps: float, causal: bool,
            threads: int = 1) -> np.ndarray:
    """All heads: Qx, Kx [B, H, N, d], V [B, H, N, dv], parameters [H, K, d] / [H, K]
    -> O [B, H, N, dv] in float64.  Heads run on ``threads`` POSIX threads."""
    Qx, Kx, V, mu, omega, alpha = map(_c, (Qx, Kx, V, mu, omega, alpha))
    B, H, N, d = Qx.shape
    K = mu.shape[1]
    dv = V.shape[3]
    out = np.empty((B, H, N, dv), dtype=np.float64)
    _check(_load().gma_oracle_forward(B, H, N, d, K, dv, _p(Qx), _p(Kx), _p(V), _p(mu), _p(omega),
                                      _p(alpha), float(var_floor), float(eps), int(causal),
                                      _p(out), int(threads)), "forward")
    return out


def diagnostics(Qx, mu, omega, alpha, var_floor: float):
    """Responsibility diagnostics (section 5.4, Eqs. 24-29) over the query
    responsibilities of every head: Qx [B, H, N, d], parameters [H, K, d] / [H, K]
    -> (p [K], H_usage, H_token, R_max, z [B, N] int32)."""
    Qx, mu, omega, alpha = map(_c, (Qx, mu, omega, alpha))
    B, H, N, d = Qx.shape
    K = mu.shape[1]
    p = np.empty((K,), dtype=np.float64)
    stats = np.empty((3,), dtype=np.float64)
    z = np.empty((B, N), dtype=np.int32)
    _check(_load().gma_oracle_diagnostics(B, H, N, d, K, _p(Qx), _p(mu), _p(omega), _p(alpha),
                                          float(var_floor), _p(p), _p(stats),
                                          z.ctypes.data_as(ctypes.POINTER(ctypes.c_int))), "diagnostics")
    return p, float(stats[0]), float(stats[1]), float(stats[2]), z


def cross_head(Qx, Ky, Vy, mu, omega, alpha, var_floor: float, eps: float) -> np.ndarray:
    """Cross-attention GMA for one head (sections 3.1, 6): queries Qx [Nq, d] read the
    memory of a context Ky [Nkv, d], Vy [Nkv, dv] -> O [Nq, dv] (Eq. 5-8, bidirectional)."""
    Qx, Ky, Vy, mu, omega, alpha = map(_c, (Qx, Ky, Vy, mu, omega, alpha))
    Nq, d = Qx.shape
    Nkv = Ky.shape[0]
    K = mu.shape[0]
    dv = Vy.shape[1]
    out = np.empty((Nq, dv), dtype=np.float64)
    _check(_load().gma_oracle_cross_head(Nq, Nkv, d, K, dv, _p(Qx), _p(Ky), _p(Vy), _p(mu), _p(omega),
                                         _p(alpha), float(var_floor), float(eps), _p(out)), "cross_head")
    return out


def backward_head(Qx, Kx, V, mu, omega, alpha, var_floor: float, eps: float, causal: bool, dO):
    """Backward pass of one head (section 4.1, Eqs. 17-20, with Eqs. 14-15 and the memory
    products of Eqs. 5-8 / 6b, 8b): given dO = dL/dO [N, dv], returns the dict of
    dL/dQx, dL/dKx [N, d], dL/dV [N, dv], dL/dmu, dL/domega [K, d], dL/dalpha [K]."""
    Qx, Kx, V, mu, omega, alpha, dO = map(_c, (Qx, Kx, V, mu, omega, alpha, dO))
    N, d = Qx.shape
    K = mu.shape[0]
    dv = V.shape[1]
    g = {"Qx": np.empty((N, d)), "Kx": np.empty((N, d)), "V": np.empty((N, dv)),
         "mu": np.empty((K, d)), "omega": np.empty((K, d)), "alpha": np.empty((K,))}
    _check(_load().gma_oracle_backward_head(N, d, K, dv, _p(Qx), _p(Kx), _p(V), _p(mu), _p(omega),
                                            _p(alpha), float(var_floor), float(eps), int(causal), _p(dO),
                                            _p(g["Qx"]), _p(g["Kx"]), _p(g["V"]), _p(g["mu"]),
                                            _p(g["omega"]), _p(g["alpha"])), "backward_head")
    return g


def project(X, Wq, Wk, Wv):
    """Input projections (section 3.1, Eq. 4): X [B, N, D], Wq and Wk [H, D, d], Wv [H, D, dv]
    -> (Qx, Kx [B, H, N, d], V [B, H, N, dv]), Qx[b, h] = X[b] Wq[h] and so on."""
    X, Wq, Wk, Wv = map(_c, (X, Wq, Wk, Wv))
    B, N, D = X.shape
    H, _, d = Wq.shape
    dv = Wv.shape[2]
    Qx = np.empty((B, H, N, d))
    Kx = np.empty((B, H, N, d))
    V = np.empty((B, H, N, dv))
    _check(_load().gma_oracle_project(B, N, D, H, d, dv, _p(X), _p(Wq), _p(Wk), _p(Wv), _p(Qx), _p(Kx), _p(V)),
           "project")
    return Qx, Kx, V

