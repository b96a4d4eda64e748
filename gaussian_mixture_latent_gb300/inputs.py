"""Seeded synthetic inputs for the Gaussian Mixture Attention forward.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no softplus, softmax, densities or contractions).  Both
the CPU oracle's tests and the CUDA path take their inputs from here.

Generator (defined here, bit-reproducible on x86-64 and aarch64 up to the
last-ulp behaviour of numpy's log/cos):

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014), used counter-style: element ``i`` of stream
  ``key`` is ``mix(key + (i + 1) * 0x9E3779B97F4A7C15)``.  Any element range
  can therefore be regenerated on its own (sampled parity checks on large
  workloads regenerate only the rows they need).
* Uniforms on (0, 1): ``((z >> 11) + 0.5) * 2**-53``.
* Normals by Box-Muller (cosine branch only): normal ``i`` of a stream uses
  uniforms ``2i`` and ``2i + 1``.

Workloads follow the configurations the method is measured on: routing
vectors Qx, Kx and values V drawn N(0, 1); means mu ~ N(0, s_mu); variance
pre-activations rho ~ N(0, 0.5); prior logits ~ N(0, 1).  ``N(a, b)`` is
read as mean a and *standard deviation* b.  The long causal workload mixes
10 % of routing rows with copies of a uniformly chosen component mean plus
N(0, 0.1) noise (independently for Qx and Kx, per head), which gives peaked
responsibilities.

bf16 tensors are returned as ``uint16`` bit patterns (round to nearest even
from float32); ``bf16_bits_to_f64`` widens them exactly.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TWO53 = float(2 ** 53)

# Stream identifiers: one per drawn tensor, fixed so any consumer can
# regenerate a tensor (or a slice of it) without drawing the others.
STREAM = {
    "Qx": 1, "Kx": 2, "V": 3, "mu": 4, "rho": 5, "alpha": 6,
    "Qx_mix_sel": 7, "Qx_mix_comp": 8, "Qx_mix_noise": 9,
    "Kx_mix_sel": 10, "Kx_mix_comp": 11, "Kx_mix_noise": 12,
    "dO": 13,                    # upstream gradient of the backward pass
    "X": 14, "Wq": 15, "Wk": 16, "Wv": 17,   # layer input and projection weights (Eq. 4)
}


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, name: str) -> np.uint64:
    """64-bit key of the stream that draws tensor ``name`` under ``seed``."""
    with np.errstate(over="ignore"):
        base = np.array([(seed * 0x100000001B3 + STREAM[name]) & 0xFFFFFFFFFFFFFFFF],
                        dtype=np.uint64)
        return _mix64(base + _GOLDEN)[0]


def splitmix64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Raw 64-bit outputs ``start .. start+count-1`` of stream ``key``."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix64(np.uint64(key) + ctr * _GOLDEN)


def uniform(key: np.uint64, start: int, count: int) -> np.ndarray:
    z = splitmix64(key, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) / _TWO53


def _normal_chunk(key, start, count):
    u = uniform(key, 2 * start, 2 * count)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def normal(key: np.uint64, start: int, count: int, threads: int | None = None) -> np.ndarray:
    """Standard normals ``start .. start+count-1`` of stream ``key`` (float64)."""
    chunk = 1 << 22
    if count <= chunk:
        return _normal_chunk(key, start, count)
    out = np.empty(count, dtype=np.float64)
    spans = [(s, min(chunk, count - s)) for s in range(0, count, chunk)]
    nthreads = threads or max(1, min(16, len(os.sched_getaffinity(0))))

    def work(span):
        s, c = span
        out[s:s + c] = _normal_chunk(key, start + s, c)

    with ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(work, spans))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape, dtype and value distributions of one synthetic GMA workload."""
    name: str
    B: int
    H: int
    N: int
    d: int
    K: int
    dv: int
    dtype: str            # "f32" or "bf16": dtype of Qx, Kx, V and of the output
    causal: bool
    mu_std: float = 1.0
    rho_std: float = 0.5
    alpha_std: float = 1.0
    mix_frac: float = 0.0  # fraction of routing rows replaced by mu rows + noise
    mix_noise: float = 0.1
    var_floor: float = 1e-4
    eps: float = 1e-6
    seed: int = 0

    @property
    def G(self) -> int:
        return self.B * self.H

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "bidir_f32_n256": Workload("bidir_f32_n256", B=1, H=1, N=256, d=16, K=8, dv=32,
                               dtype="f32", causal=False),
    "bidir_bf16_n4096": Workload("bidir_bf16_n4096", B=8, H=8, N=4096, d=64, K=64, dv=64,
                                 dtype="bf16", causal=False),
    "causal_bf16_n8192": Workload("causal_bf16_n8192", B=8, H=12, N=8192, d=64, K=64, dv=64,
                                  dtype="bf16", causal=True),
    "bidir_bf16_n65536": Workload("bidir_bf16_n65536", B=2, H=8, N=65536, d=64, K=128, dv=64,
                                  dtype="bf16", causal=False, mu_std=2.0),
    "causal_bf16_n131072": Workload("causal_bf16_n131072", B=1, H=16, N=131072, d=64, K=256,
                                    dv=128, dtype="bf16", causal=True, mix_frac=0.1),
}


def _cast(x64: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x64.astype(np.float32)
    return f32_to_bf16_bits(x32) if dtype == "bf16" else x32


def gen_params(w: Workload) -> dict:
    """mu, rho [H, K, d] and alpha [H, K], float32 (parameters are per head)."""
    H, K, d = w.H, w.K, w.d
    mu = (w.mu_std * normal(stream_key(w.seed, "mu"), 0, H * K * d)).astype(np.float32)
    rho = (w.rho_std * normal(stream_key(w.seed, "rho"), 0, H * K * d)).astype(np.float32)
    alpha = (w.alpha_std * normal(stream_key(w.seed, "alpha"), 0, H * K)).astype(np.float32)
    return {"mu": mu.reshape(H, K, d), "rho": rho.reshape(H, K, d), "alpha": alpha.reshape(H, K)}


def gen_rows(w: Workload, name: str, g: int, r0: int, r1: int, params: dict | None = None) -> np.ndarray:
    """Rows ``r0:r1`` of head ``g`` (= b*H + h) of Qx, Kx or V, float64 before the cast."""
    width = w.dv if name == "V" else w.d
    n = r1 - r0
    start = (g * w.N + r0) * width
    x = normal(stream_key(w.seed, name), start, n * width).reshape(n, width)
    if name != "V" and w.mix_frac > 0.0:
        if params is None:
            params = gen_params(w)
        h = g % w.H
        sel = uniform(stream_key(w.seed, name + "_mix_sel"), g * w.N + r0, n) < w.mix_frac
        comp = np.minimum((uniform(stream_key(w.seed, name + "_mix_comp"), g * w.N + r0, n)
                           * w.K).astype(np.int64), w.K - 1)
        noise = w.mix_noise * normal(stream_key(w.seed, name + "_mix_noise"), start, n * width
                                     ).reshape(n, width)
        mu_h = params["mu"][h].astype(np.float64)
        x = np.where(sel[:, None], mu_h[comp] + noise, x)
    return x


def gen_head(w: Workload, name: str, g: int, params: dict | None = None) -> np.ndarray:
    """One head of Qx / Kx / V in the workload dtype ([N, width])."""
    return _cast(gen_rows(w, name, g, 0, w.N, params), w.dtype)


def gen_all(w: Workload) -> dict:
    """Every input of the workload: Qx, Kx [B,H,N,d], V [B,H,N,dv] in the workload dtype
    (bf16 as uint16 bits), mu, rho [H,K,d] and alpha [H,K] float32."""
    p = gen_params(w)
    out = dict(p)
    for name in ("Qx", "Kx", "V"):
        width = w.dv if name == "V" else w.d
        arr = np.empty((w.G, w.N, width), dtype=np.uint16 if w.dtype == "bf16" else np.float32)
        for g in range(w.G):
            arr[g] = gen_head(w, name, g, p)
        out[name] = arr.reshape(w.B, w.H, w.N, width)
    return out


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 copy of an input tensor stored in ``dtype``."""
    return bf16_bits_to_f64(x) if dtype == "bf16" else np.asarray(x, dtype=np.float64)
