"""The index-checking debug build (GMA_DEBUG_BOUNDS): every forward path runs with
its global-memory indices checked on the device, on outputs and workspaces padded
with canary bytes.  A failed check posts GMA_ERR_BOUNDS to the status word
(instead of trapping), so the test asserts a clean status, untouched canaries on
both sides of every output and after every workspace, and results that still
match the fp64 oracle.  The debug library is loaded in a child process (the
GMA_LIBRARY override), so this process keeps the normal build."""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import numpy as np, torch
import gaussian_mixture_latent_gb300 as gma
import oracle
from gaussian_mixture_latent_gb300 import inputs
from tests._util import TOL, head_rel_err, oracle_head, to_device, to_f64
assert gma.library_path().endswith("libgma_debug.so"), gma.library_path()
PAD = 64                                   # canary elements on each side of an output
CANARY_F32, CANARY_BF16, CANARY_BYTE = 0x7F7A5A5A, 0x7E5A, 0xA5

def padded(shape, dtype):
    n = int(np.prod(shape))
    flat = torch.empty(n + 2 * PAD, dtype=dtype, device="cuda")
    bits = flat.view(torch.int32 if dtype == torch.float32 else torch.int16)
    bits.fill_(CANARY_F32 if dtype == torch.float32 else CANARY_BF16)
    return flat, flat[PAD:PAD + n].view(shape)

def canaries_ok(flat, dtype):
    bits = flat.view(torch.int32 if dtype == torch.float32 else torch.int16)
    want = CANARY_F32 if dtype == torch.float32 else CANARY_BF16
    return bool((bits[:PAD] == want).all() and (bits[-PAD:] == want).all())

def workspace(nbytes):
    ws = torch.full((nbytes + 4096,), CANARY_BYTE, dtype=torch.uint8, device="cuda")
    ws[:256] = 0
    return ws

def check(name, w, x, out_flat, out, ws, need, heads):
    torch.cuda.synchronize()
    st = gma.gma_get_status(ws)
    assert st == 0, (name, gma.gma_status_string(st))
    tdt = out.dtype
    assert canaries_ok(out_flat, tdt), (name, "output canaries")
    assert bool((ws[need:] == CANARY_BYTE).all()), (name, "workspace canaries")
    got = to_f64(out).reshape(w.G, w.N, w.dv)
    err = max(head_rel_err(got[g], oracle_head(w, x, g)) for g in heads)
    assert err <= TOL[w.dtype], (name, err)
    print(f"{name}: status clean, canaries intact, max relative error {err:.2e}")

cases = [
    ("bidir_k64", dict(B=1, H=3, N=700, d=64, K=64, dv=64, dtype="bf16", causal=False)),
    ("bidir_k128", dict(B=1, H=2, N=500, d=64, K=128, dv=64, dtype="bf16", causal=False)),
    ("causal_segmented", dict(B=1, H=3, N=1500, d=64, K=64, dv=64, dtype="bf16", causal=True)),
    ("causal_per_head", dict(B=2, H=48, N=300, d=64, K=64, dv=64, dtype="bf16", causal=True)),
    ("causal_sliced", dict(B=1, H=2, N=400, d=64, K=256, dv=128, dtype="bf16", causal=True)),
    ("fp32_bidir", dict(B=1, H=2, N=300, d=16, K=8, dv=32, dtype="f32", causal=False)),
    ("fp32_causal", dict(B=1, H=2, N=300, d=16, K=8, dv=32, dtype="f32", causal=True)),
]
for name, kw in cases:
    w = inputs.Workload(name, seed=7, **kw)
    x = inputs.gen_all(w)
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, w.dv, tdt, tdt, w.var_floor, 0)
    need = gma.gma_workspace_size(desc, w.causal)
    ws = workspace(need)
    out_flat, out = padded((w.B, w.H, w.N, w.dv), tdt)
    gma.gma_forward(*(to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha")), eps=w.eps,
                    causal=w.causal, var_floor=w.var_floor, out=out, workspace=ws)
    check(name, w, x, out_flat, out, ws, need, [0, w.G - 1])
print("ALL_OK")
'''


def test_debug_build_checks_indices_and_keeps_canaries():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gaussian_mixture_latent_gb300 import _build
    lib = _build.build(debug=True)
    env = dict(os.environ, GMA_LIBRARY=lib, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    print(r.stdout)
    assert r.returncode == 0 and "ALL_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
