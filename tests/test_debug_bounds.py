"""The index-checking debug build (GMA_DEBUG_BOUNDS): every forward path, the
tensor-core and general backward, the projection GEMM, the diagnostics and a
gma_forward_multi request run with their
global-memory indices checked on the device, on outputs and workspaces padded with
canary bytes.  A failed check posts GMA_ERR_BOUNDS to the status word (instead of
trapping), so the test asserts a clean status, untouched canaries on both sides of
every output and after every workspace, and results that still match the fp64 oracle.
The debug library is loaded in a child process (the GMA_LIBRARY override), so this
process keeps the normal build."""
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

# the tensor-core backward (bidirectional bf16; 252 tiles over the persistent CTAs, so CTAs
# and both compute groups cross head boundaries): canary-padded gradients and workspace
import ctypes
w = inputs.Workload("bwd_tc", seed=7, B=1, H=4, N=8000, d=64, K=64, dv=64, dtype="bf16", causal=False)
x = inputs.gen_all(w)
x["dO"] = x["V"][:, ::-1].copy()
desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, w.dv, torch.bfloat16, torch.bfloat16, w.var_floor, 0)
nb = ctypes.c_size_t(0)
assert gma._load().gma_backward_workspace_size(ctypes.byref(desc), 0, ctypes.byref(nb)) == 0
need = nb.value
ws = workspace(need)
shapes = ((w.B, w.H, w.N, w.d), (w.B, w.H, w.N, w.d), (w.B, w.H, w.N, w.dv), (w.H, w.K, w.d), (w.H, w.K, w.d),
          (w.H, w.K))
pads = [padded(shp, torch.float32) for shp in shapes]
grads = gma.gma_backward(*(to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")), eps=w.eps,
                         var_floor=w.var_floor, grads=tuple(t for _, t in pads), workspace=ws)
torch.cuda.synchronize()
st = gma.gma_get_status(ws)
assert st == 0, ("bwd_tc", gma.gma_status_string(st))
assert all(canaries_ok(f, torch.float32) for f, _ in pads), ("bwd_tc", "gradient canaries")
assert bool((ws[need:] == CANARY_BYTE).all()), ("bwd_tc", "workspace canaries")
wid = lambda a: inputs.widen(a, "bf16")
worst = 0.0
for h in (0, 3):
    ref = oracle.backward_head(wid(x["Qx"][0, h]), wid(x["Kx"][0, h]), wid(x["V"][0, h]), x["mu"][h], x["rho"][h],
                               x["alpha"][h], w.var_floor, w.eps, False, wid(x["dO"][0, h]))
    got = [t.double().cpu().numpy() for t in grads]
    floor = 1e-2 * max(np.abs(ref["Qx"]).max(), np.abs(ref["Kx"]).max())
    for i, nm in enumerate(("Qx", "Kx", "V")):
        den = max(np.abs(ref[nm]).max(), floor if nm != "V" else 0.0)
        worst = max(worst, float(np.abs(got[i][0, h] - ref[nm]).max() / den))
    for i, nm in ((3, "mu"), (4, "omega"), (5, "alpha")):
        worst = max(worst, float(np.abs(got[i][h] - ref[nm]).max() / np.abs(ref[nm]).max()))
assert worst <= TOL["bf16"], ("bwd_tc", worst)
print(f"bwd_tc: status clean, canaries intact, max relative error {worst:.2e}")

# the projection GEMM: canary-padded outputs (a ragged row tile and a partial column tile)
B, N, D, H = 2, 300, 128, 3
rng = np.random.default_rng(9)
bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()
Xh, Wqh, Wkh, Wvh = (rng.normal(size=s_) * c for s_, c in (((B, N, D), 1.0), ((H, D, 64), D ** -0.5),
                                                            ((H, D, 64), D ** -0.5), ((H, D, 64), D ** -0.5)))
ws = workspace(256)
pads = [padded((B, H, N, 64), torch.bfloat16) for _ in range(3)]
outs = gma.gma_project(bf(Xh), bf(Wqh), bf(Wkh), bf(Wvh), out=tuple(t for _, t in pads), workspace=ws)
torch.cuda.synchronize()
st = gma.gma_get_status(ws)
assert st == 0, ("project", gma.gma_status_string(st))
assert all(canaries_ok(f, torch.bfloat16) for f, _ in pads), ("project", "output canaries")
assert bool((ws[256:] == CANARY_BYTE).all()), ("project", "workspace canaries")
wd = lambda t: t.float().cpu().numpy().astype(np.float64)
refs = oracle.project(*(wd(bf(a)) for a in (Xh, Wqh, Wkh, Wvh)))
err = max(np.abs(wd(o)[b, h] - r[b, h]).max() / np.abs(r[b, h]).max() for o, r in zip(outs, refs)
          for b in range(B) for h in range(H))
assert err <= 5.5e-3, ("project", err)
print(f"project: status clean, canaries intact, max relative error {err:.2e}")

# the diagnostics (K = 64: two epilogue groups; K = 128: one), with the workspace padded
for K_, N_ in ((64, 700), (128, 300)):
    w = inputs.Workload(f"diag_k{K_}", seed=7, B=2, H=3, N=N_, d=64, K=K_, dv=64, dtype="bf16", causal=False)
    x = inputs.gen_all(w)
    desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, 1, torch.bfloat16, torch.bfloat16, w.var_floor, 0)
    nb = ctypes.c_size_t(0)
    assert gma._load().gma_diagnostics_workspace_size(ctypes.byref(desc), ctypes.byref(nb)) == 0
    ws = workspace(nb.value)
    p_, stats_, z_ = gma.gma_diagnostics(*(to_device(x[n]) for n in ("Qx", "mu", "rho", "alpha")),
                                         var_floor=w.var_floor, workspace=ws)
    torch.cuda.synchronize()
    st = gma.gma_get_status(ws)
    assert st == 0, (w.name, gma.gma_status_string(st))
    assert bool((ws[nb.value:] == CANARY_BYTE).all()), (w.name, "workspace canaries")
    rp, hu, ht, rm, rz = oracle.diagnostics(inputs.widen(x["Qx"], "bf16"), x["mu"], x["rho"], x["alpha"],
                                            w.var_floor)
    gp = p_.double().cpu().numpy()
    err = max(float(np.abs(gp - rp).max() / rp.max()),
              float(np.abs(stats_.double().cpu().numpy() - np.array([hu, ht, rm])).max()))
    agree = float((z_.cpu().numpy() == rz).mean())
    assert err <= 2e-2 and agree >= 0.99, (w.name, err, agree)
    print(f"{w.name}: status clean, canaries intact, p/stats error {err:.2e}, argmax agreement {agree:.4f}")
# the general backward (causal, K = 128: the chunk walks and the tiled products)
w = inputs.Workload("bwd_general", seed=7, B=1, H=2, N=300, d=64, K=128, dv=64, dtype="bf16", causal=True)
x = inputs.gen_all(w)
x["dO"] = x["V"][:, ::-1].copy()
desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, w.dv, torch.bfloat16, torch.bfloat16, w.var_floor, 0)
nb = ctypes.c_size_t(0)
assert gma._load().gma_backward_workspace_size(ctypes.byref(desc), 1, ctypes.byref(nb)) == 0
need = nb.value
ws = workspace(need)
shapes = ((w.B, w.H, w.N, w.d), (w.B, w.H, w.N, w.d), (w.B, w.H, w.N, w.dv), (w.H, w.K, w.d), (w.H, w.K, w.d),
          (w.H, w.K))
pads = [padded(shp, torch.float32) for shp in shapes]
grads = gma.gma_backward(*(to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha", "dO")), eps=w.eps,
                         var_floor=w.var_floor, causal=True, grads=tuple(t for _, t in pads), workspace=ws)
torch.cuda.synchronize()
st = gma.gma_get_status(ws)
assert st == 0, ("bwd_general", gma.gma_status_string(st))
assert all(canaries_ok(f, torch.float32) for f, _ in pads), ("bwd_general", "gradient canaries")
assert bool((ws[need:] == CANARY_BYTE).all()), ("bwd_general", "workspace canaries")
worst = 0.0
got = [t.double().cpu().numpy() for t in grads]
for h in (0, 1):
    ref = oracle.backward_head(wid(x["Qx"][0, h]), wid(x["Kx"][0, h]), wid(x["V"][0, h]), x["mu"][h], x["rho"][h],
                               x["alpha"][h], w.var_floor, w.eps, True, wid(x["dO"][0, h]))
    floor = 1e-2 * max(np.abs(ref["Qx"]).max(), np.abs(ref["Kx"]).max())
    for i, nm in enumerate(("Qx", "Kx", "V")):
        den = max(np.abs(ref[nm]).max(), floor if nm != "V" else 0.0)
        worst = max(worst, float(np.abs(got[i][0, h] - ref[nm]).max() / den))
    for i, nm in ((3, "mu"), (4, "omega"), (5, "alpha")):
        worst = max(worst, float(np.abs(got[i][h] - ref[nm]).max() / np.abs(ref[nm]).max()))
assert worst <= 1e-3, ("bwd_general", worst)
print(f"bwd_general: status clean, canaries intact, max relative error {worst:.2e}")

# a gma_forward_multi request: the per-head causal scan on a second stream beside the
# bidirectional forward, canary-padded outputs, every region's header zero, canaries after
w = inputs.Workload("multi", seed=7, B=2, H=48, N=300, d=64, K=64, dv=64, dtype="bf16", causal=True)
x = inputs.gen_all(w)
d_ = {n: to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha")}
pads = [padded((w.B, w.H, w.N, w.dv), torch.bfloat16) for _ in range(2)]
calls = [dict(Qx=d_["Qx"], Kx=d_["Kx"], V=d_["V"], mu=d_["mu"], rho=d_["rho"], pi_logits=d_["alpha"], eps=w.eps,
              causal=c, var_floor=w.var_floor, out=pads[k][1]) for k, c in enumerate((False, True))]
arr = (gma.gma_forward_call * 2)()
for k, c in enumerate((False, True)):
    arr[k].desc = gma._make_desc(w.B, w.H, w.N, w.d, w.K, w.dv, torch.bfloat16, torch.bfloat16, w.var_floor, 0)
    arr[k].causal = int(c)
offs = (ctypes.c_size_t * 2)()
assert gma._load().gma_forward_multi_workspace_size(arr, 2, ctypes.byref(nb), offs) == 0
need = nb.value
ws = workspace(need)
for o in offs:
    ws[o:o + 256] = 0
gma.gma_forward_multi(calls, workspace=ws, aux_stream=torch.cuda.Stream())
torch.cuda.synchronize()
for o in offs:
    st = gma._load().gma_get_status(int(ws.data_ptr()) + o, int(torch.cuda.current_stream().cuda_stream))
    assert st == 0, ("multi", gma.gma_status_string(st))
assert all(canaries_ok(f, torch.bfloat16) for f, _ in pads), ("multi", "output canaries")
assert bool((ws[need:] == CANARY_BYTE).all()), ("multi", "workspace canaries")
worst = 0.0
for (f, o), c in zip(pads, (False, True)):
    wc = w.replace(causal=c)
    gotc = to_f64(o).reshape(wc.G, wc.N, wc.dv)
    worst = max(worst, max(head_rel_err(gotc[g], oracle_head(wc, x, g)) for g in (0, 47, 95)))
assert worst <= TOL["bf16"], ("multi", worst)
print(f"multi: status clean, canaries intact, max relative error {worst:.2e}")
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
