"""The C ABI library loads and exports every entry point include/gma.h declares;
host-only argument checks return the documented codes (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_mixture_latent_gb300 as gma
    return gma._load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gma.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gma_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gma_forward", "gma_workspace_size", "gma_responsibilities",
                     "gma_get_status", "gma_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_has_sm103a_code_only():
    import subprocess
    import gaussian_mixture_latent_gb300 as gma
    r = subprocess.run(["cuobjdump", "--list-elf", gma.library_path()], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    archs = set(re.findall(r"sm_\d+a?", r.stdout))
    assert archs == {"sm_103a"}, archs


def _desc(**kw):
    import gaussian_mixture_latent_gb300 as gma
    base = dict(B=2, H=3, N=100, d=16, K=8, dv=32, in_dtype=1, out_dtype=1, var_floor=1e-4, chunk=0)
    base.update(kw)
    return gma.gma_desc(**base)


def test_workspace_size_and_argument_errors(lib):
    n = ctypes.c_size_t(0)
    assert lib.gma_workspace_size(ctypes.byref(_desc()), 0, ctypes.byref(n)) == 0
    assert n.value >= 256
    assert lib.gma_workspace_size(ctypes.byref(_desc()), 1, ctypes.byref(n)) == 0
    assert lib.gma_workspace_size(None, 0, ctypes.byref(n)) == 1
    for bad in (dict(B=0), dict(H=-1), dict(N=-5), dict(d=0), dict(K=0), dict(dv=0),
                dict(in_dtype=7), dict(var_floor=0.0), dict(var_floor=float("nan")), dict(chunk=-1)):
        assert lib.gma_workspace_size(ctypes.byref(_desc(**bad)), 0, ctypes.byref(n)) == 1, bad
    for unsup in (dict(d=257), dict(K=300), dict(dv=1024)):
        assert lib.gma_workspace_size(ctypes.byref(_desc(**unsup)), 0, ctypes.byref(n)) == 2, unsup


def test_forward_rejects_bad_arguments_before_launching(lib):
    import gaussian_mixture_latent_gb300 as gma
    d = _desc()
    p = ctypes.c_void_p(4096)      # never dereferenced: every case fails validation first
    odd = ctypes.c_void_p(4100)    # not 16-byte aligned
    f = lib.gma_forward
    args = lambda **o: [ctypes.byref(o.get("desc", d)), o.get("Q", p), p, p, p, p, p,
                        o.get("eps", 1e-6), o.get("causal", 0), o.get("out", p),
                        o.get("ws", p), o.get("wsb", 1 << 40), None]
    assert f(*args(desc=_desc(K=0))) == 1
    assert f(*args(eps=-1.0)) == 1
    assert f(*args(eps=float("inf"))) == 1
    assert f(*args(causal=2)) == 1
    assert f(*args(Q=None)) == 1
    assert f(*args(Q=odd)) == 1
    assert f(*args(out=None)) == 1
    assert f(*args(ws=None)) == 3
    assert f(*args(wsb=16)) == 3
    assert gma.gma_status_string(3).startswith("GMA_ERR_WORKSPACE")
    assert lib.gma_version() >= 100


def test_backward_and_decode_reject_bad_arguments_before_launching(lib):
    # every call below fails validation: the placeholder pointers are never dereferenced
    n = ctypes.c_size_t(0)
    ok = _desc(d=64, K=64, dv=64)
    assert lib.gma_backward_workspace_size(ctypes.byref(ok), 0, ctypes.byref(n)) == 0 and n.value > 0
    bidir = n.value
    assert lib.gma_backward_workspace_size(ctypes.byref(ok), 1, ctypes.byref(n)) == 0 and n.value > bidir
    assert lib.gma_backward_workspace_size(ctypes.byref(ok), 2, ctypes.byref(n)) == 1
    # every other shape takes the general path, except a causal state beyond shared memory
    assert lib.gma_backward_workspace_size(ctypes.byref(_desc(d=64, K=128, dv=64)), 0, ctypes.byref(n)) == 0
    assert lib.gma_backward_workspace_size(ctypes.byref(_desc(d=64, K=256, dv=256)), 0, ctypes.byref(n)) == 0
    assert lib.gma_backward_workspace_size(ctypes.byref(_desc(d=64, K=256, dv=256)), 1, ctypes.byref(n)) == 2
    assert lib.gma_backward_workspace_size(ctypes.byref(_desc(d=64, K=64, dv=64, out_dtype=0)), 0,
                                           ctypes.byref(n)) == 2
    p = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4100)
    b = lib.gma_backward
    args = lambda **o: [ctypes.byref(o.get("desc", ok)), o.get("causal", 0), o.get("Q", p), p, p, p, p, p,
                        o.get("eps", 1e-6), o.get("dO", p), p, p, p, o.get("dmu", p), p, p,
                        o.get("ws", p), o.get("wsb", 1 << 40), None]
    assert b(*args(causal=2)) == 1
    assert b(*args(eps=-1.0)) == 1
    assert b(*args(Q=None)) == 1
    assert b(*args(dO=odd)) == 1
    assert b(*args(dmu=None)) == 1
    assert b(*args(desc=_desc(d=64, K=256, dv=256), causal=1)) == 2
    assert b(*args(ws=None)) == 3
    assert b(*args(wsb=16)) == 3
    assert lib.gma_decode_workspace_size(ctypes.byref(ok), ctypes.byref(n)) == 0
    assert lib.gma_decode_workspace_size(ctypes.byref(_desc(d=64, K=256, dv=256)), ctypes.byref(n)) == 2
    dec = lib.gma_decode
    dargs = lambda **o: [ctypes.byref(o.get("desc", ok)), p, p, p, p, p, p, o.get("eps", 1e-6),
                         o.get("state", p), p, o.get("ws", p), o.get("wsb", 1 << 40), None]
    assert dec(*dargs(eps=float("nan"))) == 1
    assert dec(*dargs(state=None)) == 1
    assert dec(*dargs(state=odd)) == 1
    assert dec(*dargs(desc=_desc(d=64, K=256, dv=256))) == 2
    assert dec(*dargs(ws=None)) == 3
    assert dec(*dargs(wsb=1)) == 3


def test_chunk_is_honoured_or_refused(lib):
    # desc.chunk is the causal scan's chunk length: the tensor-core causal paths run
    # 128-row chunks and refuse any other value; the float32 CUDA-core path takes any
    # chunk whose tiles fit shared memory; bidirectional calls ignore it.
    n = ctypes.c_size_t(0)
    names = (ctypes.c_char_p * 16)()
    cnt = ctypes.c_int(0)
    ws = lambda causal, **kw: lib.gma_workspace_size(ctypes.byref(_desc(**kw)), causal, ctypes.byref(n))
    tc = dict(d=64, K=64, dv=64)
    sliced = dict(d=64, K=256, dv=128)
    for shape in (tc, sliced):
        assert ws(1, chunk=0, **shape) == 0
        assert ws(1, chunk=128, **shape) == 0
        for bad in (1, 64, 127, 256):
            assert ws(1, chunk=bad, **shape) == 2, (shape, bad)
        assert ws(0, chunk=64, **shape) == 0                       # bidirectional: ignored
        assert lib.gma_forward_plan(ctypes.byref(_desc(chunk=64, **shape)), 1, ctypes.byref(cnt), names, 16) == 2
    f32 = dict(d=16, K=8, dv=32, in_dtype=0, out_dtype=0)
    for good in (0, 1, 7, 16, 64, 128):
        assert ws(1, chunk=good, **f32) == 0, good
    assert ws(1, chunk=4096, **f32) == 2                            # tiles beyond shared memory
    assert ws(1, chunk=-1, **f32) == 1
    assert lib.gma_forward_plan(ctypes.byref(_desc(chunk=64, **f32)), 1, ctypes.byref(cnt), names, 16) == 0
    assert [names[i].decode() for i in range(cnt.value)][-1] == "simt_causal_chunk"
    # the backward: 64-row tiles at d = dv = K = 64 (chunk 0 or 64), the general path's chunk
    # otherwise while its tiles fit shared memory
    bws = lambda causal, **kw: lib.gma_backward_workspace_size(ctypes.byref(_desc(**kw)), causal, ctypes.byref(n))
    bw = dict(d=64, K=64, dv=64)
    for good in (0, 64, 16, 1, 32):
        assert bws(1, chunk=good, **bw) == 0, good
    assert bws(1, chunk=128, **bw) == 2
    assert bws(0, chunk=128, **bw) == 0
    for good in (0, 1, 16, 48):
        assert bws(1, chunk=good, **f32) == 0, good
    assert bws(1, chunk=4096, **f32) == 2


def test_project_rejects_bad_arguments_before_launching(lib):
    # every call below fails validation or launches nothing: the placeholder pointers are
    # never dereferenced
    import gaussian_mixture_latent_gb300 as gma
    p = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4100)
    pr = lib.gma_project

    def call(desc=(2, 300, 128, 3, 64, 64), X=p, Wq=p, ws=p, wsb=256):
        d = gma.gma_proj_desc(*desc)
        return pr(ctypes.byref(d), X, Wq, p, p, p, p, p, ws, wsb, None)

    assert pr(None, p, p, p, p, p, p, p, p, 256, None) == 1
    assert call(desc=(-1, 300, 128, 3, 64, 64)) == 1
    assert call(desc=(2, 300, 0, 3, 64, 64)) == 1
    assert call(desc=(2, 300, 100, 3, 64, 64)) == 2          # D not a multiple of 64
    assert call(desc=(2, 300, 128, 3, 32, 64)) == 2          # d not a multiple of 64
    assert call(desc=(2, 300, 128, 3, 64, 96)) == 2          # dv not a multiple of 64
    assert call(Wq=None) == 1
    assert call(X=None) == 1
    assert call(X=odd) == 1
    assert call(ws=None) == 3
    assert call(wsb=16) == 3
    assert call(desc=(0, 300, 128, 3, 64, 64), X=None) == 0  # B = 0: nothing to do
    assert call(desc=(2, 0, 128, 3, 64, 64), X=None) == 0    # N = 0: nothing to do


def test_forward_multi_sizes_regions_and_rejects_bad_arguments_before_launching(lib):
    import gaussian_mixture_latent_gb300 as gma
    p = 4096                       # never dereferenced: every failing case fails validation first
    calls = (gma.gma_forward_call * 3)()
    descs = (_desc(), _desc(d=64, K=64, dv=64), _desc(N=0))
    for k, (dsc, causal) in enumerate(zip(descs, (0, 1, 0))):
        calls[k].desc = dsc
        calls[k].causal = causal
        calls[k].eps = 1e-6
        for name in ("Qx", "Kx", "V", "mu", "rho", "pi_logits", "out"):
            setattr(calls[k], name, p)
    n, offs = ctypes.c_size_t(0), (ctypes.c_size_t * 3)()
    assert lib.gma_forward_multi_workspace_size(calls, 3, ctypes.byref(n), offs) == 0
    # one 256-byte aligned region per call, in order, each of the call's own workspace size
    sizes = []
    for k in range(3):
        b = ctypes.c_size_t(0)
        assert lib.gma_workspace_size(ctypes.byref(descs[k]), calls[k].causal, ctypes.byref(b)) == 0
        sizes.append((b.value + 255) // 256 * 256)
    assert list(offs) == [0, sizes[0], sizes[0] + sizes[1]] and n.value == sum(sizes)
    assert lib.gma_forward_multi_workspace_size(calls, 3, ctypes.byref(n), None) == 0
    assert lib.gma_forward_multi_workspace_size(calls, 3, None, None) == 1
    assert lib.gma_forward_multi_workspace_size(None, 2, ctypes.byref(n), None) == 1
    assert lib.gma_forward_multi_workspace_size(calls, -1, ctypes.byref(n), None) == 1
    total = n.value
    f = lib.gma_forward_multi
    assert f(calls, 0, None, 0, None, None) == 0            # nothing to do
    assert f(calls, 3, p, total - 1, None, None) == 3       # workspace too small
    assert f(calls, 3, None, total, None, None) == 3
    calls[1].causal = 2
    assert f(calls, 3, p, total, None, None) == 1
    calls[1].causal = 1
    calls[0].Qx = None
    assert f(calls, 3, p, total, None, None) == 1
    calls[0].Qx = 4100                                       # not 16-byte aligned
    assert f(calls, 3, p, total, None, None) == 1
    calls[0].Qx = p
    calls[2].n_events = 2                                    # events missing
    assert f(calls, 3, p, total, None, None) == 1
    calls[2].n_events = 0
    calls[0].eps = -1.0
    assert f(calls, 3, p, total, None, None) == 1
    calls[0].eps = 1e-6
    calls[1].desc = _desc(K=0)
    assert f(calls, 3, p, total, None, None) == 1
