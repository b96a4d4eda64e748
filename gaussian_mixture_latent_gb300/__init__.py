"""GB300 (sm_103a) Gaussian Mixture Attention forward -- Python binding.

A thin ``ctypes`` layer over the C ABI in ``include/gma.h`` (library
``libgma.so`` next to this file).  Functions carry the C names; they only
check and marshal torch tensors (device pointers, sizes, the current CUDA
stream).  Every step of the computation runs in the library's CUDA kernels:
there is no Python or CPU implementation behind these calls, and they raise
if the library has not been built.

Method: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
Probabilistic Latent Routing" (Huang & Raza, 2026), sections 3.2-3.6.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "GmaError", "gma_desc", "gma_workspace_size", "gma_workspace_init", "gma_forward",
    "gma_forward_ex", "gma_forward_plan", "gma_forward_call", "gma_forward_multi",
    "gma_responsibilities", "gma_diagnostics", "gma_forward_cross", "gma_decode", "gma_backward",
    "gma_proj_desc", "gma_project", "gma_selftest_timeout", "gma_get_status", "gma_status_string", "gma_version",
    "Workspace", "library_path",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
# GMA_LIBRARY selects another build of the library, such as the index-checking debug
# build (libgma_debug.so, _build.build(debug=True)).
_LIB_PATH = os.environ.get("GMA_LIBRARY") or os.path.join(_PKG, "libgma.so")
_lib = None

GMA_F32, GMA_BF16 = 0, 1
_DTYPES = {torch.float32: GMA_F32, torch.bfloat16: GMA_BF16}
_STATUS = {0: "GMA_OK", 1: "GMA_ERR_INVALID_ARG", 2: "GMA_ERR_UNSUPPORTED",
           3: "GMA_ERR_WORKSPACE", 4: "GMA_ERR_CUDA", 5: "GMA_ERR_TIMEOUT", 6: "GMA_ERR_BOUNDS"}


class GmaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {gma_status_string(code)}")
        self.code = code


class gma_desc(ctypes.Structure):
    """Mirror of ``gma_desc`` in include/gma.h."""
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("d", ctypes.c_int), ("K", ctypes.c_int), ("dv", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("var_floor", ctypes.c_float), ("chunk", ctypes.c_int)]


class gma_forward_call(ctypes.Structure):
    """Mirror of ``gma_forward_call`` in include/gma.h."""
    _fields_ = [("desc", gma_desc), ("causal", ctypes.c_int), ("eps", ctypes.c_float),
                ("Qx", ctypes.c_void_p), ("Kx", ctypes.c_void_p), ("V", ctypes.c_void_p),
                ("mu", ctypes.c_void_p), ("rho", ctypes.c_void_p), ("pi_logits", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("events", ctypes.POINTER(ctypes.c_void_p)), ("n_events", ctypes.c_int)]


class gma_proj_desc(ctypes.Structure):
    """Mirror of ``gma_proj_desc`` in include/gma.h."""
    _fields_ = [("B", ctypes.c_int), ("N", ctypes.c_int), ("D", ctypes.c_int), ("H", ctypes.c_int),
                ("d", ctypes.c_int), ("dv", ctypes.c_int)]


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            "libgma.so is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(the GMA forward has no fallback implementation)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, sz, i, f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    dp = ctypes.POINTER(gma_desc)
    lib.gma_workspace_size.argtypes = [dp, i, ctypes.POINTER(sz)]
    lib.gma_workspace_init.argtypes = [vp, sz, vp]
    lib.gma_forward.argtypes = [dp, vp, vp, vp, vp, vp, vp, f, i, vp, vp, sz, vp]
    lib.gma_forward_ex.argtypes = [dp, vp, vp, vp, vp, vp, vp, f, i, vp, vp, sz, vp,
                                   ctypes.POINTER(vp), i]
    lib.gma_forward_plan.argtypes = [dp, i, ctypes.POINTER(i), ctypes.POINTER(ctypes.c_char_p), i]
    lib.gma_responsibilities.argtypes = [dp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gma_diagnostics_workspace_size.argtypes = [dp, ctypes.POINTER(sz)]
    lib.gma_diagnostics.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gma_cross_workspace_size.argtypes = [dp, i, ctypes.POINTER(sz)]
    lib.gma_forward_cross.argtypes = [dp, i, vp, vp, vp, vp, vp, vp, f, vp, vp, sz, vp]
    lib.gma_decode_workspace_size.argtypes = [dp, ctypes.POINTER(sz)]
    lib.gma_decode.argtypes = [dp, vp, vp, vp, vp, vp, vp, f, vp, vp, vp, sz, vp]
    lib.gma_backward_workspace_size.argtypes = [dp, i, ctypes.POINTER(sz)]
    lib.gma_selftest_timeout.argtypes = [vp, sz, vp]
    lib.gma_backward.argtypes = [dp, i, vp, vp, vp, vp, vp, vp, f, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.gma_project.argtypes = [ctypes.POINTER(gma_proj_desc), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    cp = ctypes.POINTER(gma_forward_call)
    lib.gma_forward_multi_workspace_size.argtypes = [cp, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.gma_forward_multi.argtypes = [cp, i, vp, sz, vp, vp]
    lib.gma_get_status.argtypes = [vp, vp]
    lib.gma_status_string.argtypes = [i]
    lib.gma_status_string.restype = ctypes.c_char_p
    lib.gma_version.argtypes = []
    for fn in (lib.gma_workspace_size, lib.gma_workspace_init, lib.gma_forward,
               lib.gma_forward_ex, lib.gma_forward_plan, lib.gma_responsibilities, lib.gma_get_status, lib.gma_version,
               lib.gma_diagnostics_workspace_size, lib.gma_diagnostics, lib.gma_cross_workspace_size,
               lib.gma_forward_cross, lib.gma_decode_workspace_size, lib.gma_decode,
               lib.gma_backward_workspace_size, lib.gma_backward, lib.gma_selftest_timeout, lib.gma_project,
               lib.gma_forward_multi_workspace_size, lib.gma_forward_multi):
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


def gma_status_string(code: int) -> str:
    try:
        return _load().gma_status_string(int(code)).decode()
    except RuntimeError:
        return _STATUS.get(int(code), "unknown gma_status")


def gma_version() -> int:
    return _load().gma_version()


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _make_desc(B, H, N, d, K, dv, in_dtype, out_dtype, var_floor, chunk) -> gma_desc:
    return gma_desc(B, H, N, d, K, dv, _DTYPES[in_dtype], _DTYPES[out_dtype], float(var_floor),
                    int(chunk))


def gma_workspace_size(desc: gma_desc, causal: bool) -> int:
    n = ctypes.c_size_t(0)
    rc = _load().gma_workspace_size(ctypes.byref(desc), int(bool(causal)), ctypes.byref(n))
    if rc:
        raise GmaError(rc, "gma_workspace_size")
    return n.value


def gma_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    rc = _load().gma_workspace_init(_ptr(workspace), workspace.numel(), _stream_ptr(stream))
    if rc:
        raise GmaError(rc, "gma_workspace_init")


class Workspace:
    """A device workspace buffer that grows on demand (bytes, uint8)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int, stream=None) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            gma_workspace_init(self.buf, stream)
        return self.buf


_default_ws: dict = {}


def _workspace_for(device, nbytes, workspace, stream):
    if workspace is not None:
        if workspace.numel() < nbytes:
            raise GmaError(3, "gma_forward")
        return workspace
    key = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    ws = _default_ws.setdefault(key, Workspace(torch.device("cuda", key)))
    return ws.get(nbytes, stream)


def _check(t: torch.Tensor, name: str, shape, dtypes):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check_device_status(ws, stream, what: str) -> None:
    """Synchronise `stream` and raise GmaError when a kernel of the call posted a
    device error (a bounded wait that ran out) to the workspace's status word."""
    rc = _load().gma_get_status(_ptr(ws), _stream_ptr(stream))
    if rc:
        raise GmaError(rc, what)


def gma_forward_plan(B, H, N, d, K, dv, dtype=torch.bfloat16, causal=False, out_dtype=None,
                     var_floor: float = 1e-4, chunk: int = 0):
    """Kernel names gma_forward launches for this problem (nothing runs)."""
    desc = _make_desc(B, H, N, d, K, dv, dtype, out_dtype or dtype, var_floor, chunk)
    n = ctypes.c_int(0)
    names = (ctypes.c_char_p * 16)()
    rc = _load().gma_forward_plan(ctypes.byref(desc), int(bool(causal)), ctypes.byref(n), names, 16)
    if rc:
        raise GmaError(rc, "gma_forward_plan")
    return [names[i].decode() for i in range(min(n.value, 16))]


def gma_forward_ex(*args, events=None, **kw):
    """gma_forward with torch.cuda.Event objects recorded around each kernel launch
    (events[2i] before launch i, events[2i+1] after it)."""
    return gma_forward(*args, events=events, **kw)


def gma_forward(Qx, Kx, V, mu, rho, pi_logits, eps: float = 1e-6, causal: bool = False,
                out=None, workspace=None, var_floor: float = 1e-4, out_dtype=None,
                chunk: int = 0, stream=None, events=None, check_status: bool = False):
    """GMA forward (Eq. 5-8; causal Eq. 6b, 8b).  Qx, Kx [B,H,N,d], V [B,H,N,dv]
    (float32 or bfloat16), mu, rho [H,K,d], pi_logits [H,K] float32 -> out [B,H,N,dv].

    The call is asynchronous.  Device-side errors are posted to the workspace's
    status word, not returned: pass check_status=True to synchronise and raise
    GmaError on one, or call gma_get_status() later."""
    B, H, N, d = Qx.shape
    dv = V.shape[-1]
    K = mu.shape[1]
    in_dtype = Qx.dtype
    out_dtype = out_dtype or in_dtype
    _check(Qx, "Qx", (B, H, N, d), (torch.float32, torch.bfloat16))
    _check(Kx, "Kx", (B, H, N, d), (in_dtype,))
    _check(V, "V", (B, H, N, dv), (in_dtype,))
    _check(mu, "mu", (H, K, d), (torch.float32,))
    _check(rho, "rho", (H, K, d), (torch.float32,))
    _check(pi_logits, "pi_logits", (H, K), (torch.float32,))
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=out_dtype, device=Qx.device)
    _check(out, "out", (B, H, N, dv), (out_dtype,))
    desc = _make_desc(B, H, N, d, K, dv, in_dtype, out_dtype, var_floor, chunk)
    nbytes = gma_workspace_size(desc, causal)
    ws = _workspace_for(Qx.device, nbytes, workspace, stream)
    common = (ctypes.byref(desc), _ptr(Qx), _ptr(Kx), _ptr(V), _ptr(mu), _ptr(rho),
              _ptr(pi_logits), float(eps), int(bool(causal)), _ptr(out), _ptr(ws), ws.numel(),
              _stream_ptr(stream))
    if events is None:
        rc = _load().gma_forward(*common)
    else:
        handles = (ctypes.c_void_p * len(events))(*[e.cuda_event if e is not None else None
                                                    for e in events])
        rc = _load().gma_forward_ex(*common, handles, len(events))
    if rc:
        raise GmaError(rc, "gma_forward")
    if check_status:
        _check_device_status(ws, stream, "gma_forward")
    return out


_multi_ws: dict = {}


def gma_forward_multi(calls, workspace=None, stream=None, aux_stream=None, check_status: bool = False):
    """Several independent forwards in one request (include/gma.h, gma_forward_multi).

    calls: a list of dicts with gma_forward()'s tensor arguments Qx, Kx, V, mu, rho,
    pi_logits and optional eps (1e-6), causal (False), out, var_floor (1e-4), out_dtype,
    chunk (0), events.  With aux_stream (a torch.cuda.Stream) the library may run the
    calls that it schedules as one CTA per head on aux_stream beside the others.
    Returns the list of outputs.  workspace: None (a zeroed buffer of this module's
    cache) or a uint8 tensor of gma_forward_multi_workspace_size() bytes whose regions'
    first 256 bytes are zero.  check_status=True synchronises and raises GmaError when
    a kernel of any call posted a device error."""
    n = len(calls)
    arr = (gma_forward_call * max(n, 1))()
    outs, keep = [], []
    for k, c in enumerate(calls):
        Qx, Kx, V, mu, rho, pi = (c[name] for name in ("Qx", "Kx", "V", "mu", "rho", "pi_logits"))
        B, H, N, d = Qx.shape
        dv, K = V.shape[-1], mu.shape[1]
        out_dtype = c.get("out_dtype") or Qx.dtype
        _check(Qx, "Qx", (B, H, N, d), (torch.float32, torch.bfloat16))
        _check(Kx, "Kx", (B, H, N, d), (Qx.dtype,))
        _check(V, "V", (B, H, N, dv), (Qx.dtype,))
        _check(mu, "mu", (H, K, d), (torch.float32,))
        _check(rho, "rho", (H, K, d), (torch.float32,))
        _check(pi, "pi_logits", (H, K), (torch.float32,))
        out = c.get("out")
        if out is None:
            out = torch.empty((B, H, N, dv), dtype=out_dtype, device=Qx.device)
        _check(out, "out", (B, H, N, dv), (out_dtype,))
        outs.append(out)
        arr[k].desc = _make_desc(B, H, N, d, K, dv, Qx.dtype, out_dtype, c.get("var_floor", 1e-4), c.get("chunk", 0))
        arr[k].causal = int(bool(c.get("causal", False)))
        arr[k].eps = float(c.get("eps", 1e-6))
        for name, t in (("Qx", Qx), ("Kx", Kx), ("V", V), ("mu", mu), ("rho", rho), ("pi_logits", pi),
                        ("out", out)):
            setattr(arr[k], name, _ptr(t))
        evs = c.get("events")
        if evs is not None:
            h = (ctypes.c_void_p * len(evs))(*[e.cuda_event if e is not None else None for e in evs])
            keep.append(h)
            arr[k].events = ctypes.cast(h, ctypes.POINTER(ctypes.c_void_p))
            arr[k].n_events = len(evs)
    lib = _load()
    nbytes, offs = ctypes.c_size_t(0), (ctypes.c_size_t * max(n, 1))()
    rc = lib.gma_forward_multi_workspace_size(arr, n, ctypes.byref(nbytes), offs)
    if rc:
        raise GmaError(rc, "gma_forward_multi_workspace_size")
    if workspace is None:
        # the cached buffer's regions move with the request's calls: when the layout differs
        # from the buffer's last request, this request's region headers are zeroed first
        dev = calls[0]["Qx"].device if n else torch.device("cuda")
        key = dev.index if dev.index is not None else torch.cuda.current_device()
        ws, last = _multi_ws.get(key, (None, None))
        if ws is None or ws.numel() < nbytes.value:
            ws, last = torch.zeros(max(nbytes.value, 256), dtype=torch.uint8, device=torch.device("cuda", key)), None
        layout = tuple(offs[k] for k in range(n))
        if last is not None and last != layout:
            for o in layout:
                rc = lib.gma_workspace_init(_ptr(ws) + o, ws.numel() - o, _stream_ptr(stream))
                if rc:
                    raise GmaError(rc, "gma_workspace_init")
        _multi_ws[key] = (ws, layout)
    else:
        ws = workspace
        if ws.numel() < nbytes.value:
            raise GmaError(3, "gma_forward_multi")
    aux = None if aux_stream is None else int(aux_stream.cuda_stream)
    rc = lib.gma_forward_multi(arr, n, _ptr(ws), ws.numel(), _stream_ptr(stream), aux)
    if rc:
        raise GmaError(rc, "gma_forward_multi")
    if check_status:
        for k in range(n):
            st = lib.gma_get_status(_ptr(ws) + offs[k], _stream_ptr(stream))
            if st:
                raise GmaError(st, f"gma_forward_multi (call {k})")
    return outs


def gma_responsibilities(X, mu, rho, pi_logits, var_floor: float = 1e-4, out=None,
                         workspace=None, stream=None):
    """Responsibilities (Eq. 3) of the rows of X [B,H,N,d] -> float32 [B,H,N,K]."""
    B, H, N, d = X.shape
    K = mu.shape[1]
    _check(X, "X", (B, H, N, d), (torch.float32, torch.bfloat16))
    _check(mu, "mu", (H, K, d), (torch.float32,))
    _check(rho, "rho", (H, K, d), (torch.float32,))
    _check(pi_logits, "pi_logits", (H, K), (torch.float32,))
    if out is None:
        out = torch.empty((B, H, N, K), dtype=torch.float32, device=X.device)
    _check(out, "out", (B, H, N, K), (torch.float32,))
    desc = _make_desc(B, H, N, d, K, 1, X.dtype, X.dtype, var_floor, 0)
    nbytes = gma_workspace_size(desc, False)
    ws = _workspace_for(X.device, nbytes, workspace, stream)
    rc = _load().gma_responsibilities(ctypes.byref(desc), _ptr(X), _ptr(mu), _ptr(rho),
                                      _ptr(pi_logits), _ptr(out), _ptr(ws), ws.numel(),
                                      _stream_ptr(stream))
    if rc:
        raise GmaError(rc, "gma_responsibilities")
    return out


def gma_forward_cross(Qx, Ky, Vy, mu, rho, pi_logits, eps: float = 1e-6, var_floor: float = 1e-4, out=None,
                      workspace=None, stream=None, check_status: bool = False):
    """Cross-attention GMA (sections 3.1, 6): the queries Qx [B,H,N,d] read the memory of the
    context Ky [B,H,Nkv,d], Vy [B,H,Nkv,dv] -> out [B,H,N,dv] (bidirectional, Eq. 5-8)."""
    B, H, N, d = Qx.shape
    Nkv = Ky.shape[2]
    dv = Vy.shape[3]
    K = mu.shape[1]
    _check(Qx, "Qx", (B, H, N, d), (torch.float32, torch.bfloat16))
    _check(Ky, "Ky", (B, H, Nkv, d), (Qx.dtype,))
    _check(Vy, "Vy", (B, H, Nkv, dv), (Qx.dtype,))
    _check(mu, "mu", (H, K, d), (torch.float32,))
    _check(rho, "rho", (H, K, d), (torch.float32,))
    _check(pi_logits, "pi_logits", (H, K), (torch.float32,))
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=Qx.dtype, device=Qx.device)
    _check(out, "out", (B, H, N, dv), (Qx.dtype,))
    desc = _make_desc(B, H, N, d, K, dv, Qx.dtype, out.dtype, var_floor, 0)
    nbytes = ctypes.c_size_t(0)
    rc = _load().gma_cross_workspace_size(ctypes.byref(desc), Nkv, ctypes.byref(nbytes))
    if rc:
        raise GmaError(rc, "gma_cross_workspace_size")
    ws = _workspace_for(Qx.device, nbytes.value, workspace, stream)
    rc = _load().gma_forward_cross(ctypes.byref(desc), Nkv, _ptr(Qx), _ptr(Ky), _ptr(Vy), _ptr(mu), _ptr(rho),
                                   _ptr(pi_logits), float(eps), _ptr(out), _ptr(ws), ws.numel(),
                                   _stream_ptr(stream))
    if rc:
        raise GmaError(rc, "gma_forward_cross")
    if check_status:
        _check_device_status(ws, stream, "gma_forward_cross")
    return out


def gma_backward(Qx, Kx, V, mu, rho, pi_logits, dO, eps: float = 1e-6, var_floor: float = 1e-4, causal=False,
                 grads=None, workspace=None, stream=None, check_status: bool = False, chunk: int = 0):
    """Backward pass (section 4.1, Eqs. 17-20): given dO = dL/dO [B,H,N,dv] of the forward
    gma_forward(Qx, Kx, V, mu, rho, pi_logits), returns the float32 gradients
    (dQx, dKx, dV, dmu, drho, dpi_logits); parameter gradients are summed over the batch.
    `grads`, if given, is that tuple of preallocated outputs (overwritten)."""
    B, H, N, d = Qx.shape
    dv = V.shape[3]
    K = mu.shape[1]
    _check(Qx, "Qx", (B, H, N, d), (torch.float32, torch.bfloat16))
    _check(Kx, "Kx", (B, H, N, d), (Qx.dtype,))
    _check(V, "V", (B, H, N, dv), (Qx.dtype,))
    _check(dO, "dO", (B, H, N, dv), (Qx.dtype,))
    _check(mu, "mu", (H, K, d), (torch.float32,))
    _check(rho, "rho", (H, K, d), (torch.float32,))
    _check(pi_logits, "pi_logits", (H, K), (torch.float32,))
    if grads is None:
        f32 = dict(dtype=torch.float32, device=Qx.device)
        grads = (torch.empty((B, H, N, d), **f32), torch.empty((B, H, N, d), **f32),
                 torch.empty((B, H, N, dv), **f32), torch.empty((H, K, d), **f32),
                 torch.empty((H, K, d), **f32), torch.empty((H, K), **f32))
    shapes = ((B, H, N, d), (B, H, N, d), (B, H, N, dv), (H, K, d), (H, K, d), (H, K))
    for t, shp, name in zip(grads, shapes, ("dQx", "dKx", "dV", "dmu", "drho", "dpi_logits")):
        _check(t, name, shp, (torch.float32,))
    desc = _make_desc(B, H, N, d, K, dv, Qx.dtype, Qx.dtype, var_floor, chunk)
    nbytes = ctypes.c_size_t(0)
    rc = _load().gma_backward_workspace_size(ctypes.byref(desc), int(bool(causal)), ctypes.byref(nbytes))
    if rc:
        raise GmaError(rc, "gma_backward_workspace_size")
    ws = _workspace_for(Qx.device, nbytes.value, workspace, stream)
    rc = _load().gma_backward(ctypes.byref(desc), int(bool(causal)), _ptr(Qx), _ptr(Kx), _ptr(V), _ptr(mu),
                              _ptr(rho), _ptr(pi_logits), float(eps), _ptr(dO), *(_ptr(t) for t in grads),
                              _ptr(ws), ws.numel(), _stream_ptr(stream))
    if rc:
        raise GmaError(rc, "gma_backward")
    if check_status:
        _check_device_status(ws, stream, "gma_backward")
    return grads


def gma_project(X, Wq, Wk, Wv, out=None, workspace=None, stream=None, check_status: bool = False):
    """Input projections (section 3.1, Eq. 4): X [B, N, D], Wq and Wk [H, D, d], Wv [H, D, dv],
    all bfloat16 -> (Qx, Kx [B, H, N, d], V [B, H, N, dv]) bfloat16, Qx[b, h] = X[b] Wq[h] with
    fp32 accumulation (one tensor-core GEMM).  `out`, if given, is that tuple of preallocated
    outputs (overwritten)."""
    B, N, D = X.shape
    H, _, d = Wq.shape
    dv = Wv.shape[2]
    bf = (torch.bfloat16,)
    _check(X, "X", (B, N, D), bf)
    _check(Wq, "Wq", (H, D, d), bf)
    _check(Wk, "Wk", (H, D, d), bf)
    _check(Wv, "Wv", (H, D, dv), bf)
    if out is None:
        out = (torch.empty((B, H, N, d), dtype=torch.bfloat16, device=X.device),
               torch.empty((B, H, N, d), dtype=torch.bfloat16, device=X.device),
               torch.empty((B, H, N, dv), dtype=torch.bfloat16, device=X.device))
    for t, shp, name in zip(out, ((B, H, N, d), (B, H, N, d), (B, H, N, dv)), ("Qx", "Kx", "V")):
        _check(t, name, shp, bf)
    desc = gma_proj_desc(B, N, D, H, d, dv)
    ws = _workspace_for(X.device, 256, workspace, stream)
    rc = _load().gma_project(ctypes.byref(desc), _ptr(X), _ptr(Wq), _ptr(Wk), _ptr(Wv), *(_ptr(t) for t in out),
                             _ptr(ws), ws.numel(), _stream_ptr(stream))
    if rc:
        raise GmaError(rc, "gma_project")
    if check_status:
        _check_device_status(ws, stream, "gma_project")
    return out


def gma_decode(Qx, Kx, V, mu, rho, pi_logits, state, eps: float = 1e-6, var_floor: float = 1e-4, out=None,
               workspace=None, stream=None, check_status: bool = False):
    """Causal decode with a carried state (section 3.5, Eq. 6b / 8b as a recurrence): appends the
    N new positions of Qx, Kx [B,H,N,d], V [B,H,N,dv] to each head's sequence.  `state`
    [B,H,K,dv+1] float32 holds [S | z] of the positions so far and is updated in place;
    returns out [B,H,N,dv]."""
    B, H, N, d = Qx.shape
    dv = V.shape[3]
    K = mu.shape[1]
    _check(Qx, "Qx", (B, H, N, d), (torch.float32, torch.bfloat16))
    _check(Kx, "Kx", (B, H, N, d), (Qx.dtype,))
    _check(V, "V", (B, H, N, dv), (Qx.dtype,))
    _check(mu, "mu", (H, K, d), (torch.float32,))
    _check(rho, "rho", (H, K, d), (torch.float32,))
    _check(pi_logits, "pi_logits", (H, K), (torch.float32,))
    _check(state, "state", (B, H, K, dv + 1), (torch.float32,))
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=Qx.dtype, device=Qx.device)
    _check(out, "out", (B, H, N, dv), (torch.float32, torch.bfloat16))
    desc = _make_desc(B, H, N, d, K, dv, Qx.dtype, out.dtype, var_floor, 0)
    nbytes = ctypes.c_size_t(0)
    rc = _load().gma_decode_workspace_size(ctypes.byref(desc), ctypes.byref(nbytes))
    if rc:
        raise GmaError(rc, "gma_decode_workspace_size")
    ws = _workspace_for(Qx.device, nbytes.value, workspace, stream)
    rc = _load().gma_decode(ctypes.byref(desc), _ptr(Qx), _ptr(Kx), _ptr(V), _ptr(mu), _ptr(rho), _ptr(pi_logits),
                            float(eps), _ptr(state), _ptr(out), _ptr(ws), ws.numel(), _stream_ptr(stream))
    if rc:
        raise GmaError(rc, "gma_decode")
    if check_status:
        _check_device_status(ws, stream, "gma_decode")
    return out


_diag_ws_bytes = {}


def gma_diagnostics(Qx, mu, rho, pi_logits, var_floor: float = 1e-4, z=True, workspace=None, stream=None,
                    check_status: bool = False):
    """Responsibility diagnostics (section 5.4, Eqs. 24-29) of the query routing vectors
    Qx [B,H,N,d] (bf16, d = 64, K in {64, 128}) -> (p [K] float32, stats [3] float32 =
    (H_usage, H_token, R_max), z [B,N] int32 argmax or None), all on Qx's device."""
    B, H, N, d = Qx.shape
    K = mu.shape[1]
    _check(Qx, "Qx", (B, H, N, d), (torch.bfloat16, torch.float32))
    _check(mu, "mu", (H, K, d), (torch.float32,))
    _check(rho, "rho", (H, K, d), (torch.float32,))
    _check(pi_logits, "pi_logits", (H, K), (torch.float32,))
    p = torch.empty((K,), dtype=torch.float32, device=Qx.device)
    stats = torch.empty((3,), dtype=torch.float32, device=Qx.device)
    zt = torch.empty((B, N), dtype=torch.int32, device=Qx.device) if z else None
    desc = _make_desc(B, H, N, d, K, 1, Qx.dtype, Qx.dtype, var_floor, 0)
    key = (B, H, N, d, K, Qx.dtype)
    if key not in _diag_ws_bytes:
        nbytes = ctypes.c_size_t(0)
        rc = _load().gma_diagnostics_workspace_size(ctypes.byref(desc), ctypes.byref(nbytes))
        if rc:
            raise GmaError(rc, "gma_diagnostics_workspace_size")
        _diag_ws_bytes[key] = nbytes.value
    ws = _workspace_for(Qx.device, _diag_ws_bytes[key], workspace, stream)
    rc = _load().gma_diagnostics(ctypes.byref(desc), _ptr(Qx), _ptr(mu), _ptr(rho), _ptr(pi_logits),
                                 _ptr(p), _ptr(stats), _ptr(zt) if zt is not None else None, _ptr(ws),
                                 ws.numel(), _stream_ptr(stream))
    if rc:
        raise GmaError(rc, "gma_diagnostics")
    if check_status:
        _check_device_status(ws, stream, "gma_diagnostics")
    return p, stats, zt


def gma_selftest_timeout(workspace, stream=None):
    """Launch a kernel whose bounded wait runs out (about one second): afterwards
    gma_get_status(workspace) returns GMA_ERR_TIMEOUT (5).  `workspace` is a CUDA tensor
    of at least 256 bytes."""
    rc = _load().gma_selftest_timeout(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream_ptr(stream))
    if rc:
        raise GmaError(rc, "gma_selftest_timeout")


def gma_get_status(workspace=None, stream=None) -> int:
    """Synchronise, read and clear the device status word; returns the gma_status code."""
    if workspace is None:
        key = torch.cuda.current_device()
        if key not in _default_ws or _default_ws[key].buf is None:
            return 0
        workspace = _default_ws[key].buf
    return _load().gma_get_status(_ptr(workspace), _stream_ptr(stream))
