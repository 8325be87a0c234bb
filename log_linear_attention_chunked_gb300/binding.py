"""Thin ctypes binding of libllattn.so (argument marshalling only).

Every function here has the name of the C entry point it calls
(``include/ll_attn.h``), takes torch tensors that already live on the GPU,
passes their ``data_ptr()`` and the current CUDA stream, and raises
``LLError`` on a non-OK status.  All arithmetic happens in the library's
kernels; there is no other code path.  If the library is missing,
``lib()`` raises: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libllattn.so")

LL_F32, LL_BF16 = 0, 1
STATUS = {0: "LL_OK", 1: "LL_ERR_INVALID_ARG", 2: "LL_ERR_UNSUPPORTED", 3: "LL_ERR_CUDA",
          4: "LL_ERR_TIMEOUT", 5: "LL_ERR_WORKSPACE", 6: "LL_ERR_DEVICE"}

# every symbol the header declares
SYMBOLS = ("ll_version", "ll_status_str", "ll_last_device_error", "ll_attn_fwd_workspace_size", "ll_attn_fwd_launches",
           "ll_attn_fwd", "ll_attn_fwd_noalloc", "ll_attn_decode_step", "ll_gdn_fwd_workspace_size", "ll_gdn_fwd",
           "ll_gdn_decode_step", "ll_gdn_fwd_b_workspace_size", "ll_gdn_fwd_b", "ll_attn_fwd_cont_workspace_size",
           "ll_attn_fwd_cont", "ll_attn_bwd_workspace_size", "ll_attn_bwd_launches", "ll_attn_bwd",
           "ll_attn_fwd_level_decay_workspace_size", "ll_attn_fwd_level_decay_launches", "ll_attn_fwd_level_decay",
           "ll_attn_decode_step_level_decay",
           # test hooks (include/ll_attn_test.h)
           "ll_test_fwd_withhold_node")


class LLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class ll_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int), ("dk", ctypes.c_int),
                ("dv", ctypes.c_int), ("L", ctypes.c_int), ("chunk", ctypes.c_int), ("Ls", ctypes.c_int),
                ("io", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libllattn.so (built in-tree by ``build.py``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run log_linear_attention_chunked_gb300.build first")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, fp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
    shp = ctypes.POINTER(ll_shape)
    L.ll_version.restype = i32
    L.ll_version.argtypes = []
    L.ll_status_str.restype = ctypes.c_char_p
    L.ll_status_str.argtypes = [i32]
    L.ll_last_device_error.restype = i32
    L.ll_last_device_error.argtypes = [vp]
    L.ll_attn_fwd_workspace_size.restype = sz
    L.ll_attn_fwd_workspace_size.argtypes = [shp]
    L.ll_attn_fwd_launches.restype = i32
    L.ll_attn_fwd_launches.argtypes = [shp]
    L.ll_attn_fwd.restype = i32
    L.ll_attn_fwd.argtypes = [shp, vp, vp, vp, fp, fp, vp, fp, fp, vp, sz, vp]
    L.ll_attn_fwd_noalloc.restype = i32
    L.ll_attn_fwd_noalloc.argtypes = [shp, vp, vp, vp, fp, fp, vp, fp, fp, vp]
    L.ll_attn_decode_step.restype = i32
    L.ll_attn_decode_step.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, fp, fp, fp, fp, vp, vp]
    L.ll_attn_decode_step_level_decay.restype = i32
    L.ll_attn_decode_step_level_decay.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, fp, fp, fp, fp, vp,
                                                  vp]
    L.ll_attn_fwd_level_decay_workspace_size.restype = sz
    L.ll_attn_fwd_level_decay_workspace_size.argtypes = [shp]
    L.ll_attn_fwd_level_decay_launches.restype = i32
    L.ll_attn_fwd_level_decay_launches.argtypes = [shp]
    L.ll_attn_fwd_level_decay.restype = i32
    L.ll_attn_fwd_level_decay.argtypes = [shp, vp, vp, vp, fp, fp, vp, fp, fp, vp, sz, vp]
    L.ll_gdn_decode_step.restype = i32
    L.ll_gdn_decode_step.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, fp, fp, fp, fp, vp, vp]
    L.ll_gdn_fwd_workspace_size.restype = sz
    L.ll_gdn_fwd_workspace_size.argtypes = [shp]
    L.ll_gdn_fwd.restype = i32
    L.ll_gdn_fwd.argtypes = [shp, vp, vp, vp, fp, fp, fp, vp, vp, sz, vp]
    L.ll_attn_fwd_cont_workspace_size.restype = sz
    L.ll_attn_fwd_cont_workspace_size.argtypes = [shp, ctypes.c_longlong]
    L.ll_attn_fwd_cont.restype = i32
    L.ll_attn_fwd_cont.argtypes = [shp, ctypes.c_longlong, fp, fp, vp, vp, vp, fp, fp, vp, fp, fp, vp, sz, vp]
    L.ll_gdn_fwd_b_workspace_size.restype = sz
    L.ll_gdn_fwd_b_workspace_size.argtypes = [shp]
    L.ll_gdn_fwd_b.restype = i32
    L.ll_gdn_fwd_b.argtypes = [shp, vp, vp, vp, fp, fp, fp, vp, vp, sz, vp]
    L.ll_attn_bwd_workspace_size.restype = sz
    L.ll_attn_bwd_workspace_size.argtypes = [shp]
    L.ll_attn_bwd_launches.restype = i32
    L.ll_attn_bwd_launches.argtypes = [shp]
    L.ll_attn_bwd.restype = i32
    L.ll_attn_bwd.argtypes = [shp, vp, vp, vp, fp, fp, vp, vp, vp, vp, fp, fp, vp, sz, vp]
    L.ll_test_fwd_withhold_node.restype = i32
    L.ll_test_fwd_withhold_node.argtypes = [shp, vp, vp, vp, fp, fp, vp, vp, sz, ctypes.c_longlong,
                                            ctypes.c_ulonglong, vp]
    _lib = L
    return L


def _ptr(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _io(dtype) -> int:
    if dtype == torch.float32:
        return LL_F32
    if dtype == torch.bfloat16:
        return LL_BF16
    raise TypeError(f"unsupported io dtype {dtype}")


def _check(status: int, where: str):
    if status != 0:
        raise LLError(status, where)


def _need(x, name, dtype=None):
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")


def make_shape(B, H, T, dk, dv, L, chunk, Ls=0, io=LL_BF16) -> ll_shape:
    return ll_shape(B, H, T, dk, dv, L, chunk, Ls, io)


def ll_attn_fwd_workspace_size(shape: ll_shape) -> int:
    return int(lib().ll_attn_fwd_workspace_size(ctypes.byref(shape)))


def ll_attn_fwd_launches(shape: ll_shape) -> int:
    return int(lib().ll_attn_fwd_launches(ctypes.byref(shape)))


def ll_gdn_fwd_workspace_size(shape: ll_shape) -> int:
    return int(lib().ll_gdn_fwd_workspace_size(ctypes.byref(shape)))


def ll_gdn_fwd_b_workspace_size(shape: ll_shape) -> int:
    return int(lib().ll_gdn_fwd_b_workspace_size(ctypes.byref(shape)))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """Caller-owned scratch for a forward call (torch device memory)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def ll_attn_fwd(q, k, v, log_alpha, lam, chunk: int, *, o=None, state_out=None, scale_out=None, workspace=None):
    """Log-linear Mamba-2 forward.  q, k [B,H,T,dk]; v [B,H,T,dv] (f32 or bf16);
    log_alpha [B,H,T], lam [B,H,T,L] float32.  Returns o [B,H,T,dv]."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    io = _io(q.dtype)
    for x, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(x, n, q.dtype)
    _need(log_alpha, "log_alpha", torch.float32)
    _need(lam, "lam", torch.float32)
    Ls = 0
    if state_out is not None:
        _need(state_out, "state_out", torch.float32)
        _need(scale_out, "scale_out", torch.float32)
        Ls = state_out.shape[2]
    shape = make_shape(B, H, T, dk, dv, L, chunk, Ls, io)
    if o is None:
        o = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype)
    if workspace is None:
        workspace = alloc_workspace(ll_attn_fwd_workspace_size(shape), q.device)
    st = lib().ll_attn_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(lam), _ptr(o),
                           _ptr(state_out), _ptr(scale_out), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                           _stream(q.device))
    _check(st, "ll_attn_fwd")
    return o


def ll_attn_bwd_workspace_size(shape: ll_shape) -> int:
    return int(lib().ll_attn_bwd_workspace_size(ctypes.byref(shape)))


def ll_attn_bwd_launches(shape: ll_shape) -> int:
    return int(lib().ll_attn_bwd_launches(ctypes.byref(shape)))


def ll_attn_bwd(q, k, v, log_alpha, lam, dout, chunk: int, *, grads=None, workspace=None):
    """Backward of ll_attn_fwd for the upstream gradient dout [B,H,T,dv] (io dtype).
    Returns (dq, dk, dv, dlog_alpha, dlam); ``grads`` may pass those five
    tensors to be written in place."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    io = _io(q.dtype)
    for x, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(x, n, q.dtype)
    _need(log_alpha, "log_alpha", torch.float32)
    _need(lam, "lam", torch.float32)
    shape = make_shape(B, H, T, dk, dv, L, chunk, 0, io)
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(log_alpha),
                 torch.empty_like(lam))
    gq, gk, gv, gla, glam = grads
    for x, ref, n in ((gq, q, "dq"), (gk, k, "dk"), (gv, v, "dv"), (gla, log_alpha, "dlog_alpha"),
                      (glam, lam, "dlam")):
        _need(x, n, ref.dtype)
        if x.shape != ref.shape:
            raise ValueError(f"{n} must have shape {tuple(ref.shape)}")
    if workspace is None:
        workspace = alloc_workspace(ll_attn_bwd_workspace_size(shape), q.device)
    st = lib().ll_attn_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(lam), _ptr(dout),
                           _ptr(gq), _ptr(gk), _ptr(gv), _ptr(gla), _ptr(glam), _ptr(workspace),
                           ctypes.c_size_t(workspace.numel()), _stream(q.device))
    _check(st, "ll_attn_bwd")
    return gq, gk, gv, gla, glam


NOALLOC_SCRATCH_BYTES = 32 << 20  # LL_NOALLOC_SCRATCH_BYTES of the header


def ll_attn_fwd_noalloc(q, k, v, log_alpha, lam, chunk: int, *, o, state_out=None, scale_out=None):
    """ll_attn_fwd for callers that cannot allocate device memory: the library
    uses its own fixed scratch array (NOALLOC_SCRATCH_BYTES per device) instead
    of a workspace.  The caller passes every input and the output ``o``; this
    wrapper allocates nothing either.  Overlapping calls on one device race."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    io = _io(q.dtype)
    for x, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(x, n, q.dtype)
    _need(log_alpha, "log_alpha", torch.float32)
    _need(lam, "lam", torch.float32)
    Ls = 0
    if state_out is not None:
        _need(state_out, "state_out", torch.float32)
        _need(scale_out, "scale_out", torch.float32)
        Ls = state_out.shape[2]
    shape = make_shape(B, H, T, dk, dv, L, chunk, Ls, io)
    st = lib().ll_attn_fwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(lam),
                                   _ptr(o), _ptr(state_out), _ptr(scale_out), _stream(q.device))
    _check(st, "ll_attn_fwd_noalloc")
    return o


def ll_attn_decode_step(t, q, k, v, log_alpha, lam, states, scales, *, o=None):
    """One decode step.  t [B] int64; q, k [B,H,dk]; v [B,H,dv]; log_alpha [B,H];
    lam [B,H,Ls+1]; states [B,H,Ls,dv,dk] and scales [B,H,Ls] are updated in
    place.  Returns o [B,H,dv]."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    Ls = states.shape[2]
    io = _io(q.dtype)
    _need(t, "t", torch.int64)
    for x, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(x, n, q.dtype)
    _need(log_alpha, "log_alpha", torch.float32)
    _need(lam, "lam", torch.float32)
    _need(states, "states", torch.float32)
    _need(scales, "scales", torch.float32)
    if o is None:
        o = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    st = lib().ll_attn_decode_step(B, H, dk, dv, Ls, io, _ptr(t), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                   _ptr(lam), _ptr(states), _ptr(scales), _ptr(o), _stream(q.device))
    _check(st, "ll_attn_decode_step")
    return o


def ll_attn_fwd_level_decay_workspace_size(shape: ll_shape) -> int:
    return int(lib().ll_attn_fwd_level_decay_workspace_size(ctypes.byref(shape)))


def ll_attn_fwd_level_decay_launches(shape: ll_shape) -> int:
    return int(lib().ll_attn_fwd_level_decay_launches(ctypes.byref(shape)))


def ll_attn_fwd_level_decay(q, k, v, log_alpha, lam, chunk: int, *, o=None, state_out=None, scale_out=None,
                            workspace=None):
    """Forward with one decay per level.  As ll_attn_fwd, except log_alpha
    [B,H,T,L] float32 (column l is level l's log decay; column 0 unused)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    io = _io(q.dtype)
    for x, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(x, n, q.dtype)
    _need(log_alpha, "log_alpha", torch.float32)
    _need(lam, "lam", torch.float32)
    if tuple(log_alpha.shape) != tuple(lam.shape):
        raise ValueError("log_alpha must have the shape of lam, [B,H,T,L]")
    Ls = 0
    if state_out is not None:
        _need(state_out, "state_out", torch.float32)
        _need(scale_out, "scale_out", torch.float32)
        Ls = state_out.shape[2]
    shape = make_shape(B, H, T, dk, dv, L, chunk, Ls, io)
    if o is None:
        o = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype)
    if workspace is None:
        workspace = alloc_workspace(ll_attn_fwd_level_decay_workspace_size(shape), q.device)
    st = lib().ll_attn_fwd_level_decay(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(lam),
                                       _ptr(o), _ptr(state_out), _ptr(scale_out), _ptr(workspace),
                                       ctypes.c_size_t(workspace.numel()), _stream(q.device))
    _check(st, "ll_attn_fwd_level_decay")
    return o


def ll_attn_decode_step_level_decay(t, q, k, v, log_alpha, lam, states, scales, *, o=None):
    """One decode step with one decay per level: as ll_attn_decode_step, except
    log_alpha [B,H,Ls+1] (entry l for level l; entry 0 unused)."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    Ls = states.shape[2]
    io = _io(q.dtype)
    _need(t, "t", torch.int64)
    for x, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(x, n, q.dtype)
    _need(log_alpha, "log_alpha", torch.float32)
    _need(lam, "lam", torch.float32)
    _need(states, "states", torch.float32)
    _need(scales, "scales", torch.float32)
    if tuple(log_alpha.shape) != (B, H, Ls + 1):
        raise ValueError("log_alpha must be [B,H,Ls+1]")
    if o is None:
        o = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    st = lib().ll_attn_decode_step_level_decay(B, H, dk, dv, Ls, io, _ptr(t), _ptr(q), _ptr(k), _ptr(v),
                                               _ptr(log_alpha), _ptr(lam), _ptr(states), _ptr(scales), _ptr(o),
                                               _stream(q.device))
    _check(st, "ll_attn_decode_step_level_decay")
    return o


def ll_attn_fwd_cont_workspace_size(shape: ll_shape, t0: int) -> int:
    return int(lib().ll_attn_fwd_cont_workspace_size(ctypes.byref(shape), int(t0)))


def ll_attn_fwd_cont(t0: int, state_in, scale_in, q, k, v, log_alpha, lam, chunk: int, *, o=None, state_out=None,
                     scale_out=None, workspace=None):
    """Prefill continuation at position t0 (any t0 >= 0; a start that is not a
    multiple of the smallest power of two >= T runs as aligned pieces).
    state_in [B,H,Ls,dv,dk] / scale_in [B,H,Ls]: the decode states
    of position t0; q, k, v, log_alpha, lam: the T new tokens; optional
    state_out / scale_out receive the states of position t0 + T.  Returns o."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    Ls = state_in.shape[2]
    io = _io(q.dtype)
    for x, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(x, n, q.dtype)
    for x, n in ((log_alpha, "log_alpha"), (lam, "lam"), (state_in, "state_in"), (scale_in, "scale_in")):
        _need(x, n, torch.float32)
    shape = make_shape(B, H, T, dk, dv, L, chunk, Ls, io)
    if o is None:
        o = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(ll_attn_fwd_cont_workspace_size(shape, t0), q.device)
    st = lib().ll_attn_fwd_cont(ctypes.byref(shape), int(t0), _ptr(state_in), _ptr(scale_in), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(log_alpha), _ptr(lam), _ptr(o), _ptr(state_out), _ptr(scale_out),
                                _ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream(q.device))
    _check(st, "ll_attn_fwd_cont")
    return o


def ll_gdn_decode_step(t, q, k, v, log_alpha, beta, lam, states, *, o=None):
    """One Gated DeltaNet (reading A) decode step.  t [B] int64; q, k [B,H,dk];
    v [B,H,dv]; log_alpha, beta [B,H]; lam [B,H,Ls+1]; states [B,H,Ls,dv,dk]
    (true states) are updated in place.  Returns o [B,H,dv]."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    Ls = states.shape[2]
    io = _io(q.dtype)
    _need(t, "t", torch.int64)
    for x, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(x, n, q.dtype)
    for x, n in ((log_alpha, "log_alpha"), (beta, "beta"), (lam, "lam"), (states, "states")):
        _need(x, n, torch.float32)
    if o is None:
        o = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    st = lib().ll_gdn_decode_step(B, H, dk, dv, Ls, io, _ptr(t), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                  _ptr(beta), _ptr(lam), _ptr(states), _ptr(o), _stream(q.device))
    _check(st, "ll_gdn_decode_step")
    return o


def _gdn_forward(entry: str, size_query, q, k, v, log_alpha, beta, lam, chunk, o, workspace):
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = lam.shape[-1]
    io = _io(q.dtype)
    for x, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(x, n, q.dtype)
    for x, n in ((log_alpha, "log_alpha"), (beta, "beta"), (lam, "lam")):
        _need(x, n, torch.float32)
    shape = make_shape(B, H, T, dk, dv, L, chunk, 0, io)
    if o is None:
        o = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(size_query(shape), q.device)
    st = getattr(lib(), entry)(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                               _ptr(lam), _ptr(o), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                               _stream(q.device))
    _check(st, entry)
    return o


def ll_gdn_fwd(q, k, v, log_alpha, beta, lam, chunk: int, *, o=None, workspace=None):
    """Log-Linear Gated DeltaNet forward (reading A).  Shapes as ll_attn_fwd plus
    beta [B,H,T] float32.  Returns o [B,H,T,dv]."""
    return _gdn_forward("ll_gdn_fwd", ll_gdn_fwd_workspace_size, q, k, v, log_alpha, beta, lam, chunk, o, workspace)


def ll_gdn_fwd_b(q, k, v, log_alpha, beta, lam, chunk: int, *, o=None, workspace=None):
    """Log-Linear Gated DeltaNet forward, reading B (log-linear Mamba-2 on the
    delta-rule pseudo-values).  Arguments as ll_gdn_fwd."""
    return _gdn_forward("ll_gdn_fwd_b", ll_gdn_fwd_b_workspace_size, q, k, v, log_alpha, beta, lam, chunk, o,
                        workspace)

def ll_test_fwd_withhold_node(q, k, v, log_alpha, lam, chunk: int, node: int, timeout_ns: int, *, o=None,
                              workspace=None) -> int:
    """Test hook: the tensor-core forward with Fenwick node `node` never
    published and every bounded wait limited to `timeout_ns`.  Returns the
    launch status (the expiry itself is reported by ll_last_device_error)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    shape = make_shape(B, H, T, dk, dv, lam.shape[-1], chunk, 0, _io(q.dtype))
    if o is None:
        o = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(ll_attn_fwd_workspace_size(shape), q.device)
    return lib().ll_test_fwd_withhold_node(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                           _ptr(lam), _ptr(o), _ptr(workspace), workspace.numel(), int(node),
                                           int(timeout_ns), _stream(q.device))


def ll_last_device_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error status."""
    return int(lib().ll_last_device_error(_stream(device)))


def ll_status_str(status: int) -> str:
    return lib().ll_status_str(int(status)).decode()


def ll_version() -> int:
    return int(lib().ll_version())
