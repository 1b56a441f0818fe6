"""Python binding of libgdn_gb300.so, the sm_103a gated delta-rule library.

Argument marshalling only: each function checks that the torch tensors it is
given are contiguous fp32 CUDA tensors of the sizes the C call will touch,
derives the shape, and calls the C entry point of the same name on the
current (or given) CUDA stream.  Every step of the computation runs in the
library's CUDA kernels; there is no other implementation behind these
functions, and importing them fails loudly when the library is not built.

Layouts (see include/gdn.h):
    S [B][vh][kd][vd];  q, k [B][T][kh][kd];  v, o [B][T][vh][vd];
    g, beta [B][T][vh];  ckpt [M][B][vh][kd][vd].
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "GDNError", "gdn_step", "gdn_step_m", "gdn_mark", "gdn_rollback",
    "gdn_rollback_seq", "gdn_prefill_workspace", "gdn_prefill",
    "gdn_strerror", "gdn_version", "library_path", "load",
    "GDN_PREC_FP32", "GDN_PREC_BF16X3", "GDN_PREC_BF16", "GDN_MAX_TOKENS",
    "gdn_prefill_timeouts", "gdn_layer_prologue_m", "gdn_layer_workspace",
    "gdn_layer_step_m", "gdn_layer_hist_rollback",
    "gdn_layer_step_m_noalloc", "GDN_NOALLOC_SCRATCH_BYTES",
    "gdn_gated_rmsnorm_m",
]

GDN_OK, GDN_EINVAL, GDN_ESHAPE, GDN_EALIGN = 0, -1, -2, -3
GDN_ECUDA, GDN_ERANGE, GDN_EPTR, GDN_EALIAS = -4, -5, -6, -7
GDN_ESCRATCH = -8
GDN_PREC_FP32, GDN_PREC_BF16X3, GDN_PREC_BF16 = 0, 1, 2
GDN_MAX_TOKENS = 1 << 20
GDN_NOALLOC_SCRATCH_BYTES = 16 << 20

# Every symbol include/gdn.h declares.
EXPORTS = ("gdn_step", "gdn_step_m", "gdn_mark", "gdn_rollback",
           "gdn_rollback_seq", "gdn_prefill_workspace", "gdn_prefill",
           "gdn_prefill_timeouts", "gdn_wait_timeouts", "gdn_layer_prologue_m",
           "gdn_layer_workspace", "gdn_layer_step_m",
           "gdn_layer_hist_rollback", "gdn_gated_rmsnorm_m",
           "gdn_layer_step_m_noalloc", "gdn_strerror", "gdn_version")


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gdn_strerror(status)} (status {status})")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("kh", ctypes.c_int),
                ("vh", ctypes.c_int), ("kd", ctypes.c_int),
                ("vd", ctypes.c_int)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load libgdn_gb300.so (built by ``_build.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise ImportError(
            f"{_build.LIB} is not built; run __graft_entry__.build() "
            "(or python -m gated_deltanet_linear_gb300._build)")
    lib = ctypes.CDLL(_build.LIB)
    vp, ip, cp = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(Shape)
    sig = {
        "gdn_step": [cp] + [vp] * 7 + [vp],
        "gdn_step_m": [cp, ip] + [vp] * 9 + [vp],
        "gdn_mark": [cp, vp, vp, vp],
        "gdn_rollback": [cp, ip, ip, vp, vp, vp, vp],
        "gdn_rollback_seq": [cp, ip, vp, vp, vp, vp, vp, vp],
        "gdn_prefill": [cp, ip] + [vp] * 7 + [ip, ip, vp, ctypes.c_size_t, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.gdn_prefill_workspace.argtypes = [cp, ip, ip, ip]
    lib.gdn_prefill_workspace.restype = ctypes.c_size_t
    lib.gdn_layer_prologue_m.argtypes = [cp, ip, ip, ctypes.c_float] + [vp] * 14
    lib.gdn_layer_prologue_m.restype = ctypes.c_int
    lib.gdn_layer_workspace.argtypes = [cp, ip]
    lib.gdn_layer_workspace.restype = ctypes.c_size_t
    lib.gdn_layer_step_m.argtypes = [cp, ip, ip, ctypes.c_float] + [vp] * 13 + \
        [ctypes.c_size_t, vp]
    lib.gdn_layer_step_m.restype = ctypes.c_int
    lib.gdn_gated_rmsnorm_m.argtypes = [cp, ip, ctypes.c_float] + [vp] * 5
    lib.gdn_gated_rmsnorm_m.restype = ctypes.c_int
    lib.gdn_layer_step_m_noalloc.argtypes = [cp, ip, ip, ctypes.c_float] + \
        [vp] * 12 + [vp]
    lib.gdn_layer_step_m_noalloc.restype = ctypes.c_int
    lib.gdn_layer_hist_rollback.argtypes = [cp, ip, ip] + [vp] * 6
    lib.gdn_layer_hist_rollback.restype = ctypes.c_int
    lib.gdn_prefill_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.gdn_prefill_timeouts.restype = ctypes.c_int
    lib.gdn_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.gdn_wait_timeouts.restype = ctypes.c_int
    lib.gdn_strerror.argtypes = [ctypes.c_int]
    lib.gdn_strerror.restype = ctypes.c_char_p
    lib.gdn_version.restype = ctypes.c_int
    _lib = lib
    return lib


def gdn_strerror(status: int) -> str:
    return load().gdn_strerror(int(status)).decode()


def gdn_version() -> int:
    return load().gdn_version()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _t(x, name, numel):
    """Pointer of a contiguous fp32 CUDA tensor with exactly numel elements."""
    if x is None:
        return None
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if x.numel() != numel:
        raise ValueError(f"{name} has {x.numel()} elements, expected {numel}")
    return x.data_ptr()


def _io(x, name, numel):
    """Pointer of a token input or output: a contiguous fp32 CUDA tensor, or a
    page-locked (pinned) CPU tensor, which the kernels read or write over the
    host link."""
    if isinstance(x, torch.Tensor) and not x.is_cuda:
        if not x.is_pinned():
            raise ValueError(f"{name}: a CPU tensor must be pinned "
                             "(tensor.pin_memory())")
        if x.dtype != torch.float32 or not x.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 tensor")
        if x.numel() != numel:
            raise ValueError(f"{name} has {x.numel()} elements, expected {numel}")
        return x.data_ptr()
    return _t(x, name, numel)


def _shape(S, q):
    if S.dim() != 4:
        raise ValueError("S must be [B][vh][kd][vd]")
    B, vh, kd, vd = S.shape
    kh = q.shape[-2]
    return Shape(B, kh, vh, kd, vd)


def _check(status, where):
    if status != GDN_OK:
        raise GDNError(status, where)


def gdn_step(S, q, k, v, g, beta, o, stream=None):
    """One token for all heads; S is updated in place, o written.  The token
    tensors (q, k, v, g, beta, o) may be CUDA tensors or pinned CPU tensors."""
    sh = _shape(S, q)
    B, kh, vh, kd, vd = sh.B, sh.kh, sh.vh, sh.kd, sh.vd
    args = (_t(S, "S", B * vh * kd * vd), _io(q, "q", B * kh * kd),
            _io(k, "k", B * kh * kd), _io(v, "v", B * vh * vd),
            _io(g, "g", B * vh), _io(beta, "beta", B * vh),
            _io(o, "o", B * vh * vd))
    _check(load().gdn_step(ctypes.byref(sh), *args, _stream(stream)),
           "gdn_step")


def gdn_step_m(S_in, S_out, ckpt, q, k, v, g, beta, o, M=None, stream=None):
    """M tokens in one launch (M defaults to q.shape[1]).  The token tensors
    may be CUDA tensors or pinned CPU tensors, as for gdn_step."""
    sh = _shape(S_in, q)
    B, kh, vh, kd, vd = sh.B, sh.kh, sh.vh, sh.kd, sh.vd
    M = int(q.shape[1] if M is None else M)
    n = B * vh * kd * vd
    args = (_t(S_in, "S_in", n), _t(S_out, "S_out", n),
            _t(ckpt, "ckpt", M * n), _io(q, "q", B * M * kh * kd),
            _io(k, "k", B * M * kh * kd), _io(v, "v", B * M * vh * vd),
            _io(g, "g", B * M * vh), _io(beta, "beta", B * M * vh),
            _io(o, "o", B * M * vh * vd))
    _check(load().gdn_step_m(ctypes.byref(sh), M, *args, _stream(stream)),
           "gdn_step_m")


def gdn_mark(S, snap, kh, stream=None):
    """snap = S (device copy on the stream)."""
    B, vh, kd, vd = S.shape
    sh = Shape(B, kh, vh, kd, vd)
    n = B * vh * kd * vd
    _check(load().gdn_mark(ctypes.byref(sh), _t(S, "S", n),
                           _t(snap, "snap", n), _stream(stream)), "gdn_mark")


def gdn_rollback(S, M, m, snap, ckpt, kh, stream=None):
    """S = snap (m == 0) or ckpt[m-1] (1 <= m <= M)."""
    B, vh, kd, vd = S.shape
    sh = Shape(B, kh, vh, kd, vd)
    n = B * vh * kd * vd
    _check(load().gdn_rollback(ctypes.byref(sh), int(M), int(m),
                               _t(snap, "snap", n),
                               _t(ckpt, "ckpt", int(M) * n),
                               _t(S, "S", n), _stream(stream)), "gdn_rollback")


def gdn_rollback_seq(S, M, m_dev, snap, ckpt, kh, err_dev=None, stream=None):
    """Per-sequence rollback; m_dev is an int32 CUDA tensor [B]."""
    B, vh, kd, vd = S.shape
    sh = Shape(B, kh, vh, kd, vd)
    n = B * vh * kd * vd
    for x, name, cnt in ((m_dev, "m_dev", B), (err_dev, "err_dev", 1)):
        if x is not None and (not x.is_cuda or x.dtype != torch.int32 or
                              not x.is_contiguous() or x.numel() != cnt):
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor "
                             f"of {cnt} elements")
    _check(load().gdn_rollback_seq(
        ctypes.byref(sh), int(M), m_dev.data_ptr(), _t(snap, "snap", n),
        _t(ckpt, "ckpt", int(M) * n), _t(S, "S", n),
        None if err_dev is None else err_dev.data_ptr(), _stream(stream)),
        "gdn_rollback_seq")


def gdn_prefill_workspace(B, kh, vh, T, chunk=64, precision=GDN_PREC_FP32,
                          kd=128, vd=128):
    sh = Shape(B, kh, vh, kd, vd)
    return int(load().gdn_prefill_workspace(ctypes.byref(sh), int(T),
                                            int(chunk), int(precision)))


def gdn_prefill_timeouts():
    """Chunked-prefill CTAs that gave up waiting on the tensor cores (0)."""
    c = ctypes.c_uint(0)
    _check(load().gdn_prefill_timeouts(ctypes.byref(c)), "gdn_prefill_timeouts")
    return int(c.value)


def gdn_wait_timeouts():
    """Bounded waits that ran out in any kernel since the library was loaded
    on the current device (synchronises the device)."""
    n = ctypes.c_uint(0)
    _check(load().gdn_wait_timeouts(ctypes.byref(n)), "gdn_wait_timeouts")
    return int(n.value)


def gdn_prefill(S, q, k, v, g, beta, o, precision=GDN_PREC_FP32, chunk=64,
                workspace=None, stream=None):
    """T = q.shape[1] tokens; S updated in place (S_0 -> S_T).

    precision: GDN_PREC_FP32 (token-serial, exact to the single-step path),
    GDN_PREC_BF16X3 or GDN_PREC_BF16 (chunk-parallel on tensor cores)."""
    sh = _shape(S, q)
    B, kh, vh, kd, vd = sh.B, sh.kh, sh.vh, sh.kd, sh.vd
    T = int(q.shape[1])
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr = workspace.data_ptr()
        ws_bytes = workspace.numel() * workspace.element_size()
    args = (_t(S, "S", B * vh * kd * vd), _t(q, "q", B * T * kh * kd),
            _t(k, "k", B * T * kh * kd), _t(v, "v", B * T * vh * vd),
            _t(g, "g", B * T * vh), _t(beta, "beta", B * T * vh),
            _t(o, "o", B * T * vh * vd))
    _check(load().gdn_prefill(ctypes.byref(sh), T, *args, int(chunk),
                              int(precision), ws_ptr, ws_bytes,
                              _stream(stream)), "gdn_prefill")


def _layer_shape(hist, x, kh, vh=None, kd=128, vd=128):
    B, ck1, conv_dim = hist.shape
    vh = (conv_dim - 2 * int(kh) * kd) // vd if vh is None else vh
    return Shape(B, int(kh), vh, kd, vd), int(x.shape[1]), ck1 + 1, conv_dim


def gdn_layer_prologue_m(hist_in, hist_out, x, conv_w, a, b, A_log, dt_bias,
                         q, k, v, g, beta, kh, eps=1e-6, stream=None):
    """conv1d + SiLU with history, q/k norm and gates for M = x.shape[1]
    tokens, writing q, k, v, g, beta (the inputs of gdn_step_m)."""
    sh, M, ck, conv_dim = _layer_shape(hist_in, x, kh)
    B, vh = sh.B, sh.vh
    nh = B * (ck - 1) * conv_dim
    args = (_t(hist_in, "hist_in", nh), _t(hist_out, "hist_out", nh),
            _t(x, "x", B * M * conv_dim), _t(conv_w, "conv_w", conv_dim * ck),
            _t(a, "a", B * M * vh), _t(b, "b", B * M * vh),
            _t(A_log, "A_log", vh), _t(dt_bias, "dt_bias", vh),
            _t(q, "q", B * M * sh.kh * 128), _t(k, "k", B * M * sh.kh * 128),
            _t(v, "v", B * M * vh * 128), _t(g, "g", B * M * vh),
            _t(beta, "beta", B * M * vh))
    _check(load().gdn_layer_prologue_m(ctypes.byref(sh), M, ck, float(eps),
                                       *args, _stream(stream)),
           "gdn_layer_prologue_m")


def gdn_layer_workspace(B, kh, vh, M, kd=128, vd=128):
    sh = Shape(B, kh, vh, kd, vd)
    return int(load().gdn_layer_workspace(ctypes.byref(sh), int(M)))


def gdn_layer_step_m(S_in, S_out, ckpt, hist_in, hist_out, x, conv_w, a, b,
                     A_log, dt_bias, o, kh, workspace, eps=1e-6, stream=None):
    """Layer prologue + update over M = x.shape[1] tokens; the intermediate
    q, k, v, g, beta live in `workspace` (gdn_layer_workspace bytes)."""
    if S_in.dim() != 4:
        raise ValueError("S must be [B][vh][kd][vd]")
    B, vh, kd, vd = S_in.shape
    sh = Shape(B, int(kh), vh, kd, vd)
    M = int(x.shape[1])
    ck = int(conv_w.shape[1])
    conv_dim = 2 * int(kh) * kd + vh * vd
    n = B * vh * kd * vd
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    args = (_t(S_in, "S_in", n), _t(S_out, "S_out", n),
            _t(ckpt, "ckpt", M * n),
            _t(hist_in, "hist_in", B * (ck - 1) * conv_dim),
            _t(hist_out, "hist_out", B * (ck - 1) * conv_dim),
            _t(x, "x", B * M * conv_dim), _t(conv_w, "conv_w", conv_dim * ck),
            _t(a, "a", B * M * vh), _t(b, "b", B * M * vh),
            _t(A_log, "A_log", vh), _t(dt_bias, "dt_bias", vh),
            _t(o, "o", B * M * vh * vd))
    _check(load().gdn_layer_step_m(
        ctypes.byref(sh), M, ck, float(eps), *args, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "gdn_layer_step_m")


def gdn_gated_rmsnorm_m(o, z, w, y, eps=1e-6, stream=None):
    """Gated RMSNorm of o [B][M][vh][vd] with gate z (same shape) and
    per-channel weight w [vd] into y (y may be o)."""
    if o.dim() != 4:
        raise ValueError("o must be [B][M][vh][vd]")
    B, M, vh, vd = o.shape
    sh = Shape(B, 1, vh, 128, vd)
    n = o.numel()
    _check(load().gdn_gated_rmsnorm_m(
        ctypes.byref(sh), M, float(eps), _t(o, "o", n), _t(z, "z", n),
        _t(w, "w", vd), _t(y, "y", n), _stream(stream)),
        "gdn_gated_rmsnorm_m")


def gdn_layer_step_m_noalloc(S_in, S_out, ckpt, hist_in, hist_out, x, conv_w,
                             a, b, A_log, dt_bias, o, kh, eps=1e-6,
                             stream=None):
    """gdn_layer_step_m for callers that cannot allocate device memory: the
    intermediate q, k, v, g, beta go to the library's own static scratch of
    GDN_NOALLOC_SCRATCH_BYTES (shared by every call on the device; calls that
    overlap on the GPU race).  Larger requests raise GDNError with
    GDN_ESCRATCH."""
    if S_in.dim() != 4:
        raise ValueError("S must be [B][vh][kd][vd]")
    B, vh, kd, vd = S_in.shape
    sh = Shape(B, int(kh), vh, kd, vd)
    M = int(x.shape[1])
    ck = int(conv_w.shape[1])
    conv_dim = 2 * int(kh) * kd + vh * vd
    n = B * vh * kd * vd
    args = (_t(S_in, "S_in", n), _t(S_out, "S_out", n),
            _t(ckpt, "ckpt", M * n),
            _t(hist_in, "hist_in", B * (ck - 1) * conv_dim),
            _t(hist_out, "hist_out", B * (ck - 1) * conv_dim),
            _t(x, "x", B * M * conv_dim), _t(conv_w, "conv_w", conv_dim * ck),
            _t(a, "a", B * M * vh), _t(b, "b", B * M * vh),
            _t(A_log, "A_log", vh), _t(dt_bias, "dt_bias", vh),
            _t(o, "o", B * M * vh * vd))
    _check(load().gdn_layer_step_m_noalloc(
        ctypes.byref(sh), M, ck, float(eps), *args, _stream(stream)),
        "gdn_layer_step_m_noalloc")


def gdn_layer_hist_rollback(hist, M, m_dev, hist_snap, x, kh, kd=128, vd=128,
                            err_dev=None, stream=None):
    """Conv history after m_dev[b] of the M tokens of a layer launch."""
    B, ck1, conv_dim = hist.shape
    vh = (conv_dim - 2 * int(kh) * kd) // vd
    sh = Shape(B, int(kh), vh, kd, vd)
    for t_, name, cnt in ((m_dev, "m_dev", B), (err_dev, "err_dev", 1)):
        if t_ is not None and (not t_.is_cuda or t_.dtype != torch.int32 or
                               not t_.is_contiguous() or t_.numel() != cnt):
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor "
                             f"of {cnt} elements")
    _check(load().gdn_layer_hist_rollback(
        ctypes.byref(sh), int(M), ck1 + 1, m_dev.data_ptr(),
        _t(hist_snap, "hist_snap", hist.numel()),
        _t(x, "x", B * int(M) * conv_dim), _t(hist, "hist", hist.numel()),
        None if err_dev is None else err_dev.data_ptr(), _stream(stream)),
        "gdn_layer_hist_rollback")
