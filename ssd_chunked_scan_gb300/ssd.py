"""Python binding of libssd (include/ssd.h): argument marshalling only.

Every step of the scan runs in the CUDA library; this module checks tensor
dtypes / devices / shapes, passes raw device pointers and the current CUDA
stream through ctypes, and turns a non-zero status into ``SSDError``.  There is
no fallback: if libssd.so is missing or fails to load, importing this module
raises.
"""
import ctypes
import os

import torch

# SSD_LIB_VARIANT=check selects the debug build (index checks, see build.py)
_LIB_NAME = "libssd_check.so" if os.environ.get("SSD_LIB_VARIANT", "") == "check" else "libssd.so"
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", _LIB_NAME)

SSD_OK = 0
SSD_ERR_ARG = 1
SSD_ERR_ALIGN = 2
SSD_ERR_CHUNK = 3
SSD_ERR_UNSUPPORTED = 4
SSD_ERR_ALLOC = 5
SSD_ERR_LAUNCH = 6
SSD_ERR_TIMEOUT = 7
SSD_ERR_CUDA = 8
SSD_ERR_SCRATCH = 9
SSD_ERR_CHECK = 10
SSD_PATH_TC = 0
SSD_PATH_SIMT = 1

EXPORTED = ("ssd_fwd", "ssd_bwd", "ssd_set_path", "ssd_get_path", "ssd_set_overlap",
            "ssd_get_overlap", "ssd_strerror",
            "ssd_last_device_error", "ssd_version", "ssd_launch_count", "ssd_trace_enable",
            "ssd_trace_collect", "ssd_trace_get", "ssd_trace_reset", "ssd_fwd_noalloc",
            "ssd_fwd_noalloc_scratch_bytes", "ssd_test_stall_walks", "ssd_set_deterministic",
            "ssd_get_deterministic", "ssd_saved_bytes", "ssd_fwd_save", "ssd_bwd_saved")


class SSDError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {ssd_strerror(status)} (status {status})")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_NAME} not built at {_LIB_PATH}; run __graft_entry__.build()"
                          + (" / build_lib(check=True)" if _LIB_NAME != "libssd.so" else ""))
    lib = ctypes.CDLL(_LIB_PATH)
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.ssd_fwd.argtypes = [p] * 6 + [i64] * 7 + [p]
    lib.ssd_fwd.restype = ctypes.c_int
    lib.ssd_bwd.argtypes = [p] * 11 + [i64] * 7 + [p]
    lib.ssd_fwd_ex.argtypes = [p] * 7 + [i64] * 7 + [p]
    lib.ssd_fwd_ex.restype = ctypes.c_int
    lib.ssd_bwd_ex.argtypes = [p] * 12 + [i64] * 7 + [p]
    lib.ssd_bwd_ex.restype = ctypes.c_int
    lib.ssd_fwd_save.argtypes = [p] * 8 + [i64] * 7 + [p]
    lib.ssd_fwd_save.restype = ctypes.c_int
    lib.ssd_bwd_saved.argtypes = [p] * 14 + [i64] * 7 + [p]
    lib.ssd_bwd_saved.restype = ctypes.c_int
    lib.ssd_saved_bytes.argtypes = [i64] * 7 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.ssd_saved_bytes.restype = ctypes.c_int
    lib.ssd_bwd.restype = ctypes.c_int
    lib.ssd_set_path.argtypes = [ctypes.c_int]
    lib.ssd_set_path.restype = ctypes.c_int
    lib.ssd_get_path.argtypes = []
    lib.ssd_get_path.restype = ctypes.c_int
    lib.ssd_set_overlap.argtypes = [ctypes.c_int]
    lib.ssd_set_overlap.restype = ctypes.c_int
    lib.ssd_get_overlap.argtypes = []
    lib.ssd_get_overlap.restype = ctypes.c_int
    lib.ssd_strerror.argtypes = [ctypes.c_int]
    lib.ssd_strerror.restype = ctypes.c_char_p
    lib.ssd_last_device_error.argtypes = [p]
    lib.ssd_last_device_error.restype = ctypes.c_int
    lib.ssd_version.argtypes = []
    lib.ssd_version.restype = ctypes.c_int
    lib.ssd_launch_count.argtypes = []
    lib.ssd_launch_count.restype = ctypes.c_longlong
    lib.ssd_trace_enable.argtypes = [ctypes.c_int]
    lib.ssd_trace_collect.argtypes = []
    lib.ssd_trace_get.argtypes = [ctypes.c_int, ctypes.c_char_p, ctypes.c_int,
                                  ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_double)]
    lib.ssd_trace_reset.argtypes = []
    lib.ssd_fwd_workspace_bytes.argtypes = [i64] * 7 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.ssd_fwd_workspace_bytes.restype = ctypes.c_int
    lib.ssd_bwd_workspace_bytes.argtypes = [i64] * 7 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.ssd_bwd_workspace_bytes.restype = ctypes.c_int
    lib.ssd_pool_high_water.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    lib.ssd_pool_high_water.restype = ctypes.c_int
    lib.ssd_mamba_fwd.argtypes = [p] * 7 + [i64] * 4 + [p]
    lib.ssd_mamba_fwd.restype = ctypes.c_int
    lib.ssd_mamba_bwd.argtypes = [p] * 13 + [i64] * 4 + [p]
    lib.ssd_mamba_bwd.restype = ctypes.c_int
    lib.ssd_mamba_workspace_bytes.argtypes = [ctypes.c_int] + [i64] * 4 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.ssd_mamba_workspace_bytes.restype = ctypes.c_int
    lib.ssd_fwd_noalloc.argtypes = [p] * 6 + [i64] * 7 + [p]
    lib.ssd_fwd_noalloc.restype = ctypes.c_int
    lib.ssd_fwd_noalloc_scratch_bytes.argtypes = []
    lib.ssd_fwd_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.ssd_set_deterministic.argtypes = [ctypes.c_int]
    lib.ssd_set_deterministic.restype = ctypes.c_int
    lib.ssd_get_deterministic.argtypes = []
    lib.ssd_get_deterministic.restype = ctypes.c_int
    lib.ssd_test_stall_walks.argtypes = [ctypes.c_int]
    lib.ssd_test_stall_walks.restype = ctypes.c_int
    return lib


LIB = _load()


def ssd_strerror(status: int) -> str:
    return LIB.ssd_strerror(int(status)).decode()


def ssd_set_path(path: int) -> None:
    rc = LIB.ssd_set_path(int(path))
    if rc:
        raise SSDError(rc, "ssd_set_path")


def ssd_get_path() -> int:
    return int(LIB.ssd_get_path())


def ssd_set_overlap(on: bool) -> bool:
    """Run the tensor-core backward's dk / dv passes on the library's side
    stream (True, the default) or every kernel on the caller's stream in turn;
    returns the previous setting."""
    return bool(LIB.ssd_set_overlap(1 if on else 0))


def ssd_get_overlap() -> bool:
    return bool(LIB.ssd_get_overlap())


def ssd_set_deterministic(on: bool) -> bool:
    """Sum a group's per-head dq / dk in head order (True) instead of with
    atomic adds (False, the default) in the tensor-core backward, so that the
    sums are bitwise reproducible; returns the previous setting."""
    return bool(LIB.ssd_set_deterministic(1 if on else 0))


def ssd_get_deterministic() -> bool:
    return bool(LIB.ssd_get_deterministic())


def ssd_last_device_error(stream=None) -> int:
    return int(LIB.ssd_last_device_error(_stream(stream)))


def ssd_test_stall_walks(on: bool) -> None:
    """Failure-path test switch (include/ssd.h): while on, every tensor-core
    walk CTA stalls on a barrier nothing completes until its bounded wait gives
    up, and ssd_last_device_error then reports SSD_ERR_TIMEOUT."""
    rc = LIB.ssd_test_stall_walks(1 if on else 0)
    if rc:
        raise SSDError(rc, "ssd_test_stall_walks")


def ssd_launch_count() -> int:
    """Kernels launched by libssd in this process so far."""
    return int(LIB.ssd_launch_count())


def ssd_trace_enable(on: bool) -> None:
    LIB.ssd_trace_enable(1 if on else 0)


def ssd_trace_reset() -> None:
    LIB.ssd_trace_reset()


def ssd_trace_collect() -> dict:
    """Per-kernel {name: (launches, total_ms)} of the traced launches so far."""
    n = LIB.ssd_trace_collect()
    if n < 0:
        raise SSDError(-n, "ssd_trace_collect")
    res = {}
    buf = ctypes.create_string_buffer(128)
    for i in range(n):
        cnt, ms = ctypes.c_longlong(0), ctypes.c_double(0.0)
        rc = LIB.ssd_trace_get(i, buf, 128, ctypes.byref(cnt), ctypes.byref(ms))
        if rc:
            raise SSDError(rc, "ssd_trace_get")
        res[buf.value.decode()] = (int(cnt.value), float(ms.value))
    return res


def ssd_fwd_workspace_bytes(B, L, G, H, dk, dv, chunk=64) -> int:
    """Device workspace bytes ssd_fwd takes for this problem on the active path."""
    n = ctypes.c_size_t(0)
    rc = LIB.ssd_fwd_workspace_bytes(B, L, G, H, dk, dv, chunk, ctypes.byref(n))
    if rc:
        raise SSDError(rc, "ssd_fwd_workspace_bytes")
    return int(n.value)


def ssd_bwd_workspace_bytes(B, L, G, H, dk, dv, chunk=64) -> int:
    """Device workspace bytes ssd_bwd takes for this problem on the active path."""
    n = ctypes.c_size_t(0)
    rc = LIB.ssd_bwd_workspace_bytes(B, L, G, H, dk, dv, chunk, ctypes.byref(n))
    if rc:
        raise SSDError(rc, "ssd_bwd_workspace_bytes")
    return int(n.value)


def ssd_pool_high_water(reset=False) -> int:
    """High-water bytes of the current device's default stream-ordered pool
    (read before an optional reset to the memory in use now)."""
    n = ctypes.c_size_t(0)
    rc = LIB.ssd_pool_high_water(1 if reset else 0, ctypes.byref(n))
    if rc:
        raise SSDError(rc, "ssd_pool_high_water")
    return int(n.value)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _check(name, t, shape, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a float32 torch tensor")
    if t.device.type != "cuda":  # the library takes device pointers only
        raise ValueError(f"{name} must be a CUDA tensor, got {t.device}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dims(q, v):
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q must be [B,L,G,dk] and v [B,L,H,dv]")
    B, L, G, dk = q.shape
    H, dv = v.shape[2], v.shape[3]
    return B, L, G, H, dk, dv


def ssd_fwd(q, k, v, log_alpha, h0=None, chunk=64, out=None, stream=None):
    """out [B,L,H,dv] of the scan for q,k [B,L,G,dk], v [B,L,H,dv], log_alpha [B,L,H]."""
    B, L, G, H, dk, dv = _dims(q, v)
    dev = q.device
    _check("q", q, (B, L, G, dk), dev)
    _check("k", k, (B, L, G, dk), dev)
    _check("v", v, (B, L, H, dv), dev)
    _check("log_alpha", log_alpha, (B, L, H), dev)
    _check("h0", h0, (B, H, dk, dv), dev)
    if out is None:
        out = torch.empty((B, L, H, dv), dtype=torch.float32, device=dev)
    _check("out", out, (B, L, H, dv), dev)
    rc = LIB.ssd_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(h0), _ptr(out),
                     B, L, G, H, dk, dv, int(chunk), _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_fwd")
    return out


def _grad_buffers(B, L, G, H, dk, dv, dev, want_dh0, grads):
    shapes = {"dq": (B, L, G, dk), "dk": (B, L, G, dk), "dv": (B, L, H, dv),
              "dlog_alpha": (B, L, H), "dh0": (B, H, dk, dv)}
    g = dict(grads or {})
    for n, s in shapes.items():
        if n == "dh0" and not want_dh0:
            g[n] = None
            continue
        if g.get(n) is None:
            g[n] = torch.empty(s, dtype=torch.float32, device=dev)
        _check(n, g[n], s, dev)
    return g


def ssd_bwd(q, k, v, log_alpha, h0, dout, chunk=64, want_dh0=True, grads=None, stream=None):
    """Gradients of <dout, out>: dict dq, dk, dv, dlog_alpha, dh0 (dh0 None if not wanted).

    ``grads`` may supply preallocated output tensors under the same keys.
    """
    B, L, G, H, dk, dv = _dims(q, v)
    dev = q.device
    for n, t, s in (("q", q, (B, L, G, dk)), ("k", k, (B, L, G, dk)), ("v", v, (B, L, H, dv)),
                    ("log_alpha", log_alpha, (B, L, H)), ("h0", h0, (B, H, dk, dv)),
                    ("dout", dout, (B, L, H, dv))):
        _check(n, t, s, dev)
    g = _grad_buffers(B, L, G, H, dk, dv, dev, want_dh0, grads)
    rc = LIB.ssd_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(h0), _ptr(dout),
                     _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dlog_alpha"]),
                     _ptr(g["dh0"]), B, L, G, H, dk, dv, int(chunk), _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_bwd")
    return g


def ssd_fwd_ex(q, k, v, log_alpha, h0=None, chunk=64, out=None, hT=None, stream=None):
    """(out, hT): the forward plus the final state hT [B,H,dk,dv] = S_{L-1}."""
    B, L, G, H, dk, dv = _dims(q, v)
    dev = q.device
    for n, t, s in (("q", q, (B, L, G, dk)), ("k", k, (B, L, G, dk)), ("v", v, (B, L, H, dv)),
                    ("log_alpha", log_alpha, (B, L, H)), ("h0", h0, (B, H, dk, dv))):
        _check(n, t, s, dev)
    if out is None:
        out = torch.empty((B, L, H, dv), dtype=torch.float32, device=dev)
    if hT is None:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _check("out", out, (B, L, H, dv), dev)
    _check("hT", hT, (B, H, dk, dv), dev)
    rc = LIB.ssd_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(h0), _ptr(out),
                        _ptr(hT), B, L, G, H, dk, dv, int(chunk), _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_fwd_ex")
    return out, hT


def ssd_bwd_ex(q, k, v, log_alpha, h0, dout, dhT, chunk=64, want_dh0=True, grads=None,
               stream=None):
    """Gradients of <dout, out> + <dhT, hT> (dhT None means zero), as ssd_bwd."""
    B, L, G, H, dk, dv = _dims(q, v)
    dev = q.device
    for n, t, s in (("q", q, (B, L, G, dk)), ("k", k, (B, L, G, dk)), ("v", v, (B, L, H, dv)),
                    ("log_alpha", log_alpha, (B, L, H)), ("h0", h0, (B, H, dk, dv)),
                    ("dout", dout, (B, L, H, dv)), ("dhT", dhT, (B, H, dk, dv))):
        _check(n, t, s, dev)
    g = _grad_buffers(B, L, G, H, dk, dv, dev, want_dh0, grads)
    rc = LIB.ssd_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(h0), _ptr(dout),
                        _ptr(dhT), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                        _ptr(g["dlog_alpha"]), _ptr(g["dh0"]), B, L, G, H, dk, dv, int(chunk),
                        _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_bwd_ex")
    return g


def ssd_saved_bytes(B, L, G, H, dk, dv, chunk=64) -> int:
    """Bytes of the segment states ssd_fwd_save keeps for ssd_bwd_saved (0 when
    the active path keeps none)."""
    n = ctypes.c_size_t(0)
    rc = LIB.ssd_saved_bytes(B, L, G, H, dk, dv, chunk, ctypes.byref(n))
    if rc:
        raise SSDError(rc, "ssd_saved_bytes")
    return int(n.value)


def _check_saved(saved, n, dev):
    if saved is None:
        return
    if not isinstance(saved, torch.Tensor) or saved.dtype != torch.float32 or saved.dim() != 1:
        raise TypeError("saved must be a 1-D float32 torch tensor")
    _check("saved", saved, (n,), dev)


def ssd_fwd_save(q, k, v, log_alpha, h0=None, chunk=64, out=None, hT=None, saved=None,
                 stream=None):
    """(out, hT, saved): ssd_fwd_ex, plus the segment states for ssd_bwd_saved
    (a flat float32 tensor of ssd_saved_bytes // 4 elements, None when the
    active path keeps none)."""
    B, L, G, H, dk, dv = _dims(q, v)
    dev = q.device
    for n, t, s in (("q", q, (B, L, G, dk)), ("k", k, (B, L, G, dk)), ("v", v, (B, L, H, dv)),
                    ("log_alpha", log_alpha, (B, L, H)), ("h0", h0, (B, H, dk, dv))):
        _check(n, t, s, dev)
    if out is None:
        out = torch.empty((B, L, H, dv), dtype=torch.float32, device=dev)
    if hT is None:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    n_saved = ssd_saved_bytes(B, L, G, H, dk, dv, chunk) // 4
    if saved is None and n_saved:
        saved = torch.empty((n_saved,), dtype=torch.float32, device=dev)
    _check("out", out, (B, L, H, dv), dev)
    _check("hT", hT, (B, H, dk, dv), dev)
    _check_saved(saved, n_saved, dev)
    rc = LIB.ssd_fwd_save(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(h0), _ptr(out),
                          _ptr(hT), _ptr(saved), B, L, G, H, dk, dv, int(chunk), _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_fwd_save")
    return out, hT, saved


def ssd_bwd_saved(q, k, v, log_alpha, h0, dout, dhT, hT, saved, chunk=64, want_dh0=True,
                  grads=None, stream=None):
    """ssd_bwd_ex with the segment states ``saved`` (and final state ``hT``)
    that ssd_fwd_save returned for the same inputs."""
    B, L, G, H, dk, dv = _dims(q, v)
    dev = q.device
    for n, t, s in (("q", q, (B, L, G, dk)), ("k", k, (B, L, G, dk)), ("v", v, (B, L, H, dv)),
                    ("log_alpha", log_alpha, (B, L, H)), ("h0", h0, (B, H, dk, dv)),
                    ("dout", dout, (B, L, H, dv)), ("dhT", dhT, (B, H, dk, dv)),
                    ("hT", hT, (B, H, dk, dv))):
        _check(n, t, s, dev)
    _check_saved(saved, ssd_saved_bytes(B, L, G, H, dk, dv, chunk) // 4 if saved is not None else 0, dev)
    g = _grad_buffers(B, L, G, H, dk, dv, dev, want_dh0, grads)
    rc = LIB.ssd_bwd_saved(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(h0), _ptr(dout),
                           _ptr(dhT), _ptr(hT), _ptr(saved), _ptr(g["dq"]), _ptr(g["dk"]),
                           _ptr(g["dv"]), _ptr(g["dlog_alpha"]), _ptr(g["dh0"]), B, L, G, H, dk,
                           dv, int(chunk), _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_bwd_saved")
    return g


def ssd_fwd_noalloc(q, k, v, log_alpha, h0, out, chunk=64, stream=None):
    """Forward into a caller-provided ``out`` without any device allocation.

    For callers that cannot allocate device memory at call time (memory fully
    reserved up front by another allocator, allocation-free real-time loops,
    allocator hooks).  Runs the all-fp32 path with the library's fixed
    scratch array; problems that do not fit raise SSDError(SSD_ERR_SCRATCH).
    Calls that overlap on the GPU share that array and race.
    """
    B, L, G, H, dk, dv = _dims(q, v)
    dev = q.device
    for n, t, s in (("q", q, (B, L, G, dk)), ("k", k, (B, L, G, dk)), ("v", v, (B, L, H, dv)),
                    ("log_alpha", log_alpha, (B, L, H)), ("h0", h0, (B, H, dk, dv)),
                    ("out", out, (B, L, H, dv))):
        _check(n, t, s, dev)
    if out is None:
        raise ValueError("out must be given")
    rc = LIB.ssd_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(h0), _ptr(out),
                             B, L, G, H, dk, dv, int(chunk), _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_fwd_noalloc")
    return out


# ---- Mamba-1 selective scan (include/ssd_mamba.h) --------------------------

def _mamba_dims(x, A):
    if x.dim() != 3 or A.dim() != 2:
        raise ValueError("x must be [B,L,D] and A [D,N]")
    B, L, D = x.shape
    return B, L, D, A.shape[1]


def _mamba_check_args(x, delta, A, Bm, Cm, Dk):
    B, L, D, N = _mamba_dims(x, A)
    dev = x.device
    for n, t, sh in (("x", x, (B, L, D)), ("delta", delta, (B, L, D)), ("A", A, (D, N)),
                     ("Bm", Bm, (B, L, N)), ("Cm", Cm, (B, L, N)), ("Dk", Dk, (D,))):
        _check(n, t, sh, dev)
    return B, L, D, N, dev


def ssd_mamba_fwd(x, delta, A, Bm, Cm, Dk=None, y=None, stream=None):
    """y [B,L,D] of the selective scan for x, delta [B,L,D], A [D,N], Bm, Cm [B,L,N], Dk [D]."""
    B, L, D, N, dev = _mamba_check_args(x, delta, A, Bm, Cm, Dk)
    if y is None:
        y = torch.empty((B, L, D), dtype=torch.float32, device=dev)
    _check("y", y, (B, L, D), dev)
    rc = LIB.ssd_mamba_fwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(Dk), _ptr(y),
                           B, L, D, N, _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_mamba_fwd")
    return y


def ssd_mamba_bwd(x, delta, A, Bm, Cm, Dk, dy, grads=None, stream=None):
    """Gradients of <dy, y>: dict dx, ddelta, dA, dB, dC, dD (dD None when Dk is None)."""
    B, L, D, N, dev = _mamba_check_args(x, delta, A, Bm, Cm, Dk)
    _check("dy", dy, (B, L, D), dev)
    shapes = {"dx": (B, L, D), "ddelta": (B, L, D), "dA": (D, N), "dB": (B, L, N),
              "dC": (B, L, N), "dD": (D,)}
    g = dict(grads or {})
    for n, sh in shapes.items():
        if n == "dD" and Dk is None:
            g[n] = None
            continue
        if g.get(n) is None:
            g[n] = torch.empty(sh, dtype=torch.float32, device=dev)
        _check(n, g[n], sh, dev)
    rc = LIB.ssd_mamba_bwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(Dk), _ptr(dy),
                           _ptr(g["dx"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]),
                           _ptr(g["dC"]), _ptr(g["dD"]), B, L, D, N, _stream(stream))
    if rc:
        raise SSDError(rc, "ssd_mamba_bwd")
    return g


def ssd_mamba_workspace_bytes(bwd, B, L, D, N) -> int:
    n = ctypes.c_size_t(0)
    rc = LIB.ssd_mamba_workspace_bytes(1 if bwd else 0, B, L, D, N, ctypes.byref(n))
    if rc:
        raise SSDError(rc, "ssd_mamba_workspace_bytes")
    return int(n.value)
