"""ctypes binding of libhcread.so (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of the read: tensors are checked for device, dtype, size and
contiguity, turned into pointers, and handed to the library.  There is no
fallback: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

HC_OK, HC_ERR_ARG, HC_ERR_ALIGN, HC_ERR_SHAPE, HC_ERR_CUDA, HC_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
HC_ERR_TOO_LARGE = -6
HC_NOALLOC_MAX_T = 8

# Every symbol the C headers (include/hc_read.h, include/hc_q2.h) declare.
EXPORTS = (
    "hc_read_create", "hc_read", "hc_read_ex", "hc_read_check", "hc_read_reset",
    "hc_read_destroy", "hc_read_scratch_bytes", "hc_status_str",
    "hc_graph_begin", "hc_graph_end", "hc_graph_launch", "hc_graph_destroy",
    "hc_read_noalloc", "hc_read_batch", "hc_read_batch_persistent", "hc_read_error_word",
    "hc_read_batch_plan", "hc_read_batch_groups", "hc_read_set_batch_lanes", "hc_read_q8",
    "hc_read_batch_q8", "hc_read_batch_q8_plan", "hc_read_batch_q8_groups",
    "hc_q2_0_matvec", "hc_q2_0_matvec_batch", "hc_q2_0_matvec_batch_plan",
    "hc_read_set_wait_limit", "hc_read_set_overlap", "hc_read_noalloc_check",
    "hc_read_down_tiles_bytes", "hc_read_register_down_tiles", "hc_read_forget_down_tiles",
    "hc_read_up_tiles_bytes", "hc_read_register_up_tiles", "hc_read_forget_up_tiles",
)


class hc_read_desc(ctypes.Structure):
    """One read of hc_read_batch (field order of the C struct)."""
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "R", "w_norm", "W_down", "W_up", "gate", "pending", "out", "mean", "lo")]


class hc_read_q8_desc(ctypes.Structure):
    """One Q8_0 read of hc_read_batch_q8 (field order of the C struct)."""
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "R", "w_norm", "Wd_q", "Wd_scale", "Wu_q", "Wu_scale", "gate", "pending", "out", "mean", "lo")]


class hc_q2_0_desc(ctypes.Structure):
    """One product of hc_q2_0_matvec_batch (field order of the C struct)."""
    _fields_ = [(name, ctypes.c_void_p) for name in ("Wq", "Wscale", "x", "y")]


class HcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} ({status})")


_lib = None
_vp = ctypes.c_void_p


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libhcread.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library not built: {p}. Run __graft_entry__.build() "
            "(the read has no CPU path).")
    lib = ctypes.CDLL(p)
    lib.hc_read_create.restype = ctypes.c_int
    lib.hc_read_create.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_float, ctypes.c_int]
    lib.hc_read.restype = ctypes.c_int
    lib.hc_read.argtypes = [_vp] * 7 + [ctypes.c_int] + [_vp] * 4
    lib.hc_read_ex.restype = ctypes.c_int
    lib.hc_read_ex.argtypes = [_vp] * 7 + [ctypes.c_int] + [_vp] * 6
    lib.hc_read_check.restype = ctypes.c_int
    lib.hc_read_check.argtypes = [_vp]
    lib.hc_read_reset.restype = ctypes.c_int
    lib.hc_read_reset.argtypes = [_vp, _vp]
    lib.hc_read_destroy.restype = None
    lib.hc_read_destroy.argtypes = [_vp]
    lib.hc_read_scratch_bytes.restype = ctypes.c_int64
    lib.hc_read_scratch_bytes.argtypes = [_vp]
    lib.hc_status_str.restype = ctypes.c_char_p
    lib.hc_status_str.argtypes = [ctypes.c_int]
    lib.hc_graph_begin.restype = ctypes.c_int
    lib.hc_graph_begin.argtypes = [_vp]
    lib.hc_graph_end.restype = ctypes.c_int
    lib.hc_graph_end.argtypes = [_vp, ctypes.POINTER(_vp)]
    lib.hc_graph_launch.restype = ctypes.c_int
    lib.hc_graph_launch.argtypes = [_vp, _vp]
    lib.hc_graph_destroy.restype = None
    lib.hc_graph_destroy.argtypes = [_vp]
    lib.hc_read_noalloc.restype = ctypes.c_int
    lib.hc_read_noalloc.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float] + \
        [_vp] * 6 + [ctypes.c_int] + [_vp] * 4
    lib.hc_read_batch.restype = ctypes.c_int
    lib.hc_read_batch.argtypes = [_vp, ctypes.POINTER(hc_read_desc), ctypes.c_int, ctypes.c_int, _vp]
    lib.hc_read_batch_plan.restype = ctypes.c_int
    lib.hc_read_batch_plan.argtypes = [_vp, ctypes.POINTER(hc_read_desc), ctypes.c_int, ctypes.c_int]
    lib.hc_read_q8.restype = ctypes.c_int
    lib.hc_read_q8.argtypes = [_vp] * 9 + [ctypes.c_int] + [_vp] * 6
    lib.hc_read_set_batch_lanes.restype = ctypes.c_int
    lib.hc_read_set_batch_lanes.argtypes = [_vp, ctypes.c_int]
    lib.hc_read_batch_groups.restype = ctypes.c_int
    lib.hc_read_batch_groups.argtypes = [ctypes.POINTER(hc_read_desc), ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int)]
    lib.hc_read_batch_q8.restype = ctypes.c_int
    lib.hc_read_batch_q8.argtypes = [_vp, ctypes.POINTER(hc_read_q8_desc), ctypes.c_int, ctypes.c_int, _vp]
    lib.hc_read_batch_q8_plan.restype = ctypes.c_int
    lib.hc_read_batch_q8_plan.argtypes = [_vp, ctypes.POINTER(hc_read_q8_desc), ctypes.c_int, ctypes.c_int]
    lib.hc_read_batch_q8_groups.restype = ctypes.c_int
    lib.hc_read_batch_q8_groups.argtypes = [ctypes.POINTER(hc_read_q8_desc), ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_int)]
    lib.hc_read_error_word.restype = ctypes.c_int64
    lib.hc_read_error_word.argtypes = [_vp]
    lib.hc_q2_0_matvec.restype = ctypes.c_int
    lib.hc_q2_0_matvec.argtypes = [_vp, _vp, ctypes.c_int, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp]
    lib.hc_q2_0_matvec_batch.restype = ctypes.c_int
    lib.hc_q2_0_matvec_batch.argtypes = [ctypes.POINTER(hc_q2_0_desc), ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, _vp]
    lib.hc_q2_0_matvec_batch_plan.restype = ctypes.c_int
    lib.hc_q2_0_matvec_batch_plan.argtypes = [ctypes.POINTER(hc_q2_0_desc), ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.hc_read_batch_persistent.restype = ctypes.c_int
    lib.hc_read_batch_persistent.argtypes = [_vp, ctypes.c_int]
    lib.hc_read_set_wait_limit.restype = ctypes.c_int
    lib.hc_read_set_wait_limit.argtypes = [_vp, ctypes.c_uint64]
    lib.hc_read_set_overlap.restype = ctypes.c_int
    lib.hc_read_set_overlap.argtypes = [_vp, ctypes.c_int]
    lib.hc_read_down_tiles_bytes.restype = ctypes.c_int64
    lib.hc_read_down_tiles_bytes.argtypes = [_vp]
    lib.hc_read_register_down_tiles.restype = ctypes.c_int
    lib.hc_read_register_down_tiles.argtypes = [_vp, _vp, _vp, _vp]
    lib.hc_read_forget_down_tiles.restype = ctypes.c_int
    lib.hc_read_forget_down_tiles.argtypes = [_vp, _vp]
    lib.hc_read_up_tiles_bytes.restype = ctypes.c_int64
    lib.hc_read_up_tiles_bytes.argtypes = [_vp]
    lib.hc_read_register_up_tiles.restype = ctypes.c_int
    lib.hc_read_register_up_tiles.argtypes = [_vp, _vp, _vp, _vp]
    lib.hc_read_forget_up_tiles.restype = ctypes.c_int
    lib.hc_read_forget_up_tiles.argtypes = [_vp, _vp]
    lib.hc_read_noalloc_check.restype = ctypes.c_int
    lib.hc_read_noalloc_check.argtypes = []
    if path is None:
        _lib = lib
    return lib


def status_str(status: int) -> str:
    try:
        return load().hc_status_str(status).decode()
    except RuntimeError:
        return {0: "ok", -1: "invalid argument", -2: "pointer not 16-byte aligned",
                -3: "geometry not supported", -4: "CUDA runtime error",
                -5: "a kernel gave up on a bounded wait",
                -6: "T exceeds the no-allocation entry point's maximum"}.get(status, "unknown status")


def _check(status: int, where: str) -> None:
    if status != HC_OK:
        raise HcError(status, where)


def _stream_ptr(stream) -> int | None:
    """cudaStream_t of a torch.cuda.Stream / int / None (None = current torch stream)."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _ptr(t, name: str, dtype_names: tuple[str, ...], numel: int | None):
    """Device pointer of a tensor after checking it; None stays NULL; ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, an int pointer or None")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (the read has no CPU path)")
    if str(t.dtype).replace("torch.", "") not in dtype_names:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtype_names}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


_F32 = ("float32",)
_BF16 = ("bfloat16", "uint16", "int16")
_I8 = ("int8",)
_HALF_BITS = ("float16", "uint16", "int16")


def hc_read_create(n: int, d: int, K: int, T_max: int, eps: float = 1e-6, device: int = 0) -> int:
    """Create a handle; returns it as an integer (free with hc_read_destroy)."""
    h = _vp()
    _check(load().hc_read_create(ctypes.byref(h), n, d, K, T_max, eps, device), "hc_read_create")
    return h.value


def hc_read_ex(h: int, geometry, R, w_norm, W_down, W_up, gate, pending, T: int,
               out, mean, lo, r_out=None, rs=None, stream=None) -> None:
    """Enqueue one read (see include/hc_read.h); ``geometry`` = (n, d, K) for size checks."""
    n, d, K = geometry
    N = n * d
    args = (
        _ptr(R, "R", _F32, T * N), _ptr(w_norm, "w_norm", _F32, N),
        _ptr(W_down, "W_down", _BF16, K * N), _ptr(W_up, "W_up", _BF16, N * K),
        _ptr(gate, "gate", _F32, N), _ptr(pending, "pending", _F32, T * N),
    )
    outs = (_ptr(out, "out", _F32, T * N), _ptr(mean, "mean", _F32, T * d),
            _ptr(lo, "lo", _F32, T * K), _ptr(r_out, "r_out", _F32, T * N),
            _ptr(rs, "rs", _F32, T * n))
    _check(load().hc_read_ex(h, *args, T, *outs, _stream_ptr(stream)), "hc_read_ex")



def hc_read_q8(h: int, geometry, R, w_norm, Wd_q, Wd_scale, Wu_q, Wu_scale, gate, pending, T: int,
               out, mean, lo, r_out=None, rs=None, stream=None) -> None:
    """Enqueue one read over Q8_0 weights (see include/hc_read.h): quants int8,
    scales as binary16 bits (float16, int16 or uint16 tensors)."""
    n, d, K = geometry
    N = n * d
    args = (
        h,
        _ptr(R, "R", _F32, T * N), _ptr(w_norm, "w_norm", _F32, N),
        _ptr(Wd_q, "Wd_q", _I8, K * N), _ptr(Wd_scale, "Wd_scale", _HALF_BITS, K * N // 32),
        _ptr(Wu_q, "Wu_q", _I8, N * K), _ptr(Wu_scale, "Wu_scale", _HALF_BITS, N * K // 32),
        _ptr(gate, "gate", _F32, N), _ptr(pending, "pending", _F32, T * N), T,
        _ptr(out, "out", _F32, T * N), _ptr(mean, "mean", _F32, T * d), _ptr(lo, "lo", _F32, T * K),
        _ptr(r_out, "r_out", _F32, T * N), _ptr(rs, "rs", _F32, T * n), _stream_ptr(stream),
    )
    _check(load().hc_read_q8(*args), "hc_read_q8")

def hc_q2_0_matvec(Wq, Wscale, x, y, rows: int | None = None, cols: int | None = None,
                   ncols: int | None = None, stream=None) -> None:
    """Enqueue y = W x over Q2_0 weights (see include/hc_q2.h): Wq uint8
    [rows][cols/4], Wscale binary16 bits [rows][cols/64] (float16, int16 or
    uint16), x float32 [ncols][cols], y float32 [ncols][rows].  Sizes come
    from the tensors' shapes unless given (needed for raw pointers)."""
    if rows is None:
        rows = Wq.shape[0]
    if cols is None:
        cols = Wq.shape[-1] * 4
    if ncols is None:
        ncols = x.shape[0] if x.dim() == 2 else 1
    args = (
        _ptr(Wq, "Wq", ("uint8",), rows * cols // 4),
        _ptr(Wscale, "Wscale", _HALF_BITS, rows * (cols // 64)),
        rows, cols,
        _ptr(x, "x", _F32, ncols * cols), ncols,
        _ptr(y, "y", _F32, ncols * rows), _stream_ptr(stream),
    )
    _check(load().hc_q2_0_matvec(*args), "hc_q2_0_matvec")


def hc_q2_0_matvec_batch(products, rows: int, cols: int, ncols: int, stream=None) -> None:
    """Enqueue a batch of Q2_0 products of one shape (see include/hc_q2.h):
    ``products`` is a list of (Wq, Wscale, x, y) tensors (or int pointers)."""
    arr = (hc_q2_0_desc * max(1, len(products)))()
    for j, (Wq, Ws, x, y) in enumerate(products):
        arr[j] = hc_q2_0_desc(
            _ptr(Wq, "Wq", ("uint8",), rows * cols // 4),
            _ptr(Ws, "Wscale", _HALF_BITS, rows * (cols // 64)),
            _ptr(x, "x", _F32, ncols * cols), _ptr(y, "y", _F32, ncols * rows))
    _check(load().hc_q2_0_matvec_batch(arr, len(products), rows, cols, ncols, _stream_ptr(stream)),
           "hc_q2_0_matvec_batch")


def hc_q2_0_matvec_batch_plan(products, rows: int, cols: int, ncols: int) -> list[int]:
    """The launch each product of a batch goes to (host logic; ``products`` as
    for hc_q2_0_matvec_batch, or (Wq, Wscale, x, y) integer addresses)."""
    n = len(products)
    arr = (hc_q2_0_desc * max(1, n))()
    for j, p in enumerate(products):
        arr[j] = hc_q2_0_desc(*[v if isinstance(v, int) else v.data_ptr() for v in p])
    out = (ctypes.c_int * max(1, n))()
    rc = load().hc_q2_0_matvec_batch_plan(arr, n, rows, cols, ncols, out)
    if rc < 0:
        raise HcError(rc, "hc_q2_0_matvec_batch_plan")
    return list(out[:n])


def hc_read(h: int, geometry, R, w_norm, W_down, W_up, gate, pending, T: int,
            out, mean, lo, stream=None) -> None:
    n, d, K = geometry
    N = n * d
    args = (
        _ptr(R, "R", _F32, T * N), _ptr(w_norm, "w_norm", _F32, N),
        _ptr(W_down, "W_down", _BF16, K * N), _ptr(W_up, "W_up", _BF16, N * K),
        _ptr(gate, "gate", _F32, N), _ptr(pending, "pending", _F32, T * N),
    )
    outs = (_ptr(out, "out", _F32, T * N), _ptr(mean, "mean", _F32, T * d),
            _ptr(lo, "lo", _F32, T * K))
    _check(load().hc_read(h, *args, T, *outs, _stream_ptr(stream)), "hc_read")


def hc_read_noalloc(geometry, eps, R, w_norm, W_down, W_up, gate, pending, T: int,
                    out, mean, lo, stream=None) -> None:
    """The read without a handle or any device allocation (T <= HC_NOALLOC_MAX_T).

    For callers that cannot allocate device memory at the point of use; see
    include/hc_read.h.  The first call on a device does a one-time set-up and
    should come before any stream capture; overlapping calls race."""
    n, d, K = geometry
    N = n * d
    args = (
        _ptr(R, "R", _F32, T * N), _ptr(w_norm, "w_norm", _F32, N),
        _ptr(W_down, "W_down", _BF16, K * N), _ptr(W_up, "W_up", _BF16, N * K),
        _ptr(gate, "gate", _F32, N), _ptr(pending, "pending", _F32, T * N),
    )
    outs = (_ptr(out, "out", _F32, T * N), _ptr(mean, "mean", _F32, T * d),
            _ptr(lo, "lo", _F32, T * K))
    _check(load().hc_read_noalloc(n, d, K, eps, *args, T, *outs, _stream_ptr(stream)),
           "hc_read_noalloc")


def hc_read_noalloc_check() -> int:
    """HC_OK or HC_ERR_TIMEOUT for the hc_read_noalloc calls on the current
    device since the last check (synchronises the device, clears the record)."""
    st = load().hc_read_noalloc_check()
    if st not in (HC_OK, HC_ERR_TIMEOUT):
        _check(st, "hc_read_noalloc_check")
    return st


def hc_read_set_wait_limit(h: int, ns: int) -> None:
    """Limit (ns from the kernel's start) of the down kernels' first bulk-copy
    wait for later reads on the handle; 0 restores the default (1 s)."""
    _check(load().hc_read_set_wait_limit(h, ns), "hc_read_set_wait_limit")


def hc_read_set_overlap(h: int, enabled: bool) -> bool:
    """Whether reads on the handle may overlap their predecessor; returns the
    previous setting."""
    st = load().hc_read_set_overlap(h, 1 if enabled else 0)
    if st < 0:
        _check(st, "hc_read_set_overlap")
    return st == 1


def hc_read_down_tiles_bytes(h: int) -> int:
    """Bytes of the tile-ordered copy of a W_down for the handle's geometry."""
    n = load().hc_read_down_tiles_bytes(h)
    if n < 0:
        _check(int(n), "hc_read_down_tiles_bytes")
    return int(n)


def hc_read_register_down_tiles(h: int, geometry, W_down, tiles, stream=None) -> None:
    """Write W_down in tile order into ``tiles`` and register the pair with
    the handle (see include/hc_read.h); returns when the copy is done."""
    n, d, K = geometry
    nbytes = hc_read_down_tiles_bytes(h)
    _check(load().hc_read_register_down_tiles(
        h, _ptr(W_down, "W_down", _BF16, K * n * d), _ptr(tiles, "tiles", _BF16, nbytes // 2),
        _stream_ptr(stream)), "hc_read_register_down_tiles")


def hc_read_forget_down_tiles(h: int, W_down=None) -> None:
    """Drop the handle's tile-ordered copy of W_down (all of them for None)."""
    _check(load().hc_read_forget_down_tiles(h, _ptr(W_down, "W_down", _BF16, None)),
           "hc_read_forget_down_tiles")


def hc_read_up_tiles_bytes(h: int) -> int:
    """Bytes of the tile-ordered copy of a W_up for the handle's geometry (0: none taken)."""
    n = load().hc_read_up_tiles_bytes(h)
    if n < 0:
        _check(int(n), "hc_read_up_tiles_bytes")
    return int(n)


def hc_read_register_up_tiles(h: int, geometry, W_up, tiles, stream=None) -> None:
    """Write W_up in tile order into ``tiles`` and register the pair with the
    handle (see include/hc_read.h); returns when the copy is done."""
    n, d, K = geometry
    nbytes = hc_read_up_tiles_bytes(h)
    _check(load().hc_read_register_up_tiles(
        h, _ptr(W_up, "W_up", _BF16, K * n * d), _ptr(tiles, "tiles", _BF16, nbytes // 2),
        _stream_ptr(stream)), "hc_read_register_up_tiles")


def hc_read_forget_up_tiles(h: int, W_up=None) -> None:
    """Drop the handle's tile-ordered copy of W_up (all of them for None)."""
    _check(load().hc_read_forget_up_tiles(h, _ptr(W_up, "W_up", _BF16, None)), "hc_read_forget_up_tiles")


def _descs(geometry, reads, T: int):
    """hc_read_desc array of a list of reads (tensors checked; ints pass as addresses)."""
    n, d, K = geometry
    N = n * d
    arr = (hc_read_desc * len(reads))()
    for i, r in enumerate(reads):
        pend = r.get("pending", r.get("P"))
        arr[i] = hc_read_desc(
            _ptr(r["R"], "R", _F32, T * N), _ptr(r["w_norm"], "w_norm", _F32, N),
            _ptr(r["W_down"], "W_down", _BF16, K * N), _ptr(r["W_up"], "W_up", _BF16, N * K),
            _ptr(r["gate"], "gate", _F32, N), _ptr(pend, "pending", _F32, T * N),
            _ptr(r["out"], "out", _F32, T * N), _ptr(r["mean"], "mean", _F32, T * d),
            _ptr(r["lo"], "lo", _F32, T * K))
    return arr


def hc_read_batch(h: int, geometry, reads, T: int, stream=None) -> None:
    """Enqueue a list of reads in order (see include/hc_read.h).

    ``reads``: sequence of dicts with keys R, w_norm, W_down, W_up, gate,
    pending (or P; may be None), out, mean, lo.  A read whose R is the
    previous read's out tensor is chained."""
    arr = _descs(geometry, reads, T)
    _check(load().hc_read_batch(h, arr, len(reads), T, _stream_ptr(stream)), "hc_read_batch")


def hc_read_batch_plan(h: int, geometry, reads, T: int) -> int:
    """0: read by read on the caller's stream, 1: the persistent kernel,
    L >= 2: read by read on L internal streams."""
    st = load().hc_read_batch_plan(h, _descs(geometry, reads, T), len(reads), T)
    if st < 0:
        _check(st, "hc_read_batch_plan")
    return st


def hc_read_batch_groups(geometry, reads, T: int) -> list[int]:
    """Group index of every read (host logic; reads may give int addresses)."""
    n, d, K = geometry
    group = (ctypes.c_int * len(reads))()
    st = load().hc_read_batch_groups(_descs(geometry, reads, T), len(reads), n, d, K, T, group)
    if st < 0:
        _check(st, "hc_read_batch_groups")
    return list(group)


def _q8_descs(geometry, reads, T: int):
    """hc_read_q8_desc array of a list of Q8_0 reads (tensors checked; ints pass as addresses)."""
    n, d, K = geometry
    N = n * d
    arr = (hc_read_q8_desc * len(reads))()
    for i, r in enumerate(reads):
        pend = r.get("pending", r.get("P"))
        arr[i] = hc_read_q8_desc(
            _ptr(r["R"], "R", _F32, T * N), _ptr(r["w_norm"], "w_norm", _F32, N),
            _ptr(r["Wd_q"], "Wd_q", _I8, K * N), _ptr(r["Wd_scale"], "Wd_scale", _HALF_BITS, K * N // 32),
            _ptr(r["Wu_q"], "Wu_q", _I8, N * K), _ptr(r["Wu_scale"], "Wu_scale", _HALF_BITS, N * K // 32),
            _ptr(r["gate"], "gate", _F32, N), _ptr(pend, "pending", _F32, T * N),
            _ptr(r["out"], "out", _F32, T * N), _ptr(r["mean"], "mean", _F32, T * d),
            _ptr(r["lo"], "lo", _F32, T * K))
    return arr


def hc_read_batch_q8(h: int, geometry, reads, T: int, stream=None) -> None:
    """Enqueue a list of Q8_0 reads in order (dicts with keys R, w_norm, Wd_q,
    Wd_scale, Wu_q, Wu_scale, gate, pending or P, out, mean, lo)."""
    arr = _q8_descs(geometry, reads, T)
    _check(load().hc_read_batch_q8(h, arr, len(reads), T, _stream_ptr(stream)), "hc_read_batch_q8")


def hc_read_batch_q8_plan(h: int, geometry, reads, T: int) -> int:
    """0: read by read on the caller's stream, L >= 2: on L internal streams."""
    st = load().hc_read_batch_q8_plan(h, _q8_descs(geometry, reads, T), len(reads), T)
    if st < 0:
        _check(st, "hc_read_batch_q8_plan")
    return st


def hc_read_batch_q8_groups(geometry, reads, T: int) -> list[int]:
    """Group index of every Q8_0 read (host logic; reads may give int addresses)."""
    n, d, K = geometry
    group = (ctypes.c_int * len(reads))()
    st = load().hc_read_batch_q8_groups(_q8_descs(geometry, reads, T), len(reads), n, d, K, T, group)
    if st < 0:
        _check(st, "hc_read_batch_q8_groups")
    return list(group)


def hc_read_batch_persistent(h: int, T: int) -> bool:
    """Whether batches of T-token reads run as the persistent kernel."""
    st = load().hc_read_batch_persistent(h, T)
    if st < 0:
        _check(st, "hc_read_batch_persistent")
    return st == 1


def hc_read_check(h: int) -> int:
    """HC_OK or HC_ERR_TIMEOUT (synchronises the device)."""
    st = load().hc_read_check(h)
    if st not in (HC_OK, HC_ERR_TIMEOUT):
        _check(st, "hc_read_check")
    return st


def hc_read_error_word(h: int) -> int:
    """The raw error word (synchronises the device); bits in include/hc_read.h."""
    w = int(load().hc_read_error_word(h))
    if w < 0:
        _check(w, "hc_read_error_word")
    return w


def hc_read_reset(h: int, stream=None) -> None:
    _check(load().hc_read_reset(h, _stream_ptr(stream)), "hc_read_reset")


def hc_read_destroy(h: int) -> None:
    load().hc_read_destroy(h)


def hc_read_scratch_bytes(h: int) -> int:
    return int(load().hc_read_scratch_bytes(h))


def hc_graph_begin(stream=None) -> None:
    _check(load().hc_graph_begin(_stream_ptr(stream)), "hc_graph_begin")


def hc_graph_end(stream=None) -> int:
    g = _vp()
    _check(load().hc_graph_end(_stream_ptr(stream), ctypes.byref(g)), "hc_graph_end")
    return g.value


def hc_graph_launch(graph: int, stream=None) -> None:
    _check(load().hc_graph_launch(graph, _stream_ptr(stream)), "hc_graph_launch")


def hc_graph_destroy(graph: int) -> None:
    load().hc_graph_destroy(graph)


class Read:
    """Owning wrapper of one handle for geometry (n, d, K)."""

    def __init__(self, n: int, d: int, K: int, T_max: int, eps: float = 1e-6, device: int = 0):
        self.geometry = (n, d, K)
        self.T_max = T_max
        self.eps = eps
        self.h = hc_read_create(n, d, K, T_max, eps, device)

    def q8(self, R, w_norm, Wd_q, Wd_scale, Wu_q, Wu_scale, gate, pending, T, out, mean, lo,
           r_out=None, rs=None, stream=None) -> None:
        """One read over Q8_0 weights (hc_read_q8)."""
        hc_read_q8(self.h, self.geometry, R, w_norm, Wd_q, Wd_scale, Wu_q, Wu_scale, gate, pending, T,
                   out, mean, lo, r_out, rs, stream)

    def __call__(self, R, w_norm, W_down, W_up, gate, pending, T, out, mean, lo,
                 r_out=None, rs=None, stream=None) -> None:
        hc_read_ex(self.h, self.geometry, R, w_norm, W_down, W_up, gate, pending, T,
                   out, mean, lo, r_out, rs, stream)

    def batch(self, reads, T: int, stream=None) -> None:
        """Enqueue a list of reads (dicts, see hc_read_batch) in order."""
        hc_read_batch(self.h, self.geometry, reads, T, stream)

    def batch_q8(self, reads, T: int, stream=None) -> None:
        """Enqueue a list of Q8_0 reads (dicts, see hc_read_batch_q8) in order."""
        hc_read_batch_q8(self.h, self.geometry, reads, T, stream)

    def batch_q8_plan(self, reads, T: int) -> int:
        return hc_read_batch_q8_plan(self.h, self.geometry, reads, T)

    def batch_persistent(self, T: int) -> bool:
        return hc_read_batch_persistent(self.h, T)

    def batch_plan(self, reads, T: int) -> int:
        return hc_read_batch_plan(self.h, self.geometry, reads, T)

    def set_batch_lanes(self, lanes: int) -> int:
        """Most internal streams a batch may use (0/1: the caller's stream only)."""
        st = load().hc_read_set_batch_lanes(self.h, lanes)
        if st < 0:
            _check(st, "hc_read_set_batch_lanes")
        return st

    def check(self) -> int:
        return hc_read_check(self.h)

    def set_wait_limit(self, ns: int) -> None:
        hc_read_set_wait_limit(self.h, ns)

    def set_overlap(self, enabled: bool) -> bool:
        return hc_read_set_overlap(self.h, enabled)

    def down_tiles(self, W_down, stream=None):
        """A tile-ordered copy of W_down, registered with this handle: later
        reads with this W_down take their down weights from it (bit-identical
        results).  The returned tensor must stay alive while registered."""
        import torch
        tiles = torch.empty(hc_read_down_tiles_bytes(self.h) // 2, dtype=torch.int16, device=W_down.device)
        hc_read_register_down_tiles(self.h, self.geometry, W_down, tiles, stream)
        return tiles

    def forget_down_tiles(self, W_down=None) -> None:
        hc_read_forget_down_tiles(self.h, W_down)

    def up_tiles(self, W_up, stream=None):
        """A tile-ordered copy of W_up, registered with this handle (None at a
        geometry where no kernel takes one).  Keep the tensor alive while
        registered."""
        import torch
        nbytes = hc_read_up_tiles_bytes(self.h)
        if nbytes == 0:
            return None
        tiles = torch.empty(nbytes // 2, dtype=torch.int16, device=W_up.device)
        hc_read_register_up_tiles(self.h, self.geometry, W_up, tiles, stream)
        return tiles

    def forget_up_tiles(self, W_up=None) -> None:
        hc_read_forget_up_tiles(self.h, W_up)

    def error_word(self) -> int:
        return hc_read_error_word(self.h)

    def reset(self, stream=None) -> None:
        hc_read_reset(self.h, stream)

    def close(self) -> None:
        if self.h:
            hc_read_destroy(self.h)
            self.h = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass
