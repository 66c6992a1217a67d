"""Thin ctypes binding over libgemvfuse.so (the C ABI in include/gemvfuse.h).

Argument marshalling only: every computation runs in the library's CUDA kernels.
Arrays are passed as torch CUDA tensors (or raw integer device addresses); the
stream defaults to torch's current CUDA stream.  Importing this module loads the
library and raises ImportError if it has not been built -- there is no fallback.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgemvfuse.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libgemvfuse.so is not built (run __graft_entry__.build()): %s" % LIB_PATH)
_lib = ctypes.CDLL(LIB_PATH)

# enums (include/gemvfuse.h)
F32, F16, Q8_0, Q4_0, Q4_K = 0, 1, 2, 3, 4
EPI_NONE, EPI_SIGMOID, EPI_SILU, EPI_SILU_MUL, EPI_ADD = 0, 1, 2, 3, 4
EW_SIGMOID, EW_SILU, EW_MUL, EW_ADD = 1, 2, 3, 4
OK, ERR_INVALID, ERR_ALIAS, ERR_UNSUPPORTED, ERR_ALIGN, ERR_CUDA, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5, -6
FLAG_PDL, FLAG_NO_SPLIT_K, FLAG_NO_TENSOR_CORES = 1, 2, 4
PATH_NONE, PATH_STREAM, PATH_GENERIC, PATH_TC = 0, 1, 2, 3

_vp, _i64, _i32, _u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32


class GfOpts(ctypes.Structure):
    _fields_ = [("ncols", _i64), ("fwht_signs", _vp), ("fwht_block", _i64), ("nsigns", _i64),
                ("view_ne", _i64 * 4), ("flags", _u32), ("fwht_workspace", _vp),
                ("rms_norm_weight", _vp), ("rms_norm_eps", ctypes.c_float)]


def _sig(name, args, res=_i32):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_gemv_fused = _sig("gemv_fused", [_vp, _i32, _vp, _i64, _i64, _i32, _vp, _vp, _vp])
_gemv_fused_ex = _sig("gemv_fused_ex", [_vp, _i32, _vp, _i64, _i64, _i32, _vp, _vp,
                                        ctypes.POINTER(GfOpts), _vp])
_gemv_glu = _sig("gemv_glu", [_vp, _vp, _i32, _vp, _i64, _i64, _vp, ctypes.POINTER(GfOpts), _vp])
_fwht_signed = _sig("fwht_signed", [_vp, _vp, _vp, _i64, _i64, _i64, _vp])
_gemv_fused_fwht_noalloc = _sig("gemv_fused_fwht_noalloc", [_vp, _i32, _vp, _i64, _i64, _i32, _vp, _vp, _i64,
                                                             _vp, _i64, _i64, _u32, _vp])
NOALLOC_MAX_WORKSPACE_FLOATS = 262144
_elementwise = _sig("gf_elementwise", [_i32, _vp, _vp, _i64, _vp, _i64, _vp])
_dequantize = _sig("gf_dequantize", [_vp, _i32, _i64, _i64, _vp, _vp])
_plan = _sig("gf_plan", [_vp, _i32, _vp, _i64, _i64, _i32, _vp, _vp, ctypes.POINTER(GfOpts),
                         ctypes.POINTER(_i64 * 8)])
_plan_glu = _sig("gf_plan_glu", [_vp, _vp, _i32, _vp, _i64, _i64, _vp, ctypes.POINTER(GfOpts),
                                 ctypes.POINTER(_i64 * 8)])
_device_status = _sig("gf_device_status", [_i32])
_selftest_wait = _sig("gf_selftest_wait_timeout", [_i64, _vp, _vp])
_status_string = _sig("gf_status_string", [_i32], ctypes.c_char_p)
_last_cuda_error = _sig("gf_last_cuda_error", [])
_version = _sig("gf_version", [])
_prepare = _sig("gf_prepare", [_vp, _i32, _vp, _i64, _i64, _i32, _vp, _vp, ctypes.POINTER(GfOpts),
                               ctypes.POINTER(_vp)])
_prepare_glu = _sig("gf_prepare_glu", [_vp, _vp, _i32, _vp, _i64, _i64, _vp, ctypes.POINTER(GfOpts),
                                       ctypes.POINTER(_vp)])
_launch_prepared = _sig("gf_launch_prepared", [ctypes.POINTER(_vp), _i32, _vp])
_free_prepared = _sig("gf_free_prepared", [_vp], None)


class MultiItem(ctypes.Structure):
    _fields_ = [("W", _vp), ("M", _i64), ("epilogue", _i32), ("aux", _vp), ("dst", _vp)]


MULTI_MAX = 4
_gemv_multi = _sig("gemv_multi", [ctypes.POINTER(MultiItem), _i32, _i32, _vp, _i64, ctypes.POINTER(GfOpts), _vp])
_prepare_multi = _sig("gf_prepare_multi", [ctypes.POINTER(MultiItem), _i32, _i32, _vp, _i64,
                                           ctypes.POINTER(GfOpts), ctypes.POINTER(_vp)])
_copy = _sig("gf_copy", [_vp, _vp, _i64, _u32, _vp])
_prepare_copy = _sig("gf_prepare_copy", [_vp, _vp, _i64, _u32, ctypes.POINTER(_vp)])
_graph_create = _sig("gf_graph_create", [ctypes.POINTER(_vp), _i32, ctypes.POINTER(_vp)])
_graph_launch = _sig("gf_graph_launch", [_vp, _vp])
_graph_free = _sig("gf_graph_free", [_vp], None)

#: the raw C functions, for callers that want the status codes themselves
raw = _lib


class GemvFuseError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = "%s: %s" % (what, status_string(status))
        if status == ERR_CUDA:
            msg += " (cudaError %d)" % _last_cuda_error()
        super().__init__(msg)


def status_string(status):
    return _status_string(int(status)).decode()


def version():
    return _version()


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st, what):
    if st != OK:
        raise GemvFuseError(st, what)


def make_opts(ncols=1, fwht_signs=None, fwht_block=0, nsigns=None, view=None, pdl=False, fwht_workspace=None,
              rms_norm_weight=None, rms_norm_eps=0.0, split_k=True, tensor_cores=True):
    o = GfOpts()
    o.ncols = ncols
    o.fwht_signs = _ptr(fwht_signs)
    o.fwht_block = fwht_block
    if nsigns is None:
        nsigns = fwht_block if fwht_signs is not None and isinstance(fwht_signs, int) \
            else (fwht_signs.numel() if fwht_signs is not None else 0)
    o.nsigns = nsigns
    v = list(view or ())
    for i in range(4):
        o.view_ne[i] = v[i] if i < len(v) else 0
    o.flags = (FLAG_PDL if pdl else 0) | (0 if split_k else FLAG_NO_SPLIT_K) | \
        (0 if tensor_cores else FLAG_NO_TENSOR_CORES)
    o.fwht_workspace = _ptr(fwht_workspace)
    o.rms_norm_weight = _ptr(rms_norm_weight)
    o.rms_norm_eps = rms_norm_eps
    return o


def gemv_fused(W, wtype, x, M, K, epilogue, aux, dst, stream=None, check=True):
    st = _gemv_fused(_ptr(W), wtype, _ptr(x), M, K, epilogue, _ptr(aux), _ptr(dst), _stream(stream))
    if check:
        _check(st, "gemv_fused")
    return st


def gemv_fused_ex(W, wtype, x, M, K, epilogue, aux, dst, ncols=1, fwht_signs=None, fwht_block=0,
                  nsigns=None, view=None, pdl=False, fwht_workspace=None, rms_norm_weight=None,
                  rms_norm_eps=0.0, split_k=True, tensor_cores=True, stream=None, check=True):
    o = make_opts(ncols, fwht_signs, fwht_block, nsigns, view, pdl, fwht_workspace, rms_norm_weight,
                  rms_norm_eps, split_k, tensor_cores)
    st = _gemv_fused_ex(_ptr(W), wtype, _ptr(x), M, K, epilogue, _ptr(aux), _ptr(dst),
                        ctypes.byref(o), _stream(stream))
    if check:
        _check(st, "gemv_fused_ex")
    return st


def gemv_glu(W_gate, W_up, wtype, x, M, K, dst, ncols=1, fwht_signs=None, fwht_block=0, nsigns=None,
             view=None, pdl=False, fwht_workspace=None, rms_norm_weight=None, rms_norm_eps=0.0,
             split_k=True, stream=None, check=True):
    """dst = silu(W_gate x') * (W_up x') for each column (see include/gemvfuse.h)."""
    o = make_opts(ncols, fwht_signs, fwht_block, nsigns, view, pdl, fwht_workspace, rms_norm_weight,
                  rms_norm_eps, split_k)
    st = _gemv_glu(_ptr(W_gate), _ptr(W_up), wtype, _ptr(x), M, K, _ptr(dst), ctypes.byref(o), _stream(stream))
    if check:
        _check(st, "gemv_glu")
    return st


class Prepared:
    """A planned call (gf_prepare / gf_prepare_glu): launch() issues its kernels with no
    planning.  The buffers it was prepared with must stay allocated while it is used;
    the handle is released when the object is garbage-collected (or by close())."""

    def __init__(self, handle, keep):
        self._h = _vp(handle)
        self._keep = keep  # the options struct and tensors the handle points into

    @property
    def handle(self):
        return self._h

    def launch(self, stream=None, check=True):
        return launch_prepared([self], stream=stream, check=check)

    def close(self):
        if self._h is not None and self._h.value:
            _free_prepared(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def prepare(W, wtype, x, M, K, epilogue, aux, dst, ncols=1, fwht_signs=None, fwht_block=0, nsigns=None,
            view=None, pdl=False, fwht_workspace=None, rms_norm_weight=None, rms_norm_eps=0.0, split_k=True,
            tensor_cores=True, check=True):
    """gf_prepare: the call gemv_fused_ex(...) would make, planned once (see Prepared)."""
    o = make_opts(ncols, fwht_signs, fwht_block, nsigns, view, pdl, fwht_workspace, rms_norm_weight,
                  rms_norm_eps, split_k, tensor_cores)
    h = _vp()
    st = _prepare(_ptr(W), wtype, _ptr(x), M, K, epilogue, _ptr(aux), _ptr(dst), ctypes.byref(o), ctypes.byref(h))
    if check:
        _check(st, "gf_prepare")
    return Prepared(h.value, (W, x, aux, dst, fwht_signs, fwht_workspace, rms_norm_weight)) if st == OK else st


def prepare_glu(W_gate, W_up, wtype, x, M, K, dst, ncols=1, fwht_signs=None, fwht_block=0, nsigns=None,
                view=None, pdl=False, fwht_workspace=None, rms_norm_weight=None, rms_norm_eps=0.0, split_k=True,
                check=True):
    """gf_prepare_glu: the call gemv_glu(...) would make, planned once (see Prepared)."""
    o = make_opts(ncols, fwht_signs, fwht_block, nsigns, view, pdl, fwht_workspace, rms_norm_weight,
                  rms_norm_eps, split_k)
    h = _vp()
    st = _prepare_glu(_ptr(W_gate), _ptr(W_up), wtype, _ptr(x), M, K, _ptr(dst), ctypes.byref(o), ctypes.byref(h))
    if check:
        _check(st, "gf_prepare_glu")
    return Prepared(h.value, (W_gate, W_up, x, dst, fwht_signs, fwht_workspace, rms_norm_weight)) \
        if st == OK else st


def launch_prepared(calls, stream=None, check=True):
    """gf_launch_prepared: issue the prepared calls' kernels in order on `stream`."""
    arr = (_vp * max(1, len(calls)))(*[c.handle.value if isinstance(c, Prepared) else c for c in calls])
    st = _launch_prepared(arr, len(calls), _stream(stream))
    if check:
        _check(st, "gf_launch_prepared")
    return st


class Graph:
    """gf_graph_create: prepared calls recorded as one CUDA graph; launch() replays it."""

    def __init__(self, calls, check=True):
        arr = (_vp * max(1, len(calls)))(*[c.handle.value if isinstance(c, Prepared) else c for c in calls])
        h = _vp()
        st = _graph_create(arr, len(calls), ctypes.byref(h))
        if check:
            _check(st, "gf_graph_create")
        self.status = st
        self._h = h if st == OK else None
        self._keep = list(calls)

    def launch(self, stream=None, check=True):
        st = _graph_launch(self._h, _stream(stream))
        if check:
            _check(st, "gf_graph_launch")
        return st

    def close(self):
        if self._h is not None and self._h.value:
            _graph_free(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _multi_items(items):
    arr = (MultiItem * max(1, len(items)))()
    for i, (W, M, epi, aux, dst) in enumerate(items):
        arr[i].W, arr[i].M, arr[i].epilogue, arr[i].aux, arr[i].dst = _ptr(W), M, epi, _ptr(aux), _ptr(dst)
    return arr


def gemv_multi(items, wtype, x, K, ncols=1, fwht_signs=None, fwht_block=0, nsigns=None, pdl=False,
               fwht_workspace=None, rms_norm_weight=None, rms_norm_eps=0.0, stream=None, check=True):
    """dst_i = epilogue_i(W_i x') for items [(W, M, epilogue, aux, dst), ...] sharing x, in one
    pass (see include/gemvfuse.h)."""
    o = make_opts(ncols, fwht_signs, fwht_block, nsigns, None, pdl, fwht_workspace, rms_norm_weight, rms_norm_eps)
    st = _gemv_multi(_multi_items(items), len(items), wtype, _ptr(x), K, ctypes.byref(o), _stream(stream))
    if check:
        _check(st, "gemv_multi")
    return st


def prepare_multi(items, wtype, x, K, ncols=1, fwht_signs=None, fwht_block=0, nsigns=None, pdl=False,
                  fwht_workspace=None, rms_norm_weight=None, rms_norm_eps=0.0, check=True):
    """gf_prepare_multi: the call gemv_multi(...) would make, planned once (see Prepared)."""
    o = make_opts(ncols, fwht_signs, fwht_block, nsigns, None, pdl, fwht_workspace, rms_norm_weight, rms_norm_eps)
    h = _vp()
    st = _prepare_multi(_multi_items(items), len(items), wtype, _ptr(x), K, ctypes.byref(o), ctypes.byref(h))
    if check:
        _check(st, "gf_prepare_multi")
    return Prepared(h.value, (items, x, fwht_signs, fwht_workspace, rms_norm_weight)) if st == OK else st


def gemv_fused_fwht_noalloc(W, wtype, x, M, K, epilogue, aux, dst, ncols, fwht_signs, fwht_block, nsigns=None,
                            pdl=False, stream=None, check=True):
    """gemv_fused_ex with the signed-FWHT prologue, its workspace taken from the library's
    static device array (for callers that cannot allocate one); see include/gemvfuse.h."""
    if nsigns is None:
        nsigns = fwht_block if isinstance(fwht_signs, int) else fwht_signs.numel()
    st = _gemv_fused_fwht_noalloc(_ptr(W), wtype, _ptr(x), M, K, epilogue, _ptr(aux), _ptr(dst), ncols,
                                  _ptr(fwht_signs), fwht_block, nsigns, FLAG_PDL if pdl else 0, _stream(stream))
    if check:
        _check(st, "gemv_fused_fwht_noalloc")
    return st


def fwht_signed(x, signs, dst, n, block, nsigns=None, stream=None, check=True):
    if nsigns is None:
        nsigns = 0 if signs is None else (block if isinstance(signs, int) else signs.numel())
    st = _fwht_signed(_ptr(x), _ptr(signs), _ptr(dst), n, block, nsigns, _stream(stream))
    if check:
        _check(st, "fwht_signed")
    return st


def elementwise(op, a, b, dst, n, nb=None, stream=None, check=True):
    if nb is None:
        nb = n if b is None or isinstance(b, int) else b.numel()
    st = _elementwise(op, _ptr(a), _ptr(b), nb, _ptr(dst), n, _stream(stream))
    if check:
        _check(st, "gf_elementwise")
    return st


def dequantize(W, wtype, M, K, out, stream=None, check=True):
    st = _dequantize(_ptr(W), wtype, M, K, _ptr(out), _stream(stream))
    if check:
        _check(st, "gf_dequantize")
    return st


def plan(W, wtype, x, M, K, epilogue, aux, dst, **opts):
    """(path, info) without launching: path 1 = TMA-streamed, 2 = generic, <0 = error."""
    o = make_opts(**opts)
    info = (_i64 * 8)()
    path = _plan(_ptr(W), wtype, _ptr(x), M, K, epilogue, _ptr(aux), _ptr(dst), ctypes.byref(o),
                 ctypes.byref(info))
    return path, dict(zip(_PLAN_KEYS, list(info)))


_PLAN_KEYS = ("grid", "threads", "stage_rows", "stages", "k_chunk", "smem", "row_chunk", "split")


def plan_glu(W_gate, W_up, wtype, x, M, K, dst, **opts):
    """plan() for gemv_glu."""
    o = make_opts(**opts)
    info = (_i64 * 8)()
    path = _plan_glu(_ptr(W_gate), _ptr(W_up), wtype, _ptr(x), M, K, _ptr(dst), ctypes.byref(o),
                     ctypes.byref(info))
    return path, dict(zip(_PLAN_KEYS, list(info)))


def selftest_wait_timeout(limit_us, out, stream=None, check=True):
    """Run the bounded-wait failure self-test (see include/gemvfuse.h); out: device int32[4]."""
    st = _selftest_wait(int(limit_us), _ptr(out), _stream(stream))
    if check:
        _check(st, "gf_selftest_wait_timeout")
    return st


_repair_count = _sig("gf_repair_count", [_i32], _i64)


def repair_count(reset=False):
    """gf_repair_count: row chunks recomputed in fp32 by the integer-path kernels."""
    return _repair_count(1 if reset else 0)


def device_status(reset=False):
    return _device_status(1 if reset else 0)


def last_cuda_error():
    return _last_cuda_error()


def copy(dst, src, nbytes, pdl=False, stream=None, check=True):
    """gf_copy: nbytes from src to dst by a kernel (device memory, or host memory the
    device addresses, e.g. a pinned tensor)."""
    st = _copy(_ptr(dst), _ptr(src), nbytes, FLAG_PDL if pdl else 0, _stream(stream))
    if check:
        _check(st, "gf_copy")
    return st


def prepare_copy(dst, src, nbytes, pdl=False, check=True):
    """gf_prepare_copy: the copy gf_copy would launch, as a prepared call (a graph may hold
    it beside the GEMVs)."""
    h = _vp()
    st = _prepare_copy(_ptr(dst), _ptr(src), nbytes, FLAG_PDL if pdl else 0, ctypes.byref(h))
    if check:
        _check(st, "gf_prepare_copy")
    return Prepared(h.value, (dst, src)) if st == OK else st
