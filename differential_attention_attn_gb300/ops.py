"""ctypes binding of libdiffattn (include/diffattn.h): argument marshalling only.

Every computation runs inside the library's CUDA kernels.  PyTorch supplies
device memory and the current stream; this module only checks that tensors
have the layout the C ABI documents, then passes raw pointers.  If the shared
library has not been built, the first call raises; there is no fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdiffattn.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "diffattn.h")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = 0, 1, 2, 3, 4, 5
BF16, F32, E4M3_QK = 0, 1, 2
_DTYPE_CODE = {torch.bfloat16: BF16, torch.float32: F32}


class DiffAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libdiffattn status {status}: {message}")
        self.status = status


class Desc(ctypes.Structure):
    """Mirror of `diffattn_desc` in include/diffattn.h."""
    _fields_ = [
        ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("N", ctypes.c_int64),
        ("d", ctypes.c_int32), ("dtype", ctypes.c_int32), ("causal", ctypes.c_int32),
        ("headnorm", ctypes.c_int32), ("eps", ctypes.c_float), ("lambda_init", ctypes.c_float),
        ("status_dev", ctypes.c_void_p),
    ]


class Strides(ctypes.Structure):
    """Mirror of `diffattn_strides` (element strides of batch, head, row)."""
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("n", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libdiffattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = bind(ctypes.CDLL(path))
        return _lib


@contextlib.contextmanager
def using(lib):
    """Route this module's calls to another bound library (e.g. the
    bounds-checked debug build) for the duration of a `with` block."""
    global _lib
    with _lock:
        prev, _lib = _lib, lib
    try:
        yield lib
    finally:
        with _lock:
            _lib = prev


def bind(lib):
    """Declare the C signatures of include/diffattn.h on a loaded library."""
    vp, fp = ctypes.c_void_p, ctypes.c_void_p
    dp = ctypes.POINTER(Desc)
    lib.diffattn_fwd.restype = ctypes.c_int
    lib.diffattn_fwd.argtypes = [dp, vp, vp, vp, vp, vp, fp, fp, vp, vp]
    lib.diffattn_fwd_kv.restype = ctypes.c_int
    lib.diffattn_fwd_kv.argtypes = [dp, ctypes.c_int64, vp, vp, vp, vp, vp, fp, fp, vp,
                                    ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.diffattn_fwd_kv_plan.restype = ctypes.c_int
    lib.diffattn_fwd_kv_plan.argtypes = [dp, ctypes.c_int64, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.diffattn_fwd_kv_noalloc.restype = ctypes.c_int
    lib.diffattn_fwd_kv_noalloc.argtypes = [dp, ctypes.c_int64, vp, vp, vp, vp, vp, fp, fp,
                                            vp, ctypes.c_int, vp]
    lib.diffattn_train_sizes.restype = ctypes.c_int
    lib.diffattn_train_sizes.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t),
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.diffattn_fwd_train.restype = ctypes.c_int
    lib.diffattn_fwd_train.argtypes = [dp, vp, vp, vp, vp, vp, fp, fp, vp, vp,
                                       ctypes.c_size_t, vp]
    lib.diffattn_bwd.restype = ctypes.c_int
    lib.diffattn_bwd.argtypes = [dp, vp, vp, vp, vp, vp, fp, fp, vp, vp, vp, vp, vp, vp, vp,
                                 fp, fp, vp, ctypes.c_size_t, vp]
    lib.diffattn_fwd_host.restype = ctypes.c_int
    lib.diffattn_fwd_host.argtypes = [dp, vp, vp, vp, vp, vp, fp, fp, vp, vp, ctypes.c_size_t,
                                      vp]
    lib.diffattn_fwd_host_staging_bytes.restype = ctypes.c_int
    lib.diffattn_fwd_host_staging_bytes.argtypes = [dp, ctypes.POINTER(ctypes.c_size_t)]
    lib.diffattn_fwd_strided.restype = ctypes.c_int
    lib.diffattn_fwd_strided.argtypes = [dp, vp, vp, vp, vp, vp, fp, fp, vp,
                                         ctypes.POINTER(Strides), vp]
    lib.diffattn_fwd_train_strided.restype = ctypes.c_int
    lib.diffattn_fwd_train_strided.argtypes = [dp, vp, vp, vp, vp, vp, fp, fp, vp, vp,
                                               ctypes.c_size_t, ctypes.POINTER(Strides), vp]
    lib.diffattn_bwd_strided.restype = ctypes.c_int
    lib.diffattn_bwd_strided.argtypes = [dp, vp, vp, vp, vp, vp, fp, fp, vp, vp, vp, vp, vp, vp,
                                         vp, fp, fp, vp, ctypes.c_size_t,
                                         ctypes.POINTER(Strides), vp]
    lib.diffattn_fwd_kv_strided.restype = ctypes.c_int
    lib.diffattn_fwd_kv_strided.argtypes = [dp, ctypes.c_int64, vp, vp, vp, vp, vp, fp, fp,
                                            vp, ctypes.c_int, vp, ctypes.c_size_t,
                                            ctypes.POINTER(Strides), vp]
    lib.diffattn_selftest_wait.restype = ctypes.c_int
    lib.diffattn_selftest_wait.argtypes = [vp, ctypes.c_int64, vp]
    lib.diffattn_headnorm.restype = ctypes.c_int
    lib.diffattn_headnorm.argtypes = [dp, fp, fp, vp, vp]
    lib.diffattn_lambda_init.restype = ctypes.c_double
    lib.diffattn_lambda_init.argtypes = [ctypes.c_int]
    lib.diffattn_strerror.restype = ctypes.c_char_p
    lib.diffattn_strerror.argtypes = [ctypes.c_int]
    lib.diffattn_version.restype = ctypes.c_int
    lib.diffattn_version.argtypes = []
    return lib


def declared_symbols(header: str = HEADER_PATH) -> list[str]:
    """Names of the functions include/diffattn.h declares."""
    text = open(header).read()
    return sorted(set(re.findall(r"\b(diffattn_[a-z0-9_]+)\s*\(", text)))


def strerror(status: int) -> str:
    return load().diffattn_strerror(int(status)).decode()


def lambda_init(layer: int) -> float:
    """lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1)), computed by the library."""
    return float(load().diffattn_lambda_init(int(layer)))


def _check(status: int):
    if status != OK:
        raise DiffAttnError(status, strerror(status))


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(B, H, N, d, dtype_code, causal, headnorm, eps, lambda_init_value, status=None):
    return Desc(int(B), int(H), int(N), int(d), int(dtype_code), int(bool(causal)),
                int(headnorm), float(eps), float(lambda_init_value),
                None if status is None else status.data_ptr())


def fwd(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: int = 1, norm_w=None,
        eps: float = 1e-5, lambda_init: float = 0.0, out=None, status=None, stream=None,
        raw_status: bool = False):
    """Differential-attention head forward through `diffattn_fwd`.

    q1, k1, q2, k2: [B, H, N, d]; v: [B, H, N, 2d] (all bf16 or all fp32, CUDA,
    contiguous); lam: float32 [H]; norm_w: float32 [H, 2d] or None.  headnorm:
    0 none, 1 (or True) RMS form, 2 mean-subtracting group form.  Returns
    `out` [B, H, N, 2d] (allocated by torch when not given).  With
    raw_status=True the status code is returned instead of raising.
    """
    if q1.dim() != 4:
        raise ValueError("q1 must be [B, H, N, d]")
    B, H, N, d = q1.shape
    dtype = q1.dtype
    if dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, shape in (("k1", k1, (B, H, N, d)), ("q2", q2, (B, H, N, d)),
                           ("k2", k2, (B, H, N, d)), ("v", v, (B, H, N, 2 * d))):
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"{name} must be {shape} {dtype}")
    tensors = [q1, k1, q2, k2, v, lam] + ([norm_w] if norm_w is not None else [])
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=dtype, device=q1.device)
    tensors.append(out)
    for t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    if lam.dtype != torch.float32 or lam.numel() != H:
        raise ValueError("lam must be float32 [H]")
    if norm_w is not None and (norm_w.dtype != torch.float32 or norm_w.numel() != H * 2 * d):
        raise ValueError("norm_w must be float32 [H, 2d]")
    if tuple(out.shape) != (B, H, N, 2 * d) or out.dtype != dtype:
        raise ValueError("out must be [B, H, N, 2d] of the input dtype")
    desc = make_desc(B, H, N, d, _DTYPE_CODE[dtype], causal, headnorm, eps, lambda_init, status)
    st = load().diffattn_fwd(ctypes.byref(desc), _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v),
                             _ptr(lam), _ptr(norm_w), _ptr(out), _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return out


def fwd_host_staging_bytes(B, H, N, d, dtype=torch.bfloat16) -> int:
    """`diffattn_fwd_host_staging_bytes`: device staging bytes `fwd_host` needs."""
    desc = make_desc(B, H, N, d, _DTYPE_CODE[dtype], True, 1, 1e-5, 0.0)
    n = ctypes.c_size_t(0)
    _check(load().diffattn_fwd_host_staging_bytes(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def fwd_host(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: int = 1, norm_w=None,
             eps: float = 1e-5, lambda_init: float = 0.0, out=None, staging=None, status=None,
             stream=None, raw_status: bool = False):
    """`diffattn_fwd_host`: the forward with q1, k1, q2, k2, v and out in host memory.

    q1, k1, q2, k2, v: contiguous CPU tensors (bf16 or fp32; pinned keeps the copies
    asynchronous); lam (float32 [H]) and norm_w stay CUDA tensors; staging: a CUDA
    uint8 tensor of at least fwd_host_staging_bytes(...) bytes (allocated when not
    given).  Returns the CPU `out` [B, H, N, 2d], filled once `stream` reaches the
    end of the call.
    """
    B, H, N, d = q1.shape
    dtype = q1.dtype
    if dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, shape in (("q1", q1, (B, H, N, d)), ("k1", k1, (B, H, N, d)),
                           ("q2", q2, (B, H, N, d)), ("k2", k2, (B, H, N, d)),
                           ("v", v, (B, H, N, 2 * d))):
        if tuple(t.shape) != shape or t.dtype != dtype or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU {shape} {dtype} tensor")
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=dtype).pin_memory()
    if out.is_cuda or not out.is_contiguous() or tuple(out.shape) != (B, H, N, 2 * d):
        raise ValueError("out must be a contiguous CPU [B, H, N, 2d] tensor")
    if not lam.is_cuda or lam.dtype != torch.float32 or lam.numel() != H:
        raise ValueError("lam must be a CUDA float32 [H] tensor")
    need = fwd_host_staging_bytes(B, H, N, d, dtype)
    if staging is None:
        staging = torch.empty(need, dtype=torch.uint8, device=lam.device)
    if not staging.is_cuda or staging.numel() < need:
        raise ValueError(f"staging must be a CUDA uint8 tensor of at least {need} bytes")
    desc = make_desc(B, H, N, d, _DTYPE_CODE[dtype], causal, headnorm, eps, lambda_init, status)
    st = load().diffattn_fwd_host(ctypes.byref(desc), _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2),
                                  _ptr(v), _ptr(lam), _ptr(norm_w), _ptr(out), _ptr(staging),
                                  staging.numel(), _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return out


def fwd_fp8(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: int = 1, norm_w=None,
            eps: float = 1e-5, lambda_init: float = 0.0, out=None, status=None, stream=None,
            raw_status: bool = False):
    """`diffattn_fwd` with DIFFATTN_E4M3_QK: q1, k1, q2, k2 torch.float8_e4m3fn
    [B, H, N, 64]; v bf16 [B, H, N, 128]; returns bf16 out [B, H, N, 128]."""
    B, H, N, d = q1.shape
    for t in (q1, k1, q2, k2):
        if t.dtype != torch.float8_e4m3fn or tuple(t.shape) != (B, H, N, d):
            raise ValueError("q1, k1, q2, k2 must be float8_e4m3fn [B, H, N, d]")
    if v.dtype != torch.bfloat16 or tuple(v.shape) != (B, H, N, 2 * d):
        raise ValueError("v must be bfloat16 [B, H, N, 2d]")
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=torch.bfloat16, device=q1.device)
    _cuda_contig([q1, k1, q2, k2, v, lam, norm_w, out])
    desc = make_desc(B, H, N, d, E4M3_QK, causal, headnorm, eps, lambda_init, status)
    st = load().diffattn_fwd(ctypes.byref(desc), _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v),
                             _ptr(lam), _ptr(norm_w), _ptr(out), _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return out


def fwd_strided(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: int = 1, norm_w=None,
                eps: float = 1e-5, lambda_init: float = 0.0, out=None, status=None,
                stream=None, raw_status: bool = False):
    """`diffattn_fwd_strided`: the bf16 forward on [B, H, N, d]-shaped views of any
    layout whose rows are contiguous (e.g. x.permute(0, 2, 1, 3) of [B, N, H, d]
    storage); `out` may be such a view too (default: a contiguous tensor)."""
    B, H, N, d = q1.shape
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=q1.dtype, device=q1.device)
    ts = [q1, k1, q2, k2, v, out]
    arr = _view_strides(ts, [(B, H, N, d)] * 4 + [(B, H, N, 2 * d)] * 2, q1.dtype)
    _cuda_contig([lam, norm_w])
    desc = make_desc(B, H, N, d, _DTYPE_CODE.get(q1.dtype, -1), causal, headnorm, eps,
                     lambda_init, status)
    st = load().diffattn_fwd_strided(ctypes.byref(desc), _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2),
                                     _ptr(v), _ptr(lam), _ptr(norm_w), _ptr(out), arr,
                                     _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return out


def _view_strides(ts, shapes, dtype):
    """Checks [B, H, rows, width]-shaped CUDA views with contiguous rows and
    returns their (batch, head, row) element strides as a Strides array."""
    for t, shape in zip(ts, shapes):
        if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_cuda:
            raise ValueError(f"expected a CUDA {dtype} tensor of shape {tuple(shape)}")
        if t.stride(-1) != 1:
            raise ValueError("rows must be contiguous (last stride 1)")
    return (Strides * len(ts))(*[Strides(t.stride(0), t.stride(1), t.stride(2)) for t in ts])


def fwd_kv_plan(B, H, N, n_kv, *, causal: bool, splits: int = 0, d: int = 64,
                headnorm: bool = True, raw_status: bool = False):
    """`diffattn_fwd_kv_plan`: (split count that will run, workspace bytes)."""
    desc = make_desc(B, H, N, d, BF16, causal, headnorm, 1e-5, 0.0)
    sp, nb = ctypes.c_int(0), ctypes.c_size_t(0)
    st = load().diffattn_fwd_kv_plan(ctypes.byref(desc), int(n_kv), int(splits),
                                     ctypes.byref(sp), ctypes.byref(nb))
    if raw_status:
        return st, sp.value, nb.value
    _check(st)
    return sp.value, nb.value


def _kv_dtypes(q1):
    """(dtype code, value and output dtype) of a key/value-cache call: bf16
    throughout, or e4m3 queries/keys (DIFFATTN_E4M3_QK) with bf16 values and output."""
    if q1.dtype == torch.float8_e4m3fn:
        return E4M3_QK, torch.bfloat16
    return _DTYPE_CODE.get(q1.dtype, -1), q1.dtype


def fwd_kv(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: bool = True, norm_w=None,
           eps: float = 1e-5, lambda_init: float = 0.0, splits: int = 0, workspace=None,
           out=None, status=None, stream=None, raw_status: bool = False):
    """Forward of Nq queries against Nkv keys through `diffattn_fwd_kv` (d = 64).

    q1, q2: [B, H, Nq, 64]; k1, k2: [B, H, Nkv, 64]; v: [B, H, Nkv, 128]; the
    queries are the last Nq positions.  All bf16, or q1, k1, q2, k2
    float8_e4m3fn with bf16 v (DIFFATTN_E4M3_QK).  splits = 0 lets the library
    choose.  workspace: a CUDA tensor of at least the planned bytes, or None (a
    torch buffer of the planned size is used).  Returns bf16 out [B, H, Nq, 128].
    """
    if q1.dim() != 4 or k1.dim() != 4:
        raise ValueError("q1 and k1 must be [B, H, N, d]")
    B, H, N, d = q1.shape
    n_kv = k1.shape[2]
    code, vdtype = _kv_dtypes(q1)
    for name, t, shape, dt in (("q2", q2, (B, H, N, d), q1.dtype),
                               ("k1", k1, (B, H, n_kv, d), q1.dtype),
                               ("k2", k2, (B, H, n_kv, d), q1.dtype),
                               ("v", v, (B, H, n_kv, 2 * d), vdtype)):
        if tuple(t.shape) != shape or t.dtype != dt:
            raise ValueError(f"{name} must be {shape} {dt}")
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=vdtype, device=q1.device)
    if tuple(out.shape) != (B, H, N, 2 * d) or out.dtype != vdtype:
        raise ValueError(f"out must be [B, H, Nq, 2d] {vdtype}")
    tensors = [q1, k1, q2, k2, v, lam, out] + ([norm_w] if norm_w is not None else [])
    for t in tensors:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    if lam.dtype != torch.float32 or lam.numel() != H:
        raise ValueError("lam must be float32 [H]")
    if norm_w is not None and (norm_w.dtype != torch.float32 or norm_w.numel() != H * 2 * d):
        raise ValueError("norm_w must be float32 [H, 2d]")
    desc = make_desc(B, H, N, d, code, causal, headnorm, eps, lambda_init, status)
    lib = load()
    if workspace is None:
        sp, nb = ctypes.c_int(0), ctypes.c_size_t(0)
        st = lib.diffattn_fwd_kv_plan(ctypes.byref(desc), int(n_kv), int(splits),
                                      ctypes.byref(sp), ctypes.byref(nb))
        if st != OK:
            if raw_status:
                return st
            _check(st)
        if nb.value:
            workspace = torch.empty(nb.value, dtype=torch.uint8, device=q1.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.diffattn_fwd_kv(ctypes.byref(desc), int(n_kv), _ptr(q1), _ptr(k1), _ptr(q2),
                             _ptr(k2), _ptr(v), _ptr(lam), _ptr(norm_w), _ptr(out), int(splits),
                             _ptr(workspace), ws_bytes, _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return out


def fwd_kv_strided(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: bool = True,
                   norm_w=None, eps: float = 1e-5, lambda_init: float = 0.0, splits: int = 0,
                   workspace=None, out=None, status=None, stream=None, raw_status: bool = False):
    """`diffattn_fwd_kv_strided`: `fwd_kv` (bf16, d = 64) on [B, H, rows, width]-shaped
    views of any layout whose rows are contiguous (e.g. a [B, Nkv, H, d] cache seen
    through permute(0, 2, 1, 3)); `out` may be such a view too (default: contiguous)."""
    B, H, N, d = q1.shape
    n_kv = k1.shape[2]
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=q1.dtype, device=q1.device)
    ts = [q1, k1, q2, k2, v, out]
    shapes = [(B, H, N, d), (B, H, n_kv, d), (B, H, N, d), (B, H, n_kv, d),
              (B, H, n_kv, 2 * d), (B, H, N, 2 * d)]
    for t, shape in zip(ts, shapes):
        if tuple(t.shape) != shape or t.dtype != q1.dtype or not t.is_cuda:
            raise ValueError(f"expected a CUDA {q1.dtype} tensor of shape {shape}")
        if t.stride(-1) != 1:
            raise ValueError("rows must be contiguous (last stride 1)")
    _cuda_contig([lam, norm_w])
    arr = (Strides * 6)(*[Strides(t.stride(0), t.stride(1), t.stride(2)) for t in ts])
    desc = make_desc(B, H, N, d, _DTYPE_CODE.get(q1.dtype, -1), causal, headnorm, eps,
                     lambda_init, status)
    lib = load()
    if workspace is None:
        sp, nb = ctypes.c_int(0), ctypes.c_size_t(0)
        st = lib.diffattn_fwd_kv_plan(ctypes.byref(desc), int(n_kv), int(splits),
                                      ctypes.byref(sp), ctypes.byref(nb))
        if st != OK:
            if raw_status:
                return st
            _check(st)
        if nb.value:
            workspace = torch.empty(nb.value, dtype=torch.uint8, device=q1.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.diffattn_fwd_kv_strided(ctypes.byref(desc), int(n_kv), _ptr(q1), _ptr(k1),
                                     _ptr(q2), _ptr(k2), _ptr(v), _ptr(lam), _ptr(norm_w),
                                     _ptr(out), int(splits), _ptr(workspace), ws_bytes, arr,
                                     _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return out


def train_sizes(B, H, N, *, d: int = 64):
    """`diffattn_train_sizes`: (saved-activation bytes, backward workspace bytes)."""
    desc = make_desc(B, H, N, d, BF16, True, True, 1e-5, 0.0)
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().diffattn_train_sizes(ctypes.byref(desc), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def _check_qkv(q1, k1, q2, k2, v):
    if q1.dim() != 4:
        raise ValueError("q1 must be [B, H, N, d]")
    B, H, N, d = q1.shape
    for name, t, shape in (("k1", k1, (B, H, N, d)), ("q2", q2, (B, H, N, d)),
                           ("k2", k2, (B, H, N, d)), ("v", v, (B, H, N, 2 * d))):
        if tuple(t.shape) != shape or t.dtype != q1.dtype:
            raise ValueError(f"{name} must be {shape} {q1.dtype}")
    return B, H, N, d


def _cuda_contig(ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")


def fwd_train(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: bool = True, norm_w=None,
              eps: float = 1e-5, lambda_init: float = 0.0, out=None, saved=None, status=None,
              stream=None):
    """`diffattn_fwd_train`: the forward plus the activations the backward needs.

    Returns (out, saved); `saved` is a uint8 CUDA tensor of train_sizes()[0] bytes.
    """
    B, H, N, d = _check_qkv(q1, k1, q2, k2, v)
    saved_bytes, _ = train_sizes(B, H, N, d=d)
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=q1.dtype, device=q1.device)
    if saved is None:
        saved = torch.empty(saved_bytes, dtype=torch.uint8, device=q1.device)
    _cuda_contig([q1, k1, q2, k2, v, lam, norm_w, out, saved])
    desc = make_desc(B, H, N, d, _DTYPE_CODE.get(q1.dtype, -1), causal, headnorm, eps,
                     lambda_init, status)
    _check(load().diffattn_fwd_train(ctypes.byref(desc), _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2),
                                     _ptr(v), _ptr(lam), _ptr(norm_w), _ptr(out), _ptr(saved),
                                     saved.numel() * saved.element_size(),
                                     _stream_handle(stream)))
    return out, saved


def bwd(q1, k1, q2, k2, v, lam, saved, dy, *, causal: bool, headnorm: bool = True,
        norm_w=None, eps: float = 1e-5, lambda_init: float = 0.0, workspace=None, grads=None,
        status=None, stream=None, raw_status: bool = False):
    """`diffattn_bwd`: gradients of sum(out * dy) given fwd_train's `saved`.

    Returns dict dq1, dk1, dq2, dk2 (bf16 [B, H, N, d]), dv (bf16 [B, H, N, 2d]),
    dlam (fp32 [H]) and dw (fp32 [H, 2d], zeros without the norm).
    """
    B, H, N, d = _check_qkv(q1, k1, q2, k2, v)
    _, ws_bytes = train_sizes(B, H, N, d=d)
    dev = q1.device
    if grads is None:
        grads = {k: torch.empty((B, H, N, d), dtype=q1.dtype, device=dev)
                 for k in ("dq1", "dk1", "dq2", "dk2")}
        grads["dv"] = torch.empty((B, H, N, 2 * d), dtype=q1.dtype, device=dev)
        grads["dlam"] = torch.empty(H, dtype=torch.float32, device=dev)
        grads["dw"] = torch.zeros((H, 2 * d), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _cuda_contig([q1, k1, q2, k2, v, lam, norm_w, saved, dy, workspace, *grads.values()])
    desc = make_desc(B, H, N, d, _DTYPE_CODE.get(q1.dtype, -1), causal, headnorm, eps,
                     lambda_init, status)
    st = load().diffattn_bwd(ctypes.byref(desc), _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v),
                             _ptr(lam), _ptr(norm_w), _ptr(saved), _ptr(dy), _ptr(grads["dq1"]),
                             _ptr(grads["dk1"]), _ptr(grads["dq2"]), _ptr(grads["dk2"]),
                             _ptr(grads["dv"]), _ptr(grads["dlam"]), _ptr(grads["dw"]),
                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return grads


def fwd_train_strided(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: int = 1,
                      norm_w=None, eps: float = 1e-5, lambda_init: float = 0.0, out=None,
                      saved=None, status=None, stream=None):
    """`diffattn_fwd_train_strided`: fwd_train on [B, H, N, d]-shaped views with
    contiguous rows (`out` may be such a view too; default contiguous).
    Returns (out, saved)."""
    B, H, N, d = q1.shape
    saved_bytes, _ = train_sizes(B, H, N, d=d)
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=q1.dtype, device=q1.device)
    if saved is None:
        saved = torch.empty(saved_bytes, dtype=torch.uint8, device=q1.device)
    ts = [q1, k1, q2, k2, v, out]
    arr = _view_strides(ts, [(B, H, N, d)] * 4 + [(B, H, N, 2 * d)] * 2, q1.dtype)
    _cuda_contig([lam, norm_w, saved])
    desc = make_desc(B, H, N, d, _DTYPE_CODE.get(q1.dtype, -1), causal, headnorm, eps,
                     lambda_init, status)
    _check(load().diffattn_fwd_train_strided(ctypes.byref(desc), _ptr(q1), _ptr(k1), _ptr(q2),
                                             _ptr(k2), _ptr(v), _ptr(lam), _ptr(norm_w),
                                             _ptr(out), _ptr(saved),
                                             saved.numel() * saved.element_size(), arr,
                                             _stream_handle(stream)))
    return out, saved


def bwd_strided(q1, k1, q2, k2, v, lam, saved, dy, *, causal: bool, headnorm: int = 1,
                norm_w=None, eps: float = 1e-5, lambda_init: float = 0.0, workspace=None,
                grads=None, status=None, stream=None, raw_status: bool = False):
    """`diffattn_bwd_strided`: bwd on [B, H, N, .]-shaped views with contiguous rows;
    `grads` (dq1, dk1, dq2, dk2, dv views, plus dlam and dw) defaults to contiguous
    tensors.  Returns the grads dict as bwd does."""
    B, H, N, d = q1.shape
    _, ws_bytes = train_sizes(B, H, N, d=d)
    dev = q1.device
    if grads is None:
        grads = {k: torch.empty((B, H, N, d), dtype=q1.dtype, device=dev)
                 for k in ("dq1", "dk1", "dq2", "dk2")}
        grads["dv"] = torch.empty((B, H, N, 2 * d), dtype=q1.dtype, device=dev)
        grads["dlam"] = torch.empty(H, dtype=torch.float32, device=dev)
        grads["dw"] = torch.zeros((H, 2 * d), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ts = [q1, k1, q2, k2, v, dy, grads["dq1"], grads["dk1"], grads["dq2"], grads["dk2"],
          grads["dv"]]
    w = 2 * d
    shapes = [(B, H, N, d)] * 4 + [(B, H, N, w)] * 2 + [(B, H, N, d)] * 4 + [(B, H, N, w)]
    arr = _view_strides(ts, shapes, q1.dtype)
    _cuda_contig([lam, norm_w, saved, workspace, grads["dlam"], grads["dw"]])
    desc = make_desc(B, H, N, d, _DTYPE_CODE.get(q1.dtype, -1), causal, headnorm, eps,
                     lambda_init, status)
    st = load().diffattn_bwd_strided(ctypes.byref(desc), _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2),
                                     _ptr(v), _ptr(lam), _ptr(norm_w), _ptr(saved), _ptr(dy),
                                     _ptr(grads["dq1"]), _ptr(grads["dk1"]), _ptr(grads["dq2"]),
                                     _ptr(grads["dk2"]), _ptr(grads["dv"]), _ptr(grads["dlam"]),
                                     _ptr(grads["dw"]), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), arr,
                                     _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return grads


NOALLOC_SCRATCH_BYTES = 64 << 20


def fwd_kv_noalloc(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: bool = True,
                   norm_w=None, eps: float = 1e-5, lambda_init: float = 0.0, splits: int = 0,
                   out=None, status=None, stream=None, raw_status: bool = False):
    """`diffattn_fwd_kv_noalloc`: fwd_kv on the library's own 64 MiB scratch area.

    Same arguments and result as :func:`fwd_kv` without the workspace.  Calls
    that overlap in time race on the shared scratch; the first call on a device
    must not be inside a CUDA graph capture.
    """
    B, H, N, d = q1.shape
    n_kv = k1.shape[2]
    code, vdtype = _kv_dtypes(q1)
    if out is None:
        out = torch.empty((B, H, N, 2 * d), dtype=vdtype, device=q1.device)
    for t in [q1, k1, q2, k2, v, lam, out] + ([norm_w] if norm_w is not None else []):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    if tuple(k2.shape) != tuple(k1.shape) or tuple(q2.shape) != tuple(q1.shape) or \
            tuple(v.shape) != (B, H, n_kv, 2 * d) or tuple(out.shape) != (B, H, N, 2 * d):
        raise ValueError("q1, q2 [B, H, Nq, d]; k1, k2 [B, H, Nkv, d]; v [B, H, Nkv, 2d]; "
                         "out [B, H, Nq, 2d]")
    desc = make_desc(B, H, N, d, code, causal, headnorm, eps, lambda_init, status)
    st = load().diffattn_fwd_kv_noalloc(ctypes.byref(desc), int(n_kv), _ptr(q1), _ptr(k1),
                                        _ptr(q2), _ptr(k2), _ptr(v), _ptr(lam), _ptr(norm_w),
                                        _ptr(out), int(splits), _stream_handle(stream))
    if raw_status:
        return st
    _check(st)
    return out


def headnorm(x, *, H: int, norm_w=None, eps: float = 1e-5, lambda_init: float = 0.0,
             out_dtype=torch.bfloat16, out=None, stream=None, mode: int = 1):
    """Per-head normalisation through `diffattn_headnorm` (mode 1: RMS; mode 2:
    mean-subtracting group form).

    x: float32 [B, H, N, 2d] CUDA; returns [B, H, N, 2d] in out_dtype.
    """
    if x.dim() != 4 or x.dtype != torch.float32:
        raise ValueError("x must be float32 [B, H, N, 2d]")
    B, Hx, N, dv = x.shape
    if Hx != H or dv % 2:
        raise ValueError("x must be [B, H, N, 2d]")
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    for t in [x, out] + ([norm_w] if norm_w is not None else []):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    desc = make_desc(B, H, N, dv // 2, _DTYPE_CODE[out.dtype], False, mode, eps, lambda_init)
    _check(load().diffattn_headnorm(ctypes.byref(desc), _ptr(x), _ptr(norm_w), _ptr(out),
                                    _stream_handle(stream)))
    return out


def selftest_wait(timeout_ns: int = 50_000_000, stream=None):
    """`diffattn_selftest_wait`: returns (status code, first wait us, second wait us)."""
    st = torch.zeros(3, dtype=torch.int32, device="cuda")
    _check(load().diffattn_selftest_wait(_ptr(st), int(timeout_ns), _stream_handle(stream)))
    torch.cuda.synchronize()
    code, w0, w1 = (int(x) for x in st.cpu())
    return code, w0, w1
