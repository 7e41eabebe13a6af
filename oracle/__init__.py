"""Float64 CPU oracle for the differential-attention head forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library never loads it, and it imports nothing from the product
package.

The arithmetic lives in ``diffattn_oracle.c`` (plain C, IEEE float64, one query
row at a time with both softmax maps materialised).  This module only compiles
that file with gcc and marshals numpy arrays into it.  Source of the method:
"Differential Transformer" (Ultralytics glossary), section "How differential
attention works": ``out = (softmax(Q1 K1^T / sqrt(d)) - lambda *
softmax(Q2 K2^T / sqrt(d))) V`` with V of width 2d, then a per-head
normalisation and a ``(1 - lambda_init)`` scale,
``lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1))``.

Every function here is pinned by tests in ``tests/test_oracle.py`` against
facts the page and mathematics fix (the page's worked example, the 1 - lambda
row-sum invariant, reductions to ordinary softmax attention and to
``torch.nn.functional.rms_norm``, brute force on tiny inputs, closed forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "diffattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, no fast-math) into ``out``."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", "-o", out + ".tmp", src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _declare(lib):
    d, i, i64, p = ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
    lib.oracle_lambda_init.restype = d
    lib.oracle_lambda_init.argtypes = [i]
    lib.oracle_max_threads.restype = i
    lib.oracle_max_threads.argtypes = [i]
    lib.oracle_fwd.restype = i
    lib.oracle_fwd.argtypes = [i, i, i64, i, p, p, p, p, p, p, i, i, p, d, d, p, i]
    lib.oracle_fwd_rows.restype = i
    lib.oracle_fwd_rows.argtypes = [i, i, i64, i, p, p, p, p, p, p, i, i, p, d, d,
                                    i64, p, p, p, i]
    lib.oracle_fwd_kv_rows.restype = i
    lib.oracle_fwd_kv_rows.argtypes = [i, i, i64, i64, i, p, p, p, p, p, p, i, i, p, d, d,
                                       i64, p, p, p, i]
    lib.oracle_bwd.restype = i
    lib.oracle_bwd.argtypes = [i, i, i64, i, p, p, p, p, p, p, i, i, p, d, d, p, p, p, p, p, p,
                               p, p, i]
    lib.oracle_diff_map.restype = i
    lib.oracle_diff_map.argtypes = [i64, i, p, p, p, p, d, i, p]
    lib.oracle_groupnorm.restype = i
    lib.oracle_groupnorm.argtypes = [i64, i, i, p, p, p, d, d, p]
    lib.oracle_headnorm.restype = i
    lib.oracle_headnorm.argtypes = [i64, i, i, p, p, p, d, d, p]
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def lambda_init(layer: int, lib=None) -> float:
    """lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1)), layers numbered from 1."""
    return float((lib or load()).oracle_lambda_init(int(layer)))


def max_threads(nthreads: int = 0, lib=None) -> int:
    return int((lib or load()).oracle_max_threads(int(nthreads)))


def _check_shapes(q1, k1, q2, k2, v):
    if q1.ndim != 4:
        raise ValueError("q1 must be [B, H, N, d]")
    B, H, N, d = q1.shape
    for t in (k1, q2, k2):
        if t.shape != (B, H, N, d):
            raise ValueError("q1, k1, q2, k2 must share shape [B, H, N, d]")
    if v.shape != (B, H, N, 2 * d):
        raise ValueError("v must be [B, H, N, 2d]")
    return B, H, N, d


def fwd(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: bool,
        w=None, eps: float = 1e-5, lambda_init_value: float = 0.0,
        nthreads: int = 0, lib=None) -> np.ndarray:
    """Differential-attention head forward for every (b, h, i), float64.

    q1, k1, q2, k2: [B, H, N, d]; v: [B, H, N, 2d]; lam: [H];
    w: [H, 2d] or None (ones).  Returns out [B, H, N, 2d].
    """
    q1, k1, q2, k2, v = map(_f64, (q1, k1, q2, k2, v))
    B, H, N, d = _check_shapes(q1, k1, q2, k2, v)
    lam = _f64(lam).reshape(H)
    wv = None if w is None else _f64(w).reshape(H, 2 * d)
    out = np.zeros((B, H, N, 2 * d), dtype=np.float64)
    rc = (lib or load()).oracle_fwd(B, H, N, d, _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2),
                                    _ptr(v), _ptr(lam), int(bool(causal)), int(headnorm),
                                    _ptr(wv), float(eps), float(lambda_init_value), _ptr(out),
                                    int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_fwd failed with code {rc}")
    return out


def fwd_rows(q1, k1, q2, k2, v, lam, bh_idx, row_idx, *, causal: bool, headnorm: bool,
             w=None, eps: float = 1e-5, lambda_init_value: float = 0.0,
             nthreads: int = 0, lib=None) -> np.ndarray:
    """Output rows for selected (flat head index b*H + h, query row) pairs.

    Returns [R, 2d] float64, identical arithmetic to :func:`fwd`.
    """
    q1, k1, q2, k2, v = map(_f64, (q1, k1, q2, k2, v))
    B, H, N, d = _check_shapes(q1, k1, q2, k2, v)
    lam = _f64(lam).reshape(H)
    wv = None if w is None else _f64(w).reshape(H, 2 * d)
    bh = np.ascontiguousarray(np.asarray(bh_idx, dtype=np.int64).reshape(-1))
    ri = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64).reshape(-1))
    if bh.shape != ri.shape:
        raise ValueError("bh_idx and row_idx must have the same length")
    out = np.zeros((bh.size, 2 * d), dtype=np.float64)
    rc = (lib or load()).oracle_fwd_rows(B, H, N, d, _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2),
                                         _ptr(v), _ptr(lam), int(bool(causal)),
                                         int(headnorm), _ptr(wv), float(eps),
                                         float(lambda_init_value), bh.size, _ptr(bh), _ptr(ri),
                                         _ptr(out), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_fwd_rows failed with code {rc}")
    return out


def fwd_kv(q1, k1, q2, k2, v, lam, *, causal: bool, headnorm: bool, bh_idx=None,
           row_idx=None, w=None, eps: float = 1e-5, lambda_init_value: float = 0.0,
           nthreads: int = 0, lib=None) -> np.ndarray:
    """Key/value-cache form: Nq queries against Nkv keys of the same head.

    q1, q2: [B, H, Nq, d]; k1, k2: [B, H, Nkv, d]; v: [B, H, Nkv, 2d].  Query i is
    at sequence position Nkv - Nq + i (causal: sees keys j <= Nkv - Nq + i).
    Returns [B, H, Nq, 2d], or [R, 2d] for the selected (b*H + h, query row) pairs
    when bh_idx / row_idx are given.
    """
    q1, k1, q2, k2, v = map(_f64, (q1, k1, q2, k2, v))
    if q1.ndim != 4 or k1.ndim != 4:
        raise ValueError("q and k must be [B, H, N, d]")
    B, H, Nq, d = q1.shape
    Nkv = k1.shape[2]
    if q2.shape != q1.shape or k1.shape != (B, H, Nkv, d) or k2.shape != k1.shape:
        raise ValueError("q1, q2 must be [B, H, Nq, d] and k1, k2 [B, H, Nkv, d]")
    if v.shape != (B, H, Nkv, 2 * d):
        raise ValueError("v must be [B, H, Nkv, 2d]")
    lam = _f64(lam).reshape(H)
    wv = None if w is None else _f64(w).reshape(H, 2 * d)
    if bh_idx is None:
        bh = ri = None
        nrows = -1
        out = np.zeros((B, H, Nq, 2 * d), dtype=np.float64)
    else:
        bh = np.ascontiguousarray(np.asarray(bh_idx, dtype=np.int64).reshape(-1))
        ri = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64).reshape(-1))
        if bh.shape != ri.shape:
            raise ValueError("bh_idx and row_idx must have the same length")
        nrows = bh.size
        out = np.zeros((nrows, 2 * d), dtype=np.float64)
    rc = (lib or load()).oracle_fwd_kv_rows(B, H, Nq, Nkv, d, _ptr(q1), _ptr(k1), _ptr(q2),
                                            _ptr(k2), _ptr(v), _ptr(lam), int(bool(causal)),
                                            int(headnorm), _ptr(wv), float(eps),
                                            float(lambda_init_value), nrows, _ptr(bh),
                                            _ptr(ri), _ptr(out), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_fwd_kv_rows failed with code {rc}")
    return out


def bwd(q1, k1, q2, k2, v, lam, dy, *, causal: bool, headnorm: bool, w=None,
        eps: float = 1e-5, lambda_init_value: float = 0.0, nthreads: int = 0, lib=None):
    """Gradients of sum(y * dy) for the head forward, float64.

    Returns dict with dq1, dk1, dq2, dk2 [B, H, N, d], dv [B, H, N, 2d], dlam [H]
    and dw [H, 2d] (zeros without the norm).
    """
    q1, k1, q2, k2, v, dy = map(_f64, (q1, k1, q2, k2, v, dy))
    B, H, N, d = _check_shapes(q1, k1, q2, k2, v)
    if dy.shape != v.shape:
        raise ValueError("dy must be [B, H, N, 2d]")
    lam = _f64(lam).reshape(H)
    wv = None if w is None else _f64(w).reshape(H, 2 * d)
    g = {k: np.zeros((B, H, N, d)) for k in ("dq1", "dk1", "dq2", "dk2")}
    g["dv"] = np.zeros((B, H, N, 2 * d))
    g["dlam"] = np.zeros(H)
    g["dw"] = np.zeros((H, 2 * d))
    rc = (lib or load()).oracle_bwd(B, H, N, d, _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v),
                                    _ptr(lam), int(bool(causal)), int(headnorm), _ptr(wv),
                                    float(eps), float(lambda_init_value), _ptr(dy),
                                    _ptr(g["dq1"]), _ptr(g["dk1"]), _ptr(g["dq2"]),
                                    _ptr(g["dk2"]), _ptr(g["dv"]), _ptr(g["dlam"]),
                                    _ptr(g["dw"]), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_bwd failed with code {rc}")
    return g


def diff_map(q1, k1, q2, k2, lam: float, *, causal: bool, lib=None) -> np.ndarray:
    """The differential map map1 - lambda * map2 of one head, [N, N]."""
    q1, k1, q2, k2 = map(_f64, (q1, k1, q2, k2))
    N, d = q1.shape
    out = np.zeros((N, N), dtype=np.float64)
    rc = (lib or load()).oracle_diff_map(N, d, _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2),
                                         float(lam), int(bool(causal)), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_diff_map failed with code {rc}")
    return out


def headnorm(x, h_idx, w=None, *, H: int, eps: float, lambda_init_value: float,
             lib=None) -> np.ndarray:
    """Per-head RMS normalisation of rows x[R, dv] (head h_idx[r]), times (1 - lambda_init)."""
    x = _f64(x)
    R, dv = x.shape
    hi = np.ascontiguousarray(np.asarray(h_idx, dtype=np.int64).reshape(R))
    wv = None if w is None else _f64(w).reshape(H, dv)
    y = np.zeros_like(x)
    rc = (lib or load()).oracle_headnorm(R, dv, H, _ptr(x), _ptr(hi), _ptr(wv), float(eps),
                                         float(lambda_init_value), _ptr(y))
    if rc != 0:
        raise RuntimeError(f"oracle_headnorm failed with code {rc}")
    return y


def groupnorm(x, h_idx, w=None, *, H: int, eps: float, lambda_init_value: float,
              lib=None) -> np.ndarray:
    """Per-head group normalisation (mean-subtracting) of rows x[R, dv], times (1 - lambda_init)."""
    x = _f64(x)
    R, dv = x.shape
    hi = np.ascontiguousarray(np.asarray(h_idx, dtype=np.int64).reshape(R))
    wv = None if w is None else _f64(w).reshape(H, dv)
    y = np.zeros_like(x)
    rc = (lib or load()).oracle_groupnorm(R, dv, H, _ptr(x), _ptr(hi), _ptr(wv), float(eps),
                                          float(lambda_init_value), _ptr(y))
    if rc != 0:
        raise RuntimeError(f"oracle_groupnorm failed with code {rc}")
    return y
