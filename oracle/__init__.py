"""CSA2 oracle: a plain fp64 CPU restatement of one compressed-sparse-attention layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA library and
its Python binding never call it, and it shares no code with them.

The arithmetic lives in ``csa2_oracle.cpp`` (compiled by :func:`build` with g++ and
OpenMP); this module only marshals numpy arrays.  Every function cites the page section it
restates in the C++ source.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "csa2_oracle.cpp"
_LIB_PATH = _HERE / "_build" / "libcsa2_oracle.so"

D, DR, DI, HI, H, WIN, TOPK = 512, 64, 128, 32, 64, 128, 512


def build(force: bool = False) -> Path:
    """Compile the oracle into ``oracle/_build/libcsa2_oracle.so`` (g++, -O2, OpenMP)."""
    _LIB_PATH.parent.mkdir(parents=True, exist_ok=True)
    if not force and _LIB_PATH.exists() and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB_PATH
    tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", str(_SRC), "-o", str(tmp)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        _lib = C.CDLL(str(build()))
        _declare(_lib)
    return _lib


def _declare(L: C.CDLL) -> None:
    p = C.c_void_p
    i64, i32, f64 = C.c_int64, C.c_int, C.c_double
    L.csa2o_e2m1_value.restype = f64
    L.csa2o_e2m1_value.argtypes = [i32]
    L.csa2o_e2m1_encode.restype = i32
    L.csa2o_e2m1_encode.argtypes = [f64]
    L.csa2o_e4m3_value.restype = f64
    L.csa2o_e4m3_value.argtypes = [i32]
    L.csa2o_e4m3_encode.restype = i32
    L.csa2o_e4m3_encode.argtypes = [f64]
    L.csa2o_e4m3_encode_many.argtypes = [p, i64, p]
    L.csa2o_mx_quantize.argtypes = [p, i64, i32, p, p]
    L.csa2o_mx_dequantize.argtypes = [p, p, i64, i32, p]
    L.csa2o_rmsnorm.argtypes = [p, p, i32, f64, p]
    L.csa2o_rope.argtypes = [p, i32, f64, f64, i32]
    L.csa2o_write_seq.restype = i64
    L.csa2o_write_seq.argtypes = [i32, i32, i64, p, p, p, p, p, p, p, f64, f64, p, p, p, p, i64,
                                  p, p, p, p, p, p, p, p]
    L.csa2o_index_scores.restype = i32
    L.csa2o_index_scores.argtypes = [i32, i32, p, p, p, p, p, i64, p, i64, p, p]
    L.csa2o_topk.restype = i32
    L.csa2o_topk.argtypes = [i32, p, p, i64, i32, p, p, p]
    L.csa2o_hsi_pool.restype = i32
    L.csa2o_hsi_pool.argtypes = [i32, p, p, i64, p]
    L.csa2o_reindex_topk.restype = i32
    L.csa2o_reindex_topk.argtypes = [i32, p, p, i64, p, i32, p]
    L.csa2o_attend.restype = i32
    L.csa2o_attend.argtypes = [i32, p, p, p, p, p, i64, p, i64, i64, p, f64, i64, p, p, p]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ codecs
def e2m1_value(code: int) -> float:
    return lib().csa2o_e2m1_value(int(code))


def e2m1_encode(x: float) -> int:
    return lib().csa2o_e2m1_encode(float(x))


def e4m3_value(code: int) -> float:
    return lib().csa2o_e4m3_value(int(code))


def e4m3_encode(x) -> np.ndarray:
    x = _c(np.atleast_1d(x), np.float64)
    out = np.empty(x.shape, np.uint8)
    lib().csa2o_e4m3_encode_many(_ptr(x), x.size, _ptr(out))
    return out


def mx_quantize(v: np.ndarray):
    """Rows of n (multiple of 32) values -> (codes [rows, n/2] u8, scales [rows, n/32] u8)."""
    v = _c(v, np.float64)
    n = v.shape[-1]
    rows = v.size // n
    codes = np.empty(v.shape[:-1] + (n // 2,), np.uint8)
    scales = np.empty(v.shape[:-1] + (n // 32,), np.uint8)
    lib().csa2o_mx_quantize(_ptr(v), rows, n, _ptr(codes), _ptr(scales))
    return codes, scales


def mx_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    n = codes.shape[-1] * 2
    rows = codes.size // (n // 2)
    out = np.empty(codes.shape[:-1] + (n,), np.float64)
    lib().csa2o_mx_dequantize(_ptr(codes), _ptr(scales), rows, n, _ptr(out))
    return out


def rmsnorm(x, gamma, eps=1e-20):
    x = _c(x, np.float64)
    g = _c(gamma, np.float32)
    y = np.empty_like(x)
    lib().csa2o_rmsnorm(_ptr(x), _ptr(g), x.size, eps, _ptr(y))
    return y


def rope(x, pos, base=10000.0, inverse=False):
    x = _c(x, np.float64).copy()
    lib().csa2o_rope(_ptr(x), x.size, float(pos), float(base), int(bool(inverse)))
    return x


# ------------------------------------------------------------------ layer pieces
def write_seq(kc, gc, wa, gamma_c, w_ik, gamma_ik, gamma_w, p0, cap, *, z_codes=None,
              z_scales=None, ki_codes=None, ki_scales=None, pair_k=None, pair_g=None,
              window_prefix=None, base=10000.0, eps=1e-20, ratio=2):
    """Append T tokens (positions p0..p0+T-1) to one sequence's caches.  ``ratio`` is the
    layer's compression ratio: 2 (entry j pools tokens 2j, 2j+1) or 1 (entry j is token j).

    kc, gc, wa: [T, 512] float arrays.  The caches are created (zero) when not given and
    updated in place.  ``pair_k``/``pair_g`` hold the buffered token p0-1 when p0 is odd.
    ``window_prefix`` [127, 512] u8: FP8 rows of positions p0-127..p0-1 (zeros if None).
    Returns a dict with the caches, window [127+T,512], the new pair state (or None) and
    the fp64 pre-quantisation values (z_pre, ki_pre, win_pre) of what this call wrote.
    """
    kc, gc, wa = (_c(a, np.float32) for a in (kc, gc, wa))
    T = kc.shape[0]
    z_codes = np.zeros((cap, 256), np.uint8) if z_codes is None else z_codes
    z_scales = np.zeros((cap, 16), np.uint8) if z_scales is None else z_scales
    ki_codes = np.zeros((cap, 64), np.uint8) if ki_codes is None else ki_codes
    ki_scales = np.zeros((cap, 4), np.uint8) if ki_scales is None else ki_scales
    window = np.zeros((127 + T, D), np.uint8)
    if window_prefix is not None:
        window[:127] = window_prefix
    n_new = sum(1 for t in range(T) if (p0 + t) % ratio == ratio - 1)
    z_pre = np.zeros((max(n_new, 1), D))
    ki_pre = np.zeros((max(n_new, 1), DI))
    win_pre = np.zeros((T, D))
    pk_in = None if pair_k is None else _c(pair_k, np.float32)
    pg_in = None if pair_g is None else _c(pair_g, np.float32)
    if ratio == 2 and p0 % 2 == 1 and pk_in is None:
        raise ValueError("p0 is odd: the pair buffer (token p0-1) is required")
    pk_out = np.zeros(D, np.float32)
    pg_out = np.zeros(D, np.float32)
    g = [_c(a, np.float32) for a in (gamma_c, w_ik, gamma_ik, gamma_w)]
    n = lib().csa2o_write_seq(int(ratio), T, int(p0), _ptr(kc), _ptr(gc), _ptr(wa), *(_ptr(a) for a in g),
                              base, eps, _ptr(pk_in), _ptr(pg_in), _ptr(pk_out), _ptr(pg_out),
                              cap, _ptr(z_codes), _ptr(z_scales), _ptr(ki_codes),
                              _ptr(ki_scales), _ptr(window), _ptr(z_pre), _ptr(ki_pre),
                              _ptr(win_pre))
    if n < 0:
        raise ValueError("cache capacity too small")
    pair = (pk_out, pg_out) if ratio == 2 and (p0 + T) % 2 == 1 else None
    return dict(z_codes=z_codes, z_scales=z_scales, ki_codes=ki_codes, ki_scales=ki_scales,
                window=window, pair=pair, z_pre=z_pre[:n], ki_pre=ki_pre[:n], win_pre=win_pre,
                first_entry=p0 // ratio, n_entries=int(n))


def index_scores(pos, qi, wI, ki_codes, ki_scales, n_entries, return_qi_codes=False, ratio=2):
    """fp64 indexer scores for query rows at absolute positions ``pos``.

    qi [nq,32,128], wI [nq,32].  Returns scores [nq, max E] with NaN beyond E_r =
    floor((pos+1)/ratio).
    """
    pos = _c(pos, np.int64)
    qi = _c(qi, np.float32)
    wI = _c(wI, np.float32)
    nq = pos.size
    E = (pos + 1) // ratio
    ld = max(int(E.max()) if nq else 0, 1)
    scores = np.full((nq, ld), np.nan)
    qc = np.empty((nq, HI, 64), np.uint8) if return_qi_codes else None
    qs = np.empty((nq, HI, 4), np.uint8) if return_qi_codes else None
    rc = lib().csa2o_index_scores(int(ratio), nq, _ptr(pos), _ptr(qi), _ptr(wI), _ptr(_c(ki_codes, np.uint8)),
                                  _ptr(_c(ki_scales, np.uint8)), int(n_entries), _ptr(scores), ld,
                                  _ptr(qc), _ptr(qs))
    if rc != 0:
        raise ValueError("query position beyond the cache")
    return (scores, qc, qs) if return_qi_codes else scores


def topk(scores, E, k=TOPK):
    """(idx [nq,k] ascending, -1 padded; top scores [nq,k]; kth [nq,2] boundary scores)."""
    scores = _c(scores, np.float64)
    E = _c(E, np.int64)
    nq, ld = scores.shape
    idx = np.empty((nq, k), np.int32)
    top = np.empty((nq, k))
    kth = np.empty((nq, 2))
    lib().csa2o_topk(nq, _ptr(E), _ptr(scores), ld, k, _ptr(idx), _ptr(top), _ptr(kth))
    return idx, top, kth


def attend(pos, q, sinks, z_codes, z_scales, n_entries, window, win_p0, idx, base=10000.0,
           return_mass=False, win_start=0):
    """fp64 sink-softmax MQA for query rows at absolute positions ``pos``.

    q [nq,64,512] (already rotated), sinks [64], window [rows,512] u8 with row r <->
    position win_p0 + r, idx [nq,512].  ``win_start`` = s bounds the window rows to positions
    max(s, t-127)..t (replay from s).  Returns out [nq,64,512] (fp64).
    """
    pos = _c(pos, np.int64)
    q = _c(q, np.float32)
    sinks = _c(sinks, np.float32)
    window = _c(window, np.uint8)
    idx = _c(idx, np.int32)
    nq = pos.size
    out = np.empty((nq, H, D))
    mass = np.empty((nq, H))
    nrows = np.empty(nq, np.int32)
    rc = lib().csa2o_attend(nq, _ptr(pos), _ptr(q), _ptr(sinks), _ptr(_c(z_codes, np.uint8)),
                            _ptr(_c(z_scales, np.uint8)), int(n_entries), _ptr(window),
                            int(win_p0), window.shape[0], _ptr(idx), float(base), int(win_start),
                            _ptr(out), _ptr(mass), _ptr(nrows))
    if rc != 0:
        raise ValueError(f"attend: bad arguments ({rc})")
    return (out, mass, nrows) if return_mass else out


HSI_BLOCK, HSI_BLOCKS = 8, 2048


def hsi_pool(scores, E):
    """Hierarchical-indexer pool per row: the newest block of 8 entries plus the 2047 best other
    blocks by their best score (every block when at most 2048), ascending, -1 padded."""
    scores = _c(scores, np.float64)
    E = _c(E, np.int64)
    nq = E.size
    pool = np.empty((nq, HSI_BLOCKS), np.int32)
    lib().csa2o_hsi_pool(nq, _ptr(E), _ptr(scores), scores.shape[1], _ptr(pool))
    return pool


def reindex_topk(scores, E, pool, k=TOPK):
    """Top-k of each row's scores over its pool's visible entries (ties: lower j first)."""
    scores = _c(scores, np.float64)
    E = _c(E, np.int64)
    pool = _c(pool, np.int32)
    nq = E.size
    idx = np.empty((nq, k), np.int32)
    lib().csa2o_reindex_topk(nq, _ptr(E), _ptr(scores), scores.shape[1], _ptr(pool), k, _ptr(idx))
    return idx


# ------------------------------------------------------------------ grouped output projection
# "Inside DeepSeek V4.1", section "Attention that looks at 640 places": the outputs go back
# through 8 groups of a 1,024-wide bottleneck; [PG] o^g_{t,r} = [O-bar_{h,t}]_{h in r} W_OA,r.
# Group r holds heads 8r .. 8r+7, concatenated head after head (input k = 512 (h - 8r) + d).
OUT_GROUPS, OUT_GROUP_HEADS, OUT_GROUP_WIDTH = 8, 8, 1024


def out_group_proj(o_bar, w_oa):
    """o_bar [n, 64, 512] (the attention output), w_oa [8, 1024, 4096] (group r, output i,
    input k) -> o^g [n, 8, 1024] in fp64: o^g[:, r, i] = sum_k o_bar_r[:, k] w_oa[r, i, k]."""
    o = np.asarray(o_bar, np.float64)
    n = o.shape[0]
    o = o.reshape(n, OUT_GROUPS, OUT_GROUP_HEADS * 512)
    w = np.asarray(w_oa, np.float64)
    return np.einsum("nrk,rik->nri", o, w)

