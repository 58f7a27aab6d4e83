"""Python binding of libcsa2.so, the GB300 (sm_103a) CSA2 layer library.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
PyTorch provides device memory and streams.  The functions carry the C-ABI names of
``include/csa2.h`` and raise :class:`Csa2Error` on any non-OK status.  If the library has
not been built the import of a function fails loudly; there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

import numpy as np
import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "_build" / "libcsa2.so"

OP_WRITE_CACHE, OP_INDEX_TOPK, OP_ATTEND, OP_INDEX_POOL, OP_REINDEX_TOPK, OP_INDEX_SCORES = 0, 1, 2, 3, 4, 5
HSI_BLOCKS = 2048  # pool blocks per query row (blocks of 8 entries)
HEADS, HEAD_DIM, ROPE_DIMS, IDX_HEADS, IDX_DIM, WINDOW, TOPK = 64, 512, 64, 32, 128, 128, 512

_STATUS = {0: "ok", 1: "invalid argument", 2: "inconsistent sizes", 3: "pointer not 16-byte aligned",
           4: "workspace too small", 5: "unsupported configuration", 6: "CUDA error",
           7: "batch exceeds the fixed scratch of csa2_attend_static", 8: "a bounded wait inside a kernel gave up"}


class Csa2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_STATUS.get(status, 'unknown')} (status {status})")
        self.status = status


class csa2_config(C.Structure):
    _fields_ = [("heads", C.c_int), ("head_dim", C.c_int), ("rope_dims", C.c_int), ("idx_heads", C.c_int),
                ("idx_dim", C.c_int), ("window", C.c_int), ("topk", C.c_int), ("ratio", C.c_int),
                ("rope_base", C.c_double), ("eps", C.c_double)]


EXPORTS = ("csa2_default_config", "csa2_create", "csa2_destroy", "csa2_status_string", "csa2_kernel_launches",
           "csa2_workspace_bytes",
           "csa2_write_cache", "csa2_roll_window", "csa2_index_topk", "csa2_index_scores", "csa2_index_pool", "csa2_reindex_topk", "csa2_attend",
           "csa2_attend_replay", "csa2_attend_static", "csa2_check", "csa2_selftest_timeout",
           "csa2_out_group_proj", "csa2_tc_rate", "csa2_set_device_positions")

_lib = None


def lib() -> C.CDLL:
    """The loaded libcsa2.so.  Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(or python compressed_sparse_attention_03_gb300/build.py)")
        L = C.CDLL(str(LIB_PATH))
        p, i32, i64, sz = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
        L.csa2_default_config.argtypes = [C.POINTER(csa2_config)]
        L.csa2_create.argtypes = [C.POINTER(csa2_config), C.POINTER(p)]
        L.csa2_create.restype = i32
        L.csa2_destroy.argtypes = [p]
        L.csa2_status_string.argtypes = [i32]
        L.csa2_status_string.restype = C.c_char_p
        L.csa2_kernel_launches.argtypes = []
        L.csa2_kernel_launches.restype = C.c_uint64
        L.csa2_workspace_bytes.argtypes = [p, i32, i32, i32, i64]
        L.csa2_workspace_bytes.restype = sz
        L.csa2_write_cache.argtypes = [p] * 9 + [i32, i32] + [p] * 6 + [i64, p, p, sz, p]
        L.csa2_write_cache.restype = i32
        L.csa2_index_topk.argtypes = [p] * 5 + [i64, p, i32, i32, p, p, p, sz, p]
        L.csa2_index_topk.restype = i32
        L.csa2_roll_window.argtypes = [p, p, i32, i32, p, i32, p]
        L.csa2_roll_window.restype = i32
        L.csa2_index_scores.argtypes = [p] * 5 + [i64, p, i32, i32, p, i64, p, sz, p]
        L.csa2_index_scores.restype = i32
        L.csa2_out_group_proj.argtypes = [p, p, p, i64, p, p]
        L.csa2_out_group_proj.restype = i32
        L.csa2_tc_rate.argtypes = [p, i32, i32, C.POINTER(C.c_double), p]
        L.csa2_tc_rate.restype = i32
        L.csa2_check.argtypes = [p, p]
        L.csa2_check.restype = i32
        L.csa2_selftest_timeout.argtypes = [p, p]
        L.csa2_selftest_timeout.restype = i32
        L.csa2_index_pool.argtypes = [p] * 5 + [i64, p, i32, i32, p, p, p, p, sz, p]
        L.csa2_index_pool.restype = i32
        L.csa2_reindex_topk.argtypes = [p] * 5 + [i64, p, i32, i32, p, p, p, p, sz, p]
        L.csa2_reindex_topk.restype = i32
        L.csa2_attend.argtypes = [p] * 5 + [i64, p, p, p, i32, i32, p, p, sz, p]
        L.csa2_attend.restype = i32
        L.csa2_attend_replay.argtypes = [p] * 5 + [i64, p, p, p, p, i32, i32, p, p, sz, p]
        L.csa2_attend_replay.restype = i32
        L.csa2_attend_static.argtypes = [p] * 5 + [i64, p, p, p, i32, i32, p, p]
        L.csa2_attend_static.restype = i32
        L.csa2_set_device_positions.argtypes = [p, p, i64]
        L.csa2_set_device_positions.restype = i32
        _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise Csa2Error(fn, status)


def _dev(t, dtype, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return C.c_void_p(t.data_ptr())


def _host_p0(p0, B, h=None):
    """Host positions as int64[B]; None (passed as NULL) when the handle reads device positions
    and the call gives none."""
    if p0 is None:
        if h is not None and h.dev_p0_max is not None:
            return None
        raise ValueError("p0: required (the handle reads host positions)")
    a = np.ascontiguousarray(np.asarray(p0.cpu() if isinstance(p0, torch.Tensor) else p0, dtype=np.int64).reshape(-1))
    if a.size == 1 and B > 1:
        a = np.full(B, int(a[0]), np.int64)
    if a.size != B:
        raise ValueError(f"p0: expected {B} positions, got {a.size}")
    return a


def _p0_ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _max_entries(h, p0a, T):
    """Visible entries of the call's last query: from the host positions, else from the bound of
    the device positions."""
    if p0a is None:
        return (h.dev_p0_max + T) // h.ratio
    return int(((p0a + T) // h.ratio).max())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


class Handle:
    """Owns a csa2_handle (created on the current CUDA device)."""

    def __init__(self, rope_base: float = 10000.0, eps: float = 1e-20, ratio: int = 2):
        cfg = csa2_config()
        lib().csa2_default_config(C.byref(cfg))
        cfg.rope_base, cfg.eps, cfg.ratio = rope_base, eps, ratio
        self.ratio = ratio
        self.dev_p0_max = None  # set by csa2_set_device_positions
        h = C.c_void_p()
        _check("csa2_create", lib().csa2_create(C.byref(cfg), C.byref(h)))
        self._h = h

    @property
    def ptr(self):
        return self._h

    def close(self):
        if self._h:
            lib().csa2_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def csa2_create(rope_base: float = 10000.0, eps: float = 1e-20, ratio: int = 2) -> Handle:
    return Handle(rope_base, eps, ratio)


def csa2_kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib().csa2_kernel_launches())


def csa2_workspace_bytes(h: Handle, op: int, B: int, T: int, max_entries: int) -> int:
    return int(lib().csa2_workspace_bytes(h.ptr, op, B, T, max_entries))


def workspace(h: Handle, op: int, B: int, T: int, max_entries: int, device=None) -> torch.Tensor:
    """A uint8 CUDA tensor sized by csa2_workspace_bytes (at least 16 bytes)."""
    n = max(16, csa2_workspace_bytes(h, op, B, T, max_entries))
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def csa2_write_cache(h: Handle, kc, gc, wa, gamma_c, w_ik, gamma_ik, gamma_w, p0, z_codes, z_scales, ki_codes,
                     ki_scales, window, pair_kc=None, pair_gc=None, stream=None) -> None:
    B, T, _ = kc.shape
    p0a = _host_p0(p0, B, h)
    cap = z_codes.shape[1]
    _check("csa2_write_cache", lib().csa2_write_cache(
        h.ptr, _dev(kc, torch.bfloat16, "kc"), _dev(gc, torch.bfloat16, "gc"), _dev(wa, torch.bfloat16, "wa"),
        _dev(gamma_c, torch.float32, "gamma_c"), _dev(w_ik, torch.bfloat16, "w_ik"),
        _dev(gamma_ik, torch.float32, "gamma_ik"), _dev(gamma_w, torch.float32, "gamma_w"),
        _p0_ptr(p0a), B, T, _dev(pair_kc, torch.float32, "pair_kc"),
        _dev(pair_gc, torch.float32, "pair_gc"), _dev(z_codes, torch.uint8, "z_codes"),
        _dev(z_scales, torch.uint8, "z_scales"), _dev(ki_codes, torch.uint8, "ki_codes"),
        _dev(ki_scales, torch.uint8, "ki_scales"), cap, _dev(window, torch.uint8, "window"), None, 0,
        _stream(stream)))


def csa2_roll_window(h: Handle, window, nxt, stream=None) -> None:
    """Rows T .. T+126 of the window view [B, 127+T, 512] -> rows 0 .. 126 of the next call's view
    [B, 127+T_next, 512] (``nxt`` may be ``window`` itself when T_next == T or B == 1)."""
    B, rows, _ = window.shape
    T, T_next = rows - 127, nxt.shape[1] - 127
    if nxt.shape[0] != B or window.shape[2] != 512 or nxt.shape[2] != 512:
        raise ValueError("csa2_roll_window: views must be [B, 127+T, 512]")
    _check("csa2_roll_window", lib().csa2_roll_window(
        h.ptr, _dev(window, torch.uint8, "window"), B, T, _dev(nxt, torch.uint8, "next"), T_next, _stream(stream)))


def csa2_index_topk(h: Handle, qi, wI, ki_codes, ki_scales, p0, idx, top_scores=None, ws=None, stream=None) -> None:
    B, T = qi.shape[:2]
    p0a = _host_p0(p0, B, h)
    cap = ki_codes.shape[1]
    if ws is None:
        ws = workspace(h, OP_INDEX_TOPK, B, T, _max_entries(h, p0a, T), qi.device)
    _check("csa2_index_topk", lib().csa2_index_topk(
        h.ptr, _dev(qi, torch.bfloat16, "qi"), _dev(wI, torch.bfloat16, "wI"), _dev(ki_codes, torch.uint8, "ki_codes"),
        _dev(ki_scales, torch.uint8, "ki_scales"), cap, _p0_ptr(p0a), B, T,
        _dev(idx, torch.int32, "idx"), _dev(top_scores, torch.float32, "top_scores"), _dev(ws, torch.uint8, "ws"),
        ws.numel(), _stream(stream)))


def csa2_index_scores(h: Handle, qi, wI, ki_codes, ki_scales, p0, scores, ws=None, stream=None) -> None:
    """S^I of every visible entry: scores f32 [B, T, ld] (ld a multiple of 4, at least the largest
    visible count); entries beyond a row's visible count are left untouched."""
    B, T = qi.shape[:2]
    p0a = _host_p0(p0, B, h)
    cap = ki_codes.shape[1]
    if scores.dim() != 3 or scores.shape[:2] != (B, T):
        raise ValueError("csa2_index_scores: scores must be [B, T, ld]")
    if ws is None:
        ws = workspace(h, OP_INDEX_SCORES, B, T, _max_entries(h, p0a, T), qi.device)
    _check("csa2_index_scores", lib().csa2_index_scores(
        h.ptr, _dev(qi, torch.bfloat16, "qi"), _dev(wI, torch.bfloat16, "wI"), _dev(ki_codes, torch.uint8, "ki_codes"),
        _dev(ki_scales, torch.uint8, "ki_scales"), cap, _p0_ptr(p0a), B, T,
        _dev(scores, torch.float32, "scores"), scores.shape[2], _dev(ws, torch.uint8, "ws"), ws.numel(),
        _stream(stream)))


def csa2_index_pool(h: Handle, qi, wI, ki_codes, ki_scales, p0, idx, pool, top_scores=None, ws=None,
                    stream=None) -> None:
    """csa2_index_topk plus the hierarchical block pool [B, T, 2048] of each query."""
    B, T = qi.shape[:2]
    p0a = _host_p0(p0, B, h)
    cap = ki_codes.shape[1]
    if ws is None:
        ws = workspace(h, OP_INDEX_POOL, B, T, _max_entries(h, p0a, T), qi.device)
    _check("csa2_index_pool", lib().csa2_index_pool(
        h.ptr, _dev(qi, torch.bfloat16, "qi"), _dev(wI, torch.bfloat16, "wI"), _dev(ki_codes, torch.uint8, "ki_codes"),
        _dev(ki_scales, torch.uint8, "ki_scales"), cap, _p0_ptr(p0a), B, T,
        _dev(idx, torch.int32, "idx"), _dev(top_scores, torch.float32, "top_scores"), _dev(pool, torch.int32, "pool"),
        _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))


def csa2_reindex_topk(h: Handle, qi, wI, ki_codes, ki_scales, p0, pool, idx, top_scores=None, ws=None,
                      stream=None) -> None:
    """Top-512 of this layer's indexer scores over the entries of a given block pool."""
    B, T = qi.shape[:2]
    p0a = _host_p0(p0, B, h)
    cap = ki_codes.shape[1]
    if ws is None:
        ws = workspace(h, OP_REINDEX_TOPK, B, T, _max_entries(h, p0a, T), qi.device)
    _check("csa2_reindex_topk", lib().csa2_reindex_topk(
        h.ptr, _dev(qi, torch.bfloat16, "qi"), _dev(wI, torch.bfloat16, "wI"), _dev(ki_codes, torch.uint8, "ki_codes"),
        _dev(ki_scales, torch.uint8, "ki_scales"), cap, _p0_ptr(p0a), B, T,
        _dev(pool, torch.int32, "pool"), _dev(idx, torch.int32, "idx"), _dev(top_scores, torch.float32, "top_scores"),
        _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))


def csa2_out_group_proj(h: Handle, o, w_oa, out, stream=None) -> None:
    """o [.., 64, 512] bf16 -> out [.., 8, 1024] bf16 through the 8 grouped W_OA [8, 1024, 4096]."""
    M = o.numel() // (64 * 512)
    if out.numel() != M * 8 * 1024 or w_oa.numel() != 8 * 1024 * 4096:
        raise ValueError("csa2_out_group_proj: shapes")
    _check("csa2_out_group_proj", lib().csa2_out_group_proj(
        h.ptr, _dev(o, torch.bfloat16, "o"), _dev(w_oa, torch.bfloat16, "w_oa"), M,
        _dev(out, torch.bfloat16, "out"), _stream(stream)))


def csa2_tc_rate(h: Handle, kind: int, iters: int = 8192, stream=None) -> float:
    """Measured tensor-core rate in TFLOP/s: kind 0 kind::f16 (fp16), 1 kind::f8f6f4 (E5M2),
    2 kind::mxf4 (E2M1 with UE8M0 scales per 32).  Synchronises the stream."""
    out = C.c_double(0.0)
    _check("csa2_tc_rate", lib().csa2_tc_rate(h.ptr, int(kind), int(iters), C.byref(out), _stream(stream)))
    return out.value


def csa2_check(h: Handle, stream=None) -> int:
    """Synchronises the stream and returns what the kernels recorded since the last check: 0,
    8 (a bounded wait gave up), 2 (a device position outside 0..p0_max was read and clamped) or
    5 (an FP4 scale above 2^13, or a query beyond the fp16 range, was read).  Does not raise on
    2, 5 or 8: the caller decides."""
    st = lib().csa2_check(h.ptr, _stream(stream))
    if st not in (0, 2, 5, 8):
        _check("csa2_check", st)
    return st


def csa2_set_device_positions(h: Handle, p0_dev, p0_max: int = 0) -> None:
    """Positions from device memory (int64 CUDA tensor of B values, read by the kernels when they
    run; the calls may then pass p0=None) with the bound p0_max the host plans with; None returns
    the handle to host positions.  Call outside stream capture."""
    if p0_dev is None:
        _check("csa2_set_device_positions", lib().csa2_set_device_positions(h.ptr, None, 0))
        h.dev_p0_max = None
        return
    _check("csa2_set_device_positions", lib().csa2_set_device_positions(
        h.ptr, _dev(p0_dev, torch.int64, "p0_dev"), int(p0_max)))
    h.dev_p0_max = int(p0_max)


def csa2_selftest_timeout(h: Handle, stream=None) -> None:
    """Enqueues a kernel whose one bounded wait can never complete (a test of csa2_check)."""
    _check("csa2_selftest_timeout", lib().csa2_selftest_timeout(h.ptr, _stream(stream)))


def csa2_attend(h: Handle, q, sinks, z_codes, z_scales, window, idx, p0, out, ws=None, stream=None) -> None:
    B, T = q.shape[:2]
    p0a = _host_p0(p0, B, h)
    cap = z_codes.shape[1]
    if ws is None:
        ws = workspace(h, OP_ATTEND, B, T, 0, q.device)
    _check("csa2_attend", lib().csa2_attend(
        h.ptr, _dev(q, torch.bfloat16, "q"), _dev(sinks, torch.float32, "sinks"), _dev(z_codes, torch.uint8, "z_codes"),
        _dev(z_scales, torch.uint8, "z_scales"), cap, _dev(window, torch.uint8, "window"),
        _dev(idx, torch.int32, "idx"), _p0_ptr(p0a), B, T, _dev(out, torch.bfloat16, "out"),
        _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))


def csa2_attend_static(h: Handle, q, sinks, z_codes, z_scales, window, idx, p0, out, stream=None) -> None:
    """csa2_attend without a workspace: the library's fixed device scratch holds the split
    partials, and no call here allocates device memory (the tensors are the caller's).  Calls
    that can overlap in time share that scratch and race; see include/csa2.h."""
    B, T = q.shape[:2]
    p0a = _host_p0(p0, B, h)
    cap = z_codes.shape[1]
    _check("csa2_attend_static", lib().csa2_attend_static(
        h.ptr, _dev(q, torch.bfloat16, "q"), _dev(sinks, torch.float32, "sinks"), _dev(z_codes, torch.uint8, "z_codes"),
        _dev(z_scales, torch.uint8, "z_scales"), cap, _dev(window, torch.uint8, "window"),
        _dev(idx, torch.int32, "idx"), _p0_ptr(p0a), B, T, _dev(out, torch.bfloat16, "out"),
        _stream(stream)))


def csa2_attend_replay(h: Handle, q, sinks, z_codes, z_scales, window, idx, p0, win_start, out, ws=None,
                       stream=None) -> None:
    """csa2_attend after a bounded replay: query t of sequence b sees the window positions
    max(win_start[b], t-127)..t."""
    B, T = q.shape[:2]
    p0a = _host_p0(p0, B, h)
    wsa = _host_p0(win_start, B)
    cap = z_codes.shape[1]
    if ws is None:
        ws = workspace(h, OP_ATTEND, B, T, 0, q.device)
    _check("csa2_attend_replay", lib().csa2_attend_replay(
        h.ptr, _dev(q, torch.bfloat16, "q"), _dev(sinks, torch.float32, "sinks"), _dev(z_codes, torch.uint8, "z_codes"),
        _dev(z_scales, torch.uint8, "z_scales"), cap, _dev(window, torch.uint8, "window"),
        _dev(idx, torch.int32, "idx"), _p0_ptr(p0a), wsa.ctypes.data_as(C.c_void_p), B, T,
        _dev(out, torch.bfloat16, "out"), _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
