"""Helpers for the GPU-vs-oracle parity tests: running the oracle per sequence and the
comparison rules.

Comparison rules
  * FP4 / FP8 codes: bit-exact, except where the oracle's fp64 value before rounding lies
    within REL_BOUNDARY of a rounding midpoint, or (FP4 scale bytes) where the block maximum
    lies within REL_BOUNDARY (relative) of a power of two.  The distance to a midpoint is
    measured relative to max(|v|, rms of v's row): the rows are RMS-normalised and the fp32
    error of a rotated or pooled value follows the magnitude of its operands (about the row
    rms), not of the (possibly cancelled) result.  Exceptions are counted and returned; any
    other mismatch fails.
  * Indices: bit-exact top-512 sets; a swap is allowed only where the oracle's scores of the
    swapped entries lie within REL_TIE (relative) of the oracle's 512th score.  Swaps are
    counted and returned.
  * bf16 outputs: max-abs error <= 2e-2 and relative L2 error <= 5e-3 against fp64.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL_BOUNDARY = 1e-6
REL_TIE = 1e-6
ATOL_OUT = 2e-2
RTOL_L2_OUT = 5e-3

E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def np32(t):
    return t.detach().float().cpu().numpy()


def unpack_nibbles(codes):
    codes = np.asarray(codes, np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = codes & 15
    out[..., 1::2] = codes >> 4
    return out


def fp4_compare(g_codes, g_scales, o_codes, o_scales, pre):
    """Rows of FP4 (codes [n, d/2], scales [n, d/32]) vs the oracle; pre [n, d] fp64 values
    before quantisation.  Returns (mismatched elements, mismatched scale bytes); raises
    AssertionError on a mismatch that the boundary rule does not explain."""
    g_codes, o_codes = np.asarray(g_codes), np.asarray(o_codes)
    g_scales, o_scales = np.asarray(g_scales), np.asarray(o_scales)
    n, d = pre.shape
    gc, oc = unpack_nibbles(g_codes), unpack_nibbles(o_codes)
    bad_scale = g_scales != o_scales
    nblk = d // 32
    amax = np.abs(pre.reshape(n, nblk, 32)).max(-1)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(amax > 0, amax, 1.0))
    near_pow2 = np.abs(amax / 2.0 ** np.round(lg) - 1.0) <= REL_BOUNDARY
    unexplained = bad_scale & ~near_pow2
    assert not unexplained.any(), f"{unexplained.sum()} FP4 scale bytes differ away from a power-of-two boundary"
    bad = gc != oc
    blk_scale_bad = np.repeat(bad_scale, 32, axis=1)
    e = np.repeat(o_scales.astype(np.int64) - 127, 32, axis=1)
    x = np.abs(pre) / 2.0 ** e
    rms = np.sqrt(np.mean(pre ** 2, axis=1, keepdims=True))
    tol = REL_BOUNDARY * np.maximum(np.abs(pre), rms) / 2.0 ** e
    near_mid = (np.abs(x[..., None] - E2M1_MIDS) <= tol[..., None]).any(-1)
    # a zero that differs only in its sign bit (a value rounding to 0 from either side)
    zero_sign = ((gc & 7) == 0) & ((oc & 7) == 0) & (np.abs(x) <= 0.25 * (1 + REL_BOUNDARY))
    unexplained = bad & ~(near_mid | blk_scale_bad | zero_sign)
    assert not unexplained.any(), (f"{unexplained.sum()} FP4 codes differ away from a rounding midpoint; "
                                   f"first at {np.argwhere(unexplained)[:3].tolist()}")
    return int(bad.sum()), int(bad_scale.sum())


def e4m3_compare(g, o, pre):
    g, o = np.asarray(g), np.asarray(o)
    bad = g != o
    if not bad.any():
        return 0
    gv = np.vectorize(oracle.e4m3_value)(g[bad].astype(np.int64))
    ov = np.vectorize(oracle.e4m3_value)(o[bad].astype(np.int64))
    mid = (gv + ov) / 2
    p = pre[bad]
    rms = np.broadcast_to(np.sqrt(np.mean(pre ** 2, axis=-1, keepdims=True)), pre.shape)[bad]
    ok = np.abs(p - mid) <= REL_BOUNDARY * np.maximum(np.abs(p), rms)
    ok |= (gv == 0) & (ov == 0)
    assert ok.all(), f"{(~ok).sum()} FP8 codes differ away from a rounding midpoint"
    return int(bad.sum())


def topk_compare(g_idx, o_idx, o_scores, kth, E, n_cand=None):
    """Rows of GPU vs oracle top-512 indices.  o_scores [nq, >=E]: oracle fp64 scores;
    kth [nq, 2]: oracle 512th / 513th scores; entries lie in 0..E-1 and n_cand (default E)
    are candidates.  Returns the number of swapped entries."""
    g_idx, o_idx = np.asarray(g_idx), np.asarray(o_idx)
    swaps = 0
    for r in range(g_idx.shape[0]):
        g = g_idx[r]
        k = min(512, int(E[r] if n_cand is None else n_cand[r]))
        assert np.all(g[k:] == -1), f"row {r}: expected {512 - k} trailing -1"
        gv = g[:k]
        assert np.all(np.diff(gv) > 0) and (k == 0 or (gv[0] >= 0 and gv[-1] < E[r])), f"row {r}: not ascending / out of range"
        if np.array_equal(gv, o_idx[r, :k]):
            continue
        a, b = np.setdiff1d(gv, o_idx[r, :k]), np.setdiff1d(o_idx[r, :k], gv)
        bound = kth[r, 0]
        for j in np.concatenate([a, b]):
            assert abs(o_scores[r, j] - bound) <= REL_TIE * abs(bound), (
                f"row {r}: entry {j} swapped with oracle score {o_scores[r, j]!r} vs boundary {bound!r}")
        swaps += len(a)
    return swaps


def out_compare(g, o):
    """bf16 GPU output vs fp64 oracle: returns (max abs error, relative L2 error)."""
    g = np.asarray(g, np.float64)
    err = g - o
    mx = float(np.abs(err).max()) if err.size else 0.0
    rl2 = float(np.linalg.norm(err) / max(np.linalg.norm(o), 1e-300))
    assert mx <= ATOL_OUT, f"max abs error {mx}"
    assert rl2 <= RTOL_L2_OUT, f"relative L2 error {rl2}"
    return mx, rl2


def random_indices(B, T, p0s, seed, device="cpu"):
    """Sorted distinct entry indices per query (visible ones), -1 padded, for attention
    tests that do not depend on the indexer (drawn with a seeded generator)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    idx = torch.full((B, T, 512), -1, dtype=torch.int32)
    for b in range(B):
        for t in range(T):
            E = (int(p0s[b]) + t + 1) // 2
            k = min(512, E)
            if k:
                sel = torch.randperm(E, generator=g)[:k].sort().values
                idx[b, t, :k] = sel.to(torch.int32)
    return idx.to(device)


def pool_compare(g_pool, o_pool, scores, E, nsel=2047, nblocks=2048, block=8):
    """Rows of GPU vs oracle hierarchical pools.  A row must be ascending, -1 padded, hold
    min(blocks, nblocks) blocks and the newest block; a block present on one side only is
    allowed where its oracle block score lies within REL_TIE of the oracle's nsel-th best
    older block.  Returns the number of swapped blocks."""
    g_pool, o_pool = np.asarray(g_pool), np.asarray(o_pool)
    swaps = 0
    for r in range(g_pool.shape[0]):
        nb = (int(E[r]) + block - 1) // block
        k = min(nb, nblocks)
        g = g_pool[r]
        assert np.all(g[k:] == -1), f"row {r}: expected {nblocks - k} trailing -1"
        gv = g[:k]
        assert np.all(np.diff(gv) > 0) and (k == 0 or (gv[0] >= 0 and gv[-1] == nb - 1)), f"row {r}: pool order"
        if np.array_equal(gv, o_pool[r, :k]):
            continue
        bs = scores[r, : (nb - 1) * block].reshape(nb - 1, block).max(axis=1)
        bound = np.sort(bs)[::-1][nsel - 1]
        a, b = np.setdiff1d(gv, o_pool[r, :k]), np.setdiff1d(o_pool[r, :k], gv)
        for j in np.concatenate([a, b]):
            assert abs(bs[j] - bound) <= REL_TIE * abs(bound), (
                f"row {r}: block {j} swapped with oracle block score {bs[j]!r} vs boundary {bound!r}")
        swaps += len(a)
    return swaps


def pool_kth(scores, E, pool, k=512, block=8):
    """Oracle k-th and (k+1)-th largest scores over each row's pool entries (-inf if none)."""
    kth = np.full((scores.shape[0], 2), -np.inf)
    for r in range(scores.shape[0]):
        blks = pool[r][pool[r] >= 0].astype(np.int64)
        j = (block * blks[:, None] + np.arange(block)[None, :]).ravel()
        j = j[j < E[r]]
        v = np.sort(scores[r, j])[::-1]
        for c in range(2):
            if len(v) > k - 1 + c:
                kth[r, c] = v[k - 1 + c]
    return kth
