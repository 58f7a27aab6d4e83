"""GPU parity of the Hierarchical Sparse Indexer ("Inside DeepSeek V4.1", section "Most layers
borrow"; "Deriving the 890-Byte KV Cache", section "Hierarchical indexing bounds the later
searches"): the owner layer's block pool and a later layer's top-512 over that pool, through
the C ABI, against the fp64 oracle.  The pool a later layer searches is the oracle's, so no
GPU output feeds an oracle input.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_03_gb300 import inputs
import compressed_sparse_attention_03_gb300 as csa2
from parity_utils import np32, pool_compare, pool_kth, topk_compare
from test_gpu_parity import make_state, oracle_write, use_oracle_state

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def handle():
    return csa2.csa2_create()


@pytest.fixture(scope="module")
def handle_r1():
    return csa2.csa2_create(ratio=1)


def later_layer_queries(x, seed):
    """A second layer's indexer queries and head weights (same shapes, another seed)."""
    B, T = x["qi"].shape[:2]
    y = inputs.step_inputs(B, T, seed, DEV)
    return y["qi"], y["wI"]


def oracle_scores(x, qi, wI, b, p0, rows, ratio):
    pos = p0 + rows
    E = (pos + 1) // ratio
    n = max(int(E.max()), 1)
    kc = x["ki_codes"][b, :n].cpu().numpy()
    ks = x["ki_scales"][b, :n].cpu().numpy()
    return oracle.index_scores(pos, np32(qi[b][rows]), np32(wI[b][rows]), kc, ks, n, ratio=ratio), E


def run_pool(h, x, p0s):
    B, T = x["qi"].shape[:2]
    idx = torch.empty(B, T, 512, dtype=torch.int32, device=DEV)
    pool = torch.empty(B, T, csa2.HSI_BLOCKS, dtype=torch.int32, device=DEV)
    csa2.csa2_index_pool(h, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], p0s, idx, pool)
    return idx, pool


def check_owner_and_later(h, x, p0s, ratio=2, rows=None, seed=77):
    """Owner layer: top-512 and pool against the oracle.  Later layer: top-512 of its own
    scores over the oracle's pool (rows outside `rows` get an empty pool, all -1).  Returns
    (top-512 swaps, pool swaps, reindex swaps)."""
    B, T = x["qi"].shape[:2]
    idx, pool = run_pool(h, x, p0s)
    qi2, wI2 = later_layer_queries(x, seed)
    r_all = np.arange(T) if rows is None else np.asarray(rows)
    opools = torch.full((B, T, csa2.HSI_BLOCKS), -1, dtype=torch.int32)
    cache = {}
    for b, p0 in enumerate(p0s):
        sc, E = oracle_scores(x, x["qi"], x["wI"], b, p0, r_all, ratio)
        op = oracle.hsi_pool(sc, E)
        opools[b, r_all] = torch.from_numpy(op)
        cache[b] = (sc, E, op)
    ridx = torch.empty(B, T, 512, dtype=torch.int32, device=DEV)
    rtop = torch.empty(B, T, 512, dtype=torch.float32, device=DEV)
    csa2.csa2_reindex_topk(h, qi2, wI2, x["ki_codes"], x["ki_scales"], p0s, opools.to(DEV), ridx, rtop)
    s_top = s_pool = s_re = 0
    for b, p0 in enumerate(p0s):
        sc, E, op = cache[b]
        oidx, _, kth = oracle.topk(sc, E)
        s_top += topk_compare(idx[b][r_all].cpu().numpy(), oidx, sc, kth, E)
        s_pool += pool_compare(pool[b][r_all].cpu().numpy(), op, sc, E)
        sc2, _ = oracle_scores(x, qi2, wI2, b, p0, r_all, ratio)
        ridx_o = oracle.reindex_topk(sc2, E, op)
        g = ridx[b][r_all].cpu().numpy()
        kth2 = pool_kth(sc2, E, op)
        nvis = np.array([int(((8 * op[i][op[i] >= 0][:, None] + np.arange(8)) < E[i]).sum()) for i in range(len(r_all))])
        s_re += topk_compare(g, ridx_o, sc2, kth2, E, n_cand=nvis)
        gt_all = rtop[b][r_all].cpu().numpy()
        for i in range(len(r_all)):  # every chosen entry is one of the pool's visible entries
            chosen = g[i][g[i] >= 0]
            assert np.all(np.isin(chosen // 8, op[i])) and np.all(chosen < E[i]), f"row {r_all[i]}: entry outside pool"
            k = len(chosen)
            scale = np.abs(sc2[i, : int(E[i])]).max() if k else 0.0
            assert np.all(np.abs(gt_all[i, :k] - sc2[i, chosen]) <= 1e-5 * scale), f"row {r_all[i]} reindex scores"
            assert np.all(np.isnan(gt_all[i, k:]))
    return s_top, s_pool, s_re


@pytest.mark.parametrize("B,T,p0s", [
    (2, 1, [40001, 3000]),      # a pool of 2048 out of 2501 blocks; all 188 blocks
    (3, 1, [0, 1, 33]),         # no, one partial and a few entries
    (1, 1, [32770]),            # 16385 entries: 2049 blocks, the newest holding one entry
    (1, 1, [32768]),            # 16384 entries: exactly 2048 blocks
    (2, 64, [36000, 37]),       # prefill rows crossing 2048 blocks
    (1, 300, [0]),              # prefill from scratch
])
def test_hsi_small(handle, B, T, p0s):
    x, cap = make_state(B, T, p0s, seed=11 + T)
    if max(p0s) == 0:
        use_oracle_state(x, oracle_write(x, p0s, cap))
    sw = check_owner_and_later(handle, x, p0s)
    print(f"hsi B={B} T={T}: swaps top/pool/reindex = {sw}")


def test_hsi_block_ties(handle):
    # identical keys give identical block scores: the lower blocks must win
    p0 = 50000
    x, cap = make_state(1, 1, [p0], seed=5)
    x["ki_codes"][0, : 8 * 2500] = x["ki_codes"][0, 9]
    x["ki_scales"][0, : 8 * 2500] = x["ki_scales"][0, 9]
    idx, pool = run_pool(handle, x, [p0])
    sc, E = oracle_scores(x, x["qi"], x["wI"], 0, p0, np.arange(1), 2)
    op = oracle.hsi_pool(sc, E)
    assert np.array_equal(pool[0].cpu().numpy(), op)


def test_hsi_ratio1(handle_r1):
    p0s = [20000, 900]
    x, cap = make_state(2, 1, p0s, seed=13, ratio=1)
    sw = check_owner_and_later(handle_r1, x, p0s, ratio=1)
    print(f"hsi ratio 1: swaps top/pool/reindex = {sw}")


@pytest.mark.parametrize("name", ["decode_128k", "decode_1m"])
def test_hsi_workloads(handle, name):
    # decode_1m: 65536 blocks per row, so the pool select runs over several chunks and a merge
    wl = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(wl, DEV)
    B = min(wl.B, 4)
    for k in ("qi", "wI", "ki_codes", "ki_scales"):
        x[k] = x[k][:B].contiguous()
    sw = check_owner_and_later(handle, x, [wl.p0] * B)
    print(f"hsi {name} (B={B}): swaps top/pool/reindex = {sw}")


def test_hsi_chunk_32k_sampled(handle):
    wl = inputs.WORKLOADS["chunk_32k"]
    x = inputs.workload_inputs(wl, DEV)
    use_oracle_state(x, oracle_write(x, [wl.p0], wl.cap))
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, 1, wl.T - 1], rng.integers(0, wl.T, 9)]))
    sw = check_owner_and_later(handle, x, [wl.p0], rows=rows)
    print(f"hsi chunk_32k ({len(rows)} rows): swaps top/pool/reindex = {sw}")


def test_hsi_argument_errors(handle):
    x, cap = make_state(1, 1, [100], seed=1)
    idx = torch.empty(1, 1, 512, dtype=torch.int32, device=DEV)
    with pytest.raises(RuntimeError):
        csa2.csa2_index_pool(handle, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], [100], idx, None)
    with pytest.raises(RuntimeError):
        csa2.csa2_reindex_topk(handle, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], [100], None, idx)


def test_hsi_two_launch_groups(handle):
    # 130 sequences run as a group of 128 and a tail of 2 (its workspace and its pool rows at
    # sequence offset 128); contexts from a few blocks to more than 2048 blocks
    rng = np.random.default_rng(12)
    B = 130
    p0s = rng.integers(0, 40000, B)
    p0s[-1] = 36001  # the tail holds a row with more than 2048 blocks
    x, cap = make_state(B, 1, p0s, seed=31)
    rows = [0, 1, 64, 127, 128, 129]
    idx, pool = run_pool(handle, x, p0s)
    for b in rows:
        sc, E = oracle_scores(x, x["qi"], x["wI"], b, int(p0s[b]), np.arange(1), 2)
        oidx, _, kth = oracle.topk(sc, E)
        topk_compare(idx[b].cpu().numpy(), oidx, sc, kth, E)
        pool_compare(pool[b].cpu().numpy(), oracle.hsi_pool(sc, E), sc, E)
