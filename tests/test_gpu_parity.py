"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by element on
the same seeded inputs.  Small cases span several tiles and ragged tails; the named
workloads run at full size with sampled query rows where the oracle would be too slow.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_03_gb300 import inputs
import compressed_sparse_attention_03_gb300 as csa2
from parity_utils import (e4m3_compare, fp4_compare, np32, out_compare, random_indices, topk_compare)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def handle():
    return csa2.csa2_create()


@pytest.fixture(scope="module")
def handle_r1():
    return csa2.csa2_create(ratio=1)


def make_state(B, T, p0s, seed, cap=None, device=DEV, ratio=2):
    p0s = np.asarray(p0s, np.int64)
    cap = cap or int(((p0s + T) // ratio).max()) + 3
    x = {}
    x.update(inputs.layer_params(seed, device))
    x.update(inputs.step_inputs(B, T, seed, device))
    st = inputs.cache_state(B, T, int(p0s.max()), cap, seed, device, ratio)
    # sequences with shorter context: drop cached entries beyond their own length
    for b in range(B):
        n = int(p0s[b]) // ratio
        for k in ("z_codes", "z_scales", "ki_codes", "ki_scales"):
            st[k][b, n:] = 0
    x.update(st)
    return x, cap


def gpu_write(h, x, p0s):
    w = {k: x[k].clone() for k in ("z_codes", "z_scales", "ki_codes", "ki_scales", "window", "pair_kc", "pair_gc")}
    csa2.csa2_write_cache(h, x["kc"], x["gc"], x["wa"], x["gamma_c"], x["w_ik"], x["gamma_ik"], x["gamma_w"], p0s,
                          w["z_codes"], w["z_scales"], w["ki_codes"], w["ki_scales"], w["window"], w["pair_kc"],
                          w["pair_gc"])
    return w


def oracle_write(x, p0s, cap, ratio=2):
    res = []
    for b, p0 in enumerate(p0s):
        cpu = lambda k: np32(x[k][b]) if x[k].dtype != torch.uint8 else x[k][b].cpu().numpy().copy()
        r = oracle.write_seq(cpu("kc"), cpu("gc"), cpu("wa"), np32(x["gamma_c"]), np32(x["w_ik"]), np32(x["gamma_ik"]),
                             np32(x["gamma_w"]), int(p0), cap, z_codes=cpu("z_codes"), z_scales=cpu("z_scales"),
                             ki_codes=cpu("ki_codes"), ki_scales=cpu("ki_scales"), pair_k=cpu("pair_kc"),
                             pair_g=cpu("pair_gc"), window_prefix=cpu("window")[:127], ratio=ratio)
        res.append(r)
    return res


def use_oracle_state(x, ores):
    """Replace the caches and window views in ``x`` by what the oracle's writer produced, so
    that later stages of both sides read the same (oracle-made) state."""
    for b, r in enumerate(ores):
        for k in ("z_codes", "z_scales", "ki_codes", "ki_scales", "window"):
            x[k][b] = torch.from_numpy(r[k]).to(x[k].device)
    return x


def check_write(w, ores, p0s, T, ratio=2):
    n_code = n_scale = n_fp8 = 0
    for b, (r, p0) in enumerate(zip(ores, p0s)):
        j0, n = r["first_entry"], r["n_entries"]
        sl = slice(j0, j0 + n)
        g = {k: w[k][b].cpu().numpy() for k in ("z_codes", "z_scales", "ki_codes", "ki_scales", "window")}
        if n:
            c1, s1 = fp4_compare(g["z_codes"][sl], g["z_scales"][sl], r["z_codes"][sl], r["z_scales"][sl], r["z_pre"])
            c2, s2 = fp4_compare(g["ki_codes"][sl], g["ki_scales"][sl], r["ki_codes"][sl], r["ki_scales"][sl], r["ki_pre"])
            n_code += c1 + c2
            n_scale += s1 + s2
        # entries outside this call untouched
        assert np.array_equal(g["z_codes"][:j0], r["z_codes"][:j0])
        assert np.array_equal(g["ki_scales"][j0 + n:], r["ki_scales"][j0 + n:])
        n_fp8 += e4m3_compare(g["window"][127:], r["window"][127:], r["win_pre"])
        assert np.array_equal(g["window"][:127], r["window"][:127])
        if ratio == 2 and (p0 + T) % 2 == 1:
            assert np.array_equal(w["pair_kc"][b].cpu().numpy(), r["pair"][0])
            assert np.array_equal(w["pair_gc"][b].cpu().numpy(), r["pair"][1])
    return n_code, n_scale, n_fp8


# ------------------------------------------------------------------------ writer
@pytest.mark.parametrize("B,T,p0s", [(3, 37, [0, 5, 130]), (1, 1, [0]), (2, 1, [7, 4096]), (1, 2, [1]),
                                     (2, 300, [0, 2001])])
def test_writer_small(handle, B, T, p0s):
    x, cap = make_state(B, T, p0s, seed=B * 100 + T)
    w = gpu_write(handle, x, p0s)
    n = check_write(w, oracle_write(x, p0s, cap), p0s, T)
    print(f"writer B={B} T={T}: boundary exceptions codes/scales/fp8 = {n}")


@pytest.mark.parametrize("name", ["prefill_4k", "chunk_32k"])
def test_writer_workloads(handle, name):
    wl = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(wl, DEV)
    w = gpu_write(handle, x, [wl.p0])
    n = check_write(w, oracle_write(x, [wl.p0], wl.cap), [wl.p0], wl.T)
    print(f"writer {name}: boundary exceptions codes/scales/fp8 = {n}")


# ------------------------------------------------------------------------ window roll
@pytest.mark.parametrize("B,T,T_next,inplace", [(2, 1, 1, True), (3, 5, 5, True), (1, 200, 40, True),
                                                (2, 300, 1, False), (2, 1, 64, False)])
def test_roll_window(handle, B, T, T_next, inplace):
    g = torch.Generator(device=DEV)
    g.manual_seed(1000 * B + T)
    win = inputs.random_e4m3((B, 127 + T, 512), g, DEV)
    want = win[:, T:T + 127].clone()
    if inplace:  # the same buffer: with B = 1 the next view may be shorter
        nxt = win.view(-1)[: B * (127 + T_next) * 512].view(B, 127 + T_next, 512)
    else:
        nxt = inputs.random_e4m3((B, 127 + T_next, 512), g, DEV)
    keep = nxt[:, 127:].clone()
    csa2.csa2_roll_window(handle, win, nxt)
    assert torch.equal(nxt[:, :127], want)
    assert torch.equal(nxt[:, 127:], keep)


def test_roll_window_rejects_shared_rows():
    h = csa2.csa2_create()
    win = torch.zeros(2, 127 + 3, 512, dtype=torch.uint8, device=DEV)
    nxt = win.view(-1)[: 2 * 128 * 512].view(2, 128, 512)  # one buffer, other strides: blocks would collide
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_roll_window(h, win, nxt)
    assert e.value.status == 1


def test_decode_steps_with_roll(handle):
    """Two decode steps (T = 1 each, the window rolled in between, the pair buffer carried) write
    the same caches, window rows and pair state as one two-token call of the oracle."""
    B, p0s = 2, [4001, 300]
    x, cap = make_state(B, 2, p0s, seed=51)
    ow = oracle_write(x, p0s, cap)
    w = {k: x[k].clone() for k in ("z_codes", "z_scales", "ki_codes", "ki_scales", "pair_kc", "pair_gc")}
    view = x["window"][:, :128].clone()  # rows of positions p0-127 .. p0
    for t in range(2):
        p = [q + t for q in p0s]
        csa2.csa2_write_cache(handle, x["kc"][:, t:t + 1].contiguous(), x["gc"][:, t:t + 1].contiguous(),
                              x["wa"][:, t:t + 1].contiguous(), x["gamma_c"], x["w_ik"], x["gamma_ik"], x["gamma_w"], p,
                              w["z_codes"], w["z_scales"], w["ki_codes"], w["ki_scales"], view, w["pair_kc"],
                              w["pair_gc"])
        if t == 0:
            csa2.csa2_roll_window(handle, view, view)
    for b, r in enumerate(ow):
        j0, n = r["first_entry"], r["n_entries"]
        for k in ("z_codes", "z_scales", "ki_codes", "ki_scales"):
            g = w[k][b].cpu().numpy()
            assert np.array_equal(g[:j0], r[k][:j0]) and np.array_equal(g[j0 + n:], r[k][j0 + n:])
        fp4_compare(w["z_codes"][b, j0:j0 + n].cpu().numpy(), w["z_scales"][b, j0:j0 + n].cpu().numpy(),
                    r["z_codes"][j0:j0 + n], r["z_scales"][j0:j0 + n], r["z_pre"])
        fp4_compare(w["ki_codes"][b, j0:j0 + n].cpu().numpy(), w["ki_scales"][b, j0:j0 + n].cpu().numpy(),
                    r["ki_codes"][j0:j0 + n], r["ki_scales"][j0:j0 + n], r["ki_pre"])
        # the view of the second call holds positions p0-126 .. p0+1 = oracle rows 1 .. 128
        gv = view[b].cpu().numpy()
        assert np.array_equal(gv[:126], r["window"][1:127])  # the caller's rows, moved
        e4m3_compare(gv[126:128], r["window"][127:129], r["win_pre"])  # positions p0, p0+1
        if (p0s[b] + 2) % 2 == 1:
            assert np.array_equal(w["pair_kc"][b].cpu().numpy(), r["pair"][0])


# ------------------------------------------------------------------------ indexer + top-k
def run_index(h, x, p0s, T):
    B = x["qi"].shape[0]
    idx = torch.empty(B, T, 512, dtype=torch.int32, device=DEV)
    top = torch.empty(B, T, 512, dtype=torch.float32, device=DEV)
    csa2.csa2_index_topk(h, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], p0s, idx, top)
    return idx, top


def check_index(idx, top, x, p0s, rows=None, ratio=2):
    B, T = idx.shape[:2]
    swaps = 0
    for b, p0 in enumerate(p0s):
        r = np.arange(T) if rows is None else np.asarray(rows)
        pos = p0 + r
        E = (pos + 1) // ratio
        kc = x["ki_codes"][b, : max(int(E.max()), 1)].cpu().numpy()
        ks = x["ki_scales"][b, : max(int(E.max()), 1)].cpu().numpy()
        sc = oracle.index_scores(pos, np32(x["qi"][b][r]), np32(x["wI"][b][r]), kc, ks, kc.shape[0], ratio=ratio)
        oidx, otop, kth = oracle.topk(sc, E)
        g = idx[b][r].cpu().numpy()
        swaps += topk_compare(g, oidx, sc, kth, E)
        # the reported scores are the fp32 scores of the chosen entries; a score is a sum of 32
        # signed terms, so its fp32 error scales with the row's score magnitude
        gt = top[b][r].cpu().numpy()
        for i in range(len(r)):
            k = min(512, int(E[i]))
            ref = sc[i, g[i, :k]]
            scale = np.abs(sc[i, : int(E[i])]).max() if E[i] else 0.0
            assert np.all(np.abs(gt[i, :k] - ref) <= 1e-5 * scale), f"row {r[i]} scores"
            assert np.all(np.isnan(gt[i, k:]))
    return swaps


def check_scores(g, x, p0s, ratio=2):
    """Every visible S^I of every row (GPU fp32, [B, T, ld]) against the oracle's fp64 scores,
    within 1e-5 of the row's largest |score| (a score is a signed sum of 32 fp32 terms).
    Returns the oracle's scores per sequence."""
    B, T = g.shape[:2]
    out = []
    for b, p0 in enumerate(p0s):
        pos = p0 + np.arange(T)
        E = (pos + 1) // ratio
        n = max(int(E.max()), 1)
        sc = oracle.index_scores(pos, np32(x["qi"][b]), np32(x["wI"][b]), x["ki_codes"][b, :n].cpu().numpy(),
                                 x["ki_scales"][b, :n].cpu().numpy(), n, ratio=ratio)
        gb = g[b].cpu().numpy().astype(np.float64)
        for t in range(T):
            e = int(E[t])
            if e == 0:
                continue
            err = np.abs(gb[t, :e] - sc[t, :e])
            bound = 1e-5 * np.abs(sc[t, :e]).max()
            bad = np.nonzero(err > bound)[0]
            assert not len(bad), (f"sequence {b} query {t}: {len(bad)} scores off, first entries {bad[:4].tolist()} "
                                  f"gpu {gb[t, bad[:4]].tolist()} oracle {sc[t, bad[:4]].tolist()}")
        out.append(sc)
    return out


def run_scores(h, x, p0s, T, ratio=2):
    B = x["qi"].shape[0]
    ld = ((int(((np.asarray(p0s) + T) // ratio).max()) + 3) // 4) * 4
    g = torch.full((B, T, max(ld, 4)), float("nan"), dtype=torch.float32, device=DEV)
    csa2.csa2_index_scores(h, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], p0s, g)
    return g


@pytest.mark.parametrize("B,T,p0s", [(1, 300, [0]), (2, 5, [1000, 37]), (3, 1, [0, 1, 4001]), (2, 64, [2000, 37]),
                                     (1, 1, [70001])])
def test_index_scores_small(handle, B, T, p0s):
    """S^I alone, every visible entry of every query: the tensor-core prefill scorer (T >= 8),
    the CUDA-core scorer (T < 8) and the decode scorer (T = 1)."""
    x, cap = make_state(B, T, p0s, seed=19 + T)
    g = run_scores(handle, x, p0s, T)
    check_scores(g, x, p0s)
    # entries beyond each query's visible count are left untouched
    for b, p0 in enumerate(p0s):
        for t in range(T):
            assert torch.isnan(g[b, t, (p0 + t + 1) // 2:]).all()


@pytest.mark.parametrize("name", ["decode_512k_r1", "decode_1m"])
def test_index_scores_repeated(handle, handle_r1, name):
    """Every S^I score of the two largest decode workloads (8 x 524288 entries), from ten calls
    in one process: each call must match the oracle and repeat the first call bit for bit.  The
    selected sets and their scores alone would miss a wrong score outside the top 512."""
    wl = inputs.WORKLOADS[name]
    h = handle_r1 if wl.ratio == 1 else handle
    x = inputs.workload_inputs(wl, DEV)
    p0s = [wl.p0] * wl.B
    first = run_scores(h, x, p0s, 1, wl.ratio)
    check_scores(first, x, p0s, wl.ratio)
    E = (wl.p0 + 1) // wl.ratio
    for k in range(9):
        g = run_scores(h, x, p0s, 1, wl.ratio)
        same = torch.equal(g[..., :E].view(torch.int32), first[..., :E].view(torch.int32))
        assert same, f"call {k + 2}: {(g[..., :E] != first[..., :E]).sum().item()} scores differ from the first call"


@pytest.mark.parametrize("B,T,p0s", [(2, 1, [3001, 1000]), (1, 300, [0]), (2, 64, [2000, 37]), (3, 1, [0, 1, 2]),
                                     (1, 1, [70001])])
def test_index_small(handle, B, T, p0s):
    x, cap = make_state(B, T, p0s, seed=7 + T)
    idx, top = run_index(handle, x, p0s, T)
    swaps = check_index(idx, top, x, p0s)
    print(f"index B={B} T={T}: near-tie swaps = {swaps}")


def test_index_exact_ties(handle):
    # identical keys give identical scores: the lower indices must win
    x, cap = make_state(1, 1, [4000], seed=3)
    x["ki_codes"][0, :2000] = x["ki_codes"][0, 5]
    x["ki_scales"][0, :2000] = x["ki_scales"][0, 5]
    idx, top = run_index(handle, x, [4000], 1)
    sc = oracle.index_scores(np.array([4000]), np32(x["qi"][0]), np32(x["wI"][0]), x["ki_codes"][0].cpu().numpy(),
                             x["ki_scales"][0].cpu().numpy(), cap)
    oidx, _, kth = oracle.topk(sc, np.array([2000]))
    assert np.array_equal(idx[0, 0].cpu().numpy(), oidx[0])


def test_index_long_prefill_rows_exact_ties(handle):
    # prefill rows of >= 16,384 entries take candidate lists instead of dense score rows; the first
    # 10,000 keys are identical, so the 512th score is shared by thousands of entries and the
    # lower indices must win, as in the oracle's (score desc, j asc) sort
    T, p0 = 16, 33000
    x, cap = make_state(1, T, [p0], seed=11)
    x["ki_codes"][0, :10000] = x["ki_codes"][0, 5]
    x["ki_scales"][0, :10000] = x["ki_scales"][0, 5]
    idx, top = run_index(handle, x, [p0], T)
    pos = p0 + np.arange(T)
    sc = oracle.index_scores(pos, np32(x["qi"][0]), np32(x["wI"][0]), x["ki_codes"][0].cpu().numpy(),
                             x["ki_scales"][0].cpu().numpy(), cap)
    oidx, _, _ = oracle.topk(sc, (pos + 1) // 2)
    assert np.array_equal(idx[0].cpu().numpy(), oidx)


@pytest.mark.parametrize("name", ["decode_8k", "decode_128k", "decode_1m", "prefill_4k"])
def test_index_workloads(handle, name):
    wl = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(wl, DEV)
    if wl.p0 == 0:  # prefill from scratch: the keys come from this step's writer (the oracle's)
        use_oracle_state(x, oracle_write(x, [wl.p0], wl.cap))
    idx, top = run_index(handle, x, [wl.p0] * wl.B, wl.T)
    swaps = check_index(idx, top, x, [wl.p0] * wl.B)
    print(f"index {name}: near-tie swaps = {swaps}")


def test_index_chunk_32k_sampled(handle):
    wl = inputs.WORKLOADS["chunk_32k"]
    x = inputs.workload_inputs(wl, DEV)
    use_oracle_state(x, oracle_write(x, [wl.p0], wl.cap))
    idx, top = run_index(handle, x, [wl.p0], wl.T)
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, 1, 2, wl.T - 2, wl.T - 1], rng.integers(0, wl.T, 19)]))
    swaps = check_index(idx, top, x, [wl.p0], rows=rows)
    print(f"index chunk_32k ({len(rows)} rows): near-tie swaps = {swaps}")


def test_tail_group_workspace(handle):
    # 130 sequences run as a group of 128 and a tail of 2; the tail takes more queries per pass
    # (indexer) and more splits (attention), so the workspace must cover it too
    B, T = 130, 1
    p0s = np.random.default_rng(2).integers(0, 900, B)
    x, cap = make_state(B, T, p0s, seed=21)
    use_oracle_state(x, oracle_write(x, p0s, cap))
    idx, top = run_index(handle, x, p0s, T)
    check_index(idx, top, x, p0s)
    out = run_attend(handle, x, idx, p0s)
    print(f"tail group: max abs / rel L2 = {check_attend(out, x, idx, p0s)}")


# ------------------------------------------------------------------------ FP4 scale domain
def wide_state(B, T, p0s, seed, scale_range):
    p0s = np.asarray(p0s, np.int64)
    cap = int(((p0s + T) // 2).max()) + 3
    x = {}
    x.update(inputs.layer_params(seed, DEV))
    x.update(inputs.step_inputs(B, T, seed, DEV))
    x.update(inputs.cache_state(B, T, int(p0s.max()), cap, seed, DEV, scale_range=scale_range))
    return x, cap


@pytest.mark.parametrize("B,T,p0s", [(2, 1, [6001, 3000]), (1, 40, [2000])])
def test_index_wide_scale_range(handle, B, T, p0s):
    """K^I scale bytes uniform over 100..140 (2^-27 .. 2^13, blocks of one key up to 40 binades
    apart): every score and the top-512 sets still match the oracle.  Scales from 2^-23 up
    decode exactly; below, values under 2^-24 round away, far inside the score tolerance."""
    x, cap = wide_state(B, T, p0s, 61 + T, (100, 140))
    check_scores(run_scores(handle, x, p0s, T), x, p0s)
    idx, top = run_index(handle, x, p0s, T)
    print(f"wide-scale index B={B} T={T}: near-tie swaps = {check_index(idx, top, x, p0s)}")
    assert csa2.csa2_check(handle) == 0


def test_attend_wide_scale_range(handle):
    """Z scale bytes uniform over 100..127 (2^-27 .. 2^0; the bf16 outputs keep the absolute
    tolerance meaningful): attention still matches the oracle."""
    B, T, p0s = 3, 1, [9000, 700, 64000]
    x, cap = wide_state(B, T, p0s, 71, (100, 127))
    idx = random_indices(B, T, p0s, seed=7, device=DEV)
    out = run_attend(handle, x, idx, p0s)
    print(f"wide-scale attend: max abs / rel L2 = {check_attend(out, x, idx, p0s)}")
    assert csa2.csa2_check(handle) == 0


def test_scale_domain_is_reported(handle):
    """An FP4 scale above 2^13 (byte 141) would overflow the fp16 tensor-core operands: the
    kernels that read one record it and csa2_check returns CSA2_ERR_UNSUPPORTED once."""
    B, T, p0s = 1, 1, [5000]
    x, cap = make_state(B, T, p0s, seed=81)
    assert csa2.csa2_check(handle) == 0
    x["ki_scales"][0, 1234, 2] = 140  # the largest supported scale: no report
    run_index(handle, x, p0s, T)
    assert csa2.csa2_check(handle) == 0
    x["ki_scales"][0, 1234, 2] = 141
    run_index(handle, x, p0s, T)
    assert csa2.csa2_check(handle) == 5
    assert csa2.csa2_check(handle) == 0  # cleared
    x["ki_scales"][0, 1234, 2] = 126
    idx = random_indices(B, T, p0s, seed=8, device=DEV)
    x["z_scales"][0, int(idx[0, 0, 3]), 7] = 141
    run_attend(handle, x, idx, p0s)
    assert csa2.csa2_check(handle) == 5
    x["z_scales"][0, int(idx[0, 0, 3]), 7] = 140
    run_attend(handle, x, idx, p0s)
    assert csa2.csa2_check(handle) == 0


# ------------------------------------------------------------------------ attention
def stratified_indices(B, T, p0s, seed):
    """Sorted distinct visible entries per query: one draw per stratum of width E/512."""
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    idx = torch.full((B, T, 512), -1, dtype=torch.int32, device=DEV)
    for b in range(B):
        E = (torch.arange(T, device=DEV, dtype=torch.int64) + int(p0s[b]) + 1) // 2
        s = torch.clamp(E // 512, min=1)
        i = torch.arange(512, device=DEV)
        cand = i[None, :] * s[:, None] + (torch.rand(T, 512, generator=g, device=DEV) * s[:, None]).long()
        ok = cand < E[:, None]
        idx[b] = torch.where(ok, cand, torch.full_like(cand, -1)).to(torch.int32)
    return idx


def run_attend(h, x, idx, p0s):
    B, T = x["q"].shape[:2]
    out = torch.empty(B, T, 64, 512, dtype=torch.bfloat16, device=DEV)
    csa2.csa2_attend(h, x["q"], x["sinks"], x["z_codes"], x["z_scales"], x["window"], idx, p0s, out)
    return out


def check_attend(out, x, idx, p0s, rows=None):
    B, T = out.shape[:2]
    errs = []
    for b, p0 in enumerate(p0s):
        r = np.arange(T) if rows is None else np.asarray(rows)
        ref = oracle.attend(p0 + r, np32(x["q"][b][r]), np32(x["sinks"]), x["z_codes"][b].cpu().numpy(),
                            x["z_scales"][b].cpu().numpy(), x["z_codes"].shape[1], x["window"][b].cpu().numpy(),
                            p0 - 127, idx[b][r].cpu().numpy())
        errs.append(out_compare(np32(out[b][r]), ref))
    return max(e[0] for e in errs), max(e[1] for e in errs)


@pytest.mark.parametrize("B,T,p0s", [(1, 300, [0]), (3, 1, [8192, 20, 0]), (2, 40, [1000, 5001]), (1, 1, [1])])
def test_attend_small(handle, B, T, p0s):
    x, cap = make_state(B, T, p0s, seed=11 + T)
    use_oracle_state(x, oracle_write(x, p0s, cap))  # this step's window rows and entries
    idx = random_indices(B, T, p0s, seed=5, device=DEV)
    out = run_attend(handle, x, idx, p0s)
    print(f"attend B={B} T={T}: max abs / rel L2 = {check_attend(out, x, idx, p0s)}")


@pytest.mark.parametrize("name", ["decode_8k", "decode_128k", "decode_1m", "prefill_4k", "chunk_32k"])
def test_attend_workloads(handle, name):
    wl = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(wl, DEV)
    p0s = [wl.p0] * wl.B
    use_oracle_state(x, oracle_write(x, p0s, wl.cap))
    idx = stratified_indices(wl.B, wl.T, p0s, seed=wl.seed)
    out = run_attend(handle, x, idx, p0s)
    rows = None
    if wl.T > 64:
        rng = np.random.default_rng(wl.seed)
        rows = np.unique(np.concatenate([[0, 1, 126, 127, 1023, wl.T - 1], rng.integers(0, wl.T, 58)]))
        rows = rows[rows < wl.T]
    print(f"attend {name}: max abs / rel L2 = {check_attend(out, x, idx, p0s, rows)}")


# ------------------------------------------------------------------------ whole step
@pytest.mark.parametrize("B,T,p0s", [(1, 700, [0]), (2, 1, [2049, 6000]), (2, 33, [1100, 77])])
def test_step_end_to_end(handle, B, T, p0s):
    """write -> index/top-k -> attend on the GPU vs the same chain in the oracle."""
    x, cap = make_state(B, T, p0s, seed=17 + T)
    g = gpu_write(handle, x, p0s)
    ow = oracle_write(x, p0s, cap)
    check_write(g, ow, p0s, T)
    xg = dict(x, **g)
    idx, top = run_index(handle, xg, p0s, T)
    out = run_attend(handle, xg, idx, p0s)
    for b, p0 in enumerate(p0s):
        pos = p0 + np.arange(T)
        E = (pos + 1) // 2
        r = ow[b]
        sc = oracle.index_scores(pos, np32(x["qi"][b]), np32(x["wI"][b]), r["ki_codes"], r["ki_scales"], cap)
        oidx, _, kth = oracle.topk(sc, E)
        gidx = idx[b].cpu().numpy()
        swaps = topk_compare(gidx, oidx, sc, kth, E)
        ref = oracle.attend(pos, np32(x["q"][b]), np32(x["sinks"]), r["z_codes"], r["z_scales"], cap, r["window"],
                            p0 - 127, oidx)
        same = np.array([np.array_equal(gidx[i], oidx[i]) for i in range(T)])
        mx, rl2 = out_compare(np32(out[b])[same], ref[same])
        print(f"step b={b}: swaps={swaps} rows compared={same.sum()} max abs={mx:.3g} rel L2={rl2:.3g}")


# ------------------------------------------------------------------------ bounded replay
@pytest.mark.parametrize("B,T,p0s,starts", [(3, 40, [1000, 5001, 300], [990, 5001, 0]), (2, 1, [8192, 130], [8150, 3])])
def test_attend_replay(handle, B, T, p0s, starts):
    x, cap = make_state(B, T, p0s, seed=31 + T)
    use_oracle_state(x, oracle_write(x, p0s, cap))
    idx = random_indices(B, T, p0s, seed=6, device=DEV)
    out = torch.empty(B, T, 64, 512, dtype=torch.bfloat16, device=DEV)
    csa2.csa2_attend_replay(handle, x["q"], x["sinks"], x["z_codes"], x["z_scales"], x["window"], idx, p0s, starts,
                            out)
    errs = []
    for b, (p0, s0) in enumerate(zip(p0s, starts)):
        pos = p0 + np.arange(T)
        ref = oracle.attend(pos, np32(x["q"][b]), np32(x["sinks"]), x["z_codes"][b].cpu().numpy(),
                            x["z_scales"][b].cpu().numpy(), x["z_codes"].shape[1], x["window"][b].cpu().numpy(),
                            p0 - 127, idx[b].cpu().numpy(), win_start=s0)
        errs.append(out_compare(np32(out[b]), ref))
    print(f"attend replay B={B} T={T}: max abs / rel L2 = {max(e[0] for e in errs)}, {max(e[1] for e in errs)}")
    # no replay (s = 0) is bit-identical to csa2_attend
    zero = torch.empty_like(out)
    csa2.csa2_attend_replay(handle, x["q"], x["sinks"], x["z_codes"], x["z_scales"], x["window"], idx, p0s, [0] * B,
                            zero)
    assert torch.equal(zero, run_attend(handle, x, idx, p0s))
    with pytest.raises(csa2.Csa2Error):  # a start after p0 is not a valid bound
        csa2.csa2_attend_replay(handle, x["q"], x["sinks"], x["z_codes"], x["z_scales"], x["window"], idx, p0s,
                                [p + 1 for p in p0s], zero)


# ------------------------------------------------------------------------ compression ratio 1
@pytest.mark.parametrize("B,T,p0s", [(3, 37, [0, 5, 130]), (1, 1, [0]), (2, 1, [7, 4096]), (2, 300, [0, 2001])])
def test_writer_small_ratio1(handle_r1, B, T, p0s):
    x, cap = make_state(B, T, p0s, seed=B * 100 + T + 1, ratio=1)
    w = gpu_write(handle_r1, x, p0s)
    n = check_write(w, oracle_write(x, p0s, cap, ratio=1), p0s, T, ratio=1)
    print(f"writer ratio 1 B={B} T={T}: boundary exceptions codes/scales/fp8 = {n}")


@pytest.mark.parametrize("B,T,p0s", [(2, 1, [3001, 1000]), (1, 300, [0]), (2, 64, [2000, 37]), (3, 1, [0, 1, 2])])
def test_index_small_ratio1(handle_r1, B, T, p0s):
    x, cap = make_state(B, T, p0s, seed=9 + T, ratio=1)
    idx, top = run_index(handle_r1, x, p0s, T)
    swaps = check_index(idx, top, x, p0s, ratio=1)
    print(f"index ratio 1 B={B} T={T}: near-tie swaps = {swaps}")


@pytest.mark.parametrize("name", ["decode_512k_r1", "prefill_4k_r1"])
def test_index_workloads_ratio1(handle_r1, name):
    wl = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(wl, DEV)
    rows = None
    if wl.p0 == 0:  # prefill from scratch: the keys come from this step's writer (the oracle's)
        use_oracle_state(x, oracle_write(x, [wl.p0], wl.cap, ratio=1))
        rng = np.random.default_rng(wl.seed)
        rows = np.unique(np.concatenate([[0, 1, 510, 511, 512, wl.T - 1], rng.integers(0, wl.T, 40)]))
    idx, top = run_index(handle_r1, x, [wl.p0] * wl.B, wl.T)
    swaps = check_index(idx, top, x, [wl.p0] * wl.B, rows=rows, ratio=1)
    print(f"index {name}: near-tie swaps = {swaps}")


def test_step_end_to_end_ratio1(handle_r1):
    B, T, p0s = 2, 33, [1100, 77]
    x, cap = make_state(B, T, p0s, seed=23, ratio=1)
    g = gpu_write(handle_r1, x, p0s)
    ow = oracle_write(x, p0s, cap, ratio=1)
    check_write(g, ow, p0s, T, ratio=1)
    xg = dict(x, **g)
    idx, top = run_index(handle_r1, xg, p0s, T)
    out = run_attend(handle_r1, xg, idx, p0s)
    for b, p0 in enumerate(p0s):
        pos = p0 + np.arange(T)
        E = pos + 1
        r = ow[b]
        sc = oracle.index_scores(pos, np32(x["qi"][b]), np32(x["wI"][b]), r["ki_codes"], r["ki_scales"], cap, ratio=1)
        oidx, _, kth = oracle.topk(sc, E)
        gidx = idx[b].cpu().numpy()
        swaps = topk_compare(gidx, oidx, sc, kth, E)
        ref = oracle.attend(pos, np32(x["q"][b]), np32(x["sinks"]), r["z_codes"], r["z_scales"], cap, r["window"],
                            p0 - 127, oidx)
        same = np.array([np.array_equal(gidx[i], oidx[i]) for i in range(T)])
        mx, rl2 = out_compare(np32(out[b])[same], ref[same])
        print(f"step ratio 1 b={b}: swaps={swaps} rows compared={same.sum()} max abs={mx:.3g} rel L2={rl2:.3g}")


# ------------------------------------------------------------------------ argument errors
def test_argument_errors(handle):
    x, cap = make_state(1, 4, [0], seed=1)
    idx = torch.empty(1, 4, 512, dtype=torch.int32, device=DEV)
    with pytest.raises(csa2.Csa2Error) as e:   # cache too small for the visible entries
        csa2.csa2_index_topk(handle, x["qi"], x["wI"], x["ki_codes"][:, :1], x["ki_scales"][:, :1], [100], idx)
    assert e.value.status == 2
    with pytest.raises(csa2.Csa2Error) as e:   # workspace too small
        csa2.csa2_index_topk(handle, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], [0], idx,
                             ws=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert e.value.status == 4
    with pytest.raises(csa2.Csa2Error) as e:   # odd p0 without a pair buffer
        csa2.csa2_write_cache(handle, x["kc"], x["gc"], x["wa"], x["gamma_c"], x["w_ik"], x["gamma_ik"], x["gamma_w"],
                              [1], x["z_codes"], x["z_scales"], x["ki_codes"], x["ki_scales"], x["window"])
    assert e.value.status == 1
    out = torch.empty(4 * 64 * 512 + 8, dtype=torch.bfloat16, device=DEV)
    mis = out.view(-1)[1:1 + 4 * 64 * 512].view(1, 4, 64, 512)  # 2-byte offset: misaligned
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_attend(handle, x["q"], x["sinks"], x["z_codes"], x["z_scales"], x["window"], idx, [0], mis)
    assert e.value.status == 3
