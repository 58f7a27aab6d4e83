"""Pins of the fp64 oracle against what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: a format definition, a
library routine (torch's float8_e4m3fn cast, torch's scaled_dot_product_attention), a closed
form, an invariant, a hand-derived table or a brute force on tiny inputs.
"""
import math
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle

GOLDEN = Path(__file__).resolve().parent / "golden" / "pages_figures.txt"


def golden():
    out = {}
    for line in GOLDEN.read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        name, rest = line.split("=", 1)
        out[name.strip()] = float(rest.split("|")[0])
    return out


# ---------------------------------------------------------------- E2M1
def test_e2m1_decode_matches_format_definition():
    # E2M1: value = (-1)^s * 2^(E-1) * (1 + M/2) for E > 0, (-1)^s * M/2 for E = 0.
    for code in range(16):
        s, E, M = code >> 3, (code >> 1) & 3, code & 1
        want = (M / 2 if E == 0 else 2.0 ** (E - 1) * (1 + M / 2)) * (-1) ** s
        assert oracle.e2m1_value(code) == want


# nearest E2M1 value, ties to the even code (hand-derived from the grid 0 .5 1 1.5 2 3 4 6)
E2M1_TABLE = [(0.0, 0), (0.2, 0), (0.25, 0), (0.26, 1), (0.5, 1), (0.74, 1), (0.75, 2), (1.0, 2),
              (1.25, 2), (1.26, 3), (1.74, 3), (1.75, 4), (2.49, 4), (2.5, 4), (2.51, 5), (3.49, 5),
              (3.5, 6), (4.99, 6), (5.0, 6), (5.01, 7), (6.0, 7), (100.0, 7), (-0.3, 9), (-0.0, 8),
              (-5.0, 14), (-1e9, 15)]


@pytest.mark.parametrize("x,code", E2M1_TABLE)
def test_e2m1_encode_rounding_table(x, code):
    assert oracle.e2m1_encode(x) == code


def test_mx_block_scale_rule_and_nearest_codes():
    rng = np.random.default_rng(1)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    for trial in range(200):
        v = rng.standard_normal(64) * 10.0 ** rng.uniform(-3, 3)
        codes, scales = oracle.mx_quantize(v[None])
        deq = oracle.mx_dequantize(codes, scales)[0]
        for b in range(2):
            blk = v[32 * b:32 * b + 32]
            e = int(scales[0, b]) - 127
            amax = np.abs(blk).max()
            # OCP MX: X = 2^(floor(log2 amax) - emax), emax(E2M1) = 2  ->  amax / X in [4, 8)
            assert 4.0 <= amax / 2.0 ** e < 8.0
            # brute force: each element is the grid point nearest to |v|/X (clamped to 6)
            a = np.abs(blk) / 2.0 ** e
            best = grid[np.argmin(np.abs(a[:, None] - grid[None, :]), axis=1)]
            assert np.array_equal(np.abs(deq[32 * b:32 * b + 32]) / 2.0 ** e, best)
            assert np.all(np.sign(deq[32 * b:32 * b + 32]) * np.sign(blk) >= 0)


def test_mx_all_zero_block_and_packing_order():
    codes, scales = oracle.mx_quantize(np.zeros((1, 32)))
    assert scales[0, 0] == 0 and not codes.any()
    v = np.zeros(32)
    v[0], v[1] = 4.0, -1.0   # amax 4 -> X = 1; codes 6 and 0xA, element 0 in the low nibble
    codes, scales = oracle.mx_quantize(v[None])
    assert scales[0, 0] == 127 and codes[0, 0] == (6 | (0xA << 4))


# ---------------------------------------------------------------- E4M3
def test_e4m3_decode_matches_torch_for_all_codes():
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(400_000) * 10.0 ** rng.uniform(-4, 2.6, 400_000),
                        [0.0, -0.0, 2.0 ** -10, 2.0 ** -9.5, 2.0 ** -6, 447.9, 440.0, 416.0, -432.0]])
    x = x[np.abs(x) < 448.0]
    mine = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)
    # exact midpoints between neighbours round to the even code
    vals = np.array([oracle.e4m3_value(c) for c in range(127)])
    mids = (vals[:-1] + vals[1:]) / 2
    enc = oracle.e4m3_encode(mids)
    assert np.all(enc % 2 == 0)
    assert np.array_equal(enc, torch.from_numpy(mids).to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_e4m3_saturates():
    assert list(oracle.e4m3_encode(np.array([448.0, 470.0, 1e6, -500.0]))) == [0x7E, 0x7E, 0x7E, 0xFE]


# ---------------------------------------------------------------- RMSNorm, RoPE
def test_rmsnorm_unit_mean_square_and_bound():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(512) * 7.0
    g = (1 + 0.1 * rng.standard_normal(512)).astype(np.float32)
    y = oracle.rmsnorm(x, g)
    assert abs(np.mean((y / g) ** 2) - 1.0) < 1e-12
    # the bound behind "no number above about 22.6": |y_i| <= sqrt(512) * max|gamma|
    assert np.abs(y).max() <= math.sqrt(512) * np.abs(g).max()
    spike = np.zeros(512)
    spike[7] = 3.0
    assert abs(oracle.rmsnorm(spike, np.ones(512, np.float32))[7] - math.sqrt(512)) < 1e-9
    assert abs(math.sqrt(512) - golden()["value_bound_after_norm"]) < 0.05


def test_rope_norm_inverse_and_relative_position():
    rng = np.random.default_rng(4)
    x, y = rng.standard_normal(64), rng.standard_normal(64)
    r = oracle.rope(x, 12345)
    for i in range(32):
        assert abs(np.hypot(*r[2 * i:2 * i + 2]) - np.hypot(*x[2 * i:2 * i + 2])) < 1e-12
    assert np.allclose(oracle.rope(r, 12345, inverse=True), x, atol=1e-12)
    # <R_a x, R_b y> depends only on b - a
    d1 = oracle.rope(x, 100) @ oracle.rope(y, 130)
    d2 = oracle.rope(x, 7000) @ oracle.rope(y, 7030)
    assert abs(d1 - d2) < 1e-9
    # interleaved pairs, theta_i = 10000^(-2i/64): pair i of a unit vector turns by pos*theta_i
    e = np.zeros(64)
    e[0::2] = 1.0
    r = oracle.rope(e, 3)
    for i in (0, 1, 17, 31):
        th = 3 * 10000.0 ** (-2 * i / 64)
        assert abs(r[2 * i] - math.cos(th)) < 1e-12 and abs(r[2 * i + 1] - math.sin(th)) < 1e-12


# ---------------------------------------------------------------- writer
def _writer_params(identity_wik=False, seed=0):
    rng = np.random.default_rng(seed)
    if identity_wik:
        w = np.zeros((512, 128), np.float32)
        w[np.arange(128), np.arange(128)] = 1.0
        return dict(gamma_c=np.ones(512, np.float32), w_ik=w, gamma_ik=np.ones(128, np.float32),
                    gamma_w=np.ones(512, np.float32))
    return dict(gamma_c=(1 + 0.1 * rng.standard_normal(512)).astype(np.float32),
                w_ik=(rng.standard_normal((512, 128)) / math.sqrt(512)).astype(np.float32),
                gamma_ik=(1 + 0.1 * rng.standard_normal(128)).astype(np.float32),
                gamma_w=(1 + 0.1 * rng.standard_normal(512)).astype(np.float32))


def test_writer_constant_inputs_closed_form():
    # k^c = g^c-independent ones: k^p = 1, c = 1, Z(j=0) = 1 -> scale 2^-2 (byte 125), code 6
    T = 2
    ones = np.ones((T, 512), np.float32)
    gc = np.random.default_rng(0).standard_normal((T, 512)).astype(np.float32)
    r = oracle.write_seq(ones, gc, ones, p0=0, cap=1, **_writer_params(identity_wik=True))
    assert r["n_entries"] == 1
    assert np.all(r["z_codes"][0] == 0x66) and np.all(r["z_scales"][0] == 125)
    assert np.all(r["ki_codes"][0] == 0x66) and np.all(r["ki_scales"][0] == 125)
    # window row of token 0 (position 0, no rotation): 1.0 in E4M3 is 0x38
    assert np.all(r["window"][127] == 0x38)
    # token 1 is rotated by angle 1*theta_i on dims 448..511: pair i = (cos - sin, sin + cos)
    pre = r["win_pre"][1, 448:]
    th = 10000.0 ** (-2 * np.arange(32) / 64)
    assert np.allclose(pre[0::2], np.cos(th) - np.sin(th), atol=1e-12)
    assert np.allclose(pre[1::2], np.sin(th) + np.cos(th), atol=1e-12)


def test_writer_pair_pool_weights():
    rng = np.random.default_rng(5)
    k = rng.standard_normal(512).astype(np.float32)
    gc = rng.standard_normal((2, 512)).astype(np.float32) * 5
    prm = _writer_params(identity_wik=True)
    # equal tokens: any softmax weights summing to 1 give k^p = k
    r = oracle.write_seq(np.stack([k, k]), gc, np.ones((2, 512), np.float32), p0=0, cap=1, **prm)
    want = k / np.sqrt(np.mean(k.astype(np.float64) ** 2))
    assert np.allclose(r["z_pre"][0], want, atol=1e-12)   # j = 0: RoPE is the identity
    # equal gates: plain mean of the two tokens; a dominant gate selects its token
    k2 = rng.standard_normal((2, 512)).astype(np.float32)
    for g0, g1, kp in ((0.0, 0.0, k2.mean(0)), (40.0, -40.0, k2[0]), (-40.0, 40.0, k2[1])):
        gcs = np.stack([np.full(512, g0), np.full(512, g1)]).astype(np.float32)
        r = oracle.write_seq(k2, gcs, np.ones((2, 512), np.float32), p0=0, cap=1, **prm)
        kp = kp.astype(np.float64)
        assert np.allclose(r["z_pre"][0], kp / np.sqrt(np.mean(kp ** 2)), atol=1e-10)
    # per-channel weights: the pooled value lies between the two token values
    r0 = oracle.write_seq(k2, gc, np.ones((2, 512), np.float32), p0=0, cap=1, **prm)
    lo, hi = np.minimum(k2[0], k2[1])[:448], np.maximum(k2[0], k2[1])[:448]
    w0 = 1 / (1 + np.exp(gc[1].astype(np.float64) - gc[0]))
    rms = np.sqrt(np.mean((w0 * k2[0] + (1 - w0) * k2[1]) ** 2))
    kp_back = r0["z_pre"][0][:448] * rms
    assert np.all(kp_back >= lo - 1e-9) and np.all(kp_back <= hi + 1e-9)


def test_writer_entries_and_pair_buffer_split_calls():
    # one call over T tokens == two calls split at an odd boundary through the pair buffer
    rng = np.random.default_rng(6)
    T = 21
    kc, gc, wa = (rng.standard_normal((T, 512)).astype(np.float32) for _ in range(3))
    prm = _writer_params(seed=6)
    full = oracle.write_seq(kc, gc, wa, p0=0, cap=16, **prm)
    a = oracle.write_seq(kc[:7], gc[:7], wa[:7], p0=0, cap=16, **prm)
    assert a["pair"] is not None and a["n_entries"] == 3
    b = oracle.write_seq(kc[7:], gc[7:], wa[7:], p0=7, cap=16, z_codes=a["z_codes"], z_scales=a["z_scales"],
                         ki_codes=a["ki_codes"], ki_scales=a["ki_scales"], pair_k=a["pair"][0],
                         pair_g=a["pair"][1], **prm)
    assert b["first_entry"] == 3 and b["n_entries"] == 7
    for k in ("z_codes", "z_scales", "ki_codes", "ki_scales"):
        assert np.array_equal(full[k][:10], b[k][:10])
    assert np.array_equal(full["window"][127 + 7:], b["window"][127:])
    assert full["n_entries"] == T // 2


def test_writer_ratio1_matches_ratio2_pool_of_equal_tokens():
    # Compression ratio 1 (decoder owner layers): entry j is token j itself, rotated by j.
    # A ratio-2 entry m pooled from two copies of the same token has softmax weights summing
    # to 1, so it equals that token's ratio-1 entry when both are rotated by the same position:
    # ratio-1 entry 2m (token at position 2m) vs ratio-2 entry m (tokens 2m, 2m+1 equal).
    rng = np.random.default_rng(11)
    T = 8
    kc = rng.standard_normal((T, 512)).astype(np.float32)
    gc = rng.standard_normal((T, 512)).astype(np.float32)
    wa = rng.standard_normal((T, 512)).astype(np.float32)
    prm = _writer_params(seed=11)
    r1 = oracle.write_seq(kc, gc, wa, p0=0, cap=T, ratio=1, **prm)
    assert r1["n_entries"] == T and r1["first_entry"] == 0 and r1["pair"] is None
    kc2 = np.repeat(kc[0::2], 2, axis=0)   # tokens 2m and 2m+1 both = token 2m
    gc2 = rng.standard_normal((T, 512)).astype(np.float32)  # any gates: the weights sum to 1
    r2 = oracle.write_seq(kc2, gc2, wa, p0=0, cap=T, ratio=2, **prm)
    assert r2["n_entries"] == T // 2
    # equal up to fp64 rounding of the pooled sum (w0 k + w1 k vs k)
    assert np.allclose(r1["z_pre"][0::2], r2["z_pre"], rtol=0, atol=1e-12)
    assert np.allclose(r1["ki_pre"][0::2], r2["ki_pre"], rtol=0, atol=1e-12)
    # the window does not depend on the ratio
    assert np.array_equal(r1["window"], r2["window"])


def test_writer_ratio1_ignores_gates_and_splits_anywhere():
    rng = np.random.default_rng(12)
    T = 9
    kc, gc, wa = (rng.standard_normal((T, 512)).astype(np.float32) for _ in range(3))
    prm = _writer_params(seed=12)
    full = oracle.write_seq(kc, gc, wa, p0=5, cap=20, ratio=1, **prm)
    other_gates = oracle.write_seq(kc, -3 * gc, wa, p0=5, cap=20, ratio=1, **prm)
    for k in ("z_codes", "z_scales", "ki_codes", "ki_scales"):
        assert np.array_equal(full[k], other_gates[k])
    assert full["first_entry"] == 5 and full["n_entries"] == T
    # entries are single tokens: any split point, no pair buffer
    a = oracle.write_seq(kc[:4], gc[:4], wa[:4], p0=5, cap=20, ratio=1, **prm)
    b = oracle.write_seq(kc[4:], gc[4:], wa[4:], p0=9, cap=20, ratio=1, z_codes=a["z_codes"],
                         z_scales=a["z_scales"], ki_codes=a["ki_codes"], ki_scales=a["ki_scales"], **prm)
    for k in ("z_codes", "z_scales", "ki_codes", "ki_scales"):
        assert np.array_equal(full[k], b[k])


# The indexer-key chain of [PG] "Compressed sparse attention": k^i = c W_IK (c is the
# normalised pooled key before RoPE and FP4), k^n = gamma_IK * RMSNorm(k^i), and dims 64..127
# of K^I rotated by the entry's position (2j at ratio 2, j at ratio 1).  The inputs below make
# each stage a closed form: a pair of equal tokens of +-1 values pools to itself (the softmax
# weights sum to 1) and has mean square 1, so c = gamma_C * k exactly.
def _pm1_tokens(rng, T):
    k = np.where(rng.random(512) < 0.5, -1.0, 1.0).astype(np.float32)
    return np.repeat(k[None], T, axis=0), k.astype(np.float64)


def _rot_pairs(x, pos):
    """Dims 64..127 of x turned pair by pair by pos * 10000^(-2i/64), cos/sin written out."""
    y = np.array(x, np.float64)
    for i in range(32):
        a = pos * 10000.0 ** (-2.0 * i / 64)
        x0, x1 = x[64 + 2 * i], x[65 + 2 * i]
        y[64 + 2 * i] = x0 * math.cos(a) - x1 * math.sin(a)
        y[65 + 2 * i] = x0 * math.sin(a) + x1 * math.cos(a)
    return y


@pytest.mark.parametrize("ratio,p0,T,rope_pos", [(2, 10, 2, 10), (2, 2047, 1, 2046), (1, 7, 1, 7)])
def test_indexer_key_chain_single_tap_projection(ratio, p0, T, rope_pos):
    # W_IK with one tap per column: column o reads row r_o with weight a_o = +-0.5.  Columns
    # 0..63 read the rotated dims 448..511 of c (a permutation of them), so a k^i taken from Z
    # (after RoPE) would differ; the other columns read distinct rows below 448.  Then
    # k^i[o] = a_o c[r_o] = +-0.5, its mean square is 0.25, and k^n[o] = gamma_IK[o] * sign.
    rng = np.random.default_rng(40 + p0)
    kc, k = _pm1_tokens(rng, T)
    gc = rng.standard_normal((T, 512)).astype(np.float32) * 3
    rows = np.concatenate([448 + rng.permutation(64), rng.choice(448, 64, replace=False)])
    a = np.where(rng.random(128) < 0.5, -0.5, 0.5)
    w = np.zeros((512, 128), np.float32)
    w[rows, np.arange(128)] = a
    g_ik = (1 + 0.2 * rng.standard_normal(128)).astype(np.float32)
    prm = dict(gamma_c=np.ones(512, np.float32), w_ik=w, gamma_ik=g_ik, gamma_w=np.ones(512, np.float32))
    pair = dict(pair_k=kc[0], pair_g=gc[0]) if ratio == 2 and p0 % 2 else {}
    r = oracle.write_seq(kc, gc, kc, p0=p0, cap=p0 // ratio + 1, ratio=ratio, **pair, **prm)
    assert r["n_entries"] == 1 and r["first_entry"] * ratio == rope_pos
    kn = g_ik.astype(np.float64) * np.sign(a * k[rows])
    assert np.allclose(r["ki_pre"][0], _rot_pairs(kn, rope_pos), rtol=0, atol=1e-12)


def test_indexer_key_chain_dense_projection():
    # A dense, non-symmetric W_IK and a non-uniform gamma_C: k^i = (gamma_C * k) W_IK (a
    # library matmul), and after undoing the rotation of dims 64..127 by 2j (cos/sin written
    # out) and dividing by gamma_IK, K^I is k^i scaled to unit mean square.
    rng = np.random.default_rng(41)
    kc, k = _pm1_tokens(rng, 2)
    gc = rng.standard_normal((2, 512)).astype(np.float32)
    g_c = (1 + 0.3 * rng.standard_normal(512)).astype(np.float32)
    w = (rng.standard_normal((512, 128)) / math.sqrt(512)).astype(np.float32)
    g_ik = (1 + 0.2 * rng.standard_normal(128)).astype(np.float32)
    r = oracle.write_seq(kc, gc, kc, g_c, w, g_ik, np.ones(512, np.float32), p0=6, cap=4)
    j = r["first_entry"]
    assert j == 3 and r["n_entries"] == 1
    u = _rot_pairs(r["ki_pre"][0], -2 * j) / g_ik.astype(np.float64)
    ki = (g_c.astype(np.float64) * k) @ w.astype(np.float64)
    assert abs(np.mean(u ** 2) - 1.0) < 1e-12
    cos = u @ ki / (np.linalg.norm(u) * np.linalg.norm(ki))
    assert abs(cos - 1.0) < 1e-12
    # Z rows hold c rotated by 2j on dims 448..511 (c = gamma_C * k here)
    zc = g_c.astype(np.float64) * k
    z = np.concatenate([zc[:448], _rot_pairs(np.concatenate([np.zeros(64), zc[448:]]), 2 * j)[64:]])
    assert np.allclose(r["z_pre"][0], z, rtol=0, atol=1e-12)


def test_index_causal_bound_ratio1():
    rng = np.random.default_rng(13)
    kc, ks = oracle.mx_quantize(rng.standard_normal((60, 128)))
    pos = np.array([0, 1, 2, 58, 59])
    s = oracle.index_scores(pos, rng.standard_normal((5, 32, 128)).astype(np.float32),
                            rng.standard_normal((5, 32)).astype(np.float32), kc, ks, 60, ratio=1)
    for r, p in enumerate(pos):
        E = p + 1   # at ratio 1 every token is an entry: j <= t
        assert np.all(np.isfinite(s[r, :E])) and np.all(np.isnan(s[r, E:]))
    # the same keys at ratio 2 see only floor((t+1)/2) of them
    s2 = oracle.index_scores(pos, rng.standard_normal((5, 32, 128)).astype(np.float32),
                             rng.standard_normal((5, 32)).astype(np.float32), kc, ks, 60, ratio=2)
    assert np.isnan(s2[-1, 30:]).all() and np.isfinite(s2[-1, :30]).all()


# ---------------------------------------------------------------- indexer + top-k
def _const_keys(vals):
    """K^I rows whose 128 values all equal vals[j] (a value on the E2M1 grid, scale 1)."""
    v = np.repeat(np.asarray(vals, np.float64)[:, None], 128, axis=1)
    return oracle.mx_quantize(v)


def test_index_scores_closed_form():
    # keys j: all values c_j; Q^I heads 0..15 all +1, heads 16..31 all -1 (exact in FP4);
    # w^I = 2^-h.  q_h . k_j = +-128 c_j, so S_j = 128 |c_j| * sum over the heads of the sign
    # of c_j of 2^-h.
    c = np.array([0.5, -1.0, 1.5, -2.0, 3.0, -4.0, 6.0, 0.0, -0.5, 1.0])
    kc, ks = _const_keys(c * 2.0 ** -3)   # scale 2^-3 to exercise the block scale
    qi = np.ones((1, 32, 128), np.float32)
    qi[0, 16:] = -1.0
    wI = (2.0 ** -np.arange(32)).astype(np.float32)[None]
    pos = np.array([2 * len(c) - 1])
    s = oracle.index_scores(pos, qi, wI, kc, ks, len(c))[0]
    pos_w, neg_w = wI[0, :16].sum(), wI[0, 16:].sum()
    want = 128 * np.abs(c) * 2.0 ** -3 * np.where(c > 0, pos_w, neg_w)
    assert np.array_equal(s, want)


def test_index_causal_bound():
    rng = np.random.default_rng(7)
    kc, ks = oracle.mx_quantize(rng.standard_normal((50, 128)))
    pos = np.array([0, 1, 2, 3, 98, 99])
    s = oracle.index_scores(pos, rng.standard_normal((6, 32, 128)).astype(np.float32),
                            rng.standard_normal((6, 32)).astype(np.float32), kc, ks, 50)
    for r, p in enumerate(pos):
        E = (p + 1) // 2   # entry j is visible once token 2j+1 has arrived: j < floor((t+1)/2)
        assert np.all(np.isfinite(s[r, :E])) and np.all(np.isnan(s[r, E:]))
    with pytest.raises(ValueError):
        oracle.index_scores(np.array([101]), np.zeros((1, 32, 128), np.float32), np.zeros((1, 32), np.float32),
                            kc, ks, 50)


def test_topk_known_permutation_ties_and_short_rows():
    rng = np.random.default_rng(8)
    n = 3000
    perm = rng.permutation(n).astype(np.float64)   # distinct scores: the top 512 are known
    idx, top, kth = oracle.topk(perm[None], np.array([n]))
    assert np.array_equal(idx[0], np.sort(np.argsort(-perm)[:512]))
    assert kth[0, 0] == n - 512 and kth[0, 1] == n - 513
    # all equal: the lowest 512 indices win
    idx, _, _ = oracle.topk(np.full((1, 900), 0.25), np.array([900]))
    assert np.array_equal(idx[0], np.arange(512))
    # -0 equals +0
    s = np.zeros(600)
    s[::2] = -0.0
    idx, _, _ = oracle.topk(s[None], np.array([600]))
    assert np.array_equal(idx[0], np.arange(512))
    # fewer than 512 candidates: all kept, ascending, -1 padded
    idx, top, kth = oracle.topk(rng.standard_normal((1, 100)), np.array([100]))
    assert np.array_equal(idx[0, :100], np.arange(100)) and np.all(idx[0, 100:] == -1)
    assert np.isnan(kth[0]).all()
    # brute force on a tiny row with duplicates: every chosen score >= every unchosen one,
    # and within a tied value the chosen indices are the lowest ones
    s = rng.integers(0, 40, 700).astype(np.float64)
    idx, _, _ = oracle.topk(s[None], np.array([700]))
    chosen = idx[0]
    rest = np.setdiff1d(np.arange(700), chosen)
    assert s[chosen].min() >= s[rest].max()
    v = s[chosen].min()
    tied = np.flatnonzero(s == v)
    assert np.array_equal(np.intersect1d(tied, chosen), tied[:np.sum(s[chosen] == v)])


# ---------------------------------------------------------------- attention
def _attend_case(nq=3, seed=9, p=2000, n_entries=1200):
    rng = np.random.default_rng(seed)
    zc, zs = oracle.mx_quantize(rng.standard_normal((n_entries, 512)))
    win = oracle.e4m3_encode(rng.standard_normal((128, 512))).reshape(128, 512)
    q = rng.standard_normal((nq, 64, 512)).astype(np.float32)
    sinks = rng.standard_normal(64).astype(np.float32)
    idx = np.stack([np.sort(rng.choice(n_entries, 512, replace=False)) for _ in range(nq)]).astype(np.int32)
    pos = np.full(nq, p)
    return zc, zs, win, q, sinks, idx, pos


def _gathered(zc, zs, win, idx_row):
    G_w = np.vectorize(oracle.e4m3_value)(win.astype(np.int64))
    G_z = oracle.mx_dequantize(zc[idx_row], zs[idx_row])
    return np.concatenate([G_w, G_z])


def test_attend_matches_sdpa_with_sink_row():
    zc, zs, win, q, sinks, idx, pos = _attend_case()
    out, mass, nrows = oracle.attend(pos, q, sinks, zc, zs, len(zc), win, pos[0] - 127, idx, return_mass=True)
    assert np.all(nrows == 640) and golden()["attended_rows"] == 640 == 128 + 512
    for r in range(len(pos)):
        G = torch.from_numpy(_gathered(zc, zs, win, idx[r]))
        # a zero key/value row whose logit is s_h carries the sink: exp(s_h) joins the
        # denominator and adds nothing to the numerator
        K = torch.cat([G, torch.zeros(1, 512, dtype=torch.float64)])
        mask = torch.zeros(64, 1, K.shape[0], dtype=torch.float64)
        mask[:, 0, -1] = torch.from_numpy(sinks.astype(np.float64))
        Q = torch.from_numpy(q[r].astype(np.float64))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K[None].expand(64, -1, -1), K[None].expand(64, -1, -1),
                                                               attn_mask=mask)[:, 0, :].numpy()
        ref = np.stack([np.concatenate([ref[h, :448], oracle.rope(ref[h, 448:], pos[r], inverse=True)]) for h in range(64)])
        assert np.abs(out[r] - ref).max() < 1e-12
        assert np.all(mass[r] < 1.0)


def test_attend_without_sink_is_softmax_attention_and_single_row_closed_form():
    zc, zs, win, q, sinks, idx, pos = _attend_case(nq=1, seed=10)
    out = oracle.attend(pos, q, np.full(64, -1e4, np.float32), zc, zs, len(zc), win, pos[0] - 127, idx)
    G = torch.from_numpy(_gathered(zc, zs, win, idx[0]))
    Q = torch.from_numpy(q[0].astype(np.float64))[:, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, G[None].expand(64, -1, -1), G[None].expand(64, -1, -1))
    ref = ref[:, 0].numpy()
    ref[:, 448:] = np.stack([oracle.rope(ref[h, 448:], pos[0], inverse=True) for h in range(64)])
    assert np.abs(out[0] - ref).max() < 1e-12
    # position 0, no selected entries: one window row, A = e^S / (e^s + e^S)
    rng = np.random.default_rng(11)
    win = oracle.e4m3_encode(rng.standard_normal((128, 512))).reshape(128, 512)
    q = rng.standard_normal((1, 64, 512)).astype(np.float32)
    sinks = rng.standard_normal(64).astype(np.float32)
    out, mass, nrows = oracle.attend(np.array([0]), q, sinks, zc, zs, len(zc), win, -127,
                                     np.full((1, 512), -1, np.int32), return_mass=True)
    g = np.array([oracle.e4m3_value(c) for c in win[127]])
    S = q[0].astype(np.float64) @ g / math.sqrt(512)
    A = np.exp(S) / (np.exp(sinks.astype(np.float64)) + np.exp(S))
    assert nrows[0] == 1
    assert np.allclose(mass[0], A, rtol=1e-13, atol=0)
    assert np.allclose(out[0], A[:, None] * g[None], rtol=1e-12, atol=1e-15)   # position 0: no rotation


def test_attend_row_counts():
    zc, zs, win, q, sinks, idx, _ = _attend_case(nq=1)
    # |G_t| = min(128, t+1) window rows + min(512, floor((t+1)/2)) selected entries
    for p, want in ((0, 1), (5, 9), (126, 190), (127, 192), (1022, 639), (1023, 640), (1500, 640)):
        wrows = np.zeros((128, 512), np.uint8)
        E = (p + 1) // 2
        sel = np.full((1, 512), -1, np.int32)
        k = min(512, E)
        sel[0, :k] = np.arange(k)
        _, _, nrows = oracle.attend(np.array([p]), q, sinks, zc, zs, len(zc), wrows, p - 127, sel, return_mass=True)
        assert nrows[0] == want


def test_attend_replay_bound():
    # "Deriving the 890-Byte KV Cache", bounded replay: after a replay starting at s, query t
    # sees window positions max(s, t-127)..t only.
    zc, zs, win, q, sinks, idx, pos = _attend_case(nq=1, seed=14)
    p = int(pos[0])
    plain = oracle.attend(pos, q, sinks, zc, zs, len(zc), win, p - 127, idx)
    # a bound at or below t-127 changes nothing
    same = oracle.attend(pos, q, sinks, zc, zs, len(zc), win, p - 127, idx, win_start=p - 127)
    assert np.array_equal(plain, same)
    # row counts: min(128, t+1-s) window rows + the selected entries
    for s_, want in ((p - 127, 640), (p - 100, 613), (p - 1, 514), (p, 513)):
        _, _, nrows = oracle.attend(pos, q, sinks, zc, zs, len(zc), win, p - 127, idx, return_mass=True,
                                    win_start=s_)
        assert nrows[0] == want
    # s = t: only the query's own window row -- SDPA with the sink as a zero key/value row
    out = oracle.attend(pos, q, sinks, zc, zs, len(zc), win, p - 127, idx, win_start=p)
    G = torch.from_numpy(_gathered(zc, zs, win[-1:], idx[0]))
    K = torch.cat([G, torch.zeros(1, 512, dtype=torch.float64)])
    mask = torch.zeros(64, 1, K.shape[0], dtype=torch.float64)
    mask[:, 0, -1] = torch.from_numpy(sinks.astype(np.float64))
    Q = torch.from_numpy(q[0].astype(np.float64))[:, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K[None].expand(64, -1, -1), K[None].expand(64, -1, -1),
                                                           attn_mask=mask)[:, 0, :].numpy()
    ref = np.stack([np.concatenate([ref[h, :448], oracle.rope(ref[h, 448:], p, inverse=True)]) for h in range(64)])
    assert np.abs(out[0] - ref).max() < 1e-12
    with pytest.raises(ValueError):  # a replay start after the query is not a valid bound
        oracle.attend(pos, q, sinks, zc, zs, len(zc), win, p - 127, idx, win_start=p + 1)


def _brute_pool(s, E):
    nb = -(-E // 8)
    if nb <= 2048:
        return np.arange(nb)
    bs = s[: 8 * (nb - 1)].reshape(nb - 1, 8).max(axis=1)
    order = np.lexsort((np.arange(nb - 1), -bs))   # score desc, then block index asc
    return np.sort(np.concatenate([order[:2047], [nb - 1]]))


def test_hsi_pool_brute_force_ties_and_newest_block():
    # "Hierarchical indexing bounds the later searches": blocks of 8, 2048 blocks, 16384
    # candidates, the newest block always kept
    assert oracle.HSI_BLOCK * oracle.HSI_BLOCKS == golden()["hsi_pool"]
    rng = np.random.default_rng(15)
    E = np.array([16384 + 8 * 11 + 3, 20000, 100, 16384])
    ld = int(E.max())
    s = np.round(rng.standard_normal((4, ld)) * 4) / 4   # coarse values: many exact ties
    s[1, 8 * ((20000 - 1) // 8):] = -1e9                  # the newest block scores lowest
    pool = oracle.hsi_pool(s, E)
    for r in range(4):
        want = _brute_pool(s[r], int(E[r]))
        got = pool[r][pool[r] >= 0]
        assert np.array_equal(got, want)
        assert np.all(pool[r][len(want):] == -1)
        assert got[-1] == (E[r] - 1) // 8                 # newest block present
    assert len(pool[2][pool[2] >= 0]) == 13 and len(pool[3][pool[3] >= 0]) == 2048


def test_reindex_topk_brute_force():
    rng = np.random.default_rng(16)
    E = np.array([17000, 5000])
    s = np.round(rng.standard_normal((2, 17000)) * 8) / 8
    pool = oracle.hsi_pool(rng.standard_normal((2, 17000)), E)   # pool from another layer's scores
    idx = oracle.reindex_topk(s, E, pool)
    for r in range(2):
        blocks = pool[r][pool[r] >= 0]
        cand = np.concatenate([np.arange(8 * b, min(8 * b + 8, E[r])) for b in blocks])
        order = cand[np.lexsort((cand, -s[r, cand]))]
        want = np.sort(order[:512])
        assert np.array_equal(idx[r][idx[r] >= 0], want)
        assert set(want) <= set(cand)


# ---------------------------------------------------------------- page arithmetic
def test_kv_bytes_and_work_ratios():
    gd = golden()
    main = 512 * 4 // 8 + 512 // 16     # pages' main entry: E2M1 + one byte per 16
    idxe = 128 * 4 // 8 + 128 // 32      # indexer entry: E2M1 + one byte per 32
    assert (main, idxe, main + idxe) == (gd["main_entry_bytes"], gd["indexer_entry_bytes"], gd["entry_pair_bytes"])
    assert (3 / 2 + 1) * (main + idxe) == gd["global_bytes_per_token"]
    assert 3 * main / 2 == gd["encoder_bytes_per_token"] and 3 * idxe / 2 + idxe == gd["indexer_bytes_per_token"]
    assert gd["global_bytes_per_token"] * 2 ** 20 < 1e9
    # this library's layout (UE8M0 per 32 for both caches): the oracle's own row sizes
    zc, zs = oracle.mx_quantize(np.ones((1, 512)))
    kc, ks = oracle.mx_quantize(np.ones((1, 128)))
    assert zc.nbytes + zs.nbytes == 272 and kc.nbytes + ks.nbytes == 68
    assert (3 / 2 + 1) * (272 + 68) == 850
    assert abs((0.5 + 128 / (2 * 1e6)) - gd["ced_ratio_1e6_w128"]) < 1e-12
    assert 2048 * 8 == gd["hsi_pool"] and round(1e6 / 16384) == gd["hsi_reduction_1m"]
    assert gd["window_rows"] + gd["selected_rows"] == gd["attended_rows"]


def test_out_group_proj_selection_weights_pick_the_group_heads():
    # W_OA,r = [I_1024 | 0]: group r's output i is input k = i of the group, i.e. head
    # 8r + i // 512, dim i % 512 (heads concatenated one after another inside a group)
    rng = np.random.default_rng(3)
    o = rng.standard_normal((5, 64, 512))
    w = np.zeros((8, 1024, 4096))
    w[:, np.arange(1024), np.arange(1024)] = 1.0
    out = oracle.out_group_proj(o, w)
    for r in range(8):
        assert np.array_equal(out[:, r, :512], o[:, 8 * r])
        assert np.array_equal(out[:, r, 512:], o[:, 8 * r + 1])
    # a weight on input k of group r reads head 8r + k // 512, dim k % 512
    w2 = np.zeros((8, 1024, 4096))
    w2[5, 7, 3 * 512 + 11] = 2.0
    out2 = oracle.out_group_proj(o, w2)
    assert np.allclose(out2[:, 5, 7], 2.0 * o[:, 8 * 5 + 3, 11], rtol=0, atol=0)
    assert np.count_nonzero(out2) == np.count_nonzero(o[:, 43, 11])


def test_out_group_proj_group_locality_and_linearity():
    rng = np.random.default_rng(4)
    o = rng.standard_normal((3, 64, 512))
    w = rng.standard_normal((8, 1024, 4096)) / 64
    base = oracle.out_group_proj(o, w)
    o2 = o.copy()
    o2[:, 8 * 6 + 2] += rng.standard_normal((3, 512))  # a head of group 6 only
    moved = oracle.out_group_proj(o2, w)
    assert np.array_equal(np.delete(moved, 6, axis=1), np.delete(base, 6, axis=1))
    assert not np.allclose(moved[:, 6], base[:, 6])
    # brute force of one output against the definition's sum, element by element
    r, i, n = 2, 900, 1
    ref = sum(o[n, 8 * r + k // 512, k % 512] * w[r, i, k] for k in range(4096))
    assert abs(base[n, r, i] - ref) <= 1e-12 * max(1.0, abs(ref))
