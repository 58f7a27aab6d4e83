"""Seeded synthetic inputs for the CSA2 layer, shared by the tests, the smoke check and the
benchmark.  This module holds no arithmetic of the method: it only draws random numbers
(torch generators) with the shapes and value distributions of the workloads below, and
maps uniform random bytes to storage codes through fixed lookup tables.

Workloads (B sequences, T new tokens, p0 cached positions before the step):
  decode_8k      B=1,  p0=8192,    T=1   (4096 cached pooled entries)          seed 0
  prefill_4k     B=1,  p0=0,       T=4096                                      seed 1
  decode_128k    B=64, p0=131072,  T=1   (65536 entries per sequence)          seed 2
  decode_1m      B=8,  p0=1048576, T=1   (524288 entries per sequence)         seed 3
  chunk_32k      B=1,  p0=262144,  T=32768 (131072 cached + 16384 new entries) seed 4
  decode_512k_r1 B=8,  p0=524288,  T=1   compression ratio 1 (524288 entries)  seed 5
  prefill_4k_r1  B=1,  p0=0,       T=4096 compression ratio 1                  seed 6
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

D, DI, HI, H = 512, 128, 32, 64


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    p0: int
    seed: int
    ratio: int = 2  # compression ratio of the layer (entries per token: 1 / ratio)

    @property
    def cap(self) -> int:
        """Cache capacity (entries) that holds every entry visible to the step."""
        return (self.p0 + self.T) // self.ratio

    @property
    def cached_entries(self) -> int:
        return self.p0 // self.ratio


WORKLOADS = {
    "decode_8k": Workload("decode_8k", 1, 1, 8192, 0),
    "prefill_4k": Workload("prefill_4k", 1, 4096, 0, 1),
    "decode_128k": Workload("decode_128k", 64, 1, 131072, 2),
    "decode_1m": Workload("decode_1m", 8, 1, 1048576, 3),
    "chunk_32k": Workload("chunk_32k", 1, 32768, 262144, 4),
    "decode_512k_r1": Workload("decode_512k_r1", 8, 1, 524288, 5, ratio=1),
    "prefill_4k_r1": Workload("prefill_4k_r1", 1, 4096, 0, 6, ratio=1),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _lut_from_weights(weights) -> torch.Tensor:
    """256-entry table mapping a uniform byte to value i with probability weights[i]/256."""
    assert sum(weights) == 256
    out = []
    for v, w in enumerate(weights):
        out += [v] * w
    return torch.tensor(out, dtype=torch.uint8)


# E2M1 magnitude codes 0..7 (0, .5, 1, 1.5, 2, 3, 4, 6) as a normalised Gaussian block lands
# on them, then a sign bit; scale bytes 125/126/127 (block maxima around 2..4).
_E2M1_MAG = _lut_from_weights([26, 48, 46, 40, 52, 26, 16, 2])
_SCALE = _lut_from_weights([0] * 125 + [26, 204, 26] + [0] * 128)
# E4M3 exponent fields 3..9 (magnitudes 2^-4 .. 2^2) for the FP8 window rows.
_E4M3_EXP = _lut_from_weights([0, 0, 0, 13, 13, 26, 48, 77, 67, 12] + [0] * 6)


def _bytes(shape, g, device):
    return torch.randint(0, 256, shape, generator=g, device=device, dtype=torch.int32)


def _e2m1_nibbles(shape, g, device):
    """Random E2M1 codes: a magnitude code from the full 256-entry table, then a sign bit."""
    mag = _E2M1_MAG.to(device)[_bytes(shape, g, device)]
    sign = ((_bytes(shape, g, device) & 1) << 3).to(torch.uint8)
    return mag | sign


def random_fp4(rows_shape, n: int, g, device, scale_range=None):
    """Random FP4 rows: (codes [..., n/2] u8, scales [..., n/32] u8).  Scale bytes follow the
    table above, or are uniform over scale_range = (lo, hi) inclusive."""
    lo = _e2m1_nibbles((*rows_shape, n // 2), g, device)
    hi = _e2m1_nibbles((*rows_shape, n // 2), g, device)
    codes = (lo | (hi << 4)).to(torch.uint8)
    if scale_range is None:
        scales = _SCALE.to(device)[_bytes((*rows_shape, n // 32), g, device)]
    else:
        scales = torch.randint(scale_range[0], scale_range[1] + 1, (*rows_shape, n // 32), generator=g, device=device,
                               dtype=torch.int32).to(torch.uint8)
    return codes, scales


def random_e4m3(shape, g, device):
    """Random E4M3 codes (no NaN codes)."""
    e = _E4M3_EXP.to(device)[_bytes(shape, g, device)].to(torch.int32)
    m = torch.randint(0, 8, shape, generator=g, device=device, dtype=torch.int32)
    s = torch.randint(0, 2, shape, generator=g, device=device, dtype=torch.int32)
    return ((s << 7) | (e << 3) | m).to(torch.uint8)


def layer_params(seed: int, device="cpu"):
    """gamma_c [512], w_ik [512,128] bf16 ~N(0,1)/sqrt(512), gamma_ik [128], gamma_w [512]
    (gains ~ 1 + 0.1 N(0,1)), sinks [64] ~ N(0,1)."""
    g = _gen(10_000 + seed, device)
    f32 = dict(device=device, dtype=torch.float32, generator=g)
    gamma_c = 1.0 + 0.1 * torch.randn(D, **f32)
    w_ik = (torch.randn(D, DI, **f32) / D ** 0.5).to(torch.bfloat16)
    gamma_ik = 1.0 + 0.1 * torch.randn(DI, **f32)
    gamma_w = 1.0 + 0.1 * torch.randn(D, **f32)
    sinks = torch.randn(H, **f32)
    return dict(gamma_c=gamma_c, w_ik=w_ik, gamma_ik=gamma_ik, gamma_w=gamma_w, sinks=sinks)


def out_proj_inputs(M: int, seed: int, device="cpu"):
    """Grouped output projection: attention outputs O-bar [M,64,512] bf16 ~ 0.5 N(0,1) (the
    scale of a softmax-weighted mean of unit rows) and W_OA [8,1024,4096] bf16 ~
    N(0,1)/sqrt(4096) (group, output, input)."""
    g = _gen(40_000 + seed, device)
    f32 = dict(device=device, dtype=torch.float32, generator=g)
    o = (0.5 * torch.randn(M, H, D, **f32)).to(torch.bfloat16)
    w = (torch.randn(8, 1024, 8 * D, **f32) / (8 * D) ** 0.5).to(torch.bfloat16)
    return dict(o=o, w_oa=w)


def step_inputs(B: int, T: int, seed: int, device="cpu"):
    """Per-token inputs of one step, all bf16: k^c, g^c, w^a [B,T,512] ~N(0,1);
    Q [B,T,64,512] ~N(0,1); Q^I [B,T,32,128] ~N(0,1); w^I [B,T,32] ~N(0,1)/sqrt(128*32)."""
    g = _gen(20_000 + seed, device)
    f32 = dict(device=device, dtype=torch.float32, generator=g)
    bf = lambda *s: torch.randn(*s, **f32).to(torch.bfloat16)
    kc, gc, wa = bf(B, T, D), bf(B, T, D), bf(B, T, D)
    q = bf(B, T, H, D)
    qi = bf(B, T, HI, DI)
    wI = (torch.randn(B, T, HI, **f32) / (DI * HI) ** 0.5).to(torch.bfloat16)
    return dict(kc=kc, gc=gc, wa=wa, q=q, qi=qi, wI=wI)


def cache_state(B: int, T: int, p0: int, cap: int, seed: int, device="cpu", ratio: int = 2, scale_range=None):
    """Synthetic state before the step: FP4 caches with the p0//ratio cached entries drawn at
    random (rest zero), the window view [B,127+T,512] with random E4M3 codes in the rows of
    positions p0-127..p0-1 that exist, and a random pair buffer (used when p0 is odd).
    scale_range = (lo, hi): FP4 scale bytes uniform over lo..hi instead of the default table."""
    g = _gen(30_000 + seed, device)
    n = p0 // ratio
    z_codes = torch.zeros(B, cap, D // 2, dtype=torch.uint8, device=device)
    z_scales = torch.zeros(B, cap, D // 32, dtype=torch.uint8, device=device)
    ki_codes = torch.zeros(B, cap, DI // 2, dtype=torch.uint8, device=device)
    ki_scales = torch.zeros(B, cap, DI // 32, dtype=torch.uint8, device=device)
    if n:
        zc, zs = random_fp4((B, n), D, g, device, scale_range)
        kc, ks = random_fp4((B, n), DI, g, device, scale_range)
        z_codes[:, :n], z_scales[:, :n], ki_codes[:, :n], ki_scales[:, :n] = zc, zs, kc, ks
    window = torch.zeros(B, 127 + T, D, dtype=torch.uint8, device=device)
    first = max(0, 127 - p0)
    if first < 127:
        window[:, first:127] = random_e4m3((B, 127 - first, D), g, device)
    f32 = dict(device=device, dtype=torch.float32, generator=g)
    pair_kc = torch.randn(B, D, **f32).to(torch.bfloat16).float()
    pair_gc = torch.randn(B, D, **f32).to(torch.bfloat16).float()
    return dict(z_codes=z_codes, z_scales=z_scales, ki_codes=ki_codes, ki_scales=ki_scales, window=window,
                pair_kc=pair_kc, pair_gc=pair_gc)


def workload_inputs(w: Workload, device="cpu"):
    """Everything one step of workload ``w`` reads: params, step inputs and cache state."""
    out = {}
    out.update(layer_params(w.seed, device))
    out.update(step_inputs(w.B, w.T, w.seed, device))
    out.update(cache_state(w.B, w.T, w.p0, w.cap, w.seed, device, w.ratio))
    return out
