"""Decode steps captured once in a CUDA graph with positions in device memory
(csa2_set_device_positions), replayed at advancing positions, against the same steps called
with host positions: caches, window, pair buffers, indices and outputs bit-identical after every
step.  The host-position path is the one the oracle parity tests check."""
import pytest
import torch

import compressed_sparse_attention_03_gb300 as csa2
from compressed_sparse_attention_03_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
STATE = ("z_codes", "z_scales", "ki_codes", "ki_scales", "window", "pair_kc", "pair_gc")


def make_state(B, p0s, cap, seed, ratio):
    x = {}
    x.update(inputs.layer_params(seed, DEV))
    x.update(inputs.step_inputs(B, 1, seed, DEV))
    st = inputs.cache_state(B, 1, int(max(p0s)), cap, seed, DEV, ratio)
    for b in range(B):  # shorter sequences: no cached entries beyond their own length
        n = int(p0s[b]) // ratio
        for k in ("z_codes", "z_scales", "ki_codes", "ki_scales"):
            st[k][b, n:] = 0
    x.update(st)
    return x


class DecodePath:
    """One decode step (write, index, attend, window roll) on its own copy of the state."""

    def __init__(self, h, x, B, max_entries):
        self.h = h
        self.x = dict(x)
        for k in STATE:
            self.x[k] = x[k].clone()
        self.idx = torch.empty(B, 1, 512, dtype=torch.int32, device=DEV)
        self.out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
        self.ws_i = csa2.workspace(h, csa2.OP_INDEX_TOPK, B, 1, max_entries, DEV)
        self.ws_a = csa2.workspace(h, csa2.OP_ATTEND, B, 1, 0, DEV)

    def step(self, p0, s):
        x = self.x
        csa2.csa2_write_cache(self.h, x["kc"], x["gc"], x["wa"], x["gamma_c"], x["w_ik"], x["gamma_ik"],
                              x["gamma_w"], p0, x["z_codes"], x["z_scales"], x["ki_codes"], x["ki_scales"],
                              x["window"], x["pair_kc"], x["pair_gc"], stream=s)
        csa2.csa2_index_topk(self.h, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], p0, self.idx, ws=self.ws_i,
                             stream=s)
        csa2.csa2_attend(self.h, x["q"], x["sinks"], x["z_codes"], x["z_scales"], x["window"], self.idx, p0,
                         self.out, ws=self.ws_a, stream=s)
        csa2.csa2_roll_window(self.h, x["window"], x["window"], stream=s)

    def results(self):
        return [self.idx, self.out] + [self.x[k] for k in STATE]


def capture(fn):
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            fn(torch.cuda.current_stream())
    torch.cuda.current_stream().wait_stream(cs)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("ratio,p0s,cap_extra", [(2, [4096, 5001, 130], 8), (1, [3001, 1000], 8),
                                                  (2, [131072, 131075, 65537, 2], 8)])
def test_graph_decode_steps(ratio, p0s, cap_extra):
    B, nsteps = len(p0s), 5
    p0_max = max(p0s) + nsteps
    cap = (p0_max + 1) // ratio + cap_extra
    x = make_state(B, p0s, cap, seed=41 + B, ratio=ratio)
    max_entries = (p0_max + 1) // ratio
    h_host = csa2.csa2_create(ratio=ratio)
    h_dev = csa2.csa2_create(ratio=ratio)
    eager = DecodePath(h_host, x, B, max_entries)
    graph = DecodePath(h_dev, x, B, max_entries)
    warm = DecodePath(h_dev, x, B, max_entries)
    p0_dev = torch.tensor(p0s, dtype=torch.int64, device=DEV)
    csa2.csa2_set_device_positions(h_dev, p0_dev, p0_max)
    s = torch.cuda.current_stream()
    warm.step(None, s)  # one uncaptured step loads the kernels
    torch.cuda.synchronize()
    g = capture(lambda cs: graph.step(None, cs))
    for k in range(nsteps):
        pos = [p + k for p in p0s]
        eager.step(pos, s)
        p0_dev.copy_(torch.tensor(pos, dtype=torch.int64))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager.results(), graph.results()):
            assert torch.equal(a, b), f"step {k} (positions {pos}) differs"
    assert csa2.csa2_check(h_dev) == 0 and csa2.csa2_check(h_host) == 0
    print(f"graph decode ratio {ratio} B={B}: {nsteps} steps from one capture, bit-identical")


def test_device_position_out_of_range():
    """A device position above the bound (or below 0) is clamped into 0..p0_max, so every
    access stays within what the host validated, and csa2_check reports CSA2_ERR_SHAPE."""
    ratio, p0s = 2, [2000, 517]
    B, p0_max = len(p0s), 2100
    cap = (p0_max + 1) // ratio + 4
    x = make_state(B, p0s, cap, seed=5, ratio=ratio)
    h_host, h_dev = csa2.csa2_create(ratio=ratio), csa2.csa2_create(ratio=ratio)
    max_entries = (p0_max + 1) // ratio
    ws = csa2.workspace(h_dev, csa2.OP_INDEX_TOPK, B, 1, max_entries, DEV)
    p0_dev = torch.tensor([p0_max + 50, -3], dtype=torch.int64, device=DEV)
    csa2.csa2_set_device_positions(h_dev, p0_dev, p0_max)
    got = torch.empty(B, 1, 512, dtype=torch.int32, device=DEV)
    csa2.csa2_index_topk(h_dev, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], None, got, ws=ws)
    assert csa2.csa2_check(h_dev) == 2
    ref = torch.empty_like(got)
    csa2.csa2_index_topk(h_host, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], [p0_max, 0], ref, ws=ws)
    assert torch.equal(got, ref)
    assert csa2.csa2_check(h_dev) == 0  # the flag was cleared
    # back to host positions: the p0 argument is read again
    csa2.csa2_set_device_positions(h_dev, None)
    csa2.csa2_index_topk(h_dev, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], [p0_max, 0], got, ws=ws)
    assert torch.equal(got, ref) and csa2.csa2_check(h_dev) == 0
    with pytest.raises(ValueError):  # no positions at all
        csa2.csa2_index_topk(h_dev, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], None, got, ws=ws)
