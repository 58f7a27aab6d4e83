"""GPU parity of the grouped output projection W_OA ("Inside DeepSeek V4.1", section
"Attention that looks at 640 places"; [PG] o^g_{t,r} = [O-bar_{h,t}]_{h in r} W_OA,r) against
the fp64 oracle: bf16 output rules (max-abs <= 2e-2, relative L2 <= 5e-3), and exact
selection weights for the layout.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_03_gb300 import inputs
import compressed_sparse_attention_03_gb300 as csa2
from parity_utils import np32, out_compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def handle():
    return csa2.csa2_create()


def run(h, o, w):
    out = torch.empty(o.shape[0], 8, 1024, dtype=torch.bfloat16, device=DEV)
    csa2.csa2_out_group_proj(h, o, w, out)
    return out


@pytest.mark.parametrize("M", [1, 127, 300, 1000])
def test_out_group_proj_small(handle, M):
    # row counts below, at and across the 128-row tile, with a ragged tail
    x = inputs.out_proj_inputs(M, seed=M, device=DEV)
    out = run(handle, x["o"], x["w_oa"])
    ref = oracle.out_group_proj(np32(x["o"]), np32(x["w_oa"]))
    mx, rl2 = out_compare(np32(out), ref)
    print(f"out_group_proj M={M}: max abs {mx:.2e}, rel L2 {rl2:.2e}")


def test_out_group_proj_prefill_4k_sampled(handle):
    M = 4096
    x = inputs.out_proj_inputs(M, seed=1, device=DEV)
    out = run(handle, x["o"], x["w_oa"])
    rows = np.unique(np.concatenate([[0, 1, 127, 128, M - 1], np.random.default_rng(5).integers(0, M, 59)]))
    ref = oracle.out_group_proj(np32(x["o"][rows]), np32(x["w_oa"]))
    mx, rl2 = out_compare(np32(out[rows]), ref)
    print(f"out_group_proj M=4096 ({len(rows)} rows): max abs {mx:.2e}, rel L2 {rl2:.2e}")


def test_out_group_proj_selection_weights_exact(handle):
    # W_OA,r = [I | 0] with a second weight of 1 on input 3*512 + 11: output i < 1024 is input
    # i of the group (heads 8r and 8r+1) plus, for i = 7, head 8r+3 dim 11; bf16 inputs, exact
    M = 200
    x = inputs.out_proj_inputs(M, seed=9, device=DEV)
    w = torch.zeros(8, 1024, 4096, dtype=torch.bfloat16, device=DEV)
    w[:, torch.arange(1024), torch.arange(1024)] = 1.0
    out = run(handle, x["o"], w)
    o = x["o"].float()
    for r in range(8):
        assert torch.equal(out[:, r, :512].float(), o[:, 8 * r])
        assert torch.equal(out[:, r, 512:].float(), o[:, 8 * r + 1])
