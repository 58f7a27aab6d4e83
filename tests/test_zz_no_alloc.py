"""csa2_attend_static, the allocation-free variant of csa2_attend (its scratch is a fixed device
array of the library).  Two calls in a row must give exactly what csa2_attend gives on the same
inputs, the second call must not see the first call's partials, and once the array is set up the
calls must not change the device's free memory.

The file name keeps it last in collection, so that it also runs after every other test has
used the library; it passes alone in a fresh process as well (the first call here sets up the
scratch on this device)."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_03_gb300 import inputs
import compressed_sparse_attention_03_gb300 as csa2
from parity_utils import random_indices

pytestmark = pytest.mark.gpu
DEV = "cuda"


def attend_case(B, T, p0s, seed):
    """Attention inputs with every window row filled (codes, not a writer's output: both entry
    points read the same bytes, which is all this comparison needs)."""
    p0s = np.asarray(p0s, np.int64)
    cap = int(((p0s + T) // 2).max()) + 3
    x = inputs.step_inputs(B, T, seed, DEV)
    x["sinks"] = inputs.layer_params(seed, DEV)["sinks"]
    x.update(inputs.cache_state(B, T, int(p0s.max()), cap, seed, DEV))
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    x["window"] = inputs.random_e4m3(tuple(x["window"].shape), g, DEV)
    x["idx"] = random_indices(B, T, p0s, seed, DEV)
    x["p0s"] = p0s
    return x


def call(fn, h, x, out):
    fn(h, x["q"], x["sinks"], x["z_codes"], x["z_scales"], x["window"], x["idx"], x["p0s"], out)


def fresh_out(x):
    B, T = x["q"].shape[:2]
    return torch.full((B, T, 64, 512), float("nan"), dtype=torch.bfloat16, device=DEV)


def test_static_matches_attend_on_consecutive_calls():
    h = csa2.csa2_create()
    # first: four decode queries, split five ways, most splits with a chunk of rows;
    # second: three decode queries, the first two with one or two chunks, so most of their five
    # splits are empty and must not pick up the first call's partials
    first = attend_case(4, 1, [9000, 5001, 300, 64000], seed=41)
    second = attend_case(3, 1, [100, 0, 2500], seed=42)
    refs = []
    for x in (first, second):
        ref = fresh_out(x)
        call(csa2.csa2_attend, h, x, ref)
        refs.append(ref)

    # set-up call: resolves the scratch address on this device (may load its module)
    warm = fresh_out(first)
    call(csa2.csa2_attend_static, h, first, warm)
    torch.cuda.synchronize()
    assert torch.equal(warm, refs[0])

    outs = [fresh_out(first), fresh_out(second)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    call(csa2.csa2_attend_static, h, first, outs[0])
    call(csa2.csa2_attend_static, h, second, outs[1])
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, "csa2_attend_static changed the device's free memory"
    for out, ref in zip(outs, refs):
        assert not torch.isnan(out.float()).any()
        assert torch.equal(out, ref)


def test_static_unsplit_batch_matches_attend():
    # 160 queries are not split (one block per query): no scratch is used at all
    h = csa2.csa2_create()
    x = attend_case(2, 80, [1000, 4097], seed=43)
    ref, out = fresh_out(x), fresh_out(x)
    call(csa2.csa2_attend, h, x, ref)
    call(csa2.csa2_attend_static, h, x, out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_static_rejects_bad_arguments_before_launch():
    h = csa2.csa2_create()
    x = attend_case(1, 1, [10], seed=44)
    out = fresh_out(x)
    with pytest.raises(csa2.Csa2Error) as e:
        call(csa2.csa2_attend_static, h, dict(x, p0s=np.array([-1])), out)
    assert e.value.status == 2
    misaligned = out.view(-1)[4:]  # 8 bytes past a 16-byte boundary
    with pytest.raises(csa2.Csa2Error) as e:
        call(csa2.csa2_attend_static, h, x, misaligned)
    assert e.value.status == 3
    assert torch.isnan(out.float()).all()  # nothing was launched
