"""The tensor-core rate probe (csa2_tc_rate): the peaks the tensor-bound kernels are quoted against."""
import pytest
import torch

import compressed_sparse_attention_03_gb300 as csa2

pytestmark = pytest.mark.gpu


def test_rates_per_kind():
    h = csa2.csa2_create()
    try:
        f16, e5m2, mxf4 = (csa2.csa2_tc_rate(h, k, 4096) for k in range(3))
    finally:
        h.close()
    # the dense fp16 rate of a GB300-class part is in the PFLOP/s range; an E5M2 MMA does twice
    # the K of an fp16 one, an mxf4 MMA four times, in about the same time
    assert 800.0 < f16 < 4000.0
    assert 1.6 < e5m2 / f16 < 2.4
    assert 3.2 < mxf4 / f16 < 4.8


def test_rejects_bad_arguments():
    h = csa2.csa2_create()
    try:
        for kind, iters in ((3, 10), (-1, 10), (0, 0), (0, 1 << 17)):
            with pytest.raises(csa2.Csa2Error):
                csa2.csa2_tc_rate(h, kind, iters)
    finally:
        h.close()
