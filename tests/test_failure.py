"""Failure detection without a GPU fault: a bounded wait that runs out is
reported through the device status word and the context stays usable."""
import numpy as np
import pytest

import bi_synth as syn
from util import bits_of, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives(bi):
    assert bi.device_status() == bi.BI_OK
    bi.check_wait_timeout(20000)            # 20 ms wait on a barrier nobody arrives at
    assert bi.device_status() == bi.BI_ERR_TIMEOUT
    assert bi.device_status() == bi.BI_OK   # the read cleared it
    X, W = syn.gemm_inputs(5, 64, 64, seed=0)
    y1 = bits_of(bi.gemm_bf16(to_dev_bf16(X), to_dev_bf16(W)))
    y2 = bits_of(bi.gemm_bf16(to_dev_bf16(X), to_dev_bf16(W)))
    assert np.array_equal(y1, y2)
    assert bi.device_status() == bi.BI_OK


def test_bad_moe_offsets_are_reported(bi):
    import torch
    E, N, K, rows = 4, 64, 64, 10
    X = torch.zeros((rows, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((E, N, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((rows, N), 3.0, dtype=torch.bfloat16, device="cuda")
    for bad in ([0, 5, 3, 8, 10], [1, 2, 3, 4, 10], [0, 2, 4, 6, 9]):
        off = torch.tensor(bad, dtype=torch.int32, device="cuda")
        bi.grouped_gemm_bf16(X, W, off, Y=Y)
        assert bi.device_status() == bi.BI_ERR_INVALID_ARG
        assert torch.all(Y == 3.0), "nothing may be written for invalid offsets"
    assert bi.device_status() == bi.BI_OK


def test_host_side_errors_raise(bi):
    import torch
    X = torch.zeros((4, 60), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((16, 60), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bi.BiError) as e:
        bi.gemm_bf16(X, W)
    assert e.value.status == bi.BI_ERR_UNSUPPORTED
