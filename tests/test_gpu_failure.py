"""Failure path on the GPU without a fault: a bounded wait that nothing satisfies
gives up, the status word reports OA_ERR_TIMEOUT, and the context stays usable."""
import pytest
import torch

import oracle
import synth_inputs as si
from parity import assert_lse_close

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_context_survives(cuda_lib):
    oa = cuda_lib
    oa.sync_status()  # clean start
    oa.selftest_wait_timeout(2_000_000)  # 2 ms
    with pytest.raises(oa.OAError) as ei:
        oa.sync_status()
    assert ei.value.status == oa.OA_ERR_TIMEOUT
    assert "kernel 6" in str(ei.value)
    oa.sync_status()  # the word was cleared
    # the next real call still works
    x, *_ = si.softmax_input(8, 100, seed=1)
    _, lse = oa.softmax_rows(x.cuda())
    torch.cuda.synchronize()
    oa.sync_status()
    assert_lse_close(lse, oracle.softmax_rows(x.numpy())[1])
