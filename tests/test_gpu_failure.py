"""Device-side failure detection without a GPU fault.

Every wait in the kernels (mbarrier phases, the weight quantizer's progress
words, the GEMM's stage handoffs) is bounded: when it runs out it records
an error word and the kernel returns, so the host sees MXQ_ERR_TIMEOUT from
mxq_get_last_error and the CUDA context stays usable.  The self-test kernel
makes one such wait run out (a barrier nothing completes, 20 ms limit)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import dev_bf16, host_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from nvfp4_quantizers_gb300 import build
    build.build()
    import nvfp4_quantizers_gb300 as q
    q.lib()
    return q


def test_wait_timeout_is_reported_and_context_survives(mxq):
    assert mxq.get_last_error() == mxq.MXQ_OK
    mxq.selftest_wait_timeout()
    assert mxq.get_last_error() == mxq.MXQ_ERR_TIMEOUT
    # read and cleared
    assert mxq.get_last_error() == mxq.MXQ_OK
    # the context still runs kernels correctly
    x = W.mxfp8_small()
    r = mxq.mxfp8_quantize_rowcol(dev_bf16(x))
    torch.cuda.synchronize()
    rc, rs = O.mxfp8_quantize_rowwise(x)
    assert np.array_equal(host_u8(r.row_codes), rc)
    assert np.array_equal(host_u8(r.row_scales), O.scale_swizzle(rs))
    assert mxq.get_last_error() == mxq.MXQ_OK


def test_timeouts_do_not_accumulate(mxq):
    for _ in range(3):
        mxq.selftest_wait_timeout()
    assert mxq.get_last_error() == mxq.MXQ_ERR_TIMEOUT
    assert mxq.get_last_error() == mxq.MXQ_OK
