"""GPU parity of per-token NVFP4 with the original pretraining recipe's
stabilizers ("Miles: end-to-end MXFP8 and per-token NVFP4 RL", NVFP4
recipe section: stochastic rounding and Random Hadamard Transforms): codes,
block scales and per-token FP32 scales bit for bit against the oracle for
every combination of the two, both scale layouts, ragged shapes; without
either the bytes equal the per-token quantizer's."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import assert_bytes_equal, dev_bf16, host_u8

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


def _logical(r, T, H, lay):
    codes = host_u8(r.codes)
    sc = host_u8(r.block_scales)
    if lay == "swizzled":
        sc = O.scale_unswizzle(sc, T, H // 16)
    else:
        sc = sc.reshape(T, H // 16)
    return codes, sc, r.scales.cpu().numpy()


def check(q, x, seed, flags, lay, rows=None):
    T, H = x.shape
    r = q.nvfp4_quantize_per_token_rht_sr(dev_bf16(x), seed, flags, lay)
    torch.cuda.synchronize()
    assert q.get_last_error() == q.MXQ_OK
    codes, sc, S = _logical(r, T, H, lay)
    sel = np.arange(T) if rows is None else rows
    for lo in range(0, len(sel), 64):
        part = sel[lo:lo + 64]
        # contiguous runs keep the oracle's row index = the tensor's
        for run in np.split(part, np.nonzero(np.diff(part) != 1)[0] + 1):
            oc, osc, oS = O.nvfp4_quantize_rht_sr(x[run], seed, flags, row0=int(run[0]))
            assert_bytes_equal(codes[run], oc, f"codes flags={flags} [{lay}]")
            assert_bytes_equal(sc[run], osc, f"scales flags={flags} [{lay}]")
            assert_bytes_equal(S[run].view(np.uint32), oS.view(np.uint32),
                               f"S flags={flags} [{lay}]")
    return r


@pytest.mark.parametrize("flags", [0, 1, 2, 3])
@pytest.mark.parametrize("lay", ["swizzled", "linear"])
def test_ragged_tokens(mxq, flags, lay):
    x = W.ragged_tokens([70, 33, 101], H=256)
    check(mxq, x, 1234, flags, lay)


@pytest.mark.parametrize("H", [16, 48, 160, 1552, 2048, 2064, 4096])
def test_hidden_sizes(mxq, H):
    """Rows of up to 128 blocks keep their transformed values in registers
    between the passes (1552: 97 blocks, a ragged last step); longer rows
    (2064: 129 blocks, 4096) are transformed again in the second pass."""
    x = W.ragged_tokens([37], H=H)
    for flags in (1, 3):
        check(mxq, x, 99, flags, "swizzled")
        check(mxq, x, 99, flags, "linear")


def test_edge_tokens(mxq):
    """The per-token quantizer's edge tokens (zero, subnormal S, S = 1,
    bf16 max, a huge channel, E2M1 midpoints).  With the transform, the
    bf16-max token is outside the contract: its butterfly sums overflow
    binary32 (any block with |x| > FLT_MAX / 16 does), so it is left out."""
    x = W.tiny_token_rows(H=256)
    for flags in (0, 2):
        check(mxq, x, 5, flags, "swizzled")
    keep = np.array([0, 1, 2, 4, 5])
    for flags in (1, 3):
        check(mxq, np.ascontiguousarray(x[keep]), 5, flags, "swizzled")


def test_no_stabilizers_equals_per_token(mxq):
    x = dev_bf16(W.ragged_tokens([129, 64], H=512))
    a = mxq.nvfp4_quantize_per_token_rht_sr(x, 7, 0)
    b = mxq.nvfp4_quantize_per_token(x)
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.block_scales, b.block_scales)
    assert torch.equal(a.scales, b.scales)


def test_full_size_sampled(mxq):
    """8192 tokens x 4096 hidden with both stabilizers: 3 runs of 64
    consecutive rows (start, middle, end) against the oracle."""
    x = W.mxfp8_random(8192, 4096)
    rows = np.concatenate([np.arange(0, 64), np.arange(4000, 4064),
                           np.arange(8128, 8192)])
    check(mxq, x, 2026, 3, "swizzled", rows=rows)
