"""The allocation-free weight quantizer entry point.

nvfp4_quantize_weight_shared_noalloc serves callers that cannot allocate
device memory (plug-ins inside a framework that owns all device memory,
latency-critical loops where cudaMalloc is not allowed), so it keeps its
per-group scratch in a fixed array inside the library instead of a
caller-provided workspace.  These tests call it through the C ABI and
require its outputs to be byte-identical to those of
nvfp4_quantize_weight_shared (the workspace entry point), on two calls in a
row, so that scratch left over from the first call cannot leak into the
second.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

_p = ctypes.c_void_p
_i64 = ctypes.c_int64


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from nvfp4_quantizers_gb300 import build
    build.build()
    import nvfp4_quantizers_gb300 as q
    lib = q.lib()
    lib.nvfp4_quantize_weight_shared_noalloc.restype = ctypes.c_int
    lib.nvfp4_quantize_weight_shared_noalloc.argtypes = [
        _i64, ctypes.c_int, _p, _p, _i64, _p, _p, _p, _p, ctypes.c_int, _p]
    lib.nvfp4_quantize_weight_shared_noalloc_max_groups.restype = _i64
    lib.nvfp4_quantize_weight_shared_noalloc_max_groups.argtypes = []
    return lib


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)) \
        .view(torch.bfloat16).cuda()


def _call_noalloc(L, groups, scale_layout, S_in=None):
    import nvfp4_quantizers_gb300 as q
    G, P = len(groups), len(groups[0])
    K = groups[0][0].shape[1]
    R = sum(t.shape[0] for t in groups[0])
    ptrs = (ctypes.c_void_p * (G * P))(*[t.data_ptr() for g in groups for t in g])
    rows = (ctypes.c_int64 * P)(*[t.shape[0] for t in groups[0]])
    codes = torch.full((G, R, K // 2), 0xAB, dtype=torch.uint8, device="cuda")
    sb = q.scale_bytes(R, K // 16, scale_layout)
    scales = torch.full((G, sb), 0xAB, dtype=torch.uint8, device="cuda")
    S = torch.full((G,), -1.0, dtype=torch.float32, device="cuda")
    st = L.nvfp4_quantize_weight_shared_noalloc(
        G, P, ctypes.cast(ptrs, _p), ctypes.cast(rows, _p), K,
        codes.data_ptr(), scales.data_ptr(), S.data_ptr(),
        None if S_in is None else S_in.data_ptr(),
        q._lib._layout(scale_layout),
        torch.cuda.current_stream().cuda_stream)
    assert st == q.MXQ_OK, q.status_string(st)
    return codes, scales, S


@pytest.mark.parametrize("scale_layout", ["swizzled", "linear"])
def test_noalloc_matches_workspace_entry_point(L, scale_layout):
    import nvfp4_quantizers_gb300 as q
    experts = [W.moe_expert(e, hidden=2048, ffn=768, seed=31) for e in range(5)]
    groups = [[_dev(g), _dev(u)] for g, u, _ in experts]
    ref = q.nvfp4_quantize_weight_shared(groups, scale_layout=scale_layout)
    first = _call_noalloc(L, groups, scale_layout)
    second = _call_noalloc(L, groups, scale_layout)
    torch.cuda.synchronize()
    for got in (first, second):
        assert torch.equal(got[0], ref.codes)
        assert torch.equal(got[1], ref.block_scales)
        assert torch.equal(got[2].view(torch.int32), ref.scales.view(torch.int32))
    assert q.get_last_error() == q.MXQ_OK


def test_noalloc_second_call_sees_no_stale_scratch(L):
    """A call on larger-magnitude weights, then one on smaller ones: the
    second call's scales must come from its own data only."""
    import nvfp4_quantizers_gb300 as q
    big = [[_dev(W.to_bf16_bits(np.full((64, 128), 100.0)))] for _ in range(3)]
    small = [[_dev(W.moe_expert(e, hidden=128, ffn=64, seed=32)[0])]
             for e in range(3)]
    _call_noalloc(L, big, "swizzled")
    got = _call_noalloc(L, small, "swizzled")
    ref = q.nvfp4_quantize_weight_shared(small)
    torch.cuda.synchronize()
    assert torch.equal(got[0], ref.codes)
    assert torch.equal(got[1], ref.block_scales)
    assert torch.equal(got[2], ref.scales)


def test_noalloc_rejects_too_many_groups(L):
    import nvfp4_quantizers_gb300 as q
    cap = L.nvfp4_quantize_weight_shared_noalloc_max_groups()
    assert cap == 4096
    ptrs = (ctypes.c_void_p * 1)(0x10000)
    rows = (ctypes.c_int64 * 1)(16)
    st = L.nvfp4_quantize_weight_shared_noalloc(
        cap + 1, 1, ctypes.cast(ptrs, _p), ctypes.cast(rows, _p), 16,
        0x10000, 0x10000, 0x10000, None, 1, None)
    assert st == q.MXQ_ERR_SHAPE


def _compare(L, groups, S_in=None, scale_layout="swizzled"):
    """The no-alloc call (twice) against the workspace entry point."""
    import nvfp4_quantizers_gb300 as q
    ref = q.nvfp4_quantize_weight_shared(groups, S_in, scale_layout)
    for _ in range(2):
        got = _call_noalloc(L, groups, scale_layout, S_in)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref.codes)
        assert torch.equal(got[1], ref.block_scales)
        assert torch.equal(got[2].view(torch.int32), ref.scales.view(torch.int32))
    assert q.get_last_error() == q.MXQ_OK


def test_noalloc_more_groups_than_one_launch(L):
    """300 small groups: two launches, whose group words sit at different
    offsets of the library's array."""
    rng = np.random.default_rng(41)
    groups = [[_dev(W.to_bf16_bits(rng.standard_normal((32, 64)) * (g % 5 + 1)))]
              for g in range(300)]
    _compare(L, groups)


def test_noalloc_near_the_group_cap(L):
    """4000 groups of [16 x 16]: the array's words up to near its end."""
    rng = np.random.default_rng(42)
    host = W.to_bf16_bits(rng.standard_normal((4000, 16, 16)))
    x = _dev(host.reshape(4000 * 16, 16))
    groups = [[x[16 * g:16 * g + 16]] for g in range(4000)]
    _compare(L, groups)


def test_noalloc_scales_given_after_an_amax_call(L):
    """An amax call, then a call with group_scales_in: the array keeps the
    first call's words, which the second must not use."""
    import nvfp4_quantizers_gb300 as q
    experts = [W.moe_expert(e, hidden=512, ffn=128, seed=43) for e in range(4)]
    groups = [[_dev(g), _dev(u)] for g, u, _ in experts]
    _compare(L, groups)
    S_in = torch.tensor([0.5, 0.01, 2.0, 1e-4], dtype=torch.float32,
                        device="cuda")
    _compare(L, groups, S_in=S_in)

