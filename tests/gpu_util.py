"""Helpers shared by the GPU tests: moving bf16 bit patterns to and from the
device and comparing byte buffers with readable failure messages."""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """numpy uint16 bf16 bit patterns -> CUDA bfloat16 tensor (same bytes)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint8)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """CUDA bfloat16 tensor -> numpy uint16 bit patterns."""
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_bytes_equal(got: np.ndarray, exp: np.ndarray, what: str, cols=None):
    got = np.asarray(got)
    exp = np.asarray(exp)
    assert got.shape == exp.shape, f"{what}: shape {got.shape} != {exp.shape}"
    if np.array_equal(got, exp):
        return
    bad = np.argwhere(got != exp)
    lines = [f"{what}: {len(bad)} mismatches, first ones:"]
    for idx in bad[:10]:
        idx = tuple(int(i) for i in idx)
        lines.append(f"  at {idx}: got {got[idx]:#x} expected {exp[idx]:#x}")
    raise AssertionError("\n".join(lines))
