"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds none of the quantizers' arithmetic: it only draws random
numbers (numpy PCG64, seeded), shapes them like the workloads of "Miles:
end-to-end MXFP8 and per-token NVFP4 RL" (Qwen3-30B-A3B-style MoE: hidden
2048, expert FFN 768, 128 experts, top-8; the linear shape (2048, 2048) ->
8192 of its memory section), and rounds fp32 samples to bf16 with torch's
own cast.  Every bf16 tensor is returned as a numpy ``uint16`` array of bit
patterns so that the CPU oracle and the GPU path consume the same bytes.

The four input classes follow the quantizer-alignment section of that page
(random, quantization-boundary, all-zero, maximum-value data).
"""
from __future__ import annotations

import hashlib
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

BF16_MAX_BITS = 0x7F7F          # largest finite bf16, (2 - 2^-7) * 2^127


def to_bf16_bits(a) -> np.ndarray:
    """fp32/fp64 samples -> bf16 bit patterns (torch's round-to-nearest-even
    cast)."""
    a = np.array(a, dtype=np.float32, order="C")
    t = torch.from_numpy(a.reshape(-1))
    bits = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return bits.reshape(a.shape)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def sha256(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


# E4M3 grid facts used only to place test values (input design, not the
# quantizer): normal magnitudes (1 + m/8) * 2^e, e in [-6, 8]; midpoints
# between neighbours; subnormal steps 2^-9.
def _e4m3_midpoints() -> np.ndarray:
    vals = [m / 8.0 * 2.0 ** -6 for m in range(8)]
    for e in range(-6, 9):
        for m in range(8):
            v = (1 + m / 8.0) * 2.0 ** e
            if v <= 448.0:
                vals.append(v)
    vals = np.array(sorted(set(vals)))
    return (vals[:-1] + vals[1:]) / 2.0          # all strictly below 448


E4M3_MIDPOINTS = _e4m3_midpoints()


def _signs(rng, shape):
    return np.where(rng.random(shape) < 0.5, -1.0, 1.0)


# --------------------------------------------------------------------------
# MXFP8 small case: [256 x 512] N(0,1), last six rows replaced by edge rows.
# --------------------------------------------------------------------------
def mxfp8_small(seed: int = 0, rows: int = 256, cols: int = 512) -> np.ndarray:
    rng = _rng(seed, 1)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    nb = cols // 32
    js = np.arange(nb) - 8                      # scale exponents -8 .. 7
    # (i) block maxima exactly +-448 * 2^j, other entries E4M3 midpoints * 2^j
    r = np.empty(cols)
    for b in range(nb):
        j = js[b % len(js)]
        mids = rng.choice(E4M3_MIDPOINTS, 32) * 2.0 ** j
        mids[rng.integers(32)] = 448.0 * 2.0 ** j
        r[b * 32:(b + 1) * 32] = mids * _signs(rng, 32)
    x[rows - 6] = r
    # (ii) subnormal-range codes and ties to zero under a block max 448 * 2^j
    for b in range(nb):
        j = js[b % len(js)]
        v = np.array([2.0 ** -9 * m for m in range(1, 8)] +
                     [2.0 ** -10 * (2 * m + 1) for m in range(8)] +
                     [2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -10])
        blk = rng.choice(v, 32) * 2.0 ** j
        blk[0] = 448.0 * 2.0 ** j
        r[b * 32:(b + 1) * 32] = blk * _signs(rng, 32)
    x[rows - 5] = r
    # (iii) power-of-two block maxima 2^m, m spread over [-20, 20]
    ms = np.linspace(-20, 20, nb).round().astype(int)
    for b in range(nb):
        blk = rng.uniform(-1, 1, 32) * 2.0 ** ms[b]
        blk[rng.integers(32)] = 2.0 ** ms[b]
        r[b * 32:(b + 1) * 32] = blk
    x[rows - 4] = r
    x = to_bf16_bits(x)
    # (iv) block max 448 * 2^j +- one bf16 ulp (pins the round-up of the scale)
    row = to_bf16_bits(rng.uniform(-1, 1, cols).astype(np.float32))
    for b in range(nb):
        j = int(js[b % len(js)])
        top = int(to_bf16_bits(np.float32(448.0 * 2.0 ** j)))
        top = top + 1 if b % 2 == 0 else top - 1
        blk = to_bf16_bits(rng.uniform(-1, 1, 32) * 2.0 ** j * 200.0)
        blk[rng.integers(32)] = top
        row[b * 32:(b + 1) * 32] = blk
    x[rows - 3] = row
    # (v) all zero, (vi) all +-bf16 max
    x[rows - 2] = 0
    sgn = (rng.random(cols) < 0.5).astype(np.uint16) << 15
    x[rows - 1] = BF16_MAX_BITS | sgn
    return x


# --------------------------------------------------------------------------
# MXFP8 activation classes [M x K] (default 8192 x 4096).
# --------------------------------------------------------------------------
def mxfp8_random(M=8192, K=4096, seed=0, outlier_frac=1e-3, outlier_mul=100.0):
    """N(0,1) with a fraction of entries (chosen without replacement)
    multiplied by 100 (outliers)."""
    rng = _rng(seed, 2, M, K)
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * M * K))
    if n_out:
        idx = rng.choice(M * K, n_out, replace=False)
        x.reshape(-1)[idx] *= outlier_mul
    return to_bf16_bits(x)


def mxfp8_boundary(M=8192, K=4096, seed=0):
    """Every 32x32 tile has its diagonal at +-448 * 2^j (j cycles over
    [-10, 10] tile by tile), so every row block and every column block has
    amax 448 * 2^j; off-diagonal entries are E4M3 midpoints (normal and
    subnormal) times 2^j.  One tile in eight has its diagonal one bf16 ulp
    above 448 * 2^j (the saturation edge, where the scale steps up)."""
    rng = _rng(seed, 3, M, K)
    tm, tk = M // 32, K // 32
    j = (np.arange(tm * tk) % 21 - 10).reshape(tm, tk)
    mids = rng.choice(E4M3_MIDPOINTS, (M, K)).astype(np.float32)
    pow2 = np.repeat(np.repeat(np.ldexp(1.0, j), 32, 0), 32, 1).astype(np.float32)
    x = mids * pow2 * _signs(rng, (M, K)).astype(np.float32)
    bits = to_bf16_bits(x)
    diag_r = np.arange(M)
    diag_c = diag_r % 32                             # column offset in tile
    sgn = (rng.random((M, tk)) < 0.5).astype(np.uint16) << 15
    edge = (np.arange(tm * tk).reshape(tm, tk) % 8) == 3
    for ct in range(tk):
        jj = j[diag_r // 32, ct]
        top = to_bf16_bits((448.0 * np.ldexp(1.0, jj)).astype(np.float32))
        top = top + edge[diag_r // 32, ct].astype(np.uint16)
        bits[diag_r, ct * 32 + diag_c] = top | sgn[:, ct]
    return bits


def mxfp8_zeros(M=8192, K=4096, seed=0):
    return np.zeros((M, K), np.uint16)


def mxfp8_maxes(M=8192, K=4096, seed=0):
    """Every element +-bf16 max (0x7F7F), random signs."""
    rng = _rng(seed, 4, M, K)
    sgn = (rng.random((M, K)) < 0.5).astype(np.uint16) << 15
    return (np.uint16(BF16_MAX_BITS) | sgn).astype(np.uint16)


def fmt_maxes(M, K, value, seed=0):
    """Every element +-value (e.g. 448 for MXFP8, 2688 for NVFP4)."""
    rng = _rng(seed, 5, M, K)
    return to_bf16_bits(_signs(rng, (M, K)) * value)


MXFP8_CLASSES = {
    "random": mxfp8_random,
    "boundary": mxfp8_boundary,
    "zeros": mxfp8_zeros,
    "maxes": mxfp8_maxes,
}


def linear_input(M=2048, K=2048, seed=0):
    """The memory section's linear: input (2048, 2048), N(0, 1)."""
    return to_bf16_bits(_rng(seed, 6, M, K).standard_normal((M, K),
                                                            dtype=np.float32))


def linear_weight(N=8192, K=2048, seed=0):
    """The memory section's linear: weight [8192 x 2048], N(0, 0.02)."""
    return to_bf16_bits(0.02 * _rng(seed, 7, N, K).standard_normal(
        (N, K), dtype=np.float32))


# --------------------------------------------------------------------------
# NVFP4 activations: ragged batch of sequences, Student-t(4), sparse
# per-token outliers.
# --------------------------------------------------------------------------
def ragged_lengths(n_seq=64, lo=128, hi=4096, seed=0) -> np.ndarray:
    return _rng(seed, 8).integers(lo, hi, size=n_seq, endpoint=True)


def ragged_tokens(lengths, H=2048, seed=0, outlier_token_frac=0.02,
                  outlier_channels=4, outlier_mul=100.0) -> np.ndarray:
    """Flattened [sum(lengths) x H] bf16 activations: t(4) values; in a
    fraction of tokens a few random channels are multiplied by 100.  Every
    sequence draws from its own generator, so the sequences are made on a
    thread pool with the same result as one after the other."""
    lengths = np.asarray(lengths, np.int64)
    out = np.empty((int(np.sum(lengths)), H), np.uint16)
    starts = np.concatenate([[0], np.cumsum(lengths)])

    def one(s):
        L = int(lengths[s])
        rng = _rng(seed, 9, s)
        v = rng.standard_t(4, size=(L, H)).astype(np.float32)
        hit = np.nonzero(rng.random(L) < outlier_token_frac)[0]
        for t in hit:
            ch = rng.choice(H, outlier_channels, replace=False)
            v[t, ch] *= outlier_mul
        out[starts[s]:starts[s] + L] = to_bf16_bits(v)

    with ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(one, range(len(lengths))))
    return out


def tiny_token_rows(H=2048, seed=0) -> np.ndarray:
    """Edge tokens for NVFP4: all zero, a token whose FP32 scale is
    subnormal (amax ~ 1e-37), a token of all +-2688 (S = 1), one of all
    +-bf16 max, a token with one huge channel (block scales that round to
    zero), and one with E2M1 midpoints."""
    rng = _rng(seed, 10)
    rows = [np.zeros(H, np.float32),
            (rng.uniform(-1, 1, H) * 1e-37).astype(np.float32),
            (_signs(rng, H) * 2688.0).astype(np.float32),
            None,
            rng.uniform(-1e-6, 1e-6, H).astype(np.float32),
            (rng.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], H)
             * _signs(rng, H)).astype(np.float32)]
    rows[4][rng.integers(H)] = 3.0e4
    rows[5][0] = 6.0
    bits = []
    for r in rows:
        if r is None:
            sgn = (rng.random(H) < 0.5).astype(np.uint16) << 15
            bits.append((np.uint16(BF16_MAX_BITS) | sgn).astype(np.uint16))
        else:
            bits.append(to_bf16_bits(r))
    return np.stack(bits)


# --------------------------------------------------------------------------
# NVFP4 MoE weights: Qwen3-30B-A3B-shaped experts.
# --------------------------------------------------------------------------
def moe_expert(e: int, hidden=2048, ffn=768, seed=0, outlier_frac=1e-4,
               outlier_mul=20.0):
    """(gate [ffn x hidden], up [ffn x hidden], down [hidden x ffn]) bf16
    bits, N(0, 0.02) with a fraction of entries multiplied by 20."""
    rng = _rng(seed, 11, e)
    out = []
    for shape in ((ffn, hidden), (ffn, hidden), (hidden, ffn)):
        w = 0.02 * rng.standard_normal(shape, dtype=np.float32)
        n_out = int(round(outlier_frac * w.size))
        if n_out:
            idx = rng.choice(w.size, n_out, replace=False)
            w.reshape(-1)[idx] *= outlier_mul
        out.append(to_bf16_bits(w))
    return tuple(out)


def moe_layer(n_experts=128, hidden=2048, ffn=768, seed=0):
    """moe_expert for experts 0 .. n_experts-1 (each from its own generator),
    made on a thread pool."""
    with ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        return list(ex.map(lambda e: moe_expert(e, hidden, ffn, seed),
                           range(n_experts)))


# --------------------------------------------------------------------------
# GEMM consumer inputs.
# --------------------------------------------------------------------------
def gemm_mxfp8_inputs(M=2048, K=2048, N=8192, seed=0):
    """A [M x K] N(0,1); B [K x N] N(0, 0.02)."""
    A = to_bf16_bits(_rng(seed, 12).standard_normal((M, K), dtype=np.float32))
    B = to_bf16_bits(0.02 * _rng(seed, 13).standard_normal((K, N),
                                                           dtype=np.float32))
    return A, B


def topk_routing(n_tokens=4096, n_experts=128, k=8, seed=0) -> np.ndarray:
    """[n_tokens x k] distinct experts per token, uniform (top-k routing)."""
    rng = _rng(seed, 14)
    return np.stack([rng.choice(n_experts, k, replace=False)
                     for _ in range(n_tokens)])


def gemm_tokens(n_tokens=4096, H=2048, seed=0):
    return to_bf16_bits(_rng(seed, 15).standard_normal((n_tokens, H),
                                                       dtype=np.float32))


def expert_gather_index(route: np.ndarray, n_experts: int, pad: int = 128):
    """Rows of the grouped expert GEMM from top-k routing: expert e's group
    lists (in token order) the tokens routed to it, padded with -1 entries
    to a multiple of `pad` rows.  Returns (row_index int32 [rows],
    offsets int64 [n_experts + 1], group sizes before padding)."""
    idx, offs, sizes = [], [0], []
    for e in range(n_experts):
        toks = np.nonzero((route == e).any(axis=1))[0]
        sizes.append(len(toks))
        padded = -(-len(toks) // pad) * pad
        idx.append(np.concatenate([toks, np.full(padded - len(toks), -1)]))
        offs.append(offs[-1] + padded)
    return (np.concatenate(idx).astype(np.int32), np.array(offs, np.int64),
            np.array(sizes))
