"""Seeded synthetic inputs for the AWQ W4A16 GEMM-layout linear.

This module only draws random numbers.  It contains none of the method's
arithmetic: no nibble order, no unpacking, no dequantization, no matmul.
Both the oracle (test side) and the CUDA path (through tests and the
benchmark) consume what it produces, and nothing else is shared between
them.

Why the packed words can be drawn directly: in the AWQ GEMM layout
(tensref.org/formats/awq, "Reader" pseudo-code) every int32 word of
``qweight`` / ``qzeros`` holds eight 4-bit codes, one per nibble.  A word
whose 32 bits are uniform and independent holds eight independent codes,
each uniform on 0..15, whatever nibble order a reader applies.  Drawing
uniform 32-bit words therefore has exactly the distribution "codes and
zeros uniform 0..15, packed with ORDER" that the workloads ask for, without
this module having to know ORDER.

Workload recipe (per linear, draw order x, codes, zeros, scales, bias):
  * x      fp16 [M, K]     standard normal drawn in fp32, rounded to fp16
  * qweight int32 [K, N/8] uniform 32-bit words
  * qzeros int32 [K/G, N/8] uniform 32-bit words (0x88888888 when sym: every
           nibble 8, the symmetric zero point of GPTQModel wiki "AWQ",
           "Group quantization and zero points")
  * scales fp16 [K/G, N]   uniform [1e-3, 1e-2) drawn in fp32, rounded to fp16
  * bias   fp16 [N]        normal(0, 0.02) drawn in fp32, rounded to fp16
G = K when group_size == -1.
With dtype="bf16" the same draws are rounded to bf16 instead of fp16 (by torch's
conversion) and returned as fp32 arrays holding the bf16 values.
"""
from __future__ import annotations

import numpy as np

__all__ = ["awq_linear", "seed_for", "SYM_ZERO_WORD", "moe_inputs", "awq8_linear"]

# Every nibble equal to 8.  A word with all nibbles equal is invariant under
# any nibble permutation, so no ordering knowledge is needed to write it.
SYM_ZERO_WORD = np.uint32(0x88888888).view(np.int32)


def seed_for(config_index: int, shape_index: int) -> int:
    """Seed of one (config, shape) workload: 1000 + 100*config + shape."""
    return 1000 + 100 * int(config_index) + int(shape_index)


def _groups(K: int, group_size: int) -> int:
    G = K if group_size == -1 else group_size
    if G <= 0 or K % G != 0:
        raise ValueError(f"group_size={group_size} does not divide K={K}")
    return K // G


def awq_linear(seed: int, M: int, K: int, N: int, group_size: int = 128,
               bias: bool = False, sym: bool = False,
               x_kind: str = "normal", scale_kind: str = "uniform",
               bias_kind: str = "normal", dtype: str = "f16") -> dict:
    """Draw one synthetic AWQ linear plus an activation batch.

    Returns a dict of numpy arrays: ``x`` fp16 [M,K], ``qweight`` int32
    [K,N/8], ``qzeros`` int32 [K/G,N/8], ``scales`` fp16 [K/G,N], ``bias``
    fp16 [N] or None, plus ``group_size``.

    ``x_kind``: "normal" (N(0,1)) or "smallint" (integers in [-4, 4], used by
    the exact-arithmetic cases).  ``scale_kind``: "uniform" ([1e-3,1e-2)) or
    "pow2" (2**-p with p uniform in 4..9, also for exact cases).
    ``bias_kind``: "normal" or "dyadic" (multiples of 1/64 in [-1, 1]).
    """
    if N % 8 != 0:
        raise ValueError("N must be a multiple of 8 (eight codes per int32 word)")
    if dtype not in ("f16", "bf16"):
        raise ValueError(dtype)
    half = np.float16 if dtype == "f16" else _to_bf16
    n_groups = _groups(K, group_size)
    rng = np.random.Generator(np.random.PCG64(seed))
    if x_kind == "normal":
        x = _as(rng.standard_normal((M, K), dtype=np.float32), half)
    elif x_kind == "smallint":
        x = _as(rng.integers(-4, 5, size=(M, K)).astype(np.float32), half)
    else:
        raise ValueError(x_kind)
    qweight = rng.integers(0, 1 << 32, size=(K, N // 8), dtype=np.uint64)
    qweight = qweight.astype(np.uint32).view(np.int32)
    if sym:
        qzeros = np.full((n_groups, N // 8), SYM_ZERO_WORD, dtype=np.int32)
    else:
        qzeros = rng.integers(0, 1 << 32, size=(n_groups, N // 8), dtype=np.uint64)
        qzeros = qzeros.astype(np.uint32).view(np.int32)
    if scale_kind == "uniform":
        scales = rng.uniform(1e-3, 1e-2, size=(n_groups, N)).astype(np.float32)
        scales = _as(scales, half)
    elif scale_kind == "pow2":
        p = rng.integers(4, 10, size=(n_groups, N))
        scales = _as(np.ldexp(np.ones((n_groups, N), np.float32), -p), half)
    else:
        raise ValueError(scale_kind)
    b = None
    if bias:
        if bias_kind == "normal":
            b = _as(rng.normal(0.0, 0.02, size=N).astype(np.float32), half)
        elif bias_kind == "dyadic":
            b = _as((rng.integers(-64, 65, size=N) / 64.0).astype(np.float32), half)
        else:
            raise ValueError(bias_kind)
    return {"x": np.ascontiguousarray(x), "qweight": np.ascontiguousarray(qweight),
            "qzeros": np.ascontiguousarray(qzeros), "scales": np.ascontiguousarray(scales),
            "bias": b, "group_size": int(group_size), "M": M, "K": K, "N": N, "dtype": dtype}


def _to_bf16(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 by torch's conversion, back as fp32 arrays holding bf16 values."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _as(a: np.ndarray, half) -> np.ndarray:
    return a.astype(np.float16) if half is np.float16 else half(a)


# Workloads shaped like the 7B / 70B linears the pages discuss.  Each entry:
# (config index, shape index, name, M, K, N, group_size, bias).  Shapes only; seeds
# come from seed_for(config, shape).
_L7 = [(4096, 4096), (4096, 11008), (11008, 4096)]
_L70 = [(8192, 8192), (8192, 28672), (28672, 8192)]


def _workloads():
    out = [(0, 0, "tiny_m1_256x256", 1, 256, 256, 128, False)]
    si = 0
    for K, N in _L7:
        for b in (False, True):
            out.append((1, si, f"7b_decode_m1_{K}x{N}{'_bias' if b else ''}", 1, K, N, 128, b))
            si += 1
    si = 0
    for M in (4, 8, 16, 32):
        for K, N in _L7:
            out.append((2, si, f"7b_smallbatch_m{M}_{K}x{N}", M, K, N, 128, False))
            si += 1
    for K, N in _L7:
        out.append((2, si, f"7b_smallbatch_m8_{K}x{N}_g-1", 8, K, N, -1, False))
        si += 1
    si = 0
    for M in (512, 2048):
        for K, N in [(4096, 11008), (11008, 4096)]:
            out.append((3, si, f"7b_prefill_m{M}_{K}x{N}", M, K, N, 128, False))
            si += 1
    si = 0
    for M in (1, 16, 4096):
        for K, N in _L70:
            out.append((4, si, f"70b_m{M}_{K}x{N}", M, K, N, 128, True))
            si += 1
    return out


WORKLOADS = _workloads()


def workload(name: str):
    for w in WORKLOADS:
        if w[2] == name:
            return w
    raise KeyError(name)


def workload_inputs(name: str, dtype: str = "f16") -> dict:
    cfg, si, _, M, K, N, G, b = workload(name)
    return awq_linear(seed_for(cfg, si), M, K, N, group_size=G, bias=b, dtype=dtype)


def moe_inputs(seed: int, T: int, topk: int, E: int, K: int, N: int, group_size: int = 128,
               bias: bool = False, dtype: str = "f16") -> dict:
    """Synthetic mixture-of-experts layer: E experts' AWQ linears (each drawn as
    awq_linear, seeds seed + 1 + e) and T tokens each routed to topk distinct experts
    drawn uniformly; the routed rows (token copies) are sorted by expert (stable), so
    expert e owns rows offsets[e] .. offsets[e+1]-1.  Returns x [T*topk, K] fp16,
    qweight [E, K, N/8], qzeros [E, K/G, N/8], scales [E, K/G, N], bias [E, N] or None,
    offsets int32 [E+1], token_of_row, plus the sizes.  dtype="bf16": x, scales and bias
    rounded to bf16 instead (fp32 arrays holding bf16 values, as awq_linear)."""
    if dtype not in ("f16", "bf16"):
        raise ValueError("dtype must be 'f16' or 'bf16'")
    half = np.float16 if dtype == "f16" else _to_bf16
    rng = np.random.Generator(np.random.PCG64(seed))
    tokens = half(rng.standard_normal((T, K), dtype=np.float32))
    choice = np.stack([rng.permutation(E)[:topk] for _ in range(T)])   # [T, topk]
    expert_of_row = choice.reshape(-1)
    token_of_row = np.repeat(np.arange(T), topk)
    order = np.argsort(expert_of_row, kind="stable")
    expert_of_row, token_of_row = expert_of_row[order], token_of_row[order]
    counts = np.bincount(expert_of_row, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ex = [awq_linear(seed + 1 + e, 1, K, N, group_size=group_size, bias=bias, dtype=dtype) for e in range(E)]
    return {"x": np.ascontiguousarray(tokens[token_of_row]),
            "qweight": np.ascontiguousarray(np.stack([d["qweight"] for d in ex])),
            "qzeros": np.ascontiguousarray(np.stack([d["qzeros"] for d in ex])),
            "scales": np.ascontiguousarray(np.stack([d["scales"] for d in ex])),
            "bias": np.ascontiguousarray(np.stack([d["bias"] for d in ex])) if bias else None,
            "offsets": offsets, "token_of_row": token_of_row, "group_size": int(group_size),
            "R": int(T * topk), "E": E, "K": K, "N": N}


def awq8_linear(seed: int, M: int, K: int, N: int, group_size: int = 128, bias: bool = False,
                x_kind: str = "normal", scale_kind: str = "uniform") -> dict:
    """8-bit variant of awq_linear: qweight int32 [K, N/4] and qzeros int32 [K/G, N/4] are
    uniform 32-bit words (four independent uniform 8-bit codes each, whatever byte order
    a reader applies); x, scales, bias drawn as for 4 bits (scales uniform [1e-4, 1e-3):
    codes span 256 levels)."""
    if N % 4 != 0:
        raise ValueError("N must be a multiple of 4 (four codes per int32 word)")
    n_groups = _groups(K, group_size)
    rng = np.random.Generator(np.random.PCG64(seed))
    if x_kind == "normal":
        x = rng.standard_normal((M, K), dtype=np.float32).astype(np.float16)
    else:
        x = rng.integers(-4, 5, size=(M, K)).astype(np.float16)
    qweight = rng.integers(0, 1 << 32, size=(K, N // 4), dtype=np.uint64).astype(np.uint32).view(np.int32)
    qzeros = rng.integers(0, 1 << 32, size=(n_groups, N // 4), dtype=np.uint64).astype(np.uint32).view(np.int32)
    if scale_kind == "uniform":
        scales = rng.uniform(1e-4, 1e-3, size=(n_groups, N)).astype(np.float32).astype(np.float16)
    else:
        p = rng.integers(8, 14, size=(n_groups, N))
        scales = np.ldexp(np.ones((n_groups, N), np.float32), -p).astype(np.float16)
    b = rng.normal(0.0, 0.02, size=N).astype(np.float32).astype(np.float16) if bias else None
    return {"x": np.ascontiguousarray(x), "qweight": np.ascontiguousarray(qweight),
            "qzeros": np.ascontiguousarray(qzeros), "scales": np.ascontiguousarray(scales),
            "bias": b, "group_size": int(group_size), "M": M, "K": K, "N": N, "bits": 8}

