"""Seeded synthetic BF16 workloads shared by the tests, the oracle checks and the benchmark.

This module holds none of the coding method's arithmetic: it only draws random
numbers (numpy ``Generator``), scales them, rounds them to bfloat16 with
torch's CPU conversion, and returns the raw 16-bit patterns as ``numpy.uint16``.

The real tensors the ZipCCL summary evaluates on (Llama3-8B, Qwen3-MoE and
DeepSeek-V3 training traffic, [ZipCCL §4]) are not available; these stand in
for them with the shapes and value distributions its method section assumes:
near-Gaussian tensors [ZipCCL §2.A], gradient outliers and special values,
a Llama-3-8B per-layer parameter bucket, an MoE all-to-all payload with
imbalanced destinations [ZipCCL §2.D] and reduce-scatter shards.

Workloads (n = elements):
  gaussian      n = 2^20, N(0, 0.02), seed 1 -- the small round-trip case
  gradient      n = 2^26, N(0, 1e-3); 0.1% of positions x1000; 0.01% special
                values cycling {+0, -0, +sub, -sub, +inf, -inf, NaN} with random
                subnormal mantissas and NaN payloads; seed 2
  llama_bucket  9 tensors of a Llama-3-8B layer (q, k, v, o, gate, up, down,
                2 RMSNorm vectors), each N(0, s_t), s_t log-uniform in
                [1e-4, 5e-2]; seed 3 + tensor index
  moe_payload   16384 x 4096, 0.5 * Student-t(4); destination token counts
                Zipf(1.2) over 8 ranks (largest-remainder rounding); seed 4
  rs_shards     P = 8 shards of m = 2^25 elements, N(0, 1e-3); seed 5 + rank
  random_bits   n = 2^26 uniformly random 16-bit patterns, seed 6 -- data the
                exponent coding cannot shrink (exponents spread over all 256
                values), the case of the raw bypass
  fp8_ffn1      n = 2^26 FP8 e4m3 bytes: GELU(z), z ~ N(0, 1), scaled so the
                largest magnitude maps to 448 (the e4m3 maximum) and rounded to
                e4m3 by torch (round to nearest even); seed 7 -- a stand-in for
                the FFN1 activations of the QLC article's Gemma 2B layers
  fp8_gradient  n = 2^26 e4m3 bytes of N(0, 1) scaled the same way; seed 8
"""
from __future__ import annotations

import numpy as np
import torch

GAUSSIAN_SIGMA = 0.02
GRADIENT_SIGMA = 1e-3
RS_SIGMA = 1e-3

LLAMA3_8B_LAYER = [
    ("q_proj", (4096, 4096)),
    ("k_proj", (1024, 4096)),
    ("v_proj", (1024, 4096)),
    ("o_proj", (4096, 4096)),
    ("gate_proj", (14336, 4096)),
    ("up_proj", (14336, 4096)),
    ("down_proj", (4096, 14336)),
    ("input_layernorm", (4096,)),
    ("post_attention_layernorm", (4096,)),
]


def to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """Round float32/float64 values to bfloat16 (torch CPU, round-to-nearest-even); return uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def gaussian(n: int = 1 << 20, sigma: float = GAUSSIAN_SIGMA, seed: int = 1) -> np.ndarray:
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(n, dtype=np.float32) * np.float32(sigma)
    return to_bf16_bits(v)


def _special_patterns(rng: np.random.Generator, count: int) -> np.ndarray:
    """Cycle {+0, -0, +subnormal, -subnormal, +inf, -inf, NaN} with random payloads."""
    out = np.zeros(count, np.uint16)
    kind = np.arange(count) % 7
    sub_mant = rng.integers(1, 128, size=count, dtype=np.uint16)   # non-zero 7-bit mantissa
    nan_payload = rng.integers(1, 128, size=count, dtype=np.uint16)
    nan_sign = rng.integers(0, 2, size=count, dtype=np.uint16) << 15
    out[kind == 0] = 0x0000
    out[kind == 1] = 0x8000
    out[kind == 2] = sub_mant[kind == 2]
    out[kind == 3] = 0x8000 | sub_mant[kind == 3]
    out[kind == 4] = 0x7F80
    out[kind == 5] = 0xFF80
    out[kind == 6] = nan_sign[kind == 6] | 0x7F80 | nan_payload[kind == 6]
    return out


def gradient(n: int = 1 << 26, sigma: float = GRADIENT_SIGMA, seed: int = 2,
             outlier_frac: float = 1e-3, special_frac: float = 1e-4) -> np.ndarray:
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(n, dtype=np.float32) * np.float32(sigma)
    n_out = int(round(n * outlier_frac))
    n_spec = int(round(n * special_frac))
    pos = rng.choice(n, n_out + n_spec, replace=False)
    v[pos[:n_out]] *= np.float32(1000.0)
    x = to_bf16_bits(v)
    x[pos[n_out:]] = _special_patterns(rng, n_spec)
    return x


def llama_bucket(seed: int = 3, scale: float = 1.0):
    """Return [(name, bits uint16[n], sigma)] for one Llama-3-8B layer's parameters.

    ``scale`` < 1 shrinks every matrix's row count (for fast CPU tests) while
    keeping the nine-tensor structure, the RMSNorm vectors and the sigmas.
    """
    out = []
    for i, (name, shape) in enumerate(LLAMA3_8B_LAYER):
        rng = np.random.default_rng(seed + i)
        sigma = float(np.exp(rng.uniform(np.log(1e-4), np.log(5e-2))))
        if len(shape) == 2 and scale != 1.0:
            shape = (max(1, int(shape[0] * scale)), shape[1])
        n = int(np.prod(shape))
        v = rng.standard_normal(n, dtype=np.float32) * np.float32(sigma)
        out.append((name, to_bf16_bits(v), sigma))
    return out


def zipf_counts(total: int = 16384, ranks: int = 8, s: float = 1.2) -> list[int]:
    """Expected Zipf(s) counts over ``ranks`` destinations, largest-remainder rounded."""
    w = np.arange(1, ranks + 1, dtype=np.float64) ** (-s)
    q = total * w / w.sum()
    fl = np.floor(q).astype(np.int64)
    order = np.argsort(-(q - fl), kind="stable")
    fl[order[: total - int(fl.sum())]] += 1
    return [int(c) for c in fl]


def moe_payload(tokens: int = 16384, hidden: int = 4096, seed: int = 4, ranks: int = 8):
    """Return (bits uint16[tokens*hidden], per-destination token counts); rows contiguous per destination."""
    rng = np.random.default_rng(seed)
    v = (rng.standard_t(4, size=tokens * hidden) * 0.5).astype(np.float32)
    return to_bf16_bits(v), zipf_counts(tokens, ranks)


def rs_shards(P: int = 8, m: int = 1 << 25, sigma: float = RS_SIGMA, seed: int = 5):
    """Return a list of P uint16 arrays of m elements, shard r drawn with seed + r."""
    shards = []
    for r in range(P):
        rng = np.random.default_rng(seed + r)
        shards.append(to_bf16_bits(rng.standard_normal(m, dtype=np.float32) * np.float32(sigma)))
    return shards


def gaussian_on_device(n: int, sigma: float, seed: int, device="cuda") -> torch.Tensor:
    """N(0, sigma^2) rounded to bfloat16, drawn on the device with torch's seeded generator (for tensors too
    large to draw and copy from the host); returned as the int16 bit patterns."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return (torch.randn(n, device=device, generator=g) * sigma).to(torch.bfloat16).view(torch.int16)


def random_bits(n: int = 1 << 26, seed: int = 6) -> np.ndarray:
    """Uniformly random bf16 bit patterns (NaNs and infinities included)."""
    return np.random.default_rng(seed).integers(0, 65536, n, dtype=np.uint16)


def to_e4m3_bits(values: np.ndarray) -> np.ndarray:
    """Scale so that max |value| becomes 448, round to float8 e4m3 (torch, nearest even); return the bytes."""
    v = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    amax = float(v.abs().max()) if v.numel() else 1.0
    v = v * (448.0 / amax if amax > 0 else 1.0)
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def fp8_ffn1(n: int = 1 << 26, seed: int = 7) -> np.ndarray:
    z = torch.from_numpy(np.random.default_rng(seed).standard_normal(n, dtype=np.float32))
    return to_e4m3_bits(torch.nn.functional.gelu(z).numpy())


def fp8_gradient(n: int = 1 << 26, seed: int = 8) -> np.ndarray:
    return to_e4m3_bits(np.random.default_rng(seed).standard_normal(n, dtype=np.float32))


def all_bf16_patterns() -> np.ndarray:
    """Every 16-bit pattern once (0x0000 .. 0xFFFF)."""
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)
