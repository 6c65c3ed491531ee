"""FP8 block quantisation of the expert FFN, plain numpy -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU legs may import this
module; the product path never does.  It shares no code with the CUDA library.

Source: "Lower latency and higher throughput with multi-node DeepSeek deployment",
section "Quantization": DeepSeek-V3 runs its expert GEMMs in FP8 with block-wise scales --
weights quantised statically with one scale per 128 x 128 tile, activations dynamically
with one scale per vector of 128 elements.

Readings where the page leaves a step open (also listed in the design notes):
  * the FP8 format is E4M3 (largest finite value 448, subnormal step 2^-9), rounding to
    nearest with ties to even;
  * a block's scale is a power of two: the smallest 2^k with amax <= 448 * 2^k (k = 0 for
    an all-zero block), k kept within [-124, 127], so that every quantised value times its
    scale is exact in bf16 (down to its subnormals) and k fits one signed byte;
  * the activations quantised are the inputs of the two GEMMs of an expert: the token
    rows x (blocks of 128 along H) and h = silu(x W1) * (x W3) after it is rounded to bf16
    (blocks of 128 along I); the GEMMs then run on the dequantised values (q * 2^k) with
    fp64 sums here;
  * the router's gate GEMM is not quantised.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_values() -> np.ndarray:
    """Value of every byte of the E4M3 format (sign, 4 exponent bits with bias 7, 3
    mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN)."""
    out = np.empty(256)
    for b in range(256):
        s = -1.0 if b & 0x80 else 1.0
        e = (b >> 3) & 0xF
        m = b & 0x7
        if e == 0xF and m == 0x7:
            out[b] = np.nan
        elif e == 0:
            out[b] = s * m / 8.0 * 2.0 ** -6
        else:
            out[b] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Round float64 values (|v| <= 448) to the nearest E4M3 value, ties to even."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    if np.any(a > E4M3_MAX):
        raise ValueError("value outside the E4M3 range")
    e = np.frexp(np.where(a > 0, a, 1.0))[1] - 1  # a in [2^e, 2^(e+1)): exact
    e = np.maximum(e, -6)                         # below 2^-6 the grid step is 2^-9
    step = np.ldexp(1.0, e - 3)
    r = np.round(a / step) * step                 # numpy rounds halves to even
    return np.where(v < 0, -r, r)


K_MIN, K_MAX = -124, 127


def scale_exponent(amax: float) -> int:
    """Smallest k with amax <= 448 * 2^k (0 for amax == 0), kept within [-124, 127]."""
    if amax == 0:
        return 0
    m, e = np.frexp(float(amax))                  # amax = m 2^e, m in [0.5, 1)
    k = int(e - 9) if m <= 0.875 else int(e - 8)  # 448 = 0.875 * 2^9
    return min(max(k, K_MIN), K_MAX)


def quantize_tile(x: np.ndarray):
    """One block: (quantised E4M3 values, k); the dequantised block is q * 2^k."""
    x = np.asarray(x, dtype=np.float64)
    k = scale_exponent(float(np.abs(x).max()) if x.size else 0.0)
    return e4m3_round(x / 2.0 ** k), k


def _scale_exponents(amax: np.ndarray) -> np.ndarray:
    return np.vectorize(scale_exponent, otypes=[np.int64])(amax)


def quantize_weight(W: np.ndarray):
    """W [..., R, C] (R, C multiples of 128) -> q (same shape, E4M3 values as float64) and
    k [..., R/128, C/128] (int): each 128 x 128 tile on its own."""
    W = np.asarray(W, dtype=np.float64)
    R, C = W.shape[-2:]
    lead = W.shape[:-2]
    tiles = W.reshape(lead + (R // BLOCK, BLOCK, C // BLOCK, BLOCK))
    amax = np.abs(tiles).max(axis=(-3, -1))                     # [..., R/128, C/128]
    k = _scale_exponents(amax)
    scale = 2.0 ** k.astype(np.float64)
    q = e4m3_round(tiles / scale[..., :, None, :, None])
    return q.reshape(W.shape), k


def dequantize_weight(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    scale = 2.0 ** np.repeat(np.repeat(k.astype(np.float64), BLOCK, axis=-2), BLOCK, axis=-1)
    return q * scale


def fake_quant_rows(x: np.ndarray) -> np.ndarray:
    """Quantise then dequantise every row of x [..., n] in blocks of 128 along the row."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    v = x.reshape(x.shape[:-1] + (n // BLOCK, BLOCK))
    k = _scale_exponents(np.abs(v).max(axis=-1))
    scale = 2.0 ** k.astype(np.float64)[..., None]
    return (e4m3_round(v / scale) * scale).reshape(x.shape)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 value (ties to even), returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)                      # nearest float32
    u = f.view(np.uint32).astype(np.uint64)
    low = u & 0xFFFF
    keep = u >> 16
    # a float32 that sits exactly half-way between two bf16 values decides by the side the
    # float64 value was on (it was rounded onto the midpoint), else by the even neighbour
    above = np.abs(x) > np.abs(f.astype(np.float64))
    below = np.abs(x) < np.abs(f.astype(np.float64))
    tie_up = (low == 0x8000) & (above | (~below & ((keep & 1) == 1)))
    up = (low > 0x8000) | tie_up
    keep = keep + up.astype(np.uint64)
    return (keep << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def expert_rows_fp8(x_rows: np.ndarray, W1d: np.ndarray, W3d: np.ndarray, W2d: np.ndarray):
    """y = fq(h) W2d with h = bf16(silu(fq(x) W1d) * (fq(x) W3d)) for rows x [n, H] (bf16
    values as float64) and dequantised weights W1d, W3d [H, I], W2d [I, H]."""
    xq = fake_quant_rows(x_rows)
    u = xq @ W1d
    v = xq @ W3d
    h = u / (1.0 + np.exp(-u)) * v
    hq = fake_quant_rows(round_bf16(h))
    return hq @ W2d
