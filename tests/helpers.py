"""Shared test helpers: float64 restatements of what the method fixes in real
arithmetic (used to pin both the oracle and the CUDA path), plus record views.

Nothing here imports the CUDA binding or the oracle's internals.
"""
from functools import lru_cache

import numpy as np
import scipy.linalg

TAU = 1.0
EPS = float(np.float32(1e-30))
QMAX = 448.0


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


@lru_cache(maxsize=None)
def hadamard(B: int) -> np.ndarray:
    """Sylvester Hadamard matrix in natural order (SciPy), float64."""
    return scipy.linalg.hadamard(B).astype(np.float64)


def records(packed: np.ndarray, B: int):
    rec = np.asarray(packed, dtype=np.uint8).reshape(-1, B + 8)
    codes = rec[:, :B]
    alpha = rec[:, B:B + 4].copy().view("<f4").reshape(-1).astype(np.float64)
    s = rec[:, B + 4:B + 8].copy().view("<f4").reshape(-1).astype(np.float64)
    return codes, alpha, s


def exact_compress_quantities(G: np.ndarray, B: int):
    """Real-arithmetic values for blocks G [M, B] (float64):

    alpha = tau / sqrt(mean(G^2) + eps)            (Eqs. 6-7)
    y     = H_B G                                  (unnormalised rotation)
    u     = Z / s = Q_max * y / max|y|             (Eqs. 8-10; alpha cancels)
    s     = alpha * max|y| / (sqrt(B) * Q_max)     (Eq. 9)
    """
    G = np.asarray(G, dtype=np.float64).reshape(-1, B)
    m = (G * G).mean(axis=1)
    alpha = TAU / np.sqrt(m + EPS)
    y = G @ hadamard(B).T
    ymax = np.abs(y).max(axis=1)
    safe = np.where(ymax > 0, ymax, 1.0)
    u = np.where(ymax[:, None] > 0, QMAX * y / safe[:, None], 0.0)
    s = alpha * ymax / (np.sqrt(B) * QMAX)
    return alpha, s, u, m


def e4m3_half_ulp(u: np.ndarray) -> np.ndarray:
    """Half the E4M3 spacing at |u| (Eq. 3 with m = 3; subnormal spacing 2^-9)."""
    a = np.abs(np.asarray(u, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.where(a >= 2.0 ** -6, np.exp2(e - 3), 2.0 ** -9) / 2


def e4m3_decode_table() -> np.ndarray:
    """float64 value of each E4M3 code as PyTorch decodes it (a library routine)."""
    import torch
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def rel_l2(xhat, x) -> float:
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    xhat = np.asarray(xhat, dtype=np.float64).reshape(-1)
    nx = np.linalg.norm(x)
    return float(np.linalg.norm(xhat - x) / nx) if nx > 0 else float(np.linalg.norm(xhat))


def decode_table(code: int = 0) -> np.ndarray:
    """float64 value of each code byte: E4M3 (0) and E5M2 (1) as PyTorch
    decodes them, INT8 (2) as two's complement."""
    import torch
    if code == 2:
        return np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64)
    dt = torch.float8_e4m3fn if code == 0 else torch.float8_e5m2
    return torch.arange(256, dtype=torch.uint8).view(dt).to(torch.float64).numpy()


def code_step_distance(a: np.ndarray, b: np.ndarray, code: int = 0) -> np.ndarray:
    """Distance in grid steps between codes a and b of a format (E4M3 / E5M2:
    sign-magnitude, +0 and -0 the same value, a sign change adds the two
    magnitudes; INT8: the difference of the integers)."""
    if code == 2:
        return np.abs(np.asarray(a, dtype=np.uint8).view(np.int8).astype(np.int32)
                      - np.asarray(b, dtype=np.uint8).view(np.int8).astype(np.int32))
    a = np.asarray(a, dtype=np.int32)
    b = np.asarray(b, dtype=np.int32)
    ma, mb = a & 0x7F, b & 0x7F
    sa, sb = a >> 7, b >> 7
    same_sign = (sa == sb) | (ma == 0) | (mb == 0)
    d = np.abs(ma - mb)
    # Across zero: magnitude steps add up when the signs differ.
    d = np.where(same_sign, d, ma + mb)
    return np.where((ma == 0) & (mb == 0), 0, d)
