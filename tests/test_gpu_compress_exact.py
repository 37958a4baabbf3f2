"""The compress kernels' arithmetic on inputs whose rotation is exact.

Blocks of small integers times a power of two (bf16 exact, bf16 subnormals
included) have an exact Hadamard transform y = H G in binary32 whatever the
summation order, so the host can form what each kernel computes from y
(TACO paper, Section 4.3, Eqs. 9-10, in the rotated-domain form the kernels
use, where alpha cancels from the codes):

  ASH + DS, standard Hadamard + DS:
      k = fl(Q_max / max|y|),  codes = Cvt(fl(y * k))
      for max|y| < 2^-100 (k would overflow): k = fl(Q_max / fl(max|y| 2^64)),
      codes = Cvt(fl(fl(y 2^64) * k))
      s = fl(fl(fl(alpha * max|y|) * r_B) / Q_max)
  DS only:  s = fl(max|G| / Q_max),  codes = Cvt(fl(G / s))   (Eq. 10 as written)
  ASH only: s = 1,  codes = Cvt(fl(y * fl(alpha * r_B)))

with r_B = 1/sqrt(B) in binary32, alpha read back from the record where it
enters (ASH + DS's s and ASH only's codes) and checked against
tau / sqrt(|G|^2 / B + eps) to 1e-6; alpha = 1 exactly for the non-adaptive
variants.  Codes and s must match exactly.  A product fused into the INT8
rounding add (the integer nearest the exact product instead of the binary32
one) fails here; so would a code multiplier formed in another order.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import hadamard, records

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TAU = 1.0
EPS = float(np.float32(1e-30))
QMAX = {0: 448.0, 1: 57344.0, 2: 127.0}
VARIANTS = {0: "ash_ds", 1: "hadamard_ds", 2: "ds_only", 3: "ash_only"}
ROWS = 131                     # x 2 blocks per row: 262 blocks, several tiles and a ragged tail


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def integer_blocks(B, seed):
    """[ROWS * 2, B] float32 values k * 2^e (|k| <= 63, one e per block), exact
    in bf16: zero, single-element and constant blocks first, every seventh
    block at the bottom of the range (bf16 subnormals)."""
    rng = np.random.default_rng(seed)
    n = ROWS * 2
    kmax = rng.choice([1, 3, 7, 15, 31, 63], size=n)
    k = np.stack([rng.integers(-m, m + 1, size=B) for m in kmax]).astype(np.float64)
    e = rng.integers(-30, 31, size=n).astype(np.float64)
    tiny = np.arange(n) % 7 == 5
    e[tiny] = rng.integers(-133, -127, size=int(tiny.sum()))
    k[tiny] = np.clip(k[tiny], -7, 7)
    k[0] = 0.0
    k[1] = 0.0
    k[1, B // 3] = 5.0
    k[2] = 3.0
    X = (k * 2.0 ** e[:, None]).astype(np.float32)
    bits = X.view(np.uint32)
    assert not np.any(bits & 0xFFFF), "not exact in bf16"
    return X


def to_bf16(X):
    bits = (X.view(np.uint32) >> 16).astype(np.uint16)
    return torch.from_numpy(bits.view(np.int16).reshape(ROWS, -1)).view(torch.bfloat16).to(DEV)


def expected(X, B, variant, code, alpha_out):
    f32 = np.float32
    qmax = f32(QMAX[code])
    rB = f32(1.0 / np.sqrt(B))
    if variant == 2:
        g = X
        gmax = np.max(np.abs(g), axis=1)
        s = (gmax / qmax).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            u = np.where(s[:, None] > 0, g / np.where(s > 0, s, f32(1))[:, None], f32(0)).astype(np.float32)
        return oracle.code_encode(code, u).reshape(X.shape), s
    y64 = X.astype(np.float64) @ hadamard(B).T
    y = y64.astype(np.float32)
    assert np.array_equal(y.astype(np.float64), y64), "rotation not exact in binary32"
    ymax = np.max(np.abs(y), axis=1)
    if variant == 3:
        k = (alpha_out.astype(np.float32) * rB).astype(np.float32)
        u = (y * k[:, None]).astype(np.float32)
        return oracle.code_encode(code, u).reshape(X.shape), np.ones(len(y), np.float32)
    tiny = (ymax > 0) & (ymax < f32(2.0 ** -100))
    pre = np.where(tiny, f32(2.0 ** 64), f32(1)).astype(np.float32)
    with np.errstate(divide="ignore"):
        k = np.where(ymax > 0, qmax / (ymax * pre).astype(np.float32), f32(0)).astype(np.float32)
    u = ((y * pre[:, None]).astype(np.float32) * k[:, None]).astype(np.float32)
    alpha = alpha_out.astype(np.float32) if variant == 0 else np.ones(len(y), np.float32)
    s = np.where(ymax > 0, ((alpha * ymax).astype(np.float32) * rB).astype(np.float32) / qmax, f32(0))
    return oracle.code_encode(code, u).reshape(X.shape), s.astype(np.float32)


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("code", [0, 1, 2])
@pytest.mark.parametrize("B", [32, 64, 128, 256, 512])
def test_compress_is_the_stated_arithmetic_on_exact_rotations(taco, B, code, variant):
    X = integer_blocks(B, seed=100 * B + 10 * code + variant)
    got = taco.compress(to_bf16(X), B, variant=VARIANTS[variant], code=code).cpu().numpy()
    cg, ag, sg = records(got, B)
    want, s_want = expected(X, B, variant, code, ag)
    bad = np.argwhere(cg != want)
    assert bad.size == 0, f"{len(bad)} codes differ, first (block, element) {bad[:4].tolist()}"
    bad = np.nonzero(sg != s_want.astype(np.float64))[0]
    assert bad.size == 0, f"{bad.size} scales differ, first blocks {bad[:4].tolist()}"
    if variant in (0, 3):
        G = X.astype(np.float64)
        a_exact = TAU / np.sqrt((G * G).sum(axis=1) / B + EPS)
        assert np.max(np.abs(ag / a_exact - 1.0)) <= 1e-6
    else:
        assert np.all(ag == 1.0)
    assert taco.device_status() == 0
