"""The decompress kernels' arithmetic on records whose inverse rotation is exact.

Records with integer-valued codes (E4M3 and E5M2 codes of integers, every
INT8 code) have an exact y = H q in binary32 whatever the summation order
(|y| < 2^24), so the host can form what each kernel computes from y (TACO
paper, Eqs. 11-13, with the three scalings folded into one factor per block,
the form the kernels use):

  f = fl(fl(s * r_B) / alpha)                  (r_B = 1 for DS only, y = q)
  out = bf16(fl(y * f))
  a factor below 2^-100 (or flushed to zero) with s > 0:
      f' = fl(fl(fl(s 2^64) * r_B) / alpha),  out = bf16(fl(fl(y * f') * 2^-64))

The bf16 outputs must match bit for bit (a zero of either sign counts as
zero).  Blocks cover zero scales, ordinary factors, subnormal factors near
2^-138 and 2^-146 (kept to 11 or 3 bits in binary32, so the 2^64 rescaling
decides their outputs) and factors that underflow to zero.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import decode_table, hadamard

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
VARIANTS = {0: "ash_ds", 2: "ds_only", 3: "ash_only"}
ROWS = 131                     # x 2 blocks per row: 262 blocks, several tiles and a ragged tail


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def integer_codes(code):
    vals = decode_table(code)
    lim = 448.0 if code == 0 else 16384.0 if code == 1 else 128.0
    ok = np.isfinite(vals) & (vals == np.round(vals)) & (np.abs(vals) <= lim)
    return np.nonzero(ok)[0].astype(np.uint8)


def crafted_records(B, code, seed):
    rng = np.random.default_rng(seed)
    n = ROWS * 2
    codes = rng.choice(integer_codes(code), size=(n, B)).astype(np.uint8)
    alpha = (rng.uniform(1, 2, n) * 2.0 ** rng.integers(-20, 21, n)).astype(np.float32)
    s = (rng.uniform(1, 2, n) * 2.0 ** rng.integers(-30, 10, n)).astype(np.float32)
    kind = np.arange(n) % 9
    s[kind == 0] = 0.0                                              # zero scale: all-zero block
    for kd, ea in ((4, 35), (5, 43)):                               # subnormal factors near 2^-138, 2^-146
        s[kind == kd] = (rng.uniform(1, 2, int((kind == kd).sum())) * 2.0 ** -100).astype(np.float32)
        alpha[kind == kd] = np.float32(2.0 ** ea)
    s[kind == 7] = np.float32(2.0 ** -120)
    alpha[kind == 7] = np.float32(2.0 ** 40)                        # factor underflows to 0: rescaled
    meta = np.stack([alpha, s], axis=1).view(np.uint8).reshape(n, 8)
    return np.ascontiguousarray(np.concatenate([codes, meta], axis=1).reshape(-1)), codes, alpha, s


def expected_bits(codes, alpha, s, B, code, rotate):
    f32 = np.float32
    q = decode_table(code)[codes]
    y64 = q @ hadamard(B).T if rotate else q
    y = y64.astype(np.float32)
    assert np.array_equal(y.astype(np.float64), y64), "inverse rotation not exact in binary32"
    rr = f32(1.0 / np.sqrt(B)) if rotate else f32(1.0)
    with np.errstate(under="ignore"):
        f = ((s * rr).astype(np.float32) / alpha).astype(np.float32)
        tiny = (s > 0) & (f < f32(2.0 ** -100))
        ft = (((s * f32(2.0 ** 64)).astype(np.float32) * rr).astype(np.float32) / alpha).astype(np.float32)
        out = (y * f[:, None]).astype(np.float32)
        out_t = ((y * ft[:, None]).astype(np.float32) * f32(2.0 ** -64)).astype(np.float32)
    out = np.where(tiny[:, None], out_t, out)
    assert tiny.sum() >= 40 and (f[tiny] == 0).sum() >= 20
    return oracle.bf16_round(out.reshape(-1)).reshape(out.shape)


@pytest.mark.parametrize("variant", [0, 2, 3])
@pytest.mark.parametrize("code", [0, 1, 2])
@pytest.mark.parametrize("B", [32, 64, 128, 256, 512])
def test_decompress_is_the_stated_arithmetic_on_exact_rotations(taco, B, code, variant):
    packed, codes, alpha, s = crafted_records(B, code, seed=100 * B + 10 * code + variant)
    y = taco.decompress(torch.from_numpy(packed).to(DEV), ROWS, 2 * B, B, variant=VARIANTS[variant], code=code)
    got = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1, B)
    want = expected_bits(codes, alpha, s, B, code, rotate=variant != 2)
    zero = ((got & 0x7FFF) == 0) & ((want & 0x7FFF) == 0)
    bad = np.argwhere((got != want) & ~zero)
    assert bad.size == 0, f"{len(bad)} outputs differ, first (block, element) {bad[:4].tolist()}"
    assert taco.device_status() == 0
