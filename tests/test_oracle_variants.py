"""Pins for the oracle's ablation variants and code formats.

Variants (paper Sections 5.2.2 and 5.3.1): ASH + DS (the method), standard
Hadamard + DS (no adaptive scale, alpha = 1), DS only (no rotation either) and
ASH only (no post-rotation scale, s = 1, the rotated value cast directly).
Codes (Section 5.3.2 format ablation; Sections 2 and 6 for INT8): E4M3,
E5M2 (largest finite 57344) and INT8 (round(x / Delta), Delta = max / 127).

What pins them, independently of the oracle's own code:
- E5M2 and INT8 conversions against PyTorch's float8_e5m2 cast and NumPy's
  rint on random values, every midpoint and the saturation range;
- exact round trips built from Hadamard rows, whose codes and decoded values
  follow in closed form for every variant and code format;
- the real-arithmetic identities between variants (standard Hadamard + DS
  has the codes of ASH + DS and s / alpha of it, Note on alpha cancelling),
  the per-element error bound of each code format, and the reduce's
  idempotence, scaling and cancellation.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import bf16_to_f64, hadamard, records

VARIANTS = [oracle.ASH_DS, oracle.HADAMARD_DS, oracle.DS_ONLY, oracle.ASH_ONLY]
CODES = [oracle.E4M3, oracle.E5M2, oracle.INT8]
QMAX = {oracle.E4M3: 448.0, oracle.E5M2: 57344.0, oracle.INT8: 127.0}


def f32_to_bf16_bits(x):
    return oracle.bf16_round(np.asarray(x, dtype=np.float32))


def code_values(code, c):
    return oracle.code_value(code, np.asarray(c, dtype=np.uint8).reshape(-1))


# ---------------------------------------------------------------------------
# Code formats
# ---------------------------------------------------------------------------

def torch_e5m2_bytes(u):
    t = torch.from_numpy(np.asarray(u, dtype=np.float32)).to(torch.float8_e5m2)
    return t.view(torch.uint8).numpy()


def test_e5m2_values_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    got = code_values(oracle.E5M2, codes)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert got[0x7B] == 57344.0 and got[0xFB] == -57344.0


def test_e5m2_encode_matches_torch_in_range():
    rng = np.random.default_rng(5)
    mag = np.exp2(rng.uniform(-20, np.log2(57344.0), 200000))
    u = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    u = u[np.abs(u) < 57344.0]
    assert np.array_equal(oracle.code_encode(oracle.E5M2, u), torch_e5m2_bytes(u))


def test_e5m2_encode_midpoints_and_neighbours():
    vals = code_values(oracle.E5M2, np.arange(0, 0x7C, dtype=np.uint8))   # 0 .. 57344
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)   # exact in fp32
    pts = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
    pts = np.concatenate([pts, -pts])
    assert np.array_equal(oracle.code_encode(oracle.E5M2, pts), torch_e5m2_bytes(pts))


def test_e5m2_encode_saturates_and_keeps_sign_of_zero():
    big = np.array([57344.0, 57345.0, 61439.0, 61440.0, 1e10, 3e38], dtype=np.float32)
    assert set(oracle.code_encode(oracle.E5M2, big)) == {0x7B}
    assert set(oracle.code_encode(oracle.E5M2, -big)) == {0xFB}
    z = oracle.code_encode(oracle.E5M2, np.array([0.0, -0.0, -1e-30, 1e-30], dtype=np.float32))
    assert list(z) == [0x00, 0x80, 0x80, 0x00]


def test_int8_encode_matches_numpy_rint():
    rng = np.random.default_rng(6)
    u = rng.uniform(-140, 140, 200000).astype(np.float32)
    halves = (np.arange(-130, 131) + 0.5).astype(np.float32)
    u = np.concatenate([u, halves, np.nextafter(halves, np.float32(0)), np.nextafter(halves, np.float32(300))])
    ref = np.clip(np.rint(u.astype(np.float64)), -127, 127).astype(np.int8)
    assert np.array_equal(oracle.code_encode(oracle.INT8, u).view(np.int8), ref)
    assert np.array_equal(code_values(oracle.INT8, np.arange(256, dtype=np.uint8)),
                          np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64))


# ---------------------------------------------------------------------------
# Exact round trips (closed form)
# ---------------------------------------------------------------------------

# (a, b) with Q_max * b / a on the code grid and c * (a +- b) exact in bf16.
PAIRS = {oracle.E4M3: [(56, 48), (56, 28), (56, 7), (56, 1)],
         oracle.E5M2: [(56, 48), (56, 28), (56, 7), (56, 1)],
         oracle.INT8: [(127, 100), (127, 64), (127, 1)]}


def two_row_block(B, i, j, a, b, c):
    H = hadamard(B)
    return c * (a * H[i] + b * H[j])


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("variant", [oracle.ASH_DS, oracle.HADAMARD_DS])
@pytest.mark.parametrize("B", [64, 128, 256])
def test_rotating_ds_exact_round_trip(B, variant, code):
    """x = c (a h_i + b h_j): H x = B c (a e_i + b e_j), so the codes are
    +-Q_max at i, +-Q_max b / a at j, zero elsewhere, and decompress
    returns x exactly in bf16."""
    rng = np.random.default_rng(B + 10 * variant + 100 * code)
    blocks, expect = [], []
    for a, b in PAIRS[code]:
        i, j = rng.choice(B, 2, replace=False)
        c = 2.0 ** int(rng.integers(-12, 4))
        sb = rng.choice([-1.0, 1.0])
        blocks.append(two_row_block(B, i, j, a, sb * b, c))
        expect.append((i, j, QMAX[code] * sb * b / a))
    x = np.array(blocks)
    bits = f32_to_bf16_bits(x)
    assert np.array_equal(bf16_to_f64(bits), x.reshape(-1))
    packed = oracle.compress(bits, B, variant, code)
    codes, alpha, s = records(packed, B)
    for k, (i, j, vj) in enumerate(expect):
        v = code_values(code, codes[k])
        assert v[i] == QMAX[code] and v[j] == vj
        rest = np.delete(v, [i, j])
        assert np.all(rest == 0.0)
        if variant == oracle.HADAMARD_DS:
            assert alpha[k] == 1.0
    y = oracle.decompress(packed, bits.size, B, variant, code)
    assert np.array_equal(y, bits)


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("B", [64, 128, 256])
def test_ds_only_exact_round_trip(B, code):
    """No rotation: a block of c * {+-a, +-b, 0} has codes +-Q_max, +-Q_max b / a
    and 0, alpha = 1, s = c a / Q_max, and decodes to itself."""
    rng = np.random.default_rng(B + code)
    blocks, pat = [], []
    for a, b in PAIRS[code]:
        c = 2.0 ** int(rng.integers(-12, 4))
        v = rng.choice([0.0, a, -a, b, -b], B)
        v[rng.integers(B)] = a
        blocks.append(c * v)
        pat.append(v * QMAX[code] / a)
    bits = f32_to_bf16_bits(np.array(blocks))
    packed = oracle.compress(bits, B, oracle.DS_ONLY, code)
    codes, alpha, s = records(packed, B)
    assert np.all(alpha == 1.0)
    for k in range(len(blocks)):
        assert np.array_equal(code_values(code, codes[k]), pat[k])
    assert np.array_equal(oracle.decompress(packed, bits.size, B, oracle.DS_ONLY, code), bits)


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("B", [64, 256])
def test_ash_only_exact_round_trip(B, code):
    """x = c h_i: alpha = 1 / c, Z = sqrt(B) e_i exactly (B = 64, 256), so the
    only nonzero code is sqrt(B), s = 1, and decompress returns x."""
    rng = np.random.default_rng(B * 7 + code)
    H = hadamard(B)
    idx = rng.choice(B, 4, replace=False)
    cs = [2.0 ** int(e) for e in rng.integers(-10, 6, 4)]
    x = np.array([c * H[i] for c, i in zip(cs, idx)])
    bits = f32_to_bf16_bits(x)
    packed = oracle.compress(bits, B, oracle.ASH_ONLY, code)
    codes, alpha, s = records(packed, B)
    assert np.all(s == 1.0)
    assert np.array_equal(alpha, 1.0 / np.array(cs))
    for k, i in enumerate(idx):
        v = code_values(code, codes[k])
        assert v[i] == np.sqrt(B) and np.all(np.delete(v, i) == 0.0)
    assert np.array_equal(oracle.decompress(packed, bits.size, B, oracle.ASH_ONLY, code), bits)


# ---------------------------------------------------------------------------
# Identities and bounds on random data
# ---------------------------------------------------------------------------

def sample(B, rows=64, hidden=1024, seed=3):
    return workloads.generate("laplace_outliers", rows, hidden, seed)


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("B", [64, 128, 256])
def test_standard_hadamard_matches_ash_up_to_rounding(B, code):
    """alpha cancels from the codes (Note on Eqs. 7-10): standard Hadamard +
    DS has the codes of ASH + DS up to FP32 rounding and s_H = s_ASH / alpha_ASH."""
    bits = sample(B)
    ca, aa, sa = records(oracle.compress(bits, B, oracle.ASH_DS, code), B)
    ch, ah, sh = records(oracle.compress(bits, B, oracle.HADAMARD_DS, code), B)
    assert np.all(ah == 1.0)
    va, vh = code_values(code, ca), code_values(code, ch)
    diff = va != vh
    assert diff.mean() <= 1e-4
    # a flip moves to the adjacent grid point: at most one spacing apart
    if diff.any():
        grid = np.unique(np.abs(code_values(code, np.arange(256, dtype=np.uint8))))
        grid = grid[np.isfinite(grid)]
        ia = np.searchsorted(grid, np.abs(va[diff]))
        ih = np.searchsorted(grid, np.abs(vh[diff]))
        assert np.all(np.abs(ia - ih) <= 1)
    nz = sa > 0
    assert np.allclose(sh[nz], sa[nz] / aa[nz], rtol=1e-6, atol=0)


def half_spacing(code, u):
    """Half the grid spacing of the code format at |u| (E4M3 / E5M2: Eq. 3;
    INT8: 1/2)."""
    a = np.abs(u)
    if code == oracle.INT8:
        return np.full_like(a, 0.5)
    m, emin = (3, -6) if code == oracle.E4M3 else (2, -14)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return np.exp2(e - m) / 2


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("variant", VARIANTS)
def test_per_element_error_bound(variant, code):
    """|u - q| <= half a grid spacing of the code format for every element,
    where u is the scaled value the variant quantises (recomputed in float64
    from the stored alpha and s), up to FP32 rounding."""
    B = 128
    bits = sample(B, seed=9)
    G = bf16_to_f64(bits).reshape(-1, B)
    codes, alpha, s = records(oracle.compress(bits, B, variant, code), B)
    q = code_values(code, codes).reshape(-1, B)
    if variant == oracle.DS_ONLY:
        Z = G
    else:
        Z = (alpha[:, None] * G) @ hadamard(B).T / np.sqrt(B)
    u = Z / np.where(s > 0, s, 1.0)[:, None]
    bound = half_spacing(code, u) + 1e-5 * np.abs(u) + 1e-6
    assert np.all(np.abs(u - q) <= bound)
    if variant != oracle.ASH_ONLY:
        nz = s > 0
        assert np.all(np.abs(q[nz]).max(axis=1) == QMAX[code])   # the block maximum lands on Q_max


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("variant", [oracle.ASH_DS, oracle.HADAMARD_DS, oracle.DS_ONLY])
def test_reduce_identities(variant, code):
    """P = 1 keeps the codes; P identical shards keep the codes and scale
    s / alpha by P; a shard and its negation give all-zero blocks."""
    B = 128
    bits = sample(B, rows=16, seed=4)
    n = bits.size
    sh = oracle.compress(bits, B, variant, code)
    c0, a0, s0 = records(sh, B)
    c1, a1, s1 = records(oracle.reduce_shards([sh], n, B, variant, code), B)
    v0, v1 = code_values(code, c0), code_values(code, c1)
    assert (v0 != v1).mean() <= 1e-4
    assert np.allclose(s1 / a1, s0 / a0, rtol=2e-6)
    c4, a4, s4 = records(oracle.reduce_shards([sh] * 4, n, B, variant, code), B)
    assert (code_values(code, c4) != v0).mean() <= 1e-4
    assert np.allclose(s4 / a4, 4 * s0 / a0, rtol=2e-6)
    neg = oracle.compress(bits ^ np.uint16(0x8000), B, variant, code)
    cz, az, sz = records(oracle.reduce_shards([sh, neg], n, B, variant, code), B)
    assert np.all(sz == 0.0) and np.all(cz == 0)


@pytest.mark.parametrize("code", CODES)
def test_ash_only_reduce_of_negation_is_zero(code):
    B = 128
    bits = sample(B, rows=8, seed=2)
    sh = oracle.compress(bits, B, oracle.ASH_ONLY, code)
    neg = oracle.compress(bits ^ np.uint16(0x8000), B, oracle.ASH_ONLY, code)
    cz, az, sz = records(oracle.reduce_shards([sh, neg], bits.size, B, oracle.ASH_ONLY, code), B)
    assert np.all(sz == 1.0)
    assert np.all(code_values(code, cz) == 0.0)


def test_bad_scheme_rejected():
    bits = sample(128, rows=1, hidden=128)
    with pytest.raises(ValueError):
        oracle.compress(bits, 128, 4, 0)
    with pytest.raises(ValueError):
        oracle.compress(bits, 128, 0, 3)


def test_encode_bits_equals_the_array_encoder():
    """code_encode_bits (every input of a bit-pattern range, modulo 2^32) is
    the same encoder as code_encode on the corresponding float32 array."""
    for code in (0, 1, 2):
        for first in (0, 0x3BFFF000, 0x7F7FF000, 0xBF000000, 0xFFFFF000):
            bits = (np.arange(1 << 13, dtype=np.uint64) + first) & 0xFFFFFFFF
            u = bits.astype(np.uint32).view(np.float32)
            ref = oracle.code_encode(code, u)
            assert np.array_equal(oracle.code_encode_bits(code, first, bits.size), ref), (code, hex(first))

