"""The shard reduce sums the decoded shards as an FP32 sum should: every
product q_p * f_p rounded on its own, then added in shard order (TACO paper,
Section 4.4.2: each owner decodes the P shards it receives, sums them in FP32
and compresses the sum once; Eq. 11 gives the decode q * s / alpha).

Crafted records make that sum exactly computable on the host: every shard has
alpha = 1, so its factor s / alpha is s itself in any division, and the codes
are random finite codes of the format.  The host then forms W in float32
(numpy: correctly rounded products and adds, in shard order) and the outputs
follow from the rotated-domain reading of the reduce (compressing
(1/sqrt B) H W gives codes of Q_max W / max|W| and s' = alpha' max|W| / Q_max):

  codes = Cvt(fl(W * fl(Q_max / max|W|)))     exactly
  s'    = fl(fl(alpha' * max|W|) / Q_max)     exactly, alpha' read back
  alpha' = tau / sqrt(|W|^2 / B + eps)        within 1e-6 (FP32 energy order)

and for the ablations the same W with their own last step (the test's
docstring below).

A fused multiply-add in place of the separately rounded product changes W by
an ulp here and there, and so max|W| and s' in a fifth of the blocks: this
test sees it where the oracle-tolerance comparisons cannot.  Every fifth
block has factors near 2^-105, so that its sum lies below 2^-80 and takes the
kernel's rescaled pass (factors 2^64 s, scales taken back by 2^-64), which
scales W by a power of two and must leave the same codes and scales.  Blocks
0-9 hold a shard and its negation (the rest zero codes): W = 0 exactly and the
record is all zero.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import decode_table, records

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TAU = 1.0
EPS = float(np.float32(1e-30))
QMAX = {0: 448.0, 1: 57344.0, 2: 127.0}
NBLK = 1037          # several tiles of every kernel, an odd ragged last tile


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def finite_codes(rng, shape, code):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    if code == 0:
        c[(c & 0x7F) == 0x7F] = 0             # E4M3 NaN
    elif code == 1:
        c[(c & 0x7F) > 0x7B] = 0              # E5M2 inf / NaN
    else:
        c[c == 0x80] = 0                      # INT8 -128 has no negation
    return c


def negate(c, code):
    if code == 2:
        return (-(c.view(np.int8).astype(np.int16))).astype(np.int8).view(np.uint8)
    return c ^ np.uint8(0x80)


def crafted_shards(P, B, code, seed):
    rng = np.random.default_rng(seed)
    codes = finite_codes(rng, (P, NBLK, B), code)
    s = (rng.uniform(1, 2, size=(P, NBLK)) * 2.0 ** rng.integers(-12, -4, size=(P, NBLK))).astype(np.float32)
    tiny = np.arange(NBLK) % 5 == 3
    s[:, tiny] = (rng.uniform(1, 2, size=(P, int(tiny.sum()))) * 2.0 ** rng.integers(-110, -100, size=(P, int(tiny.sum())))).astype(np.float32)
    if P >= 2:                                 # blocks 0-9: a shard and its negation
        codes[1, :10] = negate(codes[0, :10], code)
        s[1, :10] = s[0, :10]
        codes[2:, :10] = 0
    meta = np.empty((P, NBLK, 2), np.float32)
    meta[..., 0] = 1.0
    meta[..., 1] = s
    recs = np.concatenate([codes, meta.view(np.uint8).reshape(P, NBLK, 8)], axis=2)
    return [np.ascontiguousarray(recs[p].reshape(-1)) for p in range(P)], tiny


def float32_sum(shards, B, code):
    """W = sum over shards, in order, of fl32(q * s): float32 arithmetic."""
    table = decode_table(code).astype(np.float32)      # every code value is exact in float32
    W = np.zeros((NBLK, B), np.float32)
    for sh in shards:
        c, a, s = records(sh, B)
        assert np.all(a == 1.0)
        W = W + table[c] * s.astype(np.float32)[:, None]
        assert W.dtype == np.float32
    return W


VARIANTS = {0: "ash_ds", 1: "hadamard_ds", 2: "ds_only", 3: "ash_only"}


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("code", [0, 1, 2])
@pytest.mark.parametrize("P", [2, 3, 4, 8, 16])
@pytest.mark.parametrize("B", [32, 64, 128, 256, 512])
def test_reduce_is_the_float32_sum_of_rounded_products(taco, B, P, code, variant):
    """The method (variant 0) and the ablations, whose outputs differ only in
    the last step: standard Hadamard + DS takes alpha' = 1; DS only codes
    W / s' correctly rounded with s' = fl(max|W| / Q_max) and alpha' = 1; ASH
    only stores s' = 1 and codes Cvt(fl(W * alpha'))."""
    shards, tiny = crafted_shards(P, B, code, seed=1000 * B + 10 * P + code)
    got = taco.reduce_shards([torch.from_numpy(s).to(DEV) for s in shards], NBLK, B, B,
                             variant=VARIANTS[variant], code=code).cpu().numpy()
    cg, ag, sg = records(got, B)
    W = float32_sum(shards, B, code)
    wmax = np.max(np.abs(W), axis=1)
    zero = wmax == 0
    assert np.all(zero[:10]) and not np.any(zero[10:])
    # W = 0: all codes zero; s' = 0 (1 for ASH only, which stores no scale).
    assert np.all(cg[zero] == 0) and np.all(sg[zero] == (1.0 if variant == 3 else 0.0))
    nz = ~zero
    f32 = np.float32
    qmax = f32(QMAX[code])
    ag32 = ag[nz].astype(np.float32)
    if variant == 3:
        u = (W[nz] * ag32[:, None]).astype(np.float32)
        s_want = np.ones(int(nz.sum()), np.float32)
    elif variant == 2:
        s_want = (wmax[nz] / qmax).astype(np.float32)
        u = (W[nz] / s_want[:, None]).astype(np.float32)
    else:
        alpha = ag32 if variant == 0 else np.ones_like(ag32)
        kq = (qmax / wmax[nz]).astype(np.float32)
        u = (W[nz] * kq[:, None]).astype(np.float32)
        s_want = ((alpha * wmax[nz]).astype(np.float32) / qmax).astype(np.float32)
    want = oracle.code_encode(code, u).reshape(u.shape)
    bad = np.argwhere(cg[nz] != want)
    assert bad.size == 0, f"{len(bad)} codes differ, first (block, element) {bad[:4].tolist()}"
    bad = np.nonzero(sg[nz] != s_want)[0]
    assert bad.size == 0, f"{bad.size} of {nz.sum()} scales differ (tiny blocks among them: {int(tiny[nz][bad].sum())})"
    if variant in (0, 3):
        Wd = W.astype(np.float64)
        a_exact = TAU / np.sqrt((Wd * Wd).sum(axis=1) / B + EPS)
        assert np.max(np.abs(ag[nz] / a_exact[nz] - 1.0)) <= 1e-6
    else:
        assert np.all(ag == 1.0)
    assert taco.device_status() == 0
