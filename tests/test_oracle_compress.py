"""Pins of the oracle's compress / decompress (Algorithm 1, Eqs. 5-13) against
what the paper and the mathematics fix, independently of the oracle's own code:

- Adaptive Scale hits the target energy: RMS(alpha_k G_k) = tau (Eqs. 6-7).
- The post-rotation scale equals its real-arithmetic value
  s = alpha max|H G| / (sqrt(B) Q_max) (Eqs. 8-9), alpha cancels from the codes.
- Every code lies within half an E4M3 step (Eq. 3) of the exact float64 value
  u = Q_max H G / max|H G| computed with SciPy's Hadamard matrix.
- Dual-Scale range: no code exceeds 448 and every nonzero block reaches 448.
- Special cases: one nonzero element (every code +-448), a constant block
  (one code +-448, the rest zero), an all-zero block (s = 0, codes 0, exact 0
  back), exact round trip of inputs that land on the E4M3 grid.
- Round-trip error: ||G - G'|| = (s/alpha) ||u - q|| (orthogonality, Eq. 12).
- Tiny blocks (B = 2, 4, 8): codes equal a float64 dense implementation with
  a brute-force nearest-value search.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import (QMAX, TAU, bf16_to_f64, e4m3_decode_table, e4m3_half_ulp,
                     exact_compress_quantities, hadamard, records, rel_l2)


def f32_to_bf16_bits(x):
    return oracle.bf16_round(np.asarray(x, dtype=np.float32))


def sample_inputs():
    """A few hundred rows of each workload distribution, plus zero blocks."""
    out = {}
    for dist, hidden in [("laplace_outliers", 1024), ("student_t_channels", 4096),
                         ("gaussian_sparse", 5120)]:
        out[dist] = workloads.generate(dist, 8192, hidden, seed=0, row_count=24).reshape(-1)
    return out


@pytest.fixture(scope="module")
def inputs():
    return sample_inputs()


@pytest.mark.parametrize("B", [64, 128, 256])
@pytest.mark.parametrize("dist", ["laplace_outliers", "student_t_channels", "gaussian_sparse"])
def test_scales_and_codes_against_real_arithmetic(inputs, dist, B):
    x = inputs[dist]
    G = bf16_to_f64(x).reshape(-1, B)
    codes, alpha, s = records(oracle.compress(x, B), B)
    a_ex, s_ex, u_ex, m = exact_compress_quantities(G, B)

    # Eq. 7: alpha within 1e-6 of tau / sqrt(m + eps), and the target energy.
    assert np.all(np.abs(alpha / a_ex - 1) < 1e-6)
    big = m >= 1e-24
    rms_scaled = alpha[big] * np.sqrt(m[big])
    assert np.all(np.abs(rms_scaled / TAU - 1) < 1e-6)

    # Eq. 9: s_k in real arithmetic.
    nz = s_ex > 0
    assert np.all(np.abs(s[nz] / s_ex[nz] - 1) < 2e-6)
    assert np.all(s[~nz] == 0)

    # Eq. 10 with Eq. 3: each code within half a step of the exact u (plus a
    # float32 slack far below the step at any magnitude used here).
    q = e4m3_decode_table()[codes]
    assert not np.any(np.isnan(q))
    slack = 448.0 * 4e-6
    assert np.all(np.abs(q - u_ex) <= e4m3_half_ulp(u_ex) + slack)

    # Dual-Scale range: |q| <= 448 and each nonzero block reaches 448.
    assert np.all(np.abs(q) <= QMAX)
    assert np.all(np.abs(q[nz]).max(axis=1) == QMAX)


@pytest.mark.parametrize("B", [64, 128, 256])
def test_round_trip_error_identity(inputs, B):
    """G - G' = r H (u - q) s / alpha, so ||G - G'|| = (s/alpha) ||u - q||."""
    x = inputs["student_t_channels"]
    G = bf16_to_f64(x).reshape(-1, B)
    packed = oracle.compress(x, B)
    codes, alpha, s = records(packed, B)
    _, _, u_ex, _ = exact_compress_quantities(G, B)
    q = e4m3_decode_table()[codes]
    Gp = oracle.decompress_f32(packed, x.size, B).astype(np.float64).reshape(-1, B)
    lhs = np.linalg.norm(G - Gp, axis=1)
    rhs = s / alpha * np.linalg.norm(u_ex - q, axis=1)
    gnorm = np.linalg.norm(G, axis=1)
    assert np.all(np.abs(lhs - rhs) <= 1e-3 * rhs + 2e-6 * gnorm)


@pytest.mark.parametrize("B", [64, 128, 256])
def test_decompress_matches_float64_dense_inverse(inputs, B):
    """Eqs. 11-13 in float64 with SciPy's H: G' = (1/sqrt B) H (q s) / alpha."""
    x = inputs["laplace_outliers"]
    packed = oracle.compress(x, B)
    codes, alpha, s = records(packed, B)
    q = e4m3_decode_table()[codes]
    exact = (q * s[:, None]) @ hadamard(B).T / np.sqrt(B) / alpha[:, None]
    got = oracle.decompress_f32(packed, x.size, B).astype(np.float64).reshape(-1, B)
    scale = np.abs(exact).max(axis=1, keepdims=True)
    assert np.all(np.abs(got - exact) <= 1e-6 * scale)
    # bf16 output is the nearest-even rounding of a value within the float32
    # bound above: at most half a bf16 step plus that bound from the exact G'.
    bf = bf16_to_f64(oracle.decompress(packed, x.size, B)).reshape(-1, B)
    half_step = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 1e-37))) - 8)
    assert np.all(np.abs(bf - exact) <= half_step + 1e-6 * scale)


@pytest.mark.parametrize("B", [2, 4, 8])
def test_tiny_blocks_match_dense_brute_force(B):
    table = e4m3_decode_table()
    finite = np.array([c for c in range(256) if not np.isnan(table[c])])
    rng = np.random.default_rng(100 + B)
    G32 = (rng.standard_normal((400, B)) * np.exp2(rng.uniform(-20, 4, (400, 1)))).astype(np.float32)
    x = f32_to_bf16_bits(G32)
    G = bf16_to_f64(x).reshape(-1, B)
    codes, alpha, s = records(oracle.compress(x, B), B)
    a_ex, s_ex, u_ex, _ = exact_compress_quantities(G, B)
    assert np.all(np.abs(alpha / a_ex - 1) < 1e-6)
    assert np.all(np.abs(s / s_ex - 1) < 1e-6)
    # Brute force: nearest finite value, ties to the even code.
    vals = table[finite]
    d = np.abs(u_ex.reshape(-1, 1) - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = np.where(d == best, finite[None, :], 10 ** 6)
    even = np.where((cand % 2 == 0) & (cand < 10 ** 6), cand, 10 ** 6).min(axis=1)
    brute = np.where(even < 10 ** 6, even, cand.min(axis=1)).reshape(-1, B)
    # Zeros: the sign of zero follows u; compare values, not the zero's sign.
    got_v, brute_v = table[codes], table[brute]
    # Exclude points within float32 noise of a rounding midpoint.
    sorted_vals = np.unique(np.abs(vals))
    mids = (sorted_vals[:-1] + sorted_vals[1:]) / 2
    near = np.min(np.abs(np.abs(u_ex).reshape(-1, 1) - mids[None, :]), axis=1).reshape(-1, B)
    clear = near > 448 * 1e-6
    assert np.array_equal(got_v[clear], brute_v[clear])


@pytest.mark.parametrize("B", [2, 64, 128, 256, 512])
def test_single_nonzero_element_gives_all_448(B):
    rng = np.random.default_rng(B)
    G = np.zeros((B, B), dtype=np.float32)
    vals = rng.choice([-1.0, 1.0], B) * np.exp2(rng.integers(-30, 10, B))
    G[np.arange(B), np.arange(B)] = vals          # block k has element k set
    codes, alpha, s = records(oracle.compress(f32_to_bf16_bits(G), B), B)
    H = hadamard(B)
    sign = np.sign(vals)[:, None] * H              # sign of column k of H times the value's sign
    expect = np.where(sign > 0, 0x7E, 0xFE)
    assert np.array_equal(codes, expect)


@pytest.mark.parametrize("B", [4, 64, 128, 256])
def test_constant_block(B):
    c = np.array([0.75, -3.0, 1e-20, 2.0 ** 50], dtype=np.float32)
    G = np.repeat(c[:, None], B, axis=1)
    codes, alpha, s = records(oracle.compress(f32_to_bf16_bits(G), B), B)
    assert np.array_equal(codes[:, 0], np.where(c > 0, 0x7E, 0xFE))
    assert np.all((codes[:, 1:] & 0x7F) == 0)
    # The round trip of a constant block is exact in bf16.
    back = oracle.decompress(oracle.compress(f32_to_bf16_bits(G), B), G.size, B)
    assert np.array_equal(back, f32_to_bf16_bits(G).reshape(-1))


@pytest.mark.parametrize("B", [2, 64, 128, 256])
def test_all_zero_block(B):
    x = np.zeros(3 * B, dtype=np.uint16)
    x[B:2 * B] = f32_to_bf16_bits(np.linspace(-1, 1, B, dtype=np.float32))
    packed = oracle.compress(x, B)
    codes, alpha, s = records(packed, B)
    for k in (0, 2):
        assert s[k] == 0.0
        assert np.all(codes[k] == 0)
        assert alpha[k] == np.float32(1.0) / np.sqrt(np.float32(1e-30))
    back = oracle.decompress(packed, x.size, B)
    assert np.all(back[:B] == 0) and np.all(back[2 * B:] == 0)   # +0.0 exactly


@pytest.mark.parametrize("B", [2, 4, 8, 16, 64, 128, 256, 512])
@pytest.mark.parametrize("b", [48, 28, 7, 1])
def test_exact_round_trip_on_grid_inputs(B, b):
    """x = c (a h_i + b h_j) with Hadamard rows h_i, h_j: H x = c B (a e_i + b e_j),
    so the codes are +-448 at i, +-448 b/a at j (an E4M3 value for a = 56) and
    zero elsewhere, and the bf16 round trip is exact."""
    a = 56
    H = hadamard(B)
    rng = np.random.default_rng(B * 100 + b)
    rows = []
    expect = []
    for _ in range(32):
        i, j = rng.choice(B, 2, replace=False)
        c = 2.0 ** int(rng.integers(-20, 8)) * rng.choice([-1, 1])
        rows.append(c * (a * H[i] + b * H[j]))
        e = np.zeros(B)
        e[i] = np.sign(c) * 448.0
        e[j] = np.sign(c) * 448.0 * b / a
        expect.append(e)
    X = np.array(rows, dtype=np.float32)
    x = f32_to_bf16_bits(X)
    assert np.array_equal(bf16_to_f64(x), X.astype(np.float64).reshape(-1))   # bf16-exact
    packed = oracle.compress(x, B)
    codes, _, _ = records(packed, B)
    assert np.array_equal(e4m3_decode_table()[codes], np.array(expect))
    assert np.array_equal(oracle.decompress(packed, x.size, B), x)


def test_round_trip_fidelity_of_workloads(inputs):
    """The round trip on the workload distributions loses far less than the
    bf16 -> E4M3 cast without ASH and DS (the paper's zero-collapse, Section 4.2.1)."""
    for dist, x in inputs.items():
        G = bf16_to_f64(x)
        back = bf16_to_f64(oracle.decompress(oracle.compress(x, 128), x.size, 128))
        err = rel_l2(back, G)
        direct = e4m3_decode_table()[oracle.e4m3_encode(G.astype(np.float32))]
        assert err < 0.05, (dist, err)
        assert err < 0.5 * rel_l2(direct, G), (dist, err)


def test_argument_errors():
    x = np.zeros(96, np.uint16)
    with pytest.raises(ValueError):
        oracle.compress(x, 64)        # 96 is not a multiple of 64
    with pytest.raises(ValueError):
        oracle.compress(x, 48)        # not a power of two
    with pytest.raises(ValueError):
        oracle.reduce_shards([], 64, 64)
