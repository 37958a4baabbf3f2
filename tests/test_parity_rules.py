"""CPU checks of the parity rules in tests/parity.py: each planted deviation
from the oracle's records is caught, and the FP32 rounding-order effects the
rules recognise stay bounded.  The correctly rounded exact values are pinned
against the oracle's encoder on float32-exact inputs."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import bf16_to_f64, decode_table, hadamard
from parity import compare_records, exact_values, noise_zone, near_midpoint, NOISE_REL

B = 128


def exact_u(bits, code=0):
    G = bf16_to_f64(bits).reshape(-1, B)
    y = G @ hadamard(B).T
    qmax = {0: 448.0, 1: 57344.0, 2: 127.0}[code]
    m = np.abs(y).max(axis=1, keepdims=True)
    return np.where(m > 0, qmax * y / np.where(m > 0, m, 1.0), 0.0)


@pytest.fixture(scope="module")
def case():
    bits = workloads.generate("laplace_outliers", 160, 1024, 3).reshape(-1)   # 1280 blocks, 163840 codes
    return bits, oracle.compress(bits, B)


def codes_of(packed):
    return packed.reshape(-1, B + 8)[:, :B]


def test_identical_records_pass(case):
    bits, ref = case
    st = compare_records(ref.copy(), ref, B, u_exact=exact_u(bits))
    assert st["code_mismatches"] == 0 and st["code_max_step"] == 0


def test_one_step_flips_within_budget_pass_and_beyond_fail(case):
    bits, ref = case
    n = codes_of(ref).size
    u = exact_u(bits)
    ties = near_midpoint(u).reshape(-1)
    cand = np.flatnonzero(((codes_of(ref).reshape(-1) & 0x7F) > 8) & ~ties)
    cand = cand[(codes_of(ref).reshape(-1)[cand] & 0x7F) < 0x7E]
    got = ref.copy()
    c = codes_of(got).reshape(-1)
    k = int(1e-4 * n)                                   # exactly the budget
    c[cand[:k]] += 1                                    # one step up in magnitude
    codes_of(got)[:] = c.reshape(-1, B)
    compare_records(got, ref, B)
    c[cand[k:k + 3]] += 1                               # three more: over the budget
    codes_of(got)[:] = c.reshape(-1, B)
    with pytest.raises(AssertionError):
        compare_records(got, ref, B)


def test_two_step_difference_fails_even_at_a_tie(case):
    bits, ref = case
    got = ref.copy()
    u = exact_u(bits)
    c = codes_of(got).reshape(-1)
    i = int(np.flatnonzero((c & 0x7F) == 0x40)[0])
    c[i] += 2
    codes_of(got)[:] = c.reshape(-1, B)
    with pytest.raises(AssertionError):
        compare_records(got, ref, B, u_exact=u)


def test_scale_error_fails(case):
    bits, ref = case
    got = ref.copy()
    rec = got.reshape(-1, B + 8)
    s = rec[7, B + 4:B + 8].copy().view("<f4")
    s *= np.float32(1 + 4e-6)
    rec[7, B + 4:B + 8] = s.view(np.uint8)
    with pytest.raises(AssertionError):
        compare_records(got, ref, B)


def test_tie_flips_capped_by_the_references_own_flips():
    """Blocks built so that their exact u has one rounding tie each: H x = y
    with y = 448 e_r + 432 e_(r+1), and 432 is the midpoint of the E4M3
    values 416 and 448.  Flipping tie codes passes up to the budget (1e-4 of
    the codes plus twice the ties the oracle rounded away from the correctly
    rounded value) and fails one past it."""
    H = hadamard(B)
    rows = []
    for r in range(64):
        y = np.zeros(B)
        y[r % B] = 448.0
        y[(r + 1) % B] = 432.0            # exact midpoint between the E4M3 values 416 and 448
        rows.append(y @ H / B)            # x = H y / B has H x = y
    X = np.array(rows)
    bits = oracle.bf16_round(X.astype(np.float32))
    assert np.array_equal(bf16_to_f64(bits).reshape(X.shape), X)
    ref = oracle.compress(bits, B)
    u = exact_u(bits)
    ties = near_midpoint(u)
    assert ties.sum() == 64
    ev = exact_values(u)
    table = decode_table(0)
    ref_flips = int((ties & (table[codes_of(ref)] != ev)).sum())
    # Flip the oracle's tie codes in the other direction, one by one.
    got = ref.copy()
    c = codes_of(got)
    idx = np.argwhere(ties)
    budget = int(1e-4 * c.size) + 2 * ref_flips
    for j, (bi, ei) in enumerate(idx[:min(budget, len(idx))]):
        c[bi, ei] = c[bi, ei] + 1 if table[c[bi, ei]] < 432 else c[bi, ei] - 1
    compare_records(got, ref, B, u_exact=u)
    assert budget < len(idx), (budget, ref_flips)
    bi, ei = idx[budget]
    c[bi, ei] = c[bi, ei] + 1 if table[c[bi, ei]] < 432 else c[bi, ei] - 1
    with pytest.raises(AssertionError):
        compare_records(got, ref, B, u_exact=u)


@pytest.mark.parametrize("code", [0, 1, 2])
def test_exact_values_match_the_oracle_encoder_on_float32_inputs(code):
    rng = np.random.default_rng(code)
    qmax = {0: 448.0, 1: 57344.0, 2: 127.0}[code]
    u = (rng.standard_normal(20000) * qmax / 4).astype(np.float32)
    u = np.concatenate([u, np.float32([0.0, -0.0, qmax, -qmax, 2 * qmax, 1e-30])])
    got = exact_values(u.astype(np.float64), code)
    want = decode_table(code)[oracle.code_encode(code, u)]
    assert np.array_equal(got, want)


def test_noise_zone_is_relative_to_the_block_maximum():
    u = np.zeros((2, B))
    u[0, 0] = 448.0
    u[0, 1] = 448.0 * NOISE_REL * 0.99
    u[0, 2] = 448.0 * NOISE_REL * 1.01
    u[1, 0] = 2.0
    u[1, 1] = 2.0 * NOISE_REL * 0.5
    z = noise_zone(u, B)
    assert z[0, 1] and not z[0, 2] and z[1, 1] and not z[1, 0] and z[0, 5]


def test_noise_zone_differences_are_bounded_by_value():
    """E5M2 records of constant blocks: H 1 = B e_0, so every element but the
    first is exactly zero in real arithmetic (the noise zone).  A small code
    there (FP32 noise resolved by E5M2's fine grid) passes; a value above
    2 * NOISE_REL of the block maximum fails."""
    code = 1
    X = np.full((4, B), 0.375, dtype=np.float32)
    bits = oracle.bf16_round(X)
    ref = oracle.compress(bits, B, 0, code)
    u = exact_u(bits, code)
    table = decode_table(code)
    got = ref.copy()
    c = codes_of(got)
    assert np.all(c[:, 1:] == 0)
    small = int(np.flatnonzero(np.isclose(table, 2.0 ** -10))[0])      # far below 2^-17 * 57344
    c[0, 3] = small
    st = compare_records(got, ref, B, u_exact=u, code=code)
    assert st["noise_mismatches"] == 1 and st["code_mismatches"] == 0
    big = int(np.flatnonzero(np.isclose(table, 2.0))[0])                # above 2 * 2^-17 * 57344 = 0.875
    c[1, 7] = big
    with pytest.raises(AssertionError):
        compare_records(got, ref, B, u_exact=u, code=code)


def test_exact_scales_agree_with_the_oracle():
    """The real-arithmetic scales used by the rule against the oracle's binary32
    ones: compress (every variant) and a 3-shard reduce."""
    from parity import exact_compress_scales, exact_reduce_scales
    from helpers import records
    bits = workloads.generate("student_t_channels", 32, 1024, 5).reshape(-1)
    for variant in range(4):
        for code in (0, 1, 2):
            ref = oracle.compress(bits, B, variant, code)
            _, a, s = records(ref, B)
            ae, se = exact_compress_scales(bits, B, variant, code)
            assert np.max(np.abs(a / ae - 1)) < 1e-6 and np.max(np.abs(s / se - 1)) < 1e-6, (variant, code)
    shards = [oracle.compress(workloads.generate("student_t_channels", 32, 1024, p).reshape(-1), B) for p in range(3)]
    _, a, s = records(oracle.reduce_shards(shards, 32 * 1024, B), B)
    ae, se = exact_reduce_scales(shards, B)
    assert np.max(np.abs(a / ae - 1)) < 2e-6 and np.max(np.abs(s / se - 1)) < 2e-6


def test_scale_closer_to_exact_passes_and_otherwise_fails(case):
    from parity import exact_compress_scales
    bits, ref = case
    ae, se = exact_compress_scales(bits, B)
    got = ref.copy()
    rec = got.reshape(-1, B + 8)
    ref_rec = ref.reshape(-1, B + 8)
    # Block 3: the reference's alpha moved 3e-6 off the exact value; the
    # tested alpha is the exact value rounded to binary32.
    bad_ref = ref.copy().reshape(-1, B + 8)
    bad_ref[3, B:B + 4] = np.float32(ae[3] * (1 + 3e-6)).reshape(1).view(np.uint8)
    rec[3, B:B + 4] = np.float32(ae[3]).reshape(1).view(np.uint8)
    st = compare_records(got, bad_ref.reshape(-1), B, scales_exact=(ae, se))
    assert st["scales_closer_to_exact"] == 1 and st["alpha_max_rel_vs_ref"] > 2e-6
    with pytest.raises(AssertionError):
        compare_records(got, bad_ref.reshape(-1), B)            # without the exact values
    # Tested alpha 3e-6 off both: fails.
    rec[3, B:B + 4] = np.float32(ae[3] * (1 - 3e-6)).reshape(1).view(np.uint8)
    with pytest.raises(AssertionError):
        compare_records(got, bad_ref.reshape(-1), B, scales_exact=(ae, se))


def test_exact_compress_u_matches_the_float64_restatement():
    """exact_compress_u against helpers.exact_compress_quantities (ASH + DS)
    for each code format's Q_max, and the DS-only and ASH-only forms against
    their definitions."""
    from helpers import exact_compress_quantities
    from parity import exact_compress_u
    bits = workloads.generate("laplace_outliers", 16, 1024, 9).reshape(-1)
    G = bf16_to_f64(bits).reshape(-1, B)
    _, _, u, _ = exact_compress_quantities(G, B)
    for code, qmax in ((0, 448.0), (1, 57344.0), (2, 127.0)):
        assert np.allclose(exact_compress_u(bits, B, 0, code), u * qmax / 448.0, rtol=1e-12, atol=0)
    ds = exact_compress_u(bits, B, 2, 0)
    assert np.allclose(ds, 448.0 * G / np.abs(G).max(axis=1, keepdims=True), rtol=1e-12, atol=0)
    ash = exact_compress_u(bits, B, 3, 0)
    alpha = 1.0 / np.sqrt((G * G).mean(axis=1, keepdims=True) + float(np.float32(1e-30)))
    assert np.allclose(ash, alpha * (G @ hadamard(B).T) / np.sqrt(B), rtol=1e-12, atol=0)
