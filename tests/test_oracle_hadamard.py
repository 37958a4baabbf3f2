"""Pins of the oracle's Walsh-Hadamard transform (Eq. 8, FWHT of Section 4.2.2).

- FWHT of each unit vector is the matching column of SciPy's Sylvester
  Hadamard matrix (a library routine), for every B from 2 to 512.
- H H^T = B I and H = H^T (closed form), so (1/sqrt B) H is orthogonal and
  its own inverse (Section 4.2.2).
- FWHT(FWHT(v)) = B v exactly on small integers.
- FWHT agrees with the float64 dense matrix-vector product within the
  float32 error bound of a log2(B)-stage butterfly.
"""
import numpy as np
import pytest
import scipy.linalg

import oracle

BLOCKS = [2, 4, 8, 16, 32, 64, 128, 256, 512]


@pytest.mark.parametrize("B", BLOCKS)
def test_fwht_of_identity_is_sylvester_hadamard(B):
    H = oracle.fwht(np.eye(B, dtype=np.float32), B)   # row k = FWHT(e_k) = column k of H
    ref = scipy.linalg.hadamard(B).astype(np.float32)
    assert np.array_equal(H.T, ref)


@pytest.mark.parametrize("B", BLOCKS)
def test_hadamard_is_symmetric_and_orthogonal(B):
    H = oracle.fwht(np.eye(B, dtype=np.float32), B).astype(np.float64)
    assert np.array_equal(H, H.T)
    assert np.array_equal(H @ H.T, B * np.eye(B))
    # Entries are +-1 with the sign pattern (-1)^popcount(i & j).
    i, j = np.meshgrid(np.arange(B), np.arange(B), indexing="ij")
    pop = np.vectorize(lambda v: bin(v).count("1"))(i & j)
    assert np.array_equal(H, np.where(pop % 2 == 0, 1.0, -1.0))


@pytest.mark.parametrize("B", [4, 64, 128, 256])
def test_fwht_twice_is_B_times_identity_on_integers(B):
    rng = np.random.default_rng(B)
    v = rng.integers(-1000, 1000, size=(50, B)).astype(np.float32)
    w = oracle.fwht(oracle.fwht(v, B), B)
    assert np.array_equal(w, B * v)


@pytest.mark.parametrize("B", [64, 128, 256])
def test_fwht_matches_dense_float64_within_float32_bound(B):
    rng = np.random.default_rng(7 + B)
    v = rng.standard_normal((200, B)).astype(np.float32)
    H = scipy.linalg.hadamard(B).astype(np.float64)
    exact = v.astype(np.float64) @ H.T
    got = oracle.fwht(v, B).astype(np.float64)
    # Each of log2(B) stages adds one rounding of a value bounded by the
    # stage's partial sums, which are bounded by sum |v|.
    bound = np.log2(B) * np.finfo(np.float32).eps * np.abs(v.astype(np.float64)).sum(axis=1, keepdims=True)
    assert np.all(np.abs(got - exact) <= bound)
    # Parseval (energy preservation of the normalised rotation, Section 4.2.2).
    e_in = (v.astype(np.float64) ** 2).sum(axis=1)
    e_out = (got ** 2).sum(axis=1) / B
    assert np.allclose(e_out, e_in, rtol=1e-5)
