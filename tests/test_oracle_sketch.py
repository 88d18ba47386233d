"""Pins for the SALS-style sketch selector of the oracle.

What fixes the answer: the integer dot is an exact integer (checked against
Python integer loops); symmetric rounding keeps every dequantised code
within half a step of the value it encodes and maps the block maximum to
+-7; the fp32 projection differs from the exact one by at most the
summation error bound, and its codes differ from exactly-rounded ones only
next to a rounding boundary; with an identity projection and no
quantisation the block score is the exact log of the block's softmax mass
(QSI step 3 says the LSE stands for the block's attention weight sum), so
the block masses of a sequence add up to the whole-sequence log-sum-exp,
here cross-checked with scipy's logsumexp; a Gaussian projection with
variance 1/d_s keeps q.k unbiased (Johnson-Lindenstrauss, SequenceO1 close
reading §3.1).
"""

import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import sketch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_int_dots_brute_force(rng):
    for trial in range(20):
        ds = 16
        qc = rng.integers(-127, 128, ds).astype(np.int8)
        codes = rng.integers(-7, 8, (64, ds)).astype(np.int8)
        got = sketch.int_dots(qc, codes)
        for t in range(64):
            assert got[t] == sum(int(qc[j]) * int(codes[t][j]) for j in range(ds))


def test_quantisation_error_bound(rng):
    for trial in range(50):
        x = (rng.standard_normal((64, 16)) * rng.random() * 10).astype(np.float32)
        codes, scale = sketch.quantise_block_int4(x)
        assert codes.min() >= -7 and codes.max() <= 7
        err = np.abs(codes.astype(np.float64) * float(scale) - x.astype(np.float64))
        assert err.max() <= float(scale) * (0.5 + 1e-6)
        i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert abs(int(codes[i])) == 7
        # symmetric: negating the block negates the codes
        codes_n, scale_n = sketch.quantise_block_int4(-x)
        assert scale_n == scale and (codes_n == -codes).all()


def test_zero_block_scale_is_one():
    codes, scale = sketch.quantise_block_int4(np.zeros((4, 16), np.float32))
    assert scale == 1.0 and (codes == 0).all()


def test_index_query_codes(rng):
    q = rng.standard_normal((4, 32)).astype(np.float16)
    proj = rng.standard_normal((32, 16)).astype(np.float32) / 4
    qc, sq = sketch.index_query(q, proj)
    exact = np.asarray(q, dtype=np.float64).mean(axis=0) @ proj.astype(np.float64)
    assert np.abs(qc).max() == 127
    assert np.abs(qc.astype(np.float64) * sq - exact).max() <= sq * 0.5 + 1e-5 * np.abs(exact).max()


def test_fp32_projection_within_summation_bound(rng):
    x = (rng.standard_normal((64, 128)) * 3).astype(np.float32)
    proj = (rng.standard_normal((128, 16)) / 4).astype(np.float32)
    p32 = sketch.project_fp32(x, proj).astype(np.float64)
    p64 = sketch.project_fp64(x, proj)
    bound = 128 * np.finfo(np.float32).eps * (np.abs(x).astype(np.float64) @ np.abs(proj).astype(np.float64))
    assert (np.abs(p32 - p64) <= bound).all()
    # codes from the fp32 projection equal exactly rounded codes away from ties
    codes, scale = sketch.quantise_block_int4(p32.astype(np.float32))
    ratio = p64 / float(scale)
    exact_codes = np.clip(np.rint(ratio), -7, 7)
    near = np.abs(np.abs(ratio - np.floor(ratio)) - 0.5) < 1e-4
    assert ((codes == exact_codes) | near).all()


def test_identity_projection_block_score_is_log_block_mass(rng):
    d, S, n_blocks = 16, 8, 6
    qbar = rng.standard_normal(d)
    keys = rng.standard_normal((n_blocks * S, d)) * 2
    z = keys @ qbar / math.sqrt(d)
    scores = [sketch.block_lse(z[b * S : (b + 1) * S]) for b in range(n_blocks)]
    for b in range(n_blocks):
        assert scores[b] == pytest.approx(logsumexp(z[b * S : (b + 1) * S]), rel=1e-13)
    assert logsumexp(scores) == pytest.approx(logsumexp(z), rel=1e-13)
    # block mass = softmax weight summed over the block
    w = np.exp(z - logsumexp(z))
    for b in range(n_blocks):
        assert math.exp(scores[b] - logsumexp(z)) == pytest.approx(w[b * S : (b + 1) * S].sum(), rel=1e-12)


def test_lse_bounds_and_single_token(rng):
    for n in (1, 2, 64):
        z = rng.standard_normal(n) * 5
        s = sketch.block_lse(z)
        assert z.max() <= s <= z.max() + math.log(n) + 1e-12
    assert sketch.block_lse(np.array([3.25])) == 3.25


def test_block_scores_dequantise_integer_logits(rng):
    qc = rng.integers(-127, 128, 16).astype(np.int8)
    codes = rng.integers(-7, 8, (2, 64, 16)).astype(np.int8)
    scales = np.array([0.5, 0.125], np.float32)
    s = sketch.block_scores(qc, np.float32(0.25), codes, scales, 128)
    for b in range(2):
        z = [sum(int(qc[j]) * int(codes[b, t, j]) for j in range(16)) * 0.25 * float(scales[b]) / math.sqrt(128) for t in range(64)]
        assert s[b] == pytest.approx(logsumexp(z), rel=1e-13)


def test_projection_is_unbiased_for_dot_products(rng):
    d, ds, n = 128, 16, 4000
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    est = []
    for _ in range(n):
        P = rng.standard_normal((d, ds)) / math.sqrt(ds)
        est.append((q @ P) @ (k @ P))
    est = np.array(est)
    assert abs(est.mean() - q @ k) < 4 * est.std() / math.sqrt(n)


def test_int4_packing_golden():
    cases = json.load(open(os.path.join(GOLDEN, "int4_packing.json")))["cases"]
    for c in cases:
        packed = sketch.pack_int4(np.array(c["codes"], np.int8))
        assert int(packed[0]) == c["byte"]
        assert list(sketch.unpack_int4(packed)) == c["codes"]
    allc = np.arange(-8, 8, dtype=np.int8)
    assert (sketch.unpack_int4(sketch.pack_int4(allc)) == allc).all()


def test_planted_mistake_is_caught(rng, monkeypatch):
    """Truncating instead of rounding must fail the half-step error bound."""

    def truncating(v):
        v = np.asarray(v, dtype=np.float32)
        amax = np.float32(np.max(np.abs(v)))
        scale = amax / np.float32(7.0)
        return np.clip(np.trunc(v / scale), -7, 7).astype(np.int8), np.float32(scale)

    monkeypatch.setattr(sketch, "quantise_block_int4", truncating)
    with pytest.raises(AssertionError):
        test_quantisation_error_bound(rng)


def test_dequant_golden():
    """Hand-worked int8 code x fp16 scale products (exact in fp32)."""
    g = json.load(open(os.path.join(GOLDEN, "int8_dequant.json")))
    for c in g["cases"]:
        assert float(np.float16(c["scale"])) == c["scale"], "the fixture's scales are fp16 values"
        got = sketch.dequant(np.array([[c["code"]]], np.int8), np.array([c["scale"]], np.float16))
        assert got.dtype == np.float32 and float(got[0, 0]) == c["value"]


def test_dequant_is_the_exact_product(rng):
    """Every int8 x fp16 product fits fp32: dequant equals the exact rational product,
    row by row with each row's own scale (a transposed scale would fail)."""
    from fractions import Fraction

    codes = rng.integers(-128, 128, (6, 9)).astype(np.int8)
    scales = (rng.standard_normal(6) * 0.05).astype(np.float16)
    got = sketch.dequant(codes, scales)
    for t in range(6):
        for i in range(9):
            assert Fraction(float(got[t, i])) == Fraction(int(codes[t, i])) * Fraction(float(scales[t]))


def _sketch_unit(rng, S=64, n_blocks=4, d=32):
    from oracle import decode

    P = n_blocks
    k = rng.integers(-127, 128, (P, 1, S, d)).astype(np.int8)
    v = rng.integers(-127, 128, (P, 1, S, d)).astype(np.int8)
    ks = (rng.random((P, 1, S)) * 0.02 + 0.001).astype(np.float16)
    vs = (rng.random((P, 1, S)) * 0.02 + 0.001).astype(np.float16)
    proj = (rng.standard_normal((d, 16)) / 4.0).astype(np.float32)
    q = rng.standard_normal((1, 2, d)).astype(np.float16)
    inp = decode.StepInputs(q, k, v, ks, vs, np.arange(P)[None, :], np.array([P * S]), proj)
    prm = decode.StepParams(S, 3, 0, 1, "sketch", d)
    return decode, inp, prm


def test_sketch_scores_read_the_key_scales_not_the_value_scales(rng):
    """The index key is built from the dequantised KEYS: new value scales
    leave every block score unchanged; doubling the key scales (exact in
    fp16) keeps the int4 codes, doubles each block's sketch scale, and so
    changes the scores."""
    decode, inp, prm = _sketch_unit(rng)
    base = decode.unit_sketch_scores(inp, prm, 0, 0)
    inp2 = decode.StepInputs(inp.q, inp.k_pool, inp.v_pool, inp.k_scale,
                             (inp.v_scale.astype(np.float32) * 3.0 + 0.5).astype(np.float16),
                             inp.page_table, inp.seq_lens, inp.proj)
    assert np.array_equal(decode.unit_sketch_scores(inp2, prm, 0, 0), base, equal_nan=True)
    inp3 = decode.StepInputs(inp.q, inp.k_pool, inp.v_pool, (inp.k_scale.astype(np.float32) * 2).astype(np.float16),
                             inp.v_scale, inp.page_table, inp.seq_lens, inp.proj)
    c1, s1 = decode.unit_sketch_blocks(inp, prm, 0, 0, [0, 1, 2])
    c2, s2 = decode.unit_sketch_blocks(inp3, prm, 0, 0, [0, 1, 2])
    for a, b in zip(c1, c2):
        assert np.array_equal(a, b)
    assert [2 * float(x) for x in s1] == [float(x) for x in s2]
    got = decode.unit_sketch_scores(inp3, prm, 0, 0)
    assert not np.allclose(got[:-1], base[:-1])
