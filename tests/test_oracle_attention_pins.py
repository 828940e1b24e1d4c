"""Pins of the oracle's attention forward against what the mathematics fixes.

The oracle computes O = softmax(scale * Q K^T [causal]) V per query row in
fp64 (the block "post_1787550000" builds toward: S = Q K^T and O = P V on
the tensor cores with the softmax between them, and a causal mask).  None of
these checks re-types its loop; each would fail on a plausible slip:

* an independent pure-Python brute force (math.exp / math.fsum, rows and
  keys in plain loops) on tiny shapes, causal and not, SQ != SKV -- a
  dropped scale, a transposed operand, an off-by-one in the mask;
* closed forms: zero queries give the mean of the allowed values and
  lse = log(#keys); causal row 0 of a square problem is V[0] exactly; a
  constant value column comes back unchanged (probabilities sum to 1);
* a dominant key returns its value row (and no overflow: the max shift);
* invariances: permuting keys with their values (non-causal); adding the
  same constant to every score of a row (a key offset along a direction the
  query sees as constant);
* the normaliser: Den >= |O| everywhere, Den = mean |v| for zero queries;
* scipy.special.softmax / logsumexp applied to scores formed by numpy.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)


def draw(shape, seed, dtype=torch.bfloat16, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(dtype)


def brute(q, k, v, scale, causal):
    """Independent fp64 reference with Python loops (tiny shapes only)."""
    BH, SQ, D = q.shape
    SKV = k.shape[1]
    O = np.zeros((BH, SQ, D))
    lse = np.zeros((BH, SQ))
    for b in range(BH):
        for i in range(SQ):
            keys = [j for j in range(SKV) if not causal or j <= i + SKV - SQ]
            s = [scale * math.fsum(float(q[b, i, c]) * float(k[b, j, c]) for c in range(D)) for j in keys]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            l = math.fsum(e)
            for c in range(D):
                O[b, i, c] = math.fsum(e[t] * float(v[b, keys[t], c]) for t in range(len(keys))) / l
            lse[b, i] = m + math.log(l)
    return O, lse


@pytest.mark.parametrize("SQ,SKV,causal", [(5, 5, False), (5, 5, True), (3, 7, True), (6, 4, False)])
@pytest.mark.parametrize("dtype,code", [(torch.bfloat16, oracle.BF16), (torch.float16, oracle.F16)])
def test_attention_matches_brute_force(SQ, SKV, causal, dtype, code):
    BH, D = 2, 6
    q, k, v = draw((BH, SQ, D), 1, dtype), draw((BH, SKV, D), 2, dtype), draw((BH, SKV, D), 3, dtype)
    scale = 0.37
    O, Den, lse, sden = oracle.attention(bits(q), bits(k), bits(v), code, BH, SQ, SKV, D, scale, causal)
    Ob, lseb = brute(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale, causal)
    assert np.allclose(O, Ob, rtol=0, atol=1e-13)
    assert np.allclose(lse, lseb, rtol=0, atol=1e-13)
    assert np.all(Den >= np.abs(O) - 1e-15)


def test_attention_zero_queries_give_the_mean():
    BH, SQ, SKV, D = 2, 4, 9, 8
    q = torch.zeros((BH, SQ, D), dtype=torch.bfloat16)
    k, v = draw((BH, SKV, D), 5), draw((BH, SKV, D), 6)
    O, Den, lse, sden = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, SQ, SKV, D, 1.0)
    vv = v.double().numpy()
    for i in range(SQ):
        assert np.allclose(O[:, i], vv.mean(axis=1), rtol=0, atol=1e-15)
        assert np.allclose(Den[:, i], np.abs(vv).mean(axis=1), rtol=0, atol=1e-15)
    assert np.allclose(lse, math.log(SKV), rtol=0, atol=1e-15)
    assert np.all(sden == 0)


def test_attention_zero_queries_causal_counts_allowed_keys():
    """Row i of a causal problem with SKV = SQ + 2 sees keys 0 .. i + 2."""
    BH, SQ, SKV, D = 1, 5, 7, 4
    q = torch.zeros((BH, SQ, D), dtype=torch.float16)
    k, v = draw((BH, SKV, D), 7, torch.float16), draw((BH, SKV, D), 8, torch.float16)
    O, _, lse, _ = oracle.attention(bits(q), bits(k), bits(v), oracle.F16, BH, SQ, SKV, D, 1.0, True)
    vv = v.double().numpy()[0]
    for i in range(SQ):
        n = i + 3
        assert np.allclose(O[0, i], vv[:n].mean(axis=0), rtol=0, atol=1e-15)
        assert abs(lse[0, i] - math.log(n)) < 1e-15


def test_attention_causal_first_row_is_first_value():
    BH, S, D = 3, 6, 5
    q, k, v = draw((BH, S, D), 9), draw((BH, S, D), 10), draw((BH, S, D), 11)
    O, _, _, _ = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, S, S, D, 0.5, True)
    assert np.array_equal(O[:, 0], v.double().numpy()[:, 0])


def test_attention_constant_value_column():
    BH, SQ, SKV, D = 2, 7, 11, 4
    q, k = draw((BH, SQ, D), 12), draw((BH, SKV, D), 13)
    v = draw((BH, SKV, D), 14)
    v[..., 2] = 1.5
    for causal in (False, True):
        O, _, _, _ = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, SQ, SKV, D, 0.9, causal)
        assert np.allclose(O[..., 2], 1.5, rtol=0, atol=1e-14)


def test_attention_dominant_key():
    """One key aligned with the query at a score far above the others: the
    output is that key's value row, and huge scores do not overflow."""
    BH, SQ, SKV, D = 1, 1, 8, 4
    q = torch.tensor([[[1.0, 0.0, 0.0, 0.0]]], dtype=torch.bfloat16)
    k = torch.zeros((BH, SKV, D), dtype=torch.bfloat16)
    k[0, 5, 0] = 256.0
    v = draw((BH, SKV, D), 15)
    O, _, lse, _ = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, SQ, SKV, D, 100.0)
    assert np.array_equal(O[0, 0], v.double().numpy()[0, 5])
    assert abs(lse[0, 0] - 25600.0) < 1e-9


def test_attention_key_permutation_invariance():
    BH, SQ, SKV, D = 2, 5, 9, 6
    q, k, v = draw((BH, SQ, D), 16), draw((BH, SKV, D), 17), draw((BH, SKV, D), 18)
    perm = torch.randperm(SKV, generator=torch.Generator().manual_seed(3))
    O1, _, l1, _ = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, SQ, SKV, D, 0.4)
    O2, _, l2, _ = oracle.attention(bits(q), bits(k[:, perm]), bits(v[:, perm]), oracle.BF16, BH, SQ, SKV, D, 0.4)
    assert np.allclose(O1, O2, rtol=0, atol=1e-14)
    assert np.allclose(l1, l2, rtol=0, atol=1e-13)


def test_attention_row_shift_invariance():
    """Queries q = (x, 1) and keys k_j = (y_j, t): every score of the row
    moves by the same t; O is unchanged, lse moves by t * scale."""
    BH, SQ, SKV, D = 1, 3, 6, 4
    q = draw((BH, SQ, D), 19)
    q[..., -1] = 1.0
    k, v = draw((BH, SKV, D), 20), draw((BH, SKV, D), 21)
    k[..., -1] = 0.0
    O1, _, l1, _ = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, SQ, SKV, D, 0.5)
    k2 = k.clone()
    k2[..., -1] = 8.0
    O2, _, l2, _ = oracle.attention(bits(q), bits(k2), bits(v), oracle.BF16, BH, SQ, SKV, D, 0.5)
    assert np.allclose(O1, O2, rtol=0, atol=1e-14)
    assert np.allclose(l2 - l1, 4.0, rtol=0, atol=1e-13)


def test_attention_against_scipy_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    BH, SQ, SKV, D = 3, 16, 24, 32
    q, k, v = draw((BH, SQ, D), 22), draw((BH, SKV, D), 23), draw((BH, SKV, D), 24)
    scale = 1.0 / math.sqrt(D)
    O, _, lse, _ = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, SQ, SKV, D, scale)
    S = scale * np.einsum("bic,bjc->bij", q.double().numpy(), k.double().numpy())
    P = scipy_special.softmax(S, axis=-1)
    assert np.allclose(O, P @ v.double().numpy(), rtol=0, atol=1e-13)
    assert np.allclose(lse, scipy_special.logsumexp(S, axis=-1), rtol=0, atol=1e-13)


def test_attention_sampled_rows_equal_full():
    BH, SQ, SKV, D = 2, 9, 13, 8
    q, k, v = draw((BH, SQ, D), 25), draw((BH, SKV, D), 26), draw((BH, SKV, D), 27)
    O, Den, lse, sden = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, SQ, SKV, D, 0.3, True)
    rb = np.array([1, 0, 1])
    ri = np.array([8, 0, 3])
    Os, Dens, lses, sdens = oracle.attention(bits(q), bits(k), bits(v), oracle.BF16, BH, SQ, SKV, D, 0.3,
                                             True, rows=(rb, ri))
    assert np.array_equal(Os, O[rb, ri]) and np.array_equal(Dens, Den[rb, ri])
    assert np.array_equal(lses, lse[rb, ri]) and np.array_equal(sdens, sden[rb, ri])
