"""The bf16 high/low pair that carries fp32 operands into bf16 tensor-core products (decode attention's
queries and probabilities, the prefill GEMMs' activations): x = hi + lo with hi = bf16(x) and
lo = bf16(x - hi).  These CPU tests pin the precision the parity reading relies on, from the definition
of bf16 rounding (round to nearest even on the top 16 bits of the fp32 pattern), independent of any
GPU code: the pair is within 2^-16 of x relative (2^-18 typical), products of a pair part with a bf16
value are exact in fp32, and an attention evaluated with pair products and fp32 accumulation stays
within the error the pair's 2^-16 puts on its scores (below 1e-4 of max |o| here), more than 20 times
closer to the float64 result than one bf16 per operand.
"""
import numpy as np


def bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even), returned as fp32."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def pair(x: np.ndarray):
    x = np.asarray(x, dtype=np.float32)
    hi = bf16(x)
    lo = bf16((x - hi).astype(np.float32))
    return hi, lo


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties to the even pattern (1.0)
    assert bf16(np.float32(1.0 + 2.0 ** -8)) == np.float32(1.0)
    # 1 + 3 * 2^-8 is the midpoint between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6 (even)
    assert bf16(np.float32(1.0 + 3 * 2.0 ** -8)) == np.float32(1.0 + 2.0 ** -6)
    assert bf16(np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20)) == np.float32(1.0 + 2.0 ** -7)


def test_pair_error_is_within_two_to_the_minus_16():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200_000), rng.uniform(0, 1, 200_000),
                        np.exp(rng.uniform(-30, 30, 100_000))]).astype(np.float32)
    hi, lo = pair(x)
    err = np.abs(x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    rel = err / np.abs(x.astype(np.float64))
    assert rel.max() <= 2.0 ** -16
    assert np.median(rel) <= 2.0 ** -18
    # a single bf16 is 2^8 times coarser: the pair is what makes the products fp32-accurate
    assert np.max(np.abs(x - hi) / np.abs(x)) > 2.0 ** -10


def test_products_of_pairs_with_bf16_are_exact_in_fp32():
    # bf16 x bf16 has at most 16 significant bits: exact in fp32, so only the accumulation rounds
    rng = np.random.default_rng(1)
    a = bf16(rng.standard_normal(100_000).astype(np.float32))
    b = bf16(rng.standard_normal(100_000).astype(np.float32))
    assert np.array_equal((a * b).astype(np.float64), a.astype(np.float64) * b.astype(np.float64))


def test_attention_in_pair_arithmetic_matches_float64():
    """Scores q.k and outputs sum p v with q and p as pairs, K and V bf16, fp32 accumulation (the
    tensor-core path's arithmetic), against the float64 definition.  The pair's 2^-16 relative error on
    q moves a score by at most 2^-16 * scale * sum_i |q_i k_i|, which moves its softmax weight by that
    much relatively; p's own pair error and the fp32 sums add less.  So the outputs are within twice that
    score error times max |v| -- and a single bf16 per operand is far coarser."""
    rng = np.random.default_rng(2)
    d, n, scale = 64, 513, 1.0 / 8.0
    q = (rng.standard_normal(d) * 2).astype(np.float32)
    K = bf16((rng.standard_normal((n, d)) * 2).astype(np.float32))
    V = bf16((rng.standard_normal((n, d)) * 2).astype(np.float32))
    # reference
    s64 = K.astype(np.float64) @ q.astype(np.float64) * scale
    p64 = np.exp(s64 - s64.max())
    o64 = (p64 @ V.astype(np.float64)) / p64.sum()
    # pair arithmetic: every product exact, sums in fp32 (in 16-term chunks, like an MMA's k-steps)
    qh, ql = pair(q)
    def dot32(a, b):
        acc = np.float32(0)
        for c in range(0, a.shape[-1], 16):
            acc = np.float32(acc + np.float32(np.sum((a[..., c:c + 16] * b[c:c + 16]).astype(np.float64))))
        return acc
    s = np.array([np.float32(dot32(K[j], qh) + dot32(K[j], ql)) * np.float32(scale) for j in range(n)],
                 dtype=np.float32)
    p = np.exp2((s - s.max()) * np.float32(np.log2(np.e))).astype(np.float32)
    ph, pl = pair(p)
    o = np.zeros(d, dtype=np.float32)
    for c in range(0, n, 16):
        blk = slice(c, min(n, c + 16))
        o = (o + (ph[blk].astype(np.float64) @ V[blk].astype(np.float64)).astype(np.float32)
             + (pl[blk].astype(np.float64) @ V[blk].astype(np.float64)).astype(np.float32)).astype(np.float32)
    o = o / np.float32(p.sum(dtype=np.float32))
    ds = 2.0 ** -16 * scale * np.max(np.abs(K.astype(np.float64)) @ np.abs(q.astype(np.float64)))
    err = np.max(np.abs(o - o64))
    assert err <= 2 * ds * np.max(np.abs(V))
    assert err <= 1e-4 * np.max(np.abs(o64))
    # the same with the queries and weights as single bf16 values is far coarser
    s1 = (K.astype(np.float64) @ bf16(q).astype(np.float64)) * scale
    p1 = bf16(np.exp(s1 - s1.max()).astype(np.float32)).astype(np.float64)
    o1 = (p1 @ V.astype(np.float64)) / p1.sum()
    assert np.max(np.abs(o1 - o64)) > 20 * err
