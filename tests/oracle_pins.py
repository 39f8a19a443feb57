"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each `pin_*` function takes a loaded oracle library (ctypes) and raises AssertionError when the
library disagrees with a closed form, an invariant, a brute-force float64 computation, a library
routine (torch / scipy) or a value printed on the MegaBake pages.  They are written as plain
functions so that test_oracle.py can run them against the real oracle and test_oracle_mutants.py
can run them against deliberately broken copies of it (each copy must fail at least one pin).
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch
import torch.nn.functional as F

F32 = np.float32


def _p(a):
    return a.ctypes.data


def _bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _f32_to_bf16_torch(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rand_bf16(rng, shape, std=0.5):
    return _f32_to_bf16_torch(rng.standard_normal(shape).astype(np.float32) * std)


# ---------------------------------------------------------------- bf16 rounding
def pin_bf16_rounding(lib):
    """Round-to-nearest-even fp32 -> bf16 equals torch's cast (a library routine) on random
    values, exact ties, subnormals, infinities and the largest finite values."""
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(4000).astype(F32) * 10.0) + list(rng.standard_normal(500).astype(F32) * 1e-40)
    ties = [np.uint32(0x3F808000), np.uint32(0x3F818000), np.uint32(0xBF808000), np.uint32(0x3F80FFFF),
            np.uint32(0x7F7FFFFF), np.uint32(0x00008000), np.uint32(0x00018000), np.uint32(0x7F800000),
            np.uint32(0xFF800000), np.uint32(0x80000000), np.uint32(0)]
    vals += [np.array([t], dtype=np.uint32).view(F32)[0] for t in ties]
    arr = np.array(vals, dtype=F32)
    want = _f32_to_bf16_torch(arr)
    got = np.array([lib.orc_f32_to_bf16(float(v)) for v in arr], dtype=np.uint16)
    assert np.array_equal(got, want), "bf16 rounding differs from torch's cast"
    # widening is exact: bf16 bits b -> fp32 bits b << 16
    for b in [0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049]:
        assert np.float32(lib.orc_bf16_to_f32(b)) == np.array([b << 16], dtype=np.uint32).view(F32)[0]
    nan = np.array([0x7FC00001], dtype=np.uint32).view(F32)[0]
    r = lib.orc_f32_to_bf16(float(nan))
    assert (r & 0x7F80) == 0x7F80 and (r & 0x7F) != 0, "NaN must stay NaN"


# ---------------------------------------------------------------- RMSNorm
def _rmsnorm(lib, x, g=None, eps=0.0):
    x = np.ascontiguousarray(x, dtype=F32)
    out = np.empty_like(x)
    lib.orc_rmsnorm(_p(x), None if g is None else _p(g), x.size, eps, _p(out))
    return out


def pin_rmsnorm(lib):
    """Unit RMS before the gain, scale invariance at eps = 0, the eps closed form on a constant
    vector, and the gain applied elementwise (with gain g, out / g has unit RMS)."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal(576).astype(F32) * 3.0
    y = _rmsnorm(lib, x)
    assert abs(math.sqrt(float(np.mean(y.astype(np.float64) ** 2))) - 1.0) < 1e-6
    y2 = _rmsnorm(lib, x * F32(7.5))
    assert np.allclose(y, y2, rtol=2e-6, atol=0)
    # constant vector c with eps: out = c / sqrt(c^2 + eps)
    c, eps = 0.01, 1e-4
    yc = _rmsnorm(lib, np.full(64, c, dtype=F32), eps=eps)
    assert np.allclose(yc, c / math.sqrt(c * c + eps), rtol=1e-6)
    g = _f32_to_bf16_torch(rng.uniform(0.5, 1.5, 576).astype(F32))
    yg = _rmsnorm(lib, x, g)
    gf = _bits_to_f32(g)
    assert np.allclose(yg, y * gf, rtol=1e-6, atol=1e-7)
    # against the library routine torch.nn.functional.rms_norm (float64)
    ref = F.rms_norm(torch.from_numpy(x).double(), (576,), weight=torch.from_numpy(gf).double(), eps=1e-5)
    got = _rmsnorm(lib, x, g, eps=1e-5)
    assert np.allclose(got, ref.numpy(), rtol=1e-6, atol=1e-7)


# ---------------------------------------------------------------- GEMV
def _gemv(lib, W, x, b=None):
    rows, cols = W.shape
    y = np.empty(rows, dtype=F32)
    x = np.ascontiguousarray(x, dtype=F32)
    lib.orc_gemv(_p(W), _p(x), None if b is None else _p(b), rows, cols, _p(y), 1)
    return y


def pin_gemv(lib):
    """Brute-force float64 dot products on a small [out, in] matrix (rows are outputs), a one-hot
    input selecting one column, and the bias added once per row."""
    rng = np.random.default_rng(3)
    W = _rand_bf16(rng, (37, 53))
    x = rng.standard_normal(53).astype(F32)
    Wf = _bits_to_f32(W).astype(np.float64)
    want = np.array([sum(Wf[r, k] * float(x[k]) for k in range(53)) for r in range(37)])
    assert np.allclose(_gemv(lib, W, x), want, rtol=1e-6, atol=1e-7)
    e = np.zeros(53, dtype=F32)
    e[11] = 1.0
    assert np.array_equal(_gemv(lib, W, e), _bits_to_f32(W[:, 11]))
    b = _rand_bf16(rng, (37,))
    assert np.allclose(_gemv(lib, W, x, b), want + _bits_to_f32(b), rtol=1e-6, atol=1e-7)


# ---------------------------------------------------------------- RoPE
def _rope(lib, v, n_heads, d, pos, theta):
    v = np.ascontiguousarray(v, dtype=F32).copy()
    lib.orc_rope(_p(v), n_heads, d, pos, theta)
    return v


def pin_rope(lib):
    """Identity at position 0; per-pair norms preserved; the rotate-half closed form on unit
    vectors (element i pairs with i + d/2, angle pos * theta^(-2i/d), sign of the rotation); and
    the relative-position property <R_p q, R_m k> = <R_(p-m) q, k>."""
    rng = np.random.default_rng(4)
    d, theta = 64, 10000.0
    v = rng.standard_normal(3 * d).astype(F32)
    assert np.array_equal(_rope(lib, v, 3, d, 0, theta), v)
    r = _rope(lib, v, 3, d, 37, theta).astype(np.float64).reshape(3, d)
    v3 = v.astype(np.float64).reshape(3, d)
    n0 = v3[:, : d // 2] ** 2 + v3[:, d // 2:] ** 2
    n1 = r[:, : d // 2] ** 2 + r[:, d // 2:] ** 2
    assert np.allclose(n0, n1, rtol=1e-6)
    for i in (0, 1, 5, 31):
        ang = 123 * theta ** (-2.0 * i / d)
        e = np.zeros(d, dtype=F32)
        e[i] = 1.0
        out = _rope(lib, e, 1, d, 123, theta)
        want = np.zeros(d)
        want[i], want[i + d // 2] = math.cos(ang), math.sin(ang)
        assert np.allclose(out, want, atol=1e-7), f"rope unit vector e_{i}"
        e = np.zeros(d, dtype=F32)
        e[i + d // 2] = 1.0
        out = _rope(lib, e, 1, d, 123, theta)
        want = np.zeros(d)
        want[i], want[i + d // 2] = -math.sin(ang), math.cos(ang)
        assert np.allclose(out, want, atol=1e-7), f"rope unit vector e_{i + d // 2}"
    q = rng.standard_normal(d).astype(F32)
    k = rng.standard_normal(d).astype(F32)
    a = float(np.dot(_rope(lib, q, 1, d, 50, theta).astype(np.float64), _rope(lib, k, 1, d, 20, theta).astype(np.float64)))
    b = float(np.dot(_rope(lib, q, 1, d, 30, theta).astype(np.float64), k.astype(np.float64)))
    assert abs(a - b) < 1e-5 * max(1.0, abs(b))


# ---------------------------------------------------------------- attention
def _attn(lib, q, K, V, nq, nkv, d, cap, ctx):
    o = np.empty(nq * d, dtype=F32)
    q = np.ascontiguousarray(q, dtype=F32)
    lib.orc_attention(_p(q), _p(K), _p(V), nq, nkv, d, cap, ctx, _p(o), 1)
    return o.reshape(nq, d)


def pin_attention(lib):
    """One cached key returns its V exactly; zero query (equal scores) returns the mean of V;
    query head h reads KV head h // (nq / nkv); rows at or beyond ctx are never read; and
    brute-force float64 softmax(q.K / sqrt(d)) V on small random inputs."""
    rng = np.random.default_rng(5)
    nq, nkv, d, cap = 6, 2, 64, 16
    K = _rand_bf16(rng, (nkv, cap, d))
    V = _rand_bf16(rng, (nkv, cap, d))
    q = rng.standard_normal(nq * d).astype(F32)
    o = _attn(lib, q, K, V, nq, nkv, d, cap, 1)
    for h in range(nq):
        assert np.array_equal(o[h], _bits_to_f32(V[h // 3, 0])), "single key must return its V"
    o = _attn(lib, np.zeros(nq * d, F32), K, V, nq, nkv, d, cap, 9)
    for h in range(nq):
        assert np.allclose(o[h], _bits_to_f32(V[h // 3, :9]).astype(np.float64).mean(0), rtol=1e-6, atol=1e-7)
    ctx = 11
    Kg = K.copy()
    Vg = V.copy()
    Kg[:, ctx:] = 0x7F00  # huge values beyond the context must not matter
    Vg[:, ctx:] = 0x7F00
    o1 = _attn(lib, q, Kg, Vg, nq, nkv, d, cap, ctx)
    Kf = _bits_to_f32(K).astype(np.float64)
    Vf = _bits_to_f32(V).astype(np.float64)
    for h in range(nq):
        kv = h // (nq // nkv)
        s = np.array([sum(float(q[h * d + t]) * Kf[kv, j, t] for t in range(d)) for j in range(ctx)]) / math.sqrt(d)
        a = np.exp(s - s.max())
        a /= a.sum()
        want = (a[:, None] * Vf[kv, :ctx]).sum(0)
        assert np.allclose(o1[h], want, rtol=1e-5, atol=1e-6), f"head {h}"


# ---------------------------------------------------------------- SiLU * up
def pin_silu_mul(lib):
    """silu(0) = 0, silu(z) -> z for large z, silu(z) -> 0 for very negative z, and
    silu(z) * u = z * expit(z) * u against scipy's logistic function."""
    from scipy.special import expit
    rng = np.random.default_rng(6)
    g = np.concatenate([[0.0, 30.0, -30.0], rng.standard_normal(200) * 4]).astype(F32)
    u = np.concatenate([[5.0, 1.0, 1.0], rng.standard_normal(200)]).astype(F32)
    h = np.empty_like(g)
    lib.orc_silu_mul(_p(g), _p(u), g.size, _p(h))
    assert h[0] == 0.0 and abs(h[1] - 30.0) < 1e-6 and abs(h[2]) < 1e-10
    want = g.astype(np.float64) * expit(g.astype(np.float64)) * u.astype(np.float64)
    assert np.allclose(h, want, rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------- whole decoder
def torch_restatement(wl, n_steps, kv_init=None, proj=None, lm=None):
    """An independent float64 restatement built from torch library routines (rms_norm, linear,
    scaled_dot_product_attention, silu).  Each op's result is rounded to fp32, K and V to bf16,
    which is the precision the oracle states.  kv_init: optional uint16 numpy cache to start
    from.  proj / lm: optional float64 replacements of the projection weights (proj[l][key]) and of
    the LM head matrix (FP8: the dequantized codes).  Returns (logits list, kv cache bf16 tensor)."""
    s = wl.shape
    L, H, nq, nkv, d, cap = s.n_layers, s.hidden, s.n_heads, s.n_kv_heads, s.head_dim, s.kv_capacity
    r32 = lambda t: t.float().double()  # noqa: E731
    E = wl.embed.double()
    if kv_init is None:
        kv = torch.zeros((L, 2, nkv, cap, d), dtype=torch.bfloat16)
    else:
        kv = torch.from_numpy(kv_init.view(np.int16)).view(torch.bfloat16).clone()
    inv_freq = s.rope_theta ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)

    def rot(x, pos):  # x: [heads, d]
        ang = pos * inv_freq
        cos = torch.cat([ang.cos(), ang.cos()])
        sin = torch.cat([ang.sin(), ang.sin()])
        half = torch.cat([-x[:, d // 2:], x[:, : d // 2]], dim=1)
        return x * cos + half * sin

    out = []
    for i in range(n_steps):
        tok, pos = int(wl.tokens[i]), s.pos0 + i
        x = E[tok].clone()
        for l in range(L):
            w = wl.layers[l]
            wk_ = (lambda key: proj[l][key]) if proj is not None else (lambda key: w[key].double())  # noqa: E731
            lin = lambda a, key, bkey=None: r32(F.linear(a, wk_(key),  # noqa: E731
                                                      None if (bkey is None or w[bkey] is None or not s.qkv_bias) else w[bkey].double()))
            xn = r32(F.rms_norm(x, (H,), weight=w["attn_norm"].double(), eps=s.rms_eps))
            q = lin(xn, "wq", "bq").view(nq, d)
            k = lin(xn, "wk", "bk").view(nkv, d)
            v = lin(xn, "wv", "bv").view(nkv, d)
            q = r32(rot(q, pos))
            k = r32(rot(k, pos))
            kv[l, 0, :, pos] = k.float().to(torch.bfloat16)
            kv[l, 1, :, pos] = v.float().to(torch.bfloat16)
            Kc = kv[l, 0, :, : pos + 1].double().repeat_interleave(nq // nkv, dim=0)
            Vc = kv[l, 1, :, : pos + 1].double().repeat_interleave(nq // nkv, dim=0)
            o = F.scaled_dot_product_attention(q.view(1, nq, 1, d), Kc.unsqueeze(0), Vc.unsqueeze(0))
            o = r32(o.reshape(nq * d))
            x = r32(x + lin(o, "wo"))
            xn = r32(F.rms_norm(x, (H,), weight=w["mlp_norm"].double(), eps=s.rms_eps))
            hh = r32(F.silu(lin(xn, "w_gate")) * lin(xn, "w_up"))
            x = r32(x + lin(hh, "w_down"))
        xn = r32(F.rms_norm(x, (H,), weight=wl.final_norm.double(), eps=s.rms_eps))
        out.append(r32(F.linear(xn, E if lm is None else lm)).float().numpy())
    return out, kv


def pin_decoder_vs_torch(lib_unused, wl, n_steps, decoder_cls):
    """The oracle's teacher-forced decode equals the torch restatement: logits to 1e-5 relative
    L2 every step, and identical bf16 KV caches (at most one ulp on a handful of entries)."""
    dec = decoder_cls(wl)
    ref_logits, ref_kv = torch_restatement(wl, n_steps)
    for i in range(n_steps):
        got = dec.step(int(wl.tokens[i]), wl.shape.pos0 + i)
        ref = ref_logits[i]
        rel = float(np.linalg.norm(got.astype(np.float64) - ref) / np.linalg.norm(ref))
        assert rel < 1e-5, f"step {i}: rel L2 {rel}"
    a = dec.kv.astype(np.int32)
    b = ref_kv.view(torch.int16).numpy().astype(np.int32) & 0xFFFF
    diff = a != b
    assert diff.sum() <= max(2, a.size // 100000), f"{diff.sum()} cache entries differ"


# ---------------------------------------------------------------- FP8 weight format
# E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities, S.1111.111 = NaN,
# largest finite 448; nearest code with ties to even, saturating.  Values worked out by hand.
FP8_EXACT = [(0.0, 0x00), (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (-448.0, 0xFE), (2.0 ** -6, 0x08),
             (2.0 ** -9, 0x01), (7 * 2.0 ** -9, 0x07), (3.0, 0x44), (240.0, 0x77), (256.0, 0x78), (0.3125, 0x2A)]
FP8_ROUNDED = [(1.0625, 0x38), (1.1875, 0x3A), (1.06, 0x38), (1.07, 0x39), (-0.3, 0xAA), (2.0 ** -10, 0x00),
               (1.5 * 2.0 ** -9, 0x02), (464.0, 0x7E), (1.0e6, 0x7E), (-1.0e6, 0xFE)]


def e4m3_values() -> np.ndarray:
    """Value of each of the 256 codes, from the bit fields (independent of the oracle's decoder)."""
    c = np.arange(256)
    e, m = (c >> 3) & 15, c & 7
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7))
    v = np.where(c & 0x80, -v, v)
    v[(e == 15) & (m == 7)] = np.nan
    return v


def pin_fp8_codes(lib):
    for value, code in FP8_EXACT + FP8_ROUNDED:
        assert lib.orc_fp8_from_f32(value) == code, (value, code)
    vals = e4m3_values()
    for c in range(256):
        if not np.isnan(vals[c]):
            assert lib.orc_fp8_to_f32(c) == vals[c], c
            assert lib.orc_fp8_from_f32(float(vals[c])) == c, c


def pin_fp8_quantize_and_gemv(lib, wl):
    """The oracle's codes and scales of real matrices against an exhaustive-search restatement, and
    its FP8 projection against the scaled float64 sum."""
    from oracle.oracle import bf16_bits, quantize_fp8
    vals = e4m3_values()
    pos = vals[:0x7F]
    for m in (wl.layers[0]["wq"], wl.embed[:64]):
        bits = bf16_bits(m)
        w = (bits.astype(np.uint32) << 16).view(np.float32)
        amax = np.abs(w).max(axis=1)
        s = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0)).astype(np.float32)
        x = (w / s[:, None]).astype(np.float32).astype(np.float64)
        d = np.abs(np.minimum(np.abs(x), 448.0)[..., None] - pos)
        best = d.min(axis=-1, keepdims=True)
        ties = d == best
        first = ties.argmax(axis=-1)
        nxt = np.take_along_axis(ties, np.minimum(first + 1, 0x7E)[..., None], axis=-1)[..., 0] & (first < 0x7E)
        want = np.where(nxt & (first % 2 == 1), first + 1, first).astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
        q, sc = quantize_fp8(bits, lib)
        assert np.array_equal(sc.view(np.uint32), s.view(np.uint32))
        assert np.array_equal(q, want)
        xin = np.random.default_rng(3).standard_normal(q.shape[1]).astype(F32)
        y = np.empty(q.shape[0], dtype=F32)
        lib.orc_gemv_fp8(_p(q), _p(sc), _p(xin), None, q.shape[0], q.shape[1], _p(y), 1)
        ref = (vals[q] @ xin.astype(np.float64)) * sc.astype(np.float64)
        assert np.allclose(y, ref.astype(F32), rtol=1e-6, atol=1e-12)


def pin_fp8_decoder_vs_torch(lib, wl, n_steps, decoder_cls):
    """The FP8 decode step equals the torch restatement run on the dequantized weights."""
    from oracle.oracle import FP8_SLOTS, bf16_bits, quantize_fp8
    vals = e4m3_values()

    def deq(t):
        q, s = quantize_fp8(bf16_bits(t), lib)
        return torch.from_numpy(vals[q] * s.astype(np.float64)[:, None])

    proj = [{k: deq(w[k]) for k in FP8_SLOTS} for w in wl.layers]
    ref, _ = torch_restatement(wl, n_steps, proj=proj, lm=deq(wl.embed))
    dec = decoder_cls(wl)
    for i in range(n_steps):
        got = dec.step(int(wl.tokens[i]), wl.shape.pos0 + i).astype(np.float64)
        rel = float(np.linalg.norm(got - ref[i]) / np.linalg.norm(ref[i]))
        assert rel < 1e-5, f"step {i}: rel L2 {rel}"


def pin_prefill_equals_decode_steps(lib_unused, wl, n, p0, decoder_cls, seed=21):
    """The oracle's prefill (layer-major over the prompt, causal attention through an explicit mask on
    the scores of every key of the prompt) against its teacher-forced decode steps: the prefill's
    definition is those steps, and with masked scores adding exact zeros the two agree bit for bit --
    logits of every token and every cache row.  A prefill that lets a token see a later key, hides its
    own row, rotates by the wrong position or writes a row to the wrong place differs."""
    s = wl.shape
    g = torch.Generator().manual_seed(seed)
    toks = [int(t) for t in torch.randint(0, s.vocab, (p0 + n,), generator=g)]
    a, b = decoder_cls(wl), decoder_cls(wl)
    for i in range(p0):
        a.step(toks[i], i)
        b.step(toks[i], i)
    steps = np.stack([a.step(toks[p0 + i], p0 + i) for i in range(n)])
    pre = b.prefill(toks[p0:p0 + n], p0)
    assert np.array_equal(steps.view(np.uint32), pre.view(np.uint32))
    assert np.array_equal(a.kv, b.kv)
