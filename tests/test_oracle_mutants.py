"""Planted mistakes in the oracle (on the CPU only): each mutant is a copy of mbk_oracle.c with one
plausible bug -- a dropped term, a wrong sign or index, a transposed operand -- and the pins of
oracle_pins.py must reject every one of them.  This shows the pins constrain each part of the
oracle, not just its overall shape."""
import ctypes
import os
import subprocess

import pytest

import oracle_pins as pins
from oracle import OracleDecoder
from oracle.oracle import GCC_FLAGS, bind
from persistent_decode_megakernel_gb300 import workloads

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "mbk_oracle.c")

# (name, text to find, replacement, occurrence index or None for "exactly one occurrence")
MUTANTS = [
    ("rope_sign", "x[i] = (float)(a * c - b * s);", "x[i] = (float)(a * c + b * s);", None),
    ("rope_frequency", "-(2.0 * (double)i) / (double)d", "-(1.0 * (double)i) / (double)d", None),
    ("rope_pairing", "double a = x[i], b = x[i + half];", "double a = x[i], b = x[half - 1 - i];", None),
    ("attn_scale_dropped", "s[j] = acc * scale;", "s[j] = acc;", None),
    ("gqa_mapping", "int kv = h / group;", "int kv = h % nkv;", None),
    ("attn_reads_k_as_v", "acc += s[j] * (double)orc_bf16_to_f32(Vh[(size_t)j * d + t]);",
     "acc += s[j] * (double)orc_bf16_to_f32(Kh[(size_t)j * d + t]);", None),
    ("attn_excludes_current_row", "orc_attention(q, Kc, Vc, nq, nkv, d, cap, pos + 1, o, nthreads);",
     "orc_attention(q, Kc, Vc, nq, nkv, d, cap, pos > 0 ? pos : 1, o, nthreads);", None),
    ("rms_eps_dropped", "sqrt(ss / (double)n + eps)", "sqrt(ss / (double)n + 100.0 * eps)", None),
    ("rms_sum_not_mean", "sqrt(ss / (double)n + eps)", "sqrt(ss + eps)", None),
    ("rms_gain_dropped", "double gi = g ? (double)orc_bf16_to_f32(g[i]) : 1.0;", "double gi = 1.0;", None),
    ("gemv_transposed", "acc += (double)orc_bf16_to_f32(w[k]) * (double)x[k];",
     "acc += (double)orc_bf16_to_f32(W[(size_t)k * rows + r]) * (double)x[k];", None),
    ("bias_dropped", "if (b) acc += (double)orc_bf16_to_f32(b[r]);", "(void)b;", None),
    ("attn_residual_dropped", "for (int i = 0; i < H; ++i) x[i] = (float)((double)x[i] + (double)y[i]);",
     "for (int i = 0; i < H; ++i) x[i] = y[i];", 0),
    ("mlp_residual_dropped", "for (int i = 0; i < H; ++i) x[i] = (float)((double)x[i] + (double)y[i]);",
     "for (int i = 0; i < H; ++i) x[i] = y[i];", 1),
    ("silu_is_sigmoid", "double silu = z / (1.0 + exp(-z));", "double silu = 1.0 / (1.0 + exp(-z));", None),
    ("gate_up_swapped", "orc_silu_mul(g, u, I, hbuf);", "orc_silu_mul(u, g, I, hbuf);", None),
    ("bf16_truncates", "u += 0x7fffu + lsb;", "u += 0u * lsb;", None),
    ("k_cached_unrotated", "orc_rope(k, nkv, d, pos, cfg->rope_theta);", "(void)0;", None),
    ("final_norm_gain_dropped", "orc_rmsnorm(x, final_norm, H, cfg->rms_eps, xn);", "orc_rmsnorm(x, NULL, H, cfg->rms_eps, xn);", None),
    ("v_row_from_k", "Vc[((size_t)h * cap + pos) * d + t] = orc_f32_to_bf16(v[(size_t)h * d + t]);",
     "Vc[((size_t)h * cap + pos) * d + t] = orc_f32_to_bf16(k[(size_t)h * d + t]);", None),
    # the prefill's own code (layer-major, explicit causal mask)
    ("prefill_not_causal", "if (j > p0 + t) {", "if (j > p0 + n - 1) {", None),
    ("prefill_mask_one_ahead", "if (j > p0 + t) {", "if (j > p0 + t + 1) {", None),
    ("prefill_q_rotated_by_token_index", "orc_rope(qt, nq, d, pos, cfg->rope_theta);",
     "orc_rope(qt, nq, d, t, cfg->rope_theta);", None),
    ("prefill_row_at_token_index", "Kc[((size_t)h * cap + pos) * d + i] = orc_f32_to_bf16(kr[(size_t)h * d + i]);",
     "Kc[((size_t)h * cap + t) * d + i] = orc_f32_to_bf16(kr[(size_t)h * d + i]);", None),
]


def _mutate(src: str, find: str, repl: str, occ):
    n = src.count(find)
    if occ is None:
        assert n == 1, f"mutation site must be unique, found {n}"
        return src.replace(find, repl)
    assert n > occ
    idx = -1
    for _ in range(occ + 1):
        idx = src.index(find, idx + 1)
    return src[:idx] + repl + src[idx + len(find):]


def _build(tmp_path, name, text):
    c = tmp_path / f"{name}.c"
    c.write_text(text)
    hdr_dir = os.path.dirname(SRC)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc"] + GCC_FLAGS + ["-I", hdr_dir, "-o", str(so), str(c), "-lm"], check=True)
    return bind(ctypes.CDLL(str(so)))


@pytest.fixture(scope="module")
def decoders():
    tiny = workloads.generate("tiny", seed=0)
    gains = workloads.generate("tiny", seed=1, random_gains=True)
    bias = workloads.generate(workloads.scaled_down(workloads.SHAPES["qwen2-0.5b"], n_layers=2, hidden=128,
                                                    intermediate=320, n_heads=6, n_kv_heads=2, vocab=512,
                                                    kv_capacity=32, steps=4), seed=3)
    return tiny, gains, bias


def _all_pins(lib, decoders):
    tiny, gains, bias = decoders
    checks = [
        lambda: pins.pin_bf16_rounding(lib), lambda: pins.pin_rmsnorm(lib), lambda: pins.pin_gemv(lib),
        lambda: pins.pin_rope(lib), lambda: pins.pin_attention(lib), lambda: pins.pin_silu_mul(lib),
        lambda: pins.pin_decoder_vs_torch(lib, tiny, 4, lambda wl: OracleDecoder(wl, lib=lib)),
        lambda: pins.pin_decoder_vs_torch(lib, gains, 3, lambda wl: OracleDecoder(wl, lib=lib)),
        lambda: pins.pin_decoder_vs_torch(lib, bias, 3, lambda wl: OracleDecoder(wl, lib=lib)),
        lambda: pins.pin_prefill_equals_decode_steps(lib, tiny, 12, 5, lambda wl: OracleDecoder(wl, lib=lib)),
    ]
    failed = []
    for i, chk in enumerate(checks):
        try:
            chk()
        except AssertionError:
            failed.append(i)
    return failed


def test_unmutated_copy_passes_every_pin(tmp_path, decoders):
    lib = _build(tmp_path, "clean", open(SRC).read())
    assert _all_pins(lib, decoders) == []


@pytest.mark.parametrize("name,find,repl,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, decoders, name, find, repl, occ):
    lib = _build(tmp_path, name, _mutate(open(SRC).read(), find, repl, occ))
    assert _all_pins(lib, decoders), f"mutant {name} passed every pin"


# Planted mistakes in the FP8 weight format; the FP8 pins must reject each one.
FP8_MUTANTS = [
    ("fp8_truncates", "if (a - vlo < vhi - a) c = lo;", "if (1) c = lo;", None),
    ("fp8_ties_down", "else c = (lo % 2 == 0) ? lo : lo + 1;", "else c = lo;", None),
    ("fp8_scale_not_applied", "acc *= (double)s[r];", "acc *= 1.0;", None),
    ("fp8_scale_range", "const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "const float sc = amax > 0.0f ? amax / 240.0f : 1.0f;", None),
    ("fp8_k_uses_v_codes", "project(w->wk, f8, 1,", "project(w->wk, f8, 2,", None),
    ("fp8_lm_head_bf16", "  if (fp8)\n    orc_gemv_fp8(fp8->lm_q", "  if (0)\n    orc_gemv_fp8(fp8->lm_q", None),
    ("fp8_subnormal_scale", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);", None),
    ("fp8_bias_scaled", "    acc *= (double)s[r];\n    if (b != NULL) acc += (double)orc_bf16_to_f32(b[r]);",
     "    if (b != NULL) acc += (double)orc_bf16_to_f32(b[r]);\n    acc *= (double)s[r];", None),
]


def _fp8_pins(lib):
    tiny = workloads.generate("tiny", seed=0)
    bias = workloads.generate(workloads.scaled_down(workloads.SHAPES["qwen2-0.5b"], n_layers=2, hidden=128,
                                                    intermediate=320, n_heads=6, n_kv_heads=2, vocab=512,
                                                    kv_capacity=32, steps=4), seed=3)
    checks = [
        lambda: pins.pin_fp8_codes(lib),
        lambda: pins.pin_fp8_quantize_and_gemv(lib, tiny),
        lambda: pins.pin_fp8_decoder_vs_torch(lib, tiny, 3, lambda wl: OracleDecoder(wl, lib=lib, fp8=True)),
        lambda: pins.pin_fp8_decoder_vs_torch(lib, bias, 2, lambda wl: OracleDecoder(wl, lib=lib, fp8=True)),
    ]
    failed = []
    for i, chk in enumerate(checks):
        try:
            chk()
        except AssertionError:
            failed.append(i)
    return failed


def test_unmutated_copy_passes_every_fp8_pin(tmp_path):
    lib = _build(tmp_path, "clean8", open(SRC).read())
    assert _fp8_pins(lib) == []


@pytest.mark.parametrize("name,find,repl,occ", FP8_MUTANTS, ids=[m[0] for m in FP8_MUTANTS])
def test_fp8_mutant_is_caught(tmp_path, name, find, repl, occ):
    lib = _build(tmp_path, name, _mutate(open(SRC).read(), find, repl, occ))
    assert _fp8_pins(lib), f"mutant {name} passed every FP8 pin"
