"""CPU tests of the oracle: its pins (closed forms, invariants, brute force, library routines,
the pages' printed numbers) and its self-consistency.  No GPU needed."""
import json
import os

import numpy as np
import pytest
import torch

import oracle_pins as pins
from oracle import OracleDecoder
from persistent_decode_megakernel_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_rounding(oracle_lib):
    pins.pin_bf16_rounding(oracle_lib)


def test_rmsnorm(oracle_lib):
    pins.pin_rmsnorm(oracle_lib)


def test_gemv(oracle_lib):
    pins.pin_gemv(oracle_lib)


def test_rope(oracle_lib):
    pins.pin_rope(oracle_lib)


def test_attention(oracle_lib):
    pins.pin_attention(oracle_lib)


def test_silu_mul(oracle_lib):
    pins.pin_silu_mul(oracle_lib)


@pytest.fixture(scope="module")
def tiny():
    return workloads.generate("tiny", seed=0)


@pytest.fixture(scope="module")
def tiny_gains():
    return workloads.generate("tiny", seed=1, random_gains=True)


def test_decoder_matches_torch_restatement(oracle_lib, tiny):
    pins.pin_decoder_vs_torch(oracle_lib, tiny, 32, OracleDecoder)


def test_decoder_matches_torch_restatement_with_gains(oracle_lib, tiny_gains):
    pins.pin_decoder_vs_torch(oracle_lib, tiny_gains, 12, OracleDecoder)


def test_decoder_with_bias_and_theta(oracle_lib):
    shape = workloads.scaled_down(workloads.SHAPES["qwen2-0.5b"], n_layers=2, hidden=128, intermediate=320,
                                  n_heads=6, n_kv_heads=2, vocab=512, kv_capacity=32, steps=8)
    wl = workloads.generate(shape, seed=3)
    pins.pin_decoder_vs_torch(oracle_lib, wl, 8, OracleDecoder)


def test_long_context_prefill_matches_restatement(oracle_lib):
    """A prefilled cache (K rotated by its row's position) followed by decode steps."""
    shape = workloads.scaled_down(workloads.SHAPES["smollm-135m-long"], n_layers=2, hidden=128, intermediate=256,
                                  n_heads=4, n_kv_heads=2, vocab=256, kv_capacity=96, prefill=70, pos0=70, steps=4)
    wl = workloads.generate(shape, seed=4)
    dec = OracleDecoder(wl)
    # the cache rows from K_raw: V is the bf16 cast; K at row 0 is unrotated
    vr = wl.v_raw.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kr = wl.k_raw.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(dec.kv[:, 1, :, :70], vr)
    assert np.array_equal(dec.kv[:, 0, :, 0], kr[:, :, 0])
    # rotation preserves each pair's norm (up to bf16 rounding)
    k = (dec.kv[:, 0, :, :70].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raw = wl.k_raw.numpy().astype(np.float64)
    n_k = k[..., :32] ** 2 + k[..., 32:] ** 2
    n_r = raw[..., :32] ** 2 + raw[..., 32:] ** 2
    assert np.allclose(n_k, n_r, rtol=2e-2, atol=1e-3)
    # then the decode steps agree with the restatement run on the same prefilled cache
    ref_logits, _ = pins.torch_restatement(wl, 4, kv_init=dec.kv.copy())
    for i in range(4):
        got = dec.step(int(wl.tokens[i]), 70 + i)
        rel = float(np.linalg.norm(got.astype(np.float64) - ref_logits[i]) / np.linalg.norm(ref_logits[i]))
        assert rel < 1e-5


def test_step_writes_only_its_cache_row(tiny):
    dec = OracleDecoder(tiny)
    dec.step(int(tiny.tokens[0]), 5)
    nz = np.argwhere(dec.kv != 0)
    assert set(nz[:, 3].tolist()) == {5}


def test_cache_resume_is_identical(tiny):
    """Running k steps, copying the cache into a fresh decoder and continuing gives bitwise the
    same logits as an uninterrupted run (the library keeps no state besides the cache)."""
    a = OracleDecoder(tiny)
    full = [a.step(int(tiny.tokens[i]), i) for i in range(12)]
    b = OracleDecoder(tiny)
    for i in range(7):
        b.step(int(tiny.tokens[i]), i)
    c = OracleDecoder(tiny)
    c.kv[...] = b.kv
    for i in range(7, 12):
        assert np.array_equal(c.step(int(tiny.tokens[i]), i), full[i])


def test_thread_count_does_not_change_results(tiny):
    a = OracleDecoder(tiny, nthreads=1)
    b = OracleDecoder(tiny, nthreads=3)
    for i in range(4):
        assert np.array_equal(a.step(int(tiny.tokens[i]), i), b.step(int(tiny.tokens[i]), i))
    assert np.array_equal(a.kv, b.kv)


def test_taps_bracket_the_layers(tiny):
    dec = OracleDecoder(tiny)
    logits, taps = dec.step(int(tiny.tokens[0]), 0, taps=True)
    emb = (tiny.embed[int(tiny.tokens[0])].float()).numpy()
    assert np.array_equal(taps[0], emb)
    assert taps.shape == (2 * tiny.shape.n_layers + 1, tiny.shape.hidden)
    assert np.all(np.isfinite(taps)) and np.all(np.isfinite(logits))


def test_rejects_bad_token_and_position(tiny):
    dec = OracleDecoder(tiny)
    with pytest.raises(ValueError):
        dec.step(tiny.shape.vocab, 0)
    with pytest.raises(ValueError):
        dec.step(0, tiny.shape.kv_capacity)
    with pytest.raises(ValueError):
        dec.step(-1, 0)


def test_smollm135m_parameter_count_matches_page():
    g = json.load(open(os.path.join(GOLDEN, "smollm135m_shape.json")))
    s = workloads.SHAPES["smollm-135m"]
    for k, v in g["shape"].items():
        assert getattr(s, k) == v
    assert s.param_count() == g["param_count"]
    assert round(s.param_count() * 2 / 1e6) == g["weight_megabytes_per_token_approx"]
    assert abs(s.param_count() * 2 / 2.2e12 * 1e3 - g["floor_ms_at_2p2_tbps_approx"]) < 0.005
    # the page's barrier arithmetic: (intervals per layer) * layers + 3
    assert g["intervals_per_layer_folded"] * s.n_layers + 3 == g["barriers_folded"]
    assert g["intervals_per_layer_unfolded"] * s.n_layers + 3 == g["barriers_unfolded"]


def test_workload_generation_is_seeded():
    a = workloads.generate("tiny", seed=0)
    b = workloads.generate("tiny", seed=0)
    c = workloads.generate("tiny", seed=1)
    assert torch.equal(a.embed, b.embed) and torch.equal(a.tokens, b.tokens)
    assert not torch.equal(a.embed, c.embed)
    assert a.layers[0]["bq"] is None
    assert float(a.embed.float().std()) == pytest.approx(0.02, rel=0.05)
    assert torch.all(a.layers[0]["attn_norm"].float() == 1.0)
