"""The oracle's prefill: n given tokens at positions p0 .. p0 + n - 1 computed layer by layer with an
explicit causal mask equal, bit for bit, the oracle's teacher-forced decode steps over the same tokens --
the plain definition of prefill, which the GPU prefill is compared against."""
import pytest

import oracle_pins as pins
from oracle import OracleDecoder
from persistent_decode_megakernel_gb300 import workloads


@pytest.mark.parametrize("n,p0", [(1, 0), (17, 0), (9, 30)])
def test_prefill_equals_decode_steps_tiny(n, p0):
    pins.pin_prefill_equals_decode_steps(None, workloads.generate("tiny", seed=0), n, p0, OracleDecoder)


def test_prefill_equals_decode_steps_with_bias_and_gains():
    s = workloads.scaled_down(workloads.SHAPES["qwen2-0.5b"], n_layers=2, hidden=128, intermediate=320, n_heads=6,
                              n_kv_heads=2, vocab=512, kv_capacity=64, steps=4)
    pins.pin_prefill_equals_decode_steps(None, workloads.generate(s, seed=3, random_gains=True), 20, 7, OracleDecoder)


def test_prefill_rejects_positions_outside_the_cache():
    wl = workloads.generate("tiny", seed=0)
    d = OracleDecoder(wl)
    with pytest.raises(ValueError):
        d.prefill([1, 2, 3], wl.shape.kv_capacity - 2)
    with pytest.raises(ValueError):
        d.prefill([wl.shape.vocab], 0)
