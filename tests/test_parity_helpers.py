"""CPU tests of the comparison helpers the GPU parity tests rely on."""
import numpy as np
import torch

from parity import bf16_ordinal, kv_compare


def _bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_ordinal_is_monotone_and_signed_zero_equal():
    vals = np.array([-3.0, -1.0, -1e-30, -0.0, 0.0, 1e-30, 1.0, 3.0], dtype=np.float32)
    o = bf16_ordinal(_bits(vals))
    assert np.all(np.diff(o) >= 0)
    assert o[3] == o[4] == 0


def test_kv_compare_one_ulp_passes_two_ulps_fail():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((1, 2, 1, 4, 64)).astype(np.float32)
    ob = _bits(x).reshape(x.shape)
    g = ob.copy()
    g[0, 0, 0, 1, 5] += 1                     # one ulp: fine
    r = kv_compare(torch.from_numpy(g.view(np.int16)).view(torch.bfloat16), ob, slice(0, 4))
    assert r.ok() and r.strict_violations == 0
    g[0, 1, 0, 2, 7] += 2                     # two ulps on a normal-sized entry: fails
    r = kv_compare(torch.from_numpy(g.view(np.int16)).view(torch.bfloat16), ob, slice(0, 4))
    assert not r.ok()


def test_kv_compare_tiny_entry_uses_row_scale():
    x = np.ones((1, 2, 1, 1, 64), dtype=np.float32)
    x[0, 0, 0, 0, 3] = 1e-5                   # cancels to almost nothing
    ob = _bits(x).reshape(x.shape)
    g = ob.copy()
    g[0, 0, 0, 0, 3] += 3                     # three ulps of 1e-5 is far below 1/128 of the row max
    r = kv_compare(torch.from_numpy(g.view(np.int16)).view(torch.bfloat16), ob, slice(0, 1))
    assert r.worst_scaled_ulps < 1.0 and r.strict_violations == 1
