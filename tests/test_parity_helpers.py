"""CPU tests of the comparison helpers the GPU parity tests rely on."""
import numpy as np
import torch

from parity import KvBounds, bf16_ordinal, kv_check, kv_compare, prefill_allowance


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
    assert r.ok() and r.beyond_one_ordinal == 0
    g[0, 1, 0, 2, 7] += 2                     # two ulps and no arithmetic allowance: fails
    r = kv_compare(torch.from_numpy(g.view(np.int16)).view(torch.bfloat16), ob, slice(0, 4))
    assert not r.ok() and r.violations == 1


def test_an_entry_beyond_one_ulp_passes_only_within_its_own_bound():
    o = _bits(np.array([1e-3, 1.0], dtype=np.float32))
    g = o.copy()
    g[0] += 3                                 # three ulps of 1e-3 = about 1.4e-5
    ulp = 2.0 ** (np.floor(np.log2(1e-3)) - 7)
    assert not kv_check(g, o, np.array([0.0, 0.0])).ok()
    assert not kv_check(g, o, np.array([ulp, 0.0])).ok()          # 1 + 1 ulps < 3 ulps
    r = kv_check(g, o, np.array([2.0 * ulp, 0.0]))                 # 1 + 2 ulps
    assert r.ok() and r.beyond_one_ordinal == 1 and r.worst_bound_frac <= 1.0
    g[1] += 2                                 # the other entry's allowance does not cover a 1.0-sized entry
    assert not kv_check(g, o, np.array([2.0 * ulp, 2.0 * ulp])).ok()


def test_arithmetic_allowance_is_small_for_entries_that_do_not_cancel():
    """E is the worst-case fp32 error of the entry's dot product: far below one bf16 ulp unless the
    entry is a small fraction of its terms."""
    from persistent_decode_megakernel_gb300 import workloads
    wl = workloads.generate("tiny", seed=0, steps=1)
    s = wl.shape
    x = wl.embed[int(wl.tokens[0])].to(torch.float32).numpy()
    b = KvBounds(wl)
    Ek, Ev = b.allowance(0, 5, x, None)
    from parity import _rmsnorm64
    xn = _rmsnorm64(x, wl.layers[0]["attn_norm"].to(torch.float64).numpy(), s.rms_eps)
    v = wl.layers[0]["wv"].to(torch.float64).numpy() @ xn
    assert Ev.shape == (s.n_kv_heads, s.head_dim) and Ek.shape == Ev.shape
    big = np.abs(v) > 0.1
    assert big.any() and np.all(Ev.reshape(-1)[big] < 0.5 * 2.0 ** (np.floor(np.log2(np.abs(v[big]))) - 7))
    # a layer input that differs adds ||W_i|| * ||dxn|| to every entry
    Ek2, Ev2 = b.allowance(0, 5, x, x * (1 + 1e-4))
    assert np.all(Ev2 >= Ev)


def test_prefill_allowance_covers_the_rotation_only():
    from persistent_decode_megakernel_gb300 import workloads
    shape = workloads.scaled_down(workloads.SHAPES["tiny"], prefill=8, kv_capacity=16, pos0=8, steps=1)
    wl = workloads.generate(shape, seed=0)
    E = prefill_allowance(wl)
    assert E.shape == (shape.n_layers, 2, shape.n_kv_heads, 8, shape.head_dim)
    assert np.all(E[:, 1] == 0) and np.all(E[:, 0] > 0) and E.max() < 1e-5
