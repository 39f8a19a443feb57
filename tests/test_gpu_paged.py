"""Paged KV cache (mbk_create_paged / mbk_set_page_table): the cache is a pool of pages, each holding
page_size consecutive positions of every layer and head, found through a page table.  A decoder on
a shuffled page table must give the logits and cache rows of a decoder on a contiguous cache, bit for
bit (same kernel, same order of operations; only the addresses differ)."""
import numpy as np
import pytest
import torch

from persistent_decode_megakernel_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from persistent_decode_megakernel_gb300 import build
    build.build()


def _workload(shape, n):
    if shape == "ragged-split":  # several context splits and a prefilled cache; crosses the split at 1024
        s = workloads.scaled_down(workloads.SHAPES["smollm-135m-long"], n_layers=3, vocab=4096, kv_capacity=1500,
                                  steps=n, pos0=1020, prefill=1020)
        return workloads.generate(s, seed=3)
    return workloads.generate(shape, seed=0)


def _table(n_logical, n_pool, seed):
    return np.random.default_rng(seed).permutation(n_pool)[:n_logical].tolist()


@pytest.mark.parametrize("shape,n,page", [("tiny", 24, 32), ("smollm-135m", 40, 32), ("ragged-split", 8, 64)])
def test_paged_cache_matches_contiguous(shape, n, page):
    from persistent_decode_megakernel_gb300.mbk import Decoder
    wl = _workload(shape, n)
    s = wl.shape
    n_logical = (s.kv_capacity + page - 1) // page
    pool = n_logical + 3  # some pool pages stay unused
    a = Decoder(wl)
    b = Decoder(wl, paged=(pool, page, _table(n_logical, pool, 1)))  # prefilled rows go through the table too
    toks = [int(x) for x in wl.tokens[:n]]
    la = a.steps(toks, s.pos0)
    lb = b.steps(toks, s.pos0)
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(la, lb)
    assert torch.equal(a.kv, b.logical_kv())
    # one-step launches and a greedy launch on the same handles continue identically
    p = s.pos0 + n
    if p + 4 <= s.kv_capacity:
        for i in range(2):
            assert torch.equal(a.step(toks[i], p + i).clone(), b.step(toks[i], p + i).clone())
        ta, ga = a.greedy(toks[2], 2, p + 2)
        tb, gb = b.greedy(toks[2], 2, p + 2)
        torch.cuda.synchronize()
        assert torch.equal(ta, tb) and torch.equal(ga, gb)
        assert torch.equal(a.kv, b.logical_kv())
    a.close()
    b.close()


def test_paged_cache_rejects_bad_tables_and_unmapped_positions():
    from persistent_decode_megakernel_gb300 import mbk
    wl = workloads.generate("tiny", seed=0)
    s = wl.shape
    stream = torch.cuda.current_stream().cuda_stream
    # page sizes: a power of two in [32, kv_capacity]
    for bad in (48, 16, 2 * s.kv_capacity):
        with pytest.raises(mbk.MbkError) as e:
            mbk.Decoder(wl, paged=(8, bad, [0]))
        assert e.value.code == mbk.MBK_ERR_INVALID_ARG
    d = mbk.Decoder(wl, paged=(6, 32, [5]))  # positions 0..31 mapped
    out = torch.empty(s.vocab, dtype=torch.float32, device=d.device)
    assert mbk.mbk_decode_step(d.handle, 1, 31, out.data_ptr(), stream) == mbk.MBK_OK
    assert mbk.mbk_decode_step(d.handle, 1, 32, out.data_ptr(), stream) == mbk.MBK_ERR_INVALID_ARG
    assert mbk.mbk_decode_steps(d.handle, [1, 2], 31, out.data_ptr(), stream) == mbk.MBK_ERR_INVALID_ARG
    assert mbk.mbk_set_page_table(d.handle, [5, 5], stream) == mbk.MBK_ERR_INVALID_ARG   # repeated
    assert mbk.mbk_set_page_table(d.handle, [5, 6], stream) == mbk.MBK_ERR_INVALID_ARG   # out of the pool
    assert mbk.mbk_set_page_table(d.handle, [0, 1, 2, 3, 4], stream) == mbk.MBK_ERR_INVALID_ARG  # > capacity / 32
    assert mbk.mbk_set_page_table(d.handle, [5, 0], stream) == mbk.MBK_OK
    assert mbk.mbk_decode_step(d.handle, 1, 32, out.data_ptr(), stream) == mbk.MBK_OK
    torch.cuda.synchronize()
    assert d.status() == 0
    c = mbk.Decoder(wl)  # a contiguous handle has no page table
    assert mbk.mbk_set_page_table(c.handle, [0], stream) == mbk.MBK_ERR_INVALID_ARG
    c.close()
    d.close()


@pytest.mark.parametrize("shape,page", [("smollm-135m", 32), ("smollm-135m-long", 64)])
def test_paged_cache_against_the_oracle(shape, page):
    """A decoder on a shuffled page table against the CPU oracle, every step from the oracle's state
    (sync mode, the bars of the contiguous parity tests): logits, argmax and every new cache row."""
    from parity import run_parity
    wl = workloads.generate(shape, seed=0)
    s = wl.shape
    n_logical = (s.kv_capacity + page - 1) // page
    table = _table(n_logical, n_logical + 5, seed=13)
    rep = run_parity(wl, mode="sync", paged=(n_logical + 5, page, table))
    print(f"\n{shape} paged sync: {rep}")
    print(rep.json_line().replace('"mode": "sync"', '"mode": "sync-paged"'))
    rep.check()
