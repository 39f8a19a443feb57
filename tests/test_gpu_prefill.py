"""Prefill (mbk_prefill) against the oracle.  The prefill's plain definition is teacher-forced decode
steps at positions p0 .. p0 + n - 1, so the oracle's decode steps are its reference.

"layers" mode: the residual stream entering every layer l >= 1 is the oracle's
(mbk_debug_prefill_inject), so every K/V row of every layer comes from identical inputs and must be
within one bf16 ulp entry by entry (the rule of the decode parity tests, tests/parity.py, with the
2^-17 relative error of the GEMM input's bf16 high/low pair added to the arithmetic allowance).
Unlike a decode step, a prefill's tokens attend to rows written earlier in the same call, so a
legitimate one-ulp choice of one row moves later tokens' attention by ~1e-4 relative: the logits are
held to relative L2 <= 2e-3 and max-abs <= 5e-2, and every argmax disagreement must be a near tie
of the oracle.  "e2e" mode: nothing injected; the benchmark spec's logits bars (relative L2 <= 1e-2,
max-abs <= 5e-2), and an argmax disagreement only where the oracle's gap is within twice that token's
own measured logit error.  The GEMM inputs' bf16 high/low pair (2^-17
relative) flips more bf16 K/V roundings than the decode's fp32 GEMV does, and at the first
positions attention passes a flipped V entry straight on: end to end the 135M shape's first token
is measured at 3.2e-3 relative, its last at 6e-4."""
import numpy as np
import pytest
import torch

from persistent_decode_megakernel_gb300 import workloads

pytestmark = pytest.mark.gpu

import parity  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from persistent_decode_megakernel_gb300 import build
    build.build()


def _tokens(wl, count, seed=11):
    if len(wl.tokens) >= count:
        return [int(t) for t in wl.tokens[:count]]
    g = torch.Generator().manual_seed(seed)
    return [int(t) for t in torch.randint(0, wl.shape.vocab, (count,), generator=g)]


def _copy_rows(dec, orc_kv, rows: slice):
    src = torch.from_numpy(np.ascontiguousarray(orc_kv[:, :, :, rows]).view(np.int16)).view(torch.bfloat16)
    dec.kv[:, :, :, rows] = src.to(dec.device)


def run(wl, n, p0, mode, logits="all", paged=None):
    from oracle import OracleDecoder
    from persistent_decode_megakernel_gb300 import mbk
    from persistent_decode_megakernel_gb300.mbk import Decoder

    s = wl.shape
    dec = Decoder(wl, paged=paged)
    orc = OracleDecoder(wl)
    toks = _tokens(wl, p0 + n)
    for i in range(s.prefill, p0):  # history rows the workload does not prefill
        orc.step(toks[i], i)
    if p0 > 0:
        assert paged is None, "history rows are copied into a contiguous cache"
        _copy_rows(dec, orc.kv, slice(0, p0))
    outs = [orc.step(toks[p0 + i], p0 + i, taps=True) for i in range(n)]
    ref = np.stack([o[0] for o in outs]).astype(np.float64)
    if mode == "layers":
        inject = np.stack([np.stack([o[1][2 * l] for o in outs]) for l in range(s.n_layers)])
        assert mbk.mbk_debug_prefill_inject(dec.handle, inject, n) == mbk.MBK_OK
    got = dec.prefill(toks[p0:p0 + n], p0, logits=logits)
    torch.cuda.synchronize()
    assert dec.status() == 0
    if logits == "last":
        ref = ref[-1:]
        got = got[None, :]
    got = got.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    mx = np.abs(got - ref).max()
    gi, oi = got.argmax(1), ref.argmax(1)
    tok_err = np.abs(got - ref).max(axis=1)
    # (oracle gap, that token's max-abs logit error) of every argmax disagreement
    flips = [(float(ref[r, oi[r]] - ref[r, gi[r]]), float(tok_err[r])) for r in range(len(gi)) if gi[r] != oi[r]]
    gkv = dec.kv if paged is None else dec.logical_kv()
    g_bits = gkv.view(torch.int16).cpu().numpy().view(np.uint16)
    kv = parity.KvCompare(0, 0, 0, 0.0, 0.0)
    if mode == "layers":
        bounds = parity.KvBounds(wl)
        for i in range(n):
            tok, pos = toks[p0 + i], p0 + i
            for l in range(s.n_layers):
                x = wl.embed[tok].to(torch.float32).numpy() if l == 0 else outs[i][1][2 * l]
                Ek, Ev = bounds.allowance(l, pos, x, None, input_rel=2.0 ** -17)
                kv = kv.merged(parity.kv_check(g_bits[l, 0, :, pos], orc.kv[l, 0, :, pos], Ek))
                kv = kv.merged(parity.kv_check(g_bits[l, 1, :, pos], orc.kv[l, 1, :, pos], Ev))
    dec.close()
    print(f"\nprefill n={n} p0={p0} {mode}: rel {rel.max():.2e} max-abs {mx:.2e} argmax flips {flips} kv {kv}")
    # layers mode: every layer from the oracle's input; end to end: the benchmark spec's own bars (the
    # bf16 high/low pair of every GEMM input, 2^-17 relative, flips more K/V roundings than the
    # decode's fp32 GEMV, and at the first positions attention passes a flipped V entry straight on)
    assert rel.max() <= (parity.REL_L2_TIGHT if mode == "layers" else parity.REL_L2) and mx <= parity.MAX_ABS
    # a flip is a near tie of the oracle (layers mode), or end to end within the token's own measured
    # logit error (which the bars above bound): GPU logits within e of the oracle's can swap two
    # candidates at most 2e apart, and nothing further apart
    if mode == "layers":
        assert all(gap <= parity.NEAR_TIE for gap, _ in flips), flips
    else:
        assert all(gap <= 2.0 * err for gap, err in flips), flips
    if mode == "layers":
        assert kv.ok(), kv
    return got


FULL = [("tiny", 128, 0), ("smollm-135m", 128, 0), ("qwen2-0.5b", 128, 0), ("smollm-135m-long", 64, 4096),
        ("smollm-1.7b", 64, 0)]


@pytest.mark.parametrize("name,n,p0", FULL)
@pytest.mark.parametrize("mode", ["layers", "e2e"])
def test_prefill_matches_decode_steps(name, n, p0, mode):
    run(workloads.generate(name, seed=0), n, p0, mode)


def test_prefill_ragged_tiles_after_history():
    """Two token tiles (150 = 128 + 22), after 21 cached positions."""
    s = workloads.scaled_down(workloads.SHAPES["tiny"], kv_capacity=256)
    run(workloads.generate(s, seed=3), 150, 21, "layers")


def test_prefill_paged_cache():
    s = workloads.scaled_down(workloads.SHAPES["tiny"], kv_capacity=256)
    n_logical = 256 // 32
    table = np.random.default_rng(1).permutation(n_logical + 3)[:n_logical].tolist()
    run(workloads.generate(s, seed=5), 100, 0, "layers", paged=(n_logical + 3, 32, table))


def test_prefill_last_logits_equal_the_last_row():
    s = workloads.scaled_down(workloads.SHAPES["tiny"], kv_capacity=256)
    wl = workloads.generate(s, seed=4)
    a = run(wl, 40, 0, "e2e", logits="all")
    b = run(wl, 40, 0, "e2e", logits="last")
    assert np.allclose(a[-1], b[0], rtol=0, atol=1e-6)


def test_prefill_head_dim_128_and_mqa():
    s = workloads.DecoderShape("mha128", 2, 512, 1024, 4, 2, 128, 2048, 160, 1e-5, 1e4, False, steps=12)
    run(workloads.generate(s, seed=7), 70, 5, "layers")
    s = workloads.DecoderShape("mqa", 2, 1024, 2048, 16, 1, 64, 2048, 128, 1e-5, 1e4, False, steps=12)
    run(workloads.generate(s, seed=8), 100, 0, "layers")


def test_prefill_then_decode_continues():
    """A prompt by prefill, then teacher-forced decode steps on the same cache: the steps' logits meet
    the end-to-end bars against the oracle's uninterrupted decode."""
    from oracle import OracleDecoder
    from persistent_decode_megakernel_gb300.mbk import Decoder
    wl = workloads.generate("smollm-135m", seed=0)
    s = wl.shape
    toks = _tokens(wl, 128)
    dec = Decoder(wl)
    dec.prefill(toks[:100], 0, logits=None)
    got = dec.steps(toks[100:], 100).cpu().numpy().astype(np.float64)
    assert dec.status() == 0
    orc = OracleDecoder(wl)
    for i in range(100):
        orc.step(toks[i], i)
    for i in range(28):
        ref = orc.step(toks[100 + i], 100 + i).astype(np.float64)
        assert np.linalg.norm(got[i] - ref) / np.linalg.norm(ref) <= parity.REL_L2
    dec.close()


def test_prefill_rejects_bad_arguments():
    from persistent_decode_megakernel_gb300 import mbk
    wl = workloads.generate("tiny", seed=0)
    s = wl.shape
    d = mbk.Decoder(wl)
    out = torch.empty(s.vocab, dtype=torch.float32, device=d.device)
    st = torch.cuda.current_stream().cuda_stream
    E = mbk.MBK_ERR_INVALID_ARG
    assert mbk.mbk_prefill(d.handle, [], 0, out.data_ptr(), 1, st) == E
    assert mbk.mbk_prefill(d.handle, [1, 2], s.kv_capacity - 1, out.data_ptr(), 1, st) == E
    assert mbk.mbk_prefill(d.handle, [s.vocab], 0, out.data_ptr(), 1, st) == E
    assert mbk.mbk_prefill(d.handle, [1], 0, out.data_ptr(), 3, st) == E
    assert mbk.mbk_prefill(d.handle, [1], 0, 0, 1, st) == E
    assert mbk.mbk_debug_prefill_inject(d.handle, np.zeros((s.n_layers, 2, s.hidden), np.float32), 2) == mbk.MBK_OK
    assert mbk.mbk_prefill(d.handle, [1, 2, 3], 0, out.data_ptr(), 1, st) == E   # armed for 2 tokens
    assert mbk.mbk_debug_prefill_inject(d.handle, None, 0) == mbk.MBK_OK
    assert mbk.mbk_prefill(d.handle, [1, 2, 3], 0, 0, 0, st) == mbk.MBK_OK       # cache only
    torch.cuda.synchronize()
    assert d.status() == 0
    d.close()
    f = mbk.Decoder(wl, fp8=True)
    assert mbk.mbk_prefill(f.handle, [1], 0, out.data_ptr(), 1, st) == mbk.MBK_ERR_UNSUPPORTED
    f.close()


def test_batch_step_matches_each_sequence():
    """Three sequences of one paged pool in one step (a prompt chunk after history, one decode token, a
    prompt from position 0), each against its own oracle decoder; layer inputs injected per token."""
    from oracle import OracleDecoder
    from persistent_decode_megakernel_gb300 import mbk
    from persistent_decode_megakernel_gb300.mbk import Decoder
    s = workloads.scaled_down(workloads.SHAPES["tiny"], kv_capacity=256)
    wl = workloads.generate(s, seed=9)
    ps, max_pages = 32, 256 // 32
    npool = 3 * max_pages + 2
    perm = np.random.default_rng(4).permutation(npool)
    tables = [perm[i * max_pages:(i + 1) * max_pages].tolist() for i in range(3)]
    dec = Decoder(wl, paged=(npool, ps, tables[0]))
    g = torch.Generator().manual_seed(3)
    toks = [[int(x) for x in torch.randint(0, s.vocab, (n,), generator=g)] for n in (50, 41, 20)]
    plan = [(30, 20), (40, 1), (0, 20)]
    orcs = [OracleDecoder(wl) for _ in range(3)]
    refs, taps = [], []
    pool = dec.pool
    for q, (start, cnt) in enumerate(plan):
        for i in range(start):
            orcs[q].step(toks[q][i], i)
        hist = torch.from_numpy(orcs[q].kv.view(np.int16)).view(torch.bfloat16)
        for p in range(start):  # history rows through the sequence's table
            pool[tables[q][p // ps], :, :, :, p % ps] = hist[:, :, :, p].to(dec.device)
        outs = [orcs[q].step(toks[q][start + i], start + i, taps=True) for i in range(cnt)]
        refs.append(np.stack([o[0] for o in outs]))
        taps.extend(o[1] for o in outs)
    inject = np.stack([np.stack([tp[2 * l] for tp in taps]) for l in range(s.n_layers)])
    assert mbk.mbk_debug_prefill_inject(dec.handle, inject, len(taps)) == mbk.MBK_OK
    got = dec.batch_step([(st, toks[q][st:st + c]) for q, (st, c) in enumerate(plan)], tables, logits="all")
    torch.cuda.synchronize()
    assert dec.status() == 0
    got = got.cpu().numpy().astype(np.float64)
    ref = np.concatenate(refs).astype(np.float64)
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() <= parity.REL_L2_TIGHT and (got.argmax(1) == ref.argmax(1)).all()
    bounds = parity.KvBounds(wl)
    t = 0
    for q, (start, cnt) in enumerate(plan):
        for i in range(cnt):
            pos = start + i
            g_rows = pool[tables[q][pos // ps], :, :, :, pos % ps].view(torch.int16).cpu().numpy().view(np.uint16)
            for l in range(s.n_layers):
                x = wl.embed[toks[q][pos]].to(torch.float32).numpy() if l == 0 else taps[t][2 * l]
                Ek, Ev = bounds.allowance(l, pos, x, None, input_rel=2.0 ** -17)
                assert parity.kv_check(g_rows[l, 0], orcs[q].kv[l, 0, :, pos], Ek).ok(), (q, pos, l)
                assert parity.kv_check(g_rows[l, 1], orcs[q].kv[l, 1, :, pos], Ev).ok(), (q, pos, l)
            t += 1
    dec.close()
