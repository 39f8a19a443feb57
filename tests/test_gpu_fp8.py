"""FP8 weight streaming (MBK_WEIGHTS_FP8): the library's E4M3 copies must be byte for byte the
oracle's (the format is a plain definition: scale = row max / 448, codes = nearest even, saturating),
and decoding on them must meet the parity bars against the oracle decoding on the same codes."""
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


def _gpu_quantize(w_bf16: torch.Tensor):
    from persistent_decode_megakernel_gb300 import mbk
    rows, cols = w_bf16.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    rc = mbk.mbk_quantize_fp8(w_bf16.data_ptr(), rows, cols, q.data_ptr(), s.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert rc == mbk.MBK_OK
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def test_quantization_matches_the_oracle_bit_for_bit():
    from oracle.oracle import bf16_bits, quantize_fp8
    rng = np.random.default_rng(4)
    mats = [torch.from_numpy(rng.standard_normal((37, 200)).astype(np.float32) * 0.05).to(torch.bfloat16),
            torch.from_numpy(rng.standard_normal((5, 1536)).astype(np.float32) * 3.0).to(torch.bfloat16)]
    z = mats[0].clone()
    z[3] = 0.0                                   # an all-zero row: scale 1, codes 0
    z[7, :] = 1e-5                               # small values beside a large one: subnormal E4M3 codes
    z[7, 0] = 1.0
    mats.append(z)
    wl = workloads.generate("smollm-135m", seed=0)
    mats += [wl.layers[0]["wq"], wl.layers[3]["w_down"], wl.embed[:512]]
    for m in mats:
        qg, sg = _gpu_quantize(m.contiguous().cuda())
        qo, so = quantize_fp8(bf16_bits(m.contiguous()))
        assert np.array_equal(sg.view(np.uint32), so.view(np.uint32))
        assert np.array_equal(qg, qo)


@pytest.mark.parametrize("name,steps", [("tiny", None), ("smollm-135m", 24), ("qwen2-0.5b", 4), ("smollm-135m-long", 8)])
def test_fp8_parity(name, steps):
    from parity import run_parity
    wl = workloads.generate(name, seed=0)
    rep = run_parity(wl, steps=steps, mode="sync", fp8=True)
    print(f"\n{name} fp8 sync: {rep}")
    print(rep.json_line().replace('"mode": "sync"', '"mode": "sync-fp8"'))
    rep.check()


def test_fp8_multi_step_and_greedy_match_single_steps():
    """The FP8 kernel's one-step, multi-step and greedy launches agree bit for bit."""
    from persistent_decode_megakernel_gb300.mbk import Decoder
    wl = workloads.generate("smollm-135m", seed=0)
    s = wl.shape
    a = Decoder(wl, fp8=True)
    b = Decoder(wl, fp8=True)
    toks = [int(x) for x in wl.tokens[:12]]
    singles = torch.stack([a.step(toks[i], i).clone() for i in range(12)])
    multi = b.steps(toks, 0)
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(singles, multi)
    assert torch.equal(a.kv, b.kv)
    tg, lg = a.greedy(toks[0], 4, 12)
    torch.cuda.synchronize()
    assert tg.cpu().tolist() == [int(np.argmax(r)) for r in lg.cpu().numpy()]
    a.close()
    b.close()


def test_fp8_with_a_paged_cache_matches_fp8_contiguous():
    """The weight format and the cache layout are independent: FP8 on a shuffled page table gives the
    FP8 contiguous results bit for bit (teacher-forced and greedy launches)."""
    from persistent_decode_megakernel_gb300.mbk import Decoder
    wl = workloads.generate("smollm-135m", seed=0)
    s = wl.shape
    n_logical = s.kv_capacity // 32
    table = np.random.default_rng(5).permutation(n_logical + 2)[:n_logical].tolist()
    a = Decoder(wl, fp8=True)
    b = Decoder(wl, fp8=True, paged=(n_logical + 2, 32, table))
    toks = [int(x) for x in wl.tokens[:20]]
    assert torch.equal(a.steps(toks, 0), b.steps(toks, 0))
    ta, la = a.greedy(toks[0], 6, 20)
    tb, lb = b.greedy(toks[0], 6, 20)
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(ta, tb) and torch.equal(la, lb)
    assert torch.equal(a.kv, b.logical_kv())
    a.close()
    b.close()
