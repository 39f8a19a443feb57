"""Greedy decoding on the device (mbk_decode_greedy): each step's argmax becomes the next step's
token inside one launch.  Checked against the same kernel run teacher-forced on the tokens it
chose (bit for bit), against the host argmax of its own logits, and against the CPU oracle."""
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
    if shape == "ragged-split":  # several context splits; the run crosses the split boundary at 1024
        s = workloads.scaled_down(workloads.SHAPES["smollm-135m-long"], n_layers=3, vocab=4096, kv_capacity=1500,
                                  steps=n, pos0=1020, prefill=1020)
        return workloads.generate(s, seed=3)
    return workloads.generate(shape, seed=0)


@pytest.mark.parametrize("shape,n", [("tiny", 24), ("smollm-135m", 12), ("ragged-split", 8)])
def test_greedy_matches_teacher_forced_run(shape, n):
    """The greedy launch's logits and cache rows equal those of a teacher-forced launch fed with
    the tokens the greedy launch chose, bit for bit; every chosen token is the host argmax (lowest
    index) of its step's logits."""
    from persistent_decode_megakernel_gb300.mbk import Decoder
    wl = _workload(shape, n)
    s = wl.shape
    t0 = int(wl.tokens[0])
    a = Decoder(wl)
    b = Decoder(wl)
    toks, logits = a.greedy(t0, n, s.pos0)
    torch.cuda.synchronize()
    assert a.status() == 0
    toks = toks.cpu().numpy().tolist()
    lg = logits.cpu().numpy()
    assert toks == [int(np.argmax(lg[i])) for i in range(n)]
    forced = b.steps([t0] + toks[:-1], s.pos0)
    torch.cuda.synchronize()
    assert b.status() == 0
    assert torch.equal(forced, logits)
    assert torch.equal(a.kv, b.kv)
    a.close()
    b.close()


def test_greedy_tokens_without_logits():
    """Without a logits buffer the launch chooses the same tokens."""
    from persistent_decode_megakernel_gb300.mbk import Decoder
    wl = workloads.generate("smollm-135m", seed=0)
    s = wl.shape
    a = Decoder(wl)
    b = Decoder(wl)
    ta, _ = a.greedy(int(wl.tokens[0]), 16, s.pos0)
    tb, lb = b.greedy(int(wl.tokens[0]), 16, s.pos0, want_logits=False)
    torch.cuda.synchronize()
    assert lb is None
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(ta, tb)
    assert torch.equal(a.kv, b.kv)
    a.close()
    b.close()


@pytest.mark.parametrize("shape,n", [("tiny", 16), ("smollm-135m", 64)])
def test_greedy_against_oracle(shape, n):
    """The oracle, teacher-forced on the GPU's choices (each side its own cache): the logits within
    the parity tolerances, and each chosen token is the oracle's argmax or within 1e-3 of its
    maximum (a near tie); at most one step of the run is such a near tie."""
    from oracle import OracleDecoder
    from parity import MAX_ABS, REL_L2
    from persistent_decode_megakernel_gb300.mbk import Decoder
    wl = workloads.generate(shape, seed=0)
    s = wl.shape
    d = Decoder(wl)
    toks, logits = d.greedy(int(wl.tokens[0]), n, s.pos0)
    torch.cuda.synchronize()
    assert d.status() == 0
    toks = toks.cpu().numpy().tolist()
    lg = logits.double().cpu().numpy()
    orc = OracleDecoder(wl)
    fed = [int(wl.tokens[0])] + toks[:-1]
    exact = 0
    for i in range(n):
        o = np.asarray(orc.step(fed[i], s.pos0 + i), dtype=np.float64)
        g = lg[i]
        assert np.linalg.norm(g - o) / np.linalg.norm(o) <= REL_L2
        assert np.abs(g - o).max() <= MAX_ABS
        assert o[toks[i]] >= o.max() - 1e-3
        exact += int(np.argmax(o)) == toks[i]
    assert exact >= n - 1
    d.close()


def test_greedy_rejects_bad_arguments():
    from persistent_decode_megakernel_gb300 import mbk
    wl = workloads.generate("tiny", seed=0)
    d = mbk.Decoder(wl)
    C, V = wl.shape.kv_capacity, wl.shape.vocab
    toks = torch.empty(4, dtype=torch.int32, device=d.device)
    stream = torch.cuda.current_stream().cuda_stream
    g = mbk.mbk_decode_greedy
    assert g(d.handle, 1, 4, 0, 0, 0, stream) == mbk.MBK_ERR_INVALID_ARG         # no token buffer
    assert g(d.handle, 1, 0, 0, toks.data_ptr(), 0, stream) == mbk.MBK_ERR_INVALID_ARG
    assert g(d.handle, V, 4, 0, toks.data_ptr(), 0, stream) == mbk.MBK_ERR_INVALID_ARG
    assert g(d.handle, -1, 4, 0, toks.data_ptr(), 0, stream) == mbk.MBK_ERR_INVALID_ARG
    assert g(d.handle, 1, 4, C - 3, toks.data_ptr(), 0, stream) == mbk.MBK_ERR_INVALID_ARG
    assert g(d.handle, 1, 4, -1, toks.data_ptr(), 0, stream) == mbk.MBK_ERR_INVALID_ARG
    assert g(d.handle, 1, 4, C - 4, toks.data_ptr(), 0, stream) == mbk.MBK_OK
    torch.cuda.synchronize()
    assert d.status() == 0
    d.close()
