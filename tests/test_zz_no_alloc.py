"""mbk_decode_step_static: the decode step for callers that cannot allocate device memory (code
under a caller-owned pool or budget that forbids new device allocations, or inside a runtime whose
allocator must not be re-entered).  It keeps the library's working memory in a fixed device array
inside the library instead of allocating.  Here it is called through the C ABI twice in a row and
must give the same logits and cache rows as mbk_decode_step, within the parity tolerances.

This file is collected last on purpose: the static array is shared by every call in the process,
and the test must pass both alone in a fresh process and after all the other tests.
"""
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


@pytest.mark.parametrize("name", ["tiny", "smollm-135m"])
def test_static_step_matches_handle_step_twice(name):
    from parity import MAX_ABS, REL_L2
    from persistent_decode_megakernel_gb300 import mbk

    wl = workloads.generate(name, seed=0)
    s = wl.shape
    ref = mbk.Decoder(wl)  # the existing entry point (handle-based)
    kv = torch.zeros_like(ref.kv)  # the static path's own cache
    out = torch.empty(s.vocab, dtype=torch.float32, device=ref.device)
    stream = torch.cuda.current_stream().cuda_stream
    for i in range(2):  # two calls in a row
        tok = int(wl.tokens[i])
        want = ref.step(tok, i).clone()
        rc = mbk.mbk_decode_step_static(ref.cfg, ref.weights, kv.data_ptr(), tok, i, out.data_ptr(), stream)
        assert rc == mbk.MBK_OK, mbk.mbk_error_string(rc)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        exp = want.double().cpu().numpy()
        assert np.linalg.norm(got - exp) / np.linalg.norm(exp) <= REL_L2
        assert np.abs(got - exp).max() <= MAX_ABS
        assert int(np.argmax(got)) == int(np.argmax(exp))
        # same kernel and schedule: in practice the results are bitwise equal
        assert torch.equal(out, want)
        assert torch.equal(kv[:, :, :, i], ref.kv[:, :, :, i])
    ref.close()


def test_static_step_rejects_a_shape_beyond_the_array():
    from persistent_decode_megakernel_gb300 import mbk

    wl = workloads.generate("tiny", seed=0)
    ref = mbk.Decoder(wl)
    cfg = mbk.config_from_shape(wl.shape)
    # a cache long enough that its RoPE table alone (capacity * head_dim/2 * 8 bytes) exceeds 16 MiB
    cfg.kv_capacity = 80000
    out = torch.empty(wl.shape.vocab, dtype=torch.float32, device=ref.device)
    stream = torch.cuda.current_stream().cuda_stream
    rc = mbk.mbk_decode_step_static(cfg, ref.weights, ref.kv.data_ptr(), 0, 0, out.data_ptr(), stream)
    assert rc == mbk.MBK_ERR_INVALID_ARG
    torch.cuda.synchronize()
    ref.close()
