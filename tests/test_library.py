"""CPU tests of the C-ABI library: it loads without a GPU, exports every symbol include/mbk.h
declares, and its host-side scheduler builds and checks plans for every decoder shape."""
import ctypes
import os
import re

import pytest

from persistent_decode_megakernel_gb300 import build as mbk_build
from persistent_decode_megakernel_gb300 import mbk, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbk_build.build()
    return mbk.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mbk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mbk_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for f in ("mbk_create", "mbk_decode_step", "mbk_destroy", "mbk_get_status", "mbk_error_string", "mbk_kv_fill"):
        assert f in names
    assert set(names) == set(mbk.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert mbk.mbk_error_string(code)
    assert mbk.mbk_error_string(-1) == "invalid argument"
    assert mbk.mbk_error_string(12345) == "unknown error"


@pytest.mark.parametrize("name", list(workloads.SHAPES))
@pytest.mark.parametrize("num_sms", [152, 148, 132, 7, 1])
def test_plan_builds_and_checks(lib, name, num_sms):
    s = workloads.SHAPES[name]
    info = mbk.mbk_plan_check(mbk.config_from_shape(s), num_sms)
    assert info.num_ctas == num_sms
    assert info.stage_bytes == 16384
    assert 2 <= info.num_stages <= 32
    assert info.smem_bytes <= 232448
    # every weight byte streamed exactly once per step (the check inside verifies rows; here: bytes)
    H, I, d = s.hidden, s.intermediate, s.head_dim
    qd, kvd = s.n_heads * d, s.n_kv_heads * d
    layer = (qd * H + 2 * kvd * H + H * qd + 3 * H * I) * 2
    assert info.weight_bytes == s.n_layers * layer + s.vocab * H * 2
    assert info.max_cta_bytes * num_sms >= info.weight_bytes
    if name == "smollm-135m-long":
        assert info.attn_splits == s.kv_capacity // 512
    else:
        assert info.attn_splits == 1


@pytest.mark.parametrize("shape,mma", [("tiny", 1), ("smollm-135m", 1), ("qwen2-0.5b", 1), ("smollm-1.7b", 1),
                                       ("smollm-135m-long", 1), ("mqa16", 0), ("mha128", 0)])
def test_plan_puts_attention_on_the_tensor_cores_where_the_shape_allows(lib, monkeypatch, shape, mma):
    """Head dim 64 with at most 8 query heads per KV head: tensor-core attention, with the weight ring
    at a 1024-byte aligned offset (the swizzled K/V tiles); other shapes, or MBK_ATTN_MMA=0: CUDA cores."""
    extra = {"mqa16": workloads.DecoderShape("mqa16", 2, 1024, 2048, 16, 1, 64, 2048, 96, 1e-5, 1e4, False, steps=1),
             "mha128": workloads.DecoderShape("mha128", 2, 512, 1024, 4, 4, 128, 2048, 64, 1e-5, 1e4, False, steps=1)}
    s = extra.get(shape) or workloads.SHAPES[shape]
    info = mbk.mbk_plan_check(mbk.config_from_shape(s), 152)
    assert info.attn_mma == mma
    if mma:
        assert (info.smem_bytes - info.num_stages * info.stage_bytes) % 1024 == 0
    monkeypatch.setenv("MBK_ATTN_MMA", "0")
    assert mbk.mbk_plan_check(mbk.config_from_shape(s), 152).attn_mma == 0


@pytest.mark.parametrize("capacity,groups", [(8192, 1), (16384, 2), (80000, 16)])
def test_split_combine_groups_fit_the_shared_memory(lib, capacity, groups):
    """Long caches: the split combine brings as many splits per poll as the shared memory holds next
    to a weight ring deep enough for one attention split; the rest come in further polls."""
    s = workloads.scaled_down(workloads.SHAPES["smollm-135m-long"], kv_capacity=capacity)
    info = mbk.mbk_plan_check(mbk.config_from_shape(s), 152)
    assert info.attn_splits == (capacity + 511) // 512
    assert -(-info.attn_splits // info.combine_group) == groups
    assert info.num_stages >= 512 // 64 + 1
    assert info.smem_bytes <= 232448


def test_split_context_o_projection_gets_at_least_24_rows_per_task(lib, monkeypatch):
    """A split context's O-projection tasks each poll every split's outputs; the plan gives each at
    least 24 output rows (24 tasks per layer at hidden 576) unless MBK_COMBINE_TASKS says otherwise."""
    s = workloads.SHAPES["smollm-135m-long"]
    base = mbk.mbk_plan_check(mbk.config_from_shape(s), 152).num_tasks
    monkeypatch.setenv("MBK_COMBINE_TASKS", "48")
    assert mbk.mbk_plan_check(mbk.config_from_shape(s), 152).num_tasks == base + s.n_layers * (48 - 24)
    monkeypatch.setenv("MBK_COMBINE_TASKS", "24")
    assert mbk.mbk_plan_check(mbk.config_from_shape(s), 152).num_tasks == base


@pytest.mark.parametrize("split,splits", [("256", 32), ("512", 16), ("100", None), ("32", None)])
def test_attention_split_length_knob(lib, monkeypatch, split, splits):
    monkeypatch.setenv("MBK_ATTN_SPLIT", split)
    cfg = mbk.config_from_shape(workloads.SHAPES["smollm-135m-long"])
    if splits is None:
        with pytest.raises(mbk.MbkError):
            mbk.mbk_plan_check(cfg, 152)
    else:
        assert mbk.mbk_plan_check(cfg, 152).attn_splits == splits


def test_plan_balances_bytes_across_ctas(lib):
    s = workloads.SHAPES["smollm-135m"]
    info = mbk.mbk_plan_check(mbk.config_from_shape(s), 152)
    assert info.max_cta_bytes <= 1.10 * info.weight_bytes / 152


@pytest.mark.parametrize("field,value", [("head_dim", 96), ("n_kv_heads", 3), ("hidden", 500), ("n_layers", 0),
                                         ("vocab", 0), ("intermediate", 9000)])
def test_plan_rejects_unsupported_shapes(lib, field, value):
    cfg = mbk.config_from_shape(workloads.SHAPES["tiny"])
    setattr(cfg, field, value)
    with pytest.raises(mbk.MbkError) as e:
        mbk.mbk_plan_check(cfg, 152)
    assert e.value.code == mbk.MBK_ERR_INVALID_ARG


def test_create_rejects_null_arguments_before_touching_a_gpu(lib):
    cfg = mbk.config_from_shape(workloads.SHAPES["tiny"])
    h = ctypes.c_void_p()
    assert lib.mbk_create(ctypes.byref(cfg), None, None, 0, ctypes.byref(h)) == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_decode_step(None, 0, 0, None, None) == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_get_status(None) == mbk.MBK_ERR_INVALID_ARG
    lib.mbk_destroy(None)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        mbk.load_library(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("name", list(workloads.SHAPES))
def test_fp8_plan_streams_one_byte_per_weight(lib, name):
    """MBK_WEIGHTS_FP8: the same schedule over E4M3 copies -- every weight byte once, at one byte a weight."""
    s = workloads.SHAPES[name]
    bf = mbk.mbk_plan_check(mbk.config_from_shape(s), 152)
    f8 = mbk.mbk_plan_check(mbk.config_from_shape(s, mbk.MBK_WEIGHTS_FP8), 152)
    assert f8.weight_bytes * 2 == bf.weight_bytes
    assert f8.num_tasks == bf.num_tasks
    assert f8.num_chunks <= bf.num_chunks  # twice the rows fit a stage


def test_fp8_needs_rows_of_whole_16_bytes(lib):
    cfg = mbk.config_from_shape(workloads.SHAPES["tiny"], mbk.MBK_WEIGHTS_FP8)
    cfg.intermediate = 680  # a multiple of 8 (fine for bf16) but not of 16
    with pytest.raises(mbk.MbkError) as e:
        mbk.mbk_plan_check(cfg, 152)
    assert e.value.code == mbk.MBK_ERR_INVALID_ARG
    cfg.weight_format = 7  # no such format
    cfg.intermediate = 688
    with pytest.raises(mbk.MbkError) as e:
        mbk.mbk_plan_check(cfg, 152)
    assert e.value.code == mbk.MBK_ERR_INVALID_ARG


def test_new_entry_points_reject_bad_arguments_before_touching_a_gpu(lib):
    cfg = mbk.config_from_shape(workloads.SHAPES["tiny"])
    h = ctypes.c_void_p()
    w = ctypes.c_void_p(16)
    for pages, size in [(8, 48), (8, 16), (0, 32), (8, 256), (8, 2 * cfg.kv_capacity)]:
        rc = lib.mbk_create_paged(ctypes.byref(cfg), None, w, pages, size, 0, ctypes.byref(h))
        assert rc == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_set_page_table(None, None, 1, None) == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_decode_greedy(None, 0, 1, 0, None, None, None) == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_decode_steps(None, None, 1, 0, None, None) == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_quantize_fp8(None, 4, 8, w, w, None) == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_quantize_fp8(w, 4, 7, w, w, None) == mbk.MBK_ERR_INVALID_ARG  # odd row length
    assert lib.mbk_quantize_fp8(w, 0, 8, w, w, None) == mbk.MBK_ERR_INVALID_ARG


@pytest.mark.parametrize("name", list(workloads.SHAPES))
@pytest.mark.parametrize("env", [{"MBK_FUSE_ATTENTION": "0"}, {"MBK_MAX_TASKS_PER_OP": "38"},
                                 {"MBK_MAX_TASKS_PER_OP": "1"}])
def test_schedule_variants_build_and_check(lib, monkeypatch, name, env):
    """The schedule options (O projection as tasks of its own; fewer CTAs per op, down to one) still
    give plans that pass the scheduler's own checks and stream every weight byte once."""
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    s = workloads.SHAPES[name]
    info = mbk.mbk_plan_check(mbk.config_from_shape(s), 152)
    base = (s.n_heads * s.head_dim * s.hidden + 2 * s.n_kv_heads * s.head_dim * s.hidden
            + s.hidden * s.n_heads * s.head_dim + 3 * s.hidden * s.intermediate) * 2
    assert info.weight_bytes == s.n_layers * base + s.vocab * s.hidden * 2


def test_prefill_entry_points_reject_a_null_handle_before_touching_a_gpu(lib):
    toks = (ctypes.c_int32 * 2)(1, 2)
    assert lib.mbk_prefill(None, toks, 2, 0, None, 0, None) == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_prefill(None, None, 0, 0, None, 1, None) == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_debug_prefill_inject(None, None, 0) == mbk.MBK_ERR_INVALID_ARG
    one = (ctypes.c_int32 * 1)(1)
    assert lib.mbk_batch_step(None, 1, one, one, one, one, None, 0, None) == mbk.MBK_ERR_INVALID_ARG
    assert mbk.mbk_batch_step(None, [1], [0], [5], [[0]], 0, 0, 0) == mbk.MBK_ERR_INVALID_ARG
    # the Python wrapper marshals a token sequence and the logits modes
    assert mbk.mbk_prefill(None, [1, 2, 3], 0, 0, mbk.PREFILL_LOGITS["last"], 0) == mbk.MBK_ERR_INVALID_ARG
    assert set(mbk.PREFILL_LOGITS.values()) == {0, 1, 2}


# ---- the host execution model of the exchange protocol (mbk_plan_simulate)
def _rounds_per_layer(s, fused):
    return 4 if fused else 5  # QKV, attention (+ Wo when fused), [O projection], gate/up, down


@pytest.mark.parametrize("name", list(workloads.SHAPES))
@pytest.mark.parametrize("env", [{}, {"MBK_FUSE_ATTENTION": "0"}, {"MBK_MAX_TASKS_PER_OP": "38"},
                                 {"MBK_MAX_TASKS_PER_OP": "1"}])
def test_every_plan_runs_to_completion_in_the_wait_model(lib, monkeypatch, name, env):
    """Every CTA's task list, run in order with each task waiting for the words it reads, completes at
    the first position, the last, and the boundaries of the context splits: no schedule can deadlock
    on the GPU.  Its depth is the exchange rounds per layer times the layers, plus the LM head."""
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    s = workloads.SHAPES[name]
    cfg = mbk.config_from_shape(s)
    info = mbk.mbk_plan_check(cfg, 152)
    fused = None
    positions = sorted({0, s.pos0, s.pos0 + s.steps - 1, s.kv_capacity - 1, min(1023, s.kv_capacity - 1),
                        min(1024, s.kv_capacity - 1)})
    for pos in positions:
        rc, sim = mbk.mbk_plan_simulate(cfg, 152, pos)
        assert rc == mbk.MBK_OK, (pos, sim.stuck_cta, sim.stuck_task_type, sim.stuck_layer, sim.stuck_word)
        assert sim.tasks_run == sim.tasks_total == info.num_tasks and sim.words_written_twice == 0
        depth = (sim.exchange_depth - 1) / s.n_layers
        assert depth in (4, 5), sim.exchange_depth
        fused = depth == 4 if fused is None else fused
        assert sim.exchange_depth == s.n_layers * _rounds_per_layer(s, fused) + 1
        assert sim.schedule_depth >= sim.exchange_depth
    if env.get("MBK_FUSE_ATTENTION") == "0":
        assert not fused


def test_headline_plan_has_four_exchange_rounds_per_layer(lib):
    rc, sim = mbk.mbk_plan_simulate(mbk.config_from_shape(workloads.SHAPES["smollm-135m"]), 152, 64)
    assert rc == mbk.MBK_OK and sim.exchange_depth == 30 * 4 + 1 and sim.schedule_depth == sim.exchange_depth


@pytest.mark.parametrize("drop", [0, 5, 400])
def test_a_dropped_task_leaves_its_consumers_waiting(lib, monkeypatch, drop):
    """The host-side fault injection a handle applies (one task removed from its CTA's list) shows up
    in the model as a CTA stuck on a word that nothing writes, as the GPU's bounded waits would."""
    monkeypatch.setenv("MBK_DEBUG_DROP_TASK", str(drop))
    rc, sim = mbk.mbk_plan_simulate(mbk.config_from_shape(workloads.SHAPES["smollm-135m"]), 152, 10)
    assert rc == mbk.MBK_ERR_STATE
    assert sim.tasks_run < sim.tasks_total - 1
    assert sim.stuck_cta >= 0 and sim.stuck_word >= 0 and 1 <= sim.stuck_task_type <= 6


def test_simulate_rejects_bad_arguments(lib):
    cfg = mbk.config_from_shape(workloads.SHAPES["tiny"])
    assert mbk.mbk_plan_simulate(cfg, 0, 0)[0] == mbk.MBK_ERR_INVALID_ARG
    assert mbk.mbk_plan_simulate(cfg, 152, cfg.kv_capacity)[0] == mbk.MBK_ERR_INVALID_ARG
    assert lib.mbk_plan_simulate(None, 152, 0, None) == mbk.MBK_ERR_INVALID_ARG


EDGE_SHAPES = {
    "mha128": workloads.DecoderShape("mha128", 2, 512, 1024, 4, 4, 128, 2048, 64, 1e-5, 1e4, False, steps=12),
    "mqa16": workloads.DecoderShape("mqa16", 2, 1024, 2048, 16, 1, 64, 2048, 96, 1e-5, 1e4, False, steps=12),
    "gqa128": workloads.DecoderShape("gqa128", 2, 1024, 2048, 8, 2, 128, 2048, 96, 1e-5, 1e4, False, steps=12),
    "ragged-split": workloads.scaled_down(workloads.SHAPES["smollm-135m-long"], n_layers=2, kv_capacity=1500,
                                          prefill=1494, pos0=1494, steps=6, vocab=8192),
}


@pytest.mark.parametrize("name", list(EDGE_SHAPES))
@pytest.mark.parametrize("fuse", ["-1", "0"])
@pytest.mark.parametrize("fp8", [0, 1])
def test_edge_shapes_run_to_completion_in_the_wait_model(lib, monkeypatch, name, fuse, fp8):
    """The GPU tests' edge shapes (MQA with 16 query heads per KV head, head_dim 128 as MHA and GQA, a
    ragged last context split), with either O-projection schedule and either weight format."""
    monkeypatch.setenv("MBK_FUSE_ATTENTION", fuse)
    s = EDGE_SHAPES[name]
    cfg = mbk.config_from_shape(s, weight_format=fp8)
    for pos in sorted({0, s.kv_capacity // 2, s.kv_capacity - 1, min(1024, s.kv_capacity - 1)}):
        rc, sim = mbk.mbk_plan_simulate(cfg, 152, pos)
        assert rc == mbk.MBK_OK and sim.tasks_run == sim.tasks_total, (name, pos, sim.stuck_task_type)
        assert sim.exchange_depth in (4 * s.n_layers + 1, 5 * s.n_layers + 1)


def _fake_weights(shape, misalign=None):
    """Weight and cache pointers that are never dereferenced (every case below fails its argument
    checks before any CUDA call); each tensor 64 KB apart, 16-byte aligned unless `misalign` names a
    layer field to offset by 8 bytes."""
    base = [0x7000_0000_0000]

    def nxt():
        base[0] += 0x10000
        return base[0]

    layers = (mbk.MbkLayerWeights * shape.n_layers)()
    for layer in layers:
        for k in mbk.LAYER_FIELDS:
            if k in ("bq", "bk", "bv") and not shape.qkv_bias:
                continue
            setattr(layer, k, nxt() + (8 if k == misalign else 0))
    w = mbk.MbkWeights(nxt(), nxt(), layers)
    w._keep = layers
    return w, nxt(), nxt()


def test_static_step_checks_arguments_like_create_before_touching_a_gpu(lib):
    """mbk_decode_step_static rejects, before any CUDA call, every argument mbk_create rejects
    (including a misaligned projection weight and a non-finite RoPE theta) and its own step
    arguments; the shared check also rejects the misaligned weight through mbk_create."""
    shape = workloads.SHAPES["tiny"]
    cfg = mbk.config_from_shape(shape)
    w, kv, logits = _fake_weights(shape)
    st = lib.mbk_decode_step_static
    E = mbk.MBK_ERR_INVALID_ARG
    assert st(None, ctypes.byref(w), ctypes.c_void_p(kv), 0, 0, ctypes.c_void_p(logits), None) == E
    assert st(ctypes.byref(cfg), None, ctypes.c_void_p(kv), 0, 0, ctypes.c_void_p(logits), None) == E
    assert st(ctypes.byref(cfg), ctypes.byref(w), None, 0, 0, ctypes.c_void_p(logits), None) == E
    assert st(ctypes.byref(cfg), ctypes.byref(w), ctypes.c_void_p(kv), 0, 0, None, None) == E
    for tok, pos in ((-1, 0), (shape.vocab, 0), (0, -1), (0, shape.kv_capacity)):
        assert st(ctypes.byref(cfg), ctypes.byref(w), ctypes.c_void_p(kv), tok, pos, ctypes.c_void_p(logits), None) == E
    fp8 = mbk.config_from_shape(shape)
    fp8.weight_format = mbk.MBK_WEIGHTS_FP8
    assert st(ctypes.byref(fp8), ctypes.byref(w), ctypes.c_void_p(kv), 0, 0, ctypes.c_void_p(logits), None) == E
    bad = mbk.config_from_shape(shape)
    bad.rope_theta = float("inf")
    assert st(ctypes.byref(bad), ctypes.byref(w), ctypes.c_void_p(kv), 0, 0, ctypes.c_void_p(logits), None) == E
    for field in ("wq", "wo", "w_down"):
        wm, kvm, lm = _fake_weights(shape, misalign=field)
        assert st(ctypes.byref(cfg), ctypes.byref(wm), ctypes.c_void_p(kvm), 0, 0, ctypes.c_void_p(lm), None) == E
        h = ctypes.c_void_p()
        assert lib.mbk_create(ctypes.byref(cfg), ctypes.byref(wm), ctypes.c_void_p(kvm), 0, ctypes.byref(h)) == E
        assert not h.value
    wk, kvk, lk = _fake_weights(shape)
    assert st(ctypes.byref(cfg), ctypes.byref(wk), ctypes.c_void_p(kvk + 8), 0, 0, ctypes.c_void_p(lk), None) == E
