"""ctypes binding of the C ABI in include/mbk.h (libmbk.so, built in-tree by build.py).

Argument marshalling only: every step of the decode runs in the library's CUDA kernels.  PyTorch
is used for device memory and streams.  There is no fallback: if libmbk.so is missing or cannot be
loaded, `load_library()` raises.

The functions keep the C names (mbk_create, mbk_decode_step, ...).  `Decoder` bundles a workload's
weights (copied to the GPU with torch), a KV cache and a handle for convenience.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmbk.so")

MBK_OK = 0
MBK_ERR_INVALID_ARG = -1
MBK_ERR_UNSUPPORTED = -2
MBK_ERR_CUDA = -3
MBK_ERR_TIMEOUT = -4
MBK_ERR_NOMEM = -5
MBK_ERR_STATE = -6

EXPORTED = ("mbk_create", "mbk_decode_step", "mbk_decode_step_host", "mbk_kv_fill", "mbk_get_status",
            "mbk_error_string", "mbk_destroy", "mbk_plan_check", "mbk_debug_taps", "mbk_debug_plan",
            "mbk_trace_enable", "mbk_trace_read", "mbk_debug_inject", "mbk_decode_step_static", "mbk_decode_steps",
            "mbk_decode_greedy", "mbk_create_paged", "mbk_set_page_table", "mbk_quantize_fp8", "mbk_prefill",
            "mbk_debug_prefill_inject", "mbk_plan_simulate", "mbk_batch_step")
TASK_TYPES = {1: "qkv", 2: "attn", 3: "oproj", 4: "gateup", 5: "down", 6: "lmhead"}
TRACE_STAMPS = 8  # per task: begin, inputs ready, end, first weight stage, four phase marks


class MbkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {mbk_error_string(code)} ({code})")


class MbkConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("intermediate", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("vocab", ctypes.c_int), ("kv_capacity", ctypes.c_int), ("rms_eps", ctypes.c_double),
                ("rope_theta", ctypes.c_double), ("qkv_bias", ctypes.c_int), ("weight_format", ctypes.c_int)]


MBK_WEIGHTS_BF16, MBK_WEIGHTS_FP8 = 0, 1


LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "bq", "bk", "bv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


class MbkLayerWeights(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in LAYER_FIELDS]


class MbkWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(MbkLayerWeights))]


class MbkPlanInfo(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int), ("num_tasks", ctypes.c_int), ("num_chunks", ctypes.c_int),
                ("stage_bytes", ctypes.c_int), ("num_stages", ctypes.c_int), ("attn_splits", ctypes.c_int),
                ("weight_bytes", ctypes.c_int64), ("max_cta_bytes", ctypes.c_int64), ("act_words", ctypes.c_int64),
                ("smem_bytes", ctypes.c_int), ("combine_group", ctypes.c_int), ("attn_mma", ctypes.c_int)]


class MbkSimInfo(ctypes.Structure):
    _fields_ = [("tasks_total", ctypes.c_int), ("tasks_run", ctypes.c_int), ("exchange_depth", ctypes.c_int),
                ("schedule_depth", ctypes.c_int), ("words_written_twice", ctypes.c_int64), ("stuck_cta", ctypes.c_int),
                ("stuck_task_type", ctypes.c_int), ("stuck_layer", ctypes.c_int), ("stuck_word", ctypes.c_int64)]


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmbk.so (raises if it is missing: there is no other implementation to fall back to)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is not built; run `python -m persistent_decode_megakernel_gb300.build` "
                               "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(p)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        lib.mbk_create.argtypes = [ctypes.POINTER(MbkConfig), ctypes.POINTER(MbkWeights), vp, ctypes.c_int,
                                   ctypes.POINTER(vp)]
        lib.mbk_create.restype = ctypes.c_int
        lib.mbk_decode_step.argtypes = [vp, i32, i32, vp, vp]
        lib.mbk_decode_step.restype = ctypes.c_int
        lib.mbk_decode_steps.argtypes = [vp, vp, i32, i32, vp, vp]
        lib.mbk_decode_steps.restype = ctypes.c_int
        lib.mbk_decode_greedy.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        lib.mbk_decode_greedy.restype = ctypes.c_int
        lib.mbk_prefill.argtypes = [vp, vp, i32, i32, vp, i32, vp]
        lib.mbk_prefill.restype = ctypes.c_int
        lib.mbk_debug_prefill_inject.argtypes = [vp, vp, i32]
        lib.mbk_batch_step.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, vp]
        lib.mbk_batch_step.restype = ctypes.c_int
        lib.mbk_debug_prefill_inject.restype = ctypes.c_int
        lib.mbk_create_paged.argtypes = [ctypes.POINTER(MbkConfig), ctypes.POINTER(MbkWeights), vp, i32, i32, ctypes.c_int,
                                         ctypes.POINTER(vp)]
        lib.mbk_create_paged.restype = ctypes.c_int
        lib.mbk_set_page_table.argtypes = [vp, vp, i32, vp]
        lib.mbk_set_page_table.restype = ctypes.c_int
        lib.mbk_quantize_fp8.argtypes = [vp, i32, i32, vp, vp, vp]
        lib.mbk_quantize_fp8.restype = ctypes.c_int
        lib.mbk_decode_step_host.argtypes = [vp, i32, i32, vp, vp]
        lib.mbk_decode_step_host.restype = ctypes.c_int
        lib.mbk_kv_fill.argtypes = [vp, ctypes.c_int, vp, vp, i32, i32, vp]
        lib.mbk_kv_fill.restype = ctypes.c_int
        lib.mbk_get_status.argtypes = [vp]
        lib.mbk_get_status.restype = ctypes.c_int
        lib.mbk_error_string.argtypes = [ctypes.c_int]
        lib.mbk_error_string.restype = ctypes.c_char_p
        lib.mbk_destroy.argtypes = [vp]
        lib.mbk_destroy.restype = None
        lib.mbk_plan_check.argtypes = [ctypes.POINTER(MbkConfig), ctypes.c_int, ctypes.POINTER(MbkPlanInfo)]
        lib.mbk_plan_check.restype = ctypes.c_int
        lib.mbk_plan_simulate.argtypes = [ctypes.POINTER(MbkConfig), ctypes.c_int, ctypes.c_int, ctypes.POINTER(MbkSimInfo)]
        lib.mbk_plan_simulate.restype = ctypes.c_int
        lib.mbk_debug_taps.argtypes = [vp, vp]
        lib.mbk_debug_taps.restype = ctypes.c_int
        lib.mbk_debug_plan.argtypes = [vp, vp, ctypes.c_int64]
        lib.mbk_debug_plan.restype = ctypes.c_int64
        lib.mbk_trace_enable.argtypes = [vp, ctypes.c_int]
        lib.mbk_trace_enable.restype = ctypes.c_int
        lib.mbk_trace_read.argtypes = [vp, vp, ctypes.c_int64]
        lib.mbk_trace_read.restype = ctypes.c_int64
        lib.mbk_debug_inject.argtypes = [vp, vp]
        lib.mbk_debug_inject.restype = ctypes.c_int
        lib.mbk_decode_step_static.argtypes = [ctypes.POINTER(MbkConfig), ctypes.POINTER(MbkWeights), vp, i32, i32, vp, vp]
        lib.mbk_decode_step_static.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(rc: int, where: str) -> None:
    if rc != MBK_OK:
        raise MbkError(rc, where)


def mbk_error_string(code: int) -> str:
    return load_library().mbk_error_string(int(code)).decode()


def config_from_shape(shape, weight_format: int = 0) -> MbkConfig:
    return MbkConfig(shape.n_layers, shape.hidden, shape.intermediate, shape.n_heads, shape.n_kv_heads,
                     shape.head_dim, shape.vocab, shape.kv_capacity, float(shape.rms_eps), float(shape.rope_theta),
                     int(shape.qkv_bias), int(weight_format))


def mbk_plan_check(cfg: MbkConfig, num_sms: int) -> MbkPlanInfo:
    info = MbkPlanInfo()
    _check(load_library().mbk_plan_check(ctypes.byref(cfg), int(num_sms), ctypes.byref(info)), "mbk_plan_check")
    return info


def mbk_plan_simulate(cfg: MbkConfig, num_sms: int, position: int):
    """Runs one step of the schedule through the host model of the kernel's waits: (return code, MbkSimInfo)."""
    info = MbkSimInfo()
    rc = load_library().mbk_plan_simulate(ctypes.byref(cfg), int(num_sms), int(position), ctypes.byref(info))
    return rc, info


def mbk_create(cfg: MbkConfig, weights: MbkWeights, kv_cache_ptr: int, device: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load_library().mbk_create(ctypes.byref(cfg), ctypes.byref(weights), ctypes.c_void_p(kv_cache_ptr),
                                      int(device), ctypes.byref(h)), "mbk_create")
    return h


def mbk_decode_step(h, token_id: int, position: int, logits_ptr: int, stream_ptr: int) -> int:
    return load_library().mbk_decode_step(h, int(token_id), int(position), ctypes.c_void_p(logits_ptr),
                                          ctypes.c_void_p(stream_ptr))


def mbk_decode_steps(h, tokens, position: int, logits_ptr: int, stream_ptr: int) -> int:
    """tokens: a sequence of token ids (copied into a host int32 array here)."""
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    return load_library().mbk_decode_steps(h, arr.ctypes.data_as(ctypes.c_void_p), int(arr.size), int(position),
                                           ctypes.c_void_p(logits_ptr), ctypes.c_void_p(stream_ptr))


PREFILL_LOGITS = {None: 0, "last": 1, "all": 2}  # MBK_PREFILL_LOGITS_NONE / _LAST / _ALL


def mbk_prefill(h, tokens, position: int, logits_ptr: int, logits_mode: int, stream_ptr: int) -> int:
    """tokens: a sequence of token ids (copied into a host int32 array here); logits_ptr: device fp32
    [vocab] (mode 1), [n][vocab] (mode 2), or 0 (mode 0)."""
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    return load_library().mbk_prefill(h, arr.ctypes.data_as(ctypes.c_void_p), int(arr.size), int(position),
                                      ctypes.c_void_p(logits_ptr or None), int(logits_mode), ctypes.c_void_p(stream_ptr))


def mbk_batch_step(h, counts, starts, tokens, page_tables, logits_ptr: int, logits_mode: int, stream_ptr: int) -> int:
    """counts, starts: one entry per sequence; tokens: sum(counts) ids grouped by sequence; page_tables:
    [n_seq][max_pages] pool pages (all copied into host int32 arrays here)."""
    import numpy as np
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    s = np.ascontiguousarray(np.asarray(starts, dtype=np.int32))
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    p = np.ascontiguousarray(np.asarray(page_tables, dtype=np.int32))
    vp = ctypes.c_void_p
    return load_library().mbk_batch_step(h, int(c.size), c.ctypes.data_as(vp), s.ctypes.data_as(vp),
                                         t.ctypes.data_as(vp), p.ctypes.data_as(vp), vp(logits_ptr or None),
                                         int(logits_mode), vp(stream_ptr))


def mbk_debug_prefill_inject(h, x_in, n_tokens: int) -> int:
    """x_in: host fp32 array [n_layers][n_tokens][hidden] (or None to cancel)."""
    import numpy as np
    if x_in is None:
        return load_library().mbk_debug_prefill_inject(h, None, int(n_tokens))
    arr = np.ascontiguousarray(np.asarray(x_in, dtype=np.float32))
    return load_library().mbk_debug_prefill_inject(h, arr.ctypes.data_as(ctypes.c_void_p), int(n_tokens))


def mbk_create_paged(cfg: MbkConfig, weights: MbkWeights, kv_pool_ptr: int, num_pages: int, page_size: int,
                     device: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load_library().mbk_create_paged(ctypes.byref(cfg), ctypes.byref(weights), ctypes.c_void_p(kv_pool_ptr),
                                           int(num_pages), int(page_size), int(device), ctypes.byref(h)),
           "mbk_create_paged")
    return h


def mbk_quantize_fp8(w_ptr: int, rows: int, cols: int, q_ptr: int, s_ptr: int, stream_ptr: int) -> int:
    return load_library().mbk_quantize_fp8(ctypes.c_void_p(w_ptr), int(rows), int(cols), ctypes.c_void_p(q_ptr),
                                           ctypes.c_void_p(s_ptr), ctypes.c_void_p(stream_ptr))


def mbk_set_page_table(h, pages, stream_ptr: int) -> int:
    """pages: a sequence of pool page indices (copied into a host int32 array here)."""
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(pages, dtype=np.int32))
    return load_library().mbk_set_page_table(h, arr.ctypes.data_as(ctypes.c_void_p), int(arr.size),
                                             ctypes.c_void_p(stream_ptr))


def mbk_decode_greedy(h, first_token: int, n_steps: int, position: int, tokens_out_ptr: int, logits_ptr: int,
                      stream_ptr: int) -> int:
    """tokens_out_ptr: device int32[n_steps]; logits_ptr: device float[n_steps][vocab], or 0 for none."""
    return load_library().mbk_decode_greedy(h, int(first_token), int(n_steps), int(position),
                                            ctypes.c_void_p(tokens_out_ptr), ctypes.c_void_p(logits_ptr or None),
                                            ctypes.c_void_p(stream_ptr))


def mbk_decode_step_host(h, token_id: int, position: int, logits_host_ptr: int, stream_ptr: int) -> int:
    return load_library().mbk_decode_step_host(h, int(token_id), int(position), ctypes.c_void_p(logits_host_ptr),
                                               ctypes.c_void_p(stream_ptr))


def mbk_kv_fill(h, layer: int, k_raw_ptr: int, v_raw_ptr: int, p0: int, n: int, stream_ptr: int) -> int:
    return load_library().mbk_kv_fill(h, int(layer), ctypes.c_void_p(k_raw_ptr), ctypes.c_void_p(v_raw_ptr), int(p0),
                                      int(n), ctypes.c_void_p(stream_ptr))


def mbk_get_status(h) -> int:
    return load_library().mbk_get_status(h)


def mbk_destroy(h) -> None:
    if h:
        load_library().mbk_destroy(h)


def mbk_decode_step_static(cfg: MbkConfig, weights: MbkWeights, kv_cache_ptr: int, token_id: int, position: int,
                           logits_ptr: int, stream_ptr: int) -> int:
    """One decode step that allocates no device memory (see include/mbk.h); returns the C code."""
    return load_library().mbk_decode_step_static(ctypes.byref(cfg), ctypes.byref(weights), ctypes.c_void_p(kv_cache_ptr),
                                                 int(token_id), int(position), ctypes.c_void_p(logits_ptr),
                                                 ctypes.c_void_p(stream_ptr))


def mbk_debug_taps(h, n_layers: int, hidden: int):
    import numpy as np
    out = np.empty((2 * n_layers + 1, hidden), dtype=np.float32)
    _check(load_library().mbk_debug_taps(h, out.ctypes.data), "mbk_debug_taps")
    return out


def mbk_debug_plan(h):
    import numpy as np
    lib = load_library()
    n = lib.mbk_debug_plan(h, None, 0)
    if n < 0:
        raise MbkError(int(n), "mbk_debug_plan")
    out = np.empty((n, 6), dtype=np.int32)
    lib.mbk_debug_plan(h, out.ctypes.data, n)
    return out


def mbk_debug_inject(h, x_in) -> None:
    """x_in: fp32 numpy [n_layers, hidden] (row l = input of layer l >= 1) for the next step, or None."""
    import numpy as np
    if x_in is None:
        _check(load_library().mbk_debug_inject(h, None), "mbk_debug_inject")
        return
    a = np.ascontiguousarray(x_in, dtype=np.float32)
    _check(load_library().mbk_debug_inject(h, a.ctypes.data), "mbk_debug_inject")


def mbk_trace_enable(h, enable: bool) -> None:
    _check(load_library().mbk_trace_enable(h, int(bool(enable))), "mbk_trace_enable")


def mbk_trace_read(h):
    import numpy as np
    lib = load_library()
    n = lib.mbk_debug_plan(h, None, 0)
    out = np.zeros((n, TRACE_STAMPS), dtype=np.uint64)
    r = lib.mbk_trace_read(h, out.ctypes.data, n)
    if r < 0:
        raise MbkError(int(r), "mbk_trace_read")
    return out


class Decoder:
    """A workload's weights on the GPU, a bf16 KV cache and a library handle.

    step() launches one decode step into a device logits tensor on the current torch stream.
    """

    def __init__(self, wl, device: int = 0, paged=None, fp8: bool = False):
        """paged: None for a contiguous cache, or (num_pages, page_size, pages): a pool of num_pages
        pages and the page table pages[q] for logical page q.  fp8: stream FP8 copies of the weights
        (MBK_WEIGHTS_FP8)."""
        import torch
        self.torch = torch
        s = wl.shape
        self.shape = s
        dev = torch.device("cuda", device)
        self.device = dev
        self.embed = wl.embed.to(dev)
        self.final_norm = wl.final_norm.to(dev)
        self.layers = [{k: (None if v is None else v.to(dev)) for k, v in w.items()} for w in wl.layers]
        self.paged = paged
        if paged is None:
            self.kv = torch.zeros((s.n_layers, 2, s.n_kv_heads, s.kv_capacity, s.head_dim), dtype=torch.bfloat16, device=dev)
        else:
            num_pages, page_size, _ = paged
            self.pool = torch.zeros((num_pages, s.n_layers, 2, s.n_kv_heads, page_size, s.head_dim), dtype=torch.bfloat16,
                                    device=dev)
        arr = (MbkLayerWeights * s.n_layers)()
        for i, w in enumerate(self.layers):
            for k in LAYER_FIELDS:
                t = w.get(k)
                setattr(arr[i], k, None if t is None else t.data_ptr())
        self._layer_arr = arr
        self.weights = MbkWeights(self.embed.data_ptr(), self.final_norm.data_ptr(), arr)
        self.cfg = config_from_shape(s, MBK_WEIGHTS_FP8 if fp8 else MBK_WEIGHTS_BF16)
        if paged is None:
            self.handle = mbk_create(self.cfg, self.weights, self.kv.data_ptr(), device)
        else:
            self.handle = mbk_create_paged(self.cfg, self.weights, self.pool.data_ptr(), paged[0], paged[1], device)
            self.set_pages(paged[2])
        self.logits = torch.empty(s.vocab, dtype=torch.float32, device=dev)
        if s.prefill:
            self.fill(wl.k_raw, wl.v_raw, 0)

    def set_pages(self, pages) -> None:
        stream = self.torch.cuda.current_stream(self.device).cuda_stream
        _check(mbk_set_page_table(self.handle, pages, stream), "mbk_set_page_table")
        self.pages = list(pages)

    def logical_kv(self):
        """The cache in the contiguous layout [L][2][nkv][C][d] (paged: gathered through the page table;
        unmapped positions read as zero)."""
        if self.paged is None:
            return self.kv
        torch = self.torch
        s = self.shape
        ps = self.paged[1]
        out = torch.zeros((s.n_layers, 2, s.n_kv_heads, s.kv_capacity, s.head_dim), dtype=torch.bfloat16, device=self.device)
        for q, page in enumerate(self.pages):
            a = q * ps
            b = min(s.kv_capacity, a + ps)
            if a >= b:
                break
            out[:, :, :, a:b] = self.pool[page, :, :, :, : b - a]
        return out

    def fill(self, k_raw, v_raw, p0: int) -> None:
        """Load cache rows p0.. of every layer from pre-RoPE K and V (fp32 [L][nkv][n][d])."""
        torch = self.torch
        stream = torch.cuda.current_stream(self.device).cuda_stream
        n = k_raw.shape[2]
        for l in range(self.shape.n_layers):
            kr = k_raw[l].to(self.device, torch.float32).contiguous()
            vr = v_raw[l].to(self.device, torch.float32).contiguous()
            _check(mbk_kv_fill(self.handle, l, kr.data_ptr(), vr.data_ptr(), p0, n, stream), "mbk_kv_fill")
            torch.cuda.current_stream(self.device).synchronize()

    def step(self, token: int, pos: int, logits=None):
        out = self.logits if logits is None else logits
        stream = self.torch.cuda.current_stream(self.device).cuda_stream
        _check(mbk_decode_step(self.handle, token, pos, out.data_ptr(), stream), "mbk_decode_step")
        return out

    def steps(self, tokens, pos0: int, logits=None):
        """Teacher-forced decode of len(tokens) positions from pos0 in one launch; logits [n, vocab]."""
        n = len(tokens)
        out = self.torch.empty((n, self.shape.vocab), dtype=self.torch.float32, device=self.device) if logits is None else logits
        stream = self.torch.cuda.current_stream(self.device).cuda_stream
        _check(mbk_decode_steps(self.handle, tokens, pos0, out.data_ptr(), stream), "mbk_decode_steps")
        return out

    def greedy(self, first_token: int, n: int, pos0: int, logits=None, want_logits: bool = True):
        """Greedy decode of n steps from first_token at pos0 in one launch.  Returns (tokens, logits):
        tokens[i] (device int32) is the argmax of step i's logits; logits [n, vocab] or None."""
        toks = self.torch.empty(n, dtype=self.torch.int32, device=self.device)
        out = logits
        if out is None and want_logits:
            out = self.torch.empty((n, self.shape.vocab), dtype=self.torch.float32, device=self.device)
        stream = self.torch.cuda.current_stream(self.device).cuda_stream
        _check(mbk_decode_greedy(self.handle, first_token, n, pos0, toks.data_ptr(), out.data_ptr() if out is not None else 0,
                                 stream), "mbk_decode_greedy")
        return toks, out

    def prefill(self, tokens, pos0: int, logits: str = "last", out=None):
        """Prefill len(tokens) positions from pos0 on the tensor cores (mbk_prefill); writes their cache
        rows.  logits: "last" -> [vocab], "all" -> [n, vocab], None -> no logits (returns None)."""
        n = len(tokens)
        mode = PREFILL_LOGITS[logits]
        if out is None and mode:
            shape = (self.shape.vocab,) if mode == 1 else (n, self.shape.vocab)
            out = self.torch.empty(shape, dtype=self.torch.float32, device=self.device)
        stream = self.torch.cuda.current_stream(self.device).cuda_stream
        _check(mbk_prefill(self.handle, tokens, pos0, out.data_ptr() if out is not None else 0, mode, stream),
               "mbk_prefill")
        return out

    def batch_step(self, chunks, page_tables, logits: str = "last", out=None):
        """One step over several sequences of a paged decoder (mbk_batch_step): chunks = [(start,
        [tokens...]), ...], one per sequence; page_tables [n_seq][max_pages].  logits "last" ->
        [n_seq, vocab], "all" -> [sum of tokens, vocab], None -> no logits."""
        counts = [len(t) for _, t in chunks]
        starts = [p for p, _ in chunks]
        tokens = [x for _, t in chunks for x in t]
        mode = PREFILL_LOGITS[logits]
        if out is None and mode:
            rows = len(chunks) if mode == 1 else len(tokens)
            out = self.torch.empty((rows, self.shape.vocab), dtype=self.torch.float32, device=self.device)
        stream = self.torch.cuda.current_stream(self.device).cuda_stream
        _check(mbk_batch_step(self.handle, counts, starts, tokens, page_tables, out.data_ptr() if out is not None else 0,
                              mode, stream), "mbk_batch_step")
        return out

    def status(self) -> int:
        return mbk_get_status(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            mbk_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
