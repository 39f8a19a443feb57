"""ctypes binding of the C oracle (mbk_oracle.c) -- TEST INFRASTRUCTURE ONLY.

The C file is compiled with gcc in ISO C mode with floating-point contraction off, so the
x86 and Arm builds evaluate the same expressions in the same order.  `build_oracle()` does
the compile; `OracleDecoder` runs teacher-forced decode steps over a workload.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mbk_oracle.c")
_HDR = os.path.join(_HERE, "mbk_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmbk_oracle.so")
_lock = threading.Lock()
_lib = None


GCC_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared"]


def build_oracle(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libmbk_oracle.so (skipped when up to date)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest_src:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc"] + GCC_FLAGS + ["-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("intermediate", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("vocab", ctypes.c_int), ("kv_capacity", ctypes.c_int),
                ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double), ("qkv_bias", ctypes.c_int)]


_P = ctypes.c_void_p


class _Layer(ctypes.Structure):
    _fields_ = [(k, _P) for k in ("attn_norm", "wq", "wk", "wv", "bq", "bk", "bv", "wo", "mlp_norm",
                                  "w_gate", "w_up", "w_down")]


class _Fp8Layer(ctypes.Structure):
    _fields_ = [("q", _P * 7), ("s", _P * 7)]


class _Fp8Weights(ctypes.Structure):
    _fields_ = [("layers", ctypes.POINTER(_Fp8Layer)), ("lm_q", _P), ("lm_s", _P)]


# the projections of a layer in the order of the FP8 tables
FP8_SLOTS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def bind(lib):
    """Declare the argument types of the oracle's exported functions on a loaded CDLL."""
    f = ctypes.c_float
    lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f32.restype = f
    lib.orc_f32_to_bf16.argtypes = [f]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_rmsnorm.argtypes = [_P, _P, ctypes.c_int, ctypes.c_double, _P]
    lib.orc_gemv.argtypes = [_P, _P, _P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int]
    lib.orc_rope.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double]
    lib.orc_attention.argtypes = [_P, _P, _P] + [ctypes.c_int] * 5 + [_P, ctypes.c_int]
    lib.orc_silu_mul.argtypes = [_P, _P, ctypes.c_int, _P]
    lib.orc_kv_fill.argtypes = [ctypes.POINTER(_Config), _P, _P, _P, ctypes.c_int, ctypes.c_int]
    lib.orc_decode_step.argtypes = [ctypes.POINTER(_Config), _P, _P, ctypes.POINTER(_Layer), _P,
                                    ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_int]
    lib.orc_decode_step.restype = ctypes.c_int
    lib.orc_max_threads.restype = ctypes.c_int
    lib.orc_fp8_from_f32.argtypes = [f]
    lib.orc_fp8_from_f32.restype = ctypes.c_uint8
    lib.orc_fp8_to_f32.argtypes = [ctypes.c_uint8]
    lib.orc_fp8_to_f32.restype = f
    lib.orc_quantize_fp8.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P]
    lib.orc_gemv_fp8.argtypes = [_P, _P, _P, _P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int]
    lib.orc_decode_step_fp8.argtypes = [ctypes.POINTER(_Config), _P, _P, ctypes.POINTER(_Layer),
                                        ctypes.POINTER(_Fp8Weights), _P, ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_int]
    lib.orc_decode_step_fp8.restype = ctypes.c_int
    lib.orc_prefill.argtypes = [ctypes.POINTER(_Config), _P, _P, ctypes.POINTER(_Layer), _P, _P, ctypes.c_int,
                                ctypes.c_int, _P, ctypes.c_int]
    lib.orc_prefill.restype = ctypes.c_int
    return lib


def quantize_fp8(w_bits: np.ndarray, lib=None):
    """FP8 (E4M3) codes and per-row fp32 scales of a bf16 matrix given as uint16 bit patterns [rows, cols]."""
    lib = oracle_lib() if lib is None else lib
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    rows, cols = w.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    sc = np.empty(rows, dtype=np.float32)
    lib.orc_quantize_fp8(w.ctypes.data, rows, cols, q.ctypes.data, sc.ctypes.data)
    return q, sc


def oracle_lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(ctypes.CDLL(build_oracle()))
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A contiguous uint16 numpy view of a bf16 tensor's bit patterns."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


class OracleDecoder:
    """Teacher-forced decode of one workload on the CPU.

    Holds its own bf16 KV cache [L][2][nkv][cap][d] (uint16 bit patterns).
    """

    def __init__(self, wl, nthreads: int = 0, lib=None, fp8: bool = False):
        """fp8: every projection and the LM head on FP8 (E4M3, per-row scale) copies of the weights."""
        self.lib = oracle_lib() if lib is None else lib
        s = wl.shape
        self.shape = s
        self.nthreads = nthreads
        self.cfg = _Config(s.n_layers, s.hidden, s.intermediate, s.n_heads, s.n_kv_heads, s.head_dim, s.vocab,
                           s.kv_capacity, s.rms_eps, s.rope_theta, int(s.qkv_bias))
        self._keep = []
        self.embed = bf16_bits(wl.embed)
        self.final_norm = bf16_bits(wl.final_norm)
        arr = (_Layer * s.n_layers)()
        for i, w in enumerate(wl.layers):
            for k, _ in _Layer._fields_:
                t = w.get(k)
                if t is None:
                    setattr(arr[i], k, None)
                else:
                    a = bf16_bits(t)
                    self._keep.append(a)
                    setattr(arr[i], k, a.ctypes.data)
        self.layers = arr
        self.fp8 = None
        if fp8:
            f8 = (_Fp8Layer * s.n_layers)()
            for i, w in enumerate(wl.layers):
                for j, k in enumerate(FP8_SLOTS):
                    q, sc = quantize_fp8(bf16_bits(w[k]), self.lib)
                    self._keep += [q, sc]
                    f8[i].q[j] = q.ctypes.data
                    f8[i].s[j] = sc.ctypes.data
            lq, ls = quantize_fp8(self.embed, self.lib)
            self._keep += [lq, ls, f8]
            self.fp8 = _Fp8Weights(f8, lq.ctypes.data, ls.ctypes.data)
        self.kv = np.zeros((s.n_layers, 2, s.n_kv_heads, s.kv_capacity, s.head_dim), dtype=np.uint16)
        if s.prefill:
            self.fill(wl.k_raw, wl.v_raw, 0)

    def fill(self, k_raw: torch.Tensor, v_raw: torch.Tensor, p0: int) -> None:
        """Write cache rows p0.. from pre-RoPE K and V, fp32 [L][nkv][n][d]."""
        s = self.shape
        n = k_raw.shape[2]
        for l in range(s.n_layers):
            kr = np.ascontiguousarray(k_raw[l].numpy(), dtype=np.float32)
            vr = np.ascontiguousarray(v_raw[l].numpy(), dtype=np.float32)
            self.lib.orc_kv_fill(ctypes.byref(self.cfg), self.kv[l].ctypes.data, kr.ctypes.data, vr.ctypes.data, p0, n)

    def step(self, token: int, pos: int, taps: bool = False):
        s = self.shape
        logits = np.empty(s.vocab, dtype=np.float32)
        tap = np.empty((2 * s.n_layers + 1, s.hidden), dtype=np.float32) if taps else None
        if self.fp8 is None:
            rc = self.lib.orc_decode_step(ctypes.byref(self.cfg), self.embed.ctypes.data, self.final_norm.ctypes.data,
                                          self.layers, self.kv.ctypes.data, int(token), int(pos), logits.ctypes.data,
                                          _ptr(tap), self.nthreads)
        else:
            rc = self.lib.orc_decode_step_fp8(ctypes.byref(self.cfg), self.embed.ctypes.data, self.final_norm.ctypes.data,
                                              self.layers, ctypes.byref(self.fp8), self.kv.ctypes.data, int(token), int(pos),
                                              logits.ctypes.data, _ptr(tap), self.nthreads)
        if rc != 0:
            raise ValueError(f"oracle rejected token={token} pos={pos}")
        return (logits, tap) if taps else logits

    def prefill(self, tokens, p0: int, logits: bool = True):
        """The n given tokens at positions p0 .. p0 + n - 1, layer by layer (orc_prefill); logits [n][V]."""
        if self.fp8 is not None:
            raise ValueError("the oracle's prefill takes the bf16 weights")
        s = self.shape
        toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        out = np.empty((toks.size, s.vocab), dtype=np.float32) if logits else None
        rc = self.lib.orc_prefill(ctypes.byref(self.cfg), self.embed.ctypes.data, self.final_norm.ctypes.data,
                                  self.layers, self.kv.ctypes.data, toks.ctypes.data, int(toks.size), int(p0),
                                  _ptr(out), self.nthreads)
        if rc != 0:
            raise ValueError(f"oracle rejected a prefill of {toks.size} tokens at {p0}")
        return out
