"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on the same seeded
teacher-forced stream and compare them with the stated tolerances.

Tolerances (per decode step): relative L2 error of the logits <= 1e-2 and max-abs error <= 5e-2;
greedy argmax equal on >= 99% of steps; every written KV-cache entry within one bf16 ulp.

Modes.  "sync": every GPU step starts from the oracle's state (token and cache rows below the step's
position), so each step's logits and its new cache rows are compared from identical inputs -- the
teacher-forced streams the bars are stated for.  "layers": in addition every layer reads the
oracle's input to that layer (the library's diagnostic injection), the region-by-region check of
the MegaBake article ("Where it breaks today").  "free": only the tokens are forced; each side
carries its own cache, so rounding differences also compound across steps (logits bars only).

"Within one bf16 ulp", entry by entry, with no fraction of entries exempt.  Both sides round the
same quantity to bf16; their exact values differ only by arithmetic error, so an entry passes when
its bit pattern is at most one apart from the oracle's, or when
    |gpu - oracle| <= ulp_bf16(|oracle| + E) + E,
where E bounds how far the GPU's unrounded value can be from the oracle's:
  * the fp32 rounding of the GPU's dot product of the entry's weight row with the normalised input,
    u * (H + 8) * A with A = sum_k |W_ik xn_k| (+ |bias_i|) and u = 2^-24 (the worst-case bound for
    any summation order of H terms, plus the bias, the norm scale and the rotation), and of the norm
    scale, u * (H / 2 + 4) * A;
  * in "sync" mode also the difference of the layer inputs themselves, which legitimate one-ulp
    choices of earlier layers' K/V entries move: ||W_i||_2 * ||xn_gpu - xn_oracle||_2, measured
    per layer from both sides' residual-stream taps (Cauchy-Schwarz);
  * for rotated K entries the two rows of the pair combine, |cos| E_i + |sin| E_j.
This bound is what the "fp32 math" of the oracle's definition leaves open; it is large only for
entries that cancel to a small fraction of their terms, where one bf16 ulp of the entry itself is
tiny.  Rows of a prefilled cache carry E = 3 u (|k_i cos| + |k_j sin|) (the rotation in fp32).

Argmax.  In "sync" and "layers" modes every step whose oracle top-2 gap exceeds NEAR_TIE agrees,
and every step that does not agree is such a near tie (the oracle's logit at the GPU's choice within
NEAR_TIE of its largest): a flip is then within the arithmetic noise of the logits.  The "at least
99% of steps" bar is asserted over the five decoder streams together (416 steps; a single near-tie
flip in a 64-step stream would otherwise be 98.4%).
"""
from __future__ import annotations

import dataclasses
import json
import math
import time
from typing import List, Optional

import numpy as np
import torch

REL_L2 = 1e-2
MAX_ABS = 5e-2
ARGMAX_FRACTION = 0.99
REL_L2_TIGHT = 2e-3
REL_L2_LAYERS = 1e-4
NEAR_TIE = 1e-4
FREE_ARGMAX_FLOOR = 0.95
U32 = 2.0 ** -24


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that are monotone in the value (+0 and -0 both map to 0)."""
    b = bits.astype(np.int64) & 0xFFFF
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def _bits_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp_bf16(mag: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at magnitude `mag` (normal range; subnormal spacing 2^-133)."""
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -126)))
    return 2.0 ** (e - 7)


@dataclasses.dataclass
class KvCompare:
    entries: int
    beyond_one_ordinal: int    # entries whose bit patterns are more than one apart (each within its bound)
    violations: int            # entries outside the per-entry bound: must be 0
    worst_scaled_ulps: float   # max |g - o| / ulp_bf16(|o|) (reported)
    worst_bound_frac: float    # max |g - o| / (ulp_bf16(|o| + E) + E) over entries more than one apart

    def ok(self) -> bool:
        return self.violations == 0

    def merged(self, other: "KvCompare") -> "KvCompare":
        return KvCompare(self.entries + other.entries, self.beyond_one_ordinal + other.beyond_one_ordinal,
                         self.violations + other.violations, max(self.worst_scaled_ulps, other.worst_scaled_ulps),
                         max(self.worst_bound_frac, other.worst_bound_frac))


def kv_check(g_bits: np.ndarray, o_bits: np.ndarray, allow: Optional[np.ndarray] = None) -> KvCompare:
    """Entry-by-entry comparison of bf16 bit patterns; `allow` (broadcastable, >= 0) is E above."""
    g_bits = np.asarray(g_bits).astype(np.uint16)
    o_bits = np.asarray(o_bits).astype(np.uint16)
    gf, of = _bits_f32(g_bits), _bits_f32(o_bits)
    e = np.zeros_like(of) if allow is None else np.broadcast_to(np.asarray(allow, dtype=np.float64), of.shape)
    diff = np.abs(gf - of)
    close = np.abs(bf16_ordinal(g_bits) - bf16_ordinal(o_bits)) <= 1
    bound = _ulp_bf16(np.abs(of) + e) + e
    within = close | (diff <= bound)
    far = ~close
    worst = float((diff / _ulp_bf16(np.abs(of))).max(initial=0.0))
    frac = float((diff[far] / bound[far]).max(initial=0.0))
    return KvCompare(int(o_bits.size), int(far.sum()), int((~within).sum()), worst, frac)


def kv_compare(gpu_kv: torch.Tensor, oracle_kv: np.ndarray, rows: slice, allow: Optional[np.ndarray] = None) -> KvCompare:
    """kv_check over cache rows `rows` of [L][2][nkv][C][d] caches (GPU bf16 tensor, oracle bit patterns)."""
    g = gpu_kv.view(torch.int16).cpu().numpy().view(np.uint16)[:, :, :, rows]
    return kv_check(g, oracle_kv[:, :, :, rows], allow)


def _rope_cs(shape, pos: int):
    half = shape.head_dim // 2
    i = np.arange(half, dtype=np.float64)
    ang = pos * shape.rope_theta ** (-2.0 * i / shape.head_dim)
    return np.cos(ang), np.sin(ang)


def _rmsnorm64(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    x = x.astype(np.float64)
    return x / math.sqrt(float(np.mean(x * x)) + eps) * gain


class KvBounds:
    """Per-layer allowance E of the new K (rotated) and V entries of a decode step (module docstring)."""

    def __init__(self, wl, oracle=None, fp8: bool = False):
        s = wl.shape
        self.s = s
        self.wl = wl
        self.fp8 = fp8
        self.oracle = oracle
        self._cache = {}

    def _layer(self, l: int):
        if l in self._cache:
            return self._cache[l]
        w = self.wl.layers[l]
        mats = []
        for key, bkey in (("wk", "bk"), ("wv", "bv")):
            W = w[key].to(torch.float32)
            if self.fp8:
                W = self._fp8_weights(w[key])
            absW = W.abs()
            rown = torch.linalg.vector_norm(W.to(torch.float64), dim=1).numpy()
            b = w[bkey]
            absb = np.zeros(W.shape[0]) if b is None else np.abs(b.to(torch.float64).numpy())
            mats.append((absW, rown, absb))
        gain = self.wl.layers[l]["attn_norm"].to(torch.float64).numpy()
        self._cache[l] = (mats, gain)
        return self._cache[l]

    def _fp8_weights(self, w_bf16: torch.Tensor) -> torch.Tensor:
        """The E4M3 copy both sides compute with: per-row scale times the code's value (oracle quantizer)."""
        from oracle.oracle import bf16_bits, quantize_fp8
        q, sc = quantize_fp8(bf16_bits(w_bf16), self.oracle.lib)
        lut = np.array([self.oracle.lib.orc_fp8_to_f32(c) for c in range(256)], dtype=np.float64)
        return torch.from_numpy((lut[q] * np.asarray(sc, dtype=np.float64)[:, None]).astype(np.float32))

    def allowance(self, l: int, pos: int, x_orc: np.ndarray, x_gpu: Optional[np.ndarray], input_rel: float = 0.0):
        """E for layer l's new K and V rows: arrays [nkv][d] each.  input_rel: a relative error of the
        normalised input itself on the GPU side (the prefill's bf16 high/low pair carries 2^-17)."""
        s = self.s
        (mk, mv), gain = self._layer(l)
        xn = _rmsnorm64(x_orc, gain, s.rms_eps)
        dxn = 0.0 if x_gpu is None else float(np.linalg.norm(_rmsnorm64(x_gpu, gain, s.rms_eps) - xn))
        axn = torch.from_numpy(np.abs(xn).astype(np.float32))
        out = []
        for absW, rown, absb in (mk, mv):
            A = (absW @ axn).numpy().astype(np.float64) * (1.0 + 1e-5) + absb
            E = (U32 * (1.5 * s.hidden + 12) + input_rel) * A + rown * dxn
            out.append((A.reshape(s.n_kv_heads, s.head_dim), E.reshape(s.n_kv_heads, s.head_dim)))
        (Ak, Ek), (_, Ev) = out
        c, sn = _rope_cs(s, pos)
        h = s.head_dim // 2
        Er = np.empty_like(Ek)
        Er[:, :h] = np.abs(c) * Ek[:, :h] + np.abs(sn) * Ek[:, h:] + 2 * U32 * (np.abs(c) * Ak[:, :h] + np.abs(sn) * Ak[:, h:])
        Er[:, h:] = np.abs(c) * Ek[:, h:] + np.abs(sn) * Ek[:, :h] + 2 * U32 * (np.abs(c) * Ak[:, h:] + np.abs(sn) * Ak[:, :h])
        return Er, Ev


def prefill_allowance(wl) -> np.ndarray:
    """E of the prefilled cache rows [L][2][nkv][prefill][d]: the fp32 rotation of pre-RoPE K."""
    s = wl.shape
    k = np.abs(wl.k_raw.numpy().astype(np.float64))
    pos = np.arange(s.prefill, dtype=np.float64)[:, None]
    h = s.head_dim // 2
    ang = pos * s.rope_theta ** (-2.0 * np.arange(h, dtype=np.float64) / s.head_dim)[None, :]
    c, sn = np.abs(np.cos(ang)), np.abs(np.sin(ang))
    E = np.zeros((s.n_layers, 2, s.n_kv_heads, s.prefill, s.head_dim))
    E[:, 0, :, :, :h] = 3 * U32 * (k[..., :h] * c + k[..., h:] * sn)
    E[:, 0, :, :, h:] = 3 * U32 * (k[..., h:] * c + k[..., :h] * sn)
    return E


@dataclasses.dataclass
class ParityReport:
    steps: int
    worst_rel_l2: float
    worst_max_abs: float
    argmax_agree: float
    kv: KvCompare
    prefill: KvCompare
    gpu_seconds: float
    oracle_seconds: float
    mode: str = "sync"
    disagreements: List[dict] = dataclasses.field(default_factory=list)  # {step, oracle_gap}
    name: str = ""
    decisive_steps: int = 0      # steps whose oracle top-2 gap exceeds NEAR_TIE
    decisive_agree: int = 0      # ... of which the argmax agrees

    def check(self):
        assert self.worst_rel_l2 <= REL_L2, self
        assert self.worst_max_abs <= MAX_ABS, self
        assert self.prefill.ok(), self
        if self.mode in ("sync", "layers"):
            # teacher-forced streams: the four bars of the method's comparison, entry by entry
            assert self.decisive_agree == self.decisive_steps, self
            assert all(d["oracle_gap"] <= NEAR_TIE for d in self.disagreements), self
            assert self.kv.ok(), self
            assert self.worst_rel_l2 <= (REL_L2_LAYERS if self.mode == "layers" else REL_L2_TIGHT), self
        else:
            # free running: each side's own cache; the logits bars hold, argmax disagreement stays rare
            assert self.argmax_agree >= FREE_ARGMAX_FLOOR, self

    def json_line(self) -> str:
        d = {"config": self.name, "mode": self.mode, "steps": self.steps, "rel_l2_worst": self.worst_rel_l2,
             "max_abs_worst": self.worst_max_abs, "argmax_agree": self.argmax_agree,
             "argmax_disagreements": self.disagreements, "decisive_steps": self.decisive_steps,
             "decisive_agree": self.decisive_agree, "kv_entries": self.kv.entries,
             "kv_beyond_one_ordinal": self.kv.beyond_one_ordinal, "kv_violations": self.kv.violations,
             "kv_worst_scaled_ulps": self.kv.worst_scaled_ulps, "kv_worst_bound_frac": self.kv.worst_bound_frac,
             "prefill_entries": self.prefill.entries, "prefill_violations": self.prefill.violations}
        return "PARITY_JSON " + json.dumps(d)


def _rows_to_gpu(dec, orc_kv: np.ndarray, rows: slice) -> None:
    """Oracle cache rows `rows` into the GPU cache (through the page table of a paged decoder)."""
    src = torch.from_numpy(np.ascontiguousarray(orc_kv[:, :, :, rows]).view(np.int16)).view(torch.bfloat16)
    if dec.paged is None:
        dec.kv[:, :, :, rows] = src.to(dec.device)
        return
    ps = dec.paged[1]
    a = rows.start
    while a < rows.stop:  # one copy per run of positions inside a page
        b = min(rows.stop, (a // ps + 1) * ps)
        page = dec.pages[a // ps]
        dec.pool[page, :, :, :, a % ps:a % ps + (b - a)] = src[:, :, :, a - rows.start:b - rows.start].to(dec.device)
        a = b


def _row_from_gpu(dec, pos: int) -> np.ndarray:
    """GPU cache row `pos` of every layer as bf16 bit patterns [L][2][nkv][d]."""
    row = dec.kv[:, :, :, pos] if dec.paged is None else dec.pool[dec.pages[pos // dec.paged[1]], :, :, :, pos % dec.paged[1]]
    return row.view(torch.int16).cpu().numpy().view(np.uint16)


def _step_stats(got: np.ndarray, ref: np.ndarray, i: int, rels, maxs, dis, decisive) -> int:
    diff = got - ref
    rels.append(float(np.linalg.norm(diff) / np.linalg.norm(ref)))
    maxs.append(float(np.abs(diff).max()))
    gi, oi = int(np.argmax(got)), int(np.argmax(ref))
    top2 = np.partition(ref, -2)[-2:]
    clear = float(top2[1] - top2[0]) > NEAR_TIE
    decisive[0] += int(clear)
    decisive[1] += int(clear and gi == oi)
    if gi != oi:
        dis.append({"step": i, "oracle_gap": float(ref[oi] - ref[gi])})
        return 0
    return 1


def run_parity(wl, device: int = 0, steps: int | None = None, mode: str = "sync", fp8: bool = False,
               paged=None) -> ParityReport:
    """Run `steps` teacher-forced steps of `wl` on both sides in `mode` ("sync", "layers" or "free").
    paged: None (contiguous cache) or (num_pages, page_size, table) for a paged GPU cache."""
    from oracle import OracleDecoder
    from persistent_decode_megakernel_gb300 import mbk
    from persistent_decode_megakernel_gb300.mbk import Decoder

    s = wl.shape
    n = s.steps if steps is None else steps
    dec = Decoder(wl, device=device, fp8=fp8, paged=paged)  # fp8: both sides on the FP8 copies
    orc = OracleDecoder(wl, fp8=fp8)
    prefill = KvCompare(0, 0, 0, 0.0, 0.0)
    if s.prefill:
        torch.cuda.synchronize()
        prefill = kv_compare(dec.logical_kv(), orc.kv, slice(0, s.prefill), prefill_allowance(wl))
        if mode in ("sync", "layers"):
            _rows_to_gpu(dec, orc.kv, slice(0, s.prefill))
    rels: List[float] = []
    maxs: List[float] = []
    dis: List[dict] = []
    decisive = [0, 0]
    agree = 0
    t_gpu = t_orc = 0.0
    kv = KvCompare(0, 0, 0, 0.0, 0.0)
    if mode in ("sync", "layers"):
        bounds = KvBounds(wl, orc, fp8)
        for i in range(n):
            tok, pos = int(wl.tokens[i]), s.pos0 + i
            if i > 0:
                _rows_to_gpu(dec, orc.kv, slice(pos - 1, pos))
            if mode == "layers":
                # the oracle runs first; its per-layer inputs (taps 0, 2, 4, ...) feed the GPU step
                t0 = time.perf_counter()
                ref, taps = orc.step(tok, pos, taps=True)
                t_orc += time.perf_counter() - t0
                mbk.mbk_debug_inject(dec.handle, taps[0:2 * s.n_layers:2])
            t0 = time.perf_counter()
            got = dec.step(tok, pos).cpu().numpy().astype(np.float64)
            t_gpu += time.perf_counter() - t0
            g_rows = _row_from_gpu(dec, pos)
            gtaps = None
            if mode == "sync":
                gtaps = mbk.mbk_debug_taps(dec.handle, s.n_layers, s.hidden)
                t0 = time.perf_counter()
                ref, taps = orc.step(tok, pos, taps=True)
                t_orc += time.perf_counter() - t0
            ref = ref.astype(np.float64)
            agree += _step_stats(got, ref, i, rels, maxs, dis, decisive)
            for l in range(s.n_layers):
                x_orc = wl.embed[tok].to(torch.float32).numpy() if l == 0 else taps[2 * l]
                x_gpu = None if (gtaps is None or l == 0) else gtaps[2 * l]
                Ek, Ev = bounds.allowance(l, pos, x_orc, x_gpu)
                o_rows = orc.kv[l, :, :, pos]
                kv = kv.merged(kv_check(g_rows[l, 0], o_rows[0], Ek))
                kv = kv.merged(kv_check(g_rows[l, 1], o_rows[1], Ev))
        assert dec.status() == 0, "device status reports a failed wait"
    else:
        out = torch.empty((n, s.vocab), dtype=torch.float32, device=dec.device)
        t0 = time.perf_counter()
        for i in range(n):
            dec.step(int(wl.tokens[i]), s.pos0 + i, out[i])
        torch.cuda.synchronize()
        t_gpu = time.perf_counter() - t0
        assert dec.status() == 0, "device status reports a failed wait"
        got = out.cpu().numpy().astype(np.float64)
        t0 = time.perf_counter()
        for i in range(n):
            ref = orc.step(int(wl.tokens[i]), s.pos0 + i).astype(np.float64)
            agree += _step_stats(got[i], ref, i, rels, maxs, dis, decisive)
        t_orc = time.perf_counter() - t0
        # each side's own cache: reported, not asserted (rounding choices compound across steps)
        kv = kv_compare(dec.logical_kv(), orc.kv, slice(s.pos0, s.pos0 + n))
    dec.close()
    return ParityReport(n, max(rels), max(maxs), agree / n, kv, prefill, t_gpu, t_orc, mode, dis, s.name, decisive[0], decisive[1])
