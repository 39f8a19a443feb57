"""Where a decode step's time goes, round by round, from the library's per-task trace.

Runs one decoder shape on cuda:0, traces one decode step at a chosen position (after untraced warm-up
steps) several times, and reports per exchange round of a layer (QKV, attention, O projection,
gate/up, down) medians over the middle layers and the traced repetitions:

  hop   -- from the last task of the previous round ending to the median task of this round having
           all of its inputs (the exchange: the producers' words travelling through L2 plus the
           consumers' polls and their block barrier);
  exec  -- median time from inputs ready to task end (the work, with its stage waits and barriers);
  tail  -- the last task of the round ending after the median one (imbalance and stragglers);
  span  -- the round on the critical path: from the previous round's last task to this round's.

Attention tasks also report their phases (inputs ready to the first K/V stage landed; rotation and
K/V staging; the (block, head) items; the merge of the items; the fused O rows), and the median SM
clock seen by the tasks (clock64 against globaltimer).  The trace switch adds a few globaltimer stores per task, so traced steps run a few
percent slower than untraced ones.

  python -m persistent_decode_megakernel_gb300.trace_report [--config smollm-135m] [--pos 100] [--reps 6]
"""
from __future__ import annotations

import argparse
import json

import numpy as np

ROUNDS = {1: "qkv", 2: "attn", 3: "oproj", 4: "gateup", 5: "down"}


def trace_rounds(name: str, pos: int, reps: int = 6, device: int = 0) -> dict:
    import torch

    from persistent_decode_megakernel_gb300 import mbk, workloads
    wl = workloads.generate(name, seed=0)
    s = wl.shape
    if not s.pos0 <= pos < s.kv_capacity:
        raise SystemExit(f"position {pos} outside [{s.pos0}, {s.kv_capacity})")
    dec = mbk.Decoder(wl, device=device)
    plan = mbk.mbk_debug_plan(dec.handle)
    cta, types, layer = plan[:, 0], plan[:, 1], plan[:, 2]
    res = {k: {"hop": [], "exec": [], "tail": [], "span": []} for k in ROUNDS}
    attn = {"first_stage_wait": [], "rope_and_kv_staged": [], "items": [], "merge": [], "o_rows": [],
            "combine_and_out": []}
    clocks, spans = [], []
    mid = (types == 2) & (layer >= 2) & (layer < s.n_layers - 2)
    for _ in range(reps):
        for i in range(3):
            dec.step(int(wl.tokens[i]), s.pos0 + i)
        mbk.mbk_trace_enable(dec.handle, True)
        dec.step(int(wl.tokens[3]), pos)
        torch.cuda.synchronize()
        tr = mbk.mbk_trace_read(dec.handle).astype(np.int64)
        mbk.mbk_trace_enable(dec.handle, False)
        t0 = tr[:, 0][tr[:, 0] > 0].min()
        rel = (tr - t0) / 1e3
        rel[tr == 0] = np.nan
        spans.append(float(np.nanmax(rel[:, 2])))
        for l in range(2, s.n_layers - 2):
            prev_end = None
            for ty in (5, 1, 2, 3, 4, 5):
                lay = l - 1 if (ty == 5 and prev_end is None) else l
                m = (types == ty) & (layer == lay)
                if not m.any():
                    continue
                rd, en = rel[m, 1], rel[m, 2]
                if prev_end is not None:
                    res[ty]["hop"].append(np.nanmedian(rd) - prev_end)
                    res[ty]["span"].append(np.nanmax(en) - prev_end)
                    res[ty]["exec"].append(np.nanmedian(en - rd))
                    res[ty]["tail"].append(np.nanmax(en) - np.nanmedian(en))
                prev_end = np.nanmax(en)
        r = rel[mid]
        if len(r):
            if np.isfinite(r[:, 3]).any():
                attn["first_stage_wait"].append(np.nanmedian(r[:, 3] - r[:, 1]))
            attn["rope_and_kv_staged"].append(np.nanmedian(r[:, 4] - r[:, 1]))
            attn["items"].append(np.nanmedian(r[:, 5] - r[:, 4]))
            if np.isfinite(r[:, 6]).any():
                attn["merge"].append(np.nanmedian(r[:, 6] - r[:, 5]))
                attn["o_rows"].append(np.nanmedian(r[:, 2] - r[:, 6]))
            else:
                attn["combine_and_out"].append(np.nanmedian(r[:, 2] - r[:, 5]))
        for c in np.unique(cta):
            idx = np.where((cta == c) & (types != 2))[0]
            ck, gt = tr[idx, 7].astype(np.float64), tr[idx, 2].astype(np.float64)
            ok = (ck > 0) & (gt > 0)
            if ok.sum() > 2 and gt[ok][-1] > gt[ok][0]:
                clocks.append((ck[ok][-1] - ck[ok][0]) / (gt[ok][-1] - gt[ok][0]))
    dec.close()
    out = {"workload": name, "position": pos, "traced_steps": reps, "traced_step_us": round(float(np.median(spans)), 2),
           "rounds_us": {}, "attention_phases_us": {}, "sm_clock_ghz": round(float(np.median(clocks)), 3) if clocks else None}
    layer_us = 0.0
    for ty, n in ROUNDS.items():
        if res[ty]["hop"]:
            out["rounds_us"][n] = {k: round(float(np.median(v)), 3) for k, v in res[ty].items()}
            layer_us += out["rounds_us"][n]["span"]
    out["layer_us"] = round(layer_us, 3)
    out["attention_phases_us"] = {k: round(float(np.median(v)), 3) for k, v in attn.items() if v}
    return out


def markdown(r: dict) -> str:
    lines = [f"Traced step at position {r['position']} of `{r['workload']}`: {r['traced_step_us']} us "
             f"(median of {r['traced_steps']}), SM clock {r['sm_clock_ghz']} GHz.", "",
             "| round | hop (us) | exec (us) | tail (us) | span (us) |", "|---|---|---|---|---|"]
    for n, v in r["rounds_us"].items():
        lines.append(f"| {n} | {v['hop']} | {v['exec']} | {v['tail']} | {v['span']} |")
    lines.append(f"| layer | | | | {r['layer_us']} |")
    if r["attention_phases_us"]:
        lines += ["", "Attention task phases (us): " + ", ".join(f"{k} {v}" for k, v in r["attention_phases_us"].items())]
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="smollm-135m")
    ap.add_argument("--pos", type=int, default=100)
    ap.add_argument("--reps", type=int, default=6)
    args = ap.parse_args()
    r = trace_rounds(args.config, args.pos, args.reps)
    print(markdown(r))
    print(json.dumps(r))


if __name__ == "__main__":
    main()
