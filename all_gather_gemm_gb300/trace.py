"""Timeline records of the fused all-gather matmul (ag_options.trace).

The kernels append 4-word records {t_start_ns, t_end_ns, meta, 0} to a device
buffer (word 0 is an atomic counter); ``meta = role << 56 | cta << 40 | a << 20
| b``.  This module decodes them, summarises where time went (waits on ready
flags, chunk staging, tile completion) and writes a Chrome trace-event JSON
timeline (one row per CTA) that shows the gather/GEMM overlap.

Tracing costs the recording warp a global atomic per record, so traced runs are
slower than untraced ones; use them for the shape of the timeline, not for
absolute times.

    python -m all_gather_gemm_gb300.trace --workload m16384_d8 --json out.json
"""
from __future__ import annotations

import argparse
import json
import sys

import numpy as np

ROLES = {1: "claim", 2: "wait", 3: "tile", 4: "gather", 5: "regfetch", 6: "issue"}


def new_buffer(records: int, device="cuda"):
    """A zeroed trace buffer for `records` records (torch int64 tensor)."""
    import torch
    return torch.zeros(1 + 4 * records, dtype=torch.int64, device=device)


def decode(buf) -> dict:
    """Decode a trace buffer into numpy arrays (times relative to the first record)."""
    t = buf.cpu().numpy().view(np.uint64) if hasattr(buf, "cpu") else np.asarray(buf, np.uint64)
    count = int(t[0])
    cap = (t.size - 1) // 4
    n = min(count, cap)
    rec = t[1:1 + 4 * n].reshape(-1, 4).astype(np.int64)
    t0 = int(rec[:, 0].min()) if n else 0
    meta = rec[:, 2]
    return {
        "count": count, "dropped": max(0, count - cap),
        "start": rec[:, 0] - t0, "end": rec[:, 1] - t0,
        "role": (meta >> 56) & 0xFF, "cta": (meta >> 40) & 0xFFFF,
        "a": (meta >> 20) & 0xFFFFF, "b": meta & 0xFFFFF,
    }


def summarize(d: dict, num_ctas: int | None = None) -> dict:
    """Counts and durations per role, per-CTA wait totals, completion times."""
    out = {"records": int(d["count"]), "dropped": int(d["dropped"])}
    if d["start"].size == 0:
        return out
    out["span_us"] = float(d["end"].max()) / 1e3
    ctas = num_ctas or int(d["cta"].max()) + 1
    for code, name in ROLES.items():
        m = d["role"] == code
        if not m.any():
            continue
        dur = (d["end"][m] - d["start"][m]).astype(np.float64)
        s = {"n": int(m.sum()), "mean_us": float(dur.mean()) / 1e3,
             "max_us": float(dur.max()) / 1e3,
             "first_start_us": float(d["start"][m].min()) / 1e3,
             "last_end_us": float(d["end"][m].max()) / 1e3}
        if name == "wait":
            per = np.bincount(d["cta"][m], weights=dur, minlength=ctas) / 1e3
            s["per_cta_total_us_mean"] = float(per.mean())
            s["per_cta_total_us_max"] = float(per.max())
        if name in ("tile", "claim", "regfetch", "gather"):
            s["done_by_us"] = {f"p{q}": float(np.percentile(d["end"][m], q)) / 1e3
                               for q in (10, 50, 90, 100)}
        if name == "issue":
            kind = d["b"][m] >> 16
            s["mean_us_by_kind"] = {
                k: float(dur[kind == v].mean()) / 1e3 for v, k in
                ((0, "follower"), (1, "local"), (3, "staged")) if (kind == v).any()}
        out[name] = s
    return out


def to_chrome_json(d: dict, path: str, pid: int = 0, name: str = "ag_matmul") -> None:
    """Write a Chrome trace-event file: one thread (row) per CTA."""
    ev = []
    for i in range(d["start"].size):
        role = ROLES.get(int(d["role"][i]), str(int(d["role"][i])))
        ev.append({"name": f"{role} {int(d['a'][i])}:{int(d['b'][i]) & 0xFFFF}", "cat": role,
                   "ph": "X", "pid": pid, "tid": int(d["cta"][i]),
                   "ts": float(d["start"][i]) / 1e3,
                   "dur": max(float(d["end"][i] - d["start"][i]) / 1e3, 0.01)})
    with open(path, "w") as f:
        json.dump({"traceEvents": ev, "displayTimeUnit": "ns", "otherData": {"name": name}}, f)


def main(argv=None) -> int:
    import torch

    import all_gather_gemm_gb300 as agmm
    from all_gather_gemm_gb300 import inputs as inp

    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="m16384_d8",
                    help="m16384_d8, m4096_d8_bias, m1024_d8 or cube_<n> (n a multiple of 8)")
    ap.add_argument("--layout", default="k_contiguous", choices=list(agmm.LAYOUTS))
    ap.add_argument("--k-per-flag", type=int, default=0, help="0: the library's automatic choice")
    ap.add_argument("--records", type=int, default=1 << 18)
    ap.add_argument("--json", default=None, help="write a Chrome trace of the fused call here")
    args = ap.parse_args(argv)
    table = {"m16384_d8": inp.iris_m16384, "m4096_d8_bias": inp.iris_m4096_bias,
             "m1024_d8": lambda: inp.iris_m1024(8)}
    if args.workload.startswith("cube_"):
        w = inp.cube(int(args.workload[5:]))
    else:
        w = table[args.workload]()
    x = inp.make_inputs(w)
    shards = [s.cuda() for s in x.shards]
    b = x.b.cuda()
    bias = x.bias.cuda() if x.bias is not None else None
    for _ in range(2):
        agmm.ag_matmul(shards, b, bias, layout=args.layout, k_per_flag=args.k_per_flag)
    res = {"workload": w.name, "layout": args.layout, "k_per_flag": args.k_per_flag,
           "num_sms": agmm.num_sms()}
    for label, fn in (("fused", agmm.ag_matmul), ("barrier", agmm.ag_then_matmul)):
        buf = new_buffer(args.records)
        fn(shards, b, bias, layout=args.layout, k_per_flag=args.k_per_flag, trace=buf)
        torch.cuda.synchronize()
        code, info = agmm.device_error()
        if code:
            print(f"device error {code} info {info:#x}", file=sys.stderr)
            return 1
        d = decode(buf)
        res[label] = summarize(d, agmm.num_sms())
        if label == "fused" and args.json:
            to_chrome_json(d, args.json, name=f"{w.name} fused")
    print(json.dumps(res, indent=1))
    return 0


if __name__ == "__main__":
    sys.exit(main())
