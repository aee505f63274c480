"""Per-token-bucket route-block tuning on this GPU.

The pages ship per-geometry, per-token-bucket tuning rows and adopt a row
only if it passes a gate declared before measuring (AITER #5609 "Add
DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Configuration and Performance on
the measured runtime). Here the knob is block_m: the sort block, which is
also the route tile of both GEMMs and the one tile parameter of this
implementation that is chosen per call (the library's rule picks it from
the mean routes per expert).

Gate, restated from the pages: per bucket, the default (library rule) and a
candidate are measured in P alternating pairs; one measurement is R graph
replays of the whole fused call, L2 flushed before each replay; a candidate
is adopted only with a median paired improvement >= 1 % and at least
25/31 of the pairs faster. The default is also measured against itself (an
identical-configuration control): a sound measurement does not pass it.

Table: CSV with one row per (geometry, token bucket):
H, Ip, E, topk, a16, max_tokens, block_m, default_block_m, median_gain,
wins, pairs, control_gain, control_wins, and the second knob, the weight L2
prefetch leads: prefetch1, prefetch2 (0 = the library's defaults),
prefetch_gain, prefetch_wins (``--knob prefetch`` measures them for the
rows' block_m under the same gate), and the third, the GEMMs' split
walk: split (0 = the library's choice, 1 = the split walk, 2 = whole
tiles only), split_gain, split_wins (``--knob split``, the rows' block_m
and leads fixed).
``table_for`` turns the rows of one geometry into the ``block_m_table`` of
``MoeLayer``.

  python -m block_scaled_moe_sort_gb300.tune --H 5120 --Ip 640 --E 384 --topk 6 \\
      --tokens 6 12 24 48 96 192 384 768 --buckets 8 16 32 64 128 256 512 1024 \\
      --out table.csv
"""
from __future__ import annotations

import argparse
import csv
import math
import statistics
from typing import Iterable, List, Optional, Sequence

import os

# The table measured on GB300 for the pages' geometries: the two tuned
# decode geometries (backbone 384 experts top-6, draft 128 experts top-3;
# H=5120, Ip=640; real decode rows per bucket as the pages measure them),
# the expert-parallel shard (96 of 384 experts, Ip=2304, routing over all
# 384) and a16w4 (384 top-6; 385 top-7 with the shared expert as expert
# 384; Ip=768), decode to prefill buckets.
PACKAGED_TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "block_m_gb300.csv")

MIN_GAIN = 0.01
MIN_WIN_FRACTION = 25 / 31
FIELDS = ["H", "Ip", "E", "topk", "a16", "max_tokens", "block_m", "default_block_m",
          "median_gain", "wins", "pairs", "control_gain", "control_wins",
          "prefetch1", "prefetch2", "prefetch_gain", "prefetch_wins",
          "split", "split_gain", "split_wins"]
CANDIDATES = (16, 32, 64, 128)
# (stage-1, stage-2) weight L2 prefetch leads tried against the defaults
# (a8w4 4/2, a16w4 8/8), in 128-K weight tiles
PREFETCH_CANDIDATES = ((8, 8), (24, 8), (32, 8), (16, 4), (16, 16), (4, 4))
# the GEMMs' split walk tried against the library's choice: the walk, whole tiles
SPLIT_CANDIDATES = (1, 2)


# ----------------------------------------------------------------- gate

def paired_gate(base: Sequence[float], cand: Sequence[float], min_gain: float = MIN_GAIN,
                min_win_fraction: float = MIN_WIN_FRACTION) -> dict:
    """base[i], cand[i]: the two measurements (times) of pair i. Adopt the
    candidate iff the median of (base - cand) / base is >= min_gain and the
    candidate is faster in at least ceil(min_win_fraction * pairs) pairs."""
    if len(base) != len(cand) or not base:
        raise ValueError("need the same, non-zero number of measurements on both sides")
    gains = [(b - c) / b for b, c in zip(base, cand)]
    wins = sum(1 for b, c in zip(base, cand) if c < b)
    need = math.ceil(min_win_fraction * len(base) - 1e-9)
    med = statistics.median(gains)
    return {"accept": med >= min_gain and wins >= need, "median_gain": med, "wins": wins,
            "pairs": len(base), "wins_needed": need}


# ---------------------------------------------------------------- table

# fields a row may lack (tables written before the prefetch or split knobs): 0
_OPTIONAL = {"prefetch1": 0, "prefetch2": 0, "prefetch_gain": 0.0, "prefetch_wins": 0,
             "split": 0, "split_gain": 0.0, "split_wins": 0}


def write_table(rows: Iterable[dict], path: str) -> None:
    with open(path, "w", newline="") as f:
        w = csv.DictWriter(f, fieldnames=FIELDS)
        w.writeheader()
        for r in rows:
            w.writerow({k: r.get(k, _OPTIONAL.get(k)) for k in FIELDS})


def read_table(path: str) -> List[dict]:
    with open(path, newline="") as f:
        rows = list(csv.DictReader(f))
    ints = ["H", "Ip", "E", "topk", "a16", "max_tokens", "block_m", "default_block_m", "wins",
            "pairs", "control_wins", "prefetch1", "prefetch2", "prefetch_wins", "split",
            "split_wins"]
    for r in rows:
        for k, v in _OPTIONAL.items():
            if r.get(k) in (None, ""):
                r[k] = v
        for k in ints:
            r[k] = int(r[k])
        for k in ("median_gain", "control_gain", "prefetch_gain", "split_gain"):
            r[k] = float(r[k])
    return rows


def table_for(rows: Iterable[dict], H: int, Ip: int, E: int, topk: int, a16: bool):
    """(max_tokens, block_m) rows of one geometry, by ascending max_tokens."""
    return sorted((r["max_tokens"], r["block_m"]) for r in rows
                  if (r["H"], r["Ip"], r["E"], r["topk"], r["a16"]) == (H, Ip, E, topk, int(a16)))


def packaged_table_for(H: int, Ip: int, E: int, topk: int, a16: bool):
    """The shipped GB300 rows of one geometry ([] when it was not tuned)."""
    return table_for(read_table(PACKAGED_TABLE), H, Ip, E, topk, a16)


# ------------------------------------------------------------ measuring

def random_layer(H: int, Ip: int, E: int, a16: bool, seed: int = 0, device: str = "cuda"):
    """MoeLayer with random MXFP4 weights: uniform codes, scale bytes
    127 + U{-8..-4} (the timing does not depend on the values)."""
    import torch
    from . import MoeLayer
    g = torch.Generator().manual_seed(seed)
    w1 = torch.randint(0, 256, (E, 2 * Ip, H // 2), generator=g, dtype=torch.uint8)
    w1s = (119 + torch.randint(0, 5, (E, 2 * Ip, H // 32), generator=g)).to(torch.uint8)
    w2 = torch.randint(0, 256, (E, H, Ip // 2), generator=g, dtype=torch.uint8)
    w2s = (119 + torch.randint(0, 5, (E, H, Ip // 32), generator=g)).to(torch.uint8)
    return MoeLayer(w1, w1s, w2, w2s, a16=a16, device=device)


def random_inputs(M: int, H: int, E: int, topk: int, seed: int = 0, device: str = "cuda",
                  E_route: Optional[int] = None, shared: bool = False):
    """BF16 tokens ~N(0,1), topk distinct experts per token uniformly at
    random over E_route experts (default E; an expert-parallel shard keeps
    only the ids below E, the others are dropped by the layer), routing
    weights = softmax of N(0,1) logits over the picks. shared: the last of
    the topk columns is the shared expert E - 1 with weight 1 (the routed
    picks are drawn over the other experts)."""
    import torch
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, H, generator=g).to(torch.bfloat16)
    k = topk - 1 if shared else topk
    span = E_route or (E - 1 if shared else E)
    ids = torch.argsort(torch.rand(M, span, generator=g), dim=1)[:, :k].to(torch.int32)
    w = torch.softmax(torch.randn(M, k, generator=g), dim=1)
    if shared:
        ids = torch.cat([ids, torch.full((M, 1), E - 1, dtype=torch.int32)], 1)
        w = torch.cat([w, torch.ones(M, 1)], 1)
    return x.to(device), ids.contiguous().to(device), w.contiguous().to(device)


class _Graph:
    """One captured fused call with its own output and workspace."""

    def __init__(self, layer, x, ids, w, block_m, stream, prefetch=(0, 0), split=0):
        import torch
        M, k = ids.shape
        self.out = torch.empty(M, layer.H, dtype=torch.bfloat16, device=x.device)
        from . import fused_moe_workspace_bytes
        nbytes = fused_moe_workspace_bytes(M, layer.H, layer.Ip, layer.E, k, layer.a16, block_m)
        self.ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
        with torch.cuda.stream(stream):
            for _ in range(2):
                layer(x, ids, w, out=self.out, ws=self.ws, block_m=block_m, prefetch=prefetch,
                      split=split)
            torch.cuda.synchronize()
            self.g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.g, stream=stream):
                layer(x, ids, w, out=self.out, ws=self.ws, block_m=block_m, prefetch=prefetch,
                      split=split)
        torch.cuda.synchronize()

    def measure(self, replays, flush, stream) -> float:
        """Sum of the device times of `replays` replays, L2 flushed before each."""
        import torch
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        total = 0.0
        with torch.cuda.stream(stream):
            for _ in range(replays):
                flush.zero_()
                e0.record(stream)
                self.g.replay()
                e1.record(stream)
                e1.synchronize()
                total += e0.elapsed_time(e1)
        return total


def _pairs(a: _Graph, b: _Graph, pairs, replays, flush, stream):
    ta, tb = [], []
    for i in range(pairs):
        # alternate which side goes first
        if i % 2 == 0:
            ta.append(a.measure(replays, flush, stream))
            tb.append(b.measure(replays, flush, stream))
        else:
            tb.append(b.measure(replays, flush, stream))
            ta.append(a.measure(replays, flush, stream))
    return ta, tb


def tune_geometry(H: int, Ip: int, E: int, topk: int, a16: bool, tokens: Sequence[int],
                  candidates: Sequence[int] = CANDIDATES, pairs: int = 31, replays: int = 16,
                  seed: int = 0, device: str = "cuda", log=print,
                  buckets: Optional[Sequence[int]] = None, E_route: Optional[int] = None,
                  shared: bool = False) -> List[dict]:
    """Measure at each token count of `tokens` and record the result for the
    matching entry of `buckets` (the row's max_tokens; default: the token
    count itself), as the pages measure a real decode row per bucket."""
    buckets = list(buckets) if buckets else list(tokens)
    if len(buckets) != len(tokens) or any(b < t for b, t in zip(buckets, tokens)):
        raise ValueError("one bucket bound >= each measured token count")
    import torch
    from . import fused_moe_workspace_layout
    layer = random_layer(H, Ip, E, a16, seed, device)
    stream = torch.cuda.Stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    rows = []
    for M, bucket in zip(tokens, buckets):
        x, ids, w = random_inputs(M, H, E, topk, seed + M, device, E_route, shared)
        default = fused_moe_workspace_layout(M, H, Ip, E, topk, a16)["block_m"]
        base = _Graph(layer, x, ids, w, default, stream)
        twin = _Graph(layer, x, ids, w, default, stream)
        ca, cb = _pairs(base, twin, pairs, replays, flush, stream)
        control = paired_gate(ca, cb)
        best = {"block_m": default, "median_gain": 0.0, "wins": 0, "pairs": pairs}
        for bm in candidates:
            if bm == default:
                continue
            cand = _Graph(layer, x, ids, w, bm, stream)
            tb, tc = _pairs(base, cand, pairs, replays, flush, stream)
            gate = paired_gate(tb, tc)
            log(f"M={M:6d} default {default:3d} vs {bm:3d}: median gain "
                f"{100 * gate['median_gain']:+6.2f}%  wins {gate['wins']}/{pairs}  "
                f"{'ADOPT' if gate['accept'] else 'keep'}  (base {statistics.median(tb) / replays * 1e3:8.1f} us)")
            if gate["accept"] and gate["median_gain"] > best["median_gain"]:
                best = {"block_m": bm, "median_gain": gate["median_gain"], "wins": gate["wins"],
                        "pairs": pairs}
            del cand
        log(f"M={M:6d} control: median gain {100 * control['median_gain']:+6.2f}%  "
            f"wins {control['wins']}/{pairs}  {'PASSED (bias!)' if control['accept'] else 'rejected'}")
        rows.append({"H": H, "Ip": Ip, "E": E, "topk": topk, "a16": int(a16), "max_tokens": bucket,
                     "block_m": best["block_m"], "default_block_m": default,
                     "median_gain": round(best["median_gain"], 5), "wins": best["wins"],
                     "pairs": pairs, "control_gain": round(control["median_gain"], 5),
                     "control_wins": control["wins"]})
    return rows


def tune_prefetch(rows: List[dict], candidates=PREFETCH_CANDIDATES, pairs: int = 31,
                  replays: int = 16, seed: int = 0, device: str = "cuda", log=print,
                  tokens: Optional[Sequence[int]] = None, E_route: Optional[int] = None,
                  shared: bool = False) -> List[dict]:
    """Second knob: for each row of one geometry (its block_m fixed), the
    weight L2 prefetch leads, under the same gate against the defaults.
    tokens[i] is the count measured for rows[i] (default: its max_tokens)."""
    import torch
    if not rows:
        return rows
    r0 = rows[0]
    H, Ip, E, topk, a16 = r0["H"], r0["Ip"], r0["E"], r0["topk"], bool(r0["a16"])
    tokens = list(tokens) if tokens else [r["max_tokens"] for r in rows]
    layer = random_layer(H, Ip, E, a16, seed, device)
    stream = torch.cuda.Stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    out = []
    for r, M in zip(rows, tokens):
        x, ids, w = random_inputs(M, H, E, topk, seed + M, device, E_route, shared)
        bm, sp = r["block_m"], r.get("split", 0)   # the row's split walk stays as it is
        base = _Graph(layer, x, ids, w, bm, stream, split=sp)
        best = {"prefetch": (0, 0), "median_gain": 0.0, "wins": 0}
        for pf in candidates:
            cand = _Graph(layer, x, ids, w, bm, stream, prefetch=pf, split=sp)
            tb, tc = _pairs(base, cand, pairs, replays, flush, stream)
            gate = paired_gate(tb, tc)
            log(f"M={M:6d} block_m {bm:3d} prefetch default vs {pf}: median gain "
                f"{100 * gate['median_gain']:+6.2f}%  wins {gate['wins']}/{pairs}  "
                f"{'ADOPT' if gate['accept'] else 'keep'}")
            if gate["accept"] and gate["median_gain"] > best["median_gain"]:
                best = {"prefetch": pf, "median_gain": gate["median_gain"], "wins": gate["wins"]}
            del cand
        r = dict(r)
        r["prefetch1"], r["prefetch2"] = best["prefetch"]
        r["prefetch_gain"] = round(best["median_gain"], 5)
        r["prefetch_wins"] = best["wins"]
        out.append(r)
    return out


def tune_split(rows: List[dict], candidates=SPLIT_CANDIDATES, pairs: int = 31,
               replays: int = 16, seed: int = 0, device: str = "cuda", log=print,
               tokens: Optional[Sequence[int]] = None, E_route: Optional[int] = None,
               shared: bool = False) -> List[dict]:
    """Third knob: for each row of one geometry (its block_m and prefetch
    leads fixed), the GEMMs' split walk (1 = the walk, 2 = whole tiles only)
    against the library's choice, under the same gate. tokens[i] is the count measured for
    rows[i] (default: its max_tokens)."""
    import torch
    if not rows:
        return rows
    r0 = rows[0]
    H, Ip, E, topk, a16 = r0["H"], r0["Ip"], r0["E"], r0["topk"], bool(r0["a16"])
    tokens = list(tokens) if tokens else [r["max_tokens"] for r in rows]
    layer = random_layer(H, Ip, E, a16, seed, device)
    stream = torch.cuda.Stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    out = []
    for r, M in zip(rows, tokens):
        x, ids, w = random_inputs(M, H, E, topk, seed + M, device, E_route, shared)
        bm, pf = r["block_m"], (r["prefetch1"], r["prefetch2"])
        base = _Graph(layer, x, ids, w, bm, stream, prefetch=pf)
        best = {"split": 0, "median_gain": 0.0, "wins": 0}
        for sp in candidates:
            cand = _Graph(layer, x, ids, w, bm, stream, prefetch=pf, split=sp)
            tb, tc = _pairs(base, cand, pairs, replays, flush, stream)
            gate = paired_gate(tb, tc)
            log(f"M={M:6d} block_m {bm:3d} split default vs {sp}: median gain "
                f"{100 * gate['median_gain']:+6.2f}%  wins {gate['wins']}/{pairs}  "
                f"{'ADOPT' if gate['accept'] else 'keep'}")
            if gate["accept"] and gate["median_gain"] > best["median_gain"]:
                best = {"split": sp, "median_gain": gate["median_gain"], "wins": gate["wins"]}
            del cand
        r = dict(r)
        r["split"] = best["split"]
        r["split_gain"] = round(best["median_gain"], 5)
        r["split_wins"] = best["wins"]
        out.append(r)
    return out


def main(argv: Optional[Sequence[str]] = None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--H", type=int, required=True)
    ap.add_argument("--Ip", type=int, required=True)
    ap.add_argument("--E", type=int, required=True)
    ap.add_argument("--topk", type=int, required=True)
    ap.add_argument("--a16", action="store_true")
    ap.add_argument("--tokens", type=int, nargs="+", required=True,
                    help="token counts measured")
    ap.add_argument("--buckets", type=int, nargs="+",
                    help="bucket bound (max_tokens) recorded for each measured count")
    ap.add_argument("--candidates", type=int, nargs="+", default=list(CANDIDATES))
    ap.add_argument("--pairs", type=int, default=31)
    ap.add_argument("--replays", type=int, default=16)
    ap.add_argument("--E-route", type=int, default=None,
                    help="experts the routing draws from (expert-parallel shard: the global count)")
    ap.add_argument("--shared", action="store_true",
                    help="the last routing column is the shared expert E-1 (weight 1)")
    ap.add_argument("--knob", choices=["block_m", "prefetch", "split"], default="block_m",
                    help="prefetch / split: tune the weight prefetch leads / the split walk of "
                         "the geometry's rows in --table (their other settings fixed), "
                         "measured at --tokens")
    ap.add_argument("--table", default=PACKAGED_TABLE,
                    help="rows the prefetch and split passes start from")
    ap.add_argument("--pf-candidates", nargs="+", default=None,
                    help="prefetch pass: candidate leads as STAGE1,STAGE2 (e.g. 4,4 2,2)")
    ap.add_argument("--split-candidates", type=int, nargs="+", default=list(SPLIT_CANDIDATES),
                    help="split pass: split values tried against the library's choice")
    ap.add_argument("--out", required=True)
    ap.add_argument("--append", action="store_true", help="keep the rows already in --out")
    a = ap.parse_args(argv)
    if a.knob in ("prefetch", "split"):
        mine = [r for r in read_table(a.table)
                if (r["H"], r["Ip"], r["E"], r["topk"], r["a16"]) == (a.H, a.Ip, a.E, a.topk,
                                                                       int(a.a16))]
        mine.sort(key=lambda r: r["max_tokens"])
        if len(mine) != len(a.tokens):
            raise SystemExit(f"{len(mine)} rows of this geometry in --table, {len(a.tokens)} tokens")
    if a.knob == "prefetch":
        cands = (tuple(tuple(int(v) for v in c.split(",")) for c in a.pf_candidates)
                 if a.pf_candidates else PREFETCH_CANDIDATES)
        rows = tune_prefetch(mine, candidates=cands, pairs=a.pairs, replays=a.replays,
                             tokens=a.tokens, E_route=a.E_route, shared=a.shared)
    elif a.knob == "split":
        rows = tune_split(mine, candidates=tuple(a.split_candidates), pairs=a.pairs,
                          replays=a.replays, tokens=a.tokens, E_route=a.E_route, shared=a.shared)
    else:
        rows = tune_geometry(a.H, a.Ip, a.E, a.topk, a.a16, a.tokens, a.candidates, a.pairs,
                             a.replays, buckets=a.buckets, E_route=a.E_route, shared=a.shared)
    if a.append:
        import os
        if os.path.exists(a.out):
            rows = read_table(a.out) + rows
    write_table(rows, a.out)


if __name__ == "__main__":
    main()
