"""Plain FP64 CPU reference of the block-scaled two-stage fused MoE layer.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module. It shares no
code with the CUDA path and is slow on purpose: each step is written out in
the order the pages list it, with numpy FP64 matmuls as the only library
primitive besides a stable argsort.

What one call computes (a8w4; the pages' wording is summarised in brackets):

1. sort   - group the token-expert routes by expert and pad each expert's
            group to a multiple of block_m ["the sorter", AITER #5609,
            Performance on the measured runtime; "sorting", AITER #5904,
            Fused-MoE kernel expert-parallel benchmark]
2. quant  - BF16 tokens -> FP8 E4M3 + one E8M0 scale per 1x32 along K
            [AITER #5609, Configuration: FP8 activations, per-1x32 scaling]
3. stage1 - per expert, x . W1^T with W1 the interleaved gate/up MXFP4 rows
            [AITER #5609, Configuration: MXFP4 weights, interleaved gate/up]
4. act    - SiLU(gate) * up, no routing-weight multiply; requantise to FP8
            per 1x32 ["the intermediate quantization", AITER #5904,
            Fused-MoE kernel expert-parallel benchmark; AITER #5609,
            Configuration: SiLU and no stage-one routing-weight
            multiplication]
5. stage2 - per expert, a . W2^T (down projection)
6. reduce - out[t] = sum_j w[t, j] * y[t, j], rounded once to BF16
            [AITER #5609, Configuration: BF16 output]

a16w4 (AITER #6286 "Retune gfx942 a16w4 DSv4.1 tiles for Triton 3.8",
reviewer reply: "w1 with apply_swiglu=True, w2 separate, bf16, MXFP4")
skips step 2 (activations stay BF16) and rounds the step-4 intermediate to
BF16 instead of FP8.

Readings where the pages are silent (each listed in the design notes):
E4M3 is the OCP "fn" flavour; the 1x32 scale rule is the OCP MX one; an
all-zero block has scale byte 0 and zero codes; gate/up interleave is row by
row (2j = gate_j, 2j+1 = up_j); routes to experts outside [0, E) are
dropped (expert-parallel shard); ties inside an expert keep ascending route
index r = t*topk + j; pad entries use the sentinel route M*topk and weight 0;
the final sum is rounded from FP64 straight to BF16.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

from . import mx_formats as mx


def _np(a) -> np.ndarray:
    if hasattr(a, "detach"):
        t = a.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            import torch
            return t.to(torch.float64).numpy()
        return t.numpy()
    return np.asarray(a)


# --------------------------------------------------------------------- sort

@dataclasses.dataclass
class SortResult:
    sorted_route: np.ndarray   # int32 [P]: route index r = t*topk + j, pad = M*topk
    sorted_w: np.ndarray       # float32 [P]: routing weight, pad = 0
    block_expert: np.ndarray   # int32 [P / block_m]
    expert_off: np.ndarray     # int32 [E + 1]: padded segment starts
    expert_cnt: np.ndarray     # int32 [E]: valid routes per expert
    route_pos: np.ndarray      # int32 [M*topk]: sorted position of r, -1 if dropped
    num_padded: int            # P


def moe_sort(topk_ids, topk_weights, E: int, block_m: int) -> SortResult:
    """Stable counting sort of the routes by expert id, each expert's
    segment padded up to a multiple of ``block_m`` (empty experts take no
    block). Routes whose id is outside [0, E) are dropped."""
    ids = _np(topk_ids).astype(np.int64).reshape(-1)
    w = _np(topk_weights).astype(np.float32).reshape(-1)
    R = ids.size
    r = np.arange(R, dtype=np.int64)
    valid = (ids >= 0) & (ids < E)
    cnt = np.bincount(ids[valid], minlength=E).astype(np.int64)
    padded = -(-cnt // block_m) * block_m
    off = np.zeros(E + 1, dtype=np.int64)
    off[1:] = np.cumsum(padded)
    P = int(off[E])
    sorted_route = np.full(P, R, dtype=np.int32)
    sorted_w = np.zeros(P, dtype=np.float32)
    route_pos = np.full(R, -1, dtype=np.int32)
    vr = r[valid]
    ve = ids[valid]
    order = np.argsort(ve, kind="stable")   # ascending expert, then ascending r
    vr, ve = vr[order], ve[order]
    seg_start = np.zeros(E + 1, dtype=np.int64)
    seg_start[1:] = np.cumsum(cnt)
    rank = np.arange(vr.size) - seg_start[ve]
    pos = off[ve] + rank
    sorted_route[pos] = vr
    sorted_w[pos] = w[vr]
    route_pos[vr] = pos
    block_expert = np.repeat(np.arange(E, dtype=np.int32), padded // block_m)
    return SortResult(sorted_route, sorted_w, block_expert.astype(np.int32),
                      off.astype(np.int32), cnt.astype(np.int32), route_pos, P)


# ------------------------------------------------------------ full layer

@dataclasses.dataclass
class MoeResult:
    out_bf16: np.ndarray          # float64 [M or len(tokens), H], BF16 values
    out_f64: np.ndarray           # float64 pre-rounding sum
    sort: SortResult
    inter_rows: np.ndarray        # int64: sorted positions p of the rows below
    aq: np.ndarray                # uint8 [rows, Ip] FP8 codes (a8w4) / float64 BF16 values (a16w4)
    as_: Optional[np.ndarray]     # uint8 [rows, Ip/32] (a8w4)
    tokens: np.ndarray            # int64 token ids of out rows


def _silu_mul(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return gate / (1.0 + np.exp(-gate)) * up


def fused_moe(x, topk_ids, topk_weights, w1, w1_scale, w2, w2_scale, E: int,
              a16: bool = False, block_m: int = 16,
              tokens: Optional[Sequence[int]] = None,
              experts: Optional[Sequence[int]] = None) -> MoeResult:
    """Reference output of one fused MoE call.

    ``x`` BF16 [M, H]; ``topk_ids`` int32 [M, k]; ``topk_weights`` FP32
    [M, k]; ``w1`` uint8 [E, 2*Ip, H/2]; ``w1_scale`` uint8 [E, 2*Ip, H/32];
    ``w2`` uint8 [E, H, Ip/2]; ``w2_scale`` uint8 [E, H, Ip/32].

    ``tokens`` restricts the work to those tokens' routes (outputs one row
    per listed token) so large cases can be checked on a sample; ``experts``
    restricts it further to routes of those experts (the CPU baseline uses
    this to time a bounded slice of a call).
    """
    xf = _np(x).astype(np.float64)
    ids = _np(topk_ids).astype(np.int64)
    wts = _np(topk_weights).astype(np.float32)
    M, H = xf.shape
    k = ids.shape[1]
    W1, W1s, W2, W2s = (_np(a) for a in (w1, w1_scale, w2, w2_scale))
    Ip = W2.shape[2] * 2
    assert W1.shape == (W1.shape[0], 2 * Ip, H // 2)

    srt = moe_sort(ids, wts, E, block_m)

    tok_sel = np.arange(M) if tokens is None else np.asarray(tokens, dtype=np.int64)
    want_tok = np.zeros(M, dtype=bool)
    want_tok[tok_sel] = True
    want_exp = np.ones(E, dtype=bool)
    if experts is not None:
        want_exp[:] = False
        want_exp[np.asarray(experts, dtype=np.int64)] = True

    # step 2: activation quantisation (a8w4) - dequantised operand for step 3.
    # The rule acts on each token row on its own, so only the rows of tokens
    # that have a computed route are quantised.
    if a16:
        xdq = xf                                   # BF16 values are exact in FP64
    else:
        valid = (ids >= 0) & (ids < E)
        used = want_tok & (valid & want_exp[np.where(valid, ids, 0)]).any(axis=1)
        xdq = np.zeros_like(xf)
        if used.any():
            xq, xs = mx.quant_mxfp8(xf[used])
            xdq[used] = mx.dequant_mxfp8(xq, xs)

    out = np.zeros((M, H), dtype=np.float64)
    inter_rows, aq_rows, as_rows = [], [], []

    for e in range(E):
        if not want_exp[e]:
            continue
        lo = int(srt.expert_off[e])
        p = lo + np.arange(int(srt.expert_cnt[e]))
        if p.size == 0:
            continue
        r = srt.sorted_route[p].astype(np.int64)
        t = r // k
        keep = want_tok[t]
        p, r, t = p[keep], r[keep], t[keep]
        if p.size == 0:
            continue
        # step 3: stage-one GEMM against this expert's gate/up rows
        w1dq = mx.dequant_mxfp4(W1[e], W1s[e])          # [2*Ip, H]
        h = xdq[t] @ w1dq.T                              # [n, 2*Ip]
        # step 4: SiLU(gate) * up, gate/up interleaved row by row
        act = _silu_mul(h[:, 0::2], h[:, 1::2])          # [n, Ip]
        if a16:
            adq = mx.bf16_round(act)
            aq_rows.append(adq)
        else:
            aq, as_ = mx.quant_mxfp8(act)
            adq = mx.dequant_mxfp8(aq, as_)
            aq_rows.append(aq)
            as_rows.append(as_)
        inter_rows.append(p)
        # step 5: stage-two GEMM (down projection)
        w2dq = mx.dequant_mxfp4(W2[e], W2s[e])          # [H, Ip]
        y = adq @ w2dq.T                                 # [n, H]
        # step 6: routing-weighted sum into the token rows
        wr = wts.reshape(-1)[r].astype(np.float64)
        np.add.at(out, t, wr[:, None] * y)

    out_sel = out[tok_sel]
    if inter_rows:
        rows = np.concatenate(inter_rows)
        aq_all = np.concatenate(aq_rows)
        as_all = None if a16 else np.concatenate(as_rows)
    else:
        rows = np.zeros(0, dtype=np.int64)
        aq_all = np.zeros((0, Ip), dtype=np.float64 if a16 else np.uint8)
        as_all = None if a16 else np.zeros((0, Ip // 32), dtype=np.uint8)
    return MoeResult(mx.bf16_round(out_sel), out_sel, srt, rows, aq_all, as_all, tok_sel)


# ------------------------------------------------------- shared expert

def shared_mlp(x, w1, w1_scale, w2, w2_scale, a16: bool = False) -> np.ndarray:
    """The shared expert as a dense MLP over every token, FP64 output before
    rounding [M, H]: the same steps as one expert of the layer (activation
    quantisation, gate/up GEMM, SiLU(gate)*up, intermediate requantisation,
    down projection) with routing weight 1. ``w1`` uint8 [2*Is, H/2],
    ``w1_scale`` [2*Is, H/32], ``w2`` [H, Is/2], ``w2_scale`` [H, Is/32]; Is
    may differ from the routed experts' intermediate size."""
    xf = _np(x)
    M = xf.shape[0]
    ids = np.zeros((M, 1), dtype=np.int32)
    w = np.ones((M, 1), dtype=np.float32)
    W = [np.asarray(_np(a))[None] for a in (w1, w1_scale, w2, w2_scale)]
    return fused_moe(x, ids, w, *W, 1, a16=a16).out_f64


def fused_moe_with_shared(x, topk_ids, topk_weights, w1, w1_scale, w2, w2_scale, E: int,
                          shared, a16: bool = False) -> np.ndarray:
    """Routed experts plus a separate shared expert ``shared`` = (w1,
    w1_scale, w2, w2_scale) of its own intermediate size, added with weight
    1 to every token (the "shared expert" of AITER #5609 "Add DeepSeek V4.1
    Flash TP4 gfx950 MoE tuning", Performance on the measured runtime): the
    two FP64 sums are added and rounded to BF16 once. Returns BF16 values
    (float64) [M, H]."""
    routed = fused_moe(x, topk_ids, topk_weights, w1, w1_scale, w2, w2_scale, E, a16=a16)
    return mx.bf16_round(routed.out_f64 + shared_mlp(x, *shared, a16=a16))


def shared_expert_pieces(w1, w1_scale, w2, w2_scale, Ip: int):
    """A shared expert of intermediate size Is as ceil(Is / Ip) experts of
    intermediate size Ip: piece j holds intermediate indices [j*Ip, (j+1)*Ip)
    (gate/up rows 2i, 2i+1 of w1, columns of w2), zero-padded at the end.
    SiLU(gate)*up acts on each intermediate index alone and the down
    projection sums over them, so the shared MLP is the sum of its pieces'
    outputs; Ip is a multiple of 32, so no 1x32 block of the intermediate
    straddles two pieces. Returns stacked [n, ...] arrays in the layer's
    expert layout."""
    W1, S1, W2, S2 = (np.asarray(_np(a)) for a in (w1, w1_scale, w2, w2_scale))
    Is = W2.shape[1] * 2
    n = -(-Is // Ip)
    H2 = W1.shape[1]
    p1 = np.zeros((n, 2 * Ip, H2), dtype=np.uint8)
    q1 = np.zeros((n, 2 * Ip, S1.shape[1]), dtype=np.uint8)
    p2 = np.zeros((n, W2.shape[0], Ip // 2), dtype=np.uint8)
    q2 = np.zeros((n, W2.shape[0], Ip // 32), dtype=np.uint8)
    for j in range(n):
        lo, hi = j * Ip, min((j + 1) * Ip, Is)
        p1[j, :2 * (hi - lo)] = W1[2 * lo:2 * hi]
        q1[j, :2 * (hi - lo)] = S1[2 * lo:2 * hi]
        p2[j, :, :(hi - lo) // 2] = W2[:, lo // 2:hi // 2]
        q2[j, :, :(hi - lo) // 32] = S2[:, lo // 32:hi // 32]
    return p1, q1, p2, q2

