"""Plain CPU reference of the gating step in front of the route sort.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module. It shares no
code with the CUDA path.

What it computes. The pages time the fused MoE call "including gating"
(AITER #5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Performance
on the measured runtime) but do not define the gate. The plainest reading,
and the one the synthetic routing of this repository already follows
(routing weights = softmax over the chosen experts' logits), is:

1. per token t, select the ``topk`` experts with the largest router logits
   L[t, e]; equal logits are taken in ascending expert order, and the
   selected experts are listed in that order (descending logit, then
   ascending expert);
2. the routing weight of a selected expert is the softmax of L[t, .] over
   the selected experts only (equivalently the full softmax renormalised
   over the top k);
3. optionally, a shared expert id is appended as a last column with weight
   1.0 (the 385-expert top-7 layout of AITER #6286 "Retune gfx942 a16w4
   DSv4.1 tiles for Triton 3.8", where expert 384 is always selected); a
   shared expert stored as n pieces (see ``moe.shared_expert_pieces``)
   takes n such columns, ids shared_id .. shared_id + n - 1.

The selection compares the FP32 logits themselves (an ordering, exact in
any precision); the softmax is evaluated in FP64.
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def router_topk(logits, topk: int, shared_id: Optional[int] = None, n_shared: int = 1):
    """logits float32 [M, E] -> (ids int32 [M, k'], weights float64 [M, k'])
    with k' = topk (+ n_shared with a shared expert)."""
    L = np.asarray(logits, dtype=np.float32)
    M, E = L.shape
    if not 1 <= topk <= E:
        raise ValueError("topk must be in [1, E]")
    # step 1: descending logit, ties by ascending expert (stable sort of -L)
    order = np.argsort(-L, axis=1, kind="stable")[:, :topk]
    sel = np.take_along_axis(L, order, axis=1).astype(np.float64)
    # step 2: softmax over the selected logits (shifted by their maximum,
    # which is the first selected one)
    e = np.exp(sel - sel[:, :1])
    w = e / e.sum(axis=1, keepdims=True)
    ids = order.astype(np.int32)
    if shared_id is not None:
        # step 3: the always-selected shared expert (its n_shared pieces)
        sh = np.arange(shared_id, shared_id + n_shared, dtype=np.int32)
        ids = np.concatenate([ids, np.broadcast_to(sh, (M, n_shared))], axis=1)
        w = np.concatenate([w, np.ones((M, n_shared), dtype=np.float64)], axis=1)
    return ids, w
