"""Seeded synthetic inputs for the block-scaled fused MoE layer.

This module only draws random numbers and lays them out in the byte formats
the layer consumes. It contains none of the layer's arithmetic (no decoding,
no quantisation, no sorting, no matmul), so the CPU oracle and the CUDA path
can both take their inputs from here without sharing any of the method.

Shapes follow the DeepSeek-V4.1-Flash MoE geometries the tuning pages describe:

* TP4 backbone / draft: H=5120, TP-local intermediate 576 padded to 640,
  384 experts top-6 / 128 experts top-3
  (AITER #5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Configuration).
* Expert-parallel local shard: H=5120, I=2304, 96 local experts, top-6
  (AITER #5904 "Add tuned a8w4 fused-MoE configs for DeepSeek V4.1-Flash
  (TP4 + EP, gfx950)", first paragraph).
* a16w4: w1 N=1536 (I=768) K=5120, w2 N=5120 K=768; 384 experts top-6 or
  385 experts top-7 with a fused shared expert
  (AITER #6286 "Retune gfx942 a16w4 DSv4.1 tiles for Triton 3.8", reviewer
  tables).

Byte formats produced (all row-major, C-contiguous):

* ``x``: bfloat16 [M, H], N(0, 1) rounded to bfloat16.
* ``topk_ids``: int32 [M, k]; distinct experts per token.  For the
  expert-parallel shard the ids are global (0..383) and only ids < E are local.
* ``topk_weights``: float32 [M, k], softmax of N(0, 1) logits over the k picks.
* ``w1``: uint8 [E, 2*Ip, H/2], E2M1 codes two per byte, element k in byte
  k/2, low nibble = even k. Row 2j is gate_j, row 2j+1 is up_j. Rows >= 2*I
  (intermediate padding) are zero codes.
* ``w1_scale``: uint8 [E, 2*Ip, H/32], E8M0 bytes, 127 + U{-8..-4}.
* ``w2``: uint8 [E, H, Ip/2]; columns >= I are zero codes.
* ``w2_scale``: uint8 [E, H, Ip/32].

Seeds: per-call inputs (x, routing) use ``1000*config + M + 100000*variant``;
weights use ``1000*config + 100000*variant + 7`` so a sweep over M reuses one
weight set.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

H_DSV41 = 5120


@dataclasses.dataclass(frozen=True)
class MoeShape:
    name: str
    H: int            # model dim (stage-1 K, stage-2 N)
    I: int            # logical intermediate size
    Ip: int           # stored (padded) intermediate size
    E: int            # local experts the kernels see
    topk: int         # routes per token
    E_route: int      # experts the router picks from (global for EP)
    a16: bool = False  # True: BF16 activations (a16w4); False: FP8 (a8w4)
    shared_expert: bool = False  # last column is expert E-1 with weight 1.0


# config index -> shape (variant picks b / hot where relevant)
SHAPES = {
    "draft": MoeShape("draft", H_DSV41, 576, 640, 128, 3, 128),
    "backbone": MoeShape("backbone", H_DSV41, 576, 640, 384, 6, 384),
    "ep": MoeShape("ep", H_DSV41, 2304, 2304, 96, 6, 384),
    "a16w4_384": MoeShape("a16w4_384", H_DSV41, 768, 768, 384, 6, 384, a16=True),
    "a16w4_385": MoeShape("a16w4_385", H_DSV41, 768, 768, 385, 7, 384, a16=True,
                          shared_expert=True),
}

# The token counts of each workload (decode buckets and prefill sizes).
TOKENS = {
    "draft": [5],
    "backbone": [6, 12, 24, 48, 96, 192, 384, 768],
    "backbone_boundary": [31, 32, 33, 255, 256, 257],
    "ep": [1, 4, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192, 16384],
    "a16w4": [12, 256, 1024, 1536, 4096, 16384],
    "zipf": [16384],
}

CONFIG_INDEX = {"draft": 0, "backbone": 1, "ep": 2, "a16w4_384": 3,
                "a16w4_385": 3, "zipf": 4}


def call_seed(config: int, M: int, variant: int = 0) -> int:
    return 1000 * config + M + 100000 * variant


def weight_seed(config: int, variant: int = 0) -> int:
    return 1000 * config + 100000 * variant + 7


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def make_x(M: int, H: int, g: torch.Generator) -> torch.Tensor:
    return torch.randn(M, H, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _softmax_weights(M: int, k: int, g: torch.Generator) -> torch.Tensor:
    logits = torch.randn(M, k, generator=g, dtype=torch.float32)
    return torch.softmax(logits, dim=1).contiguous()


def route_uniform(M: int, k: int, E_route: int, g: torch.Generator) -> torch.Tensor:
    """k distinct experts per token, uniformly at random."""
    if M == 0:
        return torch.zeros(0, k, dtype=torch.int32)
    u = torch.rand(M, E_route, generator=g)
    return u.topk(k, dim=1).indices.to(torch.int32).contiguous()


def route_hot(M: int, k: int, E: int, g: torch.Generator, n_hot: int = 16,
              p_hot: float = 0.8) -> torch.Tensor:
    """Concentrated routing: Binomial(k, p_hot) of each token's k distinct
    routes go to a fixed random set of ``n_hot`` experts, the rest to the
    others, so 80% of routes hit the hot set in expectation."""
    perm = torch.randperm(E, generator=g)
    hot, cold = perm[:n_hot], perm[n_hot:]
    # Binomial(k, p_hot) as a sum of k Bernoulli draws from the seeded generator
    nh = (torch.rand(M, k, generator=g) < p_hot).sum(dim=1)
    ids = torch.empty(M, k, dtype=torch.int64)
    uh = torch.rand(M, n_hot, generator=g).argsort(dim=1)
    uc = torch.rand(M, E - n_hot, generator=g).argsort(dim=1)
    for t in range(M):
        h = int(nh[t])
        ids[t, :h] = hot[uh[t, :h]]
        ids[t, h:] = cold[uc[t, :k - h]]
    # shuffle the column order so hot picks are not always first
    order = torch.rand(M, k, generator=g).argsort(dim=1)
    ids = torch.gather(ids, 1, order)
    return ids.to(torch.int32).contiguous()


def route_zipf(M: int, k: int, E: int, g: torch.Generator, s: float = 1.2) -> torch.Tensor:
    """k distinct experts per token drawn without replacement from a Zipf(s)
    popularity over a random permutation of the experts."""
    perm = torch.randperm(E, generator=g)
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    p_rank = ranks.pow(-s)
    p = torch.empty(E, dtype=torch.float64)
    p[perm] = p_rank
    p = (p / p.sum()).to(torch.float32)
    ids = torch.multinomial(p.expand(M, E).contiguous(), k, replacement=False, generator=g)
    return ids.to(torch.int32).contiguous()


def make_routing(shape: MoeShape, M: int, g: torch.Generator, mode: str = "uniform"):
    k = shape.topk
    if shape.shared_expert:
        kr = k - 1
        ids = route_uniform(M, kr, shape.E - 1, g)
        w = _softmax_weights(M, kr, g)
        ids = torch.cat([ids, torch.full((M, 1), shape.E - 1, dtype=torch.int32)], 1)
        w = torch.cat([w, torch.ones(M, 1, dtype=torch.float32)], 1)
        return ids.contiguous(), w.contiguous()
    if mode == "uniform":
        ids = route_uniform(M, k, shape.E_route, g)
    elif mode == "hot":
        ids = route_hot(M, k, shape.E_route, g)
    elif mode == "zipf":
        ids = route_zipf(M, k, shape.E_route, g)
    else:
        raise ValueError(mode)
    w = _softmax_weights(M, k, g)
    return ids, w


def _codes(n_rows: int, n_bytes: int, rng: np.random.Generator) -> torch.Tensor:
    # uniform bytes (both nibbles uniform over the 16 E2M1 codes), taken from
    # the raw 64-bit PCG64 stream, little-endian
    n = n_rows * n_bytes
    raw = rng.bit_generator.random_raw((n + 7) // 8)
    buf = raw.view(np.uint8)[:n]
    return torch.from_numpy(buf).view(n_rows, n_bytes)


def _scales(n_rows: int, n_blocks: int, rng: np.random.Generator) -> torch.Tensor:
    # E8M0 exponents uniform in [-8, -4]
    v = rng.integers(127 - 8, 127 - 3, size=(n_rows, n_blocks), dtype=np.uint8)
    return torch.from_numpy(v)


def make_weights(shape: MoeShape, seed: int, experts: Optional[int] = None):
    """MXFP4 expert weights in the canonical byte layout (see module doc).
    Drawn with numpy's PCG64 (platform-independent) for speed."""
    g = np.random.Generator(np.random.PCG64(seed))
    E = shape.E if experts is None else experts
    H, I, Ip = shape.H, shape.I, shape.Ip
    w1 = _codes(E * 2 * Ip, H // 2, g).view(E, 2 * Ip, H // 2)
    w1s = _scales(E * 2 * Ip, H // 32, g).view(E, 2 * Ip, H // 32)
    w2 = _codes(E * H, Ip // 2, g).view(E, H, Ip // 2)
    w2s = _scales(E * H, Ip // 32, g).view(E, H, Ip // 32)
    if Ip > I:
        w1[:, 2 * I:, :] = 0
        w2[:, :, I // 2:] = 0
    return dict(w1=w1.contiguous(), w1_scale=w1s.contiguous(),
                w2=w2.contiguous(), w2_scale=w2s.contiguous())


@dataclasses.dataclass
class MoeCase:
    shape: MoeShape
    M: int
    x: torch.Tensor
    topk_ids: torch.Tensor
    topk_weights: torch.Tensor
    w1: torch.Tensor
    w1_scale: torch.Tensor
    w2: torch.Tensor
    w2_scale: torch.Tensor
    seed: int


def make_case(shape_name: str, M: int, variant: int = 0, routing: str = "uniform",
              weights: Optional[dict] = None, shape: Optional[MoeShape] = None) -> MoeCase:
    """Build one seeded case. ``shape`` overrides the named geometry (used
    for reduced-size test shapes); ``weights`` reuses a weight set."""
    shp = shape if shape is not None else SHAPES[shape_name]
    cfg = CONFIG_INDEX.get(shape_name, 9)
    if routing == "zipf":
        cfg = 4
    if routing == "hot":
        variant = max(variant, 1)
    if weights is None:
        weights = make_weights(shp, weight_seed(cfg, variant))
    seed = call_seed(cfg, M, variant)
    g = _gen(seed)
    x = make_x(M, shp.H, g)
    ids, w = make_routing(shp, M, g, routing)
    return MoeCase(shp, M, x, ids, w, weights["w1"], weights["w1_scale"],
                   weights["w2"], weights["w2_scale"], seed)


def small_shape(H: int = 256, I: int = 96, Ip: int = 128, E: int = 8, topk: int = 2,
                E_route: Optional[int] = None, a16: bool = False,
                shared_expert: bool = False) -> MoeShape:
    """A reduced geometry with the same structure, for fast exhaustive tests."""
    return MoeShape("small", H, I, Ip, E, topk, E if E_route is None else E_route,
                    a16=a16, shared_expert=shared_expert)
