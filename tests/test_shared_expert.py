"""Host side of the separate shared expert: its tensors are split into
pieces of the routed intermediate size and appended to the routed experts
(shape checks included), on CPU."""
import pytest
import torch

from block_scaled_moe_sort_gb300 import shared_expert_pieces, with_shared_expert


def _tensors(E, Ip=128, H=256, seed=None):
    g = torch.Generator().manual_seed(E if seed is None else seed)
    return (torch.randint(0, 256, (E, 2 * Ip, H // 2), generator=g, dtype=torch.uint8),
            torch.randint(118, 124, (E, 2 * Ip, H // 32), generator=g, dtype=torch.uint8),
            torch.randint(0, 256, (E, H, Ip // 2), generator=g, dtype=torch.uint8),
            torch.randint(118, 124, (E, H, Ip // 32), generator=g, dtype=torch.uint8))


@pytest.mark.parametrize("squeeze", [False, True])
def test_shared_expert_of_routed_size_is_one_appended_expert(squeeze):
    routed = _tensors(5)
    shared = _tensors(1)
    if squeeze:
        shared = tuple(t[0] for t in shared)     # one expert without the leading dim
    *out, n = with_shared_expert(*routed, shared)
    assert n == 1
    for r, sh, o in zip(routed, _tensors(1), out):
        assert o.shape[0] == 6 and o.dtype == torch.uint8
        assert torch.equal(o[:5], r) and torch.equal(o[5], sh[0])


@pytest.mark.parametrize("Is", [256, 384, 96])
def test_larger_or_smaller_shared_expert_is_split_into_pieces(Is):
    Ip = 128
    routed = _tensors(3, Ip=Ip)
    w1, s1, w2, s2 = (t[0] for t in _tensors(1, Ip=Is, seed=7))
    *out, n = with_shared_expert(*routed, (w1, s1, w2, s2))
    assert n == -(-Is // Ip)
    o1, q1, o2, q2 = out
    assert o1.shape[0] == 3 + n
    for j in range(n):
        lo, hi = j * Ip, min((j + 1) * Ip, Is)
        k = hi - lo
        # gate/up rows 2i, 2i+1 of intermediate index i stay together
        assert torch.equal(o1[3 + j, :2 * k], w1[2 * lo:2 * hi])
        assert torch.equal(q1[3 + j, :2 * k], s1[2 * lo:2 * hi])
        assert torch.equal(o2[3 + j, :, :k // 2], w2[:, lo // 2:hi // 2])
        assert torch.equal(q2[3 + j, :, :k // 32], s2[:, lo // 32:hi // 32])
        # zero padding beyond the shared expert's intermediate size
        assert (o1[3 + j, 2 * k:] == 0).all() and (o2[3 + j, :, k // 2:] == 0).all()


def test_inconsistent_shared_expert_is_rejected():
    w1, s1, w2, s2 = (t[0] for t in _tensors(1, Ip=128))
    with pytest.raises(ValueError):
        shared_expert_pieces((w1[:100], s1, w2, s2), 128)
