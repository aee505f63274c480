"""Host side of the separate shared expert: its tensors are appended to the
routed experts as expert E (shape checks included), on CPU."""
import pytest
import torch

from block_scaled_moe_sort_gb300 import with_shared_expert


def _tensors(E, Ip=128, H=256):
    g = torch.Generator().manual_seed(E)
    return (torch.randint(0, 256, (E, 2 * Ip, H // 2), generator=g, dtype=torch.uint8),
            torch.randint(118, 124, (E, 2 * Ip, H // 32), generator=g, dtype=torch.uint8),
            torch.randint(0, 256, (E, H, Ip // 2), generator=g, dtype=torch.uint8),
            torch.randint(118, 124, (E, H, Ip // 32), generator=g, dtype=torch.uint8))


@pytest.mark.parametrize("squeeze", [False, True])
def test_shared_expert_appended_as_last_expert(squeeze):
    routed = _tensors(5)
    shared = _tensors(1)
    if squeeze:
        shared = tuple(t[0] for t in shared)     # one expert without the leading dim
    out = with_shared_expert(*routed, shared)
    for r, sh, o in zip(routed, _tensors(1), out):
        assert o.shape[0] == 6 and o.dtype == torch.uint8
        assert torch.equal(o[:5], r) and torch.equal(o[5], sh[0])


def test_shared_expert_shape_mismatch_is_rejected():
    routed = _tensors(4)
    bad = _tensors(1, Ip=256)
    with pytest.raises(ValueError):
        with_shared_expert(*routed, bad)
