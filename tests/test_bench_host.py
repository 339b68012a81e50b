"""Host logic of bench.py that needs no GPU: the merged weight of a layer is zero-padded to
whole blocks exactly when the block size does not divide a side (a ragged last block)."""
import torch

import bench


class _FakeLib:
    def __init__(self):
        self.calls = []

    def poetx_merge_perm(self, W0, pn, pm, Wp, scale=None, scale_p=None):
        self.calls.append(("plain", tuple(Wp.shape), None if scale_p is None else scale_p.numel()))

    def poetx_merge_perm_padded(self, W0, pn, pm, Wp, scale=None, scale_p=None):
        self.calls.append(("padded", tuple(Wp.shape),
                           None if scale_p is None else scale_p.numel()))


def test_merged_weight_pads_only_ragged_sides():
    P = _FakeLib()
    Wp, sc = bench.merged_weight(P, torch.zeros(2048, 2048), None, None, 256)
    assert tuple(Wp.shape) == (2048, 2048) and sc is None
    Wp, _ = bench.merged_weight(P, torch.zeros(2000, 1000), None, None, 256)
    assert tuple(Wp.shape) == (2048, 1024)
    Wp, sc = bench.merged_weight(P, torch.zeros(776, 528, dtype=torch.int8), None, None, 256,
                                 scale=torch.ones(776))
    assert tuple(Wp.shape) == (1024, 768) and sc.numel() == 1024
    assert [c[0] for c in P.calls] == ["plain", "padded", "padded"]
