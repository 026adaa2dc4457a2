"""Host-side helpers of the benchmark (no GPU): the packed host-to-device
transfer of a step's inputs."""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_pack_inputs_views_hold_the_tensors_at_aligned_offsets(monkeypatch):
    import bench
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self.clone())  # no CUDA here
    g = torch.Generator().manual_seed(7)
    ts = [torch.randn(3, 5, generator=g).to(torch.float16), torch.arange(7, dtype=torch.int32),
          torch.randn(2, 2, 2, generator=g).to(torch.bfloat16), torch.arange(12, dtype=torch.int64).view(3, 4)]
    dbuf, hbuf, views = bench.pack_inputs(ts, "cpu")
    assert all(v.dtype == t.dtype and v.shape == t.shape and torch.equal(v, t) for v, t in zip(views, ts))
    base = dbuf.data_ptr()
    offs = [v.data_ptr() - base for v in views]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    # no two views overlap, and the host copy is byte-identical
    for (o, v), o2 in zip(zip(offs, views), offs[1:] + [dbuf.numel()]):
        assert o + v.numel() * v.element_size() <= o2
    assert torch.equal(dbuf, hbuf)
    # writing the host buffer and copying it over refreshes every view
    hbuf.zero_()
    dbuf.copy_(hbuf)
    assert all(int(v.abs().sum()) == 0 for v in views)
