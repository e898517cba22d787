"""bench.py's host-side helpers on the CPU: the packed layout that lets one
step's inputs cross to the device in one copy."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_packed_layout_round_trip_and_alignment():
    g = torch.Generator().manual_seed(0)
    tensors = {
        "q": torch.randn((3, 2, 5), generator=g).bfloat16(),
        "beta": torch.rand((3, 2), generator=g),
        "cu_seqlens": torch.tensor([0, 1, 3], dtype=torch.int32),
        "initial_state": torch.randn((1, 2, 4, 4), generator=g),
    }
    layout, nbytes, views = bench._packed_layout(tensors)
    offs = [layout[n][0] for n in tensors]
    assert all(o % 256 == 0 for o in offs)                  # every piece 256-byte aligned
    assert offs == sorted(offs) and offs[0] == 0
    sizes = [t.numel() * t.element_size() for t in tensors.values()]
    assert nbytes == sum((sz + 255) // 256 * 256 for sz in sizes)
    for o, sz, o_next in zip(offs, sizes, offs[1:] + [nbytes]):
        assert o + sz <= o_next                             # pieces do not overlap
    buf = torch.zeros(nbytes, dtype=torch.uint8)
    for n, v in views(buf).items():
        assert v.is_contiguous() and v.dtype == tensors[n].dtype and v.shape == tensors[n].shape
        v.copy_(tensors[n])
    # a byte copy of the packed buffer carries every tensor exactly
    back = views(buf.clone())
    for n, t in tensors.items():
        assert torch.equal(back[n], t), n
    # the views alias the buffer they were made from
    v = views(buf)["beta"]
    v.fill_(7.0)
    assert torch.equal(views(buf)["beta"], torch.full_like(tensors["beta"], 7.0))
