"""Host logic of the streamed-weights stack: one layer's four projections
packed into a single buffer.  Every view starts on a 1 KB boundary (the
kernels' bulk copies and tensor maps want at least 16 bytes), no two views
overlap, the packed size covers them all, and the views round-trip the
bytes of the projections they were filled from."""
import types

import torch

from bit_group_quant_gb300 import fg
from bit_group_quant_gb300.model import HostLayerStack


def _fake_layer(h1, h2, g):
    shapes = {"qkv": (3 * h1, h1), "out": (h1, h1), "fc1": (h2, h1), "fc2": (h1, h2)}
    L = types.SimpleNamespace()
    for nm, (r, c) in shapes.items():
        codes = torch.randint(0, 256, (r, c // 2), dtype=torch.uint8, generator=g)
        meta = torch.randn((r, c // 64, 2), generator=g, dtype=torch.float32)
        setattr(L, nm, fg.Q4(codes, meta, r, c))
    return L


def test_packed_layout_aligned_disjoint_and_round_trips():
    g = torch.Generator().manual_seed(5)
    for h1, h2 in [(64, 256), (192, 768), (7168, 28672 // 16)]:
        L = _fake_layer(h1, h2, g)
        lay, size = HostLayerStack._layout(L)
        spans = []
        for nm, oc, om, rows, cols in lay:
            assert oc % HostLayerStack.ALIGN == 0 and om % HostLayerStack.ALIGN == 0
            spans.append((oc, oc + rows * cols // 2))
            spans.append((om, om + rows * cols // 64 * 8))
        spans.sort()
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 <= b0
        assert spans[-1][1] <= size and size % HostLayerStack.ALIGN == 0
        buf = torch.zeros(size, dtype=torch.uint8)
        views = HostLayerStack._views(buf, lay)
        for nm in HostLayerStack.NAMES:
            src = getattr(L, nm)
            views[nm].codes.copy_(src.codes)
            views[nm].meta.copy_(src.meta)
        for nm in HostLayerStack.NAMES:
            src = getattr(L, nm)
            v = views[nm]
            assert v.codes.is_contiguous() and v.meta.is_contiguous()
            assert torch.equal(v.codes, src.codes) and torch.equal(v.meta, src.meta)
            assert v.nbytes == src.nbytes
        payload = sum(getattr(L, nm).nbytes for nm in HostLayerStack.NAMES)
        assert size - payload < 8 * HostLayerStack.ALIGN
