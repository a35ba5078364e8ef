"""The bench line's `config` (shared by the GPU arm and the oracle's line)
computes the weight and cache footprints from the shapes; those formulas
must equal the bytes of the library's own tensors for the same shapes."""
import types

import bench
import synth
from bit_group_quant_gb300 import fg


def _tensor_footprints(wl, kv):
    h1, h2 = wl.h1, wl.h2
    per_layer = sum(fg.Q4.empty(n, k, "cpu").nbytes
                    for n, k in ((3 * h1, h1), (h1, h1), (h2, h1), (h1, h2)))
    cls = fg.KV16 if kv == "f16" else fg.KV4
    cache = cls.empty(wl.bls, wl.H, wl.d, wl.cap, "cpu", zero=False).nbytes
    return wl.layers * per_layer, wl.layers * cache


def test_footprints_equal_the_allocated_tensors():
    wl = synth.Workload("tiny", 3, 256, 4, 512, 1000, 3, 2, 20, 4, 3)
    for kv in ("g4", "f16"):
        assert bench.footprints(wl, kv) == _tensor_footprints(wl, kv)


def test_config_names_the_workload_and_options():
    args = types.SimpleNamespace(weights="hbm", no_graphs=False, kv="g4", topk=10, order="zigzag")
    cfg = bench.workload_config(synth.OPT30B, args, 1)
    assert cfg["workload"].startswith("opt-30b-shaped: 48 layers, h1 7168, 56 heads, h2 28672")
    assert "bls 144, s 512, n 32 (31 decode steps)" in cfg["workload"]
    assert cfg["decode_attention"] == "top-K sparse, 10% of the rows' V"
    assert cfg["order"] == "zigzag" and cfg["parallelism"] == "single"
    assert cfg["l2"] == "inputs larger than L2 (weights 18.5 GB, KV 33.7 GB)"
    layer = bench.workload_config(synth.OPT125M_LAYER, args, 1)
    assert layer["workload"].startswith("opt125m-layer: one decoder layer")
