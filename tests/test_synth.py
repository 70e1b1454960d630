"""Host logic of the seeded input recipe (no GPU): counts and shapes of the five workloads."""
import numpy as np

from moe_grouped_gemm_persistent_gb300 import synth


def test_workload_counts():
    d, w = synth.workload_specs("tiny")
    assert d.counts.tolist() == [256, 0, 512, 256] and d.M == 1024
    d, _ = synth.workload_specs("mixtral")
    assert d.counts.tolist() == [4352, 4096, 4096, 4096, 4096, 4352, 4352, 4096]
    assert d.M == 33536
    d, _ = synth.workload_specs("geglu")
    assert d.M == 50688 and int((d.counts == 0).sum()) == 2 and int(d.counts.max()) == 16896
    _, w = synth.workload_specs("wgrad64")
    assert w.T == 65536 and int((w.counts == 0).sum()) == 22 and int(w.counts.max()) == 24576
    d, w = synth.workload_specs("deepseek")
    assert d.M == 162304 and w.T == 162304
    assert int((d.counts == 256).sum()) == 175 and int(d.counts.max()) == 21248
    for name in synth.WORKLOADS:
        for s in synth.workload_specs(name):
            if s is not None:
                assert (s.counts % 256 == 0).all()


def test_small_inputs_shapes_and_determinism():
    spec = synth.small_dglu_spec()
    x1 = synth.make_dglu_inputs(spec)
    x2 = synth.make_dglu_inputs(spec)
    assert x1["a"].shape == (768, 320) and x1["c"].shape == (768, 320)
    assert x1["b"].shape == (3, 160, 320)
    assert (x1["a"] == x2["a"]).all() and (x1["c"] == x2["c"]).all()
    assert x1["padded_offsets"].tolist() == [256, 256, 768]
    assert float(x1["alpha"].min()) >= 0.5 and float(x1["alpha"].max()) <= 1.5
    ws = synth.small_wgrad_spec(accumulate=True)
    y = synth.make_wgrad_inputs(ws)
    assert y["a"].numel() == 192 * 1536 and y["b"].numel() == 1536 * 160
    assert y["out_old"].shape == (4, 192, 160)
    assert np.array_equal(y["offsets"].numpy(), [512, 512, 768, 1536])
