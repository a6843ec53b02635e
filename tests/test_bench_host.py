"""Host-side decisions of bench.py that shape a timing (no GPU needed)."""
import bench
from attention_prefix_scan_02_b300 import inputs


def test_l2_flush_decision_and_its_description_agree():
    expect = {"tiny": True, "bf16_4k": True, "stress": False, "long": False}
    for name, flushed in expect.items():
        wl = inputs.WORKLOADS[name]
        assert bench.needs_flush(wl) is flushed, name
        text = bench.describe(wl, wl.dtype)["l2"]
        assert text.startswith("L2 flushed" if flushed else "no flush"), (name, text)


def test_flushed_workloads_fit_in_a_few_l2s_and_unflushed_ones_do_not():
    l2 = 126 << 20
    for name, wl in inputs.WORKLOADS.items():
        if wl.kind == "stream" or name == "linattn":
            continue
        in_b = 2 if wl.dtype == "bf16" else 4
        kv = wl.heads * wl.N * wl.d * 2 * in_b
        if bench.needs_flush(wl):
            assert kv < 256 << 20
        else:
            assert kv > 2 * l2
