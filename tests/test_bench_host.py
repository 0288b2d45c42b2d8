"""Host-side pieces of bench.py: the DRAM-traffic lookup behind `roofline.traffic`."""
import os

import bench


def _rows():
    p = os.path.join(bench.ROOT, "profiles", "dram_traffic.md")
    out = {}
    for line in open(p):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[2].isdigit():
            out[(cells[0], cells[1])] = (float(cells[2]), cells[3])
    return out


def test_traffic_only_for_the_sources_it_was_taken_on():
    rows = _rows()
    assert ("bwd_dkdv", "long64k_causal") in rows
    src = bench.kernel_source_hash()
    for (kernel, workload), (value, taken_on) in rows.items():
        got = bench.recorded_traffic(kernel, workload)
        assert got == (value if taken_on == src else None)


def test_unknown_kernel_has_no_traffic():
    # the deterministic dK/dV kernel has a key of its own: the atomic kernel's
    # row (which counts the fp32 dQ accumulator) must not stand in for it
    if ("bwd_dkdv_deterministic", "long64k_causal") not in _rows():
        assert bench.recorded_traffic("bwd_dkdv_deterministic", "long64k_causal") is None
    assert bench.recorded_traffic("no_such_kernel", "long64k_causal") is None


def test_kernel_source_hash_ignores_comments_and_whitespace():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and all(c in "0123456789abcdef" for c in h)
    assert bench.code_text("int a; // note\n/* block */  int b;") == bench.code_text("int a;\nint b;")
