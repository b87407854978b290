"""Host-side checks of how bench.py ties a committed ncu summary to the
kernel source it was captured on (no GPU)."""
import os

import bench


def test_code_only_drops_comments_and_white_space():
    a = "int f(int x) {  // the sum\n  return x + 1; /* one */\n}\n"
    b = "int f(int x) {\n\n    return x + 1;\n}  // edited comment\n"
    assert bench.code_only(a) == bench.code_only(b) == "int f(int x) { return x + 1; }"


def test_code_change_is_seen():
    assert bench.code_only("return x + 1;") != bench.code_only("return x + 2;")


def test_hashed_summaries_are_well_formed():
    """A summary that names its kernel sources records their hash and the DRAM
    bytes per launch; whether it is current is reported by bench.py itself
    (`traffic` is null when the code has changed since the capture)."""
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles")
    csrc = os.path.join(os.path.dirname(root), "paged_kv_decode_07_gb300", "csrc")
    seen = 0
    for name in sorted(os.listdir(root)):
        vals = {}
        for ln in open(os.path.join(root, name)).read().splitlines():
            if ln.startswith("- ") and ":" in ln:
                k, v = ln[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
        if "kernel_sources" not in vals:
            continue
        seen += 1
        for f in vals["kernel_sources"].split():
            assert os.path.exists(os.path.join(csrc, f)), (name, f)
        h = vals.get("kernel_source_hash", "")
        assert len(h) == 16 and all(ch in "0123456789abcdef" for ch in h), name
        assert float(vals["dram_bytes_per_launch"]) > 0, name
    assert seen >= 1
