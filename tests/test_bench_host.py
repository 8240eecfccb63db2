"""bench.py's host logic that decides whether the committed ncu counters still describe the kernel."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = '''// Kernel 2: the split partial.
__device__ float f(float x) {  // scaled
  /* a block
     comment */
  asm volatile("mov.u64 %0, %%globaltimer; // not a comment" : "=l"(t));
  return x * 2.f;
}
'''


def test_comments_and_blank_lines_do_not_count():
    edited = SRC.replace("// Kernel 2: the split partial.", "// Kernel 2: the per-split partial,\n// reworded.\n\n")
    edited = edited.replace("/* a block\n     comment */", "/* another */")
    assert bench._code_only(edited) == bench._code_only(SRC)


def test_code_and_string_literals_count():
    assert bench._code_only(SRC.replace("x * 2.f", "x * 3.f")) != bench._code_only(SRC)
    # inline PTX lives in string literals: a "//" inside one is code, not a comment
    assert "// not a comment" in bench._code_only(SRC)
    assert bench._code_only(SRC.replace("%%globaltimer;", "%%clock64;")) != bench._code_only(SRC)



def test_roofline_bound_follows_the_arithmetic_intensity():
    # the ridge of the measured peaks (1,913 TFLOP/s over 6,796 GB/s) is ~281 FLOP per K/V byte:
    # bf16 decode windows sit below it (HBM), an fp8 prefill chunk of 128 rows far above (tensor)
    import workloads as wl
    peaks = (6795.8, 1913.2, "measured")
    for name, bound in (("single_row_small", "hbm"), ("verify_small", "hbm"), ("prefill_small", "tensor")):
        case = wl.make_case(name, device="cpu")
        r = bench.roofline(case, 0.1, peaks)
        assert r["bound"] == bound, name
        if bound == "tensor":
            assert r["achieved"] == round(bench.attention_flops(case) / 1e-4 / 1e12, 2)
            assert r["frac"] == round(r["achieved"] / 1913.2, 4)
        else:
            assert r["achieved"] == round(case.kv_bytes() / 1e-4 / 1e9, 2)
            assert r["frac"] == round(r["achieved"] / 6795.8, 4)


def test_profiled_traffic_scales_and_goes_stale(monkeypatch, tmp_path):
    import json
    d = {"kernel_source_hash": "abc", "workloads": {"w": {"dram_bytes_per_launch": 1010, "kv_bytes": 1000}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "decode_partial_traffic.json").write_text(json.dumps(d))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.profiled_traffic("w", 2000) == 2020      # per launch, scaled to the K/V bytes
    assert bench.profiled_traffic("other", 2000) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "changed")
    assert bench.profiled_traffic("w", 2000) is None       # the kernels changed since the capture
