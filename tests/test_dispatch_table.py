"""The kernel-choice table compiled into the library is the one the committed
generator makes from the committed sweep measurements (no hand edits), and
every row names a configuration that was measured fastest for its class."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "int4_weight_only_gemm_gb300", "csrc")


def _gen():
    spec = importlib.util.spec_from_file_location("gen_dispatch", os.path.join(CSRC, "gen_dispatch.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_table_is_generated_from_the_sweep():
    gen = _gen()
    with open(os.path.join(CSRC, "dispatch_sweep.json")) as f:
        doc = json.load(f)
    with open(os.path.join(CSRC, "dispatch_table.h")) as f:
        assert f.read() == gen.render(doc, gen.choose(doc["entries"]))


def test_each_row_is_the_measured_minimum():
    gen = _gen()
    with open(os.path.join(CSRC, "dispatch_sweep.json")) as f:
        doc = json.load(f)
    table = gen.choose(doc["entries"])
    assert table
    for (cls, M), (best, sums) in table.items():
        assert sums[best] == min(sums.values())
        if M > 8:
            assert best.startswith("tc")  # the GEMV runs M <= 8 only
