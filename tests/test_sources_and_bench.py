"""CPU checks of the library sources and of the benchmark's output contract.

* No source of the library (kernels, host code, public header) names a TMA multicast form:
  every CTA loads its own operand tiles, so the library runs unchanged under a multi-process
  launch on several GPUs.
* Both arms of the benchmark (the GPU library and the timed CPU oracle) print the same
  `config` object, so their lines describe one workload.
"""
import glob
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _library_sources():
    pats = [os.path.join(ROOT, "moe_grouped_gemm_02_gb300", "csrc", "*"), os.path.join(ROOT, "include", "*.h"),
            os.path.join(ROOT, "moe_grouped_gemm_02_gb300", "*.py")]
    files = [p for pat in pats for p in glob.glob(pat) if os.path.isfile(p)]
    assert any(p.endswith("dg_gemm_kernel.cuh") for p in files)
    return files


def test_no_multicast_in_library_sources():
    for p in _library_sources():
        with open(p, encoding="utf-8", errors="replace") as f:
            text = f.read()
        assert "multicast" not in text.lower(), f"{os.path.relpath(p, ROOT)} names a multicast form"


def test_both_bench_arms_print_one_config():
    import bench
    import synth
    w = synth.make_dense(4, 256, 256, seed=0)
    w["name"] = "dense_4x256x256"
    w["valid_rows"] = bench._valid_rows(w)
    w["flops"] = 2.0 * w["valid_rows"] * w["N"] * w["K"]
    w["bytes"] = bench._algorithmic_bytes(w)
    for world in (1, 2):
        c = bench.suite_config([w], world)
        assert c == bench.suite_config([w], world)
        assert c["workload"] == bench.WORKLOAD_NAME
        assert c["flops_per_step"] == w["flops"] and c["bytes_per_step"] == w["bytes"]
        assert ("replicas" in c["parallelism"]) == (world > 1)
    # the reference arm builds its line from the same function
    import inspect
    src = inspect.getsource(bench.run_reference)
    assert '"config": suite_config(ws, world)' in src
    src = inspect.getsource(bench.run_gpu)
    assert '"config": suite_config(ws, world)' in src
