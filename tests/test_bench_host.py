"""Host-side helpers of bench.py, on the CPU: the kernel-source digest that keys the
recorded DRAM traffic, the lookup of that traffic, and the argument defaults the
benchmark contract fixes."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _tree(tmp_path, kernels: str, internal: str = "struct X { int a; };\n"):
    d = tmp_path / "loss_scaled_adamw_gb300" / "csrc"
    d.mkdir(parents=True, exist_ok=True)
    (d / "tl_kernels.cu").write_text(kernels)
    (d / "tl_kernels_split.cu").write_text('#define TL_SPLIT_TU 1\n#include "tl_kernels.cu"\n')
    (d / "tl_internal.cuh").write_text(internal)
    (tmp_path / "profiles").mkdir(exist_ok=True)
    return tmp_path


def test_digest_ignores_comments_and_layout_but_not_code(tmp_path, monkeypatch):
    code = "int f(int x) {\n    return x + 1;\n}\n"
    commented = "// a comment\nint f(int x) {   // trailing\n\n        return x + 1;\n}\n\n"
    changed = "int f(int x) {\n    return x + 2;\n}\n"
    with_string = 'const char* s = "//not a comment";\n'
    digests = {}
    for name, src in (("code", code), ("commented", commented), ("changed", changed),
                      ("string", with_string), ("string2", 'const char* s = "//other";\n')):
        monkeypatch.setattr(bench, "ROOT", str(_tree(tmp_path / name, src)))
        digests[name] = bench.kernel_source_digest()
    assert digests["code"] == digests["commented"]
    assert digests["code"] != digests["changed"]
    assert digests["string"] != digests["string2"]       # "//" inside a string is code


def test_recorded_traffic_is_keyed_to_digest_workload_and_layout(tmp_path, monkeypatch):
    root = _tree(tmp_path, "int k;\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    digest = bench.kernel_source_digest()
    (root / "profiles" / "dram_traffic.txt").write_text(
        "# comment line\nworkload=llama_1b\nlayout=aligned\n"
        f"kernel_source_digest={digest}\nk_adamw_bf16.dram_bytes_per_launch=37019515136\n")
    assert bench.recorded_traffic("k_adamw_bf16", "llama_1b", "aligned") == 37019515136.0
    assert bench.recorded_traffic("k_unknown", "llama_1b", "aligned") is None
    assert bench.recorded_traffic("k_adamw_bf16", "ragged_100k", "aligned") is None
    assert bench.recorded_traffic("k_adamw_bf16", "llama_1b", "packed") is None
    # a kernel edit invalidates the record
    (root / "loss_scaled_adamw_gb300" / "csrc" / "tl_kernels.cu").write_text("int k2;\n")
    assert bench.recorded_traffic("k_adamw_bf16", "llama_1b", "aligned") is None


def test_recorded_traffic_without_a_summary(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(_tree(tmp_path, "int k;\n")))
    assert bench.recorded_traffic("k_adamw_bf16", "llama_1b", "aligned") is None


def test_traffic_keys_name_the_recorded_kernels():
    """Every kernel the bench can report as dominant maps to a key of the summary that
    the profile script writes."""
    recorded = {"k_accum_many_bf16_first_last", "k_adamw_bf16", "k_accumulate_first_bf16",
                "k_accumulate_bf16", "k_unscale_bf16_acc_grad"}
    assert set(bench.TRAFFIC_KEYS.values()) == recorded


def test_default_arguments_follow_the_contract():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1
    assert a.impl != "reference" and a.layout == "aligned"
    r = bench.parse_args(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert r.impl == "reference" and r.steps == 2 and r.warmup == 3


@pytest.mark.parametrize("params,steps,world,secs,want", [(1_235_814_400, 30, 1, 0.27, 137.31271111111112),
                                                          (1000, 4, 2, 0.75, 1.0666666666666667e-05)])
def test_whole_job_rate(params, steps, world, secs, want):
    assert bench.whole_job_rate(params, steps, world, secs) == pytest.approx(want, rel=1e-12)
