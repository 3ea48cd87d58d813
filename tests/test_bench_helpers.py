"""Helpers of bench.py: the kernel-source hash that ties recorded DRAM traffic to the
code it was measured on (CPU), and the plain FP8 GEMM reference rate (GPU)."""
import pytest

import bench


def test_source_hash_ignores_comments_and_layout():
    code = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    same = "/* header */\nint f(int x) { return x + 1; }\n// trailing note\n"
    other = "int f(int x) { return x + 2; }\n"
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)


def test_traffic_lookup_needs_the_recorded_hash(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# kernel hash bytes\nk_current 0123456789abcdef 1234\nk_stale 0000000000000000 99\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0123456789abcdef")
    assert bench.profiled_traffic("k_current") == 1234
    assert bench.profiled_traffic("k_stale") is None
    assert bench.profiled_traffic("k_absent") is None


@pytest.mark.gpu
def test_plain_fp8_reference_reports_its_shape(cuda_device):
    r = bench.plain_fp8_gemm_check(cuda_device, 256, 512, 1024, secs=0.05)
    assert "256x512x1024" in r["kernel"]
    assert 0.0 < r["burst_tflops"] < 20000.0
    assert 0.0 < r["sustained_tflops"] < 20000.0


def test_rescale_touches_only_tensor_rows():
    rows = {"g": {"bound": "tensor", "TFLOPs": 1000.0, "frac": 0.3, "stream_k": {"TFLOPs": 1500.0, "frac": 0.4}},
            "q": {"bound": "hbm", "GBps": 5000.0, "frac": 0.8},
            "floor": {"events_only": 1.2}}
    bench.rescale_tensor_fracs(rows, 4000.0)
    assert rows["g"]["frac"] == 0.25 and rows["g"]["stream_k"]["frac"] == 0.375
    assert rows["q"]["frac"] == 0.8
    assert rows["floor"] == {"events_only": 1.2}


def test_oracle_threads_split_rows_and_limit_blas():
    """The CPU baseline divides the oracle's quantizer over row blocks (boundaries on
    whole 128-row blocks, results concatenated in order) and limits BLAS to the thread
    count it reports."""
    import numpy as np
    from oracle import fp8_oracle as O
    x = np.random.default_rng(0).standard_normal((640, 256)).astype(np.float32)
    with bench.OracleThreads(3) as th:
        q, s = th.rows(O.quant_act_1x128, x)
        w = th.rows(O.quant_w_128x128, x)
        assert th.blas_threads in (None, 3)
    rq, rs = O.quant_act_1x128(x)
    wq, ws = O.quant_w_128x128(x)
    assert np.array_equal(q, rq) and np.array_equal(s, rs)
    assert np.array_equal(w[0], wq) and np.array_equal(w[1], ws)


def test_oracle_threads_without_threadpoolctl(monkeypatch):
    """Where threadpoolctl is missing (as on some hosts), the BLAS thread count is set and
    read back through OpenBLAS's own exported functions, and restored afterwards."""
    import builtins
    real_import = builtins.__import__

    def no_threadpoolctl(name, *args, **kwargs):
        if name == "threadpoolctl":
            raise ImportError("hidden for this test")
        return real_import(name, *args, **kwargs)

    import numpy  # noqa: F401  (the BLAS library must be loaded before it can be found)
    before = bench._openblas_threads(None)
    monkeypatch.setattr(builtins, "__import__", no_threadpoolctl)
    with bench.OracleThreads(2) as th:
        assert th.blas_threads in (None, 2)
    monkeypatch.setattr(builtins, "__import__", real_import)
    assert bench._openblas_threads(None) == before
