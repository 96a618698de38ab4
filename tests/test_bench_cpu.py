"""Host-side pieces of bench.py: the algorithmic work behind the roofline figures, and
the clock record kept to the timed window.  No GPU."""
import datetime
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
import synth  # noqa: E402


def test_algorithmic_work_closed_forms():
    """The llama8b step: fixed stride 16, 2048 references, 30720 compressed tokens."""
    w = synth.workload("llama8b")
    ref = np.arange(0, w.T, 16)
    work = bench.algorithmic_work(w, w.T, w.n_sel, ref)
    n_non = w.T - len(ref)
    # a restore: one (d_c x 2d_k) product per selected token
    assert work["rkv_reconstruct_kernel"]["flops"] == 2.0 * w.n_sel * w.d_c * w.d_kv
    # GEMM-1/2 over kv and mean rows, gate and value columns
    assert work["rkv_gemm12_swiglu_kernel"]["flops"] == 2.0 * (2 * n_non) * (2 * w.d_ff) * w.d_kv
    # retrieval: token 16k + j (j = 1..15) sees the k + 1 references at 0, 16, ..., 16k,
    # so the average pool is 15 * sum_{k<2048} (k + 1) / 30720 = 2049 / 2
    assert work["rkv_retrieve_kernel"]["flops"] == 2.0 * n_non * (2049 / 2) * w.d_kv
    # bytes of a restore: code, extremes and slots in, K and V out, W_d and the pool once
    per_tok = w.d_c * w.bits // 8 + 4 * (w.d_c // 32) + 4 * w.topk + w.d_kv * 2
    assert work["rkv_reconstruct_kernel"]["bytes"] == (
        w.n_sel * per_tok + w.d_kv * w.d_c * 2 + len(ref) * w.d_kv)


class _FakeSmi:
    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def _line(t, sm, reasons=("Not Active",) * 4):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([ts, "0", str(sm), "2070", "900.00", "0x0"] + list(reasons))


def test_clock_record_keeps_only_the_timed_window():
    t0 = 1_800_000_000.0
    lines = [
        _line(t0 - 0.5, 900, ("Not Active", "Not Active", "Not Active", "Active")),  # before
        _line(t0 + 0.05, 2070),
        _line(t0 + 0.10, 2055, ("Not Active", "Not Active", "Not Active", "Active")),
        _line(t0 + 0.15, 2070),
        _line(t0 + 0.9, 1200, ("Active", "Not Active", "Not Active", "Not Active")),  # after
    ]
    c = bench.ClockSampler(0)
    c.proc = _FakeSmi("\n".join(lines) + "\n")
    c.t0, c.t1 = t0, t0 + 0.2
    rec = c.stop()
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 2070.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"]          # the hw_slowdown sample lies outside


def test_step_config_names_the_bench_workloads():
    """Token counts per step: the qwen7b stack (28 layers x 131072 written, 64 steps x 28
    layers x 614 blocks of 64 restored) and the llama8b layer."""
    w = synth.workload("qwen7b")
    assert bench._stack_description("qwen7b").startswith("qwen7b: Qwen2.5-7B-shaped stack of 28")
    sel = synth.gen_block_selection(w.T, w.sel_block, w.sel_frac, 1)
    assert sel.numel() == 614 * 64

    class _Run(bench.StackRun):
        def __init__(self, name, n_sel):
            self.name, self.w = name, synth.workload(name)
            self.L, self.n_sel = self.w.layers, n_sel
            self.tokens_written = self.L * self.w.T
            self.tokens_read = self.w.steps * self.L * n_sel

    cfg = bench.step_config(_Run("qwen7b", 614 * 64), 1)
    assert cfg["tokens_per_step"] == 28 * 131072 + 64 * 28 * 39296
    cfg = bench.step_config(_Run("llama8b", 9830), 1)
    assert cfg["tokens_per_step"] == 32768 + 64 * 9830
    assert cfg["workload"].startswith("llama8b: ")


def test_roofline_names_the_binding_roof_against_the_burst_peak():
    """A restore at the qwen7b shape (236 flop/B) is below the burst ridge point, so HBM
    binds; at the llama8b shape (413 flop/B) the tensor peak binds, reported against the
    burst figure with the sustained one beside it."""
    peaks = {"hbm_gbs": 6785.5, "bf16_tflops": 1871.4, "bf16_tflops_sustained": 1690.7}
    for name, bound in (("qwen7b", "hbm"), ("llama8b", "tensor")):
        w = synth.workload(name)
        ref = np.arange(0, w.T, 16)
        n_sel = 39296 if name == "qwen7b" else w.n_sel
        work = bench.algorithmic_work(w, w.T, n_sel, ref)
        k = "rkv_reconstruct_kernel"
        rows = bench.kernel_rows({k: (1, 0.05)}, {k: work[k]}, 1, peaks)
        roof = bench.roofline_of(rows, {k: work[k]}, peaks, "measured", name)
        assert roof["bound"] == bound and roof["kernel"] == k
        if bound == "tensor":
            assert roof["peak"] == 1871.4 and roof["peak_sustained"] == 1690.7
            assert abs(roof["frac"] - work[k]["flops"] / 50e-6 / 1871.4e12) < 1e-4
        else:
            assert roof["peak"] == 6785.5
            assert abs(roof["frac"] - work[k]["bytes"] / 50e-6 / 6785.5e9) < 1e-4


def test_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("// header\nint f(int x) {\n  return x + 1;  // add one\n}\n")
    b.write_text("// a different header\n\nint f(int x) {\n  return x + 1;\n}\n")
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_sha1(str(a)) == bench.code_sha1(str(b))
    assert bench.code_sha1(str(a)) != bench.code_sha1(str(c))


def test_storage_report_of_the_llama8b_layer():
    """codes 256 + extremes 64 + slots 16 B per token, FP8 pool 2048 B per reference (one
    token in 16) with 8 B of norm and position per slot; the library's bf16 copy of the
    pool (4096 B per reference) shown beside it."""
    import torch
    w = synth.workload("llama8b")
    B, T, R = 1, w.T, w.T // 16

    class _Codec:
        pool_fp8 = torch.empty((B, R, w.d_kv), dtype=torch.uint8)
        pool_norm2 = torch.empty((B, R), dtype=torch.float32)
        pool_pos = torch.empty((B, R), dtype=torch.int32)
        codes = torch.empty((B, T, 256), dtype=torch.uint8)
        meta = torch.empty((B, T, 16, 2), dtype=torch.float16)
        ref_idx = torch.empty((B, T, 4), dtype=torch.int32)

        def pool_cache_bytes(self):
            return B * R * w.d_kv * 2

    rep = bench.storage_report(_Codec(), w)
    per_tok = 256 + 64 + 16 + (2048 + 8) / 16
    assert rep["bytes_per_token"] == round(per_tok, 1)
    # the page's INT4 formula with the slots added (11.33 %), plus the 8-byte norm and
    # position of each pool slot
    assert rep["fraction_of_fp16_kv"] == round(per_tok / 4096, 4) == 0.1134
    assert rep["compute_cache_bytes_per_token"] == 256.0
    assert rep["fraction_with_compute_cache"] == round((per_tok + 256) / 4096, 4)
