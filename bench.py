"""Benchmark of the ResidualKV cache codec on GB300.

Workloads (`--workload`; the default run measures all of them and prints one line whose
headline is the first):

* qwen7b     the 28-layer Qwen2.5-7B-shaped stack (2d_k = 1024, d_c = 256, d_ff = 768),
             T = 131072 per layer, stride 16, INT4.  One step = the prefill write of all
             28 layers, then 64 decode steps, each restoring in every layer 30 % of the
             tokens as 614 random contiguous 64-token blocks (39296 tokens).
* llama8b    one Llama-3.1-8B-shaped layer (2d_k = 2048, d_c = 512, d_ff = 1536),
             T = 32768: the prefill write, then 64 decode steps of 9830 random tokens.
* batched    the Llama layer shape, 16 sequences prefilled to 16384 tokens.  One step =
             one decode step: one new token per sequence written (a single-token
             compress, or a pool append at a reference position), then 30 % of every
             sequence's history restored in one call; per-step latency p50 / p99.
* long_int2  the Llama layer shape at T = 262144 with INT2 codes: prefill write, then 16
             decode steps of 30 % random tokens.
* long_bf16z the same at T = 65536 with quantisation off (bf16 z).

Inputs are resident in HBM before the timed region; L2 is flushed (a 512 MiB write)
before every timed step.  value = (tokens written + tokens restored) per second over the
timed steps, summed over ranks (weak scaling: every rank runs its own independent
sequences).  e2e = the same through the public API with the step's inputs copied from
pinned host memory inside the timed region and the last restore's K and V read back to
the host (details in each e2e record).

`--impl reference` times the CPU oracle (test infrastructure) on bounded samples of the
headline workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOAD_ORDER = ("qwen7b", "llama8b", "batched", "long_int2", "long_bf16z")
HEADLINE = "qwen7b"
METRIC = "KV tokens compressed/s + selected tokens reconstructed/s"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# reference schedule (ResidualKV notes section 2.6): alpha = 0, n_sink = 0 is the fixed
# stride of the workload; --alpha / --sink time the dynamic stride instead
SCHEDULE = {"alpha": 0.0, "sink": 0}
# 1: the encoder takes the mean's pre-activations from per-reference products kept beside
# the pool (the library's mean_precompute mode) instead of mapping the mean row
ENCODER = {"mean_precompute": 0}
BATCHED_SLACK = 1024          # decode positions a batched run may append after its prefill


def schedule_note(w) -> str:
    if SCHEDULE["alpha"] == 0.0 and SCHEDULE["sink"] == 0:
        return f"stride {w.stride}"
    return (f"dynamic stride s_0={w.stride}, alpha={SCHEDULE['alpha']}, "
            f"n_sink={SCHEDULE['sink']}")


def codec_config(rkv, w, T, batch=1):
    return rkv.Config(n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, d_c=w.d_c, d_ff=w.d_ff,
                      topk=w.topk, group=w.group, bits=w.bits, ref_stride=w.stride,
                      kv_dtype=w.kv_dtype, out_dtype=w.out_dtype, rope_base=w.rope_base,
                      batch=batch, max_tokens=T, ref_alpha=SCHEDULE["alpha"],
                      ref_sink=SCHEDULE["sink"], mean_precompute=ENCODER["mean_precompute"])


def split_positions(ref_pos, T):
    """Reference positions (from the schedule) and all the other positions below T."""
    pos = np.arange(T, dtype=np.int32)
    isref = np.zeros(T, dtype=bool)
    isref[ref_pos] = True
    return pos[isref], pos[~isref]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over the process group (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ work accounting
def per_token_bytes(w) -> dict:
    code_b = w.d_c * w.bits // 8 if w.bits != 16 else 2 * w.d_c
    meta_b = 0 if w.bits == 16 else 4 * (w.d_c // 32)
    return {"code": code_b, "meta": meta_b, "idx": 4 * w.topk,
            "out": w.d_kv * (4 if w.out_dtype == "fp32" else 2)}


def algorithmic_work(w, n_comp: int, n_sel: int, ref_pos, T: int | None = None) -> dict:
    """Flops and bytes the method itself needs: for the write kernels, summed over one
    prefill of T tokens of one sequence (n_comp = T); for the restore, one launch of
    n_sel selected tokens against a pool of len(ref_pos) references."""
    T = w.T if T is None else T
    dkv, dff, dc = w.d_kv, w.d_ff, w.d_c
    ref_pos = np.asarray(ref_pos, dtype=np.int64)
    n_ref = len(ref_pos)
    n_non = n_comp - n_ref
    b = per_token_bytes(w)
    # references visible to each non-reference token (those at earlier positions)
    before = np.searchsorted(ref_pos, np.arange(T), side="left")
    isref = np.zeros(T, dtype=bool)
    isref[ref_pos] = True
    avg_pool = float(before[~isref].sum()) / max(n_non, 1)
    return {
        "rkv_gemm12_swiglu_kernel": {"flops": 2.0 * (2 * n_non) * (2 * dff) * dkv,
                                     "bytes": 2 * n_non * dkv * 2 + 2 * dff * dkv * 2
                                     + 2 * n_non * dff * 2},
        "rkv_gemm3_quant_kernel": {"flops": 2.0 * n_non * dc * (2 * dff),
                                   "bytes": 2 * n_non * dff * 2 + n_non * (b["code"] + b["meta"])},
        "rkv_retrieve_kernel": {"flops": 2.0 * n_non * avg_pool * dkv,
                                "bytes": n_non * dkv * 2 + n_ref * dkv * 2 + n_non * b["idx"]},
        # per selected token: its code, extremes and slots in, K and V (2 d_k values) out;
        # once per launch: W_d and the FP8 reference pool
        "rkv_reconstruct_kernel": {"flops": 2.0 * n_sel * dc * dkv,
                                   "bytes": n_sel * (b["code"] + b["meta"] + b["idx"] + b["out"])
                                   + dkv * dc * 2 + n_ref * dkv},
    }


# ------------------------------------------------------------------ measured DRAM traffic
# dram__bytes_read.sum + dram__bytes_write.sum of one launch, from the ncu captures
# summarised under profiles/ (kernel-case runs of the named workload).  Reported only
# while the kernel's code is unchanged since the capture (code_sha1 below).
MEASURED_TRAFFIC = {
    ("llama8b", "rkv_reconstruct_kernel"): {"file": "k_reconstruct.cu",
                                            "code_sha1": "5f712fbabd15b4ae5b185c817fc77fbd5cd0b90b",
                                            "bytes": 10437888 + 68096},
    ("qwen7b", "rkv_reconstruct_kernel"): {"file": "k_reconstruct.cu",
                                           "code_sha1": "5f712fbabd15b4ae5b185c817fc77fbd5cd0b90b",
                                           "bytes": 15861760 + 25484032},
    # one launch over the 28 layers: a capture of the same kernel over 4 layers (157184
    # tokens, dram read 62619904 + write 266115584 bytes), scaled by 28 / 4 (every term of
    # its traffic, pools, codes and outputs, is per problem)
    ("qwen7b", "rkv_reconstruct_multi_kernel"): {"file": "k_reconstruct.cu",
                                                 "code_sha1": "5f712fbabd15b4ae5b185c817fc77fbd5cd0b90b",
                                                 "bytes": (62619904 + 266115584) * 7},
    ("llama8b", "rkv_retrieve_kernel"): {"file": "k_retrieve.cu",
                                         "code_sha1": "aa7c494b08aad67b44f721081daffd90bc65a63e",
                                         "bytes": 134541056 + 3821568},
}


def code_sha1(path: str) -> str:
    """sha1 of a source file's code: `//` comments, trailing blanks and empty lines
    removed, so that an edit to comments alone keeps a capture's counters valid."""
    import hashlib
    lines = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            code = line.split("//", 1)[0].rstrip()
            if code:
                lines.append(code)
    return hashlib.sha1("\n".join(lines).encode()).hexdigest()


def measured_traffic(workload: str, kernel: str):
    rec = MEASURED_TRAFFIC.get((workload, kernel))
    if rec is None:
        return None
    path = os.path.join(ROOT, "residual_kv_cache_gb300", "csrc", rec["file"])
    try:
        if code_sha1(path) != rec["code_sha1"]:
            return None
    except OSError:
        return None
    return rec["bytes"]


def kernel_rows(ktimes: dict, work_per_step: dict, steps: int, peaks: dict) -> dict:
    """Per kernel: launches, average launch time, share of all launch time, and the
    rates its algorithmic work per step implies over its event time per step."""
    total = sum(ms for _, ms in ktimes.values()) or 1.0
    rows = {}
    for k, (n, ms) in ktimes.items():
        r = {"launches": n, "avg_us": ms / max(n, 1) * 1e3, "share": ms / total}
        if k in work_per_step and ms > 0:
            t = ms / steps / 1e3
            wk = work_per_step[k]
            r["tflops"] = wk["flops"] / t / 1e12
            r["gbs"] = wk["bytes"] / t / 1e9
            r["tc_frac"] = r["tflops"] / peaks["bf16_tflops"]
            r["tc_frac_sustained"] = r["tflops"] / peaks["bf16_tflops_sustained"]
            r["hbm_frac"] = r["gbs"] / peaks["hbm_gbs"]
        rows[k] = {kk: (round(v, 4) if isinstance(v, float) else v) for kk, v in r.items()}
    return rows


def roofline_of(rows: dict, work_per_step: dict, peaks: dict, kind: str, workload: str):
    """The dominant kernel (largest share of launch time) against its binding roof: the
    tensor peak if its flops per byte exceed the burst ridge point, else HBM.  Per-launch
    event times, so the burst bf16 peak; the sustained one is shown beside it."""
    cands = [k for k in rows if k in work_per_step and "tflops" in rows[k]]
    if not cands:
        return None
    dom = max(cands, key=lambda k: rows[k]["share"])
    r, wk = rows[dom], work_per_step[dom]
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    base = {"kernel": dom, "traffic": measured_traffic(workload, dom),
            "flops_per_byte": round(wk["flops"] / wk["bytes"], 1), "ridge": round(ridge, 1),
            "tc_frac": r["tc_frac"], "tc_frac_sustained": r["tc_frac_sustained"],
            "hbm_frac": r["hbm_frac"]}
    if wk["flops"] / wk["bytes"] > ridge:
        return {"bound": "tensor", "achieved": round(r["tflops"], 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": r["tc_frac"],
                "peak_sustained": peaks["bf16_tflops_sustained"],
                "frac_sustained": r["tc_frac_sustained"],
                "peak_kind": f"{kind} bf16 burst (sustained beside it)", **base}
    return {"bound": "hbm", "achieved": round(r["gbs"], 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": r["hbm_frac"], "peak_kind": f"{kind} copy", **base}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 50 ms, started early (its start-up takes a while); only
    the samples whose timestamps fall inside [mark_begin, mark_end] are reported."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        import datetime
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if self.t0 is not None and not (self.t0 <= ts <= (self.t1 or ts)):
                    continue
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CUDA arm: workloads
class Ctx:
    """What every workload runner needs from the process: device, stream, barrier, the
    L2 flush buffer and the command-line arguments."""

    def __init__(self, args, dev, world, rank):
        import torch
        self.args, self.dev, self.world, self.rank = args, dev, world, rank
        self.stream = torch.cuda.current_stream(dev)
        self.flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def barrier(self):
        import torch
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(self.dev)

    def timed(self, step, steps, warmup, launches):
        """W untimed steps, then K steps each bracketed by events on the launching stream
        (L2 flushed and the device idle before each).  Returns the step times in ms and
        the number of library kernels launched inside the K timed intervals (`launches`
        reads the libraries' launch counters)."""
        import torch
        for _ in range(warmup):
            step()
        self.barrier()
        times, n_launch = [], 0
        for _ in range(steps):
            self.flush.fill_(1.0)
            self.barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            l0 = launches()
            e0.record(self.stream)
            step()
            e1.record(self.stream)
            n_launch += launches() - l0
            self.barrier()
            times.append(e0.elapsed_time(e1))
        return times, n_launch

    def kernel_times(self, codecs, step, steps):
        """The same steps again with an event pair around every launch (launches
        serialised by the events): per kernel (launches, total ms) summed over codecs."""
        for c in codecs:
            c.set_timing(True)
            c.get_timing(reset=True)
        for _ in range(steps):
            self.flush.fill_(1.0)
            self.barrier()
            step()
            self.barrier()
        out = {}
        for c in codecs:
            for k, (n, ms) in c.get_timing(reset=True).items():
                n0, ms0 = out.get(k, (0, 0.0))
                out[k] = (n0 + n, ms0 + ms)
            c.set_timing(False)
        return out


def _status(codecs) -> int:
    s = 0
    for c in codecs:
        s |= c.get_status()
    return s


class StackRun:
    """Prefill + decode-step workloads over L independent layers of one sequence each
    (qwen7b: 28 layers; llama8b, long_int2, long_bf16z: one)."""

    def __init__(self, name, ctx, seed):
        import torch
        import residual_kv_cache_gb300 as rkv
        import synth
        w = synth.workload(name)
        self.name, self.w, self.ctx = name, w, ctx
        dev = ctx.dev
        self.L = w.layers
        cfg = codec_config(rkv, w, w.T)
        self.ref, self.non = split_positions(rkv.reference_positions(cfg), w.T)
        self.ref_pos = rkv.reference_positions(cfg)
        self.zref, self.znon = np.zeros_like(self.ref), np.zeros_like(self.non)
        # per layer: its own kv rows and codec weights (seeds per layer); full-size stacks
        # draw on the device (same distribution, see synth.gen_kv)
        draw_dev = "cpu" if w.T * w.layers <= 65536 else str(dev)
        self.kv, self.codecs = [], []
        for l in range(self.L):
            s = seed + 97 * l
            self.kv.append(synth.gen_kv(w, s, device=draw_dev).to(dev))
            W = {k: v.to(dev) for k, v in synth.gen_weights(w, s + 1).items()}
            self.codecs.append(rkv.Codec(cfg, W, device=dev))
        # per decode step and layer: the selected positions
        self.sels = []
        for st in range(w.steps):
            row = []
            for l in range(self.L):
                sd = seed + 10 + st + 100003 * l
                if w.sel_block > 1:
                    row.append(synth.gen_block_selection(w.T, w.sel_block, w.sel_frac, sd).to(dev))
                else:
                    row.append(synth.gen_selection(w.T, w.n_sel, sd).to(dev))
            self.sels.append(row)
        self.n_sel = int(self.sels[0][0].numel())
        self.seq0 = torch.zeros(self.n_sel, dtype=torch.int32, device=dev)
        odt = torch.float32 if w.out_dtype == "fp32" else torch.bfloat16
        self.k_out = torch.empty((self.n_sel, w.n_kv_heads, w.head_dim), dtype=odt, device=dev)
        self.v_out = torch.empty_like(self.k_out)
        # a decode step restores every layer's selection in one launch, each layer into its
        # own K and V (rkv_reconstruct_multi); one layer uses the single restore
        self.k_outs = [self.k_out] + [torch.empty_like(self.k_out) for _ in range(self.L - 1)]
        self.v_outs = [self.v_out] + [torch.empty_like(self.k_out) for _ in range(self.L - 1)]
        self.tokens_written = self.L * w.T
        self.tokens_read = w.steps * self.L * self.n_sel
        self.read_kernel = "rkv_reconstruct_multi_kernel" if self.L > 1 else "rkv_reconstruct_kernel"

    def write(self, kvs):
        for c, kv in zip(self.codecs, kvs):
            c.reset()
            c.pool_append(kv, self.zref, self.ref, src_rows=self.ref)
            c.compress(kv, self.znon, self.non, src_rows=self.non)

    def read(self, sels, k_outs, v_outs):
        import residual_kv_cache_gb300 as rkv
        for row in sels:
            if self.L > 1:
                rkv.reconstruct_multi(self.codecs, [self.seq0] * self.L, list(row), k_outs, v_outs)
            else:
                self.codecs[0].reconstruct(self.seq0, row[0], k_outs[0], v_outs[0])

    def step(self):
        self.write(self.kv)
        self.read(self.sels, self.k_outs, self.v_outs)

    def work_per_step(self) -> dict:
        w = self.w
        one = algorithmic_work(w, w.T, self.n_sel, self.ref_pos)
        out = {}
        for k, v in one.items():
            mult = self.L * (w.steps if k == "rkv_reconstruct_kernel" else 1)
            out[self.read_kernel if k == "rkv_reconstruct_kernel" else k] = {
                "flops": v["flops"] * mult, "bytes": v["bytes"] * mult}
        return out

    def describe(self) -> str:
        w = self.w
        shape = {"qwen7b": "Qwen2.5-7B-shaped stack of 28 layers",
                 "llama8b": "Llama-3.1-8B-shaped layer",
                 "long_int2": "Llama-3.1-8B-shaped layer, long context",
                 "long_bf16z": "Llama-3.1-8B-shaped layer, quantisation off"}[self.name]
        q = "bf16 z" if w.bits == 16 else f"INT{w.bits}"
        sel = (f"{self.n_sel // w.sel_block} random {w.sel_block}-token blocks"
               if w.sel_block > 1 else f"{self.n_sel} random tokens")
        per = " per layer" if self.L > 1 else ""
        return (f"{self.name}: {shape}, T={w.T}{per}, 2d_k={w.d_kv}, d_c={w.d_c}, d_ff={w.d_ff}, "
                f"{schedule_note(w)}, {q}; prefill write + {w.steps} decode steps x {sel}{per}")

    def e2e(self):
        """Public-API path with host buffers: every step uploads its inputs (every layer's
        kv rows and every selection, from pinned host memory) and reads back the last
        restore's K and V.  Copies run on a second stream, double-buffered: the next step's
        kv rows go up while this step's write phase runs (their buffer was last read by the
        previous step's write phase), its selections once the previous step's restores
        are done, and a step's results come back while the next step computes; all K
        steps, their uploads and their read-backs lie inside one timed interval."""
        import torch
        ctx, w = self.ctx, self.w
        dev, stream = ctx.dev, ctx.stream
        kv_host = [kv.cpu().pin_memory() for kv in self.kv]
        sel_host = torch.stack([torch.stack([s.cpu() for s in row]) for row in self.sels]).pin_memory()
        kv_buf = [[torch.empty_like(kv) for kv in self.kv] for _ in range(2)]
        sel_buf = [torch.empty(sel_host.shape, dtype=torch.int32, device=dev) for _ in range(2)]
        # per layer its own K and V; the last layer's (the one read back) double-buffered
        k_dev = [self.k_outs[:-1] + [torch.empty_like(self.k_out)] for _ in range(2)]
        v_dev = [self.v_outs[:-1] + [torch.empty_like(self.k_out)] for _ in range(2)]
        k_host = torch.empty(self.k_out.shape, dtype=self.k_out.dtype).pin_memory()
        v_host = torch.empty_like(k_host).pin_memory()
        copy = torch.cuda.Stream(dev)
        uploaded = [torch.cuda.Event() for _ in range(2)]
        kv_free = [torch.cuda.Event() for _ in range(2)]
        sel_free = [torch.cuda.Event() for _ in range(2)]
        result_ready = [torch.cuda.Event() for _ in range(2)]
        result_read = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):
            kv_free[b].record(stream)
            sel_free[b].record(stream)
            result_read[b].record(stream)

        def upload(i, write_start):
            b = i % 2
            with torch.cuda.stream(copy):
                copy.wait_event(kv_free[b])
                if write_start is not None:
                    copy.wait_event(write_start)
                for dst, src in zip(kv_buf[b], kv_host):
                    dst.copy_(src, non_blocking=True)
                copy.wait_event(sel_free[b])
                sel_buf[b].copy_(sel_host, non_blocking=True)
                uploaded[b].record(copy)

        def step(i, n):
            b = i % 2
            stream.wait_event(uploaded[b])
            stream.wait_event(result_read[b])
            write_start = torch.cuda.Event()
            write_start.record(stream)
            if i + 1 < n:
                upload(i + 1, write_start)
            self.write(kv_buf[b])
            kv_free[b].record(stream)
            self.read(sel_buf[b], k_dev[b], v_dev[b])
            sel_free[b].record(stream)
            result_ready[b].record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(result_ready[b])
                k_host.copy_(k_dev[b][-1], non_blocking=True)
                v_host.copy_(v_dev[b][-1], non_blocking=True)
                result_read[b].record(copy)

        def run(n):
            upload(0, None)
            for i in range(n):
                step(i, n)
            torch.cuda.synchronize(dev)

        run(max(1, ctx.args.warmup))
        ctx.barrier()
        t0 = time.perf_counter()
        run(ctx.args.steps)
        t_step = reduce_max((time.perf_counter() - t0) / ctx.args.steps, ctx.world, dev)
        tokens = reduce_sum(self.tokens_written + self.tokens_read, ctx.world, dev)
        h2d = sum(k.numel() * k.element_size() for k in kv_host) + sel_host.numel() * 4
        d2h = 2 * k_host.numel() * k_host.element_size()
        return {"value": round(tokens / t_step, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(t_step * 1e3, 3),
                "copies": "in: every layer's kv rows and every selection of the step; out: the "
                          "K and V of the step's last restore (the other restores' K/V stay on "
                          "the device, where attention would read them); second stream, "
                          "double-buffered: the next step's kv rows go up during this step's "
                          "write phase, results come back during the next step"}


class BatchedRun:
    """Decode steps over B sequences prefilled to T tokens: per step, one new token per
    sequence written, then 30 % of each sequence's history restored in one call."""

    def __init__(self, name, ctx, seed):
        import torch
        import residual_kv_cache_gb300 as rkv
        import synth
        w = synth.workload(name)
        self.name, self.w, self.ctx = name, w, ctx
        dev = ctx.dev
        B, T0 = w.batch, w.T
        self.B, self.T0 = B, T0
        self.Tcap = T0 + BATCHED_SLACK
        cfg = codec_config(rkv, w, self.Tcap, batch=B)
        self.cfg = cfg
        self.ref_pos_all = rkv.reference_positions(cfg)
        self.isref = np.zeros(self.Tcap, dtype=bool)
        self.isref[self.ref_pos_all] = True
        W = {k: v.to(dev) for k, v in synth.gen_weights(w, seed + 1).items()}
        self.codec = rkv.Codec(cfg, W, device=dev)
        self.kv = [synth.gen_kv(w, seed + 50 + b, T=self.Tcap, device=str(dev)) for b in range(B)]
        self.new_rows = torch.stack([kv for kv in self.kv], dim=1).contiguous()   # [Tcap, B, d_kv]
        self.seq_ids = np.arange(B, dtype=np.int32)
        self.pos = T0                                       # next position to append
        self.sel_cache = {}
        self.codecs = [self.codec]
        odt = torch.float32 if w.out_dtype == "fp32" else torch.bfloat16
        n_max = B * int(round(w.sel_frac * self.Tcap)) + B
        self.k_out = torch.empty((n_max, w.n_kv_heads, w.head_dim), dtype=odt, device=dev)
        self.v_out = torch.empty_like(self.k_out)
        self.prefill()

    def prefill(self):
        """Every sequence written up to T0 (not timed)."""
        self.codec.reset()
        T0 = self.T0
        pos = np.arange(T0, dtype=np.int32)
        ref, non = pos[self.isref[:T0]], pos[~self.isref[:T0]]
        for b in range(self.B):
            self.codec.pool_append(self.kv[b], np.full(len(ref), b, np.int32), ref, src_rows=ref)
            self.codec.compress(self.kv[b], np.full(len(non), b, np.int32), non, src_rows=non)
        self.pos = T0
        self.ctx.barrier()

    def selection(self, p):
        """The restore of the step that appends position p: 30 % of each sequence's
        history [0, p] at seeded random positions (seq ids, positions)."""
        import torch
        import synth
        if p not in self.sel_cache:
            n = int(round(self.w.sel_frac * (p + 1)))
            sels = [synth.gen_selection(p + 1, n, 7919 * p + b) for b in range(self.B)]
            seq = torch.cat([torch.full((n,), b, dtype=torch.int32) for b in range(self.B)])
            self.sel_cache[p] = (seq.to(self.ctx.dev), torch.cat(sels).to(self.ctx.dev))
        return self.sel_cache[p]

    def ensure_room(self, steps):
        if self.pos + steps > self.Tcap:
            self.prefill()

    def step_at(self, p, rows, seq, pos, k_out, v_out):
        pp = np.full(self.B, p, dtype=np.int32)
        if self.isref[p]:
            self.codec.pool_append(rows, self.seq_ids, pp)
        else:
            self.codec.compress(rows, self.seq_ids, pp)
        n = seq.numel()
        self.codec.reconstruct(seq, pos, k_out[:n], v_out[:n])

    def step(self):
        p = self.pos
        seq, pos = self.selection(p)
        self.step_at(p, self.new_rows[p], seq, pos, self.k_out, self.v_out)
        self.pos += 1

    def prepare(self, steps):
        self.ensure_room(steps)
        for p in range(self.pos, self.pos + steps):
            self.selection(p)

    @property
    def tokens_per_step(self):
        return self.B + self.B * int(round(self.w.sel_frac * (self.pos + 1)))

    def work_per_step(self) -> dict:
        w = self.w
        n_sel = self.B * int(round(w.sel_frac * self.T0))
        ref_before = int(np.searchsorted(self.ref_pos_all, self.T0))
        one = algorithmic_work(w, self.T0, n_sel, self.ref_pos_all[:ref_before], T=self.T0)
        rec = one["rkv_reconstruct_kernel"]
        # B sequences' pools behind one restore; one token per sequence written
        rec = {"flops": rec["flops"], "bytes": rec["bytes"] + (self.B - 1) * ref_before * w.d_kv}
        return {"rkv_reconstruct_kernel": rec}

    def describe(self) -> str:
        w = self.w
        return (f"batched: Llama-3.1-8B layer shape, {self.B} sequences prefilled to {self.T0} "
                f"tokens, {schedule_note(w)}, INT{w.bits}; one decode step = one new token per "
                f"sequence written + 30 % of every sequence's history restored in one call")

    def e2e(self):
        """Public-API decode steps with host buffers: each step uploads its 16 new kv rows
        and its selection (pinned host memory) and reads back the restored K and V.
        Copies on a second stream, double-buffered."""
        import torch
        ctx, w = self.ctx, self.w
        dev, stream = ctx.dev, ctx.stream
        K, W_ = ctx.args.steps, max(1, ctx.args.warmup)
        self.prepare(K + W_)
        p0 = self.pos
        rows_host = self.new_rows[p0:p0 + K + W_].cpu().pin_memory()
        sels = [self.selection(p) for p in range(p0, p0 + K + W_)]
        seq_host = [s.cpu().pin_memory() for s, _ in sels]
        pos_host = [q.cpu().pin_memory() for _, q in sels]
        n_max = max(s.numel() for s, _ in sels)
        rows_buf = [torch.empty_like(self.new_rows[0]) for _ in range(2)]
        seq_buf = [torch.empty(n_max, dtype=torch.int32, device=dev) for _ in range(2)]
        pos_buf = [torch.empty(n_max, dtype=torch.int32, device=dev) for _ in range(2)]
        k_dev = [torch.empty_like(self.k_out[:n_max]) for _ in range(2)]
        v_dev = [torch.empty_like(self.k_out[:n_max]) for _ in range(2)]
        k_host = torch.empty(k_dev[0].shape, dtype=k_dev[0].dtype).pin_memory()
        v_host = torch.empty_like(k_host).pin_memory()
        copy = torch.cuda.Stream(dev)
        ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("up", "free", "ready", "read")}
        for b in range(2):
            ev["free"][b].record(stream)
            ev["read"][b].record(stream)
        h2d = d2h = 0

        def upload(i):
            nonlocal h2d
            b = i % 2
            n = seq_host[i].numel()
            with torch.cuda.stream(copy):
                copy.wait_event(ev["free"][b])
                rows_buf[b].copy_(rows_host[i], non_blocking=True)
                seq_buf[b][:n].copy_(seq_host[i], non_blocking=True)
                pos_buf[b][:n].copy_(pos_host[i], non_blocking=True)
                ev["up"][b].record(copy)
            h2d += rows_host[i].numel() * rows_host.element_size() + 8 * n

        def step(i):
            nonlocal d2h
            b = i % 2
            n = seq_host[i].numel()
            stream.wait_event(ev["up"][b])
            stream.wait_event(ev["read"][b])
            self.step_at(p0 + i, rows_buf[b], seq_buf[b][:n], pos_buf[b][:n], k_dev[b], v_dev[b])
            ev["free"][b].record(stream)
            ev["ready"][b].record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(ev["ready"][b])
                k_host[:n].copy_(k_dev[b][:n], non_blocking=True)
                v_host[:n].copy_(v_dev[b][:n], non_blocking=True)
                ev["read"][b].record(copy)
            d2h += 2 * n * k_host[0].numel() * k_host.element_size()

        def run(first, n):
            upload(first)
            for i in range(first, first + n):
                if i + 1 < first + n:
                    upload(i + 1)
                step(i)
            torch.cuda.synchronize(dev)

        run(0, W_)
        ctx.barrier()
        h2d = d2h = 0
        t0 = time.perf_counter()
        run(W_, K)
        t_step = reduce_max((time.perf_counter() - t0) / K, ctx.world, dev)
        self.pos = p0 + K + W_
        tokens = sum(self.B + seq_host[i].numel() for i in range(W_, W_ + K)) / K
        tokens = reduce_sum(tokens, ctx.world, dev)
        return {"value": round(tokens / t_step, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d / K),
                "d2h_bytes_per_step": int(d2h / K), "ms_per_step": round(t_step * 1e3, 3),
                "copies": "in: the step's new kv rows and its selection; out: every restored K "
                          "and V row of the step; second stream, double-buffered"}


def run_workload(name, ctx, seed, with_e2e=True, with_cpu=True):
    """Measure one workload: device-timed steps, per-kernel event times, roofline of the
    dominant kernel, storage, end to end, and the oracle baseline."""
    import torch
    args = ctx.args
    peaks, kind = load_peaks()
    run = BatchedRun(name, ctx, seed) if name == "batched" else StackRun(name, ctx, seed)
    codecs = run.codecs
    clocks = ClockSampler(ctx.dev.index or 0)
    clocks.start()
    if name == "batched":
        run.prepare(args.warmup + 2 * args.steps)
    run.step()                                     # first touch (outside every timing)
    ctx.barrier()
    if _status(codecs) != 0:
        raise RuntimeError(f"{name}: device status flags set")
    count = lambda: sum(c.launch_count() for c in codecs)   # noqa: E731
    clocks.mark_begin()
    t_tok0 = time.perf_counter()
    if name == "batched":
        tokens = []

        def step():
            tokens.append(run.tokens_per_step)
            run.step()
        times, launches_timed = ctx.timed(step, args.steps, args.warmup, count)
        tokens = tokens[args.warmup:]
        tok_step = float(np.mean(tokens))
    else:
        times, launches_timed = ctx.timed(run.step, args.steps, args.warmup, count)
        tok_step = run.tokens_written + run.tokens_read
    clocks.mark_end()
    clk = clocks.stop()
    wall = time.perf_counter() - t_tok0
    if name == "batched":
        run.prepare(args.steps)
    ktimes = ctx.kernel_times(codecs, run.step, args.steps)
    status = _status(codecs)
    t_ms = reduce_max(sum(times) / len(times), ctx.world, ctx.dev)
    value = reduce_sum(tok_step, ctx.world, ctx.dev) / (t_ms / 1e3)
    work = run.work_per_step()
    rows = kernel_rows(ktimes, work, args.steps, peaks)
    roof = roofline_of(rows, work, peaks, kind, name)
    read_k = ("rkv_reconstruct_kernel", "rkv_reconstruct_multi_kernel")
    read_ms = sum(ms for k, (n, ms) in ktimes.items() if k in read_k) / args.steps
    write_ms = sum(ms for k, (n, ms) in ktimes.items() if k not in read_k) / args.steps
    out = {"workload": name, "value": round(value, 1), "unit": UNIT, "ms_per_step": round(t_ms, 4),
           "config": step_config(run, ctx.world), "roofline": roof,
           "kernels": rows, "gpu_launches": int(launches_timed), "clocks": clk,
           "device_status": int(status), "timed_region_s": round(wall, 3)}
    if name == "batched":
        lat = sorted(times)
        out["latency_ms"] = {"p50": round(float(np.percentile(lat, 50)), 4),
                             "p99": round(float(np.percentile(lat, 99)), 4),
                             "max": round(lat[-1], 4), "steps": len(lat)}
        out["reconstruct_tok_s"] = round((tok_step - run.B) / (read_ms / 1e3), 1) if read_ms else None
        out["write_us_per_step"] = round(write_ms * 1e3, 2)
        out["compress_tok_s"] = round(run.B / (write_ms / 1e3), 1) if write_ms else None
    else:
        out["compress_tok_s"] = round(run.tokens_written / (write_ms / 1e3), 1) if write_ms else None
        out["reconstruct_tok_s"] = round(run.tokens_read / (read_ms / 1e3), 1) if read_ms else None
    out["storage"] = storage_report(codecs[0], run.w)
    if with_e2e:
        out["e2e"] = run.e2e()
        status |= _status(codecs)
        out["device_status"] = int(status)
    if name in Q_HEADS:
        out["sparse_attention"] = measure_attention(run, ctx)
    if with_cpu and ctx.rank == 0 and ctx.world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(name, args.cpu_seconds)
    for c in codecs:
        c.free()
    del run
    torch.cuda.empty_cache()
    return out


# query heads of the models the stacks are shaped after (Llama-3-8B: 32 over 8 key/value
# heads; Qwen2.5-7B: 28 over 4)
Q_HEADS = {"llama8b": 32, "qwen7b": 28}


def measure_attention(run, ctx):
    """The sparse layer's read after each decode step (layer 0's selection), two ways:
    rkv_reconstruct then rkv_sparse_attention (K/V written, then read back while still in
    L2), and rkv_restore_attend (K/V kept on chip, then the per-tile merge).  Each is
    timed back to back over the steps (events around the whole sequence of calls) and
    per kernel (event pairs around each launch).  Attention bytes: the K and V rows it
    reads, q in, o out."""
    import torch
    w, codec = run.w, run.codecs[0]
    hq = Q_HEADS.get(run.name, 4 * w.n_kv_heads)
    g = torch.Generator().manual_seed(4242)
    q = torch.randn(hq, w.head_dim, generator=g).to(ctx.dev)
    out = torch.empty(hq, w.head_dim, dtype=torch.float32, device=ctx.dev)
    out_f = torch.empty_like(out)
    rows = [row[0] for row in run.sels]
    unfused = lambda sel: (codec.reconstruct(run.seq0, sel, run.k_out, run.v_out),
                           codec.sparse_attention(q, run.k_out, run.v_out, out))
    fused = lambda sel: codec.restore_attend(run.seq0, sel, q, out_f)

    def back_to_back(fn):
        per = []
        for _ in range(ctx.args.steps):
            ctx.flush.fill_(1.0)
            ctx.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for sel in rows:
                fn(sel)
            e1.record()
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) / len(rows))
        return float(np.median(per)) * 1e3

    def per_kernel(fn):
        codec.set_timing(True)
        codec.get_timing(reset=True)
        for _ in range(ctx.args.steps):
            ctx.flush.fill_(1.0)
            ctx.barrier()
            for sel in rows:
                fn(sel)
            ctx.barrier()
        t = codec.get_timing(reset=True)
        codec.set_timing(False)
        return {k: ms / n * 1e3 for k, (n, ms) in t.items() if n}

    for fn in (unfused, fused):                      # warm-up
        for sel in rows[:4]:
            fn(sel)
    torch.cuda.synchronize()
    b2b_unfused, b2b_fused = back_to_back(unfused), back_to_back(fused)
    k_unfused, k_fused = per_kernel(unfused), per_kernel(fused)
    us = k_unfused["rkv_attention_kernel"]
    n = run.n_sel
    kv_bytes = 2 * n * w.n_kv_heads * w.head_dim * 2
    peaks, kind = load_peaks()
    gbs = (kv_bytes + 2 * hq * w.head_dim * 4) / (us * 1e-6) / 1e9
    d = (out - out_f).abs().max().item() / max(out.abs().max().item(), 1e-30)
    return {"tokens": n, "q_heads": hq, "kv_heads": w.n_kv_heads, "us_per_call": round(us, 2),
            "gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
            "peak_kind": f"{kind} copy",
            "note": "K/V read right after their restore (L2-resident); o is fp32",
            "restore_then_attention_us": round(b2b_unfused, 2),
            "restore_attend_us": round(b2b_fused, 2),
            "fused_speedup": round(b2b_unfused / b2b_fused, 3),
            "per_kernel_us": {k: round(v, 2) for k, v in {**k_unfused, **k_fused}.items()},
            "fused_vs_unfused_max_rel_diff": float(f"{d:.3e}"),
            "timing": "per step: one restore + attention of layer 0's selection; median over "
                      "steps of (events around all decode steps' calls) / calls; per_kernel: "
                      "event pairs around each launch"}


def storage_report(codec, w) -> dict:
    """Bytes the codec's storage keeps per token (the caller's storage tensors over B x T
    tokens: FP8 references with their norms and positions, codes, extremes, slots)
    against FP16 K and V (2 bytes per value of the 2d_k-wide row).  The library's bf16
    copy of the pool (the retrieval's tensor-core operand, a compute cache derived from
    the FP8 references) is shown beside it."""
    names = ["pool_fp8", "pool_norm2", "pool_pos", "codes", "meta", "ref_idx"]
    nbytes = {n: getattr(codec, n).numel() * getattr(codec, n).element_size() for n in names}
    tokens = codec.codes.shape[0] * codec.codes.shape[1]
    fp16 = 2 * w.d_kv
    total = sum(nbytes.values())
    cache = codec.pool_cache_bytes()
    return {"bytes_per_token": round(total / tokens, 1),
            "fraction_of_fp16_kv": round(total / tokens / fp16, 4),
            "compute_cache_bytes_per_token": round(cache / tokens, 1),
            "fraction_with_compute_cache": round((total + cache) / tokens / fp16, 4)}


def step_config(run, world: int) -> dict:
    """The workload of one step, the same on both arms of the comparison."""
    if isinstance(run, BatchedRun):
        tok = run.B + run.B * int(round(run.w.sel_frac * run.T0))
    else:
        tok = run.tokens_written + run.tokens_read
    cfg = {"workload": run.describe(), "tokens_per_step": tok,
           "l2": "flushed before every timed step",
           "parallelism": f"replicas x{world} (independent sequences)"}
    if ENCODER["mean_precompute"]:
        cfg["encoder_mean"] = "per-reference pre-activations (mean_precompute=1)"
    return cfg


# ------------------------------------------------------------------ CUDA arm: the line
def run_cuda(args):
    import torch
    from residual_kv_cache_gb300 import build as _build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    ctx = Ctx(args, dev, world, rank)
    names = [args.workload] if args.workload else list(WORKLOAD_ORDER)
    seed = 1000 * (rank + 1)
    results = {}
    for i, name in enumerate(names):
        results[name] = run_workload(name, ctx, seed + 100 * i)
    head = results[names[0]]
    out = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic", "config": head["config"],
           "compress_tok_s": head.get("compress_tok_s"),
           "reconstruct_tok_s": head.get("reconstruct_tok_s"),
           "roofline": head["roofline"], "kernels": head["kernels"], "e2e": head.get("e2e"),
           "storage": head["storage"], "gpu_launches": head["gpu_launches"],
           "clocks": head["clocks"], "device_status": head["device_status"]}
    if "cpu_baseline" in head:
        out["cpu_baseline"] = head["cpu_baseline"]
    if "sparse_attention" in head:
        out["sparse_attention"] = head["sparse_attention"]
    if len(names) > 1:
        out["configs"] = {n: results[n] for n in names[1:]}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ oracle timing
_CPU_INPUTS = {}          # the last workload's sample inputs, drawn once per process


def cpu_baseline(name: str, budget_s: float = 16.0) -> dict:
    """Time the CPU oracle (as it stands) on a bounded sample of one layer of the
    workload, per token, and scale to the step's token mix."""
    import torch
    import synth
    from oracle import codec as C

    cores = len(os.sched_getaffinity(0))
    w = synth.workload(name)
    T = min(w.T, (1 << 27) // w.d_kv)      # the sample's sequence (pool) length
    if name not in _CPU_INPUTS:
        kv = synth.gen_kv(w, 1000, T=T).to(torch.float64).numpy()
        W = {k: v.to(torch.float64).numpy() for k, v in synth.gen_weights(w, 1001).items()}
        _CPU_INPUTS.clear()
        _CPU_INPUTS[name] = (kv, W)
    kv, W = _CPU_INPUTS[name]
    sh = C.Shape(w.n_kv_heads, w.head_dim, w.d_c, w.d_ff, w.topk, w.group, w.bits, w.stride,
                 w.rope_base, SCHEDULE["alpha"], SCHEDULE["sink"])
    t0 = time.perf_counter()
    pool = C.build_pool(kv, T, w.stride, sh.ref_alpha, sh.ref_sink)
    t_pool = time.perf_counter() - t0
    rng = np.random.default_rng(0)
    nonref = np.nonzero(~C.is_reference(np.arange(T), w.stride, sh.ref_alpha, sh.ref_sink))[0]
    # compress sample: batches of 64 tokens until half the budget is used
    n_c, t_c = 0, 0.0
    enc_q, enc_meta, enc_idx, enc_pos = [], [], [], []
    while t_c < budget_s / 2 and n_c < 4096:
        p = np.sort(rng.choice(nonref, 64, replace=False))
        t0 = time.perf_counter()
        e = C.encode_tokens(kv[p], p, pool, W, sh, "operand")
        t_c += time.perf_counter() - t0
        n_c += len(p)
        enc_q.append(e["q"]); enc_meta.append(e["meta"]); enc_idx.append(e["idx"]); enc_pos.append(p)
    q = np.concatenate(enc_q); meta = np.concatenate(enc_meta); idx = np.concatenate(enc_idx)
    pos = np.concatenate(enc_pos)
    n_r, t_r = 0, 0.0
    while t_r < budget_s / 2 and n_r < 65536:
        t0 = time.perf_counter()
        zt = C.dequantize(q, meta, sh.bits, sh.group)
        means = np.stack([C.reference_mean(pool.vals, i[i >= 0]) for i in idx])
        kvh = C.decode(zt, W["Wd"], means)
        K, V = C.split_kv(kvh, sh.n_kv_heads, sh.head_dim)
        C.rope(K, pos, sh.rope_base)
        t_r += time.perf_counter() - t0
        n_r += len(pos)
    per_c = (t_c + t_pool * n_c / T) / n_c
    per_r = t_r / n_r
    if name == "batched":
        n_read = w.batch * int(round(w.sel_frac * w.T))
        written, read = w.batch, n_read
    else:
        n_sel = w.n_sel
        written, read = w.layers * w.T, w.steps * w.layers * n_sel
    t_step = per_c * written + per_r * read
    short = "" if T == w.T else f" (a {T}-token sequence: its pool has {len(pool.pos)} references)"
    return {"value": round((written + read) / t_step, 2), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{n_c} compressed tokens (random non-reference positions of one layer{short}, "
                      f"{schedule_note(w)}) and {n_r} restored tokens of the {name} workload, "
                      f"per token, scaled to the step mix ({written} written + {read} restored)",
            "compress_tok_s": round(1 / per_c, 2), "reconstruct_tok_s": round(1 / per_r, 2),
            "seconds": round(t_c + t_r + t_pool, 2)}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    name = args.workload or HEADLINE
    vals, last = [], None
    for _ in range(args.warmup):
        cpu_baseline(name, args.cpu_seconds / 4)
    for _ in range(args.steps):
        last = cpu_baseline(name, args.cpu_seconds)
        vals.append(last["value"])
    v = statistics.mean(vals)
    import synth
    w = synth.workload(name)
    if name == "batched":
        tokens = w.batch + w.batch * int(round(w.sel_frac * w.T))
        desc = (f"batched: Llama-3.1-8B layer shape, {w.batch} sequences prefilled to {w.T} "
                f"tokens, {schedule_note(w)}, INT{w.bits}; one decode step = one new token per "
                f"sequence written + 30 % of every sequence's history restored in one call")
    else:
        n_sel = (int(round(w.sel_frac * (w.T // w.sel_block))) * w.sel_block
                 if w.sel_block > 1 else w.n_sel)
        tokens = w.layers * w.T + w.steps * w.layers * n_sel
        desc = None
    cfg = {"workload": desc or _stack_description(name), "tokens_per_step": tokens,
           "l2": "flushed before every timed step",
           "parallelism": "replicas x1 (independent sequences)"}
    out = {"metric": METRIC, "value": round(v, 2), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tokens / v * 1e3, 1),
           "ms_per_step_kind": "extrapolated: each step times a bounded sample of the workload "
                               "and scales its per-token times to the step's token mix",
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference", "config": cfg,
           "cpu_baseline": {"value": round(v, 2), "unit": UNIT, "cores": last["cores"],
                            "kind": "oracle", "sample": last["sample"]},
           "e2e": {"value": round(v, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def _stack_description(name: str) -> str:
    """The description a StackRun gives, without a GPU."""
    import synth
    w = synth.workload(name)

    class _R(StackRun):
        def __init__(self):
            self.name, self.w, self.L = name, w, w.layers
            self.n_sel = (int(round(w.sel_frac * (w.T // w.sel_block))) * w.sel_block
                          if w.sel_block > 1 else w.n_sel)
    return _R().describe()


def run_kernel_case(args):
    """Minimal case for kernel captures under ncu: one layer of the workload, one
    prefill write and two decode-step restores, each followed by the sparse attention
    over its rows and by the fused restore + attention of the same selection (no timing,
    no CPU work)."""
    import torch
    import residual_kv_cache_gb300 as rkv
    from residual_kv_cache_gb300 import build as _build
    import synth

    _build.build()
    name = args.workload or HEADLINE
    w = synth.workload(name)
    if args.tokens:
        w = synth.workload(name, T=args.tokens)
    dev = torch.device("cuda", 0)
    kv = synth.gen_kv(w, 1000, device=str(dev) if w.T > 65536 else "cpu").to(dev)
    W = {k: v.to(dev) for k, v in synth.gen_weights(w, 1001).items()}
    cfg = codec_config(rkv, w, w.T)
    codec = rkv.Codec(cfg, W, device=dev)
    ref, non = split_positions(rkv.reference_positions(cfg), w.T)
    codec.pool_append(kv, np.zeros_like(ref), ref, src_rows=ref)
    codec.compress(kv, np.zeros_like(non), non, src_rows=non)
    g = torch.Generator().manual_seed(4242)
    q = torch.randn(Q_HEADS.get(name, 4 * w.n_kv_heads), w.head_dim, generator=g).to(dev)
    fuse = w.head_dim == 128 and cfg.out_dtype == "bf16"
    for s in range(2):
        if w.sel_block > 1:
            sel = synth.gen_block_selection(w.T, w.sel_block, w.sel_frac, 1010 + s).to(dev)
        else:
            sel = synth.gen_selection(w.T, w.n_sel, 1010 + s).to(dev)
        zero = torch.zeros(sel.numel(), dtype=torch.int32, device=dev)
        K, V = codec.reconstruct(zero, sel)
        codec.sparse_attention(q, K, V)             # the sparse layer's attention over them
        if fuse:
            codec.restore_attend(zero, sel, q)          # the same read, restored on chip
    # with --layers L > 1: L - 1 more layers prefilled the same way, then two decode steps
    # restoring all L layers' selections in one launch each (rkv_reconstruct_multi)
    codecs = [codec]
    for l in range(1, args.layers):
        kvl = synth.gen_kv(w, 1000 + 7 * l, device=str(dev) if w.T > 65536 else "cpu").to(dev)
        Wl = {k: v.to(dev) for k, v in synth.gen_weights(w, 1001 + 7 * l).items()}
        cl = rkv.Codec(cfg, Wl, device=dev)
        cl.pool_append(kvl, np.zeros_like(ref), ref, src_rows=ref)
        cl.compress(kvl, np.zeros_like(non), non, src_rows=non)
        codecs.append(cl)
        del kvl
    if args.layers > 1:
        for s in range(2):
            sels = [(synth.gen_block_selection(w.T, w.sel_block, w.sel_frac, 1020 + 31 * s + l)
                     if w.sel_block > 1 else synth.gen_selection(w.T, w.n_sel, 1020 + 31 * s + l)).to(dev)
                    for l in range(args.layers)]
            rkv.reconstruct_multi(codecs, [torch.zeros_like(x) for x in sels], sels)
    torch.cuda.synchronize()
    flags = 0
    for c in codecs:
        flags |= c.get_status()
    print(json.dumps({"kernel_case": name, "T": w.T, "layers": args.layers,
                      "launches": sum(c.launch_count() for c in codecs), "status": flags}))
    if flags:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--workload", default=None, choices=list(WORKLOAD_ORDER),
                    help="measure one workload only (default: all, headline first)")
    ap.add_argument("--alpha", type=float, default=0.0,
                    help="dynamic-stride growth of the reference schedule (0: fixed stride)")
    ap.add_argument("--sink", type=int, default=0, help="sink tokens of the reference schedule")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-case", action="store_true",
                    help="run one layer's prefill and two restores, for kernel captures")
    ap.add_argument("--tokens", type=int, default=0, help="override T for --kernel-case")
    ap.add_argument("--layers", type=int, default=1,
                    help="--kernel-case: layers restored together by one multi-context launch")
    ap.add_argument("--mean-precompute", action="store_true",
                    help="encoder mean from per-reference pre-activations (mean_precompute=1)")
    args = ap.parse_args()
    if args.alpha < 0 or args.sink < 0:
        ap.error("--alpha and --sink must be >= 0")
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    SCHEDULE.update(alpha=float(args.alpha), sink=int(args.sink))
    ENCODER.update(mean_precompute=1 if args.mean_precompute else 0)
    if args.kernel_case:
        run_kernel_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
