#!/usr/bin/env python
"""Benchmark of the verification pass on one GB300 (or N replicas).

One step = the whole hot path over one batch of the named workload:
ssv_rope_copy (paired RoPE index) -> ssv_verify_attn (temporal-mask
attention over prompt cache + 2B tail) -> ssv_accept (longest accepted
prefix).  Inputs are seeded and synthetic (shapes of the named workload),
resident in HBM before timing; every step is preceded by a 256 MB memset
so that no input starts in the 129 MB L2, and each step is bracketed by
CUDA events on the launching stream (the memset is outside the events).

Prints one JSON line (rank 0).  `value` = algorithmic HBM bytes of one step
(rope read+write, KV cache once per kv head + Q + K/V_new + O, every
logits / noise / draft row the acceptance needs) / device step time.
`e2e` repeats the measurement through the same public calls with the
inputs copied from pinned host memory every step and the accepted tokens
read back.  `roofline` is for the dominant op (largest device time).

--impl reference times the CPU oracle (plain numpy fp64) on the machine's host
cores, one sequence of the workload per step, same metric and unit.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from diffusion_speculative_verification_gb300 import workloads as W  # noqa: E402

METRIC = "verify-attn TFLOP/s or HBM GB/s (% of roofline); accept sequences/s"
ACCEPT_INDEX = {"tiny": 1, "gqa1p7b": 0, "gqa8b": 0, "prefill": None, "sweep": 1}
FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------
def attn_work(a: W.AttnInputs, out_bytes: int):
    es = 2 if a.dtype == W.BF16 else 4
    rows, Hq, Hkv, d = a.total_rows, a.Hq, a.Hkv, a.d
    pairs = 0.0
    for C, N, B, *_ in a.seqs:
        C, N, B = float(C), float(N), float(B)
        P = C + N
        pairs += N * (N + 1) / 2 + N * C + 2 * B * P + B * (B + 1) / 2 + B * B
    flops = pairs * Hq * 4.0 * d
    bytes_ = (a.total_cache * Hkv * d * 2 * es + rows * Hq * d * es + rows * Hkv * d * 2 * es
              + rows * Hq * d * out_bytes)
    return float(bytes_), float(flops)


def rope_bytes(a: W.AttnInputs) -> float:
    es = 2 if a.dtype == W.BF16 else 4
    return 2.0 * a.total_rows * (a.Hq + a.Hkv) * a.d * es


def accept_bytes(x) -> float:
    if x is None:
        return 0.0
    les = 2 if x.logits_dtype == W.BF16 else 4
    tot = 0.0
    for B, g in zip(x.blocks, x.gammas):
        need = min(int(g) + 1, int(B))
        tot += need * x.V * les
        if x.mode == W.MODE_REJECT:
            tot += int(g) * x.V * les
        if x.mode == W.MODE_GUMBEL and x.T != 0.0:
            tot += need * x.V * 4      # noise rows read (generated noise reads nothing more)
    return tot


def commit_bytes(a: W.AttnInputs, n_acc) -> float:
    """K and V rows read and written by the commit step: per sequence its N
    fresh prompt rows and n_acc accepted data rows."""
    es = 2 if a.dtype == W.BF16 else 4
    rows = float(np.sum(a.seqs[:, 1].astype(np.int64) + np.asarray(n_acc, np.int64)))
    return 2.0 * 2.0 * rows * a.Hkv * a.d * es


def lmhead_work(x: W.LmheadInputs):
    """Useful work of the fused LM head + acceptance: (bytes, flops, verified
    rows).  Bytes: the LM head and the hidden states read once, plus the noise
    rows of the verified slots (coupled noise at T > 0); flops: 2 V hidden per
    verified row (the kernel also multiplies the unverified and padding rows
    of its M-tiles; that work is not counted)."""
    a = x.acc
    need = [min(int(g) + 1, int(B)) for g, B in zip(a.gammas, a.blocks)]
    ver = int(sum(need))
    S = int(np.sum(a.blocks))
    b = a.V * x.hidden * 2.0 + S * x.hidden * 2.0
    if a.mode == W.MODE_GUMBEL and a.T != 0.0:
        b += ver * a.V * 4.0
    return b, 2.0 * ver * a.V * x.hidden, ver


def aggregate_ms(local_ms: float, dist_mod=None, device=None) -> float:
    """Max over ranks of a per-rank time (identity on one rank)."""
    if dist_mod is None or not dist_mod.is_available() or not dist_mod.is_initialized():
        return float(local_ms)
    if dist_mod.get_world_size() == 1:
        return float(local_ms)
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def kernel_launches(x) -> int:
    """Kernels one step launches: the rotation and the verification
    attention, then the acceptance -- the streaming reduce plus its
    completion (one finish kernel for the decision rules; for rejection
    sampling the row merge with the walk, then the three emission passes:
    normalisers, masses, the token)."""
    n = 1 + 1
    if x is not None:
        n += 5 if x.mode == W.MODE_REJECT else 2
    return n


KERNEL_OF_OP = {"verify_attn": "attn_tc_kernel", "accept": "accept_stream_kernel", "rope": "rope_copy_kernel",
                "commit": "commit_kernel", "lmhead": "lmhead_accept_kernel"}
KERNEL_SOURCES = {"attn_tc_kernel": ["attn_tc.cu", "tc_ptx.cuh", "attn.cuh", "ssv_internal.cuh"],
                  "accept_stream_kernel": ["accept_stream.cu", "accept.cuh", "tc_ptx.cuh", "noisegen.cuh", "dfloat.cuh"],
                  "accept_reduce_kernel": ["accept.cu", "accept.cuh", "dfloat.cuh", "noisegen.cuh"],
                  "accept_sample_kernel": ["accept.cu", "accept.cuh", "dfloat.cuh", "noisegen.cuh"],
                  "accept_emit_norm_kernel": ["accept.cu", "accept.cuh", "dfloat.cuh", "noisegen.cuh"],
                  "accept_locate_kernel": ["accept.cu", "accept.cuh", "dfloat.cuh", "noisegen.cuh"],
                  "rope_copy_kernel": ["rope.cu"],
                  "commit_kernel": ["commit.cu"],
                  "lmhead_accept_kernel": ["lmhead.cu", "tc_ptx.cuh", "accept.cuh", "dfloat.cuh"],
                  "lmhead_gather_kernel": ["lmhead.cu", "tc_ptx.cuh", "accept.cuh", "dfloat.cuh"],
                  "tree_attn_kernel": ["tree.cu", "accept.cuh", "dfloat.cuh", "tc_ptx.cuh"],
                  "tree_reduce_kernel": ["tree.cu", "accept.cuh", "dfloat.cuh", "tc_ptx.cuh"]}


def strip_comments(src: str) -> str:
    """C/CUDA source without its comments, whitespace runs collapsed (string
    and character literals kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def code_digest(kern: str) -> str:
    """First 16 hex digits of the sha256 of a kernel's source files, comments
    and whitespace left out: an edit of the comments keeps it, any change of
    the code alters it."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kern]:
        with open(os.path.join(ROOT, "diffusion_speculative_verification_gb300", "csrc", name)) as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(op: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json),
    or None when there is none or the kernel's code changed since it was taken."""
    kern = KERNEL_OF_OP.get(op)
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if kern is None or not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{kern}_{workload}")
    if not rec:
        return None
    if code_digest(kern) != rec.get("source_sha256_16"):
        return None
    return rec["dram_bytes_per_launch"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._th = threading.Thread(target=self._read, daemon=True)
        self._th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._th.join(timeout=2)
        self.proc = None

    def window(self, t0, t1):
        """Median SM clock, maximum clock and throttle reasons of the samples
        taken between host times t0 and t1 (the last few if none fell in)."""
        if self.proc is None and not self.lines:
            return None
        time.sleep(0.12)
        lines = list(self.lines)
        sel = [l for (t, l) in lines if t0 - 0.1 <= t <= t1 + 0.1] or [l for _, l in lines[-3:]]
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in sel:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle, one sequence per step
# ---------------------------------------------------------------------------
def _subset(a: W.AttnInputs, x, b: int):
    """Sequence b of the workload as a 1-sequence batch (attention and acceptance inputs)."""
    C, N, B, q_off, kv_off, t_off = (int(v) for v in a.seqs[b])
    rows = N + 2 * B
    sa = W.AttnInputs(a.name, a.dtype, a.Hq, a.Hkv, a.d, a.rope_base, W.seq_table([C], [N], [B]),
                      a.tau[t_off:t_off + B].copy(), a.q_raw[q_off:q_off + rows], a.k_new_raw[q_off:q_off + rows],
                      a.v_new[q_off:q_off + rows], a.k_cache[kv_off:kv_off + C], a.v_cache[kv_off:kv_off + C])
    sx = None
    if x is not None:
        so = int(x.slot_off[b])
        sl = slice(so, so + B)
        nrow = x.noise_row[sl]
        sx = W.AcceptInputs(x.name, x.mode, x.T, x.V, x.logits_dtype, x.blocks[b:b + 1], x.gammas[b:b + 1],
                            np.zeros(1, np.int32), x.tau[sl], x.logits[sl],
                            None if x.draft_logits is None else x.draft_logits[sl], x.draft_tokens[sl],
                            None if x.noise is None else x.noise[np.sort(nrow)],
                            np.argsort(np.argsort(nrow)).astype(np.int32), x.u_accept[sl], x.u_sample[b:b + 1])
    return sa, sx


def oracle_step(sa: W.AttnInputs, sx):
    import oracle.rope as orope
    import oracle.attention as oattn
    import oracle.accept as oacc
    q, k = orope.rope_copy_batch(sa.seqs, W.values_f64(sa.q_raw, sa.dtype), W.values_f64(sa.k_new_raw, sa.dtype),
                                 sa.rope_base)
    oattn.verify_attention(sa.seqs, sa.tau, q, W.values_f64(sa.k_cache, sa.dtype), W.values_f64(sa.v_cache, sa.dtype),
                           k, W.values_f64(sa.v_new, sa.dtype))
    if sx is not None:
        oacc.accept_batch(sx)


def seq_bytes(sa, sx, out_bytes):
    return rope_bytes(sa) + attn_work(sa, out_bytes)[0] + accept_bytes(sx)


def _cpu_baseline_child(config, seconds, q):
    a = W.workload_attn(config)
    xi = ACCEPT_INDEX[config]
    x = None if xi is None else W.workload_accept(config, xi)
    out_b = 2 if a.dtype == W.BF16 else 4
    done_bytes, n, t0 = 0.0, 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        sa, sx = _subset(a, x, n % a.batch)
        oracle_step(sa, sx)
        done_bytes += seq_bytes(sa, sx, out_b)
        n += 1
    dt = time.perf_counter() - t0
    q.put((done_bytes / dt / 1e9, n, dt))


def cpu_baseline(config: str, seconds: float = 12.0):
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = str(cores)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_cpu_baseline_child, args=(config, seconds, q))
    p.start()
    gbs, n, dt = q.get()
    p.join()
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} sequences of the {config} workload (rope + attention + acceptance, numpy fp64), "
                      f"{dt:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    a = W.workload_attn(args.config)
    xi = ACCEPT_INDEX[args.config]
    x = None if xi is None else W.workload_accept(args.config, xi)
    out_b = 2 if a.dtype == W.BF16 else 4
    for i in range(args.warmup):
        oracle_step(*_subset(a, x, i % a.batch))
    tot_t, tot_b = 0.0, 0.0
    for i in range(args.steps):
        sa, sx = _subset(a, x, i % a.batch)
        t0 = time.perf_counter()
        oracle_step(sa, sx)
        tot_t += time.perf_counter() - t0
        tot_b += seq_bytes(sa, sx, out_b)
    gbs = tot_b / tot_t / 1e9
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": args.config, "unit_per_step": "one sequence"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"one {args.config} sequence per step, {args.steps} steps"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class ConfigRun:
    """Device buffers, argument blocks and timed ops of one named workload:
    ssv_rope_copy, ssv_verify_attn and ssv_accept, each alone, and the whole
    step (ssv_verify_step) — plus the commit step for the headline workload."""

    def __init__(self, config, dev, with_commit):
        import torch
        from diffusion_speculative_verification_gb300 import ssv, io as sio
        self.config = config
        self.dev = dev
        a = self.a = W.workload_attn(config)
        xi = ACCEPT_INDEX[config]
        x = self.x = None if xi is None else W.workload_accept(config, xi)
        t = self.t = sio.attn_to_device(a, dev)
        acc = self.acc = None if x is None else sio.accept_to_device(x, dev)
        out_dtype = torch.bfloat16 if a.dtype == W.BF16 else torch.float32
        self.out_b = 2 if a.dtype == W.BF16 else 4
        self.qo = torch.empty_like(t["q"])
        self.ko = torch.empty_like(t["k_new"])
        self.o = torch.empty(t["q"].shape, dtype=out_dtype, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.batch = t["batch"]
        self.aargs = ssv.attn_args(self.qo, t["k_cache"], t["v_cache"], self.ko, t["v_new"], self.o, self.batch,
                                   t["tau"], 0.0, self.status)
        self.ws_attn = torch.zeros(max(256, ssv.verify_attn_workspace_bytes(self.aargs)), dtype=torch.uint8,
                                   device=dev)
        self.rargs = ssv.rope_args(t["q"], t["k_new"], self.batch, a.rope_base, q_out=self.qo, k_out=self.ko)
        self.outs = self.cargs = self.ws_acc = None
        if acc is not None:
            self.outs = (torch.empty(x.batch, dtype=torch.int32, device=dev),
                         torch.empty(x.batch, dtype=torch.int32, device=dev),
                         torch.empty(len(x.tau), dtype=torch.int32, device=dev))
            self.cargs = ssv.accept_args(acc["mode"], acc["T"], acc["logits"], acc["draft_tokens"], acc["tau"],
                                         acc["block"], acc["gamma"], acc["slot_off"], *self.outs,
                                         acc["draft_logits"], acc["noise"], acc["noise_row"], acc["u_accept"],
                                         acc["u_sample"], acc["max_block"], self.status)
            self.ws_acc = torch.zeros(ssv.accept_workspace_bytes(self.cargs), dtype=torch.uint8, device=dev)
        self.gargs = None
        if acc is not None and x.mode == W.MODE_GUMBEL and x.T != 0.0:
            # the same acceptance with the coupled noise generated on the device
            # (each slot's position = its table row index; a fixed generator key)
            self.gargs = ssv.accept_args(W.MODE_GUMBEL_GEN, acc["T"], acc["logits"], acc["draft_tokens"], acc["tau"],
                                         acc["block"], acc["gamma"], acc["slot_off"], *self.outs, None, None,
                                         acc["noise_row"], None, None, acc["max_block"], self.status,
                                         noise_seed=0x5EED5EED5EED)
        self.margs = None
        if with_commit:
            # commit step (timed on its own, not part of the step): the rotated
            # fresh rows into destination caches laid out with room, seeded
            # accepted counts
            self.n_acc_c, dst_off, dst_cap, dst_rows, _ = W.commit_layout(a, 2024)
            self.k_dst = torch.zeros((dst_rows, a.Hkv, a.d), dtype=self.ko.dtype, device=dev)
            self.v_dst = torch.zeros_like(self.k_dst)
            self.commit_in = [sio.int_tensor(v, dev) for v in (self.n_acc_c, dst_off, dst_cap)]
            self.new_len = torch.empty(a.batch, dtype=torch.int32, device=dev)
            self.margs = ssv.commit_args(self.ko, t["v_new"], self.k_dst, self.v_dst, self.batch, t["tau"],
                                         *self.commit_in, self.new_len, self.status)

    # ---- ops (each on stream s) ----
    def op_rope(self, s):
        from diffusion_speculative_verification_gb300 import ssv
        ssv.rope_copy(self.t["q"], self.t["k_new"], self.batch, self.a.rope_base, q_out=self.qo, k_out=self.ko,
                      stream=s)

    def op_attn(self, s):
        import ctypes as C
        from diffusion_speculative_verification_gb300 import ssv
        r = ssv.lib().ssv_verify_attn(C.byref(self.aargs), self.ws_attn.data_ptr(), self.ws_attn.numel(),
                                      s.cuda_stream)
        if r:
            raise ssv.SsvError(r, "ssv_verify_attn")

    def op_accept(self, s):
        import ctypes as C
        from diffusion_speculative_verification_gb300 import ssv
        if self.acc is not None:
            r = ssv.lib().ssv_accept(C.byref(self.cargs), self.ws_acc.data_ptr(), self.ws_acc.numel(), s.cuda_stream)
            if r:
                raise ssv.SsvError(r, "ssv_accept")

    def op_accept_gen(self, s):
        import ctypes as C
        from diffusion_speculative_verification_gb300 import ssv
        r = ssv.lib().ssv_accept(C.byref(self.gargs), self.ws_acc.data_ptr(), self.ws_acc.numel(), s.cuda_stream)
        if r:
            raise ssv.SsvError(r, "ssv_accept (generated noise)")

    def op_commit(self, s):
        import ctypes as C
        from diffusion_speculative_verification_gb300 import ssv
        r = ssv.lib().ssv_commit(C.byref(self.margs), s.cuda_stream)
        if r:
            raise ssv.SsvError(r, "ssv_commit")

    def op_step(self, s):
        """The whole step in one call (ssv_verify_step: the three kernels
        chained with programmatic dependent launch)."""
        from diffusion_speculative_verification_gb300 import ssv
        ssv.verify_step(self.rargs, self.aargs, self.ws_attn, self.cargs, self.ws_acc, stream=s)

    def step_eager(self, evs, s):
        for j, op in enumerate((self.op_rope, self.op_attn, self.op_accept)):
            evs[j].record(s)
            op(s)
        evs[3].record(s)

    def work(self):
        rb = rope_bytes(self.a)
        ab, af = attn_work(self.a, self.out_b)
        return rb, ab, af, accept_bytes(self.x)

    def check_status(self):
        from diffusion_speculative_verification_gb300 import ssv
        st = ssv.get_status(self.status)
        assert st == ssv.SSV_OK, f"{self.config}: device status {ssv.status_string(st)}"


class Timer:
    """Graph-replay timing on one stream.  Each graph holds K x [L2 flush,
    body]; a body's time per step is (replay - flush-only replay) / K."""

    def __init__(self, dev, stream, steps, l2_flush):
        self.dev, self.stream, self.steps, self.l2_flush = dev, stream, steps, l2_flush
        self._flush = None

    def capture(self, bodies):
        import torch
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(self.dev)
        cap.wait_stream(self.stream)
        with torch.cuda.graph(g, stream=cap):
            for _ in range(self.steps):
                self.l2_flush()
                for body in bodies:
                    body(cap)
        self.stream.wait_stream(cap)
        return g

    def replay_ms(self, g):
        import torch
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        g.replay()
        e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def flush_ms(self):
        if self._flush is None:
            self._flush = self.capture(())
            self._flush.replay()
        return self.replay_ms(self._flush)


def read_floor_ms(tm: Timer, dev, nbytes: int) -> float:
    """Achievable time of a plain streaming read of `nbytes` after the same L2
    flush, in the same graph-replay measurement (ssv_stream_read: 16-byte
    loads, two CTAs per SM).  It pays the launch and first-byte latency a
    kernel of the path pays, so on small workloads it is the floor such a
    kernel can approach, well above bytes / peak bandwidth."""
    import torch
    from diffusion_speculative_verification_gb300 import ssv
    buf = torch.ones(max((nbytes + 15) // 16, 1) * 4, dtype=torch.int32, device=dev)
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    g = tm.capture((lambda st: ssv.stream_read(buf, out, st),))
    g.replay()
    torch.cuda.synchronize()
    t = (tm.replay_ms(g) - tm.flush_ms()) / tm.steps
    del g, buf
    return t


def floors_of(tm: Timer, dev, run: ConfigRun) -> dict:
    rb, ab, af, cb = run.work()
    f = {"verify_attn": read_floor_ms(tm, dev, int(ab)), "rope": read_floor_ms(tm, dev, int(rb))}
    if run.x is not None:
        f["accept"] = read_floor_ms(tm, dev, int(cb))
    return f


def warm(run: ConfigRun, stream, l2_flush, n):
    import torch
    for _ in range(n):
        l2_flush()
        run.op_step(stream)
        if run.margs is not None:
            run.op_commit(stream)
    torch.cuda.synchronize()
    run.check_status()


def roofline_of(run: ConfigRun, op_ms, hbm_peak, tf_peak, peak_kind):
    """Roofline record of the dominant op (largest device time): HBM-bound
    ops against the measured copy bandwidth; the attention of the prefill
    workload against the measured bf16 tensor peak."""
    rb, ab, af, cb = run.work()
    ops = {"rope": (op_ms[0], rb), "verify_attn": (op_ms[1], ab), "accept": (op_ms[2], cb)}
    dom = max(ops, key=lambda k: ops[k][0])
    if dom == "verify_attn" and run.config == "prefill":
        tfs = af / (op_ms[1] * 1e-3) / 1e12
        return {"kernel": dom, "bound": "tensor", "achieved": round(tfs, 1), "peak": tf_peak, "unit": "TFLOP/s",
                "frac": round(tfs / tf_peak, 4), "traffic": measured_traffic(dom, run.config), "peak_kind": peak_kind,
                "algorithmic_flops": af}
    ach = ops[dom][1] / (ops[dom][0] * 1e-3) / 1e9
    return {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(ach / hbm_peak, 4), "traffic": measured_traffic(dom, run.config), "peak_kind": peak_kind,
            "algorithmic_bytes": ops[dom][1]}


def op_records(run: ConfigRun, op_ms, world=1, floors=None):
    rb, ab, af, cb = run.work()
    x = run.x
    recs = {
        "verify_attn": {"us": round(op_ms[1] * 1e3, 2), "gbs": round(ab / (op_ms[1] * 1e-3) / 1e9, 1),
                        "tflops": round(af / (op_ms[1] * 1e-3) / 1e12, 2), "bytes": ab, "flops": af},
        "rope": {"us": round(op_ms[0] * 1e3, 2), "gbs": round(rb / (op_ms[0] * 1e-3) / 1e9, 1), "bytes": rb},
        "accept": None if x is None else {"us": round(op_ms[2] * 1e3, 2),
                                          "gbs": round(cb / (op_ms[2] * 1e-3) / 1e9, 1), "bytes": cb,
                                          "seq_per_s": round(world * x.batch / (op_ms[2] * 1e-3), 1),
                                          "mode": {W.MODE_ARGMAX: "argmax", W.MODE_GUMBEL: "gumbel",
                                                   W.MODE_REJECT: "reject"}[x.mode], "T": x.T},
    }
    # the same bytes read by a plain streaming reduction after the same flush
    for k, i in (("rope", 0), ("verify_attn", 1), ("accept", 2)):
        if floors and recs.get(k) is not None and k in floors:
            recs[k]["read_floor_us"] = round(floors[k] * 1e3, 2)
            recs[k]["x_floor"] = round(op_ms[i] / floors[k], 2)
    return recs


def sub_record(config, args, dev, stream, l2_flush, clocks, hbm_peak, tf_peak, peak_kind):
    """One more workload of the verification pass, measured like the headline
    (CUDA-graph replays, L2 flushed before every step) with its own roofline."""
    import torch
    run = ConfigRun(config, dev, with_commit=False)
    warm(run, stream, l2_flush, max(3, args.warmup))
    K = max(1, min(args.steps, 100))
    tm = Timer(dev, stream, K, l2_flush)
    graphs = {"step": tm.capture((run.op_step,)), "rope": tm.capture((run.op_rope,)),
              "verify_attn": tm.capture((run.op_attn,))}
    if run.acc is not None:
        graphs["accept"] = tm.capture((run.op_accept,))
    for g in graphs.values():
        g.replay()
    torch.cuda.synchronize()
    t0 = time.time()
    t_flush = tm.flush_ms()
    t_step = (tm.replay_ms(graphs["step"]) - t_flush) / K
    op_ms = np.array([(tm.replay_ms(graphs[k]) - t_flush) / K if k in graphs else 0.0
                      for k in ("rope", "verify_attn", "accept")])
    t1 = time.time()
    floors = floors_of(tm, dev, run)
    run.check_status()
    rb, ab, af, cb = run.work()
    a = run.a
    rec = {"workload": config, "batch": a.batch, "Hq": a.Hq, "Hkv": a.Hkv, "head_dim": a.d, "steps": K,
           "step_us": round(t_step * 1e3, 2), "step_gbs": round((rb + ab + cb) / (t_step * 1e-3) / 1e9, 1),
           **op_records(run, op_ms, floors=floors),
           "roofline": roofline_of(run, op_ms, hbm_peak, tf_peak, peak_kind),
           "clocks": clocks.window(t0, t1) if clocks is not None else None}
    del run, graphs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch
    import torch.distributed as dist

    from diffusion_speculative_verification_gb300 import build, ssv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    ssv.lib()

    run = ConfigRun(args.config, dev, with_commit=True)
    a, x = run.a, run.x
    stream = torch.cuda.current_stream(dev)
    # L2 flush between steps: a 256 MB read (twice the 129 MB L2) leaves only
    # clean lines of an unrelated buffer, so no step inherits its inputs in L2
    # and no write-back of dirty flush lines lands inside a measured step.
    flush_buf = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.zeros((), dtype=torch.float32, device=dev)

    def l2_flush():
        torch.sum(flush_buf, dim=0, out=flush_out)

    warm(run, stream, l2_flush, args.warmup)

    # Timed region.  Default: each sequence of K steps is captured once into a
    # CUDA graph and replayed as one launch, timed by two events around the
    # replay.  Graphs: K x [flush, ssv_verify_step] (the step: rotation,
    # attention and acceptance chained by programmatic dependent launch),
    # K x [flush], and K x [flush, op] per op (each op alone); step and op
    # times are the differences with the flush-only graph, divided by K.  No
    # event sits between the kernels, and host launch latency never leaves
    # the GPU idle inside a measurement.  --eager: the three calls one at a
    # time, with events between them.
    launch = "eager" if args.eager else "cuda_graph"
    tm = Timer(dev, stream, args.steps, l2_flush)
    graphs = None
    if launch == "cuda_graph":
        graphs = {"step": tm.capture((run.op_step,)), "rope": tm.capture((run.op_rope,)),
                  "verify_attn": tm.capture((run.op_attn,)), "commit": tm.capture((run.op_commit,))}
        if run.acc is not None:
            graphs["accept"] = tm.capture((run.op_accept,))
        if run.gargs is not None:
            run.op_accept_gen(stream)
            graphs["accept_gen"] = tm.capture((run.op_accept_gen,))
        torch.cuda.synchronize()
        for g in graphs.values():  # first replay uploads the graph
            g.replay()
        torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    clocks = ClockSampler(f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local))
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    if graphs is not None:
        t_step = tm.replay_ms(graphs["step"])
        torch.cuda.synchronize()
        t1 = time.time()
        t_flush = tm.flush_ms()
        op_ms = np.array([(tm.replay_ms(graphs[k]) - t_flush) / args.steps if k in graphs else 0.0
                          for k in ("rope", "verify_attn", "accept")])
        step_total = t_step - t_flush
        commit_ms = (tm.replay_ms(graphs["commit"]) - t_flush) / args.steps
        gen_ms = (tm.replay_ms(graphs["accept_gen"]) - t_flush) / args.steps if "accept_gen" in graphs else None
    else:
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for i in range(args.steps):
            l2_flush()
            run.step_eager(events[i], stream)
        torch.cuda.synchronize()
        t1 = time.time()
        per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in events])   # ms [steps, 3]
        op_ms = per.mean(axis=0)
        step_total = float(per.sum())
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
        for i in range(args.steps):
            l2_flush()
            ev[2 * i].record(stream)
            run.op_commit(stream)
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        commit_ms = float(np.mean([ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps)]))
        gen_ms = None
    if world > 1:
        dist.barrier()
    clk = clocks.window(t0, t1) if rank == 0 else None
    floors = floors_of(tm, dev, run) if graphs is not None else None
    run.check_status()
    tot_ms = aggregate_ms(float(step_total), dist if world > 1 else None, dev)

    rb, ab, af, cb = run.work()
    mb = commit_bytes(a, run.n_acc_c)
    step_bytes = rb + ab + cb
    ms_step = tot_ms / args.steps
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    hbm_peak, tf_peak, peak_kind = load_peaks()
    roof = roofline_of(run, op_ms, hbm_peak, tf_peak, peak_kind)

    lmh = None
    if args.config in W.LMHEAD and not args.no_lmhead:
        lmh = run_lmhead(args, dev, stream, l2_flush, hbm_peak, tf_peak)

    tree = None
    if not args.no_tree and rank == 0:
        tree = run_tree(args, dev, stream, l2_flush, hbm_peak)

    # ---- end to end: host inputs -> device, run, tokens back -------------------
    e2e = run_e2e(args, run, stream)

    subs = {}
    if rank == 0 or world > 1:
        for c in [c for c in args.sub_configs.split(",") if c and c != args.config]:
            subs[c] = sub_record(c, args, dev, stream, l2_flush, clocks if rank == 0 else None, hbm_peak, tf_peak,
                                 peak_kind)
    if rank == 0:
        clocks.stop()

    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": a.dtype, "data": "synthetic (seeded)",
            "config": {"workload": args.config, "batch": a.batch, "Hq": a.Hq, "Hkv": a.Hkv, "head_dim": a.d,
                       "l2": "256 MB read before every step", "launch": launch,
                       "parallelism": f"replicas x{world}"},
            **op_records(run, op_ms, world, floors),
            "commit": {"us": round(commit_ms * 1e3, 2), "gbs": round(mb / (commit_ms * 1e-3) / 1e9, 1),
                       "bytes": mb, "frac_hbm": round(mb / (commit_ms * 1e-3) / 1e9 / hbm_peak, 4),
                       "traffic": measured_traffic("commit", args.config),
                       "note": "timed alone, not in the step; accepted counts seeded uniform on 0..B"},
            "lmhead_accept": lmh,
            "tree_verification": tree,
            "accept_noise_generated": None if gen_ms is None else {
                "us": round(gen_ms * 1e3, 2), "table_us": round(op_ms[2] * 1e3, 2),
                "speedup_vs_table": round(op_ms[2] / gen_ms, 3),
                "gbs": round(accept_bytes(run.x) / 2 / (gen_ms * 1e-3) / 1e9, 1),
                "bytes": accept_bytes(run.x) / 2,
                "note": "same acceptance, coupled noise generated on the device (Philox4x32-10 + fixed fp32 "
                        "transform) instead of read from the table; bytes = logits rows only; timed alone"},
            "seq_per_s": round(world * a.batch / (ms_step * 1e-3), 1),
            "roofline": roof,
            "gpu_launches": kernel_launches(x) * args.steps,
            "clocks": clk,
            "e2e": e2e,
            "configs": subs,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(args.config)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_lmhead(args, dev, stream, l2_flush, hbm_peak, tf_peak):
    """The fused LM head + acceptance on the workload's verified slots (timed
    alone, after the same L2 flush), beside the unfused path it replaces
    (cuBLAS bf16 GEMM to bf16 logits, then ssv_accept)."""
    import ctypes as C
    import torch
    from diffusion_speculative_verification_gb300 import ssv, io as sio
    x = W.workload_lmhead(args.config)
    d = sio.lmhead_to_device(x, dev)
    a = x.acc
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = (torch.empty(len(a.blocks), dtype=torch.int32, device=dev),
            torch.empty(len(a.blocks), dtype=torch.int32, device=dev),
            torch.empty(len(a.tau), dtype=torch.int32, device=dev))
    largs = ssv.lmhead_args(d["mode"], d["T"], d["h"], d["w"], d["draft_tokens"], d["tau"], d["block"], d["gamma"],
                            d["slot_off"], *outs, d["noise"], d["noise_row"], status)
    ws = torch.zeros(max(256, ssv.lmhead_accept_workspace_bytes(largs)), dtype=torch.uint8, device=dev)
    L = ssv.lib()

    def fused():  # on the current stream (the capture stream while a graph is captured)
        r = L.ssv_lmhead_accept(C.byref(largs), ws.data_ptr(), ws.numel(), torch.cuda.current_stream(dev).cuda_stream)
        if r:
            raise ssv.SsvError(r, "ssv_lmhead_accept")

    logits = torch.empty((d["h"].shape[0], a.V), dtype=torch.bfloat16, device=dev)
    cargs = ssv.accept_args(d["mode"], d["T"], logits, d["draft_tokens"], d["tau"], d["block"], d["gamma"],
                            d["slot_off"], *outs, None, d["noise"], d["noise_row"], None, None, 64, status)
    ws_acc = torch.zeros(ssv.accept_workspace_bytes(cargs), dtype=torch.uint8, device=dev)

    def unfused():
        torch.mm(d["h"], d["w"].t(), out=logits)
        r = L.ssv_accept(C.byref(cargs), ws_acc.data_ptr(), ws_acc.numel(), torch.cuda.current_stream(dev).cuda_stream)
        if r:
            raise ssv.SsvError(r, "ssv_accept")

    K = min(args.steps, 50)

    def graph_of(fn):
        """K x [L2 flush, fn] captured once (fn may be None: the flush alone)."""
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            for _ in range(K):
                l2_flush()
                if fn is not None:
                    fn()
        stream.wait_stream(cap)
        return g

    def replay_ms(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    # each op runs inside a CUDA graph (as the step's ops do), minus a flush-only graph
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            l2_flush()
            fused()
        torch.cuda.synchronize()
        fused_tokens = [o.clone() for o in outs]
        for _ in range(max(3, args.warmup)):
            l2_flush()
            unfused()
        torch.cuda.synchronize()
        graphs = {"fused": graph_of(fused), "unfused": graph_of(unfused), "flush": graph_of(None)}
        for g in graphs.values():
            g.replay()
        torch.cuda.synchronize()
        t_flush = replay_ms(graphs["flush"])
        t_f = (replay_ms(graphs["fused"]) - t_flush) / K
        t_u = (replay_ms(graphs["unfused"]) - t_flush) / K
    assert ssv.get_status(status) == ssv.SSV_OK
    same = all(bool(torch.equal(u, v)) for u, v in zip(fused_tokens, outs))
    nbytes, flops, ver = lmhead_work(x)
    t_hbm = nbytes / (hbm_peak * 1e9) * 1e3
    t_tc = flops / (tf_peak * 1e12) * 1e3
    lb = max(t_hbm, t_tc)
    return {"us": round(t_f * 1e3, 1), "unfused_us": round(t_u * 1e3, 1),
            "unfused": "cuBLAS bf16 GEMM to bf16 logits, then ssv_accept", "same_outputs": same,
            "mode": {W.MODE_ARGMAX: "argmax", W.MODE_GUMBEL: "gumbel"}[a.mode], "T": a.T, "V": a.V,
            "hidden": x.hidden, "slots": int(np.sum(a.blocks)), "verified_rows": ver,
            "bound": "hbm" if t_hbm >= t_tc else "tensor", "lower_bound_us": round(lb * 1e3, 1),
            "frac": round(lb / t_f, 4), "tflops": round(flops / (t_f * 1e-3) / 1e12, 1),
            "gbs": round(nbytes / (t_f * 1e-3) / 1e9, 1), "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
            "traffic": measured_traffic("lmhead", args.config),
            "launch": "cuda_graph", "note": "timed alone, not in the step; logits never written"}


def tree_work(t: W.TreeInputs, out_bytes: int):
    """Useful work of the tree pass: (bytes, flops) of the attention -- KV cache
    once per kv head, Q, new K/V and the defined output rows; 4 d flops per
    (defined row, visible key, head) -- and the logits bytes the acceptance
    reads (every (node, position) row)."""
    import oracle.tree as otree  # counting only: the tree's per-node masks
    es = 2 if t.dtype == W.BF16 else 4
    flops = 0.0
    out_rows = 0
    for s in t.seqs:
        C, N, B, E, q_off, k_off, kv_off, e_off, o_off = (int(x) for x in s)
        committed, _ = otree.tree_nodes(B, t.parent[e_off:e_off + E], t.pos[e_off:e_off + E])
        defined = sum(B - bin(c).count("1") for c in committed)
        out_rows += N + defined
        flops += (N * (N + 1) / 2 + N * C + defined * (C + N + B)) * t.Hq * 4.0 * t.d
    nq = int(np.sum(t.seqs[:, 1] + t.seqs[:, 2]))
    nk = int(np.sum(t.seqs[:, 1] + t.seqs[:, 3] + t.seqs[:, 2]))
    nc = int(np.sum(t.seqs[:, 0]))
    bytes_ = (nc * 2 + nk * 2) * t.Hkv * t.d * es + nq * t.Hq * t.d * es + out_rows * t.Hq * t.d * out_bytes
    acc_bytes = float(t.total_out - int(np.sum(t.seqs[:, 1]))) * t.V * 4.0
    return float(bytes_), float(flops), acc_bytes


TREE_WORKLOAD = dict(cache=[4096] * 4, new=[0] * 4, blocks=[32] * 4, edges=[8] * 4, Hq=32, Hkv=8, d=128, seed=1006,
                     V=W.VOCAB)


def run_tree(args, dev, stream, l2_flush, hbm_peak):
    """Tree (state-set) verification on a SPOT-like shape: block width 32, a
    draft tree of 8 edges (budget D8), the 8B-class layer with a 4096-key
    prompt cache; the attention pass over every (node, position) row, then the
    acceptance by state equality over 151936-token logits (greedy).  Timed
    alone after the same L2 flush, as CUDA-graph replays."""
    import torch
    from diffusion_speculative_verification_gb300 import ssv, io as sio
    c = TREE_WORKLOAD
    t = W.make_tree_inputs("tree", c["cache"], c["new"], c["blocks"], c["edges"], c["Hq"], c["Hkv"], c["d"], W.BF16,
                           c["seed"], V=c["V"], mode=W.MODE_ARGMAX, T=0.0)
    d = sio.tree_to_device(t, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.zeros((t.total_out, t.Hq, t.d), dtype=torch.bfloat16, device=dev)
    aargs = ssv.tree_attn_args(d["q"], d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], o, d["seqs"], d["parent"],
                               d["pos"], t.total_out, d["max_cache"], 0.0, status)
    outs = [torch.empty(t.batch, dtype=torch.int32, device=dev), torch.empty((t.batch, 64), dtype=torch.int32, device=dev),
            torch.empty(t.batch, dtype=torch.int32, device=dev), torch.empty(t.batch, dtype=torch.int32, device=dev)]
    cargs = ssv.tree_accept_args(W.MODE_ARGMAX, 0.0, d["logits"], d["seqs"], d["parent"], d["pos"], d["token"], *outs,
                                 dev_status=status)
    import ctypes as C
    L = ssv.lib()
    n = C.c_size_t(0)
    L.ssv_tree_accept_workspace(C.byref(cargs), C.byref(n))
    ws = torch.zeros(max(256, int(n.value)), dtype=torch.uint8, device=dev)
    wsa = torch.zeros(max(256, ssv.tree_verify_attn_workspace_bytes(aargs)), dtype=torch.uint8, device=dev)

    def op_attn(s):
        r = L.ssv_tree_verify_attn(C.byref(aargs), wsa.data_ptr(), wsa.numel(), s.cuda_stream)
        if r:
            raise ssv.SsvError(r, "ssv_tree_verify_attn")

    def op_acc(s):
        r = L.ssv_tree_accept(C.byref(cargs), ws.data_ptr(), ws.numel(), s.cuda_stream)
        if r:
            raise ssv.SsvError(r, "ssv_tree_accept")

    for _ in range(3):
        l2_flush()
        op_attn(stream)
        op_acc(stream)
    torch.cuda.synchronize()
    assert ssv.get_status(status) == ssv.SSV_OK
    K = max(1, min(args.steps, 20))
    tm = Timer(dev, stream, K, l2_flush)
    ga, gc = tm.capture((op_attn,)), tm.capture((op_acc,))
    ga.replay(); gc.replay()
    torch.cuda.synchronize()
    t_flush = tm.flush_ms()
    t_a = (tm.replay_ms(ga) - t_flush) / K
    t_c = (tm.replay_ms(gc) - t_flush) / K
    assert ssv.get_status(status) == ssv.SSV_OK
    ab, af, cb = tree_work(t, 2)
    res = {"workload": "batch 4, 32 q / 8 kv heads, d 128, bf16, prompt cache 4096, block 32, 8-edge draft tree, "
                       "V 151936 greedy",
           "edges": c["edges"], "output_rows": t.total_out,
           "attn_us": round(t_a * 1e3, 2), "attn_gbs": round(ab / (t_a * 1e-3) / 1e9, 1),
           "attn_tflops": round(af / (t_a * 1e-3) / 1e12, 2), "attn_bytes": ab, "attn_flops": af,
           "attn_frac_hbm": round(ab / (t_a * 1e-3) / 1e9 / hbm_peak, 4),
           "accept_us": round(t_c * 1e3, 2), "accept_gbs": round(cb / (t_c * 1e-3) / 1e9, 1), "accept_bytes": cb,
           "accept_frac_hbm": round(cb / (t_c * 1e-3) / 1e9 / hbm_peak, 4),
           "n_acc": outs[0].cpu().tolist(), "launch": "cuda_graph", "note": "timed alone, not in the step"}
    del d, o, ws, ga, gc
    torch.cuda.empty_cache()
    return res


def run_e2e(args, run: ConfigRun, stream):
    """Same calls, inputs copied from pinned host memory every step, results read back."""
    import torch
    t, acc = run.t, run.acc
    names = ["q", "k_new", "v_new", "k_cache", "v_cache", "tau"]
    host = {k: t[k].cpu().pin_memory() for k in names}
    dev_bufs = {k: t[k] for k in names}
    host["seqs"] = t["batch"].dev.cpu().pin_memory()
    dev_bufs["seqs"] = t["batch"].dev
    if acc is not None:
        for k in ("logits", "draft_tokens", "tau", "block", "gamma", "slot_off", "noise_row", "u_accept", "u_sample",
                  "draft_logits", "noise"):
            if acc[k] is not None:
                host["acc_" + k] = acc[k].cpu().pin_memory()
                dev_bufs["acc_" + k] = acc[k]
        results = list(run.outs)
    else:
        results = [run.o]
    results_host = [torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in results]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in results_host)
    steps = max(1, min(args.steps, 50))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(steps + 2):
        if i == 2:
            torch.cuda.synchronize()
            e0.record(stream)
        for k, h in host.items():
            dev_bufs[k].copy_(h, non_blocking=True)
        run.op_step(stream)
        for r, rh in zip(results, results_host):
            rh.copy_(r, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    run.check_status()
    ms = e0.elapsed_time(e1) / steps
    rb, ab, af, cb = run.work()
    del host, results_host
    return {"value": round((rb + ab + cb) / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 4), "steps": steps}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=list(W.WORKLOADS), default="sweep",
                    help="headline workload (default: sweep, the largest by bytes)")
    ap.add_argument("--sub-configs", default="prefill,gqa8b,gqa1p7b",
                    help="comma-separated workloads measured after the headline, each as a sub-record "
                         "with its own roofline ('' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-lmhead", action="store_true", help="skip the fused LM head + acceptance measurement")
    ap.add_argument("--no-tree", action="store_true", help="skip the tree verification measurement")
    ap.add_argument("--eager", action="store_true", help="launch the timed steps one call at a time")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
