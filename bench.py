"""Benchmark of one paged decode step (KV append + paged decode attention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pkv|reference]
    python bench.py --op copy_blocks [--pairs P] [--workload NAME]   # copy-on-write copy alone

Prints ONE JSON line (rank 0). A step is the whole hot path over one batch:
``kv_append`` of the step's new tokens, then ``paged_decode_attention`` (main
kernel + merge kernel). Inputs are seeded synthetic data resident in HBM. The
headline is the largest workload, ``long_splitk`` (8 sequences of 32k-131k
tokens, 2.97 GB a step); the same line carries ``per_config``: every named
workload's step (us per step, main-kernel us, GB/s, roofline fractions, ncu
traffic where pinned, the oracle's CPU baseline). A step that reads at least 2x
the L2 capacity evicts its own inputs (the K/V streams carry an evict-first hint;
with cache control off, ncu sees the main kernel read 1.00x its algorithmic bytes
from DRAM between unflushed steps at 2.3x to 23x the L2), so nothing is flushed
between its timed steps (``--l2 auto``; the headline also carries the same steps
timed after a 512 MiB memset, ``with_write_flush``); smaller steps are separated
by that memset, untimed. ``value`` is the step's algorithmic bytes (Q + K + V +
block tables + context lengths read, output written, plus the append's rows) per
second of step time, in GB/s; shared-prefix blocks count once.

``--impl reference`` times the fp64 CPU oracle on the host cores instead (the
only reference this method has), on a bounded sample of the same workload.
Under torchrun every rank runs its own copy of the workload (independent
sequences: weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import copy
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402
from paged_kv_cache_101_gb300 import roofline as R  # noqa: E402

METRIC = "paged decode-attention KV-read GB/s vs ~8 TB/s HBM peak; µs per decode step"
DEFAULT_WORKLOAD = "long_splitk"
FLUSH_BYTES = 512 << 20
L2_BYTES = 129 * 10**6  # GB300 L2 capacity
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic (read + write bytes per launch) of the main attention kernel from
# one ncu capture, keyed by workload; valid only while the kernel source hashes
# to `source_sha256` (otherwise the bench reports traffic = null).
NCU_TRAFFIC = {
    "llama3_8b_decode": {
        "bytes": 580901376 + 2423808,  # dram__bytes_read.sum + dram__bytes_write.sum
        "source_sha256": "4efd1c10e0e0af91e272fe6ce26ab7f2b292e5c09dab6cebe31b3c12d97ebbca",
    },
    "llama3_70b_mix": {
        "bytes": 1344542976 + 442624,  # dram__bytes_read.sum + dram__bytes_write.sum
        "source_sha256": "4efd1c10e0e0af91e272fe6ce26ab7f2b292e5c09dab6cebe31b3c12d97ebbca",
    },
    "long_splitk": {
        "bytes": 2968272896 + 4363776,  # dram__bytes_read.sum + dram__bytes_write.sum
        "source_sha256": "4efd1c10e0e0af91e272fe6ce26ab7f2b292e5c09dab6cebe31b3c12d97ebbca",
    },
    "spec_verify": {
        "bytes": 1406908928 + 6244352,  # dram__bytes_read.sum + dram__bytes_write.sum
        "source_sha256": "4efd1c10e0e0af91e272fe6ce26ab7f2b292e5c09dab6cebe31b3c12d97ebbca",
    },
    "llama3_8b_decode/fp8": {
        "bytes": 290347008 + 989696,  # dram__bytes_read.sum + dram__bytes_write.sum
        "source_sha256": "4efd1c10e0e0af91e272fe6ce26ab7f2b292e5c09dab6cebe31b3c12d97ebbca",
    },
    "llama3_70b_mix/fp8": {
        "bytes": 663453440 + 2262528,  # dram__bytes_read.sum + dram__bytes_write.sum
        "source_sha256": "4efd1c10e0e0af91e272fe6ce26ab7f2b292e5c09dab6cebe31b3c12d97ebbca",
    },
    "spec_verify/umma": {
        "bytes": 1442352896 + 20516864,  # dram__bytes_read.sum + dram__bytes_write.sum
        "source_sha256": "4efd1c10e0e0af91e272fe6ce26ab7f2b292e5c09dab6cebe31b3c12d97ebbca",
    },
}


def max_over_ranks(values, dist, device):
    """Each timing's maximum over all ranks (the slowest replica sets the job's
    time); the values unchanged on one rank."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_gbs(world, bytes_per_replica_step, ms_per_step):
    """Whole-job throughput: every replica moves its step's bytes in the (max over
    ranks) step time."""
    return world * bytes_per_replica_step / (ms_per_step * 1e-3) / 1e9


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in ("paged_decode.cu", "paged_decode_umma.cu", "pkv_cells.cuh", "pkv_common.cuh",
              "pkv_internal.h", "pkv_umma.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_101_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # raw samples (the JSON line carries their summary); PKV_CLOCK_LOG overrides
        self.path = os.environ.get("PKV_CLOCK_LOG") or os.path.join(
            tempfile.gettempdir(), f"pkv_clocks_gpu{gpu_index}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ pkv arm
NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s the benchmark quotes as the HBM peak


class StepRig:
    """One workload's decode step on the device: pools, inputs, workspace and the
    step (append + attention) as a user calls it, with the L2 rule between steps."""

    def __init__(self, w, args, dev, fp8=False, cascade=False):
        import torch

        import paged_kv_cache_101_gb300 as pkv
        self.torch, self.pkv, self.dev, self.args = torch, pkv, dev, args
        self.fp8, self.cascade = fp8, cascade
        self.two_calls = bool(getattr(args, "two_calls", False))
        if cascade:
            w = W.sharers_first(w)  # the sharing sequences form one consecutive group
        self.w = w

        def up(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
                torch.bfloat16)

        self.q = up(w.q)
        self.k_scale = self.v_scale = None
        if fp8:
            k8, v8, ks_h, vs_h = W.fp8_pools(w)
            self.k_cache = torch.from_numpy(k8).to(dev)
            self.v_cache = torch.from_numpy(v8).to(dev)
            self.k_scale = torch.from_numpy(ks_h).to(dev)
            self.v_scale = torch.from_numpy(vs_h).to(dev)
            del k8, v8
        else:
            self.k_cache, self.v_cache = up(w.k_cache), up(w.v_cache)
        self.k_new, self.v_new = up(w.k_new), up(w.v_new)
        self.slots = torch.from_numpy(w.slot_mapping).to(dev)
        self.tables = torch.from_numpy(w.block_tables).to(dev)
        self.lens = torch.from_numpy(w.context_lens).to(dev)
        self.out = torch.empty(self.q.shape, dtype=torch.bfloat16, device=dev)
        self.M = int(w.shared.sum()) if cascade else 0
        if cascade:
            self.groups = torch.tensor([[0, self.M, w.meta["prefix_tokens"] // 16]],
                                       dtype=torch.int32, device=dev)
            self.ws = pkv.workspace(dev, int(pkv.lib().pkv_workspace_size_cascade(
                w.num_seqs, w.n_query_per_seq, w.num_q_heads, w.num_kv_heads, w.head_dim)))
        else:
            self.ws = pkv.workspace(dev, pkv.workspace_size(
                w.num_seqs, w.n_query_per_seq, w.num_q_heads, w.num_kv_heads, w.head_dim))
        self.flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        eb = 1 if fp8 else 2
        self.attn_bytes = R.workload_bytes(w, unique=True, kv_bytes_per_element=eb)
        self.attn_bytes_logical = R.workload_bytes(w, unique=False, kv_bytes_per_element=eb)
        self.app_bytes = R.append_bytes(int(w.slot_mapping.size), w.num_kv_heads, w.head_dim,
                                        kv_bytes_per_element=eb)
        self.step_bytes = self.attn_bytes + self.app_bytes
        # Between timed steps: a step that reads at least twice the L2 capacity evicts
        # its own inputs, so nothing is flushed (no dirty flush data is written back
        # during the timed kernels); smaller steps are separated by the 512 MiB memset.
        self.l2_mode = args.l2 if args.l2 != "auto" else (
            "none" if self.step_bytes >= 2 * L2_BYTES else "flush")

    def flush(self):
        if self.l2_mode == "flush":
            self.flush_buf.zero_()

    def attend(self, q, tables, lens, out):
        pkv, w = self.pkv, self.w
        if self.fp8:
            pkv.paged_decode_attention_fp8(q, self.k_cache, self.v_cache, self.k_scale,
                                           self.v_scale, tables, lens, w.n_query_per_seq,
                                           w.scale, out, ws=self.ws)
        elif self.cascade:
            pkv.paged_decode_attention_cascade(q, self.k_cache, self.v_cache, tables, lens,
                                               w.n_query_per_seq, w.scale, out, self.groups,
                                               self.M, ws=self.ws)
        else:
            pkv.paged_decode_attention(q, self.k_cache, self.v_cache, tables, lens,
                                       w.n_query_per_seq, w.scale, out, ws=self.ws)

    def append(self, k_new, v_new, slots):
        if self.fp8:
            self.pkv.kv_append_fp8(k_new, v_new, slots, self.k_cache, self.v_cache,
                                   self.k_scale, self.v_scale)
        else:
            self.pkv.kv_append(k_new, v_new, slots, self.k_cache, self.v_cache)

    def step(self):
        if self.cascade or self.two_calls:
            self.append(self.k_new, self.v_new, self.slots)
            self.attend(self.q, self.tables, self.lens, self.out)
            return
        # one call: append, then attention (its prologue overlaps the append)
        w = self.w
        self.pkv.decode_step(self.q, self.k_new, self.v_new, self.slots, self.k_cache,
                             self.v_cache, self.tables, self.lens, w.n_query_per_seq, w.scale,
                             self.out, ws=self.ws,
                             k_scale=self.k_scale if self.fp8 else None,
                             v_scale=self.v_scale if self.fp8 else None)

    def time_steps(self, K, warmup):
        """(ms per step, main-kernel ms, append ms, attention-call ms) over K steps
        after `warmup` untimed ones.

        The timed steps run as a user runs them. Unflushed steps are timed as one
        block (an event pair around every step would add ~2 us of GPU time to each);
        flushed ones one by one, the flush outside. The main kernel's own time comes
        from a separate pass in which the library records events around it: an event
        between the append and the main kernel, or between it and the merge, keeps
        the next kernel from launching early (programmatic dependent launch), so it
        would stretch the steps it sits in. The append and the attention call
        (main kernel + merge) are timed per call in a third pass, with events
        around each; the event between them keeps the attention call from
        overlapping the append, so the two add up to a little more than a step."""
        torch, pkv = self.torch, self.pkv
        for _ in range(warmup):
            self.flush()
            self.step()
        torch.cuda.synchronize()
        ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        hook = 4
        ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(0, K, hook)]
        for a, b in ev_k:
            a.record()  # create the underlying events before the timed region
            b.record()
        torch.cuda.synchronize()
        if self.l2_mode == "none":
            ev_s[0].record()
            for _ in range(K):
                self.step()
            ev_e[0].record()
        else:
            for i in range(K):
                self.flush()
                ev_s[i].record()
                self.step()
                ev_e[i].record()
        for a, b in ev_k:
            self.flush()
            pkv.set_profiling_events(a, b)
            self.step()
            pkv.set_profiling_events(None, None)
        ev_c = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
                for _ in range(0, K, hook)]
        for e0, e1, e2 in ev_c:
            self.flush()
            e0.record()
            self.append(self.k_new, self.v_new, self.slots)
            e1.record()
            self.attend(self.q, self.tables, self.lens, self.out)
            e2.record()
        torch.cuda.synchronize()
        if self.l2_mode == "none":
            ms = ev_s[0].elapsed_time(ev_e[0]) / K
        else:
            ms = sum(a.elapsed_time(b) for a, b in zip(ev_s, ev_e)) / K
        kern = [a.elapsed_time(b) for a, b in ev_k]
        app = [e0.elapsed_time(e1) for e0, e1, _ in ev_c]
        att = [e1.elapsed_time(e2) for _, e1, e2 in ev_c]
        return ms, sum(kern) / len(kern), sum(app) / len(app), sum(att) / len(att)

    def write_flush(self, K):
        """The same steps, each after the 512 MiB memset: (ms per step, kernel ms)."""
        torch, pkv = self.torch, self.pkv
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        for i in range(K):
            self.flush_buf.zero_()
            ev[i][0].record()
            self.step()
            ev[i][1].record()
        for i in range(0, K, 4):
            self.flush_buf.zero_()
            pkv.set_profiling_events(ev[i][2], ev[i][3])
            self.step()
            pkv.set_profiling_events(None, None)
        torch.cuda.synchronize()
        f_step = sum(e[0].elapsed_time(e[1]) for e in ev) / K
        f_kern = [ev[i][2].elapsed_time(ev[i][3]) for i in range(0, K, 4)]
        return f_step, sum(f_kern) / len(f_kern)


def traffic_pin(key):
    nt = NCU_TRAFFIC.get(key)
    if nt and nt.get("source_sha256") == kernel_source_sha():
        return nt["bytes"]
    return None


def roofline_entry(rig, kern_ms, traffic, kernel_name):
    peak, peak_kind = measured_peaks()
    achieved = rig.attn_bytes / (kern_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1),
            "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_kind} hbm_gbs (burst)",
            "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": traffic, "kernel_us": round(kern_ms * 1e3, 3),
            "algorithmic_bytes_per_launch": rig.attn_bytes}


def use_cascade(w, mode):
    """The cascade for a workload with prefix sharers: forced on or off, or as the
    library's rule decides for its batch (sharers first, one group)."""
    import paged_kv_cache_101_gb300 as pkv
    if not w.shared.any() or mode == "off":
        return False
    if mode == "on":
        return True
    lens = np.concatenate([w.context_lens[w.shared], w.context_lens[~w.shared]])
    return pkv.cascade_pays(lens, [[0, int(w.shared.sum()), w.meta["prefix_tokens"] // 16]],
                            w.num_kv_heads, w.head_dim)


def run_pkv(args, rank, world, dist):
    import torch

    import paged_kv_cache_101_gb300 as pkv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    fp8 = args.kv_dtype == "fp8"
    fma = args.math == "fma"
    w0 = W.make_workload(args.workload)
    cascade = use_cascade(w0, args.cascade)
    if fma and (fp8 or cascade):
        raise SystemExit("--math fma runs the plain bf16 call only")
    pkv.set_option(pkv.PKV_OPT_MATH, 1 if fma else 0)
    pkv.set_option(pkv.PKV_OPT_PACE, 1 if args.pace else 0)
    pkv.set_option(pkv.PKV_OPT_HEADS_PER_CTA, args.heads)
    pkv.set_option(pkv.PKV_OPT_TMA_BOX, args.box)
    pkv.set_option(pkv.PKV_OPT_UMMA, 1 if args.umma else 0)
    pkv.set_option(pkv.PKV_OPT_PREFETCH, args.prefetch)
    rig = StepRig(w0, args, dev, fp8=fp8, cascade=cascade)
    del w0
    w = rig.w
    K = args.steps

    clocks = ClockSampler(dev.index)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ms_per_step, kern_mean, append_ms, attn_ms = rig.time_steps(K, args.warmup)
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()

    # the same steps again, each after the 512 MiB memset, for comparison
    write_flush = None
    if rig.l2_mode == "none":
        Kf = min(K, 300)
        f_step, f_kern = max_over_ranks(list(rig.write_flush(Kf)), dist, dev)
        write_flush = {"us_per_step": round(f_step * 1e3, 3), "kernel_us": round(f_kern * 1e3, 3),
                       "steps": Kf,
                       "note": "each step after a 512 MiB memset: its dirty lines are written "
                               "back during the timed kernels"}
    err = pkv.workspace_error(rig.ws)
    e2e_ms, e2e_mode, h2d, d2h = run_e2e(rig, args, dev)

    # max over ranks
    ms_per_step, kern_mean, e2e_ms, append_ms, attn_ms = max_over_ranks(
        [ms_per_step, kern_mean, e2e_ms, append_ms, attn_ms], dist, dev)
    # the tcgen05 kernel runs when it is opted in and the batch has 17-64 score rows per
    # kv head on bf16 pools of head_dim 128 (the library's own rule)
    umma = bool(args.umma) and not (fp8 or fma or cascade) and w.head_dim == 128 and \
        16 < w.n_query_per_seq * (w.num_q_heads // w.num_kv_heads) <= 64
    traffic = traffic_pin(args.workload + ("/fp8" if fp8 else "") +
                          ("/cascade" if cascade else "") + ("/fma" if fma else "") +
                          ("/umma" if umma else ""))
    step_bytes = rig.step_bytes
    value = job_gbs(world, step_bytes, ms_per_step)
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "us_per_step": round(ms_per_step * 1e3, 3),
        "append_us": round(append_ms * 1e3, 3),
        "attention_us": round(attn_ms * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (E4M3 KV cache, f16 products)" if fp8 else "bf16",
        "data": ("synthetic (seeded random E4M3 code pools with per-head scales, N(0,1) bf16 "
                 "Q and new rows; " if fp8 else "synthetic (seeded N(0,1) bf16 K/V/Q; ") +
                "pools in HBM; " + ("inputs several times the L2, no flush)"
                                    if rig.l2_mode == "none"
                                    else "a 512 MiB L2 flush between timed steps)"),
        "config": {
            "workload": args.workload + (" (fp8 KV cache)" if fp8 else "") +
                        (" (shared-prefix cascade)" if cascade else "") +
                        (" (CUDA-core FMA consumers)" if fma else ""),
            "kv_dtype": args.kv_dtype, "math": args.math, "pace": bool(args.pace),
            "num_seqs": w.num_seqs, "n_query_per_seq": w.n_query_per_seq,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": 16,
            "context_tokens": int(w.context_lens.sum()),
            "num_blocks": w.num_blocks, "parallelism": f"replicas x{world}",
            "l2": l2_note(rig),
            "step": ("kv_append + paged_decode_attention_cascade" if cascade else
                     "pkv_decode_step: kv_append" + ("_fp8" if fp8 else "") +
                     " + paged_decode_attention" + ("_fp8" if fp8 else "")) +
                    " (append, main + merge kernels)",
            "bytes_per_step": step_bytes, "attention_bytes_unique": rig.attn_bytes,
            "attention_bytes_logical": rig.attn_bytes_logical,
        },
        "roofline": roofline_entry(
            rig, kern_mean, traffic,
            ("paged_decode_fma_kernel" if fma else "paged_decode_umma_kernel" if umma
             else "paged_decode_kernel") +
            (" (prefix pass + main pass)" if cascade else "")),
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 6), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "path": ("pkv_decode_step_host_pipelined: " if rig.l2_mode == "none" and
                         not cascade else "pkv_decode_step_host: " if not (fp8 or cascade)
                         else "") +
                        "one pinned host arena (q, new K/V, slots, tables, lengths) -> one H2D -> "
                        "kv_append + attention -> one D2H of the output",
                "mode": e2e_mode},
        "gpu_launches": K * (4 if cascade else 3),
        "device_error_word": err,
    }
    if write_flush is not None:
        res["with_write_flush"] = write_flush
    if clk is not None:
        res["clocks"] = clk
    del rig
    torch.cuda.empty_cache()
    return res


def l2_note(rig):
    if rig.l2_mode == "none":
        return ("not flushed: each step reads %.0f MB, %.1fx the %d MB L2, so it evicts its own "
                "inputs" % (rig.step_bytes / 1e6, rig.step_bytes / L2_BYTES, L2_BYTES // 10**6))
    return "flushed between timed steps (512 MiB memset, untimed)"


def run_e2e(rig, args, dev):
    """End to end: per-step inputs from pinned host memory, output back to host.

    The step's inputs (q, new K/V rows, slots, block tables, lengths) sit in one
    pinned host arena and cross in ONE host-to-device copy into a device arena of
    the same layout; the library calls then run on views of that arena, and the
    output comes back in one device-to-host copy. The plain bf16 step goes through
    the library's host-buffer entry point (pkv_decode_step_host: both copies inside
    the C-ABI call, its arena layout); the E4M3 and cascade steps use the same
    layout with the copies made here. Returns (ms per step, mode, H2D, D2H bytes)."""
    import torch
    pkv, w = rig.pkv, rig.w
    fp8, cascade = rig.fp8, rig.cascade
    K = args.steps
    ins = [("q", rig.q), ("k_new", rig.k_new), ("v_new", rig.v_new),
           ("slot_mapping", rig.slots), ("block_tables", rig.tables),
           ("context_lens", rig.lens)]
    arena_bytes, offs = pkv.step_arena_layout(w.num_seqs, w.n_query_per_seq, w.num_q_heads,
                                              w.num_kv_heads, w.head_dim,
                                              w.block_tables.shape[1])
    h_arena = torch.empty(arena_bytes, dtype=torch.uint8).pin_memory()
    d_arena = torch.empty(arena_bytes, dtype=torch.uint8, device=dev)

    def view(buf, nm, t):
        n = t.numel() * t.element_size()
        return buf[offs[nm]:offs[nm] + n].view(t.dtype).view(t.shape)

    for nm, t in ins:
        view(h_arena, nm, t).copy_(t)
    out = rig.out
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = arena_bytes
    d2h = h_out.numel() * h_out.element_size()
    e_q, e_kn, e_vn, e_slots, e_tables, e_lens = (view(d_arena, nm, t) for nm, t in ins)

    def e2e_step():
        if not fp8 and not cascade:
            pkv.decode_step_host(h_arena, d_arena, rig.k_cache, rig.v_cache, w.num_seqs,
                                 w.n_query_per_seq, w.num_q_heads, w.block_tables.shape[1],
                                 w.scale, out, h_out, ws=rig.ws)
            return
        d_arena.copy_(h_arena, non_blocking=True)
        rig.append(e_kn, e_vn, e_slots)
        rig.attend(e_q, e_tables, e_lens, out)
        h_out.copy_(out, non_blocking=True)

    Ke = max(1, min(K, 200))
    if rig.l2_mode == "none":
        # Steps in flight two at a time: the upload, compute and download phases on
        # their own streams, two buffer slots (device arena, device output) used in
        # turn, ordered by each slot's events: a step's copies overlap its
        # neighbours' kernels, the kernels stay in order on the compute stream.
        # The timed region runs from before the first upload to after the last
        # download, so every step's copies are inside it.
        streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        slots_ev = [tuple(torch.cuda.Event() for _ in range(3)) for _ in range(2)]
        d_arenas = [d_arena, torch.empty(arena_bytes, dtype=torch.uint8, device=dev)]
        outs = [out, torch.empty_like(out)]
        h_outs = [h_out, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
        views = [tuple(view(da, nm, t) for nm, t in ins) for da in d_arenas]

        def piped_step(i):
            b = i % 2
            up, comp, down = streams
            ev_up, ev_comp, ev_down = slots_ev[b]
            if not cascade:
                pkv.decode_step_host(h_arena, d_arenas[b], rig.k_cache, rig.v_cache, w.num_seqs,
                                     w.n_query_per_seq, w.num_q_heads, w.block_tables.shape[1],
                                     w.scale, outs[b], h_outs[b], ws=rig.ws, streams=streams,
                                     events=slots_ev[b], k_scale=rig.k_scale,
                                     v_scale=rig.v_scale)
                return
            p_q, p_kn, p_vn, p_slots, p_tables, p_lens = views[b]
            up.wait_event(ev_comp)
            with torch.cuda.stream(up):
                d_arenas[b].copy_(h_arena, non_blocking=True)
                ev_up.record(up)
            comp.wait_event(ev_up)
            comp.wait_event(ev_down)
            with torch.cuda.stream(comp):
                rig.append(p_kn, p_vn, p_slots)
                rig.attend(p_q, p_tables, p_lens, outs[b])
                ev_comp.record(comp)
            down.wait_event(ev_comp)
            with torch.cuda.stream(down):
                h_outs[b].copy_(outs[b], non_blocking=True)
                ev_down.record(down)

        main = torch.cuda.current_stream(dev)
        for i in range(max(1, args.warmup)):
            piped_step(i)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(main)
        for st_ in streams:
            st_.wait_stream(main)
        for i in range(Ke):
            piped_step(i)
        for st_ in streams:
            main.wait_stream(st_)
        t1.record(main)
        torch.cuda.synchronize()
        return (t0.elapsed_time(t1) / Ke,
                "pipelined: two steps in flight, copies overlapping kernels", h2d, d2h)
    for _ in range(max(1, args.warmup)):
        rig.flush()
        e2e_step()
    torch.cuda.synchronize()
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    for i in range(Ke):
        rig.flush()
        e_s[i].record()
        e2e_step()
        e_e[i].record()
    torch.cuda.synchronize()
    return (sum(a.elapsed_time(b) for a, b in zip(e_s, e_e)) / Ke,
            "serial: one step at a time (L2 flushed between steps)", h2d, d2h)


def run_per_config(args, rank, world, dist, headline):
    """Every named workload's decode step (bf16 pools, plain call): us per step,
    main-kernel us, append and attention-call us, step and kernel GB/s, its
    `roofline` object (fractions, ncu traffic where pinned), and the oracle timed on
    a bounded sample on the host cores."""
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    entries = {}
    for name in W.WORKLOAD_ORDER:
        if name == args.workload and headline is not None:
            res = headline
            e = {"us_per_step": res["us_per_step"], "kernel_us": res["roofline"]["kernel_us"],
                 "append_us": res["append_us"], "attention_us": res["attention_us"],
                 "step_gbs": res["value"], "kernel_gbs": res["roofline"]["achieved"],
                 "frac": res["roofline"]["frac"],
                 "frac_of_8tbs": res["roofline"]["frac_of_8tbs"],
                 "traffic": res["roofline"]["traffic"],
                 "bytes_per_step": res["config"]["bytes_per_step"],
                 "attention_bytes_unique": res["config"]["attention_bytes_unique"],
                 "attention_bytes_logical": res["config"]["attention_bytes_logical"],
                 "l2": res["config"]["l2"], "steps": res["steps"],
                 "roofline": res["roofline"]}
            if "cpu_baseline" in res:
                e["cpu_baseline"] = res["cpu_baseline"]
            entries[name] = e
            continue
        rig = StepRig(W.make_workload(name), args, dev)
        ms, kern, app, att = rig.time_steps(args.steps, args.warmup)
        ms, kern, app, att = max_over_ranks([ms, kern, app, att], dist, dev)
        rf = roofline_entry(rig, kern, traffic_pin(name), "paged_decode_kernel")
        e = {"us_per_step": round(ms * 1e3, 3), "kernel_us": rf["kernel_us"],
             "append_us": round(app * 1e3, 3), "attention_us": round(att * 1e3, 3),
             "step_gbs": round(job_gbs(world, rig.step_bytes, ms), 2),
             "kernel_gbs": rf["achieved"], "frac": rf["frac"],
             "frac_of_8tbs": rf["frac_of_8tbs"], "traffic": rf["traffic"],
             "bytes_per_step": rig.step_bytes, "attention_bytes_unique": rig.attn_bytes,
             "attention_bytes_logical": rig.attn_bytes_logical, "l2": l2_note(rig),
             "steps": args.steps, "device_error_word": rig.pkv.workspace_error(rig.ws),
             "roofline": rf}
        del rig
        torch.cuda.empty_cache()
        if rank == 0 and not args.no_cpu_baseline:
            a = argparse.Namespace(**vars(args))
            a.workload = name
            a.cpu_seconds = args.cpu_seconds / 2
            e["cpu_baseline"] = cpu_baseline(a)
        entries[name] = e
    return entries


# ------------------------------------------------------------------ copy-on-write copy
COPY_METRIC = "copy-on-write block copy GB/s (bytes read + written)"


def run_copy(args, rank, world, dist):
    """Time pkv_copy_blocks alone: `--pairs` block pairs of the workload's geometry
    (16 tokens x Hkv x D bf16 in K and V per block), disjoint sources and
    destinations drawn by a seeded permutation of a pool twice that size."""
    import torch

    import oracle as O
    import paged_kv_cache_101_gb300 as pkv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    geo = W.WORKLOADS[args.workload]
    Hkv, D = geo["Hkv"], geo["D"]
    P = int(args.pairs)
    NB = 2 * P + 64
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    k_cache = torch.randint(-(1 << 15), 1 << 15, (NB, 16, Hkv, D), dtype=torch.int16, device=dev,
                            generator=g).view(torch.bfloat16)
    v_cache = torch.randint(-(1 << 15), 1 << 15, (NB, 16, Hkv, D), dtype=torch.int16, device=dev,
                            generator=g).view(torch.bfloat16)
    perm = np.random.default_rng(1234).permutation(NB).astype(np.int32)
    src = torch.from_numpy(perm[:P].copy()).to(dev)
    dst = torch.from_numpy(perm[P:2 * P].copy()).to(dev)
    block_bytes = 2 * 16 * Hkv * D * 2            # K + V of one block
    step_bytes = 2 * P * block_bytes              # read and written
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        flush.zero_()
        pkv.copy_blocks(k_cache, v_cache, src, dst)
    torch.cuda.synchronize()
    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        ev_s[i].record()
        pkv.copy_blocks(k_cache, v_cache, src, dst)
        ev_e[i].record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in zip(ev_s, ev_e)) / K

    # end to end: the pairs come from pinned host memory each step (as a block
    # manager hands them out), the pool stays on the device; 4 bytes read back
    h_src = src.cpu().pin_memory()
    h_dst = dst.cpu().pin_memory()
    h_probe = torch.empty(2, dtype=torch.int16).pin_memory()
    Ke = max(1, min(K, 200))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    for i in range(Ke):
        flush.zero_()
        e_s[i].record()
        src.copy_(h_src, non_blocking=True)
        dst.copy_(h_dst, non_blocking=True)
        pkv.copy_blocks(k_cache, v_cache, src, dst)
        h_probe.copy_(k_cache.view(torch.int16)[int(perm[P]), 0, 0, :2], non_blocking=True)
        e_e[i].record()
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in zip(e_s, e_e)) / Ke
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dist, dev)

    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9
    res = {
        "metric": COPY_METRIC, "value": round(world * achieved, 2), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "us_per_step": round(ms * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (bit copy)",
        "data": "synthetic (seeded random bf16 bit patterns; 512 MiB L2 flush between steps)",
        "config": {"workload": f"copy_blocks {P} pairs, {args.workload} geometry",
                   "num_kv_heads": Hkv, "head_dim": D, "pairs": P, "num_blocks": NB,
                   "bytes_per_step": step_bytes, "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "copy_blocks_kernel",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs (burst)", "traffic": None,
                     "kernel_us": round(ms * 1e3, 3), "algorithmic_bytes_per_launch": step_bytes},
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 6), "h2d_bytes_per_step": 8 * P,
                "d2h_bytes_per_step": 4,
                "path": "pinned host pairs -> H2D -> copy_blocks -> D2H probe"},
        "gpu_launches": K,
    }
    if clk is not None:
        res["clocks"] = clk
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle's block copy on a bounded sample of the pairs
        o = O.Oracle()
        sp = min(P, 512)
        kh = np.zeros((2 * sp + 64, 16, Hkv, D), dtype=np.uint16)
        vh = kh.copy()
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < args.cpu_seconds / 5 or n == 0:
            kh, vh = o.copy_blocks(kh, vh, np.arange(sp), np.arange(sp, 2 * sp))
            n += 1
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(n * 2 * sp * block_bytes / el / 1e9, 4),
                               "unit": "GB/s", "cores": 1, "kind": "oracle",
                               "sample": f"{n} copies of {sp} pairs in {el:.1f} s (one thread; "
                                         f"each call also copies the pools once)"}
    return res


# ------------------------------------------------------------------ tree verification
TREE_METRIC = "tree-verify attention GB/s (unique KV bytes); µs per step"


def binary_tree_masks(levels: int):
    """Ancestor-or-self bits of a complete binary tree, nodes in level order."""
    masks = []
    for node in range(2 ** levels - 1):
        m, a = 0, node
        while True:
            m |= 1 << a
            if a == 0:
                break
            a = (a - 1) // 2
        masks.append(m)
    return np.array(masks, dtype=np.uint32)


def run_tree(args, rank, world, dist):
    """Speculative tree verification on a workload's sequences: every sequence
    appends a 15-node binary candidate tree (4 levels, branching 2) and scores all
    nodes in one call; nodes see the cached context and their own ancestors.
    The 15 rows of a sequence go out as runs of at most 64 / G queries."""
    import torch

    import paged_kv_cache_101_gb300 as pkv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pkv.set_option(pkv.PKV_OPT_UMMA, 1 if args.umma else 0)
    pkv.set_option(pkv.PKV_OPT_PREFETCH, args.prefetch)
    # the 8B layer's lengths and heads unless a workload is named
    name = args.workload if args.workload_given else "llama3_8b_decode"
    base_lens = W.workload_lengths(name)[0]
    geo = W.WORKLOADS[name]
    Hq, Hkv, D = geo["Hq"], geo["Hkv"], geo["D"]
    masks = binary_tree_masks(4)
    n = masks.size
    ctx = np.asarray(base_lens, dtype=np.int64) - geo["nq"]
    T = (ctx + n).astype(np.int32)
    w = W.make_custom(len(T), n, Hq, Hkv, D, T, seed=1234 + 17)
    S = w.num_seqs
    max_q = min(64 // (Hq // Hkv), n)
    qs = (np.arange(S + 1) * n).astype(np.int32)
    split = pkv.split_queries(qs, T, max_q, tree_len=np.full(S, n, np.int32))
    V = split["table_row"].size

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    q, k_cache, v_cache = up(w.q), up(w.k_cache), up(w.v_cache)
    k_new, v_new = up(w.k_new), up(w.v_new)
    slots = torch.from_numpy(w.slot_mapping).to(dev)
    tables = torch.from_numpy(w.block_tables).to(dev)
    v_lens, v_qs, v_tr = i32(split["context_lens"]), i32(split["q_start"]), i32(split["table_row"])
    v_tl = i32(split["tree_len"])
    tmask = torch.from_numpy(np.tile(masks, S).view(np.int32)).to(dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    ws = pkv.workspace(dev, pkv.workspace_size(V, max_q, Hq, Hkv, D))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    attn_bytes = R.attention_bytes(T, n, Hq, Hkv, D) + S * n * 4
    step_bytes = attn_bytes + R.append_bytes(S * n, Hkv, D)
    l2_mode = args.l2 if args.l2 != "auto" else (
        "none" if step_bytes >= 4 * L2_BYTES else "flush")

    def flush_fn():
        if l2_mode == "flush":
            flush.zero_()

    def step():
        pkv.kv_append(k_new, v_new, slots, k_cache, v_cache)
        pkv.paged_decode_attention_varlen(q, k_cache, v_cache, tables, v_lens, v_qs, max_q,
                                          w.scale, out, tree_mask=tmask, tree_len=v_tl,
                                          table_row=v_tr, ws=ws)

    for _ in range(args.warmup):
        flush_fn()
        step()
    torch.cuda.synchronize()
    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_k0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_k1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for ev in ev_k0 + ev_k1:
        ev.record()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # timed steps as a user runs them (unflushed: one block); the main kernel's time
    # from a separate pass
    if l2_mode == "none":
        ev_s[0].record()
        for i in range(K):
            step()
        ev_e[0].record()
    else:
        for i in range(K):
            flush_fn()
            ev_s[i].record()
            step()
            ev_e[i].record()
    HOOK = 4
    for i in range(0, K, HOOK):
        flush_fn()
        pkv.set_profiling_events(ev_k0[i], ev_k1[i])
        step()
        pkv.set_profiling_events(None, None)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    if l2_mode == "none":
        ms = ev_s[0].elapsed_time(ev_e[0]) / K
    else:
        ms = sum(a.elapsed_time(b) for a, b in zip(ev_s, ev_e)) / K
    kern = [ev_k0[i].elapsed_time(ev_k1[i]) for i in range(0, K, HOOK)]
    kern_ms = sum(kern) / len(kern)
    ms, kern_ms = max_over_ranks([ms, kern_ms], dist, dev)
    peak, peak_kind = measured_peaks()
    achieved = attn_bytes / (kern_ms * 1e-3) / 1e9
    res = {
        "metric": TREE_METRIC, "value": round(world * step_bytes / (ms * 1e-3) / 1e9, 2),
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 6), "us_per_step": round(ms * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16; " + (
            "each step reads %.1fx the L2: no flush between steps)" % (step_bytes / L2_BYTES)
            if l2_mode == "none" else "512 MiB L2 flush between steps)"),
        "config": {"workload": f"tree verify: {name} lengths + 15-node binary tree",
                   "num_seqs": S, "tree_nodes": n, "runs": V, "max_queries_per_run": max_q,
                   "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D,
                   "context_tokens": int(T.sum()), "bytes_per_step": step_bytes,
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm",
                     "kernel": "paged_decode_umma_kernel" if args.umma else "paged_decode_kernel",
                     "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs (burst)", "traffic": None,
                     "kernel_us": round(kern_ms * 1e3, 3), "algorithmic_bytes_per_launch": attn_bytes},
        "gpu_launches": 3 * K,
        "device_error_word": pkv.workspace_error(ws),
    }
    if clk is not None:
        res["clocks"] = clk
    return res


# ------------------------------------------------------------------ shared system prompt
PREFIX_METRIC = "shared-prompt decode attention GB/s (unique KV bytes); µs per step"


def run_shared_prefix(args, rank, world, dist):
    """Decode step of 256 sequences (8B-layer heads) that share a system prompt
    (--prefix-tokens, 4,096 by default), each with a private suffix of 16 ..
    --suffix-max - 1 tokens: the cascade (prompt attended once per group row tile)
    and the plain call on the same inputs; the line's value is the path the
    library's rule (pkv_cascade_pays) picks."""
    import torch

    import paged_kv_cache_101_gb300 as pkv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    S, P_TOK = 256, int(args.prefix_tokens)
    if P_TOK < 16 or P_TOK % 16 or args.suffix_max <= 16:
        raise SystemExit("--prefix-tokens must be a positive multiple of 16, --suffix-max > 16")
    rng = np.random.default_rng(1234 + 23)
    lens = P_TOK + rng.integers(16, int(args.suffix_max), size=S)
    w = W.make_custom(S, 1, 32, 8, 128, lens, seed=1234 + 23, shared=np.ones(S, bool),
                      prefix_tokens=P_TOK)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k_cache, v_cache = up(w.q), up(w.k_cache), up(w.v_cache)
    k_new, v_new = up(w.k_new), up(w.v_new)
    slots = torch.from_numpy(w.slot_mapping).to(dev)
    tables = torch.from_numpy(w.block_tables).to(dev)
    lens_d = torch.from_numpy(w.context_lens).to(dev)
    groups = torch.tensor([[0, S, P_TOK // 16]], dtype=torch.int32, device=dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    ws = pkv.workspace(dev, int(pkv.lib().pkv_workspace_size_cascade(S, 1, 32, 8, 128)))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    attn_bytes = R.workload_bytes(w, unique=True)
    step_bytes = attn_bytes + R.append_bytes(S, 8, 128)

    def step_cascade():
        pkv.kv_append(k_new, v_new, slots, k_cache, v_cache)
        pkv.paged_decode_attention_cascade(q, k_cache, v_cache, tables, lens_d, 1, w.scale, out,
                                           groups, S, ws=ws)

    def step_plain():
        pkv.kv_append(k_new, v_new, slots, k_cache, v_cache)
        pkv.paged_decode_attention(q, k_cache, v_cache, tables, lens_d, 1, w.scale, out, ws=ws)

    def timed(step, K):
        for _ in range(args.warmup):
            flush.zero_()
            step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for a, b in ev:
            flush.zero_()
            a.record()
            step()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / K

    K = args.steps
    clocks = ClockSampler(dev.index)
    clocks.start()
    if dist is not None:
        dist.barrier()
    ms = timed(step_cascade, K)
    ms_plain = timed(step_plain, K)
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms_casc, ms_plain = max_over_ranks([ms, ms_plain], dist, dev)
    # the step as the library's rule runs it by default; both paths are reported
    chosen = "cascade" if pkv.cascade_pays(w.context_lens, [[0, S, P_TOK // 16]], 8,
                                           128) else "plain"
    ms = ms_casc if chosen == "cascade" else ms_plain
    peak, peak_kind = measured_peaks()
    res = {
        "metric": PREFIX_METRIC, "value": round(world * step_bytes / (ms * 1e-3) / 1e9, 2),
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 6), "us_per_step": round(ms * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16; 512 MiB L2 flush between steps)",
        "config": {"workload": f"256 sequences sharing a {P_TOK}-token system prompt, private "
                               f"suffixes U[16, {args.suffix_max}), 8B-layer heads (32/8, d 128)",
                   "context_tokens": int(w.context_lens.sum()), "bytes_per_step": step_bytes,
                   "attention_bytes_unique": attn_bytes,
                   "attention_bytes_logical": R.workload_bytes(w, unique=False),
                   "parallelism": f"replicas x{world}"},
        "chosen_by_rule": chosen,
        "cascade": {"us_per_step": round(ms_casc * 1e3, 3),
                    "value": round(world * step_bytes / (ms_casc * 1e-3) / 1e9, 2)},
        "plain_call": {"us_per_step": round(ms_plain * 1e3, 3),
                       "value": round(world * step_bytes / (ms_plain * 1e-3) / 1e9, 2)},
        "speedup_vs_plain": round(ms_plain / ms_casc, 3),
        "roofline": {"bound": "hbm", "kernel": f"step ({chosen} path)",
                     "achieved": round(step_bytes / (ms * 1e-3) / 1e9, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(step_bytes / (ms * 1e-3) / 1e9 / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs (burst)", "traffic": None},
        "gpu_launches": 4 * K + 3 * K,
        "device_error_word": pkv.workspace_error(ws),
    }
    if clk is not None:
        res["clocks"] = clk
    return res


# ------------------------------------------------------------------ oracle (CPU)
def oracle_step_fn(w, kv_dtype: str, threads: int):
    """One whole decode step of the fp64 oracle on ``w`` (bf16 or E4M3 pools) and its
    algorithmic bytes."""
    import oracle as O

    o = O.Oracle()
    eb = 1 if kv_dtype == "fp8" else 2
    step_bytes = R.workload_bytes(w, unique=True, kv_bytes_per_element=eb) + R.append_bytes(
        int(w.slot_mapping.size), w.num_kv_heads, w.head_dim, kv_bytes_per_element=eb)
    if kv_dtype != "fp8":
        return (lambda: o.step(w, threads=threads)), step_bytes
    k8, v8, ks, vs = W.fp8_pools(w)

    def step():
        k, v = o.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, k8, v8, ks, vs)
        o.paged_attention_fp8(w.q, k, v, w.block_tables, w.context_lens, w.n_query_per_seq,
                              w.scale, ks, vs, threads=threads)
    return step, step_bytes


def oracle_sample(w, budget_s: float, threads: int, kv_dtype: str = "bf16"):
    """Time the fp64 oracle on whole decode steps of ``w`` for about budget_s seconds
    (at least one pass). Returns (GB/s of algorithmic bytes, passes, seconds)."""
    step_fn, step_bytes = oracle_step_fn(w, kv_dtype, threads)
    t0 = time.perf_counter()
    passes = 0
    while True:
        step_fn()
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el * (passes + 1) / passes > 3 * budget_s:
            break
    return passes * step_bytes / el / 1e9, passes, el


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def sample_workload(name: str, max_seqs: int, max_tokens: int = 0, w=None):
    """The first ``max_seqs`` sequences of a workload (same lengths, pool and values).
    With ``max_tokens`` the sample also stops at that many context tokens: the last
    sequence kept is cut to a shorter context, its new tokens moved to that context's
    last positions, so a step over the sample is still an append + attention."""
    w = W.make_workload(name) if w is None else w
    total = len(W.workload_lengths(name)[0])
    nq = w.n_query_per_seq
    keep = min(max_seqs, w.num_seqs)
    cut = None
    if max_tokens > 0:
        run, k = 0, 0
        while k < keep:
            T = int(w.context_lens[k])
            if run + T > max_tokens:
                L = max(max_tokens - run, nq + 15)
                if k == 0 or L > nq + 15:
                    cut = (k, min(L, T))
                    k += 1
                break
            run += T
            k += 1
        keep = max(k, 1)
    nrow = keep * nq
    w.context_lens = w.context_lens[:keep].copy()
    w.block_tables = w.block_tables[:keep].copy()
    w.q = w.q[:nrow].copy()
    w.k_new = w.k_new[:nrow].copy()
    w.v_new = w.v_new[:nrow].copy()
    w.slot_mapping = w.slot_mapping[:nrow].copy()
    w.shared = w.shared[:keep].copy()
    w.num_seqs = keep
    desc = f"all {total} sequences" if keep == total else f"first {keep} of {total} sequences"
    if cut is not None and cut[1] < int(w.context_lens[cut[0]]):
        k, L = cut
        w.context_lens[k] = L
        for j in range(nq):
            pos = L - nq + j
            w.slot_mapping[k * nq + j] = int(w.block_tables[k, pos // 16]) * 16 + pos % 16
        desc += f", the last cut to its first {L} tokens"
    if keep < total or cut is not None:
        compact_pool(w)
    return w, desc


def compact_pool(w):
    """Keep only the pool blocks the sample's sequences use (same values, ids renumbered
    in order): an oracle step copies the pool for its append, so a small sample of a
    large workload must not carry the whole pool."""
    nb = (np.maximum(w.context_lens.astype(np.int64), 0) + 15) // 16
    used = set()
    for s in range(w.num_seqs):
        used.update(int(b) for b in w.block_tables[s, :nb[s]])
    used.update(int(x) // 16 for x in w.slot_mapping if x >= 0)
    ids = np.array(sorted(used), dtype=np.int64)
    remap = np.zeros(w.num_blocks, dtype=np.int64)
    remap[ids] = np.arange(ids.size)
    tables = np.zeros_like(w.block_tables)
    for s in range(w.num_seqs):
        tables[s, :nb[s]] = remap[w.block_tables[s, :nb[s]]]
    w.block_tables = tables
    w.slot_mapping = np.where(w.slot_mapping >= 0,
                              remap[np.maximum(w.slot_mapping, 0) // 16] * 16 + w.slot_mapping % 16,
                              w.slot_mapping).astype(w.slot_mapping.dtype)
    w.k_cache = np.ascontiguousarray(w.k_cache[ids])
    w.v_cache = np.ascontiguousarray(w.v_cache[ids])
    w.num_blocks = int(ids.size)


CPU_SAMPLE_SEQS = {"tiny": 4, "llama3_8b_decode": 64, "llama3_70b_mix": 64, "long_splitk": 2,
                   "spec_verify": 16}


def cpu_baseline(args):
    threads = host_cores()
    w, desc = sample_workload(args.workload, CPU_SAMPLE_SEQS.get(args.workload, 8))
    gbs, passes, el = oracle_sample(w, args.cpu_seconds, threads, args.kv_dtype)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{desc} of {args.workload} ({args.kv_dtype} KV), {passes} full decode "
                      f"step(s) (append + fp64 attention), {el:.1f} s on {threads} threads"}


REF_BUDGET_S = 120.0  # the reference arm's warm-up + timed steps, about


def run_reference(args):
    """The fp64 oracle on the host cores, --warmup + --steps steps of a sample of the
    workload sized so that the whole run takes about REF_BUDGET_S: one timed probe step
    on the usual sample, then, if (steps + warmup) of those would take longer, a
    sample of proportionally fewer context tokens."""
    threads = host_cores()
    nseq = CPU_SAMPLE_SEQS.get(args.workload, 8)
    w_full = W.make_workload(args.workload)
    w, desc = sample_workload(args.workload, nseq, w=copy.deepcopy(w_full))
    step_fn, step_bytes = oracle_step_fn(w, args.kv_dtype, threads)
    t0 = time.perf_counter()
    step_fn()  # the probe, counted as a warm-up step
    t_probe = time.perf_counter() - t0
    per_step = REF_BUDGET_S / max(1, args.steps + args.warmup)
    if t_probe > per_step:
        tokens = int(np.sum(w.context_lens))
        budget = max(int(tokens * per_step / t_probe), 1)
        w, desc = sample_workload(args.workload, nseq, max_tokens=budget, w=w_full)
        step_fn, step_bytes = oracle_step_fn(w, args.kv_dtype, threads)
    for _ in range(max(args.warmup - 1, 0)):
        step_fn()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step_fn()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = step_bytes / (ms * 1e-3) / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs)",
        "config": {"workload": args.workload + (" (fp8 KV cache)" if args.kv_dtype == "fp8"
                                                else ""),
                   "kv_dtype": args.kv_dtype, "sample": desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{desc} of {args.workload}; each step = append + fp64 attention"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.WORKLOAD_ORDER)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="step",
                    choices=["step", "copy_blocks", "tree_verify", "shared_prefix"],
                    help="step: append + attention (the headline); copy_blocks: the "
                         "copy-on-write block copy alone; tree_verify: a 15-node candidate "
                         "tree per sequence scored with tree masks")
    ap.add_argument("--pairs", type=int, default=4096, help="block pairs per copy_blocks step")
    ap.add_argument("--cascade", default="auto", choices=["auto", "on", "off"],
                    help="shared-prefix cascade for a workload with sharers (moved to the "
                         "front of the batch): auto = the library's rule "
                         "(pkv_cascade_pays), on, off")
    ap.add_argument("--prefix-tokens", type=int, default=4096,
                    help="shared_prefix op: tokens of the shared system prompt")
    ap.add_argument("--suffix-max", type=int, default=512,
                    help="shared_prefix op: private suffixes of 16 .. suffix-max - 1 tokens")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="KV pool element type (fp8 = E4M3 codes with per-head scales)")
    ap.add_argument("--l2", default="auto", choices=["auto", "flush", "none"],
                    help="between timed steps: auto = no flush when a step reads at least 2x "
                         "the L2 (it evicts its own inputs; the tree-verify op keeps 4x), "
                         "else a 512 MiB memset")
    ap.add_argument("--pace", action="store_true",
                    help="pace the attention kernel's chunks (PKV_OPT_PACE; off by default)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config entries (every named workload's step)")
    ap.add_argument("--heads", type=int, default=0,
                    help="PKV_OPT_HEADS_PER_CTA: cap on kv heads per CTA (0 = the planner's)")
    ap.add_argument("--box", type=int, default=0, choices=[0, 1, 2],
                    help="PKV_OPT_TMA_BOX: 0 = whole-block boxes when accepted, 1 = per tile")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="PKV_OPT_PREFETCH: 0 = default L2 prefetch distance, n = n - 1 blocks")
    ap.add_argument("--two-calls", action="store_true",
                    help="time each step as pkv_kv_append + the attention call instead of "
                         "one pkv_decode_step (whose attention prologue overlaps the append)")
    ap.add_argument("--umma", action="store_true",
                    help="PKV_OPT_UMMA = 1: the tcgen05 kernel for 17-64 query rows per kv head")
    ap.add_argument("--math", default="tensor", choices=["tensor", "fma"],
                    help="attention consumers: tensor cores (default) or the CUDA-core FMA "
                         "reference path (bf16 pools, plain call)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.workload_given = any(a == "--workload" or a.startswith("--workload=") for a in sys.argv)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as td
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        td.init_process_group("nccl")
        dist = td
    if args.op in ("copy_blocks", "tree_verify", "shared_prefix"):
        fn = {"copy_blocks": run_copy, "tree_verify": run_tree,
              "shared_prefix": run_shared_prefix}[args.op]
        res = fn(args, rank, world, dist)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    res = run_pkv(args, rank, world, dist)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args)
    if not args.no_per_config and args.kv_dtype == "bf16" and args.cascade == "auto" and \
            args.math == "tensor" and args.heads == 0 and args.box == 0 and not args.pace and \
            not args.umma and args.prefetch == 0:
        res["per_config"] = run_per_config(args, rank, world, dist, res)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
