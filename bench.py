#!/usr/bin/env python3
"""Benchmark of the fused attention forward library on one GB300 (or N replicas).

Default workload: single-token GQA decode over a KV cache (B=8, Hq=32, Hkv=8,
D=128, kv_len uniform in [512, 4096], cache Lmax=4096), the configuration the
decode HBM-bandwidth metric is quoted on.  One step = one ``attn_decode`` call
(split pass + log-sum-exp combine) over that batch.  Other workloads:
``--workload decode_long | decode_gqa_paged16 | decode_multi_gqa |
prefill_causal | prefill_ragged_gqa | prefill_noncausal_d64 | tiny_causal``
(``decode_multi_gqa``: 8 new tokens per sequence through ``attn_decode_multi``).

Timing: inputs resident in HBM; the case keeps enough copies of its inputs
and outputs that every step reads a copy no step has touched for at least
4x the L2 size (129 MB) of other traffic, so no step finds its K/V in L2 and
no flush is needed.  W untimed warm-up steps; then exactly K steps, cycling
the copies, captured as one CUDA graph; after a few untimed replays of that
graph, one replay is timed by a pair of CUDA events on the launching stream;
barrier + synchronize on both sides; max over ranks.  ``value`` is
algorithmic bytes (decode: K/V rows actually attended, plus q, O and lse) or
algorithmic FLOPs (prefill: 4*D per visible query/key pair) per second.
``per_launch_flushed`` repeats the measurement one launch at a time, each
between its own pair of events with a 512 MB write-then-read L2 flush before
it (it includes the per-launch event and launch floor).
``e2e`` repeats the measurement through the same call with the inputs copied
from pinned host memory and the outputs copied back inside the timed region
(one call at a time, L2 flushed before each).
``cpu_baseline`` times the fp64 oracle on a bounded sample on the host cores
(one spawn-started worker per core; each worker rebuilds the workload's
inputs from the seeded generators once, so a unit of work ships only its
indices).

``--impl reference`` times that oracle alone (the only reference this
library has) and prints the same JSON line with ``"impl": "reference"``;
each step is one bounded sample and the whole run, warm-up included, takes
about ``--ref-total`` seconds of host work (default 120).

With ``--gpus N > 1`` (launched by torch.distributed.run) every rank runs an
independent replica of the workload; nothing is exchanged ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn HBM GB/s (% of peak); prefill attn TFLOP/s (% of tensor peak)"
FLUSH_BYTES = 512 << 20
L2_BYTES = 129 * 10**6  # GB300 L2; the device property is used when it reports more
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0


# ----------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": HBM_FALLBACK_GBS, "bf16_tflops": BF16_FALLBACK_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def code_digest(path: str) -> str:
    """sha256 prefix of a kernel source with its // comments and all whitespace removed: a comment edit does
    not make committed counters stale, a code edit does."""
    import hashlib
    import re

    text = open(path, encoding="utf-8").read()
    code = "".join(line.split("//", 1)[0] for line in text.splitlines())
    return hashlib.sha256(re.sub(r"\s+", "", code).encode()).hexdigest()[:16]


def read_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` on `workload` from the committed ncu summary, or None when there is
    none or the kernel code changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if "=" in line and not line.startswith("#"):
            k, v = line.strip().split("=", 1)
            kv[k.strip()] = v.strip()
    src = os.path.join(ROOT, "attention_attn_fwd_06_gb300", "csrc", kv.get("source", ""))
    if not os.path.exists(src) or code_digest(src) != kv.get("code_sha256_16"):
        return None  # kernel changed since the counters were taken
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (t, sm, max, power, reasons)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            reasons = [n for n, v in zip(names, parts[3:7]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, mx, parts[2], reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1, label="timed"):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = label
        if not inside:
            inside = [s for s in self.samples if s[0] <= t1 + 0.5]
            window = "warmup+timed (the timed region was shorter than the sampling interval)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
        sms = sorted(s[1] for s in inside)
        reasons = sorted({r for s in inside for r in s[4]})
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------- workloads

def _pin(t):
    """Page-locked copy for the end-to-end leg; plain memory when no GPU is visible (the oracle-only arm)."""
    import torch

    return t.pin_memory() if torch.cuda.is_available() else t


class _Rotation:
    """Copies of a workload's inputs (and outputs) cycled by ``step``, so that consecutive steps read different
    addresses: with enough copies every step finds its inputs evicted from L2 by the steps in between."""

    def _init_sets(self):
        self.sets = [(self.dev, self.out, self.lse)]
        self._next = 0

    def rotate_inputs(self, l2_bytes, max_copies):
        """Enough copies that (copies - 1) steps of other traffic cover at least 4x L2, but no more copies than
        steps (a copy no step reads is no use); returns the count."""
        import torch

        n = max(2, math.ceil(4 * l2_bytes / self.touch_bytes) + 1)
        n = max(1, min(n, max_copies))
        self.l2_bytes = l2_bytes
        self.sets = [(self.dev, self.out, self.lse)] + [
            ([t.clone() for t in self.dev], torch.empty_like(self.out), torch.empty_like(self.lse))
            for _ in range(n - 1)]
        self._next = 0
        return n

    def set_bytes(self):
        dev, out, lse = self.sets[0]
        return sum(t.numel() * t.element_size() for t in dev) + out.numel() * out.element_size() + lse.numel() * 4

    def step(self):
        dev, out, lse = self.sets[self._next]
        self._next = (self._next + 1) % len(self.sets)
        self._call(dev, out, lse)

    def step_e2e(self):
        for d, h in zip(self.dev, self.host):
            d.copy_(h, non_blocking=True)
        self._call(self.dev, self.out, self.lse)
        self.out_h.copy_(self.out, non_blocking=True)
        self.lse_h.copy_(self.lse, non_blocking=True)


class _RopeMixin:
    def _rope_setup(self, w, max_pos, device):
        """RoPE tables (model constants: resident on the device, not copied per step) when the workload asks."""
        self.rope_style = w.extra.get("rope")
        self.rope_dev = None
        if self.rope_style:
            from attention_attn_fwd_06_gb300.inputs import rope_tables

            cos, sin = rope_tables(max_pos, w.D)
            self.rope_dev = (cos.to(device), sin.to(device), self.rope_style)


class DecodeCase(_Rotation, _RopeMixin):
    def __init__(self, w, device):
        import torch

        from attention_attn_fwd_06_gb300.inputs import make_decode, make_decode_multi

        self.w = w
        self.multi = w.kind == "decode_multi"
        self.Lq = w.Lq if self.multi else 1
        if self.multi:
            q, kc, vc, lens = make_decode_multi(w.B, w.Hq, w.Hkv, w.Lq, w.L, w.D, w.seed,
                                                kv_lens=w.kv_lens or None, kv_range=w.kv_range or None)
        else:
            q, kc, vc, lens = make_decode(w.B, w.Hq, w.Hkv, w.L, w.D, w.seed,
                                          kv_lens=w.kv_lens or None, kv_range=w.kv_range or None)
        self.page_size = w.extra.get("page_size")
        self._rope_setup(w, w.L, device)
        if self.page_size:
            from attention_attn_fwd_06_gb300.inputs import make_pages

            kp, vp, table = make_pages(kc, vc, self.page_size, w.seed + 7, fill_unused=0.0)
            self.host = [_pin(t) for t in (q, kp, vp, lens, table)]
        else:
            self.host = [_pin(t) for t in (q, kc, vc, lens)]
        self.dev = [t.to(device) for t in self.host]
        tok = (self.Lq,) if self.multi else ()
        self.out = torch.empty((w.B, w.Hq) + tok + (w.D,), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((w.B, w.Hq) + tok, dtype=torch.float32, device=device)
        self.out_h = _pin(torch.empty_like(self.out, device="cpu"))
        self.lse_h = _pin(torch.empty_like(self.lse, device="cpu"))
        self.lens = [int(x) for x in lens.tolist()]
        # algorithmic bytes: every attended K/V row once, q and O once, lse once
        kv_bytes = sum(self.lens) * w.Hkv * w.D * 2 * 2
        rows = w.B * w.Hq * self.Lq
        self.alg_bytes = kv_bytes + rows * w.D * 2 * 2 + rows * 4
        self.work = self.alg_bytes
        self.touch_bytes = self.alg_bytes  # bytes one step reads and writes
        self._init_sets()
        self.unit, self.kind = "GB/s", "hbm"
        self.kernel = "decode_multi" if self.multi else "decode_split"
        self.kernel_desc = ("decode_multi_kernel (one attn_decode_multi call: tcgen05 split pass with the merge fused, "
                            "event-timed)" if self.multi else
                            "decode_split_kernel (one attn_decode call: split pass with the combine fused, event-timed)")
        self.launches_per_step = 1
        self.h2d = sum(t.numel() * t.element_size() for t in self.host)
        self.d2h = self.out.numel() * 2 + self.lse.numel() * 4

    def _call(self, dev, out, lse):
        from attention_attn_fwd_06_gb300 import binding as AB

        r = self.rope_dev
        if self.page_size:
            q, kp, vp, lens, table = dev
            AB.attn_decode_paged(q, kp, vp, table, lens, out=out, lse=lse, scale=self.w.scale, rope=r)
        elif self.multi:
            q, kc, vc, lens = dev
            AB.attn_decode_multi(q, kc, vc, lens, out=out, lse=lse, scale=self.w.scale, rope=r)
        else:
            q, kc, vc, lens = dev
            AB.attn_decode(q, kc, vc, lens, out=out, lse=lse, scale=self.w.scale, rope=r)

    def oracle_sample(self, budget_s):
        """(work units done, seconds, cores, description) for the fp64 oracle on a bounded sample."""
        return run_oracle_pool(self, budget_s)


class PrefillCase(_Rotation, _RopeMixin):
    def __init__(self, w, device):
        import torch

        from attention_attn_fwd_06_gb300.inputs import make_prefill, make_varlen

        self.w = w
        self._rope_setup(w, w.L if w.kind != "varlen" else w.seq_range[1], device)
        if w.kind == "varlen":
            q, k, v, cu = make_varlen(w.B, w.Hq, w.Hkv, w.D, w.seed, seq_range=w.seq_range)
            self.cu = cu
            self.seqlens = [int(cu[i + 1] - cu[i]) for i in range(w.B)]
            self.host = [_pin(t) for t in (q, k, v, cu)]
            total = int(cu[-1])
            self.out = torch.empty((total, w.Hq, w.D), dtype=torch.bfloat16, device=device)
            self.lse = torch.empty((total, w.Hq), dtype=torch.float32, device=device)
        else:
            q, k, v = make_prefill(w.B, w.Hq, w.Hkv, w.L, w.L, w.D, w.seed)
            self.seqlens = [w.L] * w.B
            self.host = [_pin(t) for t in (q, k, v)]
            odt = torch.float32 if w.out_f32 else torch.bfloat16
            self.out = torch.empty((w.B, w.Hq, w.L, w.D), dtype=odt, device=device)
            self.lse = torch.empty((w.B, w.Hq, w.L), dtype=torch.float32, device=device)
        self.dev = [t.to(device) for t in self.host]
        self.out_h = _pin(torch.empty_like(self.out, device="cpu"))
        self.lse_h = _pin(torch.empty_like(self.lse, device="cpu"))
        pairs = sum((L * (L + 1)) // 2 if w.causal else L * L for L in self.seqlens)
        self.work = 4.0 * w.D * w.Hq * pairs
        self.unit, self.kind = "TFLOP/s", "tensor"
        self.kernel = "prefill_fwd"
        self.kernel_desc = "prefill_fwd_kernel (one attn_fwd call, event-timed)"
        # with RoPE a call launches the key- and query-rotation passes, then the attention kernel
        self.launches_per_step = 3 if self.rope_style else 1
        self.h2d = sum(t.numel() * t.element_size() for t in self.host)
        self.d2h = self.out.numel() * self.out.element_size() + self.lse.numel() * 4
        self.touch_bytes = self.h2d + self.d2h  # q, k, v read and O, lse written once per step (at least)
        self._init_sets()

    def _call(self, dev, out, lse):
        import torch

        from attention_attn_fwd_06_gb300 import binding as AB

        w = self.w
        if w.kind == "varlen":
            q, k, v, cu = dev
            mx = max(self.seqlens)
            AB.attn_fwd_varlen(q, k, v, cu, cu, mx, mx, out=out, lse=lse, causal=w.causal, scale=w.scale,
                               rope=self.rope_dev)
        else:
            q, k, v = dev
            AB.attn_fwd(q, k, v, out=out, lse=lse, causal=w.causal, scale=w.scale,
                        out_dtype=torch.float32 if w.out_f32 else torch.bfloat16, rope=self.rope_dev)

    def oracle_sample(self, budget_s):
        return run_oracle_pool(self, budget_s)


# ----------------------------------------------------------------------------- oracle (CPU) leg

_ORACLE_DATA = None  # per worker process: the workload's inputs as the oracle takes them


def _oracle_inputs(name):
    """(workload, q, k, v, lengths or cu_seqlens, rope) of a workload, rebuilt from its seeded generators: the
    same bf16 values the kernels get, as fp32 arrays (exact), which the oracle lifts to fp64."""
    from attention_attn_fwd_06_gb300.inputs import (WORKLOADS, make_decode, make_decode_multi, make_prefill,
                                                    make_varlen, rope_tables)

    w = WORKLOADS[name]
    lens = None
    if w.kind == "decode_multi":
        q, k, v, n = make_decode_multi(w.B, w.Hq, w.Hkv, w.Lq, w.L, w.D, w.seed,
                                       kv_lens=w.kv_lens or None, kv_range=w.kv_range or None)
        lens, max_pos = [int(x) for x in n.tolist()], w.L
    elif w.kind == "decode":
        q, k, v, n = make_decode(w.B, w.Hq, w.Hkv, w.L, w.D, w.seed,
                                 kv_lens=w.kv_lens or None, kv_range=w.kv_range or None)
        lens, max_pos = [int(x) for x in n.tolist()], w.L
    elif w.kind == "varlen":
        q, k, v, cu = make_varlen(w.B, w.Hq, w.Hkv, w.D, w.seed, seq_range=w.seq_range)
        lens, max_pos = [int(x) for x in cu.tolist()], w.seq_range[1]
    else:
        q, k, v = make_prefill(w.B, w.Hq, w.Hkv, w.L, w.L, w.D, w.seed)
        max_pos = w.L
    rope = None
    if w.extra.get("rope"):
        cos, sin = rope_tables(max_pos, w.D)
        rope = (cos.numpy(), sin.numpy(), w.extra["rope"])
    return w, q.float().numpy(), k.float().numpy(), v.float().numpy(), lens, rope


def _oracle_init(name):
    global _ORACLE_DATA
    os.environ["OMP_NUM_THREADS"] = "1"
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    _ORACLE_DATA = _oracle_inputs(name)


def _oracle_task(unit):
    """One unit of the workload through the oracle's own entry points; returns its seconds."""
    import oracle

    w, q, k, v, lens, rope = _ORACLE_DATA
    a, h = unit
    hk = h // (w.Hq // w.Hkv)
    t0 = time.perf_counter()
    if w.kind in ("decode", "decode_multi"):
        n = lens[a]
        args = (q[a, h][None, None], k[a, hk][None, None, :n], v[a, hk][None, None, :n], [n], w.scale)
        if w.kind == "decode":  # q [D]
            oracle.decode(*args, rope=rope)
        else:  # q [Lq, D]: bottom-right causal over the sequence's n keys
            oracle.decode_multi(*args, rope=rope)
    elif w.kind == "varlen":
        s0, s1 = lens[a], lens[a + 1]
        oracle.attention(q[s0:s1, h][None, None], k[s0:s1, hk][None, None], v[s0:s1, hk][None, None], w.scale,
                         w.causal, rope=rope)
    else:
        oracle.attention(q[a, h][None, None], k[a, hk][None, None], v[a, hk][None, None], w.scale, w.causal,
                         rope=rope)
    return time.perf_counter() - t0


class OraclePool:
    """The fp64 oracle timed on bounded, seeded samples of a case's rows, on all host cores.

    Work units are dealt to a spawn-started process pool (one BLAS thread per
    process; started once, outside every timed sample) in rounds of one unit
    per core until a sample's budget has passed; a sample's work counts the
    algorithmic work of the units finished.  Decode units are (b, hq) rows,
    each worth its share of its kv head's K/V bytes plus its q, O and lse;
    prefill units are (sequence, head) problems worth 4*D FLOPs per visible
    pair.  Samples continue through the seeded unit order where the last one
    stopped.
    """

    def __init__(self, case):
        import multiprocessing as mp

        import numpy as np

        w = case.w
        rng = np.random.default_rng(12345)
        self.cores = os.cpu_count() or 1
        units = []  # ((sequence, q head), algorithmic work)
        g = w.Hq // w.Hkv
        if isinstance(case, DecodeCase):
            Lq = case.Lq
            for b in range(w.B):
                for h in range(w.Hq):
                    units.append(((b, h), case.lens[b] * w.D * 2 * 2 / g + Lq * (w.D * 2 * 2 + 4)))
            self.what = "(b, hq) decode rows" if Lq == 1 else f"(b, hq) decode rows of {Lq} tokens"
        else:
            for a in range(w.B):
                L = case.seqlens[a]
                f = 4.0 * w.D * ((L * (L + 1)) // 2 if w.causal else L * L)
                for h in range(w.Hq):
                    units.append(((a, h), f))
            self.what = "(sequence, head) prefill problems"
        order = rng.permutation(len(units))
        self.units = [units[i] for i in order]
        self._i = 0
        # every worker rebuilds the inputs from the seeded generators once (no arrays cross the pipe per unit);
        # the start-up and a first unit per worker stay outside every timed sample
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_oracle_init, initargs=(w.name,))
        self.pool.map(_oracle_task, [self.units[0][0]] * self.cores, chunksize=1)

    def sample(self, budget_s):
        """(work units done, seconds, cores, description) for rounds of units until ``budget_s`` has passed."""
        done, work = 0, 0.0
        t0 = time.perf_counter()
        while True:
            batch = [self.units[(self._i + j) % len(self.units)] for j in range(self.cores)]
            self.pool.map(_oracle_task, [u[0] for u in batch], chunksize=1)
            self._i += self.cores
            done += len(batch)
            work += sum(u[1] for u in batch)
            if time.perf_counter() - t0 >= budget_s or done >= 50 * len(self.units):
                break
        dt = time.perf_counter() - t0
        desc = (f"{done} {self.what} (of {len(self.units)} in the workload; seeded order, repeating if all done), "
                f"fp64 numpy oracle, {self.cores} spawn worker processes x 1 BLAS thread, {dt:.1f} s")
        return work, dt, self.cores, desc

    def close(self):
        self.pool.terminate()
        self.pool.join()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def run_oracle_pool(case, budget_s):
    """One bounded sample of the fp64 oracle on all host cores (see ``OraclePool``)."""
    with OraclePool(case) as pool:
        return pool.sample(budget_s)


# ----------------------------------------------------------------------------- main

def make_case(name, device):
    from attention_attn_fwd_06_gb300.inputs import WORKLOADS

    w = WORKLOADS[name]
    return DecodeCase(w, device) if w.kind in ("decode", "decode_multi") else PrefillCase(w, device)


def workload_config(case):
    w = case.w
    cfg = {"workload": w.name, "kind": w.kind, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
           **({"rope": w.extra["rope"]} if w.extra.get("rope") else {}),
           "l2": l2_note(case)}
    if w.kind in ("decode", "decode_multi"):
        if w.kind == "decode_multi":
            cfg["Lq"] = w.Lq
        cfg.update({"Lmax": w.L, "kv_lens": "uniform [%d, %d]" % w.kv_range if w.kv_range else list(w.kv_lens),
                    "kv_tokens_total": sum(case.lens)})
        if w.extra.get("page_size"):
            cfg["page_size"] = w.extra["page_size"]
    elif w.kind == "varlen":
        cfg.update({"nseq": w.B, "seq_range": list(w.seq_range), "total_tokens": sum(case.seqlens),
                    "causal": w.causal})
    else:
        cfg.update({"L": w.L, "causal": w.causal})
    return cfg


def l2_clean(case):
    """True when every timed step reads an input copy last touched >= 4x the L2 size of traffic earlier."""
    l2 = getattr(case, "l2_bytes", None)
    return l2 is not None and (len(case.sets) - 1) * case.touch_bytes >= 4 * l2


def compact_config(case):
    """One short line naming the workload's shape."""
    c = workload_config(case)
    c.pop("l2", None)
    return " ".join(f"{k}={v}" for k, v in c.items() if k != "workload")


def l2_note(case):
    n = len(case.sets)
    l2 = getattr(case, "l2_bytes", None)
    if l2 is None:
        return "flushed between timed steps: a 512 MB buffer written, then read"
    reuse = (n - 1) * case.touch_bytes
    how = "the K steps run back to back as one CUDA graph replay between one pair of CUDA events"
    if reuse >= 4 * l2:
        return (f"not flushed: inputs larger than L2 -- {n} copies of the inputs and outputs "
                f"({n * case.set_bytes() / 1e9:.2f} GB) cycled step by step, so each step reads a copy last touched "
                f"{n - 1} steps ({reuse / 1e6:.0f} MB of other traffic, >= 4x the {l2 / 1e6:.0f} MB L2) earlier; {how}")
    return (f"not flushed, and inputs may be L2-resident: {n} copies cycled, each step's last touched {n - 1} steps "
            f"({reuse / 1e6:.1f} MB of other traffic) earlier, less than 4x the {l2 / 1e6:.0f} MB L2 (a small "
            f"configuration, or fewer steps than copies needed); {how}")


def flush_l2(flush):
    """Evict the inputs from L2: write a buffer larger than L2, then read it back.

    The read leaves L2 holding clean lines of the flush buffer, so the timed kernel does not also pay for
    writing back 129 MB of dirty flush data (traffic that is no part of attention)."""
    import torch

    flush.zero_()
    flush.view(-1, 4096).sum(dim=1, dtype=torch.int64)


def time_steps(case, steps, warmup, flush, e2e=False):
    """Each step a launch between its own pair of CUDA events, L2 flushed before it (the per-launch view)."""
    import torch

    fn = case.step_e2e if e2e else case.step
    for _ in range(warmup):
        flush_l2(flush)
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(steps):
        flush_l2(flush)
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return sum(ms), ms, t_wall0, t_wall1


def l2_bytes(device):
    import torch

    return max(int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0)), L2_BYTES)


def time_graph(case, steps, warmup, load_s=0.3):
    """K steps back to back, cycling the case's input copies, captured as one CUDA graph; one replay is timed
    by one pair of CUDA events.  W eager warm-up steps come first (they also size the library workspace, so
    the captured calls allocate nothing), then untimed replays of the same graph for ``load_s`` seconds (graph
    upload, clocks under this load, and clock samples for a timed region shorter than the sampling interval).
    Returns (milliseconds for the K steps, wall time of the first loaded replay, wall time after the timed one)."""
    import torch

    for _ in range(warmup):
        case.step()
    torch.cuda.synchronize()
    case._next = 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            case.step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t_load = time.time()
    while True:
        graph.replay()
        torch.cuda.synchronize()
        if time.time() - t_load >= load_s:
            break
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(stream)
    graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    ms = start.elapsed_time(end)
    del graph
    return ms, t_load, t_wall1


_dist = None


def barrier():
    if _dist is not None:
        _dist.barrier()


def max_over_ranks(x: float) -> float:
    """The largest of every rank's value (the slowest replica sets the job's time)."""
    if _dist is None:
        return x
    import torch

    device = "cuda" if _dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    _dist.all_reduce(t, op=_dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args):
    global _dist
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        _dist = dist
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)

    from attention_attn_fwd_06_gb300 import binding as AB

    AB.load()
    pk = peaks()
    case = make_case(args.workload, device)
    case.rotate_inputs(l2_bytes(device), max_copies=args.steps)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    time.sleep(0.2)
    total_ms, tw0, tw1 = time_graph(case, args.steps, args.warmup)
    if AB.attn_get_device_status() != AB.ATTN_OK:
        raise RuntimeError("device status reported an error during the timed steps")
    clk = clocks.summary(tw0, tw1, "untimed replays of the timed CUDA graph (same load) and the timed replay")
    n_side = max(3, args.steps // 4)
    launch_ms, _, _, _ = time_steps(case, n_side, 3, flush)
    e2e_ms, _, _, _ = time_steps(case, n_side, 2, flush, e2e=True)
    clocks.stop()
    if AB.attn_get_device_status() != AB.ATTN_OK:
        raise RuntimeError("device status reported an error during the per-launch or end-to-end steps")

    total_ms = max_over_ranks(total_ms)
    launch_ms = max_over_ranks(launch_ms)
    e2e_ms = max_over_ranks(e2e_ms)
    sec_per_step = total_ms / 1e3 / args.steps
    scale_unit = 1e9 if case.unit == "GB/s" else 1e12
    value = world * case.work / sec_per_step / scale_unit
    per_gpu = case.work / sec_per_step / scale_unit
    e2e_value = world * case.work / (e2e_ms / 1e3 / n_side) / scale_unit
    launch_value = case.work / (launch_ms / 1e3 / n_side) / scale_unit
    if case.kind == "hbm":
        peak, peak_src = pk["hbm_gbs"], pk["source"]
        roof = {"bound": "hbm", "achieved": per_gpu, "peak": peak, "unit": "GB/s", "frac": per_gpu / peak,
                "traffic": read_traffic(case.kernel, case.w.name), "peak_source": peak_src,
                "kernel": case.kernel_desc}
    else:
        peak, peak_src = pk["bf16_tflops"], pk["source"]
        roof = {"bound": "tensor", "achieved": per_gpu, "peak": peak, "unit": "TFLOP/s", "frac": per_gpu / peak,
                "traffic": read_traffic(case.kernel, case.w.name), "peak_source": peak_src,
                "kernel": case.kernel_desc}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": case.unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec_per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) rounded to bf16)",
        "config": dict(workload_config(case), parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "e2e": {"value": e2e_value, "unit": case.unit, "h2d_bytes_per_step": case.h2d,
                "d2h_bytes_per_step": case.d2h},
        "gpu_launches": case.launches_per_step * args.steps,
        "roofline": roof,
        "per_launch_flushed": {"value": launch_value, "unit": case.unit, "ms_per_step": launch_ms / n_side,
                               "frac": launch_value / peak, "steps": n_side,
                               "how": "each step one launch between its own pair of CUDA events, L2 flushed "
                                      "(512 MB written, then read) before it; includes the per-launch event floor"},
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        work, dt, cores, desc = case.oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": work / dt / scale_unit, "unit": case.unit, "cores": cores,
                                "kind": "oracle", "sample": desc, "seconds": dt}
    if rank == 0 and args.also:
        # Every extra workload is timed like the main one (a CUDA-graph replay over rotating input copies) and
        # reported by a few short numbers; the shapes and the shared timing note come first, in "also_config",
        # so the per-workload results close the line.
        also, also_cfg = {}, {}
        for name in args.also.split(","):
            if not name or name == args.workload:
                continue
            try:
                c2 = make_case(name, device)
                n2 = max(8, args.steps // 4)
                c2.rotate_inputs(l2_bytes(device), max_copies=n2)
                t_ms, _, _ = time_graph(c2, n2, 3, load_s=0.05)
                l_ms, _, _, _ = time_steps(c2, n2, 3, flush)
                s_step = t_ms / 1e3 / n2
                su = 1e9 if c2.unit == "GB/s" else 1e12
                v2 = c2.work / s_step / su
                pkv = pk["hbm_gbs"] if c2.kind == "hbm" else pk["bf16_tflops"]
                traffic = read_traffic(c2.kernel, name)
                also[name] = {"value": round(v2, 1), "unit": c2.unit, "ms_per_step": round(s_step * 1e3, 5),
                              "frac": round(v2 / pkv, 4), "traffic": traffic, "l2_clean": l2_clean(c2),
                              "flushed_ms": round(l_ms / n2, 5)}
                also_cfg[name] = compact_config(c2)
                del c2
                torch.cuda.empty_cache()
            except Exception as e:  # a workload whose kernel is not built yet is reported, not fatal
                also[name] = {"error": str(e)[:200]}
        also_cfg["timing"] = ("value, ms_per_step: max(8, steps/4) steps back to back as one CUDA-graph replay over "
                              "rotating input copies (l2_clean: each step's copy last touched >= 4x the L2 size "
                              "of traffic earlier); flushed_ms: one launch between its own CUDA events after a "
                              "512 MB L2 flush; frac: value / the measured peak of the roofline column")
        line["also_config"] = also_cfg
        line["also"] = also
    if rank == 0:
        print(json.dumps(line), flush=True)
    if _dist is not None:
        _dist.destroy_process_group()


def run_reference(args):
    """The oracle timed as it stands on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch  # noqa: F401

    case = make_case(args.workload, "cpu")
    # each step is one bounded sample; the whole run (warm-up included) stays within about --ref-total seconds
    budget = min(args.ref_budget, args.ref_total / max(1, args.steps + args.warmup))
    per_step, work_sum = [], 0.0
    desc, cores = "", 0
    with OraclePool(case) as pool:
        for i in range(args.warmup + args.steps):
            work, dt, cores, desc = pool.sample(budget)
            if i >= args.warmup:
                per_step.append(dt)
                work_sum += work
    scale_unit = 1e9 if case.unit == "GB/s" else 1e12
    sec = sum(per_step) / len(per_step)
    value = work_sum / sum(per_step) / scale_unit
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": case.unit,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) rounded to bf16)",
        "config": dict(workload_config(case), l2="not applicable: the oracle runs on the host cores"),
        "cpu_baseline": {"value": value, "unit": case.unit, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": case.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_gqa")
    ap.add_argument("--also", default="decode_long,decode_gqa_paged16,decode_gqa_rope,decode_multi_gqa,decode_multi_long,"
                                      "prefill_causal,prefill_causal_rope,prefill_ragged_gqa,prefill_noncausal_d64",
                    help="comma-separated extra workloads measured in the same run (rank 0, N=1 style)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of host work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=5.0, help="at most this many seconds of host work per "
                                                                  "reference step")
    ap.add_argument("--ref-total", type=float, default=120.0,
                    help="seconds of host work for the whole reference run (warm-up steps included)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
