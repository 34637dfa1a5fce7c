#!/usr/bin/env python3
"""Benchmark of the OSCAR decode hot path on GB300 (one JSON line on rank 0).

A step is one full decode step of the workload: for every layer, the fused
eviction of the oldest recent token of every sequence into the INT2 history
(with the ring append of the new token) followed by decode attention over
sink + INT2 history + recent window.  The state advances every step
(history +1 token per sequence and layer).  Inputs are synthetic, seeded,
and already resident in HBM when the timed region starts; every layer has
its own pool (far larger than the 129 MB L2), so no L2 flush is needed.

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the float64 CPU oracle arm

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
sequences are independent); no collective is on the data path, and timing
takes the max over ranks ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_evict_gb300 import synth as S  # noqa: E402

METRIC = "decode context-tokens/s attended"
UNIT = "tokens/s"
HIST_BYTES_PER_TOKEN_HEAD = 96      # 2 x 32 B codes + 2 x 4 x (fp16 s, fp16 z) at 32 positions per group
BOOST_RECORD_BYTES = 16             # K channel boost: 8 x (position, 4-bit code) entries per K token-vector


def hist_bytes_per_token_head(g: int) -> int:
    """INT2 history bytes per (token, KV head): K and V codes + (s, z) pairs."""
    return 2 * 32 + 2 * (128 // g) * 4
BF16_BYTES_PER_TOKEN_HEAD = 2 * 128 * 2
DEFAULT_WORKLOAD = "qwen3_8b_36l"

# DRAM traffic of int2_kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum of one launch: the one-layer version of the
# workload, the bench's own launch configuration, captured with
# `ncu --set full -k regex:int2_kernel -c 1`), with the algorithmic bytes of
# the captured launch.  Reported, scaled to the bench's mean launch by the
# units processed, only while the kernel source is the one captured.
INT2_TRAFFIC_CAPTURE = {
    "workload": "qwen3_8b_36l",
    "source_sha256_16": "23a75730b702d91a",     # csrc/decode.cu + csrc/oscar_common.cuh, comments removed
    "traffic_bytes": 917.45e6 + 12.07e6,
    "algorithmic_bytes": 911.11e6,
}


def kernel_source_hash() -> str:
    """sha256 prefix of the INT2 kernel's sources with comments and blank
    lines removed (the captured counters depend on the code, not on its
    comments)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("decode.cu", "oscar_common.cuh"):
        with open(os.path.join(ROOT, "bit_kv_cache_evict_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        for line in text.splitlines():
            code = re.sub(r"//.*$", "", line).rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def int2_traffic(workload: str, int2_bytes: float):
    cap = INT2_TRAFFIC_CAPTURE
    if workload != cap["workload"] or kernel_source_hash() != cap["source_sha256_16"]:
        return None
    return int2_bytes * cap["traffic_bytes"] / cap["algorithmic_bytes"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["oscar", "reference"], default="oscar")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(S.WORKLOADS))
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (testing)")
    ap.add_argument("--cpu-tokens", type=int, default=60000,
                    help="history tokens in the oracle's bounded sample")
    ap.add_argument("--cpu-steps", type=int, default=12,
                    help="oracle steps timed for cpu_baseline (about 10 s of host work)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the one-layer side records (gate, frac_by_workload) of a 1-GPU run")
    ap.add_argument("--calibrate", action="store_true",
                    help="time the offline rotation calibration (oscar_calibrate_rotation) instead of a decode "
                         "step: one JSON line, the float64 oracle timed on the same inputs")
    ap.add_argument("--codebook", type=float, default=None, metavar="A",
                    help="Lloyd-Max levels {0, A, 3-A, 3} for every head instead of the uniform grid")
    ap.add_argument("--boost", action="store_true",
                    help="K channel precision boost: eight positions per K token-vector at 4 bits")
    ap.add_argument("--quant-group", type=int, default=32, choices=[32, 64, 128],
                    help="stored positions per fp16 scale/zero pair (32 is the configured format)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------

def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend)


def reduce_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(t_ms: float, units: float, world: int, device=None):
    """Whole-job throughput of a weak-scaling replica run: the slowest
    rank's time (max over ranks) and the units all ranks processed (sum).
    Returns (value in units/s, max time in ms)."""
    t_max = reduce_max(t_ms, world, device)
    total = reduce_sum(float(units), world, device)
    return total / (t_max / 1e3), t_max


def reference_budget(args) -> int:
    """History tokens of the oracle's sample per reference-arm step: about
    six million attended tokens over the whole --steps/--warmup run (a few
    minutes on the host cores), at most --cpu-tokens, at least 8000."""
    return int(min(args.cpu_tokens, max(8000, 6e6 / max(1, args.steps + args.warmup))))


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 8]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1].split()[0]))
                smax = float(r[2].split()[0])
                power.append(float(r[3].split()[0]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if "Active" in v and "Not" not in v:
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no samples"]}
        # samples under load: power within 35% of the peak seen
        pmax = max(power) if power else 0
        loaded = [s for s, p in zip(sm, power) if p >= 0.65 * pmax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": pmax}


# ---------------------------------------------------------------------------
# workload state on the GPU
# ---------------------------------------------------------------------------

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


class GpuState:
    """Pools, BF16 segments, queries and per-step metadata for every layer."""

    def __init__(self, w: S.Workload, layers: int, steps_total: int, rank: int, quant_group: int = 32,
                 codebook: float | None = None, boost: bool = False):
        import torch
        from bit_kv_cache_evict_gb300 import oscar as O
        self.O, self.torch = O, torch
        self.w, self.L = w, layers
        dev = torch.device("cuda")
        self.dev = dev
        B, Hq, Hk, d = w.batch, w.hq, w.hk, S.D
        self.shape = O.make_shape(Hq, Hk, quant_group=quant_group)
        # K channel boost: one 16-byte record per K token-vector beside the pool
        self.boost = boost
        self.hist_tok_bytes = hist_bytes_per_token_head(quant_group) + (BOOST_RECORD_BYTES if boost else 0)
        ctx = S.context_lengths(w)
        self.ctx0 = ctx
        hist0 = np.maximum(ctx - S.NSLOT, 0).astype(np.int64)
        self.hist0 = hist0
        cap = hist0 + steps_total + 1
        self.max_pages = int((cap.max() + S.PAGE - 1) // S.PAGE)
        grp = None
        if w.prefix_seqs:
            grp = np.full(B, -1, np.int32)
            grp[: w.prefix_seqs] = 0
        perm_seed = (w.seed * 7919 + 1) if w.shuffled else 0
        table, self.num_pages, self.pool_bytes = O.oscar_pool_layout(self.shape, cap, grp, w.shared_hist_tokens,
                                                                     perm_seed, self.max_pages)
        self.table = torch.from_numpy(table).to(dev)
        self.B, self.Hq, self.Hk = B, Hq, Hk
        # per-step metadata (device): eviction target position, ring row,
        # history length after the step
        steps = np.arange(steps_total, dtype=np.int64)[:, None]
        self.hist_before = torch.from_numpy((hist0[None, :] + steps).astype(np.int32)).to(dev)
        self.hist_after = torch.from_numpy((hist0[None, :] + steps + 1).astype(np.int32)).to(dev)
        rows = np.arange(B)[None, :] * S.NSLOT + S.SINK + (steps % S.RECENT)
        self.src_row = torch.from_numpy(rows.astype(np.int32)).to(dev)
        self.seqs = torch.arange(B, dtype=torch.int32, device=dev)
        self.bf16_len = torch.full((B,), S.NSLOT, dtype=torch.int32, device=dev)
        self.sm_scale = 1.0 / math.sqrt(d)
        self.ws = torch.empty(O.oscar_decode_workspace_bytes(self.shape, B, self.max_pages), dtype=torch.uint8,
                              device=dev)
        # Lloyd-Max levels {0, a, 3 - a, 3} with one a for every head (None: uniform levels)
        self.cb = None if codebook is None else torch.full((Hk, 2), float(codebook), dtype=torch.float32,
                                                           device=dev)
        self.layers = []
        gen = torch.Generator(device=dev)
        for layer in range(layers):
            gen.manual_seed(w.seed * 100003 + 1009 * layer + 7 * rank)
            U = torch.from_numpy(S.rotation_U(w, layer).astype(np.float32)).to(dev)
            clip = torch.from_numpy(S.clip_ratios(w).astype(np.float32)).to(dev)
            prof = torch.from_numpy(S.channel_profile(w, layer).astype(np.float32)).to(dev)
            pool = torch.empty(self.pool_bytes, dtype=torch.uint8, device=dev)
            brec = (torch.empty(self.num_pages * Hk * O.BOOST_BLOCK_BYTES, dtype=torch.uint8, device=dev)
                    if boost else None)
            self._fill_history(pool, brec, U, clip, prof, gen, hist0, grp)
            kv = S.kv_tokens_torch(w, B * S.NSLOT, gen, prof, dev).view(B, S.NSLOT, Hk, 2, d).contiguous()
            q = torch.randn((B, Hq, d), generator=gen, device=dev).to(torch.bfloat16)
            new_kv = S.kv_tokens_torch(w, B, gen, prof, dev).contiguous()
            out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
            self.layers.append(dict(U=U, clip=clip, pool=pool, boost=brec, kv=kv, q=q, new_kv=new_kv, out=out))
        torch.cuda.synchronize()

    def _fill_history(self, pool, brec, U, clip, prof, gen, hist0, grp):
        """Bulk-evict each sequence's initial history (shared prefix pages
        once, by the first sharer) in chunks."""
        torch = self.torch
        seqs, poss = [], []
        for b in range(self.B):
            start = 0
            if grp is not None and grp[b] >= 0 and b != int(np.argmax(grp == grp[b])):
                start = self.w.shared_hist_tokens
            n = int(hist0[b]) - start
            if n > 0:
                seqs.append(np.full(n, b, np.int32))
                poss.append(np.arange(start, start + n, dtype=np.int32))
        if not seqs:
            return
        seq = np.concatenate(seqs)
        pos = np.concatenate(poss)
        chunk = 1 << 19
        for i in range(0, seq.size, chunk):
            n = min(chunk, seq.size - i)
            toks = S.kv_tokens_torch(self.w, n, gen, prof, self.dev).contiguous()
            sq = torch.from_numpy(seq[i:i + n]).to(self.dev)
            ps = torch.from_numpy(pos[i:i + n]).to(self.dev)
            if brec is not None:
                self.O.oscar_evict_quantize_boost(self.shape, toks, sq, ps, U, clip, pool, brec, self.table, self.B,
                                                  self.max_pages, self.num_pages)
            elif self.cb is None:
                self.O.oscar_evict_quantize(self.shape, toks, sq, ps, U, clip, pool, self.table, self.B,
                                            self.max_pages, self.num_pages)
            else:
                self.O.oscar_evict_quantize_codebook(self.shape, toks, sq, ps, U, clip, self.cb, pool, self.table,
                                                     self.B, self.max_pages, self.num_pages)

    def layer_step(self, layer: int, s: int, int2_events=None):
        O = self.O
        st = self.layers[layer]
        flat = st["kv"].view(self.B * S.NSLOT, self.Hk, 2, S.D)
        if self.boost:
            O.oscar_evict_quantize_boost(self.shape, flat, self.seqs, self.hist_before[s], st["U"], st["clip"],
                                         st["pool"], st["boost"], self.table, self.B, self.max_pages,
                                         self.num_pages, src_row=self.src_row[s], new_kv=st["new_kv"])
        elif self.cb is None:
            O.oscar_evict_quantize(self.shape, flat, self.seqs, self.hist_before[s], st["U"], st["clip"], st["pool"],
                                   self.table, self.B, self.max_pages, self.num_pages, src_row=self.src_row[s],
                                   new_kv=st["new_kv"])
        else:
            O.oscar_evict_quantize_codebook(self.shape, flat, self.seqs, self.hist_before[s], st["U"], st["clip"],
                                            self.cb, st["pool"], self.table, self.B, self.max_pages, self.num_pages,
                                            src_row=self.src_row[s], new_kv=st["new_kv"])
        if int2_events is not None:
            O.oscar_time_next_int2(*int2_events)
        if self.boost:
            O.oscar_decode_attn_boost(self.shape, st["q"], st["kv"], self.bf16_len, st["pool"], st["boost"],
                                      self.table, self.max_pages, self.num_pages, self.hist_after[s], st["U"],
                                      self.sm_scale, st["out"], self.ws)
        elif self.cb is None:
            O.oscar_decode_attn(self.shape, st["q"], st["kv"], self.bf16_len, st["pool"], self.table,
                                self.max_pages, self.num_pages, self.hist_after[s], st["U"], self.sm_scale,
                                st["out"], self.ws)
        else:
            O.oscar_decode_attn_codebook(self.shape, st["q"], st["kv"], self.bf16_len, st["pool"], self.table,
                                         self.max_pages, self.num_pages, self.hist_after[s], st["U"], self.cb,
                                         self.sm_scale, st["out"], self.ws)

    # algorithmic bytes (per layer) of the step with index s
    def hist_tokens_after(self, s: int) -> int:
        return int((self.hist0 + s + 1).sum())

    def attended_tokens(self, s: int) -> int:
        return self.hist_tokens_after(s) + self.B * S.NSLOT

    def bits_per_element(self, s: int) -> dict:
        """Stored bits per K/V element after step s: the INT2 history alone,
        and over every token of every sequence (BF16 sink + recent included),
        with shared prefix pages counted per sequence and once."""
        hist = self.hist0 + s + 1
        elems = float((hist + S.NSLOT).sum()) * 2 * S.D
        hist_bits = float(hist.sum()) * self.hist_tok_bytes * 8
        bf16_bits = float(self.B * S.NSLOT) * BF16_BYTES_PER_TOKEN_HEAD * 8
        out = {"int2_history": self.hist_tok_bytes * 8 / (2 * S.D),
               "all_tokens": (hist_bits + bf16_bits) / elems}
        if self.w.prefix_seqs:
            dup = (self.w.prefix_seqs - 1) * self.w.shared_hist_tokens * self.hist_tok_bytes * 8
            out["all_tokens_shared_pages_once"] = (hist_bits - dup + bf16_bits) / elems
        return out

    def step_bytes(self, s: int) -> float:
        hist = self.hist_tokens_after(s) * self.Hk * self.hist_tok_bytes
        bf16 = self.B * S.NSLOT * self.Hk * BF16_BYTES_PER_TOKEN_HEAD
        qo = self.B * self.Hq * S.D * (2 + 4)
        evict = self.B * self.Hk * 2 * (S.D * 2 * 2 + 48)    # read old + write new row, write codes + s/z
        return float(hist + bf16 + qo + evict)


# ---------------------------------------------------------------------------
# oracle (float64 CPU) on a bounded sample of the workload
# ---------------------------------------------------------------------------

class OracleSample:
    """The first sequences of layer 0 whose history totals about
    ``budget`` tokens, with their history written by the oracle's own
    eviction; one timed step = evict one token per sampled sequence + decode
    all their heads."""

    def __init__(self, w: S.Workload, budget: int):
        import oracle
        self.orc = oracle.get()
        ctx = S.context_lengths(w)
        hist = np.maximum(ctx - S.NSLOT, 0)
        n = 1
        while n < w.batch and hist[:n].sum() < budget:
            n += 1
        self.n = n
        self.ctx = ctx[:n]
        self.hist = hist[:n].astype(np.int32)
        self.shape = oracle.Shape(S.D, S.GROUP, S.SINK, S.RECENT, S.PAGE, w.hq, w.hk)
        rng = S.rng_for(w, 11)
        prof = S.channel_profile(w)
        cap = self.hist + 64
        self.max_pages = int((cap.max() + 63) // 64)
        rc, self.table, npages, nbytes = self.orc.pool_layout(self.shape, cap, max_pages=self.max_pages)
        self.pool = np.zeros(nbytes, np.uint8)
        self.U = S.rotation_U(w).astype(np.float32).astype(np.float64)
        self.clip = S.clip_ratios(w)
        for b in range(n):
            h = int(self.hist[b])
            toks = S.kv_tokens(w, h, rng, prof)
            self.orc.evict(self.shape, toks, np.full(h, b, np.int32), np.arange(h, dtype=np.int32), self.U,
                           self.clip, self.pool, self.table, self.max_pages)
        self.kv = S.kv_tokens(w, n * S.NSLOT, rng, prof).reshape(n, S.NSLOT, w.hk, 2, S.D)
        self.new = S.kv_tokens(w, n, rng, prof)
        self.q = S.queries(w, rng, n)
        self.bf16_len = np.full(n, S.NSLOT, np.int32)
        self.threads = self.orc.num_threads()

    def step(self):
        rows = (np.arange(self.n) * S.NSLOT + S.SINK).astype(np.int32)
        flat = self.kv.reshape(self.n * S.NSLOT, -1, 2, S.D)
        pool = self.pool.copy()   # keep the sample's state fixed across steps
        self.orc.evict(self.shape, flat, np.arange(self.n, dtype=np.int32), self.hist, self.U, self.clip, pool,
                       self.table, self.max_pages, src_row=rows)
        self.orc.decode(self.shape, self.q, self.kv, self.bf16_len, pool, self.table, self.max_pages,
                        self.hist + 1, self.U, 1.0 / math.sqrt(S.D))
        return int((self.hist + 1).sum() + self.n * S.NSLOT)

    def time(self, steps: int, warmup: int = 0):
        for _ in range(warmup):
            self.step()
        t0 = time.perf_counter()
        toks = 0
        for _ in range(steps):
            toks += self.step()
        dt = time.perf_counter() - t0
        return toks / dt, dt

    def time_one_thread(self):
        """One step on a single host thread (the same sample)."""
        self.orc.set_num_threads(1)
        try:
            return self.time(1, 0)
        finally:
            self.orc.set_num_threads(self.threads)

    def describe(self) -> str:
        return (f"layer 0 of the workload: sequences 0..{self.n - 1} (history {int(self.hist.sum())} tokens, "
                f"{self.shape.num_q_heads} query / {self.shape.num_kv_heads} KV heads), one eviction per "
                f"sequence + decode of all heads per step, float64")


def cpu_info() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "processor\t: 0")) and ":" in line:
                    if "model name" in line.lower():
                        return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, rank: int, world: int) -> None:
    if rank != 0:
        return
    w = S.WORKLOADS[args.workload]
    samp = OracleSample(w, reference_budget(args))
    tps, dt = samp.time(args.steps, args.warmup)
    ms = dt / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": UNIT, "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.layers or w.layers),
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": samp.threads, "kind": "oracle",
                         "sample": samp.describe(), "cpu": cpu_info()},
        "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w: S.Workload, layers: int, quant_group: int = 32, codebook: float | None = None,
              boost: bool = False) -> dict:
    ctx = {"fixed": f"{w.ctx_lo}", "uniform": f"uniform[{w.ctx_lo},{w.ctx_hi}]",
           "loguniform": f"loguniform[{w.ctx_lo},{w.ctx_hi}]"}[w.ctx_kind]
    cfg = {"workload": w.name, "batch_per_gpu": w.batch, "layers": layers, "q_heads": w.hq, "kv_heads": w.hk,
           "head_dim": S.D, "context": ctx, "sink": S.SINK, "recent": S.RECENT, "quant_group": quant_group,
           "page": S.PAGE, "page_table": "shuffled" if w.shuffled else "contiguous",
           "kv_values": w.dist, "l2": "inputs larger than L2 (a distinct pool per layer)",
           "parallelism": "replicas (independent sequences per GPU)"}
    if codebook is not None:
        cfg["levels"] = f"Lloyd-Max {{0, {codebook:g}, {3 - codebook:g}, 3}}"
    if boost:
        cfg["k_boost"] = "8 of 128 K positions per token at 4 bits (16-byte record)"
    if w.prefix_seqs:
        cfg["prefix_sharing"] = f"{w.prefix_seqs} sequences share a {w.prefix_tokens}-token prefix"
    return cfg


# One-layer side records of a 1-GPU run: the INT2 kernel's roofline fraction
# on the other single-GPU workloads, measured in the same process after the
# main timed region.  Each pool is larger than L2 (qwen3_4b's 0.2 GB layer
# is rotated over four layers, so consecutive steps read different pools).
SIDE_RECORDS = (("gate", 1), ("qwen3_4b", 4), ("qwen3_32b", 1), ("stress", 1))


def side_record(name: str, layers: int, steps: int, warmup: int, peak_gbs: float) -> dict:
    """INT2 launch time (CUDA events on the launching stream, every launch)
    and whole-step time of a short run of workload ``name``."""
    import torch
    w = S.WORKLOADS[name]
    st = GpuState(w, layers, warmup + steps, 0)
    stream = torch.cuda.current_stream()
    for s in range(warmup):
        for layer in range(layers):
            st.layer_step(layer, s)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps * layers)]
    for a, b in evs:   # materialise the events (torch creates them at their first record)
        a.record(stream)
        b.record(stream)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(steps):
        for layer in range(layers):
            st.layer_step(layer, warmup + k, evs[k * layers + layer])
    stop.record(stream)
    torch.cuda.synchronize()
    int2_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    step_ms = start.elapsed_time(stop) / steps
    int2_bytes = statistics.mean(st.hist_tokens_after(warmup + k) * st.Hk * st.hist_tok_bytes for k in range(steps))
    step_bytes = statistics.mean(st.step_bytes(warmup + k) for k in range(steps)) * layers
    att = statistics.mean(st.attended_tokens(warmup + k) for k in range(steps)) * layers
    del st
    torch.cuda.empty_cache()
    int2_gbs = int2_bytes / (int2_ms * 1e-3) / 1e9
    step_gbs = step_bytes / (step_ms * 1e-3) / 1e9
    return {"workload": name, "layers": layers, "batch": w.batch, "q_heads": w.hq, "kv_heads": w.hk,
            "int2_launch_ms": int2_ms, "int2_bytes_per_launch": int2_bytes, "int2_gbs": int2_gbs,
            "int2_frac": int2_gbs / peak_gbs, "step_ms": step_ms, "step_algorithmic_gbs": step_gbs,
            "step_frac": step_gbs / peak_gbs, "context_tokens_per_s": att / (step_ms * 1e-3),
            "steps": steps, "warmup": warmup}


def run_oscar(args, rank: int, world: int, local: int) -> None:
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    from bit_kv_cache_evict_gb300 import build as Bld
    if local == 0:     # one rank per node compiles (if the library is stale); the others then find it built
        Bld.build()
    barrier(world)
    Bld.build()
    w = S.WORKLOADS[args.workload]
    L = args.layers or w.layers
    K, W = args.steps, args.warmup
    e2e_steps = 0 if args.no_e2e else K
    total_steps = W + K + e2e_steps
    t0 = time.time()
    st = GpuState(w, L, total_steps, rank, args.quant_group, args.codebook, args.boost)
    setup_s = time.time() - t0
    stream = torch.cuda.current_stream()

    for s in range(W):
        for layer in range(L):
            st.layer_step(layer, s)
    torch.cuda.synchronize()
    barrier(world)

    # int2-kernel events around the launches of three layers per step in the
    # timed region (an event between two kernels ends their programmatic
    # overlap, so the other layers run without them; every layer carries the
    # same history lengths).  The end-to-end region records the same events
    # on the same layers, so that the two regions carry the same
    # instrumentation.
    stride = max(1, L // 3)
    timed_layers = [layer for layer in range(L) if layer % stride == 0][:3]
    evs = {(k, layer): (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for k in range(K) for layer in timed_layers}
    e2e_evs = {(k, layer): (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for k in range(e2e_steps) for layer in timed_layers}
    for a, b in list(evs.values()) + list(e2e_evs.values()):   # materialise the events
        a.record(stream)
        b.record(stream)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(K):
        s = W + k
        for layer in range(L):
            st.layer_step(layer, s, evs.get((k, layer)))
    stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    t_ms = start.elapsed_time(stop)
    int2_ms = [a.elapsed_time(b) for a, b in evs.values()]

    att = sum(st.attended_tokens(W + k) for k in range(K)) * L
    value, t_ms_max = aggregate(t_ms, att, world, dev)
    ms_per_step = t_ms_max / K
    step_bytes = sum(st.step_bytes(W + k) for k in range(K)) * L / K
    hist_bytes = [st.hist_tokens_after(W + k) * st.Hk * st.hist_tok_bytes for k in range(K)]
    int2_avg_ms = statistics.mean(int2_ms)
    int2_median_ms = statistics.median(int2_ms)
    int2_bytes = statistics.mean(hist_bytes)
    peaks = load_peaks()
    achieved = int2_bytes / (int2_avg_ms * 1e-3) / 1e9

    # end to end through the C ABI from pinned host buffers: per layer, copy
    # the step's query and new token in, run the step, copy the output out.
    # When a layer's kernels run long enough to hide the extra host work
    # (0.2 ms), the copies run on two copy streams ordered with events, so
    # that the next layer's upload and the previous layer's download overlap
    # the current layer's kernels (as a serving loop would); otherwise they
    # run in the compute stream.
    e2e = None
    overlap_copies = ms_per_step / L > 0.2
    if e2e_steps:
        hq = [torch.empty_like(l["q"], device="cpu").pin_memory() for l in st.layers]
        hn = [torch.empty_like(l["new_kv"], device="cpu").pin_memory() for l in st.layers]
        ho = [torch.empty_like(l["out"], device="cpu").pin_memory() for l in st.layers]
        for layer in range(L):
            hq[layer].copy_(st.layers[layer]["q"])
            hn[layer].copy_(st.layers[layer]["new_kv"])
        torch.cuda.synchronize()
        barrier(world)
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(L)]     # layer's inputs uploaded
        ev_done = [torch.cuda.Event() for _ in range(L)]   # layer's step finished: inputs free, output ready
        ev_out = [torch.cuda.Event() for _ in range(L)]    # layer's output downloaded
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for ev in ev_done + ev_out:
            ev.record(stream)
        for k in range(e2e_steps):
            s = W + K + k
            for layer in range(L):
                lay = st.layers[layer]
                if not overlap_copies:
                    lay["q"].copy_(hq[layer], non_blocking=True)
                    lay["new_kv"].copy_(hn[layer], non_blocking=True)
                    st.layer_step(layer, s, e2e_evs.get((k, layer)))
                    ho[layer].copy_(lay["out"], non_blocking=True)
                    continue
                with torch.cuda.stream(h2d_s):
                    h2d_s.wait_event(ev_done[layer])
                    lay["q"].copy_(hq[layer], non_blocking=True)
                    lay["new_kv"].copy_(hn[layer], non_blocking=True)
                    ev_in[layer].record(h2d_s)
                stream.wait_event(ev_in[layer])
                stream.wait_event(ev_out[layer])
                st.layer_step(layer, s, e2e_evs.get((k, layer)))
                ev_done[layer].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(ev_done[layer])
                    ho[layer].copy_(lay["out"], non_blocking=True)
                    ev_out[layer].record(d2h_s)
        stream.wait_stream(d2h_s)
        e1.record(stream)
        torch.cuda.synchronize()
        e_att = sum(st.attended_tokens(W + K + k) for k in range(e2e_steps)) * L
        e_value, e_ms = aggregate(e0.elapsed_time(e1), e_att, world, dev)
        h2d = L * (st.layers[0]["q"].numel() * 2 + st.layers[0]["new_kv"].numel() * 2)
        d2h = L * st.layers[0]["out"].numel() * 4
        e2e = {"value": e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / e2e_steps,
               "copies": "overlapped on copy streams" if overlap_copies else "in the compute stream"}

    cpu = None
    if rank == 0 and not args.no_cpu:
        samp = OracleSample(w, args.cpu_tokens)
        tps, dt = samp.time(args.cpu_steps, 0)
        tps1, dt1 = samp.time_one_thread()
        cpu = {"value": tps, "unit": UNIT, "cores": samp.threads, "kind": "oracle",
               "sample": f"{args.cpu_steps} steps of " + samp.describe(), "seconds": dt, "cpu": cpu_info(),
               "value_1_thread": tps1, "seconds_1_thread": dt1}

    # one-layer side records (1-GPU runs only): the 32K batch-64 layer the
    # INT2 roofline target is stated on, and the other single-GPU shapes
    bpe = st.bits_per_element(W + K - 1)
    side = None
    if world == 1 and not args.no_side:
        del st
        torch.cuda.empty_cache()
        side = {}
        for name, layers in SIDE_RECORDS:
            if name != w.name:
                side[name] = side_record(name, layers, 20, 3, peaks["hbm_gbs"])

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int2 codes x fp16 hi/lo operands (q', p*s) on tensor cores, fp32 accumulate", "data": "synthetic",
            "config": config_of(w, L, args.quant_group, args.codebook, args.boost),
            "decode_tokens_per_s": world * w.batch * K / (t_ms_max / 1e3),
            "bits_per_element": bpe,
            "step_algorithmic_gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
            "step_frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "roofline": {"kernel": "int2_kernel (split-K INT2 history attention)", "bound": "hbm",
                         "achieved": achieved, "peak": peaks["hbm_gbs"], "peak_source": peaks["source"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": int2_traffic(w.name if args.quant_group == 32 and args.codebook is None and not args.boost
                                                else "", int2_bytes),
                         "bytes_per_launch": int2_bytes, "launch_ms": int2_avg_ms,
                         "launch_ms_median": int2_median_ms,
                         "share_of_step": int2_avg_ms * L / ms_per_step,
                         "launches_timed": len(int2_ms)},
            "cpu_baseline": cpu, "e2e": e2e,
            "gate": side.get("gate") if side else None,
            "frac_by_workload": ({w.name: achieved / peaks["hbm_gbs"],
                                  **{k: v["int2_frac"] for k, v in side.items()}} if side else None),
            "side_records": side,
            "gpu_launches": K * L * 5,
            "clocks": clk, "setup_s": setup_s,
        }
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


CALIB_CONFIG = {"workload": "qwen3_8b_calibration", "query_tokens": 1024, "query_heads": 32, "kv_heads": 8,
                "tokens": 2048, "head_dim": S.D}


def run_calibrate(args, rank: int) -> None:
    """Offline rotation calibration of one layer (Qwen3-8B heads): attention
    outputs of 1024 calibration query tokens x 32 heads over 2048 tokens,
    the K and V covariances of the 8 KV groups and their eigenvectors.  The
    metric is the time of one calibration; the clip-ratio search with the
    calibrated U is timed beside it, and the float64 oracle's rotation
    calibration runs once on the same inputs for cpu_baseline."""
    import torch
    from bit_kv_cache_evict_gb300 import build as B
    from bit_kv_cache_evict_gb300 import oscar as O
    if rank != 0:
        return
    B.build()
    cfg = CALIB_CONFIG
    nq, nt, hq, hk = cfg["query_tokens"], cfg["tokens"], cfg["query_heads"], cfg["kv_heads"]
    qb, kvb = S.calibration_inputs(1800, nq, nt, hq, hk)
    sh = O.make_shape(hq, hk)
    dev = torch.device("cuda", 0)
    q_t = torch.from_numpy(qb.view(np.int16)).to(dev).view(torch.bfloat16)
    kv_t = torch.from_numpy(kvb.view(np.int16)).to(dev).view(torch.bfloat16)
    U_t = torch.empty((hk, 2, S.D, S.D), dtype=torch.float32, device=dev)
    ws = torch.zeros(O.oscar_calibrate_workspace_bytes(sh, nq), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(S.D)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        O.oscar_calibrate_rotation(sh, q_t, kv_t, scale, U_t, ws, dev_status=status, stream=stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(0)
    clocks.start()
    for a, b in ev:
        a.record(stream)
        O.oscar_calibrate_rotation(sh, q_t, kv_t, scale, U_t, ws, dev_status=status, stream=stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    # clip-ratio search with the calibrated U (11 candidates, 0.50 .. 1.00)
    grid_np = np.round(np.arange(0.50, 1.0001, 0.05), 4).astype(np.float32)
    grid_t = torch.from_numpy(grid_np).to(dev)
    clip_t = torch.empty((hk, 2), dtype=torch.float32, device=dev)
    cws = torch.zeros(O.oscar_calibrate_clip_workspace_bytes(sh, nt, int(grid_np.size)), dtype=torch.uint8,
                      device=dev)
    for _ in range(3):
        O.oscar_calibrate_clip(sh, kv_t, U_t, grid_t, clip_t, workspace=cws, stream=stream)
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in cev:
        a.record(stream)
        O.oscar_calibrate_clip(sh, kv_t, U_t, grid_t, clip_t, workspace=cws, stream=stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    clip_ms = statistics.median(a.elapsed_time(b) for a, b in cev)
    flops = 2.0 * nq * hq * nt * S.D * 2          # logits and weighted sum of the attention outputs
    from oracle import calibrate as OC
    q64 = S.bf16_to_f32(qb).astype(np.float64)
    kv64 = S.bf16_to_f32(kvb).astype(np.float64)
    t0 = time.perf_counter()
    OC.calibrate(q64, kv64, scale)
    cpu_s = time.perf_counter() - t0
    print(json.dumps({
        "metric": "offline rotation calibration time per layer", "value": ms, "unit": "ms",
        "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "dtype": "f32", "data": "synthetic", "config": cfg, "vs_baseline": None,
        "status": int(status.item()), "attention_gflop": flops / 1e9,
        "clip_search_ms": clip_ms, "clip_candidates": int(grid_np.size),
        "clips_chosen": sorted(set(float(c) for c in clip_t.cpu().numpy().ravel())),
        "cpu_baseline": {"value": cpu_s * 1e3, "unit": "ms", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "the same calibration, float64 numpy (BLAS threads)"},
        "clocks": clk}))


def main():
    args = parse_args()
    rank, world, local = dist_info()
    if args.calibrate:
        run_calibrate(args, rank)
        return
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_oscar(args, rank, world, local)


if __name__ == "__main__":
    main()
