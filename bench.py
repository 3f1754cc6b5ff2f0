#!/usr/bin/env python
"""Decode-step benchmark: KV GB/s of quantized-cache decode attention with the fused meter.

A step is one decode step of the whole model: for every layer, append the new
token's K/V and run the decode attention over [shared prefix ++ live suffix]
(one kvq_decode_attn_append call, which does the append inside the decode
kernel; --separate-append times kvq_append + kvq_decode_attn instead); then
kvq_meter finalises the meter of every (layer, sequence, head).
The default workload is the Qwen3-8B-shaped cartridge decode (batch 16, 36
layers, 8 kv heads, 32 q heads, 632-token K16/V8 shared prefix with a x10 sink,
11,996-token BF16 live suffix = 12,628 attended tokens).

value = algorithmic bytes of the step (every live token's K, V, scales and
witness once per (layer, kv head); the shared prefix once per layer) / step
time.  Inputs are resident in HBM before the timed region and larger than L2
(no flush needed).  `e2e` is the same metric through the public API with host
buffers: pinned host->device copies of the step's queries and new K/V, and a
device->host read of the outputs and meter, inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "decode-attn KV GB/s (% of GB300 HBM peak) with meter on; attended tok/s"
SM_SCALE = float(np.float32(1.0 / math.sqrt(128)))
# device sources of decode_split_kernel (the roofline kernel): its recorded DRAM traffic is valid only
# for the code it was captured from (comments and blank lines aside)
# and for its launch plan (decode.cu picks the warps per CTA, the stage count and the split plan) and build
# flags (build.py)
KERNEL_SOURCES = ["quantized_kv_cache_kvq_gb300/csrc/decode_kernel.cuh", "quantized_kv_cache_kvq_gb300/csrc/kvq_common.cuh",
                  "quantized_kv_cache_kvq_gb300/csrc/decode_instances.inc", "quantized_kv_cache_kvq_gb300/csrc/decode.cu",
                  "quantized_kv_cache_kvq_gb300/build.py"]
# the second workload the default run times after the headline (same steps and warm-up)
SECOND_WORKLOAD = "int8_7b_certified"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="qwen3_8b_cartridge", choices=sorted(W.WORKLOADS))
    p.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--eager", action="store_true", help="launch the step eagerly instead of replaying a CUDA graph")
    p.add_argument("--value-side", action="store_true",
                   help="meter the value side too (value witness read, output-error bound from kvq_meter)")
    p.add_argument("--meter-off", action="store_true",
                   help="decode without the meter (no witness read, no kvq_meter): the meter's marginal cost, as "
                        "time per step against the default")
    p.add_argument("--shapes", action="store_true",
                   help="alternative bound shapes too (two-sided meter and det-tanh from kvq_meter)")
    p.add_argument("--gate", action="store_true",
                   help="gate support too: per-page contributions from kvq_decode_attn_ex and a kvq_gate plan per layer")
    p.add_argument("--bypass", type=int, default=0, metavar="M",
                   help="INT8 keys: M massive RoPE pairs per (layer, kv head) injected (x30) and kept in fp16 by the "
                        "fixed-channel bypass")
    p.add_argument("--int8-groups", action="store_true",
                   help="INT8 keys and values with one fp16 scale per token per 32-channel group (WitCert 6.2.3, "
                        "G_c = 32) instead of one per token")
    p.add_argument("--separate-append", action="store_true",
                   help="kvq_append + kvq_decode_attn per layer instead of the fused kvq_decode_attn_append")
    p.add_argument("--layers", type=int, default=0, help="override layer count (profiling only; not a bench line)")
    p.add_argument("--batch", type=int, default=0,
                   help="override the batch (the first sequences of the workload; profiling only, not a bench line)")
    p.add_argument("--no-second", action="store_true",
                   help=f"time only the headline workload (the default run also times {SECOND_WORKLOAD} after it)")
    p.add_argument("--resident-layers", type=int, default=0,
                   help="keep only this many layers' caches in HBM and run every layer call on cache l %% R "
                        "(for workloads whose caches exceed HBM; each call still streams a full layer)")
    return p.parse_args()


CODE_BYTES = {"bf16": 2, "e4m3": 1, "e4m3s": 1, "int8": 1, "int8g32": 1}
SCALE_BYTES = {"bf16": 0, "e4m3": 0, "e4m3s": 2, "int8": 2, "int8g32": 8}   # fp16 scales per token per kv head


def token_head_bytes(k_fmt, v_fmt, meter=True, value_side=False, bypass=0) -> int:
    """Bytes one token of one kv head costs the decode: K and V codes, fp16 scales, 32-byte witness
    (+ the 4-byte value witness with the value side of the output bound, + the fp16 key outlier tile of
    the fixed-channel bypass: 8 columns for up to 4 pairs, 16 for up to 8)."""
    return (128 * (CODE_BYTES[k_fmt] + CODE_BYTES[v_fmt]) + SCALE_BYTES[k_fmt] + SCALE_BYTES[v_fmt] + 32 * meter
            + 4 * value_side + (0 if not bypass else 16 if bypass <= 4 else 32))


def step_bytes(w, lens, value_side=False, meter=True) -> int:
    """Algorithmic bytes of one decode step: live tokens once per (layer, kv head), the prefix once per layer."""
    live = int(np.sum(lens)) * token_head_bytes(w.k_fmt, w.v_fmt, meter=meter, value_side=value_side,
                                                bypass=w.bypass_pairs)
    pre = (w.prefix_len * token_head_bytes(w.prefix_k_fmt, w.prefix_v_fmt, meter=meter, value_side=value_side)
           if w.prefix_len else 0)
    return w.n_layers * w.n_kv_heads * (live + pre)


def code_only(text: str) -> str:
    """C++ source without comments and blank lines: what decides the compiled kernel (an edit of a comment
    leaves the recorded counters valid)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_hash(read=None) -> str:
    """Fingerprint of the decode kernel's code; ``read(path)`` returns a source's text (default: the working
    tree)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(code_only(text).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Issue roofline of a path bound by integer arithmetic and instruction issue (the INT8-dithered decode
# regenerates every element's dither with Philox4x32-10): each SM has 4 schedulers that each issue at most
# one warp-instruction per clock.  The SM count is the device's (cudaDevAttrMultiProcessorCount through
# torch) and the clock its maximum SM clock as nvidia-smi reports it during the run; the GB300 figures below
# (152 SMs, 2070 MHz) stand in only where the device cannot be asked (CPU tests).
SCHEDULERS_PER_SM = 4
FALLBACK_SMS, FALLBACK_MAX_SM_MHZ = 152, 2070.0


def issue_peak_winst_per_s(sms: int, sm_mhz: float) -> float:
    return sms * SCHEDULERS_PER_SM * sm_mhz * 1e6


def max_sm_mhz(clocks: dict) -> tuple[float, str]:
    """The SM clock ceiling for the issue peak: nvidia-smi's clocks.max.sm sampled during the run, else the
    measured figure in MEASURED_PEAKS.json, else the GB300 maximum."""
    if clocks and clocks.get("sm_max_mhz"):
        return float(clocks["sm_max_mhz"]), "nvidia-smi clocks.max.sm during the run"
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("sm_max_mhz"):
            return float(d["sm_max_mhz"]), "MEASURED_PEAKS.json sm_max_mhz"
    return FALLBACK_MAX_SM_MHZ, "GB300 maximum SM clock (fallback)"


def runs_a_variant(args, w) -> bool:
    """True when a switch or the workload runs another decode instance than the plain one the ncu records
    describe (value side, bound shapes, gate support, key outlier bypass, meter off, group scales)."""
    return bool(args.value_side or args.shapes or args.gate or w.bypass_pairs or args.meter_off
                or getattr(args, "int8_groups", False))


def traffic_record(workload: str, variant: bool = False):
    """The ncu record of the plain decode kernel of a workload; none for variants (value side, bound
    shapes, gate support, bypass: other kernel instances or extra outputs)."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if variant:
        return None
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(workload)
    if not rec or rec.get("kernel_hash") != kernel_hash():
        return None
    return rec


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"kvq_clocks_{os.getpid()}_{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def wait_started(self, limit_s: float = 3.0):
        """Return once nvidia-smi has written its first sample (or after ``limit_s``)."""
        t0 = time.perf_counter()
        while self.proc is not None and time.perf_counter() - t0 < limit_s:
            self.fh.flush()
            if os.path.exists(self.path) and os.path.getsize(self.path) > 0:
                return
            time.sleep(0.02)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sms.append(float(parts[0]))
                    mx = float(parts[1])
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------------------------------------ GPU arm
class Model:
    """All layers' caches of one workload, filled through kvq_append, plus the step's buffers."""

    def __init__(self, w, device, seed_base=0, n_layers=None, resident=0, value_side=False, shapes=False,
                 gate=False, meter=True, lens=None):
        self.separate_append = False
        self.meter_on = meter
        self.value_side = value_side
        self.gate = gate
        import torch

        import quantized_kv_cache_kvq_gb300 as kvq

        self.kvq, self.torch, self.w, self.dev = kvq, torch, w, device
        self.L = n_layers or w.n_layers
        self.R = min(self.L, resident) if resident else self.L   # caches resident in HBM
        B, Hkv, Hq = w.batch, w.n_kv_heads, w.n_q_heads
        self.lens = W.seq_lengths(w) if lens is None else np.asarray(lens, dtype=np.int64)
        assert len(self.lens) == B
        pages = (self.lens + W.PAGE - 1) // W.PAGE
        bt = W.block_table_for(w, self.lens)
        self.num_pages = int(pages.sum())
        self.bt = torch.from_numpy(bt).to(device)
        self.seq_lens = torch.from_numpy(self.lens.astype(np.int32)).to(device)
        # the step's new token sits at the last position of every sequence
        last = self.lens - 1
        self.new_slots = torch.from_numpy(np.array([W.slot_mapping(bt, s, [last[s]])[0] for s in range(B)],
                                                   dtype=np.int32)).to(device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        g = torch.Generator(device=device)
        self.caches, self.prefixes = [], []
        total = int(self.lens.sum())
        pos = torch.cat([torch.arange(w.prefix_len, w.prefix_len + int(n), device=device) for n in self.lens])
        slots = torch.cat([torch.from_numpy(W.slot_mapping(bt, s, np.arange(n))) for s, n in
                           enumerate(self.lens)]).to(device)
        for l in range(self.R):
            g.manual_seed(W.unit_seed(w, 100_000 + 1000 * seed_base + l))
            opairs = torch.from_numpy(W.bypass_pair_table(w, l)).to(device) if w.bypass_pairs else None
            c = kvq.PagedCache(w.k_fmt, w.v_fmt, Hkv, self.num_pages, layer=l,
                               seed=(0x5EED << 20) + 97 * l + seed_base, value_witness=value_side,
                               outlier_pairs=opairs)
            chunk = 1 << 18
            for a in range(0, total, chunk):
                b = min(total, a + chunk)
                k, v = W.gen_tokens_gpu(w, l, pos[a:b], g, device)
                kvq.append(c, k, v, slots[a:b].contiguous(), self.err)
            self.caches.append(c)
            if w.prefix_len:
                p = kvq.PagedCache(w.prefix_k_fmt, w.prefix_v_fmt, Hkv, (w.prefix_len + 15) // 16, layer=l,
                                   seed=(0xCA47 << 20) + l, value_witness=value_side)
                k, v = W.gen_tokens_gpu(w, l, torch.arange(w.prefix_len, device=device), g, device, sink=True)
                kvq.append(p, k, v, torch.arange(w.prefix_len, dtype=torch.int32, device=device), self.err)
                self.prefixes.append(p)
            else:
                self.prefixes.append(None)
        # the step's inputs: queries and new K/V of every layer
        qd = torch.bfloat16 if w.q_dtype == "bf16" else torch.float32
        g.manual_seed(W.unit_seed(w, 200_000 + seed_base))
        self.q = torch.randn((self.L, B, Hq, 128), generator=g, device=device).to(qd).contiguous()
        self.k_new = torch.randn((self.L, B, Hkv, 128), generator=g, device=device)
        self.v_new = torch.randn((self.L, B, Hkv, 128), generator=g, device=device)
        self.out = torch.empty((self.L, B, Hq, 128), device=device)
        self.state = torch.empty((self.L, B, Hq, 8), device=device)
        self.meter_a = torch.empty((self.L, B, Hq), device=device)
        self.raw_a = torch.empty((self.L, B, Hq), device=device)
        self.cert_b = torch.empty((self.L, B, Hq), device=device) if w.tier_b else None
        self.counts = torch.zeros(4, dtype=torch.int32, device=device)
        self.ranking = (torch.empty((B, self.L * Hq), dtype=torch.int32, device=device)
                        if w.n_outliers else None)
        self.ws = torch.empty(kvq.decode_workspace_size(B, Hkv, Hq), dtype=torch.uint8, device=device)
        tiers = (kvq.TIER_A | (kvq.TIER_B if w.tier_b else 0) | (kvq.TIER_V if value_side else 0)
                 | (kvq.TIER_S if shapes else 0))
        self.out_bound = torch.empty((self.L, B, Hq), device=device) if value_side else None
        self.two_sided = torch.empty((self.L, B, Hq), device=device) if shapes else None
        self.det_tanh = torch.empty((self.L, B, Hq), device=device) if shapes else None
        # gate support: per-page log contributions to A - 1 of every (sequence, query head), and the greedy
        # page-in plan's length per (layer, sequence, query head)
        self.contrib = self.n_page_in = None
        if gate:
            stride = int(pages.max()) + (w.prefix_len + W.PAGE - 1) // W.PAGE
            self.contrib = torch.empty((self.L, B, Hq, stride), device=device)
            self.n_page_in = torch.empty((self.L, B, Hq), dtype=torch.int32, device=device)
        self.mp = kvq.meter_params(tiers, w.n_layers, Hq, w.n_steps, w.delta_req, w.tau)
        torch.cuda.synchronize()
        if self.err.item() != 0:
            raise RuntimeError(f"append reported {kvq.STATUS.get(self.err.item())}")

    def step(self, q=None, k_new=None, v_new=None, events=None):
        kvq, w = self.kvq, self.w
        q = self.q if q is None else q
        k_new = self.k_new if k_new is None else k_new
        v_new = self.v_new if v_new is None else v_new
        for l in range(self.L):
            c = l % self.R
            kw = dict(prefix=self.prefixes[c], prefix_len=w.prefix_len, sm_scale=SM_SCALE,
                      meter=self.mp if self.meter_on else None, meter_state=self.state[l] if self.meter_on else None,
                      err=self.err)
            if self.separate_append:
                kvq.append(self.caches[c], k_new[l], v_new[l], self.new_slots, self.err)
            if events is not None:
                events[l][0].record()
                kvq.debug_time_decode(events[l][2], events[l][3])
            if self.gate:
                kvq.decode_attn_ex(self.caches[c], q[l], self.bt, self.seq_lens, self.out[l], self.ws, k_new=k_new[l],
                                   v_new=v_new[l], page_log_contrib=self.contrib[l], **kw)
            elif self.separate_append:
                kvq.decode_attn(self.caches[c], q[l], self.bt, self.seq_lens, self.out[l], self.ws, **kw)
            else:
                kvq.decode_attn_append(self.caches[c], k_new[l], v_new[l], q[l], self.bt, self.seq_lens, self.out[l],
                                       self.ws, **kw)
            if events is not None:
                events[l][1].record()
                kvq.debug_time_decode(None, None)
            if self.gate:
                kvq.gate(self.contrib[l], self.state[l], self.seq_lens, w.prefix_len, w.tau, self.n_page_in[l])
        if not self.meter_on:
            return
        kvq.meter(self.state, self.L, w.batch, w.n_q_heads, self.mp, self.meter_a, self.raw_a, self.counts,
                  cert_b=self.cert_b, ranking=self.ranking, out_bound=self.out_bound, two_sided=self.two_sided,
                  det_tanh=self.det_tanh)

    def launches_per_step(self) -> int:
        meter = (1 + (1 if self.ranking is not None else 0)) if self.meter_on else 0
        return self.L * (3 if self.separate_append else 2) + meter + (self.L if self.gate else 0)


def rank_share(w, rank: int, world: int):
    """This rank's sequences of the job: the global batch is world x w.batch sequences (weak scaling: the
    per-GPU work stays one workload's batch), assigned to ranks by ``dist.shard_sequences`` (balanced
    attended tokens, deterministic).  Returns (the rank's workload, its live lengths, its global sequence
    indices).  The units are independent, so no collective touches the data path."""
    from quantized_kv_cache_kvq_gb300.dist import shard_sequences

    if world == 1:
        lens = W.seq_lengths(w)
        return w, lens, np.arange(len(lens))
    lens_g = W.seq_lengths(W.reduced(w, batch=w.batch * world))
    idx = shard_sequences(lens_g, world, prefix_len=w.prefix_len)[rank]
    return W.reduced(w, batch=len(idx)), lens_g[idx], idx


def job_totals(per_rank, counts, world: int, cpu_group=None):
    """Sum the ranks' per-step figures (step bytes, attended tokens, ...) and meter counters over the ranks
    (host-side, after the timed region)."""
    vals = [float(x) for x in np.atleast_1d(per_rank)]
    if world == 1:
        return vals, [int(c) for c in counts]
    import torch
    import torch.distributed as dist

    from quantized_kv_cache_kvq_gb300.dist import reduce_meter_counts

    t = torch.tensor(vals, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=cpu_group)
    return t.tolist(), [int(c) for c in reduce_meter_counts(counts, group=cpu_group).tolist()]


def run_gpu(args, w, init_dist=True):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cpu_group = None
    if world > 1:
        import torch.distributed as dist

        if init_dist and not dist.is_initialized():
            dist.init_process_group("nccl")
        cpu_group = dist.new_group(backend="gloo")  # host-side sums (meter counters, step bytes)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import quantized_kv_cache_kvq_gb300 as kvq

    kvq.load()
    resident = args.resident_layers
    if not resident and w.name == "ragged_paged":
        resident = 4  # 36 layers of this workload need ~413 GB of cache: rotate 4 resident layers
    if args.meter_off and (args.value_side or args.shapes or args.gate):
        raise SystemExit("--meter-off excludes the meter's extensions")
    wr, lens, _ = rank_share(w, rank, world)
    m = Model(wr, dev, seed_base=rank, n_layers=args.layers or None, resident=resident, value_side=args.value_side,
              shapes=args.shapes, gate=args.gate, meter=not args.meter_off, lens=lens)
    m.separate_append = args.separate_append
    per_step_bytes = step_bytes(wr, m.lens, value_side=args.value_side, meter=not args.meter_off) * m.L // w.n_layers
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        m.step()
    barrier()
    graph = None
    if not args.eager:
        # the whole step (append + decode + merge per layer, meter) as one CUDA graph
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            m.step()
        for _ in range(args.warmup):
            graph.replay()
        barrier()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # the sampler needs a moment to start; untimed steps keep the GPU loaded meanwhile, so the samples
        # bracket the timed region under the same load
        clk.wait_started()
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 0.3:
            graph.replay() if graph is not None else m.step()
            torch.cuda.synchronize()
        barrier()
        start.record()
        for s in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                m.step()
        stop.record()
        barrier()
    ms = start.elapsed_time(stop)
    # per-launch duration of the decode kernel (the dominant one): CUDA events the library records on
    # the call's stream right before and after that kernel's launch (kvq_debug_time_decode), eager
    # steps; plus events around each whole call (append + decode + merge)
    n_ev = max(1, min(args.steps, 20))
    events = [[tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(m.L)]
              for _ in range(n_ev)]
    for st in events:
        for e4 in st:
            for e in e4:
                e.record()  # creates the underlying CUDA event
    torch.cuda.synchronize()
    barrier()
    for s in range(n_ev):
        m.step(events=events[s])
    barrier()
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    if m.err.item() != 0:
        raise RuntimeError(f"device error {kvq.STATUS.get(m.err.item())}")
    ms_step = ms / args.steps
    rank_attended = float(np.sum(m.lens) + w.prefix_len * wr.batch) * m.L * w.n_kv_heads
    (job_bytes, attended), job_counts = job_totals([per_step_bytes, rank_attended], m.counts.cpu().tolist(), world,
                                                   cpu_group)
    value = job_bytes / (ms_step * 1e-3) / 1e9
    layer_ms = [e[2].elapsed_time(e[3]) for st in events for e in st]
    call_ms = [e[0].elapsed_time(e[1]) for st in events for e in st]
    layer_bytes = per_step_bytes / m.L
    achieved = layer_bytes / (statistics.mean(layer_ms) * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    tr = traffic_record(w.name, variant=runs_a_variant(args, w))
    res = dict(value=value, ms_step=ms_step, achieved=achieved, graph=graph is not None, layer_ms_mean=statistics.mean(layer_ms),
               call_ms_mean=statistics.mean(call_ms),
               layer_ms_median=statistics.median(layer_ms), peak=peak, peak_kind=peak_kind, traffic=tr,
               clocks=clk.summary(), launches=m.launches_per_step() * args.steps, attended=attended,
               per_step_bytes=per_step_bytes, world=world, rank=rank, counts=job_counts, sms=sms,
               resident=m.R, job_bytes=job_bytes, rank_batch=wr.batch)
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, m, per_step_bytes, world, use_graph=graph is not None, cpu_group=cpu_group)
    return res


def roofline_of(r, w, args) -> dict:
    """Roofline object of the dominant kernel (decode_split_kernel): HBM-bound layouts against the measured
    copy peak; the INT8-dithered layout (record marked "alu") against the issue peak, with its HBM figures
    alongside."""
    rec = r["traffic"]
    launch_s = r["layer_ms_mean"] * 1e-3
    hbm = {"bound": "hbm", "achieved": r["achieved"], "peak": r["peak"], "unit": "GB/s",
           "frac": r["achieved"] / r["peak"], "traffic": (rec["bytes_per_launch"] if rec else None),
           "kernel": "decode_split_kernel (CUDA events around its launch, eager steps)",
           "peak_source": f"{r['peak_kind']} hbm_gbs",
           "algorithmic_bytes_per_launch": r["per_step_bytes"] // (args.layers or w.n_layers),
           "launch_ms_mean": r["layer_ms_mean"], "call_ms_mean": r["call_ms_mean"]}
    if not rec or rec.get("bound") != "alu":
        return hbm
    achieved = rec["warp_inst_per_launch"] / launch_s
    sms = int(r.get("sms") or FALLBACK_SMS)
    mhz, mhz_src = max_sm_mhz(r.get("clocks"))
    peak = issue_peak_winst_per_s(sms, mhz)
    sms_src = "the device's SM count" if r.get("sms") else "GB300 SM count (fallback)"
    out = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "warp-instructions/s", "frac": achieved / peak,
           "traffic": rec["bytes_per_launch"], "kernel": hbm["kernel"],
           "peak_source": f"{sms} SMs ({sms_src}) x {SCHEDULERS_PER_SM} schedulers x 1 warp-instruction/clock x "
                          f"{mhz:.0f} MHz ({mhz_src})",
           "warp_inst_per_launch": rec["warp_inst_per_launch"],
           "hbm_achieved_gbs": r["achieved"], "hbm_frac": r["achieved"] / r["peak"],
           "algorithmic_bytes_per_launch": hbm["algorithmic_bytes_per_launch"],
           "launch_ms_mean": r["layer_ms_mean"], "call_ms_mean": r["call_ms_mean"]}
    return out


def run_e2e(args, m, per_step_bytes, world, use_graph=True, cpu_group=None):
    """Same metric through the public API with pinned host buffers and copies in the timed region."""
    torch = m.torch
    hq = torch.empty(m.q.shape, dtype=m.q.dtype, pin_memory=True).copy_(m.q)
    hk = torch.empty(m.k_new.shape, dtype=m.k_new.dtype, pin_memory=True).copy_(m.k_new)
    hv = torch.empty(m.v_new.shape, dtype=m.v_new.dtype, pin_memory=True).copy_(m.v_new)
    ho = torch.empty(m.out.shape, dtype=m.out.dtype, pin_memory=True)
    hm = torch.empty(m.meter_a.shape, dtype=m.meter_a.dtype, pin_memory=True)
    hc = torch.empty(4, dtype=torch.int32, pin_memory=True)
    dq, dk, dv = torch.empty_like(m.q), torch.empty_like(m.k_new), torch.empty_like(m.v_new)
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            m.step(dq, dk, dv)

    def one():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        if graph is not None:
            graph.replay()
        else:
            m.step(dq, dk, dv)
        ho.copy_(m.out, non_blocking=True)
        if m.meter_on:
            hm.copy_(m.meter_a, non_blocking=True)
            hc.copy_(m.counts, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
        torch.cuda.current_stream().synchronize()  # the host reads the step's result
    el = (time.perf_counter() - t0) / args.steps
    h2d = (hq.numel() * hq.element_size() + hk.numel() * 4 + hv.numel() * 4)
    d2h = ho.numel() * 4 + ((hm.numel() * 4 + 16) if m.meter_on else 0)
    job_bytes = per_step_bytes
    if world > 1:
        import torch.distributed as dist

        t = torch.tensor([el], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=cpu_group)
        el = float(t.item())
        (job_bytes,), _ = job_totals([per_step_bytes], [0, 0, 0, 0], world, cpu_group)
    return {"value": job_bytes / el / 1e9, "unit": "GB/s", "ms_per_step": el * 1e3,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ------------------------------------------------------------------------------------------ CPU oracle
def oracle_units(w, n_units: int, seed_base: int = 0):
    """Time the float64 oracle's decode of n (sequence, kv head) units of layer 0 at full context."""
    from oracle import attention as OA
    from oracle.encoders import fp16_value
    from tests.parity import oracle_cache_rows

    lens = W.seq_lengths(w)
    bts = W.identity_block_table(lens)
    total_bytes, elapsed = 0, 0.0
    for u in range(n_units):
        s = (u + seed_base) % w.batch
        n = int(lens[s])
        k32, v32, q = W.gen_unit_cpu(w, s, 0, n, first_pos=w.prefix_len)
        g = u % w.n_kv_heads
        k1, v1 = k32[:, g:g + 1], v32[:, g:g + 1]
        slots = W.slot_mapping(bts, s, np.arange(n))
        pre = None
        if w.prefix_len:
            pk, pv, _ = W.gen_unit_cpu(w, 0, 0, w.prefix_len, seed_unit=777_777)
            pre = (pk[:, g:g + 1], pv[:, g:g + 1])
        t0 = time.perf_counter()
        rows = oracle_cache_rows(k1, v1, slots, w.k_fmt, w.v_fmt, 1234, 0)
        kk, kh, vh, ww = k1[:, 0], rows["kh"][:, 0], rows["vh"][:, 0], fp16_value(rows["w16"][:, 0])
        sk = fp16_value(rows["ksb"][:, 0]) if rows["ksb"] is not None else None
        if pre is not None:
            pr = oracle_cache_rows(pre[0], pre[1], np.arange(w.prefix_len), w.prefix_k_fmt, w.prefix_v_fmt, 99, 0)
            kk = np.concatenate([pre[0][:, 0], kk])
            kh = np.concatenate([pr["kh"][:, 0], kh])
            vh = np.concatenate([pr["vh"][:, 0], vh])
            ww = np.concatenate([fp16_value(pr["w16"][:, 0]), ww])
        G = w.group
        tb = dict(delta_req=w.delta_req, n_layers=w.n_layers, n_q_heads=w.n_q_heads, n_steps=w.n_steps) \
            if w.tier_b else None
        OA.decode_head(q[g * G:(g + 1) * G].astype(np.float64), kk, kh, vh, ww, SM_SCALE, s_k=sk, tier_b=tb)
        elapsed += time.perf_counter() - t0
        total_bytes += n * token_head_bytes(w.k_fmt, w.v_fmt)
        if w.prefix_len:
            total_bytes += w.prefix_len * token_head_bytes(w.prefix_k_fmt, w.prefix_v_fmt)
    return total_bytes, elapsed


def blas_threads() -> int:
    """Threads of the BLAS pool the oracle's matrix products run on."""
    try:
        import threadpoolctl

        info = threadpoolctl.threadpool_info()
        n = max([i.get("num_threads", 1) for i in info] or [1])
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def host_cores() -> dict:
    """The host's logical CPUs (os.cpu_count()) and the BLAS threads the oracle actually used."""
    return {"cores": os.cpu_count() or 1, "blas_threads": blas_threads()}


def cpu_baseline(w, budget_s: float = 15.0):
    """Oracle GB/s on a bounded sample: as many full-context units as fit in ~budget_s."""
    b1, t1 = oracle_units(w, 1)
    n = max(1, min(4 * w.n_kv_heads, int(budget_s / max(t1, 1e-3))))
    b, t = oracle_units(w, n, seed_base=1)
    return {"value": b / t / 1e9, "unit": "GB/s", **host_cores(), "kind": "oracle",
            "sample": f"{n} (sequence, kv head) units of layer 0 at full context ({w.name}): float64 oracle "
                      f"dequantize + compressed/exact attention + TV + meter; {b / 1e6:.1f} MB of KV in {t:.1f} s"}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_units(w, 1)
    b, t = 0, 0.0
    for s in range(args.steps):
        bb, tt = oracle_units(w, 1, seed_base=s)
        b += bb
        t += tt
    value = b / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "GB/s", **host_cores(), "kind": "oracle",
                             "sample": f"each step: one (sequence, kv head) unit of layer 0 at full context"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def workload_config(w, world: int = 1):
    """The workload of a line: with N ranks the job is a global batch of N x w.batch sequences, sharded by
    balanced attended tokens (``dist.shard_sequences``)."""
    lens = W.seq_lengths(W.reduced(w, batch=w.batch * world))
    cfg = {"workload": w.name, "batch": w.batch * world, "layers": w.n_layers, "kv_heads": w.n_kv_heads,
           "q_heads": w.n_q_heads, "head_dim": 128, "page_size": 16,
           "layout": f"K {w.k_fmt} / V {w.v_fmt}", "meter": "tier A" + (" + tier B" if w.tier_b else ""),
           "context_tokens": int(lens.mean()) + w.prefix_len, "l2": "inputs larger than L2 (no flush)"}
    if world > 1:
        cfg["batch_per_gpu"] = w.batch
        cfg["parallelism"] = f"dp{world}: sequences sharded across ranks by attended tokens, no data-path collective"
    if w.prefix_len:
        cfg["prefix"] = f"{w.prefix_len} shared tokens, K {w.prefix_k_fmt} / V {w.prefix_v_fmt}, sink x{w.sink_scale:g}"
    return cfg


def times_second_workload(args) -> bool:
    """The default run (the headline workload with no switch) also times the second target workload."""
    return (args.workload == "qwen3_8b_cartridge" and not args.no_second and not args.layers and not args.batch
            and not args.resident_layers and not args.separate_append and not args.eager
            and not runs_a_variant(args, W.WORKLOADS[args.workload]) and not args.bypass)


def second_object(args, w, r) -> dict:
    """The second target workload's figures, timed in the same process after the headline with the same
    steps and warm-up: its own value, step time, roofline (issue and HBM), clocks, e2e and cpu baseline."""
    line = bench_line(args, w, r)
    keep = ("value", "unit", "ms_per_step", "pct_of_hbm_peak", "attended_kv_tok_per_s", "seq_tok_per_s", "roofline",
            "clocks", "e2e", "config", "gpu_launches", "meter_counts", "launch_mode", "cpu_baseline")
    return {k: line[k] for k in keep if k in line}


def main():
    args = parse()
    w = W.WORKLOADS[args.workload]
    if args.bypass:
        if w.k_fmt != "int8" or w.prefix_len:
            raise SystemExit("--bypass needs a workload with INT8-dithered keys and no shared prefix")
        w = W.reduced(w, massive_pairs=args.bypass, massive_scale=30.0, bypass_pairs=args.bypass)
    if args.int8_groups:
        if w.k_fmt != "int8" or w.v_fmt != "int8" or w.prefix_len or w.bypass_pairs:
            raise SystemExit("--int8-groups needs a workload with INT8-dithered keys and values, no shared prefix "
                             "and no outlier bypass")
        w = W.reduced(w, k_fmt="int8g32", v_fmt="int8g32")
    if args.batch:
        w = W.reduced(w, batch=args.batch)
    if args.impl == "reference":
        run_reference(args, w)
        return
    r = run_gpu(args, w)
    line = bench_line(args, w, r) if r["rank"] == 0 else None
    if times_second_workload(args):
        import gc

        import torch

        gc.collect()
        torch.cuda.empty_cache()   # the headline's caches are released before the second workload's are built
        w2 = W.WORKLOADS[SECOND_WORKLOAD]
        r2 = run_gpu(args, w2)
        if line is not None:
            line[SECOND_WORKLOAD] = second_object(args, w2, r2)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line))


def bench_line(args, w, r) -> dict:
    """The JSON object of one bench run (rank 0) from run_gpu's result ``r``."""
    line = {"metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": r["world"], "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(w, r["world"]),
            "pct_of_hbm_peak": 100.0 * r["value"] / r["world"] / r["peak"],
            "attended_kv_tok_per_s": r["attended"] / (r["ms_step"] * 1e-3),
            "seq_tok_per_s": w.batch * r["world"] / (r["ms_step"] * 1e-3),
            "roofline": roofline_of(r, w, args),
            "gpu_launches": r["launches"], "clocks": r["clocks"], "meter_counts": r["counts"],
            "launch_mode": "cuda_graph" if r["graph"] else "eager"}
    if args.meter_off:
        line["config"]["meter"] = "off (no witness read, no kvq_meter)"
    if args.value_side:
        line["config"]["meter"] += " + value side (output-error bound)"
    if args.shapes:
        line["config"]["meter"] += " + alternative bound shapes (two-sided, det-tanh)"
    if args.gate:
        line["config"]["meter"] += " + gate support (per-page contributions, greedy page-in plan per layer)"
    if w.bypass_pairs:
        line["config"]["layout"] += (f" + fixed-channel key bypass of {w.bypass_pairs} massive RoPE pairs "
                                     f"(x{w.massive_scale:g}, fp16)")
    if r["resident"] < (args.layers or w.n_layers):
        line["config"]["resident_layers"] = r["resident"]
    if "e2e" in r:
        line["e2e"] = r["e2e"]
    if args.layers or args.batch:
        line["note"] = (f"profiling run with {args.layers or w.n_layers} layers, batch {w.batch}: not a bench line")
    if r["world"] == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
        extra = [n for n, on in (("value side", args.value_side), ("bound shapes", args.shapes),
                                 ("gate support", args.gate), ("outlier bypass", w.bypass_pairs)) if on]
        if extra:
            line["cpu_baseline"]["sample"] += (f"; the plain decode of this workload (the oracle sample leaves out the "
                                               f"{', '.join(extra)} work of the GPU line)")
    return line


if __name__ == "__main__":
    main()
