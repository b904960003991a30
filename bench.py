"""Benchmark of the ring-attention hot path on GB300.

One step = one pass of the whole path over one batch of the 128K causal striped
workload (B=1, H=8, L=131072, d=128, N=16 virtual ranks).  By default that pass
is a single launch: the fused ring sweep reads Q, K and V in token order and
writes O and LSE in token order, the striped assignment being the addresses of
its tiles, so the shard and un-shard permutes are part of the sweep's loads and
stores.  ``--explicit-permutes`` runs them as separate permute kernels around a
sweep on shard stacks instead (six launches per step).  Inputs are synthetic
(seeded N(0, 1) bf16) and larger than L2, so nothing is reused from cache
between steps.

The metric is algorithmic TFLOP/s: 4 * B * H * d * L(L+1)/2 flops per step
(the causal pairs, counted once per layout; skipped and masked work is not
counted).  Besides the device-resident number the JSON line carries:
  * roofline  -- the attention kernel alone: its CUDA-event time per launch
                 against the measured dense-bf16 burst peak (the kernel is timed
                 in a region well under a second), with the fraction of the
                 sustained peak beside it;
  * e2e       -- the same metric through the same public calls with the step's
                 inputs copied from pinned host memory and O / LSE copied back;
  * cpu_baseline -- the fp64 CPU oracle, timed on a bounded sample of query rows;
  * clocks    -- SM clocks and throttle reasons sampled during the timed region.

``--impl reference`` times the CPU oracle itself on the same workload and metric.
Under torchrun (N > 1) every rank runs its own replica of the workload.
"""
import argparse
import contextlib
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from synthetic_inputs import WORKLOADS, make_cu_seqlens, make_dout, make_qkv  # noqa: E402

METRIC = "causal ring-attention fwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 peak"
METRIC_BWD = "causal ring-attention bwd TFLOP/s (bf16, 1×GB300; algorithmic 8·B·H·d·pairs)"
DEFAULT_WORKLOAD = "striped_B1_H8_L131072_d128_N16"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_striped_128k_traffic.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "sequence_blockwise_softmax_gb300", "csrc", f)
                  for f in ("attn_sm103.cu", "ra_device.cuh", "ra_positions.cuh", "ra_internal.h")]


def algorithmic_flops(B, L, H, d, causal):
    pairs = L * (L + 1) // 2 if causal else L * L
    return 4.0 * B * H * d * pairs


def _code_only(text):
    """C++ source with comments and whitespace removed, so that the hash moves only
    when the code does.  String literals are kept whole."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join("".join(out).split())


def kernel_source_hash():
    """Hash of the attention kernel's code (comments and whitespace excluded)."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def read_traffic():
    """Per-launch DRAM bytes of the attention kernel from the committed ncu summary,
    or None when the kernel source changed since it was taken."""
    try:
        fields = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    key, val = line.split(":", 1)
                    fields[key.strip()] = val.strip()
        if fields.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return float(fields["dram_bytes_per_full_launch"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------- clocks
REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        cmd = ["nvidia-smi", "-i", str(self.index),
               "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "200"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 4:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                bits = int(parts[3], 16)
            except ValueError:
                continue
            for bit, name in REASON_BITS.items():
                if bits & bit and name != "gpu_idle":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- the GPU path
class Workload:
    def __init__(self, ra, name, layout, dev, shape=None, stepwise=False, kv_heads=None, varlen=None,
                 seq_order=True, loopback=False):
        w = dict(WORKLOADS[name])
        if shape is not None:
            w.update(B=shape[0], L=shape[1], H=shape[2], d=shape[3], N=shape[4])
        self.ra, self.name, self.layout, self.dev = ra, name, layout, dev
        self.B, self.L, self.H, self.d, self.N = w["B"], w["L"], w["H"], w["d"], w["N"]
        self.U = w.get("U", 1)
        self.causal = w["causal"]
        B, L, H, d, N, U = self.B, self.L, self.H, self.d, self.N, self.U
        self.Hkv = kv_heads or H
        # token-order sweep (RA_FLAG_SEQ_ORDER): the layout is the tiles' addresses and no
        # permute runs; the Ulysses split, the stepwise sweep and zigzag chunks that are not
        # a multiple of 128 rows take the explicit permutes
        self.seq_order = (seq_order and U == 1 and not stepwise and not loopback and
                          not (layout == "zigzag" and (L // N // 2) % 128))
        self.loopback = loopback
        q, k, v, _ = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])
        if self.Hkv != H:
            # grouped-query attention: the first H_kv heads of the drawn K and V
            k, v = k[:, :, :self.Hkv].contiguous(), v[:, :, :self.Hkv].contiguous()
        with near_gpu(dev) as cpus:
            self.host = [t.pin_memory() for t in (q, k, v)]
            self.o_host = torch.empty((B, L, H, d), dtype=torch.float32).pin_memory()
            self.lse_host = torch.empty((B, H, L), dtype=torch.float32).pin_memory()
            self.hosts_out = [(self.o_host, self.lse_host),
                              (torch.empty_like(self.o_host).pin_memory(),
                               torch.empty_like(self.lse_host).pin_memory())]
        self.host_cpus = cpu_list(cpus) if cpus else None
        self.seq = [t.to(dev) for t in self.host]
        P = U * N
        self.heads = [H, self.Hkv, self.Hkv]
        self.shard = [torch.empty((P, B, L // P, hx, d), dtype=torch.bfloat16, device=dev)
                      for hx in self.heads]
        if U > 1:
            self.head = [torch.empty((N, U, B, L // N, hx // U, d), dtype=torch.bfloat16, device=dev)
                         for hx in self.heads]
        self.Bq, self.Hq = U * B, H // U
        ring_in = self.head if U > 1 else self.shard
        self.o_ring = torch.empty(ring_in[0].shape, dtype=torch.float32, device=dev)
        self.lse_ring = torch.empty((N, self.Bq, self.Hq, L // N), dtype=torch.float32, device=dev)
        self.o_shard = (torch.empty(self.shard[0].shape, dtype=torch.float32, device=dev)
                        if U > 1 else None)
        self.o_seq = torch.empty((B, L, H, d), dtype=torch.float32, device=dev)
        self.lse_seq = torch.empty((B, H, L), dtype=torch.float32, device=dev)
        self.flags = ra.RA_FLAG_STEPWISE if stepwise else (ra.RA_FLAG_SEQ_ORDER if self.seq_order else 0)
        self.ws = ra.new_workspace(ra.ra_ring_attn_workspace_bytes(self.Bq, L, self.Hq, d, N, self.flags),
                                   device=dev)
        self.flops = algorithmic_flops(B, L, H, d, self.causal)
        self.cu = None
        if varlen:
            if B != 1 or U != 1:
                raise ValueError("packed sequences need B = 1 and no Ulysses split")
            cu = make_cu_seqlens(L, varlen, w["seed"])
            lens = (cu[1:] - cu[:-1]).double()
            pairs = float((lens * (lens + 1) / 2).sum()) if self.causal else float((lens * lens).sum())
            self.flops = 4.0 * H * d * pairs
            self.cu = cu.to(torch.int32).to(dev)
        attn_launches = (2 * N - 1) if stepwise else 1     # N block sweeps + N-1 merges
        self.launches = 3 * (2 if U > 1 else 1) + attn_launches + (2 if U > 1 else 1) + 1
        if self.seq_order:
            self.launches = 1
        if loopback:
            # the multi-GPU ring driver with its N ranks on this GPU (device-to-device
            # copies on a copy stream in place of the transfers)
            if U != 1 or varlen:
                raise ValueError("the loopback ring runs plain ring layouts")
            from sequence_blockwise_softmax_gb300 import ring
            self.ring = ring
            self.ring_ranks = ring.loopback_ranks(*self.shard, N, layout, self.causal, o=self.o_ring,
                                                  lse=self.lse_ring)
            self.comm_stream = torch.cuda.Stream(device=dev)
            active = sum(1 for r in self.ring_ranks for st, j, p in r.schedule if st == 0 or p)
            self.launches = 3 + (2 * active - N) + 2
            self.ring_bytes = ring.ring_bytes_per_step(B, L // N, self.Hkv, d) * N * (N - 1)
        self.attn_events = []

    def step(self, time_attention=False, slot=0):
        ra, B, L, H, d, N, U = self.ra, self.B, self.L, self.H, self.d, self.N, self.U
        seq, o_seq, lse_seq = self.slots[slot] if slot else (self.seq, self.o_seq, self.lse_seq)
        if self.seq_order:
            # one launch: the sweep reads q/k/v and writes O / LSE in token order
            if time_attention:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
            if self.cu is not None:
                ra.ra_ring_attn_fwd_varlen(*seq, o_seq, lse_seq, self.cu, L, H, self.Hkv, d, N, self.layout,
                                           self.causal, flags=self.flags, workspace=self.ws)
            else:
                ra.ra_ring_attn_fwd_gqa(*seq, o_seq, lse_seq, B, L, H, self.Hkv, d, N, self.layout, self.causal,
                                        flags=self.flags, workspace=self.ws)
            if time_attention:
                e1.record()
                self.attn_events.append((e0, e1))
            return
        for i in range(3):
            hx = self.heads[i]
            ra.ra_shard_permute(seq[i], self.shard[i], ra.RA_SEQ_TO_SHARDS, self.layout, B, L, hx, d, N, U)
            if U > 1:
                ra.ra_shard_permute(self.shard[i], self.head[i], ra.RA_ULYSSES_SEQ_TO_HEAD, self.layout,
                                    B, L, hx, d, N, U)
        ring_in = self.head if U > 1 else self.shard
        if time_attention:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
        if self.loopback:
            self.ring.run_ring(self.ring_ranks, self.ring.LoopbackRing(), self.comm_stream)
        elif self.cu is not None:
            ra.ra_ring_attn_fwd_varlen(*ring_in, self.o_ring, self.lse_ring, self.cu, L, H, self.Hkv, d, N,
                                       self.layout, self.causal, flags=self.flags, workspace=self.ws)
        elif self.Hkv == H:
            ra.ra_ring_attn_fwd(*ring_in, self.o_ring, self.lse_ring, self.Bq, L, self.Hq, d, N, self.layout,
                                self.causal, flags=self.flags, workspace=self.ws)
        else:
            ra.ra_ring_attn_fwd_gqa(*ring_in, self.o_ring, self.lse_ring, self.Bq, L, self.Hq, self.Hkv // U,
                                    d, N, self.layout, self.causal, flags=self.flags, workspace=self.ws)
        if time_attention:
            e1.record()
            self.attn_events.append((e0, e1))
        o = self.o_ring
        if U > 1:
            ra.ra_shard_permute(o, self.o_shard, ra.RA_ULYSSES_HEAD_TO_SEQ, self.layout, B, L, H, d, N, U)
            o = self.o_shard
        ra.ra_shard_permute(o, o_seq, ra.RA_SHARDS_TO_SEQ, self.layout, B, L, H, d, N, U)
        ra.ra_lse_to_seq(self.lse_ring, lse_seq, self.layout, B, L, H, N, U)

    def prepare_backward(self):
        """Forward once (saved activations), then buffers for the backward step."""
        ra, B, L, H, d, N = self.ra, self.B, self.L, self.H, self.d, self.N
        if self.U != 1 or self.cu is not None:
            raise ValueError("the backward bench runs plain ring layouts")
        self.step()
        self.do_seq = make_dout(B, L, H, d).to(self.dev)
        self.bws = ra.new_workspace(ra.ra_ring_attn_bwd_workspace_bytes(B, L, H, d, N), device=self.dev)
        self.flops = 2.0 * self.flops
        self.dq_seq = torch.empty((B, L, H, d), dtype=torch.float32, device=self.dev)
        self.dk_seq = torch.empty((B, L, self.Hkv, d), dtype=torch.float32, device=self.dev)
        self.dv_seq = torch.empty_like(self.dk_seq)
        if self.seq_order:
            # token order: D = rowsum(dO * O), the dK/dV pass and the dQ pass, no permutes
            self.launches = 3
            return
        self.do_shard = torch.empty_like(self.shard[0])
        S = L // N
        self.dq = torch.empty((N, B, S, H, d), dtype=torch.float32, device=self.dev)
        self.dk = torch.empty((N, B, S, self.Hkv, d), dtype=torch.float32, device=self.dev)
        self.dv = torch.empty_like(self.dk)
        self.launches = 1 + 3 + 3

    def step_bwd(self, time_attention=False):
        ra, B, L, H, d, N = self.ra, self.B, self.L, self.H, self.d, self.N
        if self.seq_order:
            if time_attention:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
            ra.ra_ring_attn_bwd(*self.seq, self.o_seq, self.do_seq, self.lse_seq, self.dq_seq, self.dk_seq,
                                self.dv_seq, B, L, H, self.Hkv, d, N, self.layout, self.causal, workspace=self.bws,
                                flags=ra.RA_FLAG_SEQ_ORDER)
            if time_attention:
                e1.record()
                self.attn_events.append((e0, e1))
            return
        ra.ra_shard_permute(self.do_seq, self.do_shard, ra.RA_SEQ_TO_SHARDS, self.layout, B, L, H, d, N)
        if time_attention:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
        ra.ra_ring_attn_bwd(*self.shard, self.o_ring, self.do_shard, self.lse_ring, self.dq, self.dk, self.dv,
                            B, L, H, self.Hkv, d, N, self.layout, self.causal, workspace=self.bws)
        if time_attention:
            e1.record()
            self.attn_events.append((e0, e1))
        ra.ra_shard_permute(self.dq, self.dq_seq, ra.RA_SHARDS_TO_SEQ, self.layout, B, L, H, d, N)
        ra.ra_shard_permute(self.dk, self.dk_seq, ra.RA_SHARDS_TO_SEQ, self.layout, B, L, self.Hkv, d, N)
        ra.ra_shard_permute(self.dv, self.dv_seq, ra.RA_SHARDS_TO_SEQ, self.layout, B, L, self.Hkv, d, N)

    def run_e2e(self, steps, world, dev):
        """End to end through the same calls: every step uploads its q, k, v from pinned host
        memory and downloads its O and LSE.  Steps alternate between two buffer slots and the
        copies run on their own streams (upload and download engines), so the upload of step
        i+1 and the download of step i-1 overlap the compute of step i.  Returns ms per step
        over the whole timed region, copies included."""
        if not hasattr(self, "slots"):
            self.slots = [None, ([torch.empty_like(t) for t in self.seq], torch.empty_like(self.o_seq),
                                 torch.empty_like(self.lse_seq))]
            self.up, self.down = torch.cuda.Stream(), torch.cuda.Stream()
        compute = torch.cuda.current_stream()
        dev_bufs = [(self.seq, self.o_seq, self.lse_seq), self.slots[1]]
        Ev = lambda: torch.cuda.Event()
        up_done, comp_done, down_done = [Ev(), Ev()], [Ev(), Ev()], [Ev(), Ev()]
        Tv = lambda: torch.cuda.Event(enable_timing=True)
        copy_times = []          # per step: (upload start, end), (download start, end)
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(compute)
        self.up.wait_event(e0)
        self.down.wait_event(e0)
        for i in range(steps):
            k = i % 2
            seq, o_seq, lse_seq = dev_bufs[k]
            with torch.cuda.stream(self.up):
                if i >= 2:
                    self.up.wait_event(comp_done[k])        # step i-2 has read these inputs
                u0, u1 = Tv(), Tv()
                u0.record(self.up)
                for h, dbuf in zip(self.host, seq):
                    dbuf.copy_(h, non_blocking=True)
                u1.record(self.up)
                up_done[k].record(self.up)
            compute.wait_event(up_done[k])
            if i >= 2:
                compute.wait_event(down_done[k])            # step i-2's outputs are on the host
            c0, c1 = Tv(), Tv()
            c0.record(compute)
            self.step(slot=k)
            c1.record(compute)
            comp_done[k].record(compute)
            with torch.cuda.stream(self.down):
                self.down.wait_event(comp_done[k])
                d0, d1 = Tv(), Tv()
                d0.record(self.down)
                self.hosts_out[k][0].copy_(o_seq, non_blocking=True)
                self.hosts_out[k][1].copy_(lse_seq, non_blocking=True)
                d1.record(self.down)
                down_done[k].record(self.down)
            copy_times.append(((u0, u1), (d0, d1), (c0, c1)))
        compute.wait_stream(self.down)
        compute.wait_stream(self.up)
        e1.record(compute)
        torch.cuda.synchronize()
        barrier(world)
        # the copy engines' rates (median over the steps), to read the end-to-end number by
        up_ms = float(np.median([a.elapsed_time(b) for (a, b), _, _ in copy_times]))
        down_ms = float(np.median([a.elapsed_time(b) for _, (a, b), _ in copy_times]))
        # the step's own kernels while the copies run beside them (power and link sharing)
        self.e2e_step_ms = float(np.median([a.elapsed_time(b) for _, _, (a, b) in copy_times]))
        self.copy_gbs = (self.h2d_bytes() / up_ms / 1e6 if up_ms > 0 else None,
                         self.d2h_bytes() / down_ms / 1e6 if down_ms > 0 else None)
        return max_over_ranks(e0.elapsed_time(e1), world, dev) / steps

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host)

    def d2h_bytes(self):
        return self.o_host.numel() * 4 + self.lse_host.numel() * 4


# ----------------------------------------------------------------- host memory
def gpu_local_cpus(dev):
    """The CPUs of the socket the GPU hangs off (sysfs local_cpulist of its PCI function),
    limited to the ones this process may use; None when unknown."""
    if getattr(dev, "type", None) != "cuda" or not torch.cuda.is_available():
        return None
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open("/sys/bus/pci/devices/%s/local_cpulist" % bus) as f:
            text = f.read().strip()
        cpus = set()
        for part in text.split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
        return (cpus & os.sched_getaffinity(0)) or None
    except (OSError, AttributeError, ValueError, RuntimeError):
        return None


@contextlib.contextmanager
def near_gpu(dev):
    """Pinned host buffers allocated inside are placed in the memory of the CPUs the GPU
    is attached to (the process runs on those CPUs while the pages are pinned, then
    returns to its own set), so that the step's copies do not cross sockets."""
    cpus = gpu_local_cpus(dev)
    saved = os.sched_getaffinity(0)
    if cpus:
        os.sched_setaffinity(0, cpus)
    try:
        yield cpus
    finally:
        if cpus:
            os.sched_setaffinity(0, saved)


def cpu_list(cpus):
    """'0-71' style text for a set of CPU numbers."""
    out, run = [], []
    for c in sorted(cpus):
        if run and c == run[-1] + 1:
            run.append(c)
        else:
            if run:
                out.append("%d-%d" % (run[0], run[-1]) if len(run) > 1 else str(run[0]))
            run = [c]
    if run:
        out.append("%d-%d" % (run[0], run[-1]) if len(run) > 1 else str(run[0]))
    return ",".join(out)


# ----------------------------------------------------------------- ring balance
def ring_pair_counts(layout, N, S, causal):
    """Allowed (query, key) pairs that rank i computes at ring step s, where it meets the
    key/value shard of rank j = (i - s) mod N: an [N, N] table indexed [i, s].

    Counted from the token positions of each layout ("From Ring Attention to DeepSpeed
    Ulysses to USP", §3.4 contiguous, §4 striped, §6.1 zigzag): contiguous rank r holds
    r*S .. r*S+S-1, so an earlier rank's shard is all visible, its own is a triangle and a
    later one is hidden; striped local token a of rank r sits at a*N + r, so a key shard
    j <= i gives the triangle c <= a and j > i the strict one c < a; zigzag rank r holds
    chunks r and 2N-1-r of S/2 tokens, which makes every step half a block, plus the two
    diagonal chunk triangles' extra S/2 on step 0."""
    c = np.zeros((N, N), dtype=np.int64)
    for i in range(N):
        for s in range(N):
            j = (i - s) % N
            if not causal:
                c[i, s] = S * S
            elif layout == "contiguous":
                c[i, s] = S * S if j < i else (S * (S + 1) // 2 if j == i else 0)
            elif layout == "striped":
                c[i, s] = S * (S + 1) // 2 if j <= i else S * (S - 1) // 2
            else:
                C = S // 2
                c[i, s] = 2 * C * C + (C if j == i else 0)
    return c


def balance_table(layout, N, S, causal):
    """The ring's critical path in pairs: with one device per rank a step lasts as long as
    its busiest rank, so the sweep costs sum_s max_i pairs(i, s) against the ideal total / N."""
    c = ring_pair_counts(layout, N, S, causal)
    crit = int(c.max(axis=0).sum())
    ideal = float(c.sum()) / N
    return {"pairs_total": int(c.sum()), "pairs_step_max": c.max(axis=0).tolist(),
            "pairs_critical_path": crit, "pairs_ideal": ideal, "pairs_ratio": crit / ideal}


def measure_ring_steps(ra, wl, reps=3):
    """The per-rank stepwise loop, each rank as if it had the whole GPU: for every rank i
    and step s, one ra_block_attn_fwd against key/value rank (i - s) mod N plus, from step
    1 on, one ra_lse_merge into the rank's accumulator, timed with CUDA events.  Returns
    [N, N] milliseconds indexed [i, s] (median over ``reps`` sweeps)."""
    N, Bq, Hq, d, L = wl.N, wl.Bq, wl.Hq, wl.d, wl.L
    S = L // N
    ring = [t.view(N, Bq, S, t.shape[-2], d) for t in (wl.head if wl.U > 1 else wl.shard)]
    o_acc = torch.empty((Bq, S, Hq, d), dtype=torch.float32, device=wl.dev)
    lse_acc = torch.empty((Bq, Hq, S), dtype=torch.float32, device=wl.dev)
    o_b, lse_b = torch.empty_like(o_acc), torch.empty_like(lse_acc)
    out = np.zeros((reps, N, N))
    for rep in range(reps):
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(N)] for _ in range(N)]
        for i in range(N):
            for s in range(N):
                j = (i - s) % N
                o, lse = (o_acc, lse_acc) if s == 0 else (o_b, lse_b)
                ev[i][s][0].record()
                if wl.Hkv == wl.H:
                    ra.ra_block_attn_fwd(ring[0][i], ring[1][j], ring[2][j], o, lse, Bq, S, Hq, d, N, i, j,
                                         wl.layout, wl.causal, workspace=wl.ws)
                else:
                    ra.ra_block_attn_fwd_gqa(ring[0][i], ring[1][j], ring[2][j], o, lse, Bq, S, Hq,
                                             wl.Hkv // wl.U, d, N, i, j, wl.layout, wl.causal, workspace=wl.ws)
                if s:
                    ra.ra_lse_merge_bshd(o_acc, lse_acc, o_b, lse_b, Bq, S, Hq, d)
                ev[i][s][1].record()
        torch.cuda.synchronize()
        out[rep] = [[a.elapsed_time(b) for a, b in row] for row in ev]
    ra.ra_check_status(wl.ws)
    return np.median(out, axis=0)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, dev):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_rank, world, ms_per_step_max):
    """Whole-job TFLOP/s: every rank's replica counts, timed by the slowest rank."""
    return flops_per_rank * world / (ms_per_step_max * 1e-3) / 1e12


def timed(fn, steps, world, dev):
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1), world, dev)


# ----------------------------------------------------------------- CPU oracle timing
def oracle_sample_run(name, budget_s, seed=0, cache={}):
    """Time the fp64 oracle on a random sample of query rows (all batches and heads)
    sized to about ``budget_s`` seconds.  Returns (flops, seconds, rows, threads)."""
    import oracle
    w = WORKLOADS[name]
    B, L, H, d = w["B"], w["L"], w["H"], w["d"]
    key = (name,)
    if key not in cache:
        cache[key] = make_qkv(B, L, H, d, w["seed"], w["k_scale_frac"])[:3]
    q, k, v = cache[key]
    rng = np.random.default_rng(seed)

    def run(n):
        rows = np.sort(rng.integers(0, L, n))
        t0 = time.perf_counter()
        oracle.full_attention(q, k, v, causal=w["causal"], rows=rows)
        dt = time.perf_counter() - t0
        keys = (rows + 1).sum() if w["causal"] else n * L
        return 4.0 * B * H * d * float(keys), dt, n

    fl, dt, n = run(4)                       # calibration
    rate = fl / max(dt, 1e-6)
    per_row = 4.0 * B * H * d * (L / 2 if w["causal"] else L)
    n = max(4, int(budget_s * rate / per_row))
    fl, dt, n = run(n)
    return fl, dt, n, oracle.num_threads()


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    name = args.workload
    w = WORKLOADS[name]
    layout = args.layout or w["layouts"][0]
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_sample_run(name, per_step, seed=100 + i)
    fl_tot, t_tot, rows_tot, threads = 0.0, 0.0, 0, 1
    for i in range(args.steps):
        fl, dt, n, threads = oracle_sample_run(name, per_step, seed=i)
        fl_tot += fl
        t_tot += dt
        rows_tot += n
    value = fl_tot / t_tot / 1e12
    sample = ("%d random query rows (all %d heads) of the %s workload, %d steps of ~%.0f s"
              % (rows_tot, w["H"], name, args.steps, per_step))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_tot / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": name, "layout": layout, "B": w["B"], "L": w["L"], "H": w["H"],
                   "d": w["d"], "N": w["N"], "causal": w["causal"]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(WORKLOADS))
    ap.add_argument("--config", type=int, default=None, choices=range(1, len(WORKLOADS) + 1),
                    help="select the workload by its number, 1-5 (tiny non-causal, causal 8K, zigzag 2x32K, "
                         "striped 128K, USP 256K); overrides --workload")
    ap.add_argument("--layout", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--stepwise", action="store_true",
                    help="run the sweep as N block launches + N-1 LSE merges (the pages' per-step loop)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward (ra_ring_attn_bwd) on saved forward outputs instead")
    ap.add_argument("--explicit-permutes", action="store_true",
                    help="run the forward on shard stacks with the permute kernels around the sweep "
                         "instead of the token-order sweep")
    ap.add_argument("--ring-loopback", action="store_true",
                    help="run the multi-GPU ring driver (sequence_blockwise_softmax_gb300.ring) with its N ranks "
                         "on this GPU: per rank and step a block call and a merge, the K/V shift as "
                         "device-to-device copies on a copy stream")
    ap.add_argument("--varlen", type=int, default=None,
                    help="pack this many variable-length sequences (seeded cut points) into the workload")
    ap.add_argument("--kv-heads", type=int, default=None,
                    help="grouped-query attention with this many key/value heads")
    ap.add_argument("--shape", default=None,
                    help="B,L,H,d,N override of the workload's sizes (a smaller case for profiling)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.config is not None:
        args.workload = list(WORKLOADS)[args.config - 1]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import sequence_blockwise_softmax_gb300 as ra
    ra.lib()  # fails loudly when the library is missing
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)

    w = WORKLOADS[args.workload]
    layout = args.layout or w["layouts"][0]
    shape = tuple(int(x) for x in args.shape.split(",")) if args.shape else None
    wl = Workload(ra, args.workload, layout, dev, shape, stepwise=args.stepwise, kv_heads=args.kv_heads,
                  varlen=args.varlen, seq_order=not args.explicit_permutes, loopback=args.ring_loopback)

    step = wl.step
    if args.backward:
        wl.prepare_backward()
        step = wl.step_bwd
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ra.ra_check_status(wl.ws)

    # device-resident timed region
    wl.attn_events = []
    with ClockSampler(local_rank) as clocks:
        ms = timed(lambda: step(time_attention=True), args.steps, world, dev)
    ms_step = ms / args.steps
    attn_ms = float(np.mean([a.elapsed_time(b) for a, b in wl.attn_events]))
    attn_ms = max_over_ranks(attn_ms, world, dev)
    ra.ra_check_status(wl.ws)

    # end to end through the same calls, host buffers in and out
    if args.backward:
        ms_e2e = None
    else:
        wl.run_e2e(2, world, dev)
        ms_e2e = wl.run_e2e(args.steps, world, dev)
        ra.ra_check_status(wl.ws)

    value = job_value(wl.flops, world, ms_step)
    e2e_value = job_value(wl.flops, world, ms_e2e) if ms_e2e else None

    peaks, peak_src = measured_peaks()
    # the timed region is well under a second of back-to-back launches: the burst peak
    peak = float(peaks["bf16_tflops"])
    peak_sustained = float(peaks.get("bf16_tflops_sustained", peak))
    achieved = wl.flops / (attn_ms * 1e-3) / 1e12
    # the committed DRAM figure is for the default forward launch only
    default_launch = not (args.backward or args.stepwise or args.ring_loopback or args.varlen or args.kv_heads or shape
                          or args.workload != DEFAULT_WORKLOAD or layout != "striped")
    traffic = read_traffic() if default_launch else None

    line = {
        "metric": METRIC_BWD if args.backward else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload + ("" if shape is None else " (resized)"), "layout": layout, "B": wl.B, "L": wl.L, "H": wl.H,
                   "d": wl.d, "N": wl.N, "U": wl.U, "H_kv": wl.Hkv, "causal": wl.causal,
                   "packed_sequences": args.varlen,
                   "parallelism": "replicas" if world > 1 else "single GPU, %d virtual ranks" % wl.N,
                   "sweep": ("ring driver, N ranks on one GPU (loopback transfers)" if args.ring_loopback
                             else "stepwise" if args.stepwise else "fused"),
                   "io": ("token order: the layout is the sweep's tile addressing, no permute kernels"
                          if wl.seq_order else "shard stacks with explicit permute kernels"),
                   "l2": "inputs larger than L2 (q/k/v %.0f MiB)" % (wl.h2d_bytes() / 2 ** 20)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "frac_of_sustained": achieved / peak_sustained,
                     "traffic": traffic,
                     "kernel": ("ra_ring_attn_bwd: bwd_dot + attn_bwd_dkv + attn_bwd_dq" if args.backward else
                                "ring driver: per rank and step attn_fwd_kernel<fp32 partial> + lse_merge_kernel, "
                                "K/V copies on a copy stream" if args.ring_loopback else
                                "ra_ring_attn_fwd stepwise: N x attn_fwd_kernel<fp32 partial> + N-1 x lse_merge_kernel"
                                if args.stepwise else "attn_fwd_kernel<128, fp32 O> (ra_ring_attn_fwd)"),
                     "kernel_ms": attn_ms,
                     "peak_source": "%s bf16_tflops (burst); frac_of_sustained against %s "
                                    "bf16_tflops_sustained" % (peak_src, peak_src)},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": wl.h2d_bytes(),
                "d2h_bytes_per_step": wl.d2h_bytes(), "ms_per_step": ms_e2e,
                "copies": "every step uploads q/k/v and downloads O/LSE; two buffer slots, copies "
                          "on their own streams overlap the neighbouring steps' compute",
                "step_kernels_ms": getattr(wl, "e2e_step_ms", None),
                "h2d_gbs": getattr(wl, "copy_gbs", (None, None))[0],
                "d2h_gbs": getattr(wl, "copy_gbs", (None, None))[1],
                "host_buffers": ("pinned, placed by the GPU's local CPUs %s" % wl.host_cpus if wl.host_cpus
                                 else "pinned")},
        "gpu_launches": wl.launches * args.steps,
        "clocks": clocks.summary(),
    }

    if args.ring_loopback:
        per = wl.ring.ring_bytes_per_step(wl.B, wl.L // wl.N, wl.Hkv, wl.d)
        line["ring_driver"] = {
            "bytes_per_rank_step": per, "copy_bytes_per_sweep": per * wl.N * (wl.N - 1),
            "transport": "device-to-device copies on a copy stream (one GPU holds all ranks); on N GPUs "
                         "the same driver moves these bytes with NCCL point-to-point (not measured here)"}
    if wl.cu is None:
        bal = balance_table(layout, wl.N, wl.L // wl.N, wl.causal)
        if args.stepwise:
            # measured after the timed region: every (rank, step) block + merge on the whole GPU
            t = measure_ring_steps(ra, wl)
            step_max = t.max(axis=0)
            bal.update({
                "step_ms_max": step_max.tolist(), "step_ms_mean": t.mean(axis=0).tolist(),
                "critical_path_ms": float(step_max.sum()), "ideal_ms": float(t.sum()) / wl.N,
                "ms_ratio": float(step_max.sum()) / (float(t.sum()) / wl.N),
                "per_rank_tflops_critical_path": wl.flops / wl.N / (step_max.sum() * 1e-3) / 1e12,
                "timing": "each rank's block + merge launched alone on the whole GPU, as if every "
                          "rank had its own; a step lasts as long as its slowest rank"})
        line["ring_balance"] = bal

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, dt, n, threads = oracle_sample_run(args.workload, args.cpu_budget)
        line["cpu_baseline"] = {
            "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "%d random query rows x %d heads of the workload (%.1f s of fp64 work)"
                      % (n, wl.H, dt)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
