#!/usr/bin/env python3
"""Benchmark of the DGQ INT8 paged KV-cache hot path on GB300.

One step = dgq_compress of every layer's K/V (bf16 -> uint8 codes in paged blocks plus
segment records), dgq_paged_decode_attn over every layer's INT8 cache, then dgq_append of the
step's own key and value into every layer's cache, for one
synthetic workload (default: the largest, the MHA high-concurrency decode batch, 32 layers, 100
requests of 256..2048 tokens, Hq = Hkv = 32, block size 16, shuffled blocks).  Inputs are
generated on the GPU by the seeded generator before timing and stay resident in HBM; each layer
has its own buffers, so one step touches far more than L2 (no flush needed).  After the main
line's measurements, the other workloads (2, 4, 5, 5p) are set up and timed the same way for a
per-workload table (`other_workloads`).

Prints ONE JSON line (rank 0).  `value` is decode-attention algorithmic GB/s over all ranks;
`compress_gbs` the same for dgq_compress.  `--impl reference` times the CPU oracle instead.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 3] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT8 paged decode-attn HBM GB/s (% of peak); dgq_compress GB/s"
D = 128
REC = 128  # bytes per segment record
APPEND_ROOM = 64  # tokens each request may grow by through dgq_append during a run
APPEND_PAIR_BYTES = 2 * 2 * D + 2 * REC + 4 + 2 * D  # k_new + v_new, record in/out, table entry, codes


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="3", help="workload id: 1..5 or 5p (default 3, the largest: MHA, "
                    "100 requests)")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the per-workload table (workloads 2, 4, 5, 5p timed after the main line)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the two-phase (chunked prefill) compression timing after the timed steps")
    ap.add_argument("--no-formats", action="store_true",
                    help="skip the comparison encodings (fixed64, sym_int8, fp8_e4m3) after the timed steps")
    ap.add_argument("--paged-input", action="store_true",
                    help="compress from a bf16 paged cache (dgq_compress_paged) instead of packed rows")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers (profiling captures; 0 = all of the workload's layers)")
    return ap.parse_args()


def workload(cfg):
    from synth import configs
    key = int(cfg) if cfg.isdigit() else cfg
    w = configs.WORKLOADS[key]
    lens = configs.seq_lens(w)
    bt, nb = configs.block_tables(w, lens)
    return w, lens, bt, nb, configs.cu_seqlens(lens)


def with_append_room(bt, nb, lens, bs, room):
    """The block table widened so that every request can grow by `room` tokens: fresh blocks
    (ids from nb upward) in the columns past each request's last block."""
    import numpy as np
    need = [(int(L) + room + bs - 1) // bs for L in lens]
    out = np.zeros((bt.shape[0], max(max(need), bt.shape[1])), dtype=np.int32)
    out[:, :bt.shape[1]] = bt
    nxt = nb
    for b, L in enumerate(lens):
        for j in range((int(L) + bs - 1) // bs, need[b]):
            out[b, j] = nxt
            nxt += 1
    return out, nxt


def algorithmic_bytes(w, lens):
    """Per layer: (decode bytes, compress bytes), from the shapes."""
    dec = 0
    for L in lens:
        L = int(L)
        dec += w.hkv * (2 * L * D + REC) + 4 * ((L + w.block_size - 1) // w.block_size)
        dec += w.hq * D * 2 * 2 + 2 * w.hkv * D * 2  # q in, out, k_new, v_new
    elems = 2 * int(sum(lens)) * w.hkv * D          # K and V elements
    comp = elems * 2 + elems * 1 + len(lens) * w.hkv * REC + 4 * len(lens)  # read bf16, write codes + records
    return dec, comp


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s)"


def src_hash(name):
    """Hash of a kernel's source file and of every shared device header it may include."""
    csrc = os.path.join(ROOT, "int8_group_quantized_gb300", "csrc")
    h = hashlib.sha256()
    for f in [name] + sorted(x for x in os.listdir(csrc) if x.endswith(".cuh")):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def ncu_traffic(kernel_src, workload_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    h = src_hash(kernel_src)
    with open(p) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split("\t")
            if len(parts) >= 4 and parts[0] == kernel_src and parts[1] == workload_name and parts[2] == h:
                return float(parts[3])
    return None


class ClockSampler:
    """SM clock, power and throttle reasons sampled while the timed region runs (read-only
    queries).  NVML through ctypes every 20 ms when the driver's NVML library loads (the GPU
    picked by its PCI bus id), else `nvidia-smi -lms 50`."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}  # nvmlClocksEventReason* masks

    def __init__(self, dev_index):
        self.proc = None
        self.dev = dev_index
        self.thread = None
        self.samples = []
        self.smax = None
        self.source = None

    def _nvml_handle(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None, None
        h = ctypes.c_void_p()
        try:
            import torch
            pr = torch.cuda.get_device_properties(self.dev)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                raise RuntimeError("no NVML device for that bus id")
        except Exception:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.dev), ctypes.byref(h)) != 0:
                return None, None
        return nv, h

    def _poll(self, nv, h):
        import ctypes
        clk, mw, reasons = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag:
            ok = nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0  # NVML_CLOCK_SM
            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
            get_reasons(h, ctypes.byref(reasons))
            if ok:
                self.samples.append((float(clk.value), mw.value / 1e3, int(reasons.value)))
            time.sleep(0.02)

    def start(self):
        import threading
        try:
            import ctypes
            nv, h = self._nvml_handle()
            if nv is not None:
                mx = ctypes.c_uint()
                if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                    self.smax = float(mx.value)
                self.stop_flag = False
                self.thread = threading.Thread(target=self._poll, args=(nv, h), daemon=True)
                self.thread.start()
                t0 = time.time()
                while not self.samples and time.time() - t0 < 2.0:  # the first sample is in
                    time.sleep(0.005)
                self.source = "nvml, 20 ms"
                return
        except Exception:
            self.thread = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 50 ms"
        except Exception:
            self.proc = None

    def stop(self):
        sm, reasons, smax, power = [], set(), self.smax, []
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join(timeout=2)
            for mhz, w, bits in self.samples:
                sm.append(mhz)
                power.append(w)
                for n, b in self.REASON_BITS.items():
                    if bits & b:
                        reasons.add(n)
        elif self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                return None
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax = float(f[2])
                    power.append(float(f[3]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "sm_mhz_min": min(sm),
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": round(max(power), 1) if power else None,
                "source": self.source}


# ------------------------------------------------------------------------------ CPU oracle

class OracleSample:
    """A bounded sample of the workload (the first `requests` requests of the first `layers`
    layers), generated once on the host; run() times the oracle's compress and fp64 decode
    attention over it."""

    def __init__(self, w, lens, layers=4, requests=8):
        import numpy as np
        import synth
        from synth import configs
        self.w = w
        self.sub = np.asarray(lens[:requests], dtype=np.int32)
        self.cu = configs.cu_seqlens(self.sub)
        nblk = [(int(L) + w.block_size - 1) // w.block_size for L in self.sub]
        self.bt = np.zeros((len(self.sub), max(1, max(nblk))), dtype=np.int32)
        off = 0
        for b, n in enumerate(nblk):
            self.bt[b, :n] = np.arange(off, off + n)
            off += n
        self.nb = max(off, 1)
        self.dec_b, self.comp_b = algorithmic_bytes(w, self.sub)
        self.layers = []
        for layer in range(layers):
            tabs = synth.span_tables(w.seed, layer, self.sub, w.hkv, w.rule)
            B = len(self.sub)
            self.layers.append((
                synth.fill_layer(w.seed, synth.STREAM_K, layer, self.cu, w.hkv, tabs),
                synth.fill_layer(w.seed, synth.STREAM_V, layer, self.cu, w.hkv, tabs),
                synth.fill_heads(w.seed, synth.STREAM_Q, layer, B, w.hq, 1.0),
                synth.fill_heads(w.seed, synth.STREAM_KNEW, layer, B, w.hkv, 0.15),
                synth.fill_heads(w.seed, synth.STREAM_VNEW, layer, B, w.hkv, 0.15)))
        self.desc = (f"oracle (single-threaded C) on {requests} of {len(lens)} requests x {layers} of "
                     f"{w.layers} layers of workload '{w.name}'")

    def run(self):
        """Returns (decode_bytes, decode_s, compress_bytes, compress_s)."""
        import oracle
        td = tc = 0.0
        for k, v, q, kn, vn in self.layers:
            t0 = time.perf_counter()
            kp, vp, table = oracle.compress(k, v, self.cu, self.w.hkv, self.w.block_size, self.bt, self.nb)
            t1 = time.perf_counter()
            oracle.paged_decode_attn(q, kn, vn, kp, vp, table, self.bt, self.sub)
            t2 = time.perf_counter()
            tc += t1 - t0
            td += t2 - t1
        n = len(self.layers)
        return self.dec_b * n, td, self.comp_b * n, tc


def host_cpu():
    """The host's CPU model and logical core count (the oracle baseline runs on one core)."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part") and not model:
                    model = line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    arm_parts = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
                 "0xd49": "Arm Neoverse N2"}  # /proc/cpuinfo "CPU part" of Arm server cores
    model = arm_parts.get(model.lower(), model)
    return {"model": model or platform.processor() or "unknown", "arch": platform.machine(),
            "nproc": os.cpu_count()}


def max_over_ranks(values, device, world):
    """The slowest rank's value of each timing (a replica run is as fast as its slowest GPU)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_gbs(bytes_per_step, steps, world, max_ms):
    """Whole-job GB/s of `world` replicas that each moved `bytes_per_step` per step."""
    return world * bytes_per_step * steps / (max_ms / 1e3) / 1e9


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w, lens, _, _, _ = workload(args.config)
    tot_d = tot_c = bd = bc = 0.0
    sample = OracleSample(w, lens, layers=1, requests=4)
    desc = sample.desc
    for i in range(args.warmup + args.steps):
        db, dt, cb, ct = sample.run()
        if i >= args.warmup:
            bd += db
            tot_d += dt
            bc += cb
            tot_c += ct
    value = bd / tot_d / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * (tot_d + tot_c) / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": f"{min(4, len(lens))} requests x 1 layer per step"},
        "compress_gbs": round(bc / tot_c / 1e9, 4),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc,
                         "host": host_cpu()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ GPU path

def setup_layers(w, lens, bt, nb, cu, dev, sp, nl, paged_input=False):
    """Every layer's inputs drawn on the GPU by the seeded generator (K/V, the step's q / k_new /
    v_new), and its own zeroed INT8 pools and records.  The step inputs of all layers sit in one
    buffer and the outputs in another, so that an end-to-end step moves each with one copy."""
    import numpy as np
    import torch
    import synth
    B, Hq, Hkv, bs = w.batch, w.hq, w.hkv, w.block_size
    T = int(cu[-1])
    d_cu = torch.from_numpy(cu).to(dev)
    d_bt = torch.from_numpy(bt).to(dev)
    d_lens = torch.from_numpy(lens).to(dev)
    layers = []
    n_q, n_kv = B * Hq * D, B * Hkv * D
    step_in = torch.empty(nl * (n_q + 2 * n_kv), dtype=torch.bfloat16, device=dev)
    step_out = torch.empty(nl * n_q, dtype=torch.bfloat16, device=dev)
    for l in range(nl):
        n, st, sg = synth.span_tables(w.seed, l, lens, Hkv, w.rule)
        tabs = tuple(torch.from_numpy(x).to(dev) for x in (n, st, sg))
        k = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
        v = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
        synth.dev_fill_layer(w.seed, synth.STREAM_K, l, d_cu, Hkv, tabs, T, k, sp)
        synth.dev_fill_layer(w.seed, synth.STREAM_V, l, d_cu, Hkv, tabs, T, v, sp)
        base = l * (n_q + 2 * n_kv)
        q = step_in[base:base + n_q].view(B, Hq, D)
        kn = step_in[base + n_q:base + n_q + n_kv].view(B, Hkv, D)
        vn = step_in[base + n_q + n_kv:base + n_q + 2 * n_kv].view(B, Hkv, D)
        synth.dev_fill_heads(w.seed, synth.STREAM_Q, l, B, Hq, 1.0, q, sp)
        synth.dev_fill_heads(w.seed, synth.STREAM_KNEW, l, B, Hkv, 0.15, kn, sp)
        synth.dev_fill_heads(w.seed, synth.STREAM_VNEW, l, B, Hkv, 0.15, vn, sp)
        layers.append(dict(
            k=k, v=v, q=q, kn=kn, vn=vn,
            kp=torch.zeros((nb, Hkv, bs, D), dtype=torch.uint8, device=dev),
            vp=torch.zeros((nb, Hkv, bs, D), dtype=torch.uint8, device=dev),
            table=torch.zeros((B, Hkv, REC), dtype=torch.uint8, device=dev),
            out=step_out[l * n_q:(l + 1) * n_q].view(B, Hq, D)))
    if paged_input:  # the same tokens in a bf16 paged cache laid out like the INT8 pools
        tok_blk = torch.from_numpy(np.concatenate(
            [bt[b, np.arange(int(L)) // bs] for b, L in enumerate(lens)]).astype(np.int64)).to(dev)
        tok_slot = torch.from_numpy(np.concatenate(
            [np.arange(int(L)) % bs for L in lens]).astype(np.int64)).to(dev)
        for L in layers:
            for name in ("k", "v"):
                src = torch.zeros((nb, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
                src[tok_blk, :, tok_slot, :] = L[name]
                L[name + "_src"] = src
    return layers, step_in, step_out, d_cu, d_bt, d_lens


class StepFns:
    """The three phases of a step over every layer, through the C ABI binding."""

    def __init__(self, dgq, layers, d_cu, d_bt, d_lens, max_seqlen, bs, cws, aws, pws, sp, paged_input=False):
        self.__dict__.update(dgq=dgq, layers=layers, d_cu=d_cu, d_bt=d_bt, d_lens=d_lens, ms=max_seqlen, bs=bs,
                             cws=cws, aws=aws, pws=pws, sp=sp, paged=paged_input)

    def compress_all(self):
        dgq = self.dgq
        for L in self.layers:
            if self.paged:
                dgq.dgq_compress_paged(L["k_src"], L["v_src"], self.d_bt, self.d_cu, self.ms, self.bs, self.d_bt,
                                       L["kp"], L["vp"], L["table"], self.cws, self.sp)
            else:
                dgq.dgq_compress(L["k"], L["v"], self.d_cu, self.ms, self.bs, self.d_bt, L["kp"], L["vp"], L["table"],
                                 self.cws, self.sp)

    def decode_all(self):
        for L in self.layers:
            self.dgq.dgq_paged_decode_attn(L["q"], L["kn"], L["vn"], L["kp"], L["vp"], L["table"], self.d_bt,
                                           self.d_lens, self.ms, L["out"], self.aws, self.sp)

    def append_all(self):  # the step's own token of every layer into its cache
        for L in self.layers:
            self.dgq.dgq_append(L["kn"], L["vn"], self.bs, self.d_bt, L["kp"], L["vp"], L["table"], self.pws,
                                self.sp)


def time_other_workload(cfg, dev, sp, peak, steps=5, warmup=2):
    """Compress and decode of every layer of another workload, timed like the main run (CUDA
    events on the launching stream around each phase; inputs resident in HBM, each layer its own
    buffers), for the per-workload table.  Frees everything before it returns."""
    import torch
    import int8_group_quantized_gb300 as dgq
    w, lens, bt, nb, cu = workload(cfg)
    B, Hq, Hkv, bs, nl = w.batch, w.hq, w.hkv, w.block_size, w.layers
    ms = int(lens.max())
    layers, step_in, step_out, d_cu, d_bt, d_lens = setup_layers(w, lens, bt, nb, cu, dev, sp, nl)
    cws = torch.zeros(dgq.dgq_compress_workspace_size(B, ms, Hkv), dtype=torch.uint8, device=dev)
    aws = torch.zeros(dgq.dgq_attn_workspace_size(B, Hq, Hkv, ms), dtype=torch.uint8, device=dev)
    fn = StepFns(dgq, layers, d_cu, d_bt, d_lens, ms, bs, cws, aws, None, sp)
    for _ in range(warmup):
        fn.compress_all()
        fn.decode_all()
    torch.cuda.synchronize()
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    stream = torch.cuda.current_stream()
    for e0, e1, e2 in ev:
        e0.record(stream)
        fn.compress_all()
        e1.record(stream)
        fn.decode_all()
        e2.record(stream)
    torch.cuda.synchronize()
    comp_ms = sum(a.elapsed_time(b) for a, b, _ in ev)
    dec_ms = sum(b.elapsed_time(c) for _, b, c in ev)
    err = dgq.dgq_workspace_error(cws, sp) or dgq.dgq_workspace_error(aws, sp)
    dec_b, comp_b = algorithmic_bytes(w, lens)
    dec_us, comp_us = dec_ms / (steps * nl) * 1e3, comp_ms / (steps * nl) * 1e3
    del layers, step_in, step_out, cws, aws, fn
    torch.cuda.empty_cache()
    return {"workload": w.name, "layers": nl, "steps": steps, "warmup": warmup,
            "decode_us_per_layer": round(dec_us, 2), "decode_gbs": round(dec_b / dec_us / 1e3, 1),
            "decode_frac_of_peak": round(dec_b / dec_us / 1e3 / peak, 4),
            "decode_token_heads_per_s": round(sum(int(L) + 1 for L in lens) * Hq / (dec_us / 1e6), 1),
            "compress_us_per_layer": round(comp_us, 2), "compress_gbs": round(comp_b / comp_us / 1e3, 1),
            "compress_frac_of_peak": round(comp_b / comp_us / 1e3 / peak, 4),
            "compress_kernel": "compress_cluster_kernel" if ms <= 4096 else "compress_kernel",
            "decode_bytes_per_layer": dec_b, "compress_bytes_per_layer": comp_b, "device_error": err}


def time_graph_step(dgq, layers, d_cu, d_bt, d_lens, max_seqlen, bs, cws, aws, pws, paged, dec_b, comp_b, peak,
                    steps, warmup=3):
    """The step (compress, decode, append of every layer) captured into three CUDA graphs, one per
    phase, and replayed: the same launches as the main run without the per-launch host and
    submission cost.  Timed like the main run (CUDA events around each phase's replay)."""
    import torch
    s = torch.cuda.Stream()
    fn = StepFns(dgq, layers, d_cu, d_bt, d_lens, max_seqlen, bs, cws, aws, pws, s.cuda_stream, paged)
    s.wait_stream(torch.cuda.current_stream())
    graphs = []
    for phase in (fn.compress_all, fn.decode_all, fn.append_all):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            phase()
        graphs.append(g)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    for _ in range(warmup):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in evs:
        for i, g in enumerate(graphs):
            e[i].record(cur)
            g.replay()
        e[3].record(cur)
    torch.cuda.synchronize()
    err = dgq.dgq_workspace_error(cws) or dgq.dgq_workspace_error(aws) or dgq.dgq_workspace_error(pws)
    nl = len(layers)
    us = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / (steps * nl) * 1e3 for i in range(3)]
    return {"what": "each phase of the step (every layer's launches) captured into one CUDA graph and replayed; "
                    "CUDA events around each replay",
            "steps": steps, "compress_us_per_layer": round(us[0], 2),
            "compress_gbs": round(comp_b / us[0] / 1e3, 1), "decode_us_per_layer": round(us[1], 2),
            "decode_gbs": round(dec_b / us[1] / 1e3, 1), "decode_frac_of_peak": round(dec_b / us[1] / 1e3 / peak, 4),
            "append_us_per_layer": round(us[2], 2), "device_error": int(err)}


def time_compress_e2e(w, layers, d_cu, d_bt, max_seqlen, bs, cws, sp, comp_b, nlayers=4, reps=3):
    """Compression end to end through the C ABI: per layer, the bf16 K and V come from pinned host
    memory (one copy each, on two copy streams, into one of two device buffer pairs, so that a
    layer's copies overlap the previous layer's compression), dgq_compress writes the layer's
    pools and records, and the records go back to pinned host memory; CUDA events around
    `nlayers` layers, `reps` passes after one warm pass.  Context for the compress figure: in
    serving, K/V are produced on the GPU by prefill and never cross the host link (the
    device-resident figure is compress_gbs)."""
    import torch
    import int8_group_quantized_gb300 as dgq
    use = layers[:nlayers]
    dev = use[0]["k"].device
    h_k = torch.empty(use[0]["k"].shape, dtype=torch.bfloat16).pin_memory()
    h_v = torch.empty_like(h_k).pin_memory()
    h_k.copy_(use[0]["k"])
    h_v.copy_(use[0]["v"])
    d_k = [torch.empty_like(use[0]["k"]) for _ in range(2)]
    d_v = [torch.empty_like(use[0]["v"]) for _ in range(2)]
    h_tab = torch.empty((len(use),) + tuple(use[0]["table"].shape), dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream()
    ks, vs = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_k = [torch.cuda.Event() for _ in range(2)]
    ev_v = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]  # buffer pair no longer read by a compression
    for e in ev_free:
        e.record(stream)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    n = 0
    for r in range(reps + 1):
        if r == 1:
            ev[0].record(stream)
            ks.wait_event(ev[0])  # no copy of the timed passes starts before the clock
            vs.wait_event(ev[0])
        for i, L in enumerate(use):
            b = n % 2
            n += 1
            for cs, dst, src, done in ((ks, d_k[b], h_k, ev_k[b]), (vs, d_v[b], h_v, ev_v[b])):
                cs.wait_event(ev_free[b])
                with torch.cuda.stream(cs):
                    dst.copy_(src, non_blocking=True)
                    done.record(cs)
            stream.wait_event(ev_k[b])
            stream.wait_event(ev_v[b])
            dgq.dgq_compress(d_k[b], d_v[b], d_cu, max_seqlen, bs, d_bt, L["kp"], L["vp"], L["table"], cws, sp)
            ev_free[b].record(stream)
            h_tab[i].copy_(L["table"], non_blocking=True)
    ev[1].record(stream)
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / (reps * len(use))
    h2d = 2 * h_k.numel() * 2
    d2h = h_tab[0].numel()
    del d_k, d_v
    return {"value": round(comp_b / (ms / 1e3) / 1e9, 1), "unit": "GB/s", "us_per_layer": round(ms * 1e3, 2),
            "h2d_bytes_per_layer": h2d, "d2h_bytes_per_layer": d2h, "layers": len(use), "reps": reps,
            "what": "dgq_compress with the layer's bf16 K/V copied from pinned host memory (K and V on two "
                    "copy streams, overlapping the previous layer's compression) and its records copied "
                    "back, per layer; GB/s over compression's algorithmic bytes"}


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import int8_group_quantized_gb300 as dgq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dgq.lib()

    w, lens, bt, nb, cu = workload(args.config)
    B, Hq, Hkv, bs, nl = w.batch, w.hq, w.hkv, w.block_size, w.layers
    bt, nb = with_append_room(bt, nb, lens, bs, APPEND_ROOM)
    if args.layers:
        nl = min(nl, args.layers)
    max_seqlen = int(lens.max())
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    layers, step_in, step_out, d_cu, d_bt, d_lens = setup_layers(w, lens, bt, nb, cu, dev, sp, nl,
                                                                  args.paged_input)
    cws = torch.zeros(dgq.dgq_compress_workspace_size(B, max_seqlen, Hkv), dtype=torch.uint8, device=dev)
    aws = torch.zeros(dgq.dgq_attn_workspace_size(B, Hq, Hkv, max_seqlen), dtype=torch.uint8, device=dev)
    pws = torch.zeros(dgq.dgq_append_workspace_size(), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    fn = StepFns(dgq, layers, d_cu, d_bt, d_lens, max_seqlen, bs, cws, aws, pws, sp, args.paged_input)
    compress_all, decode_all, append_all = fn.compress_all, fn.decode_all, fn.append_all

    for _ in range(args.warmup):
        compress_all()
        decode_all()
        append_all()
    torch.cuda.synchronize()

    # ---- timed region: K steps, each = compress all layers + decode all layers + append the
    # step's token to every layer's cache
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for e0, e1, e2, e3 in evs:
        e0.record(stream)
        compress_all()
        e1.record(stream)
        decode_all()
        e2.record(stream)
        append_all()
        e3.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    comp_ms = sum(e0.elapsed_time(e1) for e0, e1, _, _ in evs)
    dec_ms = sum(e1.elapsed_time(e2) for _, e1, e2, _ in evs)
    app_ms = sum(e2.elapsed_time(e3) for _, _, e2, e3 in evs)
    # medians over the timed steps (per step: all layers of the phase)
    medians = {"step_ms": statistics.median(e0.elapsed_time(e3) for e0, _, _, e3 in evs),
               "compress_ms": statistics.median(e0.elapsed_time(e1) for e0, e1, _, _ in evs),
               "decode_ms": statistics.median(e1.elapsed_time(e2) for _, e1, e2, _ in evs),
               "append_ms": statistics.median(e2.elapsed_time(e3) for _, _, e2, e3 in evs)}
    if clk:
        clk["timed_region_ms"] = round(total_ms, 2)
        clk["ms_x_median_mhz"] = round(total_ms * clk["sm_mhz"], 1)
    # parity spot check outside the timed region (layer 0 compressed again: the appends above
    # have grown its records)
    dgq.dgq_compress(layers[0]["k"], layers[0]["v"], d_cu, max_seqlen, bs, d_bt, layers[0]["kp"],
                     layers[0]["vp"], layers[0]["table"], cws, sp)
    torch.cuda.synchronize()
    checked = spot_check(w, lens, cu, bt, layers[0], rank)
    # segment counts of layer 0's (request, head) pairs, as the article's per-layer debug output
    n_seg = layers[0]["table"][:, :, 0:4].contiguous().view(torch.int32).cpu().numpy().ravel()
    seg_hist = {int(k): int(c) for k, c in zip(*np.unique(n_seg, return_counts=True))}
    err = (dgq.dgq_workspace_error(cws, sp) or dgq.dgq_workspace_error(aws, sp)
           or dgq.dgq_workspace_error(pws, sp))

    dec_b, comp_b = algorithmic_bytes(w, lens)
    dec_b_step, comp_b_step = dec_b * nl, comp_b * nl

    # ---- end-to-end through the public API: per step the step's decode inputs (q, k_new, v_new
    # of every layer) come from pinned host memory and the outputs go back to pinned host memory.
    # The copies run on two copy streams, one per direction, layer by layer: layer l's decode
    # waits only for layer l's inputs, and layer l's outputs travel while layer l + 1 decodes.
    h_in = torch.empty(step_in.shape, dtype=step_in.dtype, device="cpu").pin_memory()
    h_out = torch.empty(step_out.shape, dtype=step_out.dtype, device="cpu").pin_memory()
    h_in.copy_(step_in)
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    per_in, per_out = B * Hq * D + 2 * B * Hkv * D, B * Hq * D
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(nl)]
    ev_dec = [torch.cuda.Event() for _ in range(nl)]
    ev_start, ev_out = torch.cuda.Event(), torch.cuda.Event()

    def e2e_step():
        ev_start.record(stream)  # the previous step's readers of step_in / writers of step_out
        h2d_s.wait_event(ev_start)
        d2h_s.wait_event(ev_start)
        with torch.cuda.stream(h2d_s):
            for l in range(nl):
                step_in[l * per_in:(l + 1) * per_in].copy_(h_in[l * per_in:(l + 1) * per_in], non_blocking=True)
                ev_in[l].record(h2d_s)
        for l, L in enumerate(layers):
            stream.wait_event(ev_in[l])
            dgq.dgq_paged_decode_attn(L["q"], L["kn"], L["vn"], L["kp"], L["vp"], L["table"], d_bt, d_lens,
                                      max_seqlen, L["out"], aws, sp)
            ev_dec[l].record(stream)
        with torch.cuda.stream(d2h_s):
            for l in range(nl):
                d2h_s.wait_event(ev_dec[l])
                h_out[l * per_out:(l + 1) * per_out].copy_(step_out[l * per_out:(l + 1) * per_out],
                                                             non_blocking=True)
            ev_out.record(d2h_s)
        append_all()
        stream.wait_event(ev_out)  # the step ends once its outputs are in host memory

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(5, min(args.steps, 50))
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a0.elapsed_time(a1) / e2e_steps
    del h_in, h_out
    comp_e2e = time_compress_e2e(w, layers, d_cu, d_bt, max_seqlen, bs, cws, sp, comp_b) if rank == 0 else None

    ref0 = request0_reference(w, lens, layers[0]) if rank == 0 else None
    fidelity = fidelity_check(w, layers[0], ref0) if rank == 0 else None
    prefill = None
    if not args.no_prefill:
        prefill = time_prefill(w, lens, cu, bt, layers, d_cu, d_bt, d_lens, max_seqlen, sp, comp_b,
                               max(2, min(args.steps, 5)))
    split_v = None
    if not args.no_prefill:
        split_v = time_split_v(w, lens, layers, d_cu, d_bt, d_lens, max_seqlen, aws, sp, dec_b, comp_b, ref0,
                               max(2, min(args.steps, 5)))
    formats = None
    if not args.no_formats:
        formats = time_formats(w, lens, layers, d_cu, d_bt, d_lens, max_seqlen, aws, sp, dec_b, ref0,
                               max(3, min(args.steps, 10)))

    peak, peak_src = measured_peak()
    graph = None
    if rank == 0:
        graph = time_graph_step(dgq, layers, d_cu, d_bt, d_lens, max_seqlen, bs, cws, aws, pws, args.paged_input,
                                dec_b, comp_b, peak, max(5, min(args.steps, 20)))
    total_ms, comp_ms, dec_ms, app_ms, e2e_ms = max_over_ranks([total_ms, comp_ms, dec_ms, app_ms, e2e_ms], dev,
                                                              world)
    others = None
    if world == 1 and not args.no_others:  # the other workloads, each with every layer resident
        del layers, step_in, step_out, fn, compress_all, decode_all, append_all
        torch.cuda.empty_cache()
        others = {}
        for cfg in ("2", "4", "5", "5p"):
            if cfg != str(args.config):
                others[cfg] = time_other_workload(cfg, dev, sp, peak)

    if rank == 0:
        K = args.steps
        dec_gbs = replica_gbs(dec_b_step, K, world, dec_ms)
        comp_gbs = replica_gbs(comp_b_step, K, world, comp_ms)
        dec_launch_us = dec_ms / (K * nl) * 1e3
        comp_launch_us = comp_ms / (K * nl) * 1e3
        app_launch_us = app_ms / (K * nl) * 1e3
        app_b = B * Hkv * APPEND_PAIR_BYTES
        # the library compresses a call whose requests are all at most 4096 tokens with its
        # cluster kernel, longer ones with the grid-wide kernel
        comp_name, comp_src = (("compress_cluster_kernel", "dgq_compress_cluster.cu") if max_seqlen <= 4096
                               else ("compress_kernel", "dgq_compress.cu"))
        kernels = {
            "attn_kernel": {"bytes_per_launch": dec_b, "avg_launch_us": round(dec_launch_us, 2),
                            "achieved_gbs": round(dec_b / dec_launch_us / 1e3, 1), "src": "dgq_attn.cu",
                            "timed_with": "combine_kernel (merge of split pairs)"},
            comp_name: {"bytes_per_launch": comp_b, "avg_launch_us": round(comp_launch_us, 2),
                        "achieved_gbs": round(comp_b / comp_launch_us / 1e3, 1), "src": comp_src},
            "append_kernel": {"bytes_per_launch": app_b, "avg_launch_us": round(app_launch_us, 2),
                              "achieved_gbs": round(app_b / app_launch_us / 1e3, 1), "src": "dgq_append.cu",
                              "bound": "launch latency (one warp per (request, head) pair)"},
        }
        dom = max(kernels, key=lambda k: kernels[k]["avg_launch_us"])
        ach = kernels[dom]["achieved_gbs"]
        roofline = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                    "traffic": ncu_traffic(kernels[dom]["src"], w.name), "kernel": dom, "peak_source": peak_src}
        line = {
            "metric": METRIC, "value": round(dec_gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4),
            "median_ms": {k: round(v, 4) for k, v in medians.items()}, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": w.name, "layers": nl, "batch": B, "q_heads": Hq, "kv_heads": Hkv,
                       "head_dim": D, "block_size": bs, "seq_len": int(max_seqlen) if len(set(lens.tolist())) == 1
                       else f"{int(lens.min())}..{int(lens.max())}", "parallelism": f"replicas x{world}",
                       "compress_source": "bf16 paged cache" if args.paged_input else "packed bf16 rows",
                       "l2": "inputs larger than L2 (each layer has its own buffers; one step reads "
                             f"{(dec_b_step + comp_b_step) / 1e9:.1f} GB)"},
            "decode_frac_of_peak": round(dec_gbs / world / peak, 4),
            "compress_gbs": round(comp_gbs, 1),
            "compress_frac_of_peak": round(comp_gbs / world / peak, 4),
            "decode_token_heads_per_s": round(world * sum(int(L) + 1 for L in lens) * Hq * nl * K / (dec_ms / 1e3), 1),
            "roofline": roofline,
            "kernels": kernels,
            "e2e": {"value": round(world * dec_b_step / (e2e_ms / 1e3) / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "what": "decode step via the C ABI: every layer's q/k_new/v_new copied from pinned host "
                            "memory and its output copied back, per layer on two copy streams overlapping the "
                            "decode of the other layers, the decode of every layer, the step's token appended "
                            "to every layer's cache"},
            "segments": {"n_seg_histogram": seg_hist, "over": "(request, KV head) pairs of layer 0"},
            "fidelity": fidelity,
            "prefill_two_phase": prefill,
            "independent_v_segmentation": split_v,
            "formats": formats,
            "compress_e2e": comp_e2e,
            "graph": graph,
            "other_workloads": others,
            "gpu_launches": 4 * nl * K,  # per layer: compress, attention, merge, append
            "clocks": clk,
            "device_error": err,
            "parity_spot_check": checked,
        }
        if world == 1 and not args.no_cpu_baseline:
            sample = OracleSample(w, lens)
            db = dt = cb = ct = 0.0
            while dt + ct < 10.0:  # about 10 s of single-core oracle work
                a_, b_, c_, d_ = sample.run()
                db, dt, cb, ct = db + a_, dt + b_, cb + c_, ct + d_
            line["cpu_baseline"] = {"value": round(db / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                    "host": host_cpu(),
                                    "sample": sample.desc + f", repeated for {dt + ct:.1f} s",
                                    "compress_gbs": round(cb / ct / 1e9, 4)}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def spot_check(w, lens, cu, bt, layer0, rank):
    """Compress codes of request 0 / head 0 of layer 0 bit-exact vs the oracle (host-generated)."""
    if rank != 0:
        return None
    import numpy as np
    import oracle
    import synth
    L = int(lens[0])
    n, st, sg = synth.spans(w.seed, 0, 0, 0, L, w.rule)
    k = synth.fill_pair(w.seed, synth.STREAM_K, 0, 0, 0, L, n, st, sg)
    v = synth.fill_pair(w.seed, synth.STREAM_V, 0, 0, 0, L, n, st, sg)
    rec, kc, vc = oracle.compress_pair(k, v)
    kp = layer0["kp"].cpu().numpy()
    t = np.arange(L)
    gk = kp[bt[0, t // w.block_size], 0, t % w.block_size]
    grec = layer0["table"][0, 0].cpu().numpy().tobytes()
    return bool(np.array_equal(gk, kc) and grec == rec.tobytes())


def request0_reference(w, lens, layer0):
    """Request 0 of layer 0: its bf16 K/V (regenerated on the host), the step's q / k_new / v_new,
    and fp64 attention of all its query heads over the unquantised K/V."""
    import numpy as np
    import oracle
    import synth
    L = int(lens[0])
    k = np.zeros((L, w.hkv, D), dtype=np.uint16)
    v = np.zeros((L, w.hkv, D), dtype=np.uint16)
    for h in range(w.hkv):
        n, st, sg = synth.spans(w.seed, 0, 0, h, L, w.rule)
        k[:, h] = synth.fill_pair(w.seed, synth.STREAM_K, 0, 0, h, L, n, st, sg)
        v[:, h] = synth.fill_pair(w.seed, synth.STREAM_V, 0, 0, h, L, n, st, sg)
    q = layer0["q"][:1].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    kn = layer0["kn"][:1].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    vn = layer0["vn"][:1].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    cu = np.array([0, L], dtype=np.int32)
    lens1 = np.array([L], dtype=np.int32)
    raw = oracle.decode_attn_unquantised(q, kn, vn, k, v, cu, lens1)
    return dict(L=L, k=k, v=v, q=q, kn=kn, vn=vn, raw=raw)


def out0(layer0):
    """fp64 values of request 0's decode output (bf16) on layer 0."""
    import numpy as np
    got = layer0["out"][:1].contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    return (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def err_stats(a, b):
    import numpy as np
    d = np.abs(a - b)
    return {"max_abs": float(f"{d.max():.3e}"), "mean_abs": float(f"{d.mean():.3e}")}


def fidelity_check(w, layer0, ref):
    """Request 0 of layer 0, all query heads: the GPU's decode output against fp64 attention over
    the unquantised bf16 K/V (the encoding's error, reported as context) and against the oracle's
    fp64 attention over its own compressed cache (the kernel's error)."""
    import numpy as np
    import oracle
    L, k, v, q, kn, vn, raw = (ref[x] for x in ("L", "k", "v", "q", "kn", "vn", "raw"))
    got = out0(layer0)
    cu = np.array([0, L], dtype=np.int32)
    lens1 = np.array([L], dtype=np.int32)
    nb = (L + w.block_size - 1) // w.block_size
    bt = np.arange(nb, dtype=np.int32)[None]
    kp, vp, table = oracle.compress(k, v, cu, w.hkv, w.block_size, bt, nb)
    cache = oracle.paged_decode_attn(q, kn, vn, kp, vp, table, bt, lens1)
    err = err_stats
    comparison = {}  # the same attention with K/V through other 8-bit quantisers, fp64
    for scheme in oracle.COMPARISON_QUANTISERS:
        kd = np.stack([oracle.dequant_comparison(k[:, h], scheme) for h in range(w.hkv)], axis=1)
        vd = np.stack([oracle.dequant_comparison(v[:, h], scheme) for h in range(w.hkv)], axis=1)
        comparison[scheme] = err(oracle.decode_attn_dense(q[0], kn[0], vn[0], kd, vd), raw[0])
    return {"gpu_vs_unquantised": err(got, raw), "dgq_fp64_vs_unquantised": err(cache, raw),
            "gpu_vs_oracle": err(got, cache), "others_fp64_vs_unquantised": comparison,
            "sample": f"request 0 ({L} tokens), all {w.hq} query heads, layer 0; unquantised = fp64 "
                      "attention over the original bf16 K/V"}


def time_prefill(w, lens, cu, bt, layers, d_cu, d_bt, d_lens, max_seqlen, sp, comp_b, reps, max_layers=8):
    """Compression in two phases as chunked prefill would run it, outside the timed steps.  Per
    layer (up to `max_layers`), chunk by chunk: the chunk's bf16 K/V are written into a bf16 paged
    cache (standing in for the prefill kernels; not timed), then dgq_prefill_chunk_stats on that
    chunk (timed: the chunk is in L2, as right after prefill wrote it); at the end
    dgq_prefill_finish (timed).  Against it, dgq_compress_paged on a complete cache (launched back
    to back, as in the timed steps).  The
    chunk covers about 64 MB of K+V (at most 16384 tokens per request)."""
    import numpy as np
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = layers[0]["k"].device
    B, Hkv, bs = w.batch, w.hkv, w.block_size
    nb = layers[0]["kp"].shape[0]
    C = int(min(16384, max(16, (64 << 20) // (B * Hkv * 512)))) // 16 * 16
    nchunks = (int(lens.max()) + C - 1) // C
    chunks = []
    for c in range(nchunks):  # packed rows, blocks and slots of chunk c's tokens
        rows, blks, slots = [], [], []
        for b, L in enumerate(lens):
            t = np.arange(min(c * C, int(L)), min((c + 1) * C, int(L)))
            rows.append(int(cu[b]) + t)
            blks.append(bt[b, t // bs])
            slots.append(t % bs)
        beg = np.minimum(c * C, lens).astype(np.int32)
        end = np.minimum((c + 1) * C, lens).astype(np.int32)
        chunks.append(tuple(torch.from_numpy(np.concatenate(x).astype(np.int64)).to(dev) for x in (rows, blks, slots))
                      + (torch.from_numpy(beg).to(dev), torch.from_numpy(end).to(dev)))
    use = layers[:max_layers]
    ks = torch.zeros((nb, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    vs = torch.zeros_like(ks)
    W = (max_seqlen + 15) // 16
    stats = torch.zeros((B, Hkv, W, 8), dtype=torch.float32, device=dev)
    ws = torch.zeros(dgq.dgq_prefill_workspace_size(B, Hkv), dtype=torch.uint8, device=dev)
    cws = torch.zeros(dgq.dgq_compress_workspace_size(B, max_seqlen, Hkv), dtype=torch.uint8, device=dev)
    t_stats = t_fin = t_one = 0.0
    same = True
    for r in range(reps + 1):  # the first pass warms up
        for L in use:
            evs = []  # no synchronisation between chunks: each statistics launch queues behind the
            for rows, blks, slots, beg, end in chunks:  # chunk's write, so its events time the kernel
                ks[blks, :, slots, :] = L["k"][rows]  # the prefill's write of this chunk
                vs[blks, :, slots, :] = L["v"][rows]
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                dgq.dgq_prefill_chunk_stats(ks, vs, d_bt, beg, end, max_seqlen, stats, ws, sp)
                e1.record()
                evs.append((e0, e1))
            e2, e3 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            e2.record()
            dgq.dgq_prefill_finish(ks, vs, d_bt, d_lens, max_seqlen, stats, d_bt, L["kp"], L["vp"], L["table"], ws, sp)
            e3.record()
            torch.cuda.synchronize()
            s_ms = sum(a.elapsed_time(b) for a, b in evs)
            if r == reps and L is use[0]:  # the same records as the one-shot compress of the complete cache
                tab = L["table"].clone()
                dgq.dgq_compress_paged(ks, vs, d_bt, d_cu, max_seqlen, bs, d_bt, L["kp"], L["vp"], L["table"],
                                       cws, sp)
                torch.cuda.synchronize()
                same = bool(torch.equal(tab, L["table"]))
            if r > 0:
                t_stats += s_ms
                t_fin += e2.elapsed_time(e3)
    # the one-shot compress of the last layer's complete cache, launched back to back
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for r in range(reps + 1):
        if r == 1:
            ev[0].record()
        dgq.dgq_compress_paged(ks, vs, d_bt, d_cu, max_seqlen, bs, d_bt, use[-1]["kp"], use[-1]["vp"],
                               use[-1]["table"], cws, sp)
    ev[1].record()
    torch.cuda.synchronize()
    t_one = ev[0].elapsed_time(ev[1]) * len(use)
    # one layer's statistics calls (every chunk, on the complete cache) captured into a CUDA graph
    # and replayed: their device-side cost without the host's cost per call, which the timing
    # above includes whenever a call is too short to keep the GPU ahead of the host
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        for rows, blks, slots, beg, end in chunks:
            dgq.dgq_prefill_chunk_stats(ks, vs, d_bt, beg, end, max_seqlen, stats, ws, gs.cuda_stream)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for i in range(2):
        ev[i].record()
        if i == 0:
            for _ in range(reps):
                g.replay()
    torch.cuda.synchronize()
    t_graph = ev[0].elapsed_time(ev[1]) / reps
    n = reps * len(use)
    err = dgq.dgq_workspace_error(ws, sp) or dgq.dgq_workspace_error(cws, sp)
    st_us, fin_us, one_us = t_stats / n * 1e3, t_fin / n * 1e3, t_one / n * 1e3
    return {"chunk_tokens": C, "chunks": nchunks, "layers_timed": len(use),
            "stats_us_per_layer": round(st_us, 2), "finish_us_per_layer": round(fin_us, 2),
            "stats_graph_us_per_layer": round(t_graph * 1e3, 2),
            "total_us_per_layer": round(st_us + fin_us, 2), "gbs": round(comp_b / (st_us + fin_us) / 1e3, 1),
            "one_shot_paged_us_per_layer": round(one_us, 2), "one_shot_gbs": round(comp_b / one_us / 1e3, 1),
            "records_identical_to_one_shot": same, "device_error": err,
            "what": "statistics per prefill chunk right after the chunk is written (L2-hot), then one "
                    "finishing pass; bytes as for compress (2 B read + 1 B written per K/V value)"}


def time_split_v(w, lens, layers, d_cu, d_bt, d_lens, max_seqlen, aws, sp, dec_b, comp_b, ref0, reps):
    """Independent V segmentation (a group-selection variant) on the same workload, outside the
    timed steps: each layer compressed in two phases from a bf16 paged copy of its K/V (one
    statistics call over whole requests with V's variance, then the finish with a V record
    table), then decoded by the split instance of the decode kernel; CUDA-event time per layer
    over `reps` passes, and on rank 0 the GPU output of request 0 against fp64 attention over
    the unquantised K/V."""
    import numpy as np
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = layers[0]["k"].device
    B, Hkv, bs = w.batch, w.hkv, w.block_size
    nb = layers[0]["kp"].shape[0]
    bt = d_bt.cpu().numpy()
    cu = d_cu.cpu().numpy()
    blk = torch.from_numpy(np.concatenate([bt[b, np.arange(int(L)) // bs] for b, L in enumerate(lens)])
                           .astype(np.int64)).to(dev)
    slot = torch.from_numpy(np.concatenate([np.arange(int(L)) % bs for L in lens]).astype(np.int64)).to(dev)
    rows = torch.from_numpy(np.concatenate([int(cu[b]) + np.arange(int(L)) for b, L in enumerate(lens)])
                            .astype(np.int64)).to(dev)
    ks = torch.zeros((nb, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    vs = torch.zeros_like(ks)
    stats = torch.zeros((B, Hkv, (max_seqlen + 15) // 16, 8), dtype=torch.float32, device=dev)
    ws = torch.zeros(dgq.dgq_prefill_workspace_size(B, Hkv), dtype=torch.uint8, device=dev)
    vtab = torch.zeros_like(layers[0]["table"])
    zeros = torch.zeros(B, dtype=torch.int32, device=dev)
    t_st = t_fin = t_dec = 0.0
    use = layers[:8]
    for r in range(reps + 1):
        for L in use:
            ks[blk, :, slot, :] = L["k"][rows]
            vs[blk, :, slot, :] = L["v"][rows]
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            ev[0].record()
            dgq.dgq_prefill_chunk_stats(ks, vs, d_bt, zeros, d_lens, max_seqlen, stats, ws, sp, v_variance=True)
            ev[1].record()
            dgq.dgq_prefill_finish(ks, vs, d_bt, d_lens, max_seqlen, stats, d_bt, L["kp"], L["vp"], L["table"], ws,
                                   sp, v_seg_table=vtab)
            ev[2].record()
            dgq.dgq_paged_decode_attn_split(L["q"], L["kn"], L["vn"], L["kp"], L["vp"], L["table"], vtab, d_bt,
                                            d_lens, max_seqlen, L["out"], aws, sp)
            ev[3].record()
            torch.cuda.synchronize()
            if r > 0:
                t_st += ev[0].elapsed_time(ev[1])
                t_fin += ev[1].elapsed_time(ev[2])
                t_dec += ev[2].elapsed_time(ev[3])
            if r == reps and L is use[0] and ref0 is not None:
                fid = err_stats(out0(L), ref0["raw"])
    n = reps * len(use)
    st_us, fin_us, dec_us = t_st / n * 1e3, t_fin / n * 1e3, t_dec / n * 1e3
    res = {"stats_us_per_layer": round(st_us, 2), "finish_us_per_layer": round(fin_us, 2),
           "compress_gbs": round(comp_b / (st_us + fin_us) / 1e3, 1), "decode_us_per_layer": round(dec_us, 2),
           "decode_gbs": round(dec_b / dec_us / 1e3, 1),
           "device_error": dgq.dgq_workspace_error(ws, sp) or dgq.dgq_workspace_error(aws, sp),
           "what": "statistics with V's variance over whole requests + finish with V's own segments; decode "
                   "with both record tables"}
    if ref0 is not None:
        res["gpu_vs_unquantised"] = fid
    return res


def time_formats(w, lens, layers, d_cu, d_bt, d_lens, max_seqlen, aws, sp, dec_b, ref0, reps):
    """The comparison encodings on the same workload, outside the timed steps: every layer's bf16
    K/V encoded into its own pools (overwriting the DGQ cache), then the same decode over all
    layers; CUDA-event time per layer over `reps` passes, decode GB/s over the bytes each format
    reads (codes, plus the per-token parameters of fixed64), and, on rank 0, the GPU output of
    request 0 against fp64 attention over the unquantised K/V."""
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = layers[0]["k"].device
    B, Hkv, bs = w.batch, w.hkv, w.block_size
    nb = layers[0]["kp"].shape[0]
    ews = torch.zeros(dgq.dgq_encode_format_workspace_size(B, Hkv), dtype=torch.uint8, device=dev)
    par_bytes = 2 * 16 * Hkv * int(sum(int(L) for L in lens))  # fixed64: (min, scale) x 2 halves x K, V per token
    res = {}
    for fmt in ("fixed64", "sym_int8", "fp8_e4m3"):
        pars = [(torch.empty((nb, Hkv, bs, 4), dtype=torch.float32, device=dev),
                 torch.empty((nb, Hkv, bs, 4), dtype=torch.float32, device=dev)) if fmt == "fixed64"
                else (None, None) for _ in layers]

        def enc_all():
            for L, (kpar, vpar) in zip(layers, pars):
                dgq.dgq_encode_format(fmt, L["k"], L["v"], d_cu, max_seqlen, bs, d_bt, L["kp"], L["vp"], L["table"],
                                      ews, kpar, vpar, sp)

        def dec_all():
            for L, (kpar, vpar) in zip(layers, pars):
                dgq.dgq_paged_decode_attn_format(fmt, L["q"], L["kn"], L["vn"], L["kp"], L["vp"], L["table"], d_bt,
                                                 d_lens, max_seqlen, L["out"], aws, kpar, vpar, sp)
        for _ in range(2):
            enc_all()
            dec_all()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        enc_ms = dec_ms = 0.0
        for _ in range(reps):
            ev[0].record()
            enc_all()
            ev[1].record()
            dec_all()
            ev[2].record()
            torch.cuda.synchronize()
            enc_ms += ev[0].elapsed_time(ev[1])
            dec_ms += ev[1].elapsed_time(ev[2])
        err = dgq.dgq_workspace_error(ews, sp) or dgq.dgq_workspace_error(aws, sp)
        n = reps * len(layers)
        dec_us, enc_us = dec_ms / n * 1e3, enc_ms / n * 1e3
        rd = dec_b + (par_bytes if fmt == "fixed64" else 0)
        entry = {"encode_us_per_layer": round(enc_us, 2), "decode_us_per_layer": round(dec_us, 2),
                 "decode_bytes_per_layer": rd, "decode_gbs": round(rd / dec_us / 1e3, 1), "device_error": err}
        if ref0 is not None:
            import numpy as np
            import oracle
            got = out0(layers[0])
            kd = np.stack([oracle.dequant_comparison(ref0["k"][:, h], fmt) for h in range(Hkv)], axis=1)
            vd = np.stack([oracle.dequant_comparison(ref0["v"][:, h], fmt) for h in range(Hkv)], axis=1)
            want = oracle.decode_attn_dense(ref0["q"][0], ref0["kn"][0], ref0["vn"][0], kd, vd)
            entry["gpu_vs_unquantised"] = err_stats(got, ref0["raw"])
            entry["gpu_vs_oracle"] = err_stats(got[0], want)
        res[fmt] = entry
    return res


def torch_int16():
    import torch
    return torch.int16


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
