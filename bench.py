"""Benchmark of the MLA decode hot path (absorb -> latent attention -> W_UV up-projection).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dsv3_decode|tiny|ragged_paged|long_splitkv|mtp_causal]

Prints ONE JSON line (rank 0).  A step is one pass of the whole path over one batch
of the workload; the workload is DeepSeek-V3-shaped decode (B=64, H=128, T=4096,
d_c=512, d_r=64) unless --workload says otherwise.  With N>1 (torchrun) every rank
runs the same batch on its own GPU (independent sequences: weak scaling, no
collective on the data path); `value` is the whole-job tokens/s over the slowest rank.

--impl reference times the fp64 CPU oracle on this host's cores on a bounded sample
of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mla_latent_kv_70_b300 import inputs as I  # noqa: E402

METRIC = "MLA decode tokens/s (one attention layer: absorb + latent attention + W_UV)"
UNIT = "tokens/s"
ROW_BYTES = 1152
EVENT_EVERY = 4
E2E_SETS = 8
L2_BYTES = 126e6
DECODE_SOURCES = ["mla_latent_kv_70_b300/csrc/decode_sm103.cu",
                  "mla_latent_kv_70_b300/csrc/ptx_sm103.cuh",
                  "mla_latent_kv_70_b300/csrc/common.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv3_decode", choices=sorted(I.WORKLOADS) + sorted(EXTRA))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, world, device=None):
    """The largest of `x` over all ranks: a job takes as long as its slowest rank.  Uses the
    initialised process group (NCCL on GPUs: pass the rank's device; gloo: the CPU)."""
    if world <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_step, ms_per_step):
    """Units per second over the whole job: every rank processes `units_per_step` per step."""
    return world * units_per_step / (ms_per_step / 1e3)


def algorithmic(case):
    """Bytes and FLOPs of one latent-attention launch, by definition (no overheads)."""
    pairs = 0
    for T in case.seqlens:
        for s in range(case.S):
            pairs += T if not case.causal else max(0, min(T, T - case.S + s + 1))
    cache_bytes = ROW_BYTES * case.total_tokens
    io_bytes = case.B * case.S * case.H * (576 * 2 + 512 * 4 + 4)
    flops = 2.0 * case.H * (576 + 512) * pairs
    return cache_bytes, cache_bytes + io_bytes, flops


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get(
            "bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


def source_sha():
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        p = os.path.join(ROOT, rel)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, num_splits=None):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on the
    current kernel source with the same split count (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except ValueError:
        return None
    e = d.get(workload)
    if not e or e.get("source_sha") != source_sha():
        return None
    if num_splits is not None and e.get("num_splits") not in (None, num_splits):
        return None
    return e.get("dram_bytes_per_launch")


class CtypesNvml:
    """The few read-only NVML queries the clock sampler needs, called straight from the
    driver's libnvidia-ml through ctypes (for hosts where the pynvml module is missing).
    Mirrors the pynvml names ClockSampler uses; raises if the library or device is absent."""
    NVML_CLOCK_SM = 1

    def __init__(self, pci_bus_id: str):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.handle = ctypes.c_void_p()
        rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.handle))
        if rc != 0:
            raise RuntimeError(f"nvmlDeviceGetHandleByPciBusId_v2: {rc}")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _uint(self, fn, *args):
        v = self.ct.c_uint()
        if fn(self.handle, *args, self.ct.byref(v)) != 0:
            raise RuntimeError(fn.__name__)
        return v.value

    def nvmlDeviceGetClockInfo(self, h, clock):
        return self._uint(self.lib.nvmlDeviceGetClockInfo, self.ct.c_int(clock))

    def nvmlDeviceGetMaxClockInfo(self, h, clock):
        return self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.ct.c_int(clock))

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self.ct.c_ulonglong()
        if self.reasons_fn(self.handle, self.ct.byref(v)) != 0:
            raise RuntimeError("clock event reasons")
        return v.value


class ClockSampler:
    """SM clock and clock-event reasons sampled while `active` is set.

    NVML through pynvml (handle found by the device's UUID, so CUDA_VISIBLE_DEVICES
    remapping is harmless), else through ctypes on libnvidia-ml (handle found by the
    device's PCI bus id); if NVML is unusable, `nvidia-smi -lms` on that bus id, started
    before the warm-up and filtered to the samples stamped inside the timed region (or the
    two that bracket it, when the region is shorter than the sampling period)."""
    REASONS = {0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, dev):
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.active = False
        self.window = [None, None]   # host wall-clock times of the timed region
        self.error = None
        self._stop = False
        self.nv = None
        self.proc = None
        props = torch.cuda.get_device_properties(dev)
        try:
            import pynvml
            pynvml.nvmlInit()
            uuid = str(props.uuid)
            h = None
            for cand in (uuid, "GPU-" + uuid):
                try:
                    h = pynvml.nvmlDeviceGetHandleByUUID(cand)
                    break
                except Exception:  # noqa: BLE001
                    continue
            if h is None:
                h = pynvml.nvmlDeviceGetHandleByIndex(dev.index)
            self.h = h
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)
            self.nv = pynvml
        except Exception as e:  # noqa: BLE001
            self.error = f"nvml: {e!r}"
        self.bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        if self.nv is None:
            try:
                nv = CtypesNvml(self.bus)
                self.h = None
                self.max_mhz = nv.nvmlDeviceGetMaxClockInfo(None, nv.NVML_CLOCK_SM)
                self.nv = nv
                self.NVML_CLOCK_SM = nv.NVML_CLOCK_SM
                self.error = None
            except Exception as e:  # noqa: BLE001
                self.error = (self.error + "; " if self.error else "") + f"libnvidia-ml: {e!r}"
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()

    def _run(self):
        while not self._stop and self.nv is not None:
            if self.active:
                try:
                    self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                    r = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                    for bit in range(1, 64):       # bit 0 is gpu_idle
                        if r >> bit & 1:
                            self.reasons.add(self.REASONS.get(1 << bit, f"0x{1 << bit:x}"))
                except Exception as e:  # noqa: BLE001
                    self.error = f"nvml sample: {e!r}"
            time.sleep(0.0002)

    def begin(self):
        self.window[0] = time.time()
        self.active = True

    def end(self):
        self.active = False
        self.window[1] = time.time()

    SMI_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def start_smi(self):
        """Fallback sampler: nvidia-smi on this device, 20 ms period, from now on."""
        if self.nv is not None or self.proc is not None:
            return
        import shutil
        import subprocess
        if not shutil.which("nvidia-smi"):
            return
        self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.bus}", f"--query-gpu={self.SMI_FIELDS}",
                                      "--format=csv,noheader,nounits", "-lms", "20"],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

    def stop(self):
        self._stop = True
        self.t.join(timeout=1)
        if self.proc is not None:
            self.proc.terminate()
            out = self.proc.communicate(timeout=5)[0]
            mhz, max_mhz, reasons, how = smi_window(out.splitlines(), *self.window)
            self.samples += mhz
            self.max_mhz = max_mhz if max_mhz is not None else self.max_mhz
            self.reasons |= reasons
            if how:
                self.error = how
        d = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
             "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
             "samples": len(self.samples)}
        if self.error:
            d["note" if self.samples else "error"] = self.error
        return d


def smi_window(lines, t0, t1):
    """Samples of `nvidia-smi --query-gpu=<ClockSampler.SMI_FIELDS> --format=csv,noheader,
    nounits` stamped inside [t0, t1] (host epoch seconds).  When none falls inside (a region
    shorter than the period), the last sample before and the first after are used instead.
    Returns (sm MHz list, max MHz, reason names, note or None)."""
    import datetime
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    rows = []
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 7 or not f[1].isdigit():
            continue
        try:
            ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            continue
        rows.append((ts, f))
    if not rows or t0 is None or t1 is None:
        return [], None, set(), "nvidia-smi: no samples"
    inside = [f for ts, f in rows if t0 <= ts <= t1]
    note = None
    if not inside:
        before = [f for ts, f in rows if ts < t0][-1:]
        after = [f for ts, f in rows if ts > t1][:1]
        inside = before + after
        note = "nvidia-smi: region shorter than the 20 ms period; bracketing samples"
    max_mhz = None
    reasons = set()
    for f in inside:
        max_mhz = int(f[2]) if f[2].isdigit() else max_mhz
        for name, v in zip(names, f[3:]):
            if v.lower() == "active":
                reasons.add(name)
    return [int(f[1]) for f in inside], max_mhz, reasons, note


def blas_threads():
    """Threads the oracle's BLAS uses (numpy's OpenBLAS/MKL), else the usable cores."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def cpu_baseline(case, min_seconds=10.0, max_seqs=None):
    """Time the fp64 oracle (as it stands) over whole sequences of the workload."""
    import numpy as np  # noqa: F401
    import oracle as O
    w_uk, w_uv = (w.double().numpy() for w in I.weights(case))
    cores = blas_threads()
    tokens = 0
    seqs = 0
    t0 = time.perf_counter()
    b = 0
    max_seqs = max_seqs or 4 * case.B
    while seqs == 0 or (time.perf_counter() - t0 < min_seconds and seqs < max_seqs):
        T = case.seqlens[b]
        rows = I.seq_rows(case, b)[:T].double().numpy()
        qn, qr = I.seq_queries(case, b)
        qn, qr = qn.double().numpy(), qr.double().numpy()
        if case.rope:
            import numpy as np
            rows[:, 512:] = O.rope_interleaved(rows[:, 512:], np.arange(T), case.theta)
            pos = np.array([T - case.S + s for s in range(case.S)], dtype=np.float64)
            qr = O.rope_interleaved(qr, pos[:, None], case.theta)
        q_lat = O.absorb_q(qn, w_uk)
        o_lat, _ = O.decode_absorbed_seq(q_lat, qr, rows[:, :512], rows[:, 512:], case.scale,
                                         case.causal)
        O.out_proj_uv(o_lat, w_uv)
        tokens += case.S
        seqs += 1
        b = (b + 1) % case.B
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{seqs} whole sequences of {case.name} (T={case.seqlens[0] if len(set(case.seqlens)) == 1 else 'ragged'}, "
                      f"H={case.H}) through absorb + fp64 absorbed attention + W_UV, {dt:.1f} s"}


def run_reference(args, case):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    times = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(case, min_seconds=0.0, max_seqs=1)  # one sequence per step
        if i >= args.warmup:
            times.append(case.S / r["value"])
    step_s = sum(times) / len(times)
    value = case.S / step_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "B": case.B, "S": case.S, "H": case.H,
                       "T": case.seqlens[0], "step": "one sequence of the batch per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                             "cores": r["cores"],
                             "sample": "one whole sequence per step (absorb + fp64 absorbed attention + W_UV)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# The two paths beside the decode step: prefill of a 4096-token prompt in the expanded
# order, and the DeepSeek-V3 decode step on pre-fused weights (W_UQ W_UK^T, W_UV W_O).
# ----------------------------------------------------------------------------
EXTRA = {
    "prefill_4k": "prefill of one 4096-token prompt, H=128 (mla_prefill: K_h, V_h built, causal attention)",
    "dsv3_fused": "DeepSeek-V3 decode step on pre-fused weights: c^Q W_UQK -> latent attention -> "
                  "sum_h z_h W_UVO[h] (d_cq=1536, d_model=4096)",
    "dsv3_fp8": "DeepSeek-V3 decode step over the FP8 latent cache (E4M3 latent + bf16 k^R, 640-byte rows, "
                "power-of-two scale per row, quantized by mla_quantize_fp8 before timing)",
}


def prefill_flops(B, T_q, T_kv, H):
    pairs = B * sum(min(T_kv, T_kv - T_q + i + 1) for i in range(T_q))
    return 2.0 * H * pairs * (192 + 128) + 2.0 * B * T_kv * 512 * 256 * H


def cpu_baseline_extra(name, case, min_seconds=10.0):
    """The oracle on a bounded sample of the extra workloads (a few heads of the prompt,
    or whole sequences of the fused decode), scaled to the workload's unit."""
    import numpy as np
    import oracle as O
    cores = blas_threads()
    t0 = time.perf_counter()
    d = lambda t: t.double().numpy()
    if name == "prefill_4k":
        T = case.seqlens[0]
        rows = d(I.seq_rows(case, 0)[:T])
        qn, qr = (d(t) for t in I.seq_queries(case, 0))
        w_uk, w_uv = (d(w) for w in I.weights(case))
        heads = 0
        while heads == 0 or (time.perf_counter() - t0 < min_seconds and heads < case.H):
            h = [heads]
            O.decode_expanded_seq(qn[:, h], qr[:, h], rows[:, :512], rows[:, 512:], w_uk[h], w_uv[h],
                                  case.scale, causal=True)
            heads += 1
        dt = time.perf_counter() - t0
        value = case.S / (dt * case.H / heads)
        sample = f"{heads} of {case.H} heads of the {T}-token prompt (fp64 expanded attention), {dt:.1f} s, scaled to all heads"
    elif name == "dsv3_fp8":
        w_uk, w_uv = (d(w) for w in I.weights(case))
        seqs = 0
        while seqs == 0 or (time.perf_counter() - t0 < min_seconds and seqs < case.B):
            T = case.seqlens[seqs]
            codes, kr, scales = O.quantize_fp8_rows(d(I.seq_rows(case, seqs)[:T]))
            rows = O.dequantize_fp8_rows(codes, kr, scales)
            qn, qr = (d(t) for t in I.seq_queries(case, seqs))
            o_lat, _ = O.decode_absorbed_seq(O.absorb_q(qn, w_uk), qr, rows[:, :512], rows[:, 512:], case.scale)
            O.out_proj_uv(o_lat, w_uv)
            seqs += 1
        dt = time.perf_counter() - t0
        value = seqs * case.S / dt
        sample = f"{seqs} whole sequences (E4M3 quantization, absorbed fp64 attention, W_UV), {dt:.1f} s"
    else:
        w_uk, w_uv = (d(w) for w in I.weights(case))
        w_uq, w_o = d(I.query_side_weights(case)), d(I.output_weights(case))
        seqs = 0
        while seqs == 0 or (time.perf_counter() - t0 < min_seconds and seqs < case.B):
            T = case.seqlens[seqs]
            rows = d(I.seq_rows(case, seqs)[:T])
            q_nope = np.einsum("si,hik->shk", d(I.seq_c_q(case, seqs)), w_uq)
            q_lat = O.absorb_q(q_nope, w_uk)
            o_lat, _ = O.decode_absorbed_seq(q_lat, d(I.seq_queries(case, seqs)[1]), rows[:, :512], rows[:, 512:],
                                             case.scale)
            O.out_proj_heads(O.out_proj_uv(o_lat, w_uv), w_o)
            seqs += 1
        dt = time.perf_counter() - t0
        value = seqs * case.S / dt
        sample = f"{seqs} whole sequences (c^Q W_UQ, absorbed fp64 attention, W_UV, W_O), {dt:.1f} s"
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}


def pipelined_e2e(sets, pinned, steps, warmup, stream, barrier, lanes=8):
    """Time `steps` end-to-end steps through the public API, as a serving loop runs them.

    `sets` holds buffer sets (device inputs, device result, step(stream)); `pinned` the step's
    inputs in pinned host memory, one per device input.  Consecutive steps take the sets in
    turn.  The compute of the steps runs in order on one stream, as in the device-timed run,
    each step one CUDA graph replay.  A step's inputs are copied in on a copy-in stream ahead
    of its compute, and its result is copied out to pinned host memory on a copy-out stream
    behind it (set k uses copy streams k mod `lanes`).  Both copies go by the copy engine and
    overlap the compute of the neighbouring steps; events keep a set's buffers from being
    overwritten while an earlier step still uses them.  The streams are the loop's own
    (created here, non-blocking), joined to `stream` by events at the start and the end.
    Returns (ms for all steps, bytes in per step, bytes out per step).
    """
    from cuda.bindings import runtime as rt

    def check(res):
        err = res[0] if isinstance(res, tuple) else res
        assert err == rt.cudaError_t.cudaSuccess, err
        return res[1] if isinstance(res, tuple) and len(res) > 1 else None

    n, lanes = len(sets), min(lanes, len(sets))
    torch.cuda.synchronize()                      # the sets' buffers were filled on `stream`

    def new_stream():
        return check(rt.cudaStreamCreateWithFlags(rt.cudaStreamNonBlocking))
    h_comp = new_stream()
    h_in = [new_stream() for _ in range(lanes)]
    h_out = [new_stream() for _ in range(lanes)]
    comp = torch.cuda.ExternalStream(int(h_comp))
    outs = [torch.empty(res.shape, dtype=res.dtype).pin_memory() for _, res, _ in sets]
    graphs = []
    for _, _, run in sets:
        run(comp)                                 # one eager step per set before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=comp):
            run(comp)
        graphs.append(g)

    # The loop calls the runtime directly (no torch wrappers): eleven calls per step, each
    # well under a microsecond on the host.
    def events(count):
        return [check(rt.cudaEventCreateWithFlags(rt.cudaEventDisableTiming)) for _ in range(count)]
    landed, done, read = events(n), events(n), events(n)   # per set: inputs on the device,
    #                                                         compute finished, result on the host
    fork, joins = events(1)[0], events(1 + 2 * lanes)
    execs = [rt.cudaGraphExec_t(init_value=g.raw_cuda_graph_exec()) for g in graphs]
    to_dev, to_host = rt.cudaMemcpyKind.cudaMemcpyHostToDevice, rt.cudaMemcpyKind.cudaMemcpyDeviceToHost
    copies_in = [[(dst.data_ptr(), src.data_ptr(), src.numel() * src.element_size())
                  for src, dst in zip(pinned, ins)] for ins, _, _ in sets]
    copy_out = [(out.data_ptr(), res.data_ptr(), out.numel() * out.element_size())
                for out, (_, res, _) in zip(outs, sets)]
    ours = [h_comp] + h_in + h_out

    def one(i):
        k = i % n
        c_in, c_out = h_in[k % lanes], h_out[k % lanes]
        check(rt.cudaStreamWaitEvent(c_in, done[k], 0))       # the set's last step read its inputs
        for dst, src, nbytes in copies_in[k]:
            check(rt.cudaMemcpyAsync(dst, src, nbytes, to_dev, c_in))
        check(rt.cudaEventRecord(landed[k], c_in))
        check(rt.cudaStreamWaitEvent(h_comp, landed[k], 0))
        check(rt.cudaStreamWaitEvent(h_comp, read[k], 0))     # the set's last result was read back
        check(rt.cudaGraphLaunch(execs[k], h_comp))
        check(rt.cudaEventRecord(done[k], h_comp))
        check(rt.cudaStreamWaitEvent(c_out, done[k], 0))
        dst, src, nbytes = copy_out[k]
        check(rt.cudaMemcpyAsync(dst, src, nbytes, to_host, c_out))
        check(rt.cudaEventRecord(read[k], c_out))

    # Every set's graph is launched (and so uploaded) at least once before the timed steps.
    for i in range(max(warmup, n)):
        one(i)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    check(rt.cudaEventRecord(fork, stream.cuda_stream))
    for h in ours:
        check(rt.cudaStreamWaitEvent(h, fork, 0))
    for i in range(steps):
        one(i)
    for h, ev in zip(ours, joins):
        check(rt.cudaEventRecord(ev, h))
        check(rt.cudaStreamWaitEvent(stream.cuda_stream, ev, 0))
    e1.record(stream)
    barrier()
    for ev in landed + done + read + joins + [fork]:
        check(rt.cudaEventDestroy(ev))
    del graphs, comp
    for h in ours:
        check(rt.cudaStreamDestroy(h))
    h2d = sum(t.numel() * t.element_size() for t in pinned)
    return e0.elapsed_time(e1), h2d, outs[0].numel() * outs[0].element_size()


def run_extra(args):
    name = args.workload
    rank, world, local = dist_env()
    if name == "prefill_4k":
        case = I.make_case("prefill_4k", 1, 4096, 128, [4096], causal=True)
    else:
        case = I.dsv3()
    if args.impl == "reference":
        if rank == 0:
            r = cpu_baseline_extra(name, case, min_seconds=2.0)
            print(json.dumps({"impl": "reference", "metric": METRIC_EXTRA[name], "value": r["value"], "unit": UNIT,
                              "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": case.B * case.S / r["value"] * 1e3, "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                              "config": {"workload": name, "description": EXTRA[name]}, "cpu_baseline": r,
                              "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
        return
    import mla_latent_kv_70_b300 as mla
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    assert args.warmup >= 3, "at least 3 warm-up steps"
    B, S, H = case.B, case.S, case.H
    w_uk, w_uv = (w.to(dev) for w in I.weights(case))
    qn_h, qr_h = I.queries(case)
    kv = I.cache(case, device=dev)
    # make_set() allocates one set of the step's per-step buffers (device inputs, output,
    # scratch) and returns (device inputs, result, step(stream, marks)); the weights and the
    # cache are shared by all sets.
    if name == "prefill_4k":
        T = case.seqlens[0]
        inputs_h = [qn_h, qr_h]

        def make_set():
            q_nope, q_rope = qn_h.to(dev), qr_h.to(dev)
            o = torch.empty(B, S, H, 128, device=dev)
            lse = torch.empty(B, S, H, device=dev)
            ws = torch.empty(mla.mla_prefill_workspace_bytes(B, case.t_cap, H), dtype=torch.uint8, device=dev)

            def step(st, marks=None):
                if marks:
                    marks(0)
                mla.mla_prefill(q_nope, q_rope, kv, T, w_uk, w_uv, o, lse, scale=case.scale, workspace=ws,
                                stream=st)
                if marks:
                    marks(1)
            return [q_nope, q_rope], o, step
        flops = prefill_flops(B, S, T, H)
        alg_bytes = B * T * 1152 + B * S * H * (192 * 2 + 128 * 4 + 4) + 2 * H * 512 * 128 * 2
        kernel = "mla_prefill (K_h, V_h expansion + causal attention)"
        kernels_per_step = 2        # k_expand_kv, k_prefill_attn
    elif name == "dsv3_fp8":
        kv8 = torch.empty(case.B, case.t_cap, I.FP8_ROW, dtype=torch.uint8, device=dev)
        kv_sc = torch.empty(case.B, case.t_cap, device=dev)
        mla.mla_quantize_fp8(kv.view(-1, I.ROW), kv8.view(-1, I.FP8_ROW), kv_sc.view(-1))
        del kv
        seqlens = torch.tensor(case.seqlens, dtype=torch.int32, device=dev)
        inputs_h = [qn_h, qr_h]

        def make_set():
            q_nope, q_rope = qn_h.to(dev), qr_h.to(dev)
            dstep = mla.DecodeStep(B, S, H, w_uk, w_uv, max_seqlen=max(case.seqlens), seqlens=case.seqlens)

            def step(st, marks=None):
                mla.mla_absorb_q(q_nope, q_rope, w_uk, None, case.theta, dstep.q_cat, st)
                if marks:
                    marks(0)
                mla.mla_decode_latent_fp8(dstep.q_cat, kv8, kv_sc, seqlens, dstep.o_lat, dstep.lse,
                                          scale=case.scale, max_seqlen=dstep.max_seqlen,
                                          num_splits=dstep.num_splits, workspace=dstep.workspace,
                                          status=dstep.status, stream=st)
                if marks:
                    marks(1)
                mla.mla_out_proj_uv(dstep.o_lat, w_uv, dstep.o, st)
            return [q_nope, q_rope], dstep.o, step
        rows_read = sum(case.seqlens)
        flops = 2.0 * B * S * H * (576 + 512) * rows_read / B
        alg_bytes = rows_read * (I.FP8_ROW + 4) + B * S * H * (1152 + 2048 + 4)
        kernel = "mla_decode_latent_fp8 (E4M3 tiles widened to bf16 in shared memory)"
        kernels_per_step = 3        # k_absorb_q, k_decode_sm103, k_out_proj_uv
    else:
        w_uq, w_o = I.query_side_weights(case).to(dev), I.output_weights(case).to(dev)
        d_cq, d_model = w_uq.shape[1], w_o.shape[2]
        w_uqk = torch.empty(H, d_cq, 512, dtype=torch.bfloat16, device=dev)
        w_uvo = torch.empty(H, 512, d_model, dtype=torch.bfloat16, device=dev)
        mla.mla_fuse_weights(w_uq, w_uk, w_uv, w_o, w_uqk, w_uvo)
        c_q_h = I.c_q(case)
        seqlens = torch.tensor(case.seqlens, dtype=torch.int32, device=dev)
        splits = mla.mla_decode_num_splits(B, S, H, max(case.seqlens))
        dws_bytes = max(mla.mla_decode_workspace_bytes(B, S, H, splits, max(case.seqlens)), 16)
        inputs_h = [c_q_h, qr_h]

        def make_set():
            c_q, q_rope = c_q_h.to(dev), qr_h.to(dev)
            q_cat = torch.empty(B, S, H, 576, dtype=torch.bfloat16, device=dev)
            o_lat = torch.empty(B, S, H, 512, device=dev)
            lse = torch.empty(B, S, H, device=dev)
            out = torch.empty(B, S, d_model, device=dev)
            ws = torch.empty(mla.mla_out_proj_fused_workspace_bytes(B, S, H), dtype=torch.uint8, device=dev)
            dws = torch.empty(dws_bytes, dtype=torch.uint8, device=dev)

            def step(st, marks=None):
                mla.mla_absorb_q_fused(c_q, q_rope, w_uqk, None, case.theta, q_cat, st)
                mla.mla_decode_latent(q_cat, kv, seqlens, o_lat, lse, scale=case.scale,
                                      max_seqlen=max(case.seqlens), num_splits=splits, workspace=dws, stream=st)
                if marks:
                    marks(0)
                mla.mla_out_proj_fused(o_lat, w_uvo, out, ws, st)
                if marks:
                    marks(1)
            return [c_q, q_rope], out, step
        flops = 2.0 * B * S * H * 512 * d_model
        alg_bytes = H * 512 * d_model * 2 + B * S * H * 512 * (4 + 2 + 2) + B * S * d_model * 4
        kernel = "mla_out_proj_fused (sum_h z_h W_UVO[h], the dominant call)"
        # k_gemm + k_rope_slice (absorb), k_decode_sm103, k_f32_to_bf16 + k_gemm (output
        # projection; a driver memset zeroes the split-K output beside them)
        kernels_per_step = 5
    set0 = make_set()
    step = set0[2]

    stream = torch.cuda.current_stream()
    clocks = ClockSampler(dev)
    clocks.start_smi()
    for _ in range(args.warmup):
        step(stream)
    torch.cuda.synchronize()
    from cuda.bindings import runtime as cudart
    # Event nodes around the dominant call of every EVENT_EVERY-th step give its duration
    # inside the timed run.  An event node between two kernels keeps the second from
    # starting early under programmatic dependent launch, so the other steps carry none.
    evs = {i: (cudart.cudaEventCreate()[1], cudart.cudaEventCreate()[1]) for i in range(0, args.steps, EVENT_EVERY)}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
        cs = torch.cuda.current_stream()
        for i in range(args.steps):
            def marks(j, i=i):
                err = cudart.cudaEventRecordWithFlags(evs[i][j], cs.cuda_stream, cudart.cudaEventRecordExternal)[0]
                assert err == cudart.cudaError_t.cudaSuccess, err
            step(cs, marks if i in evs else None)
    graph.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.begin()
    start.record(stream)
    graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    clocks.end()
    total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    part_s = statistics.mean(cudart.cudaEventElapsedTime(a, b)[1] for a, b in evs.values()) / 1e3
    for a, b in evs.values():
        cudart.cudaEventDestroy(a)
        cudart.cudaEventDestroy(b)
    clock_info = clocks.stop()

    # End to end through the public API over several buffer sets (pipelined_e2e), as for the
    # decode workload.  A prefill set holds ~0.75 GB, so that workload takes three sets.
    n_sets = 3 if name == "prefill_4k" else E2E_SETS
    sets = [set0] + [make_set() for _ in range(n_sets - 1)]

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
    e2e_ms, h2d, d2h = pipelined_e2e(sets, [t.pin_memory() for t in inputs_h], args.steps, args.warmup,
                                     stream, barrier)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    hbm, tf_burst, _, peak_kind = measured_peaks()
    t_hbm, t_tc = alg_bytes / (hbm * 1e9), flops / (tf_burst * 1e12)
    if t_tc >= t_hbm:
        roof = {"bound": "tensor", "achieved": flops / part_s / 1e12, "peak": tf_burst, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": alg_bytes / part_s / 1e9, "peak": hbm, "unit": "GB/s"}
    roof.update({"frac": roof["achieved"] / roof["peak"],
                 "traffic": recorded_traffic(name, 1) if name == "dsv3_fp8" else None, "kernel": kernel,
                 "peak_source": f"{peak_kind} (MEASURED_PEAKS.json burst)", "kernel_us": part_s * 1e6,
                 "algorithmic_bytes": alg_bytes, "flops": flops, "roofline_us": max(t_hbm, t_tc) * 1e6})
    tokens = B * S
    line = {"metric": METRIC_EXTRA[name], "value": whole_job_rate(world, tokens, total_ms / args.steps),
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": name, "description": EXTRA[name], "B": B, "S": S, "H": H,
                       "T": case.seqlens[0], "l2": "inputs larger than L2",
                       "timing": f"cuda graph of the timed steps; the dominant call timed by event "
                                 f"nodes on every {EVENT_EVERY}th step",
                       "parallelism": f"dp{world} (independent replicas, no collective)"},
            "clocks": clock_info,
            "e2e": {"value": whole_job_rate(world, tokens, e2e_ms / args.steps), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * kernels_per_step,
            "roofline": roof}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_extra(name, case)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


METRIC_EXTRA = {"prefill_4k": "MLA prefill tokens/s (one attention layer, expanded order)",
                "dsv3_fused": "MLA decode tokens/s on pre-fused weights (one attention layer: "
                              "c^Q W_UQK + latent attention + sum_h z_h W_UVO[h])",
                "dsv3_fp8": "MLA decode tokens/s over the FP8 latent cache (one attention layer: "
                            "absorb + latent attention + W_UV)"}


def main():
    args = parse()
    if args.workload in EXTRA:
        run_extra(args)
        return
    case = I.WORKLOADS[args.workload]()
    if args.impl == "reference":
        run_reference(args, case)
        return

    import mla_latent_kv_70_b300 as mla
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    assert args.warmup >= 3, "at least 3 warm-up steps"

    # Inputs resident in HBM before timing.  A cache smaller than L2 is replicated so
    # that consecutive timed steps read different copies, more bytes in all than L2
    # holds, and each step's cache reads come from HBM.
    kv = I.cache(case, device=dev)
    cache_b, _, _ = algorithmic(case)
    n_copies = 1 if cache_b > L2_BYTES else min(256, math.ceil(2 * L2_BYTES / cache_b))
    qn, qr = I.queries(case)
    w_uk, w_uv = (w.to(dev) for w in I.weights(case))
    q_nope, q_rope = qn.to(dev), qr.to(dev)
    seqlens = torch.tensor(case.seqlens, dtype=torch.int32, device=dev)
    block_table = case.block_table.to(dev) if case.paged else None
    q_pos = case.q_positions().to(dev) if case.rope else None
    if case.rope:
        pos = (I.pool_positions(case).to(dev) if case.paged else
               torch.arange(case.t_cap, dtype=torch.int32, device=dev).repeat(case.B))
        mla.mla_rope_inplace(kv, 576, pos.numel(), 512, pos, case.theta)
    kvs = [kv] + [kv.clone() for _ in range(n_copies - 1)]
    step = mla.DecodeStep(case.B, case.S, case.H, w_uk, w_uv, max_seqlen=max(case.seqlens),
                          num_splits=case.num_splits, causal=case.causal, rope_theta=case.theta,
                          total_rows=case.total_tokens, seqlens=case.seqlens)
    stream = torch.cuda.current_stream()

    def run_step(st, marks=None, kv=kv):
        """One step on stream `st`; `marks(i)` records the decode boundaries."""
        mla.mla_absorb_q(q_nope, q_rope, w_uk, q_pos, case.theta, step.q_cat, st)
        if marks:
            marks(0)
        mla.mla_decode_latent(step.q_cat, kv, seqlens, step.o_lat, step.lse, scale=case.scale,
                              max_seqlen=step.max_seqlen, block_table=block_table,
                              causal=case.causal, num_splits=step.num_splits,
                              workspace=step.workspace, status=step.status, stream=st)
        if marks:
            marks(1)
        mla.mla_out_proj_uv(step.o_lat, w_uv, step.o, st)

    clocks = ClockSampler(dev)
    clocks.start_smi()          # no-op with NVML; nvidia-smi needs a moment to start
    for _ in range(args.warmup):
        run_step(stream)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # The K timed steps are captured once into a CUDA graph (the library makes no host
    # synchronisation, so a decode step is capturable, as serving engines run it) and
    # replayed as one launch: no host launch gaps between the kernels.  Event-record
    # nodes around the decode of every fourth step give the decode kernel's duration
    # inside the same run.  An event node between two kernels stops the next kernel from
    # starting early under programmatic dependent launch (about 12 us per step here), so
    # the other steps carry none and keep the overlap a serving loop gets.
    timing = (f"cuda graph of the timed steps; decode timed by event nodes on every "
              f"{EVENT_EVERY}th step")
    try:
        from cuda.bindings import runtime as cudart
        sampled = list(range(0, args.steps, EVENT_EVERY))
        evs = {i: (cudart.cudaEventCreate()[1], cudart.cudaEventCreate()[1]) for i in sampled}
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.graph(graph, stream=cap):
            cs = torch.cuda.current_stream()
            for i in range(args.steps):
                def marks(j, i=i):
                    err = cudart.cudaEventRecordWithFlags(evs[i][j], cs.cuda_stream,
                                                          cudart.cudaEventRecordExternal)[0]
                    assert err == cudart.cudaError_t.cudaSuccess, err
                run_step(cs, marks if i in evs else None, kv=kvs[i % n_copies])
        graph.replay()                      # one untimed replay
        torch.cuda.synchronize()
        use_graph = True
    except Exception as e:  # noqa: BLE001
        timing = f"eager launches (graph capture failed: {e!r})"
        use_graph = False

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    clocks.begin()
    start.record(stream)
    if use_graph:
        graph.replay()
    else:
        dec_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(args.steps)]
        for i in range(args.steps):
            run_step(stream, lambda j, i=i: dec_events[i][j].record(stream), kv=kvs[i % n_copies])
    end.record(stream)
    barrier()
    clocks.end()
    total_ms = start.elapsed_time(end)
    if use_graph:
        dec_ms = [cudart.cudaEventElapsedTime(a, b)[1] for a, b in evs.values()]
        for a, b in evs.values():
            cudart.cudaEventDestroy(a)
            cudart.cudaEventDestroy(b)
    else:
        dec_ms = [a.elapsed_time(b) for a, b in dec_events]
    total_ms = max_over_ranks(total_ms, world, dev)
    status = int(step.status.item())
    clock_info = clocks.stop()

    # End to end through the public API, as a serving loop runs it: every step copies its
    # queries in from pinned host memory, runs the public DecodeStep and reads its output
    # back, with the copies of E2E_SETS buffer sets overlapping the compute (pipelined_e2e).
    # A single 3 MB host-to-device copy is faster by SM loads of the mapped buffer
    # (mla_copy_from_host) than by the copy engine, but those loads take SMs from the
    # compute that runs beside them, and copy-engine copies on several streams overlap.
    def make_set(k):
        kv_k = kvs[k % n_copies]
        st = step if k == 0 else mla.DecodeStep(
            case.B, case.S, case.H, w_uk, w_uv, max_seqlen=max(case.seqlens), num_splits=case.num_splits,
            causal=case.causal, rope_theta=case.theta, total_rows=case.total_tokens, seqlens=case.seqlens)
        qn_k, qr_k = (q_nope, q_rope) if k == 0 else (q_nope.clone(), q_rope.clone())
        return ([qn_k, qr_k], st.o,
                lambda s_: st(qn_k, qr_k, kv_k, seqlens, block_table=block_table, q_pos=q_pos, stream=s_))
    # Step i reads cache copy i mod n_copies, as in the device-timed run: the number of sets
    # is a multiple of n_copies.
    n_sets = n_copies * math.ceil(E2E_SETS / n_copies)
    e2e_ms, h2d, d2h = pipelined_e2e([make_set(k) for k in range(n_sets)], [qn.pin_memory(), qr.pin_memory()],
                                     args.steps, args.warmup, stream, barrier)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    ms_per_step = total_ms / args.steps
    tokens_per_step = case.B * case.S
    value = whole_job_rate(world, tokens_per_step, ms_per_step)
    e2e_value = whole_job_rate(world, tokens_per_step, e2e_ms / args.steps)

    _, alg_b, flops = algorithmic(case)
    hbm, tf_burst, tf_sus, peak_kind = measured_peaks()
    dec_avg_s = statistics.mean(dec_ms) / 1e3
    achieved_gbs = alg_b / dec_avg_s / 1e9
    achieved_tf = flops / dec_avg_s / 1e12
    t_hbm = alg_b / (hbm * 1e9)
    t_tc = flops / (tf_burst * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    traffic = recorded_traffic(case.name, step.num_splits)
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                "frac": achieved_gbs / hbm}
    else:
        roof = {"bound": "tensor", "achieved": achieved_tf, "peak": tf_burst, "unit": "TFLOP/s",
                "frac": achieved_tf / tf_burst}
    roof.update({"traffic": traffic, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json burst)",
                 "kernel": "mla_decode_latent", "decode_us": dec_avg_s * 1e6,
                 "algorithmic_bytes": alg_b, "cache_bytes": cache_b, "flops": flops,
                 "tflops": achieved_tf, "tensor_frac": achieved_tf / tf_burst,
                 "roofline_us": max(t_hbm, t_tc) * 1e6,
                 "frac_of_min_roofline": max(t_hbm, t_tc) / dec_avg_s})

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": case.name, "B": case.B, "S": case.S, "H": case.H,
                       "T": case.seqlens[0] if len(set(case.seqlens)) == 1 else "ragged",
                       "total_cached_rows": case.total_tokens, "d_c": 512, "d_r": 64,
                       "num_splits": step.num_splits, "paged": case.paged,
                       "causal": case.causal, "rope": case.rope,
                       "l2": f"inputs larger than L2: {cache_b / 1e6:.0f} MB cache read per step"
                             if n_copies == 1 else
                             f"{n_copies} copies of the {cache_b / 1e6:.2f} MB cache read in turn "
                             f"({n_copies * cache_b / 1e6:.0f} MB > L2)",
                       "timing": timing,
                       "parallelism": f"dp{world} (independent replicas, no collective)"},
            "clocks": clock_info,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * step.kernels_per_step,
            "decode_steps_timed": len(dec_ms),
            "device_status": status,
            "roofline": roof}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
