"""Benchmark of the PagedAttention hot path on one GB300 (or N replicas).

One step = one pass of the whole path over the Llama-3-70B-shaped decode
batch (256 sequences, 64 query / 8 KV heads, head_dim 128, 32-token blocks,
bf16, log-normal context lengths, split-KV partitions of 512 tokens): one
pa_decode_write call, which stores the 256 new tokens' K/V in their slots and
runs paged decode over every sequence (plan + decode launches).  The metric
is decode KV bandwidth: algorithmic K+V bytes read per step / step time, plus
decode tokens/s per layer.  Under torchrun every rank runs its own replica
(weak scaling); the step time is the slowest rank's.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle instead
(bounded samples of the same workload on the host cores).

``other_decodes`` is pa_decode alone on the 8B-shaped, shared-prefix and
mixed fp8 decode workloads and on fp8 caches (K+V bytes / time);
``decode_cuda_cores`` the step through the CUDA-core decode kernel;
``mixed_step`` the chunked-prefill mixed batch as two calls and as one
pa_mixed_step launch; ``block_manager`` the host block manager's numbers;
``e2e`` the step with host buffers.  The line also carries
``prefill``: the tensor-core chunked-prefill kernel
timed on its own (CUDA events, inputs resident), as useful causal TFLOP/s
(4 * head_dim * Hq * sum over query rows of the keys each row attends to)
against the measured dense bf16 peak, for the 512-token chunk of the
chunked-prefill mixed batch (fp8 KV) and for a batch that fills every SM.
``--prefill-only`` prints just that measurement (used for profiling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV GB/s and tokens/s/layer on 1 GB300; % of HBM roofline"
UNIT = "GB/s"
WORKLOAD = "Llama-3-70B-shaped decode layer"
NOMINAL_HBM_GBPS = 7900.0     # GB300 HBM3e, vendor figure (context; the roofline uses the measured copy rate)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _tensor_peak():
    """Dense bf16 TFLOP/s for a kernel timed on its own (burst figure)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    return 1900.0, "fallback"


def _causal_flops(b) -> float:
    """Useful FLOPs of one pa_prefill_chunk call: Q.K^T and P.V over the keys each row sees."""
    p = b.prefill
    keys = 0
    for c in range(len(p.q_start)):
        n = int(p.cu_q_lens[c + 1] - p.cu_q_lens[c])
        keys += n * int(p.q_start[c]) + n * (n + 1) // 2
    return 4.0 * b.head_dim * b.num_q_heads * keys


# the chunk of the chunked-prefill mixed batch (fp8 KV, bf16 q: one 512-row chunk over 4096 tokens), then the
# prefill-only batches of workloads.PREFILL_WORKLOADS (2048 / 256-token chunks, MHA, every SM busy)
MIXED_CHUNK_DESC = ("chunked-prefill mixed batch, fp8 KV: 512-token chunk at position 4096, GQA 32/8, "
                    "head_dim 128, block 16")


def measure_block_manager() -> dict:
    """The host block manager (pa_bm_*) on the pages' block arithmetic: slots wasted on the
    Llama-3-8B-shaped lengths, blocks saved by sharing a 2048-token prefix among 4 branches, and
    the rate of single-token appends (the decode step's bookkeeping) on one host thread."""
    import time
    import paged_kv_cache_writes_gb300 as pa
    rng = np.random.default_rng(101)
    lens = rng.integers(512, 4097, size=64)
    bm = pa.BlockManager(20000, 16, shuffle_seed=1)
    seqs = [bm.new_sequence() for _ in lens]
    for s_, L in zip(seqs, lens):
        bm.append(s_, int(L))
    st = bm.stats()
    waste = 1.0 - st.logical_tokens / (st.used_blocks * 16)
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < 0.2:
        for s_ in seqs:
            bm.append(s_, 1)
        n += len(seqs)
    rate = n / (time.perf_counter() - t0)
    bm.close()
    tails = np.random.default_rng(11).integers(0, 257, size=(32, 4))
    bm = pa.BlockManager(8192, 16, shuffle_seed=1)
    for pr in range(32):
        root = bm.new_sequence()
        bm.append(root, 2048)
        for b_, s_ in enumerate([root] + [bm.fork(root) for _ in range(3)]):
            bm.append(s_, int(tails[pr, b_]))
    st2 = bm.stats()
    bm.close()
    return {"waste_frac_llama8b_lengths": waste, "blocks_used_llama8b": st.used_blocks,
            "shared_prefix_saving": 1.0 - st2.used_blocks / st2.logical_blocks,
            "appends_per_s_one_thread": rate,
            "note": "host C++ through the C ABI (ctypes call per append included)"}


def measure_other_decodes(dev_name: str, steps: int, warmup: int) -> dict:
    """pa_decode alone on the other decode workloads: algorithmic K+V bytes / CUDA-event time."""
    import torch
    import workloads as W
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    peak, kind = _peaks()
    res = {}
    cases = (("llama8b", W.cfg_llama8b), ("shared_prefix", W.cfg_shared_prefix),
             ("mixed_fp8_decodes", W.cfg_mixed_fp8),
             ("llama8b_fp8_cache", lambda: W.cfg_llama8b(kv_dtype="fp8")),
             ("llama70b_fp8_cache", lambda: W.cfg_llama70b(kv_dtype="fp8")),
             ("llama70b_fp8_cache_head_scales", lambda: W.cfg_llama70b(kv_dtype="fp8", fp8_scales="head")),
             ("head_dim64_32_8", W.cfg_d64), ("head_dim64_64_8", lambda: W.cfg_d64(num_q_heads=64)),
             ("head_dim64_64_8_fp8_cache", lambda: W.cfg_d64(num_q_heads=64, kv_dtype="fp8")),
             ("gqa3_24_8", lambda: W.cfg_gqa(24)), ("gqa5_40_8", lambda: W.cfg_gqa(40)))
    for key, fn in cases:
        b = fn()
        db = DeviceBatch(b, dev_name)
        db.run_setup()
        db.write_step()
        for _ in range(warmup):
            db.decode()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            db.decode()
        e1.record(s)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        ms = e0.elapsed_time(e1) / steps
        gbs = b.decode_kv_bytes() / (ms * 1e-3) / 1e9
        r = {"workload": b.name, "kv_dtype": b.kv_dtype, "num_seqs": b.num_seqs,
             "heads": f"{b.num_q_heads}/{b.num_kv_heads}", "kv_bytes": b.decode_kv_bytes(), "ms": ms,
             "GBps": gbs, "frac_of_hbm": gbs / peak, "peak_source": kind, "note": None}
        if key == "shared_prefix":
            # logical bytes count each shared prefix block once per branch that reads it; the unique
            # bytes count each physical block once (a floor for the DRAM traffic, re-reads may hit L2)
            uniq = unique_kv_bytes(b)
            r.pop("frac_of_hbm")
            r.update({"GBps_logical": r.pop("GBps"), "frac_of_hbm_logical": gbs / peak, "kv_bytes_unique": uniq,
                      "GBps_unique": uniq / (ms * 1e-3) / 1e9, "frac_of_hbm_unique": uniq / (ms * 1e-3) / 1e9 / peak,
                      "note": "kv_bytes counts the shared prefix once per branch (logical); kv_bytes_unique "
                              "counts each physical block once"})
        res[key] = r
        del db
        torch.cuda.empty_cache()
    return res


def unique_kv_bytes(b) -> int:
    """K+V bytes of the physical blocks a decode pass reads, each block once (the most tokens of it
    that any sequence reads), for batches whose sequences share blocks."""
    used = {}
    for i, L in enumerate(b.seq_lens.astype(np.int64)):
        for j in range(int(-(-L // b.block_size))):
            blk = int(b.block_tables[i, j])
            used[blk] = max(used.get(blk, 0), int(min(b.block_size, L - j * b.block_size)))
    return sum(used.values()) * 2 * b.num_kv_heads * b.head_dim * b.kv_elem_bytes


def measure_mixed_step(dev_name: str, steps: int, warmup: int) -> dict:
    """The chunked-prefill mixed batch (one 512-row chunk + 128 decodes, fp8 KV): its attention as two
    calls (pa_prefill_chunk, then pa_decode) against one pa_mixed_step (prefill tiles and decode CTAs in
    one grid), and each part alone, each timed with CUDA events over the same number of back-to-back
    steps.  vs_longer_part: the one launch's time over the longer part's alone (1.0 would be a perfect
    overlap of the shorter part)."""
    import torch
    import workloads as W
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    b = W.cfg_mixed_fp8()
    db = DeviceBatch(b, dev_name)
    db.run_setup()
    db.write_step()

    def two():
        db.prefill_chunk()
        db.decode()

    res = {"workload": "chunked-prefill mixed batch, fp8 KV: 512-token chunk at 4096 + 128 decodes "
                       "(256..8192 tokens), GQA 32/8, head_dim 128, block 16",
           "kv_bytes_decode": b.decode_kv_bytes(), "useful_tflop_prefill": _causal_flops(b) / 1e12}
    s = torch.cuda.current_stream()
    for key, fn in (("two_calls", two), ("one_launch", db.mixed_attention), ("prefill_alone", db.prefill_chunk),
                    ("decode_alone", db.decode)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        res[key + "_ms"] = e0.elapsed_time(e1) / steps
    res["speedup"] = res["two_calls_ms"] / res["one_launch_ms"]
    res["vs_longer_part"] = res["one_launch_ms"] / max(res["prefill_alone_ms"], res["decode_alone_ms"])
    del db
    torch.cuda.empty_cache()
    return res


def measure_prefill(dev_name: str, steps: int, warmup: int) -> dict:
    import torch
    import workloads as W
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    peak, kind = _tensor_peak()
    res = {}
    cases = [("mixed_fp8_chunk", MIXED_CHUNK_DESC, W.cfg_mixed_fp8)]
    cases += [(k, d, f) for k, (d, f) in W.PREFILL_WORKLOADS.items()]
    for key, desc, make in cases:
        b = make()
        db = DeviceBatch(b, dev_name)
        db.run_setup()
        db.write_step()
        for _ in range(warmup):
            db.prefill_chunk()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            db.prefill_chunk()
        e1.record(s)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        ms = e0.elapsed_time(e1) / steps
        tf = _causal_flops(b) / (ms * 1e-3) / 1e12
        res[key] = {"workload": desc, "kv_dtype": b.kv_dtype, "ms": ms, "useful_tflop": _causal_flops(b) / 1e12,
                    "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                                 "frac": tf / peak, "peak_source": kind,
                                 "kernel": "prefill_tc_kernel (pa_prefill_chunk)"}}
        del db
        torch.cuda.empty_cache()
    return res


# the sources of the decode kernel the bench times (their hash dates the committed capture)
DECODE_SOURCES = ("pa_decode_tc.cuh", "pa_tcgen05.cuh", "pa_decode.cuh", "pa_attention.cuh", "pa_common.cuh")


def _sources_hash(names) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in names:
        with open(os.path.join(ROOT, "paged_kv_cache_writes_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profile_figures(profile: str, sources) -> dict | None:
    """The ``name: number`` lines of a committed ncu summary under profiles/, or None when the
    summary is missing or the kernel's sources changed since it was captured (source_sha256_16)."""
    import re
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"^source_sha256_16:\s*([0-9a-f]{16})\s*$", text, re.M)
    if not m or m.group(1) != _sources_hash(sources):
        return None
    return {k: float(v) for k, v in re.findall(r"^([a-z][a-z0-9_]*):\s*([0-9.eE+-]+)\s*$", text, re.M)}


def _profiled_traffic(kv_bytes: int):
    """DRAM bytes per decode launch, scaled from the committed ncu capture of the
    decode kernel -- or None if the decode sources changed since that capture."""
    f = _profile_figures("decode_tc_kernel__llama70b_decode.md", DECODE_SOURCES)
    if not f or "traffic_per_kv_byte" not in f:
        return None
    return f["traffic_per_kv_byte"] * kv_bytes


def _config(b, extra=None):
    name = WORKLOAD if b.num_seqs == 256 else f"{WORKLOAD} (reduced to {b.num_seqs} sequences)"
    cfg = {"workload": name, "num_seqs": b.num_seqs, "num_q_heads": b.num_q_heads,
           "num_kv_heads": b.num_kv_heads, "head_dim": b.head_dim, "block_size": b.block_size,
           "kv_dtype": b.kv_dtype, "partition_size": b.partition_size or 512,
           "context_tokens": int(b.seq_lens.astype(np.int64).sum()), "max_seq_len": b.max_seq_len,
           "lengths": "log-normal, median 1000, sigma 1.0, cap 8192 (seeded)",
           "l2": "inputs larger than L2 (KV read per step >> 129 MB L2)"}
    if extra:
        cfg.update(extra)
    return cfg


_NVML_REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, clock-event reasons)."""

    def __init__(self, cuda_index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        bus = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(cuda_index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except Exception:
            bus = None
        ok = bus is not None and self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        try:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self) -> int:
        v = self.c.c_uint()
        return v.value if self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.c.byref(v)) == 0 else -1

    def sm_max_mhz(self) -> int:
        v = self.c.c_uint()
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.c.byref(v)) == 0 else -1

    def reasons(self) -> int:
        v = self.c.c_ulonglong()
        return v.value if self.reasons_fn(self.h, self.c.byref(v)) == 0 else 0


class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region: NVML read in a
    thread of this process every ~0.5 ms (the timed region can be a few ms long),
    and nvidia-smi every 200 ms when NVML cannot be loaded."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.nvml = None
        self.lines = []
        self.samples = []       # (sm MHz, reason bits)
        self.stop = threading.Event()

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.index)
            self.max_mhz = self.nvml.sm_max_mhz()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _poll(self):
        while not self.stop.is_set():
            self.samples.append((self.nvml.sm_mhz(), self.nvml.reasons()))
            time.sleep(0.0005)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        self.stop.set()
        if self.nvml is not None:
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.nvml is not None:
            sm = [m for m, _ in self.samples if m > 0]
            reasons = sorted({n for _, r in self.samples for bit, n in _NVML_REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(sm), "source": "NVML, every ~0.5 ms"}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, every 200 ms"}


def measure_stream_copy(dev_name: str) -> dict:
    """Device-to-device copy of 2 GiB (torch copy_, bytes read + written), best of 10 with CUDA events:
    the HBM figure of this run, beside the measured peak and the nominal one."""
    import torch
    n = 1 << 30
    a = torch.empty(n, dtype=torch.bfloat16, device=dev_name).fill_(1.0)
    bb = torch.empty_like(a)
    for _ in range(3):
        bb.copy_(a)
    torch.cuda.synchronize()
    best = None
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        bb.copy_(a)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        best = t if best is None else min(best, t)
    del a, bb
    torch.cuda.empty_cache()
    peak, kind = _peaks()
    return {"GBps": 2 * 2 * n / (best * 1e-3) / 1e9, "how": "torch copy_ of 1 Gi bf16 elements (read + write bytes), "
            "best of 10, CUDA events", "measured_peak_GBps": peak, "measured_peak_source": kind,
            "nominal_hbm3e_GBps": NOMINAL_HBM_GBPS}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(x: float, device) -> float:
    """The largest x over the ranks of the process group (x itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(units_per_rank: float, ms: float, world_size: int) -> float:
    """Whole-job rate of a weak-scaling run: every rank processes units_per_rank
    units (its own replica of the workload) and ms is the slowest rank's time."""
    return units_per_rank * world_size / (ms * 1e-3)


def _time_oracle(b, kp, vp, ids) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.decode_batch(b, kp, vp, seq_ids=ids)
    return time.perf_counter() - t0


def _sample_ids(b, budget_bytes, rng):
    """Random sequences whose KV bytes add up to about ``budget_bytes``."""
    per = b.seq_lens.astype(np.int64) * 2 * b.num_kv_heads * b.head_dim * b.kv_elem_bytes
    ids, tot = [], 0
    for i in rng.permutation(b.num_seqs):
        ids.append(int(i))
        tot += int(per[i])
        if tot >= budget_bytes:
            break
    return np.array(sorted(ids), dtype=np.int32), tot


def cpu_oracle_rate(b, seconds: float = 15.0):
    """The oracle as it stands, on the host cores, over a bounded sample."""
    import oracle
    import workloads as W
    kp, vp = W.empty_pools(b)
    oracle.populate(b, kp, vp)
    rng = np.random.default_rng(0)
    ids, nbytes = _sample_ids(b, 8 << 20, rng)          # calibrate on ~8 MB of KV
    t = _time_oracle(b, kp, vp, ids)
    target = max(1 << 20, int(nbytes * seconds / max(t, 1e-3)))
    ids, nbytes = _sample_ids(b, target, rng)
    t = _time_oracle(b, kp, vp, ids)
    res = {"value": nbytes / t / 1e9, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
           "sample": f"{len(ids)} of {b.num_seqs} sequences ({nbytes / 1e6:.0f} MB of KV), fp64 C, OpenMP, "
                     f"{t:.1f} s"}
    # the same oracle on one thread, over a smaller sample (reference point only)
    cores = oracle.max_threads()
    oracle.set_threads(1)
    try:
        ids1, nb1 = _sample_ids(b, max(1 << 20, target // max(1, cores) // 3), rng)
        t1 = _time_oracle(b, kp, vp, ids1)
    finally:
        oracle.set_threads(cores)
    res["one_thread"] = {"value": nb1 / t1 / 1e9, "unit": UNIT,
                         "sample": f"{len(ids1)} sequences ({nb1 / 1e6:.0f} MB of KV), {t1:.1f} s"}
    return res


def run_reference(args):
    """--impl reference: the oracle timed per step on bounded samples."""
    import oracle
    import workloads as W
    ws, rank, _ = _dist()
    if rank != 0:
        return
    b = W.cfg_llama70b()
    kp, vp = W.empty_pools(b)
    oracle.populate(b, kp, vp)
    rng = np.random.default_rng(1)
    budget = 6 << 20
    for _ in range(args.warmup):
        ids, _ = _sample_ids(b, budget, rng)
        _time_oracle(b, kp, vp, ids)
    tot_b, tot_t, tot_seq = 0, 0.0, 0
    for _ in range(args.steps):
        ids, nb = _sample_ids(b, budget, rng)
        tot_t += _time_oracle(b, kp, vp, ids)
        tot_b += nb
        tot_seq += len(ids)
    value = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) K/V/q, seeded block tables)",
            "config": _config(b, {"sample_per_step": f"~{budget >> 20} MB of KV (random sequences)"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"{tot_seq} sequences over {args.steps} steps, ~{budget >> 20} MB KV each"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_ours(args):
    import torch
    import workloads as W
    from paged_kv_cache_writes_gb300 import build_lib
    build_lib.build()
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev_name = f"cuda:{local}"

    b = W.cfg_llama70b(batch=args.batch)
    db = DeviceBatch(b, dev_name)
    db.run_setup()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    kv_bytes = b.decode_kv_bytes()
    # algorithmic bytes of one fused step (pa_decode_write): K+V once per KV head, q in, out, tables,
    # lengths, and the new tokens' K/V read and stored
    eb_q = 2
    new_bytes = 2 * b.num_seqs * b.num_kv_heads * b.head_dim * eb_q * 2 + b.num_seqs * 8
    dec_bytes = (kv_bytes + 2 * b.num_seqs * b.num_q_heads * b.head_dim * eb_q +
                 int(np.ceil(b.seq_lens / b.block_size).sum()) * 4 + b.num_seqs * 4 + new_bytes)

    # one step = one pa_decode_write call: the 256 new tokens stored, then decode (plan + decode launches)
    for _ in range(args.warmup):
        db.decode_write()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            db.decode_write()
            ev[i][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    ms = start.elapsed_time(end) / args.steps
    dec_all = sorted(a.elapsed_time(z) for a, z in ev)
    dec_ms = statistics.mean(dec_all)

    def pct(q):
        return dec_all[min(len(dec_all) - 1, int(q * (len(dec_all) - 1) + 0.5))]
    assert pa.pa_get_device_error() == 0
    ms = _max_over_ranks(ms, dev_name)

    # end to end through the public API with host buffers (pinned), copies inside the timed region:
    # every step copies its inputs (q, the new tokens' K/V and slots, tables, lengths) from pinned host
    # memory and reads its output back.  Two device buffer sets and separate copy streams let step i+1's
    # inputs and step i-1's output move while step i computes (the copy engines run beside the kernels).
    k_new, v_new, slots_new = db.fused_step_tensors()
    srcs = {"q": db.q, "bt": db.block_tables, "sl": db.seq_lens, "k": k_new, "v": v_new, "s": slots_new}
    host = {k: v.cpu().pin_memory() for k, v in srcs.items()}
    out_h = [torch.empty(db.out.shape, dtype=db.out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h[0].numel() * out_h[0].element_size()
    bufs = [{k: torch.empty_like(v) for k, v in srcs.items()} for _ in range(2)]
    for bset in bufs:
        bset["out"] = torch.empty_like(db.out)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    for i in range(2):   # the buffers start free
        ev_done[i].record(stream)
        ev_read[i].record(stream)

    def e2e_step(i):
        bset = bufs[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_done[i % 2])            # the step that last used this set has computed
            for k in ("q", "bt", "sl", "k", "v", "s"):
                bset[k].copy_(host[k], non_blocking=True)
            ev_in[i % 2].record(s_in)
        stream.wait_event(ev_in[i % 2])
        stream.wait_event(ev_read[i % 2])              # its output has been read back
        pa.pa_decode_write(bset["q"], bset["k"], bset["v"], bset["s"], db.k_cache, db.v_cache, db.desc,
                           bset["bt"], bset["sl"], int(b.seq_lens.max()), b.scale, bset["out"], db.workspace,
                           b.partition_size, stream=stream)
        ev_done[i % 2].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[i % 2])
            out_h[i % 2].copy_(bset["out"], non_blocking=True)
            ev_read[i % 2].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_stream(s_out)                          # the last output is back on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    assert torch.equal(out_h[(args.steps - 1) % 2].view(torch.int32), bufs[(args.steps - 1) % 2]["out"].cpu().view(torch.int32))
    e2e_ms = _max_over_ranks(e2e_ms, dev_name)

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    peak, peak_kind = _peaks()
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    value = _job_rate(kv_bytes, ms, ws) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) K/V/q rounded to bf16, seeded shuffled block tables)",
        "config": _config(b, {"parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}),
        "tokens_per_s_per_layer": _job_rate(b.num_seqs, ms, ws),
        "decode_ms": dec_ms,
        "decode_ms_p10_p50_p90": [pct(0.1), pct(0.5), pct(0.9)],
        "step": "one pa_decode_write call: the new tokens' cache write fused into the decode launch",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": _profiled_traffic(kv_bytes),
                     "kernel": "decode_tc_kernel (pa_decode_write: plan + decode launches, timed together)",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": _job_rate(kv_bytes, e2e_ms, ws) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": "pa_decode_write per step; inputs copied from pinned host memory and the output read "
                        "back every step, on copy streams overlapping the neighbouring steps' compute"},
        "gpu_launches": 2 * args.steps,  # per step: decode plan, decode (the cache write is inside)
        "clocks": clocks.summary(),
    }
    prof = _profile_figures("decode_tc_kernel__llama70b_decode.md", DECODE_SOURCES)
    if prof:
        # pipe figures of the committed ncu capture of this kernel (same sources)
        line["roofline"]["ncu"] = {k: v for k, v in prof.items() if k != "traffic_per_kv_byte"}
    if ws == 1:
        # the same step through the CUDA-core decode kernel (selectable; the default uses the tensor cores)
        with pa.decode_kernel("cuda_cores"):
            for _ in range(args.warmup):
                db.decode_write()
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n_cc = max(5, args.steps // 5)
            c0.record(stream)
            for _ in range(n_cc):
                db.decode_write()
            c1.record(stream)
            torch.cuda.synchronize()
        cc_ms = c0.elapsed_time(c1) / n_cc
        assert pa.pa_get_device_error() == 0
        line["decode_cuda_cores"] = {
            "kernel": "paged_decode_kernel (pa_set_decode_kernel(PA_DECODE_KERNEL_CUDA_CORES))",
            "ms": cc_ms, "achieved": dec_bytes / (cc_ms * 1e-3) / 1e9, "unit": "GB/s",
            "frac": dec_bytes / (cc_ms * 1e-3) / 1e9 / peak}
        del db
        torch.cuda.empty_cache()
        line["prefill"] = measure_prefill(dev_name, max(5, args.steps // 5), args.warmup)
        line["other_decodes"] = measure_other_decodes(dev_name, max(5, args.steps // 5), args.warmup)
        line["mixed_step"] = measure_mixed_step(dev_name, max(5, args.steps // 5), args.warmup)
        line["block_manager"] = measure_block_manager()
        line["stream_copy"] = measure_stream_copy(dev_name)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_rate(b, args.cpu_seconds)
    print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_case(args):
    """--case NAME: W warm-up and K timed calls of one kernel on one workload, for ncu captures.
    decode_bf16 / decode_fp8 / decode_fp8_head: pa_decode on the Llama-3-70B-shaped batch (--batch
    sequences); decode_write: pa_decode_write on it; prefill:<key>: pa_prefill_chunk on the mixed
    batch's chunk (mixed_fp8_chunk) or a batch of workloads.PREFILL_WORKLOADS; mixed: pa_mixed_step
    on the chunked-prefill mixed batch; mixed_two: its pa_prefill_chunk + pa_decode."""
    import torch
    import workloads as W
    from paged_kv_cache_writes_gb300 import build_lib
    build_lib.build()
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    torch.cuda.set_device(0)
    c = args.case
    if c.startswith("decode"):
        kv = "fp8" if "fp8" in c else "bf16"
        b = W.cfg_llama70b(batch=args.batch, kv_dtype=kv, fp8_scales="head" if c.endswith("_head") else "tensor")
    elif c.startswith("prefill:"):
        key = c.split(":", 1)[1]
        b = W.cfg_mixed_fp8() if key == "mixed_fp8_chunk" else W.PREFILL_WORKLOADS[key][1]()
    elif c in ("mixed", "mixed_two"):
        b = W.cfg_mixed_fp8()
    else:
        raise SystemExit(f"unknown case {c}")
    db = DeviceBatch(b, "cuda:0")
    db.run_setup()
    if c != "decode_write":
        db.write_step()

    def two():
        db.prefill_chunk()
        db.decode()
    fn = {"decode_write": db.decode_write, "mixed": db.mixed_attention, "mixed_two": two}.get(
        c, db.prefill_chunk if c.startswith("prefill:") else db.decode)
    with pa.decode_kernel(args.decode_kernel):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ms = e0.elapsed_time(e1) / args.steps
    out = {"case": c, "workload": b.name, "ms": ms, "steps": args.steps, "warmup": args.warmup,
           "decode_kernel": args.decode_kernel}
    if c.startswith("decode"):
        out["kv_bytes"] = b.decode_kv_bytes()
        out["GBps"] = b.decode_kv_bytes() / (ms * 1e-3) / 1e9
    elif c.startswith("prefill:"):
        out["useful_tflop"] = _causal_flops(b) / 1e12
        out["TFLOPs"] = _causal_flops(b) / (ms * 1e-3) / 1e12
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--batch", type=int, default=256,
                    help="sequences in the decode batch (256 = the named workload; smaller only for profiling)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the tensor-core prefill kernel (profiling)")
    ap.add_argument("--case", default=None,
                    help="time one kernel alone (profiling): decode_bf16, decode_fp8, decode_fp8_head, "
                         "decode_write, prefill:<key>, mixed, mixed_two")
    ap.add_argument("--decode-kernel", choices=["auto", "cuda_cores"], default="auto",
                    help="with --case: the decode kernel pa_set_decode_kernel selects")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case:
        run_case(args)
        return
    if args.prefill_only:
        import torch
        from paged_kv_cache_writes_gb300 import build_lib
        build_lib.build()
        torch.cuda.set_device(0)
        print(json.dumps({"metric": "prefill useful TFLOP/s", "prefill": measure_prefill("cuda:0", args.steps,
                                                                                       args.warmup)}))
        return
    (run_reference if args.impl == "reference" else run_ours)(args)


if __name__ == "__main__":
    main()
