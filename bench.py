"""Benchmark of the paged-KV decode step on GB300.

A step is one pass of the decode hot path over one batch: kv_append of each
sequence's newest K/V row, then paged_attention_decode (split-K partial kernel
plus log-sum-exp reduction).  Default workload: the long-context decode
(bf16, batch 8, lengths uniform in [32768, 65536], 32/8 heads, head_dim 128,
block size 16, random physical placement, split-K over blocks), the largest
steady decode configuration.

Prints one JSON line (rank 0).  `value` is decode KV GB/s: algorithmic K/V
bytes of the visible rows (4096 B per token row for this layer) per step over
the device-timed step time.  `e2e` is the same metric through the C ABI with
the per-step inputs copied from pinned host memory and the output read back
inside the timed region.  On one GPU the default run also measures, as extra
keys of the same line, a read-only HBM streaming peak and the other
configured workloads (the Llama-shaped layer, long context at block size 64,
the 200-step churn trace, the shared-prefix batch, the prefix tree, eight
query heads per kv head, and both over MXFP8 pools), each with its own
roofline.

--impl reference times the CPU oracle on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import signal
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = ("llama", "llama_mxfp8", "long_bs16", "long_bs64", "long_bs64_k16", "shared", "churn",
             "gqa8", "gqa8_mxfp8", "tree", "append", "block_copy")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="long_bs16", choices=WORKLOADS)
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch size (small cases for profiling)")
    ap.add_argument("--prefix-len", type=int, default=0,
                    help="shared workload: prefix tokens (default 2048)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the read peak and the other workloads of the default run")
    ap.add_argument("--cpu-sample-seconds", type=float, default=12.0)
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


def kernel_traffic(kernel_file, summary):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    src = os.path.join(ROOT, "paged_kv_cache_41_gb300", "csrc", "kernels", kernel_file)
    summ = os.path.join(ROOT, "profiles", summary)
    if not (os.path.exists(src) and os.path.exists(summ)):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    text = open(summ).read()
    m_h = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_h or not m_t or m_h.group(1) != h:
        return None
    return float(m_t.group(1))


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for ln in open(self.path):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def all_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def make_batch(name, device, seed_offset=0, batch=0):
    from paged_kv_cache_41_gb300 import workloads as wl
    if name in ("llama", "llama_mxfp8"):
        return wl.llama_batch(device=device, seed=2 + seed_offset, batch=batch or 64)
    if name == "long_bs16":
        return wl.long_batch(device=device, block_size=16, seed=3 + seed_offset, batch=batch or 8)
    if name in ("long_bs64", "long_bs64_k16"):
        return wl.long_batch(device=device, block_size=64, seed=3 + seed_offset, batch=batch or 8)
    if name in ("gqa8", "gqa8_mxfp8"):
        # the Llama-shaped lengths with eight query heads per kv head (64 / 8)
        rng = np.random.default_rng(2 + seed_offset)
        lens = rng.integers(512, 8192, size=batch or 64, endpoint=True)
        b = wl.custom_batch(lens, dtype="bf16", hq=64, hkv=8, d=128, p=16, seed=2 + seed_offset,
                            device=device)
        b.name = "gqa8"
        return b
    if name == "churn":
        # the lengths of the churn trace's first decode step, as a plain batch
        step = next(wl.ChurnTrace(seed=4 + seed_offset, steps=1).run())
        return wl.custom_batch(step.seq_lens, dtype="bf16", hq=32, hkv=8, d=128, p=16,
                               seed=4 + seed_offset, device=device)
    raise ValueError(name)


DECODE_WORKLOAD_NAMES = {
    "llama": "llama3-8b-shaped decode layer",
    "llama_mxfp8": "llama3-8b-shaped decode layer over MXFP8 K/V pools",
    "long_bs16": "long-context decode, block size 16",
    "long_bs64": "long-context decode, block size 64",
    "long_bs64_k16": "long-context decode, block size 64 read as 16-row kernel blocks "
                     "(tables expanded per step)",
    "gqa8": "decode layer with 8 query heads per kv head (64/8)",
    "gqa8_mxfp8": "decode layer with 8 query heads per kv head (64/8) over MXFP8 K/V pools",
    "churn": "churn trace decode",
}


def decode_config(workload, b, partition_size, world):
    """The config of a decode workload, the same for both arms."""
    kblock = 16 if workload == "long_bs64_k16" else b.block_size
    mx = workload.endswith("_mxfp8")
    row_bytes = 2 * b.num_kv_heads * b.head_dim * 33 // 32 if mx else kv_row_bytes(b)
    return {
        "workload": DECODE_WORKLOAD_NAMES[workload],
        "batch": b.num_seqs, "num_q_heads": b.num_q_heads, "num_kv_heads": b.num_kv_heads,
        "head_dim": b.head_dim, "block_size": b.block_size, "kernel_block_size": kblock,
        "seq_len_min": int(b.seq_lens.min()), "seq_len_max": int(b.seq_lens.max()),
        "total_tokens": int(b.seq_lens.sum()), "pool_blocks": b.num_blocks,
        "partition_size": partition_size,
        "kv_bytes_per_step": int(b.seq_lens.astype(np.int64).sum()) * row_bytes,
        "l2": "inputs larger than L2 (K/V read per step >> 129 MB)",
        "parallelism": f"replicas x{world} (sequences shard, no collective)",
    }


def kv_row_bytes(b):
    return 2 * b.num_kv_heads * b.head_dim * (2 if b.dtype == "bf16" else 4)


# ------------------------------------------------------------------ CPU oracle timing
_SAMPLE_POOLS = {}  # (batch, sequence, tokens, mx) -> the oracle's private pool, reused


def oracle_sample(b, seconds, nthreads, mx=False, max_tokens=None):
    """Time the CPU oracle decoding whole sequences of the batch (or their
    first max_tokens tokens) until about `seconds` of CPU work; returns
    (kv_bytes, rows, elapsed, sample description).  mx: the sequences are
    quantized into MXFP8 pools and the oracle decodes their exact values (the
    time includes reading them out of the pool).  With max_tokens the private
    pools are kept for later calls (steps of the reference arm)."""
    import oracle
    from paged_kv_cache_41_gb300 import workloads as wl
    order = np.random.default_rng(0).permutation(b.num_seqs)
    kh_all, vh_all = b.k_hist, b.v_hist
    q_all = wl.to_numpy_storage(b.q)
    shape_blk = (b.block_size, b.num_kv_heads, b.head_dim)
    done_bytes = done_rows = 0
    elapsed = 0.0

    def private_pool(r, t):
        """A pool holding only sequence r's first t rows, paged through its
        own table 0, 1, ...: (table, K pool, V pool, q)."""
        key = (id(b), int(r), t, mx)
        if key in _SAMPLE_POOLS:
            return _SAMPLE_POOLS[key]
        lo = int(b.hist_offsets[r])
        nblk = max(1, oracle.num_blocks(t, b.block_size))
        table = np.arange(nblk, dtype=np.int32)
        kh = wl.to_numpy_storage(kh_all[lo:lo + t])
        vh = wl.to_numpy_storage(vh_all[lo:lo + t])
        i = np.arange(t, dtype=np.int64)
        slots = table[i // b.block_size].astype(np.int64) * b.block_size + i % b.block_size
        if mx:
            shape = (nblk,) + shape_blk
            kc = np.zeros(oracle.mxfp8_pool_bytes(*shape), np.uint8)
            vc = kc.copy()
            oracle.kv_append_mxfp8(kc, vc, shape, kh, vh, slots)
            q = np.ascontiguousarray(wl.to_numpy_storage(b.q[r:r + 1].float()))
        else:
            kc = np.zeros((nblk,) + shape_blk, dtype=kh.dtype)
            vc = np.zeros_like(kc)
            oracle.kv_append(kc, vc, kh, vh, slots)
            q = np.ascontiguousarray(q_all[r:r + 1])
        entry = (table, kc, vc, q)
        if max_tokens is not None:
            _SAMPLE_POOLS[key] = entry
        return entry

    for r in order:
        t = int(b.seq_lens[r]) if max_tokens is None else min(int(b.seq_lens[r]), max_tokens)
        table, kc, vc, q = private_pool(r, t)
        t0 = time.perf_counter()
        if mx:
            shape = (len(table),) + shape_blk
            kc, vc = oracle.mxfp8_to_f32(kc, shape), oracle.mxfp8_to_f32(vc, shape)
        oracle.paged_decode(q, kc, vc, table.reshape(1, -1), np.array([t], np.int32), b.scale,
                            nthreads=nthreads)
        elapsed += time.perf_counter() - t0
        done_bytes += t * (2 * b.num_kv_heads * b.head_dim * 33 // 32 if mx else kv_row_bytes(b))
        done_rows += 1
        if elapsed >= seconds:
            break
    desc = (f"{done_rows} of {b.num_seqs} sequences"
            f"{'' if max_tokens is None else f' (their first {max_tokens} tokens)'} "
            f"({done_bytes / 1e6:.1f} MB of {'MXFP8 ' if mx else ''}K/V), "
            f"all {b.num_q_heads} heads, fp64 oracle")
    return done_bytes, done_rows, elapsed, desc


def cpu_model():
    """The host CPU's model name, as /proc/cpuinfo gives it (or its part
    number on Arm), for the baseline's record."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return None
    for key in ("model name", "CPU part"):
        m = re.search(rf"^{key}\s*:\s*(.+)$", info, re.M)
        if m:
            return m.group(1).strip() if key == "model name" else f"Arm CPU part {m.group(1).strip()}"
    return None


def cpu_baseline(b, seconds, mx=False):
    """The oracle on all host cores of the affinity mask, then on one core
    (a shorter sample)."""
    nthreads = len(os.sched_getaffinity(0))
    nbytes, rows, el, desc = oracle_sample(b, seconds, nthreads, mx)
    nb1, rows1, el1, desc1 = oracle_sample(b, max(2.0, seconds / 4), 1, mx)
    return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": desc, "rows_per_s": rows / el,
            "single_thread": {"value": nb1 / el1 / 1e9, "unit": "GB/s", "sample": desc1},
            "cpu_model": cpu_model()}


# ------------------------------------------------------------------ GPU arm
def run_pkv(args, rank, world, local):
    import torch
    from paged_kv_cache_41_gb300 import pkv

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    pkv.load_library()
    b = make_batch(args.workload, dev, seed_offset=rank, batch=args.batch)
    B = b.num_seqs
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    dt = b.k_hist.dtype
    mx = args.workload.endswith("_mxfp8")  # the same layer over MXFP8 pools
    if mx:
        kc = pkv.MxPool(*shape, device=dev)
        vc = pkv.MxPool(*shape, device=dev)
    else:
        kc = torch.zeros(shape, dtype=dt, device=dev)
        vc = torch.zeros(shape, dtype=dt, device=dev)
    slots = torch.from_numpy(b.slots).to(dev)
    pre = torch.from_numpy(b.prefill_rows()).to(dev)
    pkv.kv_append(kc, vc, b.k_hist[pre], b.v_hist[pre], slots[pre])
    last_np = b.last_rows()
    last = torch.from_numpy(last_np).to(dev)
    new_k = b.k_hist[last].contiguous()
    new_v = b.v_hist[last].contiguous()
    step_slots = slots[last].contiguous()
    bt = torch.from_numpy(b.block_tables).to(dev)
    sl = torch.from_numpy(b.seq_lens).to(dev)
    q = b.q.contiguous()
    out = torch.empty_like(q)
    # long_bs64_k16: the bs64 allocator pool read as bs16 kernel blocks
    # ([M5.3] 0x0AC); each step expands the tables on the device first.
    kblock = 16 if args.workload == "long_bs64_k16" else b.block_size
    ratio = b.block_size // kblock
    kview = (b.num_blocks * ratio, kblock, b.num_kv_heads, b.head_dim)
    kck, vck = (kc, vc) if mx else (kc.view(kview), vc.view(kview))
    btk = torch.empty(B, b.max_blocks * ratio, dtype=torch.int32, device=dev)

    def decode_call(qq, tables, lens, o=None):
        if ratio > 1:
            pkv.expand_block_tables(tables, b.block_size, kblock, out=btk)
            tables = btk
        pkv.paged_attention_decode(qq, kck, vck, tables, lens, b.scale,
                                   out=out if o is None else o, partition_size=psize, workspace=ws)

    psize = args.partition_size
    ctas = pkv.decode_num_ctas(kck, B, b.num_q_heads, b.max_blocks * ratio, psize)
    ws_bytes = pkv.decode_workspace_bytes(kck, B, b.num_q_heads, b.max_blocks * ratio, psize)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    stream = torch.cuda.current_stream()

    def step():
        pkv.kv_append(kc, vc, new_k, new_v, step_slots)
        decode_call(q, bt, sl)

    # algorithmic bytes: K and V of the visible rows; an MXFP8 row is one byte
    # per element plus one scale byte per 32
    row_bytes = 2 * b.num_kv_heads * b.head_dim * 33 // 32 if mx else kv_row_bytes(b)
    kv_bytes = int(b.seq_lens.astype(np.int64).sum()) * row_bytes
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)

    clocks = ClockSampler(local)
    clocks.start()
    # the step time: events at the ends only, so that nothing stands between
    # a step's append and its decode (the decode's launch overlaps the
    # append's tail)
    torch.cuda.synchronize()
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        pkv.kv_append(kc, vc, new_k, new_v, step_slots)
        decode_call(q, bt, sl)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = all_max(t0.elapsed_time(t1), world)
    # each kernel's own time (the roofline's decode duration), in a second pass
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        ea, eb, ec = ev[i]
        ea.record(stream)
        pkv.kv_append(kc, vc, new_k, new_v, step_slots)
        eb.record(stream)
        decode_call(q, bt, sl)
        ec.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    decode_ms = all_max(float(np.mean([ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)])),
                        world)
    append_ms = float(np.mean([ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]))
    assert pkv.get_device_error() == 0
    ms_step = total_ms / args.steps

    # ---- end to end through the C ABI with host buffers.  Every step copies
    # its inputs (q, the new K/V rows and their slots, tables, lengths) from
    # pinned host memory and reads its output back, inside the timed region.
    # As a serving loop would, the copies are double-buffered on their own
    # streams: step i's inputs go to buffer set i % 2 while step i - 1
    # computes, once step i - 2's decode has finished with that set.
    h_q = q.cpu().pin_memory()
    h_k = new_k.cpu().pin_memory()
    h_v = new_v.cpu().pin_memory()
    h_slots = step_slots.cpu().pin_memory()
    h_bt = bt.cpu().pin_memory()
    h_sl = sl.cpu().pin_memory()
    h_outs = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    sets = [(torch.empty_like(q), torch.empty_like(new_k), torch.empty_like(new_v),
             torch.empty_like(step_slots), torch.empty_like(bt), torch.empty_like(sl))
            for _ in range(2)]
    d_outs = [torch.empty_like(out) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_slots, h_bt, h_sl))
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    landed = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        j = i % 2
        d_q, d_k, d_v, d_slots, d_bt, d_sl = sets[j]
        with torch.cuda.stream(up):
            if used[j]:
                up.wait_event(done[j])  # step i - 2's decode has read this set
            for d, h in ((d_q, h_q), (d_k, h_k), (d_v, h_v), (d_slots, h_slots), (d_bt, h_bt),
                         (d_sl, h_sl)):
                d.copy_(h, non_blocking=True)
            landed[j].record(up)
        stream.wait_event(landed[j])
        if used[j]:
            stream.wait_event(read[j])  # step i - 2's output has been read back
        pkv.kv_append(kc, vc, d_k, d_v, d_slots)
        decode_call(d_q, d_bt, d_sl, d_outs[j])
        done[j].record(stream)
        used[j] = True
        with torch.cuda.stream(down):
            down.wait_event(done[j])
            h_outs[j].copy_(d_outs[j], non_blocking=True)
            read[j].record(down)

    for i in range(max(3, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    up.wait_event(s0)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_stream(down)
    stream.wait_stream(up)
    s1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = all_max(s0.elapsed_time(s1), world) / args.steps
    assert pkv.get_device_error() == 0

    peak, peak_kind = load_peaks()
    achieved = kv_bytes / (decode_ms * 1e-3) / 1e9
    summaries = {"llama": ("decode.cu", "decode_partial_llama.md"),
                 "llama_mxfp8": ("decode.cu", "decode_partial_mxfp8.md"),
                 "long_bs16": ("decode.cu", "decode_partial_long_bs16.md"),
                 "long_bs64": ("decode.cu", "decode_partial_long_bs64.md"),
                 "gqa8": ("decode_tc.cu", "decode_tc_gqa8.md"),
                 "gqa8_mxfp8": ("decode_tc_mx.cu", "decode_tc_mx_gqa8.md")}
    traffic = (kernel_traffic(*summaries[args.workload]) if args.workload in summaries and
               not args.batch else None)
    res = {
        "metric": "paged-decode KV GB/s (% of HBM peak) and decode rows/s at 1 GB300",
        "value": world * kv_bytes / (ms_step * 1e-3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp8 K/V, bf16 q/out" if mx else b.dtype,
        "data": "synthetic (seeded N(0,1) q/k/v, seeded lengths and block placement)",
        "config": decode_config(args.workload, b, psize, world),
        "decode_ctas": ctas,
        "rows_per_s": world * B / (ms_step * 1e-3),
        "pct_of_hbm_peak": 100.0 * (kv_bytes / (ms_step * 1e-3) / 1e9) / peak,
        "decode_ms": decode_ms,
        "append_ms": append_ms,
        "roofline": {"bound": "hbm",
                     "kernel": {"gqa8": "decode_tc_kernel",
                                "gqa8_mxfp8": "decode_tc_mx_kernel"}.get(
                                    args.workload, "decode_partial_kernel") + " + decode_reduce_kernel",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": kv_bytes},
        "e2e": {"value": world * kv_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "double-buffered: step i's inputs copied on a side stream while step "
                          "i - 1 computes; outputs read back on a third stream"},
        "gpu_launches": args.steps * (3 + (ratio > 1)),  # append, [expand,] partial, reduce
        "clocks": clk,
    }
    return res, b


# ------------------------------------------------------------------ shared prefix
def run_shared(args, rank, world, local):
    """Shared-prefix batch: 128 requests on one 2048-token prefix (128 full
    blocks) plus private suffixes U{16..512} whose first 8 rows were copied on
    write from the parent's shared tail block."""
    import torch
    from paged_kv_cache_41_gb300 import pkv
    from paged_kv_cache_41_gb300 import workloads as wl

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    pkv.load_library()
    sp = wl.shared_prefix_batch(device=dev, seed=5 + rank, batch=args.batch or 128,
                                **({"prefix_len": args.prefix_len} if args.prefix_len else {}))
    shape = (sp.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    pkv.kv_append(kc, vc, sp.parent_k, sp.parent_v, torch.from_numpy(sp.parent_slots).to(dev))
    pairs = torch.from_numpy(sp.cow_pairs).to(dev)
    pkv.kv_block_copy(kc, vc, pairs)
    pkv.kv_append(kc, vc, sp.child_k, sp.child_v, torch.from_numpy(sp.child_slots).to(dev))
    pre = torch.from_numpy(sp.prefix_block_ids).to(dev)
    st = torch.from_numpy(sp.suffix_tables).to(dev)
    sl = torch.from_numpy(sp.suffix_lens).to(dev)
    B, Hq, D = sp.num_seqs, sp.num_q_heads, sp.head_dim
    out = torch.empty_like(sp.q)
    ws = torch.empty(pkv.shared_prefix_workspace_bytes(kc, B, Hq, sp.prefix_len, st.shape[1]),
                     dtype=torch.uint8, device=dev)
    split = pkv.prefix_split_len(kc, B, Hq, sp.prefix_len)
    nsplit = -(-sp.prefix_len // split)
    so = torch.empty(B, Hq, nsplit, D, dtype=torch.float32, device=dev)
    sls = torch.empty(B, Hq, nsplit, dtype=torch.float32, device=dev)
    # > L2 (129 MB); long enough (~150 us) that the host is always ahead of the GPU
    flush = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    stream = torch.cuda.current_stream()

    def prefix_call():
        pkv.prefix_attention_states(sp.q, kc, vc, pre, sp.prefix_len, sp.scale, split_len=split,
                                    states_o=so, states_lse=sls)

    def full_call():
        pkv.shared_prefix_attention(sp.q, kc, vc, pre, sp.prefix_len, st, sl, sp.scale, out=out,
                                    workspace=ws)

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            flush.fill_(1)  # evict the prefix K/V and q from L2 before each call
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))

    for _ in range(args.warmup):
        prefix_call()
        full_call()
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    n = max(args.steps, 20)
    prefix_ms = all_max(timed(prefix_call, n), world)
    full_ms = all_max(timed(full_call, n), world)
    clk = clocks.stop()
    assert pkv.get_device_error() == 0

    # end to end: q, tables and lengths from pinned host memory, output back
    h_q, h_st, h_sl = sp.q.cpu().pin_memory(), st.cpu().pin_memory(), sl.cpu().pin_memory()
    h_pre = pre.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    d_q, d_st, d_sl, d_pre = (torch.empty_like(x) for x in (sp.q, st, sl, pre))
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_st, h_sl, h_pre))
    d2h = h_out.numel() * h_out.element_size()

    def e2e():
        d_q.copy_(h_q, non_blocking=True)
        d_st.copy_(h_st, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        d_pre.copy_(h_pre, non_blocking=True)
        pkv.shared_prefix_attention(d_q, kc, vc, d_pre, sp.prefix_len, d_st, d_sl, sp.scale,
                                    out=out, workspace=ws)
        h_out.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e()
    e2e_ms = timed(e2e, n)
    assert pkv.get_device_error() == 0

    flops = 4.0 * B * Hq * sp.prefix_len * D
    tflops = flops / (prefix_ms * 1e-3) / 1e12
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(peaks.get("bf16_tflops", 1900.0))
    row = kv_row_bytes_dims(sp.num_kv_heads, D, 2)
    logical = B * (sp.prefix_len + float(sp.suffix_lens.mean())) * row
    unique = (sp.prefix_len + float(sp.suffix_lens.sum())) * row
    res = {
        "metric": "shared-prefix TFLOP/s (prefix contraction on tensor cores, % of dense bf16 peak)",
        "value": world * tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": n,
        "warmup": args.warmup, "ms_per_step": full_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, seeded suffix lengths and block placement)",
        "config": {"workload": "shared-prefix batch", "batch": B, "prefix_len": sp.prefix_len,
                   "suffix_len_mean": float(sp.suffix_lens.mean()), "num_q_heads": Hq,
                   "num_kv_heads": sp.num_kv_heads, "head_dim": D, "block_size": sp.block_size,
                   "prefix_split_len": split, "prefix_splits": nsplit,
                   "cow_pairs": int(sp.cow_pairs.shape[0]),
                   "l2": "flushed (1 GiB write) before every timed call"},
        "prefix_ms": prefix_ms,
        "shared_prefix_call_ms": full_ms,
        "logical_kv_bytes": logical, "unique_kv_bytes": unique,
        "effective_kv_gbps": logical / (full_ms * 1e-3) / 1e9,
        "roofline": {"bound": "tensor", "kernel": "prefix_attention_kernel",
                     "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "peak_kind": "measured bf16_tflops (burst, kernel timed alone)",
                     "traffic": kernel_traffic("prefix_tc.cu", "prefix_attention_shared.md"),
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": world * logical / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s (logical K/V)",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": n * 5,  # prefix states; prefix, plan, partial, reduce
        "clocks": clk,
    }
    return res, sp


# ------------------------------------------------------------------ prefix tree
TREE_SHAPE = dict(root_len=2048, groups=4, group_len=1024, leaf_lo=16, leaf_hi=512)


def tree_batch(device, seed, batch):
    from paged_kv_cache_41_gb300 import workloads as wl
    tree = wl.multi_level_tree(batch=batch, seed=seed, **TREE_SHAPE)
    return wl.prefix_tree_batch(tree, device=device, seed=seed)


def run_tree(args, rank, world, local):
    """Multi-level shared prefixes: 128 requests under one 2048-token root,
    four groups of 32 under their own chunk of 512..1024 tokens, and a private
    leaf of 16..512 tokens each.  One call attends every request over its
    whole path (chunk-first tensor-core phase, decode of the leaves, merge)."""
    import torch
    from paged_kv_cache_41_gb300 import pkv

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    pkv.load_library()
    tb = tree_batch(dev, 6 + rank, args.batch or 128)
    shape = (tb.num_blocks, tb.block_size, tb.num_kv_heads, tb.head_dim)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    pkv.kv_append(kc, vc, tb.k_rows, tb.v_rows, torch.from_numpy(tb.slots).to(dev))
    B, Hq, D = tb.num_seqs, tb.num_q_heads, tb.head_dim
    plan = pkv.chunk_tree_plan(kc, tb.chunks, tb.block_ids, B, Hq)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    out = torch.empty_like(tb.q)
    flush = torch.empty(1 << 30, dtype=torch.uint8, device=dev)  # > L2 (129 MB)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    stream = torch.cuda.current_stream()

    def call():
        pkv.chunk_tree_attention(tb.q, kc, vc, plan, tb.scale, out=out, workspace=ws)

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            flush.fill_(1)  # evict the K/V, states and q from L2 before each call
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    n = max(args.steps, 20)
    call_ms = all_max(timed(call, n), world)
    clk = clocks.stop()
    assert pkv.get_device_error() == 0

    # end to end: each step re-plans the snapshot on the host (the leaves grow
    # every decode step), copies the plan and q from pinned memory, attends
    # and reads the output back.  Two pinned plan buffers alternate; a buffer
    # is re-planned only after the copy that read it has run.
    cap = int(plan.host.numel()) + 4096
    h_plans = [torch.empty(cap, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    d_plans = [torch.empty(cap, dtype=torch.uint8, device=dev) for _ in range(2)]
    copied = [None, None]
    h_q = tb.q.cpu().pin_memory()
    d_q = torch.empty_like(tb.q)
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    step = [0]

    def e2e():
        i = step[0] % 2
        step[0] += 1
        if copied[i] is not None:
            copied[i].synchronize()
        p = pkv.chunk_tree_plan(kc, tb.chunks, tb.block_ids, B, Hq, host_buffer=h_plans[i],
                                device_buffer=d_plans[i])
        copied[i] = torch.cuda.Event()
        copied[i].record(stream)
        d_q.copy_(h_q, non_blocking=True)
        pkv.chunk_tree_attention(d_q, kc, vc, p, tb.scale, out=out, workspace=ws)
        h_out.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e()
    e2e_ms = timed(e2e, n)
    assert pkv.get_device_error() == 0
    h2d = int(plan.host.numel()) + h_q.numel() * h_q.element_size()
    d2h = h_out.numel() * h_out.element_size()

    hbm, kind = load_peaks()
    row = kv_row_bytes_dims(tb.num_kv_heads, D, 2)
    ch = tb.chunks.astype(np.int64)
    cov = ch[:, 3] - ch[:, 2]
    logical = float((ch[:, 1] * cov).sum()) * row
    unique = float(ch[:, 1].sum()) * row
    shared = cov > 1
    flops_cf = 4.0 * float((ch[shared, 1] * cov[shared]).sum()) * Hq * D
    achieved = unique / (call_ms * 1e-3) / 1e9
    res = {
        "metric": "prefix-tree attention: logical KV GB/s (K/V bytes per-request decode "
                  "would read / call time)",
        "value": world * logical / (call_ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": call_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, seeded chunk lengths and block placement)",
        "config": {"workload": "three-level prefix tree", "batch": B, **TREE_SHAPE,
                   "chunks": int(len(ch)), "num_q_heads": Hq, "num_kv_heads": tb.num_kv_heads,
                   "head_dim": D, "block_size": tb.block_size, "threshold": 1,
                   "l2": "flushed (1 GiB write) before every timed call"},
        "tree_call_ms": call_ms,
        "logical_kv_bytes": logical, "unique_kv_bytes": unique,
        "saved_kv_reads": logical - unique,
        "chunk_first_flops": flops_cf,
        "roofline": {"bound": "hbm", "kernel": "whole call (prefix_attention_kernel, "
                     "decode_partial_kernel, decode_reduce_kernel, tree_merge_kernel)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_kind": f"{kind} hbm_gbs (copy)", "traffic": None,
                     "algorithmic_bytes_per_launch": unique},
        "e2e": {"value": world * logical / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s (logical K/V)",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "includes": "host planning of the snapshot every step"},
        "gpu_launches": n * 4,  # chunk-first, decode partial, reduce, merge
        "clocks": clk,
    }
    return res, tb


# ------------------------------------------------------------------ append / block copy
COPY_PAIRS = 16384  # copy-on-write (src, dst) block pairs per block_copy call


def cache_ops_inputs(args, dev, seed_offset):
    """The Llama-shaped batch's pool and rows; for block_copy also a filled
    pool and COPY_PAIRS (src, dst) pairs over disjoint blocks."""
    b = make_batch("llama", dev, seed_offset=seed_offset, batch=args.batch)
    pairs = None
    if args.workload == "block_copy":
        rng = np.random.default_rng(7 + seed_offset)
        n = min(COPY_PAIRS, b.num_blocks // 2)
        perm = rng.permutation(b.num_blocks)
        pairs = np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int64)
    return b, pairs


def run_cache_ops(args, rank, world, local):
    """kv_append of every history row of the Llama-shaped batch (a prefill's
    scatter, 294k rows), or kv_block_copy of COPY_PAIRS whole blocks (K and
    V): byte copies, bound by HBM read + write."""
    import torch
    from paged_kv_cache_41_gb300 import pkv
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    pkv.load_library()
    b, pairs = cache_ops_inputs(args, dev, rank)
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    kc = torch.zeros(shape, dtype=b.k_hist.dtype, device=dev)
    vc = torch.zeros_like(kc)
    slots = torch.from_numpy(b.slots).to(dev)
    row = b.num_kv_heads * b.head_dim * b.k_hist.element_size()  # bytes of one K (or V) row
    stream = torch.cuda.current_stream()
    append = args.workload == "append"
    if append:
        nbytes = 2 * 2 * b.k_hist.shape[0] * row  # K and V, read + written

        def call():
            pkv.kv_append(kc, vc, b.k_hist, b.v_hist, slots)
    else:
        pkv.kv_append(kc, vc, b.k_hist, b.v_hist, slots)
        d_pairs = torch.from_numpy(pairs).to(dev)
        nbytes = 2 * 2 * len(pairs) * b.block_size * row

        def call():
            pkv.kv_block_copy(kc, vc, d_pairs)

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, e in evs:
            a.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(e) for a, e in evs]))

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    n = max(args.steps, 20)
    ms = all_max(timed(call, n), world)
    clk = clocks.stop()
    assert pkv.get_device_error() == 0

    # end to end: the step's inputs from pinned host memory (the rows and
    # their slots, or the pairs), the call, and a read of the device error
    # word as the step's result
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    h_err = torch.empty(1, dtype=torch.int32, pin_memory=True)
    if append:
        h_k, h_v = b.k_hist.cpu().pin_memory(), b.v_hist.cpu().pin_memory()
        h_s = slots.cpu().pin_memory()
        d_k, d_v, d_s = torch.empty_like(b.k_hist), torch.empty_like(b.v_hist), torch.empty_like(slots)
        h2d = h_k.numel() * h_k.element_size() * 2 + h_s.numel() * 8

        def e2e():
            d_k.copy_(h_k, non_blocking=True)
            d_v.copy_(h_v, non_blocking=True)
            d_s.copy_(h_s, non_blocking=True)
            pkv.kv_append(kc, vc, d_k, d_v, d_s)
            h_err.copy_(err, non_blocking=True)
    else:
        h_p = torch.from_numpy(pairs).pin_memory()
        d_p = torch.empty_like(d_pairs)
        h2d = h_p.numel() * 8

        def e2e():
            d_p.copy_(h_p, non_blocking=True)
            pkv.kv_block_copy(kc, vc, d_p)
            h_err.copy_(err, non_blocking=True)

    for _ in range(3):
        e2e()
    e2e_ms = timed(e2e, n)
    assert pkv.get_device_error() == 0

    hbm, kind = load_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    kname = "kv_append_kernel" if append else "kv_block_copy_kernel"
    summary = "kv_append_prefill.md" if append else "kv_block_copy.md"
    traffic = kernel_traffic("append_copy.cu", summary) if not args.batch else None
    res = {
        "metric": ("kv_append" if append else "kv_block_copy") +
                  " GB/s (K/V bytes read + written per call / call time)",
        "value": world * achieved, "unit": "GB/s", "n_gpus": world, "steps": n,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": b.dtype,
        "data": "synthetic (seeded N(0,1) k/v rows, seeded block placement)",
        "config": {"workload": ("prefill-scale append: every history row of the "
                                "llama3-8b-shaped batch" if append else
                                f"copy-on-write of {len(pairs)} whole blocks (K and V) of the "
                                "llama3-8b-shaped pool"),
                   "rows": int(b.k_hist.shape[0]), "num_kv_heads": b.num_kv_heads,
                   "head_dim": b.head_dim, "block_size": b.block_size,
                   "pool_blocks": b.num_blocks, "bytes_per_call": nbytes,
                   "l2": f"inputs larger than L2 ({nbytes / 2e9:.2f} GB read per call)",
                   "parallelism": f"replicas x{world} (no collective)"},
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm,
                     "peak_kind": f"{kind} hbm_gbs (copy: read + write bytes)",
                     "traffic": traffic, "algorithmic_bytes_per_launch": nbytes},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
        "gpu_launches": n,
        "clocks": clk,
    }
    return res, (b, pairs)


def cache_ops_cpu_sample(b, pairs, workload, seconds):
    """The oracle's kv_append (or kv_block_copy) on samples of the same rows
    (or pairs) until about `seconds` of CPU work: (bytes, elapsed, sample)."""
    import oracle
    from paged_kv_cache_41_gb300 import workloads as wl
    kh_all, vh_all = wl.to_numpy_storage(b.k_hist.cpu()), wl.to_numpy_storage(b.v_hist.cpu())
    row = kh_all[0].nbytes
    done = 0
    elapsed = 0.0
    calls = 0
    if workload == "append":
        n = min(16384, kh_all.shape[0])
        kc = np.zeros((n // b.block_size + 1, b.block_size) + kh_all.shape[1:], kh_all.dtype)
        vc = np.zeros_like(kc)
        slots = np.random.default_rng(0).permutation(n).astype(np.int64)
        while elapsed < seconds:
            lo = (calls * n) % max(1, kh_all.shape[0] - n)
            k, v = kh_all[lo:lo + n], vh_all[lo:lo + n]
            t0 = time.perf_counter()
            oracle.kv_append(kc, vc, k, v, slots)
            elapsed += time.perf_counter() - t0
            done += 4 * n * row
            calls += 1
        desc = f"{calls} calls of {n} rows into a private pool"
    else:
        nb = 2 * min(1024, len(pairs))
        shape = (nb, b.block_size) + kh_all.shape[1:]
        kc = np.zeros(shape, kh_all.dtype)
        kc.reshape(-1)[:] = np.resize(kh_all.reshape(-1), kc.size)  # rows repeated as needed
        vc = kc.copy()
        pp = np.stack([np.arange(nb // 2), np.arange(nb // 2, nb)], axis=1).astype(np.int64)
        while elapsed < seconds:
            t0 = time.perf_counter()
            oracle.kv_block_copy(kc, vc, pp)
            elapsed += time.perf_counter() - t0
            done += 4 * len(pp) * b.block_size * row
            calls += 1
        desc = f"{calls} calls of {len(pp)} block pairs in a private pool"
    return done, elapsed, desc + ", single-threaded C oracle"


def tree_cpu_baseline(tb, seconds):
    """The oracle's definition on whole requests of the tree batch."""
    import oracle
    from paged_kv_cache_41_gb300 import workloads as wl
    nthreads = len(os.sched_getaffinity(0))
    shape = (tb.num_blocks, tb.block_size, tb.num_kv_heads, tb.head_dim)
    hk = np.zeros(shape, np.uint16)
    hv = np.zeros(shape, np.uint16)
    slots = np.concatenate([
        np.array([oracle.slot_for_position(tb.block_ids[f:], tb.block_size, t)
                  for t in range(int(n))], np.int64) for f, n, _, _ in tb.chunks])
    oracle.kv_append(hk, hv, wl.to_numpy_storage(tb.k_rows), wl.to_numpy_storage(tb.v_rows), slots)
    q = wl.to_numpy_storage(tb.q)
    row = kv_row_bytes_dims(tb.num_kv_heads, tb.head_dim, 2)
    done, el, nbytes = 0, 0.0, 0.0
    while el < seconds and done < tb.num_seqs:
        r = done
        mine = [c for c in tb.chunks if c[2] <= r < c[3]]
        sub = np.array([(f, n, 0, 1) for f, n, _, _ in mine], np.int32)
        t0 = time.perf_counter()
        oracle.chunk_tree(np.ascontiguousarray(q[r:r + 1]), hk, hv, sub, tb.block_ids, tb.scale,
                          nthreads=nthreads)
        el += time.perf_counter() - t0
        nbytes += sum(int(n) for _, n, _, _ in mine) * row
        done += 1
    return {"value": nbytes / el / 1e9, "unit": "GB/s (logical K/V)", "cores": nthreads,
            "kind": "oracle", "seconds": el,
            "sample": f"{done} of {tb.num_seqs} requests, all heads, whole path, fp64 oracle"}


# ------------------------------------------------------------------ churn trace
def run_churn(args, rank, world, local, want_batch=True):
    """256 concurrent requests; each step appends one row per request, then
    decodes.  Requests finish (geometric output lengths) and are replaced by
    arrivals whose whole prompt is appended first (untimed, as prefill).  The
    first W steps are warm-up; the next K are timed per step with CUDA events
    around the step's append and around its decode."""
    import torch
    from paged_kv_cache_41_gb300 import pkv
    from paged_kv_cache_41_gb300 import workloads as wl

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    pkv.load_library()
    tr = wl.ChurnTrace(seed=4 + rank, steps=args.warmup + args.steps)
    hkv, d, hq, p = 8, 128, 32, tr.block_size
    shape = (tr.num_blocks, p, hkv, d)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    gen = wl.make_generator(4 + rank, dev)
    B = tr.concurrency
    q = wl.randn((B, hq, d), "bf16", gen, dev)
    out = torch.empty_like(q)
    row = 2 * hkv * d * 2
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    t_app = t_dec = t_e2e = 0.0
    kv_bytes = 0
    h2d = d2h = 0
    n_timed = 0
    ws = None
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    for i, st in enumerate(tr.run()):
        timed = i >= args.warmup
        if i == args.warmup:
            torch.cuda.synchronize()
            barrier(world)
            clocks.start()
        if st.arrival_rows:
            ak = wl.randn((st.arrival_rows, hkv, d), "bf16", gen, dev)
            av = wl.randn((st.arrival_rows, hkv, d), "bf16", gen, dev)
            pkv.kv_append(kc, vc, ak, av, torch.from_numpy(st.arrival_slots).to(dev))
        nk = wl.randn((B, hkv, d), "bf16", gen, dev)
        nv = wl.randn((B, hkv, d), "bf16", gen, dev)
        h_slots = torch.from_numpy(st.step_slots).pin_memory()
        h_bt = torch.from_numpy(st.block_tables).pin_memory()
        h_sl = torch.from_numpy(st.seq_lens).pin_memory()
        h_k, h_v = nk.cpu().pin_memory(), nv.cpu().pin_memory()
        need = pkv.decode_workspace_bytes(kc, B, hq, h_bt.shape[1])
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        # end to end: this step's inputs from pinned host memory, output back
        ev[0].record(stream)
        d_slots = h_slots.to(dev, non_blocking=True)
        d_bt = h_bt.to(dev, non_blocking=True)
        d_sl = h_sl.to(dev, non_blocking=True)
        d_k = h_k.to(dev, non_blocking=True)
        d_v = h_v.to(dev, non_blocking=True)
        ev[1].record(stream)
        pkv.kv_append(kc, vc, d_k, d_v, d_slots)
        ev[2].record(stream)
        pkv.paged_attention_decode(q, kc, vc, d_bt, d_sl, 1.0 / math.sqrt(d), out=out,
                                   workspace=ws)
        ev[3].record(stream)
        h_out.copy_(out, non_blocking=True)
        ev[4].record(stream)
        if timed:
            torch.cuda.synchronize()
            t_app += ev[1].elapsed_time(ev[2])
            t_dec += ev[2].elapsed_time(ev[3])
            t_e2e += ev[0].elapsed_time(ev[4])
            kv_bytes += int(st.seq_lens.astype(np.int64).sum()) * row
            h2d += sum(t.numel() * t.element_size() for t in (h_slots, h_bt, h_sl, h_k, h_v))
            d2h += h_out.numel() * h_out.element_size()
            n_timed += 1
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert pkv.get_device_error() == 0
    t_dec = all_max(t_dec, world)
    t_app = all_max(t_app, world)
    t_e2e = all_max(t_e2e, world)
    peak, peak_kind = load_peaks()
    achieved = kv_bytes / (t_dec * 1e-3) / 1e9
    ms_step = (t_app + t_dec) / n_timed
    res = {
        "metric": "paged-decode KV GB/s (% of HBM peak) and decode rows/s at 1 GB300",
        "value": world * achieved, "unit": "GB/s", "n_gpus": world, "steps": n_timed,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded churn trace: lognormal prompts, geometric outputs, N(0,1) q/k/v)",
        "config": {"workload": "churn trace decode", "concurrency": B, "num_q_heads": hq,
                   "num_kv_heads": hkv, "head_dim": d, "block_size": p,
                   "pool_blocks": tr.num_blocks, "kv_bytes_timed": kv_bytes,
                   "l2": "inputs larger than L2 (K/V read per step >> 129 MB)",
                   "parallelism": f"replicas x{world} (sequences shard, no collective)"},
        "rows_per_s": world * B * n_timed / ((t_app + t_dec) * 1e-3),
        "pct_of_hbm_peak": 100.0 * achieved / peak,
        "decode_ms": t_dec / n_timed, "append_ms": t_app / n_timed,
        "roofline": {"bound": "hbm", "kernel": "decode_partial_kernel + decode_reduce_kernel",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy)", "traffic": None,
                     "algorithmic_bytes_per_launch": kv_bytes / max(1, n_timed)},
        "e2e": {"value": world * kv_bytes / (t_e2e * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": t_e2e / n_timed, "h2d_bytes_per_step": h2d // max(1, n_timed),
                "d2h_bytes_per_step": d2h // max(1, n_timed)},
        "gpu_launches": n_timed * 3,  # append, partial, reduce
        "clocks": clk,
    }
    return res, (make_batch("churn", "cpu", seed_offset=rank) if want_batch else None)


def kv_row_bytes_dims(hkv, d, elem):
    return 2 * hkv * d * elem


def shared_cpu_baseline(sp, seconds):
    """The oracle on whole requests of the shared-prefix batch (its own pool)."""
    import oracle
    from paged_kv_cache_41_gb300 import workloads as wl
    nthreads = len(os.sched_getaffinity(0))
    shape = (sp.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
    hk = np.zeros(shape, np.uint16)
    hv = np.zeros(shape, np.uint16)
    n_par = sp.prefix_len + sp.shared_tail
    ps = np.array([oracle.slot_for_position(sp.parent_table, sp.block_size, t)
                   for t in range(n_par)], np.int64)
    oracle.kv_append(hk, hv, wl.to_numpy_storage(sp.parent_k), wl.to_numpy_storage(sp.parent_v), ps)
    oracle.kv_block_copy(hk, hv, sp.cow_pairs)
    ck, cv = wl.to_numpy_storage(sp.child_k), wl.to_numpy_storage(sp.child_v)
    for r in range(sp.num_seqs):
        table = np.concatenate([sp.prefix_block_ids, sp.suffix_tables[r]])
        lo, hi = sp.child_offsets[r], sp.child_offsets[r + 1]
        cs = np.array([oracle.slot_for_position(table, sp.block_size, n_par + i)
                       for i in range(hi - lo)], np.int64)
        oracle.kv_append(hk, hv, np.ascontiguousarray(ck[lo:hi]), np.ascontiguousarray(cv[lo:hi]), cs)
    q = wl.to_numpy_storage(sp.q)
    done = 0
    el = 0.0
    flops = 0.0
    while el < seconds and done < sp.num_seqs:
        r = done
        t0 = time.perf_counter()
        oracle.shared_prefix(np.ascontiguousarray(q[r:r + 1]), hk, hv, sp.prefix_block_ids,
                             sp.prefix_len, np.ascontiguousarray(sp.suffix_tables[r:r + 1]),
                             np.ascontiguousarray(sp.suffix_lens[r:r + 1]), sp.scale,
                             nthreads=nthreads)
        el += time.perf_counter() - t0
        flops += 4.0 * sp.num_q_heads * sp.prefix_len * sp.head_dim
        done += 1
    return {"value": flops / el / 1e12, "unit": "TFLOP/s (prefix part)", "cores": nthreads,
            "kind": "oracle", "seconds": el,
            "sample": f"{done} of {sp.num_seqs} requests, all heads, prefix + suffix, fp64 oracle"}



# ------------------------------------------------------------------ read peak, extras
def hbm_read_peak(dev, reps=10):
    """Read-only HBM streaming peak of this GPU: the better of the two probes
    of libpkv_probe (16-byte loads that skip L1; 32 KiB bulk copies into
    shared memory), each streaming a ~4 GB buffer (>> L2) once per launch,
    best of `reps` launches timed with CUDA events on the launching stream."""
    import ctypes
    import torch
    from paged_kv_cache_41_gb300 import build as pkv_build
    lib = ctypes.CDLL(pkv_build.build_probe())
    for fn in (lib.pkv_probe_hbm_read_lsu, lib.pkv_probe_hbm_read_bulk):
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                       ctypes.c_void_p]
    lib.pkv_probe_error.restype = ctypes.c_int
    lib.pkv_probe_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nbytes = sms * 32768 * 800
    buf = torch.ones(nbytes // 4, dtype=torch.int32, device=dev)
    sink = torch.zeros(sms * 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    res = {}
    for name, fn, ctas in (("lsu", lib.pkv_probe_hbm_read_lsu, sms * 4),
                           ("bulk", lib.pkv_probe_hbm_read_bulk, sms)):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps + 2)]
        for a, b in evs:
            a.record(stream)
            rc = fn(buf.data_ptr(), nbytes, ctas, sink.data_ptr(), stream.cuda_stream)
            b.record(stream)
            assert rc == 0, f"read probe {name} failed to launch"
        torch.cuda.synchronize()
        ms = min(a.elapsed_time(b) for a, b in evs[2:])
        res[name] = nbytes / (ms * 1e-3) / 1e9
    err = ctypes.c_uint(0)
    assert lib.pkv_probe_error(ctypes.byref(err)) == 0 and err.value == 0
    del buf
    torch.cuda.empty_cache()
    best = max(res.values())
    return {"value": best, "unit": "GB/s", "lsu": res["lsu"], "bulk": res["bulk"],
            "bytes_per_launch": nbytes,
            "how": "read-only streaming of a buffer >> L2 once per launch, writing nothing "
                   f"but one word per CTA; best of {reps} launches (CUDA events); the better "
                   "of 16-byte L1-bypassing loads (4 CTAs x 512 threads per SM) and 32 KiB "
                   "cp.async.bulk copies into a 4-slot shared-memory ring (1 CTA per SM)"}


def _compact(r, read_peak=None):
    """The keys of a workload's result that an extra entry keeps."""
    keep = ("value", "unit", "ms_per_step", "steps", "warmup", "rows_per_s", "decode_ms",
            "append_ms", "pct_of_hbm_peak", "prefix_ms", "shared_prefix_call_ms", "tree_call_ms",
            "effective_kv_gbps", "unique_kv_bytes", "roofline", "clocks", "gpu_launches",
            "decode_ctas", "config")
    d = {k: r[k] for k in keep if k in r}
    d["e2e"] = {k: r["e2e"][k] for k in ("value", "unit", "ms_per_step") if k in r["e2e"]}
    if read_peak and d.get("roofline", {}).get("bound") == "hbm":
        d["roofline"] = dict(d["roofline"], read_peak=read_peak,
                             frac_of_read_peak=d["roofline"]["achieved"] / read_peak)
    return d


def run_extras(args, local):
    """The other configured workloads, measured in the same run (one GPU):
    each keeps its own timing rules (L2 flushed or inputs larger than L2) and
    its own roofline."""
    import torch

    def sub(**kw):
        d = dict(vars(args))
        d.update(kw)
        return argparse.Namespace(**d)

    out = {}
    peak = hbm_read_peak(torch.device(f"cuda:{local}"))
    out["hbm_read_peak"] = peak
    rp = peak["value"]
    for name in ("llama", "long_bs64", "gqa8", "llama_mxfp8", "gqa8_mxfp8"):
        r, _ = run_pkv(sub(workload=name, batch=0, partition_size=0), 0, 1, local)
        out[name] = _compact(r, rp)
        torch.cuda.empty_cache()
    # the churn trace as configured: 200 decode steps, the first 5 untimed
    r, _ = run_churn(sub(workload="churn", warmup=5, steps=195), 0, 1, local, want_batch=False)
    out["churn"] = _compact(r, rp)
    torch.cuda.empty_cache()
    r, _ = run_shared(sub(workload="shared", batch=0, prefix_len=0), 0, 1, local)
    out["shared"] = _compact(r, rp)
    torch.cuda.empty_cache()
    r, _ = run_tree(sub(workload="tree", batch=0), 0, 1, local)
    out["tree"] = _compact(r, rp)
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        if rank != 0:
            return
        res = run_reference(args)
        print(json.dumps(res), flush=True)
        return
    if args.workload == "shared":
        res, sp = run_shared(args, rank, world, local)
        if rank == 0 and not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = shared_cpu_baseline(sp, args.cpu_sample_seconds)
    elif args.workload == "tree":
        res, tb = run_tree(args, rank, world, local)
        if rank == 0 and not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = tree_cpu_baseline(tb, args.cpu_sample_seconds)
    elif args.workload in ("append", "block_copy"):
        res, (b, pairs) = run_cache_ops(args, rank, world, local)
        if rank == 0 and not args.no_cpu_baseline and world == 1:
            nb_, el, desc = cache_ops_cpu_sample(b, pairs, args.workload, args.cpu_sample_seconds)
            res["cpu_baseline"] = {"value": nb_ / el / 1e9, "unit": "GB/s", "cores": 1,
                                   "kind": "oracle", "sample": desc}
    elif args.workload == "churn":
        res, b = run_churn(args, rank, world, local)
        if rank == 0 and not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = cpu_baseline(b, args.cpu_sample_seconds)
    else:
        res, b = run_pkv(args, rank, world, local)
        if rank == 0 and not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = cpu_baseline(b, args.cpu_sample_seconds,
                                               args.workload.endswith("_mxfp8"))
        del b
        if (world == 1 and args.workload == "long_bs16" and not args.batch
                and not args.no_extras):
            extras = run_extras(args, local)
            rp = extras["hbm_read_peak"]["value"]
            res["roofline"]["read_peak"] = rp
            res["roofline"]["frac_of_read_peak"] = res["roofline"]["achieved"] / rp
            res["hbm_read_peak"] = extras.pop("hbm_read_peak")
            res["also_measured"] = extras
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle, as it stands, on bounded samples of the same workload."""
    if args.workload in ("append", "block_copy"):
        b, pairs = cache_ops_inputs(args, "cpu", 0)
        per_step = min(6.0, 150.0 / max(1, args.steps + args.warmup))
        cache_ops_cpu_sample(b, pairs, args.workload, per_step / 4)
        nb_ = el = 0.0
        for _ in range(args.steps):
            x, y, desc = cache_ops_cpu_sample(b, pairs, args.workload, per_step)
            nb_ += x
            el += y
        v = nb_ / el / 1e9
        return {"impl": "reference",
                "metric": ("kv_append" if args.workload == "append" else "kv_block_copy") +
                          " GB/s (K/V bytes read + written per call / call time)",
                "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16 (byte copies)", "data": "synthetic",
                "config": {"workload": args.workload},
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": f"per step: {desc}"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
    # about 150 s in all: with many steps each is a short sample (a
    # sequence's first 512 tokens)
    per_step = min(6.0, 150.0 / max(1, args.steps + args.warmup))
    max_tok = None if per_step >= 1.0 else 512
    if args.workload in ("shared", "tree"):
        # the oracle's whole-request definition, as the GPU arm's cpu_baseline
        from paged_kv_cache_41_gb300 import workloads as wl
        if args.workload == "shared":
            sp = wl.shared_prefix_batch(device="cpu", seed=5, batch=args.batch or 128,
                                        **({"prefix_len": args.prefix_len} if args.prefix_len else {}))
            cb = shared_cpu_baseline(sp, per_step * args.steps)
            metric, unit = ("shared-prefix TFLOP/s (prefix contraction on tensor cores, % of "
                            "dense bf16 peak)"), "TFLOP/s"
        else:
            cb = tree_cpu_baseline(tree_batch("cpu", 6, args.batch or 128), per_step * args.steps)
            metric, unit = ("prefix-tree attention: logical KV GB/s (K/V bytes per-request "
                            "decode would read / call time)"), "GB/s"
        v = cb["value"]
        return {"impl": "reference", "metric": metric, "value": v, "unit": unit, "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * cb["seconds"] / max(1, args.steps),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "config": {"workload": args.workload},
                "cpu_baseline": cb,
                "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    b = make_batch(args.workload, "cpu", batch=args.batch)
    mx = args.workload.endswith("_mxfp8")
    nthreads = len(os.sched_getaffinity(0))
    for _ in range(args.warmup):
        oracle_sample(b, per_step / 4, nthreads, mx, max_tok)
    tot_b = tot_r = tot_t = 0.0
    desc = ""
    for _ in range(args.steps):
        nb_, nr_, el, desc = oracle_sample(b, per_step, nthreads, mx, max_tok)
        tot_b += nb_
        tot_r += nr_
        tot_t += el
    v = tot_b / tot_t / 1e9
    return {
        "impl": "reference",
        "metric": "paged-decode KV GB/s (% of HBM peak) and decode rows/s at 1 GB300",
        "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(args.workload, b, args.partition_size,
                                int(os.environ.get("WORLD_SIZE", "1"))),
        "rows_per_s": tot_r / tot_t,
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


if __name__ == "__main__":
    main()
