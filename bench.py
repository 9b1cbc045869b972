"""Benchmark of the batched cache-aware Conformer streaming step on GB300.

Workload (default): the Parakeet-EOU-120M-shaped encoder (17 layers, d_model
512, 8 heads, ff 2048, bf16 weights, fp32 accumulation) serving 256 concurrent
synthetic streams of 60 s.  Every step pushes 160 ms (16 mel frames, 2 encoder
frames) for all 256 streams through the C-ABI (cac_stream_push), with caches
resident on the GPU, random per-stream resets at 1 % per step, and stream start
offsets drawn on 0..499 frames (even) and reached by an untimed pre-roll.

One JSON line on rank 0:  value = streamed audio-seconds per second over all
ranks (max time over ranks), e2e = the same from page-locked host buffers
(cac_stream_push_host_async: each push queued before the host reads the
previous push's frames; the one-call-at-a-time cac_stream_push_host beside it),
roofline of the dominant kernel class (CUDA events on the
launching stream, in a profiled pass of the same steps), the fp64 oracle timed
on the host cores as cpu_baseline, and the SM clocks sampled during the timed
region.  `--impl reference` times the oracle itself as the reference arm.

Multi-GPU (torchrun): every rank serves its own 256 streams (its own seeds) on
its own replica; no collective on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
from dataclasses import replace
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import WORKLOADS, FRAME_SEC, EOU_DECODER  # noqa: E402

METRIC = "streamed audio-sec/sec (B streams, 160 ms chunks) + % of tensor/HBM roofline"
UNIT = "audio-s/s"


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; barrier + max over ranks)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, local, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(ms_local: float, streams: int, frames: int, steps: int, device=None):
    """Whole-job audio-s/s: every rank streams `streams` x `frames` encoder frames
    per step (weak scaling); the job takes as long as the slowest rank."""
    import torch.distributed as dist
    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    ms_max = max_over_ranks(ms_local, device)
    audio = world * streams * frames * FRAME_SEC * steps
    return audio / (ms_max / 1e3), ms_max


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on the host cores (spawned workers)
# ---------------------------------------------------------------------------
def _oracle_worker(conn, blob_path, cfg, mel, push_mel):
    """One oracle instance stepped on command: a stream pushing `push_mel` mel
    frames per step (the provisional-tail encoder when the model has right
    context), or, with push_mel 0, one offline window encoded per step."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    from oracle import conformer as O
    blob = np.load(blob_path, mmap_mode="r")
    W = O.weights_f64(synth.unpack_weights(cfg, blob))
    enc = None
    if push_mel:
        enc = O.ProvisionalTailEncoder(W, cfg) if cfg.right_context > 0 else O.StreamingEncoder(W, cfg)
    k = 0
    conn.send("ready")
    while True:
        cmd = conn.recv()
        if cmd is None:
            break
        for _ in range(cmd):
            if push_mel:
                r = k % (mel.shape[0] // push_mel)  # an utterance shorter than the sample repeats
                enc.push(mel[push_mel * r: push_mel * (r + 1)])
                k += 1
            else:
                O.encode_offline(mel, W, cfg)
        conn.send("done")


def oracle_workers(blob, units: int) -> int:
    """Workers of a bounded oracle sample: one per host core, at most one per
    stream (or window) of the workload, and at most what half the host memory
    holds (a worker keeps the weights in fp32 and in fp64)."""
    n = max(1, min(cpu_cores(), units))
    try:
        mem = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    except (ValueError, OSError, AttributeError):
        return n
    return max(1, min(n, int(mem // 2 // (12 * blob.size + (1 << 28)))))


def workload_mel(wl, sid: int) -> np.ndarray:
    """Stream (or window) `sid`'s mel as the GPU legs generate it."""
    n = wl.offline_mel if wl.offline_batch else (int(round(wl.seconds * 100)) // wl.push_mel) * wl.push_mel
    return synth.make_mel(n, sid, silence_frac=wl.silence_frac)


class OracleFarm:
    """One worker process per stream (or offline window) of a sample, each
    stepping its own oracle instance on command."""

    def __init__(self, cfg, blob, mels, push_mel: int):
        import multiprocessing as mp
        for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"
        ctx = mp.get_context("spawn")
        self.tmp = tempfile.mkdtemp(prefix="cac_oracle_")
        self.blob_path = os.path.join(self.tmp, "w.npy")
        np.save(self.blob_path, blob)
        self.cores = len(mels)
        self.procs, self.conns = [], []
        for mel in mels:
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(b, self.blob_path, cfg, mel, push_mel), daemon=True)
            p.start()
            self.procs.append(p)
            self.conns.append(a)
        for a in self.conns:
            assert a.recv() == "ready"

    def step(self, chunks: int = 1) -> float:
        t = time.perf_counter()
        for a in self.conns:
            a.send(chunks)
        for a in self.conns:
            assert a.recv() == "done"
        return time.perf_counter() - t

    def step_one(self, chunks: int = 1) -> float:
        """Worker 0 alone (the others idle): the one-core figure."""
        t = time.perf_counter()
        self.conns[0].send(chunks)
        assert self.conns[0].recv() == "done"
        return time.perf_counter() - t

    def close(self):
        for a in self.conns:
            a.send(None)
        for p in self.procs:
            p.join(timeout=30)
        try:
            os.unlink(self.blob_path)
            os.rmdir(self.tmp)
        except OSError:
            pass


def cpu_cores() -> int:
    return max(1, min(os.cpu_count() or 1, 16))


# ---------------------------------------------------------------------------
# roofline bookkeeping: algorithmic work per launch of each kernel class
# ---------------------------------------------------------------------------
def algorithmic_work(cfg, S, n, mean_lc):
    """Per launch: ('tensor', flops) for GEMMs, ('hbm', bytes) for the rest.
    S = streams one launch covers (a sub-batch's share when the step runs as
    concurrent sub-batches); n = frames pushed per stream; the layer stack runs
    over n rows per stream (emit + lookahead rows per pass in the
    provisional-tail variant)."""
    D, F, J, L, H = cfg.d_model, cfg.ff_dim, cfg.joint_dim, cfg.n_layers, cfg.n_heads
    rows = cfg.emit_frames + cfg.lookahead_frames if cfg.provisional else n
    M = S * rows
    W1, W2, W3 = 14 + 8 * n, 4 * n + 6, 2 * n + 2
    sub_flops = 2 * D * (S * (W1 // 2) * 3 * 128 + S * (W2 // 2) * 3 * D + S * (W3 // 2) * 3 * D) / 3.0
    kv = S * (mean_lc + rows) * D * 2 * 2               # K and V rows read, bf16
    nr = cfg.att_left + cfg.att_chunk                   # position-table rows
    return {
        "gemm_ff_up": ("tensor", 2.0 * M * F * D),
        "gemm_ff_down": ("tensor", 2.0 * M * D * F),
        "gemm_qkv": ("tensor", 2.0 * M * 3 * D * D),
        "gemm_out_proj": ("tensor", 2.0 * M * D * D),
        "gemm_pw1_glu": ("tensor", 2.0 * M * 2 * D * D),
        "gemm_pw2": ("tensor", 2.0 * M * D * D),
        "gemm_joint": ("tensor", 2.0 * M * J * D),
        "gemm_sub_out": ("tensor", 2.0 * M * D * D),
        "gemm_subsample": ("tensor", sub_flops),
        # q fp32 in, K/V cache + new rows, output as a split (hi, lo) bf16 pair, bf16 position table
        "attention": ("hbm", kv + M * D * 4 + M * D * 4 + nr * D * 2),
        # GLU rows in, conv tail (8 rows) in, n rows committed, output
        "dwconv": ("hbm", M * D * 2 + S * 8 * D * 2 + M * D * 2 + M * D * 2 + 12 * D * 4),
        # per launch, averaged over the step's LayerNorm launches.  bf16: the
        # attention, conv and FF2 LayerNorms run inside the GEMMs after them, so
        # the launches are the first FF1 LayerNorm (x in 4 B, split (hi, lo)
        # bf16 out 4 B), ln_out fused with the next FF1 LayerNorm for L - 1
        # layers (x in, x in place, split out: 12 B) and the last ln_out (x in,
        # fp32 frames + plain bf16 out: 10 B).  fp32: 1 + 3L plain LayerNorms
        # as well (8 B).
        "layernorm": ("hbm", M * D * (8 + (L - 1) * 12 + 10) / (L + 1) if cfg.dtype == "bf16"
                      else M * D * ((1 + 3 * L) * 8 + (L - 1) * 12 + 10) / (4 * L + 1)),
        "stage_mel": ("hbm", S * (8 * n + 14) * 128 * 4 + S * W1 * 128 * 2 + S * 14 * 128 * 2),
        # chained steps: every projection of the layer stack, the subsampling
        # output linear and the joint run inside the chain launches; per STEP
        # (divided by the chain launches per step where it is used)
        "chain_step": ("tensor", 2.0 * M * (L * (2 * F * D + 2 * D * F + 3 * D * D + D * D + 2 * D * D + D * D)
                                            + D * D + J * D)),
    }


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of one
# ncu capture of the kernel on this workload, with the source files it was
# built from; reported only while those files are unchanged (see profiles/).
NCU_TRAFFIC = {
    # one 64-stream sub-batch launch (M = 128, 128-column tiles split 4 ways over K), as the timed steps run it
    "gemm_ff_down": (2.932480e6, {"csrc/gemm_tc.cu": "3ee627b20cf39f3b64578fd19447b597f4357505349f915fbb061634946c2f6d",
                                  "csrc/gemm.cuh": "a972a38b741b4b87d703c97f987cdb576f9d9cb0a2ffb7498fe7da05ea0ffb14",
                                  "csrc/common.cuh": "99bbe108d6f42c2d09d40fa1de59d0a862e2406fb6b9cceb8827e50bdaf781b3"}),
}


def measured_traffic(kernel_class: str, workload: str):
    """ncu DRAM bytes per launch for the 256-stream workload, or None when not
    captured for this class or when its sources changed since the capture."""
    import hashlib
    if workload != "eou120m_256streams_60s" or kernel_class not in NCU_TRAFFIC:
        return None
    nbytes, files = NCU_TRAFFIC[kernel_class]
    pkg = os.path.join(ROOT, "cache_aware_conformer_gb300")
    for rel, digest in files.items():
        with open(os.path.join(pkg, rel), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return nbytes


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops_sustained"], "measured"
    return 6800.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# the streaming workload
# ---------------------------------------------------------------------------
class StreamWorkload:
    """S synthetic streams of `seconds` of audio pushed `push_mel` mel frames at a
    time; start offsets reached by an untimed pre-roll; per-step resets."""

    def __init__(self, wl, rank: int, device, steps_needed: int, workers: int):
        import torch
        from cache_aware_conformer_gb300 import native
        self.wl, self.cfg = wl, wl.model
        self.S = wl.streams
        self.dev = device
        self.push_mel = wl.push_mel
        self.n = wl.push_mel // 8
        self.chunks = int(round(wl.seconds * 100)) // self.push_mel        # pushes per utterance
        base = rank * self.S
        self.offsets = synth.start_offsets(self.S, wl.max_start_offset, seed=7 + rank)
        self.pre = (self.offsets // self.n).astype(np.int64)                # pre-roll pushes per stream
        W = synth.make_weights_parallel(self.cfg, seed=0, workers=workers)
        self.blob = synth.pack_weights(self.cfg, W)
        del W
        mel = synth.make_mels_parallel(self.chunks * self.push_mel, range(base, base + self.S), wl.silence_frac, workers)
        self.mel = torch.from_numpy(mel).to(device).view(self.S, self.chunks, self.push_mel, 128)
        del mel
        self.model = native.Model(self.cfg, self.blob)
        self.pool = native.Pool(self.model, self.S, max_frames_per_step=max(2, min(8, self.n)))
        self.ids = [self.pool.create_stream() for _ in range(self.S)]
        # pre-roll: stream s pushes its first pre[s] chunks (untimed, eager)
        for r in range(int(self.pre.max()) if self.S else 0):
            sel = np.nonzero(self.pre > r)[0]
            chunk = self.mel[torch.from_numpy(sel).to(device), r].contiguous()
            self.pool.push([self.ids[i] for i in sel], chunk, joint=False)
        self.pool.check()
        # per-step inputs: chunk index of every stream, arranged contiguously per step;
        # an utterance that ends restarts (reset) at its first chunk
        self.t = 0
        self.steps = steps_needed
        cidx = (self.pre[None, :] + np.arange(steps_needed)[:, None]) % self.chunks      # [steps, S]
        ar = torch.arange(self.S, device=device)
        self.step_mel = torch.stack([self.mel[ar, torch.from_numpy(c).to(device)] for c in cidx])
        self.cidx = cidx
        self.resets = [np.nonzero(synth.reset_mask(self.S, t, wl.reset_prob, seed=11 + rank) | (cidx[t] == 0))[0]
                       for t in range(steps_needed)]
        self.staging = torch.empty(self.S, self.push_mel, 128, device=device)
        self.host_out = None  # (enc, joint) host buffers of the end-to-end pass
        self.enc = torch.empty(self.S, self.n, self.cfg.d_model, device=device)
        self.joint = torch.empty(self.S, self.n, self.cfg.joint_dim, device=device)
        self.lc_hist = []
        self.subT = self.pre * self.n

    def step(self):
        """One timed step: resets drawn for this step, then one push of all streams."""
        t = self.t
        r = self.resets[t]
        if len(r):
            self.pool.reset([self.ids[i] for i in r])
            self.subT[r] = 0
        self.lc_hist.append(float(np.minimum(self.subT, self.cfg.att_left).mean()))
        self.staging.copy_(self.step_mel[t])
        self.pool.push_into(self.ids, self.staging, self.enc, self.joint)
        self.subT += self.n
        self.t += 1

    def step_host(self, mel_host):
        t = self.t
        r = self.resets[t]
        if len(r):
            self.pool.reset([self.ids[i] for i in r])
            self.subT[r] = 0
        enc, joint, _ = self.pool.push_host(self.ids, mel_host, out=self.host_out)
        self.subT += self.n
        self.t += 1
        return enc, joint

    def step_host_async(self, mel_host, out):
        """Queue one host-buffer push into `out` (frames there once the
        default stream has passed it)."""
        t = self.t
        r = self.resets[t]
        if len(r):
            self.pool.reset([self.ids[i] for i in r])
            self.subT[r] = 0
        self.pool.push_host_async(self.ids, mel_host, out)
        self.subT += self.n
        self.t += 1


class OfflineWorkload:
    """B windows of offline_mel mel frames encoded in one cac_encode_offline call per step."""

    def __init__(self, wl, rank: int, device, workers: int):
        import torch
        from cache_aware_conformer_gb300 import native
        self.wl, self.cfg = wl, wl.model
        self.B, self.T = wl.offline_batch, wl.offline_mel
        W = synth.make_weights_parallel(self.cfg, seed=0, workers=workers)
        self.blob = synth.pack_weights(self.cfg, W)
        del W
        base = rank * self.B
        mel = synth.make_mels_parallel(self.T, range(base, base + self.B), wl.silence_frac, workers)
        self.mel = torch.from_numpy(mel).to(device)
        self.lens = [self.T] * self.B
        self.model = native.Model(self.cfg, self.blob)
        T3 = self.T
        for _ in range(3):
            T3 = (T3 + 1) // 2
        self.T3 = T3
        self.enc = torch.empty(self.B, T3, self.cfg.d_model, device=device)
        self.joint = torch.empty(self.B, T3, self.cfg.joint_dim, device=device)

    def step(self):
        self.model.encode_offline(self.mel, self.lens, out=(self.enc, self.joint))


def run_offline(args, wl):
    import torch
    rank, local, world = dist_init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K, Wm = args.steps, args.warmup
    w = OfflineWorkload(wl, rank, dev, max(1, min(cpu_cores(), 16)))
    for _ in range(Wm):
        w.step()
    torch.cuda.synchronize()
    barrier()
    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip().isdigit()]
    clocks = ClockSampler(int(vis[local]) if local < len(vis) else local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    e0.record()
    for _ in range(K):
        w.step()
    e1.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    w.model.check()
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    audio = world * w.B * w.T * 0.01 * K
    value = audio / (ms / 1e3)
    # e2e: host mel in, host frames out, through the same entry point
    mel_h = w.mel.cpu().pin_memory()
    t0 = time.perf_counter()
    for _ in range(max(1, K // 4)):
        m = mel_h.to(dev, non_blocking=True)
        w.model.encode_offline(m, w.lens, out=(w.enc, w.joint))
        enc_h, joint_h = w.enc.cpu(), w.joint.cpu()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    e2e = {"value": world * w.B * w.T * 0.01 * max(1, K // 4) / e2e_s, "unit": UNIT,
           "h2d_bytes_per_step": w.B * w.T * 128 * 4, "d2h_bytes_per_step": w.B * w.T3 * (w.cfg.d_model + w.cfg.joint_dim) * 4}
    # tensor roofline of the whole encode (GEMM FLOPs per window)
    _, tf_peak, peak_src = load_peaks()
    D, F, J, L = w.cfg.d_model, w.cfg.ff_dim, w.cfg.joint_dim, w.cfg.n_layers
    flops = 2.0 * w.B * w.T3 * (L * (2 * 2 * D * F + 3 * D * D + D * D + 2 * D * D + D * D) + J * D)
    ach = flops / (ms / K * 1e-3) / 1e12
    roofline = {"kernel": "whole offline encode (GEMM FLOPs only)", "bound": "tensor", "achieved": ach,
                "peak": tf_peak, "unit": "TFLOP/s", "frac": ach / tf_peak, "traffic": None,
                "peak_source": f"{peak_src} (bf16 sustained)"}
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            try:
                cpu = cpu_baseline(wl, w.blob, 1)
            except Exception as exc:  # reported beside the GPU figures, never instead of them
                cpu = {"error": f"{type(exc).__name__}: {exc}"[:300], "kind": "oracle"}
        print(json.dumps({"metric": workload_metric(wl), "value": value, "unit": UNIT,
                          "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms / K, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                          "config": {"workload": wl.name, "windows": w.B, "mel_frames": w.T, "frames": w.T3,
                                     "layers": L, "d_model": D, "parallelism": f"replicas x{world}"},
                          "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": None,
                          "clocks": clk}), flush=True)


def run_ours(args, wl):
    import torch
    rank, local, world = dist_init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K, Wm = args.steps, args.warmup
    Kp = min(K, args.profile_steps)
    Ke = min(K, args.e2e_steps)
    Kd = min(K, args.decode_steps) if wl.model.joint_dim == EOU_DECODER.joint_dim and not wl.model.provisional else 0
    E_WARM = 3 if Ke else 0  # untimed host-buffer pushes before the e2e leg (its staging buffers and graph)
    total_steps = Wm + K + 2 * Kp + E_WARM + 2 * Ke + (Kd + 3 if Kd else 0)
    workers = max(1, min(cpu_cores(), 16))
    w = StreamWorkload(wl, rank, dev, total_steps, workers)
    w.pool.set_graphs(True)
    for _ in range(Wm):
        w.step()
    torch.cuda.synchronize()
    # ---- timed region: K steps, device-timed with CUDA events on the launching stream
    barrier()
    torch.cuda.synchronize()
    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip().isdigit()]
    clocks = ClockSampler(int(vis[local]) if local < len(vis) else local)
    clocks.start()
    time.sleep(0.3)
    launches0 = w.pool.launch_count()
    lc0 = len(w.lc_hist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    e0.record()
    for _ in range(K):
        w.step()
    e1.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    ms = e0.elapsed_time(e1)
    launches = w.pool.launch_count() - launches0
    mean_lc = float(np.mean(w.lc_hist[lc0:]))
    w.pool.check()
    value, ms_max = aggregate_throughput(ms, w.S, w.n, K, dev)

    # ---- per-push latency: one push at a time (graph replay), CUDA events
    # around each push, synchronized between pushes
    lat = []
    for _ in range(Kp):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        w.step()
        a1.record()
        a1.synchronize()
        lat.append(a0.elapsed_time(a1))
    latency = {"p50_ms": float(np.percentile(lat, 50)), "p95_ms": float(np.percentile(lat, 95)),
               "pushes": len(lat), "note": "one push of all streams, graph replay, device time"} if lat else None

    # ---- profiled pass of the same steps: per-kernel-class CUDA events (the
    # timed steps' sub-batches, eager launches; NVTX range "profiled")
    w.pool.set_profile(True)
    w.pool.read_profile()
    torch.cuda.nvtx.range_push("profiled")
    for _ in range(Kp):
        w.step()
    torch.cuda.nvtx.range_pop()
    prof = w.pool.read_profile()
    w.pool.set_profile(False)
    hbm_peak, tf_peak, peak_src = load_peaks()
    # a launch covers one sub-batch: S / G streams when the step runs as G
    # concurrent sub-batches (the profiled steps keep the timed steps' split)
    G = w.pool.sub_batches(w.S, w.n)
    work = algorithmic_work(w.cfg, w.S / G, w.n, mean_lc)
    if "chain" in prof and prof["chain"][1]:
        # chained steps: the chain launches carry the step's projection FLOPs
        work["chain"] = ("tensor", work["chain_step"][1] / (prof["chain"][1] / max(Kp, 1)))
    kernels = {}
    for name, (tot, cnt) in prof.items():
        if cnt == 0:
            continue
        ent = {"total_ms_per_step": tot / Kp, "launches_per_step": cnt / Kp, "avg_us": 1e3 * tot / cnt}
        if name in work:
            bound, amount = work[name]
            if bound == "tensor":
                ach = amount / (tot / cnt * 1e-3) / 1e12
                ent.update(bound="tensor", achieved=ach, unit="TFLOP/s", frac=ach / tf_peak)
            else:
                ach = amount / (tot / cnt * 1e-3) / 1e9
                ent.update(bound="hbm", achieved=ach, unit="GB/s", frac=ach / hbm_peak)
        kernels[name] = ent
    roofline = None
    bounded = [k for k in kernels if "bound" in kernels[k]]
    if bounded:
        dom = max(bounded, key=lambda k: kernels[k]["total_ms_per_step"])
        d = kernels[dom]
        roofline = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"],
                    "peak": tf_peak if d["bound"] == "tensor" else hbm_peak, "unit": d["unit"], "frac": d["frac"],
                    "traffic": measured_traffic(dom, wl.name),
                    "peak_source": f"{peak_src} ({'bf16 sustained' if d['bound'] == 'tensor' else 'HBM copy'})",
                    "per_launch": work[dom][1], "avg_launch_us": d["avg_us"],
                    "measured_in": (f"profiled pass in the timed steps' launch configuration: {G} concurrent "
                                    f"sub-batch(es) of {w.S // G} streams, each on its own stream, launched eagerly "
                                    "instead of replayed from graphs; CUDA events on the launching stream around "
                                    "every launch (overlapping launches of different sub-batches each count their "
                                    "own duration)")}

    # ---- end to end through the C-ABI with host buffers (copies inside the timed region)
    # inputs and results in page-locked host memory (copied directly by the library).
    # The first host-buffer pushes allocate the library's staging buffers and
    # capture the step's graph for them, so a few run untimed first, as the
    # device-timed leg's warm-up steps do.  Timed: each step's push is queued
    # (cac_stream_push_host_async) before the host waits for the previous
    # step's frames and reads them from the other of two output buffers; the
    # last step's frames are waited for and read inside the timed region.
    # Beside it, the same steps one synchronous cac_stream_push_host at a time.
    host_mels = [w.step_mel[w.t + i].cpu().pin_memory() for i in range(E_WARM + 2 * Ke)]
    outs = [(torch.empty(w.S, w.n, w.cfg.d_model).pin_memory(),
             torch.empty(w.S, w.n, w.cfg.joint_dim).pin_memory()) for _ in range(2)]
    w.host_out = outs[0]
    for i in range(E_WARM):
        w.step_host(host_mels[i])
    host_mels = host_mels[E_WARM:]
    evs = [torch.cuda.Event(), torch.cuda.Event()]
    out_np = [(e.numpy(), j.numpy()) for e, j in outs]  # host reads through numpy views of the pinned buffers
    seen = float(out_np[0][1][:, -1, 0].sum())
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for i in range(Ke):
        w.step_host_async(host_mels[i], outs[i % 2])
        evs[i % 2].record()
        if i:
            evs[(i - 1) % 2].synchronize()
            seen += float(out_np[(i - 1) % 2][1][:, -1, 0].sum())  # the host reads the step's joint frames
    if Ke:
        evs[(Ke - 1) % 2].synchronize()
        seen += float(out_np[(Ke - 1) % 2][1][:, -1, 0].sum())
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for i in range(Ke):
        w.step_host(host_mels[Ke + i])
    e2e_sync_s = max_over_ranks(time.perf_counter() - t0, dev)
    e2e = None  # not measured with --e2e-steps 0
    if Ke:
        e2e = {"value": world * w.S * w.n * FRAME_SEC * Ke / e2e_s, "unit": UNIT,
               "h2d_bytes_per_step": w.S * w.push_mel * 128 * 4,
               "d2h_bytes_per_step": w.S * w.n * (w.cfg.d_model + w.cfg.joint_dim) * 4,
               "mode": ("cac_stream_push_host_async: step k+1 queued before the host waits for and reads "
                        "step k's frames (two page-locked output buffers); host wall time"),
               "one_call_at_a_time": {"value": world * w.S * w.n * FRAME_SEC * Ke / e2e_sync_s, "unit": UNIT,
                                      "what": "cac_stream_push_host, synchronous, the same number of steps"},
               "finite": bool(np.isfinite(seen))}
    w.pool.check()

    decode = None
    if Kd:
        try:
            decode = measure_decode(w, Kd, dev, clk)
        except Exception as exc:  # the decoder leg is reported beside the encoder, never instead of it
            decode = {"error": f"{type(exc).__name__}: {exc}"[:300]}

    legs = {}
    for name, steps, fn in (("frontend", args.frontend_steps,
                             lambda: measure_frontend(w.S, args.frontend_steps, dev, load_peaks()[0])),
                            ("beam", args.beam_steps, lambda: measure_beam(w.S, args.beam_steps, dev)),
                            ("palette", args.palette_steps if w.cfg.dtype == "bf16" and not w.cfg.provisional else 0,
                             lambda: measure_palette(w, args.palette_steps, dev))):
        if steps > 0:
            try:
                legs[name] = fn()
            except Exception as exc:  # reported beside the encoder, never instead of it
                legs[name] = {"error": f"{type(exc).__name__}: {exc}"[:300]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(wl, w.blob, args.cpu_chunks)
        except Exception as exc:  # reported beside the GPU figures, never instead of them
            cpu = {"error": f"{type(exc).__name__}: {exc}"[:300], "kind": "oracle"}
    if rank == 0:
        line = {"metric": workload_metric(wl),
                "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": Wm,
                "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": dict(workload_config(wl, world), mean_Lc=mean_lc),
                "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
                "latency": latency, "gpu_launches": launches, "clocks": clk, "decode": decode}
        line.update(legs)
        print(json.dumps(line), flush=True)


def fp32_alu_peak(sm_mhz: float) -> float:
    """FP32 FMA peak, TFLOP/s: SMs x 128 FP32 lanes x 2 FLOP x SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def measure_decode(w, Kd: int, dev, clk):
    """The greedy RNN-T + EOU decoder (fp32, include/cac_decode.h), 2 frames
    per stream per step: (a) encoder step + decode step back to back, (b) the
    decode step alone, CUDA events on the launching stream; decisions and
    emissions per step from an untimed pass over the same frames.  The decoder
    reads seeded projected frames (synth.make_joint_frames, about 0.3
    emissions per frame with the synthetic decoder weights) resident on the
    device, not the random-weight encoder's projections, on which a blank
    always wins."""
    import torch
    from cache_aware_conformer_gb300 import native
    dc = EOU_DECODER
    Wd = synth.make_decoder_weights(dc, 0)
    dec = native.Decoder(dc, synth.pack_decoder_weights(dc, Wd), w.S)
    ids = list(range(w.S))
    T = w.n
    tok = torch.empty(w.S, T * dc.max_symbols, dtype=torch.int32, device=dev)
    fr = torch.empty_like(tok)
    cn = torch.empty(w.S, dtype=torch.int32, device=dev)
    nz = Kd + 3
    zs = torch.from_numpy(np.stack([synth.make_joint_frames(nz * T, s, dc.joint_dim) for s in ids])).to(dev)
    frames_of = lambda i: zs[:, (i % nz) * T:(i % nz + 1) * T]
    for i in range(3):
        w.step()
        dec.step_into(ids, frames_of(i), tok, fr, cn)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(Kd):
        w.step()
        dec.step_into(ids, frames_of(3 + i), tok, fr, cn)
    e1.record()
    torch.cuda.synchronize()
    both_ms = e0.elapsed_time(e1) / Kd
    dec.reset(ids)
    e0.record()
    for i in range(Kd):
        dec.step_into(ids, frames_of(i), tok, fr, cn)
    e1.record()
    torch.cuda.synchronize()
    dec_ms = e0.elapsed_time(e1) / Kd
    dec.reset(ids)
    em = dcs = 0
    for i in range(Kd):
        dec.step_into(ids, frames_of(i), tok, fr, cn)
        c = cn.cpu().numpy()
        f = fr.cpu().numpy()
        forced = sum(int(np.sum(np.bincount(f[b, :c[b]], minlength=T) == dc.max_symbols)) for b in range(w.S))
        em += int(c.sum())
        dcs += int(c.sum()) + w.S * T - forced
    dec.check()
    dec.close()
    em, dcs = em / Kd, dcs / Kd
    C, P, J = dc.classes, dc.pred_dim, dc.joint_dim
    flops = dcs * 2.0 * C * J + em * (2.0 * 4 * P * P + 2.0 * J * P)   # joint per decision, LSTM + projection per emission
    peak = fp32_alu_peak(clk.get("sm_max_mhz") or 2070.0)
    ach = flops / (dec_ms * 1e-3) / 1e12
    return {"what": "greedy RNN-T + EOU decode of the step's 2 frames per stream (fp32, one cooperative launch)",
            "dtype": "f32", "ms_per_step": dec_ms, "decisions_per_step": dcs, "emissions_per_step": em,
            "encode_plus_decode": {"value": w.S * T * FRAME_SEC / (both_ms * 1e-3), "unit": UNIT,
                                   "ms_per_step": both_ms},
            "roofline": {"bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                         "traffic": None,
                         "peak_source": "derived: SMs x 128 FP32 lanes x 2 FLOP x max SM clock"}}


def measure_palette(w, Kp: int, dev):
    """The encoder with its weight matrices as 6-bit palettes
    (cac_model_create_palette; tables by cache_aware_conformer_gb300.palette)
    against the dense encoder on the same decoded weights: the workload's
    streams, one 160 ms push per step, graphs on, device-timed with CUDA
    events; weight bytes per step read by the projections (dense bf16: 2 B
    a weight, palette: 0.75 B)."""
    import torch
    from cache_aware_conformer_gb300 import native, palette
    cfg = w.cfg
    Wd, tables = palette.palettize_model(cfg, synth.make_weights(cfg, 0))
    blob = synth.pack_weights(cfg, Wd)
    mel = torch.from_numpy(np.stack([synth.make_mel(w.push_mel, s) for s in range(w.S)])).to(dev)
    F = w.push_mel // 8
    enc = torch.empty(w.S, F, cfg.d_model, device=dev)
    jt = torch.empty(w.S, F, cfg.joint_dim, device=dev)
    n_w = sum(np.asarray(Wd[n]).size for n in palette.matrix_names(cfg.n_layers) if not n.endswith("att.wpos"))
    out = {"what": "encoder step with 6-bit palette weights vs dense on the same decoded weights "
                   f"({w.S} streams, one {w.push_mel * 10} ms push per step, graphs)",
           "matrix_weights": int(n_w),
           "weight_bytes_per_step": {"dense_bf16": 2 * n_w, "palette": int(0.75 * n_w)}}
    for name, tab in (("palette", tables), ("dense", None)):
        model = native.Model(cfg, blob, tables=tab)
        pool = native.Pool(model, w.S, max(2, F))
        pool.set_graphs(True)
        ids = [pool.create_stream() for _ in range(w.S)]
        for _ in range(3):
            pool.push_into(ids, mel, enc, jt)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(Kp):
            pool.push_into(ids, mel, enc, jt)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / Kp
        pool.check()
        out[name] = {"ms_per_step": ms, "value": w.S * F * FRAME_SEC / (ms * 1e-3), "unit": UNIT}
        pool.close()
        model.close()
    return out


def measure_frontend(S: int, Kf: int, dev, peak_gbs: float):
    """The streaming log-mel front end (include/cac_frontend.h): Kf pushes of
    160 ms (2560 samples) for S streams of seeded speech-like audio resident on
    the device, CUDA events on the launching stream.  HBM bytes per push and
    stream: the new audio read, the frames written, the 512-sample tail read
    and rewritten."""
    import torch
    from cache_aware_conformer_gb300 import native
    fe = native.Frontend(S)
    ids, ns = list(range(S)), 2560
    n_push = Kf + 4
    audio = torch.from_numpy(np.stack([synth.make_audio(n_push * ns, s) for s in ids])).to(dev)
    mel = torch.empty((S, 20, 128), dtype=torch.float32, device=dev)
    frames = 0
    for i in range(3):
        frames = sum(fe.push_into(ids, audio[:, i * ns:(i + 1) * ns], mel))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(3, 3 + Kf):
        frames = sum(fe.push_into(ids, audio[:, i * ns:(i + 1) * ns], mel))
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / Kf
    fe.close()
    nbytes = S * (ns * 4 + (frames / S) * 128 * 4 + 2 * 512 * 4)
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"what": "streaming log-mel front end: 160 ms of 16 kHz audio per stream per push (fp32, one launch)",
            "dtype": "f32", "ms_per_push": ms, "value": S * 0.16 / (ms * 1e-3), "unit": UNIT,
            "frames_per_push": frames,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak_gbs, "unit": "GB/s", "frac": ach / peak_gbs,
                         "traffic": None}}


def measure_beam(S: int, Kb: int, dev, beam: int = 8):
    """The batched MALSD beam search (include/cac_beam.h, beam 8) over 2 seeded
    projected frames per stream per step, CUDA events around Kb steps."""
    import torch
    from cache_aware_conformer_gb300 import native
    dc = EOU_DECODER
    Wd = synth.make_decoder_weights(dc, 0)
    bd = native.BeamDecoder(dc, synth.pack_decoder_weights(dc, Wd), beam, S, max_tokens=256)
    ids, T = list(range(S)), 2
    zs = torch.from_numpy(np.stack([synth.make_joint_frames((Kb + 3) * T, s, dc.joint_dim) for s in ids])).to(dev)
    for i in range(3):
        bd.step(ids, zs[:, i * T:(i + 1) * T])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(3, 3 + Kb):
        bd.step(ids, zs[:, i * T:(i + 1) * T])
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / Kb
    bd.check()
    bd.close()
    return {"what": f"MALSD beam search, beam {beam}, 2 projected frames per stream per step (fp32, cooperative "
                    f"launch)", "dtype": "f32", "ms_per_step": ms, "value": S * T * FRAME_SEC / (ms * 1e-3),
            "unit": UNIT,
            "roofline": None,
            "roofline_note": "not reported: the joint evaluations and label expansions per step depend on the "
                             "search and are not counted on the device"}


def cpu_baseline(wl, blob, chunks: int):
    """The oracle as it stands on a bounded sample of the workload: streams
    0 .. C-1 (one per host core), `chunks` pushes each after an untimed first
    one; offline workloads: windows 0 .. C-1, `chunks` encodes each."""
    cfg = wl.model
    units = wl.offline_batch or wl.streams
    n = oracle_workers(blob, units)
    farm = OracleFarm(cfg, blob, [workload_mel(wl, sid) for sid in range(n)], 0 if wl.offline_batch else wl.push_mel)
    try:
        if not wl.offline_batch:
            farm.step(1)                  # first push (stream start) untimed
        secs = farm.step(chunks)
        one = farm.step_one(chunks)       # the same work on one core, the others idle
    finally:
        farm.close()
    what = f"{cfg.n_layers}-layer d_model-{cfg.d_model} model, fp64 numpy"
    if wl.offline_batch:
        sec = wl.offline_mel * 0.01
        sample = f"windows 0..{n - 1} of {units} x {chunks} offline encodes of {wl.offline_mel} mel frames"
        sample1 = f"1 window x {chunks} offline encodes"
    else:
        sec = wl.push_mel * 0.01
        sample = f"streams 0..{n - 1} of {units} x {chunks} pushes of {10 * wl.push_mel} ms"
        sample1 = f"1 stream x {chunks} pushes of {10 * wl.push_mel} ms"
    return {"value": n * chunks * sec / secs, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{sample} (one per core, {what}); {secs:.1f} s wall",
            "single_core": {"value": chunks * sec / one, "unit": UNIT, "cores": 1,
                            "sample": f"{sample1}; {one:.1f} s wall"}}


def workload_metric(wl) -> str:
    if wl.offline_batch:
        return f"offline encode audio-sec/sec ({wl.name})"
    return METRIC if wl.name == "eou120m_256streams_60s" else f"streamed audio-sec/sec ({wl.name})"


def workload_config(wl, world: int) -> dict:
    """The static description of a streaming workload, shared by both arms."""
    cfg = wl.model
    return {"workload": wl.name, "streams_per_gpu": wl.streams, "chunk_ms": 10 * wl.push_mel,
            "layers": cfg.n_layers, "d_model": cfg.d_model, "heads": cfg.n_heads, "ff": cfg.ff_dim,
            "att_left": cfg.att_left, "att_chunk": cfg.att_chunk, "reset_prob": wl.reset_prob,
            "start_offsets": f"even, 0..{max(wl.max_start_offset - 1, 0)}", "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2: each step reads all K/V rings and all weights",
            "knobs": {k: os.environ[k] for k in ("CAC_PDL", "CAC_GROUPS", "CAC_SPLIT_TARGET", "CAC_CHAIN",
                                                 "CAC_CHAIN_MAX_SPLITS",
                                                 "CAC_SPLIT_MIN_SLICES") if os.environ.get(k)}}


def run_reference(args, wl):
    """Reference arm: the fp64 oracle itself on the host cores, same metric and
    config.  Each step = one push of a sample of the workload's streams (one per
    core); offline workloads: one encode of a sample of its windows."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    cfg = wl.model
    W = synth.make_weights_parallel(cfg, seed=0, workers=cpu_cores())
    blob = synth.pack_weights(cfg, W)
    del W
    units = wl.offline_batch or wl.streams
    n = oracle_workers(blob, units)
    if wl.offline_batch:  # a window is seconds of fp64 work: fewer steps
        K, Wm = min(args.steps, args.ref_steps, 2), 1
    else:
        K, Wm = min(args.steps, args.ref_steps), min(args.warmup, 3)
    farm = OracleFarm(cfg, blob, [workload_mel(wl, sid) for sid in range(n)], 0 if wl.offline_batch else wl.push_mel)
    try:
        farm.step(Wm if wl.offline_batch else 1 + Wm)
        secs = farm.step(K)
    finally:
        farm.close()
    sec = (wl.offline_mel if wl.offline_batch else wl.push_mel) * 0.01
    value = n * K * sec / secs
    unit_name = "windows" if wl.offline_batch else "streams"
    step_name = "offline encodes" if wl.offline_batch else f"pushes of {10 * wl.push_mel} ms"
    config = (dict(workload=wl.name, windows=wl.offline_batch, mel_frames=wl.offline_mel, layers=cfg.n_layers,
                   d_model=cfg.d_model, parallelism=f"replicas x{world}") if wl.offline_batch
              else workload_config(wl, world))
    line = {"impl": "reference", "metric": workload_metric(wl), "value": value, "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": Wm, "ms_per_step": 1e3 * secs / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(config, **{f"{unit_name}_sampled": n}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "kind": "oracle",
                             "sample": f"{unit_name} 0..{n - 1} of {units}, {K} {step_name} each"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="eou120m_256streams_60s", choices=sorted(WORKLOADS))
    ap.add_argument("--profile-steps", type=int, default=40)
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--cpu-chunks", type=int, default=100)
    ap.add_argument("--ref-steps", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=40)
    ap.add_argument("--frontend-steps", type=int, default=20, help="log-mel front-end pushes to time (0: skip)")
    ap.add_argument("--beam-steps", type=int, default=10, help="beam-search steps to time (0: skip)")
    ap.add_argument("--palette-steps", type=int, default=20,
                    help="steps of the palette-weight encoder and its dense twin to time (0: skip)")
    ap.add_argument("--streams", type=int, default=0,
                    help="override the workload's stream count (small cases for profiler captures; 0: the workload's)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = WORKLOADS[args.workload]
    if args.streams > 0:
        wl = replace(wl, streams=args.streams)
    if args.impl == "reference":
        run_reference(args, wl)
    elif wl.offline_batch:
        run_offline(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
