"""Benchmark of the fused normalisation path on GB300.

One step = one pass of the fused step over one batch: 256 uint8 images of
224x224x3 (NHWC) -> FP16 NHWC, ImageNet mean/std, per-image flip (p=0.5) and
RandomErasing (p=0.5, scale [0.02, 0.33], ratio [0.3, 3.3]) records sampled
on the host from a seed.  Prints ONE JSON line.

  value      images/s of the CUDA kernel with inputs resident in HBM; the
             timed steps are replays of a CUDA graph of launches that rotate
             over enough distinct (src, dst, records) sets to exceed L2 four
             times, so no step reads what the previous one left in L2.  The
             batches share no buffer, so each launch overlaps the previous
             one's drain (TR_LAUNCH_OVERLAP_PREVIOUS); isolated_launches
             times the same launches each waiting for the one before.
  roofline   algorithmic bytes per launch (N*H*W*C*(1 + out_bytes) minus the
             erased source reads) / average launch time, against the measured
             HBM copy bandwidth (MEASURED_PEAKS.json).
  e2e        images/s through the transfer station with pinned host buffers:
             every step copies its uint8 batch and records host->device, runs
             the kernel and copies the FP16 result device->host.
  cpu_baseline  the CPU oracle on a bounded sample of the same workload, on
             the host's cores.

Multi-GPU (torchrun, one process per GPU): every rank runs its own replica
of the workload (images are independent; no data-path collective); the
timing is the max over ranks and value sums the images of all ranks.

--impl reference times the CPU oracle as the reference arm instead.
"""
import argparse
import concurrent.futures as cf
import ctypes
import hashlib
import json
import re
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "images/sec and achieved HBM GB/s (fraction of peak) at 256×224×224×3"
FALLBACK_HBM_GBS = 6800.0
SPACER_CYCLES = 200_000   # about 0.1 ms at GB300's 2.07 GHz SM clock


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4])
    ap.add_argument("--layout", default=None, help="override the config's output layout (nhwc/nchw/nhwc4)")
    ap.add_argument("--batch", type=int, default=None, help="override the config's batch size N")
    ap.add_argument("--crop", type=int, default=0,
                    help="read each image as a window of an SxS source (random origins when the workload "
                         "flips/erases, else the centre): tr_fused_norm_crop")
    ap.add_argument("--size", default=None,
                    help="override the config's image size as HxW (e.g. 299x299: rows of 897 bytes, the "
                         "odd-row form of the tiled kernel)")
    ap.add_argument("--variant", type=int, default=0, help="0 auto, 1 tiled, 2 generic")
    ap.add_argument("--static", action="store_true", help="static band schedule (no workspace)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="each launch waits for the previous one to complete before touching memory (no "
                         "TR_LAUNCH_OVERLAP_PREVIOUS); by default consecutive batches, which share no buffer, "
                         "overlap one launch's drain with the next one's first copies")
    ap.add_argument("--fused-sampling", action="store_true",
                    help="records drawn inside the fused kernel each step (tr_fused_norm_sampled)")
    ap.add_argument("--device-sampling", action="store_true",
                    help="each step samples its records on the GPU (tr_sample_aug_params_device) before the kernel")
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-pipeline", action="store_true",
                    help="skip the 64-batch pinned-host stream (reported under 'pipeline')")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-batched", action="store_true",
                    help="skip the launches of 1, 4 and 8 headline batches each (tr_fused_norm_batches), "
                         "reported under 'batched_launches', the headline batches with their records sampled in "
                         "the same call ('fused_sampling') and the 299x299 odd-row batches ('odd_rows')")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other batch workloads (16x32x32x3, 200x28x28x1, 256x224x224x3 -> f32 NHWC/NCHW) "
                         "reported under 'per_config'")
    ap.add_argument("--no-clocks", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------ helpers -----

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        import torch
        if not torch.cuda.is_available():
            backend = "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, local, world, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value, device):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate_images_per_s(world, n_per_rank, steps, max_ms):
    """Whole-job images/s: every rank's images over the slowest rank's time."""
    return world * n_per_rank * steps / (max_ms / 1000.0)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "hbm_gbs" in d:
            return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """sha256[:16] of the kernel's source (fused_norm.cu + internal.h) with
    comments and whitespace removed: what the compiler sees, so a profile
    stays attached to the code it measured across comment edits."""
    h = hashlib.sha256()
    for fn in ("fused_norm.cu", "internal.h"):
        with open(os.path.join(ROOT, "image_preprocessing_gb300", "csrc", fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, enabled=True):
        self.index = index
        self.proc = None
        self.enabled = enabled
        self.lines = []

    def start(self):
        if not self.enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------- workloads -----

def workload(args):
    from image_preprocessing_gb300 import synth
    cfg = dict(synth.CONFIGS[args.config])
    layout = args.layout or cfg["layouts"][0]
    cfg["layout"] = layout
    name = cfg["name"]
    if args.layout:
        name += "_" + layout
    if args.batch:
        name = name.replace("n%d_" % cfg["N"], "n%d_" % args.batch, 1)
        cfg["N"] = args.batch
    size = getattr(args, "size", None)
    if size:
        H, W = (int(v) for v in size.lower().split("x"))
        if H < 1 or W < 1:
            raise SystemExit("--size wants HxW with H, W >= 1")
        name = name.replace("_%dx%dx%d_" % (cfg["H"], cfg["W"], cfg["C"]), "_%dx%dx%d_" % (H, W, cfg["C"]), 1)
        cfg["H"], cfg["W"] = H, W
    cfg["crop"] = getattr(args, "crop", 0)
    if cfg["crop"]:
        name += "_crop_from_%dx%d" % (cfg["crop"], cfg["crop"])
    cfg["workload"] = name
    return cfg


def algorithmic_bytes(cfg, recs):
    """N*H*W*C*(1 + out_bytes) minus the erased source reads (h*w*C per erased
    image, rectangles clipped to the image)."""
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    ob = 2 if cfg["out_dtype"] == "f16" else 4
    out_ch = 4 if cfg["layout"] == "nhwc4" else C
    total = N * H * W * (C + out_ch * ob)
    if recs is not None:
        h = np.clip(recs[:, 3], 0, None).astype(np.int64)
        w = np.clip(recs[:, 4], 0, None).astype(np.int64)
        total -= int(np.sum(np.where((h > 0) & (w > 0), h * w, 0))) * C
    return total


def host_batch(cfg, seed):
    from image_preprocessing_gb300 import synth
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    if cfg["pixels"] == "uniform":
        return synth.pixels_uniform(seed, N, H, W, C)
    if cfg["pixels"] == "sparse":
        return synth.pixels_sparse(seed, N, H, W, C)
    return synth.pixels_gaussian(seed, N, H, W, C)


def sample_records(cfg, seed, offset, impl_sampler):
    if not (cfg["flip"] or cfg["erase"]):
        return None, offset
    return impl_sampler(seed, offset, cfg["N"], cfg["H"], cfg["W"], flip=cfg["flip"], erase=cfg["erase"],
                        erase_p=cfg["erase_p"])


# -------------------------------------------------------------- ours ------

def run_ours(args, rank, local, world, pg):
    import torch
    import image_preprocessing_gb300 as trfn

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workload(args)
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    dt = trfn.OUT_F16 if cfg["out_dtype"] == "f16" else trfn.OUT_F32
    layout = {"nhwc": trfn.LAYOUT_NHWC, "nchw": trfn.LAYOUT_NCHW, "nhwc4": trfn.LAYOUT_NHWC4}[cfg["layout"]]
    tdt = torch.float16 if dt == trfn.OUT_F16 else torch.float32
    mean = np.array(cfg["mean"], np.float32)
    std = np.array(cfg["std"], np.float32)
    out_shape = trfn.out_shape(N, H, W, C, layout)

    # distinct buffer sets whose total footprint is at least 4x L2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    S = cfg["crop"]
    src_img = (S * S * C) if S else (H * W * C)
    set_bytes = N * src_img + int(np.prod(out_shape)) * (2 if dt == trfn.OUT_F16 else 4)
    nsets = max(2, int(np.ceil(4 * l2 / set_bytes)))
    srcs, dsts, augs, recs_all, crops = [], [], [], [], []
    offset = rank * 10 ** 9
    for j in range(nsets):
        hb = host_batch(dict(cfg, H=S, W=S) if S else cfg, 1000 + args.config + 100 * j + 7919 * rank)
        srcs.append(torch.from_numpy(hb).to(dev))
        if S:
            g = np.random.default_rng(3000 + j)
            if cfg["flip"] or cfg["erase"]:
                c = np.stack([g.integers(0, S - H + 1, N), g.integers(0, S - W + 1, N)], axis=1)
            else:
                c = np.tile([(S - H) // 2, (S - W) // 2], (N, 1))
            crops.append(torch.from_numpy(c.astype(np.int32)).to(dev))
        dsts.append(torch.empty(out_shape, dtype=tdt, device=dev))
        recs, offset = sample_records(cfg, 2000 + args.config, offset, trfn.tr_sample_aug_params)
        recs_all.append(recs)
        augs.append(torch.from_numpy(recs).to(dev) if recs is not None else None)
    if (args.device_sampling or args.fused_sampling) and (cfg["flip"] or cfg["erase"]):
        # the records each step samples on the GPU (same seeds as launch(j) below)
        import oracle
        recs_all = [oracle.sample_aug_params_blocked(4000 + j, 0, N, H, W, flip=cfg["flip"], erase=cfg["erase"],
                                                     erase_p=cfg["erase_p"])[0] for j in range(nsets)]
    alg_bytes = [algorithmic_bytes(cfg, r) for r in recs_all]

    stream = torch.cuda.Stream(device=dev)
    # scheduling workspaces that differ from one launch to the next, so that a
    # launch may overlap the one before it (TR_LAUNCH_OVERLAP_PREVIOUS: the
    # batches share no buffer).  Full graphs (even length) alternate 0/1;
    # shorter runs (eager remainders, the tail graph, any length) alternate
    # 2/1, so they start on another workspace than a full graph ends on (1)
    # and end on another than one starts on (0).  --static measures the
    # workspace-free schedule.
    wss = [None] * 3 if args.static else [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device=dev)
                                          for _ in range(3)]

    dev_sampling = args.device_sampling and (cfg["flip"] or cfg["erase"])
    fused_sampling = args.fused_sampling and (cfg["flip"] or cfg["erase"]) and not S
    # records sampled by a separate call launch without the option (the
    # kernel reads records the call before it wrote); the one-call form
    # (tr_fused_norm_sampled) overlaps its sampler with the previous launch
    overlap_ok = not dev_sampling
    overlap = {"on": overlap_ok and not args.no_overlap}

    def launch(j, k=0, part=False):
        ws = wss[(2, 1)[k % 2]] if part else wss[k % 2]
        if fused_sampling:
            trfn.tr_fused_norm_sampled(srcs[j], dsts[j], mean, std, 4000 + j, 0, augs[j], flip=cfg["flip"],
                                       erase=cfg["erase"], erase_p=cfg["erase_p"], out_dtype=dt, layout=layout,
                                       stream=stream, variant=args.variant, workspace=ws,
                                       overlap_previous=overlap["on"])
            return
        if dev_sampling:
            trfn.tr_sample_aug_params_device(4000 + j, 0, N, H, W, augs[j], flip=cfg["flip"], erase=cfg["erase"],
                                             erase_p=cfg["erase_p"], stream=stream)
        if S:
            trfn.tr_fused_norm_crop(srcs[j], S, S, S * C, S * S * C, dsts[j], N, H, W, C, mean, std, crop=crops[j],
                                    aug=augs[j], out_dtype=dt, layout=layout, stream=stream, variant=args.variant,
                                    workspace=ws, overlap_previous=overlap["on"])
        else:
            trfn.tr_fused_norm(srcs[j], dsts[j], mean, std, augs[j], out_dtype=dt, layout=layout, stream=stream,
                               variant=args.variant, workspace=ws, overlap_previous=overlap["on"])

    # warm the library's per-kernel caches (ending on an odd launch index, so
    # the next launch takes the other workspace), then capture graphs of
    # launches; G is even, so workspaces alternate across replays too
    with torch.cuda.stream(stream):
        for k in range(nsets + nsets % 2):
            launch(k % nsets, k)
    torch.cuda.synchronize()
    G = nsets * max(1, 60 // nsets)
    G += G % 2

    def capture(count, part=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(count):
                launch(k % nsets, k, part)
        return g

    launches_before = trfn.tr_launch_count()
    g_full = capture(G)
    K, Wm = args.steps, args.warmup
    g_tail = capture(K % G, part=True) if K % G else None
    captured = trfn.tr_launch_count() - launches_before

    def run_steps(steps, exact_tail=None, marks=None):
        # full graph replays, then the remainder as one tail graph (timed
        # region) or as eager launches (warm-up); all on `stream`, where the
        # timing events are recorded (a replay goes to the current stream).
        # marks: (replay index, event) pairs recorded before that replay
        marks = dict(marks or [])
        with torch.cuda.stream(stream):
            for i in range(steps // G):
                if i in marks:
                    marks[i].record(stream)
                g_full.replay()
            rem = steps % G
            if rem and exact_tail is not None:
                exact_tail.replay()
            elif rem:
                for k in range(rem):
                    launch(k % nsets, k, part=True)

    def spacer():
        # the GPU spins (bounded, about a millisecond) while the host queues
        # the timed region behind it, so the region does not include the
        # host's time to submit its first graph
        with torch.cuda.stream(stream):
            torch.cuda._sleep(SPACER_CYCLES)

    run_steps(Wm)
    # every graph object the timed region replays runs (three times) before
    # it: the first replay of a graph uploads it, a one-time cost that would
    # otherwise fall into the region (about 64 us per 20 launches)
    with torch.cuda.stream(stream):
        for _ in range(3):
            if K >= G:
                g_full.replay()
            if g_tail is not None:
                g_tail.replay()
    warm_graph_replays = 3 * (int(K >= G) + int(g_tail is not None))
    torch.cuda.synchronize()
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    clocks.start()
    # keep the GPU busy while the sampler starts
    run_steps(min(Wm, 4 * G) if Wm else 0)
    time.sleep(0.15)
    barrier(pg)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    # five trials: events between graph replays inside the timed region when
    # it holds at least five replays, else four repeats of the timed region
    # after it (same graphs, same launches)
    replays = K // G
    trial_at = [replays * t // 5 for t in range(1, 5)] if replays >= 5 else []
    trial_ev = [torch.cuda.Event(enable_timing=True) for _ in trial_at]
    # the host waited above: run the timed region's launches once, untimed,
    # right before it (a GPU left idle for a while measured its next region
    # about 0.6 % slower than the same region repeated)
    spacer()
    run_steps(min(K, G), g_tail if K < G else None)
    spacer()
    ev0.record(stream)
    run_steps(K, g_tail, marks=list(zip(trial_at, trial_ev)))
    ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    barrier(pg)
    ms = ev0.elapsed_time(ev1)
    trials = None
    if trial_ev:
        bounds = [ev0] + trial_ev + [ev1]
        steps_in = [(b - a) * G for a, b in zip([0] + trial_at, trial_at + [replays])]
        steps_in[-1] += K % G
        per = [bounds[t].elapsed_time(bounds[t + 1]) / steps_in[t] for t in range(len(steps_in))]
        trials = {"count": len(per), "ms_per_step": per, "median_ms_per_step": float(np.median(per)),
                  "how": "five parts of the timed region"}
    else:
        per = [ms / K]
        for _ in range(4):
            e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            spacer()
            e_a.record(stream)
            run_steps(K, g_tail)
            e_b.record(stream)
            e_b.synchronize()
            per.append(e_a.elapsed_time(e_b) / K)
        trials = {"count": len(per), "ms_per_step": per, "median_ms_per_step": float(np.median(per)),
                  "how": "the timed region, then four repeats of it (same graphs and launches)"}
    trials["spread"] = float(max(per) / min(per) - 1.0)
    clk = clocks.stop()
    ms_max = max_over_ranks(pg, ms, dev)
    per_launch_s = (ms / 1000.0) / K
    # average algorithmic bytes per launch over the rotation actually timed
    seq = [k % nsets for k in range(K)]
    avg_bytes = float(np.mean([alg_bytes[j] for j in seq]))
    achieved_gbs = avg_bytes / per_launch_s / 1e9
    peak, peak_kind = measured_peaks()

    # sampled parity of the last outputs against the oracle (bench's own launch configuration)
    parity = parity_sample(cfg, srcs, dsts, recs_all, mean, std, dt, layout, nsets, crops)

    # the same launches, each waiting for the previous one to complete before
    # it touches memory (no overlap): a graph replayed for about a fifth of the
    # timed steps, reported beside the main figure
    isolated = None
    if overlap["on"]:
        overlap["on"] = False
        g_iso = capture(G)
        reps = max(1, min(K // G, 200) // 5)
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g_iso.replay()
            e_a.record(stream)
            for _ in range(reps):
                g_iso.replay()
            e_b.record(stream)
        e_b.synchronize()
        iso_s = e_a.elapsed_time(e_b) / 1000.0 / (reps * G)
        iso_gbs = float(np.mean([alg_bytes[k % nsets] for k in range(G)])) / iso_s / 1e9
        isolated = {"ms_per_step": iso_s * 1000.0, "images_per_s": N / iso_s, "achieved": iso_gbs,
                    "frac": iso_gbs / peak, "steps": reps * G,
                    "launch": "each launch waits for the previous one to complete (no TR_LAUNCH_OVERLAP_PREVIOUS)"}
        overlap["on"] = True
        del g_iso

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, cfg, dev, mean, std, dt, layout, tdt, out_shape, rank, pg)
    headline = args.config == 3 and not S and not args.batch and not args.layout and not args.size
    pipeline = None
    if not args.no_pipeline and headline:
        pipeline = run_pipeline(dev, rank, pg)
    per_config = None
    if not args.no_per_config and headline and world == 1:
        per_config = run_per_config(dev, measured_peaks()[0], args.cpu_seconds / 4, not args.no_cpu)
    batched = sampled = odd_rows = None
    if not args.no_batched and headline and world == 1 and not (dev_sampling or fused_sampling):
        batched = run_batched(dev, measured_peaks()[0])
        sampled = run_sampled(dev, measured_peaks()[0])
        odd_rows = run_odd_rows(dev, measured_peaks()[0])

    value = aggregate_images_per_s(world, N, K, ms_max)
    res = {
        "metric": METRIC,
        "value": value,
        "unit": "images/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": ms_max / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": cfg["workload"], "N": N, "H": H, "W": W, "C": C, "in": "u8 NHWC",
            "out": cfg["out_dtype"] + " " + cfg["layout"].upper(),
            "flip_p": 0.5 if cfg["flip"] else 0.0, "erase_p": cfg["erase_p"],
            "l2": l2_note(K, nsets, set_bytes, l2),
            "launch": "CUDA graph of %d launches replayed (%s); variant %d; %s" % (
                G, "timed: %d replays + a graph of the %d remaining launches; every timed graph replayed "
                   "three times in warm-up (%d replays beyond the %d warm-up steps), and %d launches of the "
                   "region run untimed just before it" % (K // G, K % G, warm_graph_replays, Wm, min(K, G)),
                args.variant,
                "consecutive launches overlap (tr_fused_norm_ex, TR_LAUNCH_OVERLAP_PREVIOUS: independent batches, "
                "workspaces differing from one launch to the next)" if overlap["on"]
                else "each launch waits for the previous one to complete"),
            "schedule": "static (tr_fused_norm)" if args.static else "dynamic bands (tr_fused_norm_ws)",
            "source": ("%dx%d windows of %dx%d images (tr_fused_norm_crop)" % (H, W, S, S)) if S else "compact",
            "records": ("sampled inside the fused kernel every step (tr_fused_norm_sampled)" if fused_sampling
                        else "sampled on the GPU every step (tr_sample_aug_params_device)" if dev_sampling
                        else "sampled on the host (tr_sample_aug_params), uploaded once"),
            "parallelism": "replicas" if world > 1 else "single",
        },
        "hbm_gbs": achieved_gbs,
        "roofline": {
            "bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
            "frac": achieved_gbs / peak, "peak_kind": peak_kind,
            "frac_of_nominal_8000": achieved_gbs / 8000.0,
            "algorithmic_bytes_per_launch": avg_bytes,
            "traffic": profiled_traffic(cfg["workload"]),
        },
        "gpu_launches": K * (2 if (dev_sampling or fused_sampling) else 1),   # sampler + fused kernel
        "captured_launches": int(captured),
        "parity_sample": parity,
    }
    if clk is not None:
        res["clocks"] = clk
    if trials is not None:
        res["trials"] = trials
    if isolated is not None:
        res["isolated_launches"] = isolated
    if e2e is not None:
        res["e2e"] = e2e
    if pipeline is not None:
        res["pipeline"] = pipeline
    if per_config is not None:
        res["per_config"] = per_config
    if batched is not None:
        res["batched_launches"] = batched
    if sampled is not None:
        res["fused_sampling"] = sampled
    if odd_rows is not None:
        res["odd_rows"] = odd_rows
    return res


def l2_note(K, nsets, set_bytes, l2):
    """How the timed region stands against L2: its K launches walk the
    rotating sets in order, so they touch min(K, nsets) of them.  Below 4x L2
    of distinct bytes the region's inputs are L2-resident (small workloads at
    small step counts; `per_config` times those over every set)."""
    touched = min(K, nsets) * set_bytes
    if touched >= 4 * l2:
        return "inputs larger than L2: %d rotating buffer sets, %.0f MB >= 4x L2 (%.0f MB)" % (
            nsets, nsets * set_bytes / 1e6, l2 / 1e6)
    return ("L2-resident: the timed region's %d launches touch %d of the %d rotating buffer sets, "
            "%.0f MB < 4x L2 (%.0f MB); per_config times the small workloads over every set" % (
                K, min(K, nsets), nsets, touched / 1e6, l2 / 1e6))


def parity_sample(cfg, srcs, dsts, recs_all, mean, std, dt, layout, nsets, crops=None):
    """A few images of the last written buffer set against the oracle."""
    import oracle
    import torch
    j = (nsets - 1)
    idx = [0, cfg["N"] // 2, cfg["N"] - 1]
    src = srcs[j][idx].cpu().numpy()
    recs = recs_all[j][idx] if recs_all[j] is not None else None
    got = dsts[j][idx].cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if dt == 1 else got.numpy()
    if crops:
        S, H, W, C = cfg["crop"], cfg["H"], cfg["W"], cfg["C"]
        ref = oracle.fused_norm_crop(src.reshape(-1), S * S * C, S * C, S, S, len(idx), H, W, C, mean, std,
                                     crops[j][idx].cpu().numpy(), recs, dt, layout)
    else:
        ref = oracle.fused_norm(src, mean, std, recs, out_dtype=dt, layout=layout)
    if dt == 1:
        def ordered(b):
            b = b.astype(np.int32)
            return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
        err = int(np.max(np.abs(ordered(got) - ordered(ref))))
        ok = err <= 1 and bool(np.all(got[ref == 0] == 0))
        return {"images": len(idx), "max_f16_ulp": err, "ok": ok}
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    ok = err <= 2e-6 and bool(np.all(got.view(np.uint32)[ref.view(np.uint32) == 0] == 0))
    return {"images": len(idx), "max_abs": err, "ok": ok}


def run_e2e(args, cfg, dev, mean, std, dt, layout, tdt, out_shape, rank, pg):
    """Through the public API with pinned host buffers: each step copies its
    uint8 batch and its records host->device, runs the kernel, and copies the
    result device->host (tr_ts_submit)."""
    import torch
    import image_preprocessing_gb300 as trfn
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    nh = 4
    h_src = [torch.from_numpy(host_batch(cfg, 5000 + b + 7919 * rank)).pin_memory() for b in range(nh)]
    offset = 0
    h_par = []
    for b in range(nh):
        recs, offset = sample_records(cfg, 2005, offset, trfn.tr_sample_aug_params)
        h_par.append(torch.from_numpy(recs).pin_memory() if recs is not None else None)
    slot_bytes = trfn.tr_ts_slot_bytes(N, H, W, C)
    slots = [torch.empty(slot_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty(out_shape, dtype=tdt, device=dev) for _ in range(2)]
    h_out = [torch.empty(out_shape, dtype=tdt).pin_memory() for _ in range(2)]
    s_copy, s_comp, s_d2h = (torch.cuda.Stream(device=dev) for _ in range(3))
    ts = trfn.TransferStation(dev.index, slots, s_copy, s_comp, s_d2h)

    def steps(k0, count):
        for k in range(k0, k0 + count):
            ts.submit(h_src[k % nh], d_out[k % 2], mean, std, h_params=h_par[k % nh], h_dst=h_out[k % 2],
                      out_dtype=dt, layout=layout)

    steps(0, 4)
    assert ts.sync(60000)
    K = args.e2e_steps
    # three runs of K steps; the median is reported (host memory and its link
    # are shared with the machine's other jobs, so a single run can catch
    # their traffic)
    runs = []
    for t in range(3):
        barrier(pg)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        steps(4 + t * K, K)
        ok = ts.sync(120000)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        assert ok, "transfer station did not finish"
        runs.append(max_over_ranks(pg, t1 - t0, dev))
    ts.close()
    sec = float(np.median(runs))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    ob = 2 if dt == 1 else 4
    h2d = N * H * W * C + (N * 20 if h_par[0] is not None else 0)
    d2h = int(np.prod(out_shape)) * ob
    # the bound the station runs against: the same steps' copies alone (the
    # batch in on the copy stream, the result out on the d2h stream, both
    # directions at once), no kernel
    img = N * H * W * C
    reps = 16
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    main = torch.cuda.current_stream(dev)
    e_a.record(main)
    s_copy.wait_stream(main)
    s_d2h.wait_stream(main)
    for k in range(reps):
        with torch.cuda.stream(s_copy):
            slots[k % 2][:img].copy_(h_src[k % nh].view(-1), non_blocking=True)
        with torch.cuda.stream(s_d2h):
            h_out[k % 2].copy_(d_out[k % 2], non_blocking=True)
    main.wait_stream(s_copy)
    main.wait_stream(s_d2h)
    e_b.record(main)
    e_b.synchronize()
    copies_s = e_a.elapsed_time(e_b) / 1e3 / reps
    return {"value": world * N * K / sec, "unit": "images/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K,
            "runs_images_per_s": [world * N * K / r for r in runs],
            "how": "median of three runs of %d steps" % K,
            "path": "tr_ts_submit: pinned host u8 + records -> device slot A/B (copy stream) -> kernel "
                    "(compute stream) -> pinned host output (d2h stream)",
            "link_gbs": (h2d + d2h) * K / sec / 1e9,
            "copies_alone": {"us_per_step": copies_s * 1e6, "link_gbs": (img + d2h) / copies_s / 1e9,
                             "frac": copies_s / (sec / K),
                             "how": "the step's uint8 batch in and result out, both directions at once, %d steps, "
                                    "no kernel" % reps}}


def run_pipeline(dev, rank, pg):
    """The 64-batch stream: 64 distinct pinned host batches of 256x224x224x3
    uint8 (and their records, flip 0.5, erase 0.5, Philox offsets running on
    across batches) go through the transfer station to fp16 NHWC on the
    device; the copy of batch k+1 (copy stream) overlaps the kernel on batch
    k (compute stream).  Outputs stay on the device (two alternating output
    buffers).  Reports images/s from the first copy to the last kernel (CUDA
    events; the median of three passes), a lone 38.5 MB pinned copy, the
    kernel alone, and the overlap efficiency (T_copy + T_kernel) /
    T_pipelined over the 64 batches."""
    import torch
    import image_preprocessing_gb300 as trfn
    from image_preprocessing_gb300 import synth
    cfg = synth.CONFIGS[5]
    B, N, H, W, C = cfg["batches"], cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    mean = np.array(cfg["mean"], np.float32)
    std = np.array(cfg["std"], np.float32)
    # clipped-Gaussian pixels (seed 5000 + b), drawn straight into the pinned
    # buffers by host threads (numpy drops the GIL while it draws)
    h_src = [torch.empty((N, H, W, C), dtype=torch.uint8).pin_memory() for _ in range(B)]
    t_draw = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(lambda b: synth.pixels_gaussian_into(5000 + b + 7919 * rank, h_src[b].numpy()), range(B)))
    t_draw = time.perf_counter() - t_draw
    h_par, offset = [], 0
    for b in range(B):
        recs, offset = trfn.tr_sample_aug_params(2005, offset, N, H, W, flip=True, erase=True,
                                                 erase_p=cfg["erase_p"])
        h_par.append(torch.from_numpy(recs).pin_memory())
    slot_bytes = trfn.tr_ts_slot_bytes(N, H, W, C)
    slots = [torch.empty(slot_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty((N, H, W, C), dtype=torch.float16, device=dev) for _ in range(2)]
    s_copy, s_comp = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def events():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    # every host batch is copied once before anything is timed: the first
    # device access to freshly pinned pages costs several times a later one,
    # and a running pipeline reuses its pinned buffers
    img_bytes = N * H * W * C
    with torch.cuda.stream(s_copy):
        for b in range(B):
            slots[b & 1][:img_bytes].copy_(h_src[b].view(-1), non_blocking=True)
    torch.cuda.synchronize()
    # a lone pinned host-to-device copy of one batch (8 batches, averaged;
    # the median of three such runs)
    lone = []
    for _ in range(3):
        e0, e1 = events()
        with torch.cuda.stream(s_copy):
            e0.record(s_copy)
            for b in range(8):
                slots[b & 1][:img_bytes].copy_(h_src[b].view(-1), non_blocking=True)
            e1.record(s_copy)
        e1.synchronize()
        lone.append(e0.elapsed_time(e1) / 8 / 1e3)
    t_copy = float(np.median(lone))
    # the kernel alone on a slot, dynamically scheduled as in the station (16
    # launches, averaged)
    d_par = h_par[0].to(dev)
    src0 = slots[0][:img_bytes].view(N, H, W, C)
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device=dev)
    e0, e1 = events()
    with torch.cuda.stream(s_comp):
        trfn.tr_fused_norm(src0, d_out[0], mean, std, d_par, out_dtype=trfn.OUT_F16, stream=s_comp, workspace=ws)
        e0.record(s_comp)
        for k in range(16):
            trfn.tr_fused_norm(src0, d_out[k & 1], mean, std, d_par, out_dtype=trfn.OUT_F16, stream=s_comp,
                               workspace=ws)
        e1.record(s_comp)
    e1.synchronize()
    t_kernel = e0.elapsed_time(e1) / 16 / 1e3
    # the pipelined stream
    ts = trfn.TransferStation(dev.index, slots, s_copy, s_comp, None)
    for b in range(2):   # warm-up: the station's first batch also saves its filler
        ts.submit(h_src[b], d_out[b & 1], mean, std, h_params=h_par[b], out_dtype=trfn.OUT_F16)
    assert ts.sync(60000)
    # the stream of B batches, three times; the median is reported (host
    # memory and its link are shared with the machine's other jobs)
    passes = []
    for _ in range(3):
        barrier(pg)
        torch.cuda.synchronize()
        e0, e1 = events()
        e0.record(s_copy)
        launches = trfn.tr_launch_count()
        for b in range(B):
            ts.submit(h_src[b], d_out[b & 1], mean, std, h_params=h_par[b], out_dtype=trfn.OUT_F16)
        e1.record(s_comp)
        launches = trfn.tr_launch_count() - launches
        e1.synchronize()
        assert ts.sync(60000)
        passes.append(max_over_ranks(pg, e0.elapsed_time(e1) / 1e3, dev))
    ts.close()
    t_pipe = float(np.median(passes))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    h2d = img_bytes + N * 20
    # the last two batches' outputs are still on the device (batch b wrote
    # d_out[b & 1]): images first, middle and last of each against the oracle
    parity = {"batches": [B - 2, B - 1], "images": [0, N // 2, N - 1], "ok": True, "max_f16_ulp": 0}
    for b in (B - 2, B - 1):
        one = parity_sample(dict(cfg, layout="nhwc"), [h_src[b]], [d_out[b & 1]], [h_par[b].numpy()], mean, std,
                            trfn.OUT_F16, trfn.LAYOUT_NHWC, 1)
        parity["ok"] = parity["ok"] and one["ok"]
        parity["max_f16_ulp"] = max(parity["max_f16_ulp"], one["max_f16_ulp"])
    return {
        "workload": cfg["name"], "batches": B, "images_per_s": world * B * N / t_pipe,
        "passes_images_per_s": [world * B * N / t for t in passes], "how": "median of three passes",
        "ms_pipelined": t_pipe * 1e3, "h2d_gbs_lone_copy": img_bytes / t_copy / 1e9,
        "us_copy_per_batch": t_copy * 1e6, "us_kernel_per_batch": t_kernel * 1e6,
        "overlap_efficiency": B * (t_copy + t_kernel) / t_pipe,
        "overlap_efficiency_bound": (t_copy + t_kernel) / max(t_copy, t_kernel),
        "h2d_gbs_pipelined": B * h2d / t_pipe / 1e9,
        "h2d_bytes_per_batch": h2d, "gpu_launches": int(launches),
        "path": "tr_ts_submit: pinned host u8 + records -> device slot A/B (copy stream) -> kernel "
                "(compute stream); outputs stay on the device",
        "pixels": "rint(Normal(110, 60)) clipped to [0, 255] (seed 5000 + b), drawn in %.1f s on host threads" % t_draw,
        "parity_sample": parity,
    }


def run_config(k, layout_name, dev, peak):
    """One of the other batch workloads (16x32x32x3 -> f32, 200x28x28x1 ->
    f32, 256x224x224x3 -> f32 NHWC or NCHW): a CUDA graph of launches
    rotating over enough buffer sets to exceed L2 four times, timed with the
    launches overlapping the previous one (independent batches) and with each
    waiting for the previous one; three trials each, median reported; three
    images of the last written set against the oracle."""
    import torch
    import image_preprocessing_gb300 as trfn
    from image_preprocessing_gb300 import synth
    cfg = dict(synth.CONFIGS[k])
    cfg["layout"] = layout_name
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    dt = trfn.OUT_F16 if cfg["out_dtype"] == "f16" else trfn.OUT_F32
    layout = {"nhwc": trfn.LAYOUT_NHWC, "nchw": trfn.LAYOUT_NCHW, "nhwc4": trfn.LAYOUT_NHWC4}[layout_name]
    mean = np.array(cfg["mean"], np.float32)
    std = np.array(cfg["std"], np.float32)
    pixels = synth.config_pixels(k)
    recs = None
    if cfg["flip"] or cfg["erase"]:
        recs, _ = trfn.tr_sample_aug_params(2000 + k, 0, N, H, W, flip=cfg["flip"], erase=cfg["erase"],
                                            erase_p=cfg["erase_p"])
    out_shape = trfn.out_shape(N, H, W, C, layout)
    ob = 2 if dt == trfn.OUT_F16 else 4
    in_bytes, out_bytes = N * H * W * C, int(np.prod(out_shape)) * ob
    in_stride, out_stride = -(-in_bytes // 256) * 256, -(-out_bytes // 256) * 256
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(2, int(np.ceil(4 * l2 / (in_bytes + out_bytes))))
    G = nsets * max(1, 60 // nsets)
    G += G % 2
    # every set holds the same pixels at its own address
    src_all = torch.empty((nsets, in_stride), dtype=torch.uint8, device=dev)
    src_all[:, :in_bytes].copy_(torch.from_numpy(pixels).reshape(1, -1).to(dev).expand(nsets, -1))
    dst_all = torch.empty((nsets, out_stride), dtype=torch.uint8, device=dev)
    aug = torch.from_numpy(recs).to(dev) if recs is not None else None
    s0, d0 = src_all.data_ptr(), dst_all.data_ptr()
    stream = torch.cuda.Stream(device=dev)
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device=dev) for _ in range(2)]
    kernel = trfn.tr_fused_norm_plan(s0, d0, N, H, W, C, dt, layout)

    def launch(j, overlap):
        trfn.tr_fused_norm(s0 + (j % nsets) * in_stride, d0 + (j % nsets) * out_stride, mean, std, aug,
                           out_dtype=dt, layout=layout, stream=stream, shape=(N, H, W, C), workspace=wss[j % 2],
                           overlap_previous=overlap)

    with torch.cuda.stream(stream):
        for j in range(nsets + nsets % 2):
            launch(j, False)
    torch.cuda.synchronize()
    alg = algorithmic_bytes(cfg, recs)
    res = {"workload": cfg["name"].replace("_nhwc_nchw", "_" + layout_name), "N": N, "H": H, "W": W, "C": C,
           "out": cfg["out_dtype"] + " " + layout_name.upper(),
           "kernel": {trfn.VARIANT_TILED: "tiled", trfn.VARIANT_GENERIC: "per-element"}.get(kernel, str(kernel)),
           "algorithmic_bytes_per_launch": alg,
           "l2": "%d rotating buffer sets, %.0f MB >= 4x L2" % (nsets, nsets * (in_bytes + out_bytes) / 1e6)}
    reps = max(1, -(-240 // G))
    for mode, overlap in (("overlapping", True), ("waiting", False)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(G):
                launch(j, overlap)
        with torch.cuda.stream(stream):
            g.replay()
        per = []
        for _ in range(3):
            e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                torch.cuda._sleep(SPACER_CYCLES)
                e_a.record(stream)
                for _ in range(reps):
                    g.replay()
                e_b.record(stream)
            e_b.synchronize()
            per.append(e_a.elapsed_time(e_b) / (reps * G))
        ms = float(np.median(per))
        gbs = alg / (ms / 1e3) / 1e9
        res[mode] = {"ms_per_step": ms, "images_per_s": N / (ms / 1e3), "achieved_gbs": gbs, "frac": gbs / peak,
                     "trials_ms_per_step": per, "launches_timed": reps * G}
        del g
    torch.cuda.synchronize()
    last = (G - 1) % nsets
    got = dst_all[last, :out_bytes].view(torch.float16 if dt == trfn.OUT_F16 else torch.float32).view(out_shape)
    res["parity_sample"] = parity_sample(cfg, [torch.from_numpy(pixels)], [got], [recs], mean, std, dt, layout, 1)
    res["launch"] = "CUDA graph of %d launches, %d replay(s) per trial after one untimed replay" % (G, reps)
    return res


def run_batched(dev, peak, Ks=(1, 4, 8)):
    """The headline workload (256 x 224x224x3 -> f16 NHWC, flip + erase) as
    launches of K batches each (tr_fused_norm_batches): 2*max(K) distinct
    buffer sets, each launch taking the next K; per-batch time and roofline
    fraction with each launch waiting for the previous one and with launches
    overlapping; three trials each (median); the first batch of the last
    launch against the oracle."""
    import torch
    import image_preprocessing_gb300 as trfn
    from image_preprocessing_gb300 import synth
    cfg = dict(synth.CONFIGS[3], layout="nhwc")
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    mean = np.array(cfg["mean"], np.float32)
    std = np.array(cfg["std"], np.float32)
    nsets = 2 * max(Ks)
    px = synth.config_pixels(3)
    src0 = torch.from_numpy(px).to(dev)
    srcs = [src0.clone() for _ in range(nsets)]
    dsts = [torch.empty((N, H, W, C), dtype=torch.float16, device=dev) for _ in range(nsets)]
    recs, augs, offset = [], [], 0
    for j in range(nsets):
        r, offset = trfn.tr_sample_aug_params(2003, offset, N, H, W, erase_p=cfg["erase_p"])
        recs.append(r)
        augs.append(torch.from_numpy(r).to(dev))
    alg = [algorithmic_bytes(cfg, r) for r in recs]
    stream = torch.cuda.Stream(device=dev)
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device=dev) for _ in range(2)]
    out = {}
    last = None
    for K in Ks:
        per_cycle = nsets // K   # launches per pass over the sets
        L = per_cycle * max(1, 32 // (per_cycle * K))   # about 32 batches per graph

        def launch(i, overlap):
            sel = [(i * K + t) % nsets for t in range(K)]
            trfn.tr_fused_norm_batches([(srcs[j], dsts[j], augs[j]) for j in sel], mean, std,
                                       out_dtype=trfn.OUT_F16, layout=trfn.LAYOUT_NHWC, stream=stream,
                                       workspace=wss[i % 2], overlap_previous=overlap)
            return sel

        res = {}
        for mode, overlap in (("waiting", False), ("overlapping", True)):
            with torch.cuda.stream(stream):
                for i in range(L):
                    last = launch(i, overlap)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(L):
                    launch(i, overlap)
            with torch.cuda.stream(stream):
                g.replay()
            per = []
            reps = 4
            for _ in range(3):
                e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    torch.cuda._sleep(SPACER_CYCLES)
                    e_a.record(stream)
                    for _ in range(reps):
                        g.replay()
                    e_b.record(stream)
                e_b.synchronize()
                per.append(e_a.elapsed_time(e_b) / (reps * L * K))
            ms = float(np.median(per))
            avg = float(np.mean([alg[(i * K + t) % nsets] for i in range(L) for t in range(K)]))
            gbs = avg / (ms / 1e3) / 1e9
            res[mode] = {"us_per_batch": ms * 1e3, "images_per_s": N / (ms / 1e3), "achieved_gbs": gbs,
                         "frac": gbs / peak, "trials_us_per_batch": [v * 1e3 for v in per]}
            del g
        res["launches_per_graph"] = L
        out["K=%d" % K] = res
    torch.cuda.synchronize()
    j = last[0]
    parity = parity_sample(cfg, [srcs[j]], [dsts[j]], [recs[j]], mean, std, trfn.OUT_F16, trfn.LAYOUT_NHWC, 1)
    out["parity_sample"] = parity
    out["path"] = ("tr_fused_norm_batches: K batches of 256x224x224x3 -> f16 NHWC (flip + erase) per launch, "
                   "dynamic schedule, %d rotating buffer sets" % nsets)
    return out


def time_graph_modes(stream, launch, G, reps, per_launch_units=1):
    """Median milliseconds per unit (a launch, or per_launch_units batches of
    it) of a CUDA graph of G launches, replayed reps times per trial, three
    trials, with the launches overlapping the previous one and with each
    waiting for it: {mode: (median, trials)}.  launch(k, overlap) issues
    launch k on stream; one untimed replay precedes the trials."""
    import torch
    out = {}
    for mode, overlap in (("overlapping", True), ("waiting", False)):
        with torch.cuda.stream(stream):
            for k in range(G):
                launch(k, overlap)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(G):
                launch(k, overlap)
        with torch.cuda.stream(stream):
            g.replay()
        per = []
        for _ in range(3):
            e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                torch.cuda._sleep(SPACER_CYCLES)
                e_a.record(stream)
                for _ in range(reps):
                    g.replay()
                e_b.record(stream)
            e_b.synchronize()
            per.append(e_a.elapsed_time(e_b) / (reps * G * per_launch_units))
        out[mode] = (float(np.median(per)), per)
        del g
    torch.cuda.synchronize()
    return out


def run_sampled(dev, peak):
    """The headline workload with its records drawn on the GPU in the same
    call (tr_fused_norm_sampled: the sampler grid, then the fused kernel,
    whose CTAs make their first records themselves when the call overlaps
    the previous one): per-batch time and roofline fraction overlapping and
    waiting; the records and three images of the last written set against
    the oracle."""
    import torch
    import image_preprocessing_gb300 as trfn
    from image_preprocessing_gb300 import synth
    cfg = dict(synth.CONFIGS[3], layout="nhwc")
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    mean = np.array(cfg["mean"], np.float32)
    std = np.array(cfg["std"], np.float32)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(2, int(np.ceil(4 * l2 / (N * H * W * C * 3))))
    src0 = torch.from_numpy(synth.config_pixels(3)).to(dev)
    srcs = [src0.clone() for _ in range(nsets)]
    dsts = [torch.empty((N, H, W, C), dtype=torch.float16, device=dev) for _ in range(nsets)]
    recs = [torch.zeros((N, 5), dtype=torch.int32, device=dev) for _ in range(nsets)]
    stream = torch.cuda.Stream(device=dev)
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device=dev) for _ in range(2)]
    G = nsets * max(1, 60 // nsets)
    G += G % 2

    def launch(k, overlap):
        j = k % nsets
        trfn.tr_fused_norm_sampled(srcs[j], dsts[j], mean, std, 4000 + j, 0, recs[j], flip=cfg["flip"],
                                   erase=cfg["erase"], erase_p=cfg["erase_p"], out_dtype=trfn.OUT_F16,
                                   layout=trfn.LAYOUT_NHWC, stream=stream, workspace=wss[k % 2],
                                   overlap_previous=overlap)

    t = time_graph_modes(stream, launch, G, max(1, -(-240 // G)))
    got_recs = [r.cpu().numpy() for r in recs]   # the records the sampler wrote (bytes of the erased spans)
    alg = float(np.mean([algorithmic_bytes(cfg, got_recs[k % nsets]) for k in range(G)]))
    out = {"workload": cfg["name"] + "_records_sampled_in_call", "algorithmic_bytes_per_launch": alg,
           "l2": "%d rotating buffer sets >= 4x L2" % nsets}
    for mode, (ms, per) in t.items():
        gbs = alg / (ms / 1e3) / 1e9
        out[mode] = {"us_per_batch": ms * 1e3, "images_per_s": N / (ms / 1e3), "achieved_gbs": gbs,
                     "frac": gbs / peak, "trials_us_per_batch": [v * 1e3 for v in per]}
    import oracle
    j = (G - 1) % nsets
    ref_recs = oracle.sample_aug_params_blocked(4000 + j, 0, N, H, W, flip=cfg["flip"], erase=cfg["erase"],
                                                erase_p=cfg["erase_p"])[0]
    par = parity_sample(cfg, [srcs[j]], [dsts[j]], [ref_recs], mean, std, trfn.OUT_F16, trfn.LAYOUT_NHWC, 1)
    par["records_equal"] = bool(np.array_equal(got_recs[j], ref_recs))
    par["ok"] = par["ok"] and par["records_equal"]
    out["parity_sample"] = par
    out["path"] = ("tr_fused_norm_sampled: records sampled on the GPU (Philox4x32-10 counters) and the fused step "
                   "in one call, graph of %d calls" % G)
    return out


def run_odd_rows(dev, peak):
    """256 x 299x299x3 -> f16 NHWC, f16 NCHW and f32 NCHW, flip + erase:
    source rows of 897 bytes and NCHW output rows of 598 / 1196, the tiled
    kernel's odd-row form; per batch overlapping and waiting, three images of
    the last set against the oracle."""
    import torch
    import image_preprocessing_gb300 as trfn
    from image_preprocessing_gb300 import synth
    out = {}
    N, H, W, C = 256, 299, 299, 3
    for layout_name, dt_name in (("nhwc", "f16"), ("nchw", "f16"), ("nchw", "f32")):
        cfg = dict(synth.CONFIGS[3], H=H, W=W, layout=layout_name, out_dtype=dt_name)
        cfg["name"] = "n256_299x299x3_%s_%s_flip_erase" % (dt_name, layout_name)
        layout = trfn.LAYOUT_NHWC if layout_name == "nhwc" else trfn.LAYOUT_NCHW
        dt = trfn.OUT_F16 if dt_name == "f16" else trfn.OUT_F32
        ob = 2 if dt_name == "f16" else 4
        mean = np.array(cfg["mean"], np.float32)
        std = np.array(cfg["std"], np.float32)
        shape = trfn.out_shape(N, H, W, C, layout)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        nsets = max(2, int(np.ceil(4 * l2 / (N * H * W * C * (1 + ob)))))
        px = synth.pixels_uniform(1299, N, H, W, C)
        src0 = torch.from_numpy(px).to(dev)
        srcs = [src0.clone() for _ in range(nsets)]
        dsts = [torch.empty(shape, dtype=torch.float16 if ob == 2 else torch.float32, device=dev)
                for _ in range(nsets)]
        recs_all, augs, offset = [], [], 0
        for j in range(nsets):
            r, offset = trfn.tr_sample_aug_params(2299, offset, N, H, W, erase_p=cfg["erase_p"])
            recs_all.append(r)
            augs.append(torch.from_numpy(r).to(dev))
        stream = torch.cuda.Stream(device=dev)
        wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device=dev) for _ in range(2)]
        G = nsets * max(1, 60 // nsets)
        G += G % 2

        def launch(k, overlap):
            j = k % nsets
            trfn.tr_fused_norm(srcs[j], dsts[j], mean, std, augs[j], out_dtype=dt, layout=layout,
                               stream=stream, workspace=wss[k % 2], overlap_previous=overlap)

        t = time_graph_modes(stream, launch, G, max(1, -(-120 // G)))
        alg = float(np.mean([algorithmic_bytes(cfg, recs_all[k % nsets]) for k in range(G)]))
        geo = trfn.tr_fused_norm_geometry(N, H, W, C, out_dtype=dt, layout=layout, overlap_previous=True)
        # geometry's grid is the static schedule's; these launches carry a
        # workspace, so they take every resident slot (or one CTA per band)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        geo["grid_launched"] = min(N * -(-H // geo["rows"]), geo["ctas_per_sm"] * sms)
        r = {"workload": cfg["name"], "algorithmic_bytes_per_launch": alg,
             "kernel": "tiled, odd-row form" if geo.get("odd_form") else "tiled", "geometry": geo,
             "l2": "%d rotating buffer sets >= 4x L2" % nsets}
        for mode, (ms, per) in t.items():
            gbs = alg / (ms / 1e3) / 1e9
            r[mode] = {"us_per_batch": ms * 1e3, "images_per_s": N / (ms / 1e3), "achieved_gbs": gbs,
                       "frac": gbs / peak, "trials_us_per_batch": [v * 1e3 for v in per]}
        j = (G - 1) % nsets
        r["parity_sample"] = parity_sample(cfg, [srcs[j]], [dsts[j]], [recs_all[j]], mean, std, dt, layout, 1)
        out[cfg["name"]] = r
        del srcs, dsts
        torch.cuda.empty_cache()
    return out


def run_per_config(dev, peak, cpu_seconds, with_cpu):
    """The other batch workloads beside the headline, keyed by workload name;
    for the 256x224x224x3 -> f32 validation batch also the oracle on the
    host's cores (all of them and one)."""
    from image_preprocessing_gb300 import synth
    out = {}
    for k, lay in ((1, "nhwc"), (2, "nhwc"), (4, "nhwc"), (4, "nchw")):
        r = run_config(k, lay, dev, peak)
        if with_cpu and k == 4:
            cfg = dict(synth.CONFIGS[4], layout=lay)
            v, threads, sample = oracle_images_per_s(cfg, cpu_seconds)
            v1, _, sample1 = oracle_images_per_s(cfg, max(1.0, cpu_seconds / 2), threads=1)
            per_image = r["algorithmic_bytes_per_launch"] / r["N"]
            r["cpu_baseline"] = {"value": v, "unit": "images/s", "cores": threads, "kind": "oracle",
                                 "algorithmic_gbs": v * per_image / 1e9, "sample": sample,
                                 "single_core": {"value": v1, "algorithmic_gbs": v1 * per_image / 1e9,
                                                 "sample": sample1}}
        out[r["workload"]] = r
    return out


# ------------------------------------------------------------- oracle -----

def cpu_model():
    """The host CPU as /proc/cpuinfo names it (model name, else the Arm part)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown"
    arm_parts = {"0xd4f": "Neoverse V2", "0xd40": "Neoverse V1", "0xd0c": "Neoverse N1"}
    for line in info.splitlines():
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    for line in info.splitlines():
        if line.lower().startswith("cpu part"):
            part = line.split(":", 1)[1].strip().lower()
            return "Arm part %s (%s)" % (part, arm_parts.get(part, "unlisted"))
    return "unknown"


def oracle_images_per_s(cfg, seconds, threads=None):
    """The oracle as it stands on a bounded sample of the workload, split by
    image over host threads (ctypes releases the GIL).  Returns
    (images/s, threads, sample text)."""
    import oracle
    import image_preprocessing_gb300 as trfn
    threads = threads or os.cpu_count() or 1
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    m = min(N, max(threads, 8))
    src = host_batch(dict(cfg, N=m), 1000 + 3)
    recs = None
    if cfg["flip"] or cfg["erase"]:
        recs, _ = oracle.sample_aug_params(2003, 0, m, H, W, flip=cfg["flip"], erase=cfg["erase"],
                                           erase_p=cfg["erase_p"])
    mean = np.array(cfg["mean"], np.float32)
    std = np.array(cfg["std"], np.float32)
    dt = oracle.OUT_F16 if cfg["out_dtype"] == "f16" else oracle.OUT_F32
    layout = {"nhwc": 0, "nchw": 1, "nhwc4": 2}[cfg["layout"]]
    done = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while time.perf_counter() - t0 < seconds:
            futs = [ex.submit(oracle.fused_norm, src[i:i + 1], mean, std,
                              None if recs is None else recs[i:i + 1], dt, layout) for i in range(m)]
            for f in futs:
                f.result()
            done += m
    el = time.perf_counter() - t0
    sample = "%d passes over %d of the %d images (%dx%dx%d), %.1f s on %d threads" % (
        done // m, m, N, H, W, C, el, threads)
    return done / el, threads, sample


def run_reference(args, rank, world, pg):
    """The oracle as the reference arm: each step runs the oracle over one
    image per host thread of the workload (a bounded sample of the batch);
    up to --steps steps, stopping early once --cpu-seconds have passed."""
    cfg = workload(args)
    if rank != 0:
        return None
    import oracle
    threads = os.cpu_count() or 1
    N, H, W, C = cfg["N"], cfg["H"], cfg["W"], cfg["C"]
    m = min(N, threads)
    src = host_batch(cfg, 1000 + args.config)[:m].copy()
    recs = None
    if cfg["flip"] or cfg["erase"]:
        recs, _ = oracle.sample_aug_params(2000 + args.config, 0, m, H, W, flip=cfg["flip"], erase=cfg["erase"],
                                           erase_p=cfg["erase_p"])
    mean = np.array(cfg["mean"], np.float32)
    std = np.array(cfg["std"], np.float32)
    dt = oracle.OUT_F16 if cfg["out_dtype"] == "f16" else oracle.OUT_F32
    layout = {"nhwc": 0, "nchw": 1, "nhwc4": 2}[cfg["layout"]]
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        def step():
            futs = [ex.submit(oracle.fused_norm, src[i:i + 1], mean, std, None if recs is None else recs[i:i + 1],
                              dt, layout) for i in range(m)]
            for f in futs:
                f.result()
        for _ in range(min(args.warmup, 3)):
            step()
        done = 0
        t0 = time.perf_counter()
        while done < args.steps and (done == 0 or time.perf_counter() - t0 < args.cpu_seconds):
            step()
            done += 1
        el = time.perf_counter() - t0
    value = m * done / el
    sample = "%d steps of %d of the %d images (%dx%dx%d, one per thread), %.1f s on %d threads" % (
        done, m, N, H, W, C, el, threads)
    return {"metric": METRIC, "value": value, "unit": "images/s", "n_gpus": world, "steps": done,
            "warmup": args.warmup, "ms_per_step": el * 1000 / max(1, done), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg["workload"], "N": N, "H": H, "W": W, "C": C},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "images/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "images/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, local, world, pg = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, rank, world, pg)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
        return
    res = run_ours(args, rank, local, world, pg)
    if rank == 0:
        if not args.no_cpu and world == 1:
            cfg = workload(args)
            v, threads, sample = oracle_images_per_s(cfg, args.cpu_seconds)
            v1, _, sample1 = oracle_images_per_s(cfg, max(1.0, args.cpu_seconds / 4), threads=1)
            # the GPU line's mean algorithmic bytes per image (its sampled rectangles)
            per_image = res["roofline"]["algorithmic_bytes_per_launch"] / res["config"]["N"]
            res["cpu_baseline"] = {"value": v, "unit": "images/s", "cores": threads, "kind": "oracle",
                                   "algorithmic_gbs": v * per_image / 1e9, "sample": sample,
                                   "single_core": {"value": v1, "algorithmic_gbs": v1 * per_image / 1e9,
                                                   "sample": sample1},
                                   "cpu_model": cpu_model()}
        print(json.dumps(res), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
