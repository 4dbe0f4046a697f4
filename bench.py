"""Benchmark of the GDN decode-step front: µs per launch and achieved HBM
bandwidth at 1..16 rows on one GB300, through the C ABI.

A step is one launch of the whole path (residual add + norm, in_proj_qkvz /
in_proj_ba, conv update, gates, gated delta rule, gated norm) over one batch
of rows. Launches are replayed from a CUDA graph; every launch reads another
copy of the layer weights (the copies together exceed L2) and another set of
state slots, so each launch streams its weights and state from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--rows R] [--workload full]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

The headline is the full unsharded layer (H=8192, 16 key / 64 value heads,
dk=dv=128, 512 slots of f32 state) at 16 rows: the largest configuration of
the method that runs on one GPU. The same line carries per-width tables of
every workload (the shard, the full layer, the shard with a bf16 state in
its first-layer variant with a quarter of the rows padding, and the dense
MXFP4 layer over a rotated 48-layer stack).

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN decode-block µs/launch and achieved HBM GB/s (% of peak) at rows 1–16"
PAGES_NOTE = ("pages report 13.3-34.7 µs/launch at 1-16 rows on MI355X TP8 with MXFP4 weights "
              "(other hardware and format: context only)")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="full")
    ap.add_argument("--rows", type=int, default=16, help="rows of the headline step")
    ap.add_argument("--widths", default="1,2,4,8,16", help="widths of the per-width tables")
    ap.add_argument("--tables",
                    default="shard,full,shard_bf16,dense_mxfp4,dense_mxfp6,shard_wide,shard_verify,shard_out,full_out",
                    help="workloads of the per-width tables ('' for none)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--engine", default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-child", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e nominal


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# Per-width table recipe of each workload: widths, the pad fraction, the
# first-layer variant, the least number of weight copies the launches rotate
# over (the dense MXFP4 layer rotates a 48-layer stack).
TABLES = {
    "shard": {"widths": [1, 2, 4, 8, 16]},
    "full": {"widths": [1, 2, 4, 8, 16]},
    "shard_bf16": {"widths": [1, 3, 8, 9, 16], "pad": 0.25, "first_layer": True},
    "dense_mxfp4": {"widths": [1, 2, 4, 8, 16], "min_copies": 48},
    "dense_mxfp6": {"widths": [1, 2, 4, 8, 16], "min_copies": 48},
    # steps wider than one launch (one launch per 16-row tile)
    "shard_wide": {"shape": "shard", "max_rows": 64, "widths": [16, 24, 32, 48, 64]},
    # the step with out_proj folded in
    "shard_out": {"shape": "shard", "widths": [1, 4, 8, 16], "out_proj": True},
    "full_out": {"shape": "full", "widths": [1, 16], "out_proj": True},
    # verify steps: (sequences, tokens) with a state slot per token
    "shard_verify": {"shape": "shard", "verify": [(1, 2), (1, 4), (2, 4), (4, 4), (8, 2), (2, 8)]},
}


# ----------------------------------------------------------------- CPU oracle

def oracle_inputs(shape, rows, seed):
    import torch
    from gated_deltanet_layer_gb300 import workloads as WL
    w = WL.make_weights(shape, seed)
    st = WL.make_state(shape, seed + 1)
    stp = WL.make_step(shape, rows, seed + 2)
    f64 = lambda t: None if t is None else (t.numpy() if t.dtype == torch.uint8 else t.to(torch.float64).numpy())
    return (f64(stp["x"]), f64(stp["residual"]), {k: f64(v) for k, v in w.items()},
            stp["state_indices"].numpy(), f64(st["conv_state"]), f64(st["ssm_state"]))


def cpu_child(args):
    """Time the oracle (as it stands) for about --cpu-seconds; print a JSON line."""
    from gated_deltanet_layer_gb300 import workloads as WL
    from oracle import gdn_oracle as O
    shape = WL.SHAPES[args.workload]
    x, res, w, idx, conv, ssm = oracle_inputs(shape, args.rows, 777)
    n, t0 = 0, time.perf_counter()
    limit = args.steps if args.impl == "reference" else None
    while True:
        O.gdn_step(shape, x, res, w, idx, conv, ssm)
        n += 1
        el = time.perf_counter() - t0
        if (limit is not None and n >= limit) or (limit is None and el >= args.cpu_seconds):
            break
    print(json.dumps({"n": n, "seconds": el, "us_per_step": el / n * 1e6}))


def run_cpu_baseline(args, steps=None, seconds=None):
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-child", "--workload", args.workload,
           "--rows", str(args.rows), "--cpu-seconds", str(seconds or args.cpu_seconds)]
    if steps is not None:
        cmd += ["--impl", "reference", "--steps", str(steps)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d, cores


# ----------------------------------------------------------------- traffic


def kernel_source_hash() -> str:
    """sha256 (16 hex digits) of the kernel sources and the C header."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "gated_deltanet_layer_gb300", "csrc", "*")) +
                   glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, rows: int):
    """DRAM bytes (read + write) per launch of the step kernel from the
    committed ncu record in profiles/, if it was taken on these kernel sources
    with this workload and row count; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha") != kernel_source_hash() or rec.get("workload") != workload or rec.get("rows") != rows:
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- clocks

class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        busy = sorted(sm)
        med = busy[len(busy) // 2]
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- ranks

def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's `value` (the slowest rank's time); the value
    itself on a single process (dist None)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- GPU arm

class Rig:
    """One workload on the device: weight copies the launches rotate over
    (together larger than 3x L2, and at least `min_copies`), the conv and SSM
    state of every slot, and a handle."""

    def __init__(self, shape, g, l2, engine, min_copies=4, out_proj=False):
        import torch
        from gated_deltanet_layer_gb300 import GdnDecode
        self.shape, self.g = shape, g
        self.out_proj = out_proj
        wbytes = shape.weight_bytes() + (shape.out_proj_bytes(0) if out_proj else 0)
        self.ncopy = max(min_copies, int((3 * l2 + wbytes - 1) // wbytes) + 1)
        self.wbytes = wbytes
        H, Hv = shape.hidden, shape.num_v_heads

        def qkvz():
            if shape.qkvz_format in ("mxfp4", "mxfp6"):
                # codes uniform; block exponents U{-8..-4} (MXFP4) or U{-10..-6} (MXFP6)
                nbytes, elo = (H // 2, -8) if shape.qkvz_format == "mxfp4" else (H * 3 // 4, -10)
                return {"qkvz": torch.randint(0, 256, (shape.n_qkvz, nbytes), generator=g, device="cuda",
                                              dtype=torch.uint8),
                        "qkvz_scales": (127 + torch.randint(elo, elo + 5, (shape.n_qkvz, H // 32), generator=g,
                                                            device="cuda")).to(torch.uint8)}
            return {"qkvz": self.bf16(shape.n_qkvz, H, std=0.02), "qkvz_scales": None}

        self.copies = []
        for _ in range(self.ncopy):
            self.copies.append({
                "input_norm_w": self.bf16(H, std=0.1),
                **qkvz(),
                "ba": self.bf16(shape.n_ba, H, std=0.02),
                "conv_w": self.bf16(shape.conv_channels, shape.conv_kernel, std=0.02),
                "A_log": -2.0 * torch.rand(Hv, generator=g, device="cuda"),
                "dt_bias": self.bf16(Hv, std=0.5),
                "gated_norm_w": self.bf16(shape.head_v_dim, std=0.1),
                "out_proj": self.bf16(H, Hv * shape.head_v_dim, std=0.02) if out_proj else None,
            })
        sdt = torch.bfloat16 if shape.ssm_dtype == "bf16" else torch.float32
        self.conv = self.bf16(shape.num_slots, shape.conv_channels, shape.conv_kernel - 1, std=1.0)
        self.ssm = (torch.randn(shape.num_slots, Hv, shape.head_v_dim, shape.head_k_dim, generator=g,
                                device="cuda") * 0.1).to(sdt)
        self.layer = GdnDecode(shape, engine=engine)
        self.wstructs = [self.layer.weights_struct(c) for c in self.copies]

    def bf16(self, *s, std):
        import torch
        return (torch.randn(*s, generator=self.g, device="cuda") * std).to(torch.bfloat16)

    def batch(self, rows, n, pad=0.0, first_layer=False):
        """n distinct step inputs of `rows` rows with fresh random slots each;
        round(pad * rows) of the rows are pad rows (index 0)."""
        import torch
        sh = self.shape
        npad = int(round(pad * rows))
        out = []
        for _ in range(n):
            perm = torch.randperm(sh.num_slots - 1, generator=self.g, device="cuda")[:rows] + 1
            if npad:
                perm[torch.randperm(rows, generator=self.g, device="cuda")[:npad]] = 0
            out.append((self.bf16(rows, sh.hidden, std=1.0), None if first_layer else self.bf16(rows, sh.hidden, std=1.0),
                        perm.to(torch.int32).contiguous(),
                        torch.empty(rows, sh.num_v_heads * sh.head_v_dim, dtype=torch.bfloat16, device="cuda"),
                        torch.empty(rows, sh.hidden, dtype=torch.bfloat16, device="cuda"),
                        torch.empty(rows, sh.hidden, dtype=torch.bfloat16, device="cuda") if self.out_proj else None))
        return out

    def capture(self, rows, n, pad=0.0, first_layer=False):
        """A CUDA graph of n launches, each on the next weight copy."""
        import torch
        batch = self.batch(rows, min(n, 64), pad, first_layer)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        def one(k, b):
            x, r, i, c, ro, o = b
            if self.out_proj:
                self.layer.step_out(x, r, self.copies[k % self.ncopy], i, self.conv, self.ssm, c, ro, o,
                                    weights_struct=self.wstructs[k % self.ncopy])
            else:
                self.layer.step(x, r, self.copies[k % self.ncopy], i, self.conv, self.ssm, c, ro,
                                weights_struct=self.wstructs[k % self.ncopy])

        with torch.cuda.stream(s):
            one(0, batch[0])  # one eager launch first (lazy set-up outside the capture)
            torch.cuda.current_stream().synchronize()
            with torch.cuda.graph(graph, stream=s):
                for k in range(n):
                    one(k, batch[k % len(batch)])
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return graph

    def capture_verify(self, seqs, tokens, n):
        """A CUDA graph of n verify steps (seqs sequences of `tokens` tokens,
        fresh random input and per-token output slots each), each on the next
        weight copy."""
        import torch
        sh = self.shape
        steps = []
        for _ in range(min(n, 64)):
            perm = torch.randperm(sh.num_slots - 1, generator=self.g, device="cuda")[:seqs * (tokens + 1)] + 1
            perm = perm.to(torch.int32)
            rows = seqs * tokens
            steps.append((self.bf16(rows, sh.hidden, std=1.0), self.bf16(rows, sh.hidden, std=1.0),
                          perm[:seqs].contiguous(), perm[seqs:].reshape(seqs, tokens).contiguous(),
                          torch.empty(rows, sh.num_v_heads * sh.head_v_dim, dtype=torch.bfloat16, device="cuda"),
                          torch.empty(rows, sh.hidden, dtype=torch.bfloat16, device="cuda")))
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            x, r, si, so, c, ro = steps[0]
            self.layer.verify(x, r, self.copies[0], si, so, self.conv, self.ssm, c, ro, weights_struct=self.wstructs[0])
            torch.cuda.current_stream().synchronize()
            with torch.cuda.graph(graph, stream=s):
                for k in range(n):
                    x, r, si, so, c, ro = steps[k % len(steps)]
                    self.layer.verify(x, r, self.copies[k % self.ncopy], si, so, self.conv, self.ssm, c, ro,
                                      weights_struct=self.wstructs[k % self.ncopy])
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return graph

    def check(self):
        st, detail = self.layer.check()
        if st != 0:
            raise RuntimeError(f"device error word 0x{detail:08x} ({self.shape.name})")


def native(args):
    import torch
    from gated_deltanet_layer_gb300 import workloads as WL

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    shape = WL.SHAPES[args.workload]
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    peak, peak_kind = peaks()
    g = torch.Generator(device="cuda")
    g.manual_seed(1234 + rank)

    def time_graph(graph):
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(st)
        graph.replay()
        e1.record(st)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        return e0.elapsed_time(e1)  # ms

    def row_of(sh, u, rows, live, first_layer, extra=0):
        b = sh.launch_bytes(rows, live, first_layer=first_layer) + extra
        gbs = b / u / 1e3
        return {"us": round(u, 3), "GBps": round(gbs, 1), "frac_of_" + peak_kind: round(gbs / peak, 4),
                "frac_of_nominal_8TBps": round(gbs / NOMINAL_HBM_GBS, 4), "bytes": b, "live_rows": live,
                "launches": -(-rows // 16)}

    def width_table(rig, widths, pad=0.0, first_layer=False):
        extra = (lambda r: rig.shape.out_proj_bytes(r)) if rig.out_proj else (lambda r: 0)
        """µs per launch of a graph of 100 launches, median of replays over
        ~0.3 s (so the clock sampler sees the GPU under load)."""
        out = {}
        for wdt in widths:
            gg = rig.capture(wdt, 100, pad, first_layer)
            times = []
            t_end = time.time() + 0.3
            while time.time() < t_end or len(times) < 5:
                times.append(time_graph(gg) * 10.0)  # µs per launch
            times.sort()
            live = wdt - int(round(pad * wdt))
            out[str(wdt)] = row_of(rig.shape, times[len(times) // 2], wdt, live, first_layer, extra(wdt))
            del gg
        rig.check()
        return out

    K, Wm = args.steps, args.warmup
    clocks = Clocks(local)
    rig = Rig(shape, g, l2, args.engine)
    # warm-up: W untimed steps
    gw = rig.capture(args.rows, max(3, Wm))
    gw.replay()
    torch.cuda.synchronize()
    # headline: exactly K timed steps
    gk = rig.capture(args.rows, K)
    ms = max_over_ranks(time_graph(gk), dist, "cuda")
    us = ms * 1e3 / K
    bytes_launch = shape.launch_bytes(args.rows, args.rows)
    rig.check()
    del gw, gk

    e2e = None
    if not args.no_e2e:
        # end to end through the public API with host buffers: per step, copy this
        # step's inputs from pinned host memory, launch, read the outputs back
        H, Hv = shape.hidden, shape.num_v_heads
        Bi = args.rows * H * 2 * 2 + args.rows * 4
        Bo = args.rows * Hv * shape.head_v_dim * 2 + args.rows * H * 2
        hx = torch.empty(args.rows, H, dtype=torch.bfloat16).pin_memory()
        hr = torch.empty(args.rows, H, dtype=torch.bfloat16).pin_memory()
        hi = torch.randperm(shape.num_slots - 1)[:args.rows].add(1).to(torch.int32).pin_memory()
        hx.copy_(torch.randn(args.rows, H).to(torch.bfloat16))
        hr.copy_(torch.randn(args.rows, H).to(torch.bfloat16))
        hc = torch.empty(args.rows, Hv * shape.head_v_dim, dtype=torch.bfloat16).pin_memory()
        ho = torch.empty(args.rows, H, dtype=torch.bfloat16).pin_memory()
        dx, dr, di = (torch.empty_like(hx, device="cuda"), torch.empty_like(hr, device="cuda"),
                      torch.empty_like(hi, device="cuda"))
        dc, do = torch.empty_like(hc, device="cuda"), torch.empty_like(ho, device="cuda")

        def e2e_step(k):
            dx.copy_(hx, non_blocking=True)
            dr.copy_(hr, non_blocking=True)
            di.copy_(hi, non_blocking=True)
            rig.layer.step(dx, dr, rig.copies[k % rig.ncopy], di, rig.conv, rig.ssm, dc, do,
                           weights_struct=rig.wstructs[k % rig.ncopy])
            hc.copy_(dc, non_blocking=True)
            ho.copy_(do, non_blocking=True)

        for k in range(max(3, Wm)):
            e2e_step(k)
        torch.cuda.synchronize()
        st0 = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st0)
        for k in range(K):
            e2e_step(k)
        e1.record(st0)
        torch.cuda.synchronize()
        rig.check()
        # host cost of one call through the binding (argument marshalling, the
        # C entry point and the launch enqueue; the GPU runs behind)
        h0 = time.perf_counter()
        for k in range(K):
            rig.layer.step(dx, dr, rig.copies[k % rig.ncopy], di, rig.conv, rig.ssm, dc, do,
                           weights_struct=rig.wstructs[k % rig.ncopy])
        host_us = (time.perf_counter() - h0) * 1e6 / K
        torch.cuda.synchronize()
        rig.check()
        e2e = {"value": round(e0.elapsed_time(e1) * 1e3 / K, 3), "unit": "µs/launch", "h2d_bytes_per_step": Bi,
               "d2h_bytes_per_step": Bo, "host_us_per_call": round(host_us, 2),
               "how": "eager gdn_decode_step via the Python binding with pinned-host copies in and out each step"}
    n_ctas, engine = rig.layer.launch_info(args.rows)
    ncopy, wbytes = rig.ncopy, rig.wbytes

    # per-width tables, one workload at a time (outside the headline timed region)
    tables = {}
    widths = [int(v) for v in args.widths.split(",") if v]
    for name in [t for t in args.tables.split(",") if t]:
        rec = TABLES[name]
        if name != args.workload or rig is None:
            rig = None
            torch.cuda.empty_cache()
            tshape = WL.SHAPES[rec.get("shape", name)].with_(max_rows=rec.get("max_rows", 16))
            rig = Rig(tshape, g, l2, args.engine, rec.get("min_copies", 4), rec.get("out_proj", False))
        if "verify" in rec:
            vt = {}
            for S, T in rec["verify"]:
                gg = rig.capture_verify(S, T, 100)
                times = []
                t_end = time.time() + 0.3
                while time.time() < t_end or len(times) < 5:
                    times.append(time_graph(gg) * 10.0)
                times.sort()
                u = times[len(times) // 2]
                b = rig.shape.verify_bytes(S, T)
                vt[f"{S}x{T}"] = {"us": round(u, 3), "GBps": round(b / u / 1e3, 1),
                                  "frac_of_" + peak_kind: round(b / u / 1e3 / peak, 4), "bytes": b,
                                  "rows": S * T, "launches": -(-S // (16 // T))}
                del gg
            rig.check()
            tables[name] = {"copies": rig.ncopy, "verify": vt}
            rig = None
            continue
        ws = rec["widths"] if name != args.workload else sorted(set(rec["widths"]) | set(widths))
        tables[name] = {"copies": rig.ncopy, "first_layer": rec.get("first_layer", False),
                        "pad_fraction": rec.get("pad", 0.0),
                        "widths": width_table(rig, ws, rec.get("pad", 0.0), rec.get("first_layer", False))}
        rig = None
    clk = clocks.stop()

    result = {
        "metric": METRIC, "value": round(us, 3), "unit": "µs/launch", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None,
        "dtype": shape.qkvz_format + " weights, f32 math, " + shape.ssm_dtype + " state",
        "data": "synthetic (seeded random weights and states of the layer's shapes)",
        "config": {"workload": f"{shape.name}: H={shape.hidden} Hk={shape.num_k_heads} Hv={shape.num_v_heads} "
                               f"dk=dv={shape.head_k_dim} slots={shape.num_slots} {shape.ssm_dtype} state, "
                               f"{shape.qkvz_format} in_proj_qkvz",
                   "rows": args.rows, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: weights rotated over {ncopy} copies "
                         f"({ncopy * wbytes / 1e6:.0f} MB vs {l2 / 1e6:.0f} MB L2), fresh slots per launch",
                   "timing": "CUDA graph of K launches, CUDA events on the launching stream",
                   "grid": n_ctas, "engine": engine,
                   "launch": "persistent grid, one CTA per SM; programmatic dependent launch between steps"},
        "achieved_GBps": round(bytes_launch / us / 1e3, 1),
        "frac_of_nominal_8TBps": round(bytes_launch / us / 1e3 / NOMINAL_HBM_GBS, 4),
        "widths": tables,
        "roofline": {"bound": "hbm", "achieved": round(bytes_launch / us / 1e3, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(bytes_launch / us / 1e3 / peak, 4),
                     "traffic": measured_traffic(args.workload, args.rows), "peak_kind": peak_kind,
                     "bytes_per_launch": bytes_launch},
        "e2e": e2e,
        "gpu_launches": K,
        "clocks": clk,
        "context": PAGES_NOTE,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        d, cores = run_cpu_baseline(args)
        result["cpu_baseline"] = {"value": round(d["us_per_step"], 1), "unit": "µs/launch", "cores": cores,
                                  "kind": "oracle", "sample": f"{d['n']} oracle steps of the same workload "
                                  f"({args.rows} rows) in {d['seconds']:.1f} s, float64 numpy"}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gated_deltanet_layer_gb300 import workloads as WL
    shape = WL.SHAPES[args.workload]
    # warm-up steps are not timed
    run_cpu_baseline(args, steps=max(1, args.warmup))
    d, cores = run_cpu_baseline(args, steps=args.steps)
    v = round(d["us_per_step"], 1)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "µs/launch", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{shape.name}", "rows": args.rows},
        "cpu_baseline": {"value": v, "unit": "µs/launch", "cores": cores, "kind": "oracle",
                         "sample": f"{d['n']} oracle steps ({args.rows} rows) in {d['seconds']:.1f} s"},
        "e2e": {"value": v, "unit": "µs/launch", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    args = parse()
    if args.cpu_child:
        cpu_child(args)
    elif args.impl == "reference":
        reference(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
