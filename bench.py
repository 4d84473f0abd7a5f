#!/usr/bin/env python
"""Benchmark of the group-affine quantized projection (libaffqmm) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line on rank 0.  A step is one pass of the projection path
over one batch of synthetic input with the weights resident in HBM:

  gate_up_decode (default)  M=1, K=3840, N=30720 (stacked gate/up), 4-bit g64
  decode_step               a 60-layer decoder's projections + tied head, M=1
  prompt_chunk              M=128 through one layer's four projection shapes
  prompt_step               M=128 through all 60 layers' projections (the aggregate)
  lane_sweep                M in {2,4,8,16} at 4-bit g64 and M=16 at 8b/3b/2b
  tiny                      M=1, K=256, N=512, 4-bit g64
  embed_rows                4096 scaled embedding rows gathered from the tied head's table
                            (its row-contiguous copy)
  embed_rows_blocks         the same gather read from the packed blocks themselves

`value` is packed-weight bytes (codes + bf16 scales + biases) per second for
the decode workloads and TFLOP/s for the prompt chunk.  Weight copies rotate
so that the bytes touched between two reads of one copy exceed the 129 MB L2.
Steps are replayed from CUDA graphs and timed with CUDA events on the stream
that launches them.  `e2e` times the same steps end to end with host
buffers: a one-projection step is one call of the C ABI's host-buffer entry
point (affqmm_run_host: x uploaded from pinned host memory, the projection,
y read back); a step of several projections, the exact-codes form and the
embedding gather upload the step's inputs, run it through the Python API
and read its outputs back.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload on the host cores.  Under torchrun every rank runs an
independent replica (the path needs no exchange) and rank 0 reports the
aggregate over ranks with the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "affine-4bit qmm packed-weight GB/s vs HBM peak (M=1..16); TFLOP/s at M=128"
L2_BYTES = 129 * 10 ** 6
KERNEL_SOURCES = ["group_affine_bit_gb300/csrc/decode.cu", "group_affine_bit_gb300/csrc/prompt.cu",
                  "group_affine_bit_gb300/csrc/embed.cu",
                  "group_affine_bit_gb300/csrc/affqmm_format.cuh", "group_affine_bit_gb300/csrc/affqmm_tc.cuh",
                  "group_affine_bit_gb300/csrc/affqmm_async.cuh",
                  "group_affine_bit_gb300/csrc/plan.cu"]   # the host planner: how a launch is cut


# ----------------------------------------------------------------------------- setup
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: per workload)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="gate_up_decode",
                    choices=["gate_up_decode", "decode_step", "prompt_chunk", "prompt_step", "lane_sweep", "tiny",
                             "embed_rows", "embed_rows_blocks", "gate_up_exact"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="no nvidia-smi sampling (for runs under a profiler)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle sample")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_max(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def aggregate(per_rank_units: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank processed the same units."""
    return per_rank_units * world / max_seconds


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


SHARED_KERNEL_HEADERS = KERNEL_SOURCES[3:]


def source_digest(kernel: str | None = None) -> str:
    """Hash of the kernel sources: of one kernel ("decode", "prompt", "embed":
    its .cu, the shared device headers and the host planner that cuts its
    launches), or of all of them."""
    h = hashlib.sha256()
    rels = KERNEL_SOURCES if kernel is None else [f"group_affine_bit_gb300/csrc/{kernel}.cu", *SHARED_KERNEL_HEADERS]
    for rel in rels:
        p = os.path.join(ROOT, rel)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def committed_traffic(key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(key)
    if not d or d.get("src_digest") != source_digest(key.split()[0]):
        return None
    return d.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the GPU is busy."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.2)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[2]), smax=float(parts[3]), power=float(parts[4]),
                                 hw=parts[6], hwth=parts[7], swth=parts[8], swpc=parts[9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r["power"] > 0.3 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwth", "hw_thermal_slowdown"),
                              ("swth", "sw_thermal_slowdown"), ("swpc", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy),
                "power_w_max": max(r["power"] for r in rows)}


# ----------------------------------------------------------------------------- workloads
def copies_for(bytes_per_copy: int) -> int:
    """Rotating copies so that more than twice the L2 is touched between two
    reads of one copy."""
    return max(4, math.ceil(2 * L2_BYTES / max(1, bytes_per_copy)))


class Case:
    """One resident projection: `copies` packed copies of one seeded affine
    table (the same values), its activations and its output."""

    def __init__(self, api, synth, label, bits, group, M, N, K, seed, copies, device):
        import torch
        self.api = api
        self.label, self.bits, self.group, self.M, self.N, self.K, self.seed = label, bits, group, M, N, K, seed
        self.copies = copies
        g = synth.generator(seed, device)
        codes, s, b = synth.affine_table(bits, group, N, K, g, device)
        self.ws = [api.pack(codes, s, b, bits, group) for _ in range(copies)]
        del codes, s, b
        self.x = synth.activations(M, K, g, device)
        self.y = torch.empty(M, N, dtype=torch.bfloat16, device=device)

    exact = False  # the exact-codes form (affqmm_run_exact) instead of rounded weights

    def run(self, i: int, workspace):
        if self.exact:
            self.api.run_exact(self.ws[i % self.copies], self.x, y=self.y, workspace=workspace)
        else:
            self.api.run(self.ws[i % self.copies], self.x, y=self.y, workspace=workspace)

    @property
    def packed_bytes(self) -> int:   # codes + bf16 scale and bias per group
        return self.N * self.K * self.bits // 8 + 4 * self.N * self.K // self.group

    @property
    def algorithmic_bytes(self) -> int:
        return self.packed_bytes + 2 * self.M * self.K + 2 * self.M * self.N

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def launches(self) -> int:
        """Launches of the dominant kernel (decode or prompt kernel)."""
        return 1 if self.M <= 16 else -(-self.M // 128)

    @property
    def kernels(self) -> int:
        """All of the library's kernel launches: a prompt chunk also launches its merge kernel."""
        return 1 if self.M <= 16 else 2 * (-(-self.M // 128))

    def oracle_shape(self):
        return dict(bits=self.bits, group=self.group, M=self.M, N=self.N, K=self.K, seed=self.seed)


class Workload:
    """A step = every case run once, in order, on one stream."""
    name = ""
    unit = "GB/s"
    default_steps = 3000

    def __init__(self, api, synth, device):
        self.api = api
        self.workspace = api.Workspace(device)
        self.cases = self.make_cases(api, synth, device)
        self.x_arena = self.y_arena = None
        if len(self.cases) > 1:
            self._arenas(device)

    def _arenas(self, device):
        """A step's activations and outputs in one contiguous buffer each (the
        cases' x and y become views of them, 16-byte aligned, same values), as
        an engine keeps a step's activations: the step's inputs go up in one
        copy and its outputs come back in one."""
        import torch

        def carve(shapes):
            offs, n = [], 0
            for rows, cols in shapes:
                offs.append(n)
                n += -(-rows * cols // 8) * 8          # 16-byte aligned views
            return offs, n
        xo, xn = carve([(c.M, c.K) for c in self.cases])
        yo, yn = carve([(c.M, c.N) for c in self.cases])
        self.x_arena = torch.empty(xn, dtype=torch.bfloat16, device=device)
        self.y_arena = torch.empty(yn, dtype=torch.bfloat16, device=device)
        for c, a, b in zip(self.cases, xo, yo):
            xv = self.x_arena[a:a + c.M * c.K].view(c.M, c.K)
            xv.copy_(c.x)
            c.x = xv
            c.y = self.y_arena[b:b + c.M * c.N].view(c.M, c.N)

    def make_cases(self, api, synth, device):
        raise NotImplementedError

    def step(self, i: int):
        for c in self.cases:
            c.run(i, self.workspace)

    @property
    def launches_per_step(self) -> int:
        return sum(c.launches for c in self.cases)

    @property
    def kernels_per_step(self) -> int:
        return sum(c.kernels for c in self.cases)

    @property
    def units_per_step(self) -> float:
        """Units of the metric: packed-weight bytes, or FLOPs for prompt rows."""
        if self.unit == "TFLOP/s":
            return float(sum(c.flops for c in self.cases))
        return float(sum(c.packed_bytes for c in self.cases))

    @property
    def scale(self) -> float:
        return 1e12 if self.unit == "TFLOP/s" else 1e9

    def roofline_info(self):
        c0 = self.cases[0]
        if self.unit == "TFLOP/s":
            return dict(kernel=f"prompt_kernel<{c0.bits},{c0.group}>", bound="tensor",
                        units_per_step=float(sum(c.flops for c in self.cases)), unit="TFLOP/s",
                        traffic_key=f"prompt {self.name}")
        nb = 2 if max(c.M for c in self.cases) > 8 else 1
        exact = "true" if getattr(c0, "exact", False) else "false"
        return dict(kernel=f"decode_kernel<{c0.bits},{c0.group},{nb},{exact}>", bound="hbm",
                    units_per_step=float(sum(c.algorithmic_bytes for c in self.cases)), unit="GB/s",
                    traffic_key=f"decode {self.name}")

    def l2_note(self) -> str:
        touched = sum(c.packed_bytes for c in self.cases)
        rot = max(c.copies for c in self.cases)
        if rot > 1:
            return (f"inputs larger than L2: {rot} rotating weight copies per case "
                    f"({rot * touched / 1e6:.0f} MB touched per rotation > 129 MB L2)")
        return f"inputs larger than L2: {touched / 1e6:.0f} MB of distinct packed weights per step > 129 MB L2"

    def describe(self) -> str:
        return self.name

    def config(self):
        return {"workload": self.describe(), "cases": [
            f"{c.label}: M={c.M} N={c.N} K={c.K} {c.bits}-bit g{c.group} seed {c.seed}" for c in self.cases],
            "l2": self.l2_note(), "parallelism": "replicas"}

    def e2e_io(self):
        if self.x_arena is not None:
            return [self.x_arena], [self.y_arena]
        return [c.x for c in self.cases], [c.y for c in self.cases]

    def oracle_shape(self):
        return self.cases[0].oracle_shape()


class GateUpDecode(Workload):
    name = "gate_up_decode"

    def make_cases(self, api, synth, device, shape=None):
        c = shape or synth.GATE_UP_DECODE
        one = c["N"] * c["K"] * c["bits"] // 8 + 4 * c["N"] * c["K"] // c["group"]
        return [Case(api, synth, self.name, c["bits"], c["group"], c["M"], c["N"], c["K"], c["seed"],
                     copies_for(one), device)]

    def describe(self):
        c = self.cases[0]
        return f"{self.name}: M={c.M} K={c.K} N={c.N} {c.bits}-bit group {c.group}"


class GateUpExact(GateUpDecode):
    """The gate/up decode shape through the exact-codes form (the pages' lane
    projection: exact codes, group sums of x)."""
    name = "gate_up_exact"

    def make_cases(self, api, synth, device, shape=None):
        cases = super().make_cases(api, synth, device, shape)
        for c in cases:
            c.exact = True
        return cases


class Tiny(GateUpDecode):
    name = "tiny"

    def make_cases(self, api, synth, device):
        return super().make_cases(api, synth, device, synth.TINY)


class DecodeStep(Workload):
    """A 60-layer decoder's projections (qkv, o, gate/up, down) and the tied
    head, M = 1: every weight distinct, about 16 GB read per step."""
    name = "decode_step"
    default_steps = 200

    def make_cases(self, api, synth, device):
        bits, group, seed = 4, 64, synth.DECODE_STEP_SEED
        cases = []
        for layer in range(synth.N_LAYERS):
            for j, (label, (N, K)) in enumerate(synth.DECODER_LAYER_SHAPES.items()):
                cases.append(Case(api, synth, f"L{layer}.{label}", bits, group, 1, N, K,
                                  synth.step_seed(seed, layer, j), 1, device))
        N, K = synth.HEAD_SHAPE
        cases.append(Case(api, synth, "head", bits, group, 1, N, K, synth.step_seed(seed, synth.N_LAYERS, 0), 1,
                          device))
        return cases

    def describe(self):
        return (f"{self.name}: {synth_n_layers(self)} layers x (qkv, o, gate_up, down) + tied head, M=1, "
                f"hidden 5376, 4-bit group 64, {len(self.cases)} projections")

    def config(self):
        d = super().config()
        d["cases"] = d["cases"][:4] + [d["cases"][-1], f"... {len(self.cases)} projections in all"]
        d["packed_gb_per_step"] = round(self.units_per_step / 1e9, 3)
        return d

    def oracle_shape(self):
        return self.cases[2].oracle_shape()   # a gate/up projection


def synth_n_layers(wl) -> int:
    return (len(wl.cases) - 1) // 4


class PromptChunk(Workload):
    """M = 128 activation rows through one decoder layer's four projections."""
    name = "prompt_chunk"
    unit = "TFLOP/s"
    default_steps = 500

    def make_cases(self, api, synth, device):
        c = synth.PROMPT_CHUNK
        return [Case(api, synth, label, c["bits"], c["group"], c["M"], N, K, synth.step_seed(c["seed"], 0, j), 1,
                     device) for j, (label, (N, K)) in enumerate(synth.DECODER_LAYER_SHAPES.items())]

    def describe(self):
        return f"{self.name}: M=128 through qkv, o, gate_up, down (hidden 5376), 4-bit group 64"


class PromptStep(Workload):
    """M = 128 activation rows through all 60 layers' four projections (every
    weight distinct, 15.4 GB a step): the aggregate rate of a prompt chunk's
    forward over the decoder."""
    name = "prompt_step"
    unit = "TFLOP/s"
    default_steps = 100

    def make_cases(self, api, synth, device):
        c = synth.PROMPT_CHUNK
        return [Case(api, synth, f"L{layer}.{label}", c["bits"], c["group"], c["M"], N, K,
                     synth.step_seed(c["seed"], layer, j), 1, device)
                for layer in range(synth.N_LAYERS)
                for j, (label, (N, K)) in enumerate(synth.DECODER_LAYER_SHAPES.items())]

    def describe(self):
        return (f"{self.name}: M=128 through {len(self.cases) // 4} layers x (qkv, o, gate_up, down), hidden 5376, "
                f"4-bit group 64, {len(self.cases)} projections")

    def config(self):
        d = super().config()
        d["cases"] = d["cases"][:4] + [f"... {len(self.cases)} projections in all"]
        d["packed_gb_per_step"] = round(sum(c.packed_bytes for c in self.cases) / 1e9, 3)
        return d


class LaneSweep(Workload):
    """M in {2, 4, 8, 16} at 4-bit g64 and M = 16 at 8-bit g32, 3-bit g64 and
    2-bit g128 on K = 3840, N = 15360."""
    name = "lane_sweep"
    default_steps = 1000

    def make_cases(self, api, synth, device):
        c = synth.SWEEP_SHAPE
        out = []
        for j, (M, bits, group) in enumerate(synth.SWEEP_CASES):
            one = c["N"] * c["K"] * bits // 8 + 4 * c["N"] * c["K"] // group
            out.append(Case(api, synth, f"M{M} {bits}b g{group}", bits, group, M, c["N"], c["K"], c["seed"] + j,
                            copies_for(one), device))
        return out

    def describe(self):
        return f"{self.name}: K=3840 N=15360, (M, bits, group) in {[(c.M, c.bits, c.group) for c in self.cases]}"


class EmbedRows(Workload):
    """Scaled embedding rows: 4096 token ids gathered from the tied head's table
    (262144 x 5376, 4-bit g64) times bf16(sqrt(5376)), read from the table's
    row-contiguous copy (affqmm_embed_rows_copy; the copy is made once, before
    timing, like the packing).  Bytes = the gathered rows' packed bytes + the
    ids + the bf16 output.  Steps rotate over 16 id sets and 4 output buffers
    so that neither the rows nor the output stay in L2 between steps."""
    name = "embed_rows"
    default_steps = 500
    T = 4096
    ID_SETS = 16
    OUT_SETS = 4
    from_copy = True

    def make_cases(self, api, synth, device):
        import torch
        N, K = synth.HEAD_SHAPE
        g = synth.generator(synth.EMBED_SEED, device)
        codes, s, b = synth.affine_table(4, 64, N, K, g, device)
        self.w = api.pack(codes, s, b, 4, 64)
        del codes, s, b
        self.rows = api.pack_rows(self.w) if self.from_copy else None
        self.ids = [torch.randint(0, N, (self.T,), generator=g, device=device, dtype=torch.int32)
                    for _ in range(self.ID_SETS)]
        self.outs = [torch.empty(self.T, K, dtype=torch.bfloat16, device=device) for _ in range(self.OUT_SETS)]
        self.N, self.K = N, K
        return []

    def gather(self, ids, out):
        if self.from_copy:
            self.api.embed_rows_copy(self.w, self.rows, ids, math.sqrt(5376.0), out=out)
        else:
            self.api.embed_rows(self.w, ids, math.sqrt(5376.0), out=out)

    def step(self, i: int):
        self.gather(self.ids[i % self.ID_SETS], self.outs[i % self.OUT_SETS])

    def step_e2e(self, i: int):
        """The end-to-end step: the ids uploaded to and the rows read back from
        the first buffers."""
        self.gather(self.ids[0], self.outs[0])

    launches_per_step = 1
    kernels_per_step = 1

    @property
    def packed_row_bytes(self) -> int:
        return self.K * 4 // 8 + 4 * self.K // 64

    @property
    def units_per_step(self) -> float:
        return float(self.T * (self.packed_row_bytes + 4 + 2 * self.K))

    def roofline_info(self):
        kernel = f"embed_kernel<4,64,{'true' if self.from_copy else 'false'}>"
        return dict(kernel=kernel, bound="hbm", units_per_step=self.units_per_step, unit="GB/s",
                    traffic_key=f"embed {self.name}")

    def l2_note(self) -> str:
        rot = self.ID_SETS * self.T * self.packed_row_bytes + self.OUT_SETS * self.T * self.K * 2
        return (f"inputs larger than L2: steps rotate over {self.ID_SETS} sets of {self.T} random rows of a 1.5 GB "
                f"table and {self.OUT_SETS} output buffers ({rot / 1e6:.0f} MB touched per rotation > 129 MB L2)")

    def describe(self):
        src = "its row-contiguous copy" if self.from_copy else "the packed blocks"
        return (f"{self.name}: T={self.T} ids into {self.N}x{self.K} 4-bit g64 (read from {src}), "
                f"scale bf16(sqrt(5376))")

    def config(self):
        return {"workload": self.describe(), "T": self.T, "N": self.N, "K": self.K, "bits": 4, "group": 64,
                "l2": self.l2_note(), "parallelism": "replicas"}

    def e2e_io(self):
        return [self.ids[0]], [self.outs[0]]


class EmbedRowsBlocks(EmbedRows):
    """The same gather read from the packed blocks (the tied head's own layout, no copy)."""
    name = "embed_rows_blocks"
    from_copy = False


WORKLOADS = {"gate_up_decode": GateUpDecode, "decode_step": DecodeStep, "prompt_chunk": PromptChunk,
             "prompt_step": PromptStep,
             "lane_sweep": LaneSweep, "tiny": Tiny, "embed_rows": EmbedRows, "embed_rows_blocks": EmbedRowsBlocks,
             "gate_up_exact": GateUpExact}


# ----------------------------------------------------------------------------- timing
def graph_of(fn, first: int, count: int):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(first, first + count):
            fn(i)
    return g


def time_steps(wl, steps: int, warmup: int, dist, device):
    """Device time of exactly `steps` steps replayed from CUDA graphs (at most
    about 2000 launches per graph)."""
    import torch
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        for i in range(warmup):       # eager warm-up (also initializes the library)
            wl.step(i)
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize(device)
    chunk = max(1, min(steps, 2000 // max(1, wl.launches_per_step)))
    full = graph_of(wl.step, 0, chunk)
    rest = graph_of(wl.step, 0, steps % chunk) if steps % chunk else None
    for _ in range(max(1, warmup // chunk)):
        full.replay()
    torch.cuda.synchronize(device)
    stream = torch.cuda.current_stream(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(device)
    # Keep the GPU busy (a spin of ~0.1 ms) while the host enqueues the start
    # event and the graphs, so that the timed region starts when the GPU
    # reaches the work, not when the host finishes submitting it.
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(200_000)
    e0.record(stream)
    for _ in range(steps // chunk):
        full.replay()
    if rest is not None:
        rest.replay()
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist)
    seconds = e0.elapsed_time(e1) * 1e-3
    return seconds, (full, rest, chunk)


def time_cases(wl, device, launches: int = 40, replays: int = 5):
    """Rate of each case of a few-case workload timed alone (graph replay of
    `launches` launches over its rotating copies, CUDA events): the per-case
    figures beside the step's aggregate."""
    import torch
    out = {}
    stream = torch.cuda.current_stream(device)
    for c in wl.cases:
        g = graph_of(lambda i, c=c: c.run(i, wl.workspace), 0, launches)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(device)
        sec = e0.elapsed_time(e1) * 1e-3 / (launches * replays)
        units = c.flops if wl.unit == "TFLOP/s" else c.packed_bytes
        out[c.label] = round(units / sec / wl.scale, 1)
        del g
    return out


def sustain_for_clocks(graphs, device, seconds: float = 1.0):
    """Replay the timed graphs for about `seconds` so the clock sampler sees
    the same load when the timed region itself is too short to sample."""
    import torch
    full, rest, chunk = graphs
    t0 = time.time()
    while time.time() - t0 < seconds:
        full.replay()
        torch.cuda.synchronize(device)


class HostCalls:
    """One step of a workload as C calls of affqmm_run_host with host buffers:
    per projection, x is uploaded from pinned host memory, the projection runs
    and y is read back into pinned host memory -- one call of the C ABI, its
    arguments marshalled once (ctypes, no per-call Python checks)."""

    def __init__(self, wl, h_in, h_out, stream_ptr: int):
        import ctypes
        api = wl.api
        L = api.lib()
        self.fn = L.affqmm_run_host
        self.steps = []   # per weight copy: the argument tuples of every case
        need = max(api.workspace_bytes(c.ws[0], c.M) for c in wl.cases)
        buf = wl.workspace.get(need)
        ws_ptr, ws_n = (buf.data_ptr() if need else None), buf.numel()
        self._keep = []
        copies = max(c.copies for c in wl.cases)
        for i in range(copies):
            calls = []
            for c, hx, hy in zip(wl.cases, h_in, h_out):
                cw = c.ws[i % c.copies].cstruct()
                self._keep.append(cw)
                calls.append((ctypes.byref(cw), hx.data_ptr(), c.M, hy.data_ptr(), c.x.data_ptr(), c.y.data_ptr(),
                              ws_ptr, ws_n, stream_ptr))
            self.steps.append(calls)

    def step(self, i: int):
        fn = self.fn
        for args in self.steps[i % len(self.steps)]:
            rc = fn(*args)
            if rc:
                raise RuntimeError(f"affqmm_run_host failed with status {rc}")


def time_e2e(wl, steps: int, device):
    """Same steps end to end with host buffers: the step's activations uploaded
    from pinned host memory at its start and its outputs read back to pinned
    host memory at its end, inside the timed region.  A step of one projection
    is one call of the C ABI's host-buffer entry point (affqmm_run_host: upload,
    projection, read-back).  A step of several projections uploads all of its
    inputs, runs its projections through the Python API (affqmm_run) and reads
    all of its outputs back: one host call per projection would put two copies
    between every pair of launches (about 14 us more per projection on the
    GPU).  The exact-codes form and the embedding gather, which have no
    host-buffer call, take the second form too."""
    import torch
    ins, outs = wl.e2e_io()
    h_in = [t.detach().cpu().pin_memory() for t in ins]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = sum(t.numel() * t.element_size() for t in h_out)
    stream = torch.cuda.current_stream(device)
    cases = getattr(wl, "cases", [])
    host = None
    if len(cases) == 1 and not getattr(cases[0], "exact", False):
        host = HostCalls(wl, h_in, h_out, int(stream.cuda_stream))
    for i in range(3):
        if host is not None:
            host.step(i)
        else:
            wl.step(i)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(steps):
        if host is not None:
            host.step(i)
            continue
        for d, h in zip(ins, h_in):
            d.copy_(h, non_blocking=True)
        getattr(wl, "step_e2e", wl.step)(i)
        for d, h in zip(outs, h_out):
            h.copy_(d, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    via = ("affqmm_run_host (C ABI, host buffers)" if host is not None
           else "step inputs uploaded, Python API (affqmm_run), step outputs read back (torch copies)")
    return max(wall, e0.elapsed_time(e1) * 1e-3), bi, bo, via


# ----------------------------------------------------------------------------- oracle
class OracleSample:
    """The CPU oracle on a bounded sample of a workload: whole output rows of
    one of its projections (same seed, same values), threaded over rows on
    all host cores.  Rate = packed-weight bytes (GB/s) or FLOPs (TFLOP/s) of
    the sampled rows per second."""

    def __init__(self, shape: dict, unit: str):
        import oracle
        from group_affine_bit_gb300 import synth
        self.orc = oracle.load()
        self.unit = unit
        self.bits, self.group = shape["bits"], shape["group"]
        self.M, self.N, self.K = shape["M"], shape["N"], shape["K"]
        x, codes, s, b = synth.problem(self.bits, self.group, self.M, self.N, self.K, shape["seed"])
        self.xb, self.cb = synth.bits_u16(x), codes.numpy()
        self.sb, self.bb = synth.bits_u16(s), synth.bits_u16(b)
        self.threads = host_cores()
        self.embed = bool(shape.get("embed"))
        self.exact = bool(shape.get("exact"))
        if self.exact:
            self.threads = 1  # the exact-codes oracle is not threaded
        if self.embed:
            self.threads = 1
            self.embed_scale = int(synth.bits_u16(torch_bf16_scalar(math.sqrt(self.K)))[0])

    def units(self, rows: int) -> float:
        if self.embed:
            return rows * (self.K * self.bits // 8 + 4 * self.K // self.group + 4 + 2 * self.K) / 1e9
        if self.unit == "TFLOP/s":
            return 2.0 * self.M * rows * self.K / 1e12
        return (rows * self.K * self.bits // 8 + 4 * rows * self.K // self.group) / 1e9

    def run(self, rows: int) -> float:
        t0 = time.perf_counter()
        if self.embed:   # rows of the table gathered (one thread: the oracle's gather is not threaded)
            import numpy as np
            ids = np.arange(rows, dtype=np.int32)
            self.orc.embed_rows(self.bits, self.group, self.cb[:rows], self.sb[:rows], self.bb[:rows], ids,
                                self.embed_scale)
        elif self.exact:
            self.orc.qmm_groupsum(self.bits, self.group, self.xb, self.cb[:rows], self.sb[:rows], self.bb[:rows])
        else:
            self.orc.qmm(self.bits, self.group, self.xb, self.cb[:rows], self.sb[:rows], self.bb[:rows],
                         nthreads=self.threads)
        return time.perf_counter() - t0

    def rows_for(self, seconds: float) -> int:
        n = min(self.N, 64)
        dt = max(self.run(n), 1e-5)
        return int(max(1, min(self.N, n * seconds / dt)))

    def describe(self, rows: int, reps: int) -> str:
        if self.embed:
            return (f"{reps} x {rows} gathered rows of K={self.K}, {self.bits}-bit g{self.group} times a bf16 "
                    f"scale; oracle on one thread")
        if self.exact:
            return (f"{reps} x {rows} of {self.N} output rows of one projection of the workload (M={self.M}, "
                    f"K={self.K}, {self.bits}-bit g{self.group}); float64 exact-codes oracle on one thread")
        how = f"threaded over rows on {self.threads} cores" if self.threads > 1 else "on one thread"
        return (f"{reps} x {rows} of {self.N} output rows of one projection of the workload (M={self.M}, "
                f"K={self.K}, {self.bits}-bit g{self.group}); float64 oracle {how}")

    def rate(self, seconds: float):
        rows = self.rows_for(seconds)
        reps, total = 0, 0.0
        while total < seconds or reps == 0:
            total += self.run(rows)
            reps += 1
        return self.units(rows) * reps / total, self.describe(rows, reps), total


WORKLOAD_ORACLE_SHAPES = {   # the projection each workload's oracle sample takes rows of
    "gate_up_decode": lambda s: s.GATE_UP_DECODE,
    "tiny": lambda s: s.TINY,
    "decode_step": lambda s: dict(bits=4, group=64, M=1, N=s.DECODER_LAYER_SHAPES["gate_up"][0],
                                  K=s.DECODER_LAYER_SHAPES["gate_up"][1], seed=s.step_seed(s.DECODE_STEP_SEED, 0, 2)),
    "prompt_chunk": lambda s: dict(bits=4, group=64, M=128, N=s.DECODER_LAYER_SHAPES["qkv"][0],
                                   K=s.DECODER_LAYER_SHAPES["qkv"][1], seed=s.step_seed(s.PROMPT_CHUNK["seed"], 0, 0)),
    "prompt_step": lambda s: dict(bits=4, group=64, M=128, N=s.DECODER_LAYER_SHAPES["qkv"][0],
                                  K=s.DECODER_LAYER_SHAPES["qkv"][1], seed=s.step_seed(s.PROMPT_CHUNK["seed"], 0, 0)),
    "lane_sweep": lambda s: dict(bits=4, group=64, M=2, N=s.SWEEP_SHAPE["N"], K=s.SWEEP_SHAPE["K"],
                                 seed=s.SWEEP_SHAPE["seed"]),
    "embed_rows": lambda s: dict(bits=4, group=64, M=1, N=4096, K=s.HEAD_SHAPE[1], seed=s.EMBED_SEED, embed=True),
    "embed_rows_blocks": lambda s: dict(bits=4, group=64, M=1, N=4096, K=s.HEAD_SHAPE[1], seed=s.EMBED_SEED,
                                        embed=True),
    "gate_up_exact": lambda s: dict(s.GATE_UP_DECODE, exact=True),
}


def torch_bf16_scalar(v: float):
    import torch
    return torch.tensor([v], dtype=torch.float32).to(torch.bfloat16)


def workload_unit(name: str) -> str:
    return WORKLOADS[name].unit


# ----------------------------------------------------------------------------- main
def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: rank 0 only; each step is one
    bounded sample of the workload."""
    if rank != 0:
        return 0
    from group_affine_bit_gb300 import synth
    unit = workload_unit(args.workload)
    steps = args.steps if args.steps is not None else 20
    smp = OracleSample(WORKLOAD_ORACLE_SHAPES[args.workload](synth), unit)
    per_step = max(0.02, args.cpu_seconds / max(1, steps + args.warmup))
    rows = smp.rows_for(per_step)
    for _ in range(args.warmup):
        smp.run(rows)
    total = 0.0
    for _ in range(steps):
        total += smp.run(rows)
    value = smp.units(rows) * steps / total
    sample = smp.describe(rows, 1) + " per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": 1,
            "steps": steps, "warmup": args.warmup, "ms_per_step": total / max(1, steps) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, "sample": sample},
            "cpu_baseline": {"value": value, "unit": unit, "cores": smp.threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    from group_affine_bit_gb300 import api, build, synth
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    if rank == 0:
        build.build()
    barrier(dist)
    api.lib()

    wl = WORKLOADS[args.workload](api, synth, device)
    steps = args.steps if args.steps is not None else wl.default_steps
    warmup = max(3, args.warmup)

    sampler = ClockSampler(local) if rank == 0 and not args.no_clocks else None
    if sampler:
        sampler.start()
    seconds, graphs = time_steps(wl, steps, warmup, dist, device)
    clocks = None
    if sampler:
        if seconds < 1.0:
            sustain_for_clocks(graphs, device, 1.0)
        clocks = sampler.stop()
    t_max = reduce_max(dist, seconds, device)
    value = aggregate(wl.units_per_step * steps, world, t_max) / wl.scale

    info = wl.roofline_info()
    peaks = measured_peaks()
    launches = steps * wl.launches_per_step
    per_launch_s = seconds / launches
    units_per_launch = info["units_per_step"] / wl.launches_per_step
    if info["bound"] == "hbm":
        achieved = units_per_launch / per_launch_s / 1e9
        peak, peak_name = peaks["hbm_gbs"], "hbm_gbs (copy)"
    else:
        achieved = units_per_launch / per_launch_s / 1e12
        sustained = seconds >= 1.0
        peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        peak_name = "bf16_tflops_sustained (cuBLAS)" if sustained else "bf16_tflops burst (cuBLAS)"
    roofline = {"bound": info["bound"], "kernel": info["kernel"], "achieved": achieved, "peak": peak,
                "unit": info["unit"], "frac": achieved / peak, "peak_source": f"{peaks['source']} {peak_name}",
                "traffic": committed_traffic(info["traffic_key"]),
                ("bytes_per_launch" if info["bound"] == "hbm" else "flop_per_launch"): units_per_launch,
                "launch_us": per_launch_s * 1e6}

    e2e = None
    if not args.no_e2e:
        e2e_steps = min(steps, 2000)
        t_e2e, bi, bo, via = time_e2e(wl, e2e_steps, device)
        t_e2e = reduce_max(dist, t_e2e, device)
        e2e = {"value": aggregate(wl.units_per_step * e2e_steps, world, t_e2e) / wl.scale, "unit": wl.unit,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": e2e_steps, "via": via}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(WORKLOAD_ORACLE_SHAPES[args.workload](synth), wl.unit)
        r, sample, dt = smp.rate(args.cpu_seconds)
        cpu = {"value": r, "unit": wl.unit, "cores": smp.threads, "kind": "oracle", "sample": sample,
               "seconds": round(dt, 2)}
        if smp.threads > 1:   # the same oracle on one host core
            smp.threads = 1
            r1, sample1, dt1 = smp.rate(args.cpu_seconds)
            cpu["single_thread"] = {"value": r1, "unit": wl.unit, "cores": 1, "sample": sample1,
                                    "seconds": round(dt1, 2)}

    if rank == 0:
        config = wl.config()
        if 1 < len(getattr(wl, "cases", [])) <= 8 and world == 1:
            config["per_case_" + wl.unit.replace("/", "")] = time_cases(wl, device)
        codes_only = None   # the same rate counting the code bytes alone (no scales and biases)
        if wl.unit == "GB/s" and getattr(wl, "cases", None):
            codes_only = value * sum(c.N * c.K * c.bits // 8 for c in wl.cases) / sum(c.packed_bytes for c in wl.cases)
        line = {"metric": METRIC, "value": value, "unit": wl.unit, "n_gpus": world, "steps": steps,
                "warmup": warmup, "ms_per_step": t_max / steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": steps * wl.kernels_per_step, "clocks": clocks, "kernel_src_digest": source_digest(),
                "codes_only_gbs": codes_only}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
