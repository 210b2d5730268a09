"""Benchmark: Transformer-XL relative attention + memory rollover on GB300.

One step = one pass of the hot path over one batch of the workload: every
segment of the workload's chain, and in each segment every layer's q, k, v
projections of [memory; h] (txl_project_qkv), its relative attention and
its memory rollover (one txl_rel_attn_fwd_mem call for 64-wide heads, else
txl_rel_attn_fwd and txl_mem_update), the rollover feeding the next
segment's keys and values and each layer's output feeding the next layer (``--attn-only``: the attention and rollover alone on fixed
per-layer inputs).  Inputs are seeded and synthetic, resident in HBM before
the timed region; the per-step working set is far larger than L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the float64 CPU oracle
    python bench.py --recompute-vs-reuse     # eval cost per token, window recompute vs memory reuse

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
(weak scaling: independent sequences, no data-path collective); timing is the
max over ranks.  ``--gpus N`` run without a launcher starts the N ranks
itself (torch.distributed.run on 127.0.0.1).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from transformer_xl_relative_rel_gb300 import inputs  # noqa: E402
from transformer_xl_relative_rel_gb300.workloads import DEFAULT_BENCH, WORKLOADS, Workload  # noqa: E402

METRIC = "rel-attn query-tokens/s and TFLOP/s (% of BF16 tensor peak), 1 GB300"
UNIT = "query-tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "rel_attn_bf16_char_train.md")
KERNEL_SRC = os.path.join(ROOT, "transformer_xl_relative_rel_gb300", "csrc", "attn_bf16.cu")


# --------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, cpu: bool = False):
    if world <= 1:
        return None
    import torch.distributed as dist
    backend = "nccl" if (torch.cuda.is_available() and not cpu) else "gloo"
    dist.init_process_group(backend=backend)
    return dist


def free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(n: int, argv) -> int:
    """``--gpus N`` without a launcher around it: start N ranks on this node
    (torch.distributed.run, rendezvous on 127.0.0.1), one replica per GPU;
    rank 0 prints the line.  Returns the launcher's exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__)] + list(argv)
    env = dict(os.environ)
    env.setdefault("OMP_NUM_THREADS", "1")
    return subprocess.call(cmd, env=env)


def dry_run(args, rank: int, world: int) -> int:
    """The launcher and the cross-rank timing without a GPU: each rank times
    a fixed amount of host work per step (no CUDA call), the step time is the
    max over ranks (gloo), and rank 0 prints the line with ``n_gpus`` = the
    world size and ``value`` = all ranks' units over that time."""
    init_dist(world, cpu=True)
    units = 1000.0
    x = np.ones(1 << 16)
    for _ in range(args.warmup):
        x = np.sqrt(x + 1.0)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x = np.sqrt(x + 1.0)
    local_s = time.perf_counter() - t0
    barrier(world)
    step_s = max_over_ranks(local_s, world) / args.steps
    value = aggregate_rate(units * args.steps, local_s, world)
    if rank == 0:
        print(json.dumps({"metric": "dry run: host work per rank, no GPU", "value": value, "unit": "units/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": step_s * 1e3, "scaling": "weak", "dry_run": True}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the slowest rank sets the time)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_rate(units_per_rank: float, local_seconds: float, world: int) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    t = max_over_ranks(local_seconds, world)
    return units_per_rank * world / t


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes of one layer call of the attention kernel (a launch's bytes
    over the calls it carries) from the committed ncu summary, if it was
    taken on the current kernel source and this workload."""
    try:
        text = open(PROFILE_TRAFFIC).read()
    except OSError:
        return None
    m_src = re.search(r"kernel source sha256\[:16\]:\s*([0-9a-f]{16})", text)
    m_wl = re.search(r"workload:\s*(\S+)", text)
    m_b = re.search(r"dram bytes per (?:launch|call) \(read\+write\):\s*([0-9.eE+]+)", text)
    if not (m_src and m_wl and m_b):
        return None
    if m_src.group(1) != kernel_hash() or m_wl.group(1) != workload:
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except OSError:
            pass
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ------------------------------------------------------------------ workload
class AttnChain:
    """``--attn-only``: every layer's attention on fixed q, k, v, r (drawn
    once, outside the timed region) and the rollover of its extended
    context, which no later attention reads.  Device buffers of one replica:
    per layer q, k, v, r, u, v-bias, the attention output and two
    extended-context buffers [M+L, B, d_model] that trade places every
    segment."""

    graph_steps = 1
    step_desc = ("per segment, per layer: attention on fixed q, k, v (txl_rel_attn_fwd) and the rollover of "
                 "the layer's extended context (no recurrence into k, v)")

    def __init__(self, w: Workload, device, ring: bool = False, pad: int = 0, fused: bool = False):
        s = w.shape
        self.w = w
        self.ring = ring
        # attention and rollover of a layer in one call (txl_rel_attn_fwd_mem)
        self.fused = fused and not ring and not (pad and pad != s.d_head)
        self.pad = pad if pad and pad != s.d_head else 0
        self.dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        B, H, D, L, M, T, dm = s.batch, s.heads, s.d_head, s.seg_len, s.mem_len, s.klen, s.d_model
        g = torch.Generator(device=device).manual_seed(w.seed)
        self.layers = []
        sin = torch.from_numpy(inputs.sinusoid(T, dm)).float().to(device)
        for n in range(w.layers):
            if w.init == "unit":
                q = torch.randn(L, B, H, D, generator=g, device=device)
                k = torch.randn(T, B, H, D, generator=g, device=device)
                v = torch.randn(T, B, H, D, generator=g, device=device)
                wr = torch.randn(dm, dm, generator=g, device=device) * math.sqrt(2.0 / dm)
                u = torch.randn(H, D, generator=g, device=device)
                wb = torch.randn(H, D, generator=g, device=device)
                ext = torch.randn(T, B, dm, generator=g, device=device)
            else:   # hidden states N(0,1), projection weights N(0, 0.02^2)
                ext = torch.randn(T, B, dm, generator=g, device=device)
                wq, wk, wv, wr = (torch.randn(dm, dm, generator=g, device=device) * 0.02 for _ in range(4))
                q = (ext[M:] @ wq).view(L, B, H, D)
                k = (ext @ wk).view(T, B, H, D)
                v = (ext @ wv).view(T, B, H, D)
                u = torch.randn(H, D, generator=g, device=device) * 0.02
                wb = torch.randn(H, D, generator=g, device=device) * 0.02
            r = (sin @ wr).flip(0).reshape(T, H, D)
            if self.pad:
                # head vectors stored with `pad` elements (zeros past D), the
                # layout txl_project_heads / txl_rel_table write
                def padh(x):
                    return torch.nn.functional.pad(x, (0, self.pad - D))
                q, k, v, r, u, wb = (padh(x) for x in (q, k, v, r, u, wb))
            self.layers.append(dict(
                q=q.to(self.dtype).contiguous(), k=k.to(self.dtype).contiguous(),
                v=v.to(self.dtype).contiguous(), r=r.to(self.dtype).contiguous(),
                u=u.float().contiguous(), w=wb.float().contiguous(),
                out=torch.empty(L, B, H, self.pad or D, dtype=self.dtype, device=device), start=0,
                ext=[ext.to(self.dtype).contiguous(), torch.empty(T, B, dm, dtype=self.dtype, device=device)]))
        torch.cuda.synchronize()

    def step(self, txl, attn_events=None):
        launches = 0
        for _seg in range(self.w.segments):
            for lay in self.layers:
                launches += self.layer(txl, lay, attn_events)
        return launches

    def layer(self, txl, lay, attn_events=None) -> int:
        """One layer of one segment: the attention call and the memory
        update, in one library call when the chain is fused (the events
        then bracket both); returns the kernels launched."""
        if attn_events is not None:
            attn_events.begin()
        if self.fused:
            M = self.w.shape.mem_len
            txl.rel_attn_fwd_mem(lay["q"], lay["k"], lay["v"], lay["r"], lay["u"], lay["w"], mem_len=M,
                                 mem_next=lay["ext"][1], ext_ctx=lay["ext"][0], out=lay["out"])
            lay["ext"].reverse()
            mem_launches = 0 if self.rollover_in_attention else 1
        else:
            self.attn(txl, lay)
            mem_launches = None
        if attn_events is not None:
            attn_events.end()
        if mem_launches is None:
            mem_launches = self.memory(txl, lay)
        return 1 + self.attn_extra_launches + mem_launches

    def attn(self, txl, lay):
        """The layer's attention call in this chain's storage mode."""
        M = self.w.shape.mem_len
        if self.ring:
            txl.rel_attn_fwd_ring(lay["q"], lay["k"], lay["v"], lay["r"], lay["u"], lay["w"],
                                  mem_len=M, kv_start=lay["start"], out=lay["out"])
        elif self.pad:
            txl.rel_attn_fwd_padded(lay["q"], lay["k"], lay["v"], lay["r"], lay["u"], lay["w"],
                                    mem_len=M, d_head=self.w.shape.d_head, out=lay["out"])
        else:
            txl.rel_attn_fwd(lay["q"], lay["k"], lay["v"], lay["r"], lay["u"], lay["w"],
                             mem_len=M, out=lay["out"])

    def memory(self, txl, lay) -> int:
        """The layer's memory update; returns the kernels it launched."""
        M, L = self.w.shape.mem_len, self.w.shape.seg_len
        T = M + L
        if self.ring:
            # the context is a ring of T rows: the segment's L rows replace the
            # oldest L (the hidden states here; a k / v ring takes its
            # projected rows the same way)
            w0 = (lay["start"] + M) % T
            txl.ring_append(lay["ext"][0], lay["ext"][1][:L], w0)
            lay["start"] = (lay["start"] + L) % T
            return 2 if w0 + L > T else 1
        txl.mem_update(lay["ext"][1], lay["ext"][0], mem_len=M)
        lay["ext"].reverse()
        return 1

    @property
    def working_set_bytes(self) -> int:
        tot = 0
        for lay in self.layers:
            for key in ("q", "k", "v", "r", "out"):
                tot += lay[key].numel() * lay[key].element_size()
            tot += sum(x.numel() * x.element_size() for x in lay["ext"])
        return tot

    def oracle_layer(self) -> dict:
        lay = self.layers[0]
        if not self.pad:
            return lay
        D = self.w.shape.d_head
        return {k: lay[k][..., :D] for k in ("q", "k", "v", "r", "u", "w")}

    def e2e(self, txl, steps: int, world: int) -> dict:
        return measure_e2e(self.w, self, txl, steps, world)

    attn_extra_launches = 0
    rollover_in_attention = False


class EagerMarks:
    """CUDA events around each attention call of an eagerly launched step."""

    def __init__(self):
        self.pairs = []
        self.calls = []       # layer calls inside each interval

    def begin(self):
        self._e0 = torch.cuda.Event(enable_timing=True)
        self._e0.record()

    def end(self, calls: int = 1):
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record()
        self.pairs.append((self._e0, e1))
        self.calls.append(calls)

    def intervals_ms(self):
        return [a.elapsed_time(b) for a, b in self.pairs]


class GraphMarks:
    """Event pairs around each attention call of a captured step, recorded by
    the replayed graph itself: external event-record nodes through the
    driver API (an event recorded by torch during a capture only orders
    streams).  The times are then those of the graph-replayed step, with no
    host work between the kernels; after the replays they hold the last one."""
    RECORD_EXTERNAL = 1

    def __init__(self):
        import ctypes
        self._c = ctypes
        cu = ctypes.CDLL("libcuda.so.1")
        vp = ctypes.c_void_p
        cu.cuEventCreate.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
        cu.cuEventRecordWithFlags.argtypes = [vp, vp, ctypes.c_uint]
        self._elapsed = getattr(cu, "cuEventElapsedTime_v2", None) or cu.cuEventElapsedTime
        self._elapsed.argtypes = [ctypes.POINTER(ctypes.c_float), vp, vp]
        self._destroy = getattr(cu, "cuEventDestroy_v2", None) or cu.cuEventDestroy
        self._destroy.argtypes = [vp]
        self.cu = cu
        self.pairs = []
        self.calls = []       # layer calls inside each interval

    def _check(self, r, what):
        if r != 0:
            raise RuntimeError(f"{what}: CUresult {r}")

    def _record(self):
        c = self._c
        ev = c.c_void_p()
        self._check(self.cu.cuEventCreate(c.byref(ev), 0), "cuEventCreate")
        stream = c.c_void_p(torch.cuda.current_stream().cuda_stream)
        self._check(self.cu.cuEventRecordWithFlags(ev, stream, self.RECORD_EXTERNAL), "cuEventRecordWithFlags")
        return ev

    def begin(self):
        self._e0 = self._record()

    def end(self, calls: int = 1):
        self.pairs.append((self._e0, self._record()))
        self.calls.append(calls)

    def intervals_ms(self):
        c = self._c
        out = []
        for a, b in self.pairs:
            ms = c.c_float()
            self._check(self._elapsed(c.byref(ms), a, b), "cuEventElapsedTime")
            out.append(ms.value)
        return out

    def close(self):
        for a, b in self.pairs:
            self._destroy(a)
            self._destroy(b)
        self.pairs = []


def qkv_launches(w: Workload, dp: int, ring: bool) -> int:
    """Launches of a layer's q, k, v projections under txl_project_qkv's
    rule (include/txl.h): bf16 TMA-addressable operands put the three in one
    launch; the ring variant projects q on its own."""
    s = w.shape
    n_out = s.heads * dp
    bn = 256 if n_out >= 256 else (n_out + 15) // 16 * 16
    fused = (w.dtype == "bf16" and s.d_model % 8 == 0 and (n_out * 2) % 16 == 0 and dp <= 256
             and bn % dp == 0)
    if not fused:
        return 3
    return 2 if ring else 1


def qkv_cells_launches(w: Workload, dp: int, cells: int) -> int:
    """Launches of txl_project_qkv_cells over ``cells`` layer calls: where a
    call's q, k and v go in one launch, up to eight calls share a launch;
    otherwise each call is projected as txl_project_qkv projects it."""
    one = qkv_launches(w, dp, False)
    if one == 1 and cells >= 2:
        return (cells + 7) // 8
    return cells * one


class LayerChain:
    """The recurrence of the pages, every step a library call.  Per segment
    and layer n (Transformer-XL Sections 3.2-3.3): q = h W_q^T on the
    segment's states, k = h~ W_kE^T and v = h~ W_v^T on the extended context
    h~ = [memory; h] (txl_project_qkv), the relative attention over h~,
    and the rollover that keeps the newest M rows of h~ as the next
    segment's memory (inside the attention call, txl_rel_attn_fwd_mem, or
    txl_mem_update), so each segment's keys and values
    are projected from the memory the previous segment left.  Layer n+1's
    segment states are layer n's attention output, written by the
    attention straight into layer n+1's extended context (the output
    projection, residual, LayerNorm and feed-forward between layers are not
    on this path and are left out); layer 0's are the segment's input
    states, copied in by the library (txl_ring_append of L rows).  Head
    vectors other than 64 wide are stored padded to 64 (the layout the
    projections write); their layers n >= 1 read fixed synthetic states,
    because the padded output is not a d_model-wide row.  The relative
    table of each layer depends on neither batch nor segment and is built
    once (txl_rel_table), outside the timed region."""

    def __init__(self, w: Workload, device, txl, ring: bool = False, fused: bool = False):
        s = w.shape
        self.w = w
        self.txl = txl
        B, H, D, L, M, T, dm = s.batch, s.heads, s.d_head, s.seg_len, s.mem_len, s.klen, s.d_model
        self.dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.dp = 64 if (D != 64 and w.dtype == "bf16") else D
        if (ring or fused) and self.dp != D:
            raise SystemExit("--ring / --fused-rollover need unpadded heads (d_head 64)")
        self.ring, self.fused = ring, fused
        dt, dp = self.dtype, self.dp
        g = torch.Generator(device=device).manual_seed(w.seed)
        # the segments' input states (layer 0), N(0, 1)
        self.h0 = [torch.randn(L, B, dm, generator=g, device=device).to(dt) for _ in range(w.segments)]
        self.layers = []
        for _n in range(w.layers):
            def wt():
                return (0.02 * torch.randn(H * D, dm, generator=g, device=device)).to(dt).contiguous()
            wq, wk, wv, wr = wt(), wt(), wt(), wt()
            u = torch.zeros(H, dp, device=device)
            wb = torch.zeros(H, dp, device=device)
            u[:, :D] = 0.02 * torch.randn(H, D, generator=g, device=device)
            wb[:, :D] = 0.02 * torch.randn(H, D, generator=g, device=device)
            r = txl.rel_table(wr, T, H, D, dp)
            # the first memory, and fixed segment states in rows M.. where no
            # earlier layer writes them: N(0, 1)
            ext0 = torch.randn(T, B, dm, generator=g, device=device).to(dt)
            ext = [ext0] if ring else [ext0, ext0.clone()]
            self.layers.append(dict(
                wq=wq, wk=wk, wv=wv, r=r, u=u, w=wb, ext=ext, start=0, hin=None,
                q=torch.empty(L, B, H, dp, dtype=dt, device=device),
                k=torch.empty(T, B, H, dp, dtype=dt, device=device),
                v=torch.empty(T, B, H, dp, dtype=dt, device=device),
                out=torch.empty(L, B, H, dp, dtype=dt, device=device)))
        self.cur = 0
        self.proj_launches = qkv_launches(w, dp, ring)
        torch.cuda.synchronize()

    # every other step starts from the other buffer of each ping-pong pair
    # when the segment count is odd: a graph then holds two steps
    @property
    def graph_steps(self) -> int:
        return 1 if (self.ring or self.w.segments % 2 == 0) else 2

    @property
    def step_desc(self) -> str:
        roll = ("ring append of the L new rows (txl_ring_append)" if self.ring else
                "rollover in the attention call (a diagonal's calls in shared launches of up to 8 calls, "
                "txl_rel_attn_fwd_mem_cells)" if self.attn_grouped else
                "rollover in the attention call (txl_rel_attn_fwd_mem)" if self.fused else
                "rollover of the extended context (txl_mem_update)")
        order = ("" if self.ring else
                 "; the (layer, segment) cells run as a wavefront over the diagonals layer + segment, "
                 "each diagonal's projections (txl_project_qkv_cells, up to 8 cells a launch) then its "
                 "attention calls")
        return ("per segment: layer 0's input states copied in (txl_ring_append); per layer: q, k, v "
                "projections of [memory; h] (txl_project_qkv, tcgen05: x read once for the three), "
                "attention, " + roll +
                "; layer n's output is layer n+1's input" + order)

    def _ring_in(self, lay, rows) -> int:
        """Append a segment's L states to a layer's ring (the oldest L rows)."""
        s = self.w.shape
        T = s.klen
        pos = (lay["start"] + s.mem_len) % T
        self.txl.ring_append(lay["ext"][0], rows, pos)
        lay["hin"] = rows
        return 2 if pos + s.seg_len > T else 1

    def step(self, txl, attn_events=None, inputs=None) -> int:
        """One pass over the workload's segments.  With the memory copied
        between ping-pong buffers the (layer, segment) cells run as a
        wavefront: cell (n, tau) needs layer n-1's output of segment tau and
        layer n's memory from segment tau-1, so the cells with the same
        n + tau are independent; each such diagonal runs its projections,
        then its attention calls back to back.  Every call gets exactly the
        inputs of the segment-by-segment order.  ``inputs``: optional
        (ready, used) CUDA events per segment around layer 0's input copy."""
        if self.ring:
            launches = 0
            for tau in range(self.w.segments):
                launches += self.segment(txl, tau, attn_events)
            return launches
        launches = 0
        cur0, nl, S = self.cur, len(self.layers), self.w.segments
        for d in range(nl + S - 1):
            cells = [(n, d - n) for n in range(nl) if 0 <= d - n < S]
            for n, tau in cells:
                if n == 0:
                    launches += self._input(txl, tau, (cur0 + tau) & 1, inputs)
            launches += self._project_cells(txl, [(n, (cur0 + tau) & 1) for n, tau in cells])
            if self.attn_grouped:
                launches += self._attend_cells(txl, [(n, (cur0 + tau) & 1) for n, tau in cells], attn_events)
                continue
            for n, tau in cells:
                launches += self._attend(txl, n, (cur0 + tau) & 1, attn_events)
        self.cur = (cur0 + S) & 1
        return launches

    def _input(self, txl, tau: int, par: int, inputs=None) -> int:
        """Layer 0's segment states into its extended context (L rows)."""
        M = self.w.shape.mem_len
        if inputs is not None:
            torch.cuda.current_stream().wait_event(inputs[0][tau])
        txl.ring_append(self.layers[0]["ext"][par][M:], self.h0[tau], 0)     # a plain copy of L rows
        if inputs is not None:
            inputs[1][tau].record(torch.cuda.current_stream())
        return 1

    def _project_cells(self, txl, cells) -> int:
        """The projections of a diagonal's (layer, buffer) cells in grouped
        launches (txl_project_qkv_cells)."""
        s = self.w.shape
        lays = [self.layers[n] for n, _ in cells]
        txl.project_qkv_cells([lay["ext"][par] for lay, (_, par) in zip(lays, cells)],
                              [lay["wq"] for lay in lays], [lay["wk"] for lay in lays],
                              [lay["wv"] for lay in lays], s.heads, s.d_head, self.dp, q_from=s.mem_len,
                              qs=[lay["q"] for lay in lays], ks=[lay["k"] for lay in lays],
                              vs=[lay["v"] for lay in lays])
        return qkv_cells_launches(self.w, self.dp, len(cells))

    def _attend_cells(self, txl, cells, attn_events=None) -> int:
        """The attention and rollover of a diagonal's (layer, buffer) cells
        in shared launches (txl_rel_attn_fwd_mem_cells, up to 8 calls each):
        each call as _attend makes it."""
        s = self.w.shape
        B, H, D, L, M = s.batch, s.heads, s.d_head, s.seg_len, s.mem_len
        nl = len(self.layers)
        lays = [self.layers[n] for n, _ in cells]
        outs = [self.layers[n + 1]["ext"][par][M:].view(L, B, H, D) if n + 1 < nl else self.layers[n]["out"]
                for n, par in cells]
        if attn_events is not None:
            attn_events.begin()
        txl.rel_attn_fwd_mem_cells([lay["q"] for lay in lays], [lay["k"] for lay in lays],
                                   [lay["v"] for lay in lays], [lay["r"] for lay in lays],
                                   [lay["u"] for lay in lays], [lay["w"] for lay in lays], M,
                                   [lay["ext"][1 - par] for lay, (_, par) in zip(lays, cells)],
                                   [lay["ext"][par] for lay, (_, par) in zip(lays, cells)], outs=outs)
        if attn_events is not None:
            attn_events.end(len(cells))
        k = len(cells)
        launches = (k + 7) // 8 if k >= 2 else 1 + self.attn_extra_launches
        return launches + (0 if self.rollover_in_attention else k)

    def _attend(self, txl, n: int, par: int, attn_events=None) -> int:
        """Layer n's attention (its output straight into layer n+1's
        extended context) and the rollover of its extended context into the
        other buffer, the next segment's memory."""
        s = self.w.shape
        B, H, D, L, M = s.batch, s.heads, s.d_head, s.seg_len, s.mem_len
        lay = self.layers[n]
        ext = lay["ext"][par]
        nxt = self.layers[n + 1] if n + 1 < len(self.layers) else None
        out = lay["out"]
        if nxt is not None and self.dp == D:
            out = nxt["ext"][par][M:].view(L, B, H, D)
        if attn_events is not None:
            attn_events.begin()
        args = (lay["q"], lay["k"], lay["v"], lay["r"], lay["u"], lay["w"])
        if self.fused:
            txl.rel_attn_fwd_mem(*args, mem_len=M, mem_next=lay["ext"][1 - par], ext_ctx=ext, out=out)
        elif self.dp != D:
            txl.rel_attn_fwd_padded(*args, mem_len=M, d_head=D, out=out)
        else:
            txl.rel_attn_fwd(*args, mem_len=M, out=out)
        if attn_events is not None:
            attn_events.end()
        launches = 1 + self.attn_extra_launches
        if self.fused:
            return launches + (0 if self.rollover_in_attention else 1)
        txl.mem_update(lay["ext"][1 - par], ext, mem_len=M)
        return launches + 1

    def segment(self, txl, tau: int, attn_events=None) -> int:
        s = self.w.shape
        B, H, D, L, M, dm = s.batch, s.heads, s.d_head, s.seg_len, s.mem_len, s.d_model
        dp, cur, nl = self.dp, self.cur, len(self.layers)
        launches = 0
        first = self.layers[0]
        if self.ring:
            launches += self._ring_in(first, self.h0[tau])
        else:
            txl.ring_append(first["ext"][cur][M:], self.h0[tau], 0)     # a plain copy of L rows
            launches += 1
        for n, lay in enumerate(self.layers):
            ext = lay["ext"][0 if self.ring else cur]
            if self.ring:   # the segment's states are not the ring's last rows
                txl.project_heads(lay["hin"], lay["wq"], H, D, dp, out=lay["q"])
                txl.project_qkv(ext, None, lay["wk"], lay["wv"], H, D, dp, k=lay["k"], v=lay["v"])
            else:
                txl.project_qkv(ext, lay["wq"], lay["wk"], lay["wv"], H, D, dp, q_from=M,
                                q=lay["q"], k=lay["k"], v=lay["v"])
            launches += self.proj_launches
            nxt = self.layers[n + 1] if n + 1 < nl else None
            out = lay["out"]
            if nxt is not None and dp == D and not self.ring:
                out = nxt["ext"][cur][M:].view(L, B, H, D)      # straight into the next layer's h~
            if attn_events is not None:
                attn_events.begin()
            args = (lay["q"], lay["k"], lay["v"], lay["r"], lay["u"], lay["w"])
            if self.ring:
                txl.rel_attn_fwd_ring(*args, mem_len=M, kv_start=lay["start"], out=out)
            elif self.fused:
                txl.rel_attn_fwd_mem(*args, mem_len=M, mem_next=lay["ext"][1 - cur], ext_ctx=ext, out=out)
            elif dp != D:
                txl.rel_attn_fwd_padded(*args, mem_len=M, d_head=D, out=out)
            else:
                txl.rel_attn_fwd(*args, mem_len=M, out=out)
            if attn_events is not None:
                attn_events.end()
            launches += 1 + self.attn_extra_launches
            if self.ring:
                lay["start"] = (lay["start"] + L) % s.klen
                if nxt is not None:
                    launches += self._ring_in(nxt, out.view(L, B, dm))
            elif self.fused:
                launches += 0 if self.rollover_in_attention else 1
            else:
                txl.mem_update(lay["ext"][1 - cur], ext, mem_len=M)
                launches += 1
        return launches

    @property
    def working_set_bytes(self) -> int:
        tot = sum(x.numel() * x.element_size() for x in self.h0)
        for lay in self.layers:
            for key in ("wq", "wk", "wv", "r", "q", "k", "v", "out"):
                tot += lay[key].numel() * lay[key].element_size()
            tot += sum(x.numel() * x.element_size() for x in lay["ext"])
        return tot

    def oracle_layer(self) -> dict:
        """Layer 0's last attention inputs (first d_head columns), for the
        CPU oracle's timing sample."""
        D = self.w.shape.d_head
        lay = self.layers[0]
        return {k: lay[k][..., :D] for k in ("q", "k", "v", "r", "u", "w")}

    def e2e(self, txl, steps: int, world: int) -> dict:
        """The same step through the public API with each segment's input
        states in pinned host memory: every step copies them host->device
        (on a side stream, a segment ahead) and reads the last layer's
        output of the last segment back; CUDA events around the steps."""
        host = [x.cpu().pin_memory() for x in self.h0]
        last = self.layers[-1]["out"]
        out_host = torch.empty_like(last, device="cpu").pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in host)
        d2h = out_host.numel() * out_host.element_size()
        main = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        S = self.w.segments
        copied = [torch.cuda.Event() for _ in range(S)]
        used = [torch.cuda.Event() for _ in range(S)]

        def one():
            side.wait_stream(main)
            if self.ring:
                for tau in range(S):
                    side.wait_event(used[tau])
                    with torch.cuda.stream(side):
                        self.h0[tau].copy_(host[tau], non_blocking=True)
                        copied[tau].record(side)
                    main.wait_event(copied[tau])
                    self.segment(txl, tau)
                    used[tau].record(main)
            else:
                # every segment's copy is queued up front on the side
                # stream; layer 0's input copy of segment tau waits for it
                for tau in range(S):
                    side.wait_event(used[tau])
                    with torch.cuda.stream(side):
                        self.h0[tau].copy_(host[tau], non_blocking=True)
                        copied[tau].record(side)
                self.step(txl, inputs=(copied, used))
            out_host.copy_(last, non_blocking=True)

        one()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            one()
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        sec = e0.elapsed_time(e1) / 1e3
        tokens = self.w.shape.batch * self.w.shape.seg_len * S * steps
        return {"value": aggregate_rate(tokens, sec, world), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": steps}

    def projection_flops_per_step(self) -> float:
        s = self.w.shape
        per_layer = 2.0 * s.batch * s.d_model * s.heads * s.d_head * (s.seg_len + 2 * s.klen)
        return per_layer * self.w.layers * self.w.segments

    attn_extra_launches = 0
    rollover_in_attention = False
    attn_grouped = False


def rollover_fuses(w: Workload, splits: int) -> bool:
    """Mirror of the library's choice to do the rollover inside the
    attention launch (for the launch count only): bf16, d_head 64, 16-byte
    rows, and a CTA's share of the copy at 8 GB/s within half of its share
    of the tiles at 1.6 us each."""
    s = w.shape
    if w.dtype != "bf16" or s.d_head != 64:
        return False
    row = s.batch * s.d_model * 2
    nbytes = s.mem_len * row
    if (s.seg_len * row) % 16 or nbytes % 16 or nbytes == 0:
        return False
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    nqt = (s.seg_len + 127) // 128
    items = s.batch * s.heads * nqt * splits
    G = min(items, sms)
    tiles = 0.0
    for qt in range(nqt):
        kend = s.mem_len + qt * 128 + min(128, s.seg_len - qt * 128)
        tiles += (kend + 127) // 128 + splits
    tiles *= s.batch * s.heads / G
    return nbytes / G / 8e3 <= 0.5 * tiles * 1.6


# ------------------------------------------------------------- e2e measurement
def measure_e2e(w: Workload, chain: "AttnChain", txl, steps: int, world: int):
    """The same step through the public API with the inputs in pinned host
    memory: every step copies each layer's q, k, v, r, biases and extended
    context host->device, runs the calls, and reads the last layer's output
    back.  Timed with CUDA events around the whole step.

    The copies run on a second stream, one layer ahead: a layer's copies wait
    (event) until that layer's previous calls have finished with its device
    buffers, and its calls wait (event) for its copies, so the host link
    (the bound: every input crosses it) never waits for the kernels."""
    host = []
    for lay in chain.layers:
        host.append({key: lay[key].cpu().pin_memory() for key in ("q", "k", "v", "r", "u", "w")}
                    | {"ext": lay["ext"][0].cpu().pin_memory()})
    out_host = torch.empty_like(chain.layers[-1]["out"], device="cpu").pin_memory()
    M = w.shape.mem_len
    h2d = sum(t.numel() * t.element_size() for hl in host for t in hl.values()) * w.segments
    d2h = out_host.numel() * out_host.element_size()

    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    nl = len(chain.layers)
    copied = [torch.cuda.Event() for _ in range(nl)]   # a layer's inputs are on the device
    used = [torch.cuda.Event() for _ in range(nl)]     # a layer's calls are done with its buffers

    def one():
        side.wait_stream(main)      # nothing of a step starts before the step's start event
        for _seg in range(w.segments):
            for n, (lay, hl) in enumerate(zip(chain.layers, host)):
                side.wait_event(used[n])
                with torch.cuda.stream(side):
                    for key in ("q", "k", "v", "r", "u", "w"):
                        lay[key].copy_(hl[key], non_blocking=True)
                    lay["ext"][0].copy_(hl["ext"], non_blocking=True)
                    copied[n].record(side)
                main.wait_event(copied[n])
                chain.layer(txl, lay)
                used[n].record(main)
        out_host.copy_(chain.layers[-1]["out"], non_blocking=True)

    one()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    sec = e0.elapsed_time(e1) / 1e3
    tokens = w.shape.batch * w.shape.seg_len * w.segments * steps
    return {"value": aggregate_rate(tokens, sec, world), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps}


# ------------------------------------------------------------ oracle (CPU) leg
_ORACLE_INPUTS = {}


def oracle_rate(w: Workload, budget_s: float, layer=None):
    """The float64 oracle, as it stands, on a bounded sample of one layer call
    of the workload: random (b, h, i) rows.  Returns query-tokens/s in the
    benchmark's unit (a query token = one position through every head of
    every layer), the rows done and the threads used."""
    import oracle
    s = w.shape
    key = (w.name, id(layer))
    host = _ORACLE_INPUTS.get(key)
    if host is None:
        if layer is None:
            p = inputs.unit_layer(s, w.seed)
            host = {k: v.astype(np.float64) for k, v in p.items()}
        else:
            host = {k: layer[k].double().cpu().numpy() for k in ("q", "k", "v", "r", "u", "w")}
        _ORACLE_INPUTS.clear()
        _ORACLE_INPUTS[key] = host
    g = np.random.Generator(np.random.PCG64(w.seed + 1))
    threads = oracle.max_threads()
    n = max(threads, 16)
    done, spent = 0, 0.0
    while spent < budget_s:
        rows = np.stack([g.integers(0, s.batch, n), g.integers(0, s.heads, n),
                         g.integers(0, s.seg_len, n)], 1)
        t0 = time.perf_counter()
        oracle.rel_attn_rows(host["q"], host["k"], host["v"], host["r"], host["u"], host["w"],
                             mem_len=s.mem_len, rows=rows)
        dt = time.perf_counter() - t0
        done += n
        spent += dt
        if dt < budget_s / 8:
            n *= 2
    rows_per_s = done / spent
    return rows_per_s / (s.heads * w.layers), done, threads, spent


def config_of(w: Workload, world: int, working_set: int = 0, ring: bool = False, pad: int = 0,
              rollover: str = ""):
    s = w.shape
    c = {"workload": w.name, "batch": s.batch, "heads": s.heads, "d_head": s.d_head,
         "seg_len": s.seg_len, "mem_len": s.mem_len, "layers": w.layers, "segments": w.segments,
         "parallelism": f"replicas x{world} (batch-independent, no collective)"}
    if rollover:
        c["rollover"] = rollover
    if ring:
        c["memory"] = "ring (txl_rel_attn_fwd_ring + txl_ring_append of L rows)"
    if pad and pad != s.d_head:
        c["head_storage"] = f"padded to {pad} (txl_project_heads writes it, txl_rel_attn_fwd_padded reads it)"
    if working_set:
        c["l2"] = f"per-step working set {working_set / 1e9:.2f} GB > 129 MB L2 (inputs larger than L2, no flush)"
    return c


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    per_step = max(0.5, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rate(w, per_step / 4)
    rates, spent = [], 0.0
    rows = 0
    threads = 1
    for _ in range(args.steps):
        r, n, threads, t = oracle_rate(w, per_step)
        rates.append(r)
        rows += n
        spent += t
    value = rows / spent / (w.shape.heads * w.layers)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{rows} random (b,h,i) rows of one layer call, unit-variance "
                                       f"inputs; rate scaled to whole query tokens (x{w.shape.heads} heads "
                                       f"x{w.layers} layers)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------ main
# ------------------------------------------------- recompute vs reuse (Table 9)
TABLE9_PAPER = {3800: 1874, 2800: 1409, 1800: 773, 800: 363}   # Transformer-XL, Table 9 (whole model)


def recompute_vs_reuse(args, local: int):
    """Per-token evaluation cost of the attention, the two ways the paper
    compares in its evaluation-speed section: the vanilla model re-runs a
    whole window of W positions for every prediction (one call with L = W,
    M = 0 gives B new tokens), Transformer-XL runs a 128-token segment against
    a cached memory of W (one call with L = 128, M = W gives 128*B tokens).
    Both through txl_rel_attn_fwd on the char-LM head shape (H 8, D 64).
    One JSON line per attention length; the paper's ratio is for the whole
    model on its own hardware (context, not a target)."""
    import transformer_xl_relative_rel_gb300 as txl
    B, H, D, seg = args.batch_t9, 8, 64, 128
    gen = torch.Generator(device="cuda").manual_seed(9)
    dev = torch.device("cuda", local)

    def layer(L, M):
        T = L + M
        def rnd(*shape):
            return (0.45 * torch.randn(*shape, generator=gen, device=dev)).to(torch.bfloat16)
        return dict(q=rnd(L, B, H, D), k=rnd(T, B, H, D), v=rnd(T, B, H, D), r=rnd(T, H, D),
                    u=0.02 * torch.randn(H, D, generator=gen, device=dev),
                    w=0.02 * torch.randn(H, D, generator=gen, device=dev),
                    out=torch.empty(L, B, H, D, dtype=torch.bfloat16, device=dev), M=M)

    def time_call(lay, reps):
        call = lambda: txl.rel_attn_fwd(lay["q"], lay["k"], lay["v"], lay["r"], lay["u"], lay["w"],
                                        mem_len=lay["M"], out=lay["out"])
        for _ in range(args.warmup):
            call()
        txl.check()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        txl.check()
        return e0.elapsed_time(e1) / 1e3 / reps

    def flops(L, M):
        return 6.0 * D * B * H * (L * M + L * (L + 1) / 2)

    for W in sorted(TABLE9_PAPER):
        reuse = layer(seg, W)
        t_reuse = time_call(reuse, max(5, args.steps))
        del reuse
        recompute = layer(W, 0)
        t_recompute = time_call(recompute, max(3, args.steps // 4))
        del recompute
        torch.cuda.empty_cache()
        per_tok_reuse = t_reuse / (B * seg)
        per_tok_recompute = t_recompute / B
        print(json.dumps({
            "metric": "eval attention time per token: recompute the window (vanilla) vs reuse the memory",
            "attn_len": W, "batch": B, "heads": H, "d_head": D, "seg_len": seg, "dtype": "bf16",
            "data": "synthetic",
            "reuse_us_per_token": per_tok_reuse * 1e6, "recompute_us_per_token": per_tok_recompute * 1e6,
            "slowdown": per_tok_recompute / per_tok_reuse,
            "flop_ratio_per_token": (flops(W, 0) / B) / (flops(seg, W) / (B * seg)),
            "reuse_call_us": t_reuse * 1e6, "recompute_call_us": t_recompute * 1e6,
            "recompute_tflops": flops(W, 0) / t_recompute / 1e12, "reuse_tflops": flops(seg, W) / t_reuse / 1e12,
            "paper_slowdown_whole_model": TABLE9_PAPER[W]}), flush=True)
    return 0


def backward(args, local: int):
    """Time txl_rel_attn_bwd (the gradients of one layer call) at the
    workload's per-call shape: unit-variance bf16 inputs and output gradient,
    workspace and outputs allocated once, CUDA events over the timed calls
    (per-call working set > L2).  Algorithmic work of the backward: 16*D
    FLOPs per visible (query, key) pair -- the content and position scores
    recomputed (2D + 2D), dP, dV, dK (2D each), dQ through the keys and
    through the table (2D each), the table gradient (2D).

    Three timings: the backward that runs its own forward (the headline
    value), the backward fed the forward's saved output and row log-sum-exp,
    and a training layer's forward (with log-sum-exp) plus that backward."""
    import transformer_xl_relative_rel_gb300 as txl
    w = WORKLOADS[args.workload]
    s = w.shape
    B, H, D, L, M = s.batch, s.heads, s.d_head, s.seg_len, s.mem_len
    T = L + M
    gen = torch.Generator(device="cuda").manual_seed(11)
    dev = torch.device("cuda", local)
    rnd = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(torch.bfloat16)
    q, k, v, r, dout = rnd(L, B, H, D), rnd(T, B, H, D), rnd(T, B, H, D), rnd(T, H, D), rnd(L, B, H, D)
    u = torch.randn(H, D, generator=gen, device=dev)
    wb = torch.randn(H, D, generator=gen, device=dev)
    nbytes = txl.rel_attn_bwd_workspace_bytes(B, M, L, H, D, txl.TXL_BF16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    fwd = lambda: txl.rel_attn_fwd(q, k, v, r, u, wb, mem_len=M, out=out, lse=lse)
    fwd()
    grads = txl.rel_attn_bwd(q, k, v, r, u, wb, dout, mem_len=M, workspace=ws)
    bwd = lambda: txl.rel_attn_bwd(q, k, v, r, u, wb, dout, mem_len=M, workspace=ws, grads=grads)
    bwd_saved = lambda: txl.rel_attn_bwd(q, k, v, r, u, wb, dout, mem_len=M, workspace=ws, grads=grads,
                                         out=out, lse=lse)

    def layer():
        fwd()
        bwd_saved()

    def timed(call):
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            call()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / args.steps

    txl.check()
    clocks = ClockSampler(local)
    clocks.start()
    t = timed(bwd)
    t_saved = timed(bwd_saved)
    t_layer = timed(layer)
    clk = clocks.stop()
    txl.check()
    pairs = L * M + L * (L + 1) / 2
    flops = 16.0 * D * B * H * pairs
    peaks, src = load_peaks()
    peak = peaks["bf16_tflops"]
    print(json.dumps({
        "metric": "rel-attn backward query-tokens/s and TFLOP/s (16*D flops per visible pair), 1 GB300",
        "value": B * L / t, "unit": "query-tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_call": t * 1e3, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": w.name, "batch": B, "heads": H, "d_head": D,
                                       "seg_len": L, "mem_len": M,
                                       "l2": f"workspace {nbytes / 1e9:.2f} GB > 129 MB L2 (no flush)"},
        "tflops": flops / t / 1e12, "frac_bf16_peak": flops / t / 1e12 / peak, "peak": peak,
        "peak_source": src, "launches_per_call": 10,
        "saved_forward": {"ms_per_call": t_saved * 1e3, "tflops": flops / t_saved / 1e12,
                          "frac_bf16_peak": flops / t_saved / 1e12 / peak, "launches_per_call": 9},
        "forward_plus_backward": {"ms_per_call": t_layer * 1e3,
                                  "tflops": (flops + 6.0 * D * B * H * pairs) / t_layer / 1e12},
        "design": "tcgen05 scores kernel (P, dA, table-frame dA in bf16) + five tcgen05 contraction launches "
                  "(the library's own; see profiles/)",
        "clocks": clk}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_BENCH, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="txl", choices=["txl", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count")
    ap.add_argument("--segments", type=int, default=0, help="override the workload's segment count")
    ap.add_argument("--recompute-vs-reuse", action="store_true",
                    help="per-token eval attention cost, sliding-window recompute vs memory reuse (Table 9)")
    ap.add_argument("--batch-t9", type=int, default=22, help="batch for --recompute-vs-reuse")
    ap.add_argument("--pad", type=int, default=0,
                    help="store head vectors padded to this many elements (txl_rel_attn_fwd_padded)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the eager step only (no CUDA-graph replay of the step)")
    ap.add_argument("--backward", action="store_true",
                    help="time txl_rel_attn_bwd (gradients of one layer call) at the workload's shape")
    ap.add_argument("--fused-rollover", action="store_true",
                    help="--attn-only: attention and memory update of a layer in one call "
                         "(txl_rel_attn_fwd_mem; the recurrence step does this by default); the roofline's "
                         "launch time then includes the rollover copy")
    ap.add_argument("--separate-rollover", action="store_true",
                    help="recurrence step: the memory update as its own call (txl_mem_update) instead of "
                         "inside the attention call")
    ap.add_argument("--ring", action="store_true",
                    help="memory as a ring: each layer appends its L new rows instead of copying M")
    ap.add_argument("--attn-only", action="store_true",
                    help="time attention + rollover on fixed per-layer q, k, v (no projections, no recurrence "
                         "into k, v)")
    ap.add_argument("--dry-run", action="store_true",
                    help="no GPU: exercise the rank launcher and the max-over-ranks timing on host work")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one replica per GPU: this process becomes the launcher of N ranks
        return launch_ranks(args.gpus, sys.argv[1:] if argv is None else argv)
    rank, world, local = dist_env()
    if args.dry_run:
        return dry_run(args, rank, world)
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import transformer_xl_relative_rel_gb300 as txl
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    init_dist(world)
    try:
        txl.load_library()
    except txl.TxlError:
        from transformer_xl_relative_rel_gb300 import _build
        _build.build()
        txl.load_library()

    if args.recompute_vs_reuse:
        return recompute_vs_reuse(args, local)
    if args.backward:
        return backward(args, local)

    w = WORKLOADS[args.workload]
    if args.layers or args.segments:
        import dataclasses
        w = dataclasses.replace(w, layers=args.layers or w.layers, segments=args.segments or w.segments)
    s = w.shape
    dev = torch.device("cuda", local)
    if args.attn_only:
        chain = AttnChain(w, dev, ring=args.ring, pad=args.pad, fused=args.fused_rollover)
        padded = bool(chain.pad)
    else:
        # the attention and the memory update of a layer in one call wherever
        # the chain allows it (64-wide heads, a copied memory)
        fused = not args.separate_rollover and not args.ring and (s.d_head == 64 or w.dtype != "bf16")
        chain = LayerChain(w, dev, txl, ring=args.ring, fused=fused or args.fused_rollover)
        padded = chain.dp != s.d_head
    # the library's own plan for this call shape: key splits and launches
    splits, call_launches = txl.rel_attn_fwd_plan(s.batch, s.mem_len, s.seg_len, s.heads, s.d_head,
                                                  txl.TXL_BF16 if w.dtype == "bf16" else txl.TXL_F32)
    # (head vectors stored padded go straight to the kernel: no padding copies)
    chain.attn_extra_launches = (1 if splits > 1 else 0) if padded else call_launches - 1
    chain.rollover_in_attention = chain.fused and rollover_fuses(w, splits)
    # a diagonal's attention calls share launches where the library groups
    # them: bf16, 64-wide heads, unsplit, the fused rollover call
    if isinstance(chain, LayerChain):
        chain.attn_grouped = (chain.fused and not chain.ring and w.dtype == "bf16" and chain.dp == s.d_head == 64
                              and splits == 1)
    for _ in range(args.warmup * chain.graph_steps):
        chain.step(txl)
    txl.check()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    attn_events = EagerMarks()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    launches = 0
    for _ in range(args.steps):
        launches += chain.step(txl, attn_events)
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    txl.check()
    local_s = e0.elapsed_time(e1) / 1e3
    eager_step_s = max_over_ranks(local_s, world) / args.steps
    # The same step captured in a CUDA graph and replayed: the kernels, their
    # arguments and their order are those of the eager step; the per-call
    # host work (binding checks, launch calls) leaves the timed region.  A
    # chain whose ping-pong buffers return to their start only every second
    # step (odd segment count) is captured as two steps and replayed half as
    # often, with one captured single step first when K is odd.  Falls back
    # to the eager timing if the capture fails.
    timing = {"mode": "eager", "eager_ms_per_step": eager_step_s * 1e3}
    attn_ms = attn_events.intervals_ms()
    attn_calls = list(attn_events.calls)
    attn_timing = "CUDA events around each attention launch of the eagerly launched timed steps"
    gmarks = None
    if not args.no_graph and not args.ring:
        try:
            gs = chain.graph_steps
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for _ in range(gs):
                    chain.step(txl)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            # captured on the stream that ran the warm-up step: the library's
            # split scratch is kept per stream and was sized there
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=side):
                for _ in range(gs):
                    chain.step(txl)
            # the same step with an event pair around each attention call,
            # replayed after the timed region (the event nodes cost the step
            # about 5%, so the timed graph has none)
            gmarks = GraphMarks()
            gph_m = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph_m, stream=side):
                for _ in range(gs):
                    chain.step(txl, gmarks)
            g1 = None
            if gs > 1 and args.steps % gs:
                # one more step, replayed after the pairs: it leaves the buffers
                # where this capture leaves the chain's host-side parity
                g1 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g1, stream=side):
                    chain.step(txl)
            for _ in range(args.warmup):
                gph.replay()
            torch.cuda.synchronize()
            txl.check()
            clocks = ClockSampler(local)
            clocks.start()
            barrier(world)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(args.steps // gs):
                gph.replay()
            if g1 is not None:
                g1.replay()
            e1.record()
            torch.cuda.synchronize()
            barrier(world)
            clk = clocks.stop()
            txl.check()
            local_s = e0.elapsed_time(e1) / 1e3
            timing["mode"] = "cuda_graph"
            for _ in range(2):
                gph_m.replay()
            torch.cuda.synchronize()
            txl.check()
            attn_ms = gmarks.intervals_ms()
            attn_calls = list(gmarks.calls)
            attn_timing = ("event-record nodes around each attention launch of the step's graph, replayed "
                           "after the timed region (the last replay; eager-step events gave "
                           f"{sum(attn_events.intervals_ms()) / sum(attn_events.calls) * 1e3:.1f} us per call)")
            del gph, g1, gph_m
        except Exception as ex:   # keep the eager numbers
            torch.cuda.synchronize()
            timing["graph_error"] = str(ex)[:160]
    tokens_per_step = s.batch * s.seg_len * w.segments
    value = aggregate_rate(tokens_per_step * args.steps, local_s, world)
    step_s = max_over_ranks(local_s, world) / args.steps
    if gmarks is not None:
        gmarks.close()
    # a marked interval holds one launch of one layer call, or of several
    # (grouped calls): per-call time = total time / calls
    attn_avg_s = sum(attn_ms) / len(attn_ms) / 1e3
    attn_call_s = sum(attn_ms) / sum(attn_calls) / 1e3

    flops_call = w.flops_per_call()
    calls_per_step = w.layers * w.segments
    tflops_step = flops_call * calls_per_step / step_s / 1e12
    peaks, peak_kind = load_peaks()
    ai = flops_call / w.bytes_per_call()
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if ai >= ridge:
        achieved = flops_call / attn_call_s / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak}
    else:
        achieved = w.bytes_per_call() / attn_call_s / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak}
    roof["traffic"] = profiled_traffic(w.name)
    if getattr(chain, "rollover_in_attention", False):
        s_ = w.shape
        roof["traffic_note"] = ("the launch also copies the layer's memory rollover "
                                f"({2 * 2 * s_.mem_len * s_.batch * s_.d_model / 1e6:.1f} MB algorithmic)")
    if w.dtype == "bf16":
        roof["issued_to_algorithmic_flops"] = w.issued_flops_per_call(splits) / flops_call
    roof["kernel"] = "rel_attn_bf16_kernel" if w.dtype == "bf16" else "rel_attn_f32_kernel"
    roof["launch_avg_us"] = attn_avg_s * 1e6
    roof["calls_per_launch"] = sum(attn_calls) / len(attn_calls)
    roof["call_avg_us"] = attn_call_s * 1e6
    if roof["calls_per_launch"] > 1:
        roof["per_call"] = ("launches carry 1-8 layer calls (txl_rel_attn_fwd_mem_cells): achieved is the "
                            "calls' algorithmic work over the launches' total time; traffic is per call")
    roof["launch_timing"] = attn_timing
    roof["peak_source"] = f"{peak_kind} ({'MEASURED_PEAKS.json burst' if peak_kind == 'measured' else 'fallback'})"

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": config_of(w, world, chain.working_set_bytes, args.ring,
                                args.pad if args.attn_only else (chain.dp if chain.dp != s.d_head else 0),
                                "in the attention launch (txl_rel_attn_fwd_mem)" if chain.rollover_in_attention
                                else ("own launch (txl_rel_attn_fwd_mem)" if chain.fused
                                      else "own launch (txl_mem_update)")),
            "tflops": tflops_step, "pct_bf16_peak": tflops_step / peaks["bf16_tflops"] * 100.0,
            "roofline": roof, "clocks": clk, "gpu_launches": launches, "timing": timing}
    line["config"]["step"] = chain.step_desc
    if isinstance(chain, LayerChain):
        pf = chain.projection_flops_per_step()
        line["projection_tflops"] = pf / step_s / 1e12
        line["step_tflops_with_projections"] = (flops_call * calls_per_step + pf) / step_s / 1e12

    e2e_steps = args.e2e_steps or max(2, min(args.steps, 5))
    line["e2e"] = chain.e2e(txl, e2e_steps, world)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows, threads, spent = oracle_rate(w, 12.0, layer=chain.oracle_layer())
        line["cpu_baseline"] = {
            "value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{rows} random (b,h,i) rows of layer 0's inputs ({spent:.1f} s of CPU); rate scaled "
                      f"to whole query tokens (x{s.heads} heads x{w.layers} layers)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
