"""Benchmark of split-K paged-attention decode on GB300.

Prints ONE JSON line (rank 0).  A step is one decode call over one batch of
the workload: phase 1 (attention over every partition) and phase 2 (the
log-sum-exp merge) for V2, or the single pass for V1 -- whichever the V1/V2
dispatch picks for the workload.  The metric is effective KV-read bandwidth:
the K and V bytes a decode must read (sum over sequences of
seq_len * num_kv_heads * head_dim * 2 * 2 bytes) divided by the time per call.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                        [--impl reference]
Under torchrun (N > 1) every rank decodes its own replica of the workload
(no data exchange: the path has none) and the slowest rank's time is used.
``--impl reference`` times the fp64 CPU oracle instead, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import ctypes
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
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "paged-decode attention effective KV-read GB/s (% of HBM peak); µs per call"
DEFAULT_CONFIG = "batch_decode"
# Timed after the headline in the same run: the 100K-token decode at both
# partition sizes and the largest workload (4.3 GB of K/V).
PER_CONFIG = ("long_100k", "long_100k_p1024", "stress")
# Calls in each per_config timed region (the headline times --steps).
PER_CONFIG_STEPS = 100
# The HBM3e figure quoted for the part (about 8 TB/s); the measured copy
# bandwidth is the roofline's denominator, this one is reported beside it.
NOMINAL_HBM_GBS = 8000.0
# Sources of each kernel family, hashed to void a recorded ncu traffic figure
# once the kernel changes.
KERNEL_SOURCES = {
    "pa_attn": ["paged_kv_decode_v2_gb300/csrc/pa_attn.cuh",
                "paged_kv_decode_v2_gb300/csrc/pa_device.cuh"],
    "pa_simt": ["paged_kv_decode_v2_gb300/csrc/pa_simt.cuh",
                "paged_kv_decode_v2_gb300/csrc/pa_device.cuh"],
    "pa_tc": ["paged_kv_decode_v2_gb300/csrc/pa_tc.cuh",
              "paged_kv_decode_v2_gb300/csrc/pa_tc2.cuh",
              "paged_kv_decode_v2_gb300/csrc/pa_tcgen05.cuh",
              "paged_kv_decode_v2_gb300/csrc/pa_device.cuh"],
}
# From this many query rows per KV head the library runs the tcgen05 kernel.
TC_MIN_ROWS = 32
# From this many (bf16, two tiles) it writes the binary16 copy of V.
VH_MIN_ROWS = 1024
# pa_set_rows_kernel mode of this run (--rows-kernel).
ROWS_KERNEL = 0


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(x: float, world: int, device) -> float:
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


# ---------------------------------------------------------------- peaks, clocks, traffic

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor TFLOP/s: the measured burst figure (a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the GPU is under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed: edits to
    comments leave the code, and so the hash, unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(family: str = "pa_attn") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[f"{kernel}/{workload}"]
    except Exception:
        return None
    if rec.get("source_hash") != kernel_source_hash(kernel.split("_v")[0]):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- the read floor

# A plain load kernel over a decode workload's own caches and block table: one
# CTA per (partition, KV head, sequence) reads the K and V tiles of its blocks
# (UNROLL blocks per round, every load of a round issued before any is used,
# nothing computed).  Its time is what reading exactly the decode's bytes in
# its paged layout costs on this GPU: the floor phase 1 is compared with.
READ_FLOOR_SRC = r"""
#include <cstdint>
#include <cuda_runtime.h>
template <int UNROLL, int R>
__global__ void rf_gather(const uint4 *__restrict__ kc, const uint4 *__restrict__ vc,
                          const int *__restrict__ table, const int *__restrict__ seq_lens,
                          int max_blocks, int bs, int KV, int bpp, long long pool, unsigned *sink)
{
    const int p = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int per = R * blockDim.x;
    const int L = seq_lens[s];
    const int nb = (L + bs - 1) / bs;
    const int b0 = p * bpp;
    const int b1 = b0 + bpp < nb ? b0 + bpp : nb;
    const int *row = table + (size_t)s * max_blocks;
    unsigned acc = 0;
    for (int b = b0; b < b1; b += UNROLL) {
        uint4 v[2 * UNROLL * R];
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const int id = b + k < b1 ? row[b + k] : -1;
            const bool ok = id >= 0 && id < pool;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const size_t off = ((size_t)(ok ? id : 0) * KV + h) * per + r * blockDim.x + threadIdx.x;
                v[2 * (k * R + r)] = ok ? __ldcs(kc + off) : make_uint4(0, 0, 0, 0);
                v[2 * (k * R + r) + 1] = ok ? __ldcs(vc + off) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int j = 0; j < 2 * UNROLL * R; ++j)
            acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
    }
    if (acc == 0x9e3779b9u)
        sink[0] = acc;
}
extern "C" int rf_launch(const void *kc, const void *vc, const int *table, const int *seq_lens,
                         int S, int max_blocks, int bs, int KV, int D, int bpp, int np,
                         long long pool, unsigned *sink, int block, int unroll, void *stream)
{
    const int per = bs * D * 2 / 16;
    if (block <= 0 || per % block || (per / block != 1 && per / block != 2))
        return 1;
    dim3 grid(np, KV, S);
    cudaStream_t st = (cudaStream_t)stream;
    const uint4 *k = (const uint4 *)kc, *v = (const uint4 *)vc;
    if (per / block == 1) {
        if (unroll == 8) rf_gather<8, 1><<<grid, block, 0, st>>>(k, v, table, seq_lens, max_blocks, bs, KV, bpp, pool, sink);
        else rf_gather<2, 1><<<grid, block, 0, st>>>(k, v, table, seq_lens, max_blocks, bs, KV, bpp, pool, sink);
    } else {
        if (unroll == 8) rf_gather<8, 2><<<grid, block, 0, st>>>(k, v, table, seq_lens, max_blocks, bs, KV, bpp, pool, sink);
        else rf_gather<2, 2><<<grid, block, 0, st>>>(k, v, table, seq_lens, max_blocks, bs, KV, bpp, pool, sink);
    }
    return (int)cudaGetLastError();
}
"""


def read_floor(dec, k1_ms: float) -> dict:
    """Best time of the plain gather over the workload's caches (a few launch shapes), beside
    phase 1's time on the same bytes; single-token decode workloads only."""
    import subprocess
    w, inp = dec.w, dec.inp
    build = os.path.join(ROOT, "paged_kv_decode_v2_gb300", "_build")
    os.makedirs(build, exist_ok=True)
    src, so = os.path.join(build, "read_floor.cu"), os.path.join(build, "read_floor.so")
    with open(src, "w") as f:
        f.write(READ_FLOOR_SRC)
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                           "-Xcompiler", "-fPIC", src, "-o", so])
    lib = ctypes.CDLL(so)
    V, LL, I = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int
    lib.rf_launch.argtypes = [V, V, V, V, I, I, I, I, I, I, I, LL, V, I, I, V]
    S, maxb = inp.block_tables.shape
    assert int(inp.seq_lens.max()) <= maxb * w.block_size
    bpp = max(1, w.partition_size // w.block_size)
    np_ = -(-dec.max_seq_len // (bpp * w.block_size))
    per = w.block_size * w.head_dim * 2 // 16
    sink = torch.zeros(4, dtype=torch.int32, device=dec.device)
    stream = torch.cuda.current_stream().cuda_stream
    best = None
    for block, unroll in ((per, 2), (per // 2, 8), (per, 8), (per // 2, 2)):
        if not 32 <= block <= 1024:
            continue

        def fn(k, block=block, unroll=unroll):
            kc, vc = dec.caches[k % dec.copies]
            rc = lib.rf_launch(kc.data_ptr(), vc.data_ptr(), inp.block_tables.data_ptr(),
                               inp.seq_lens.data_ptr(), S, maxb, w.block_size, w.num_kv_heads,
                               w.head_dim, bpp, np_, inp.key_cache.shape[0], sink.data_ptr(),
                               block, unroll, stream)
            if rc:
                raise RuntimeError(f"read-floor probe launch failed ({rc})")
        for k in range(5):
            fn(k)
        torch.cuda.synchronize()
        ms = min(time_calls(fn, 5, 50) for _ in range(3))
        if best is None or ms < best[0]:
            best = (ms, block, unroll)
    peak, _ = hbm_peak()
    gbs = dec.kv_bytes / (best[0] * 1e-3) / 1e9
    return {"us": round(best[0] * 1e3, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
            "launch": f"{best[1]} threads, {best[2]} blocks per round",
            "phase1_over_floor": round(best[0] / k1_ms, 4),
            "what": "plain loads of the same K/V tiles through the same block table, one CTA per "
                    "(partition, KV head, sequence), nothing computed"}


# ---------------------------------------------------------------- the CUDA path

class Decoder:
    """One workload on one GPU: inputs (rotated copies when small vs L2) and workspace."""

    def __init__(self, w: wl.Workload, device):
        import paged_kv_decode_v2_gb300 as pa
        self.pa = pa
        pa.load()
        self.w = w
        self.device = device
        base = wl.make_inputs(w, device=device)
        self.kv_bytes = base.kv_bytes
        # Inputs larger than L2 between reuses: rotate through R copies of the caches.
        self.copies = max(1, math.ceil(3 * L2_BYTES / max(1, self.kv_bytes)))
        self.caches = [(base.key_cache, base.value_cache)]
        for r in range(1, self.copies):
            g = torch.Generator(device=device).manual_seed(w.seed + 100 + r)
            k = torch.randn(base.key_cache.shape, generator=g, device=device).to(base.key_cache.dtype)
            v = torch.randn(base.value_cache.shape, generator=g, device=device).to(base.value_cache.dtype)
            self.caches.append((k, v))
        self.inp = base
        self.sum_seq_len = int(base.seq_lens.sum().item())
        S, H, D = base.query.shape[0], w.num_heads, w.head_dim
        self.cap = base.block_tables.shape[1] * w.block_size
        self.max_seq_len = base.max_seq_len
        self.np = pa.num_partitions(self.max_seq_len, w.partition_size)
        self.out = torch.empty_like(base.query)
        if w.q_len > 1:
            # several new tokens: the multi-query dispatch entry point
            self.variant = pa.pa_decode_mq_choose(S, w.q_len, w.num_heads, w.num_kv_heads, D,
                                                  self.max_seq_len, w.partition_size)
        else:
            self.variant = pa.pa_decode_choose(S, w.num_kv_heads, self.max_seq_len,
                                               w.partition_size)
        self.launches_per_step = 2 if self.variant == 2 else 1
        # V1 with several new tokens never touches the intermediates: one slot suffices.
        np_alloc = 1 if (w.q_len > 1 and self.variant == 1) else max(1, self.np)
        self.tmp, self.es, self.ml = pa.alloc_workspace(S, H, D, np_alloc, device=device,
                                                        q_len=w.q_len)
        # Algorithmic FLOPs of a call: 4 * head_dim per (query row, head, visible
        # key) -- Q.K and P.V, 2 * head_dim each; new token i of a sequence of
        # L tokens sees L - q_len + i + 1 keys.
        vis = 0
        for L in base.seq_lens.tolist():
            for i in range(w.q_len):
                vis += max(0, min(L - w.q_len + i + 1, L))
        self.flops = 4 * w.head_dim * w.num_heads * vis
        rows = w.q_len * w.group_size
        self.family = ("pa_tc" if rows >= TC_MIN_ROWS else
                       "pa_simt" if rows <= 8 and ROWS_KERNEL == 5 else "pa_attn")
        self.vh_copy = w.q_len > 1 and self._makes_v_half_copy(pa, S, H, D)
        if self.vh_copy:
            # the offsets and copy passes, the two-tile kernel (binary16 or, when the
            # copy's flag is set, bf16 P), the merge for V2
            self.launches_per_step = 4 if self.variant == 2 else 3

    def _makes_v_half_copy(self, pa, S, H, D) -> bool:
        """Whether pa_decode_mq writes the binary16 copy of V for this workload: the rule
        include/pa_decode.h states (bf16 rows on the two-tile kernel under fp16's rule,
        and room past the partials for the block offsets, the flag and at least one block;
        whether the packed copy then fits is the device's decision, the launches are the
        same either way)."""
        w = self.w
        rows = w.q_len * w.group_size
        mode = ROWS_KERNEL
        uses_tc = mode in (2, 3, 4, 6) or (mode in (0, 5) and rows >= TC_MIN_ROWS)
        two = D <= 128 and uses_tc and mode not in (3, 6) and (
            mode == 4 or (rows > 128 and self.max_seq_len >= 1024))
        # 1024 rows per KV head at least, unless mode 4 forces two tiles
        if w.dtype != wl.BF16 or not two or (rows < VH_MIN_ROWS and mode != 4):
            return False
        part = pa.pa_decode_mq_partition(S, w.q_len, H, w.num_kv_heads, D, self.max_seq_len,
                                         w.partition_size)
        np_used = pa.num_partitions(self.max_seq_len, part) if self.variant == 2 else 0
        r256 = lambda x: (x + 255) // 256 * 256
        off = r256(S * w.q_len * H * np_used * D * 4) + r256(4 * (S + 1))
        block = w.num_kv_heads * w.block_size * D * 2
        return off + block <= self.tmp.numel() * 4

    def free(self):
        """Drop the device buffers (the caller then empties torch's cache)."""
        for name in ("caches", "inp", "out", "tmp", "es", "ml", "e2e_dev_in", "e2e_views",
                     "e2e_out", "_call_args", "_k1_args", "_e2e_args"):
            if hasattr(self, name):
                delattr(self, name)

    def call(self, i: int):
        """One decode call on copy i % R through the public dispatch entry point of the
        C ABI (pa_decode, or pa_decode_mq for several new tokens), its arguments
        marshalled once per copy as a C caller would hold them."""
        if not hasattr(self, "_call_args"):
            pa, w, inp = self.pa, self.w, self.inp
            lib = pa.load()
            self._call_fn = lib.pa_decode_mq if w.q_len > 1 else lib.pa_decode
            shape = pa._lib._shape_args_mq if w.q_len > 1 else pa._lib._shape_args
            self._call_args = []
            for kc, vc in self.caches:
                args = shape(inp.query, kc, vc, inp.block_tables, inp.seq_lens, self.max_seq_len,
                             w.scale)
                self._call_args.append(tuple(args) + (
                    int(w.partition_size), pa._lib._DTYPE[inp.query.dtype],
                    ctypes.c_void_p(self.out.data_ptr()), ctypes.c_void_p(self.tmp.data_ptr()),
                    ctypes.c_void_p(self.es.data_ptr()), ctypes.c_void_p(self.ml.data_ptr()),
                    self.tmp.shape[-2], None))
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = self._call_fn(*self._call_args[i % self.copies], stream)
        if rc != 0:
            raise RuntimeError(f"decode returned {rc}")

    def kernel1_call(self, i: int):
        """Kernel 1 of the call alone, through the C ABI with arguments marshalled once:
        pa_decode_v2_phase1 for V2, the whole call otherwise (V1 is one kernel; the
        multi-query V2 has no separate phase-1 entry point)."""
        if self.w.q_len > 1 or self.variant != 2:
            return self.call(i)
        if not hasattr(self, "_k1_args"):
            pa, w, inp = self.pa, self.w, self.inp
            self._k1_fn = pa.load().pa_decode_v2_phase1
            self._k1_args = []
            for kc, vc in self.caches:
                args = pa._lib._shape_args(inp.query, kc, vc, inp.block_tables, inp.seq_lens,
                                           self.max_seq_len, w.scale)
                self._k1_args.append(tuple(args) + (
                    int(w.partition_size), pa._lib._DTYPE[inp.query.dtype],
                    ctypes.c_void_p(self.tmp.data_ptr()), ctypes.c_void_p(self.es.data_ptr()),
                    ctypes.c_void_p(self.ml.data_ptr()), self.tmp.shape[-2], None))
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = self._k1_fn(*self._k1_args[i % self.copies], stream)
        if rc != 0:
            raise RuntimeError(f"phase 1 returned {rc}")

    def pack_host_inputs(self):
        """One pinned host buffer holding a step's query, block tables and lengths;
        two device copies of it and two outputs (double buffering)."""
        inp = self.inp
        parts = [inp.query, inp.block_tables, inp.seq_lens]
        sizes = [t.numel() * t.element_size() for t in parts]
        offs = [0]
        for n in sizes:
            offs.append(offs[-1] + (n + 255) // 256 * 256)
        host_in = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
        for t, o, n in zip(parts, offs, sizes):
            host_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        self.e2e_dev_in, self.e2e_views, self.e2e_out, self.e2e_host_out = [], [], [], []
        for _ in range(2):
            dev_in = torch.empty(offs[-1], dtype=torch.uint8, device=self.device)
            self.e2e_dev_in.append(dev_in)
            self.e2e_views.append([dev_in[o:o + n].view(t.dtype).view(t.shape)
                                   for t, o, n in zip(parts, offs, sizes)])
            self.e2e_out.append(torch.empty_like(self.out))
            self.e2e_host_out.append(torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory())
        self.copy_stream = torch.cuda.Stream(device=self.device)
        self.compute_stream = torch.cuda.Stream(device=self.device)
        return host_in

    def e2e_steps(self, k0: int, n: int, host_in):
        """n decode steps through the C ABI with host buffers, pipelined as a
        serving loop does, with two buffer sets.  The copy stream moves step
        k + 1's inputs host -> device (one packed copy) while step k decodes on
        the compute stream, then step k's `out` device -> host once it is done;
        the next step's input copy is queued ahead of this step's output copy
        so it never waits behind a decode.  Every step moves its own bytes.  The
        copies, events and the decode entry point are called through ctypes
        with arguments marshalled once, so the host keeps ahead of the GPU.
        Returns (start, end) events bracketing all copies and decodes."""
        rt, lib = _cudart(), self.pa.load()
        cs, ks = self.copy_stream, self.compute_stream
        csh, ksh = ctypes.c_void_p(cs.cuda_stream), ctypes.c_void_p(ks.cuda_stream)
        if not hasattr(self, "_e2e_events"):
            evs = []
            for _ in range(4):
                e = ctypes.c_void_p()
                _rt_check(rt.cudaEventCreateWithFlags(ctypes.byref(e), 2))  # no timing
                evs.append(e)
            self._e2e_events = evs
            self._e2e_args = [[self._decode_args(j, c, ksh) for c in range(self.copies)]
                              for j in range(2)]
        h2d_ev, dec_ev = self._e2e_events[0:2], self._e2e_events[2:4]
        entry = lib.pa_decode_mq if self.w.q_len > 1 else lib.pa_decode
        nbytes_in = host_in.numel()
        nbytes_out = self.e2e_out[0].numel() * self.e2e_out[0].element_size()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        cs.wait_stream(torch.cuda.current_stream())
        ks.wait_stream(torch.cuda.current_stream())

        def h2d(k):
            # Set k % 2 was last read by step k - 2, whose decode has ended.
            j = k % 2
            if k - k0 >= 2:
                _rt_check(rt.cudaStreamWaitEvent(csh, dec_ev[j], 0))
            _rt_check(rt.cudaMemcpyAsync(ctypes.c_void_p(self.e2e_dev_in[j].data_ptr()),
                                         ctypes.c_void_p(host_in.data_ptr()), nbytes_in, 1, csh))
            _rt_check(rt.cudaEventRecord(h2d_ev[j], csh))

        start.record(cs)
        h2d(k0)
        for k in range(k0, k0 + n):
            j = k % 2
            # Step k's inputs have landed; they were queued after step k - 2's
            # output copy, so out[j] is free again as well.
            _rt_check(rt.cudaStreamWaitEvent(ksh, h2d_ev[j], 0))
            rc = entry(*self._e2e_args[j][k % self.copies])
            if rc != 0:
                raise RuntimeError(f"decode returned {rc}")
            _rt_check(rt.cudaEventRecord(dec_ev[j], ksh))
            if k + 1 < k0 + n:
                h2d(k + 1)
            _rt_check(rt.cudaStreamWaitEvent(csh, dec_ev[j], 0))
            _rt_check(rt.cudaMemcpyAsync(ctypes.c_void_p(self.e2e_host_out[j].data_ptr()),
                                         ctypes.c_void_p(self.e2e_out[j].data_ptr()), nbytes_out, 2,
                                         csh))
        cs.wait_stream(ks)
        end.record(cs)
        return start, end

    def _decode_args(self, j: int, c: int, stream):
        """ctypes arguments of one pa_decode / pa_decode_mq call on buffer set j, cache copy c."""
        pa, w = self.pa, self.w
        q, bt, sl = self.e2e_views[j]
        kc, vc = self.caches[c]
        if w.q_len > 1:
            args = pa._lib._shape_args_mq(q, kc, vc, bt, sl, self.max_seq_len, w.scale)
        else:
            args = pa._lib._shape_args(q, kc, vc, bt, sl, self.max_seq_len, w.scale)
        return tuple(args) + (int(w.partition_size), pa._lib._DTYPE[q.dtype],
                              ctypes.c_void_p(self.e2e_out[j].data_ptr()),
                              ctypes.c_void_p(self.tmp.data_ptr()),
                              ctypes.c_void_p(self.es.data_ptr()),
                              ctypes.c_void_p(self.ml.data_ptr()), self.tmp.shape[-2], None,
                              stream)


_CUDART = None


def _cudart():
    """The CUDA runtime, for stream-ordered copies and events in the end-to-end loop."""
    global _CUDART
    if _CUDART is None:
        import glob
        cands = ["libcudart.so", "libcudart.so.13"]
        for d in (os.environ.get("CUDA_HOME", "/usr/local/cuda"), "/usr/local/cuda"):
            cands += sorted(glob.glob(os.path.join(d, "lib64", "libcudart.so*")))
            cands += sorted(glob.glob(os.path.join(d, "targets", "*", "lib", "libcudart.so*")))
        for c in cands:
            try:
                lib = ctypes.CDLL(c)
                break
            except OSError:
                continue
        else:
            raise RuntimeError("libcudart not found")
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        lib.cudaMemcpyAsync.argtypes = [vp, vp, sz, ctypes.c_int, vp]
        lib.cudaEventRecord.argtypes = [vp, vp]
        lib.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]
        lib.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
        _CUDART = lib
    return _CUDART


def _rt_check(rc: int):
    if rc != 0:
        raise RuntimeError(f"CUDA runtime error {rc}")


def soak(dec, i0: int, seconds: float) -> int:
    """Back-to-back calls for a while (untimed), so clock samples see the GPU under this load."""
    i = i0
    t_end = time.time() + seconds
    while time.time() < t_end:
        dec.call(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return i


# Cycles of the GPU spin that precedes a timed region (about 50 us at 2 GHz).
SPACER_CYCLES = 100_000


def time_calls(fn, i0: int, n: int) -> float:
    """ms per call of n back-to-back calls fn(i0 + k), between two CUDA events on the
    current stream (the stream every launch goes to).  A short GPU spin is queued
    first, outside the timed region: the stream is then busy while the host records
    the start event and queues the first call, so the region measures the calls
    back to back and not the host's launch latency after an idle stream."""
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(SPACER_CYCLES)
    t0.record()
    for k in range(n):
        fn(i0 + k)
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / n


def roofline(dec, k1_ms: float, ms_step: float, w: wl.Workload):
    """The dominant kernel (kernel 1) against its bound: HBM bytes or tensor FLOPs,
    whichever takes longer at its peak."""
    peak, peak_kind = hbm_peak()
    tpeak, tpeak_kind = bf16_peak()
    kernel = dec.family + ("_v2_phase1" if dec.variant == 2 else "_v1")
    k1_gbs = dec.kv_bytes / (k1_ms * 1e-3) / 1e9
    k1_tflops = dec.flops / (k1_ms * 1e-3) / 1e12
    tensor_bound = dec.flops / (tpeak * 1e12) > dec.kv_bytes / (peak * 1e9)
    if tensor_bound:
        r = {"bound": "tensor", "kernel": kernel, "achieved": round(k1_tflops, 2), "peak": tpeak,
             "peak_kind": tpeak_kind + (" dense bf16 (burst)" if w.dtype == wl.BF16 else
                                        " dense bf16 (burst) x 1, fp16's nominal ratio"),
             "unit": "TFLOP/s", "frac": round(k1_tflops / tpeak, 4)}
    else:
        r = {"bound": "hbm", "kernel": kernel, "achieved": round(k1_gbs, 2), "peak": peak,
             "peak_kind": peak_kind + " copy bandwidth", "unit": "GB/s",
             "frac": round(k1_gbs / peak, 4),
             "frac_of_nominal": round(k1_gbs / NOMINAL_HBM_GBS, 4)}
    split = w.q_len == 1 and dec.variant == 2
    r |= {"traffic": recorded_traffic(w.name, kernel),
          "algorithmic_bytes_per_launch": dec.kv_bytes,
          "algorithmic_flops_per_launch": dec.flops,
          "kernel_us": round(k1_ms * 1e3, 3),
          "timing": ("kernel 1 alone: pa_decode_v2_phase1 called back to back between two CUDA "
                     "events on its stream, so consecutive launches keep the programmatic "
                     "dependent launch overlap they have inside the timed call")
                    if split else
                    "the whole call (its one kernel for V1; both kernels for the multi-query V2), "
                    "the timed region's own events",
          "merge_us": round(max(0.0, ms_step - k1_ms) * 1e3, 3) if split else None}
    return r


def measure(dec, w: wl.Workload, i0: int, K: int, W: int, world: int, local: int):
    """W warm-up calls, then the timed region (K calls, barrier and synchronize on both
    sides, clocks sampled under load) and kernel 1 alone over K calls after it.
    Returns (ms per call over the slowest rank, kernel-1 ms per launch, clocks, next i)."""
    for k in range(W):
        dec.call(i0 + k)
    torch.cuda.synchronize()
    i = i0 + W
    with ClockSampler(local) as clk:
        # keep the GPU loaded around the timed region so the clock samples describe it
        i = soak(dec, i, 1.0)
        barrier(world)
        torch.cuda.synchronize()
        ms_step = time_calls(dec.call, i, K)
        barrier(world)
        i += K
        for k in range(W):
            dec.kernel1_call(i + k)
        i += W
        k1_ms = time_calls(dec.kernel1_call, i, K)
        i += K
        i = soak(dec, i, 0.5)
    clocks = clk.summary()
    return max_over_ranks(ms_step, world, dec.device), k1_ms, clocks, i


def config_line(dec, w: wl.Workload, ms_step: float, k1_ms: float, clocks, world: int):
    """The per-workload fields shared by the headline and the per_config entries."""
    peak, _ = hbm_peak()
    gbs = world * dec.kv_bytes / (ms_step * 1e-3) / 1e9
    return {"us_per_call": round(ms_step * 1e3, 3), "value": round(gbs, 2), "unit": "GB/s",
            "pct_of_hbm_peak": round(100.0 * gbs / world / peak, 2),
            "pct_of_nominal_hbm": round(100.0 * gbs / world / NOMINAL_HBM_GBS, 2),
            "variant": f"v{dec.variant}", "kv_bytes_per_step": dec.kv_bytes,
            "roofline": roofline(dec, k1_ms, ms_step, w), "clocks": clocks}


def time_gpu(args, w: wl.Workload):
    world, rank, local = dist_env()
    init_dist(world, "nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dec = Decoder(w, device)
    K, W = args.steps, args.warmup

    ms_step, k1_ms, clocks, _ = measure(dec, w, 0, K, W, world, local)
    head = config_line(dec, w, ms_step, k1_ms, clocks, world)
    if args.read_floor and w.q_len == 1:
        head["read_floor"] = read_floor(dec, k1_ms)

    # End to end through the public API with host buffers: each step copies its
    # inputs (query, block tables, sequence lengths, packed in one pinned
    # buffer) host -> device in one copy, decodes, and reads `out` back to
    # pinned host memory; copies of one step overlap the decode of the next.
    host_in = dec.pack_host_inputs()
    dec.e2e_steps(0, W, host_in)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = dec.e2e_steps(W, K, host_in)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device) / K
    h2d = host_in.numel()
    d2h = dec.e2e_host_out[0].numel() * dec.e2e_host_out[0].element_size()

    result = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_step, 6),
        "us_per_call": head["us_per_call"],
        "pct_of_hbm_peak": head["pct_of_hbm_peak"],
        "pct_of_nominal_hbm": head["pct_of_nominal_hbm"],
        "peaks": {"hbm_gbs": hbm_peak()[0], "hbm_kind": hbm_peak()[1] + " copy bandwidth "
                  "(read + write)", "nominal_hbm_gbs": NOMINAL_HBM_GBS},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.DTYPE_NAME[w.dtype],
        "data": "synthetic (seeded N(0,1) queries and paged K/V caches, random block placement)",
        "config": workload_config(dec, w, world),
        "e2e": {"value": round(world * dec.kv_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 6), "h2d_bytes_per_step": h2d,
                "pipelined": "two buffer sets; step k + 1's input copy and step k - 1's output copy overlap step k's decode",
                "d2h_bytes_per_step": d2h},
        "gpu_launches": K * dec.launches_per_step,
        "roofline": head["roofline"],
        "clocks": clocks,
    }
    if "read_floor" in head:
        result["read_floor"] = head["read_floor"]
    del host_in
    dec.free()
    del dec
    torch.cuda.empty_cache()

    # The other decode workloads the >= 70% target names (the 100K-token sequence
    # at both partition sizes) and the largest one, each timed the same way after
    # the headline's timed region, within the same process.
    if not args.no_per_config and world == 1:
        per = {}
        for name in PER_CONFIG:
            if name == w.name:
                continue
            wc = wl.ALL[name]
            d = Decoder(wc, device)
            ms_c, k1_c, clk_c, _ = measure(d, wc, 0, PER_CONFIG_STEPS, W, world, local)
            per[name] = config_line(d, wc, ms_c, k1_c, clk_c, world) | {
                "steps": PER_CONFIG_STEPS, "config": workload_config(d, wc, world)}
            if args.read_floor and wc.q_len == 1:
                per[name]["read_floor"] = read_floor(d, k1_c)
            d.free()
            del d
            torch.cuda.empty_cache()
        result["per_config"] = per
    return result, rank, world


def workload_config(dec, w: wl.Workload, world: int):
    return {
        "workload": w.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
        "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
        "partition_size": w.partition_size, "q_len": w.q_len, "max_seq_len": dec.max_seq_len,
        "sum_seq_len": dec.sum_seq_len, "kv_bytes_per_step": dec.kv_bytes,
        "variant": f"v{dec.variant}", "accumulate": "f32",
        "binary16_v_copy": bool(getattr(dec, "vh_copy", False)),
        "l2": (f"inputs larger than L2: {dec.copies} rotating K/V cache copies, "
               f"{dec.copies * dec.kv_bytes / 1e6:.0f} MB read between reuses vs 129 MB L2"),
        "parallelism": "replicas" if world > 1 else "single GPU",
    }


# ---------------------------------------------------------------- the oracle on the host

def time_oracle(w: wl.Workload, budget_s: float = 12.0):
    """The fp64 oracle as it stands, on all host cores, over a bounded sample of the workload.

    The sample is a seeded random subset of the (query row, head) pairs; the
    time of the whole workload is extrapolated by the keys the pairs see, and
    the line's GB/s is the workload's K/V bytes over that time.
    """
    import oracle
    inp = wl.make_inputs(w, device="cpu")
    prob = oracle.Problem.from_arrays(wl.to_oracle_arrays(inp))
    cores = os.cpu_count() or 1
    S, Q, H = w.num_seqs, w.q_len, w.num_heads
    lens = inp.seq_lens.tolist()
    keys = [max(0, min(lens[r // Q] - Q + r % Q + 1, lens[r // Q])) for r in range(S * Q)]
    total_keys = sum(keys) * H
    order = torch.randperm(S * Q * H, generator=torch.Generator().manual_seed(w.seed)).tolist()
    # grow the sample of (row, head) pairs until one pass takes a noticeable time
    n = max(1, min(len(order), 64))
    while True:
        pairs = [(i // H, i % H) for i in order[:n]]
        t = time.perf_counter()
        oracle.decode(prob, pairs=pairs, num_threads=cores)
        dt = time.perf_counter() - t
        if dt > budget_s / 4 or n == len(order):
            break
        n = min(len(order), n * 4)
    reps = max(1, int(budget_s / max(dt, 1e-3) / 2))
    t = time.perf_counter()
    for _ in range(reps):
        oracle.decode(prob, pairs=pairs, num_threads=cores)
    dt = (time.perf_counter() - t) / reps
    sample_keys = max(1, sum(keys[r] for r, _ in pairs))
    full_s = dt * total_keys / sample_keys
    gbs = inp.kv_bytes / full_s / 1e9
    desc = (f"{len(pairs)} of {S * Q * H} (query row, head) pairs of {w.name}"
            f"{' (all)' if len(pairs) == S * Q * H else ''}, {reps} timed passes of {dt:.2f} s, "
            f"extrapolated by visible keys")
    return gbs, cores, desc, full_s


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(wl.ALL))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows-kernel", type=int, default=0, choices=range(6),
                    help="pa_set_rows_kernel mode (0 = the library's choice; 5 = the CUDA-core "
                         "kernel up to 8 query rows per KV head)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the chosen workload (no per_config entries)")
    ap.add_argument("--read-floor", action="store_true",
                    help="also time a plain load kernel over each decode workload's own caches "
                         "and block table (built with nvcc on the spot): the read floor that "
                         "phase 1 is compared with")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = wl.ALL[args.config]
    world, rank, _ = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return
        gbs, cores, desc, full_s = time_oracle(w)
        line = {"metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(full_s * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded)", "impl": "reference",
                "config": {"workload": w.name},
                "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                                 "kind": "oracle", "sample": desc},
                "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    global ROWS_KERNEL
    ROWS_KERNEL = args.rows_kernel
    if ROWS_KERNEL:
        import paged_kv_decode_v2_gb300 as pa
        pa.pa_set_rows_kernel(ROWS_KERNEL)
    result, rank, world = time_gpu(args, w)
    if ROWS_KERNEL:
        result["rows_kernel"] = ROWS_KERNEL
    if rank == 0:
        if not args.no_cpu_baseline:
            gbs, cores, desc, _ = time_oracle(w)
            result["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                                      "kind": "oracle", "sample": desc}
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
