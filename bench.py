"""Benchmark of the paged KV-cache decode path on GB300.

Default workload: Llama-2-70B-shaped GQA decode, one layer -- batch 64, 64 query /
8 KV heads (m = 8), head_dim 128, cached lengths uniform in [512, 8192], bf16
K/V, block size 16, shuffled physical blocks, a cycle of 32 consecutive decode
steps that each append one token per sequence.  One bench step = one decode step
of the whole path through pkv_decode_step: the 64 new tokens appended to the cache
and the attention (split-K partials + log-sum-exp merge) for all 64 x 64 heads, in
one launch (the block that reads a sequence's last page writes its new token
first).  Workloads the library cannot fuse call kv_append, then the attention.

Metric: KV-cache bytes read per second (logical bytes: every cached token's K and
V of every KV head, 2 bytes each), with tokens/s per layer beside it.  Other
workloads (--workload) print the same line for the 7B MHA, long-context GQA/MQA
and varlen-prefill configurations.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun every rank runs the same per-GPU workload (weak scaling, no
collective on the data path); rank 0 prints one JSON line with the max time over
ranks.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload instead (the reference arm).
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
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import gen  # noqa: E402

METRIC = "paged GQA decode: KV-cache read GB/s (% of HBM peak); tokens/s per layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------- utilities

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash(files):
    """Identity of the kernels' code: the sources with comments, trailing blanks and empty
    lines removed, so that a comment edit keeps a profile summary valid."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_165_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.rstrip() for line in text.splitlines() if line.strip()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(summary_name, source_hash):
    """DRAM bytes per launch recorded in a profile summary, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_val = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_val or m_hash.group(1) != source_hash:
        return None
    return float(m_val.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU is under load."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].strip() not in ("", "[N/A]"))}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: each rank contributes its own and all receive the max."""
    if not torch.distributed.is_available() or not torch.distributed.is_initialized() or \
            torch.distributed.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_ms: float) -> float:
    """Units all ranks processed (independent replicas: weak scaling) per second of the
    slowest rank."""
    return units_per_rank * world / (max_ms / 1e3)


# ------------------------------------------------------------------ workloads

class DecodeWorkload:
    """Decode steps over a paged cache: append one token per sequence, then attend."""

    def __init__(self, spec, lengths, cycle, label, window=0, fp8=False, qlen=1, spare_blocks=0):
        self.spec, self.lengths, self.cycle, self.label = spec, list(lengths), cycle, label
        self.spare_blocks = spare_blocks   # physical blocks no sequence uses (free pool)
        self.num_splits = 0
        self.window = window   # > 0: sliding window of this many tokens
        self.fp8 = fp8         # E4M3 codes + one fp32 scale per cached row
        self.qlen = qlen       # new tokens per sequence per step, all verified at once
        self.copies = None     # copy-on-write block pairs run before each step's appends

    # bytes of K and V read by one step c of the cycle (every visible cached token, every
    # KV head; FP8: the code bytes and the row's 4-byte scale)
    def kv_bytes(self, c):
        row = self.spec.head_dim + 4 if self.fp8 else \
            self.spec.head_dim * (2 if self.spec.cache_dtype == torch.bfloat16 else 4)
        q = self.qlen
        seen = [n + q * (c + 1) if self.window <= 0 else min(n + q * (c + 1), self.window + q - 1)
                for n in self.lengths]
        return sum(seen) * self.spec.kv_heads * 2 * row

    # attention flops of step c (4 Hq d per visible (query, key) pair: scores and P.V)
    def attn_flops(self, c):
        q, s = self.qlen, self.spec
        pairs = sum(q * (n + q * c) + q * (q + 1) // 2 for n in self.lengths) if self.window <= 0 else None
        return None if pairs is None else 4 * s.q_heads * s.head_dim * pairs

    def sample_flops(self, n_seq):
        """Attention flops of one step of the oracle sample (its first n_seq sequences)."""
        q, s = self.qlen, self.spec
        return 4 * s.q_heads * s.head_dim * sum(q * n + q * (q + 1) // 2 for n in self.lengths[:n_seq])

    def tensor_bound(self, hbm_gbs, bf16_tflops):
        """Many query rows per sequence put the step above the bf16 / HBM ridge: it is then
        measured in attention TFLOP/s against the tensor roofline."""
        f = self.attn_flops(0) if self.qlen > 1 else None
        return bool(f) and f / self.kv_bytes(0) > bf16_tflops * 1e3 / hbm_gbs

    def describe(self):
        s = self.spec
        return {"workload": self.label, "batch": s.batch, "q_heads": s.q_heads, "kv_heads": s.kv_heads,
                "head_dim": s.head_dim, "block_size": s.block_size,
                "cache_dtype": "e4m3 codes + fp32 row scales" if self.fp8 else
                ("bf16" if s.cache_dtype == torch.bfloat16 else "fp32"),
                "q_dtype": "fp32", "mean_cached_len": sum(self.lengths) / len(self.lengths),
                "decode_steps_cycle": self.cycle, "window": self.window, "new_tokens_per_step": self.qlen,
                "kv_gb_per_step": self.kv_bytes(self.cycle // 2) / 1e9,
                "l2": "inputs larger than L2: each step reads %.2f GB of K/V vs 129 MB L2"
                      % (self.kv_bytes(0) / 1e9)}

    def setup(self, device):
        import paged_kv_cache_165_gb300 as pkv
        s = self.spec
        bs = s.block_size
        g = gen.generator(s.seed)
        nb = sum(gen.blocks_needed(n + self.cycle * self.qlen, bs) for n in self.lengths) + self.spare_blocks
        bm = pkv.BlockManager(nb, bs, order=gen.permutation(g, nb))
        for b, n in enumerate(self.lengths):
            bm.add_sequence(b, n)
        slots, clens = [], []
        for c in range(self.cycle):
            step = []
            for _ in range(self.qlen):   # token-major within a sequence: rows b*qlen + i
                sl, copies = bm.append_step(range(s.batch))
                assert not copies
                step.append(sl)
            slots.append(torch.tensor(step, dtype=torch.int64).t().reshape(-1))
            clens.append(bm.context_lens(range(s.batch)))
        self._finish_setup(device, pkv, bm, nb, slots, clens)

    def _finish_setup(self, device, pkv, bm, nb, slots, clens):
        s = self.spec
        bs = s.block_size
        self.nb = nb
        self.released_blocks = 0
        if self.window > 0:
            # blocks before every query's window go back to the pool (their table entries
            # become -1): this step's queries see positions len - window .. len - 1
            for b in range(s.batch):
                self.released_blocks += len(bm.release_outside_window(b, self.window))
        self.table = bm.block_table(range(s.batch)).to(device)
        self.slots_h = [t.pin_memory() for t in slots]
        self.clens_h = [t.pin_memory() for t in clens]
        self.slots = [t.to(device) for t in slots]
        self.clens = [t.to(device) for t in clens]
        cg = torch.Generator(device=device)
        cg.manual_seed(s.seed)
        shape = (nb, s.kv_heads, bs, s.head_dim)
        self.k_cache = torch.randn(shape, generator=cg, device=device, dtype=torch.float32).to(s.cache_dtype)
        self.v_cache = torch.randn(shape, generator=cg, device=device, dtype=torch.float32).to(s.cache_dtype)
        if self.fp8:
            # the same values quantised through the public append (all slots at once)
            rows = (nb * bs, s.kv_heads, s.head_dim)
            kq = torch.empty(shape, dtype=torch.uint8, device=device)
            vq = torch.empty_like(kq)
            self.k_scale = torch.empty(shape[:3], device=device)
            self.v_scale = torch.empty_like(self.k_scale)
            all_slots = torch.arange(nb * bs, device=device, dtype=torch.int64)
            pkv.kv_append_fp8(self.k_cache.transpose(1, 2).reshape(rows).contiguous(),
                              self.v_cache.transpose(1, 2).reshape(rows).contiguous(),
                              kq, vq, self.k_scale, self.v_scale, all_slots)
            self.k_cache, self.v_cache = kq, vq
        B, Hq, Hkv, d = s.batch, s.q_heads, s.kv_heads, s.head_dim
        R = B * self.qlen                # query rows per step
        new_dt = torch.bfloat16 if self.fp8 else s.cache_dtype
        self.q = torch.randn((self.cycle, R, Hq, d), generator=cg, device=device)
        self.k_new = torch.randn((self.cycle, R, Hkv, d), generator=cg, device=device).to(new_dt)
        self.v_new = torch.randn((self.cycle, R, Hkv, d), generator=cg, device=device).to(new_dt)
        self.out = torch.empty((R, Hq, d), device=device)
        self.lse = torch.empty((R, Hq), device=device)
        self.cu_q = torch.arange(B + 1, dtype=torch.int32, device=device) * self.qlen
        ws = pkv.paged_attention_workspace_bytes(B, R, self.qlen, Hq, Hkv, d, bs, self.table.shape[1],
                                                 self.window, self.num_splits)
        ws = max(ws, pkv.decode_workspace_bytes(B, Hq, Hkv, d, bs, self.table.shape[1], self.num_splits))
        self.ws = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)   # zeroed once
        self.splits = 1 if ws == 0 else None
        # end-to-end arm: each step's inputs (q, new K/V rows, slot mapping, context lengths)
        # packed into one pinned host buffer, as a serving loop stages them, so that one
        # host->device copy brings a step; the output returns into pinned host memory
        parts = [self.q.cpu(), self.k_new.cpu(), self.v_new.cpu(), torch.stack(slots), torch.stack(clens)]
        sizes = [t[0].numel() * t[0].element_size() for t in parts]
        offs = [0]
        for n in sizes:
            offs.append((offs[-1] + n + 255) // 256 * 256)
        self.stage_h = torch.empty((self.cycle, offs[-1]), dtype=torch.uint8).pin_memory()
        for c in range(self.cycle):
            for t, o, n in zip(parts, offs, sizes):
                self.stage_h[c, o:o + n] = t[c].contiguous().view(-1).view(torch.uint8)
        # two device staging buffers and two outputs: step k+1's inputs come in and step
        # k-1's output goes out on a copy stream while step k computes
        self.stage_d = [torch.empty(offs[-1], dtype=torch.uint8, device=device) for _ in range(2)]
        self.views = [[sd[o:o + n].view(t.dtype).view(t.shape[1:]) for t, o, n in zip(parts, offs, sizes)]
                      for sd in self.stage_d]
        self.out_e = [torch.empty((R, Hq, d), device=device) for _ in range(2)]
        self.out_h = [torch.empty((R, Hq, d)).pin_memory() for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=device)
        self.pkv = pkv
        # a plain decode step (one new token per sequence, no window) goes through
        # pkv_decode_step where the library appends inside the attention launch (as many
        # launches as the attention alone); otherwise kv_append, then the attention call, so
        # that the timed attention call is the attention's launches alone
        # (pkv_decode_step_fp8 on an FP8 cache, quantising the bf16 new rows)
        mbs = self.table.shape[1]
        if self.fp8:
            step_launches = pkv.decode_step_fp8_kernel_launches(B, Hq, Hkv, d, bs, mbs, nb, torch.bfloat16,
                                                                self.num_splits)
            attn_launches = pkv.decode_kernel_launches(B, Hq, Hkv, d, bs, mbs, nb, torch.uint8, self.num_splits)
        else:
            step_launches = pkv.decode_step_kernel_launches(B, Hq, Hkv, d, bs, mbs, nb, s.cache_dtype,
                                                            self.num_splits)
            attn_launches = pkv.decode_kernel_launches(B, Hq, Hkv, d, bs, mbs, nb, s.cache_dtype, self.num_splits)
        self.step_call = self.qlen == 1 and self.window <= 0 and step_launches == attn_launches
        if self.step_call:
            self.launches_per_step = step_launches
        else:
            self.launches_per_step = 1 + pkv.paged_attention_kernel_launches(
                B, R, self.qlen, Hq, Hkv, d, bs, self.table.shape[1], nb,
                torch.uint8 if self.fp8 else s.cache_dtype, self.window, self.num_splits)

    def decode(self, out, q, clens, lse=None):
        """The public decode call: pkv_paged_decode_attention, with a sliding window
        pkv_paged_attention (one query per sequence), or on an FP8 cache
        pkv_paged_decode_attention_fp8."""
        if self.fp8:
            self.pkv.paged_decode_attention_fp8(out, q, self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                                                self.table, clens, self.spec.scale, window=self.window, lse=lse,
                                                num_splits=self.num_splits, workspace=self.ws)
        elif self.qlen > 1:
            self.pkv.paged_attention(out, q, self.k_cache, self.v_cache, self.table, clens, self.spec.scale,
                                     cu_q=self.cu_q, max_q=self.qlen, window=self.window, lse=lse,
                                     num_splits=self.num_splits, workspace=self.ws)
        elif self.window <= 0:
            self.pkv.paged_decode_attention(out, q, self.k_cache, self.v_cache, self.table, clens,
                                            self.spec.scale, lse=lse, num_splits=self.num_splits,
                                            workspace=self.ws)
        else:
            self.pkv.paged_attention(out, q, self.k_cache, self.v_cache, self.table, clens, self.spec.scale,
                                     window=self.window, lse=lse, num_splits=self.num_splits,
                                     workspace=self.ws)

    def append(self, c):
        self.cache_append(self.k_new[c], self.v_new[c], self.slots[c])

    def cache_append(self, k_new, v_new, slots):
        """Copy-on-write of shared blocks, then the appends (which a decode step does itself)."""
        if self.copies is not None:   # copy-on-write of shared blocks before the writes
            self.pkv.kv_block_copy(self.k_cache, self.v_cache, self.copies)
        if self.step_call:
            return
        if self.fp8:
            self.pkv.kv_append_fp8(k_new, v_new, self.k_cache, self.v_cache, self.k_scale, self.v_scale, slots)
        else:
            self.pkv.kv_append(k_new, v_new, self.k_cache, self.v_cache, slots)

    def attend_call(self, out, q, k_new, v_new, slots, clens, lse=None):
        """The attention (with the step's appends, for a decode step) through the public API."""
        if self.step_call and self.fp8:
            self.pkv.decode_step_fp8(out, q, k_new, v_new, slots, self.k_cache, self.v_cache, self.k_scale,
                                     self.v_scale, self.table, clens, self.spec.scale, lse=lse,
                                     num_splits=self.num_splits, workspace=self.ws)
        elif self.step_call:
            self.pkv.decode_step(out, q, k_new, v_new, slots, self.k_cache, self.v_cache, self.table, clens,
                                 self.spec.scale, lse=lse, num_splits=self.num_splits, workspace=self.ws)
        else:
            self.decode(out, q, clens, lse=lse)

    def attend(self, c):
        self.attend_call(self.out, self.q[c], self.k_new[c], self.v_new[c], self.slots[c], self.clens[c],
                         lse=self.lse)

    def e2e_capture(self):
        """One CUDA graph per (cycle step c, buffer parity) of the public API calls a serving
        loop makes per step: compute of step k (decode_step, or kv_append + the attention, on the
        inputs in staging buffer k % 2) alongside, on a copy stream, the host->device copy of
        step k+1's inputs from pinned host memory into the other buffer and the
        device->host copy of step k-1's output.  Replaying them keeps the host out of the
        step's critical path (a few microseconds of host work per step)."""
        comp, cp = torch.cuda.current_stream(), self.copy_stream
        self.graphs = {}
        for c in range(self.cycle):
            for buf in range(2):
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream(device=self.stage_d[0].device)
                side.wait_stream(comp)
                with torch.cuda.graph(g, stream=side):
                    cs = torch.cuda.current_stream()
                    fork = torch.cuda.Event()
                    fork.record(cs)
                    cp.wait_event(fork)
                    with torch.cuda.stream(cp):
                        self.stage_d[1 - buf].copy_(self.stage_h[(c + 1) % self.cycle], non_blocking=True)
                        self.out_h[1 - buf].copy_(self.out_e[1 - buf], non_blocking=True)
                    q, kn, vn, sl, cl = self.views[buf]
                    self.cache_append(kn, vn, sl)
                    self.attend_call(self.out_e[buf], q, kn, vn, sl, cl)
                    join = torch.cuda.Event()
                    join.record(cp)
                    cs.wait_event(join)
                comp.wait_stream(side)
                self.graphs[(c, buf)] = g
        torch.cuda.synchronize()

    def e2e_steps(self, first, steps):
        """`steps` decode steps from pinned host inputs to the output in pinned host memory:
        the first step's inputs are copied in, each step's graph computes it while moving
        the neighbouring steps' inputs and outputs, and the last output is copied out."""
        self.stage_d[0].copy_(self.stage_h[first % self.cycle], non_blocking=True)
        for k in range(steps):
            self.graphs[((first + k) % self.cycle, k % 2)].replay()
        last = (steps - 1) % 2
        self.out_h[last].copy_(self.out_e[last], non_blocking=True)

    def e2e_bytes(self):
        return self.stage_h[0].numel(), self.out_h[0].numel() * 4

    # ---- CPU oracle on a bounded sample (same shapes and distribution, own draws)
    def oracle_sample(self, n_seq, steps=1):
        import oracle
        s = self.spec
        steps = max(steps, self.qlen)
        sub = gen.DecodeSpec(s.name + "_sample", s.seed + 77, n_seq, s.q_heads, s.kv_heads, s.head_dim,
                             s.cache_dtype, s.block_size, steps)
        inp = gen.decode_inputs(sub, self.lengths[:n_seq], steps=steps)
        bs = s.block_size
        threads = os.cpu_count() or 1
        if self.fp8:
            kq, ks = oracle.quantize_rows_e4m3(inp.k_cache)
            vq, vs = oracle.quantize_rows_e4m3(inp.v_cache)

        def run_verify(c):
            # qlen new tokens per sequence appended, then attended causally at once
            q = self.qlen
            for i in range(q):
                slots = torch.tensor([oracle.slot_of(inp.block_table[b], n + i, bs)
                                      for b, n in enumerate(inp.cached)])
                oracle.kv_append(inp.k_cache, inp.v_cache, inp.k_new[i], inp.v_new[i], slots)
            lens = torch.tensor([n + q for n in inp.cached], dtype=torch.int32)
            rows = torch.stack([inp.q[i] for i in range(q)], 1).reshape(-1, s.q_heads, s.head_dim)
            cu = torch.arange(len(inp.cached) + 1, dtype=torch.int32) * q
            oracle.paged_attention(rows, inp.k_cache, inp.v_cache, inp.block_table, lens, cu, s.scale,
                                   window=self.window, nthreads=threads)
            return int(lens.sum()) * s.kv_heads * s.head_dim * 2 * (2 if s.cache_dtype == torch.bfloat16 else 4)

        if self.qlen > 1:
            return run_verify, threads

        def run(c):
            slots = torch.tensor([oracle.slot_of(inp.block_table[b], n + c, bs)
                                  for b, n in enumerate(inp.cached)])
            lens = torch.tensor([n + c + 1 for n in inp.cached], dtype=torch.int32)
            if self.fp8:
                oracle.kv_append_fp8(kq, vq, ks, vs, inp.k_new[c], inp.v_new[c], slots)
                kc, vc = oracle.dequantize_fp8(kq, ks), oracle.dequantize_fp8(vq, vs)
            else:
                oracle.kv_append(inp.k_cache, inp.v_cache, inp.k_new[c], inp.v_new[c], slots)
                kc, vc = inp.k_cache, inp.v_cache
            if self.window <= 0:
                oracle.paged_decode(inp.q[c], kc, vc, inp.block_table, lens, s.scale, nthreads=threads)
                seen = lens
            else:
                cu = torch.arange(len(inp.cached) + 1, dtype=torch.int32)
                oracle.paged_attention(inp.q[c], kc, vc, inp.block_table, lens, cu, s.scale,
                                       window=self.window, nthreads=threads)
                seen = lens.clamp(max=self.window)
            row = s.head_dim + 4 if self.fp8 else s.head_dim * (2 if s.cache_dtype == torch.bfloat16 else 4)
            return int(seen.sum()) * s.kv_heads * 2 * row
        return run, threads


class MixWorkload(DecodeWorkload):
    """Continuous-batching mix: 256 sequences with lognormal lengths; sequences 0..63 share
    one 4096-token prefix and form 32 fork pairs that share their whole history, so the
    step's appends first copy each pair's shared partial last block (copy-on-write)."""

    def __init__(self):
        super().__init__(gen.MIX, gen.mix_lengths(), 1,
                         "continuous-batching mix: batch 256, 32 q / 8 kv heads, d 128, lognormal lengths "
                         "(median 1024, sigma 1, [16, 32768]); 64 sequences share a 4096-token prefix as "
                         "32 fork pairs, copy-on-write before the appends, bs 16, bf16 KV")

    def kv_bytes(self, c):
        # logical bytes: every sequence's tokens, shared or not (after this step's append)
        return sum(n + 1 for n in self.lengths) * self.spec.kv_heads * self.spec.head_dim * 2 * 2

    def setup(self, device):
        import paged_kv_cache_165_gb300 as pkv
        s = self.spec
        bs, B = s.block_size, s.batch
        P, S = gen.MIX_PREFIX_TOKENS, gen.MIX_PREFIX_SEQS
        unique = P + sum(n - (P if b < S else 0) for b, n in enumerate(self.lengths)
                         if not (b < S and b % 2 == 1))
        nb = gen.blocks_needed(unique, bs) + 2 * B + 64
        bm = pkv.BlockManager(nb, bs, order=gen.permutation(gen.generator(s.seed), nb))
        root = B                                    # the shared prefix, outside the batch
        bm.add_sequence(root, P)
        for b, n in enumerate(self.lengths):
            if b < S and b % 2 == 1:
                bm.fork(b - 1, b)                   # the pair shares its whole history
                continue
            if b < S:
                bm.fork(root, b)
                start = P
            else:
                bm.add_sequence(b, 0)
                start = 0
            for _ in range(start, n):
                bm.append_slot(b)
        bm.free_sequence(root)
        sl, copies = bm.append_step(range(B))
        bm.audit()
        # bytes of the distinct blocks read (the shared prefix and pair histories once)
        used = {}
        for b in range(B):
            n = bm.lengths[b]
            for j, blk in enumerate(bm.tables[b]):
                used[blk] = max(used.get(blk, 0), min(bs, n - j * bs))
        self.unique_bytes = sum(used.values()) * s.kv_heads * s.head_dim * 2 * 2
        self.n_copies = len(copies)
        self._finish_setup(device, pkv, bm, nb, [torch.tensor(sl, dtype=torch.int64)],
                           [bm.context_lens(range(B))])
        self.copies = torch.tensor(copies, dtype=torch.int32, device=device)
        # the 64 rows that start with the same physical blocks: their shared prefix is read once
        # per step (pkv_decode_step_shared_prefix), the rest of each row by the decode
        groups = bm.shared_prefix_groups(range(B))
        self.groups = groups.to(device)
        self.n_groups, self.prefix_tokens = groups.n_groups, groups.max_prefix_tokens
        mbs = self.table.shape[1]
        ws = pkv.decode_step_shared_prefix_workspace_bytes(B, s.q_heads, s.kv_heads, s.head_dim, bs, mbs, self.groups,
                                                           self.num_splits)
        if ws > self.ws.numel():
            self.ws = torch.zeros(ws, dtype=torch.uint8, device=device)
        self.step_call = True
        self.launches_per_step = 1 + pkv.decode_step_shared_prefix_kernel_launches(   # + kv_block_copy
            B, s.q_heads, s.kv_heads, s.head_dim, bs, mbs, nb, s.cache_dtype, self.groups, self.num_splits)

    def attend_call(self, out, q, k_new, v_new, slots, clens, lse=None):
        """The step's appends and attention through pkv_decode_step_shared_prefix."""
        self.pkv.decode_step_shared_prefix(out, q, k_new, v_new, slots, self.k_cache, self.v_cache, self.table,
                                           clens, self.spec.scale, self.groups, lse=lse, num_splits=self.num_splits,
                                           workspace=self.ws)

    def describe(self):
        d = super().describe()
        d.update({"cow_copies_per_step": getattr(self, "n_copies", None),
                  "unique_gb_per_step": getattr(self, "unique_bytes", 0) / 1e9,
                  "shared_prefix": {"groups": getattr(self, "n_groups", None),
                                    "prefix_tokens": getattr(self, "prefix_tokens", None),
                                    "call": "pkv_decode_step_shared_prefix"}})
        return d


class PrefillWorkload:
    """Varlen causal prefill of 8 prompts (lengths uniform in [256, 4096]) writing the cache."""

    def __init__(self):
        self.lengths = gen.long_prefill_lengths()
        self.hq, self.hkv, self.d, self.bs = 64, 8, 128, 16
        self.label = "long-context prefill: 8 prompts U[256,4096], 64 q / 8 kv heads, d 128, bf16"

    def flops(self):
        # causal: sum_b L(L+1)/2 query-key pairs x Hq x (2d for q.k + 2d for p.v)
        return sum(n * (n + 1) // 2 for n in self.lengths) * self.hq * 4 * self.d

    def describe(self):
        return {"workload": self.label, "prompt_lengths": self.lengths, "q_heads": self.hq,
                "kv_heads": self.hkv, "head_dim": self.d, "tflop_per_step": self.flops() / 1e12,
                "l2": "K/V of all prompts (%.0f MB) re-read from L2 across query tiles"
                      % (sum(self.lengths) * self.hkv * self.d * 4 / 1e6)}

    def setup(self, device):
        import paged_kv_cache_165_gb300 as pkv
        self.pkv = pkv
        p = gen.prefill_inputs(self.lengths, self.hq, self.hkv, self.d, torch.bfloat16, seed=4)
        self.p = p
        self.q, self.k, self.v = p.q.to(device), p.k.to(device), p.v.to(device)
        self.cu = p.cu_seqlens.to(device)
        nb = sum(gen.blocks_needed(n) for n in self.lengths)
        bm = pkv.BlockManager(nb, self.bs, order=gen.permutation(gen.generator(4), nb))
        for s, n in enumerate(self.lengths):
            bm.add_sequence(s, n)
        self.slots = torch.cat([bm.slot_mapping(s, range(n)) for s, n in enumerate(self.lengths)]).to(device)
        self.kc = torch.zeros((nb, self.hkv, self.bs, self.d), dtype=torch.bfloat16, device=device)
        self.vc = torch.zeros_like(self.kc)
        self.out = torch.empty((p.q.shape[0], self.hq, self.d), device=device)
        self.launches_per_step = 2

    def step(self, c):
        self.pkv.prefill_attention(self.out, self.q, self.k, self.v, self.cu, max(self.lengths),
                                   1 / math.sqrt(self.d), k_cache=self.kc, v_cache=self.vc,
                                   slot_mapping=self.slots)

    # ---- end to end: the step's inputs (q, k, v, slot mapping, cu_seqlens) copied in from
    # one pinned host buffer, the public call, the fp32 output copied back to pinned memory
    def e2e_setup(self):
        parts = [self.p.q, self.p.k, self.p.v, self.slots.cpu(), self.p.cu_seqlens]
        sizes = [t.numel() * t.element_size() for t in parts]
        offs = [0]
        for n in sizes:
            offs.append((offs[-1] + n + 255) // 256 * 256)
        self.stage_h = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
        for t, o, n in zip(parts, offs, sizes):
            self.stage_h[o:o + n] = t.contiguous().view(-1).view(torch.uint8)
        self.stage_d = torch.empty(offs[-1], dtype=torch.uint8, device=self.q.device)
        self.views = [self.stage_d[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, sizes)]
        self.out_h = torch.empty(tuple(self.out.shape)).pin_memory()

    def e2e_step(self):
        q, k, v, slots, cu = self.views
        self.stage_d.copy_(self.stage_h, non_blocking=True)
        self.pkv.prefill_attention(self.out, q, k, v, cu, max(self.lengths), 1 / math.sqrt(self.d),
                                   k_cache=self.kc, v_cache=self.vc, slot_mapping=slots)
        self.out_h.copy_(self.out, non_blocking=True)

    def e2e_bytes(self):
        return self.stage_h.numel(), self.out_h.numel() * 4

    # ---- CPU oracle on a bounded sample: the shortest prompts, about 300 GFLOP (seconds of fp64)
    def oracle_sample(self, flops=3e11):
        import oracle
        order = sorted(range(len(self.lengths)), key=lambda i: self.lengths[i])
        pick, fl = [], 0
        for i in order:
            pick.append(i)
            fl += self.lengths[i] * (self.lengths[i] + 1) // 2 * self.hq * 4 * self.d
            if fl >= flops:
                break
        lens = [self.lengths[i] for i in pick]
        p = gen.prefill_inputs(lens, self.hq, self.hkv, self.d, torch.bfloat16, seed=44)
        threads = os.cpu_count() or 1

        def run():
            oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 1 / math.sqrt(self.d), nthreads=threads)
            return fl
        return run, threads, lens


WORKLOADS = {
    "gqa70b": lambda: DecodeWorkload(gen.GQA_70B, gen.gqa_70b_lengths(), 32,
                                     "llama2-70b-shaped GQA decode: batch 64, 64 q / 8 kv heads, d 128, "
                                     "lengths U[512,8192], 32-step append+attend cycle, bs 16, bf16 KV"),
    "mha7b": lambda: DecodeWorkload(gen.MHA_7B, [gen.MHA_7B_LENGTH] * gen.MHA_7B.batch, 1,
                                    "llama2-7b-shaped MHA decode: batch 32, 32 q = 32 kv heads, d 128, "
                                    "2048 cached tokens, one append+attend step, bs 16, bf16 KV"),
    "long_gqa": lambda: DecodeWorkload(gen.LONG_GQA, [gen.LONG_LENGTH] * 4, 1,
                                       "long-context split-K GQA decode: batch 4, 64 q / 8 kv heads, d 128, "
                                       "131072 cached tokens, bs 16, bf16 KV"),
    "long_mqa": lambda: DecodeWorkload(gen.LONG_MQA, [gen.LONG_LENGTH] * 4, 1,
                                       "long-context split-K MQA decode: batch 4, 64 q / 1 kv head, d 128, "
                                       "131072 cached tokens, bs 16, bf16 KV"),
    "gqa70b_fp8": lambda: DecodeWorkload(gen.GQA_70B, gen.gqa_70b_lengths(), 32,
                                         "llama2-70b-shaped GQA decode on an FP8 cache (E4M3 codes, fp32 scale "
                                         "per row): batch 64, 64 q / 8 kv heads, d 128, lengths U[512,8192], "
                                         "32-step append+attend cycle, bs 16", fp8=True),
    "verify4": lambda: DecodeWorkload(gen.GQA_70B, gen.gqa_70b_lengths(), 1,
                                      "llama2-70b-shaped GQA verification step: batch 64, 64 q / 8 kv heads, "
                                      "d 128, lengths U[512,8192], 4 new tokens per sequence appended and "
                                      "attended causally, bs 16, bf16 KV", qlen=4),
    "prefix_chunk": lambda: DecodeWorkload(gen.PREFIX_CHUNK, [gen.PREFIX_LENGTH] * gen.PREFIX_CHUNK.batch, 1,
                                           "chunked prefill on a cached prefix: batch 8, 4096 cached tokens each, "
                                           "512 new tokens per sequence appended and attended causally (bottom-"
                                           "right), 64 q / 8 kv heads, d 128, bs 16, bf16 KV, fp32 q",
                                           qlen=gen.PREFIX_CHUNK_LEN),
    "tiny": lambda: DecodeWorkload(gen.TINY, list(gen.TINY_LENGTHS), 1,
                                   "tiny decode step: batch 2, 8 q / 2 kv heads, d 64, lengths {17, 40} + 1 "
                                   "appended, bs 16, 8 physical blocks in seeded-permutation order, fp32 q/K/V",
                                   spare_blocks=gen.TINY_NUM_BLOCKS - sum(gen.blocks_needed(n + 1)
                                                                          for n in gen.TINY_LENGTHS)),
    "mix": MixWorkload,
    "swa": lambda: DecodeWorkload(gen.SWA, [gen.SWA_LENGTH] * gen.SWA.batch, 1,
                                  "mistral-7b-shaped sliding-window decode: batch 64, 32 q / 8 kv heads, d 128, "
                                  "16384 cached tokens, window 4096 (blocks outside released), bs 16, bf16 KV",
                                  window=gen.SWA_WINDOW),
    "prefill": PrefillWorkload,
}


# ------------------------------------------------------------------- our arm

def measure(name, wl, args, device, world, rank, steps, warmup, soak, with_e2e=True, cpu_sample=None,
            cpu_seconds=0.0):
    """Set the workload up, warm it up, time exactly `steps` steps (events on the launching
    stream, barriers and the max over ranks around them) with clocks sampled meanwhile, and
    return the result keys of one JSON line.  cpu_sample: None for no CPU baseline, else the
    oracle sample size (sequences for a decode workload, fp64 flops for the prefill), run
    again and again until cpu_seconds have passed."""
    import paged_kv_cache_165_gb300 as pkv
    if hasattr(wl, "num_splits"):
        wl.num_splits = args.num_splits
    wl.setup(device)
    is_decode = isinstance(wl, DecodeWorkload)
    stream = torch.cuda.current_stream()

    def step(i):
        c = i % wl.cycle if is_decode else 0
        if is_decode:
            wl.append(c)
            wl.attend(c)
        else:
            wl.step(c)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    # soak (untimed) so that clocks settle and the sampler sees the GPU under load
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    t_end = time.time() + soak
    i = warmup
    while time.time() < t_end:
        step(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # ---- timed region: exactly `steps` steps, events on the launching stream
    first = i
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(steps):
        c = (first + k) % wl.cycle if is_decode else 0
        if is_decode:
            wl.append(c)
            ev_a[k].record(stream)
            wl.attend(c)
            ev_b[k].record(stream)
        else:
            ev_a[k].record(stream)
            wl.step(c)
            ev_b[k].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    elapsed_ms = start.elapsed_time(stop)
    kernel_ms = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error during the timed region")
    max_ms = max_over_ranks(elapsed_ms, device)

    hbm, bf16, bf16_sus, peak_kind = peaks()
    ms_per_step = max_ms / steps
    res = {"metric": METRIC, "impl": "ours"}
    step_flops = None
    if is_decode:
        step_bytes = [wl.kv_bytes((first + k) % wl.cycle) for k in range(steps)]
        value = whole_job_rate(sum(step_bytes), world, max_ms) / 1e9
        kern_avg_ms = sum(kernel_ms) / len(kernel_ms)
        # bytes HBM has to deliver per launch: with shared blocks (a common prefix, forked
        # histories) each distinct block once, the logical bytes staying the metric's value
        alg_bytes = getattr(wl, "unique_bytes", None) or sum(step_bytes) / len(step_bytes)
        achieved = alg_bytes / (kern_avg_ms / 1e3) / 1e9
        files = ["decode.cu", "decode_kparams.cuh", "decode_epilogue.cuh", "common.cuh"]
        if wl.fp8:
            files += ["decode_fp8.cu", "fp8_codes.cuh"]
        elif getattr(wl, "groups", None) is not None:
            files.append("paged_prefill.cu")    # the shared-prefix kernel and merge
        elif wl.qlen >= 64 and wl.window <= 0:
            files.append("paged_prefill.cu")    # the chunked-prefill kernel (many query rows)
        elif wl.spec.q_heads // wl.spec.kv_heads > 8 or wl.qlen > 1:
            files.append("decode_umma.cu")      # the tcgen05 kernel (large groups, query rows)
        src = kernel_source_hash(files)
        traffic = profiled_traffic(f"decode_{name}.md", src)
        res.update({
            "value": value, "unit": "GB/s", "pct_hbm_peak": 100 * value / hbm,
            "tokens_per_s_per_layer": wl.spec.batch * wl.qlen * world / (ms_per_step / 1e3),
            **({"attention_tflops": world * sum(wl.attn_flops((first + k) % wl.cycle) for k in range(steps))
                / (max_ms / 1e3) / 1e12}
               if wl.qlen > 1 and wl.window <= 0 else {}),
            **({"unique_gb_per_s": whole_job_rate(wl.unique_bytes * steps, world, max_ms) / 1e9}
               if hasattr(wl, "unique_bytes") else {}),
            "roofline": {"bound": "hbm", "kernel": "paged_decode_attention (split-K partials + LSE merge)",
                         "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s",
                         "algorithmic_bytes_per_launch": alg_bytes,
                         **({"logical_bytes_per_launch": sum(step_bytes) / len(step_bytes)}
                            if hasattr(wl, "unique_bytes") else {}),
                         "avg_launch_ms": kern_avg_ms,
                         "traffic": traffic, "kernel_source_sha256_16": src},
        })
        step_flops = [wl.attn_flops((first + k) % wl.cycle) for k in range(steps)] \
            if wl.qlen > 1 and wl.window <= 0 else None
        if step_flops and wl.tensor_bound(hbm, bf16):
            # many query rows per sequence (chunked prefill on a cached prefix): the work is
            # above the bf16 / HBM ridge, so the metric is attention TFLOP/s against the
            # tensor roofline; the cache-read rate stays as a key of its own
            flops = sum(step_flops) / len(step_flops)
            ach = flops / (kern_avg_ms / 1e3) / 1e12
            res.update({
                "metric": "chunked prefill on a cached prefix: attention TFLOP/s (4*Hq*d per visible query-key pair)",
                "value": res["attention_tflops"], "unit": "TFLOP/s", "kv_read_gb_per_s": value,
                "roofline": {"bound": "tensor", "kernel": "paged_attention (query rows over the cache)",
                             "achieved": ach, "peak": bf16, "unit": "TFLOP/s", "frac": ach / bf16,
                             "peak_source": "measured bf16_tflops (burst)" if peak_kind == "measured"
                             else "fallback 1.9 PFLOP/s",
                             "frac_of_sustained": ach / bf16_sus, "peak_sustained": bf16_sus,
                             "algorithmic_flops_per_launch": flops, "avg_launch_ms": kern_avg_ms,
                             "traffic": traffic, "kernel_source_sha256_16": src},
            })
    else:
        flops = wl.flops()
        value = whole_job_rate(flops * steps, world, max_ms) / 1e12
        kern_avg_ms = sum(kernel_ms) / len(kernel_ms)
        achieved = flops / (kern_avg_ms / 1e3) / 1e12
        src = kernel_source_hash(["prefill.cu", "common.cuh"])
        res.update({
            "metric": "varlen causal prefill TFLOP/s (4*Hq*d per causal query-key pair)",
            "value": value, "unit": "TFLOP/s",
            "prompt_tokens_per_s_per_layer": sum(wl.lengths) * world / (ms_per_step / 1e3),
            "roofline": {"bound": "tensor", "kernel": "prefill_attention (cache write + attention)",
                         "achieved": achieved, "peak": bf16, "unit": "TFLOP/s", "frac": achieved / bf16,
                         "peak_source": f"{peak_kind} bf16_tflops (burst)",
                         # the step loop runs seconds under the power cap: the sustained GEMM rate
                         "frac_of_sustained": achieved / bf16_sus, "peak_sustained": bf16_sus,
                         "avg_launch_ms": kern_avg_ms,
                         "traffic": profiled_traffic("prefill.md", src), "kernel_source_sha256_16": src},
        })
    res.update({
        "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if not is_decode or wl.spec.cache_dtype == torch.bfloat16 else "fp32",
        "accumulate": "fp32", "data": "synthetic (seeded N(0,1), shuffled blocks)",
        "config": dict(wl.describe(), parallelism=f"replicas x{world} (independent batches)",
                       soak_s=soak, num_splits=args.num_splits),
        "gpu_launches": wl.launches_per_step * steps,
        "clocks": clocks,
    })

    # ---- end to end through the public API with pinned host buffers
    if with_e2e and is_decode:
        wl.e2e_capture()
        # warm-up: the very steps the timed region replays, so that every graph it uses has
        # been launched (uploaded to the device) once; the steps are idempotent (the same
        # appends to the same slots)
        wl.e2e_steps(first, steps)
        torch.cuda.synchronize()
        e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e_start.record(stream)
        wl.e2e_steps(first, steps)
        e_stop.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e_start.elapsed_time(e_stop), device)
        # the last step's output, as it reached host memory, equals the same step run eagerly
        last_c, last_buf = (first + steps - 1) % wl.cycle, (steps - 1) % 2
        wl.append(last_c)
        wl.attend(last_c)
        if not torch.equal(wl.out_h[last_buf], wl.out.cpu()):
            raise RuntimeError("end-to-end output differs from the eager step")
        h2d, d2h = wl.e2e_bytes()
        tb = res["unit"] == "TFLOP/s"   # the tensor-bound query-row workload: the same metric
        res["e2e"] = {"value": whole_job_rate(sum(step_flops) if tb else sum(step_bytes), world, e_ms)
                      / (1e12 if tb else 1e9), "unit": res["unit"],
                      "ms_per_step": e_ms / steps, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h,
                      "kind": "pipelined throughput: steps back to back, each step's copies overlapped "
                              "with its neighbours' compute; not the host-to-host latency of one step",
                      "path": "public API calls (decode_step, or kv_append then the attention) replayed as one "
                              "CUDA graph per step; step k+1's inputs copied in from pinned host "
                              "memory and step k-1's output copied out on a second stream while "
                              "step k computes"}
    elif with_e2e:
        wl.e2e_setup()
        for _ in range(2):
            wl.e2e_step()
        torch.cuda.synchronize()
        e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e_start.record(stream)
        for _ in range(steps):
            wl.e2e_step()
        e_stop.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e_start.elapsed_time(e_stop), device)
        # the output, as it reached host memory, equals the same step run on device inputs
        wl.step(0)
        if not torch.equal(wl.out_h, wl.out.cpu()):
            raise RuntimeError("end-to-end output differs from the eager step")
        h2d, d2h = wl.e2e_bytes()
        res["e2e"] = {"value": whole_job_rate(wl.flops() * steps, world, e_ms) / 1e12, "unit": "TFLOP/s",
                      "ms_per_step": e_ms / steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "kind": "one step after another on one stream (copy in, compute, copy out)",
                      "path": "public API call (prefill_attention writing the cache) on inputs copied in "
                              "from one pinned host buffer, the fp32 output copied back to pinned host "
                              "memory, one step after another"}

    # ---- CPU oracle baseline (rank 0, one GPU only)
    if world == 1 and rank == 0 and cpu_sample is not None and not is_decode:
        run, threads, lens = wl.oracle_sample(cpu_sample)
        t0 = time.perf_counter()
        fl, reps = 0, 0
        while reps == 0 or time.perf_counter() - t0 < cpu_seconds:
            fl += run()
            reps += 1
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                               "sample": f"causal prefill of the {len(lens)} shortest prompts (lengths {lens}, "
                                         f"same shapes, own seeded draws), {reps} times, fp64 C oracle, "
                                         f"{threads} threads, {dt:.2f} s"}
    if world == 1 and rank == 0 and cpu_sample is not None and is_decode:
        tb = wl.tensor_bound(hbm, bf16)
        n_seq = 1 if tb else min(cpu_sample, wl.spec.batch)
        csteps = wl.cycle if wl.qlen == 1 else 1
        run, threads = wl.oracle_sample(n_seq, steps=csteps)
        t0 = time.perf_counter()
        nbytes, reps = 0, 0
        while reps == 0 or time.perf_counter() - t0 < cpu_seconds:
            nbytes += run(reps % csteps)   # the cycle's steps in order, then again (idempotent appends)
            reps += 1
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": wl.sample_flops(n_seq) * reps / dt / 1e12 if tb else nbytes / dt / 1e9,
                               "unit": "TFLOP/s" if tb else "GB/s", "cores": threads,
                               "kind": "oracle",
                               "sample": f"{reps} append+attend steps of {n_seq} of the {wl.spec.batch} "
                                         f"sequences (same lengths and shapes, own seeded draws), "
                                         f"fp64 C oracle, {threads} threads, {dt:.2f} s"}
    return res


# The five configurations of the workload set, with the CPU-oracle sample each is timed on
# beside it (sequences of a decode step, or fp64 flops of the shortest prompts), repeated for
# --config-cpu-seconds.
CONFIG_SET = [
    ("1_tiny", "tiny", 2),   # 60 KB of K/V: the time is launch latency, not HBM
    ("2_llama2_7b_mha", "mha7b", 8),
    ("3_llama2_70b_gqa", "gqa70b", 16),
    ("4_mix_prefix_share", "mix", 16),
    ("5_long_gqa", "long_gqa", 1),
    ("5_long_mqa", "long_mqa", 1),
    ("5_prefill", "prefill", 5e10),
]

CONFIG_KEYS = ("workload", "value", "unit", "ms_per_step", "pct_hbm_peak", "tokens_per_s_per_layer",
               "prompt_tokens_per_s_per_layer", "unique_gb_per_s", "gpu_launches", "cpu_baseline")


def config_summary(res):
    """The keys of one workload's line that the configs object carries."""
    out = {k: res[k] for k in CONFIG_KEYS if k in res}
    out["workload"] = res["config"]["workload"]
    r = res["roofline"]
    out["roofline"] = {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac", "avg_launch_ms")}
    out["steps"], out["warmup"] = res["steps"], res["warmup"]
    out["clocks"] = {k: res["clocks"].get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")} \
        if res.get("clocks") else None
    return out


def bench_ours(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    import paged_kv_cache_165_gb300 as pkv
    from paged_kv_cache_165_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    pkv.lib()

    cpu = None if args.no_cpu_baseline else (args.cpu_seqs if args.workload != "prefill" else 3e11)
    res = measure(args.workload, WORKLOADS[args.workload](), args, device, world, rank, args.steps, args.warmup, args.soak,
                  with_e2e=True, cpu_sample=cpu, cpu_seconds=args.cpu_seconds)
    torch.cuda.empty_cache()

    # ---- every configuration of the workload set at one GPU, each with its CPU-oracle
    # baseline: the same measurement, fewer steps, no end-to-end pass
    if world == 1 and rank == 0 and not args.no_configs and args.workload == "gqa70b":
        configs = {}
        for key, name, sample in CONFIG_SET:
            if name == args.workload:
                line = dict(res)
            else:
                line = measure(name, WORKLOADS[name](), args, device, 1, 0, args.config_steps, args.warmup,
                               args.config_soak, with_e2e=False,
                               cpu_sample=None if args.no_cpu_baseline else sample,
                               cpu_seconds=args.config_cpu_seconds)
                torch.cuda.empty_cache()
            configs[key] = config_summary(line)
            if name == "tiny":
                configs[key]["note"] = ("correctness-size step (60 KB of K/V): its time is launch latency, "
                                        "so its GB/s and roofline fraction say nothing about HBM")
        res["configs"] = configs
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))


# ------------------------------------------------------------ reference arm

def bench_reference(args):
    """The fp64 CPU oracle as the reference arm, on a bounded sample per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]()
    if not isinstance(wl, DecodeWorkload):
        print(json.dumps({"impl": "reference", "unavailable": "reference arm covers the decode workloads"}))
        return
    hbm, bf16, _, _ = peaks()
    tb = wl.tensor_bound(hbm, bf16)
    n_seq = 1 if tb else args.ref_seqs
    run, threads = wl.oracle_sample(n_seq, steps=wl.cycle)
    for k in range(args.warmup):
        run(k % wl.cycle)
    t0 = time.perf_counter()
    nbytes = 0
    for k in range(args.steps):
        nbytes += run((args.warmup + k) % wl.cycle)
    dt = time.perf_counter() - t0
    value = wl.sample_flops(n_seq) * args.steps / dt / 1e12 if tb else nbytes / dt / 1e9
    unit = "TFLOP/s" if tb else "GB/s"
    metric = ("chunked prefill on a cached prefix: attention TFLOP/s (4*Hq*d per visible query-key pair)"
              if tb else METRIC)
    sample = (f"each step: one append+attend step of {n_seq} of the {wl.spec.batch} sequences "
              f"(same lengths and shapes, own seeded draws), fp64 C oracle, {threads} threads")
    print(json.dumps({
        "metric": metric, "impl": "reference", "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": wl.describe(),
        "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gqa70b", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--num-splits", type=int, default=0,
                    help="decode split-K chunks per sequence (0: the library's plan)")
    ap.add_argument("--soak", type=float, default=1.5, help="untimed seconds before the timed steps")
    ap.add_argument("--cpu-seqs", type=int, default=64,
                    help="sequences in the CPU-baseline sample (one step)")
    ap.add_argument("--ref-seqs", type=int, default=8,
                    help="sequences per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration measurements of the default run")
    ap.add_argument("--config-steps", type=int, default=20, help="timed steps of each configuration")
    ap.add_argument("--config-soak", type=float, default=0.3, help="untimed seconds before each configuration")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="the CPU-oracle baseline repeats its sample for at least this long")
    ap.add_argument("--config-cpu-seconds", type=float, default=4.0,
                    help="the same for each configuration of the default run")
    args = ap.parse_args()
    args.warmup_requested = args.warmup
    args.warmup = max(args.warmup, 3)     # at least three untimed warm-up steps
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
