"""Benchmark: MASW draft-attention decode steps/s and HBM GB/s vs full-KV
attention at a 32K prefix, on the 3B-draft-shaped workload (28 layers, batch 8,
24 query / 8 kv heads, head_dim 128, bf16, S=4 sink, W=1024 window, r=512).

One bench step = one speculative draft iteration of L_draft = 5 decode steps:
per step and layer, append the new token's K/V and run draft attention over the
compressed memory; at the fourth step every sequence crosses the compression
boundary tau_62 = 32772, so a slot is written per layer right after that step's
attention; the iteration ends by rolling the 5 speculative tokens back (as
after a fully rejected draft), so every iteration starts from the same 32K
state.  The iteration is captured once as a CUDA graph and replayed.  `value`
counts decode steps (5 per bench step) per second.  The full-KV contrast runs
the same loop with full-KV decode attention over the uncompressed cache.

Inputs are synthetic N(0,1) bf16 (no datasets or weights are involved); the
per-step working set (about 1 GB of K/V) is larger than the 129 MB L2, so no
explicit flush is needed between iterations.
"""
from __future__ import annotations

import argparse
import functools
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "draft3b_28l_b8"
METRIC = "MASW draft-attn decode steps/s (28 layers x batch 8, 32K prefix)"
UNIT = "decode steps/s"


def _code_only(src: str) -> str:
    """C/CUDA source with comments, trailing blanks and empty lines removed."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip())


def _code_hash(paths):
    """sha256 (first 16 hex) of the code of C/CUDA sources: edits to comments
    leave it unchanged."""
    import hashlib
    h = hashlib.sha256()
    for path in paths:
        with open(path) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _recorded_traffic():
    """dram read+write bytes per launch of the fused-step kernel from the
    committed ncu summary, if the kernel code is unchanged since (code hash of
    masw_decode_mma.cu + masw_internal.cuh); None otherwise."""
    import re
    try:
        csrc = os.path.join(ROOT, "compressed_draft_kv_gb300", "csrc")
        code = _code_hash([os.path.join(csrc, n) for n in ("masw_decode_mma.cu", "masw_internal.cuh")])
        with open(os.path.join(ROOT, "profiles", "decode_mma_step_b8_32k.md")) as f:
            txt = f.read()
        rec = re.search(r"first 16 hex\): `([0-9a-f]{16})`", txt)
        val = re.search(r"traffic_bytes_per_launch: (\d+)", txt)
        if rec and val and rec.group(1) == code:
            return int(val.group(1))
    except OSError:
        pass
    return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _peaks_tensor():
    """Dense bf16 tensor peak: the measured cuBLAS burst figure (prefill launches
    are timed in short bursts), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (burst)"
    except Exception:
        return 1900.0, "fallback"


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during a timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- GPU bench --

def workload_prefixes(w: dict, synth) -> list[int]:
    """Per-sequence prefix lengths.  Fixed-prefix workloads: the same prefix for
    every sequence.  Ragged workloads: uniform on [prefix_lo, prefix_hi], each
    snapped down to the nearest length at which sequence b reaches a
    compression boundary at draft step (b mod steps) + 1, so every iteration
    crosses boundaries at staggered steps."""
    if "prefix" in w:
        return [w["prefix"]] * w["batch"]
    base = synth.ragged_prefixes(w["batch"], w["prefix_lo"], w["prefix_hi"], w["seed"])
    out = []
    for b, p0 in enumerate(base):
        s_b = b % w["steps"] + 1
        target = (w["S"] + w["W"] - s_b) % w["r"]
        out.append(p0 - ((p0 - target) % w["r"]))
    return out


class DraftBench:
    """One speculative draft iteration of a workload, captured as a CUDA graph."""

    def __init__(self, torch, capi, synth, workload: str, prefix: int | None = None, batch: int | None = None):
        self.torch, self.capi = torch, capi
        w = dict(synth.WORKLOADS[workload])
        if prefix is not None:
            w["prefix"] = prefix
            w.pop("prefix_lo", None)
        if batch is not None:
            w["batch"] = batch
        self.w = w
        self.L, self.B, self.Hq, self.Hkv, self.D = w["layers"], w["batch"], w["Hq"], w["Hkv"], w["D"]
        self.S, self.W, self.r = w["S"], w["W"], w["r"]
        self.steps = w["steps"]
        self.R = 16                      # the pages' 16-token raw-KV rollback window
        self.prefixes = workload_prefixes(w, synth)
        pmax = max(self.prefixes)
        self.dev = torch.device("cuda", torch.cuda.current_device())
        dt = torch.bfloat16
        self.h = capi.masw_mem_create(self.S, self.W, self.r, self.Hkv, self.D, self.L, batch=self.B,
                                      dtype=capi.MASW_BF16, max_seq_len=pmax + 32, full_kv=True,
                                      rollback_reserve=self.R)
        nmax = max(0, (pmax - self.S - self.W) // self.r)
        g = torch.Generator(device=self.dev)
        g.manual_seed(2)
        # four distinct seeded N(0,1) draws, reused across (layer, sequence) blocks
        draws = []
        for _ in range(4):
            kr = torch.randn(pmax, self.Hkv, self.D, generator=g, device=self.dev).to(dt)
            vr = torch.randn(pmax, self.Hkv, self.D, generator=g, device=self.dev).to(dt)
            ks = torch.randn(max(nmax, 1), self.Hkv, self.D, generator=g, device=self.dev).to(dt)
            vs = torch.randn(max(nmax, 1), self.Hkv, self.D, generator=g, device=self.dev).to(dt)
            draws.append((kr, vr, ks, vs))
        for l in range(self.L):
            for b in range(self.B):
                kr, vr, ks, vs = draws[(l * self.B + b) % 4]
                t = self.prefixes[b]
                n = max(0, (t - self.S - self.W) // self.r)
                capi.masw_mem_load(self.h, l, b, kr[:t], vr[:t], ks[:n] if n else None, vs[:n] if n else None)
        del draws
        torch.cuda.empty_cache()
        rn = lambda *shape: torch.randn(*shape, generator=g, device=self.dev).to(dt)
        self.q = [[rn(self.B, self.Hq, self.D) for _ in range(self.L)] for _ in range(self.steps)]
        self.k = [[rn(self.B, self.Hkv, self.D) for _ in range(self.L)] for _ in range(self.steps)]
        self.v = [[rn(self.B, self.Hkv, self.D) for _ in range(self.L)] for _ in range(self.steps)]
        self.qg = [rn(self.B, self.Hq, self.D) for _ in range(self.L)]
        self.kg = [rn(self.B, self.Hkv, self.D) for _ in range(self.L)]
        self.vg = [rn(self.B, self.Hkv, self.D) for _ in range(self.L)]
        self.o = [[torch.empty(self.B, self.Hq, self.D, device=self.dev) for _ in range(self.L)]
                  for _ in range(self.steps)]
        self.lse = [[torch.empty(self.B, self.Hq, device=self.dev) for _ in range(self.L)]
                    for _ in range(self.steps)]
        self.og = [torch.empty(self.B, self.Hq, self.D, device=self.dev) for _ in range(self.L)]
        self.seqs = list(range(self.B))
        # sequences that reach a compression boundary at each draft step
        self.due = []
        for s_ in range(self.steps):
            d = []
            for b in range(self.B):
                t = self.prefixes[b] + s_ + 1
                if t >= self.S + self.W + self.r and (t - self.S - self.W) % self.r == 0:
                    d.append(b)
            self.due.append(d)
        self.stream = torch.cuda.Stream(device=self.dev)

    # one speculative iteration through the C-ABI: per step and layer one fused
    # append + attention launch (carrying the slot writes of the sequences at a
    # boundary), then the rollback of the speculative tokens
    def iteration(self, full: bool = False):
        c = self.capi
        launches = 0
        for s_ in range(self.steps):
            due = self.due[s_]
            for l in range(self.L):
                if full:
                    c.masw_full_step(self.h, l, self.q[s_][l], self.k[s_][l], self.v[s_][l], self.o[s_][l],
                                     self.lse[s_][l])
                elif due:
                    n = len(due)
                    c.masw_draft_step_slot(self.h, l, self.q[s_][l], self.k[s_][l], self.v[s_][l], self.o[s_][l],
                                           due, self.qg[l][:n], self.kg[l][:n], self.vg[l][:n], self.og[l][:n],
                                           lse=self.lse[s_][l])
                else:
                    c.masw_draft_step(self.h, l, self.q[s_][l], self.k[s_][l], self.v[s_][l], self.o[s_][l],
                                      self.lse[s_][l])
                launches += 1
        c.masw_rollback(self.h, self.seqs, self.prefixes)
        return launches + 1

    def capture(self, fn):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            fn()                     # eager warm-up (also configures kernels)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            n = fn()
        torch.cuda.synchronize()
        return g, n

    def time_graph(self, g, warmup: int, steps: int, barrier=None):
        """Seconds for `steps` back-to-back replays (first to last event), after
        `warmup` untimed ones; an event between replays also gives each replay's
        own duration, whose median is kept in self.last_median_s."""
        torch = self.torch
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        if barrier:
            barrier()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        with torch.cuda.stream(self.stream):
            ev[0].record(self.stream)
            for i in range(steps):
                g.replay()
                ev[i + 1].record(self.stream)
        torch.cuda.synchronize()
        if barrier:
            barrier()
        torch.cuda.synchronize()
        per = [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(steps)]
        self.last_median_s = statistics.median(per)
        return ev[0].elapsed_time(ev[steps]) / 1e3

    def kv_bytes_per_decode_step(self, full: bool = False):
        """K/V bytes one decode step reads over all layers and sequences (at the
        first draft step of the iteration)."""
        E = 2 * self.Hkv * self.D * 2
        tot = 0
        for t0 in self.prefixes:
            t = t0 + 1
            if full:
                rows = t
            else:
                rows = min(self.S, t) + max(0, min(self.W, t - self.S)) + max(0, (t - self.S - self.W) // self.r)
            tot += rows * E
        return tot * self.L

    def algorithmic_bytes_per_draft_launch(self):
        """One fused draft step of one layer at t = prefix+1: the working set
        (sink + window + slots, K and V, 2*Hkv*D*2 bytes per entry) of every
        sequence, plus Q (bf16), the new token's K/V (read once, written to the
        pool and to the full-KV cache) and O, LSE (fp32)."""
        E = 2 * self.Hkv * self.D * 2
        kv = self.kv_bytes_per_decode_step() // self.L
        other = self.B * self.Hq * self.D * 2 + self.B * E * 3 + self.B * self.Hq * (self.D + 1) * 4
        return kv + other, kv, other

    def time_draft_kernel(self, reps: int):
        """Average duration of one fused masw_draft_step launch, timed with
        CUDA events on the launching stream over `reps` replays of a graph of
        the per-layer launches of one decode step followed by the one-token
        rollback that restores the state (counted against the step launches)."""
        c = self.capi

        def step():
            for l in range(self.L):
                c.masw_draft_step(self.h, l, self.q[0][l], self.k[0][l], self.v[0][l], self.o[0][l],
                                  self.lse[0][l])
            c.masw_rollback(self.h, self.seqs, self.prefixes)
            return self.L
        g, n = self.capture(step)
        secs = self.time_graph(g, 3, reps)
        return secs / (reps * n), n * reps

    def e2e(self, iters: int):
        """The same iteration through the public API with host buffers: every
        iteration copies all of its inputs (q, k, v of every decode step and
        layer, the slot tokens' q, k, v) in from a pinned host buffer, makes the
        library calls eagerly (no graph), and reads every O back into a pinned
        host buffer, all inside the timed region.  Device and host buffers are
        doubled so that, on a second stream, iteration i+1's inputs are copied in
        and iteration i's outputs copied out while iteration i+1 computes (one
        copy each way per iteration, ordered by events)."""
        torch, c = self.torch, self.capi
        ins = [x for row in self.q for x in row] + [x for row in self.k for x in row] + \
              [x for row in self.v for x in row] + list(self.qg) + list(self.kg) + list(self.vg)
        offs, tot = [], 0
        for x in ins:
            offs.append(tot)
            tot += x.numel() * x.element_size()
        SL = self.steps * self.L
        n_out = SL * self.B * self.Hq * self.D + self.L * self.qg[0].shape[0] * self.Hq * self.D
        per = self.B * self.Hq * self.D
        pg = self.qg[0].shape[0] * self.Hq * self.D
        host_in = torch.empty(tot, dtype=torch.uint8).pin_memory()
        for x, o_ in zip(ins, offs):
            n = x.numel() * x.element_size()
            host_in[o_:o_ + n].copy_(x.reshape(-1).view(torch.uint8).cpu())
        host_out = [torch.empty(n_out).pin_memory() for _ in range(2)]
        bufs = []
        for _ in range(2):
            dev_in = torch.empty(tot, dtype=torch.uint8, device=self.dev)
            views = [dev_in[o_:o_ + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for x, o_ in zip(ins, offs)]
            dev_out = torch.empty(n_out, device=self.dev)
            bufs.append({
                "in": dev_in, "out": dev_out,
                "q": [views[i * self.L:(i + 1) * self.L] for i in range(self.steps)],
                "k": [views[SL + i * self.L:SL + (i + 1) * self.L] for i in range(self.steps)],
                "v": [views[2 * SL + i * self.L:2 * SL + (i + 1) * self.L] for i in range(self.steps)],
                "qg": views[3 * SL:3 * SL + self.L], "kg": views[3 * SL + self.L:3 * SL + 2 * self.L],
                "vg": views[3 * SL + 2 * self.L:],
                "o": [[dev_out[(s_ * self.L + l) * per:(s_ * self.L + l + 1) * per].view(self.B, self.Hq, self.D)
                       for l in range(self.L)] for s_ in range(self.steps)],
                "og": [dev_out[SL * per + l * pg:SL * per + (l + 1) * pg].view(-1, self.Hq, self.D)
                       for l in range(self.L)],
            })
        st = self.stream
        cs = torch.cuda.Stream(device=self.dev)
        ev = lambda: torch.cuda.Event()
        h2d, d2h = tot, n_out * 4

        # each buffer's iteration as a list of bound library calls (built once,
        # so the timed loop spends its host time in the calls themselves)
        sh = st.cuda_stream
        for bf in bufs:
            calls = []
            for s_ in range(self.steps):
                due = self.due[s_]
                for l in range(self.L):
                    if due:
                        n = len(due)
                        calls.append(functools.partial(
                            c.masw_draft_step_slot, self.h, l, bf["q"][s_][l], bf["k"][s_][l], bf["v"][s_][l],
                            bf["o"][s_][l], due, bf["qg"][l][:n], bf["kg"][l][:n], bf["vg"][l][:n],
                            bf["og"][l][:n], stream=sh))
                    else:
                        calls.append(functools.partial(c.masw_draft_step, self.h, l, bf["q"][s_][l],
                                                       bf["k"][s_][l], bf["v"][s_][l], bf["o"][s_][l], stream=sh))
            calls.append(functools.partial(c.masw_rollback, self.h, self.seqs, self.prefixes, stream=sh))
            bf["calls"] = calls

        def compute(bf):
            for call in bf["calls"]:
                call()

        def run(n_it):
            in_ready = [None, None]      # H2D of the buffer's current iteration done
            done = [None, None]          # compute of the buffer's current iteration done
            out_done = [None, None]      # D2H of the buffer's last outputs done
            with torch.cuda.stream(cs):
                bufs[0]["in"].copy_(host_in, non_blocking=True)
                in_ready[0] = ev()
                in_ready[0].record(cs)
            for i in range(n_it):
                cur, nxt = i % 2, (i + 1) % 2
                st.wait_event(in_ready[cur])
                if out_done[cur] is not None:
                    st.wait_event(out_done[cur])        # this buffer's previous outputs are on the host
                compute(bufs[cur])
                done[cur] = ev()
                done[cur].record(st)
                with torch.cuda.stream(cs):
                    if i + 1 < n_it:
                        if i >= 1:
                            cs.wait_event(done[nxt])    # iteration i-1 no longer reads that buffer
                        bufs[nxt]["in"].copy_(host_in, non_blocking=True)
                        in_ready[nxt] = ev()
                        in_ready[nxt].record(cs)
                    cs.wait_event(done[cur])
                    host_out[cur].copy_(bufs[cur]["out"], non_blocking=True)
                    out_done[cur] = ev()
                    out_done[cur].record(cs)

        run(2)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        run(iters)
        e1.record(cs)      # after the last D2H, which follows the last iteration's compute
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3, h2d, d2h

    def close(self):
        self.capi.masw_mem_destroy(self.h)


def run_verify(torch, capi, synth, reps: int = 5):
    """Target verify attention for the 8B-target shape: batch 4, Lq = 6 (L_draft
    + 1), 32 query / 8 kv heads, head_dim 128, 32768 + 6 keys, 32 layers with
    distinct caches (17.2 GB, larger than L2), timed as a graph of 32 launches."""
    w = synth.WORKLOADS["verify8b_32k"]
    B, Lq, Hq, Hkv, D, L = w["batch"], w["Lq"], w["Hq"], w["Hkv"], w["D"], w["layers"]
    T = w["prefix"] + Lq
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    caches = []
    for _ in range(L):
        kc = torch.randn(B, Hkv, T, D, generator=g, device=dev).to(torch.bfloat16)
        vc = torch.randn(B, Hkv, T, D, generator=g, device=dev).to(torch.bfloat16)
        caches.append((kc, vc))
    q = [torch.randn(B, Lq, Hq, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    kl = torch.full((B,), T, dtype=torch.int32, device=dev)
    o = torch.empty(B, Lq, Hq, D, device=dev)
    ws = torch.zeros(capi.masw_verify_workspace_bytes(B, Lq, Hq, Hkv, D, T), dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)

    def run():
        for l in range(L):
            capi.masw_verify_attn(q[l], caches[l][0], caches[l][1], kl, o, workspace=ws)
    with torch.cuda.stream(st):
        run()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=st):
        run()
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(reps):
            gr.replay()
        e1.record(st)
    torch.cuda.synchronize()
    secs = e0.elapsed_time(e1) / 1e3 / reps
    kv_bytes = L * B * Hkv * T * D * 2 * 2
    flops = L * B * Hkv * 4 * (Hq // Hkv) * sum(T - Lq + 1 + j for j in range(Lq)) * D
    del caches
    torch.cuda.empty_cache()
    return {"ms_per_verify": secs * 1e3, "layers": L, "batch": B, "lq": Lq, "keys": T,
            "kv_bytes": kv_bytes, "gbs": kv_bytes / secs / 1e9, "tflops": flops / secs / 1e12,
            "launches": L}


def run_accept(torch, capi, reps: int = 20):
    """Greedy acceptance of verified blocks: batch 8, L_draft = 5 (6 logit rows
    per sequence), a 128,256-token vocabulary (Llama-3), bf16 logits.  24
    distinct logit buffers (295 MB, larger than L2) are cycled inside a graph so
    every call reads its logits from HBM."""
    B, L, V, nbuf = 8, 5, 128256, 24
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    logits = [torch.randn(B, L + 1, V, generator=g, device=dev).to(torch.bfloat16) for _ in range(nbuf)]
    draft = torch.randint(0, V, (B, L), generator=g, device=dev, dtype=torch.int32)
    tokens = torch.empty(B, L + 1, dtype=torch.int32, device=dev)
    n_emit = torch.empty(B, dtype=torch.int32, device=dev)
    ws = torch.zeros(capi.masw_greedy_workspace_bytes(B, L, V), dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)

    def run():
        for x in logits:
            capi.masw_greedy_accept(x, draft, tokens, n_emit, workspace=ws, stream=st.cuda_stream)
    with torch.cuda.stream(st):
        run()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=st):
        run()
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(reps):
            gr.replay()
        e1.record(st)
    torch.cuda.synchronize()
    per_call = e0.elapsed_time(e1) / 1e3 / (reps * nbuf)
    nbytes = B * (L + 1) * V * 2
    del logits
    torch.cuda.empty_cache()
    return {"batch": B, "l_draft": L, "vocab": V, "dtype": "bf16", "us_per_call": per_call * 1e6,
            "bytes_per_call": nbytes, "gbs": nbytes / per_call / 1e9, "launches": 1}


def prefill_flops(T, S, W, r, Hq, D, self_attend=False):
    """Algorithmic flops of one (layer, sequence) prefill: 4 D flops (QK^T and PV)
    per query head per visible (query, key) pair of the structured mask."""
    def slots(t):
        return max(0, (t - S - W) // r)
    pairs = 0
    for i in range(1, T + 1):
        pairs += min(S, i) + (i - max(S + 1, i - W + 1) + 1 if i > S else 0) + slots(i - 1)
    M = slots(T)
    for m in range(1, M + 1):
        pairs += S + W + (m if self_attend else m - 1)
    return 4 * D * Hq * pairs, pairs


def run_prefill(torch, capi, synth, workload: str, T: int, reps: int = 3):
    """Draft prefill of a T-token prefix through every layer of the draft model
    for one sequence (one masw_prefill per layer: attention of all raw and slot
    rows under the structured mask, then M_0 stored), timed with CUDA events."""
    w = synth.WORKLOADS[workload]
    L, Hq, Hkv, D, S, W, r = w["layers"], w["Hq"], w["Hkv"], w["D"], w["S"], w["W"], w["r"]
    M = max(0, (T - S - W) // r)
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    mk = lambda *shape: torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
    qr, kr, vr = mk(T, Hq, D), mk(T, Hkv, D), mk(T, Hkv, D)
    qs, ks, vs = mk(max(M, 1), Hq, D), mk(max(M, 1), Hkv, D), mk(max(M, 1), Hkv, D)
    o_r = torch.empty(T, Hq, D, device=dev)
    l_r = torch.empty(T, Hq, device=dev)
    o_s = torch.empty(max(M, 1), Hq, D, device=dev)
    l_s = torch.empty(max(M, 1), Hq, device=dev)
    h = capi.masw_mem_create(S, W, r, Hkv, D, L, batch=1, dtype=capi.MASW_BF16, max_seq_len=T + 64,
                             rollback_reserve=16)
    st = torch.cuda.Stream(device=dev)

    def run():
        for l in range(L):
            capi.masw_prefill(h, l, 0, qr, kr, vr, qs, ks, vs, o_r, l_r, o_s, l_s, stream=st)
    with torch.cuda.stream(st):
        run()
        run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(reps):
            run()
        e1.record(st)
    torch.cuda.synchronize()
    secs = e0.elapsed_time(e1) / 1e3 / reps
    capi.masw_mem_destroy(h)
    flops, pairs = prefill_flops(T, S, W, r, Hq, D)
    per_launch = secs / L
    return {"workload": workload, "prefix": T, "layers": L, "slots": M, "ms_per_prefill": secs * 1e3,
            "ms_per_layer": per_launch * 1e3, "tokens_per_s": T / secs,
            "tflops": flops / per_launch / 1e12, "flops_per_layer": flops, "visible_pairs_per_head": pairs,
            "launches": 2 * L}


# ------------------------------------------------------ ranks (replicas) --

def max_over_ranks(timings, world: int, device: str = "cpu"):
    """Each timing's maximum over the ranks of the job (the slowest replica sets
    the job's time); a single process returns its own timings."""
    if world <= 1:
        return list(timings)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in timings], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world: int, units_per_rank: float, secs: float) -> float:
    """Units processed by all ranks (weak scaling: every replica does the same
    work) per second of the slowest rank."""
    return world * units_per_rank / secs


# ------------------------------------------------------------ CPU oracle --

class OracleIteration:
    """The CPU oracle, as it stands, on one (layer, sequence) pair of the
    default workload's 32K state, running the GPU arm's speculative iteration:
    L_draft x (append + draft attention), the slot write at the step that
    reaches the compression boundary, and the rollback of the speculative
    tokens after the last step.  unit() is one (layer, sequence) decode step;
    a decode step of the workload is layers x batch units (slot writes and
    rollbacks come in the GPU arm's proportion: one per L_draft units)."""

    def __init__(self):
        import oracle.masw_oracle as orc
        from compressed_draft_kv_gb300 import synth
        self.orc, self.synth = orc, synth
        w = synth.WORKLOADS[WORKLOAD]
        self.w = w
        S, W, r, Hkv, D, prefix = w["S"], w["W"], w["r"], w["Hkv"], w["D"], w["prefix"]
        n = orc.slot_count(prefix, S, W, r)
        kr = synth.normal((prefix, Hkv, D), "bf16", "cpu-sample", "k").float().numpy()
        vr = synth.normal((prefix, Hkv, D), "bf16", "cpu-sample", "v").float().numpy()
        ks = synth.normal((n, Hkv, D), "bf16", "cpu-sample", "ks").float().numpy()
        vs = synth.normal((n, Hkv, D), "bf16", "cpu-sample", "vs").float().numpy()
        self.mem = orc.MaswOracle(S, W, r, Hkv, D, 1, 1, reserve=16)
        self.mem.load(0, 0, kr, vr, ks, vs)
        self.prefix = prefix
        self.i = 0
        self.units = 0
        self.slot_writes = 0
        self.rollbacks = 0

    def unit(self):
        orc, synth, w = self.orc, self.synth, self.w
        Hkv, Hq, D = w["Hkv"], w["Hq"], w["D"]
        s_ = self.i % w["steps"]
        k = synth.normal((1, Hkv, D), "bf16", "cpu-sample", "k1", s_).float().numpy()
        v = synth.normal((1, Hkv, D), "bf16", "cpu-sample", "v1", s_).float().numpy()
        q = synth.normal((1, Hq, D), "bf16", "cpu-sample", "q1", s_).float().numpy()
        self.mem.append(0, k, v)
        self.mem.draft_attn(0, q)
        t = self.mem.t(0, 0)
        if orc.is_boundary(t, w["S"], w["W"], w["r"]) and self.mem.m(0, 0) == orc.slot_count(t, w["S"], w["W"], w["r"]) - 1:
            g = synth.normal((1, Hq, D), "bf16", "cpu-sample", "qg").float().numpy()
            kg = synth.normal((1, Hkv, D), "bf16", "cpu-sample", "kg").float().numpy()
            self.mem.materialize_slot(0, [0], g, kg, kg)
            self.slot_writes += 1
        if s_ == w["steps"] - 1:
            self.mem.rollback([0], [self.prefix])
            self.rollbacks += 1
        self.i += 1
        self.units += 1


def _cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def oracle_sample(seconds_budget: float = 12.0):
    """cpu_baseline of the GPU arm: the oracle's speculative iteration
    (OracleIteration) for about `seconds_budget` seconds, as decode steps/s."""
    it = OracleIteration()
    w = it.w
    t0 = time.perf_counter()
    while True:
        it.unit()
        el = time.perf_counter() - t0
        if el > seconds_budget or it.units >= 400:
            break
    steps_per_s = it.units / el / (w["layers"] * w["batch"])
    return {"value": steps_per_s, "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"{it.units} (layer, sequence) decode steps of one pair at a {it.prefix}-token prefix "
                      f"(append + draft attention, {it.slot_writes} slot writes, {it.rollbacks} rollbacks: "
                      f"the GPU arm's iteration) in {el:.1f} s; a decode step is {w['layers']} x {w['batch']} "
                      f"such units; numpy fp64, default BLAS threading"}


def reference_arm(steps: int, warmup: int):
    """The reference arm: the CPU oracle timed as it stands.  One reference
    step = one sequence's decode step through all layers (`layers` units of
    OracleIteration), i.e. 1/batch of a decode step of the workload; `warmup`
    untimed steps, then `steps` timed ones."""
    it = OracleIteration()
    w = it.w
    for _ in range(warmup * w["layers"]):
        it.unit()
    u0 = it.units
    t0 = time.perf_counter()
    for _ in range(steps * w["layers"]):
        it.unit()
    el = time.perf_counter() - t0
    ms_per_step = el * 1e3 / steps
    value = steps / el / w["batch"]            # decode steps (all layers x batch) per second
    sample = (f"{steps} timed reference steps after {warmup} untimed; a reference step is one sequence's "
              f"decode step through all {w['layers']} layers ({w['layers']} x append + draft attention on one "
              f"(layer, sequence) pair at a {it.prefix}-token prefix, with the GPU arm's slot writes and "
              f"rollbacks: {it.slot_writes} and {it.rollbacks} in all), 1/{w['batch']} of a decode step; "
              f"{it.units - u0} units in {el:.1f} s; numpy fp64, default BLAS threading")
    return {"value": value, "ms_per_step": ms_per_step, "secs": el, "sample": sample, "cores": _cores()}


# ------------------------------------------------------- profiling case --

def profile_case(kind: str, prefix: int):
    """A few launches of one kernel on the benchmark's per-launch shape (batch 8,
    24q/8kv heads, 32K prefix) over 4 layers, for an ncu capture: each launch
    reads a different layer's data, and ncu flushes caches between passes."""
    import torch
    from compressed_draft_kv_gb300 import capi, synth
    capi.load()
    w = synth.WORKLOADS[WORKLOAD]
    L, B, Hq, Hkv, D, S, W, r = 4, w["batch"], w["Hq"], w["Hkv"], w["D"], w["S"], w["W"], w["r"]
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    if kind == "prefill":
        T = prefix
        M = max(0, (T - S - W) // r)
        mk = lambda *shape: torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
        h = capi.masw_mem_create(S, W, r, Hkv, D, 1, batch=1, dtype=capi.MASW_BF16, max_seq_len=T + 64)
        qr, kr, vr, qs, ks, vs = mk(T, Hq, D), mk(T, Hkv, D), mk(T, Hkv, D), mk(M, Hq, D), mk(M, Hkv, D), mk(M, Hkv, D)
        o_r, o_s = torch.empty(T, Hq, D, device=dev), torch.empty(max(M, 1), Hq, D, device=dev)
        for _ in range(3):
            capi.masw_prefill(h, 0, 0, qr, kr, vr, qs, ks, vs, o_r, None, o_s, None)
        torch.cuda.synchronize()
        capi.masw_mem_destroy(h)
        return
    if kind == "accept":
        # greedy acceptance on the bench's shape (batch 8, L_draft = 5, a
        # 128,256-token vocabulary, bf16): one call on each of 4 logit buffers
        ab, al, av = 8, 5, 128256
        logits = [torch.randn(ab, al + 1, av, generator=g, device=dev).to(torch.bfloat16) for _ in range(4)]
        draft = torch.randint(0, av, (ab, al), generator=g, device=dev, dtype=torch.int32)
        tokens = torch.empty(ab, al + 1, dtype=torch.int32, device=dev)
        n_emit = torch.empty(ab, dtype=torch.int32, device=dev)
        ws = torch.zeros(capi.masw_greedy_workspace_bytes(ab, al, av), dtype=torch.uint8, device=dev)
        for x in logits:
            capi.masw_greedy_accept(x, draft, tokens, n_emit, workspace=ws)
        torch.cuda.synchronize()
        return
    if kind == "verify":
        vb, Lq, Hq8 = 4, 6, 32
        T = prefix + Lq
        kc = torch.randn(vb, Hkv, T, D, generator=g, device=dev).to(torch.bfloat16)
        vc = torch.randn(vb, Hkv, T, D, generator=g, device=dev).to(torch.bfloat16)
        q = torch.randn(vb, Lq, Hq8, D, generator=g, device=dev).to(torch.bfloat16)
        kl = torch.full((vb,), T, dtype=torch.int32, device=dev)
        o = torch.empty(vb, Lq, Hq8, D, device=dev)
        for _ in range(4):
            capi.masw_verify_attn(q, kc, vc, kl, o)
        torch.cuda.synchronize()
        return
    if kind == "step_b1":
        # the pages' decoding setting: one sequence through all 28 layers of the
        # 3B-draft memory (4.5 MB per layer, 126 MB per decode step, about the
        # size of L2), three iterations of 28 fused steps and the rollback, so a
        # capture of the second iteration's launches sees what the first left in L2
        L1 = w["layers"]
        h = capi.masw_mem_create(S, W, r, Hkv, D, L1, batch=1, dtype=capi.MASW_BF16, max_seq_len=prefix + 32,
                                 rollback_reserve=16)
        n = max(0, (prefix - S - W) // r)
        kr = torch.randn(prefix, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
        vr = torch.randn(prefix, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
        ks = torch.randn(n, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
        for l in range(L1):
            capi.masw_mem_load(h, l, 0, kr, vr, ks, ks)
        q = [torch.randn(1, Hq, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(L1)]
        kn = [torch.randn(1, Hkv, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(L1)]
        o = torch.empty(1, Hq, D, device=dev)
        for _ in range(3):
            for l in range(L1):
                capi.masw_draft_step(h, l, q[l], kn[l], kn[l], o)
            capi.masw_rollback(h, [0], [prefix])
        torch.cuda.synchronize()
        capi.masw_mem_destroy(h)
        return
    full = kind == "full"
    h = capi.masw_mem_create(S, W, r, Hkv, D, L, batch=B, dtype=capi.MASW_BF16, max_seq_len=prefix + 8,
                             full_kv=full)
    n = max(0, (prefix - S - W) // r)
    kr = torch.randn(prefix, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
    ks = torch.randn(n, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
    for l in range(L):
        for b in range(B):
            capi.masw_mem_load(h, l, b, kr, kr, ks, ks)
    q = torch.randn(B, Hq, D, generator=g, device=dev).to(torch.bfloat16)
    o = torch.empty(B, Hq, D, device=dev)
    kn = torch.randn(B, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
    for l in range(L):
        if kind == "step":
            capi.masw_draft_step(h, l, q, kn, kn, o)
        else:
            (capi.masw_full_attn if full else capi.masw_draft_attn)(h, l, q, o)
    torch.cuda.synchronize()
    capi.masw_mem_destroy(h)


# ------------------------------------------------------------------ main --

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="masw", choices=["masw", "reference"])
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["draft3b_28l_b8", "draft3b_28l_b1", "draft8b_b32_ragged", "draft3b_1layer_8k", "paper_s128_w128_r4",
                             "paper_s128_w128_r8", "swa_w1024"])
    ap.add_argument("--prefix", type=int, default=None, help="override the prefix (all sequences)")
    ap.add_argument("--batch", type=int, default=None, help="override the number of sequences")
    ap.add_argument("--sweep", action="store_true",
                    help="MASW vs full-KV decode steps/s at prefixes 4K..32K (one JSON line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-verify", action="store_true")
    ap.add_argument("--e2e-iters", type=int, default=20)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--prefill-only", action="store_true",
                    help="only the draft prefill of one sequence through all layers (one JSON line)")
    ap.add_argument("--profile-case", choices=["draft", "step", "step_b1", "full", "verify", "prefill", "accept"],
                    default=None,
                    help="run a few launches of one kernel on a small state (4 layers) for an ncu capture")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from compressed_draft_kv_gb300 import synth
    wl = dict(synth.WORKLOADS[args.workload])
    if args.batch is not None:
        if args.batch < 1:
            raise SystemExit("--batch must be at least 1")
        wl["batch"] = args.batch
    prefix = args.prefix or wl.get("prefix", 32768)

    if args.profile_case:
        profile_case(args.profile_case, prefix)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        ref = reference_arm(args.steps, args.warmup)
        cb = {"value": ref["value"], "unit": UNIT, "cores": ref["cores"], "kind": "oracle", "sample": ref["sample"]}
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": ref["value"], "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ref["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "prefix": prefix,
                       "reference_step": "one sequence's decode step through all layers (1/batch of a decode step)"},
            "cpu_baseline": cb,
            "e2e": {"value": ref["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    import torch
    from compressed_draft_kv_gb300 import capi
    capi.load()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = dist.barrier

    if args.prefill_only:
        with ClockSampler(local) as clk:
            pf = run_prefill(torch, capi, synth, args.workload, prefix, reps=max(1, args.steps // 20))
        peak = _peaks_tensor()
        pf["roofline"] = {"bound": "tensor", "achieved": pf["tflops"], "peak": peak[0], "unit": "TFLOP/s",
                          "frac": pf["tflops"] / peak[0], "peak_kind": peak[1]}
        pf["clocks"] = clk.summary()
        if rank == 0:
            print(json.dumps({"metric": "draft prefill tokens/s (one sequence, all layers)", "value": pf["tokens_per_s"],
                              "unit": "tokens/s", "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                              "prefill": pf}))
        return

    if args.sweep:
        rows = []
        for pf in (4096, 8192, 16384, 24576, 32768):
            bench = DraftBench(torch, capi, synth, args.workload, pf)
            g_d, _ = bench.capture(bench.iteration)
            g_f, _ = bench.capture(lambda: bench.iteration(full=True))
            sd = bench.time_graph(g_d, args.warmup, max(10, args.steps // 4))
            sf = bench.time_graph(g_f, 3, 5)
            kd = bench.kv_bytes_per_decode_step()
            kf = bench.kv_bytes_per_decode_step(full=True)
            ns = bench.steps
            rows.append({"prefix": pf, "masw_steps_per_s": max(10, args.steps // 4) * ns / sd,
                         "full_steps_per_s": 5 * ns / sf,
                         "masw_ms_per_step": sd / (max(10, args.steps // 4) * ns) * 1e3,
                         "full_ms_per_step": sf / (5 * ns) * 1e3,
                         "masw_kv_gb_per_step": kd / 1e9, "full_kv_gb_per_step": kf / 1e9})
            bench.close()
            del bench, g_d, g_f
            torch.cuda.empty_cache()
        if rank == 0:
            print(json.dumps({"metric": METRIC + " vs prefix", "unit": UNIT, "workload": args.workload,
                              "sweep": rows}))
        return

    bench = DraftBench(torch, capi, synth, args.workload, args.prefix, args.batch)
    g_draft, launches = bench.capture(bench.iteration)
    g_full, launches_full = bench.capture(lambda: bench.iteration(full=True))
    full_iters = max(3, args.steps // 5)
    with ClockSampler(local) as clk:
        secs = bench.time_graph(g_draft, args.warmup, args.steps, barrier)
        median_step_s = bench.last_median_s
        secs_full = bench.time_graph(g_full, 3, full_iters, barrier)
    kern_s, _ = bench.time_draft_kernel(reps=50)
    e2e_s, h2d, d2h = bench.e2e(args.e2e_iters)
    capi.masw_sync(bench.h)
    total_b, kv_b, qo_b = bench.algorithmic_bytes_per_draft_launch()
    kv_step = bench.kv_bytes_per_decode_step()
    kv_step_full = bench.kv_bytes_per_decode_step(full=True)
    prefixes = list(bench.prefixes)
    due_steps = [s_ + 1 for s_ in range(bench.steps) if bench.due[s_]]
    bench.close()
    del g_draft, g_full, bench
    torch.cuda.empty_cache()
    verify = None
    if not args.no_verify and args.workload == WORKLOAD:
        verify = run_verify(torch, capi, synth)
    accept = None
    if not args.no_verify and args.workload == WORKLOAD:
        accept = run_accept(torch, capi)
        accept["hbm_frac"] = accept["gbs"] / _peaks()[0]
    prefill = None
    if not args.no_prefill and args.workload == WORKLOAD:
        prefill = run_prefill(torch, capi, synth, args.workload, prefix)
        tp = _peaks_tensor()
        prefill["tensor_frac"] = prefill["tflops"] / tp[0]
        prefill["tensor_peak_kind"] = tp[1]

    secs, secs_full, e2e_per = max_over_ranks([secs, secs_full, e2e_s / args.e2e_iters], world, "cuda")
    dsteps = wl["steps"]
    value = whole_job_rate(world, args.steps * dsteps, secs)
    full_value = whole_job_rate(world, full_iters * dsteps, secs_full)
    peak, peak_kind = _peaks()
    achieved = total_b / kern_s / 1e9
    traffic = _recorded_traffic() if args.workload == WORKLOAD and args.batch is None and args.prefix is None else None
    line = {
        "metric": (METRIC if args.workload == WORKLOAD and args.batch is None and args.prefix is None
                   else f"MASW draft-attn decode steps/s ({args.workload}, batch {wl['batch']}, prefix {prefix})"),
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "ms_per_step_median": median_step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "layers": wl["layers"], "batch": wl["batch"], "q_heads": wl["Hq"],
                   "kv_heads": wl["Hkv"], "head_dim": wl["D"],
                   "prefix": prefixes[0] if len(set(prefixes)) == 1 else f"ragged {min(prefixes)}..{max(prefixes)}",
                   "S": wl["S"], "W": wl["W"], "r": wl["r"], "rollback_reserve": 16,
                   "decode_steps_per_bench_step": dsteps, "boundary_steps": due_steps,
                   "kv_gb_per_decode_step": kv_step / 1e9,
                   "l2": "working set per decode step > 129 MB L2; no flush",
                   "launch": "CUDA graph of one speculative iteration", "parallelism": f"replicas x{world}"},
        "full_kv": {"value": full_value, "unit": UNIT, "ms_per_step": secs_full / full_iters * 1e3,
                    "kv_gb_per_decode_step": kv_step_full / 1e9,
                    "gbs": kv_step_full * full_iters * dsteps / secs_full / 1e9},
        "speedup_vs_full_kv": value / full_value,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "traffic_source": ("recorded, not measured in this run: ncu dram__bytes_read.sum + "
                                        "dram__bytes_write.sum per launch from profiles/decode_mma_step_b8_32k.md, "
                                        "whose kernel code hash matches the built sources" if traffic is not None
                                        else "none: no ncu capture of the current kernel code for this workload"),
                     "peak_kind": peak_kind,
                     "kernel": "decode_mma_kernel<128, NST> (masw_draft_step: fused append + draft attention; NST = 2 stages, 3 when each CTA streams a long run of keys)",
                     "bytes_per_launch": total_b, "kv_bytes_per_launch": kv_b,
                     "us_per_launch": kern_s * 1e6, "frac_of_8tbs": achieved / 8000.0},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
        "e2e": {"value": world * dsteps / e2e_per, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "per iteration: one copy of all q/k/v inputs from pinned host memory, eager C-ABI calls "
                       "(no graph), one copy of every O back to pinned host memory; buffers doubled so that "
                       "iteration i+1's inputs come in and iteration i's outputs go out on a copy stream "
                       "while iteration i+1 computes"},
    }
    if verify:
        # draft / target attention time per sequence: L_draft draft steps of the
        # 3B-draft memory (batch 8) against one 8B-target verify (batch 4)
        draft_per_seq = (secs / args.steps) / wl["batch"]
        verify_per_seq = verify["ms_per_verify"] / 1e3 / verify["batch"]
        verify["draft_over_verify_per_sequence"] = draft_per_seq / verify_per_seq
        verify["hbm_frac"] = verify["gbs"] / peak
        line["verify"] = verify
        # Eq. 1 of the pages with this run's attention-only latencies: t_d = one
        # draft decode step per sequence, t_t = one verify per sequence, and the
        # pages' tokens per iteration (3B draft, 32K; [EN] §5 draft-cost table)
        t_d = (secs / args.steps) / dsteps / wl["batch"]
        t_t = verify["ms_per_verify"] / 1e3 / verify["batch"]
        t_d_full = (secs_full / full_iters) / dsteps / wl["batch"]
        line["eq1_illustration"] = {
            "note": "attention-only latencies measured here (draft memory S=4, W=1024, r=512) with the pages' "
                    "Tok./Iter; an illustration of Eq. 1, not a measured model speedup",
            "l_draft": dsteps, "t_draft_over_t_target": t_d / t_t, "t_full_draft_over_t_target": t_d_full / t_t,
            "tok_per_iter_pages": {"full_kv_draft": 4.05, "masw_4x": 3.65, "masw_8x": 3.43},
            "speedup_masw_4x": capi.masw_eq1_speedup(3.65 - 1.0, dsteps, t_d, t_t),
            "speedup_masw_8x": capi.masw_eq1_speedup(3.43 - 1.0, dsteps, t_d, t_t),
            "speedup_full_kv_draft": capi.masw_eq1_speedup(4.05 - 1.0, dsteps, t_d_full, t_t),
        }
    if accept:
        line["greedy_accept"] = accept
    if prefill:
        line["prefill"] = prefill
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == WORKLOAD:
        line["cpu_baseline"] = oracle_sample()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
