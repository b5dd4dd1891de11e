#!/usr/bin/env python
"""Benchmark of the KDA token step on GB300 (one JSON line on stdout).

Headline: serving-scale decode, 256 sequences x 64 heads x d=128, one token
per call (fp32 state, 1 GiB, larger than L2, so calls run back to back),
starting from the state 32 warm-up tokens leave; metric = state GB/s (2 * d
* d * 4 bytes per sequence, head and token, over the device time of one
call).  The same line carries: that workload's 128 calls replayed as one
CUDA graph; its end-to-end figure through the C ABI with host buffers; the
batched decode (64 x 32 heads, 128 MiB of state, L2 flushed between timed
calls by a 256 MiB write and a 256 MiB read); the batched prefill (8 x 64
heads x 8192 tokens) and the single-sequence prefill (1 x 32 heads x 4096
tokens), chunk 64, bf16 q/k/v, as tokens/s; the packed variable-length
prefill; each with its roofline; and the fp64 CPU oracle timed on this
host's cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun), each rank runs an independent replica of the workload
on its own GPU (the (sequence, head) units never interact); value is the
units of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA decode state GB/s (% of HBM peak); prefill tokens/s (% tensor peak)"
HEADLINE_WL = "decode_b256_h64_x128"     # serving-scale decode, 1 GiB of state
DECODE_WL = "decode_b64_h32_x256"       # batched decode, 128 MiB of state (L2 flushed)
PREFILL_WL = "prefill_b8_h64_t8192"     # batched prefill
PREFILL1_WL = "prefill_b1_h32_t4096"    # single-sequence prefill
D = 128
STATE_BYTES = 2 * D * D * 4          # read + write of one 128x128 fp32 state
FLUSH_BYTES = 256 << 20
PREFILL_FLOP_PER_TOKEN_HEAD = 140.6e3  # algorithmic, triangles counted once


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "src": "fallback"}


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "kda_delta_rule_token_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


PROJ_MD = "proj_decode_b64_h32_prefill_b8_h64_traffic.md"


def profile_traffic(md_name, sha, label="per launch (full workload)"):
    """DRAM bytes per launch (or per call, by `label`) recorded by an ncu
    capture in profiles/<md_name>, or None when missing or taken on another
    version of the kernel source."""
    p = os.path.join(ROOT, "profiles", md_name)
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_sha = re.search(r"kernel source sha256\[:16\]:\s*([0-9a-f]{16})", text)
    m_tr = re.search(r"dram bytes " + re.escape(label) + r":\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != sha:
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi samples (200 ms) of the SM clock and throttle reasons."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        text = self.file.read()
        os.unlink(self.file.name)
        return parse_clocks(text)


def parse_clocks(text):
    """Median SM clock, maximum SM clock and the throttle reasons seen in
    `nvidia-smi --format=csv,noheader,nounits` lines of ClockSampler.Q
    (malformed lines are skipped)."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        r = [x.strip() for x in line.split(",")]
        if len(r) < 9:
            continue
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
        except ValueError:
            continue
        for name, val in zip(names, r[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
            "samples": len(sm)}


def replica_aggregate(local_ms, units_per_rank, dist=None, device="cpu"):
    """Replicas across ranks: returns (slowest rank's ms, units of all ranks per s).

    Each rank runs an independent replica of the workload (the (sequence,
    head) units never interact), so the job's throughput is the units all
    ranks processed over the slowest rank's time.
    """
    world = 1
    ms = float(local_ms)
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * units_per_rank / (ms * 1e-3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- our arm

class Ours:
    def __init__(self, args, world, rank, local):
        import torch
        import kda_delta_rule_token_gb300 as kda
        from kda_delta_rule_token_gb300 import synth
        self.torch, self.kda, self.synth = torch, kda, synth
        self.args, self.world, self.rank = args, world, rank
        torch.cuda.set_device(local)
        self.dev = torch.device("cuda", local)
        self.local = local
        kda.load()
        self.stream = torch.cuda.current_stream()
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl", device_id=self.dev)
            self.dist = dist
        else:
            self.dist = None
        self.flush_w = torch.empty(FLUSH_BYTES // 4, device=self.dev)
        self.flush_r = torch.ones(FLUSH_BYTES // 4, device=self.dev)
        self.sink = torch.empty((), device=self.dev)

    def barrier_sync(self):
        self.torch.cuda.synchronize()
        if self.dist is not None:
            self.dist.barrier()
        self.torch.cuda.synchronize()

    def max_over_ranks(self, x):
        return replica_aggregate(x, 1, self.dist, self.dev)[0]

    def flush_l2(self):
        self.flush_w.fill_(1.0)
        self.torch.sum(self.flush_r, 0, out=self.sink)

    # ---------------------------------------------------------------- decode
    def decode(self, wl_name, flush, graph=False, e2e=True, state_bf16=False):
        """Decode calls of one workload, one launch per call, device-timed.

        flush: write and read 256 MiB between timed calls (for workloads whose
        state fits in L2); otherwise calls run back to back.  Workloads with
        warm-up tokens start from the state the decode kernel reaches after
        them (the GPU tests check that warm-up against the oracle).  graph:
        also time the workload's calls captured once as a CUDA graph and
        replayed (per-call time = replay time / calls).  e2e: the same calls
        through the C ABI with the inputs copied in from pinned host memory
        and o copied out, inside the timed region.  state_bf16: the state is
        kept as bf16 (kda_decode_step_bf16state; a workload whose initial
        state is zero, so that its bf16 form needs no conversion).
        """
        torch, kda, synth = self.torch, self.kda, self.synth
        wl = synth.WORKLOADS[wl_name]
        p = synth.make_params(wl, self.dev)
        st = synth.make_state(wl, self.dev)
        S, cs = st["S"], st["conv_state"]
        if state_bf16:
            assert wl.s0_std == 0 and not graph and not e2e
            S = torch.zeros(S.shape, dtype=torch.int16, device=self.dev)
            del st
        step_fn = kda.kda_decode_step_bf16state if state_bf16 else kda.kda_decode_step
        state_bytes = STATE_BYTES // 2 if state_bf16 else STATE_BYTES
        B, H = wl.B, wl.H
        o = torch.empty((B, H, D), device=self.dev)
        ctx = kda.kda_create(H, p["conv_w"], p["dt_bias"], p["A_log"], p["gamma"])
        K, W = self.args.steps, self.args.warmup

        def run(tk, t, out=o, stream=None):
            step_fn(ctx, B, tk["q"][t], tk["k"][t], tk["v"][t], tk["z"][t],
                    tk["beta_logit"][t], tk["gate_logit"][t], cs, S, out, None,
                    self.stream if stream is None else stream)

        if wl.warmup_tokens:
            warm = synth.make_tokens(wl, self.dev, T=wl.warmup_tokens, warm=True)
            for t in range(wl.warmup_tokens):
                run(warm, t)
            del warm
        tk = synth.make_tokens(wl, self.dev)
        for i in range(W):
            if flush:
                self.flush_l2()
            run(tk, i % wl.T)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        self.barrier_sync()
        l0 = kda.kda_launch_count()
        t_wall = time.perf_counter()
        for i in range(K):
            if flush:
                self.flush_l2()
            ev[i][0].record(self.stream)
            run(tk, (W + i) % wl.T)
            ev[i][1].record(self.stream)
        self.barrier_sync()
        t_wall = time.perf_counter() - t_wall
        launches = kda.kda_launch_count() - l0
        times = [a.elapsed_time(b) for a, b in ev]
        ms = self.max_over_ranks(statistics.fmean(times))
        assert kda.kda_sync_status(ctx, self.stream) == kda.KDA_OK

        ms_graph, graph_launches = None, 0
        if graph:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device=self.dev)
            side.wait_stream(self.stream)
            with torch.cuda.graph(g, stream=side):
                for t in range(wl.T):
                    run(tk, t, stream=torch.cuda.current_stream())
            self.stream.wait_stream(side)
            R = 3
            for _ in range(W):
                g.replay()
            evg = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(R)]
            self.barrier_sync()
            for i in range(R):
                evg[i][0].record(self.stream)
                g.replay()
                evg[i][1].record(self.stream)
            self.barrier_sync()
            ms_graph = self.max_over_ranks(statistics.fmean(a.elapsed_time(b) for a, b in evg)) / wl.T
            graph_launches = R * wl.T
            assert kda.kda_sync_status(ctx, self.stream) == kda.KDA_OK
            del g

        # End to end through the C ABI with pinned host buffers, the way a
        # serving loop runs it: every step copies its inputs in from pinned
        # host memory, decodes and copies o out, and the next step's inputs
        # are staged while this step decodes.  The batch is split into
        # `--e2e-split` groups of sequences; a group's six inputs sit back to
        # back in one pinned host buffer (each at a 16-byte multiple), so a
        # group is one host-to-device copy, one decode call on views of the
        # device copy and one device-to-host copy of its o, on three streams.
        # Device input packs and outputs alternate between two buffers: a
        # step's copy-in waits for the decode two steps back that read the
        # same pack, its decode for the copy-out two steps back of the same
        # output.  Value: the time of Ke steps / Ke (events on the decode
        # stream around the whole loop, the other streams wait for the start).
        ms_e2e, h2d, d2h = None, 0, 0
        if e2e:
            nh = min(8, wl.T)
            names = ("q", "k", "v", "z", "gate_logit", "beta_logit")
            nsplit = max(1, min(self.args.e2e_split, B))
            groups = [(B * j // nsplit, B * (j + 1) // nsplit) for j in range(nsplit)]
            layout = []                                     # (group, name) -> (offset, shape)
            off = 0
            for (b0, b1) in groups:
                ent = {}
                for n in names:
                    shp = tk[n][0][b0:b1].shape
                    n_el = tk[n][0][b0:b1].numel()
                    ent[n] = (off, n_el, shp)
                    off += (n_el + 3) // 4 * 4
                layout.append((off, ent))
            total = off
            host = []
            for t in range(nh):
                hb = torch.empty(total, dtype=torch.float32, pin_memory=True)
                for (b0, b1), (_, ent) in zip(groups, layout):
                    for n, (a, n_el, _s) in ent.items():
                        hb[a:a + n_el].copy_(tk[n][t][b0:b1].reshape(-1))
                host.append(hb)
            dpack = [torch.empty(total, dtype=torch.float32, device=self.dev) for _ in range(2)]
            seg = []                                        # (start, end) of each group in a pack
            start = 0
            for (end, _ent) in layout:
                seg.append((start, end))
                start = end
            dv = [[{n: dp[a:a + n_el].view(shp) for n, (a, n_el, shp) in ent.items()} for (_e, ent) in layout]
                  for dp in dpack]
            od = [torch.empty((B, H, D), device=self.dev) for _ in range(2)]
            o_host = [torch.empty((B, H, D), pin_memory=True) for _ in range(2)]
            h2d = total * 4
            d2h = B * H * D * 4
            s_in = torch.cuda.Stream(device=self.dev)
            s_out = torch.cuda.Stream(device=self.dev)
            ev_dec, ev_out = {}, {}

            def steps(i0, n):
                for i in range(i0, i0 + n):
                    p = i % 2
                    hb = host[i % nh]
                    if flush:
                        self.flush_l2()
                    for j, (b0, b1) in enumerate(groups):
                        a0, a1 = seg[j]
                        if (i - 2, j) in ev_dec:
                            s_in.wait_event(ev_dec.pop((i - 2, j)))
                        with torch.cuda.stream(s_in):
                            dpack[p][a0:a1].copy_(hb[a0:a1], non_blocking=True)
                        e_in = torch.cuda.Event()
                        e_in.record(s_in)
                        self.stream.wait_event(e_in)
                        if (i - 2, j) in ev_out:
                            self.stream.wait_event(ev_out.pop((i - 2, j)))
                        g_ = dv[p][j]
                        kda.kda_decode_step(ctx, b1 - b0, g_["q"], g_["k"], g_["v"], g_["z"],
                                            g_["beta_logit"], g_["gate_logit"], cs[b0:b1], S[b0:b1],
                                            od[p][b0:b1], None, self.stream)
                        e_d = torch.cuda.Event()
                        e_d.record(self.stream)
                        ev_dec[(i, j)] = e_d
                        s_out.wait_event(e_d)
                        with torch.cuda.stream(s_out):
                            o_host[p][b0:b1].copy_(od[p][b0:b1], non_blocking=True)
                        e_o = torch.cuda.Event()
                        e_o.record(s_out)
                        ev_out[(i, j)] = e_o

            Ke = max(3, min(K, 200))
            steps(0, W)
            self.barrier_sync()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            s_in.wait_event(e0)
            s_out.wait_event(e0)
            steps(W, Ke)
            self.stream.wait_stream(s_out)
            e1.record(self.stream)
            self.barrier_sync()
            ms_e2e = self.max_over_ranks(e0.elapsed_time(e1) / Ke)
            assert kda.kda_sync_status(ctx, self.stream) == kda.KDA_OK
            del host, dpack, dv, od, o_host
        kda.kda_destroy(ctx)

        units = B * H                                   # (sequence, head) pairs per call
        alg_bytes = units * (state_bytes + 5 * D * 4 + 4 + D * 4 + 2 * 9 * D * 4) + H * 7680
        res = {
            "wl": wl, "ms": ms, "times": times, "launches": launches, "wall": t_wall,
            "state_elem_bytes": 2 if state_bf16 else 4,
            "state_gbs": self.world * units * state_bytes / (ms * 1e-3) / 1e9,
            "alg_gbs": alg_bytes / (ms * 1e-3) / 1e9, "alg_bytes": alg_bytes,
            "ms_graph": ms_graph, "graph_launches": graph_launches,
        }
        if ms_graph is not None:
            res["state_gbs_graph"] = self.world * units * STATE_BYTES / (ms_graph * 1e-3) / 1e9
            res["alg_gbs_graph"] = alg_bytes / (ms_graph * 1e-3) / 1e9
        if ms_e2e is not None:
            res.update({"e2e_gbs": self.world * units * STATE_BYTES / (ms_e2e * 1e-3) / 1e9,
                        "ms_e2e": ms_e2e, "h2d": h2d, "d2h": d2h})
        del tk, S, cs
        torch.cuda.empty_cache()
        return res

    # ---------------------------------------------------------- low-rank decode
    def decode_lowrank(self, wl_name):
        """kda_decode_step_lowrank (front-end GEMMs + decode kernel) per call,
        and the front-end alone (kda_lowrank), on a decode workload with the
        default low-rank widths; L2 flushed between timed calls."""
        torch, kda, synth = self.torch, self.kda, self.synth
        wl = synth.WORKLOADS[wl_name]
        p = synth.make_params(wl, self.dev)
        st = synth.make_state(wl, self.dev)
        S, cs = st["S"], st["conv_state"]
        tk = synth.make_tokens(wl, self.dev)
        lr = synth.make_lowrank(wl, self.dev)
        B, H = wl.B, wl.H
        o = torch.empty((B, H, D), device=self.dev)
        ctx = kda.kda_create(H, p["conv_w"], p["dt_bias"], p["A_log"], p["gamma"])
        kda.kda_bind_lowrank(ctx, lr["hidden"], lr["rank"], lr["W_fa"], lr["W_fb"], lr["W_bp"])
        ws = torch.empty(kda.kda_decode_lowrank_workspace_bytes(ctx, B), dtype=torch.uint8, device=self.dev)
        wsf = torch.empty(kda.kda_lowrank_workspace_bytes(ctx, B), dtype=torch.uint8, device=self.dev)
        z = torch.empty((B, H, D), device=self.dev)
        bl = torch.empty((B, H), device=self.dev)
        K, W = min(self.args.steps, 500), self.args.warmup

        def step(i):
            t = i % wl.T
            kda.kda_decode_step_lowrank(ctx, B, lr["x"][t], tk["q"][t], tk["k"][t], tk["v"][t],
                                        tk["gate_logit"][t], cs, S, o, None, ws, 0, self.stream)

        def front(i):
            kda.kda_lowrank(ctx, B, lr["x"][i % wl.T], z, bl, wsf, 0, self.stream)

        out = {}
        for name, fn in (("step", step), ("frontend", front)):
            for i in range(W):
                self.flush_l2()
                fn(i)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            self.barrier_sync()
            l0 = kda.kda_launch_count()
            for i in range(K):
                self.flush_l2()
                ev[i][0].record(self.stream)
                fn(W + i)
                ev[i][1].record(self.stream)
            self.barrier_sync()
            out[name] = (self.max_over_ranks(statistics.fmean(a.elapsed_time(b) for a, b in ev)),
                         kda.kda_launch_count() - l0)
        assert kda.kda_sync_status(ctx, self.stream) == kda.KDA_OK
        kda.kda_destroy(ctx)
        hid, rank = lr["hidden"], lr["rank"]
        fe_bytes = 4 * ((rank + H) * hid + H * D * rank + B * hid + B * H * D + B * H)
        fe_flop = 2 * B * ((rank + H) * hid + H * D * rank)
        units = B * H
        res = {"wl": wl, "hidden": hid, "rank": rank, "ms_step": out["step"][0], "launches_step": out["step"][1],
               "ms_frontend": out["frontend"][0], "launches_frontend": out["frontend"][1],
               "fe_bytes": fe_bytes, "fe_flop": fe_flop,
               "state_gbs": self.world * units * STATE_BYTES / (out["step"][0] * 1e-3) / 1e9}
        del tk, S, cs, lr
        torch.cuda.empty_cache()
        return res

    # ---------------------------------------------------------------- projections
    def projections(self, wl_name, with_cublas=True):
        """kda_project_qkvg (bf16 q/k/v and fp32 gate logits for prefill
        workloads, fp32 for decode ones) and kda_project_o on the tokens of
        one call of a workload (hidden 7168); cuBLAS bf16 GEMMs of the same
        shapes are timed beside them for context.  Inputs larger than L2 (or
        the weights, at decode size)."""
        torch, kda, synth = self.torch, self.kda, self.synth
        wl = synth.WORKLOADS[wl_name]
        pr = synth.make_projections(wl, self.dev)
        N, H, hid = pr["x"].shape[0], wl.H, pr["hidden"]
        HD = H * D
        p = synth.make_params(wl, self.dev)
        ctx = kda.kda_create(H, p["conv_w"], p["dt_bias"], p["A_log"], p["gamma"])
        kda.kda_bind_projections(ctx, hid, pr["W_qkvg"].view(torch.int16), pr["W_o"].view(torch.int16))
        f32 = wl.mode == "decode"
        dt = torch.float32 if f32 else torch.bfloat16
        q, k, v = (torch.empty((N, HD), device=self.dev, dtype=dt) for _ in range(3))
        g = torch.empty((N, HD), device=self.dev)
        y = torch.empty((N, hid), device=self.dev)
        ws = torch.empty(kda.kda_project_o_workspace_bytes(ctx, N), dtype=torch.uint8, device=self.dev)
        xi = pr["x"].view(torch.int16)
        K = 5 if N > 4096 else 50
        W = max(3, self.args.warmup)

        def timed(fn, n):
            for _ in range(W):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            self.barrier_sync()
            l0 = kda.kda_launch_count()
            for i in range(n):
                ev[i][0].record(self.stream)
                fn()
                ev[i][1].record(self.stream)
            self.barrier_sync()
            return (self.max_over_ranks(statistics.fmean(a.elapsed_time(b) for a, b in ev)),
                    kda.kda_launch_count() - l0)

        ms_in, l_in = timed(lambda: kda.kda_project_qkvg(ctx, N, xi, q, k, v, g, qkv_f32=f32, stream=self.stream), K)
        ms_out, l_out = timed(lambda: kda.kda_project_o(ctx, N, pr["o_in"], y, ws, 0, self.stream), K)
        assert kda.kda_sync_status(ctx, self.stream) == kda.KDA_OK
        kda.kda_destroy(ctx)
        res = {"wl": wl, "N": N, "hidden": hid, "H": H, "ms_in": ms_in, "launches_in": l_in,
               "ms_out": ms_out, "launches_out": l_out,
               "flop_in": 2.0 * N * 4 * HD * hid, "flop_out": 2.0 * N * HD * hid,
               "bytes_in": 2 * (N * hid + 4 * HD * hid) + N * HD * (3 * (4 if f32 else 2) + 4),
               "bytes_out": 2 * hid * HD + N * HD * (4 + 2 + 2) + 4 * N * hid}
        if with_cublas:
            Wt = pr["W_qkvg"]
            with torch.cuda.stream(self.stream):
                ms_cb, _ = timed(lambda: torch.matmul(pr["x"], Wt.t()), K)
            res["ms_cublas_in"] = ms_cb
        del pr, q, k, v, g, y, ws
        torch.cuda.empty_cache()
        return res

    # ---------------------------------------------------------------- prefill
    def prefill(self, wl_name, e2e=True):
        torch, kda, synth = self.torch, self.kda, self.synth
        wl = synth.WORKLOADS[wl_name]
        if self.args.prefill_shape:   # profiling: a smaller case of the workload
            sB, sH, sT = (int(x) for x in self.args.prefill_shape.split(","))
            wl = synth.shrink(wl, B=sB, H=sH, T=sT)
        p = synth.make_params(wl, self.dev)
        tk = synth.make_tokens(wl, self.dev)
        st = synth.make_state(wl, self.dev)
        S, cs = st["S"], st["conv_state"]
        B, T, H = wl.B, wl.T, wl.H
        o = torch.empty((B, T, H, D), device=self.dev)
        q, k, v = (tk[n].view(torch.int16) for n in ("q", "k", "v"))
        ctx = kda.kda_create(H, p["conv_w"], p["dt_bias"], p["A_log"], p["gamma"])
        nws = kda.kda_prefill_workspace_bytes(ctx, B, T)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=self.dev)
        W = max(3, self.args.warmup)
        K = max(3, min(self.args.steps, self.args.prefill_steps))

        def call(qq, kk, vv, zz, bb, gg, out):
            S.zero_()
            cs.zero_()
            kda.kda_prefill(ctx, B, T, qq, kk, vv, zz, bb, gg, cs, S, out, ws, nws, self.stream)

        for _ in range(W):
            call(q, k, v, tk["z"], tk["beta_logit"], tk["gate_logit"], o)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        self.barrier_sync()
        l0 = kda.kda_launch_count()
        for i in range(K):
            S.zero_()
            cs.zero_()
            ev[i][0].record(self.stream)
            kda.kda_prefill(ctx, B, T, q, k, v, tk["z"], tk["beta_logit"], tk["gate_logit"],
                            cs, S, o, ws, nws, self.stream)
            ev[i][1].record(self.stream)
        self.barrier_sync()
        launches = kda.kda_launch_count() - l0
        times = [a.elapsed_time(b) for a, b in ev]
        ms = self.max_over_ranks(statistics.fmean(times))
        assert kda.kda_sync_status(ctx, self.stream) == kda.KDA_OK

        ms_e2e, h2d, d2h = None, 0, 0
        if e2e:
            # End to end with pinned host buffers (inputs in, o out, every
            # call), as a serving loop runs it: within a call, group j's inputs
            # are copied in on one stream while group j - 1 runs (one
            # kda_prefill call per group of sequences) and finished groups'
            # outputs are copied out on a third stream; across calls, the next
            # call's copies overlap this call's kernels and copy-out.  Device
            # inputs and outputs alternate between two sets: a copy-in waits
            # for the kernel two calls back that read its buffers, a kernel
            # for the copy-out two calls back of its output.  Value: the time
            # of Ke calls / Ke (events on the kernel stream around the loop).
            names = ("q", "k", "v", "z", "beta_logit", "gate_logit")
            host = {n: tk[n].to("cpu").pin_memory() for n in names}
            o_host = torch.empty((B, T, H, D), pin_memory=True)
            h2d = sum(x.numel() * x.element_size() for x in host.values())
            d2h = o_host.numel() * 4
            dbuf = [tk, {n: torch.empty_like(tk[n]) for n in names}]
            obuf = [o, torch.empty_like(o)]
            groups = [(b, min(B, b + max(1, B // 4))) for b in range(0, B, max(1, B // 4))]
            s_in = torch.cuda.Stream(device=self.dev)
            s_out = torch.cuda.Stream(device=self.dev)
            ev_k, ev_o = {}, {}

            def calls(i0, n):
                for i in range(i0, i0 + n):
                    p = i % 2
                    db, ob = dbuf[p], obuf[p]
                    S.zero_()
                    cs.zero_()
                    for j, (b0, b1) in enumerate(groups):
                        if (i - 2, j) in ev_k:
                            s_in.wait_event(ev_k.pop((i - 2, j)))
                        with torch.cuda.stream(s_in):
                            for nm in names:
                                db[nm][b0:b1].copy_(host[nm][b0:b1], non_blocking=True)
                        e_in = torch.cuda.Event()
                        e_in.record(s_in)
                        self.stream.wait_event(e_in)
                        if (i - 2, j) in ev_o:
                            self.stream.wait_event(ev_o.pop((i - 2, j)))
                        kda.kda_prefill(ctx, b1 - b0, T, db["q"][b0:b1].view(torch.int16),
                                        db["k"][b0:b1].view(torch.int16), db["v"][b0:b1].view(torch.int16),
                                        db["z"][b0:b1], db["beta_logit"][b0:b1], db["gate_logit"][b0:b1],
                                        cs[b0:b1], S[b0:b1], ob[b0:b1], ws, nws, self.stream)
                        e_k = torch.cuda.Event()
                        e_k.record(self.stream)
                        ev_k[(i, j)] = e_k
                        s_out.wait_event(e_k)
                        with torch.cuda.stream(s_out):
                            o_host[b0:b1].copy_(ob[b0:b1], non_blocking=True)
                        e_o = torch.cuda.Event()
                        e_o.record(s_out)
                        ev_o[(i, j)] = e_o

            Ke = 3
            calls(0, 1)                                     # warm-up
            self.barrier_sync()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            s_in.wait_event(e0)
            s_out.wait_event(e0)
            calls(1, Ke)
            self.stream.wait_stream(s_out)
            e1.record(self.stream)
            self.barrier_sync()
            ms_e2e = self.max_over_ranks(e0.elapsed_time(e1) / Ke)
            del dbuf, obuf, host, o_host
        kda.kda_destroy(ctx)
        th = B * T * H
        io_bytes = th * (3 * D * 2 + 3 * D * 4 + 4) + B * H * (STATE_BYTES + 2 * 9 * D * 4) \
            + H * 7680
        per_call = launches // K
        kernels = ("kda_prefill_kernel" if nws == 0 else
                   "kda_prefill_split_kernel" if per_call == 1 else
                   "kda_prefill_kernel + kda_prefill_split_kernel (last partial wave)")
        res = {"wl": wl, "ms": ms, "launches": launches, "kernels": kernels, "workspace_bytes": nws,
               "tokens_s": self.world * B * T / (ms * 1e-3),
               "e2e_tokens_s": None if ms_e2e is None else self.world * B * T / (ms_e2e * 1e-3),
               "ms_e2e": ms_e2e, "h2d": h2d, "d2h": d2h, "alg_bytes": io_bytes,
               "alg_gbs": io_bytes / (ms * 1e-3) / 1e9,
               "alg_tflops": th * PREFILL_FLOP_PER_TOKEN_HEAD / (ms * 1e-3) / 1e12}
        del tk, S, cs, o
        torch.cuda.empty_cache()
        return res


    # ------------------------------------------------------- packed-sequence prefill
    def prefill_varlen(self):
        """kda_prefill_varlen on 32 packed sequences of mixed lengths (64 heads):
        lengths 2^U(8, 13) rounded (seed 5), q/k/v bf16 N(0, 1), the
        prefill_b8_h64_t8192 parameter recipe, zero initial state."""
        torch, kda, synth = self.torch, self.kda, self.synth
        import numpy as np
        lengths = synth.packed_lengths()
        total = int(lengths.sum())
        wl = synth.packed_workload(lengths)
        p = synth.make_params(wl, self.dev)
        tk = synth.make_tokens(wl, self.dev)
        H = wl.H
        Bs = len(lengths)
        S = torch.zeros((Bs, H, D, D), device=self.dev)
        cs = torch.zeros((Bs, 3, 3 * H * D), device=self.dev)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=self.dev)
        q, k, v = (tk[n][0].view(torch.int16) for n in ("q", "k", "v"))
        z, bl, g = tk["z"][0], tk["beta_logit"][0], tk["gate_logit"][0]
        o = torch.empty((total, H, D), device=self.dev)
        ctx = kda.kda_create(H, p["conv_w"], p["dt_bias"], p["A_log"], p["gamma"])
        W = max(3, self.args.warmup)
        K = max(3, min(self.args.steps, self.args.prefill_steps))
        for _ in range(W):
            S.zero_()
            cs.zero_()
            kda.kda_prefill_varlen(ctx, Bs, cu, total, q, k, v, z, bl, g, cs, S, o, self.stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        self.barrier_sync()
        l0 = kda.kda_launch_count()
        for i in range(K):
            S.zero_()
            cs.zero_()
            ev[i][0].record(self.stream)
            kda.kda_prefill_varlen(ctx, Bs, cu, total, q, k, v, z, bl, g, cs, S, o, self.stream)
            ev[i][1].record(self.stream)
        self.barrier_sync()
        launches = kda.kda_launch_count() - l0
        ms = self.max_over_ranks(statistics.fmean(a.elapsed_time(b) for a, b in ev))
        assert kda.kda_sync_status(ctx, self.stream) == kda.KDA_OK
        kda.kda_destroy(ctx)
        th = total * H
        io_bytes = th * (3 * D * 2 + 3 * D * 4 + 4) + Bs * H * (STATE_BYTES + 2 * 9 * D * 4) + H * 7680
        res = {"sequences": Bs, "H": H, "total_tokens": total, "min_len": int(lengths.min()),
               "max_len": int(lengths.max()), "ms": ms, "launches": launches,
               "tokens_s": self.world * total / (ms * 1e-3), "alg_bytes": io_bytes,
               "alg_gbs": io_bytes / (ms * 1e-3) / 1e9}
        del tk, S, cs, o
        torch.cuda.empty_cache()
        return res


# ----------------------------------------------------------------------------- oracle arm

def oracle_decode(wl_name, budget_s, calls_cap, pairs=None, threads=None):
    """Time the fp64 oracle on decode calls of a workload.

    Each call covers the first ``pairs`` (sequence, head) pairs in (b, h)
    order (all of them when None), so a call is a bounded sample of the
    workload's call; the inputs of the first calls are cycled.
    """
    import numpy as np
    from kda_delta_rule_token_gb300 import synth
    import oracle
    wl = synth.WORKLOADS[wl_name]
    nthreads = threads or oracle.cpu_count()
    Bs = wl.B if pairs is None else max(1, min(wl.B, pairs // wl.H))
    small = synth.shrink(wl, B=Bs)
    p = {k: v.numpy().astype(np.float64) for k, v in synth.make_params(small, "cpu").items()}
    st = {k: v.numpy().astype(np.float64) for k, v in synth.make_state(small, "cpu").items()}
    ncalls = max(1, min(wl.T, calls_cap, 16))
    tk = synth.make_tokens(small, "cpu", T=ncalls)
    S, cs = st["S"], st["conv_state"]
    done, elapsed = 0, 0.0
    per_call = []
    while done < calls_cap and elapsed < budget_s:
        t = done % ncalls
        one = {n: tk[n][t:t + 1].transpose(0, 1).contiguous().numpy().astype(np.float64)
               for n in ("q", "k", "v", "z", "gate_logit", "beta_logit")}
        t0 = time.perf_counter()
        out = oracle.run(**one, conv_w=p["conv_w"], dt_bias=p["dt_bias"], A_log=p["A_log"],
                         gamma=p["gamma"], conv_state=cs, S=S, nthreads=nthreads)
        dt = time.perf_counter() - t0
        S, cs = out.S, out.conv_state
        per_call.append(dt)
        elapsed += dt
        done += 1
    units = Bs * wl.H
    return {"gbs": done * units * STATE_BYTES / elapsed / 1e9, "calls": done,
            "per_call": per_call, "threads": nthreads, "units": units,
            "sample": f"{done} decode calls over {Bs} of the {wl.B} sequences x {wl.H} heads "
                      f"({units} pairs per call; the first {ncalls} calls' inputs cycled), fp64, "
                      f"{nthreads} threads, state GB/s of the pairs processed"}


def oracle_prefill(wl_name, tokens, heads=None):
    """Time the fp64 oracle on one sequence of ``tokens`` tokens over ``heads``
    heads of a prefill workload's shape (heads = this host's cores by default,
    one head per thread); tokens/s is scaled to the workload's head count."""
    import numpy as np
    from kda_delta_rule_token_gb300 import synth
    import oracle
    wl = synth.WORKLOADS[wl_name]
    nthreads = oracle.cpu_count()
    heads = heads or max(nthreads, 1)
    small = synth.shrink(wl, B=1, H=heads, T=tokens)
    p = {k: v.numpy().astype(np.float64) for k, v in synth.make_params(small, "cpu").items()}
    tk = {k: v.float().numpy().astype(np.float64) for k, v in
          synth.make_tokens(small, "cpu").items()}
    st = {k: v.numpy().astype(np.float64) for k, v in synth.make_state(small, "cpu").items()}
    t0 = time.perf_counter()
    oracle.run(**tk, conv_w=p["conv_w"], dt_bias=p["dt_bias"], A_log=p["A_log"],
               gamma=p["gamma"], conv_state=st["conv_state"], S=st["S"], nthreads=nthreads)
    dt = time.perf_counter() - t0
    token_heads = heads * tokens
    return {"tokens_s": token_heads / wl.H / dt, "threads": min(nthreads, heads), "seconds": dt,
            "sample": f"1 sequence x {heads} heads x {tokens} tokens of the "
                      f"{wl.B}x{wl.H}x{wl.T} prefill shape (fp64 sequential per head, "
                      f"{min(nthreads, heads)} threads; tokens/s scaled by {heads}/{wl.H} heads)"}


REF_PAIRS = 2048   # (sequence, head) pairs per reference-arm step: a bounded sample of a call


def run_reference(args, world, rank):
    """--impl reference: the fp64 oracle as it stands, on this host's cores,
    on the headline workload's decode calls (each step one call over a
    bounded sample of its (sequence, head) pairs)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    W, K = args.warmup, args.steps
    calls = W + K
    from kda_delta_rule_token_gb300 import synth
    wl = synth.WORKLOADS[HEADLINE_WL]
    r = oracle_decode(HEADLINE_WL, budget_s=float("inf"), calls_cap=calls, pairs=REF_PAIRS)
    timed = r["per_call"][W:]
    ms = statistics.fmean(timed) * 1e3
    value = r["units"] * STATE_BYTES / (ms * 1e-3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": HEADLINE_WL, "B": wl.B, "H": wl.H, "d": D,
                   "calls_cycled": wl.T, "state_MiB": wl.B * wl.H * D * D * 4 / 2**20,
                   "l2": "n/a (CPU)", "parallelism": "rank 0 only",
                   "pairs_per_step": r["units"]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": r["threads"],
                         "kind": "oracle", "sample": r["sample"]},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main

def decode_block(res, peaks, md_name, sha, flush_note, kernel="kda_decode_kernel"):
    wl = res["wl"]
    hb = peaks["hbm_gbs"]
    out = {
        "workload": wl.name, "B": wl.B, "H": wl.H, "d": D, "calls_cycled": wl.T,
        "state_MiB": wl.B * wl.H * D * D * res["state_elem_bytes"] / 2**20, "l2": flush_note,
        "initial_state": f"after {wl.warmup_tokens} warm-up tokens" if wl.warmup_tokens else
                         "N(0, 0.01) state, N(0, 1) window",
        "ms_per_call": round(res["ms"], 5), "state_gbs": round(res["state_gbs"], 1),
        "gpu_launches": res["launches"],
        "roofline": {"bound": "hbm", "achieved": round(res["alg_gbs"], 1), "peak": hb,
                     "unit": "GB/s", "frac": round(res["alg_gbs"] / hb, 4),
                     "traffic": profile_traffic(md_name, sha),
                     "kernel": kernel, "peak_src": peaks["src"] + " hbm_gbs",
                     "alg_bytes_per_launch": res["alg_bytes"]},
    }
    if res.get("ms_graph") is not None:
        out["graph"] = {"calls_per_graph": wl.T, "ms_per_call": round(res["ms_graph"], 5),
                        "state_gbs": round(res["state_gbs_graph"], 1),
                        "frac": round(res["alg_gbs_graph"] / hb, 4),
                        "gpu_launches": res["graph_launches"]}
    if res.get("ms_e2e") is not None:
        out["e2e"] = {"value": round(res["e2e_gbs"], 2), "unit": "GB/s",
                      "ms_per_step": round(res["ms_e2e"], 5),
                      "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"]}
    return out


def prefill_block(pre, peaks, steps, md_name, sha, cpu=None):
    pw = pre["wl"]
    tf32_peak = peaks["bf16_tflops"] * 0.5
    blk = {
        "workload": pw.name, "B": pw.B, "H": pw.H, "T": pw.T, "chunk": pw.chunk,
        "value": round(pre["tokens_s"], 1), "unit": "tokens/s",
        "ms_per_step": round(pre["ms"], 4), "steps": steps,
        "dtype": "bf16 in, f32 compute/state/out",
        "l2": f"inputs and output {pre['alg_bytes'] / 1e9:.2f} GB > L2",
        "gpu_launches": pre["launches"],
        "roofline": {"bound": "hbm", "achieved": round(pre["alg_gbs"], 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(pre["alg_gbs"] / peaks["hbm_gbs"], 4),
                     "traffic": profile_traffic(md_name, sha),
                     "kernel": pre["kernels"], "peak_src": peaks["src"] + " hbm_gbs",
                     "alg_bytes_per_launch": pre["alg_bytes"]},
        "workspace_bytes": pre["workspace_bytes"],
        "tensor": {"achieved_tflops": round(pre["alg_tflops"], 2),
                   "pct_of_bf16_peak": round(100 * pre["alg_tflops"] / peaks["bf16_tflops"], 2),
                   "pct_of_tf32_peak": round(100 * pre["alg_tflops"] / tf32_peak, 2),
                   "flop_per_token_head": PREFILL_FLOP_PER_TOKEN_HEAD},
    }
    if pre.get("ms_e2e") is not None:
        blk["e2e"] = {"value": round(pre["e2e_tokens_s"], 1), "unit": "tokens/s",
                      "ms_per_step": round(pre["ms_e2e"], 3),
                      "h2d_bytes_per_step": pre["h2d"], "d2h_bytes_per_step": pre["d2h"]}
    if cpu is not None:
        blk["cpu_baseline"] = {"value": round(cpu["tokens_s"], 3), "unit": "tokens/s",
                               "cores": cpu["threads"], "kind": "oracle", "sample": cpu["sample"]}
    return blk


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill-steps", type=int, default=10)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip every decode line (profiling only)")
    ap.add_argument("--prefill-workload", default=None,
                    help="profiling only: time this prefill workload alone")
    ap.add_argument("--prefill-shape", default=None,
                    help="profiling only: with --prefill-workload, 'B,H,T' of a smaller case of it")
    ap.add_argument("--decode-workload", default=None,
                    help="profiling only: time this decode workload alone (no e2e, no graph)")
    ap.add_argument("--bf16-state", action="store_true",
                    help="profiling only: with --decode-workload, the bf16-state decode")
    ap.add_argument("--varlen-only", action="store_true",
                    help="profiling only: time the packed-sequence prefill alone")
    ap.add_argument("--lowrank-only", action="store_true",
                    help="profiling only: time the low-rank front-end decode line alone")
    ap.add_argument("--proj-only", default=None,
                    help="profiling only: time the projections on this workload's tokens alone")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-split", type=int, default=1,
                    help="groups of sequences the decode end-to-end step is pipelined over")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    ours = Ours(args, world, rank, local)
    peaks = load_peaks()
    if args.prefill_workload or args.decode_workload or args.lowrank_only or args.proj_only or args.varlen_only:
        # profiling runs
        out = {"profiling_only": True}
        if args.proj_only:
            r = ours.projections(args.proj_only, with_cublas=False)
            out.update(proj_workload=args.proj_only, proj_in_ms=round(r["ms_in"], 4), proj_out_ms=round(r["ms_out"], 4))
        if args.lowrank_only:
            r = ours.decode_lowrank(DECODE_WL)
            out.update(lowrank_step_ms=round(r["ms_step"], 5), lowrank_frontend_ms=round(r["ms_frontend"], 5))
        if args.varlen_only:
            r = ours.prefill_varlen()
            out.update(varlen_ms=round(r["ms"], 4), varlen_tokens=r["total_tokens"])
        if args.prefill_workload:
            r = ours.prefill(args.prefill_workload, e2e=False)
            out.update(prefill_workload=args.prefill_workload, prefill_ms=round(r["ms"], 4))
        if args.decode_workload:
            r = ours.decode(args.decode_workload, flush=False, e2e=False, state_bf16=args.bf16_state)
            out.update(decode_workload=args.decode_workload, decode_ms=round(r["ms"], 5),
                       bf16_state=args.bf16_state)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return

    clocks = ClockSampler(local)
    clocks.start()
    head = None if args.no_decode else ours.decode(HEADLINE_WL, flush=False, graph=True)
    dec = None if args.no_decode else ours.decode(DECODE_WL, flush=True, e2e=False)
    d16 = None if args.no_decode else ours.decode(HEADLINE_WL, flush=False, e2e=False, state_bf16=True)
    dlr = None if args.no_decode else ours.decode_lowrank(DECODE_WL)
    psteps = max(3, min(args.steps, args.prefill_steps))
    pre = None if args.no_prefill else ours.prefill(PREFILL_WL)
    pre1 = None if args.no_prefill else ours.prefill(PREFILL1_WL, e2e=False)
    pvl = None if args.no_prefill else ours.prefill_varlen()
    prj = None if args.no_prefill else ours.projections(PREFILL_WL)
    prd = None if args.no_decode else ours.projections(DECODE_WL, with_cublas=False)
    clk = clocks.stop()

    if rank != 0:
        return
    cpu_head = None if (args.no_cpu_baseline or head is None) else \
        oracle_decode(HEADLINE_WL, budget_s=10.0, calls_cap=100000, pairs=None)
    cpu_pre = None if (args.no_cpu_baseline or pre is None) else oracle_prefill(PREFILL_WL, 8192)
    cpu_pre1 = None if (args.no_cpu_baseline or pre1 is None) else oracle_prefill(PREFILL1_WL, 4096)

    dsha = source_sha("decode.cu")
    psha = source_sha("prefill.cu", "ptx.cuh", "tc.cuh")
    lsha = source_sha("lowrank.cu", "ptx.cuh", "tc.cuh")
    prsha = source_sha("proj.cu", "ptx.cuh", "tc.cuh")
    line = {"metric": METRIC}
    if head is not None:
        wl = head["wl"]
        hb = decode_block(head, peaks, "decode_b256_h64_kda_decode_kernel.md", dsha,
                          "state 1 GiB > L2, calls back to back")
        line.update({
            "value": round(head["state_gbs"], 2), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(head["ms"], 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": HEADLINE_WL, "B": wl.B, "H": wl.H, "d": D,
                       "calls_cycled": wl.T, "state_MiB": wl.B * wl.H * D * D * 4 / 2**20,
                       "initial_state": hb["initial_state"],
                       "l2": "inputs larger than L2 (1 GiB of state read and written per call)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "state_pct_of_hbm_peak": round(100 * head["state_gbs"] / world / peaks["hbm_gbs"], 2),
            "roofline": hb["roofline"],
            "e2e": hb["e2e"],
            "gpu_launches": head["launches"],
            "graph": hb["graph"],
        })
    line["clocks"] = clk
    if cpu_head is not None:
        line["cpu_baseline"] = {"value": round(cpu_head["gbs"], 4), "unit": "GB/s",
                                "cores": cpu_head["threads"], "kind": "oracle",
                                "sample": cpu_head["sample"]}
    if dec is not None:
        line["decode_b64_h32"] = decode_block(
            dec, peaks, "decode_b64_h32_kda_decode_kernel.md", dsha,
            "state 128 MiB < L2: flushed between timed calls (256 MiB write + 256 MiB read)")
    if d16 is not None:
        blk = decode_block(d16, peaks, "decode_b256_h64_bf16state_kda_decode_kernel.md", dsha,
                           "state 512 MiB > L2, calls back to back",
                           kernel="kda_decode_kernel<bf16 state>")
        blk["dtype"] = "bf16 state, f32 compute and I/O"
        blk["state_bytes_per_head_step"] = STATE_BYTES // 2
        line["decode_bf16state"] = blk
    if dlr is not None:
        w = dlr["wl"]
        fe_gbs = dlr["fe_bytes"] / (dlr["ms_frontend"] * 1e-3) / 1e9
        line["decode_lowrank"] = {
            "workload": w.name + f" through the low-rank front-end (hidden {dlr['hidden']}, rank {dlr['rank']})",
            "B": w.B, "H": w.H, "l2": "flushed between timed calls",
            "ms_per_call": round(dlr["ms_step"], 5), "state_gbs": round(dlr["state_gbs"], 1),
            "gpu_launches": dlr["launches_step"],
            "frontend": {
                "ms_per_call": round(dlr["ms_frontend"], 5), "gpu_launches": dlr["launches_frontend"],
                "tflops_algorithmic": round(dlr["fe_flop"] / (dlr["ms_frontend"] * 1e-3) / 1e12, 3),
                "roofline": {"bound": "hbm", "achieved": round(fe_gbs, 1), "peak": peaks["hbm_gbs"],
                             "unit": "GB/s", "frac": round(fe_gbs / peaks["hbm_gbs"], 4),
                             "traffic": profile_traffic("lowrank_b64_h32_kda_lowrank_gemm_kernel.md", lsha),
                             "kernel": "kda_lowrank_gemm_kernel + kda_lowrank_reduce_kernel",
                             "alg_bytes_per_call": dlr["fe_bytes"]},
            },
        }
    if pre is not None:
        line["prefill"] = prefill_block(pre, peaks, psteps, "prefill_b8_h64_kernel.md", psha, cpu_pre)
    if pre1 is not None:
        line["prefill_single"] = prefill_block(pre1, peaks, psteps, "prefill_b1_h32_kernel.md", psha,
                                               cpu_pre1)
    if pvl is not None:
        line["prefill_varlen"] = {
            "workload": "32 packed sequences, lengths 2^U(8,13) (seed 5), H=64, chunk 64",
            "sequences": pvl["sequences"], "H": pvl["H"], "total_tokens": pvl["total_tokens"],
            "min_len": pvl["min_len"], "max_len": pvl["max_len"],
            "value": round(pvl["tokens_s"], 1), "unit": "tokens/s", "ms_per_step": round(pvl["ms"], 4),
            "gpu_launches": pvl["launches"],
            "roofline": {"bound": "hbm", "achieved": round(pvl["alg_gbs"], 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(pvl["alg_gbs"] / peaks["hbm_gbs"], 4),
                         "traffic": profile_traffic("prefill_varlen_kernel.md", psha),
                         "kernel": "kda_prefill_kernel",
                         "alg_bytes_per_launch": pvl["alg_bytes"]},
        }
    for key, r in (("projections", prj), ("projections_decode", prd)):
        if r is None:
            continue
        w = r["wl"]
        tin = r["flop_in"] / (r["ms_in"] * 1e-3) / 1e12
        tout = r["flop_out"] / (r["ms_out"] * 1e-3) / 1e12
        gin = r["bytes_in"] / (r["ms_in"] * 1e-3) / 1e9
        gout = r["bytes_out"] / (r["ms_out"] * 1e-3) / 1e9
        big = r["N"] > 4096
        tr_in = profile_traffic(PROJ_MD, prsha, f"per call (qkvg, {w.name})")
        tr_out = profile_traffic(PROJ_MD, prsha, f"per call (o, {w.name})")
        blk = {
            "workload": f"{w.name}: {r['N']} tokens, hidden {r['hidden']}, H={r['H']}, bf16 operands, fp32 accumulation",
            "qkvg": {"ms_per_call": round(r["ms_in"], 4), "tflops": round(tin, 1), "gbs": round(gin, 1),
                     "gpu_launches": r["launches_in"],
                     "roofline": ({"bound": "tensor", "achieved": round(tin, 1), "peak": peaks["bf16_tflops"],
                                   "unit": "TFLOP/s", "frac": round(tin / peaks["bf16_tflops"], 4),
                                   "peak_src": peaks["src"] + " bf16_tflops (burst)", "traffic": tr_in}
                                  if big else
                                  {"bound": "hbm", "achieved": round(gin, 1), "peak": peaks["hbm_gbs"],
                                   "unit": "GB/s", "frac": round(gin / peaks["hbm_gbs"], 4),
                                   "peak_src": peaks["src"] + " hbm_gbs", "traffic": tr_in}),
                     "kernel": "kda_proj_gemm_kernel"},
            "o": {"ms_per_call": round(r["ms_out"], 4), "tflops": round(tout, 1), "gbs": round(gout, 1),
                  "gpu_launches": r["launches_out"],
                  "roofline": ({"bound": "tensor", "achieved": round(tout, 1), "peak": peaks["bf16_tflops"],
                                "unit": "TFLOP/s", "frac": round(tout / peaks["bf16_tflops"], 4),
                                "peak_src": peaks["src"] + " bf16_tflops (burst)", "traffic": tr_out}
                               if big else
                               {"bound": "hbm", "achieved": round(gout, 1), "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": round(gout / peaks["hbm_gbs"], 4),
                                "peak_src": peaks["src"] + " hbm_gbs", "traffic": tr_out}),
                  "kernel": "kda_to_bf16_kernel + kda_proj_gemm_kernel"},
        }
        if "ms_cublas_in" in r:
            blk["qkvg"]["context_cublas_bf16_ms"] = round(r["ms_cublas_in"], 4)
        line[key] = blk
    print(json.dumps(line), flush=True)
    if ours.dist is not None:
        ours.dist.destroy_process_group()


if __name__ == "__main__":
    main()
