"""Benchmark: VeriCache draft decode-attention throughput on GB300.

One step = one VeriCache round of one attention layer for the 8B-shaped
workload (batch 8, 32 query / 8 kv heads, head_dim 128, 32768-token context,
KV_comp = every token at 2-bit group-32):
  for i in 0..x-1:  vc_draft_step append drafted token i's K / V rows to
                                  KV_comp (2-bit) and attend over its
                                  N + i + 1 entries, one launch (+ combine)
  vc_verify_attn    the x = 32 block queries over bf16 KV_full (causal):
                    the pending token and the first x - 1 drafts, whose
                    predictions check all x drafts (the workload's "verify
                    x = 32 queries"; no bonus prediction in this timing)
  vc_accept         LM-head argmax (mean of the query-head outputs, d 128,
                    vocab 32000) + longest matching prefix
value = drafted tokens per second = batch * x / step time (whole round, all
kernels), inputs resident in HBM.  The roofline object reports the draft
kernel alone: algorithmic bytes (KV_comp bytes read per call) / its mean
CUDA-event duration inside the timed region.

e2e: the same round through the same C-ABI calls with host buffers: per step
the queries are copied from pinned host memory, KV_full (the page's
"full KV in CPU memory") is staged host->device on a side stream while the
drafting runs, and the verified / emitted tokens are copied back.

other_workloads: after the headline's timed region, rank 0 times the other
workloads of the path on the device (CUDA events): the 70B-shaped layer
(draft over bf16 token-drop KV_comp, 40-query verify over a 131072-token
KV_full, GPU token selection) with the 40k-context verify point, one
staggered mixed launch of the 32-request 3-bit workload, and the headline's
draft step at 3 and 4 bits.  Beside each, unless --no-cpu-baseline, a
`cpu_baseline`: the oracle on a bounded sample of the same shape (about 2 s
each; drafted tokens/s, or verified query-head rows/s, matching the device
key it sits beside).

--impl reference: the CPU oracle on this machine's cores, a bounded sample
of the same workload per step (draft attention of one request).
Multi-GPU (torchrun): independent replicas, weak scaling, no data-path
collective; timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft decode-attn tokens/s and achieved HBM TB/s (% of peak), 8B-shape 32k ctx"
WORKLOAD = "8b_32k_2bit"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """nvidia-smi samples during the timed region: the sampler is started and
    its first line awaited before the region begins (nvidia-smi takes longer
    to start than a short timed region lasts), that line is dropped, and the
    GPU is polled every 10 ms."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.skip = 0

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.perf_counter()
            while not self.lines and time.perf_counter() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.005)
            self.skip = len(self.lines)
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

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.skip:]:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return rank, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allmax(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# workload construction (device-resident)
# ---------------------------------------------------------------------------

def build(w, seed, device):
    import torch
    import lossless_compressed_kv_gb300 as vc
    B, hq, hkv, d, N, x, bits = w["batch"], w["hq"], w["hkv"], w["d"], w["ctx"], w["x"], w["bits"]
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    L = N + x                                  # prefix + verification block of x queries
    npg = (L + 15) // 16
    P = B * npg
    perm = torch.randperm(P, generator=g, device=device).to(torch.int32)
    table = perm.view(B, npg).contiguous()
    oc = torch.randperm(d, generator=g, device=device)[:w["outliers"]]
    kp = torch.empty((P, hkv, 16, d), dtype=torch.bfloat16, device=device)
    vp = torch.empty_like(kp)
    for s in range(0, P, 512):                 # fp32 draws -> bf16 (round to nearest even)
        e = min(P, s + 512)
        kk = torch.randn((e - s, hkv, 16, d), generator=g, device=device)
        kk[..., oc] *= w["outlier_scale"]
        kp[s:e] = kk.to(torch.bfloat16)
        vp[s:e] = torch.randn((e - s, hkv, 16, d), generator=g, device=device).to(torch.bfloat16)
    full = vc.PagedKV(kp.view(torch.uint8).view(P, -1), vp.view(torch.uint8).view(P, -1), table,
                      torch.full((B,), L, dtype=torch.int32, device=device), hkv, d, 16)
    cpg = (N + x + 15) // 16
    cperm = torch.randperm(B * cpg, generator=g, device=device).to(torch.int32)
    comp = vc.PagedKV.allocate(B * cpg, hkv, d, bits, cperm.view(B, cpg).contiguous(),
                               torch.full((B,), N, dtype=torch.int32, device=device), device=device)
    # registration: KV_comp of the N-token prefix (every token kept)
    offs = torch.arange(0, B * N + 1, N, dtype=torch.int32, device=device)
    idx = torch.arange(N, dtype=torch.int32, device=device).repeat(B)
    vc.compress(full, offs, idx, comp, N)
    q = torch.randn((x, B, hq, d), generator=g, device=device).to(torch.bfloat16)
    qv = q.permute(1, 0, 2, 3).contiguous()    # [B][x][Hq][D] verify block (same queries as the drafts)
    # the K / V rows of drafted token i (position N + i), as a model step
    # hands them over: [x][B][Hkv][D]
    kn = torch.stack([kp[table[:, (N + i) // 16].long(), :, (N + i) % 16, :] for i in range(x)]).contiguous()
    vn = torch.stack([vp[table[:, (N + i) // 16].long(), :, (N + i) % 16, :] for i in range(x)]).contiguous()
    lm = torch.randn((d, w["vocab"]), generator=g, device=device) * w["lm_std"]
    drafts = torch.randint(0, w["vocab"], (B, x), generator=g, device=device).to(torch.int32)
    return dict(full=full, comp=comp, q=q, qv=qv, kn=kn, vn=vn, lm=lm, drafts=drafts, oc=oc, L=L)


class Round:
    """One VeriCache round for one attention layer (all buffers preallocated)."""

    def __init__(self, w, st, device):
        import torch
        import lossless_compressed_kv_gb300 as vc
        self.vc, self.w, self.st = vc, w, st
        B, hq, d, N, x = w["batch"], w["hq"], w["d"], w["ctx"], w["x"]
        self.B, self.N, self.x, self.hq, self.d = B, N, x, hq, d
        full, comp = st["full"], st["comp"]
        self.scale = 1.0 / math.sqrt(d)
        # per draft step: the new entry's KV_comp position and the attended lengths
        self.app_start = [torch.full((B,), N + i, dtype=torch.int32, device=device) for i in range(x)]
        self.comp_i = [vc.PagedKV(comp.k_pages, comp.v_pages, comp.block_table,
                                  torch.full((B,), N + i + 1, dtype=torch.int32, device=device),
                                  comp.num_kv_heads, comp.head_dim, comp.bits) for i in range(x)]
        self.dout = torch.empty((B, hq, d), dtype=torch.float32, device=device)
        self.dws = torch.empty(vc.draft_workspace_bytes(comp, hq, N + x), dtype=torch.uint8, device=device)
        self.vout = torch.empty((B, x, hq, d), dtype=torch.float32, device=device)
        self.vws = torch.empty(vc.verify_workspace_bytes(full, x, hq, st["L"]), dtype=torch.uint8,
                               device=device)
        self.ver = torch.empty((B, x), dtype=torch.int32, device=device)
        self.alen = torch.empty((B,), dtype=torch.int32, device=device)
        self.emit = torch.empty((B, x + 1), dtype=torch.int32, device=device)
        self.aws = torch.empty(vc.accept_workspace_bytes(B, x, w["vocab"], d), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # kernels per round: x x (draft step + its reduce), verify + its
        # reduce, accept's mean + logits + finalize
        self.launches = x * 2 + 2 + 3

    def run(self, q=None, qv=None, ev=None, full=None, verify_wait=None):
        import torch
        vc, st = self.vc, self.st
        q = st["q"] if q is None else q
        qv = st["qv"] if qv is None else qv
        full = st["full"] if full is None else full
        # ev: {call index: (event recorded before it or None, event after it or None)}
        for i in range(self.x):
            if ev is not None and i in ev and ev[i][0] is not None:
                ev[i][0].record()
            vc.draft_step(q[i], self.comp_i[i], st["kn"][i], st["vn"][i], self.app_start[i], self.scale, self.dout,
                          self.N + self.x, self.dws, status=self.status)
            if ev is not None and i in ev and ev[i][1] is not None:
                ev[i][1].record()
        if verify_wait is not None:
            torch.cuda.current_stream().wait_event(verify_wait)
        vc.verify_attn(qv, full, self.scale, self.vout, st["L"], self.vws, status=self.status)
        vc.accept(self.vout, st["lm"], st["drafts"], self.ver, self.alen, self.emit, self.aws,
                  hidden_group=self.hq)


    def stage_calls(self):
        """The round split into its stages (each a list of API calls)."""
        vc, st = self.vc, self.st
        draft = [lambda i=i: vc.draft_step(st["q"][i], self.comp_i[i], st["kn"][i], st["vn"][i], self.app_start[i],
                                           self.scale, self.dout, self.N + self.x, self.dws, status=self.status)
                 for i in range(self.x)]
        verify = [lambda: vc.verify_attn(st["qv"], st["full"], self.scale, self.vout, st["L"], self.vws,
                                         status=self.status)]
        accept = [lambda: vc.accept(self.vout, st["lm"], st["drafts"], self.ver, self.alen, self.emit, self.aws,
                                    hidden_group=self.hq)]
        return {"draft_step": draft, "verify_attn": verify, "accept": accept}

    def breakdown(self, reps=5):
        """Per-stage device time: each stage's calls captured in a CUDA graph
        and its replays timed with CUDA events (no host gaps between calls)."""
        import torch
        out = {}
        for name, calls in self.stage_calls().items():
            g = capture(lambda: [c() for c in calls])
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g.replay()
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / reps
            out[name] = {"us_per_round": us, "us_per_call": us / len(calls)}
        return out


def capture(fn):
    """CUDA graph of the work `fn` enqueues on the current stream."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def draft_bytes(w, n_entries):
    """Algorithmic bytes of one draft call: every KV_comp entry of every kv
    head, K and V, codes + fp16 scale + fp16 zero."""
    d, bits, hkv = w["d"], w["bits"], w["hkv"]
    per_tok_head = 2 * (d * bits // 8 + 2 * 2 * d // 32)
    return w["batch"] * n_entries * hkv * per_tok_head


def bits_measure(w, device, bit_widths=(3, 4)):
    """The draft step (vc_draft_step: append + draft + reduce) of the
    headline workload's shape at other code widths: per call device time
    over graph replays of the x calls of a round, algorithmic bytes and the
    fraction of the measured HBM rate."""
    import torch
    peak, _ = peaks()
    out = {}
    for bits in bit_widths:
        w2 = dict(w, bits=bits)
        st2 = build(w2, 1234, device)
        rnd2 = Round(w2, st2, device)
        calls = rnd2.stage_calls()["draft_step"]
        us = _graph_us(torch, lambda: [c() for c in calls], 5) / len(calls)
        nb = float(np.mean([draft_bytes(w2, w2["ctx"] + i + 1) for i in range(len(calls))]))
        out["%d_bit" % bits] = {"us_per_call": us, "bytes_per_call": nb, "GBps": nb / us / 1e3,
                                "frac_hbm_measured": nb / us / 1e3 / peak,
                                "tokens_per_s": w["batch"] / (us * 1e-6)}
        del st2, rnd2
        torch.cuda.empty_cache()
    return out


def headline_config(w):
    """The `config` object of the headline line, the same for both arms."""
    N, x = w["ctx"], w["x"]
    span = (x // 4, (3 * x) // 4)
    comp_mb = float(np.mean([draft_bytes(w, N + i + 1) for i in range(*span)])) / 1e6
    full_mb = w["batch"] * ((N + x + 15) // 16) * 16 * w["hkv"] * w["d"] * 2 * 2 / 1e6
    return {"workload": WORKLOAD, "batch": w["batch"], "ctx": N, "q_heads": w["hq"], "kv_heads": w["hkv"],
            "head_dim": w["d"], "bits": w["bits"], "group": 32, "page": 16, "x": x, "verify_n_q": x,
            "lm_head": [w["d"], w["vocab"]], "parallelism": "replicas",
            "l2": "inputs larger than L2: KV_comp %.0f MB per draft call, KV_full %.0f MB per verify"
                  % (comp_mb, full_mb)}


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------

def oracle_sample(w, st, seconds_target=15.0, max_requests=128):
    """Time the oracle's draft attention on whole requests of the same
    workload (KV_comp built by the oracle's own compress from the same
    KV_full) until about `seconds_target` of CPU work."""
    import torch
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    N, d, hkv = w["ctx"], w["d"], w["hkv"]
    full = st["full"]
    done, t_total, n_threads = 0, 0.0, oracle.threads()
    with ThreadPoolExecutor(n_threads) as pool:
        cache = {}
        for it in range(max_requests):
            b = it % w["batch"]
            if b in cache:
                q, comp = cache[b]
                t0 = time.perf_counter()
                oracle.draft_attn(q, comp, float(np.float32(1 / math.sqrt(d))), pool=pool)
                t_total += time.perf_counter() - t0
                done += 1
                if t_total >= seconds_target:
                    break
                continue
            pages = full.block_table[b, :N // 16].long()
            k = full.k_pages[pages].view(torch.int16).view(-1, hkv, 16, d).permute(0, 2, 1, 3).reshape(N, hkv, d)
            v = full.v_pages[pages].view(torch.int16).view(-1, hkv, 16, d).permute(0, 2, 1, 3).reshape(N, hkv, d)
            k = k.cpu().numpy().view(np.uint16)
            v = v.cpu().numpy().view(np.uint16)
            q = st["q"][0, b].view(torch.int16).cpu().numpy().view(np.uint16)
            comp = oracle.compress(k, v, np.arange(N, dtype=np.int32), w["bits"])
            cache[b] = (q, comp)
            t0 = time.perf_counter()
            oracle.draft_attn(q, comp, float(np.float32(1 / math.sqrt(d))), pool=pool)
            t_total += time.perf_counter() - t0
            done += 1
            if t_total >= seconds_target:
                break
    return {"value": done / t_total, "unit": "tokens/s", "cores": n_threads, "kind": "oracle",
            "sample": "%d request-steps (cycling over the 8 requests) x 1 draft step (32 query heads over 32768 2-bit KV_comp entries); "
                      "KV_comp from the oracle's own compress; %.1f s of CPU time" % (done, t_total)}


def _oracle_reps(fn, seconds):
    """Call fn until about `seconds` of wall time; (calls, seconds)."""
    n, t = 0, 0.0
    while t < seconds:
        t0 = time.perf_counter()
        fn()
        t += time.perf_counter() - t0
        n += 1
    return n, t


def oracle_extras(seconds=2.0):
    """Bounded oracle samples beside the other workloads' device numbers, in
    the same units (drafted tokens/s; verified query-head rows/s), on seeded
    synthetic inputs of the same shapes (timing only: the values are not
    compared here).  Each sample runs for about `seconds`."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    import synth
    nt = oracle.threads()

    def entry(value, unit, sample):
        return {"value": value, "unit": unit, "cores": nt, "kind": "oracle", "sample": sample}

    def draft_leg(pool, k, v, bits, hq, what):
        n, hkv, d = k.shape
        comp = oracle.compress(k, v, np.arange(n, dtype=np.int32), bits)
        q = synth.normal_bf16(rng, (hq, d))
        scale = float(np.float32(1 / math.sqrt(d)))
        c, t = _oracle_reps(lambda: oracle.draft_attn(q, comp, scale, pool=pool), seconds)
        return entry(c / t, "tokens/s", "%d request-steps x 1 draft step (%d query heads over %d %s entries of "
                     "one request); %.1f s" % (c, hq, n, what, t))

    def verify_leg(pool, n_ctx, n_q, hq, hkv, d, rows, what):
        # one kv head's K / V (a row reads only its own head), rows of the
        # block's last query spread over that head's group
        k = synth.normal_bf16(rng, (n_ctx, 1, d))
        v = synth.normal_bf16(rng, (n_ctx, 1, d))
        grp = hq // hkv
        q = synth.normal_bf16(rng, (n_q, grp, d))
        qs = list(range(n_q - rows // grp, n_q)) if rows >= grp else [n_q - 1]
        scale = float(np.float32(1 / math.sqrt(d)))
        c, t = _oracle_reps(lambda: oracle.verify_attn(q, k, v, scale, queries=qs, pool=pool), seconds)
        nrows = c * len(qs) * grp
        return entry(nrows / t, "query-head rows/s", "%d rows (query x head) over %d keys each (%s); %.1f s"
                     % (nrows, n_ctx, what, t))

    out = {}
    with ThreadPoolExecutor(nt) as pool:
        w = dict(synth.WORKLOADS["70b_128k_drop4"])
        rng = synth.rng_for("70b_128k_drop4", 11)
        hq, hkv, d, nk, N, x = w["hq"], w["hkv"], w["d"], w["kept_total"], w["ctx"], w["x"]
        k = synth.normal_bf16(rng, (nk, hkv, d))
        v = synth.normal_bf16(rng, (nk, hkv, d))
        out["70b_draft"] = draft_leg(pool, k, v, 16, hq, "kept bf16")
        del k, v
        out["70b_verify"] = verify_leg(pool, N + x, x, hq, hkv, d, 32, "the 70B-shaped block's last queries")
        out["verify_40k"] = verify_leg(pool, 40960 + 40, 40, 32, hkv, d, 32, "the 40k point's last queries")
        w = dict(synth.WORKLOADS["mixed_32req_3bit"])
        rng = synth.rng_for("mixed_32req_3bit", 11)
        n_mean = (w["ctx_lo"] + w["ctx_hi"]) // 2
        k = synth.normal_bf16(rng, (n_mean, w["hkv"], w["d"]))
        v = synth.normal_bf16(rng, (n_mean, w["hkv"], w["d"]))
        out["mixed_draft"] = draft_leg(pool, k, v, w["bits"], w["hq"], "3-bit (the mean context)")
        del k, v
        vr = verify_leg(pool, n_mean + w["x"], w["x"], w["hq"], w["hkv"], w["d"], 32,
                        "the mean context, the block's last queries")
        vr.update(value=vr["value"] / w["hq"], unit="verified tokens/s (all query heads of a query)")
        out["mixed_verify"] = vr
        w = dict(synth.WORKLOADS[WORKLOAD])
        rng = synth.rng_for(WORKLOAD, 11)
        k = synth.normal_bf16(rng, (w["ctx"], w["hkv"], w["d"]))
        v = synth.normal_bf16(rng, (w["ctx"], w["hkv"], w["d"]))
        for bits in (3, 4):
            out["%d_bit" % bits] = draft_leg(pool, k, v, bits, w["hq"], "%d-bit" % bits)
    return out


def attach_oracle(extras, cpu):
    """Put each oracle sample beside the device number it matches."""
    big = extras["70b_128k_drop4"]
    big["draft"]["cpu_baseline"] = cpu["70b_draft"]
    c = big["config"]
    big["verify"]["rows_per_s"] = c["batch"] * c["x"] * c["q_heads"] / (big["verify"]["us_per_call"] * 1e-6)
    big["verify"]["cpu_baseline"] = cpu["70b_verify"]
    v40 = big["verify_40k"]
    c = v40["config"]
    v40["rows_per_s"] = c["batch"] * c["n_q"] * c["q_heads"] / (v40["us_per_call"] * 1e-6)
    v40["cpu_baseline"] = cpu["verify_40k"]
    extras["mixed_32req_3bit"]["cpu_baseline"] = {"draft_tokens_per_s": cpu["mixed_draft"],
                                                  "verify_tokens_per_s": cpu["mixed_verify"]}
    for bits in (3, 4):
        extras["draft_8b_32k_other_bits"]["%d_bit" % bits]["cpu_baseline"] = cpu["%d_bit" % bits]


def reference_main(args, rank, ws):
    if rank != 0:
        return
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    import synth
    w = dict(synth.WORKLOADS[WORKLOAD])
    N, d, hkv, hq = w["ctx"], w["d"], w["hkv"], w["hq"]
    rng = synth.rng_for(WORKLOAD, 7)
    k = synth.normal_bf16(rng, (N, hkv, d))
    v = synth.normal_bf16(rng, (N, hkv, d))
    q = synth.normal_bf16(rng, (hq, d))
    comp = oracle.compress(k, v, np.arange(N, dtype=np.int32), w["bits"])
    scale = float(np.float32(1 / math.sqrt(d)))
    with ThreadPoolExecutor(oracle.threads()) as pool:
        for _ in range(args.warmup):
            oracle.draft_attn(q, comp, scale, pool=pool)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle.draft_attn(q, comp, scale, pool=pool)
        dt = time.perf_counter() - t0
    val = args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": headline_config(w),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": "1 request x 1 draft step per step (32 query heads over 32768 2-bit "
                                       "KV_comp entries)"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="vc", choices=["vc", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads' device timings (70B-shaped layer, 40k verify, mixed launch)")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=[WORKLOAD, "mixed_32req_3bit", "toy_e2e", "staging", "70b_128k_drop4",
                             "stagger_32req_3bit", "remote_prefix_8req_3bit", "verify_40k"])
    ap.add_argument("--cycles", type=int, default=2, help="measured cycles of the staggering workload")
    args = ap.parse_args()
    rank, ws = dist_init()
    if args.impl == "reference":
        reference_main(args, rank, ws)
        return
    if args.workload != WORKLOAD:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        {"mixed_32req_3bit": mixed_main, "toy_e2e": toy_main, "staging": staging_main,
         "70b_128k_drop4": big_main, "stagger_32req_3bit": stagger_main,
         "remote_prefix_8req_3bit": remote_main, "verify_40k": verify40k_main}[args.workload](args)
        return
    import torch
    import synth
    import lossless_compressed_kv_gb300 as vc
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = dict(synth.WORKLOADS[WORKLOAD])
    st = build(w, 1234 + rank, device)
    rnd = Round(w, st, device)
    B, x, N = w["batch"], w["x"], w["ctx"]

    for _ in range(max(3, args.warmup)):
        rnd.run()
    torch.cuda.synchronize()
    assert rnd.status.item() == 0, "device status %d" % rnd.status.item()

    # the whole round as one CUDA graph: the host launches it once per step.
    # Two event-record nodes, before draft call x/4 and after call 3x/4 - 1,
    # time the middle half of the draft calls of the timed replays
    # themselves (the last replay's values are read after).  An event node
    # splits the graph's programmatic launch edge and costs a few us, so the
    # span carries only these two.
    span = (x // 4, (3 * x) // 4)
    try:
        span_ev = (torch.cuda.Event(enable_timing=True, external=True),
                   torch.cuda.Event(enable_timing=True, external=True))
        marks = {span[0]: (span_ev[0], None), span[1] - 1: (None, span_ev[1])}
    except TypeError:
        marks = None
    graph = capture(lambda: rnd.run(ev=marks))
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        start.record()
        for s in range(args.steps):
            graph.replay()
        stop.record()
        torch.cuda.synchronize()
    barrier(ws)
    assert rnd.status.item() == 0, "device status %d" % rnd.status.item()
    t_ms = allmax(start.elapsed_time(stop), ws)
    ms_step = t_ms / args.steps
    stages = rnd.breakdown()
    # algorithmic bytes of call i: N + i + 1 entries
    if marks is not None:
        draft_src = ("CUDA events before draft call %d and after call %d of 0..%d inside the timed graph "
                     "replays; per call = span / %d" % (span[0], span[1] - 1, x - 1, span[1] - span[0]))
        bytes_avg = float(np.mean([draft_bytes(w, N + i + 1) for i in range(*span)]))
        t_draft = span_ev[0].elapsed_time(span_ev[1]) * 1e-3 / (span[1] - span[0])
    else:
        draft_src = "CUDA events around replays of a graph of the round's draft calls"
        bytes_avg = float(np.mean([draft_bytes(w, N + i + 1) for i in range(x)]))
        t_draft = stages["draft_step"]["us_per_call"] * 1e-6
    peak, peak_kind = peaks()
    achieved = bytes_avg / t_draft / 1e9
    value = ws * B * x / (ms_step * 1e-3)

    e2e = None
    if not args.no_e2e:
        e2e = e2e_measure(w, st, rnd, args, ws, device)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_sample(w, st)
    extras = None
    if rank == 0 and not args.no_extras:
        # the other workloads of the path, timed on the device (CUDA events
        # around graph replays / launches), after the headline's timed region
        extras = {"70b_128k_drop4": big_measure(),
                  "mixed_32req_3bit": mixed_measure(args.steps, args.warmup, staging=False),
                  "draft_8b_32k_other_bits": bits_measure(w, device)}
        if not args.no_cpu_baseline:
            attach_oracle(extras, oracle_extras())
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "draft_attn_traffic.txt")) as f:
            tj = json.load(f)
        if tj.get("kernel_source_hash") == source_hash():
            traffic = tj["bytes_per_launch"]
    except Exception:
        pass
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f16 mma / fp32 accumulate on 2-bit codes", "data": "synthetic",
                "config": headline_config(w),
                "draft_attn": {"tokens_per_s": ws * B / t_draft, "us_per_call": t_draft * 1e6,
                               "bytes_per_call": bytes_avg, "timing": draft_src},
                "stages": stages,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                             "kernel": "draft_kernel<2,128> (incl. the step's append) + draft_reduce_kernel"},
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": rnd.launches * args.steps,
                "clocks": clk.summary(), "other_workloads": extras}
        print(json.dumps(line), flush=True)


def e2e_measure(w, st, rnd, args, ws, device):
    """Host-buffer round: pinned queries H2D, KV_full staged H2D on a side
    stream (overlapping the drafting), emitted tokens D2H."""
    import torch
    import lossless_compressed_kv_gb300 as vc
    full = st["full"]
    B, x = w["batch"], w["x"]
    hk = torch.empty(full.k_pages.shape, dtype=torch.uint8, pin_memory=True)
    hv = torch.empty(full.v_pages.shape, dtype=torch.uint8, pin_memory=True)
    hk.copy_(full.k_pages)
    hv.copy_(full.v_pages)
    hq = torch.empty(st["q"].shape, dtype=torch.bfloat16, pin_memory=True)
    hq.copy_(st["q"])
    hqv = torch.empty(st["qv"].shape, dtype=torch.bfloat16, pin_memory=True)
    hqv.copy_(st["qv"])
    hout = torch.empty((B, x + 1), dtype=torch.int32, pin_memory=True)
    hlen = torch.empty((B,), dtype=torch.int32, pin_memory=True)
    # two staging buffers: round i stages into buffer i % 2 while round i - 1
    # verifies from the other; a copy waits for the verify that last read its
    # buffer
    bufs = []
    for _ in range(2):
        sk, sv = torch.empty_like(full.k_pages), torch.empty_like(full.v_pages)
        bufs.append((sk, sv, vc.PagedKV(sk, sv, full.block_table, full.seq_lens, full.num_kv_heads,
                                        full.head_dim, 16)))
    # the step's queries, double-buffered like KV_full: copied on the staging
    # stream right after the previous round's KV_full.  Host->device copies
    # share one copy-engine queue, so a small copy on the compute stream would
    # wait behind a half-gigabyte staging copy and hold the drafting back; on
    # the staging stream it lands exactly when the drafting may start anyway.
    qbufs = [(torch.empty_like(st["q"]), torch.empty_like(st["qv"])) for _ in range(2)]
    side = torch.cuda.Stream(device=device)
    staged_ev = [torch.cuda.Event(), torch.cuda.Event()]
    verified_ev = [torch.cuda.Event(), torch.cuda.Event()]
    q_ev = [torch.cuda.Event(), torch.cuda.Event()]
    nbytes = hk.numel()
    it = [0]

    def step():
        i = it[0] % 2
        sk, sv, staged = bufs[i]
        qd, qvd = qbufs[i]
        if it[0] >= 2:
            side.wait_event(verified_ev[i])
        with torch.cuda.stream(side):
            qd.copy_(hq, non_blocking=True)
            qvd.copy_(hqv, non_blocking=True)
            q_ev[i].record(side)
        vc.stage_async(sk, hk, nbytes, side)
        vc.stage_async(sv, hv, nbytes, side, staged_ev[i])
        torch.cuda.current_stream().wait_event(q_ev[i])
        rnd.run(q=qd, qv=qvd, full=staged, verify_wait=staged_ev[i])
        verified_ev[i].record()
        hout.copy_(rnd.emit, non_blocking=True)
        hlen.copy_(rnd.alen, non_blocking=True)
        it[0] += 1

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    dt = allmax(time.perf_counter() - t0, ws)
    h2d = 2 * nbytes + hq.numel() * 2 + hqv.numel() * 2
    d2h = hout.numel() * 4 + hlen.numel() * 4
    staged_gbps = h2d * args.steps / dt / 1e9  # host -> device bytes over the loop's wall time
    return {"value": ws * B * x * args.steps / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "h2d_GBps": staged_gbps,
            "note": "KV_full (%.2f GB) staged from pinned host memory on a side stream each round "
                    "into one of two device buffers, overlapping the drafting; host -> device bytes "
                    "moved at %.0f GB/s over the loop" % (2 * nbytes / 1e9, staged_gbps)}


# ---------------------------------------------------------------------------
# other workloads (not the headline line): staggered mixed batch, toy loop,
# host -> device staging bandwidth
# ---------------------------------------------------------------------------

def _bf16_pools(vc, torch, g, device, b, n_tok, nkv, d):
    """Random bf16 KV_full of b requests x n_tok tokens, pages in a seeded
    permuted order."""
    npg = (n_tok + 15) // 16
    perm = torch.randperm(b * npg, generator=g, device=device).to(torch.int32)
    kp = torch.empty((b * npg, nkv, 16, d), dtype=torch.bfloat16, device=device)
    vp = torch.empty_like(kp)
    for s0 in range(0, b * npg, 1024):
        e = min(b * npg, s0 + 1024)
        kp[s0:e] = torch.randn((e - s0, nkv, 16, d), generator=g, device=device).to(torch.bfloat16)
        vp[s0:e] = torch.randn((e - s0, nkv, 16, d), generator=g, device=device).to(torch.bfloat16)
    return vc.PagedKV(kp.view(torch.uint8).view(b * npg, -1), vp.view(torch.uint8).view(b * npg, -1),
                      perm.view(b, npg).contiguous(), torch.full((b,), n_tok, dtype=torch.int32, device=device),
                      nkv, d, 16)


def _graph_us(torch, fn, reps):
    """Mean device time of fn over replays of a CUDA graph of it (us)."""
    gr = capture(fn)
    a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gr.replay()
    a.record()
    for _ in range(reps):
        gr.replay()
    b2.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b2) / reps * 1e3


def _verify_40k(vc, torch, g, device, d, hkv, peak, tpeak, reps):
    """The 40k-context verify point: batch 8, 32q/8kv, context 40960, a block
    of 40 queries (160 rows per kv head: one two-tile row block)."""
    B2, hq2, N2, x2 = 8, 32, 40960, 40
    L2 = N2 + x2
    scale = 1.0 / math.sqrt(d)
    full2 = _bf16_pools(vc, torch, g, device, B2, L2, hkv, d)
    qv2 = torch.randn((B2, x2, hq2, d), generator=g, device=device).to(torch.bfloat16)
    vout2 = torch.empty((B2, x2, hq2, d), dtype=torch.float32, device=device)
    vws2 = torch.empty(vc.verify_workspace_bytes(full2, x2, hq2, L2), dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    t_ver2 = _graph_us(torch, lambda: vc.verify_attn(qv2, full2, scale, vout2, L2, vws2, status=status), reps)
    torch.cuda.synchronize()
    assert status.item() == 0, "device status %d" % status.item()
    v2_bytes = B2 * L2 * hkv * 2 * d * 2
    v2_flops = 2 * 2 * B2 * x2 * hq2 * L2 * d
    return {"config": {"batch": B2, "q_heads": hq2, "kv_heads": hkv, "ctx": N2, "n_q": x2},
            "us_per_call": t_ver2, "GBps": v2_bytes / t_ver2 / 1e3,
            "frac_hbm_measured": v2_bytes / t_ver2 / 1e3 / peak, "TFLOPs": v2_flops / t_ver2 / 1e6,
            "frac_bf16_measured": v2_flops / t_ver2 / 1e6 / tpeak}


def verify40k_main(args):
    """Only the 40k-context verify point (for profiling it alone)."""
    import torch
    import lossless_compressed_kv_gb300 as vc
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    g = torch.Generator(device=device)
    g.manual_seed(78)
    peak, _ = peaks()
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        tpeak = float(json.load(f)["bf16_tflops"])
    r = _verify_40k(vc, torch, g, device, 128, 8, peak, tpeak, max(1, args.steps))
    print(json.dumps({"metric": "40k-context verify: 8 requests x 40 queries, 32q/8kv, D 128, bf16 KV_full",
                      "workload": "verify_40k", "verify_40k": r,
                      "timing": "CUDA events around replays of a CUDA graph of the call; flops count the causal "
                                "block as full"}), flush=True)


def big_main(args):
    """70B-shaped layer (batch 4, 64q/8kv, D 128, 131072-token context,
    32768 kept in bf16: 64 sink + 512 recent + top by a seeded score): the
    draft call over KV_comp and the 40-query verify over KV_full, plus the
    40k-context verify point (batch 8, 32q/8kv, context 40960, 40 queries).
    Each call is captured in a CUDA graph and timed over replays."""
    print(json.dumps(big_measure()), flush=True)


def big_measure():
    """The measurements of big_main as one JSON-ready dict."""
    import torch
    import synth
    import lossless_compressed_kv_gb300 as vc
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    w = dict(synth.WORKLOADS["70b_128k_drop4"])
    B, hq, hkv, d, N, x = w["batch"], w["hq"], w["hkv"], w["d"], w["ctx"], w["x"]
    g = torch.Generator(device=device)
    g.manual_seed(77)
    peak, _ = peaks()
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        tpeak = float(json.load(f)["bf16_tflops"])

    def pools(b, n_tok, nkv):
        return _bf16_pools(vc, torch, g, device, b, n_tok, nkv, d)

    def timed(fn, reps):
        return _graph_us(torch, fn, reps)

    scale = 1.0 / math.sqrt(d)
    L = N + x
    full = pools(B, L, hkv)
    # kept lists on the GPU (vc_select_kept) from the seeded scores; the
    # workload generator's lists are the same (tests/test_gpu_select.py)
    nk = w["kept_total"]
    scores = np.zeros((B, N), np.float32)
    for b in range(B):
        r = np.random.default_rng([w["seed"], 1, b])
        scores[b, w["sink"]:N - w["recent"]] = r.random(N - w["sink"] - w["recent"], dtype=np.float32)
    scores_d = torch.from_numpy(scores).to(device)
    offs_d = torch.arange(0, (B + 1) * nk, nk, dtype=torch.int32, device=device)
    idx_d = torch.empty(B * nk, dtype=torch.int32, device=device)
    sel_status = torch.zeros(1, dtype=torch.int32, device=device)
    t_sel = timed(lambda: vc.select_kept(full, offs_d, idx_d, w["sink"], w["recent"], scores=scores_d,
                                         status=sel_status), 10)
    sws = torch.empty(vc.select_workspace_bytes(B, N), dtype=torch.uint8, device=device)
    idx_kn = torch.empty(B * nk, dtype=torch.int32, device=device)
    t_sel_kn = timed(lambda: vc.select_kept(full, offs_d, idx_kn, w["sink"], w["recent"], score_stride=N,
                                            workspace=sws, status=sel_status), 5)
    torch.cuda.synchronize()
    assert sel_status.item() == 0
    offs, idx = offs_d.cpu().numpy(), idx_d.cpu().numpy()
    cpg = (nk + x + 15) // 16
    cperm = torch.randperm(B * cpg, generator=g, device=device).to(torch.int32)
    comp = vc.PagedKV.allocate(B * cpg, hkv, d, 16, cperm.view(B, cpg).contiguous(),
                               torch.full((B,), nk, dtype=torch.int32, device=device), device=device)
    vc.compress(full, torch.from_numpy(offs).to(device), torch.from_numpy(idx).to(device), comp, nk)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    q = torch.randn((B, hq, d), generator=g, device=device).to(torch.bfloat16)
    dout = torch.empty((B, hq, d), dtype=torch.float32, device=device)
    dws = torch.empty(vc.draft_workspace_bytes(comp, hq, nk), dtype=torch.uint8, device=device)
    t_draft = timed(lambda: vc.draft_attn(q, comp, scale, dout, nk, dws, status=status), 20)
    draft_bytes_ = B * nk * hkv * 2 * d * 2
    qv = torch.randn((B, x, hq, d), generator=g, device=device).to(torch.bfloat16)
    vout = torch.empty((B, x, hq, d), dtype=torch.float32, device=device)
    vws = torch.empty(vc.verify_workspace_bytes(full, x, hq, L), dtype=torch.uint8, device=device)
    t_ver = timed(lambda: vc.verify_attn(qv, full, scale, vout, L, vws, status=status), 10)
    ver_bytes = B * L * hkv * 2 * d * 2
    ver_flops = 2 * 2 * B * x * hq * L * d
    del full, comp, dws, vws
    torch.cuda.empty_cache()
    # the 40k-context verify point
    v40 = _verify_40k(vc, torch, g, device, d, hkv, peak, tpeak, 10)
    torch.cuda.synchronize()
    assert status.item() == 0, "device status %d" % status.item()
    return {
        "metric": "70B-shaped layer: draft over bf16 token-drop KV_comp and 40-query verify; 40k-context verify",
        "workload": "70b_128k_drop4",
        "config": {"batch": B, "q_heads": hq, "kv_heads": hkv, "head_dim": d, "ctx": N, "kept": nk, "x": x},
        "select_kept": {"us_seeded_scores": t_sel, "us_keynorm_scores": t_sel_kn,
                        "keynorm_GBps": B * N * hkv * d * 2 / t_sel_kn / 1e3,
                        "note": "4 x 131072 positions, 64 sink + 512 recent + top by score, 32768 kept per "
                                "request; key-norm path reads every K row"},
        "draft": {"us_per_call": t_draft, "bytes": draft_bytes_, "GBps": draft_bytes_ / t_draft / 1e3,
                  "frac_hbm_measured": draft_bytes_ / t_draft / 1e3 / peak,
                  "tokens_per_s": B / (t_draft * 1e-6)},
        "verify": {"us_per_call": t_ver, "bytes": ver_bytes, "GBps": ver_bytes / t_ver / 1e3,
                   "frac_hbm_measured": ver_bytes / t_ver / 1e3 / peak, "TFLOPs": ver_flops / t_ver / 1e6,
                   "frac_bf16_measured": ver_flops / t_ver / 1e6 / tpeak},
        "verify_40k": v40,
        "timing": "CUDA events around replays of a CUDA graph of the call; flops count the causal block as full",
    }


def staging_main(args):
    """Pinned host -> device copy bandwidth, one stream and four streams."""
    import torch
    import lossless_compressed_kv_gb300 as vc
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    res = {}
    for ns in (1, 2, 4):
        streams = [torch.cuda.Stream() for _ in range(ns)]
        part = n // ns
        for it in range(args.warmup + 1):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i, st in enumerate(streams):
                vc.stage_async(d[i * part:], h[i * part:], part, st)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
        res["streams_%d_GBps" % ns] = n / dt / 1e9
    print(json.dumps({"metric": "pinned host -> device staging GB/s", "bytes": n, **res}), flush=True)


def mixed_main(args):
    print(json.dumps(mixed_measure(args.steps, args.warmup, staging=True)), flush=True)


def mixed_measure(steps, warmup, staging):
    """Staggered mixed batch: 32 requests, contexts U[8192, 65536], 32q/8kv,
    D 128, 3-bit KV_comp; even requests draft, odd ones verify x = 25 in one
    launch, while the NEXT round's verifying requests' KV_full (odd requests
    of the other parity set) is staged from pinned host memory on a side
    stream.  Reports tokens/s of both halves, each half timed alone in the
    same launch (the other role's requests idle), the staging bandwidth and
    the overlap efficiency (t_mixed + t_stage) / t_wall."""
    import torch
    import synth
    import lossless_compressed_kv_gb300 as vc
    w = dict(synth.WORKLOADS["mixed_32req_3bit"])
    B, hq, hkv, d, x, bits = w["batch"], w["hq"], w["hkv"], w["d"], w["x"], w["bits"]
    rng = np.random.default_rng(w["seed"])
    lens = rng.integers(w["ctx_lo"], w["ctx_hi"] + 1, size=B).astype(np.int64)
    role = np.array([b % 2 for b in range(B)], np.int32)
    full_lens = lens + x                            # verifying requests hold the block too
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(w["seed"])
    npg = [(int(n) + 15) // 16 for n in full_lens]
    maxb = max(npg)
    table = torch.full((B, maxb), -1, dtype=torch.int32)
    o = 0
    for b in range(B):
        table[b, :npg[b]] = torch.arange(o, o + npg[b], dtype=torch.int32)
        o += npg[b]
    P = o
    pb = vc.page_bytes(hkv, d, 16)
    kp = torch.empty((P, pb // 2), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    for s0 in range(0, P, 4096):
        e = min(P, s0 + 4096)
        kp[s0:e] = torch.randn((e - s0, pb // 2), generator=g, device=dev).to(torch.bfloat16)
        vp[s0:e] = torch.randn((e - s0, pb // 2), generator=g, device=dev).to(torch.bfloat16)
    tdev = table.to(dev)
    full = vc.PagedKV(kp.view(torch.uint8), vp.view(torch.uint8), tdev,
                      torch.tensor(full_lens, dtype=torch.int32, device=dev), hkv, d, 16)
    comp = vc.PagedKV.allocate(P, hkv, d, bits, tdev, torch.tensor(lens, dtype=torch.int32, device=dev))
    kept = [np.arange(n, dtype=np.int32) for n in lens]
    offs, idx = synth.csr(kept)
    vc.compress(full, torch.from_numpy(offs).to(dev), torch.from_numpy(idx).to(dev), comp, int(lens.max()))
    qd = torch.randn((B, hq, d), generator=g, device=dev).to(torch.bfloat16)
    qv = torch.randn((B, x, hq, d), generator=g, device=dev).to(torch.bfloat16)
    od = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
    ov = torch.empty((B, x, hq, d), dtype=torch.float32, device=dev)
    msl = int(full_lens.max())
    wsb = torch.empty(vc.mixed_workspace_bytes(comp, full, x, hq, msl), dtype=torch.uint8, device=dev)
    roled = torch.from_numpy(role).to(dev)
    # staging: the verifying requests' KV_full for the next round, pinned host -> device
    ver_pages = sum(npg[b] for b in range(B) if role[b] == 1)
    stage_bytes = ver_pages * pb
    if staging:
        hk = torch.empty(stage_bytes, dtype=torch.uint8, pin_memory=True)
        hv = torch.empty(stage_bytes, dtype=torch.uint8, pin_memory=True)
        hk.fill_(0)
        hv.fill_(0)
        sk = torch.empty(stage_bytes, dtype=torch.uint8, device=dev)
        sv = torch.empty(stage_bytes, dtype=torch.uint8, device=dev)
        side = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def mixed():
        vc.mixed_attn(roled, qd, comp, od, qv, full, ov, 1.0 / math.sqrt(d), msl, wsb, status=status)

    def stage():
        vc.stage_async(sk, hk, stage_bytes, side)
        vc.stage_async(sv, hv, stage_bytes, side)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn, n):
        torch.cuda.synchronize()
        ev[0].record()
        for _ in range(n):
            fn()
        ev[1].record()
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / n

    for _ in range(max(3, warmup)):
        mixed()
    t_mixed = timed(mixed, max(steps, 3))
    # each half alone in the same launch (the other role's requests idle)
    halves = {}
    for name, keep in (("draft", 0), ("verify", 1)):
        rh = torch.from_numpy(np.where(role == keep, role, 2).astype(np.int32)).to(dev)
        halves[name] = timed(lambda: vc.mixed_attn(rh, qd, comp, od, qv, full, ov, 1.0 / math.sqrt(d), msl, wsb,
                                                   status=status), max(steps, 3))
    t_stage = t_wall = None
    if staging:
        t0 = time.perf_counter()
        for _ in range(steps):
            stage()
        torch.cuda.synchronize()
        t_stage = (time.perf_counter() - t0) * 1e3 / steps
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            stage()
            mixed()
        torch.cuda.synchronize()
        t_wall = (time.perf_counter() - t0) * 1e3 / steps
    assert status.item() == 0
    nd = int((role == 0).sum())
    nv = int((role == 1).sum())
    comp_bytes = sum(int(lens[b]) for b in range(B) if role[b] == 0) * hkv * 2 * (d * bits // 8 + 4 * d // 32)
    full_bytes = sum(int(full_lens[b]) for b in range(B) if role[b] == 1) * hkv * 2 * d * 2
    flops = sum(2 * 2 * x * hq * int(full_lens[b]) * d for b in range(B) if role[b] == 1)
    line = {"metric": "staggered mixed batch: draft + verify attention in one launch", "workload": "mixed_32req_3bit",
            "config": {"batch": B, "ctx": "U[%d,%d]" % (w["ctx_lo"], w["ctx_hi"]), "q_heads": hq, "kv_heads": hkv,
                       "head_dim": d, "bits": bits, "x": x, "drafting": nd, "verifying": nv},
            "ms_mixed_launch": t_mixed, "ms_stage": t_stage, "ms_wall_stage_and_mixed": t_wall,
            "overlap_efficiency": (t_mixed + t_stage) / t_wall if staging else None,
            "draft_tokens_per_s": nd / (t_mixed * 1e-3), "verify_tokens_per_s": nv * x / (t_mixed * 1e-3),
            "algorithmic_GBps": (comp_bytes + full_bytes) / (t_mixed * 1e-3) / 1e9,
            "ms_draft_half_alone": halves["draft"], "draft_half_GBps": comp_bytes / (halves["draft"] * 1e-3) / 1e9,
            "ms_verify_half_alone": halves["verify"],
            "verify_half_GBps": full_bytes / (halves["verify"] * 1e-3) / 1e9,
            "verify_tflops": flops / (t_mixed * 1e-3) / 1e12,
            "stage_GBps": 2 * stage_bytes / (t_stage * 1e-3) / 1e9 if staging else None,
            "stage_bytes": 2 * stage_bytes,
            "timing": "CUDA events around %d mixed launches" % max(steps, 3)}
    return line


def stagger_main(args):
    """Staggering scheduler on the 32-request, 2-layer workload: lock step
    (every request drafts x tokens, then all verify; one staging buffer for
    all of KV_full) against the balanced staggered plan (two staging slots),
    both at x = 25, and the staggered plan at the scheduler's smallest
    stall-free horizon.  Each run: one warm-up cycle, then `--cycles`
    measured cycles.  The scheduler's cost model is calibrated from timed
    all-draft / all-verify / idle ticks and the measured link rate; its
    predictions are printed beside the measurements."""
    import torch
    import synth
    import lossless_compressed_kv_gb300 as vc
    from lossless_compressed_kv_gb300.stagger import phase_schedule
    w = dict(synth.WORKLOADS["stagger_32req_3bit"])
    dev = torch.device("cuda")
    t0 = time.perf_counter()
    from synth.rigs import stagger_rig
    eng, qd, qv = stagger_rig(w, dev)
    t_build = time.perf_counter() - t0
    B, L, x, mx = w["batch"], w["layers"], w["x"], w["max_x"]
    cycles = max(1, args.cycles)

    def qvx(n):
        return [q[:, :n].contiguous() for q in qv]

    # cost model: ms per tick (all layers) with fixed roles
    it = 5
    t_idle = eng.time_roles(np.full(B, 2), x, it, qd, qvx(x))
    t_draft = eng.time_roles(np.zeros(B), x, it, qd, qvx(x))
    fulls = eng.device_full(x)
    t_verify = eng.time_roles(np.ones(B), x, it, qd, qvx(x), fulls)
    del fulls
    torch.cuda.empty_cache()
    cb = eng.comp_bytes().astype(np.float64)
    fb = eng.pages(x).astype(np.float64)
    d_ns = (t_draft - t_idle) * 1e6 * cb / cb.sum()
    v_ns = (t_verify - t_idle) * 1e6 * fb / fb.sum()
    tick_ns = t_idle * 1e6
    sb = eng.stage_bytes(x)
    P = x + 1

    def one(phase, n_phases, xx, slots):
        roles = phase_schedule(phase, n_phases, cycles + 1)
        r = eng.run(roles, xx, slots, qd, qvx(xx), measure_from=n_phases)
        r["cycle_ms"] = r["wall_ms"] / cycles
        r["draft_tokens_per_s"] = r["draft_tokens"] / (r["wall_ms"] * 1e-3)
        r["stall_ms_per_cycle"] = r["stall_ms"] / cycles
        r["stage_ms_per_cycle"] = r["stage_ms"] / cycles
        return r

    lock = one(np.full(B, P - 1, np.int32), P, x, 1)
    bw = lock["link_GBps"]                                       # bytes per ns
    pred = lambda ph, n_ph, slots, s=sb: vc.stagger_simulate(  # noqa: E731
        ph, n_ph, s, d_ns, v_ns, bw, n_slots=slots, n_layers=L, tick_ns=tick_ns)
    lock["predicted"] = pred(np.full(B, P - 1, np.int32), P, 1)
    ph, phb = vc.stagger_plan(sb, P)
    stag = one(ph, P, x, 2)
    stag["predicted"] = pred(ph, P, 2)
    stag["max_phase_requests"] = int(np.bincount(ph, minlength=P).max())
    sbm = eng.stage_bytes(mx)
    xh, phh, predh = vc.stagger_horizon(sbm, d_ns, v_ns, bw, 1, mx, n_slots=2, n_layers=L, tick_ns=tick_ns)
    hor = one(phh, xh + 1, xh, 2)
    hor["predicted"] = pred(phh, xh + 1, 2, eng.stage_bytes(xh))
    hor["x"] = xh
    # the guide's per-token swap cost T_swap / L for the mean request at x
    t_swap_ms = float(sb.mean()) / (bw * 1e6)
    keep = ("cycle_ms", "stall_ms_per_cycle", "stage_ms_per_cycle", "overlap", "link_GBps", "max_tick_ms",
            "mean_tick_ms", "draft_tokens_per_s", "peak_stage_bytes", "launches")
    pk = ("cycle_ns", "stall_ns", "stage_ns", "overlap", "peak_stage_bytes")

    def pick(r):
        out = {k: r[k] for k in keep}
        out["predicted"] = {k: r["predicted"][k] for k in pk}
        for k in ("x", "max_phase_requests"):
            if k in r:
                out[k] = r[k]
        return out

    line = {"metric": "staggered verification across requests, layers and rounds: cycle time, staging stall "
                      "and overlap (lock step vs balanced stagger vs scheduler horizon)",
            "workload": "stagger_32req_3bit",
            "config": {"batch": B, "ctx": "U[%d,%d]" % (w["ctx_lo"], w["ctx_hi"]), "layers": L, "q_heads": w["hq"],
                       "kv_heads": w["hkv"], "head_dim": w["d"], "bits": w["bits"], "x": x, "cycles": cycles,
                       "kv_full_host_GB": float(eng.stage_bytes(mx).sum()) / 1e9},
            "cost_model_ms": {"idle_tick": t_idle, "all_draft_tick": t_draft, "all_verify_tick": t_verify,
                              "link_GBps": bw},
            "t_swap_mean_request_ms": t_swap_ms, "t_swap_per_drafted_token_ms": t_swap_ms / x,
            "lock_step": pick(lock), "staggered": pick(stag), "staggered_at_horizon": pick(hor),
            "build_s": t_build}
    print(json.dumps(line), flush=True)


def remote_main(args):
    """Remote prefix caching: time to the first drafted token and to the
    first verified block when only KV_comp crosses the slow link (KV_full on
    a fast link), against one-token decoding after KV_full crossed the slow
    link; the same number of tokens (every draft accepted) for both."""
    import torch
    import synth
    w = dict(synth.WORKLOADS["remote_prefix_8req_3bit"])
    dev = torch.device("cuda")
    from synth.rigs import remote_rig
    eng, qd, qv, q1, ones = remote_rig(w, dev)
    rate, chunk = w["slow_GBps"], int(w["chunk_MB"]) << 20
    # warm-up (module loading, first launches) on an unthrottled link
    eng.run_vericache(qd, qv, 1, 1000.0, chunk)
    eng.run_full_kv_remote(q1, ones, 2, 1000.0, chunk)
    vr = eng.run_vericache(qd, qv, w["rounds"], rate, chunk)
    steps = w["rounds"] * (w["x"] + 1)
    br = eng.run_full_kv_remote(q1, ones, steps, rate, chunk)
    line = {"metric": "remote prefix caching: startup and time to N tokens, KV_comp over a slow link vs KV_full "
                      "over it", "workload": "remote_prefix_8req_3bit",
            "config": {k: w[k] for k in ("batch", "hq", "hkv", "d", "ctx", "layers", "bits", "x", "rounds",
                                         "slow_GBps", "chunk_MB")},
            "slow_link_bytes": {"vericache_kv_comp": vr["slow_bytes"], "baseline_kv_full": vr["fast_bytes"]},
            "compression_ratio": vr["fast_bytes"] / vr["slow_bytes"],
            "vericache": vr, "full_kv_remote": br,
            "startup_speedup": br["first_token_ms"] / vr["first_draft_ms"],
            "time_to_tokens_speedup": br["total_ms"] / vr["total_ms"],
            "note": "attention work of the schedule only; token counts assume every draft accepted; both links "
                    "share this machine's host->device path"}
    print(json.dumps(line), flush=True)


def toy_main(args):
    """End-to-end toy loop (batch 4, 16384-token prompt, 512 tokens, x = 32,
    4-bit KV_comp): wall time of the VeriCache rounds and of full-KV greedy
    decoding from the same prefilled state, identical outputs checked."""
    import torch
    import synth
    from lossless_compressed_kv_gb300 import toy
    w = dict(synth.WORKLOADS["toy_e2e"])
    t0 = time.perf_counter()
    r = toy.run(w, timed=True)
    line = {"metric": "toy decoder greedy tokens/s: VeriCache rounds vs full-KV decoding", "workload": "toy_e2e",
            "config": {k: w[k] for k in ("batch", "layers", "d_model", "hq", "hkv", "d", "ffn", "vocab", "prompt",
                                         "bits", "x", "gen")},
            "identical_outputs": bool(np.array_equal(r["vericache"].numpy(), r["full"].numpy())),
            "rounds": r["stats"]["rounds"], "mean_accepted_per_round": r["stats"]["mean_accepted"],
            "vericache_tokens_per_s": w["batch"] * w["gen"] / r["stats"]["t_vericache"],
            "full_kv_tokens_per_s": w["batch"] * w["gen"] / r["stats"]["t_full"],
            "note": "host loop in Python driving the C ABI; KV_full resident in HBM; wall %.1f s" %
                    (time.perf_counter() - t0)}
    print(json.dumps(line), flush=True)


def source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("draft_attn.cu", "draft_impl.cuh", "vc_internal.cuh", "quant_row.cuh", "comp_layout.cuh"):
        with open(os.path.join(ROOT, "lossless_compressed_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
