"""Cross-resource staggering across requests, layers and rounds on one GPU.

"VeriCache: Making Lossy KV Compression Exact", "Verifying Without Giving
Back the Speedup" and Figure 2: requests do not all draft and then all verify;
while some verify against their full cache, the others keep drafting from the
compressed one.  Study notes "VeriCache: Turning Lossy KV Cache into Lossless
LLM Inference", case 2: KV_comp stays in HBM, KV_full lives in host memory
and is brought in only for verification, and who verifies is staggered so
that few full caches are on the link at once.  "VeriCache Guide": the
dual-stream engine (full KV reloaded on a swap stream while drafting goes on)
and "Best Practice 2" (page-locked host memory).

The engine runs an explicit schedule: one role per request per tick (0 draft
one token, 1 verify, 2 idle).  A tick runs every layer as one vc_mixed_attn
launch on the compute stream (drafting requests over that layer's KV_comp,
verifying requests over their staged KV_full).  The verifying requests of a
tick form one staging job: a side stream copies their KV_full, layer by layer,
from page-locked host memory into a ring of staging slots (vc_stage_async),
as far ahead as free slots allow; layer l of the tick waits only for layer l
of its job, and the slot is handed back after the tick's last layer.  Events
recorded on the compute stream before and after each wait measure the stall;
events on the side stream measure each job's link time.

Phase plans for the schedule and the model that predicts its stall come from
the library's scheduler (vc_stagger_plan / vc_stagger_simulate /
vc_stagger_horizon).  This module only issues library calls and CUDA stream /
event operations; all arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import PagedKV, mixed_attn, mixed_workspace_bytes, page_bytes, stage_async

DRAFT, VERIFY, IDLE = 0, 1, 2


def phase_schedule(phase, n_phases: int, n_cycles: int) -> np.ndarray:
    """Roles [n_cycles * n_phases][n] of a phase plan: request r verifies at
    the ticks t with t mod n_phases == phase[r] and drafts at the others."""
    phase = np.asarray(phase, np.int32)
    t = np.arange(n_cycles * n_phases)[:, None]
    return np.where(t % n_phases == phase[None, :], VERIFY, DRAFT).astype(np.int32)


class StaggerEngine:
    """KV_comp resident per layer, KV_full per layer in page-locked host memory.

    comp: one PagedKV per layer (the same batch, block table and lengths for
      every layer; seq_lens = context lengths);
    host_k / host_v: one page-locked uint8 tensor [pages, page_bytes] per
      layer holding the bf16 KV_full pages;
    first_page: int [n] -- request r's pages are host pages
      first_page[r] .. first_page[r] + ceil((ctx[r] + x) / 16) - 1 of every layer
      (room for the largest block length max_x is the caller's);
    ctx: int [n] context lengths (a verifying request's KV_full holds ctx + x
      tokens, the last x being the drafted block)."""

    def __init__(self, comp, host_k, host_v, first_page, ctx, num_kv_heads: int, head_dim: int, num_q_heads: int,
                 max_x: int, device=None):
        self.L = len(comp)
        if not (self.L == len(host_k) == len(host_v)) or self.L == 0:
            raise ValueError("one KV_comp and one host KV_full pair per layer")
        for t in list(host_k) + list(host_v):
            if not t.is_pinned():
                raise ValueError("KV_full must be in page-locked host memory")
        self.comp = comp
        self.host_k, self.host_v = host_k, host_v
        self.first = np.asarray(first_page, np.int64)
        self.ctx = np.asarray(ctx, np.int64)
        self.n = len(self.ctx)
        self.hkv, self.d, self.hq, self.max_x = num_kv_heads, head_dim, num_q_heads, max_x
        self.pb = page_bytes(num_kv_heads, head_dim, 16)
        if host_k[0].shape[1] != self.pb:
            raise ValueError("host page size does not match the format")
        self.dev = torch.device("cuda") if device is None else device
        self.compute = torch.cuda.Stream(self.dev)
        self.side = torch.cuda.Stream(self.dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.max_len = int(self.ctx.max()) + max_x
        self.max_blocks = (self.max_len + 15) // 16

    # -- sizes ---------------------------------------------------------------
    def pages(self, x: int) -> np.ndarray:
        return (self.ctx + x + 15) // 16

    def stage_bytes(self, x: int) -> np.ndarray:
        """KV_full bytes (K and V, every layer) staged for one verification."""
        return self.pages(x) * self.pb * 2 * self.L

    def comp_bytes(self) -> np.ndarray:
        """KV_comp bytes read by one draft step of each request (all layers)."""
        hb = self.comp[0].k_pages.shape[1] // self.hkv     # one head block
        return ((self.ctx + 15) // 16) * hb * self.hkv * 2 * self.L

    # -- one run -------------------------------------------------------------
    def run(self, roles, x: int, n_slots: int, q_draft, q_verify, measure_from: int = 0, snapshot=None) -> dict:
        """Execute the schedule `roles` [T][n] with drafted blocks of x tokens.

        q_draft: per layer bf16 [n][Hq][D]; q_verify: per layer bf16
        [n][x][Hq][D].  measure_from: first tick of the measured window.
        snapshot(t, l, out_draft, out_verify): optional, called after layer l
        of tick t is enqueued on the compute stream (for checks; it must
        enqueue its work on that stream, the current one while it runs).
        Returns measured times (ms) over the window."""
        roles = np.asarray(roles, np.int32)
        T = roles.shape[0]
        if roles.shape[1] != self.n or not (1 <= x <= self.max_x) or n_slots < 1:
            raise ValueError("bad schedule, block length or slot count")
        L, dev, pb = self.L, self.dev, self.pb
        npg = self.pages(x)
        # staging jobs: the verifying requests of each tick that has any
        job_tick, job_reqs = [], []
        for t in range(T):
            rs = np.nonzero(roles[t] == VERIFY)[0]
            if len(rs):
                job_tick.append(t)
                job_reqs.append(rs)
        tick_job = {t: i for i, t in enumerate(job_tick)}
        slot_pages = max([int(npg[rs].sum()) for rs in job_reqs], default=1)
        # slot layout: [layer][pages of the job's requests, in request order]
        slot_k = [torch.empty((L * slot_pages, pb), dtype=torch.uint8, device=dev) for _ in range(n_slots)]
        slot_v = [torch.empty((L * slot_pages, pb), dtype=torch.uint8, device=dev) for _ in range(n_slots)]
        # per job: block table into the slot's layer region, roles
        tables, role_dev = [], [None] * T
        role_cache = {}
        for t in range(T):
            key = roles[t].tobytes()
            if key not in role_cache:
                role_cache[key] = torch.from_numpy(roles[t].copy()).to(dev)
            role_dev[t] = role_cache[key]
        for rs in job_reqs:
            tab = np.full((self.n, self.max_blocks), -1, np.int32)
            off = 0
            for r in rs:
                tab[r, :npg[r]] = np.arange(off, off + npg[r], dtype=np.int32)
                off += int(npg[r])
            tables.append(torch.from_numpy(tab).to(dev))
        full_lens = torch.from_numpy((self.ctx + x).astype(np.int32)).to(dev)
        od = torch.empty((self.n, self.hq, self.d), dtype=torch.float32, device=dev)
        ov = torch.empty((self.n, x, self.hq, self.d), dtype=torch.float32, device=dev)
        probe = PagedKV(slot_k[0][:slot_pages], slot_v[0][:slot_pages], tables[0] if tables else
                        torch.full((self.n, self.max_blocks), -1, dtype=torch.int32, device=dev), full_lens,
                        self.hkv, self.d, 16)
        ws = torch.empty(max(1, mixed_workspace_bytes(self.comp[0], probe, x, self.hq, self.max_len)),
                         dtype=torch.uint8, device=dev)
        scale = 1.0 / float(np.sqrt(self.d))

        ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        staged = [[torch.cuda.Event() for _ in range(L)] for _ in range(n_slots)]
        free = [torch.cuda.Event() for _ in range(n_slots)]
        j_start = [ev() for _ in job_tick]
        j_end = [ev() for _ in job_tick]
        stall_ev = {}
        t_ev = [ev() for _ in range(T + 1)]

        def enqueue_job(i):
            s = i % n_slots
            with torch.cuda.stream(self.side):
                if i >= n_slots:
                    self.side.wait_event(free[s])       # recorded after job i - n_slots' tick
                j_start[i].record(self.side)
                for l in range(L):
                    off = l * slot_pages
                    for r in job_reqs[i]:
                        a, c = int(self.first[r]), int(npg[r])
                        stage_async(slot_k[s][off:off + c], self.host_k[l][a:a + c], c * pb, self.side)
                        stage_async(slot_v[s][off:off + c], self.host_v[l][a:a + c], c * pb, self.side)
                        off += c
                    staged[s][l].record(self.side)
                j_end[i].record(self.side)

        self.status.zero_()
        torch.cuda.current_stream(dev).synchronize()   # slots, tables and roles are ready
        for i in range(min(n_slots, len(job_tick))):
            enqueue_job(i)
        with torch.cuda.stream(self.compute):
            for t in range(T):
                t_ev[t].record(self.compute)
                i = tick_job.get(t)
                s = None if i is None else i % n_slots
                for l in range(L):
                    if i is not None:
                        a_ev, b_ev = ev(), ev()
                        a_ev.record(self.compute)
                        self.compute.wait_event(staged[s][l])
                        b_ev.record(self.compute)
                        stall_ev[(t, l)] = (a_ev, b_ev)
                        full = PagedKV(slot_k[s][l * slot_pages:(l + 1) * slot_pages],
                                       slot_v[s][l * slot_pages:(l + 1) * slot_pages], tables[i], full_lens,
                                       self.hkv, self.d, 16)
                    else:
                        full = probe
                    mixed_attn(role_dev[t], q_draft[l], self.comp[l], od, q_verify[l], full, ov, scale,
                               self.max_len, ws, status=self.status, stream=self.compute)
                    if snapshot is not None:
                        snapshot(t, l, od, ov)
                if i is not None:
                    free[s].record(self.compute)
                if i is not None and i + n_slots < len(job_tick):
                    enqueue_job(i + n_slots)
            t_ev[T].record(self.compute)
        torch.cuda.synchronize(dev)
        if int(self.status.item()) != 0:
            raise RuntimeError("device status %d during the staggered run" % int(self.status.item()))

        m0 = measure_from
        wall = t_ev[m0].elapsed_time(t_ev[T])
        stall = sum(a.elapsed_time(b) for (t, _), (a, b) in stall_ev.items() if t >= m0)
        stage = sum(j_start[i].elapsed_time(j_end[i]) for i, t in enumerate(job_tick) if t >= m0)
        staged_bytes = sum(int(npg[job_reqs[i]].sum()) * pb * 2 * L for i, t in enumerate(job_tick) if t >= m0)
        ticks = [t_ev[t].elapsed_time(t_ev[t + 1]) for t in range(m0, T)]
        win = roles[m0:]
        return {
            "ticks": T - m0, "wall_ms": wall, "stall_ms": stall, "stage_ms": stage,
            "overlap": 1.0 - stall / stage if stage > 0 else 1.0,
            "link_GBps": staged_bytes / (stage * 1e-3) / 1e9 if stage > 0 else None,
            "max_tick_ms": max(ticks) if ticks else 0.0, "mean_tick_ms": float(np.mean(ticks)) if ticks else 0.0,
            "draft_tokens": int((win == DRAFT).sum()), "verify_tokens": int((win == VERIFY).sum()) * x,
            "staged_bytes": staged_bytes, "peak_stage_bytes": n_slots * slot_pages * pb * 2 * L,
            "launches": (T - m0) * L * 2,
        }

    def device_full(self, x: int):
        """Every request's KV_full (ctx + x tokens) copied to the device, one
        PagedKV per layer (for calibration and checks)."""
        npg = self.pages(x)
        tab = np.full((self.n, self.max_blocks), -1, np.int32)
        off = 0
        for r in range(self.n):
            tab[r, :npg[r]] = np.arange(off, off + npg[r], dtype=np.int32)
            off += int(npg[r])
        tabd = torch.from_numpy(tab).to(self.dev)
        lens = torch.from_numpy((self.ctx + x).astype(np.int32)).to(self.dev)
        out = []
        for l in range(self.L):
            k = torch.empty((off, self.pb), dtype=torch.uint8, device=self.dev)
            v = torch.empty_like(k)
            o = 0
            for r in range(self.n):
                a, c = int(self.first[r]), int(npg[r])
                k[o:o + c].copy_(self.host_k[l][a:a + c])
                v[o:o + c].copy_(self.host_v[l][a:a + c])
                o += c
            out.append(PagedKV(k, v, tabd, lens, self.hkv, self.d, 16))
        return out

    def time_roles(self, role, x: int, n_iter: int, q_draft, q_verify, full_layers=None) -> float:
        """Mean ms of one tick (every layer) with fixed roles: calibrates the
        scheduler's cost model.  full_layers: per layer a PagedKV of KV_full
        for the verifying requests (device resident)."""
        dev = self.dev
        roled = torch.from_numpy(np.asarray(role, np.int32).copy()).to(dev)
        full_lens = torch.from_numpy((self.ctx + x).astype(np.int32)).to(dev)
        if full_layers is None:
            dummy = torch.empty((1, self.pb), dtype=torch.uint8, device=dev)
            tab = torch.full((self.n, self.max_blocks), -1, dtype=torch.int32, device=dev)
            full_layers = [PagedKV(dummy, dummy, tab, full_lens, self.hkv, self.d, 16)] * self.L
        od = torch.empty((self.n, self.hq, self.d), dtype=torch.float32, device=dev)
        ov = torch.empty((self.n, x, self.hq, self.d), dtype=torch.float32, device=dev)
        ws = torch.empty(max(1, mixed_workspace_bytes(self.comp[0], full_layers[0], x, self.hq, self.max_len)),
                         dtype=torch.uint8, device=dev)
        scale = 1.0 / float(np.sqrt(self.d))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.compute):
            for it in range(n_iter + 2):
                if it == 2:
                    a.record(self.compute)
                for l in range(self.L):
                    mixed_attn(roled, q_draft[l], self.comp[l], od, q_verify[l], full_layers[l], ov, scale,
                               self.max_len, ws, status=self.status, stream=self.compute)
            b.record(self.compute)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / n_iter
