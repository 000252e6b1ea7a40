"""Remote prefix caching emulated on one GPU.

"VeriCache: Making Lossy KV Compression Exact", the two serving settings
(remote prefix caching), and study notes "VeriCache: Turning Lossy KV Cache
into Lossless LLM Inference", case 3: a store holds the precomputed KV of
long prefixes; the serving GPU receives only the compressed cache over the
slow link and starts drafting from it, while the full cache reaches the
verifier over a fast link.  Decoding can start about a compression ratio
sooner than if the full cache had to cross the slow link first.

One machine plays both sides.  The slow link is a paced copy
(vc_stage_paced_async) of KV_comp from page-locked host memory; the fast link
is a plain staging copy (vc_stage_async) of KV_full on a second stream.  The
compute stream drafts (vc_draft_attn, every layer per drafted token) as soon
as each layer's KV_comp has landed, and verifies each block of x drafts
(vc_verify_attn, every layer) once that layer's KV_full is there.  The
baseline sends KV_full over the slow link and decodes one token at a time over
it (vc_verify_attn with a one-query block).  This is the attention work of the
schedule only: the drafted tokens are not produced by a model, so the token
counts assume every draft accepted (x + 1 tokens per round).
"""
from __future__ import annotations

import torch

from . import (draft_attn, draft_workspace_bytes, link_clock, stage_async, stage_paced_async,
               verify_attn, verify_workspace_bytes)


class RemotePrefixEngine:
    """comp: per layer a PagedKV of KV_comp on the device (the destination of
    the slow link; seq_lens = prefix lengths); full: per layer a PagedKV of
    bf16 KV_full on the device (the destination of the fast link; seq_lens =
    prefix + x); comp_host / full_host: per layer (K, V) page-locked uint8
    tensors with the bytes of the matching device pools (the store)."""

    def __init__(self, comp, full, comp_host, full_host, num_q_heads: int, max_seq_len: int):
        self.L = len(comp)
        if not (self.L == len(full) == len(comp_host) == len(full_host)) or self.L == 0:
            raise ValueError("one KV_comp and one KV_full per layer")
        for pair, dev in zip(list(comp_host) + list(full_host), list(comp) + list(full)):
            for h, d in zip(pair, (dev.k_pages, dev.v_pages)):
                if not h.is_pinned() or h.numel() != d.numel():
                    raise ValueError("host store must be page-locked and match the device pools")
        self.comp, self.full = comp, full
        self.comp_host, self.full_host = comp_host, full_host
        self.hq = num_q_heads
        self.max_len = max_seq_len
        self.dev = comp[0].k_pages.device
        self.compute = torch.cuda.Stream(self.dev)
        self.slow = torch.cuda.Stream(self.dev)
        self.fast = torch.cuda.Stream(self.dev)
        self.origin = torch.zeros(1, dtype=torch.int64, device=self.dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)

    def bytes(self, which):
        pools = self.comp if which == "comp" else self.full
        return sum(p.k_pages.numel() + p.v_pages.numel() for p in pools)

    @staticmethod
    def _poison(pools):
        """0xFF over the destinations (NaN bit patterns in bf16 and fp16), so
        that a layer read before it has landed shows in the outputs."""
        for p in pools:
            p.k_pages.fill_(255)
            p.v_pages.fill_(255)

    def _send(self, pools, host, stream, paced, rate, chunk):
        """Copies of every layer's K and V on `stream`; returns per-layer
        events."""
        ready = []
        off = 0
        with torch.cuda.stream(stream):
            for l in range(self.L):
                for dst, src in ((pools[l].k_pages, host[l][0]), (pools[l].v_pages, host[l][1])):
                    n = src.numel()
                    if paced:
                        stage_paced_async(dst, src, n, chunk, rate, self.origin, off, stream)
                    else:
                        stage_async(dst, src, n, stream)
                    off += n
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                ready.append(e)
        return ready

    def _start(self):
        """Time origin: the link clock, then an event all streams wait for."""
        torch.cuda.synchronize(self.dev)
        t0 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.slow):
            link_clock(self.origin, self.slow)
            t0.record(self.slow)
        for s in (self.fast, self.compute):
            s.wait_event(t0)
        return t0

    def run_vericache(self, q_draft, q_verify, rounds: int, slow_bytes_per_ns: float, chunk_bytes: int,
                      poison: bool = True, outputs=None) -> dict:
        """q_draft: per layer bf16 [B][Hq][D]; q_verify: per layer bf16
        [B][x][Hq][D].  Times (ms) from the link origin."""
        x = q_verify[0].shape[1]
        B = q_draft[0].shape[0]
        od = torch.empty((B, self.hq, q_draft[0].shape[2]), dtype=torch.float32, device=self.dev)
        ov = torch.empty((B, x, self.hq, q_draft[0].shape[2]), dtype=torch.float32, device=self.dev)
        dws = torch.empty(draft_workspace_bytes(self.comp[0], self.hq, self.max_len), dtype=torch.uint8,
                          device=self.dev)
        vws = torch.empty(verify_workspace_bytes(self.full[0], x, self.hq, self.max_len), dtype=torch.uint8,
                          device=self.dev)
        scale = 1.0 / float(q_draft[0].shape[2]) ** 0.5
        step_end, round_end = [], []
        self.status.zero_()
        if poison:
            self._poison(self.comp)
            self._poison(self.full)
        t0 = self._start()
        comp_ready = self._send(self.comp, self.comp_host, self.slow, True, slow_bytes_per_ns, chunk_bytes)
        full_ready = self._send(self.full, self.full_host, self.fast, False, 0.0, 0)
        with torch.cuda.stream(self.compute):
            for r in range(rounds):
                for i in range(x):
                    for l in range(self.L):
                        if r == 0 and i == 0:
                            self.compute.wait_event(comp_ready[l])
                        draft_attn(q_draft[l], self.comp[l], scale, od, self.max_len, dws, status=self.status,
                                   stream=self.compute)
                    e = torch.cuda.Event(enable_timing=True)
                    e.record(self.compute)
                    step_end.append(e)
                for l in range(self.L):
                    if r == 0:
                        self.compute.wait_event(full_ready[l])
                    verify_attn(q_verify[l], self.full[l], scale, ov, self.max_len, vws, status=self.status,
                                stream=self.compute)
                e = torch.cuda.Event(enable_timing=True)
                e.record(self.compute)
                round_end.append(e)
            if outputs is not None:
                outputs.append((od.clone(), ov.clone()))
        torch.cuda.synchronize(self.dev)
        if int(self.status.item()) != 0:
            raise RuntimeError("device status %d" % int(self.status.item()))
        ms = lambda e: t0.elapsed_time(e)  # noqa: E731
        return {"first_draft_ms": ms(step_end[0]), "first_verified_ms": ms(round_end[0]),
                "total_ms": ms(round_end[-1]), "comp_arrived_ms": ms(comp_ready[-1]),
                "full_arrived_ms": ms(full_ready[-1]), "rounds": rounds, "x": x,
                "tokens_if_all_accepted": rounds * (x + 1) * B,
                "round_ms": (round_end[0].elapsed_time(round_end[-1]) / (rounds - 1)) if rounds > 1 else None,
                "slow_bytes": self.bytes("comp"), "fast_bytes": self.bytes("full")}

    def run_full_kv_remote(self, q_one, full_one, steps: int, slow_bytes_per_ns: float, chunk_bytes: int,
                           poison: bool = True, outputs=None) -> dict:
        """Baseline: KV_full over the slow link, then one-token decoding over
        it.  q_one: per layer bf16 [B][1][Hq][D]; full_one: per layer PagedKV
        over the same pools as the engine's KV_full, seq_lens = prefix + 1."""
        B = q_one[0].shape[0]
        ov = torch.empty((B, 1, self.hq, q_one[0].shape[3]), dtype=torch.float32, device=self.dev)
        vws = torch.empty(verify_workspace_bytes(full_one[0], 1, self.hq, self.max_len), dtype=torch.uint8,
                          device=self.dev)
        scale = 1.0 / float(q_one[0].shape[3]) ** 0.5
        step_end = []
        self.status.zero_()
        if poison:
            self._poison(full_one)
        t0 = self._start()
        full_ready = self._send(full_one, self.full_host, self.slow, True, slow_bytes_per_ns, chunk_bytes)
        with torch.cuda.stream(self.compute):
            for i in range(steps):
                for l in range(self.L):
                    if i == 0:
                        self.compute.wait_event(full_ready[l])
                    verify_attn(q_one[l], full_one[l], scale, ov, self.max_len, vws, status=self.status,
                                stream=self.compute)
                e = torch.cuda.Event(enable_timing=True)
                e.record(self.compute)
                step_end.append(e)
            if outputs is not None:
                outputs.append(ov.clone())
        torch.cuda.synchronize(self.dev)
        if int(self.status.item()) != 0:
            raise RuntimeError("device status %d" % int(self.status.item()))
        ms = lambda e: t0.elapsed_time(e)  # noqa: E731
        return {"first_token_ms": ms(step_end[0]), "total_ms": ms(step_end[-1]), "steps": steps,
                "tokens": steps * B, "full_arrived_ms": ms(full_ready[-1]),
                "step_ms": (step_end[0].elapsed_time(step_end[-1]) / (steps - 1)) if steps > 1 else None}
