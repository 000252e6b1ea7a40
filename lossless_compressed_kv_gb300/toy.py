"""End-to-end VeriCache greedy loop on a small random-init decoder.

"VeriCache: Making Lossy KV Compression Exact", section "The Core Idea":
draft x tokens with the compressed cache, verify the block (pending token +
x drafts) in one pass over the full cache, emit the longest matching prefix
plus the verifier's correction or bonus token; the output must equal greedy
decoding with the full cache.  The study notes add the commit step: resume
from the last accepted token.

Model (random weights, exactness is relative to the same model): d_model
layers of pre-RMSNorm attention (GQA, rotary embedding, theta 500000) and a
SwiGLU MLP, bf16 weights and bf16 activations between layers, fp32 LM head.
Every computation runs in libvc through the C ABI; this module only
allocates buffers and sequences the calls (the host loop of the method).

Commit rule: after a round with a accepted drafts the full cache keeps the
verifier's K/V of the pending token and the a accepted drafts (positions P ..
P + a); the compressed cache is rolled back to its length before the round
and re-filled with those a + 1 entries compressed from the full cache; the
emitted correction / bonus token becomes the next pending token.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

import lossless_compressed_kv_gb300 as vc

ROPE_THETA = 500000.0
EPS = 1e-5


def _dev_bf16(a: np.ndarray, device):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def _graph(fn):
    """CUDA graph of the work `fn` enqueues (run once on a side stream first,
    which is also the first execution of that work)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@dataclass
class ToyShape:
    layers: int
    d_model: int
    hq: int
    hkv: int
    d: int
    ffn: int
    vocab: int
    bits: int
    x: int


class ToyDecoder:
    def __init__(self, shape: ToyShape, weights: dict, device="cuda"):
        self.s, self.dev = shape, device
        self.embed_t = torch.from_numpy(weights["embed"]).to(device)
        self.lm_head = torch.from_numpy(weights["lm_head"]).to(device)
        self.final_norm = torch.from_numpy(weights["final_norm"]).to(device)
        self.layers = []
        for lw in weights["layers"]:
            self.layers.append({
                "attn_norm": torch.from_numpy(lw["attn_norm"]).to(device),
                "mlp_norm": torch.from_numpy(lw["mlp_norm"]).to(device),
                "wqkv": _dev_bf16(lw["wqkv"], device), "wo": _dev_bf16(lw["wo"], device),
                "wgu": _dev_bf16(lw["wgu"], device), "wd": _dev_bf16(lw["wd"], device)})
        self.scale = 1.0 / math.sqrt(shape.d)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self._bufs = {}

    # -- buffers ----------------------------------------------------------
    def _buf(self, name, shape, dtype=torch.float32):
        key = (name, tuple(shape), dtype)
        t = self._bufs.get(key)
        if t is None:
            t = torch.empty(shape, dtype=dtype, device=self.dev)
            self._bufs[key] = t
        return t

    def new_full(self, batch: int, capacity: int):
        """Per layer a bf16 paged cache; request b owns pages [b*np, (b+1)*np)."""
        npg = (capacity + 15) // 16
        table = torch.arange(batch * npg, dtype=torch.int32, device=self.dev).view(batch, npg)
        lens = torch.zeros(batch, dtype=torch.int32, device=self.dev)
        return [vc.PagedKV.allocate(batch * npg, self.s.hkv, self.s.d, 16, table, lens, device=self.dev)
                for _ in range(self.s.layers)]

    def new_comp(self, batch: int, capacity: int):
        npg = (capacity + 15) // 16
        table = torch.arange(batch * npg, dtype=torch.int32, device=self.dev).view(batch, npg)
        lens = torch.zeros(batch, dtype=torch.int32, device=self.dev)
        return [vc.PagedKV.allocate(batch * npg, self.s.hkv, self.s.d, self.s.bits, table, lens, device=self.dev)
                for _ in range(self.s.layers)]

    @staticmethod
    def view(kv: vc.PagedKV, lens: torch.Tensor, b0: int = 0, b1=None):
        bt = kv.block_table if (b0 == 0 and b1 is None) else kv.block_table[b0:b1]
        return vc.PagedKV(kv.k_pages, kv.v_pages, bt, lens, kv.num_kv_heads, kv.head_dim, kv.bits)

    # -- one forward pass over m rows -------------------------------------
    def forward(self, ids, row_req, row_pos, full, attn):
        """ids/row_req/row_pos: device int32 [m], rows grouped by request.
        attn(layer, q bf16 [m][hq][d], o fp32 [m][hq*d]) fills o.
        Returns the final-norm hidden states fp32 [m][d_model]."""
        s, m = self.s, int(ids.numel())
        x = self._buf("x", (m, s.d_model))
        h = self._buf("h", (m, s.d_model))
        qkv = self._buf("qkv", (m, (s.hq + 2 * s.hkv) * s.d))
        q = self._buf("q", (m, s.hq, s.d), torch.bfloat16)
        o = self._buf("o", (m, s.hq * s.d))
        gu = self._buf("gu", (m, 2 * s.ffn))
        act = self._buf("act", (m, s.ffn))
        vc.embed(ids, self.embed_t, x, status=self.status)
        for li, L in enumerate(self.layers):
            vc.rmsnorm(x, L["attn_norm"], h, EPS)
            vc.linear(h, L["wqkv"], qkv)
            vc.rope_kv_write(qkv, row_req, row_pos, s.hq, ROPE_THETA, q, full[li], status=self.status)
            attn(li, q, o)
            vc.linear(o, L["wo"], x, accumulate=True)
            vc.rmsnorm(x, L["mlp_norm"], h, EPS)
            vc.linear(h, L["wgu"], gu)
            vc.swiglu(gu, act)
            vc.linear(act, L["wd"], x, accumulate=True)
        out = self._buf("hidden", (m, s.d_model))
        vc.rmsnorm(x, self.final_norm, out, EPS)
        return out

    def argmax(self, hidden, batch: int, n_pred: int, drafts=None):
        """LM-head argmax (and, with drafts, the accept rule) of [batch][n_pred] rows."""
        x = 0 if drafts is None else int(drafts.shape[1])
        ver = self._buf("ver", (batch, n_pred), torch.int32)
        al = self._buf("al", (batch,), torch.int32)
        em = self._buf("em", (batch, x + 1), torch.int32)
        ws = self._buf("aws", (vc.accept_workspace_bytes(batch, n_pred, self.s.vocab, self.s.d_model),), torch.uint8)
        dr = drafts if drafts is not None else self._buf("nodraft", (batch, 0), torch.int32)
        vc.accept(hidden.view(batch, n_pred, 1, -1), self.lm_head, dr, ver, al, em, ws)
        return ver, al, em

    # -- prefill ------------------------------------------------------------
    def prefill(self, prompt: torch.Tensor, full, chunk: int = 64):
        """prompt int32 [B][P] on the device.  Writes K/V of every prompt
        position into `full` (all layers) and returns the first generated
        token per request (int32 [B])."""
        s = self.s
        B, P = int(prompt.shape[0]), int(prompt.shape[1])
        m = B * P
        ids = prompt.reshape(-1).contiguous()
        row_req = torch.arange(B, dtype=torch.int32, device=self.dev).repeat_interleave(P)
        row_pos = torch.arange(P, dtype=torch.int32, device=self.dev).repeat(B)
        n_chunks = (P + chunk - 1) // chunk
        ends = [min(P, (c + 1) * chunk) for c in range(n_chunks)]
        lens_c = [torch.full((1,), e, dtype=torch.int32, device=self.dev) for e in ends]
        vws = self._buf("pre_vws", (vc.verify_workspace_bytes(self.view(full[0], lens_c[0], 0, 1), chunk, s.hq, P),),
                        torch.uint8)
        vout = self._buf("pre_vout", (1, chunk, s.hq, s.d))

        def attn(li, q, o):
            for b in range(B):
                for c in range(n_chunks):
                    r0, n = b * P + c * chunk, ends[c] - c * chunk
                    kv = self.view(full[li], lens_c[c], b, b + 1)
                    out = o[r0:r0 + n].view(1, n, s.hq, s.d)
                    vc.verify_attn(q[r0:r0 + n].view(1, n, s.hq, s.d), kv, self.scale, out, ends[c], vws,
                                   status=self.status)

        hidden = self.forward(ids, row_req, row_pos, full, attn)
        last = hidden.view(B, P, -1)[:, P - 1].contiguous()
        for kv in full:
            kv.seq_lens.fill_(P)
        ver, _, _ = self.argmax(last, B, 1)
        return ver[:, 0].clone()

    # -- full-KV greedy decoding (the reference) ---------------------------
    def greedy_full(self, first: torch.Tensor, full, start: int, n_tokens: int):
        """One token per step with the full cache; every step is the same
        CUDA graph (positions advanced on the device), replayed."""
        s, B = self.s, int(first.numel())
        outs = torch.empty((B, n_tokens), dtype=torch.int32, device=self.dev)
        outs[:, 0] = first
        tok = self._buf("g_tok", (B,), torch.int32)
        tok.copy_(first)
        row_req = torch.arange(B, dtype=torch.int32, device=self.dev)
        row_pos = self._buf("g_pos", (B,), torch.int32)
        row_pos.fill_(start)
        lens = self._buf("g_lens", (B,), torch.int32)
        ws = self._buf("g_vws", (vc.verify_workspace_bytes(full[0], 1, s.hq, start + n_tokens + 1),), torch.uint8)

        def attn(li, q, o):
            vc.verify_attn(q.view(B, 1, s.hq, s.d), self.view(full[li], lens), self.scale,
                           o.view(B, 1, s.hq, s.d), start + n_tokens + 1, ws, status=self.status)

        def step():
            torch.add(row_pos, 1, out=lens)
            hidden = self.forward(tok, row_req, row_pos, full, attn)
            ver, _, _ = self.argmax(hidden, B, 1)
            tok.copy_(ver[:, 0])
            row_pos.add_(1)

        if n_tokens > 1:
            g = _graph(step)  # the first step runs while the graph is captured
            outs[:, 1] = tok
            for i in range(2, n_tokens):
                g.replay()
                outs[:, i] = tok
        return outs  # [B][n_tokens]

    # -- VeriCache rounds ----------------------------------------------------
    def vericache(self, first: torch.Tensor, full, comp, start: int, n_tokens: int, stats=None):
        """Draft x tokens per round on KV_comp, verify x + 1 on KV_full,
        accept, commit.  KV_comp must already hold the compressed prompt.
        The x draft steps of a round are one CUDA graph and the verification
        pass another, both replayed every round with the round's positions
        in device buffers; the host reads the accepted lengths once per
        round and commits."""
        s, B, x = self.s, int(first.numel()), self.s.x
        dev = self.dev
        P = [start] * B                 # position of the pending token
        Cn = [start] * B                # KV_comp length
        pending = first.cpu().tolist()
        gen = [[t] for t in pending]
        cap = start + n_tokens + 2 * x + 2     # a finished request re-drafts from a frozen position
        capl = torch.full((B,), cap, dtype=torch.int32, device=dev)   # positions compress may read
        dws = self._buf("d_ws", (vc.draft_workspace_bytes(comp[0], s.hq, cap),), torch.uint8)
        vws = self._buf("v_ws", (vc.verify_workspace_bytes(full[0], x + 1, s.hq, cap),), torch.uint8)
        row_req1 = torch.arange(B, dtype=torch.int32, device=dev)
        row_reqv = torch.arange(B, dtype=torch.int32, device=dev).repeat_interleave(x + 1)
        offs1 = torch.arange(B + 1, dtype=torch.int32, device=dev)
        jv = torch.arange(x + 1, dtype=torch.int32, device=dev)
        # the round's inputs (set before the graphs run)
        p_dev = self._buf("r_p", (B,), torch.int32)          # P
        c_dev = self._buf("r_c", (B,), torch.int32)          # Cn
        pend = self._buf("r_pend", (B,), torch.int32)        # pending tokens
        # buffers the graphs use
        tok = self._buf("r_tok", (B,), torch.int32)
        drafts = self._buf("r_drafts", (B, x), torch.int32)
        row_pos = self._buf("r_pos", (B,), torch.int32)
        clens = self._buf("r_clens", (B,), torch.int32)
        cstart = self._buf("r_cstart", (B,), torch.int32)
        ids = self._buf("r_ids", (B, x + 1), torch.int32)
        vpos = self._buf("r_vpos", (B, x + 1), torch.int32)
        flens = self._buf("r_flens", (B,), torch.int32)
        res = {}

        def draft_round():
            tok.copy_(pend)
            for i in range(x):
                torch.add(p_dev, i, out=row_pos)
                torch.add(c_dev, i + 1, out=clens)
                torch.add(c_dev, i, out=cstart)

                def attn(li, q, o):
                    # the token's K/V was just written into KV_full at P + i:
                    # compress it into KV_comp's next slot, then attend
                    vc.compress(self.view(full[li], capl), offs1, row_pos, comp[li], 1, comp_start=cstart,
                                status=self.status)
                    vc.draft_attn(q, self.view(comp[li], clens), self.scale, o.view(B, s.hq, s.d), cap, dws,
                                  status=self.status)

                hidden = self.forward(tok, row_req1, row_pos, full, attn)
                ver, _, _ = self.argmax(hidden, B, 1)
                drafts[:, i] = ver[:, 0]
                tok.copy_(ver[:, 0])

        def vattn(li, q, o):
            vc.verify_attn(q.view(B, x + 1, s.hq, s.d), self.view(full[li], flens), self.scale,
                           o.view(B, x + 1, s.hq, s.d), cap, vws, status=self.status)

        def verify_round():
            # verify the block [pending, d_0 .. d_{x-1}] with the full cache
            ids[:, 0] = pend
            ids[:, 1:] = drafts
            torch.add(p_dev[:, None], jv[None, :], out=vpos)
            torch.add(p_dev, x + 1, out=flens)
            hidden = self.forward(ids.view(-1), row_reqv, vpos.view(-1), full, vattn)
            res["ver"], res["al"], res["em"] = self.argmax(hidden, B, x + 1, drafts)

        g_draft = g_verify = None
        rounds = accepted = 0
        while min(len(g) for g in gen) < n_tokens:
            p_dev.copy_(torch.tensor(P, dtype=torch.int32))
            c_dev.copy_(torch.tensor(Cn, dtype=torch.int32))
            pend.copy_(torch.tensor(pending, dtype=torch.int32))
            if g_draft is None:
                g_draft = _graph(draft_round)  # the first round runs while the graphs are captured
                g_verify = _graph(verify_round)
            else:
                g_draft.replay()
                g_verify.replay()
            al_h, em_h = res["al"].cpu().tolist(), res["em"].cpu().tolist()
            # ---- commit: KV_full keeps P..P+a, KV_comp re-filled from it ----
            done = [len(gen[b]) >= n_tokens for b in range(B)]
            kept = [list(range(P[b], P[b] + (0 if done[b] else al_h[b]) + 1)) for b in range(B)]
            offs = torch.tensor(np.cumsum([0] + [len(k) for k in kept]), dtype=torch.int32, device=dev)
            idx = torch.tensor([i for k in kept for i in k], dtype=torch.int32, device=dev)
            cst = torch.tensor(Cn, dtype=torch.int32, device=dev)
            for li in range(s.layers):
                vc.compress(self.view(full[li], capl), offs, idx, comp[li], max(len(k) for k in kept),
                            comp_start=cst, status=self.status)
            for b in range(B):
                if len(gen[b]) >= n_tokens:   # finished: keep its state frozen
                    continue
                a = al_h[b]
                emitted = [t for t in em_h[b] if t >= 0]
                gen[b].extend(emitted)
                P[b] += a + 1
                Cn[b] += a + 1
                pending[b] = emitted[-1]
                accepted += a
            rounds += 1
        if stats is not None:
            stats.update(rounds=rounds, mean_accepted=accepted / max(1, rounds * B))
        return torch.tensor([g[:n_tokens] for g in gen], dtype=torch.int32)


def run(w: dict, device="cuda", prompt=None, n_gen=None, batch=None, seed=None, timed=False):
    """Prefill, then decode n_gen tokens per request twice from the same
    state: with VeriCache rounds and with plain full-KV greedy decoding.
    Returns dict(vericache ids, full-KV ids, stats, first tokens)."""
    import synth
    s = ToyShape(w["layers"], w["d_model"], w["hq"], w["hkv"], w["d"], w["ffn"], w["vocab"], w["bits"], w["x"])
    rng = np.random.default_rng([w["seed"] if seed is None else seed, 0])
    weights = synth.toy_weights(rng, w)
    B = w["batch"] if batch is None else batch
    P = w["prompt"] if prompt is None else prompt
    G = w["gen"] if n_gen is None else n_gen
    ids = synth.token_ids(rng, (B, P), w["vocab"])
    model = ToyDecoder(s, weights, device)
    cap = P + G + 2 * s.x + 2
    full_a = model.new_full(B, cap)
    first = model.prefill(torch.from_numpy(ids).to(device), full_a)
    full_b = [vc.PagedKV(f.k_pages.clone(), f.v_pages.clone(), f.block_table, f.seq_lens.clone(), f.num_kv_heads,
                         f.head_dim, f.bits) for f in full_a]
    comp = model.new_comp(B, cap)
    offs = torch.arange(0, B * P + 1, P, dtype=torch.int32, device=device)
    idx = torch.arange(P, dtype=torch.int32, device=device).repeat(B)
    lensP = torch.full((B,), P, dtype=torch.int32, device=device)
    for li in range(s.layers):
        vc.compress(model.view(full_a[li], lensP), offs, idx, comp[li], P, status=model.status)
    stats = {}
    import time
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ids_vc = model.vericache(first, full_a, comp, P, G, stats)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    ids_ref = model.greedy_full(first, full_b, P, G).cpu()
    torch.cuda.synchronize()
    stats["t_vericache"], stats["t_full"] = t1 - t0, time.perf_counter() - t1
    stats["status"] = int(model.status.item())
    return dict(vericache=ids_vc, full=ids_ref, stats=stats, prompt=ids, weights=weights, first=first.cpu())
