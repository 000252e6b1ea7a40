"""Seeded synthetic rigs for the staggering and remote-prefix workloads:
paged KV_full / KV_comp of every layer (drawn with torch's seeded device
generator, N(0,1) bf16), their bytes in page-locked host memory where the
workload stages them, per-layer queries, and the engine of the package that
runs the workload.  Used by the benchmark and the GPU tests alike; holds
none of the method's arithmetic (compression runs in the library)."""
from __future__ import annotations

import numpy as np


def stagger_rig(w, device):
    """The staggering workload: per layer, KV_full of every request (bf16,
    N(0,1), room for blocks of up to max_x tokens, a request's pages
    contiguous) in page-locked host memory and KV_comp of its context (every
    token, w["bits"]) resident on the device; per-layer queries.  Returns
    (engine, q_draft per layer [B][Hq][D], q_verify per layer [B][max_x][Hq][D])."""
    import torch
    import synth
    import lossless_compressed_kv_gb300 as vc
    from lossless_compressed_kv_gb300.stagger import StaggerEngine
    B, hq, hkv, d, bits, L, mx = w["batch"], w["hq"], w["hkv"], w["d"], w["bits"], w["layers"], w["max_x"]
    rng = np.random.default_rng(w["seed"])
    ctx = rng.integers(w["ctx_lo"], w["ctx_hi"] + 1, size=B).astype(np.int64)
    npg = (ctx + mx + 15) // 16
    first = np.concatenate([[0], np.cumsum(npg)[:-1]]).astype(np.int64)
    P = int(npg.sum())
    pb = vc.page_bytes(hkv, d, 16)
    tab = np.full((B, int(npg.max())), -1, np.int32)
    for b in range(B):
        tab[b, :npg[b]] = np.arange(first[b], first[b] + npg[b], dtype=np.int32)
    cpg = (ctx + 15) // 16
    ctab = np.full((B, int(cpg.max())), -1, np.int32)
    c0 = np.concatenate([[0], np.cumsum(cpg)[:-1]])
    for b in range(B):
        ctab[b, :cpg[b]] = np.arange(c0[b], c0[b] + cpg[b], dtype=np.int32)
    tabd, ctabd = torch.from_numpy(tab).to(device), torch.from_numpy(ctab).to(device)
    lens_full = torch.from_numpy((ctx + mx).astype(np.int32)).to(device)
    lens_comp = torch.from_numpy(ctx.astype(np.int32)).to(device)
    offs, idx = synth.csr([np.arange(n, dtype=np.int32) for n in ctx])
    offs, idx = torch.from_numpy(offs).to(device), torch.from_numpy(idx).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(w["seed"])
    comps, hk, hv = [], [], []
    for _ in range(L):
        kp = torch.empty((P, pb // 2), dtype=torch.bfloat16, device=device)
        vp = torch.empty_like(kp)
        for s0 in range(0, P, 4096):
            e = min(P, s0 + 4096)
            kp[s0:e] = torch.randn((e - s0, pb // 2), generator=g, device=device).to(torch.bfloat16)
            vp[s0:e] = torch.randn((e - s0, pb // 2), generator=g, device=device).to(torch.bfloat16)
        full = vc.PagedKV(kp.view(torch.uint8), vp.view(torch.uint8), tabd, lens_full, hkv, d, 16)
        comp = vc.PagedKV.allocate(int(cpg.sum()), hkv, d, bits, ctabd, lens_comp, device=device)
        vc.compress(full, offs, idx, comp, int(ctx.max()))
        comps.append(comp)
        for src, dst in ((kp, hk), (vp, hv)):
            h = torch.empty((P, pb), dtype=torch.uint8, pin_memory=True)
            h.copy_(src.view(torch.uint8))
            dst.append(h)
        del kp, vp, full
    torch.cuda.synchronize()
    qd = [torch.randn((B, hq, d), generator=g, device=device).to(torch.bfloat16) for _ in range(L)]
    qv = [torch.randn((B, mx, hq, d), generator=g, device=device).to(torch.bfloat16) for _ in range(L)]
    eng = StaggerEngine(comps, hk, hv, first, ctx, hkv, d, hq, mx, device=device)
    return eng, qd, qv


def remote_rig(w, device):
    """Remote prefix caching workload: per layer bf16 KV_full (prefix + x
    tokens, N(0,1)) and its KV_comp (every prefix token, w["bits"]) on the
    device, and their bytes in page-locked host memory (the store).  Returns
    (engine, q_draft, q_verify [B][x], q_one [B][1], KV_full views with
    seq_lens = prefix + 1 for the one-token baseline), all per layer."""
    import torch
    import synth
    import lossless_compressed_kv_gb300 as vc
    from lossless_compressed_kv_gb300.remote import RemotePrefixEngine
    B, hq, hkv, d, bits, L, n, x = (w["batch"], w["hq"], w["hkv"], w["d"], w["bits"], w["layers"], w["ctx"],
                                    w["x"])
    npg, cpg = (n + x + 15) // 16, (n + 15) // 16
    pb = vc.page_bytes(hkv, d, 16)
    tabd = torch.arange(B * npg, dtype=torch.int32, device=device).view(B, npg).contiguous()
    ctabd = torch.arange(B * cpg, dtype=torch.int32, device=device).view(B, cpg).contiguous()
    full_lens = torch.full((B,), n + x, dtype=torch.int32, device=device)
    one_lens = torch.full((B,), n + 1, dtype=torch.int32, device=device)
    comp_lens = torch.full((B,), n, dtype=torch.int32, device=device)
    offs, idx = synth.csr([np.arange(n, dtype=np.int32)] * B)
    offs, idx = torch.from_numpy(offs).to(device), torch.from_numpy(idx).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(w["seed"])
    fulls, comps, ones, fh, ch = [], [], [], [], []

    def pinned(t):
        h = torch.empty(t.numel(), dtype=torch.uint8, pin_memory=True)
        h.copy_(t.view(-1))
        return h

    for _ in range(L):
        kp = torch.empty((B * npg, pb // 2), dtype=torch.bfloat16, device=device)
        vp = torch.empty_like(kp)
        for s0 in range(0, B * npg, 4096):
            e = min(B * npg, s0 + 4096)
            kp[s0:e] = torch.randn((e - s0, pb // 2), generator=g, device=device).to(torch.bfloat16)
            vp[s0:e] = torch.randn((e - s0, pb // 2), generator=g, device=device).to(torch.bfloat16)
        full = vc.PagedKV(kp.view(torch.uint8), vp.view(torch.uint8), tabd, full_lens, hkv, d, 16)
        comp = vc.PagedKV.allocate(B * cpg, hkv, d, bits, ctabd, comp_lens, device=device)
        vc.compress(full, offs, idx, comp, n)
        torch.cuda.synchronize()
        fulls.append(full)
        comps.append(comp)
        ones.append(vc.PagedKV(full.k_pages, full.v_pages, tabd, one_lens, hkv, d, 16))
        fh.append((pinned(full.k_pages), pinned(full.v_pages)))
        ch.append((pinned(comp.k_pages), pinned(comp.v_pages)))
    qd = [torch.randn((B, hq, d), generator=g, device=device).to(torch.bfloat16) for _ in range(L)]
    qv = [torch.randn((B, x, hq, d), generator=g, device=device).to(torch.bfloat16) for _ in range(L)]
    q1 = [torch.randn((B, 1, hq, d), generator=g, device=device).to(torch.bfloat16) for _ in range(L)]
    eng = RemotePrefixEngine(comps, fulls, ch, fh, hq, n + x)
    return eng, qd, qv, q1, ones
