"""Test-side helpers: build paged caches from the seeded generators, move
them to the GPU, and read GPU page pools back into the oracle's logical
layout (byte offsets from the page format in include/vc.h).  Holds none of
the method's arithmetic."""
from __future__ import annotations

import numpy as np
import torch

import synth

PAGE = synth.PAGE
GROUP = 32


def hb(d: int, bits: int) -> int:
    return PAGE * d * 2 if bits == 16 else 2 * d * (bits + 1)


def to_dev(a: np.ndarray, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def full_cache(rng, lens, hkv, d, outliers=(), oscale=1.0, capacity=None, spare_pages=0):
    """Random bf16 KV_full in pages.  Returns (PagedKV on the GPU, dict of
    numpy pools / table / lens for the oracle side)."""
    import lossless_compressed_kv_gb300 as vc
    lens = np.asarray(lens, dtype=np.int32)
    table, total = synth.block_tables(rng, lens, capacity)
    total += spare_pages
    k, v = synth.kv_pools(rng, total, hkv, d, outliers, oscale)
    kd = to_dev(k.view(np.uint8).reshape(total, -1))
    vd = to_dev(v.view(np.uint8).reshape(total, -1))
    full = vc.PagedKV(kd, vd, to_dev(table), to_dev(lens), hkv, d, 16)
    return full, dict(k=k, v=v, table=table, lens=lens)


def logical_full(h: dict, b: int, n=None):
    n = int(h["lens"][b]) if n is None else n
    return (synth.logical_from_pages(h["k"], h["table"][b], n),
            synth.logical_from_pages(h["v"], h["table"][b], n))


def comp_cache(rng, batch, capacity, hkv, d, bits, zero=False):
    """Empty KV_comp pools with a random block table covering `capacity`
    slots per request (seq_lens set by the caller)."""
    import lossless_compressed_kv_gb300 as vc
    cap = np.broadcast_to(np.asarray(capacity), (batch,)).astype(np.int64)
    table, total = synth.block_tables(rng, cap)
    lens = torch.zeros(batch, dtype=torch.int32, device="cuda")
    comp = vc.PagedKV.allocate(total, hkv, d, bits, to_dev(table), lens, zero=zero)
    return comp, table


def read_comp(pool: torch.Tensor, table_row: np.ndarray, n: int, hkv: int, d: int, bits: int) -> dict:
    """GPU comp pool -> oracle.compress-style logical dict for one request."""
    p = pool.cpu().numpy()
    B = hb(d, bits)
    npg = (n + PAGE - 1) // PAGE
    blk = p.reshape(p.shape[0], hkv, B)[table_row[:npg]]          # [npg][hkv][B]
    if bits == 16:
        x = blk.view(np.uint16).reshape(npg, hkv, PAGE, d).transpose(0, 2, 1, 3).reshape(npg * PAGE, hkv, d)
        return dict(bits=16, x16=x[:n])
    cb, ng = d * bits // 8, d // GROUP
    codes = blk[:, :, :PAGE * cb].reshape(npg, hkv, PAGE, cb).transpose(0, 2, 1, 3).reshape(npg * PAGE, hkv, cb)
    sc = blk[:, :, PAGE * cb:PAGE * cb + PAGE * ng * 2].copy().view(np.uint16).reshape(npg, hkv, PAGE, ng)
    ze = blk[:, :, PAGE * cb + PAGE * ng * 2:].copy().view(np.uint16).reshape(npg, hkv, PAGE, ng)
    sc = sc.transpose(0, 2, 1, 3).reshape(npg * PAGE, hkv, ng)
    ze = ze.transpose(0, 2, 1, 3).reshape(npg * PAGE, hkv, ng)
    return dict(bits=bits, packed=codes[:n], scales=sc[:n], zeros=ze[:n])


def read_comp_kv(comp, table: np.ndarray, b: int, n: int) -> dict:
    """Both K and V of request b in the layout of oracle.compress."""
    kk = read_comp(comp.k_pages, table[b], n, comp.num_kv_heads, comp.head_dim, comp.bits)
    vv = read_comp(comp.v_pages, table[b], n, comp.num_kv_heads, comp.head_dim, comp.bits)
    if comp.bits == 16:
        return dict(bits=16, k16=kk["x16"], v16=vv["x16"])
    return dict(bits=comp.bits, k_packed=kk["packed"], k_scales=kk["scales"], k_zeros=kk["zeros"],
                v_packed=vv["packed"], v_scales=vv["scales"], v_zeros=vv["zeros"])


def row_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max_i |got - ref| / ||ref||_2 (rows = last axis)."""
    g = got.reshape(-1, got.shape[-1]).astype(np.float64)
    r = ref.reshape(-1, ref.shape[-1]).astype(np.float64)
    nrm = np.linalg.norm(r, axis=1)
    nrm = np.where(nrm == 0, 1.0, nrm)
    return float((np.abs(g - r).max(axis=1) / nrm).max())


TOL = 2e-3  # attention: max abs error <= 2e-3 * ||o_ref||_2 per output row
