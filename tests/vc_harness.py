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


# Code placement inside a quantised head block (the page format in
# include/vc.h): bit offset of each (token, channel) code, per plane.
def k_bit(bits: int, d: int, s, c, plane: int = 0):
    s, c = np.asarray(s), np.asarray(c)
    ks, t, e = c >> 4, (c >> 2) & 3, c & 3
    r, half = 2 * ks + (e >> 1), e & 1
    if bits == 2:
        return s * 2 * d + t * (d // 2) + 32 * (r >> 3) + 16 * half + 2 * (r & 7)
    if bits == 4:
        return s * 4 * d + t * d + 32 * (r >> 2) + 16 * half + 4 * (r & 3)
    if plane == 0:
        return s * 3 * d + t * (d // 2) + 32 * (r >> 3) + 16 * half + 2 * (r & 7)
    u, j = r >> 3, r & 7
    beta = 2 * (j & 3) + np.array([0, 1, 8, 9])[2 * (u & 1) + (j >> 2)]
    if d == 64:
        return s * 3 * d + 2 * d + t * 16 + 8 * half + beta
    return s * 3 * d + 2 * d + t * (d // 4) + 32 * (u >> 1) + 16 * half + beta


def v_bit(bits: int, d: int, tau, c, plane: int = 0):
    tau, c = np.asarray(tau), np.asarray(c)
    g, row8, mt = c & 7, (c >> 3) & 1, c >> 4
    t, hi, half = (tau >> 1) & 3, tau >> 3, tau & 1
    region = g * 4 + t
    if bits == 4:
        return 32 * (region * (d // 16) + mt) + 16 * half + 8 * row8 + 4 * hi
    u, m = mt >> 1, mt & 1
    if bits == 2 or plane == 0:
        return 32 * (region * (d // 32) + u) + 16 * half + 8 * m + 4 * row8 + 2 * hi
    j = 2 * row8 + hi
    beta = 2 * j + np.array([0, 1, 8, 9])[2 * (u & 1) + m]
    return 32 * d + 32 * (region * (d // 64) + (u >> 1)) + 16 * half + beta


def v_param(g: int, tau, gr):
    tau, gr = np.asarray(tau), np.asarray(gr)
    return (((tau >> 1) & 3) * g + gr) * 4 + 2 * (tau >> 3) + (tau & 1)


def _bits_at(region: np.ndarray, off: np.ndarray, width: int) -> np.ndarray:
    """region: [..., nbytes] uint8; off: bit offsets (broadcast over the
    leading axes) -> unsigned fields of `width` bits (never straddling a byte
    pair boundary within a 32-bit word)."""
    w = region.view("<u4")
    word = w[..., off >> 5]
    return ((word >> (off & 31).astype(np.uint32)) & np.uint32((1 << width) - 1)).astype(np.uint8)


def _pack_le(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes [..., D] -> little-endian packing (channel i at bits [bits*i,
    bits*i + bits) of the row's byte string), the oracle's logical layout."""
    d = codes.shape[-1]
    bitv = ((codes[..., :, None] >> np.arange(bits, dtype=np.uint8)) & 1).reshape(*codes.shape[:-1], d * bits)
    return np.packbits(bitv, axis=-1, bitorder="little")


def decode_codes(blk: np.ndarray, d: int, bits: int, kind: str) -> np.ndarray:
    """Code regions of quantised K ("k") or V ("v") head blocks [n, HB] ->
    codes [n][16 tokens][d] uint8."""
    s = np.arange(PAGE)[:, None]
    c = np.arange(d)[None, :]
    reg = np.ascontiguousarray(blk[:, :PAGE * d * bits // 8])
    f = k_bit if kind == "k" else v_bit
    if bits == 3:
        return _bits_at(reg, f(3, d, s, c, 0), 2) | (_bits_at(reg, f(3, d, s, c, 1), 1) << 2)
    return _bits_at(reg, f(bits, d, s, c), bits)


def read_comp(pool: torch.Tensor, table_row: np.ndarray, n: int, hkv: int, d: int, bits: int,
              kind: str = "k") -> dict:
    """GPU comp pool -> oracle.compress-style logical dict for one request
    (`kind` "k" or "v": the two pools place codes and parameters
    differently)."""
    p = pool.cpu().numpy()
    B = hb(d, bits)
    npg = (n + PAGE - 1) // PAGE
    blk = p.reshape(p.shape[0], hkv, B)[table_row[:npg]].reshape(npg * hkv, B)   # [npg*hkv][B]
    if bits == 16:
        x = blk.view(np.uint16).reshape(npg, hkv, PAGE, d).transpose(0, 2, 1, 3).reshape(npg * PAGE, hkv, d)
        return dict(bits=16, x16=x[:n])
    cb, ng = d * bits // 8, d // GROUP
    codes = decode_codes(blk, d, bits, kind)
    codes = codes.reshape(npg, hkv, PAGE, d).transpose(0, 2, 1, 3).reshape(npg * PAGE, hkv, d)
    par = blk[:, PAGE * cb:].copy().view(np.uint16).reshape(npg * hkv, 2, PAGE * ng)
    if kind == "k":
        sc, ze = par[:, 0].reshape(npg * hkv, PAGE, ng), par[:, 1].reshape(npg * hkv, PAGE, ng)
    else:
        idx = v_param(ng, np.arange(PAGE)[:, None], np.arange(ng)[None, :])
        sc, ze = par[:, 0][:, idx], par[:, 1][:, idx]
    sc = sc.reshape(npg, hkv, PAGE, ng).transpose(0, 2, 1, 3).reshape(npg * PAGE, hkv, ng)
    ze = ze.reshape(npg, hkv, PAGE, ng).transpose(0, 2, 1, 3).reshape(npg * PAGE, hkv, ng)
    return dict(bits=bits, packed=_pack_le(codes[:n], bits), scales=sc[:n], zeros=ze[:n])


def read_comp_kv(comp, table: np.ndarray, b: int, n: int) -> dict:
    """Both K and V of request b in the layout of oracle.compress."""
    kk = read_comp(comp.k_pages, table[b], n, comp.num_kv_heads, comp.head_dim, comp.bits, "k")
    vv = read_comp(comp.v_pages, table[b], n, comp.num_kv_heads, comp.head_dim, comp.bits, "v")
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
