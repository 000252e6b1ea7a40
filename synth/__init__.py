"""Seeded synthetic inputs for the VeriCache attention-step operations.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark.  It only draws random numbers and lays them out (pages, block
tables, kept-index lists); it holds none of the arithmetic of the method
(no quantisation, attention, argmax or acceptance).

Workload shapes follow the pages' long-context settings (Llama-3.1-8B/70B
shaped attention, 32k-128k context, 4x compression, 25-40 token drafts); the
five named workloads are in ``WORKLOADS``.  Values: K, V, Q ~ N(0, 1) rounded
to bf16 (round to nearest even), a few K "outlier" channels multiplied by a
constant before rounding, LM-head weights ~ N(0, sigma) in fp32.
"""
from __future__ import annotations

import numpy as np

PAGE = 16  # tokens per KV page (paged KV block size)

# ----------------------------------------------------------------------------
# bf16 bit helpers (input rounding only)
# ----------------------------------------------------------------------------


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0,
                chunk: int = 1 << 24) -> np.ndarray:
    """N(0, std^2) samples rounded to bf16 bits, drawn in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = bf16_bits(x)
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# paged KV pools and block tables
# ----------------------------------------------------------------------------


def pages_for(n: int) -> int:
    return (n + PAGE - 1) // PAGE


def block_tables(rng: np.random.Generator, lens, capacity=None):
    """Random page assignment.

    lens: tokens each request must hold; capacity: tokens to reserve per
    request (>= lens), default lens.  Returns (table int32 [B][max_blocks],
    total_pages).  Unused slots hold -1.  Physical pages are a seeded
    permutation, so consecutive logical pages are scattered in the pool.
    """
    lens = np.asarray(lens, dtype=np.int64)
    cap = lens if capacity is None else np.maximum(np.asarray(capacity), lens)
    nblk = [pages_for(int(c)) for c in cap]
    total = int(sum(nblk))
    maxb = max(1, max(nblk) if nblk else 1)
    perm = rng.permutation(total).astype(np.int32)
    table = np.full((len(lens), maxb), -1, dtype=np.int32)
    o = 0
    for b, k in enumerate(nblk):
        table[b, :k] = perm[o:o + k]
        o += k
    return table, total


def kv_pools(rng: np.random.Generator, num_pages: int, hkv: int, d: int,
             outlier_channels=(), outlier_scale: float = 1.0):
    """K and V page pools, bf16 bits, layout [page][kv_head][16][d].

    Every slot is an independent N(0,1) draw, so a request's logical K/V is
    whatever its block table points at.  K's outlier channels are multiplied
    by ``outlier_scale`` before rounding to bf16.
    """
    shape = (num_pages, hkv, PAGE, d)
    v = normal_bf16(rng, shape)
    if len(outlier_channels) == 0:
        k = normal_bf16(rng, shape)
    else:
        n = int(np.prod(shape))
        k = np.empty(n, dtype=np.uint16)
        chunk = (1 << 24) // d * d
        mult = np.ones(d, dtype=np.float32)
        mult[list(outlier_channels)] = np.float32(outlier_scale)
        for s in range(0, n, chunk):
            e = min(n, s + chunk)
            x = rng.standard_normal(e - s, dtype=np.float32).reshape(-1, d)
            x *= mult
            k[s:e] = bf16_bits(x).reshape(-1)
        k = k.reshape(shape)
    return k, v


def outlier_channels(rng: np.random.Generator, d: int, count: int):
    return sorted(int(c) for c in rng.choice(d, size=count, replace=False))


def logical_from_pages(pool: np.ndarray, table_row: np.ndarray, n: int) -> np.ndarray:
    """Gather one request's first n tokens: pool [P][H][16][d] -> [n][H][d]."""
    npg = pages_for(n)
    if n == 0:
        return np.zeros((0,) + (pool.shape[1], pool.shape[3]), dtype=pool.dtype)
    pg = pool[table_row[:npg]]                       # [npg][H][16][d]
    pg = pg.transpose(0, 2, 1, 3).reshape(npg * PAGE, pool.shape[1], pool.shape[3])
    return pg[:n]


def pages_from_logical(pool: np.ndarray, table_row: np.ndarray, x: np.ndarray, start: int = 0):
    """Write logical tokens x [n][H][...] into pool pages from token ``start``."""
    for j in range(x.shape[0]):
        t = start + j
        pool[table_row[t // PAGE], :, t % PAGE] = x[j]


# ----------------------------------------------------------------------------
# kept-index lists (token-drop); the selection heuristics of the pages are
# out of scope, so a seeded stand-in picks the positions
# ----------------------------------------------------------------------------


def kept_sink_recent_random(rng, n: int, sink: int, recent: int, n_random: int) -> np.ndarray:
    """sink tokens + recent tokens + n_random distinct seeded draws from the
    middle, sorted ascending (shared by all kv-heads of the request)."""
    mid = np.arange(sink, n - recent)
    pick = rng.choice(mid, size=min(n_random, mid.size), replace=False)
    idx = np.concatenate([np.arange(sink), pick, np.arange(n - recent, n)])
    return np.unique(idx).astype(np.int32)


def kept_sink_recent_topk(rng, n: int, sink: int, recent: int, total: int) -> np.ndarray:
    """sink + recent + the highest seeded uniform scores of the middle so the
    list holds ``total`` positions; equal scores keep the lower index."""
    mid_n = n - sink - recent
    k = total - sink - recent
    score = rng.random(mid_n, dtype=np.float32)
    order = np.lexsort((np.arange(mid_n), -score))   # score desc, index asc
    pick = sink + np.sort(order[:k])
    idx = np.concatenate([np.arange(sink), pick, np.arange(n - recent, n)])
    return idx.astype(np.int32)


def csr(lists):
    offs = np.zeros(len(lists) + 1, dtype=np.int32)
    for i, l in enumerate(lists):
        offs[i + 1] = offs[i] + len(l)
    idx = np.concatenate([np.asarray(l, dtype=np.int32) for l in lists]) if lists else np.zeros(0, np.int32)
    return offs, idx.astype(np.int32)


# ----------------------------------------------------------------------------
# other inputs
# ----------------------------------------------------------------------------


def lm_head(rng, d: int, vocab: int, std: float) -> np.ndarray:
    return (rng.standard_normal((d, vocab), dtype=np.float32) * np.float32(std)).astype(np.float32)


def token_ids(rng, shape, vocab: int) -> np.ndarray:
    return rng.integers(0, vocab, size=shape, dtype=np.int64).astype(np.int32)


# ----------------------------------------------------------------------------
# the five named workloads (shapes, seeds)
# ----------------------------------------------------------------------------

WORKLOADS = {
    "tiny": dict(
        desc="1 request, 4q/1kv heads, head_dim 64, context 512, 2 K outlier "
             "channels x8; 128 kept (16 sink + 48 recent + 64 random) at 4-bit; "
             "x=8; LM head 64x1000 ~N(0,0.05)",
        batch=1, hq=4, hkv=1, d=64, ctx=512, outliers=2, outlier_scale=8.0,
        bits=4, sink=16, recent=48, n_random=64, x=8, vocab=1000, lm_std=0.05, seed=1),
    "8b_32k_2bit": dict(
        desc="Llama-3.1-8B-shaped attention layer: batch 8, 32q/8kv, head_dim 128, "
             "context 32768, page 16, 4 K outlier channels x10; KV_comp = all "
             "tokens at 2-bit group 32; x=32",
        batch=8, hq=32, hkv=8, d=128, ctx=32768, outliers=4, outlier_scale=10.0,
        bits=2, x=32, vocab=32000, lm_std=0.05, seed=2),
    "70b_128k_drop4": dict(
        desc="Llama-3.1-70B-shaped attention layer: batch 4, 64q/8kv, head_dim 128, "
             "context 131072; KV_comp = 32768 kept (64 sink + 512 recent + top "
             "seeded scores) in bf16; x=40",
        batch=4, hq=64, hkv=8, d=128, ctx=131072, outliers=0, outlier_scale=1.0,
        bits=16, sink=64, recent=512, kept_total=32768, x=40, vocab=32000, lm_std=0.05, seed=3),
    "mixed_32req_3bit": dict(
        desc="staggered mixed batch: 32 requests, context U[8192,65536], 32q/8kv, "
             "head_dim 128, 3-bit group-32 KV_comp; even requests draft, odd "
             "requests verify x=25 over KV_full staged from pinned host memory",
        batch=32, hq=32, hkv=8, d=128, ctx_lo=8192, ctx_hi=65536, outliers=0,
        outlier_scale=1.0, bits=3, x=25, seed=4),
    "stagger_32req_3bit": dict(
        desc="staggering scheduler across requests, layers and rounds: 32 requests, "
             "context U[8192,65536], 2 attention layers of 32q/8kv, head_dim 128, "
             "3-bit group-32 KV_comp resident, bf16 KV_full in page-locked host "
             "memory staged for each verification; x=25 (block of 25 queries), "
             "room for blocks up to 64",
        batch=32, hq=32, hkv=8, d=128, ctx_lo=8192, ctx_hi=65536, layers=2, bits=3, x=25,
        max_x=64, seed=6),
    "remote_prefix_8req_3bit": dict(
        desc="remote prefix caching on one box: 8 stored prefixes of 32768 tokens, 2 "
             "attention layers of 32q/8kv, head_dim 128; the 3-bit KV_comp crosses a "
             "slow link paced at 25 GB/s, the bf16 KV_full a fast link (plain staging); "
             "x=25, 4 rounds; baseline: KV_full over the slow link, one-token decoding",
        batch=8, hq=32, hkv=8, d=128, ctx=32768, layers=2, bits=3, x=25, rounds=4,
        slow_GBps=25.0, chunk_MB=4, seed=7),
    "toy_e2e": dict(
        desc="2-layer decoder d_model 1024, 8q/2kv heads, head_dim 128, SwiGLU 4096, "
             "vocab 32000, weights N(0,0.02); batch 4, prompt 16384; 4-bit KV_comp; "
             "x=32; 512 generated tokens",
        batch=4, layers=2, d_model=1024, hq=8, hkv=2, d=128, ffn=4096, vocab=32000,
        w_std=0.02, prompt=16384, bits=4, x=32, gen=512, seed=5),
}


def rng_for(name: str, salt: int = 0) -> np.random.Generator:
    return np.random.default_rng([WORKLOADS[name]["seed"], salt])


def toy_weights(rng, w: dict) -> dict:
    """Random-init weights of the toy decoder, N(0, w_std): bf16 projection
    matrices [in][out], fp32 embedding table and LM head, unit norm weights."""
    dm, hq, hkv, d, f, vocab, std = w["d_model"], w["hq"], w["hkv"], w["d"], w["ffn"], w["vocab"], w["w_std"]
    out = {"embed": (rng.standard_normal((vocab, dm), dtype=np.float32) * np.float32(std)).astype(np.float32),
           "lm_head": (rng.standard_normal((dm, vocab), dtype=np.float32) * np.float32(std)).astype(np.float32),
           "final_norm": np.ones(dm, np.float32), "layers": []}
    for _ in range(w["layers"]):
        out["layers"].append({
            "attn_norm": np.ones(dm, np.float32),
            "wqkv": normal_bf16(rng, (dm, (hq + 2 * hkv) * d), std),
            "wo": normal_bf16(rng, (hq * d, dm), std),
            "mlp_norm": np.ones(dm, np.float32),
            "wgu": normal_bf16(rng, (dm, 2 * f), std),
            "wd": normal_bf16(rng, (f, dm), std),
        })
    return out
