"""Oracle of the toy decoder used by the end-to-end greedy loop.

TEST INFRASTRUCTURE ONLY (tests import it; the library never does).  Plain
numpy, fp64 arithmetic; values are rounded to bf16 where the model stores
them as bf16 (activations entering a projection, q / k / v), the attention is
the oracle's causal verification attention (vc_oracle.c), and the LM head is
fp64.  Source: "VeriCache: Making Lossy KV Compression Exact", The Core Idea
(drafter and verifier are the same model; greedy decoding).  Model choices
(not on the pages; any fixed model works because exactness is relative to
the same model): pre-RMSNorm (eps 1e-5), rotary embedding (theta 500000,
channel i paired with i + D/2), grouped-query attention, SwiGLU MLP.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

THETA = 500000.0
EPS = 1e-5


def _bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 (round to nearest even) -> value in fp64."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return (((u + r) >> 16) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def _bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


def _w(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm(x, w):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS) * w


def rope(x, pos, d):
    """x [n][h][d] fp64, rotate-half pairs (i, i + d/2)."""
    half = d // 2
    inv = THETA ** (-2.0 * np.arange(half) / d)
    ang = pos[:, None] * inv[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x0, x1 = x[..., :half], x[..., half:]
    return np.concatenate([x0 * c - x1 * s, x1 * c + x0 * s], axis=-1)


def forward(weights: dict, shape: dict, ids: np.ndarray) -> np.ndarray:
    """One request, tokens ids [n] at positions 0..n-1 (causal).  Returns
    the final-norm hidden states fp64 [n][d_model]."""
    hq, hkv, d, f = shape["hq"], shape["hkv"], shape["d"], shape["ffn"]
    n = ids.size
    pos = np.arange(n, dtype=np.float64)
    x = weights["embed"][ids].astype(np.float64)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    for L in weights["layers"]:
        h = rmsnorm(x, L["attn_norm"].astype(np.float64))
        qkv = _bf16(h) @ _w(L["wqkv"])
        q = qkv[:, :hq * d].reshape(n, hq, d)
        k = qkv[:, hq * d:(hq + hkv) * d].reshape(n, hkv, d)
        v = qkv[:, (hq + hkv) * d:].reshape(n, hkv, d)
        qb, kb, vb = _bits(rope(q, pos, d)), _bits(rope(k, pos, d)), _bits(v)
        o = oracle.verify_attn_block(qb, kb, vb, scale).reshape(n, hq * d)
        x = x + _bf16(o) @ _w(L["wo"])
        h = rmsnorm(x, L["mlp_norm"].astype(np.float64))
        gu = _bf16(h) @ _w(L["wgu"])
        g, u = gu[:, :f], gu[:, f:]
        act = g / (1.0 + np.exp(-g)) * u
        x = x + _bf16(act) @ _w(L["wd"])
    return rmsnorm(x, weights["final_norm"].astype(np.float64))


def greedy_choices(weights: dict, shape: dict, tokens: np.ndarray, start: int):
    """Teacher-forced over `tokens` (prompt + generated): for each position
    p >= start - 1 the fp64 argmax of the next-token logits and its margin
    to the runner-up.  Returns (argmax [n - start + 1], margin [...])."""
    h = forward(weights, shape, tokens)
    logits = h[start - 1:] @ weights["lm_head"].astype(np.float64)
    top2 = np.argsort(-logits, axis=1, kind="stable")[:, :2]
    rows = np.arange(logits.shape[0])
    return top2[:, 0], logits[rows, top2[:, 0]] - logits[rows, top2[:, 1]]
