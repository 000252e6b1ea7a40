"""End-to-end pin of one VeriCache round inside the oracle: with KV_comp
equal to KV_full (every token kept, 16-bit storage) every drafted token is
accepted and the bonus token is emitted (x + 1 tokens).

Source: "VeriCache: Making Lossy KV Compression Exact", The Core Idea (draft x
tokens with the compressed cache, verify them in one pass with x + 1
predictions, accept the longest matching prefix plus correction or bonus).
Attention-only reading: a position's hidden vector is the mean over query
heads of its attention output; the drafted token at step i is the argmax of
the LM head applied to the draft output of query i.
"""
import numpy as np

import oracle
from synth import bf16_bits


def test_identical_caches_accept_everything():
    rng = np.random.default_rng(21)
    n_prefix, x, hkv, grp, d, vocab = 30, 6, 2, 2, 32, 200
    hq = hkv * grp
    n_ctx = n_prefix + x + 1
    k = bf16_bits(rng.standard_normal((n_ctx, hkv, d)).astype(np.float32))
    v = bf16_bits(rng.standard_normal((n_ctx, hkv, d)).astype(np.float32))
    q = bf16_bits(rng.standard_normal((x + 1, hq, d)).astype(np.float32))
    w = (rng.standard_normal((d, vocab)) * 0.05).astype(np.float32)
    scale = float(np.float32(1 / np.sqrt(d)))
    drafts = []
    for i in range(x):
        n_comp = n_prefix + i + 1          # prefix + tokens appended so far + self
        comp = oracle.compress(k[:n_comp], v[:n_comp], np.arange(n_comp, dtype=np.int32), 16)
        o = oracle.draft_attn(q[i], comp, scale).astype(np.float32)
        r = oracle.accept(o[None, :, :], w, np.zeros(0, np.int32))
        drafts.append(int(r["verified"][0]))
    ov = oracle.verify_attn_block(q, k, v, scale).astype(np.float32)     # [x+1][hq][d]
    r = oracle.accept(ov, w, np.array(drafts, np.int32))
    assert r["accept_len"] == x and r["n_emitted"] == x + 1
    assert list(r["emitted"][:x]) == drafts
    assert r["emitted"][x] == r["verified"][x]


def test_corrupted_cache_is_corrected_by_verifier():
    """Whatever the drafter proposes, the emitted tokens are the verifier's
    own predictions up to and including the first mismatch."""
    rng = np.random.default_rng(22)
    x, vocab, d = 8, 50, 16
    h = rng.standard_normal((x + 1, d)).astype(np.float32)
    w = rng.standard_normal((d, vocab)).astype(np.float32)
    ver = oracle.accept(h, w, np.zeros(0, np.int32))["verified"]
    for bad in range(x):
        drafts = ver[:x].copy()
        drafts[bad] = (drafts[bad] + 1) % vocab
        r = oracle.accept(h, w, drafts)
        assert r["accept_len"] == bad
        assert list(r["emitted"][:bad + 1]) == list(ver[:bad + 1])
