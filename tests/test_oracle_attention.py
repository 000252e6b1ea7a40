"""Pins of the oracle's attention (single-query draft attention over the
compressed cache and causal block verification over the full cache) against
closed forms and invariants that do not come from the oracle itself.

Sources: "VeriCache: Making Lossy KV Compression Exact", The Core Idea (draft
with KV_comp; one verification pass over KV_full gives a prediction for each
drafted position and one more); "KV Cache and Speculative Decoding",
Autoregressive Decoding and the KV Cache (a query attends causally to itself
and every earlier position; grouped-query attention shares K/V heads).
"""
import math

import numpy as np
import pytest

import oracle
from synth import bf16_bits, bf16_to_f32


def bf(x):
    return bf16_bits(np.asarray(x, np.float32))


def f(b):
    return bf16_to_f32(b).astype(np.float64)


# ---------------------------------------------------------------- attend

def test_single_key_returns_its_value():
    rng = np.random.default_rng(0)
    q, k, v = rng.standard_normal(8), rng.standard_normal((1, 8)), rng.standard_normal((1, 8))
    o, w = oracle.attend(q, k, v, 0.3, want_weights=True)
    assert np.array_equal(o, v[0]) and w[0] == 1.0


def test_identical_keys_give_mean_value():
    rng = np.random.default_rng(1)
    k = np.tile(rng.standard_normal(16), (9, 1))
    v = rng.standard_normal((9, 16))
    o = oracle.attend(rng.standard_normal(16), k, v, 0.25)
    assert np.allclose(o, v.mean(0), rtol=0, atol=1e-15)


def test_two_keys_closed_form():
    """q.k0 - q.k1 = delta -> weight of k0 = 1 / (1 + exp(-scale delta))."""
    q = np.array([1.0, 0, 0, 0])
    k = np.array([[3.0, 1, 0, 0], [1.0, 0, 5, 0]])
    v = np.array([[1.0, 0, 0, 2], [0.0, 1, 0, -2]])
    scale = 0.5
    a = 1.0 / (1.0 + math.exp(-scale * 2.0))
    o = oracle.attend(q, k, v, scale)
    assert np.allclose(o, a * v[0] + (1 - a) * v[1], rtol=0, atol=1e-15)


def test_dominant_key_and_underflow():
    q = np.ones(4)
    k = np.zeros((5, 4))
    k[3] = 400.0                      # scores 0,0,0,1600*scale,0
    v = np.arange(20.0).reshape(5, 4)
    o = oracle.attend(q, k, v, 1.0)
    assert np.array_equal(o, v[3])    # exp(-1600) underflows to exactly 0


def test_weights_sum_to_one_and_convexity():
    rng = np.random.default_rng(2)
    for n in (1, 2, 7, 100, 1000):
        k, v = rng.standard_normal((n, 32)) * 3, rng.standard_normal((n, 32))
        o, w = oracle.attend(rng.standard_normal(32), k, v, 1 / math.sqrt(32), want_weights=True)
        assert abs(w.sum() - 1.0) <= 1e-12 and np.all(w >= 0)
        assert np.all(o <= v.max(0) + 1e-12) and np.all(o >= v.min(0) - 1e-12)


def test_key_permutation_invariance():
    rng = np.random.default_rng(3)
    k, v, q = rng.standard_normal((33, 16)), rng.standard_normal((33, 16)), rng.standard_normal(16)
    p = rng.permutation(33)
    assert np.allclose(oracle.attend(q, k, v, 0.2), oracle.attend(q, k[p], v[p], 0.2),
                       rtol=0, atol=1e-14)


def test_brute_force_tiny_against_enumerated_logsumexp():
    """N <= 16, D = 4: the weights satisfy log p_t = s_t - logsumexp(s) where
    the log-sum-exp is taken with math.fsum over all terms (exact summation);
    o is compared with an fsum of p_t v_t per channel."""
    rng = np.random.default_rng(4)
    for n in range(1, 17):
        q, k, v = rng.standard_normal(4), rng.standard_normal((n, 4)), rng.standard_normal((n, 4))
        o, w = oracle.attend(q, k, v, 0.7, want_weights=True)
        s = [0.7 * math.fsum(q[i] * k[t, i] for i in range(4)) for t in range(n)]
        lse = math.log(math.fsum(math.exp(x) for x in s))
        pw = [math.exp(x - lse) for x in s]
        assert np.allclose(w, pw, rtol=1e-13, atol=0)
        for c in range(4):
            assert abs(o[c] - math.fsum(pw[t] * v[t, c] for t in range(n))) <= 1e-13


# ---------------------------------------------------------------- verify

def test_verify_causal_mask_against_dominant_key():
    """Keys are all zero except one at position p with a huge score.  A query
    at position >= p sees it (output = v_p); a query before p does not, and
    with equal scores its output is the mean of V[0..pos]."""
    n_ctx, n_q, d = 24, 8, 8
    p = 19
    k = np.zeros((n_ctx, 1, d), np.float32)
    k[p, 0, :] = 64.0
    v = np.random.default_rng(5).standard_normal((n_ctx, 1, d)).astype(np.float32)
    kb, vb = bf(k), bf(v)
    q = bf(np.ones((n_q, 1, d), np.float32))
    out = oracle.verify_attn(q, kb, vb, 1.0)
    vf = f(vb)[:, 0]
    for i in range(n_q):
        pos = n_ctx - n_q + i
        if pos >= p:
            assert np.array_equal(out[i, 0], vf[p])
        else:
            assert np.allclose(out[i, 0], vf[:pos + 1].mean(0), rtol=0, atol=1e-14)


def test_verify_gqa_head_mapping():
    """V is constant c_g on kv head g, so every query head h outputs exactly
    c_{h // G} (weights sum to one), whatever the scores."""
    rng = np.random.default_rng(6)
    hkv, grp, d, n_ctx, n_q = 3, 4, 16, 40, 5
    k = bf(rng.standard_normal((n_ctx, hkv, d)))
    c = np.array([1.5, -2.0, 0.25])
    v = bf(np.broadcast_to(c[None, :, None], (n_ctx, hkv, d)).astype(np.float32))
    q = bf(rng.standard_normal((n_q, hkv * grp, d)))
    out = oracle.verify_attn_block(q, k, v, 0.125)
    for h in range(hkv * grp):
        assert np.allclose(out[:, h], c[h // grp], rtol=0, atol=1e-14)


def test_verify_rows_equal_single_query_attention():
    rng = np.random.default_rng(7)
    n_ctx, n_q, hkv, grp, d = 37, 9, 2, 2, 32
    k = bf(rng.standard_normal((n_ctx, hkv, d)))
    v = bf(rng.standard_normal((n_ctx, hkv, d)))
    q = bf(rng.standard_normal((n_q, hkv * grp, d)))
    blk = oracle.verify_attn_block(q, k, v, 0.17)
    per = oracle.verify_attn(q, k, v, 0.17)
    assert np.array_equal(blk, per)
    for i in (0, 4, 8):
        for h in range(hkv * grp):
            pos = n_ctx - n_q + i
            o = oracle.attend(f(q[i, h]), f(k[:pos + 1, h // grp]), f(v[:pos + 1, h // grp]), 0.17)
            assert np.array_equal(o, blk[i, h])


# ---------------------------------------------------------------- draft

def test_draft_ratio_one_bf16_equals_full_attention():
    """Compression ratio 1 with 16-bit storage (every token kept, bf16) must
    reproduce full attention: the draft output equals the verification output
    of a one-query block at the last position."""
    rng = np.random.default_rng(8)
    n, hkv, grp, d = 50, 2, 4, 64
    k = bf(rng.standard_normal((n, hkv, d)))
    v = bf(rng.standard_normal((n, hkv, d)))
    q = bf(rng.standard_normal((hkv * grp, d)))
    comp = oracle.compress(k, v, np.arange(n, dtype=np.int32), 16)
    dr = oracle.draft_attn(q, comp, 0.125)
    ve = oracle.verify_attn_block(q[None], k, v, 0.125)[0]
    assert np.array_equal(dr, ve)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_draft_quantised_on_exact_grid_equals_bf16(bits):
    """K/V rows that lie exactly on a 2^-3 grid with all 2^b levels present in
    every group quantise losslessly, so the b-bit draft equals the bf16 draft
    on the same kept tokens (pins unpack + dequant + gather order)."""
    rng = np.random.default_rng(9 + bits)
    n, hkv, grp, d = 40, 2, 2, 64
    q_levels = (1 << bits)

    def grid(shape):
        lv = rng.integers(0, q_levels, shape)
        lv[..., 0::32] = 0
        lv[..., 1::32] = q_levels - 1
        off = rng.integers(-8, 8, shape[:-1] + (d // 32,))
        return (np.repeat(off, 32, axis=-1) + lv) * 0.125

    k, v = bf(grid((n, hkv, d))), bf(grid((n, hkv, d)))
    kept = np.array([0, 2, 3, 10, 11, 12, 30, 39], np.int32)
    q = bf(rng.standard_normal((hkv * grp, d)))
    a = oracle.draft_attn(q, oracle.compress(k, v, kept, bits), 0.2)
    b = oracle.draft_attn(q, oracle.compress(k, v, kept, 16), 0.2)
    assert np.allclose(a, b, rtol=0, atol=1e-13)


def test_draft_gqa_head_mapping():
    rng = np.random.default_rng(12)
    n, hkv, grp, d = 20, 4, 2, 32
    k = bf(rng.standard_normal((n, hkv, d)))
    c = np.array([0.5, -1.0, 2.0, 3.0])
    v = bf(np.broadcast_to(c[None, :, None], (n, hkv, d)).astype(np.float32))
    q = bf(rng.standard_normal((hkv * grp, d)))
    out = oracle.draft_attn(q, oracle.compress(k, v, np.arange(0, n, 3, dtype=np.int32), 16), 0.3)
    for h in range(hkv * grp):
        assert np.allclose(out[h], c[h // grp], rtol=0, atol=1e-14)
