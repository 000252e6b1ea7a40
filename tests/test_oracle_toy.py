"""Pins of the toy-decoder oracle's building blocks against closed forms:
the rotary embedding is the identity at position 0, preserves each rotated
pair's norm, and makes q.k depend only on the position difference; RMSNorm
with unit weight yields unit root-mean-square; SwiGLU of a zero gate is 0."""
import numpy as np

from oracle import toy_model as T


def test_rope_identity_at_zero_and_norm_preserving():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 128))
    assert np.allclose(T.rope(x, np.zeros(5), 128), x, rtol=0, atol=0)
    y = T.rope(x, np.arange(5, dtype=float) * 1000.0, 128)
    n_x = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_y = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.allclose(n_x, n_y, rtol=1e-12, atol=1e-12)


def test_rope_dot_product_depends_on_relative_position_only():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((1, 1, 128)), rng.standard_normal((1, 1, 128))
    dots = []
    for p in (0.0, 7.0, 12345.0):
        qr = T.rope(q, np.array([p + 30.0]), 128)
        kr = T.rope(k, np.array([p]), 128)
        dots.append(float((qr * kr).sum()))
    assert np.allclose(dots, dots[0], rtol=1e-9, atol=1e-9)


def test_rmsnorm_unit_rms_and_swiglu_zero_gate():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 1024)) * 7
    y = T.rmsnorm(x, np.ones(1024))
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-6)
    g = np.zeros(8)
    assert np.all(g / (1.0 + np.exp(-g)) * np.arange(8) == 0)


# ---------------------------------------------------------------------------
# The composed forward pass ("VeriCache: Making Lossy KV Compression Exact",
# The Core Idea: drafter and verifier are the same model, so the loop's
# output is pinned to this model's greedy decoding).  Tiny hand-built models
# whose outputs have closed forms; each catches one plausible mistake in
# forward(): a dropped residual, a wrong norm weight, a misordered q / k / v
# split, gate and up halves swapped, a missing output projection.
# ---------------------------------------------------------------------------

def _bits(x):
    return T._bits(np.asarray(x, dtype=np.float64))


def _model(rng, hq=2, hkv=1, d=4, f=3, vocab=11, dm=None):
    dm = hq * d if dm is None else dm
    shape = dict(hq=hq, hkv=hkv, d=d, ffn=f)
    layer = dict(attn_norm=np.ones(dm, np.float32), mlp_norm=np.ones(dm, np.float32),
                 wqkv=_bits(np.zeros((dm, (hq + 2 * hkv) * d))), wo=_bits(np.zeros((hq * d, dm))),
                 wgu=_bits(np.zeros((dm, 2 * f))), wd=_bits(np.zeros((f, dm))))
    w = dict(embed=rng.standard_normal((vocab, dm)).astype(np.float32),
             final_norm=(0.5 + rng.random(dm)).astype(np.float32), lm_head=np.zeros((dm, vocab), np.float32),
             layers=[layer])
    return w, shape


def _rms(x, w):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + T.EPS) * w


def test_forward_with_silent_blocks_is_the_normed_embedding():
    """Zero output projections: both residual branches add nothing, so the
    result is the final RMSNorm (with its own, non-unit weight) of the
    embedding rows.  A dropped residual gives zeros; a wrong norm weight a
    different scale."""
    rng = np.random.default_rng(10)
    w, shape = _model(rng)
    w["layers"][0]["wqkv"] = _bits(rng.standard_normal(w["layers"][0]["wqkv"].shape))
    w["layers"][0]["wgu"] = _bits(rng.standard_normal(w["layers"][0]["wgu"].shape))
    w["layers"][0]["attn_norm"] = (1 + rng.random(8)).astype(np.float32)
    ids = np.array([3, 1, 4, 1, 5])
    got = T.forward(w, shape, ids)
    want = _rms(w["embed"][ids].astype(np.float64), w["final_norm"].astype(np.float64))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_forward_attention_takes_v_from_the_last_slice_and_averages_causally():
    """q and k columns of wqkv zero, v columns = the identity on the first d
    model dimensions: every score is 0, so position i attends uniformly to
    positions 0..i, and with wo = [I; I] (both query heads of the group
    project back onto the same d dimensions) the residual stream gains twice
    the causal mean of bf16(normed x)[:d].  A split that took v from the q
    or k columns gives zeros or non-uniform weights; a missing wo nothing."""
    rng = np.random.default_rng(11)
    hq, hkv, d = 2, 1, 4
    w, shape = _model(rng, hq, hkv, d)
    dm = hq * d
    L = w["layers"][0]
    wqkv = np.zeros((dm, (hq + 2 * hkv) * d))
    wqkv[:d, (hq + hkv) * d:] = np.eye(d)                  # v = h[:, :d]
    L["wqkv"] = _bits(wqkv)
    wo = np.zeros((hq * d, dm))
    wo[:d, :d] = np.eye(d)
    wo[d:, :d] = np.eye(d)
    L["wo"] = _bits(wo)
    w["final_norm"] = np.ones(dm, np.float32)
    ids = np.array([2, 7, 0, 9])
    got = T.forward(w, shape, ids)
    x = w["embed"][ids].astype(np.float64)
    h = T._bf16(_rms(x, 1.0))[:, :d]
    v = T._bf16(h)                                          # stored as bf16
    mean = np.cumsum(v, axis=0) / np.arange(1, len(ids) + 1)[:, None]
    x2 = x.copy()
    x2[:, :d] += 2 * T._bf16(mean)
    assert np.allclose(got, _rms(x2, 1.0), rtol=1e-9, atol=1e-9)


def test_forward_mlp_gate_is_the_first_half():
    """Attention silent; wgu maps model dim 0 to the gate of unit 0 with
    weight a and to its up input with weight b (a != b); wd returns unit 0 to
    model dim 1.  The residual gains silu(a h0) * (b h0) on dim 1, which is
    not silu(b h0) * (a h0) (halves swapped)."""
    rng = np.random.default_rng(12)
    w, shape = _model(rng, f=3)
    dm, f = 8, 3
    L = w["layers"][0]
    a, b = 1.5, -0.75
    wgu = np.zeros((dm, 2 * f))
    wgu[0, 0], wgu[0, f] = a, b
    L["wgu"] = _bits(wgu)
    wd = np.zeros((f, dm))
    wd[0, 1] = 1.0
    L["wd"] = _bits(wd)
    w["final_norm"] = np.ones(dm, np.float32)
    ids = np.array([4, 6])
    got = T.forward(w, shape, ids)
    x = w["embed"][ids].astype(np.float64)
    h0 = T._bf16(_rms(x, 1.0))[:, 0]
    g, u = a * h0, b * h0
    act = g / (1 + np.exp(-g)) * u
    x2 = x.copy()
    x2[:, 1] += T._bf16(act)
    assert np.allclose(got, _rms(x2, 1.0), rtol=1e-9, atol=1e-9)
    g2, u2 = b * h0, a * h0                                  # the swapped reading differs
    assert not np.allclose(g2 / (1 + np.exp(-g2)) * u2, act)


def test_greedy_choices_argmax_and_margin():
    """LM head = a scaled copy of the identity on the first vocab rows: the
    argmax of each position's logits is the model dimension with the largest
    normed value; the margin is its gap to the runner-up."""
    rng = np.random.default_rng(13)
    w, shape = _model(rng, vocab=11)
    w["lm_head"][:, :8] = 3.0 * np.eye(8, dtype=np.float32)
    ids = np.array([1, 2, 3, 4])
    arg, margin = T.greedy_choices(w, shape, ids, 2)
    h = T.forward(w, shape, ids)[1:]
    logits = np.concatenate([3.0 * h, np.zeros((h.shape[0], 3))], axis=1)
    srt = np.sort(logits, axis=1)
    assert np.array_equal(arg, np.argmax(logits, axis=1))
    assert np.allclose(margin, srt[:, -1] - srt[:, -2], rtol=1e-12, atol=1e-12)
