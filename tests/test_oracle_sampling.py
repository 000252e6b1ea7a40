"""Pins of the oracle's rejection-sampling acceptance ("VeriCache Guide",
"Mathematical Guarantee of Lossless Correctness") that do not reuse its
code: identical draft and target distributions accept every draft and draw
the bonus by an inverse CDF written with numpy; the emitted token's
distribution equals the target distribution (the guarantee itself, Monte
Carlo); a zero draft probability is always accepted; the fp32 logits match
the greedy path's arithmetic."""
import numpy as np

import oracle


def softmax64(l, tau):
    z = l.astype(np.float64) / tau
    e = np.exp(z - z.max())
    return e / e.sum()


def test_identical_distributions_accept_all_and_draw_the_bonus():
    rng = np.random.default_rng(1)
    x, vocab, tau = 5, 50, 0.7
    tl = rng.standard_normal((x + 1, vocab)).astype(np.float32)
    drafts = rng.integers(0, vocab, x).astype(np.int32)
    u = rng.random(x).astype(np.float32) * 0.999
    v = rng.random(x + 1).astype(np.float32)
    r = oracle.accept_sampled(tl, tl[:x], drafts, u, v, tau)
    assert r["accept_len"] == x
    p = softmax64(tl[x], tau)
    bonus = int(np.searchsorted(np.cumsum(p), float(v[x]) * p.sum(), side="right"))
    assert list(r["emitted"]) == list(drafts) + [bonus]


def test_emitted_token_follows_the_target_distribution():
    """P(emit t) = p_target(t) when the draft token is drawn from p_draft."""
    rng = np.random.default_rng(2)
    vocab, tau, trials = 6, 1.0, 40000
    tl = np.array([[1.0, 0.2, -0.5, 2.0, 0.0, -1.0], [0.0] * 6], np.float32)
    dl = np.array([[0.0, 1.5, 0.3, -0.2, 1.0, -0.3]], np.float32)
    pt, pd = softmax64(tl[0], tau), softmax64(dl[0], tau)
    counts = np.zeros(vocab)
    for _ in range(trials):
        d = int(rng.choice(vocab, p=pd))
        r = oracle.accept_sampled(tl, dl, np.array([d], np.int32), rng.random(1, dtype=np.float32),
                                  rng.random(2, dtype=np.float32), tau)
        counts[r["emitted"][0]] += 1
    emp = counts / trials
    sd = np.sqrt(pt * (1 - pt) / trials)
    assert np.all(np.abs(emp - pt) < 5 * sd + 1e-4), (emp, pt)


def test_zero_draft_probability_is_accepted():
    tl = np.zeros((2, 4), np.float32)
    dl = np.array([[0.0, 0.0, -1e30, 0.0]], np.float32)      # p_draft(2) = 0
    r = oracle.accept_sampled(tl, dl, np.array([2], np.int32), np.array([0.99], np.float32),
                              np.array([0.5, 0.5], np.float32), 1.0)
    assert r["accept_len"] == 1 and r["emitted"][0] == 2


def test_logits_are_the_greedy_path_logits():
    rng = np.random.default_rng(4)
    hidden = rng.standard_normal((3, 4, 32)).astype(np.float32)
    w = (rng.standard_normal((32, 200)) * 0.05).astype(np.float32)
    lg = oracle.logits(hidden, w)
    ver = oracle.accept(hidden, w, np.zeros(0, np.int32))["verified"]
    assert np.array_equal(lg.argmax(axis=1), ver)
    ref = (hidden.astype(np.float64).mean(axis=1) @ w.astype(np.float64))
    assert np.allclose(lg, ref, rtol=1e-4, atol=1e-5)
