"""Pins of the oracle's greedy acceptance against the pages' worked example,
the rule's stated cases and constructed LM heads whose argmax is known.

Source: "VeriCache: Making Lossy KV Compression Exact", The Core Idea: the
drafts are compared with the verifier's predictions left to right; at the
first mismatch the verified prefix plus the verifier's token is emitted and
the rest is discarded; if every draft matches, the whole draft plus the
verifier's extra (bonus) prediction is emitted.
"""
import os

import numpy as np

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "accept_worked_example.txt")


def onehot_head(vocab_targets, dm, vocab):
    """Hidden rows are one-hot e_i and W[i, t_i] = 1, so logits row i peaks at
    t_i with margin 1 and argmax is t_i."""
    w = np.zeros((dm, vocab), np.float32)
    h = np.zeros((len(vocab_targets), dm), np.float32)
    for i, t in enumerate(vocab_targets):
        h[i, i] = 1.0
        w[i, t] = 1.0
    return h, w


def test_pages_worked_example():
    rows = {}
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        key, val = line.split(":", 1)
        rows[key.strip()] = val.split()
    names = sorted(set(rows["draft"]) | {t for t in rows["verify"] if t != "..."} | {"Q"})
    tok = {n: i for i, n in enumerate(names)}
    drafts = np.array([tok[t] for t in rows["draft"]], np.int32)
    x = len(drafts)
    verify = [tok[t] if t != "..." else tok["Q"] for t in rows["verify"]]
    verify = verify + [tok["Q"]] * (x + 1 - len(verify))       # unspecified tail
    h, w = onehot_head(verify, x + 1, len(names))
    r = oracle.accept(h, w, drafts)
    assert list(r["verified"]) == verify
    emit = [tok[t] for t in rows["emit"]]
    assert r["n_emitted"] == len(emit) and list(r["emitted"][:len(emit)]) == emit
    assert r["accept_len"] == 5 and np.all(r["emitted"][len(emit):] == -1)
    assert not r["ambiguous"].any()


def test_all_match_emits_draft_plus_bonus():
    x = 6
    drafts = np.array([4, 9, 1, 1, 0, 7], np.int32)
    h, w = onehot_head(list(drafts) + [3], x + 1, 10)
    r = oracle.accept(h, w, drafts)
    assert r["accept_len"] == x and r["n_emitted"] == x + 1
    assert list(r["emitted"]) == list(drafts) + [3]


def test_all_match_without_bonus_prediction():
    """n_pred = x: no bonus is available; the draft alone is emitted."""
    drafts = np.array([2, 2, 5], np.int32)
    h, w = onehot_head(list(drafts), 3, 8)
    r = oracle.accept(h, w, drafts)
    assert r["accept_len"] == 3 and r["n_emitted"] == 3 and list(r["emitted"]) == [2, 2, 5, -1]


def test_first_position_mismatch_emits_one_token():
    drafts = np.array([1, 2, 3, 4], np.int32)
    h, w = onehot_head([0, 2, 3, 4, 5], 5, 6)
    r = oracle.accept(h, w, drafts)
    assert r["accept_len"] == 0 and r["n_emitted"] == 1 and r["emitted"][0] == 0


def test_argmax_tie_takes_lowest_id():
    w = np.zeros((2, 10), np.float32)
    w[0, [3, 7]] = 2.0
    w[1, [1, 3, 7]] = 1.0
    h = np.array([[1.0, 0.0], [0.0, 1.0]], np.float32)
    r = oracle.accept(h, w, np.array([3], np.int32))
    assert list(r["verified"]) == [3, 1]
    assert r["ambiguous"].all()          # exact ties are near-ties


def test_hidden_group_mean():
    """hidden rows given as hg vectors are averaged: mean of (+e_0, +e_0,
    -e_0, +e_1 * 3) = (0.25, 0.75) selects the column favouring e_1."""
    w = np.zeros((2, 4), np.float32)
    w[0, 0] = 1.0
    w[1, 2] = 1.0
    hid = np.array([[[1, 0], [1, 0], [-1, 0], [0, 3]]], np.float32)
    r = oracle.accept(hid, w, np.array([2], np.int32))
    assert r["verified"][0] == 2 and r["accept_len"] == 1


def test_random_logits_match_brute_force_fp32_argmax():
    """The oracle's logits are fp32 fused multiply-adds in index order; a
    numpy loop doing the same per column with np.float32 gives the same
    argmax ids (brute force over the vocabulary)."""
    rng = np.random.default_rng(0)
    dm, vocab, n = 16, 50, 5
    h = rng.standard_normal((n, dm)).astype(np.float32)
    w = rng.standard_normal((dm, vocab)).astype(np.float32)
    r = oracle.accept(h, w, np.zeros(n - 1, np.int32))
    l64 = h.astype(np.float64) @ w.astype(np.float64)
    for i in range(n):
        if not r["ambiguous"][i]:
            assert r["verified"][i] == int(np.argmax(l64[i]))
