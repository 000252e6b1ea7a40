"""GPU vc_accept against the oracle.  Both compute every logit as fp32
fused multiply-adds in increasing hidden index from the same fp32 mean of
the hidden group, so verified ids, acceptance lengths and emitted tokens
must be bit-exact (no near-tie exclusion is needed; the oracle's near-tie
flags are still reported)."""
import os

import numpy as np
import pytest
import torch

import oracle
from tests import vc_harness as H

pytestmark = pytest.mark.gpu


def gpu_accept(hidden, w, drafts, hg=1):
    import lossless_compressed_kv_gb300 as vc
    hd = H.to_dev(hidden.astype(np.float32))
    wd = H.to_dev(w.astype(np.float32))
    b, n_pred = hidden.shape[0], hidden.shape[1]
    x = drafts.shape[1]
    dd = H.to_dev(drafts.astype(np.int32)) if x else torch.zeros((b, 0), dtype=torch.int32, device="cuda")
    ver = torch.full((b, n_pred), -7, dtype=torch.int32, device="cuda")
    al = torch.full((b,), -7, dtype=torch.int32, device="cuda")
    em = torch.full((b, x + 1), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(vc.accept_workspace_bytes(b, n_pred, w.shape[1], w.shape[0]), dtype=torch.uint8, device="cuda")
    vc.accept(hd, wd, dd, ver, al, em, ws, hidden_group=hg)
    torch.cuda.synchronize()
    return ver.cpu().numpy(), al.cpu().numpy(), em.cpu().numpy()


def check(hidden, w, drafts, hg=1):
    ver, al, em = gpu_accept(hidden, w, drafts, hg)
    for b in range(hidden.shape[0]):
        h = hidden[b] if hg > 1 else hidden[b][:, None, :]
        r = oracle.accept(h, w, drafts[b])
        assert np.array_equal(ver[b], r["verified"]), b
        assert al[b] == r["accept_len"], b
        assert np.array_equal(em[b], r["emitted"]), b
    return ver, al, em


@pytest.mark.parametrize("bonus", [True, False])
@pytest.mark.parametrize("hg", [1, 4])
def test_accept_random_with_planted_mismatches(bonus, hg):
    rng = np.random.default_rng(3 + hg + bonus)
    B, x, d, vocab = 5, 9, 64, 1000
    n_pred = x + 1 if bonus else x
    shape = (B, n_pred, hg, d) if hg > 1 else (B, n_pred, d)
    hidden = rng.standard_normal(shape).astype(np.float32)
    w = (rng.standard_normal((d, vocab)) * 0.05).astype(np.float32)
    drafts = np.zeros((B, x), np.int32)
    for b in range(B):
        h = hidden[b] if hg > 1 else hidden[b][:, None, :]
        ver = oracle.accept(h, w, np.zeros(0, np.int32))["verified"]
        drafts[b] = ver[:x]
        if b < x and b < B - 1:
            drafts[b, b] = (drafts[b, b] + 1) % vocab     # first mismatch at position b
    ver, al, em = check(hidden, w, drafts, hg)
    assert al[B - 1] == x                                    # the untouched request accepts all


def test_accept_pages_worked_example_on_gpu():
    """Draft A..H, verifier A B C D E X ...: emit A B C D E X."""
    names = "ABCDEFGHXQ"
    tok = {c: i for i, c in enumerate(names)}
    drafts = np.array([[tok[c] for c in "ABCDEFGH"]], np.int32)
    verify = [tok[c] for c in "ABCDEX"] + [tok["Q"]] * 3
    hidden = np.zeros((1, 9, 9), np.float32)
    w = np.zeros((9, len(names)), np.float32)
    for i, t in enumerate(verify):
        hidden[0, i, i] = 1.0
        w[i, t] = 1.0
    ver, al, em = check(hidden, w, drafts)
    assert al[0] == 5 and [names[t] for t in em[0] if t >= 0] == list("ABCDEX")


def test_accept_vocab_tail_and_ties():
    """Vocabulary not a multiple of the 256-column tile, equal maxima in
    different tiles: the lowest id wins."""
    d, vocab = 8, 777
    w = np.zeros((d, vocab), np.float32)
    w[0, [5, 300, 776]] = 3.0
    w[1, 776] = 1.0
    hidden = np.zeros((1, 2, d), np.float32)
    hidden[0, 0, 0] = 1.0
    hidden[0, 1, 1] = 1.0
    ver, al, em = check(hidden, w, np.array([[5]], np.int32))
    assert list(ver[0]) == [5, 776] and al[0] == 1 and list(em[0]) == [5, 776]


def test_accept_toy_e2e_size():
    """The toy decoder's LM head (d 1024, vocab 32000), 4 requests x 33 rows."""
    rng = np.random.default_rng(9)
    B, x, d, vocab = 4, 32, 1024, 32000
    hidden = rng.standard_normal((B, x + 1, d)).astype(np.float32)
    w = (rng.standard_normal((d, vocab)) * 0.02).astype(np.float32)
    drafts = rng.integers(0, vocab, (B, x)).astype(np.int32)
    ver, _, _ = gpu_accept(hidden, w, np.zeros((B, x), np.int32))
    drafts[:, :20] = ver[:, :20]
    drafts[1] = ver[1, :x]
    check(hidden, w, drafts)
