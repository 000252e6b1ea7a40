"""GPU vc_accept_sampled against the oracle.  The logits are the same fp32
bits on both sides (checked); the softmax sums and the inverse CDF run in
fp32 on the GPU and fp64 in the oracle, so each request is compared
decision by decision up to its first decision whose margin (the oracle's
relative distance to flipping it) is below MARGIN -- ten times the typical
fp32 error of a 32000-term softmax sum.  With near-uniform 32000-way
distributions the inverse-CDF boundaries lie ~1/32000 apart, so most draws
there are marginal; the 2000-way cases compare whole rounds."""
import numpy as np
import pytest
import torch

import oracle
from tests import vc_harness as H

pytestmark = pytest.mark.gpu

# a decision is compared when the oracle's distance to flipping it is at
# least this (relative); the GPU's fp32 softmax and cumulative sums are
# typically within ~2e-6 of the fp64 values
MARGIN = 2e-5


def gpu_sampled(th, dh, w, drafts, u, v, tau, hg):
    import lossless_compressed_kv_gb300 as vc
    b, x = th.shape[0], th.shape[1] - 1
    d, vocab = w.shape
    al = torch.empty(b, dtype=torch.int32, device="cuda")
    em = torch.empty((b, x + 1), dtype=torch.int32, device="cuda")
    ws = torch.empty(vc.accept_sampled_workspace_bytes(b, x, vocab, d), dtype=torch.uint8, device="cuda")
    vc.accept_sampled(H.to_dev(th), H.to_dev(dh) if x else None, H.to_dev(w), H.to_dev(drafts) if x else None,
                      H.to_dev(u) if x else None, H.to_dev(v), tau, al, em, ws, hidden_group=hg)
    torch.cuda.synchronize()
    rt, rd = b * (x + 1), b * x
    lt = ws.view(torch.float32)[(rt + rd) * d:(rt + rd) * d + rt * vocab].view(rt, vocab).cpu().numpy()
    return al.cpu().numpy(), em.cpu().numpy(), lt


def compare(th, dh, w, drafts, u, v, tau, hg, al, em, lt):
    """Checks every decision up to each request's first marginal one;
    returns (decisions compared, decisions taken)."""
    b, x = th.shape[0], th.shape[1] - 1
    compared = total = 0
    for i in range(b):
        tl = oracle.logits(th[i], w)
        assert np.array_equal(lt[i * (x + 1):(i + 1) * (x + 1)].view(np.uint32), tl.view(np.uint32)), i
        dl = oracle.logits(dh[i], w) if x else np.zeros((0, w.shape[1]), np.float32)
        r = oracle.accept_sampled(tl, dl, drafts[i], u[i], v[i], tau)
        steps = r["accept_len"] + 1
        total += steps
        ok = 0
        for s in range(steps):
            if r["margins"][s] < MARGIN:
                break
            ok = s + 1
        compared += ok
        if ok == steps:
            assert al[i] == r["accept_len"], i
            assert np.array_equal(em[i], r["emitted"]), i
        else:
            # the first ok decisions were kept drafts: same ids, and the GPU
            # did not stop earlier
            assert al[i] >= ok, i
            assert np.array_equal(em[i][:ok], r["emitted"][:ok]), i
    return compared, total


@pytest.mark.parametrize("tau,noise,vocab", [(0.8, 0.02, 32000), (1.0, 0.2, 32000), (0.3, 0.05, 2000),
                                             (1.0, 0.3, 2000)])
def test_sampled_accept_matches_oracle(tau, noise, vocab):
    rng = np.random.default_rng(int(tau * 100) + int(noise * 1000) + vocab)
    B, x, hg, d = 8, 16, 4, 128
    w = (rng.standard_normal((d, vocab)) * 0.05).astype(np.float32)
    th = rng.standard_normal((B, x + 1, hg, d)).astype(np.float32)
    dh = (th[:, :x] + noise * rng.standard_normal((B, x, hg, d))).astype(np.float32)
    drafts = np.empty((B, x), np.int32)
    for i in range(B):           # drafts drawn from the draft distribution
        dl = oracle.logits(dh[i], w).astype(np.float64) / tau
        p = np.exp(dl - dl.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        drafts[i] = [rng.choice(vocab, p=p[j]) for j in range(x)]
    u = rng.random((B, x), dtype=np.float32)
    v = rng.random((B, x + 1), dtype=np.float32)
    al, em, lt = gpu_sampled(th, dh, w, drafts, u, v, tau, hg)
    compared, total = compare(th, dh, w, drafts, u, v, tau, hg, al, em, lt)
    assert compared >= total // 2, (compared, total)


def test_sampled_identical_distributions_keep_all_drafts():
    rng = np.random.default_rng(11)
    B, x, hg, d, vocab = 4, 8, 2, 64, 1000
    w = (rng.standard_normal((d, vocab)) * 0.05).astype(np.float32)
    th = rng.standard_normal((B, x + 1, hg, d)).astype(np.float32)
    dh = th[:, :x].copy()
    drafts = rng.integers(0, vocab, (B, x)).astype(np.int32)
    u = (rng.random((B, x), dtype=np.float32) * 0.99).astype(np.float32)
    v = rng.random((B, x + 1), dtype=np.float32)
    al, em, lt = gpu_sampled(th, dh, w, drafts, u, v, 0.9, hg)
    assert (al == x).all()
    assert np.array_equal(em[:, :x], drafts)
    compared, total = compare(th, dh, w, drafts, u, v, 0.9, hg, al, em, lt)
    assert compared >= total - B      # every kept draft; the bonus draws may be marginal


def test_sampled_bad_draft_id_is_rejected_and_x0_draws_bonus():
    rng = np.random.default_rng(12)
    B, x, d, vocab = 2, 3, 32, 100
    w = (rng.standard_normal((d, vocab)) * 0.1).astype(np.float32)
    th = rng.standard_normal((B, x + 1, 1, d)).astype(np.float32)
    dh = th[:, :x].copy()
    drafts = np.array([[5, 7, 9], [-1, 7, 9]], np.int32)
    u = np.full((B, x), 0.5, np.float32)
    v = rng.random((B, x + 1), dtype=np.float32)
    al, em, _ = gpu_sampled(th, dh, w, drafts, u, v, 1.0, 1)
    assert al[0] == 3 and al[1] == 0
    # x = 0: only the bonus draw
    al0, em0, lt0 = gpu_sampled(th[:, :1], dh[:, :0], w, np.zeros((B, 0), np.int32), np.zeros((B, 0), np.float32),
                                v[:, :1].copy(), 1.0, 1)
    assert (al0 == 0).all()
    for i in range(B):
        r = oracle.accept_sampled(oracle.logits(th[i, :1], w), np.zeros((0, vocab), np.float32),
                                  np.zeros(0, np.int32), np.zeros(0, np.float32), v[i, :1], 1.0)
        if r["margins"][0] >= MARGIN:
            assert em0[i, 0] == r["emitted"][0]
