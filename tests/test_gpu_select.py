"""GPU vc_select_kept against the oracle: key-norm scores bit-exact, kept
lists bit-exact (key-norm scores computed on the GPU, or seeded scores
passed in), ragged lengths, windows larger than the request, ties, the
70B-shaped workload's lists at full size, and the slot-count check."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import vc_harness as H

pytestmark = pytest.mark.gpu


def keep_counts(lens, sink, recent, keeps):
    out = []
    for n, k in zip(lens, keeps):
        s = min(sink, n)
        r = min(recent, n - s)
        out.append(s + r + max(0, min(n - s - r, k - s - r)))
    return out


def run(full, counts, sink, recent, scores=None, stride=None):
    import lossless_compressed_kv_gb300 as vc
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    idx = torch.full((max(1, int(offs[-1])),), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    if scores is None:
        ws = torch.empty(vc.select_workspace_bytes(full.batch, stride), dtype=torch.uint8, device="cuda")
    vc.select_kept(full, H.to_dev(offs), idx, sink, recent, scores=scores, score_stride=stride, workspace=ws,
                   status=st)
    torch.cuda.synchronize()
    return offs, idx.cpu().numpy(), int(st.item()), ws


@pytest.mark.parametrize("d,hkv,lens,sink,recent,frac", [
    (128, 8, [1000, 37, 4096, 1], 16, 64, 4),
    (64, 2, [300, 16, 17], 4, 8, 3),
    (128, 1, [5000], 64, 512, 4),
    (64, 4, [10, 3], 8, 8, 2),            # windows cover the whole request
])
def test_select_keynorm_matches_oracle(d, hkv, lens, sink, recent, frac):
    rng = np.random.default_rng(d + hkv + len(lens))
    full, hf = H.full_cache(rng, lens, hkv, d, synth.outlier_channels(rng, d, 2), 8.0)
    stride = max(lens)
    counts = keep_counts(lens, sink, recent, [max(1, n // frac) for n in lens])
    offs, got, st, ws = run(full, counts, sink, recent, stride=stride)
    assert st == 0
    sc = ws.view(torch.float32)[: len(lens) * stride].view(len(lens), stride).cpu().numpy()
    for b, n in enumerate(lens):
        k, _ = H.logical_full(hf, b)
        ref_s = oracle.keynorm_scores(k)
        assert np.array_equal(sc[b, :n].view(np.uint32), ref_s.view(np.uint32)), b
        ref = oracle.select_kept(ref_s, sink, recent, counts[b])
        assert np.array_equal(got[offs[b]:offs[b + 1]], ref), b


def test_select_seeded_scores_with_ties():
    rng = np.random.default_rng(5)
    lens = [3000, 1, 700, 2048]
    stride = 3072
    full, _ = H.full_cache(rng, lens, 1, 64)
    scores = (rng.integers(0, 5, (len(lens), stride)) * 0.5).astype(np.float32)   # heavy ties
    scores[0, 100:200] = -1.5                                                      # negatives order too
    counts = keep_counts(lens, 10, 20, [900, 1, 700, 100])
    offs, got, st, _ = run(full, counts, 10, 20, scores=H.to_dev(scores), stride=stride)
    assert st == 0
    for b, n in enumerate(lens):
        ref = oracle.select_kept(scores[b, :n], 10, 20, counts[b])
        assert np.array_equal(got[offs[b]:offs[b + 1]], ref), b


def test_select_70b_workload_lists_full_size():
    """The 70B-shaped workload: 4 x 131072 positions, 64 sink + 512 recent +
    the top of a seeded uniform score, 32768 kept -- the same lists as the
    workload generator."""
    w = synth.WORKLOADS["70b_128k_drop4"]
    B, n = w["batch"], w["ctx"]
    lens = [n] * B
    table, total = synth.block_tables(np.random.default_rng(0), np.array(lens))
    import lossless_compressed_kv_gb300 as vc
    dummy = torch.zeros((total, 16 * 2 * 8), dtype=torch.uint8, device="cuda")   # K pages unused
    full = vc.PagedKV(dummy, dummy, H.to_dev(table), H.to_dev(np.array(lens, np.int32)), 1, 8, 16)
    scores = np.zeros((B, n), np.float32)
    ref = []
    for b in range(B):
        rng = np.random.default_rng([99, b])
        ref.append(synth.kept_sink_recent_topk(rng, n, w["sink"], w["recent"], w["kept_total"]))
        rng = np.random.default_rng([99, b])
        scores[b, w["sink"]:n - w["recent"]] = rng.random(n - w["sink"] - w["recent"], dtype=np.float32)
    offs, got, st, _ = run(full, [w["kept_total"]] * B, w["sink"], w["recent"], scores=H.to_dev(scores),
                           stride=n)
    assert st == 0
    for b in range(B):
        assert np.array_equal(got[offs[b]:offs[b + 1]], ref[b]), b


def test_select_rejects_a_count_the_rule_cannot_fill():
    rng = np.random.default_rng(9)
    full, _ = H.full_cache(rng, [100, 50], 1, 64)
    scores = rng.random((2, 100), dtype=np.float32)
    # request 1 asks for 60 of 50 positions
    offs, got, st, _ = run(full, [30, 60], 4, 4, scores=H.to_dev(scores), stride=100)
    assert st == 1                          # VC_ERR_INVALID_ARG
    assert (got[offs[1]:offs[2]] == -7).all()   # nothing written for it
    ref = oracle.select_kept(scores[0], 4, 4, 30)
    assert np.array_equal(got[offs[0]:offs[1]], ref)
