"""Pins of the oracle's token selection ("VeriCache Guide", the compressor
class of "Implementing VeriCache in Python and PyTorch": key-norm importance
averaged over heads, the top tokens kept in position order), independent of
its own code: exact closed forms, a float64 reference within the fp32 error
bound, and a brute-force selection written a different way (lexsort)."""
import numpy as np
import pytest

import oracle
import synth


def test_keynorm_closed_forms():
    # constant rows: sum of squares c^2 * d exact, square root exact
    d, hkv = 64, 2
    x = np.empty((3, hkv, d), np.float32)
    x[0, 0], x[0, 1] = 1.0, 0.5          # norms 8 and 4 -> mean 6
    x[1, 0], x[1, 1] = 2.0, 2.0          # 16, 16 -> 16
    x[2, 0], x[2, 1] = 0.0, 0.25         # 0, 2 -> 1
    s = oracle.keynorm_scores(synth.bf16_bits(x))
    assert s.tolist() == [6.0, 16.0, 1.0]


def test_keynorm_matches_float64_within_fp32_bound():
    rng = np.random.default_rng(3)
    n, hkv, d = 50, 8, 128
    k = synth.normal_bf16(rng, (n, hkv, d), std=3.0)
    got = oracle.keynorm_scores(k).astype(np.float64)
    ref = np.linalg.norm(synth.bf16_to_f32(k).astype(np.float64), axis=-1).mean(axis=-1)
    # fp32 sum of d squares: relative error <= d*u; sqrt and the head mean add
    # a few more roundings
    assert np.all(np.abs(got - ref) <= (d + 8) * 2.0 ** -24 * ref)


def brute_select(score, sink, recent, keep):
    n = len(score)
    sink = min(sink, n)
    recent = min(recent, n - sink)
    mid = np.arange(sink, n - recent)
    top = max(0, min(len(mid), keep - sink - recent))
    order = np.lexsort((mid, -score[mid].astype(np.float64)))   # score desc, position asc
    keep_mid = mid[order[:top]]
    pos = np.concatenate([np.arange(sink), keep_mid, np.arange(n - recent, n)])
    return np.unique(pos).astype(np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 400))
    sink, recent = int(rng.integers(0, 20)), int(rng.integers(0, 40))
    keep = int(rng.integers(0, n + 10))
    # few distinct values: many ties
    score = (rng.integers(0, 7, n) * 0.125).astype(np.float32)
    got = oracle.select_kept(score, sink, recent, keep)
    assert np.array_equal(got, brute_select(score, sink, recent, keep))


def test_select_special_cases():
    s = np.arange(10, dtype=np.float32)[::-1].copy()      # decreasing: earlier = higher
    assert np.array_equal(oracle.select_kept(s, 0, 0, 100), np.arange(10))   # keep >= n: all
    assert np.array_equal(oracle.select_kept(s, 2, 3, 1), [0, 1, 7, 8, 9])   # keep below the windows
    assert np.array_equal(oracle.select_kept(s, 2, 3, 7), [0, 1, 2, 3, 7, 8, 9])
    assert np.array_equal(oracle.select_kept(np.ones(6, np.float32), 0, 0, 3), [0, 1, 2])  # ties -> lowest
    assert np.array_equal(oracle.select_kept(s, 20, 5, 3), np.arange(10))   # sink clamped to n


def test_select_agrees_with_the_workload_generator():
    """The 70B workload's kept list (sink + recent + top by a seeded score) is
    the oracle's selection over the same seeded scores."""
    rng = np.random.default_rng(12345)
    n, sink, recent, total = 5000, 64, 512, 1250
    idx = synth.kept_sink_recent_topk(rng, n, sink, recent, total)
    rng = np.random.default_rng(12345)
    score = np.zeros(n, np.float32)
    score[sink:n - recent] = rng.random(n - sink - recent, dtype=np.float32)
    assert np.array_equal(oracle.select_kept(score, sink, recent, total), idx)
