"""GPU vc_compress against the oracle: bit-exact packed codes, fp16 scales
and zeros (and bf16 rows for the token-drop format), for ragged kept lists,
append offsets, several head dims / bit widths, the tiny workload and the
full 8B-shaped 32k workload."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import vc_harness as H

pytestmark = pytest.mark.gpu


def run_compress(full, comp, kept_lists, comp_start=None):
    import lossless_compressed_kv_gb300 as vc
    offs, idx = synth.csr(kept_lists)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs = None if comp_start is None else H.to_dev(np.asarray(comp_start, np.int32))
    vc.compress(full, H.to_dev(offs), H.to_dev(idx), comp, max(len(k) for k in kept_lists), comp_start=cs,
                status=st)
    torch.cuda.synchronize()
    return int(st.item())


def check(comp, ctable, hfull, kept_lists, bits, start=None):
    for b, kept in enumerate(kept_lists):
        k, v = H.logical_full(hfull, b)
        ref = oracle.compress(k, v, np.asarray(kept, np.int32), bits)
        s0 = 0 if start is None else int(start[b])
        got = H.read_comp_kv(comp, ctable, b, s0 + len(kept))
        got = {key: (val if key == "bits" else val[s0:]) for key, val in got.items()}
        for key in ref:
            if key != "bits":
                assert np.array_equal(got[key], ref[key]), (b, key)


SHAPES = [(bits, d) for bits in (2, 3, 4, 16) for d in (32, 64, 128, 256) if bits == 16 or d % 64 == 0]


@pytest.mark.parametrize("bits,d", SHAPES)
def test_compress_random_shapes(bits, d):
    rng = np.random.default_rng(100 + bits * 7 + d)
    lens = [37, 500, 16, 1]
    hkv = 2
    full, hf = H.full_cache(rng, lens, hkv, d, outliers=synth.outlier_channels(rng, d, 2), oscale=10.0)
    kept = [np.sort(rng.choice(n, size=max(1, n // 3), replace=False)).astype(np.int32) for n in lens]
    kept[1] = np.arange(500, dtype=np.int32)       # everything kept, several pages + ragged tail
    comp, ctable = H.comp_cache(rng, len(lens), [len(k) + 40 for k in kept], hkv, d, bits)
    assert run_compress(full, comp, kept) == 0
    check(comp, ctable, hf, kept, bits)


@pytest.mark.parametrize("bits,d", [(2, 128), (3, 128), (4, 128), (2, 64), (3, 64), (4, 64)])
def test_compress_append_offsets(bits, d):
    """Append mode: entries go to slots comp_start[b] + j (drafted tokens
    appended to an existing KV_comp); slots before comp_start are untouched."""
    rng = np.random.default_rng(7)
    lens, hkv = [70, 33], 3
    full, hf = H.full_cache(rng, lens, hkv, d)
    comp, ctable = H.comp_cache(rng, 2, 100, hkv, d, bits, zero=True)
    kept = [np.arange(60, 70, dtype=np.int32), np.arange(30, 33, dtype=np.int32)]
    start = [23, 50]
    assert run_compress(full, comp, kept, comp_start=start) == 0
    check(comp, ctable, hf, kept, bits, start=start)
    before = H.read_comp(comp.k_pages, ctable[0], 23, hkv, d, bits, "k")
    assert not before["packed"].any() and not before["scales"].any()
    vbefore = H.read_comp(comp.v_pages, ctable[0], 23, hkv, d, bits, "v")
    assert not vbefore["packed"].any() and not vbefore["zeros"].any()


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_compress_one_token_appends_match_bulk(bits):
    """Appending one token per call (the draft loop's path) builds the same
    bytes as compressing the whole range at once (the page-parallel path)."""
    rng = np.random.default_rng(11)
    lens, d, hkv = [45, 40], 128, 2
    full, hf = H.full_cache(rng, lens, hkv, d)
    kept = [np.arange(40, dtype=np.int32), np.arange(40, dtype=np.int32)]
    c1, t1 = H.comp_cache(rng, 2, 48, hkv, d, bits, zero=True)
    assert run_compress(full, c1, kept) == 0
    c2, _ = H.comp_cache(rng, 2, 48, hkv, d, bits, zero=True)
    import lossless_compressed_kv_gb300 as vc
    c2 = vc.PagedKV(c2.k_pages, c2.v_pages, c1.block_table, c2.seq_lens, hkv, d, bits)
    for i in range(40):
        assert run_compress(full, c2, [np.array([i], np.int32)] * 2, comp_start=[i, i]) == 0
    assert torch.equal(c1.k_pages, c2.k_pages) and torch.equal(c1.v_pages, c2.v_pages)


def test_compress_bad_indices_are_reported_and_skipped():
    rng = np.random.default_rng(8)
    full, hf = H.full_cache(rng, [40], 1, 64)
    comp, ctable = H.comp_cache(rng, 1, 64, 1, 64, 4, zero=True)
    kept = [np.array([0, 39, 40, 5], np.int32)]       # 40 >= seq_len
    assert run_compress(full, comp, kept) == 3        # VC_ERR_BAD_INDEX
    good = H.read_comp_kv(comp, ctable, 0, 4)
    k, v = H.logical_full(hf, 0)
    ref = oracle.compress(k, v, np.array([0, 39, 5], np.int32), 4)
    for key in ("k_packed", "k_scales", "v_zeros"):
        assert np.array_equal(good[key][[0, 1, 3]], ref[key])
        assert not good[key][2].any()                  # skipped entry never written


def test_compress_tiny_workload():
    w = synth.WORKLOADS["tiny"]
    rng = synth.rng_for("tiny")
    oc = synth.outlier_channels(rng, w["d"], w["outliers"])
    full, hf = H.full_cache(rng, [w["ctx"]], w["hkv"], w["d"], oc, w["outlier_scale"])
    kept = [synth.kept_sink_recent_random(rng, w["ctx"], w["sink"], w["recent"], w["n_random"])]
    assert len(kept[0]) == 128
    comp, ctable = H.comp_cache(rng, 1, 128 + 16, w["hkv"], w["d"], w["bits"])
    assert run_compress(full, comp, kept) == 0
    check(comp, ctable, hf, kept, w["bits"])


def test_compress_8b_32k_full_size():
    """The 8B-shaped workload at full size (8 x 32768 tokens x 8 kv heads,
    every token kept, 2-bit): every entry bit-exact."""
    w = synth.WORKLOADS["8b_32k_2bit"]
    rng = synth.rng_for("8b_32k_2bit")
    oc = synth.outlier_channels(rng, w["d"], w["outliers"])
    lens = [w["ctx"]] * w["batch"]
    full, hf = H.full_cache(rng, lens, w["hkv"], w["d"], oc, w["outlier_scale"])
    kept = [np.arange(w["ctx"], dtype=np.int32)] * w["batch"]
    comp, ctable = H.comp_cache(rng, w["batch"], w["ctx"], w["hkv"], w["d"], w["bits"])
    assert run_compress(full, comp, kept) == 0
    check(comp, ctable, hf, kept, w["bits"])


@pytest.mark.parametrize("bits,d", [(2, 128), (3, 128), (4, 128), (3, 64), (2, 256)])
def test_gpu_page_read_through_the_exported_helpers(bits, d):
    """A C caller's view of KV_comp: head blocks written by vc_compress on
    the GPU, copied to the host and converted by vc_comp_block_decode (no
    test-side layout code), equal the oracle's packed little-endian codes,
    scales and zeros byte for byte."""
    import lossless_compressed_kv_gb300 as vc
    rng = np.random.default_rng(900 + bits + d)
    hkv, n = 2, 16 * 5 + 7
    full, hf = H.full_cache(rng, [n], hkv, d, outliers=synth.outlier_channels(rng, d, 2), oscale=10.0)
    kept = [np.arange(n, dtype=np.int32)]
    comp, ctable = H.comp_cache(rng, 1, n, hkv, d, bits)
    assert run_compress(full, comp, kept) == 0
    k, v = H.logical_full(hf, 0)
    ref = oracle.compress(k, v, kept[0], bits)
    hb = vc.head_block_bytes(d, bits)
    pools = {"k": comp.k_pages.cpu().numpy().reshape(-1, hkv, hb), "v": comp.v_pages.cpu().numpy().reshape(-1, hkv, hb)}
    for kind in ("k", "v"):
        for p in range((n + 15) // 16):
            for h in range(hkv):
                codes, sc, ze = vc.comp_block_decode(pools[kind][ctable[0][p], h], d, bits, kind)
                s = np.arange(16 * p, min(n, 16 * p + 16))
                m = len(s)
                assert np.array_equal(codes[:m], ref[kind + "_packed"][s, h]), (kind, p, h)
                assert np.array_equal(sc[:m], ref[kind + "_scales"][s, h]), (kind, p, h)
                assert np.array_equal(ze[:m], ref[kind + "_zeros"][s, h]), (kind, p, h)
