"""GPU vc_draft_attn / vc_verify_attn / vc_mixed_attn against the oracle.

Tolerance (attention outputs, fp32 accumulation over bf16 / dequantised
inputs): per output row max_i |o_gpu - o_ref| <= 2e-3 * ||o_ref||_2.
Shapes span several pages, context chunks and a ragged tail; the edge cases
are a single token, an exact page, an empty request and every GQA group
size up to 8.  The full-size workloads are checked on every draft row and on
sampled verification rows."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import vc_harness as H

pytestmark = pytest.mark.gpu


def vc():
    import lossless_compressed_kv_gb300 as m
    return m


def compress_all(full, comp, kept_lists):
    offs, idx = synth.csr(kept_lists)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    vc().compress(full, H.to_dev(offs), H.to_dev(idx), comp, max(1, max(len(k) for k in kept_lists)), status=st)
    comp.seq_lens.copy_(torch.tensor([len(k) for k in kept_lists], dtype=torch.int32))
    torch.cuda.synchronize()
    assert st.item() == 0


def gpu_draft(comp, q, scale, max_len):
    m = vc()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, m.draft_workspace_bytes(comp, q.shape[1], max_len)), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.draft_attn(q, comp, scale, out, max_len, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out.cpu().numpy()


def gpu_verify(full, q, scale, max_len):
    m = vc()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, m.verify_workspace_bytes(full, q.shape[1], q.shape[2], max_len)), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.verify_attn(q, full, scale, out, max_len, ws, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


def q_bf16(rng, shape):
    qn = synth.normal_bf16(rng, shape)
    return qn, H.to_dev(qn.view(np.int16)).view(torch.bfloat16)


# --------------------------------------------------------------- draft

DRAFT_CASES = [
    # bits, d, hkv, grp, lens
    (2, 128, 2, 4, [1, 16, 17, 700, 5000]),
    (3, 128, 2, 4, [33, 4097]),
    (4, 128, 1, 8, [300, 64]),
    (16, 128, 2, 8, [2100, 15]),
    (2, 64, 3, 1, [90, 1000]),
    (3, 64, 1, 2, [129]),
    (4, 64, 2, 4, [1, 2, 3]),
    (16, 64, 1, 4, [513, 31]),
    (2, 128, 1, 8, [3000, 47]),          # 2-bit with the full 8-head group
    (3, 128, 4, 3, [1500, 16]),          # an odd group size
]


@pytest.mark.parametrize("bits,d,hkv,grp,lens", DRAFT_CASES)
def test_draft_matches_oracle(bits, d, hkv, grp, lens):
    rng = np.random.default_rng(bits * 1000 + d + hkv * 10 + grp)
    full, hf = H.full_cache(rng, lens, hkv, d, synth.outlier_channels(rng, d, 2), 8.0)
    kept = [np.arange(n, dtype=np.int32) if n < 100 else
            np.sort(rng.choice(n, size=n // 2, replace=False)).astype(np.int32) for n in lens]
    comp, ctable = H.comp_cache(rng, len(lens), [len(k) for k in kept], hkv, d, bits)
    compress_all(full, comp, kept)
    hq = hkv * grp
    qn, qd = q_bf16(rng, (len(lens), hq, d))
    scale = 1.0 / math.sqrt(d)
    got = gpu_draft(comp, qd, scale, max(len(k) for k in kept))
    for b in range(len(lens)):
        k, v = H.logical_full(hf, b)
        ref = oracle.draft_attn(qn[b], oracle.compress(k, v, kept[b], bits), float(np.float32(scale)))
        assert H.row_err(got[b], ref) <= H.TOL, (b, H.row_err(got[b], ref))


@pytest.mark.parametrize("bits", [2, 3, 4, 16])
@pytest.mark.parametrize("qstd", [1.0 / 64, 64.0, 1024.0])
def test_draft_query_range(bits, qstd):
    """Queries far from N(0, 1): rotary-embedded queries of real models reach
    tens to hundreds, and small ones lose bits in narrow formats.  q ~
    N(0, qstd^2) with 4 K outlier channels x10 against the oracle: the
    quantised path carries q in f16 operands pre-scaled per register, so the
    small end tests its subnormal range and the large end its overflow
    headroom (|q| up to several thousand at qstd 1024)."""
    rng = np.random.default_rng(int(qstd * 64) + bits)
    d, hkv, grp = 128, 2, 4
    lens = [3000, 17, 700]
    full, hf = H.full_cache(rng, lens, hkv, d, synth.outlier_channels(rng, d, 4), 10.0)
    kept = [np.arange(n, dtype=np.int32) for n in lens]
    comp, _ = H.comp_cache(rng, len(lens), lens, hkv, d, bits)
    compress_all(full, comp, kept)
    qn = synth.normal_bf16(rng, (len(lens), hkv * grp, d), std=qstd)
    qd = H.to_dev(qn.view(np.int16)).view(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    got = gpu_draft(comp, qd, scale, max(lens))
    assert np.isfinite(got).all()
    for b in range(len(lens)):
        k, v = H.logical_full(hf, b)
        ref = oracle.draft_attn(qn[b], oracle.compress(k, v, kept[b], bits), float(np.float32(scale)))
        assert H.row_err(got[b], ref) <= H.TOL, (b, H.row_err(got[b], ref))


def test_draft_empty_request_gives_zeros():
    rng = np.random.default_rng(5)
    full, hf = H.full_cache(rng, [40, 40], 1, 64)
    comp, _ = H.comp_cache(rng, 2, 64, 1, 64, 4)
    compress_all(full, comp, [np.arange(40, dtype=np.int32), np.zeros(0, np.int32)])
    qn, qd = q_bf16(rng, (2, 4, 64))
    got = gpu_draft(comp, qd, 0.125, 40)
    assert np.all(got[1] == 0) and np.all(np.isfinite(got[0]))


def test_empty_batch_through_the_binding():
    """Batch 0 with zero-size tensors (null data pointers): every call is a
    no-op that returns VC_OK and leaves the status word and the pools alone."""
    m = vc()
    rng = np.random.default_rng(9)
    d, hkv, hq = 128, 2, 8
    full, _ = H.full_cache(rng, [40], hkv, d)
    comp, _ = H.comp_cache(rng, 1, 64, hkv, d, 3)
    k0, v0 = comp.k_pages.clone(), comp.v_pages.clone()
    bt = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    ln = torch.zeros(0, dtype=torch.int32, device="cuda")
    c0 = m.PagedKV(comp.k_pages, comp.v_pages, bt, ln, hkv, d, 3)
    f0 = m.PagedKV(full.k_pages, full.v_pages, bt, ln, hkv, d, 16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = lambda *shape, dt=torch.float32: torch.empty(shape, dtype=dt, device="cuda")
    m.draft_attn(e(0, hq, d, dt=torch.bfloat16), c0, 0.1, e(0, hq, d), 64, e(0, dt=torch.uint8), status=st)
    m.draft_step(e(0, hq, d, dt=torch.bfloat16), c0, e(0, hkv, d, dt=torch.int16), e(0, hkv, d, dt=torch.int16),
                 e(0, dt=torch.int32), 0.1, e(0, hq, d), 64, e(0, dt=torch.uint8), status=st)
    m.verify_attn(e(0, 9, hq, d, dt=torch.bfloat16), f0, 0.1, e(0, 9, hq, d), 64, e(0, dt=torch.uint8), status=st)
    m.compress(f0, torch.zeros(1, dtype=torch.int32, device="cuda"), e(0, dt=torch.int32), c0, 0, status=st)
    m.mixed_attn(e(0, dt=torch.int32), e(0, hq, d, dt=torch.bfloat16), c0, e(0, hq, d),
                 e(0, 9, hq, d, dt=torch.bfloat16), f0, e(0, 9, hq, d), 0.1, 64, e(0, dt=torch.uint8), status=st)
    lm = torch.zeros((d, 1000), dtype=torch.float32, device="cuda")
    m.accept(e(0, 9, hq, d), lm, e(0, 8, dt=torch.int32), e(0, 9, dt=torch.int32), e(0, dt=torch.int32),
             e(0, 9, dt=torch.int32), e(0, dt=torch.uint8), hidden_group=hq)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(comp.k_pages, k0) and torch.equal(comp.v_pages, v0)


@pytest.mark.parametrize("bits,n,bad_page", [(2, 64, 2), (2, 60, 3), (3, 200, 0), (16, 60, 3)])
def test_draft_bad_page_id_reported(bits, n, bad_page):
    """An out-of-range block-table entry (a full page in the middle, the
    ragged last page, the first page) is reported; the request's output
    stays finite and the other request's rows match the oracle."""
    rng = np.random.default_rng(6 + bits + n)
    lens = [n, 90]
    full, hf = H.full_cache(rng, lens, 1, 64)
    comp, ctable = H.comp_cache(rng, 2, lens, 1, 64, bits)
    kept = [np.arange(k, dtype=np.int32) for k in lens]
    compress_all(full, comp, kept)
    bt = comp.block_table.clone()
    bt[0, bad_page] = comp.num_pages + 5                # out of range: reported, never read
    bad = vc().PagedKV(comp.k_pages, comp.v_pages, bt, comp.seq_lens, 1, 64, bits)
    qn, qd = q_bf16(rng, (2, 4, 64))
    m = vc()
    out = torch.empty((2, 4, 64), dtype=torch.float32, device="cuda")
    ws = torch.empty(m.draft_workspace_bytes(bad, 4, max(lens)), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.draft_attn(qd, bad, 0.125, out, max(lens), ws, status=st)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert st.item() == 3 and np.isfinite(got).all()
    k, v = H.logical_full(hf, 1)
    ref = oracle.draft_attn(qn[1], oracle.compress(k, v, kept[1], bits), float(np.float32(0.125)))
    assert H.row_err(got[1], ref) <= H.TOL


def test_draft_tiny_workload():
    w = synth.WORKLOADS["tiny"]
    rng = synth.rng_for("tiny")
    oc = synth.outlier_channels(rng, w["d"], w["outliers"])
    full, hf = H.full_cache(rng, [w["ctx"]], w["hkv"], w["d"], oc, w["outlier_scale"])
    kept = [synth.kept_sink_recent_random(rng, w["ctx"], w["sink"], w["recent"], w["n_random"])]
    comp, _ = H.comp_cache(rng, 1, 128, w["hkv"], w["d"], w["bits"])
    compress_all(full, comp, kept)
    qn, qd = q_bf16(rng, (1, w["hq"], w["d"]))
    scale = 1.0 / math.sqrt(w["d"])
    got = gpu_draft(comp, qd, scale, 128)
    k, v = H.logical_full(hf, 0)
    ref = oracle.draft_attn(qn[0], oracle.compress(k, v, kept[0], w["bits"]), float(np.float32(scale)))
    assert H.row_err(got[0], ref) <= H.TOL


@pytest.mark.parametrize("name", ["8b_32k_2bit", "70b_128k_drop4"])
def test_draft_full_size_workloads(name):
    """Every row of the full-size workloads (the launch configuration the
    benchmark times), against the oracle over the same KV_comp."""
    from concurrent.futures import ThreadPoolExecutor
    w = synth.WORKLOADS[name]
    rng = synth.rng_for(name)
    oc = synth.outlier_channels(rng, w["d"], w["outliers"]) if w["outliers"] else ()
    lens = [w["ctx"]] * w["batch"]
    full, hf = H.full_cache(rng, lens, w["hkv"], w["d"], oc, w["outlier_scale"])
    if w["bits"] == 16:
        kept = [synth.kept_sink_recent_topk(rng, w["ctx"], w["sink"], w["recent"], w["kept_total"])
                for _ in lens]
    else:
        kept = [np.arange(w["ctx"], dtype=np.int32)] * w["batch"]
    comp, _ = H.comp_cache(rng, w["batch"], len(kept[0]), w["hkv"], w["d"], w["bits"])
    compress_all(full, comp, kept)
    qn, qd = q_bf16(rng, (w["batch"], w["hq"], w["d"]))
    scale = 1.0 / math.sqrt(w["d"])
    got = gpu_draft(comp, qd, scale, len(kept[0]))
    del full, comp
    with ThreadPoolExecutor(oracle.threads()) as pool:
        for b in range(w["batch"]):
            k, v = H.logical_full(hf, b)
            ref = oracle.draft_attn(qn[b], oracle.compress(k, v, kept[b], w["bits"]), float(np.float32(scale)),
                                    pool=pool)
            assert H.row_err(got[b], ref) <= H.TOL, (b, H.row_err(got[b], ref))


@pytest.mark.parametrize("name", ["8b_32k_2bit", "70b_128k_drop4"])
def test_draft_step_full_size_workloads(name):
    """The call the benchmark's round makes (vc_draft_step: append the step's
    entry at slot ctx, then attend) at full size, every row against the
    oracle over the cache with that entry."""
    from concurrent.futures import ThreadPoolExecutor
    m = vc()
    w = synth.WORKLOADS[name]
    rng = synth.rng_for(name, 5)
    n = w["ctx"]
    lens = [n + 1] * w["batch"]
    full, hf = H.full_cache(rng, lens, w["hkv"], w["d"])
    if w["bits"] == 16:
        kept = [synth.kept_sink_recent_topk(rng, n, w["sink"], w["recent"], w["kept_total"]) for _ in lens]
    else:
        kept = [np.arange(n, dtype=np.int32)] * w["batch"]
    cap = len(kept[0]) + 1
    comp, _ = H.comp_cache(rng, w["batch"], cap, w["hkv"], w["d"], w["bits"])
    compress_all(full, comp, kept)
    slot = np.full(w["batch"], len(kept[0]), np.int32)
    kvn = [H.logical_full(hf, b) for b in range(w["batch"])]
    kn = np.stack([k[n] for k, _ in kvn])
    vn = np.stack([v[n] for _, v in kvn])
    lens_c = H.to_dev(slot + 1)
    c = m.PagedKV(comp.k_pages, comp.v_pages, comp.block_table, lens_c, w["hkv"], w["d"], w["bits"])
    qn, qd = q_bf16(rng, (w["batch"], w["hq"], w["d"]))
    scale = 1.0 / math.sqrt(w["d"])
    out = torch.empty((w["batch"], w["hq"], w["d"]), dtype=torch.float32, device="cuda")
    ws = torch.empty(m.draft_workspace_bytes(c, w["hq"], cap), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.draft_step(qd, c, H.to_dev(kn.view(np.int16)), H.to_dev(vn.view(np.int16)), H.to_dev(slot), scale, out, cap,
                 ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = out.cpu().numpy()
    del full, comp
    with ThreadPoolExecutor(oracle.threads()) as pool:
        for b in range(w["batch"]):
            k, v = kvn[b]
            kb = np.concatenate([kept[b], np.array([n], np.int32)])
            ref = oracle.draft_attn(qn[b], oracle.compress(k, v, kb, w["bits"]), float(np.float32(scale)), pool=pool)
            assert H.row_err(got[b], ref) <= H.TOL, (b, H.row_err(got[b], ref))


# --------------------------------------------------------------- verify

VERIFY_CASES = [
    # d, hkv, grp, n_q, lens
    (128, 2, 4, 8, [8, 9, 100, 4200]),
    (128, 1, 8, 40, [40, 41, 1300]),
    (128, 2, 4, 25, [25, 8193]),
    (64, 1, 4, 9, [512, 9, 16]),
    (64, 2, 2, 1, [1, 17, 3648, 3649, 4097]),   # a split ends after 3648 keys
    (128, 3, 1, 33, [700]),
    (64, 1, 8, 64, [64, 200]),
    (128, 2, 4, 40, [40, 4200, 8200]),   # 160 rows: two 128-row tiles
    (64, 1, 8, 24, [24, 700]),           # 192 rows: two tiles, head_dim 64
    # a one-tile last row block behind two-tile blocks runs as a second
    # launch of one-tile CTAs: 256 + 128, 256 + 94 and (head_dim 64) 256 + 24 rows
    (128, 1, 8, 48, [48, 4300]),
    (128, 2, 7, 50, [50, 51, 2000]),
    (64, 2, 5, 56, [56, 5000]),
    (128, 1, 8, 64, [64, 3000]),         # the largest block: 64 queries x 8 heads = 512 rows
]


@pytest.mark.parametrize("d,hkv,grp,n_q,lens", VERIFY_CASES)
def test_verify_matches_oracle(d, hkv, grp, n_q, lens):
    rng = np.random.default_rng(d + hkv * 3 + grp * 17 + n_q)
    full, hf = H.full_cache(rng, lens, hkv, d, synth.outlier_channels(rng, d, 2), 8.0)
    hq = hkv * grp
    qn, qd = q_bf16(rng, (len(lens), n_q, hq, d))
    scale = 1.0 / math.sqrt(d)
    got, st = gpu_verify(full, qd, scale, max(lens))
    assert st == 0
    for b in range(len(lens)):
        k, v = H.logical_full(hf, b)
        ref = oracle.verify_attn_block(qn[b], k, v, float(np.float32(scale)))
        assert H.row_err(got[b], ref) <= H.TOL, (b, H.row_err(got[b], ref))


def test_verify_short_request_reports_bad_index():
    rng = np.random.default_rng(3)
    full, hf = H.full_cache(rng, [4, 30], 1, 64)
    qn, qd = q_bf16(rng, (2, 8, 4, 64))
    got, st = gpu_verify(full, qd, 0.125, 30)
    assert st == 3 and np.all(got[0] == 0) and np.all(np.isfinite(got[1]))


@pytest.mark.parametrize("grp,n_q,rows_i", [(4, 33, (0, 7, 32)), (8, 40, (0, 31, 32, 39)),
                                             (7, 50, (0, 36, 37, 49))])
def test_verify_rows_invariant_to_block_and_batch(grp, n_q, rows_i):
    """A query's output is the same bits whether it is verified alone (n_q =
    1, batch 1, one 128-row tile) or as row i of a block of n_q in a batch of
    3 (two tiles; with grp 8 and 40 queries 320 rows, so queries 32.. sit in
    a one-tile row block of a second launch; with grp 7 and 50 queries,
    query 36 straddles the two launches):
    split boundaries are fixed by position and rows are independent."""
    rng = np.random.default_rng(11 + grp)
    d, hkv = 128, 2
    lens = [5000, 9000, 333]
    full, hf = H.full_cache(rng, lens, hkv, d)
    qn, qd = q_bf16(rng, (3, n_q, hkv * grp, d))
    blk, _ = gpu_verify(full, qd, 0.088, max(lens))
    m = vc()
    for i in rows_i:
        # request 1 alone, truncated so that query i is the last position
        L = lens[1] - n_q + i + 1
        one = m.PagedKV(full.k_pages, full.v_pages, full.block_table[1:2].contiguous(),
                        torch.tensor([L], dtype=torch.int32, device="cuda"), hkv, d, 16)
        alone, st = gpu_verify(one, qd[1:2, i:i + 1].contiguous(), 0.088, L)
        assert st == 0
        assert np.array_equal(alone[0, 0], blk[1, i])


@pytest.mark.parametrize("name,n_q", [("8b_32k_2bit", 32), ("8b_32k_2bit", 33), ("70b_128k_drop4", 40)])
def test_verify_full_size_sampled(name, n_q):
    """Full-size verification in the benchmark's launch configuration; 48
    seeded (request, query, head) rows are recomputed one by one."""
    from concurrent.futures import ThreadPoolExecutor
    w = synth.WORKLOADS[name]
    rng = synth.rng_for(name, 1)
    lens = [w["ctx"] + n_q] * w["batch"]
    full, hf = H.full_cache(rng, lens, w["hkv"], w["d"])
    qn, qd = q_bf16(rng, (w["batch"], n_q, w["hq"], w["d"]))
    scale = 1.0 / math.sqrt(w["d"])
    got, st = gpu_verify(full, qd, scale, max(lens))
    assert st == 0
    del full
    samp = np.random.default_rng(0)
    with ThreadPoolExecutor(oracle.threads()) as pool:
        for b in range(w["batch"]):
            k, v = H.logical_full(hf, b)
            qs = sorted(set([0, n_q - 1] + list(samp.integers(0, n_q, 2))))
            hs = sorted(set(samp.integers(0, w["hq"], 3)))
            ref = oracle.verify_attn(qn[b], k, v, float(np.float32(scale)), heads=hs, queries=qs, pool=pool)
            for i in qs:
                for h in hs:
                    e = H.row_err(got[b, i, h], ref[i, h])
                    assert e <= H.TOL, (b, i, h, e)


# --------------------------------------------------------------- mixed

@pytest.mark.parametrize("bits,d,grp", [(3, 128, 4), (2, 128, 8), (4, 64, 4), (16, 128, 4), (2, 64, 2), (16, 64, 8)])
def test_mixed_launch_matches_oracle_and_standalone(bits, d, grp):
    """Staggered batch: even requests draft over KV_comp, odd requests
    verify x = 25 over KV_full, in one launch (every code width and head
    size the launch instantiates).  Draft and verify rows match the oracle;
    verify rows are also bit-identical to the standalone verification
    kernel."""
    rng = np.random.default_rng(44 + bits + d + grp)
    hkv, n_q = 2, 25
    lens = [3000, 2100, 700, 4500, 1234, 90]
    role = np.array([b % 2 for b in range(len(lens))], np.int32)
    full, hf = H.full_cache(rng, lens, hkv, d)
    kept = [np.arange(n, dtype=np.int32) for n in lens]
    comp, _ = H.comp_cache(rng, len(lens), lens, hkv, d, bits)
    compress_all(full, comp, kept)
    hq = hkv * grp
    qdn, qdd = q_bf16(rng, (len(lens), hq, d))
    qvn, qvd = q_bf16(rng, (len(lens), n_q, hq, d))
    scale = 1.0 / math.sqrt(d)
    m = vc()
    od = torch.full((len(lens), hq, d), 7.0, device="cuda")
    ov = torch.full((len(lens), n_q, hq, d), 7.0, device="cuda")
    ws = torch.empty(m.mixed_workspace_bytes(comp, full, n_q, hq, max(lens)), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.mixed_attn(H.to_dev(role), qdd, comp, od, qvd, full, ov, scale, max(lens), ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    od, ov = od.cpu().numpy(), ov.cpu().numpy()
    alone, _ = gpu_verify(full, qvd, scale, max(lens))
    for b in range(len(lens)):
        if role[b] == 0:
            k, v = H.logical_full(hf, b)
            ref = oracle.draft_attn(qdn[b], oracle.compress(k, v, kept[b], bits), float(np.float32(scale)))
            assert H.row_err(od[b], ref) <= H.TOL
            assert np.all(ov[b] == 7.0)           # other role's buffer untouched
        else:
            k, v = H.logical_full(hf, b)
            ref = oracle.verify_attn_block(qvn[b], k, v, float(np.float32(scale)))
            assert H.row_err(ov[b], ref) <= H.TOL
            assert np.array_equal(ov[b], alone[b])
            assert np.all(od[b] == 7.0)


def test_mixed_launch_full_size_workload():
    """The staggered mixed workload at its stated size, in one vc_mixed_attn
    call: 32 requests with contexts drawn uniformly from [8192, 65536], 32
    query / 8 kv heads, head_dim 128, 3-bit group-32 KV_comp; even requests
    draft, odd requests verify a block of x = 25 over KV_full.  Every draft
    row is checked against the oracle over the same KV_comp, and 4 seeded
    (query, head) rows of each verifying request (64 rows) against the
    oracle's causal attention over KV_full."""
    from concurrent.futures import ThreadPoolExecutor
    w = synth.WORKLOADS["mixed_32req_3bit"]
    B, hq, hkv, d, x, bits = w["batch"], w["hq"], w["hkv"], w["d"], w["x"], w["bits"]
    rng = synth.rng_for("mixed_32req_3bit", 1)
    ctx = rng.integers(w["ctx_lo"], w["ctx_hi"] + 1, size=B).astype(np.int64)
    role = np.array([b % 2 for b in range(B)], np.int32)
    full_lens = [int(n) + x for n in ctx]            # a verifying request holds its block too
    full, hf = H.full_cache(rng, full_lens, hkv, d)
    kept = [np.arange(int(n), dtype=np.int32) for n in ctx]
    comp, _ = H.comp_cache(rng, B, [len(k) for k in kept], hkv, d, bits)
    compress_all(full, comp, kept)
    qdn, qdd = q_bf16(rng, (B, hq, d))
    qvn, qvd = q_bf16(rng, (B, x, hq, d))
    scale = 1.0 / math.sqrt(d)
    m = vc()
    msl = max(full_lens)
    od = torch.full((B, hq, d), 7.0, device="cuda")
    ov = torch.full((B, x, hq, d), 7.0, device="cuda")
    ws = torch.empty(m.mixed_workspace_bytes(comp, full, x, hq, msl), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.mixed_attn(H.to_dev(role), qdd, comp, od, qvd, full, ov, scale, msl, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    od, ov = od.cpu().numpy(), ov.cpu().numpy()
    del full, comp, ws
    samp = np.random.default_rng(2)
    sc = float(np.float32(scale))
    with ThreadPoolExecutor(oracle.threads()) as pool:
        for b in range(B):
            k, v = H.logical_full(hf, b)
            if role[b] == 0:
                ref = oracle.draft_attn(qdn[b], oracle.compress(k[:ctx[b]], v[:ctx[b]], kept[b], bits), sc,
                                        pool=pool)
                assert H.row_err(od[b], ref) <= H.TOL, (b, H.row_err(od[b], ref))
                assert np.all(ov[b] == 7.0)
            else:
                qs = [0, x - 1] + [int(i) for i in samp.integers(1, x - 1, 2)]
                hs = [int(h) for h in samp.integers(0, hq, 4)]
                rows = list(zip(qs, hs))
                ref = oracle.verify_attn(qvn[b], k, v, sc, heads=sorted(set(hs)), queries=sorted(set(qs)),
                                         pool=pool)
                for i, h in rows:
                    e = H.row_err(ov[b, i, h], ref[i, h])
                    assert e <= H.TOL, (b, i, h, e)
                assert np.all(od[b] == 7.0)


@pytest.mark.parametrize("bits,n_q", [(2, 9), (16, 9), (2, 40)])
def test_garbage_past_the_end_never_leaks(bits, n_q):
    """Slots past a request's length may hold any bytes (memory reused from
    earlier work): fill them with NaN bit patterns and check that draft and
    verification outputs stay finite and match the oracle (n_q 40: two
    128-row tiles, each with its own MMA warp)."""
    rng = np.random.default_rng(77)
    d, hkv, grp = 128, 2, 4
    lens = [max(37, n_q), 100, 16 * 9 + 3]
    full, hf = H.full_cache(rng, lens, hkv, d)
    # poison every slot of the last page past each request's length
    for b, n in enumerate(lens):
        page = int(hf["table"][b][(n - 1) // 16])
        for pool in (full.k_pages, full.v_pages):
            blk = pool[page].view(torch.int16).view(hkv, 16, d)
            blk[:, n % 16 or 16:, :] = -1          # 0xFFFF = bf16 NaN
    qn, qd = q_bf16(rng, (len(lens), n_q, hkv * grp, d))
    got, st = gpu_verify(full, qd, 0.088, max(lens))
    assert st == 0 and np.isfinite(got).all()
    for b in range(len(lens)):
        k, v = H.logical_full(hf, b)
        ref = oracle.verify_attn_block(qn[b], k, v, float(np.float32(0.088)))
        assert H.row_err(got[b], ref) <= H.TOL
    kept = [np.arange(n, dtype=np.int32) for n in lens]
    comp, ctable = H.comp_cache(rng, len(lens), lens, hkv, d, bits)
    compress_all(full, comp, kept)
    for b, n in enumerate(lens):                    # poison KV_comp tails too
        if n % 16:
            page = int(ctable[b][(n - 1) // 16])
            comp.k_pages[page].fill_(255)
            comp.v_pages[page].fill_(255)
    # re-write the valid slots of the poisoned pages, leaving the tails poisoned
    compress_all(full, comp, kept)
    qdn, qdd = q_bf16(rng, (len(lens), hkv * grp, d))
    gd = gpu_draft(comp, qdd, 0.088, max(lens))
    assert np.isfinite(gd).all()
    for b in range(len(lens)):
        k, v = H.logical_full(hf, b)
        ref = oracle.draft_attn(qdn[b], oracle.compress(k, v, kept[b], bits), float(np.float32(0.088)))
        assert H.row_err(gd[b], ref) <= H.TOL
