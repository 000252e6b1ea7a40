"""GPU vc_draft_step (append the step's new entry to KV_comp, then draft
attention, in one launch) against the two separate calls it replaces
(vc_compress appending the same rows at the same position, then
vc_draft_attn): KV_comp bytes and draft outputs bit-identical, step after
step, for every format, ragged lengths and slots at page boundaries; the
oracle on the final cache; an out-of-range slot is reported."""
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


def rows_at(hf, pos):
    """bf16 K / V rows of position pos[b] of every request: [B][Hkv][D]."""
    ks, vs = [], []
    for b, p in enumerate(pos):
        k, v = H.logical_full(hf, b, int(p) + 1)
        ks.append(k[p])
        vs.append(v[p])
    return np.stack(ks), np.stack(vs)


@pytest.mark.parametrize("bits,d,hkv,grp", [(2, 128, 2, 4), (3, 128, 2, 4), (4, 64, 1, 8), (16, 128, 2, 4),
                                            (2, 64, 2, 2), (16, 64, 1, 4)])
def test_draft_step_equals_append_then_draft(bits, d, hkv, grp):
    m = vc()
    rng = np.random.default_rng(bits * 10 + d + hkv)
    n0 = np.array([300, 15, 1000, 64], np.int64)        # prefixes (ragged, page-aligned 64)
    steps = 18                                           # crosses page boundaries
    B, hq = len(n0), hkv * grp
    full, hf = H.full_cache(rng, n0 + steps, hkv, d)
    cap = n0 + steps
    comp_a, ctable = H.comp_cache(rng, B, cap, hkv, d, bits)
    comp_b = m.PagedKV(comp_a.k_pages.clone(), comp_a.v_pages.clone(), comp_a.block_table,
                       torch.zeros(B, dtype=torch.int32, device="cuda"), hkv, d, bits)
    offs, idx = synth.csr([np.arange(n, dtype=np.int32) for n in n0])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c in (comp_a, comp_b):
        m.compress(full, H.to_dev(offs), H.to_dev(idx), c, int(n0.max()), status=st)
    scale = 1.0 / math.sqrt(d)
    msl = int(cap.max())
    ws = torch.empty(m.draft_workspace_bytes(comp_a, hq, msl), dtype=torch.uint8, device="cuda")
    for i in range(steps):
        pos = n0 + i
        lens = H.to_dev((pos + 1).astype(np.int32))
        qn = synth.normal_bf16(rng, (B, hq, d))
        q = H.to_dev(qn.view(np.int16)).view(torch.bfloat16)
        # a: append with vc_compress, then vc_draft_attn
        o1, i1 = synth.csr([np.array([p], np.int32) for p in pos])
        m.compress(full, H.to_dev(o1), H.to_dev(i1), comp_a, 1, comp_start=H.to_dev(pos.astype(np.int32)),
                   status=st)
        ca = m.PagedKV(comp_a.k_pages, comp_a.v_pages, comp_a.block_table, lens, hkv, d, bits)
        out_a = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
        m.draft_attn(q, ca, scale, out_a, msl, ws, status=st)
        # b: one vc_draft_step with the same rows
        kn, vn = rows_at(hf, pos)
        cb = m.PagedKV(comp_b.k_pages, comp_b.v_pages, comp_b.block_table, lens, hkv, d, bits)
        out_b = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
        m.draft_step(q, cb, H.to_dev(kn.view(np.int16)), H.to_dev(vn.view(np.int16)),
                     H.to_dev(pos.astype(np.int32)), scale, out_b, msl, ws, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert torch.equal(comp_a.k_pages, comp_b.k_pages), i
        assert torch.equal(comp_a.v_pages, comp_b.v_pages), i
        assert torch.equal(out_a, out_b), i
    # the final step's output against the oracle over the appended cache
    for b in range(B):
        k, v = H.logical_full(hf, b, int(n0[b] + steps))
        ref_comp = oracle.compress(k, v, np.arange(n0[b] + steps, dtype=np.int32), bits)
        ref = oracle.draft_attn(qn[b], ref_comp, float(np.float32(scale)))
        assert H.row_err(out_b[b].cpu().numpy(), ref) <= H.TOL


def test_draft_step_slot_out_of_range_is_reported():
    m = vc()
    rng = np.random.default_rng(3)
    d, hkv, hq, bits = 128, 1, 4, 2
    n0 = np.array([100, 40], np.int64)
    full, hf = H.full_cache(rng, n0 + 1, hkv, d)
    comp, _ = H.comp_cache(rng, 2, n0 + 1, hkv, d, bits, zero=True)
    before_k, before_v = comp.k_pages.clone(), comp.v_pages.clone()
    lens = H.to_dev(n0.astype(np.int32))             # slot == seq_len: outside the attended range
    c = m.PagedKV(comp.k_pages, comp.v_pages, comp.block_table, lens, hkv, d, bits)
    kn, vn = rows_at(hf, n0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(m.draft_workspace_bytes(c, hq, 101), dtype=torch.uint8, device="cuda")
    out = torch.empty((2, hq, d), dtype=torch.float32, device="cuda")
    q = torch.zeros((2, hq, d), dtype=torch.bfloat16, device="cuda")
    m.draft_step(q, c, H.to_dev(kn.view(np.int16)), H.to_dev(vn.view(np.int16)),
                 H.to_dev(n0.astype(np.int32)), 0.1, out, 101, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 1                             # VC_ERR_INVALID_ARG
    assert torch.equal(comp.k_pages, before_k) and torch.equal(comp.v_pages, before_v)
