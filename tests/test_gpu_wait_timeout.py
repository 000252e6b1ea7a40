"""The bounded device waits, made to run out on purpose (host-side fault
injection, no GPU fault): with vc_debug_set_wait_fault(limit, skip_copies)
the draft, draft-step, verification and mixed kernels issue none of their
KV page copies, so each wait on a copy can only reach its limit.  Each call
must then report VC_ERR_TIMEOUT in its status word, give finite (zero)
outputs, leave no copy in flight and no TMEM allocated (the verification
kernel's warps leave their waits one after another and still free TMEM
together), and the next call with the switch off must be exact again."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import vc_harness as H

pytestmark = pytest.mark.gpu

TIMEOUT = 6
LIMIT_NS = 20_000          # 20 us per wait


def vc():
    import lossless_compressed_kv_gb300 as m
    return m


@pytest.fixture
def fault():
    m = vc()
    yield m.debug_set_wait_fault
    m.debug_set_wait_fault(0, False)


def _caches(rng, lens, hkv=2, d=128, bits=2):
    full, hf = H.full_cache(rng, lens, hkv, d)
    kept = [np.arange(n, dtype=np.int32) for n in lens]
    comp, _ = H.comp_cache(rng, len(lens), lens, hkv, d, bits)
    offs, idx = synth.csr(kept)
    vc().compress(full, H.to_dev(offs), H.to_dev(idx), comp, max(lens))
    comp.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
    return full, hf, comp, kept


def test_waits_time_out_and_the_next_call_is_clean(fault):
    m = vc()
    rng = np.random.default_rng(31)
    d, hkv, grp, n_q, bits = 128, 2, 4, 40, 2
    lens = [40, 3000, 900]               # every request holds the 40-query block
    full, hf, comp, kept = _caches(rng, lens, hkv, d, bits)
    hq = hkv * grp
    qn = synth.normal_bf16(rng, (len(lens), hq, d))
    qd = H.to_dev(qn.view(np.int16)).view(torch.bfloat16)
    qvn = synth.normal_bf16(rng, (len(lens), n_q, hq, d))
    qv = H.to_dev(qvn.view(np.int16)).view(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    msl = max(lens)
    od = torch.empty((len(lens), hq, d), dtype=torch.float32, device="cuda")
    ov = torch.empty((len(lens), n_q, hq, d), dtype=torch.float32, device="cuda")
    dws = torch.empty(m.draft_workspace_bytes(comp, hq, msl), dtype=torch.uint8, device="cuda")
    vws = torch.empty(m.verify_workspace_bytes(full, n_q, hq, msl), dtype=torch.uint8, device="cuda")
    role = H.to_dev(np.array([0, 1, 0], np.int32))
    mws = torch.empty(m.mixed_workspace_bytes(comp, full, 25, hq, msl), dtype=torch.uint8, device="cuda")
    om = torch.empty((len(lens), 25, hq, d), dtype=torch.float32, device="cuda")

    with pytest.raises(m.VCError):
        fault(-1, True)                                     # out of range: refused
    fault(LIMIT_NS, True)
    roles = np.array([0, 1, 0])
    calls = [   # (call, outputs it writes and the rows written)
        (lambda st: m.draft_attn(qd, comp, scale, od, msl, dws, status=st), [(od, [0, 1, 2])]),
        (lambda st: m.verify_attn(qv, full, scale, ov, msl, vws, status=st), [(ov, [0, 1, 2])]),   # two 128-row tiles
        (lambda st: m.verify_attn(qv[:, :25].contiguous(), full, scale, om, msl, vws, status=st),
         [(om, [0, 1, 2])]),                                                                        # one tile
        (lambda st: m.mixed_attn(role, qd, comp, od, qv[:, :25].contiguous(), full, om, scale, msl, mws, status=st),
         [(od, list(np.nonzero(roles == 0)[0])), (om, list(np.nonzero(roles == 1)[0]))]),
    ]
    for call, outs in calls:
        for t in (od, ov, om):
            t.fill_(float("nan"))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        call(st)
        torch.cuda.synchronize()
        assert st.item() == TIMEOUT
        for t, rows in outs:                                # every row the call owns: written, zero
            assert bool((t[rows] == 0).all())

    fault(0, False)                                         # back to normal: exact again
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.draft_attn(qd, comp, scale, od, msl, dws, status=st)
    m.verify_attn(qv, full, scale, ov, msl, vws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    god, gov = od.cpu().numpy(), ov.cpu().numpy()
    for b in range(len(lens)):
        k, v = H.logical_full(hf, b)
        ref = oracle.draft_attn(qn[b], oracle.compress(k, v, kept[b], bits), float(np.float32(scale)))
        assert H.row_err(god[b], ref) <= H.TOL
        ref = oracle.verify_attn_block(qvn[b], k, v, float(np.float32(scale)))
        assert H.row_err(gov[b], ref) <= H.TOL
