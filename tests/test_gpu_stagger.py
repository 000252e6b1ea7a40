"""GPU: the staggered engine (KV_full staged layer by layer from page-locked
host memory into a ring of slots while other requests draft) gives, at every
tick and layer, verification rows bit-identical to vc_verify_attn over a
device-resident KV_full and draft rows equal to vc_draft_attn over KV_comp
within the attention tolerance (the two launches split pages over warps
differently).  A missing or misplaced
wait on a staged layer would read another job's pages: the ring reuses slots
within the run.  Lock step (one slot for every request's KV_full) and a
schedule with idle requests are checked the same way."""
import math

import numpy as np
import pytest
import torch

from tests import vc_harness as H

pytestmark = pytest.mark.gpu

SPEC = dict(batch=6, hq=8, hkv=2, d=128, ctx_lo=600, ctx_hi=3000, layers=2, bits=3, x=5, max_x=8, seed=3)


@pytest.fixture(scope="module")
def rig():
    from synth.rigs import stagger_rig
    eng, qd, qv = stagger_rig(SPEC, torch.device("cuda"))
    return eng, qd, qv


def references(eng, qd, qv, x):
    import lossless_compressed_kv_gb300 as vc
    scale = 1.0 / math.sqrt(eng.d)
    fulls = eng.device_full(x)
    rv, rd = [], []
    for l in range(eng.L):
        q = qv[l][:, :x].contiguous()
        out = torch.empty((eng.n, x, eng.hq, eng.d), dtype=torch.float32, device="cuda")
        ws = torch.empty(vc.verify_workspace_bytes(fulls[l], x, eng.hq, eng.max_len), dtype=torch.uint8,
                         device="cuda")
        vc.verify_attn(q, fulls[l], scale, out, eng.max_len, ws)
        rv.append(out.cpu().numpy())
        od = torch.empty((eng.n, eng.hq, eng.d), dtype=torch.float32, device="cuda")
        ws = torch.empty(vc.draft_workspace_bytes(eng.comp[l], eng.hq, eng.max_len), dtype=torch.uint8,
                         device="cuda")
        vc.draft_attn(qd[l], eng.comp[l], scale, od, eng.max_len, ws)
        rd.append(od.cpu().numpy())
    torch.cuda.synchronize()
    return rd, rv


def run_and_check(rig, roles, x, slots):
    eng, qd, qv = rig
    snaps = []

    def snap(t, l, od, ov):
        snaps.append((t, l, od.clone(), ov.clone()))

    r = eng.run(roles, x, slots, qd, [q[:, :x].contiguous() for q in qv], measure_from=0, snapshot=snap)
    rd, rv = references(eng, qd, qv, x)
    assert len(snaps) == roles.shape[0] * eng.L
    n_ver = n_dr = 0
    for t, l, od, ov in snaps:
        od, ov = od.cpu().numpy(), ov.cpu().numpy()
        for b in range(eng.n):
            if roles[t, b] == 1:
                assert np.array_equal(ov[b], rv[l][b]), (t, l, b)
                n_ver += 1
            elif roles[t, b] == 0:
                # different page-to-warp splits round P to fp16 against
                # different running maxima: equal within the oracle tolerance
                assert H.row_err(od[b], rd[l][b]) <= H.TOL, (t, l, b)
                n_dr += 1
    assert n_ver > 0 and n_dr > 0
    assert r["link_GBps"] > 0 and r["stage_ms"] > 0 and r["wall_ms"] > 0
    return r


def test_staggered_plan_two_slots(rig):
    import lossless_compressed_kv_gb300 as vc
    from lossless_compressed_kv_gb300.stagger import phase_schedule
    eng = rig[0]
    x = SPEC["x"]
    ph, pb = vc.stagger_plan(eng.stage_bytes(x), x + 1)
    roles = phase_schedule(ph, x + 1, 2)
    r = run_and_check(rig, roles, x, 2)
    assert r["peak_stage_bytes"] == 2 * pb.max()


def test_staggered_single_slot_and_lock_step(rig):
    from lossless_compressed_kv_gb300.stagger import phase_schedule
    eng = rig[0]
    x = 3
    roles = phase_schedule(np.arange(eng.n) % (x + 1), x + 1, 2)
    run_and_check(rig, roles, x, 1)
    lock = phase_schedule(np.full(eng.n, x), x + 1, 2)
    r = run_and_check(rig, lock, x, 1)
    assert r["peak_stage_bytes"] == eng.stage_bytes(x).sum()


def test_idle_requests_and_chunked_verification(rig):
    """Lock step under a staging budget: after the draft ticks, the requests
    verify in chunks while the rest wait (role 2)."""
    eng = rig[0]
    x = SPEC["x"]
    n = eng.n
    roles = []
    for _ in range(2):
        roles += [[0] * n] * x
        for c in range(0, n, 2):
            roles.append([1 if c <= b < c + 2 else 2 for b in range(n)])
    run_and_check(rig, np.array(roles, np.int32), x, 2)
