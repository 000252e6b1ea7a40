"""GPU: the paced copy of the emulated slow link (vc_link_clock +
vc_stage_paced_async) delivers the bytes no faster than its rate, offsets
included; the remote-prefix engine's draft and verification outputs, computed
while KV_comp crosses the slow link and KV_full the fast one (destinations
filled with NaN bit patterns first), equal vc_draft_attn / vc_verify_attn over
the landed data, and drafting starts only once the compressed cache can have
arrived."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SPEC = dict(batch=2, hq=8, hkv=2, d=128, ctx=3000, layers=2, bits=3, x=5, rounds=2, seed=11)


def test_paced_copy_rate_and_bytes():
    import lossless_compressed_kv_gb300 as vc
    n = 16 << 20
    src = torch.randint(0, 256, (n,), dtype=torch.uint8).pin_memory()
    dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
    origin = torch.zeros(1, dtype=torch.int64, device="cuda")
    side = torch.cuda.Stream()
    rate = 4.0                                    # bytes per ns = 4 GB/s
    for offset in (0, 8 << 20):
        dst.zero_()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        vc.link_clock(origin, side)
        a.record(side)
        vc.stage_paced_async(dst, src, n, 1 << 20, rate, origin, offset, side, b)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        assert ms >= 0.97 * (offset + n) / rate / 1e6, ms
        assert ms <= 10 * (offset + n) / rate / 1e6 + 50.0, ms      # it does finish
        assert torch.equal(dst.cpu(), src)


def test_paced_copy_argument_errors():
    import lossless_compressed_kv_gb300 as vc
    src = torch.zeros(1024, dtype=torch.uint8).pin_memory()
    dst = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    origin = torch.zeros(1, dtype=torch.int64, device="cuda")
    side = torch.cuda.Stream()
    with pytest.raises(vc.VCError):
        vc.stage_paced_async(dst, src, 1024, 0, 1.0, origin, 0, side)           # chunk 0
    with pytest.raises(vc.VCError):
        vc.stage_paced_async(dst, src, 1024, 256, 0.0, origin, 0, side)         # no rate
    with pytest.raises(vc.VCError):
        vc.stage_paced_async(dst, src, 1024, 256, 1e-9, origin, 0, side)        # span > 60 s
    with pytest.raises(vc.VCError):
        vc.stage_paced_async(dst, torch.zeros(1024, dtype=torch.uint8), 1024, 256, 1.0, origin, 0, side)


def test_remote_prefix_engine_outputs_and_pacing():
    from synth.rigs import remote_rig
    import lossless_compressed_kv_gb300 as vc
    eng, qd, qv, q1, ones = remote_rig(SPEC, torch.device("cuda"))
    rate, chunk = 2.0, 64 << 10
    outs = []
    vr = eng.run_vericache(qd, qv, SPEC["rounds"], rate, chunk, outputs=outs)
    od, ov = outs[0]
    assert vr["first_draft_ms"] >= 0.97 * eng.bytes("comp") / rate / 1e6
    assert vr["first_verified_ms"] >= vr["first_draft_ms"] and vr["round_ms"] > 0
    # references over the landed data (last layer: the outputs hold it)
    l = eng.L - 1
    scale = 1.0 / np.sqrt(SPEC["d"])
    rd = torch.empty_like(od)
    ws = torch.empty(vc.draft_workspace_bytes(eng.comp[l], SPEC["hq"], eng.max_len), dtype=torch.uint8,
                     device="cuda")
    vc.draft_attn(qd[l], eng.comp[l], scale, rd, eng.max_len, ws)
    rv = torch.empty_like(ov)
    ws = torch.empty(vc.verify_workspace_bytes(eng.full[l], SPEC["x"], SPEC["hq"], eng.max_len), dtype=torch.uint8,
                     device="cuda")
    vc.verify_attn(qv[l], eng.full[l], scale, rv, eng.max_len, ws)
    torch.cuda.synchronize()
    assert torch.isfinite(od).all() and torch.isfinite(ov).all()
    assert torch.equal(od, rd) and torch.equal(ov, rv)
    # baseline: KV_full over the slow link, one-token steps
    outs = []
    br = eng.run_full_kv_remote(q1, ones, 3, rate, chunk, outputs=outs)
    assert br["first_token_ms"] >= 0.97 * eng.bytes("full") / rate / 1e6
    r1 = torch.empty_like(outs[0])
    ws = torch.empty(vc.verify_workspace_bytes(ones[l], 1, SPEC["hq"], eng.max_len), dtype=torch.uint8,
                     device="cuda")
    vc.verify_attn(q1[l], ones[l], scale, r1, eng.max_len, ws)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], r1)
