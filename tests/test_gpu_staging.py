"""Staging of KV_full from host memory ("VeriCache Guide", the dual-stream
engine and "Best Practice 2": the full cache is reloaded on a side stream
from page-locked host memory, which is what lets the copy engines run at
full rate and overlap the drafting).  vc_stage_async and its paced variant
must refuse a source that is not page-locked host memory with
VC_ERR_STAGING, copy nothing in that case, and copy the bytes exactly when
the source is pinned."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def vc():
    import lossless_compressed_kv_gb300 as m
    return m


def _dst(n):
    return torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")


def test_stage_refuses_pageable_and_device_sources():
    m = vc()
    n = 1 << 20
    side = torch.cuda.Stream()
    pageable = torch.arange(n, dtype=torch.int64).to(torch.uint8)     # ordinary (pageable) host memory
    assert not pageable.is_pinned()
    on_device = torch.ones(n, dtype=torch.uint8, device="cuda")
    for src in (pageable, on_device):
        dst = _dst(n)
        with pytest.raises(m.VCError) as e:
            m.stage_async(dst, src, n, side)
        assert m.STATUS[e.value.code] == "VC_ERR_STAGING"
        origin = torch.zeros(1, dtype=torch.int64, device="cuda")
        m.link_clock(origin, side)
        with pytest.raises(m.VCError) as e:
            m.stage_paced_async(dst, src, n, 1 << 18, 100.0, origin, 0, side)
        assert m.STATUS[e.value.code] == "VC_ERR_STAGING"
        torch.cuda.synchronize()
        assert bool((dst == 0xAB).all())                             # nothing was copied


def test_stage_pinned_copies_exactly():
    m = vc()
    n = (1 << 20) + 48
    side = torch.cuda.Stream()
    src = torch.from_numpy(np.random.default_rng(3).integers(0, 256, n, dtype=np.uint8)).pin_memory()
    dst = _dst(n)
    done = torch.cuda.Event()
    m.stage_async(dst, src, n, side, done)
    torch.cuda.current_stream().wait_event(done)
    assert torch.equal(dst.cpu(), src)
    dst2 = _dst(n)
    origin = torch.zeros(1, dtype=torch.int64, device="cuda")
    m.link_clock(origin, side)
    m.stage_paced_async(dst2, src, n, 1 << 18, 100.0, origin, 0, side)   # 100 GB/s: about 10 us
    side.synchronize()
    assert torch.equal(dst2.cpu(), src)
