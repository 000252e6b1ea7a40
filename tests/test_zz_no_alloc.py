"""vc_draft_attn_static — the draft attention without a caller workspace,
for callers that cannot allocate device memory at the call site (a plugin
inside an engine that owns all device memory, or a path that must not call
cudaMalloc because it can synchronise the device).  Called through the C
ABI; its output must match vc_draft_attn (which takes a workspace) within
the attention tolerance used by the other tests, on two calls in a row that
share the library's fixed scratch array.  Collected last so that a failure
here does not hide the others."""
import ctypes as C
import gc
import math

import numpy as np
import pytest
import torch

import synth
from tests import vc_harness as H

pytestmark = pytest.mark.gpu


def _setup(seed, lens, hkv=2, d=128, grp=4, bits=2):
    rng = np.random.default_rng(seed)
    full, hf = H.full_cache(rng, lens, hkv, d, synth.outlier_channels(rng, d, 2), 8.0)
    kept = [np.arange(n, dtype=np.int32) for n in lens]
    comp, _ = H.comp_cache(rng, len(lens), lens, hkv, d, bits)
    import lossless_compressed_kv_gb300 as vc
    offs, idx = synth.csr(kept)
    vc.compress(full, H.to_dev(offs), H.to_dev(idx), comp, max(lens))
    comp.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
    q = H.to_dev(synth.normal_bf16(rng, (len(lens), hkv * grp, d)).view(np.int16)).view(torch.bfloat16)
    return comp, q


def _static_call(lib, q, comp, scale, out, max_len, status):
    s = comp.struct()
    return lib.vc_draft_attn_static(C.c_void_p(q.data_ptr()), int(q.shape[1]), C.byref(s), C.c_float(scale),
                                    C.c_void_p(out.data_ptr()), int(max_len), C.c_void_p(status.data_ptr()),
                                    C.c_void_p(torch.cuda.current_stream().cuda_stream))


def _reference(comp, q, scale, max_len):
    import lossless_compressed_kv_gb300 as vc
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(vc.draft_workspace_bytes(comp, q.shape[1], max_len), dtype=torch.uint8, device="cuda")
    vc.draft_attn(q, comp, scale, out, max_len, ws)
    return out


def test_static_scratch_draft_matches_workspace_draft_twice():
    import lossless_compressed_kv_gb300 as vc
    lib = vc.library()
    lib.vc_draft_attn_static.restype = C.c_int
    lib.vc_draft_attn_static.argtypes = [C.c_void_p, C.c_int32, C.POINTER(vc.PagedKVStruct), C.c_float,
                                         C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]
    lib.vc_static_scratch_bytes.restype = C.c_size_t
    assert lib.vc_static_scratch_bytes() == 8 << 20
    # two calls in a row with different shapes / data: the second must not see
    # anything left over from the first in the shared array
    for i, (seed, lens) in enumerate(((1, [3000, 17, 900]), (2, [40, 5000, 2047, 1, 600]))):
        comp, q = _setup(seed, lens)
        scale = 1.0 / math.sqrt(128)
        need = vc.draft_workspace_bytes(comp, q.shape[1], max(lens))
        assert need <= lib.vc_static_scratch_bytes()
        # the partials of more than one context chunk per row go through the
        # array, so the combine pass reads what this call wrote there
        assert need // (len(lens) * q.shape[1] * (128 + 2) * 4) > 1
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        # no garbage collection inside the measured window: freed tensors of
        # earlier calls must not show up as a change
        gc.collect()
        gc.disable()
        try:
            torch.cuda.synchronize()
            free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
            rc = _static_call(lib, q, comp, scale, out, max(lens), st)
            torch.cuda.synchronize()
            free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        finally:
            gc.enable()
        assert rc == 0, vc.STATUS.get(rc, rc)
        if i == 1:   # device set up by the first call: the second allocates nothing
            assert free1 == free0
            assert alloc1 == alloc0
        ref = _reference(comp, q, scale, max(lens))
        torch.cuda.synchronize()
        assert st.item() == 0
        got, want = out.cpu().numpy(), ref.cpu().numpy()
        assert np.isfinite(got).all()
        assert H.row_err(got, want) <= H.TOL


def test_static_scratch_empty_batch_with_null_pointers():
    """Batch 0: the format is checked and VC_OK returned before any pointer
    is looked at, as vc_draft_attn does (zero-size tensors carry null data
    pointers)."""
    import lossless_compressed_kv_gb300 as vc
    lib = vc.library()
    lib.vc_draft_attn_static.restype = C.c_int
    lib.vc_draft_attn_static.argtypes = [C.c_void_p, C.c_int32, C.POINTER(vc.PagedKVStruct), C.c_float,
                                         C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]
    s = vc.PagedKVStruct(None, None, 0, None, None, 0, 0, vc.KVFormat(2, 128, 2))
    assert lib.vc_draft_attn_static(None, 8, C.byref(s), C.c_float(0.1), None, 64, None, None) == 0
    s.fmt = vc.KVFormat(2, 96, 2)         # an unsupported head_dim is still refused
    assert vc.STATUS[lib.vc_draft_attn_static(None, 8, C.byref(s), C.c_float(0.1), None, 64, None,
                                              None)] == "VC_ERR_UNSUPPORTED"


def test_static_scratch_rejects_oversized_calls():
    """A call that would need more than the fixed array is refused before any
    launch, with VC_ERR_WORKSPACE."""
    import lossless_compressed_kv_gb300 as vc
    lib = vc.library()
    lib.vc_draft_attn_static.restype = C.c_int
    lib.vc_draft_attn_static.argtypes = [C.c_void_p, C.c_int32, C.POINTER(vc.PagedKVStruct), C.c_float,
                                         C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]
    batch, hkv, d = 4096, 8, 128        # thousands of requests x 64 heads: partials >> 8 MiB
    bt = torch.zeros((batch, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(batch, dtype=torch.int32, device="cuda")
    comp = vc.PagedKV.allocate(1, hkv, d, 2, bt, lens)
    need = vc.draft_workspace_bytes(comp, 64, 1 << 16)
    assert need > lib.vc_static_scratch_bytes()
    q = torch.zeros((batch, 64, d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((batch, 64, d), dtype=torch.float32, device="cuda")
    s = comp.struct()
    rc = lib.vc_draft_attn_static(C.c_void_p(q.data_ptr()), 64, C.byref(s), C.c_float(0.1),
                                  C.c_void_p(out.data_ptr()), 1 << 16, None, None)
    assert vc.STATUS[rc] == "VC_ERR_WORKSPACE"
