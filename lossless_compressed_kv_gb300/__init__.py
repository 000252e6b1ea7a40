"""VeriCache attention step for GB300 (sm_103a): Python binding of libvc.so.

The C ABI is declared in include/vc.h.  This module only marshals torch
tensors (device memory owned by the caller) and CUDA streams into that ABI;
every step of the computation runs in the library's CUDA kernels.  There is
no fallback: importing raises when libvc.so has not been built
(``python lossless_compressed_kv_gb300/build.py``).

Operations (see the header for their exact definitions and the pages they
follow): ``compress`` (KV_full -> KV_comp gather / 2-3-4-bit quantisation),
``draft_attn`` (decode attention over KV_comp), ``verify_attn`` (causal
block attention over KV_full), ``accept`` (argmax + longest matching prefix
+ correction / bonus), ``stage_async`` (pinned host -> device copy on a side
stream) and ``mixed_attn`` (draft and verify requests in one launch); the
staggering scheduler (``stagger_plan`` / ``stagger_simulate`` /
``stagger_horizon``, host code in the library; engine in ``stagger.py``) and
the paced copy of an emulated slow link (``link_clock`` /
``stage_paced_async``; remote-prefix engine in ``remote.py``).
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvc.so")
PAGE = 16
GROUP = 32

if not os.path.exists(LIB_PATH):
    raise ImportError("libvc.so is not built: run `python lossless_compressed_kv_gb300/build.py`")


class KVFormat(C.Structure):
    _fields_ = [("num_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("bits", C.c_int32)]


class PagedKVStruct(C.Structure):
    _fields_ = [("k_pages", C.c_void_p), ("v_pages", C.c_void_p), ("num_pages", C.c_int64),
                ("block_table", C.c_void_p), ("seq_lens", C.c_void_p), ("batch", C.c_int32),
                ("max_blocks", C.c_int32), ("fmt", KVFormat)]


class StaggerModel(C.Structure):
    _fields_ = [("n_requests", C.c_int32), ("stage_bytes", C.c_void_p), ("draft_ns", C.c_void_p),
                ("verify_ns", C.c_void_p), ("tick_ns", C.c_double), ("link_bytes_per_ns", C.c_double),
                ("n_slots", C.c_int32), ("n_layers", C.c_int32)]


class StaggerResult(C.Structure):
    _fields_ = [("cycle_ns", C.c_double), ("compute_ns", C.c_double), ("stall_ns", C.c_double),
                ("stage_ns", C.c_double), ("overlap", C.c_double), ("peak_stage_bytes", C.c_int64),
                ("draft_tokens_per_cycle", C.c_int64)]


_P = C.c_void_p
_lib = C.CDLL(LIB_PATH)
_SIG = {
    "vc_page_bytes": (C.c_size_t, [C.POINTER(KVFormat)]),
    "vc_head_block_bytes": (C.c_size_t, [C.POINTER(KVFormat)]),
    "vc_compress": (C.c_int, [C.POINTER(PagedKVStruct), _P, _P, _P, C.c_int32, C.POINTER(PagedKVStruct), _P, _P]),
    "vc_select_workspace_bytes": (C.c_size_t, [C.c_int32, C.c_int32]),
    "vc_accept_sampled_workspace_bytes": (C.c_size_t, [C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "vc_accept_sampled": (C.c_int, [_P, _P, C.c_int32, C.c_int32, C.c_int32, _P, C.c_int32, C.c_int32, C.c_float,
                                    _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "vc_select_kept": (C.c_int, [C.POINTER(PagedKVStruct), _P, C.c_int32, _P, C.c_int32, C.c_int32, _P, _P,
                                 C.c_size_t, _P, _P]),
    "vc_draft_workspace_bytes": (C.c_size_t, [C.POINTER(PagedKVStruct), C.c_int32, C.c_int32]),
    "vc_draft_attn": (C.c_int, [_P, C.c_int32, C.POINTER(PagedKVStruct), C.c_float, _P, C.c_int32, _P,
                                C.c_size_t, _P, _P]),
    "vc_draft_step": (C.c_int, [_P, C.c_int32, C.POINTER(PagedKVStruct), _P, _P, _P, C.c_float, _P, C.c_int32, _P,
                                C.c_size_t, _P, _P]),
    "vc_verify_workspace_bytes": (C.c_size_t, [C.POINTER(PagedKVStruct), C.c_int32, C.c_int32, C.c_int32]),
    "vc_verify_attn": (C.c_int, [_P, C.c_int32, C.c_int32, C.POINTER(PagedKVStruct), C.c_float, _P, C.c_int32,
                                 _P, C.c_size_t, _P, _P]),
    "vc_accept_workspace_bytes": (C.c_size_t, [C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "vc_accept": (C.c_int, [_P, C.c_int32, C.c_int32, C.c_int32, _P, C.c_int32, C.c_int32, _P, C.c_int32, _P, _P,
                            _P, _P, C.c_size_t, _P]),
    "vc_stage_async": (C.c_int, [_P, _P, C.c_size_t, _P, _P]),
    "vc_link_clock": (C.c_int, [_P, _P]),
    "vc_stage_paced_async": (C.c_int, [_P, _P, C.c_size_t, C.c_size_t, C.c_double, _P, C.c_size_t, _P, _P]),
    "vc_mixed_workspace_bytes": (C.c_size_t, [C.POINTER(PagedKVStruct), C.POINTER(PagedKVStruct), C.c_int32,
                                              C.c_int32, C.c_int32]),
    "vc_mixed_attn": (C.c_int, [_P, _P, C.POINTER(PagedKVStruct), _P, _P, C.c_int32, C.POINTER(PagedKVStruct), _P,
                                C.c_int32, C.c_float, C.c_int32, _P, C.c_size_t, _P, _P]),
    "vc_embed": (C.c_int, [_P, C.c_int32, _P, C.c_int32, C.c_int32, _P, _P, _P]),
    "vc_rmsnorm": (C.c_int, [_P, C.c_int32, C.c_int32, _P, C.c_float, _P, _P]),
    "vc_linear": (C.c_int, [_P, _P, _P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _P]),
    "vc_swiglu": (C.c_int, [_P, C.c_int32, C.c_int32, _P, _P]),
    "vc_rope_kv_write": (C.c_int, [_P, C.c_int32, _P, _P, C.c_int32, C.c_float, _P, C.POINTER(PagedKVStruct), _P,
                                   _P]),
    "vc_draft_attn_static": (C.c_int, [_P, C.c_int32, C.POINTER(PagedKVStruct), C.c_float, _P, C.c_int32, _P, _P]),
    "vc_static_scratch_bytes": (C.c_size_t, []),
    "vc_stagger_plan": (C.c_int, [_P, C.c_int32, C.c_int32, _P, _P]),
    "vc_stagger_simulate": (C.c_int, [C.POINTER(StaggerModel), C.c_int32, _P, C.c_int32, C.POINTER(StaggerResult)]),
    "vc_stagger_horizon": (C.c_int, [C.POINTER(StaggerModel), C.c_int32, C.c_int32, C.c_int32,
                                     C.POINTER(C.c_int32), _P, C.POINTER(StaggerResult)]),
    "vc_debug_set_wait_fault": (C.c_int, [C.c_int64, C.c_int32]),
    "vc_comp_block_decode": (C.c_int, [C.POINTER(KVFormat), C.c_int32, _P, _P, _P, _P]),
    "vc_comp_block_encode": (C.c_int, [C.POINTER(KVFormat), C.c_int32, _P, _P, _P, _P]),
    "vc_status_string": (C.c_char_p, [C.c_int]),
    "vc_version": (C.c_char_p, []),
}
for _n, (_r, _a) in _SIG.items():
    _f = getattr(_lib, _n)
    _f.restype = _r
    _f.argtypes = _a

STATUS = {0: "VC_OK", 1: "VC_ERR_INVALID_ARG", 2: "VC_ERR_UNSUPPORTED", 3: "VC_ERR_BAD_INDEX",
          4: "VC_ERR_CUDA", 5: "VC_ERR_STAGING", 6: "VC_ERR_TIMEOUT", 7: "VC_ERR_WORKSPACE"}


class VCError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (%s)" % (where, STATUS.get(code, code),
                                          _lib.vc_status_string(code).decode()))


def _check(code: int, where: str):
    if code != 0:
        raise VCError(code, where)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(s):
    if s is None:
        s = torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def version() -> str:
    return _lib.vc_version().decode()


def library():
    """The loaded ctypes handle (for ABI tests)."""
    return _lib


def comp_block_decode(block, head_dim: int, bits: int, kind: str):
    """vc_comp_block_decode of one stored head block (host bytes, numpy
    uint8 [vc_head_block_bytes]); kind "k" or "v".  Returns (codes uint8
    [16][head_dim * bits / 8] little-endian per slot, scales, zeros fp16 bits
    [16][head_dim / 32])."""
    import numpy as np
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    codes = np.empty((PAGE, head_dim * bits // 8), np.uint8)
    sc = np.empty((PAGE, head_dim // GROUP), np.uint16)
    ze = np.empty_like(sc)
    f = KVFormat(1, head_dim, bits)
    _check(_lib.vc_comp_block_decode(C.byref(f), 0 if kind == "k" else 1, blk.ctypes.data, codes.ctypes.data,
                                     sc.ctypes.data, ze.ctypes.data), "vc_comp_block_decode")
    return codes, sc, ze


def comp_block_encode(codes, scales, zeros, head_dim: int, bits: int, kind: str):
    """vc_comp_block_encode: logical content -> one stored head block (numpy uint8)."""
    import numpy as np
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint16)
    ze = np.ascontiguousarray(zeros, dtype=np.uint16)
    f = KVFormat(1, head_dim, bits)
    blk = np.empty(2 * head_dim * (bits + 1), np.uint8)
    _check(_lib.vc_comp_block_encode(C.byref(f), 0 if kind == "k" else 1, codes.ctypes.data, sc.ctypes.data,
                                     ze.ctypes.data, blk.ctypes.data), "vc_comp_block_encode")
    return blk


def debug_set_wait_fault(wait_limit_ns: int = 0, skip_copies: bool = False):
    """vc_debug_set_wait_fault (tests of the bounded device waits only)."""
    _check(_lib.vc_debug_set_wait_fault(int(wait_limit_ns), int(bool(skip_copies))), "vc_debug_set_wait_fault")


def head_block_bytes(head_dim: int, bits: int) -> int:
    f = KVFormat(1, head_dim, bits)
    return int(_lib.vc_head_block_bytes(C.byref(f)))


def page_bytes(num_kv_heads: int, head_dim: int, bits: int) -> int:
    f = KVFormat(num_kv_heads, head_dim, bits)
    return int(_lib.vc_page_bytes(C.byref(f)))


@dataclass
class PagedKV:
    """A paged K/V cache in the layout of include/vc.h.

    k_pages / v_pages: uint8 device tensors [num_pages, page_bytes];
    block_table: int32 [batch, max_blocks]; seq_lens: int32 [batch]."""
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    num_kv_heads: int
    head_dim: int
    bits: int

    @property
    def batch(self) -> int:
        return int(self.block_table.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    def struct(self) -> PagedKVStruct:
        for t, dt in ((self.block_table, torch.int32), (self.seq_lens, torch.int32)):
            if t.dtype != dt or not t.is_contiguous():
                raise ValueError("block_table / seq_lens must be contiguous int32")
        for t in (self.k_pages, self.v_pages):
            if not t.is_contiguous():
                raise ValueError("page pools must be contiguous")
        return PagedKVStruct(self.k_pages.data_ptr(), self.v_pages.data_ptr(), self.num_pages,
                             self.block_table.data_ptr(), self.seq_lens.data_ptr(), self.batch,
                             int(self.block_table.shape[1]), KVFormat(self.num_kv_heads, self.head_dim, self.bits))

    @staticmethod
    def allocate(num_pages: int, num_kv_heads: int, head_dim: int, bits: int, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, device="cuda", zero: bool = False) -> "PagedKV":
        pb = page_bytes(num_kv_heads, head_dim, bits)
        mk = torch.zeros if zero else torch.empty
        return PagedKV(mk((num_pages, pb), dtype=torch.uint8, device=device),
                       mk((num_pages, pb), dtype=torch.uint8, device=device),
                       block_table, seq_lens, num_kv_heads, head_dim, bits)


def compress(full: PagedKV, kept_offsets, kept_idx, comp: PagedKV, max_kept: int, comp_start=None,
             status=None, stream=None):
    fs, cs = full.struct(), comp.struct()
    _check(_lib.vc_compress(C.byref(fs), _ptr(kept_offsets), _ptr(kept_idx), _ptr(comp_start), int(max_kept),
                            C.byref(cs), _ptr(status), _stream(stream)), "vc_compress")


def select_workspace_bytes(batch: int, score_stride: int) -> int:
    return int(_lib.vc_select_workspace_bytes(int(batch), int(score_stride)))


def select_kept(full: PagedKV, kept_offsets, kept_idx, sink: int, recent: int, scores=None, score_stride=None,
                workspace=None, status=None, stream=None):
    """Kept-index list per request into kept_idx (CSR by kept_offsets):
    sink + recent windows plus the middle positions of highest score (key
    norm averaged over heads when scores is None)."""
    fs = full.struct()
    stride = int(score_stride if score_stride is not None else (scores.shape[-1] if scores is not None else 0))
    nb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.vc_select_kept(C.byref(fs), _ptr(scores), stride, _ptr(kept_offsets), int(sink), int(recent),
                               _ptr(kept_idx), _ptr(workspace), nb, _ptr(status), _stream(stream)),
           "vc_select_kept")


def draft_workspace_bytes(comp: PagedKV, num_q_heads: int, max_seq_len: int) -> int:
    cs = comp.struct()
    return int(_lib.vc_draft_workspace_bytes(C.byref(cs), num_q_heads, int(max_seq_len)))


def draft_attn(q, comp: PagedKV, softmax_scale: float, out, max_seq_len: int, workspace, status=None,
               stream=None):
    cs = comp.struct()
    _check(_lib.vc_draft_attn(_ptr(q), int(q.shape[-2]), C.byref(cs), float(softmax_scale), _ptr(out),
                              int(max_seq_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _ptr(status), _stream(stream)), "vc_draft_attn")


def draft_step(q, comp: PagedKV, k_new, v_new, slot, softmax_scale: float, out, max_seq_len: int, workspace,
               status=None, stream=None):
    """vc_draft_step: write each request's new entry (bf16 K / V rows
    [B][Hkv][D]) to KV_comp position slot[b], then draft attention."""
    cs = comp.struct()
    _check(_lib.vc_draft_step(_ptr(q), int(q.shape[1]), C.byref(cs), _ptr(k_new), _ptr(v_new), _ptr(slot),
                              float(softmax_scale), _ptr(out), int(max_seq_len), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)),
           "vc_draft_step")


def verify_workspace_bytes(full: PagedKV, n_q: int, num_q_heads: int, max_seq_len: int) -> int:
    fs = full.struct()
    return int(_lib.vc_verify_workspace_bytes(C.byref(fs), n_q, num_q_heads, int(max_seq_len)))


def verify_attn(q, full: PagedKV, softmax_scale: float, out, max_seq_len: int, workspace, status=None,
                stream=None):
    fs = full.struct()
    _check(_lib.vc_verify_attn(_ptr(q), int(q.shape[1]), int(q.shape[2]), C.byref(fs), float(softmax_scale),
                               _ptr(out), int(max_seq_len), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)),
           "vc_verify_attn")


def accept_workspace_bytes(batch: int, n_pred: int, vocab: int, d: int) -> int:
    return int(_lib.vc_accept_workspace_bytes(batch, n_pred, vocab, d))


def accept(hidden, lm_head, drafts, verified, accept_len, emitted, workspace, hidden_group: int = 1,
           stream=None):
    """hidden [B][n_pred][hidden_group][d] (or [B][n_pred][d]) fp32; lm_head [d][V] fp32."""
    b, n_pred = int(hidden.shape[0]), int(hidden.shape[1])
    d, vocab = int(lm_head.shape[0]), int(lm_head.shape[1])
    x = int(drafts.shape[1]) if drafts is not None and drafts.dim() == 2 else 0
    _check(_lib.vc_accept(_ptr(hidden), b, n_pred, int(hidden_group), _ptr(lm_head), d, vocab,
                          _ptr(drafts) if x else None, x, _ptr(verified), _ptr(accept_len), _ptr(emitted),
                          _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "vc_accept")


def accept_sampled_workspace_bytes(batch: int, x: int, vocab: int, d: int) -> int:
    return int(_lib.vc_accept_sampled_workspace_bytes(int(batch), int(x), int(vocab), int(d)))


def accept_sampled(target_hidden, draft_hidden, lm_head, drafts, u, v, temperature: float, accept_len, emitted,
                   workspace, hidden_group: int = 1, stream=None):
    """Rejection-sampling acceptance.  target_hidden [B][x+1][hg][d] (or
    [B][x+1][d]), draft_hidden [B][x][hg][d], drafts [B][x] int32, u [B][x],
    v [B][x+1] fp32 uniforms."""
    b, x = int(target_hidden.shape[0]), int(target_hidden.shape[1]) - 1
    d, vocab = int(lm_head.shape[0]), int(lm_head.shape[1])
    _check(_lib.vc_accept_sampled(_ptr(target_hidden), _ptr(draft_hidden) if x else None, b, x, int(hidden_group),
                                  _ptr(lm_head), d, vocab, float(temperature), _ptr(drafts) if x else None,
                                  _ptr(u) if x else None, _ptr(v), _ptr(accept_len), _ptr(emitted),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "vc_accept_sampled")


def stage_async(dst, pinned_src, nbytes: int, side_stream, done_event=None):
    """vc_stage_async; done_event (a torch.cuda.Event, created lazily by
    torch) is recorded on side_stream after the copy."""
    _check(_lib.vc_stage_async(C.c_void_p(dst.data_ptr()), C.c_void_p(pinned_src.data_ptr()), int(nbytes),
                               C.c_void_p(side_stream.cuda_stream), None), "vc_stage_async")
    if done_event is not None:
        done_event.record(side_stream)


def link_clock(origin, stream=None):
    """Write the device timer (ns) into origin (int64 device tensor, 1 element)."""
    if origin.dtype != torch.int64:
        raise ValueError("origin must be an int64 device tensor")
    _check(_lib.vc_link_clock(_ptr(origin), _stream(stream)), "vc_link_clock")


def stage_paced_async(dst, pinned_src, nbytes: int, chunk_bytes: int, bytes_per_ns: float, origin,
                      link_offset_bytes: int, side_stream, done_event=None):
    """vc_stage_async paced as a link of bytes_per_ns that has carried
    link_offset_bytes since the origin written by link_clock."""
    _check(_lib.vc_stage_paced_async(C.c_void_p(dst.data_ptr()), C.c_void_p(pinned_src.data_ptr()), int(nbytes),
                                     int(chunk_bytes), float(bytes_per_ns), _ptr(origin), int(link_offset_bytes),
                                     C.c_void_p(side_stream.cuda_stream), None), "vc_stage_paced_async")
    if done_event is not None:
        done_event.record(side_stream)


def mixed_workspace_bytes(comp: PagedKV, full: PagedKV, n_q: int, num_q_heads: int, max_seq_len: int) -> int:
    cs, fs = comp.struct(), full.struct()
    return int(_lib.vc_mixed_workspace_bytes(C.byref(cs), C.byref(fs), n_q, num_q_heads, int(max_seq_len)))


def mixed_attn(role, q_draft, comp: PagedKV, out_draft, q_verify, full: PagedKV, out_verify,
               softmax_scale: float, max_seq_len: int, workspace, status=None, stream=None):
    cs, fs = comp.struct(), full.struct()
    _check(_lib.vc_mixed_attn(_ptr(role), _ptr(q_draft), C.byref(cs), _ptr(out_draft), _ptr(q_verify),
                              int(q_verify.shape[1]), C.byref(fs), _ptr(out_verify), int(q_draft.shape[1]),
                              float(softmax_scale), int(max_seq_len), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)),
           "vc_mixed_attn")


# ---------------------------------------------------------------------------
# staggering scheduler (host code in the library; numpy in, numpy / dict out)
# ---------------------------------------------------------------------------

def _np_ptr(a):
    return C.c_void_p(a.ctypes.data)


def stagger_plan(stage_bytes, n_phases: int):
    """Balanced verify phases (vc_stagger_plan): returns (phase [n] int32,
    phase_bytes [n_phases] int64)."""
    import numpy as np
    sb = np.ascontiguousarray(stage_bytes, dtype=np.int64)
    ph = np.zeros(max(1, len(sb)), np.int32)
    pb = np.zeros(n_phases, np.int64)
    _check(_lib.vc_stagger_plan(_np_ptr(sb), len(sb), int(n_phases), _np_ptr(ph), _np_ptr(pb)), "vc_stagger_plan")
    return ph[:len(sb)], pb


class _Model:
    """Keeps the numpy arrays a vc_stagger_model points to alive."""

    def __init__(self, stage_bytes, draft_ns, verify_ns, link_bytes_per_ns, n_slots, n_layers, tick_ns):
        import numpy as np
        self.sb = np.ascontiguousarray(stage_bytes, dtype=np.int64)
        self.d = np.ascontiguousarray(draft_ns, dtype=np.float64)
        self.v = np.ascontiguousarray(verify_ns, dtype=np.float64)
        if not (len(self.sb) == len(self.d) == len(self.v)):
            raise ValueError("stage_bytes, draft_ns and verify_ns differ in length")
        self.s = StaggerModel(len(self.sb), self.sb.ctypes.data, self.d.ctypes.data, self.v.ctypes.data,
                              float(tick_ns), float(link_bytes_per_ns), int(n_slots), int(n_layers))


def _result(r: StaggerResult) -> dict:
    return {f: getattr(r, f) for f, _ in StaggerResult._fields_}


def stagger_simulate(phase, n_phases: int, stage_bytes, draft_ns, verify_ns, link_bytes_per_ns: float,
                     n_slots: int = 2, n_layers: int = 1, tick_ns: float = 0.0, n_cycles: int = 4) -> dict:
    """Steady-state cycle of a phase plan under the staging model (vc_stagger_simulate)."""
    import numpy as np
    m = _Model(stage_bytes, draft_ns, verify_ns, link_bytes_per_ns, n_slots, n_layers, tick_ns)
    ph = np.ascontiguousarray(phase, dtype=np.int32)
    r = StaggerResult()
    _check(_lib.vc_stagger_simulate(C.byref(m.s), int(n_phases), _np_ptr(ph), int(n_cycles), C.byref(r)),
           "vc_stagger_simulate")
    return _result(r)


def stagger_horizon(stage_bytes, draft_ns, verify_ns, link_bytes_per_ns: float, x_lo: int, x_hi: int,
                    n_slots: int = 2, n_layers: int = 1, tick_ns: float = 0.0, n_cycles: int = 4):
    """Smallest stall-free draft horizon in [x_lo, x_hi] (vc_stagger_horizon):
    returns (x, phase [n] int32, result dict)."""
    import numpy as np
    m = _Model(stage_bytes, draft_ns, verify_ns, link_bytes_per_ns, n_slots, n_layers, tick_ns)
    ph = np.zeros(max(1, len(m.sb)), np.int32)
    x = C.c_int32(0)
    r = StaggerResult()
    _check(_lib.vc_stagger_horizon(C.byref(m.s), int(x_lo), int(x_hi), int(n_cycles), C.byref(x), _np_ptr(ph),
                                   C.byref(r)), "vc_stagger_horizon")
    return int(x.value), ph[:len(m.sb)], _result(r)


# ---------------------------------------------------------------------------
# decoder-layer operations (end-to-end loop)
# ---------------------------------------------------------------------------

def embed(ids, table, out, status=None, stream=None):
    _check(_lib.vc_embed(_ptr(ids), int(ids.numel()), _ptr(table), int(table.shape[1]), int(table.shape[0]),
                         _ptr(out), _ptr(status), _stream(stream)), "vc_embed")


def rmsnorm(x, weight, out, eps: float = 1e-5, stream=None):
    _check(_lib.vc_rmsnorm(_ptr(x), int(x.shape[0]), int(x.shape[1]), _ptr(weight), float(eps), _ptr(out),
                           _stream(stream)), "vc_rmsnorm")


def linear(x, w_bf16, out, accumulate: bool = False, stream=None):
    """out[m][n] (+)= bf16(x) @ W, x fp32 [m][k], W bf16 [k][n], out fp32."""
    m, k = int(x.shape[0]), int(x.shape[1])
    _check(_lib.vc_linear(_ptr(x), _ptr(w_bf16), _ptr(out), m, k, int(w_bf16.shape[1]), int(bool(accumulate)),
                          _stream(stream)), "vc_linear")


def swiglu(gu, out, stream=None):
    _check(_lib.vc_swiglu(_ptr(gu), int(gu.shape[0]), int(out.shape[1]), _ptr(out), _stream(stream)), "vc_swiglu")


def rope_kv_write(qkv, row_req, row_pos, num_q_heads: int, theta: float, q_out, full: PagedKV, status=None,
                  stream=None):
    fs = full.struct()
    _check(_lib.vc_rope_kv_write(_ptr(qkv), int(qkv.shape[0]), _ptr(row_req), _ptr(row_pos), int(num_q_heads),
                                 float(theta), _ptr(q_out), C.byref(fs), _ptr(status), _stream(stream)),
           "vc_rope_kv_write")
