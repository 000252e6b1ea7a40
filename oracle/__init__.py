"""CPU oracle for the VeriCache attention-step operations.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the library under
``lossless_compressed_kv_gb300`` never imports it.  The arithmetic lives in
``vc_oracle.c`` (plain loops, fp64 attention, exact fp32 quantisation); this
module only builds it with gcc, loads it with ctypes and loops over requests
and heads.  Pages followed (titles, sections): "VeriCache: Making Lossy KV
Compression Exact" (The Core Idea: draft, verify with x+1 predictions, accept
rule and its worked example); "VeriCache Guide" (The Uniform Compressor
Interface; the compressor's sorted kept-index gather shared by all heads);
"KV Cache and Speculative Decoding" (causal attention).

Every function here is pinned by tests/test_oracle_*.py against closed forms,
library routines, brute force and the pages' worked example.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vc_oracle.c")
_LIB = os.path.join(_HERE, "libvc_oracle.so")
GROUP = 32

_lib = None


def build(force: bool = False) -> str:
    """Compile vc_oracle.c with gcc (-ffp-contract=off keeps fp32 steps
    unfused) into oracle/libvc_oracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        P = C.c_void_p
        L.vco_f32_to_f16_rn.restype = C.c_uint16
        L.vco_f32_to_f16_rn.argtypes = [C.c_float]
        L.vco_f16_to_f32.restype = C.c_float
        L.vco_f16_to_f32.argtypes = [C.c_uint16]
        L.vco_f32_to_f16_array.argtypes = [P, P, C.c_size_t]
        L.vco_f16_to_f32_array.argtypes = [P, P, C.c_size_t]
        L.vco_quantize_group.argtypes = [P, C.c_int, C.c_int, P, P, P]
        L.vco_quantize_row.argtypes = [P, C.c_int, C.c_int, P, P, P]
        L.vco_pack_codes.argtypes = [P, C.c_int, C.c_int, P]
        L.vco_unpack_codes.argtypes = [P, C.c_int, C.c_int, P]
        L.vco_dequant_row.argtypes = [P, P, P, C.c_int, P]
        L.vco_compress.restype = C.c_int
        L.vco_compress.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P, C.c_int, C.c_int,
                                   P, P, P, P, P, P, P, P]
        L.vco_attend.argtypes = [P, P, P, C.c_int, C.c_int, C.c_double, P, P]
        L.vco_draft_attn.restype = C.c_int
        L.vco_draft_attn.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                     P, P, P, P, P, P, P, P, C.c_double, P]
        L.vco_verify_attn.restype = C.c_int
        L.vco_verify_attn.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                      P, P, C.c_double, P]
        L.vco_accept.restype = C.c_int
        L.vco_keynorm_scores.argtypes = [P, C.c_int, C.c_int, C.c_int, P]
        L.vco_select_kept.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, P]
        L.vco_select_kept.restype = C.c_int
        L.vco_logits.argtypes = [P, C.c_int, C.c_int, P, C.c_int, C.c_int, P]
        L.vco_accept_sampled.argtypes = [P, P, C.c_int, C.c_float, P, C.c_int, P, P, P, P, P]
        L.vco_accept_sampled.restype = C.c_int
        L.vco_accept.argtypes = [P, C.c_int, C.c_int, P, C.c_int, C.c_int, P, C.c_int,
                                 P, P, P, P]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# scalar / row level
# ---------------------------------------------------------------------------

def f32_to_f16(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().vco_f32_to_f16_array(_p(x), _p(out), x.size)
    return out


def f16_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().vco_f16_to_f32_array(_p(h), _p(out), h.size)
    return out


def quantize_group(x, bits: int):
    """x: fp32 values of one group.  Returns (codes uint8, scale fp16 bits,
    zero fp16 bits)."""
    x = _c(x, np.float32)
    codes = np.empty(x.size, dtype=np.uint8)
    s = np.zeros(1, dtype=np.uint16)
    z = np.zeros(1, dtype=np.uint16)
    lib().vco_quantize_group(_p(x), x.size, bits, _p(codes), _p(s), _p(z))
    return codes, int(s[0]), int(z[0])


def quantize_row(x_bf16, bits: int):
    x = _c(x_bf16, np.uint16)
    d = x.size
    codes = np.empty(d, dtype=np.uint8)
    s = np.empty(d // GROUP, dtype=np.uint16)
    z = np.empty(d // GROUP, dtype=np.uint16)
    lib().vco_quantize_row(_p(x), d, bits, _p(codes), _p(s), _p(z))
    return codes, s, z


def pack_codes(codes, bits: int) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.size * bits // 8, dtype=np.uint8)
    lib().vco_pack_codes(_p(c), c.size, bits, _p(out))
    return out


def unpack_codes(packed, d: int, bits: int) -> np.ndarray:
    p = _c(packed, np.uint8)
    out = np.empty(d, dtype=np.uint8)
    lib().vco_unpack_codes(_p(p), d, bits, _p(out))
    return out


def dequant_row(codes, scales, zeros) -> np.ndarray:
    c = _c(codes, np.uint8)
    s = _c(scales, np.uint16)
    z = _c(zeros, np.uint16)
    out = np.empty(c.size, dtype=np.float64)
    lib().vco_dequant_row(_p(c), _p(s), _p(z), c.size, _p(out))
    return out


def attend(q, keys, vals, scale: float, want_weights: bool = False):
    q = _c(q, np.float64)
    k = _c(keys, np.float64)
    v = _c(vals, np.float64)
    n, d = k.shape
    out = np.empty(d, dtype=np.float64)
    w = np.empty(max(n, 1), dtype=np.float64) if want_weights else None
    lib().vco_attend(_p(q), _p(k), _p(v), n, d, scale, _p(out), _p(w))
    return (out, w[:n]) if want_weights else out


# ---------------------------------------------------------------------------
# request level (logical layouts; the page layout is unpacked by the caller)
# ---------------------------------------------------------------------------

def compress(k, v, kept, bits: int) -> dict:
    """One request.  k, v: [n][hkv][d] bf16 bits; kept: positions.

    bits 2/3/4 -> dict(k_packed [m][hkv][d*b/8] u8, k_scales, k_zeros
    [m][hkv][d/32] fp16 bits, and the same for v).  bits 16 -> dict(k16, v16)
    gathered [m][hkv][d] bf16 bits."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    kept = _c(kept, np.int32)
    n, hkv, d = k.shape
    m = kept.size
    L = lib()
    if bits == 16:
        k16 = np.empty((m, hkv, d), np.uint16)
        v16 = np.empty((m, hkv, d), np.uint16)
        rc = L.vco_compress(_p(k), _p(v), n, hkv, d, _p(kept), m, 16,
                            None, None, None, None, None, None, _p(k16), _p(v16))
        if rc:
            raise ValueError("kept index out of range")
        return dict(bits=16, k16=k16, v16=v16)
    pb = d * bits // 8
    out = dict(bits=bits,
               k_packed=np.empty((m, hkv, pb), np.uint8), v_packed=np.empty((m, hkv, pb), np.uint8),
               k_scales=np.empty((m, hkv, d // GROUP), np.uint16),
               k_zeros=np.empty((m, hkv, d // GROUP), np.uint16),
               v_scales=np.empty((m, hkv, d // GROUP), np.uint16),
               v_zeros=np.empty((m, hkv, d // GROUP), np.uint16))
    rc = L.vco_compress(_p(k), _p(v), n, hkv, d, _p(kept), m, bits,
                        _p(out["k_packed"]), _p(out["k_scales"]), _p(out["k_zeros"]),
                        _p(out["v_packed"]), _p(out["v_scales"]), _p(out["v_zeros"]), None, None)
    if rc:
        raise ValueError("kept index out of range")
    return out


def comp_concat(a: dict, b: dict) -> dict:
    """Append compressed entries b after a (draft tokens appended to KV_comp)."""
    return {k: (a[k] if k == "bits" else np.concatenate([a[k], b[k]], axis=0)) for k in a}


def comp_slice(c: dict, sl) -> dict:
    return {k: (c[k] if k == "bits" else c[k][sl]) for k in c}


def _draft_one(q, comp, kv, grp, d, scale):
    """One kv head of one request: q [grp][d]."""
    bits = comp["bits"]
    sel = lambda a: _c(a[:, kv:kv + 1], a.dtype)
    n = (comp["k16"] if bits == 16 else comp["k_packed"]).shape[0]
    out = np.empty((grp, d), dtype=np.float64)
    q = _c(q, np.uint16)
    L = lib()
    if bits == 16:
        k16, v16 = sel(comp["k16"]), sel(comp["v16"])
        rc = L.vco_draft_attn(_p(q), grp, 1, d, n, 16, None, None, None, None, None, None,
                              _p(k16), _p(v16), scale, _p(out))
    else:
        a = [sel(comp[x]) for x in ("k_packed", "k_scales", "k_zeros", "v_packed", "v_scales", "v_zeros")]
        rc = L.vco_draft_attn(_p(q), grp, 1, d, n, bits, *[_p(t) for t in a], None, None, scale, _p(out))
    assert rc == 0
    return out


def draft_attn(q, comp: dict, scale: float, pool: ThreadPoolExecutor | None = None) -> np.ndarray:
    """One request.  q [hq][d] bf16 bits; comp as returned by compress
    (n_comp entries).  Returns [hq][d] fp64."""
    q = _c(q, np.uint16)
    hq, d = q.shape
    hkv = (comp["k16"] if comp["bits"] == 16 else comp["k_packed"]).shape[1]
    grp = hq // hkv
    jobs = [(q[g * grp:(g + 1) * grp], comp, g, grp, d, scale) for g in range(hkv)]
    if pool is None:
        parts = [_draft_one(*j) for j in jobs]
    else:
        parts = list(pool.map(lambda j: _draft_one(*j), jobs))
    return np.concatenate(parts, axis=0)


def verify_attn(q, k, v, scale: float, heads=None, queries=None,
                pool: ThreadPoolExecutor | None = None) -> np.ndarray:
    """One request.  q [n_q][hq][d]; k, v [n_ctx][hkv][d] (the last n_q are
    the block).  Returns [n_q][hq][d] fp64 (NaN where not computed when a
    subset of heads / queries is asked for)."""
    q = _c(q, np.uint16)
    k = np.asarray(k)
    v = np.asarray(v)
    n_q, hq, d = q.shape
    n_ctx, hkv, _ = k.shape
    grp = hq // hkv
    heads = range(hq) if heads is None else heads
    queries = range(n_q) if queries is None else queries
    out = np.full((n_q, hq, d), np.nan)
    L = lib()

    def one(iq_h):
        i, h = iq_h
        g = h // grp
        pos = n_ctx - n_q + i
        kk = _c(k[:pos + 1, g:g + 1], np.uint16)
        vv = _c(v[:pos + 1, g:g + 1], np.uint16)
        qq = _c(q[i:i + 1, h:h + 1], np.uint16)
        o = np.empty((1, 1, d))
        rc = L.vco_verify_attn(_p(qq), 1, 1, 1, d, pos + 1, _p(kk), _p(vv), scale, _p(o))
        assert rc == 0
        return i, h, o[0, 0]

    jobs = [(i, h) for i in queries for h in heads]
    res = map(one, jobs) if pool is None else pool.map(one, jobs)
    for i, h, o in res:
        out[i, h] = o
    return out


def verify_attn_block(q, k, v, scale: float) -> np.ndarray:
    """Whole-block call of the C routine (used to pin the per-query path)."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    n_q, hq, d = q.shape
    n_ctx, hkv, _ = k.shape
    out = np.empty((n_q, hq, d))
    rc = lib().vco_verify_attn(_p(q), n_q, hq, hkv, d, n_ctx, _p(k), _p(v), scale, _p(out))
    if rc:
        raise ValueError("bad verify arguments")
    return out


def accept(hidden, w, drafts, want_ambiguous: bool = True):
    """One request.  hidden [n_pred][hg][dm] fp32, w [dm][V] fp32, drafts [x].
    Returns dict(verified [n_pred], accept_len, emitted [x+1] (-1 padded),
    n_emitted, ambiguous [n_pred] bool)."""
    h = _c(hidden, np.float32)
    if h.ndim == 2:
        h = h[:, None, :]
    n_pred, hg, dm = h.shape
    w = _c(w, np.float32)
    vocab = w.shape[1]
    dr = _c(drafts, np.int32)
    x = dr.size
    ver = np.empty(n_pred, np.int32)
    al = np.zeros(1, np.int32)
    em = np.empty(x + 1, np.int32)
    amb = np.zeros(n_pred, np.uint8) if want_ambiguous else None
    ne = lib().vco_accept(_p(h), n_pred, hg, _p(w), dm, vocab, _p(dr), x, _p(ver), _p(al),
                          _p(em), _p(amb))
    return dict(verified=ver, accept_len=int(al[0]), emitted=em, n_emitted=int(ne),
                ambiguous=(amb.astype(bool) if amb is not None else None))


def keynorm_scores(k) -> np.ndarray:
    """Token importance: mean over kv heads of the fp32 key L2 norm.
    k: bf16 bits [n][hkv][d] -> fp32 [n] (the guide's compressor)."""
    k = _c(k, np.uint16)
    n, hkv, d = k.shape
    out = np.empty(n, np.float32)
    lib().vco_keynorm_scores(_p(k), n, hkv, d, _p(out))
    return out


def select_kept(score, sink: int, recent: int, keep: int) -> np.ndarray:
    """Ascending kept-index list: sink and recent positions plus the middle
    positions of highest score (ties: lower position)."""
    score = _c(score, np.float32)
    n = int(score.shape[0])
    out = np.empty(max(n, 1), np.int32)
    c = lib().vco_select_kept(_p(score), n, int(sink), int(recent), int(keep), _p(out))
    return out[:c].copy()


def logits(hidden, w) -> np.ndarray:
    """fp32 logits of hidden rows [rows][hg][d] (group mean, then one fused
    multiply-add per hidden index in increasing order) -> [rows][vocab]."""
    hidden = _c(hidden, np.float32)
    if hidden.ndim == 2:
        hidden = hidden[:, None, :]
    w = _c(w, np.float32)
    rows, hg, dm = hidden.shape
    out = np.empty((rows, w.shape[1]), np.float32)
    lib().vco_logits(_p(hidden), rows, hg, _p(w), dm, w.shape[1], _p(out))
    return out


def accept_sampled(target_logits, draft_logits, drafts, u, v, tau: float) -> dict:
    """Rejection-sampling acceptance of one request (x drafts, x + 1 target
    rows): accept_len, emitted [x + 1] (-1 padded), margins [x + 1]."""
    tl = _c(target_logits, np.float32)
    x = int(tl.shape[0]) - 1
    vocab = int(tl.shape[1])
    dl = _c(draft_logits, np.float32).reshape(max(x, 1), vocab) if x else np.zeros((1, vocab), np.float32)
    dr = _c(drafts, np.int32).reshape(-1)
    u = _c(u, np.float32).reshape(-1)
    v = _c(v, np.float32).reshape(-1)
    al = np.zeros(1, np.int32)
    em = np.empty(x + 1, np.int32)
    mg = np.empty(x + 1, np.float64)
    lib().vco_accept_sampled(_p(tl), _p(dl), vocab, float(tau), _p(dr), x, _p(u), _p(v), _p(al), _p(em), _p(mg))
    return dict(accept_len=int(al[0]), emitted=em, margins=mg)
