"""The C-ABI library loads, exports every entry point include/vc.h declares,
and rejects bad arguments on the host before any CUDA work (no GPU needed:
these paths return before touching the device)."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vc.h")


def _build():
    import __graft_entry__
    return __graft_entry__._builder().build()


@pytest.fixture(scope="module")
def vc():
    _build()
    import lossless_compressed_kv_gb300 as m
    return m


def declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"VC_API[^;(]*?\b(vc_\w+)\s*\(", txt)))


def test_header_declares_the_four_operations():
    names = declared()
    for n in ("vc_compress", "vc_draft_attn", "vc_verify_attn", "vc_accept"):
        assert n in names


def test_every_declared_symbol_is_exported(vc):
    out = subprocess.run(["nm", "-D", "--defined-only", vc.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(vc_\w+)", out))
    missing = [n for n in declared() if n not in exported]
    assert not missing, missing
    for n in declared():
        getattr(vc.library(), n)


def test_page_sizes_follow_the_layout(vc):
    # bf16: 16 x D x 2 bytes per head; b bits: codes 16*D*b/8 + scales/zeros 2*16*D/32*2
    assert vc.head_block_bytes(128, 16) == 4096
    assert vc.head_block_bytes(128, 2) == 768
    assert vc.head_block_bytes(128, 3) == 1024
    assert vc.head_block_bytes(128, 4) == 1280
    assert vc.head_block_bytes(64, 4) == 640
    assert vc.page_bytes(8, 128, 2) == 8 * 768
    assert vc.head_block_bytes(128, 5) == 0          # unsupported width
    assert vc.head_block_bytes(32, 16) == 1024
    assert vc.head_block_bytes(32, 2) == 0           # quantised formats need head_dim % 64 == 0


def test_struct_layout_matches_c(vc):
    assert C.sizeof(vc.KVFormat) == 12
    assert C.sizeof(vc.PagedKVStruct) == 64
    assert C.sizeof(vc.StaggerModel) == 56      # static_assert'ed in the library too
    assert C.sizeof(vc.StaggerResult) == 56


def test_host_side_argument_errors(vc):
    L = vc.library()
    assert L.vc_compress(None, None, None, None, 0, None, None, None) == 1
    assert L.vc_draft_attn(None, 4, None, 1.0, None, 0, None, 0, None, None) == 1
    assert L.vc_verify_attn(None, 1, 4, None, 1.0, None, 0, None, 0, None, None) == 1
    assert L.vc_accept(None, 1, 1, 1, None, 1, 1, None, 0, None, None, None, None, 0, None) == 1
    fake = C.c_void_p(16)   # never dereferenced: validation fails first
    fmt = vc.KVFormat(2, 128, 5)                      # 5 bits: unsupported
    s = vc.PagedKVStruct(fake.value, fake.value, 4, fake.value, fake.value, 1, 1, fmt)
    assert L.vc_draft_attn(fake, 4, C.byref(s), 1.0, fake, 16, fake, 1 << 20, None, None) == 2
    fmt = vc.KVFormat(2, 128, 16)
    s = vc.PagedKVStruct(fake.value, fake.value, 4, fake.value, fake.value, 1, 1, fmt)
    assert L.vc_verify_attn(fake, 65, 4, C.byref(s), 1.0, fake, 16, fake, 1 << 20, None, None) == 2  # n_q > 64
    assert L.vc_verify_attn(fake, 4, 5, C.byref(s), 1.0, fake, 16, fake, 1 << 20, None, None) == 2   # 5 % 2 != 0
    # accept: n_pred must be x or x + 1
    assert L.vc_accept(fake, 1, 5, 1, fake, 4, 10, fake, 2, fake, fake, fake, fake, 1 << 20, None) == 1
    assert vc.STATUS[L.vc_accept(fake, 1, 3, 1, fake, 4, 10, fake, 2, fake, fake, fake, None, 0, None)] \
        == "VC_ERR_WORKSPACE"
    assert L.vc_status_string(7) == b"workspace missing or too small"


def test_empty_batch_is_ok_with_null_data(vc):
    """Batch 0: formats and sizes are checked, nothing is launched, VC_OK;
    the per-request pointers may be NULL (a zero-size tensor's data pointer).
    No CUDA call happens on this path, so it runs without a GPU."""
    L = vc.library()
    comp = vc.PagedKVStruct(None, None, 0, None, None, 0, 0, vc.KVFormat(8, 128, 2))
    full = vc.PagedKVStruct(None, None, 0, None, None, 0, 0, vc.KVFormat(8, 128, 16))
    assert L.vc_draft_attn(None, 32, C.byref(comp), 1.0, None, 0, None, 0, None, None) == 0
    assert L.vc_draft_step(None, 32, C.byref(comp), None, None, None, 1.0, None, 0, None, 0, None, None) == 0
    assert L.vc_verify_attn(None, 32, 32, C.byref(full), 1.0, None, 0, None, 0, None, None) == 0
    assert L.vc_mixed_attn(None, None, C.byref(comp), None, None, 25, C.byref(full), None, 32, 1.0, 0, None, 0,
                           None, None) == 0
    assert L.vc_compress(C.byref(full), None, None, None, 0, C.byref(comp), None, None) == 0
    assert L.vc_select_kept(C.byref(full), None, 1, None, 64, 512, None, None, 0, None, None) == 0
    fake = C.c_void_p(16)   # never dereferenced
    assert L.vc_accept(None, 0, 33, 1, fake, 128, 32000, None, 32, None, None, None, None, 0, None) == 0
    assert L.vc_accept_sampled(None, None, 0, 4, 1, fake, 128, 32000, 1.0, None, None, None, None, None, None, 0,
                               None) == 0
    # the formats are still checked: an unsupported width or block length is refused
    bad = vc.PagedKVStruct(None, None, 0, None, None, 0, 0, vc.KVFormat(8, 128, 5))
    assert L.vc_draft_attn(None, 32, C.byref(bad), 1.0, None, 0, None, 0, None, None) == 2
    assert L.vc_verify_attn(None, 65, 32, C.byref(full), 1.0, None, 0, None, 0, None, None) == 2
    assert L.vc_accept(None, 0, 5, 1, fake, 128, 32000, None, 32, None, None, None, None, 0, None) == 1
    # ... and with requests, a NULL query is an argument error again
    one = vc.PagedKVStruct(fake.value, fake.value, 4, fake.value, fake.value, 1, 1, vc.KVFormat(8, 128, 2))
    assert L.vc_draft_attn(None, 32, C.byref(one), 1.0, fake, 16, fake, 1 << 20, None, None) == 1


def test_oracle_and_library_share_no_code():
    """The CUDA sources and the oracle do not include or import each other."""
    csrc = os.path.join(ROOT, "lossless_compressed_kv_gb300", "csrc")
    for f in os.listdir(csrc):
        assert "oracle" not in open(os.path.join(csrc, f)).read().lower()
    for f in ("vc_oracle.c", "__init__.py"):
        txt = open(os.path.join(ROOT, "oracle", f)).read()
        assert not re.search(r"(import|from)\s+lossless_compressed_kv_gb300", txt)
        assert "#include \"vc" not in txt and "libvc.so" not in txt
    pkg = open(os.path.join(ROOT, "lossless_compressed_kv_gb300", "__init__.py")).read()
    assert "import oracle" not in pkg and "from oracle" not in pkg


# ---------------------------------------------------------------------------
# KV_comp head blocks: stored order <-> logical content (host helpers)
# ---------------------------------------------------------------------------

def _header_k_bit(bits, d, s, c, plane):
    """The K code placement exactly as the layout notes of include/vc.h
    write it (bit offset of the code's low bit; plane 1 = top bit of a 3-bit
    code)."""
    ks, t, e = c // 16, (c // 4) % 4, c % 4
    r, h = 2 * ks + e // 2, e % 2
    if bits == 2:
        return s * 2 * d + t * d // 2 + 32 * (r // 8) + 16 * h + 2 * (r % 8)
    if bits == 4:
        return s * 4 * d + t * d + 32 * (r // 4) + 16 * h + 4 * (r % 4)
    if plane == 0:
        return s * 3 * d + t * d // 2 + 32 * (r // 8) + 16 * h + 2 * (r % 8)
    u, j = r // 8, r % 8
    beta = 2 * (j % 4) + [0, 1, 8, 9][2 * (u % 2) + j // 4]
    if d == 64:
        return s * 3 * d + 2 * d + 16 * t + 8 * h + beta
    return s * 3 * d + 2 * d + t * d // 4 + 32 * (u // 2) + 16 * h + beta


def _header_v_bit(bits, d, s, c, plane):
    g, w, m = c % 8, (c // 8) % 2, c // 16
    t, hi, h = (s // 2) % 4, s // 8, s % 2
    R = 4 * g + t
    if bits == 4:
        return 32 * (R * d // 16 + m) + 16 * h + 8 * w + 4 * hi
    u, n = m // 2, m % 2
    if bits == 2 or plane == 0:
        return 32 * (R * d // 32 + u) + 16 * h + 8 * n + 4 * w + 2 * hi
    j = 2 * w + hi
    return 32 * d + 32 * (R * d // 64 + u // 2) + 16 * h + 2 * j + [0, 1, 8, 9][2 * (u % 2) + n]


def _header_param(kind, g, s, gr, bits):
    if kind == "k":
        return s * g + gr
    return (((s // 2) % 4) * g + gr) * 4 + 2 * (s // 8) + (s % 2)


@pytest.mark.parametrize("bits,d", [(2, 64), (2, 128), (3, 64), (3, 128), (3, 256), (4, 64), (4, 128)])
@pytest.mark.parametrize("kind", ["k", "v"])
def test_comp_block_helpers_follow_the_header(vc, bits, d, kind):
    """One code of value 2^b - 1 (or, for 3 bits, each plane's bit) at a time:
    the stored block vc_comp_block_encode writes has exactly those bits set,
    at the offsets the header's formulas give; scales and zeros land at the
    header's parameter indices; decode inverts encode."""
    import numpy as np
    rng = np.random.default_rng(bits * 100 + d + (kind == "v"))
    g = d // 32
    row, cr = d * bits // 8, 16 * d * bits // 8
    f = _header_k_bit if kind == "k" else _header_v_bit
    z16 = np.zeros((16, g), np.uint16)
    for s, c in [(0, 0), (15, d - 1)] + [tuple(x) for x in rng.integers(0, [16, d], (12, 2))]:
        codes = np.zeros((16, row), np.uint8)
        for j in range(bits):           # code 2^b - 1: all its bits
            bit = bits * c + j
            codes[s, bit // 8] |= 1 << (bit % 8)
        blk = vc.comp_block_encode(codes, z16, z16, d, bits, kind)
        want = set()
        for j in range(bits):
            want.add(f(bits, d, s, c, 1) if bits == 3 and j == 2 else f(bits, d, s, c, 0) + j)
        got = set(np.nonzero(np.unpackbits(blk[:cr], bitorder="little"))[0].tolist())
        assert got == want, (s, c)
        assert not blk[cr:].any()
        back = vc.comp_block_decode(blk, d, bits, kind)
        assert np.array_equal(back[0], codes)
    sc = rng.integers(0, 1 << 16, (16, g)).astype(np.uint16)
    ze = rng.integers(0, 1 << 16, (16, g)).astype(np.uint16)
    blk = vc.comp_block_encode(np.zeros((16, row), np.uint8), sc, ze, d, bits, kind)
    par = blk[cr:].view(np.uint16)
    for s in range(16):
        for gr in range(g):
            i = _header_param(kind, g, s, gr, bits)
            assert par[i] == sc[s, gr] and par[16 * g + i] == ze[s, gr]
    # every bit of a random stored block is used: decode then encode is the identity
    rand = rng.integers(0, 256, 2 * d * (bits + 1)).astype(np.uint8)
    assert np.array_equal(vc.comp_block_encode(*vc.comp_block_decode(rand, d, bits, kind), d, bits, kind), rand)


def test_comp_block_helpers_reject_bad_arguments(vc):
    import numpy as np
    blk = np.zeros(768, np.uint8)
    for d, bits in ((128, 16), (96, 2), (32, 2), (128, 5)):
        with pytest.raises(vc.VCError):
            vc.comp_block_decode(blk, d, bits, "k")
    f = vc.KVFormat(1, 128, 2)
    lib = vc.library()
    z = np.zeros(4096, np.uint8)
    assert lib.vc_comp_block_decode(C.byref(f), 2, z.ctypes.data, z.ctypes.data, z.ctypes.data,
                                    z.ctypes.data) == 1
    assert lib.vc_comp_block_encode(C.byref(f), 0, None, z.ctypes.data, z.ctypes.data, z.ctypes.data) == 1
