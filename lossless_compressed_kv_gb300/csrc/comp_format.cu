// Host-side conversions between a stored KV_comp head block and the
// logical format of include/vc.h (vc_comp_block_decode / _encode): codes as a
// little-endian bit string per token slot (channel i at bits [b i, b i + b)),
// fp16 scales and zeros as [16 slots][D/32 groups].  The stored block holds
// the same codes, scales and zeros in the order comp_layout.cuh defines (the
// order the draft kernel's tensor-core operands want); these helpers let a C
// caller read or write a page without knowing that order.  Plain host code:
// no CUDA call, no allocation.
#include <cstring>

#include "comp_layout.cuh"
#include "vc_internal.cuh"

namespace {

bool fmt_ok(const vc_kv_format *f) {
    return f && (f->bits == 2 || f->bits == 3 || f->bits == 4) && f->head_dim >= 64 && f->head_dim <= 256 &&
           f->head_dim % 64 == 0;
}

inline unsigned get_bit(const uint8_t *p, int bit) { return (p[bit >> 3] >> (bit & 7)) & 1u; }
inline void put_bit(uint8_t *p, int bit, unsigned v) {
    if (v)
        p[bit >> 3] = (uint8_t)(p[bit >> 3] | (1u << (bit & 7)));
    else
        p[bit >> 3] = (uint8_t)(p[bit >> 3] & ~(1u << (bit & 7)));
}

// bit offset in the stored code region of bit j (0 = least significant) of
// the code of (slot s, channel c)
int stored_bit(int kind, int bits, int d, int s, int c, int j) {
    if (bits == 3) {
        const int plane = j == 2 ? 1 : 0, jj = j == 2 ? 0 : j;
        return (kind == 0 ? vc::layout::k_bit(3, d, s, c, plane) : vc::layout::v_bit(3, d, s, c, plane)) + jj;
    }
    return (kind == 0 ? vc::layout::k_bit(bits, d, s, c, 0) : vc::layout::v_bit(bits, d, s, c, 0)) + j;
}

// index (in fp16 units from the start of the scale array) of the parameter
// of (slot s, group gr)
int stored_param(int kind, int groups, int s, int gr) {
    return kind == 0 ? s * groups + gr : vc::layout::v_param(groups, s, gr);
}

}  // namespace

extern "C" {

vc_status vc_comp_block_decode(const vc_kv_format *fmt, int32_t kind, const void *block, uint8_t *codes,
                               uint16_t *scales, uint16_t *zeros) {
    if (!fmt_ok(fmt) || (kind != 0 && kind != 1) || !block || !codes || !scales || !zeros)
        return VC_ERR_INVALID_ARG;
    const int b = fmt->bits, d = fmt->head_dim, g = d / VC_GROUP;
    const uint8_t *blk = static_cast<const uint8_t *>(block);
    const int row = d * b / 8, cr = VC_PAGE_TOKENS * row;
    std::memset(codes, 0, (size_t)cr);
    for (int s = 0; s < VC_PAGE_TOKENS; ++s)
        for (int c = 0; c < d; ++c)
            for (int j = 0; j < b; ++j)
                put_bit(codes + s * row, b * c + j, get_bit(blk, stored_bit(kind, b, d, s, c, j)));
    const uint8_t *par = blk + cr;
    for (int s = 0; s < VC_PAGE_TOKENS; ++s)
        for (int gr = 0; gr < g; ++gr) {
            const int i = stored_param(kind, g, s, gr);
            std::memcpy(scales + s * g + gr, par + 2 * i, 2);
            std::memcpy(zeros + s * g + gr, par + 2 * (VC_PAGE_TOKENS * g + i), 2);
        }
    return VC_OK;
}

vc_status vc_comp_block_encode(const vc_kv_format *fmt, int32_t kind, const uint8_t *codes, const uint16_t *scales,
                               const uint16_t *zeros, void *block) {
    if (!fmt_ok(fmt) || (kind != 0 && kind != 1) || !block || !codes || !scales || !zeros)
        return VC_ERR_INVALID_ARG;
    const int b = fmt->bits, d = fmt->head_dim, g = d / VC_GROUP;
    uint8_t *blk = static_cast<uint8_t *>(block);
    const int row = d * b / 8, cr = VC_PAGE_TOKENS * row;
    std::memset(blk, 0, (size_t)vc::head_block_bytes(b, d));
    for (int s = 0; s < VC_PAGE_TOKENS; ++s)
        for (int c = 0; c < d; ++c)
            for (int j = 0; j < b; ++j)
                put_bit(blk, stored_bit(kind, b, d, s, c, j), get_bit(codes + s * row, b * c + j));
    uint8_t *par = blk + cr;
    for (int s = 0; s < VC_PAGE_TOKENS; ++s)
        for (int gr = 0; gr < g; ++gr) {
            const int i = stored_param(kind, g, s, gr);
            std::memcpy(par + 2 * i, scales + s * g + gr, 2);
            std::memcpy(par + 2 * (VC_PAGE_TOKENS * g + i), zeros + s * g + gr, 2);
        }
    return VC_OK;
}

}  // extern "C"
