// Placement of the quantised codes inside a KV_comp head block (bits 2, 3
// and 4; head_dim D a multiple of 64).  The same bytes hold the same codes
// as a plain little-endian packing would; only their order differs, chosen
// so that the draft kernel turns packed words into tensor-core operands with
// one mask (sometimes one shift) per 32-bit operand register:
//
//  * K codes, 16 token rows of D*bits/8 bytes.  A row is split into four
//    thread regions t = 0..3; region t holds the codes of channels
//    16 ks + 4 t + e (ks < D/16, e < 4), i.e. the four channels that thread t
//    of an m16n8k16 fragment supplies in k-step ks.  Channel 16 ks + 4 t + e
//    is operand register r = 2 ks + (e >> 1), half e & 1: the two codes of a
//    register sit at the same bit position of the two 16-bit halves of one
//    word, so a mask leaves two f16 subnormals that are exactly code * 2^(p-24).
//  * V codes: channel-major (see v_bit), so that a thread holding one channel
//    reads that channel's codes of a page in one or two words.
//  * 3 bits (K): the low two bits of each code use the 2-bit placement, the
//    high bit a separate plane placed so that one shift and mask put it right
//    above the low bits of its register.
//
// Offsets are in bits from the start of the head block's code region (K) or
// the V block's code region; every code of a plane lies inside one 32-bit
// word.  Scales and zeros: fp16 [16 tokens][G] for K and V.
#pragma once

namespace vc {
namespace layout {

// K code of channel c of token row s; plane 1 = high bit of a 3-bit code.
__host__ __device__ inline int k_bit(int bits, int D, int s, int c, int plane) {
    const int ks = c >> 4, t = (c >> 2) & 3, e = c & 3;
    const int r = 2 * ks + (e >> 1), half = e & 1;
    if (bits == 2) return s * 2 * D + t * (D / 2) + 32 * (r >> 3) + 16 * half + 2 * (r & 7);
    if (bits == 4) return s * 4 * D + t * D + 32 * (r >> 2) + 16 * half + 4 * (r & 3);
    // 3 bits
    if (plane == 0) return s * 3 * D + t * (D / 2) + 32 * (r >> 3) + 16 * half + 2 * (r & 7);
    const int u = r >> 3, j = r & 7;
    const int set = 2 * (u & 1) + (j >> 2);
    const int beta = 2 * (j & 3) + (set == 0 ? 0 : set == 1 ? 1 : set == 2 ? 8 : 9);
    if (D == 64) return s * 3 * D + 2 * D + t * 16 + 8 * half + beta;
    return s * 3 * D + 2 * D + t * (D / 4) + 32 * (u >> 1) + 16 * half + beta;
}

// V code of token tau of channel c; plane 1 = high bit of a 3-bit code.
// Channel-major: the tensor-memory operand of the tcgen05 draft kernel (lane
// = channel, column = token pair) comes out of a channel's words with one
// mask (or one shift and a mask, plus for 3 bits one merge) per column.
//  * bits 2: one 32-bit word per channel, token tau at bit 16 (tau & 1) +
//    2 (tau >> 1).
//  * bits 3: the low two bits as bits 2 (words 0 .. D-1), then one 32-bit
//    high-bit word per channel pair, bit 16 (tau & 1) + 2 (tau >> 1) + (c & 1).
//  * bits 4: two words per channel (tokens 0-7, 8-15), token tau at bit
//    16 (tau & 1) + 4 ((tau & 7) >> 1) of word 2 c + (tau >> 3).
__host__ __device__ inline int v_bit(int bits, int D, int tau, int c, int plane) {
    if (bits == 4) return 32 * (2 * c + (tau >> 3)) + 16 * (tau & 1) + 4 * ((tau & 7) >> 1);
    if (bits == 2 || plane == 0) return 32 * c + 16 * (tau & 1) + 2 * (tau >> 1);
    return 32 * D + 32 * (c >> 1) + 16 * (tau & 1) + 2 * (tau >> 1) + (c & 1);
}

// Element index (in fp16 units from the start of the V scale array) of the
// scale / zero of token tau, group gr; G = D / 32 groups: [16][G], a token's
// parameters together (as for K).
__host__ __device__ inline int v_param(int bits, int G, int tau, int gr) {
    (void)bits;
    return tau * G + gr;
}

}  // namespace layout
}  // namespace vc
