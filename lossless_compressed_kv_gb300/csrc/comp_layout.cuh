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
//  * V codes, regions per fragment thread (g, t) of the V^T P^T product:
//    thread (g, t) owns the codes of channels {16 mt + g, 16 mt + 8 + g}
//    (all m-tiles mt) for tokens {2t, 2t+1, 2t+8, 2t+9}.  An operand
//    register holds one channel of tokens (2t, 2t+1) or (2t+8, 2t+9); the
//    four registers of an m-tile sit at positions p, p+VHI (second token
//    pair) and, for the row g+8 channel, 4 higher (2- and 3-bit) or one
//    byte higher (4-bit).
//  * 3 bits: the low two bits of each code use the 2-bit placement, the high
//    bit a separate plane placed so that one shift and mask put it right
//    above the low bits of its register.
//
// Offsets are in bits from the start of the head block's code region (K) or
// the V block's code region; every code of a plane lies inside one 32-bit
// word.  Scales and zeros: K as fp16 [16 tokens][G], V as fp16
// [4][G][4] with entry [t][group][i] for token 2t + (i & 1) + 8 (i >> 1).
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
__host__ __device__ inline int v_bit(int bits, int D, int tau, int c, int plane) {
    const int g = c & 7, row8 = (c >> 3) & 1, mt = c >> 4;
    const int t = (tau >> 1) & 3, hi = tau >> 3, half = tau & 1;
    const int region = g * 4 + t;
    if (bits == 4) return 32 * (region * (D / 16) + mt) + 16 * half + 8 * row8 + 4 * hi;
    const int u = mt >> 1, m = mt & 1;  // word of the region: one 32-channel group
    if (plane == 0) return 32 * (region * (D / 32) + u) + 16 * half + 8 * m + 4 * row8 + 2 * hi;
    // 3 bits, high bit of the register at low-plane position p = 2 j (j < 4)
    // of word u, shift 8 m: placed in a high-plane word so that one of four
    // shifts lines it up at p + 2
    const int j = 2 * row8 + hi;
    const int set = 2 * (u & 1) + m;
    const int beta = 2 * j + (set == 0 ? 0 : set == 1 ? 1 : set == 2 ? 8 : 9);
    return 32 * D + 32 * (region * (D / 64) + (u >> 1)) + 16 * half + beta;
}

// Element index (in fp16 units from the start of the V scale array) of the
// scale / zero of token tau, group gr; G = D / 32 groups.
__host__ __device__ inline int v_param(int G, int tau, int gr) {
    const int t = (tau >> 1) & 3, i = 2 * (tau >> 3) + (tau & 1);
    return (t * G + gr) * 4 + i;
}

}  // namespace layout
}  // namespace vc
