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
//  * V codes, one string of 16 token codes per channel (channel-major), the
//    D/8 strings that one fragment row-thread g needs stored contiguously.
//    Token tau is operand k-slot tau; the string puts tokens (2t, 2t+1) and
//    (2t+8, 2t+9) of thread t at the same position of the two halves.
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

// Index of channel c's string among the D V strings.
__host__ __device__ inline int v_string(int D, int c) {
    const int g = c & 7, hi8 = (c >> 3) & 1, mt = c >> 4;
    return g * (D / 8) + 2 * mt + hi8;
}

// V code of token tau of channel c; plane 1 = high bit of a 3-bit code.
__host__ __device__ inline int v_bit(int bits, int D, int tau, int c, int plane) {
    const int lam = v_string(D, c);
    const int t = (tau >> 1) & 3, h = tau >> 3, half = tau & 1;
    if (bits == 2) return 32 * lam + 16 * half + 4 * t + 2 * h;
    if (bits == 4) return 32 * (D * (t >> 1) + lam) + 16 * half + 8 * (t & 1) + 4 * h;
    if (plane == 0) return 32 * lam + 16 * half + 4 * t + 2 * h;
    const int sp = t == 0 ? 0 : t == 1 ? 1 : t == 2 ? 4 : 5;
    return 32 * D + 16 * lam + 8 * half + sp + 2 * h;
}

// Element index (in fp16 units from the start of the V scale array) of the
// scale / zero of token tau, group gr; G = D / 32 groups.
__host__ __device__ inline int v_param(int G, int tau, int gr) {
    const int t = (tau >> 1) & 3, i = 2 * (tau >> 3) + (tau & 1);
    return (t * G + gr) * 4 + i;
}

}  // namespace layout
}  // namespace vc
