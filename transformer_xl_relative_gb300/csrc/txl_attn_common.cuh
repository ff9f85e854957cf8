// txl_attn_common.cuh -- pieces shared by the two fused tcgen05 relative-attention kernels (one
// CTA per query tile, and the persistent one): shared-memory / TMEM layout constants, the query
// permutation of TMEM lanes, the per-row BD ring and the branch-free logits loop.
#pragma once

#include <cuda_bf16.h>

#include "txl_ptx.cuh"

namespace txl {
namespace attn {

constexpr int kTile = 16384;                 // 128 rows x 128 B: one swizzle-atom column
constexpr int kBdPitchWords = 132;           // per-row ring of 256 bf16 + 4 exchange words
constexpr int kBdBytes = 128 * kBdPitchWords * 4;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColBD = 256, kColO = 384;
constexpr uint32_t kColP = 448;             // P of the current tile when D <= 64 (see kSeparateP)
constexpr float kRescaleThreshold = 8.0f;    // log2 units: P values stay below 2^8

__device__ __forceinline__ int query_of_row(int li) { return 2 * (li & 63) + (li >> 6); }

// The two threads of row li meet at named barrier 2 + li/32 (64 threads: one warp per half).
__device__ __forceinline__ void pair_bar(int li) { named_bar_sync(2 + (li >> 5), 64); }

// ---------------------------------------------------------------------------------------------
// Logits of one thread's 64 columns of a tile (log2 domain): s = AC + BD(remapped), in place,
// returning their maximum.  The ring already carries the mask (-inf) and the clamp (the value of
// r[clamp_len]) in the positions concerned, so every tile runs this one branch-free loop.
__device__ __forceinline__ float logits_interior(float* s, const uint32_t* bdrow, int wbase)
{
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int m = 0; m < 32; ++m) {
        const uint32_t w = bdrow[(wbase - m) & 127];
        const float x0 = add_bf16hi_f32(w, s[2 * m]);
        const float x1 = add_bf16lo_f32(w, s[2 * m + 1]);
        s[2 * m] = x0;
        s[2 * m + 1] = x1;
        switch (m & 3) {
        case 0: m0 = fmax3(m0, x0, x1); break;
        case 1: m1 = fmax3(m1, x0, x1); break;
        case 2: m2 = fmax3(m2, x0, x1); break;
        default: m3 = fmax3(m3, x0, x1); break;
        }
    }
    return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// Copy this thread's half of a new BD chunk (64 fp32 columns, in registers) into the row's ring
// as bf16.  Chunk column c lives at ring position (128*(t&1) + c + sh) mod 256 (two positions per
// 32-bit word, the even one in the low half).  With sh = 1 the column pairs straddle words, so
// the words shared with the other half, or with the other ring slot, are written per 16 bits.
__device__ __forceinline__ void ring_write_half(uint32_t* bdrow, uint32_t row_saddr, const uint32_t* v,
                                                int t, int hf, int sh)
{
    uint32_t* slot = bdrow + 64 * (t & 1);
    const uint32_t slot_saddr = row_saddr + 256u * (t & 1);
    if (sh == 0) {
        // word 32hf + k = (lo: column 64hf + 2k, hi: column 64hf + 2k + 1)
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(__uint_as_float(v[8 * q4 + 2 * e]), __uint_as_float(v[8 * q4 + 2 * e + 1]));
            *reinterpret_cast<uint4*>(slot + 32 * hf + 4 * q4) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        // word 32hf + k = (lo: column 64hf + 2k - 1, hi: column 64hf + 2k)
        const uint16_t first = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[0])));
        const uint16_t last = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[63])));
        sts_u16(slot_saddr + 4u * (32 * hf) + 2u, first);             // hi half of word 32hf
#pragma unroll
        for (int k = 1; k < 4; ++k)
            slot[32 * hf + k] = pack_bf16x2(__uint_as_float(v[2 * k - 1]), __uint_as_float(v[2 * k]));
#pragma unroll
        for (int q4 = 1; q4 < 8; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 4 * q4 + e;
                w[e] = pack_bf16x2(__uint_as_float(v[2 * k - 1]), __uint_as_float(v[2 * k]));
            }
            *reinterpret_cast<uint4*>(slot + 32 * hf + 4 * q4) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        // column 64hf + 63 is the lo half of word 32hf + 32: word 32 of this slot for hf = 0,
        // word 0 of the other slot (ring position 128((t+1)&1)) for hf = 1
        const uint32_t dst = hf == 0 ? slot_saddr + 4u * 32 : row_saddr + 256u * ((t + 1) & 1);
        sts_u16(dst, last);
    }
}

}  // namespace attn
}  // namespace txl
