// Gather-side definitions shared by the lookup kernels (pg_lookup.cu) and the one-launch
// decode step (pg_decode_step.cu): the gather geometry, the NF4 levels, sign masks, and the
// per-sequence body of the streaming decode lookup, so that both produce bit-identical e_t.
// Sources: PageGram report sections 3.1 (page-local rows), 3.3 (NF4 rows); Engram notes
// (arXiv 2601.07372) sections 3.2 (multi-head hashing), 3.5 (addressing known ahead).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pg_hash.cuh"

namespace pg {
namespace {

constexpr int kMaxItems = 32;       // (order, head) items per token
constexpr int kMaxSignWords = 128;  // items * sign words per token

struct GatherGeom {
  int64_t N;            // tokens
  uint32_t L;           // sequence length
  uint64_t fm_L;        // fastmod constant of L
  int items;            // O * H
  int W;                // sign words per item
  int tb;               // tokens per batch
  int per_tok;          // chunks (or NF4 tasks) per token
  uint32_t tok_magic;   // floor(c / per_tok) = umulhi(c, tok_magic)
  uint32_t rc;          // 16-byte chunks per stored row (multi-head f32/bf16), or per row (flat)
  uint32_t rc_magic;
  uint32_t row_bytes;
  uint32_t e_bytes;     // bytes of one token's e_t
  int64_t nbatch;
  uint64_t table_bytes; // NF4: bytes of the table (the last rows' 16-byte windows stop there)
};

// NF4 levels: QLoRA's NormalFloat-4 values as printed in its paper (Dettmers et al. 2023,
// Appendix E; the PageGram report, section 3.3, names the data type): normal quantiles at
// evenly spaced probabilities (7 negative, exact zero, 8 positive), scaled to [-1, 1].
__constant__ uint32_t c_nf4_bits[16] = {
    0xbf800000u, 0xbf3239b1u, 0xbf066b30u, 0xbeca32a0u, 0xbe91a24du, 0xbe3d353fu,
    0xbdba7871u, 0x00000000u, 0x3da2faffu, 0x3e24cae3u, 0x3e7c04ddu, 0x3ead033au,
    0x3ee1a4b8u, 0x3f1007abu, 0x3f3913b3u, 0x3f800000u};

// XOR masks that negate 4 fp32 from 4 sign bits.
__device__ __forceinline__ uint4 f32_sign_mask(uint32_t bits) {
  return make_uint4((bits & 1u) << 31, (bits & 2u) << 30, (bits & 4u) << 29, (bits & 8u) << 28);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ streaming decode lookup

// One new token of sequence b, by one warp. With t = pos[b], the window is the token's
// canonical ID (c_0) and, for 1 <= j <= t, the ID ring's slot (t - j) mod 4 (kPad before
// the start of the sequence: the same window item_row reads from a [B, L] batch). Lanes <
// items hash one (order, head) item each into s_rows / s_signs (the warp's own); the warp
// then walks the token's e_t in the gather kernels' units (16-byte chunks of a stored row;
// NF4: 8-element pieces) with their arithmetic, so e_t (written to out_tok, global or shared
// memory) is bit-identical to pg_gather_sign_concat's. The gather ends with a __syncwarp
// (every lane has read pos and the ring and is done with s_rows); the caller then writes
// ids[b][t mod 4] and pos[b]. A negative t is reported as device error bit 512 and nothing
// is written.

// The window of sequence b's new token, by one warp: returns t = pos[b] and the token's
// canonical ID in *c0_out (both in every lane), lanes < 4 the ID ring's slot `lane` in
// *slot_out. Only loads: the hash constants are not needed yet.
__device__ __forceinline__ int decode_token_window(const HashParams& P, int b, int lane,
                                                   const int32_t* __restrict__ tokens,
                                                   const uint32_t* __restrict__ canon_map, const int32_t* pos,
                                                   const uint32_t* ids, int32_t* err, uint32_t* c0_out,
                                                   uint32_t* slot_out) {
  int t = 0;
  uint32_t c0 = 0, slot_id = 0;
  if (lane < 4) slot_id = ids[4 * static_cast<int64_t>(b) + lane];
  if (lane == 0) {
    t = pos[b];
    c0 = canon_token(tokens, canon_map, P.vocab, b, err);
  }
  *c0_out = __shfl_sync(0xffffffffu, c0, 0);
  *slot_out = slot_id;
  return __shfl_sync(0xffffffffu, t, 0);
}

// The hashes and the gather of sequence b from its window (t, c0, the lanes' ID ring
// slots). Returns t.
template <int ROWT, int OUTT, bool FLAT>
__device__ __forceinline__ int decode_token_gather(const HashParams& P, const GatherGeom& g,
                                                   const ItemConst* __restrict__ s_ic, const float* s_nf4,
                                                   uint32_t* s_rows, uint64_t* s_signs, int lane, int t,
                                                   uint32_t c0, uint32_t slot_id,
                                                   const uint8_t* __restrict__ table, uint8_t* out_tok,
                                                   int* err_word) {
  const int items = g.items;
  if (t < 0) {  // not a position any call writes: the sequence is left as it is
    if (lane == 0 && err_word) atomicOr(err_word, 512);
    return t;
  }
  uint64_t c[4];
  c[0] = c0;
#pragma unroll
  for (int j = 1; j < 4; ++j) {
    const uint32_t id = __shfl_sync(0xffffffffu, slot_id, (t - j) & 3);
    c[j] = t >= j ? id : kPad;
  }
  if (lane < items) {
    uint64_t hs;
    s_rows[lane] = item_row_ids(s_ic[lane], P.mode, c, &hs);
    for (int q = 0; q < g.W; ++q) s_signs[lane * g.W + q] = mix64(hs + kGolden * static_cast<uint64_t>(q + 1));
  }
  __syncwarp();
  const uint32_t* rows = s_rows;
  const uint64_t* signs = s_signs;
  for (int cc = lane; cc < g.per_tok; cc += 32) {
    if constexpr (ROWT == PG_NF4) {
      // piece cc & 7 of item cc >> 3: codes of elements 8 piece .. 8 piece + 7, the row's scale
      const int it = cc >> 3, piece = cc & 7;
      const uint8_t* w = table + static_cast<uint64_t>(rows[it]) * 34u;
      const uint32_t codes = static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(w + 4 * piece))) |
                             (static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(w + 4 * piece + 2)))
                              << 16);
      const float scale = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const uint16_t*>(w + 32))));
      const uint32_t bits = static_cast<uint32_t>(signs[it * g.W] >> (8 * piece)) & 0xFFu;
      float x[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float val = s_nf4[(codes >> (4 * q)) & 15u] * scale;
        x[q] = ((bits >> q) & 1u) ? -val : val;
      }
      if constexpr (OUTT == PG_F32) {
        uint8_t* dst = out_tok + cc * 32u;
        *reinterpret_cast<uint4*>(dst) = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                                                    __float_as_uint(x[2]), __float_as_uint(x[3]));
        *reinterpret_cast<uint4*>(dst + 16) = make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]),
                                                         __float_as_uint(x[6]), __float_as_uint(x[7]));
      } else {
        *reinterpret_cast<uint4*>(out_tok + cc * 16u) = make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                                                                   pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
      }
    } else {
      constexpr int E = ROWT == PG_F32 ? 4 : 8;  // elements per 16-byte chunk
      if constexpr (FLAT) {
        // chunk cc of the d-wide row of every order, signed and summed in order
        float acc[E];
        for (int o = 0; o < items; ++o) {
          const uint4 x4 = ldg_stream(table + static_cast<uint64_t>(rows[o]) * g.row_bytes + cc * 16u);
          const uint32_t e0 = cc * E;
          const uint32_t bb = static_cast<uint32_t>(signs[o * g.W + (e0 >> 6)] >> (e0 & 63)) & ((1u << E) - 1u);
          float x[E];
          if constexpr (ROWT == PG_F32) {
            const uint4 f = xor4(x4, f32_sign_mask(bb));
            x[0] = __uint_as_float(f.x); x[1] = __uint_as_float(f.y);
            x[2] = __uint_as_float(f.z); x[3] = __uint_as_float(f.w);
          } else {
            const uint4 f = xor4(x4, bf16_sign_mask(bb));
            x[0] = bf16_lo(f.x); x[1] = bf16_hi(f.x); x[2] = bf16_lo(f.y); x[3] = bf16_hi(f.y);
            x[4] = bf16_lo(f.z); x[5] = bf16_hi(f.z); x[6] = bf16_lo(f.w); x[7] = bf16_hi(f.w);
          }
#pragma unroll
          for (int q = 0; q < E; ++q) acc[q] = (o == 0) ? x[q] : __fadd_rn(acc[q], x[q]);
        }
        if constexpr (OUTT == PG_F32) {
#pragma unroll
          for (int q = 0; q < E; q += 4)
            *reinterpret_cast<uint4*>(out_tok + (cc * E + q) * 4u) =
                make_uint4(__float_as_uint(acc[q]), __float_as_uint(acc[q + 1]), __float_as_uint(acc[q + 2]),
                           __float_as_uint(acc[q + 3]));
        } else {
          *reinterpret_cast<uint4*>(out_tok + cc * 16u) =
              make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                         pack_bf16(acc[6], acc[7]));
        }
      } else {
        const uint32_t it = cc / g.rc, piece = cc - it * g.rc;
        const uint4 v = ldg_stream(table + static_cast<uint64_t>(rows[it]) * g.row_bytes + piece * 16u);
        const uint32_t e0 = piece * E;
        const uint32_t bb = static_cast<uint32_t>(signs[it * g.W + (e0 >> 6)] >> (e0 & 63)) & ((1u << E) - 1u);
        if constexpr (ROWT == PG_F32) {
          *reinterpret_cast<uint4*>(out_tok + cc * 16u) = xor4(v, f32_sign_mask(bb));
        } else if constexpr (OUTT == PG_BF16) {
          *reinterpret_cast<uint4*>(out_tok + cc * 16u) = xor4(v, bf16_sign_mask(bb));
        } else {
          const uint4 f = xor4(v, bf16_sign_mask(bb));
          uint8_t* dst = out_tok + cc * 32u;
          *reinterpret_cast<uint4*>(dst) = make_uint4(f.x << 16, f.x & 0xFFFF0000u, f.y << 16, f.y & 0xFFFF0000u);
          *reinterpret_cast<uint4*>(dst + 16) = make_uint4(f.z << 16, f.z & 0xFFFF0000u, f.w << 16, f.w & 0xFFFF0000u);
        }
      }
    }
  }
  __syncwarp();  // every lane is done with s_rows / s_signs and has read pos and the ring
  return t;
}

// Both parts: returns t and the canonical ID in *c0_out.
template <int ROWT, int OUTT, bool FLAT>
__device__ __forceinline__ int decode_token_lookup(const HashParams& P, const GatherGeom& g,
                                                   const ItemConst* __restrict__ s_ic, const float* s_nf4,
                                                   uint32_t* s_rows, uint64_t* s_signs, int b, int lane,
                                                   const int32_t* __restrict__ tokens,
                                                   const uint32_t* __restrict__ canon_map,
                                                   const uint8_t* __restrict__ table, const int32_t* pos,
                                                   const uint32_t* ids, uint8_t* out_tok, int32_t* err,
                                                   int* err_word, uint32_t* c0_out) {
  uint32_t slot_id;
  const int t = decode_token_window(P, b, lane, tokens, canon_map, pos, ids, err, c0_out, &slot_id);
  return decode_token_gather<ROWT, OUTT, FLAT>(P, g, s_ic, s_nf4, s_rows, s_signs, lane, t, *c0_out, slot_id,
                                               table, out_tok, err_word);
}

}  // namespace
}  // namespace pg
