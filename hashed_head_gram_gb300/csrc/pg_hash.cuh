// Device-side hashing helpers shared by the lookup kernels (pg_lookup.cu) and the fused
// lookup + projection kernel (pg_project.cu). Hash definition: hash_version 1 (pg.h).
#pragma once

#include <cuda_bf16.h>

#include "pg_internal.cuh"

namespace pg {

__device__ __forceinline__ uint32_t fold32(uint64_t h) { return static_cast<uint32_t>(h ^ (h >> 32)); }

// Odd multiplier m_{kind,o,k,j} of hash_version 1.
__host__ __device__ __forceinline__ uint64_t multiplier(uint64_t seed, int kind, int o, int k, int j) {
  const uint64_t fid = static_cast<uint64_t>(((kind * 4 + o) * 64 + k) * 4 + j);
  return mix64(seed + kGolden * (1ull + fid)) | 1ull;
}

// Reads the canonical ID of token `src` (flat index); out-of-range IDs are reported
// through err (smallest flat index wins) and read as ID 0.
__device__ __forceinline__ uint32_t canon_token(const int32_t* __restrict__ tokens,
                                                const uint32_t* __restrict__ canon_map,
                                                uint32_t vocab, int64_t src, int32_t* err) {
  int32_t x = __ldg(tokens + src);
  if (x < 0 || static_cast<uint32_t>(x) >= vocab) {
    if (err) atomicMin(reinterpret_cast<unsigned int*>(err), static_cast<unsigned int>(src));
    x = 0;
  }
  return canon_map ? __ldg(canon_map + x) : static_cast<uint32_t>(x);
}

// Remainder by direct computation (Lemire, Kaser & Kurz, "Faster remainder by direct
// computation", Software: Practice and Experience 2019): with c = ceil(2^64 / d),
// a mod d = floor(((c * a) mod 2^64) * d / 2^64), exact for all 32-bit a and d >= 1
// (d = 1 gives c = 0 and the remainder 0).
__host__ __device__ __forceinline__ uint64_t fastmod_constant(uint32_t d) { return ~0ull / d + 1ull; }

__device__ __forceinline__ uint32_t fastmod(uint32_t a, uint64_t c, uint32_t d) {
  return static_cast<uint32_t>(__umul64hi(c * a, d));
}

// Per-(order, head) item constants, kept in shared memory by the kernels.
struct ItemConst {
  uint64_t mp[4], mh[4], ms[4];  // multipliers: page hash, head hash, sign hash
  uint64_t fm_main, fm_slot;     // fastmod constants of div_main and S
  uint32_t div_main;             // P_n (PageGram), M_{n,k} (Engram), R_n (flat)
  uint32_t slots;                // S (PageGram), 1 otherwise
  uint32_t stride;               // K * S (PageGram)
  uint32_t base;                 // row of (page 0, head k, slot 0) / subtable start
  int32_t n;                     // n-gram order
  int32_t pad;
};

__host__ __device__ __forceinline__ void init_item_const(ItemConst& it, const HashParams& P, uint64_t seed,
                                                         int item) {
  const int o = item / P.H, k = item - (item / P.H) * P.H;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    it.mp[j] = multiplier(seed, 0, o, 0, j);
    it.mh[j] = multiplier(seed, 1, o, k, j);
    it.ms[j] = multiplier(seed, 2, o, k, j);
  }
  const bool paged = P.mode == PG_PAGEGRAM;
  it.div_main = paged ? P.divisor[o][0] : P.divisor[o][P.mode == PG_ENGRAM ? k : 0];
  it.slots = paged ? static_cast<uint32_t>(P.S) : 1u;
  it.stride = paged ? static_cast<uint32_t>(P.K * P.S) : 0u;
  it.base = paged ? P.base[o][0] + static_cast<uint32_t>(k * P.S) : P.base[o][P.mode == PG_ENGRAM ? k : 0];
  it.fm_main = fastmod_constant(it.div_main);
  it.fm_slot = fastmod_constant(it.slots);
  it.n = P.order_n[o];
}

// Row of item `it` from the canonical IDs c_j of positions t - j (kPad before the start of
// the sequence; only j < n is read), and the 64-bit sign hash h_{2,o,k} through *hs:
//   PageGram  base_n + ((H_page mod P_n) K + k) S + (H_head mod S)
//   Engram    base_{n,k} + H_head mod M_{n,k};   flat  base_n + H_head mod R_n
__device__ __forceinline__ uint32_t item_row_ids(const ItemConst& it, int mode, const uint64_t (&c)[4], uint64_t* hs) {
  uint64_t hp = 0, hh = 0, h2 = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j < it.n) {
      hp ^= c[j] * it.mp[j];
      hh ^= c[j] * it.mh[j];
      h2 ^= c[j] * it.ms[j];
    }
  }
  *hs = h2;
  if (mode == PG_PAGEGRAM)
    return it.base + fastmod(fold32(hp), it.fm_main, it.div_main) * it.stride +
           fastmod(fold32(hh), it.fm_slot, it.slots);
  return it.base + fastmod(fold32(hh), it.fm_main, it.div_main);
}

// The same for token `tok` (position t in its sequence), reading the IDs it needs.
__device__ __forceinline__ uint32_t item_row(const ItemConst& it, int mode, const int32_t* __restrict__ tokens,
                                             const uint32_t* __restrict__ canon_map, uint32_t vocab, int64_t tok,
                                             uint32_t t, int32_t* err, uint64_t* hs) {
  uint64_t c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    c[j] = (j < it.n && t >= static_cast<uint32_t>(j)) ? canon_token(tokens, canon_map, vocab, tok - j, err) : kPad;
  return item_row_ids(it, mode, c, hs);
}

// XOR masks that negate 8 packed bf16 (two per 32-bit word) from 8 sign bits.
__device__ __forceinline__ uint4 bf16_sign_mask(uint32_t bits) {
  uint4 m;
  m.x = ((bits & 1u) << 15) | ((bits & 2u) << 30);
  m.y = ((bits & 4u) << 13) | ((bits & 8u) << 28);
  m.z = ((bits & 16u) << 11) | ((bits & 32u) << 26);
  m.w = ((bits & 64u) << 9) | ((bits & 128u) << 24);
  return m;
}

// 16 bytes of a table row: read-only, not kept in L1 (rows are rarely reused by one SM).
__device__ __forceinline__ uint4 ldg_stream(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

__device__ __forceinline__ uint4 xor4(uint4 a, uint4 b) {
  return make_uint4(a.x ^ b.x, a.y ^ b.y, a.z ^ b.z, a.w ^ b.w);
}

}  // namespace pg
