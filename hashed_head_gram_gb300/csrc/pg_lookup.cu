// Hashing and gather kernels of the N-gram lookup (sm_103a).
//
// pg_canon_hash          one thread per (token, order, head): writes x'_t, rows, sign words.
// pg_gather_sign_concat  one warp per token (grid-stride, persistent grid):
//   phase A  lanes 0..3 read the token window and canonicalise it; lane l owns item
//            l = (order o, head k), whose multipliers it computed once at kernel start,
//            and hashes it to a row (+ the 64-bit sign hash); sign words follow.
//   phase B  the token's rows are streamed in 16-byte chunks: chunk c covers bytes
//            [16c, 16c+16) of the token's concatenated e_t, so every warp store writes
//            512 contiguous bytes and every load reads 16 bytes of one row. In PageGram
//            mode all K rows of an order lie in one K*S-row page block (4 KiB for
//            bf16 r=64, S=4; 1088 B for NF4), so each order is served from one
//            contiguous segment (PageGram tech report, section 3.1).
// Sources: PageGram report sections 2.1, 2.2, 3.1, 3.3; Engram notes (arXiv 2601.07372)
// section 3.2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pg_internal.cuh"

namespace pg {
namespace {

constexpr int kWarps = 8;            // warps per block of the gather kernel
constexpr int kMaxItems = 32;        // (order, head) items per token in the gather kernel
constexpr int kMaxSignWords = 128;   // items * sign words per token in the gather kernel

// NF4 levels: normal quantiles at evenly spaced probabilities (7 negative, exact zero,
// 8 positive; outermost probability 1 - (1/30 + 1/32)/2), scaled to [-1, 1]; the
// QLoRA NormalFloat-4 construction (PageGram report 3.3 names the data type).
__constant__ uint32_t c_nf4_bits[16] = {
    0xbf800000u, 0xbf3239b1u, 0xbf066b2eu, 0xbeca329eu, 0xbe91a24bu, 0xbe3d353du,
    0xbdba7869u, 0x00000000u, 0x3da2fb01u, 0x3e24cadfu, 0x3e7c04dau, 0x3ead0336u,
    0x3ee1a4b5u, 0x3f1007a9u, 0x3f3913b0u, 0x3f800000u};

__device__ __forceinline__ uint32_t fold32(uint64_t h) { return static_cast<uint32_t>(h ^ (h >> 32)); }

__device__ __forceinline__ uint64_t multiplier(uint64_t seed, int kind, int o, int k, int j) {
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

// Row of item (o, k) from its head (and page) hash; `hh` = H of the head hash,
// `hp` = H of the page hash (PageGram only).
__device__ __forceinline__ uint32_t row_from_hashes(const HashParams& p, int o, int k,
                                                    uint32_t hp, uint32_t hh) {
  if (p.mode == PG_PAGEGRAM) {
    const uint32_t page = hp % p.divisor[o][0];
    const uint32_t slot = hh % static_cast<uint32_t>(p.S);
    return p.base[o][0] + (page * static_cast<uint32_t>(p.K) + static_cast<uint32_t>(k)) *
                              static_cast<uint32_t>(p.S) + slot;
  }
  if (p.mode == PG_ENGRAM) return p.base[o][k] + hh % p.divisor[o][k];
  return p.base[o][0] + hh % p.divisor[o][0];
}

// ------------------------------------------------------------------ K1: canon + hash

__global__ void __launch_bounds__(256) canon_hash_kernel(
    const __grid_constant__ HashParams P, uint64_t seed, const int32_t* __restrict__ tokens,
    int64_t B, int64_t L, const uint32_t* __restrict__ canon_map, uint32_t* __restrict__ canon_out,
    uint32_t* __restrict__ rows_out, uint64_t* __restrict__ sign_out, int32_t* err) {
  const int items = P.O * P.H;
  const int64_t total = B * L * items;
  for (int64_t gid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; gid < total;
       gid += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = gid / items;
    const int item = static_cast<int>(gid - tok * items);
    const int o = item / P.H, k = item - (item / P.H) * P.H;
    const int64_t b = tok / L, t = tok - b * L;
    const int n = P.order_n[o];
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      c[j] = (j < n || (P.hash_kind == PG_HASH_TOY && j < 2))
                 ? (t - j >= 0 ? canon_token(tokens, canon_map, P.vocab, b * L + t - j, err) : kPad)
                 : kPad;
    if (canon_out && item == 0) canon_out[tok] = c[0];
    uint32_t row;
    uint64_t hs = 0;
    if (P.hash_kind == PG_HASH_TOY) {
      row = t >= 1 ? static_cast<uint32_t>((3ull * c[1] + c[0]) % P.toy_m) : PG_NO_ROW;
    } else {
      uint64_t hp = 0, hh = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < n) {
          hp ^= static_cast<uint64_t>(c[j]) * multiplier(seed, 0, o, 0, j);
          hh ^= static_cast<uint64_t>(c[j]) * multiplier(seed, 1, o, k, j);
          hs ^= static_cast<uint64_t>(c[j]) * multiplier(seed, 2, o, k, j);
        }
      row = row_from_hashes(P, o, k, fold32(hp), fold32(hh));
    }
    rows_out[gid] = row;
    if (sign_out)
      for (int q = 0; q < P.W; ++q)
        sign_out[gid * P.W + q] =
            P.hash_kind == PG_HASH_TOY ? 0ull : mix64(hs + kGolden * static_cast<uint64_t>(q + 1));
  }
}

// ------------------------------------------------------------------ K2: fused gather

struct WarpScratch {
  uint32_t row[kMaxItems];
  uint64_t hsign[kMaxItems];
  uint64_t sign[kMaxSignWords];
};

__device__ __forceinline__ uint4 ldg_stream(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

__device__ __forceinline__ uint16_t ldg_u16(const void* ptr) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(ptr));
  return v;
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

// XOR masks that negate 4 fp32 from 4 sign bits.
__device__ __forceinline__ uint4 f32_sign_mask(uint32_t bits) {
  return make_uint4((bits & 1u) << 31, (bits & 2u) << 30, (bits & 4u) << 29, (bits & 8u) << 28);
}

__device__ __forceinline__ uint4 xor4(uint4 a, uint4 b) {
  return make_uint4(a.x ^ b.x, a.y ^ b.y, a.z ^ b.z, a.w ^ b.w);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Registers are capped so that NCH <= 4 variants keep 32 warps per SM resident.
template <int ROWT, int OUTT, bool FLAT, int NCH>
__global__ void __launch_bounds__(kWarps * 32, NCH <= 4 ? 4 : (NCH <= 8 ? 2 : 1)) gather_kernel(
    const __grid_constant__ HashParams P, uint64_t seed, const int32_t* __restrict__ tokens,
    int64_t B, int64_t L, const uint32_t* __restrict__ canon_map,
    const uint8_t* __restrict__ table, uint32_t row_bytes, uint32_t rc, uint32_t rc_magic,
    uint8_t* __restrict__ e_out, uint32_t e_bytes, int32_t* err) {
  __shared__ WarpScratch scratch[kWarps];
  __shared__ float s_nf4[16];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  WarpScratch& ws = scratch[warp];
  if (ROWT == PG_NF4 && threadIdx.x < 16) s_nf4[threadIdx.x] = __uint_as_float(c_nf4_bits[threadIdx.x]);
  __syncthreads();

  const int items = P.O * P.H;
  const int W = P.W;
  // This lane's item and its multipliers (fixed for the whole kernel).
  const bool has_item = lane < items;
  const int io = has_item ? lane / P.H : 0;
  const int ik = has_item ? lane - io * P.H : 0;
  const int n = P.order_n[io];
  int nmax = 0;
  for (int o = 0; o < P.O; ++o) nmax = max(nmax, P.order_n[o]);
  uint64_t mp[4], mh[4], ms[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mp[j] = multiplier(seed, 0, io, 0, j);
    mh[j] = multiplier(seed, 1, io, ik, j);
    ms[j] = multiplier(seed, 2, io, ik, j);
  }
  // Row of this lane's item = lane_base + (H_page mod div_main) * stride + H_head mod S
  // (PageGram), or lane_base + H_head mod div_main (Engram, flat).
  const bool paged = P.mode == PG_PAGEGRAM;
  const uint32_t div_main = paged ? P.divisor[io][0] : P.divisor[io][P.mode == PG_ENGRAM ? ik : 0];
  const uint32_t slots = static_cast<uint32_t>(P.S);
  const uint32_t stride = static_cast<uint32_t>(P.K) * slots;
  const uint32_t lane_base = paged ? P.base[io][0] + static_cast<uint32_t>(ik) * slots
                                   : P.base[io][P.mode == PG_ENGRAM ? ik : 0];

  const int64_t N = B * L;
  const int64_t warp_stride = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * kWarps + warp; tok < N; tok += warp_stride) {
    const int64_t b = tok / L, t = tok - b * L;
    // ---- phase A: window, hashes, rows, sign words
    uint32_t cj = kPad;
    if (lane < nmax && t - lane >= 0) cj = canon_token(tokens, canon_map, P.vocab, tok - lane, err);
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = __shfl_sync(0xffffffffu, cj, j);
    if (has_item) {
      uint64_t hp = 0, hh = 0, hs = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < n) {
          const uint64_t cv = c[j];
          hp ^= cv * mp[j];
          hh ^= cv * mh[j];
          hs ^= cv * ms[j];
        }
      const uint32_t h32 = fold32(hh);
      ws.row[lane] = paged ? lane_base + (fold32(hp) % div_main) * stride + h32 % slots
                           : lane_base + h32 % div_main;
      ws.hsign[lane] = hs;
    }
    __syncwarp();
    for (int s = lane; s < items * W; s += 32) {
      const int it = s / W;
      ws.sign[s] = mix64(ws.hsign[it] + kGolden * static_cast<uint64_t>(s - it * W + 1));
    }
    __syncwarp();

    // ---- phase B: gather, dequantise, sign, concat (or flat sum)
    uint8_t* out_tok = e_out + static_cast<uint64_t>(tok) * e_bytes;
    if constexpr (FLAT) {
      // rc chunks of 16 bytes per row; every order contributes to every chunk.
      constexpr int E = ROWT == PG_F32 ? 4 : 8;   // elements per chunk
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int cidx = lane + 32 * i;
        if (cidx < static_cast<int>(rc)) {
          float acc[E];
          for (int o = 0; o < P.O; ++o) {
            const uint4 v = ldg_stream(table + static_cast<uint64_t>(ws.row[o]) * row_bytes +
                                       static_cast<uint32_t>(cidx) * 16u);
            const int e0 = cidx * E;
            const uint32_t bits =
                static_cast<uint32_t>(ws.sign[o * W + (e0 >> 6)] >> (e0 & 63)) & ((1u << E) - 1u);
            float x[E];
            if constexpr (ROWT == PG_F32) {
              const uint4 f = xor4(v, f32_sign_mask(bits));
              x[0] = __uint_as_float(f.x); x[1] = __uint_as_float(f.y);
              x[2] = __uint_as_float(f.z); x[3] = __uint_as_float(f.w);
            } else {
              const uint4 f = xor4(v, bf16_sign_mask(bits));
              x[0] = bf16_lo(f.x); x[1] = bf16_hi(f.x); x[2] = bf16_lo(f.y); x[3] = bf16_hi(f.y);
              x[4] = bf16_lo(f.z); x[5] = bf16_hi(f.z); x[6] = bf16_lo(f.w); x[7] = bf16_hi(f.w);
            }
#pragma unroll
            for (int q = 0; q < E; ++q) acc[q] = (o == 0) ? x[q] : __fadd_rn(acc[q], x[q]);
          }
          if constexpr (OUTT == PG_F32) {
#pragma unroll
            for (int q = 0; q < E; q += 4)
              *reinterpret_cast<uint4*>(out_tok + (static_cast<uint32_t>(cidx) * E + q) * 4u) =
                  make_uint4(__float_as_uint(acc[q]), __float_as_uint(acc[q + 1]),
                             __float_as_uint(acc[q + 2]), __float_as_uint(acc[q + 3]));
          } else {
            uint4 o4;
            o4.x = pack_bf16(acc[0], acc[1]);
            o4.y = pack_bf16(acc[2], acc[3]);
            o4.z = pack_bf16(acc[4], acc[5]);
            o4.w = pack_bf16(acc[6], acc[7]);
            *reinterpret_cast<uint4*>(out_tok + static_cast<uint32_t>(cidx) * 16u) = o4;
          }
        }
      }
    } else if constexpr (ROWT == PG_NF4) {
      // task c = (item, piece of 8 elements); codes at bytes [4*piece, 4*piece + 4) of
      // the 34-byte row (2-byte aligned), scale at bytes 32..33.
      const int tasks = items * 8;
      uint32_t codes[NCH];
      uint16_t sbits[NCH];
      uint32_t bits[NCH];
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int cidx = lane + 32 * i;
        if (cidx < tasks) {
          const int it = cidx >> 3, piece = cidx & 7;
          const uint8_t* rowp = table + static_cast<uint64_t>(ws.row[it]) * 34u;
          const uint32_t lo = ldg_u16(rowp + 4 * piece);
          const uint32_t hi = ldg_u16(rowp + 4 * piece + 2);
          codes[i] = lo | (hi << 16);
          sbits[i] = ldg_u16(rowp + 32);
          bits[i] = static_cast<uint32_t>(ws.sign[it * W] >> (piece * 8)) & 0xFFu;
        }
      }
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int cidx = lane + 32 * i;
        if (cidx < tasks) {
          const float scale = __half2float(__ushort_as_half(sbits[i]));
          float x[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float v = s_nf4[(codes[i] >> (4 * q)) & 15u] * scale;
            x[q] = ((bits[i] >> q) & 1u) ? -v : v;
          }
          if constexpr (OUTT == PG_F32) {
            uint8_t* dst = out_tok + static_cast<uint32_t>(cidx) * 32u;
            *reinterpret_cast<uint4*>(dst) = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                                                        __float_as_uint(x[2]), __float_as_uint(x[3]));
            *reinterpret_cast<uint4*>(dst + 16) = make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]),
                                                             __float_as_uint(x[6]), __float_as_uint(x[7]));
          } else {
            uint4 o4;
            o4.x = pack_bf16(x[0], x[1]);
            o4.y = pack_bf16(x[2], x[3]);
            o4.z = pack_bf16(x[4], x[5]);
            o4.w = pack_bf16(x[6], x[7]);
            *reinterpret_cast<uint4*>(out_tok + static_cast<uint32_t>(cidx) * 16u) = o4;
          }
        }
      }
    } else {
      // multi-head f32 / bf16 rows: chunk c = (item, piece); item = c / rc.
      constexpr int E = ROWT == PG_F32 ? 4 : 8;
      const int chunks = items * static_cast<int>(rc);
      uint4 v[NCH];
      uint32_t bits[NCH];
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const uint32_t cidx = static_cast<uint32_t>(lane + 32 * i);
        if (cidx < static_cast<uint32_t>(chunks)) {
          const uint32_t it = rc == 1u ? cidx : __umulhi(cidx, rc_magic);
          const uint32_t piece = cidx - it * rc;
          v[i] = ldg_stream(table + static_cast<uint64_t>(ws.row[it]) * row_bytes + piece * 16u);
          const uint32_t e0 = piece * E;
          bits[i] = static_cast<uint32_t>(ws.sign[it * W + (e0 >> 6)] >> (e0 & 63)) & ((1u << E) - 1u);
        }
      }
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const uint32_t cidx = static_cast<uint32_t>(lane + 32 * i);
        if (cidx < static_cast<uint32_t>(chunks)) {
          if constexpr (ROWT == PG_F32) {
            *reinterpret_cast<uint4*>(out_tok + cidx * 16u) = xor4(v[i], f32_sign_mask(bits[i]));
          } else if constexpr (OUTT == PG_BF16) {
            *reinterpret_cast<uint4*>(out_tok + cidx * 16u) = xor4(v[i], bf16_sign_mask(bits[i]));
          } else {
            const uint4 f = xor4(v[i], bf16_sign_mask(bits[i]));
            uint8_t* dst = out_tok + cidx * 32u;
            *reinterpret_cast<uint4*>(dst) = make_uint4(f.x << 16, f.x & 0xFFFF0000u,
                                                        f.y << 16, f.y & 0xFFFF0000u);
            *reinterpret_cast<uint4*>(dst + 16) = make_uint4(f.z << 16, f.z & 0xFFFF0000u,
                                                             f.w << 16, f.w & 0xFFFF0000u);
          }
        }
      }
    }
    __syncwarp();
  }
}

using GatherFn = void (*)(const HashParams, uint64_t, const int32_t*, int64_t, int64_t,
                          const uint32_t*, const uint8_t*, uint32_t, uint32_t, uint32_t, uint8_t*,
                          uint32_t, int32_t*);

template <int ROWT, int OUTT, bool FLAT>
GatherFn pick_nch(int nch) {
  if (nch <= 2) return gather_kernel<ROWT, OUTT, FLAT, 2>;
  if (nch <= 4) return gather_kernel<ROWT, OUTT, FLAT, 4>;
  if (nch <= 8) return gather_kernel<ROWT, OUTT, FLAT, 8>;
  if (nch <= 16) return gather_kernel<ROWT, OUTT, FLAT, 16>;
  return nullptr;
}

GatherFn pick_gather(int row_dtype, int out_dtype, bool flat, int nch) {
  if (flat) {
    if (row_dtype == PG_F32 && out_dtype == PG_F32) return pick_nch<PG_F32, PG_F32, true>(nch);
    if (row_dtype == PG_BF16 && out_dtype == PG_BF16) return pick_nch<PG_BF16, PG_BF16, true>(nch);
    if (row_dtype == PG_BF16 && out_dtype == PG_F32) return pick_nch<PG_BF16, PG_F32, true>(nch);
    return nullptr;
  }
  if (row_dtype == PG_F32 && out_dtype == PG_F32) return pick_nch<PG_F32, PG_F32, false>(nch);
  if (row_dtype == PG_BF16 && out_dtype == PG_BF16) return pick_nch<PG_BF16, PG_BF16, false>(nch);
  if (row_dtype == PG_BF16 && out_dtype == PG_F32) return pick_nch<PG_BF16, PG_F32, false>(nch);
  if (row_dtype == PG_NF4 && out_dtype == PG_BF16) return pick_nch<PG_NF4, PG_BF16, false>(nch);
  if (row_dtype == PG_NF4 && out_dtype == PG_F32) return pick_nch<PG_NF4, PG_F32, false>(nch);
  return nullptr;
}

pg_status prepare_err(int32_t* err_index, cudaStream_t stream) {
  if (!err_index) return PG_OK;
  if (reinterpret_cast<uintptr_t>(err_index) % 4) return PG_ERR_ALIGN;
  // 0xFFFFFFFF reads as -1; the kernels lower it with an unsigned atomicMin.
  cudaError_t e = cudaMemsetAsync(err_index, 0xFF, sizeof(int32_t), stream);
  return e == cudaSuccess ? PG_OK : cuda_fail(e);
}

}  // namespace
}  // namespace pg

extern "C" {

pg_status pg_canon_hash(const pg_table_desc* desc, const int32_t* tokens, int32_t B, int32_t L,
                        const uint32_t* canon_map, uint32_t* canon_out, uint32_t* rows_out,
                        uint64_t* sign_out, int32_t* err_index, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  Geometry g;
  pg_status st = validate_desc(desc, &g);
  if (st != PG_OK) return st;
  if (B < 0 || L < 0) return PG_ERR_SHAPE;
  const int64_t N = static_cast<int64_t>(B) * L;
  if (N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (N == 0) return PG_OK;
  if (!tokens || !rows_out) return PG_ERR_NULL;
  if (sm_count() == 0) return cuda_fail(cudaGetLastError());
  st = prepare_err(err_index, stream);
  if (st != PG_OK) return st;
  HashParams P;
  fill_hash_params(desc, g, &P);
  const int64_t total = N * g.O * g.H;
  const int64_t want = (total + 255) / 256;
  const int blocks = static_cast<int>(want < sm_count() * 8ll ? want : sm_count() * 8ll);
  canon_hash_kernel<<<blocks, 256, 0, stream>>>(P, desc->hash_seed, tokens, B, L, canon_map,
                                                canon_out, rows_out, sign_out, err_index);
  return after_launch(1);
}

pg_status pg_gather_sign_concat(const pg_table_desc* desc, const int32_t* tokens, int32_t B,
                                int32_t L, const uint32_t* canon_map, const void* table,
                                uint64_t table_bytes, void* e_out, int32_t out_dtype,
                                int32_t* err_index, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  Geometry g;
  pg_status st = validate_desc(desc, &g);
  if (st != PG_OK) return st;
  if (desc->hash_kind != PG_HASH_MULXOR) return PG_ERR_UNSUPPORTED;
  if (B < 0 || L < 0) return PG_ERR_SHAPE;
  const int64_t N = static_cast<int64_t>(B) * L;
  if (N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (N == 0) return PG_OK;
  if (!tokens || !table || !e_out) return PG_ERR_NULL;
  if (table_bytes < g.rows * g.row_bytes) return PG_ERR_RANGE;
  if (reinterpret_cast<uintptr_t>(table) % 16 || reinterpret_cast<uintptr_t>(e_out) % 16)
    return PG_ERR_ALIGN;
  if (out_dtype != PG_F32 && out_dtype != PG_BF16) return PG_ERR_DTYPE;
  const bool flat = desc->mode == PG_FLAT;
  const int items = g.O * g.H;
  if (items > kMaxItems || items * g.W > kMaxSignWords) return PG_ERR_UNSUPPORTED;
  if (desc->row_dtype != PG_NF4 && g.row_bytes % 16) return PG_ERR_UNSUPPORTED;
  uint32_t rc = desc->row_dtype == PG_NF4 ? 8u : g.row_bytes / 16u;
  int nch;
  if (flat) nch = (static_cast<int>(rc) + 31) / 32;
  else nch = (items * static_cast<int>(rc) + 31) / 32;
  GatherFn fn = pick_gather(desc->row_dtype, out_dtype, flat, nch);
  if (!fn) return desc->row_dtype == PG_F32 && out_dtype == PG_BF16 ? PG_ERR_DTYPE : PG_ERR_UNSUPPORTED;
  const uint32_t out_size = out_dtype == PG_F32 ? 4u : 2u;
  const uint32_t e_bytes = g.e_width * out_size;
  // item = umulhi(chunk, magic) = floor(chunk / rc), exact while chunk * rc < 2^32
  const uint32_t rc_magic = rc == 1u ? 0u : static_cast<uint32_t>((1ull << 32) / rc + 1ull);
  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  st = prepare_err(err_index, stream);
  if (st != PG_OK) return st;
  HashParams P;
  fill_hash_params(desc, g, &P);
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, reinterpret_cast<const void*>(fn), kWarps * 32, 0);
  if (e != cudaSuccess) return cuda_fail(e);
  if (per_sm < 1) per_sm = 1;
  const int64_t want = (N + kWarps - 1) / kWarps;
  const int blocks = static_cast<int>(want < static_cast<int64_t>(nsm) * per_sm ? want
                                                                              : static_cast<int64_t>(nsm) * per_sm);
  fn<<<blocks, kWarps * 32, 0, stream>>>(P, desc->hash_seed, tokens, B, L, canon_map,
                                         static_cast<const uint8_t*>(table), g.row_bytes, rc, rc_magic,
                                         static_cast<uint8_t*>(e_out), e_bytes, err_index);
  return after_launch(1);
}

}  // extern "C"
