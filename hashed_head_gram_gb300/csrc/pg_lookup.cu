// Hashing and gather kernels of the N-gram lookup (sm_103a).
//
// pg_canon_hash          one thread per (token, order, head): writes x'_t, rows, sign words.
// pg_gather_sign_concat  persistent grid of 256-thread blocks:
//   Each warp takes batches of tb tokens (2 for K = 8 heads x 2 orders), independently:
//   phase A  one lane per (token, item = (order o, head k)): canonical window, the page /
//            head / sign multiply-XOR hashes, the row (remainders by direct computation)
//            and the sign words, into the warp's double-buffered shared memory;
//   phase B  the batch is streamed in 16-byte chunks, 8 per lane: chunk c of a token covers
//            bytes [16c, 16c+16) of its concatenated e_t, so 32 consecutive chunks are 512
//            contiguous bytes of e_t and 4 whole 128-byte rows of one page (PageGram: all K
//            rows of an order lie in one K*S-row page block, PageGram report section 3.1);
//   phase A of the warp's next batch runs while phase B's loads are in flight. A batch's
//   token IDs are read ahead of it by a few lanes (raw IDs two batches ahead, canonical IDs
//   one ahead) and handed to the hashing lanes by shuffles, so phase A issues no loads
//   (batches of one token keep per-lane ID reads).
//   NF4 rows (34 bytes) take their own kernel: windows copied into shared memory by
//   cp.async three batches ahead, dequantised from there (see gather_nf4_kernel).
// Sources: PageGram report sections 2.1, 2.2, 3.1, 3.3; Engram notes (arXiv 2601.07372)
// section 3.2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pg_conv_math.cuh"
#include "pg_gather.cuh"
#include "pg_hash.cuh"

namespace pg {
namespace {

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

// The IDs of a warp batch (tb consecutive tokens from flat position tb * batch) are loaded
// ahead of the batch, once per warp: lane q < tb + 3 holds the token at flat position
// tb * batch - 3 + q, which covers every n-gram window of the batch (n <= 4). Its raw ID is
// read first and its canonical ID from that later, each load in flight while the warp
// works on an earlier batch; the hashing lanes then take their n-gram's IDs by shuffles.
// tb <= kMaxBatchTokens keeps the window within the 32 lanes.
constexpr int kMaxBatchTokens = 32 - 3;

__device__ __forceinline__ bool window_has(const GatherGeom& g, int tb, int64_t batch, int lane) {
  const int64_t f = batch * tb - 3 + lane;
  return batch < g.nbatch && lane < tb + 3 && f >= 0 && f < g.N;
}

__device__ __forceinline__ int32_t window_raw_id(const GatherGeom& g, int tb, const int32_t* __restrict__ tokens,
                                                 int64_t batch, int lane) {
  return window_has(g, tb, batch, lane) ? __ldg(tokens + (batch * tb - 3 + lane)) : 0;
}

// The canonical ID of raw ID x at this lane's window position (kPad where there is none).
// An out-of-range ID reads as ID 0 and is reported by the batch that owns its position.
__device__ __forceinline__ uint32_t window_canon_id(const GatherGeom& g, int tb, uint32_t vocab,
                                                    const uint32_t* __restrict__ canon_map, int64_t batch, int lane,
                                                    int32_t x, int32_t* err) {
  if (!window_has(g, tb, batch, lane)) return kPad;
  if (x < 0 || static_cast<uint32_t>(x) >= vocab) {
    if (err && lane >= 3)
      atomicMin(reinterpret_cast<unsigned int*>(err), static_cast<unsigned int>(batch * tb - 3 + lane));
    x = 0;
  }
  return canon_map ? __ldg(canon_map + x) : static_cast<uint32_t>(x);
}

// Row and sign hash of (token s of the batch, item `ic`) from the window's canonical IDs
// `cid`. Every lane of the warp calls it (shuffles); `valid` lanes get the row.
__device__ __forceinline__ uint32_t window_row(const ItemConst& ic, int mode, const GatherGeom& g, int64_t tok, int s,
                                               uint32_t cid, bool valid, uint64_t* hs) {
  uint64_t c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) c[j] = __shfl_sync(0xffffffffu, cid, s - j + 3);
  if (!valid) return 0u;
  const uint32_t t = fastmod(static_cast<uint32_t>(tok), g.fm_L, g.L);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (!(j < ic.n && t >= static_cast<uint32_t>(j))) c[j] = kPad;
  return item_row_ids(ic, mode, c, hs);
}

constexpr int kThreads = 256;       // threads per gather block
constexpr int kChunksPerThread = 8; // 16-byte chunks (or NF4 tasks) per lane per warp batch

// Phase A: rows and sign words of every (token, item) of one warp batch, one lane each.
template <int ITEMS, int TB>
__device__ __forceinline__ void hash_batch(const ItemConst* __restrict__ ic, const GatherGeom& g, int mode,
                                           int64_t batch, int lane, const int32_t* __restrict__ tokens,
                                           const uint32_t* __restrict__ canon_map, uint32_t vocab,
                                           uint32_t* s_rows, uint64_t* s_signs, int32_t* err) {
  const int p = lane;
  const int items = ITEMS ? ITEMS : g.items;
  const int tb = ITEMS ? TB : g.tb;
  if (p >= tb * items) return;
  const int s = p / items;  // once per lane and batch
  const int item = p - s * items;
  const int64_t tok = batch * tb + s;
  if (tok >= g.N) return;
  const uint32_t t = fastmod(static_cast<uint32_t>(tok), g.fm_L, g.L);
  uint64_t hs;
  s_rows[p] = item_row(ic[item], mode, tokens, canon_map, vocab, tok, t, err, &hs);
  for (int q = 0; q < g.W; ++q) s_signs[p * g.W + q] = mix64(hs + kGolden * static_cast<uint64_t>(q + 1));
}

// Warp-batch geometry: tb tokens whose (token, item) pairs fit 32 lanes and whose chunks
// fit kChunksPerThread per lane (the host computes the same numbers).
__host__ __device__ constexpr int batch_tokens(int per_tok, int items) {
  return (32 * kChunksPerThread / per_tok) < (32 / items) ? (32 * kChunksPerThread / per_tok) : (32 / items);
}

// RC (16-byte chunks per row, or 8-element NF4 tasks per row) and ITEMS (items per token)
// fixed at compile time turn the chunk -> (token, item, piece) mapping into shifts for the
// layouts the workloads use; RC = ITEMS = 0 is the general, runtime-geometry version.
template <int ROWT, int OUTT, bool FLAT, int RC, int ITEMS>
__global__ void __launch_bounds__(kThreads, (RC > 0 && ITEMS > 0) ? 3 : 2) gather_kernel(
    const __grid_constant__ HashParams P, uint64_t seed, const GatherGeom g, const int32_t* __restrict__ tokens,
    const uint32_t* __restrict__ canon_map, const uint8_t* __restrict__ table, uint8_t* __restrict__ e_out,
    int32_t* err) {
  constexpr bool CT = RC > 0 && ITEMS > 0;
  constexpr int PT = CT ? (FLAT ? RC : ITEMS * RC) : 1;
  constexpr int TBC = CT ? batch_tokens(PT, ITEMS) : 1;
  constexpr int NCH = CT ? (TBC * PT + 31) / 32 : kChunksPerThread;
  static_assert(TBC <= kMaxBatchTokens, "the batch's ID window fits the lanes");
  const int per_tok = CT ? PT : g.per_tok;
  const int items = CT ? ITEMS : g.items;
  const int tb = CT ? TBC : g.tb;
  const uint32_t rc = CT ? RC : g.rc;
  constexpr int kWarpsPerBlock = kThreads / 32;
  __shared__ ItemConst s_ic[kMaxItems];
  // per warp, double-buffered: rows [2][32], sign words [2][kMaxSignWords]
  __shared__ uint32_t s_rows_all[kWarpsPerBlock][2][32];
  __shared__ uint64_t s_signs_all[kWarpsPerBlock][2][kMaxSignWords];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x < g.items) init_item_const(s_ic[threadIdx.x], P, seed, threadIdx.x);
  __syncthreads();

  // phase A of a batch: lane p = (token s, item) hashes its row and sign words from the
  // window's canonical IDs `cid` (no loads)
  auto hash_to = [&](int64_t batch, uint32_t cid, uint32_t* s_rows, uint64_t* s_signs) {
    const int p = lane;
    const int s = p < tb * items ? p / items : 0;
    const int item = p - s * items;
    const int64_t tok = batch * tb + s;
    const bool valid = batch < g.nbatch && p < tb * items && tok < g.N;
    uint64_t hs;
    const uint32_t row = window_row(s_ic[valid ? item : 0], P.mode, g, tok, s, cid, valid, &hs);
    if (valid) {
      s_rows[p] = row;
      for (int q = 0; q < g.W; ++q) s_signs[p * g.W + q] = mix64(hs + kGolden * static_cast<uint64_t>(q + 1));
    }
  };
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
  // IDs: raw IDs two batches ahead of the one hashed, canonical IDs one ahead. Batches of
  // one token keep per-lane ID reads instead (each hashing lane reads its n-gram's IDs while
  // the previous batch's rows are in flight): there the window's bookkeeping costs more
  // issue slots than the reads' latency, which the row loads hide (measured).
  constexpr bool kWindow = !CT || TBC > 1;
  int32_t raw_ahead = 0;
  uint32_t cid_ahead = kPad;
  if constexpr (kWindow) {
    raw_ahead = window_raw_id(g, tb, tokens, first, lane);
    const int32_t raw1 = window_raw_id(g, tb, tokens, first + nwarps, lane);
    const uint32_t cid0 = window_canon_id(g, tb, P.vocab, canon_map, first, lane, raw_ahead, err);
    cid_ahead = window_canon_id(g, tb, P.vocab, canon_map, first + nwarps, lane, raw1, err);
    raw_ahead = window_raw_id(g, tb, tokens, first + 2 * nwarps, lane);
    hash_to(first, cid0, s_rows_all[warp][0], s_signs_all[warp][0]);
  } else if (first < g.nbatch) {
    hash_batch<ITEMS, TBC>(s_ic, g, P.mode, first, lane, tokens, canon_map, P.vocab, s_rows_all[warp][0],
                           s_signs_all[warp][0], err);
  }
  __syncwarp();
  const int chunks = tb * per_tok;
  int cur = 0;
  for (int64_t batch = first; batch < g.nbatch; batch += nwarps) {
    const uint32_t* rows = s_rows_all[warp][cur];
    const uint64_t* signs = s_signs_all[warp][cur];
    uint32_t cid_next = kPad;
    // a batch is streamed in rounds of 32 * NCH chunks (one round unless a token's e_t
    // is wider than a round)
    for (int base = 0; base < chunks; base += 32 * NCH) {
    // ---- phase B, issue: loads of this round's chunks
    uint4 v[NCH];
    uint32_t bits[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const uint32_t c = base + lane + 32 * i;
      if (c < static_cast<uint32_t>(chunks)) {
        const uint32_t s = CT ? c / PT : __umulhi(c, g.tok_magic);
        const uint32_t cc = c - s * per_tok;
        if (batch * tb + s < g.N) {
          if constexpr (FLAT) {
            // chunk cc of the d-wide row, for every order: loaded and summed at use
            v[i] = make_uint4(0, 0, 0, 0);
            bits[i] = 0;
          } else {
            constexpr int E = ROWT == PG_F32 ? 4 : 8;
            const uint32_t it = CT ? cc / RC : (rc == 1u ? cc : __umulhi(cc, g.rc_magic));
            const uint32_t piece = cc - it * rc;
            v[i] = ldg_stream(table + static_cast<uint64_t>(rows[s * items + it]) * (CT ? RC * 16u : g.row_bytes) +
                              piece * 16u);
            const uint32_t e0 = piece * E;
            bits[i] = static_cast<uint32_t>(signs[(s * items + it) * g.W + (e0 >> 6)] >> (e0 & 63)) &
                      ((1u << E) - 1u);
          }
        }
      }
    }
    // ---- IDs of later batches, then phase A of the next batch, while the loads are in flight
    if constexpr (kWindow) {
      if (base == 0) {
        cid_next = window_canon_id(g, tb, P.vocab, canon_map, batch + 2 * nwarps, lane, raw_ahead, err);
        raw_ahead = window_raw_id(g, tb, tokens, batch + 3 * nwarps, lane);
        hash_to(batch + nwarps, cid_ahead, s_rows_all[warp][cur ^ 1], s_signs_all[warp][cur ^ 1]);
      }
    } else if (base == 0 && batch + nwarps < g.nbatch) {
      hash_batch<ITEMS, TBC>(s_ic, g, P.mode, batch + nwarps, lane, tokens, canon_map, P.vocab,
                             s_rows_all[warp][cur ^ 1], s_signs_all[warp][cur ^ 1], err);
    }
    // ---- phase B, finish: dequantise, sign, (sum), store
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const uint32_t c = base + lane + 32 * i;
      if (c >= static_cast<uint32_t>(chunks)) continue;
      const uint32_t s = CT ? c / PT : __umulhi(c, g.tok_magic);
      const uint32_t cc = c - s * per_tok;
      const int64_t tok = batch * tb + s;
      if (tok >= g.N) continue;
      uint8_t* out_tok = e_out + static_cast<uint64_t>(tok) * g.e_bytes;
      if constexpr (FLAT) {
        constexpr int E = ROWT == PG_F32 ? 4 : 8;
        const int O = items;
        float acc[E];
        for (int o = 0; o < O; ++o) {
          const uint4 x4 =
              ldg_stream(table + static_cast<uint64_t>(rows[s * O + o]) * (CT ? RC * 16u : g.row_bytes) + cc * 16u);
          const uint32_t e0 = cc * E;
          const uint32_t b = static_cast<uint32_t>(signs[(s * O + o) * g.W + (e0 >> 6)] >> (e0 & 63)) &
                             ((1u << E) - 1u);
          float x[E];
          if constexpr (ROWT == PG_F32) {
            const uint4 f = xor4(x4, f32_sign_mask(b));
            x[0] = __uint_as_float(f.x); x[1] = __uint_as_float(f.y);
            x[2] = __uint_as_float(f.z); x[3] = __uint_as_float(f.w);
          } else {
            const uint4 f = xor4(x4, bf16_sign_mask(b));
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
      } else if constexpr (ROWT == PG_F32) {
        *reinterpret_cast<uint4*>(out_tok + cc * 16u) = xor4(v[i], f32_sign_mask(bits[i]));
      } else if constexpr (OUTT == PG_BF16) {
        *reinterpret_cast<uint4*>(out_tok + cc * 16u) = xor4(v[i], bf16_sign_mask(bits[i]));
      } else {
        const uint4 f = xor4(v[i], bf16_sign_mask(bits[i]));
        uint8_t* dst = out_tok + cc * 32u;
        *reinterpret_cast<uint4*>(dst) = make_uint4(f.x << 16, f.x & 0xFFFF0000u, f.y << 16, f.y & 0xFFFF0000u);
        *reinterpret_cast<uint4*>(dst + 16) =
            make_uint4(f.z << 16, f.z & 0xFFFF0000u, f.w << 16, f.w & 0xFFFF0000u);
      }
    }
    }  // rounds
    __syncwarp();
    cur ^= 1;
    cid_ahead = cid_next;
  }
}

// ------------------------------------------------------------------ K2, E4M3 output

// The gather with the FP8 projection's operand as its output (Engram notes section 3.4:
// the fused projection runs in FP8): e_t of bf16 rows, quantised per token as
// pg_fp8_quantize does it, q_i = E4M3(x_i / s) with s = max |x| / 448 (correctly rounded
// fp32 division, round to nearest even, saturating; s = 0 stores zeros), so codes and
// scales equal pg_gather_sign_concat (bf16) followed by pg_fp8_quantize bit for bit. The
// batch, hash and load phases are the bf16 gather's; a warp batch holds whole tokens in
// registers, so each token's max |x| is a warp reduction over the bf16 magnitudes (as
// 15-bit patterns, whose integer order is their numeric order; NaN patterns left out).
template <int RC, int ITEMS>
__global__ void __launch_bounds__(kThreads, 3) gather_e4m3_kernel(
    const __grid_constant__ HashParams P, uint64_t seed, const GatherGeom g, const int32_t* __restrict__ tokens,
    const uint32_t* __restrict__ canon_map, const uint8_t* __restrict__ table, uint8_t* __restrict__ q_out,
    float* __restrict__ scale_out, int32_t* err) {
  constexpr int PT = ITEMS * RC;
  constexpr int TBC = batch_tokens(PT, ITEMS);
  constexpr int NCH = (TBC * PT + 31) / 32;
  static_assert(TBC == 1 || PT % 32 == 0, "a lane's chunks of one step belong to one token");
  constexpr int kWarpsPerBlock = kThreads / 32;
  constexpr int E = 8;  // bf16 elements per 16-byte chunk
  __shared__ ItemConst s_ic[kMaxItems];
  __shared__ uint32_t s_rows_all[kWarpsPerBlock][2][32];
  __shared__ uint64_t s_signs_all[kWarpsPerBlock][2][kMaxSignWords];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x < g.items) init_item_const(s_ic[threadIdx.x], P, seed, threadIdx.x);
  __syncthreads();

  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
  if (first < g.nbatch)
    hash_batch<ITEMS, TBC>(s_ic, g, P.mode, first, lane, tokens, canon_map, P.vocab, s_rows_all[warp][0],
                           s_signs_all[warp][0], err);
  __syncwarp();
  int cur = 0;
  for (int64_t batch = first; batch < g.nbatch; batch += nwarps) {
    const uint32_t* rows = s_rows_all[warp][cur];
    const uint64_t* signs = s_signs_all[warp][cur];
    uint4 v[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const uint32_t c = lane + 32 * i;
      v[i] = make_uint4(0, 0, 0, 0);
      if (c < static_cast<uint32_t>(TBC * PT)) {
        const uint32_t sidx = c / PT, cc = c - sidx * PT;
        if (batch * TBC + sidx < g.N) {
          const uint32_t it = cc / RC, piece = cc - it * RC;
          v[i] = ldg_stream(table + static_cast<uint64_t>(rows[sidx * ITEMS + it]) * (RC * 16u) + piece * 16u);
        }
      }
    }
    const int64_t next = batch + nwarps;
    if (next < g.nbatch)
      hash_batch<ITEMS, TBC>(s_ic, g, P.mode, next, lane, tokens, canon_map, P.vocab, s_rows_all[warp][cur ^ 1],
                             s_signs_all[warp][cur ^ 1], err);
    // sign, then each token's largest magnitude
    uint32_t amax[TBC];
#pragma unroll
    for (int t = 0; t < TBC; ++t) amax[t] = 0u;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const uint32_t c = lane + 32 * i;
      const uint32_t sidx = c / PT, cc = c - sidx * PT;
      if (c >= static_cast<uint32_t>(TBC * PT)) continue;
      const uint32_t it = cc / RC, piece = cc - it * RC;
      const uint32_t e0 = piece * E;
      const uint32_t bits =
          static_cast<uint32_t>(signs[(sidx * ITEMS + it) * g.W + (e0 >> 6)] >> (e0 & 63)) & ((1u << E) - 1u);
      v[i] = xor4(v[i], bf16_sign_mask(bits));
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      uint32_t m = 0u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t lo = w[q] & 0x7FFFu, hi = (w[q] >> 16) & 0x7FFFu;
        m = max(m, lo > 0x7F80u ? 0u : lo);
        m = max(m, hi > 0x7F80u ? 0u : hi);
      }
      const int t = TBC == 1 ? 0 : static_cast<int>((32 * i) / PT);  // PT % 32 == 0 when TBC > 1
      amax[t] = max(amax[t], m);
    }
    // scale s, and its correctly rounded reciprocal for the quotients (Markstein's division:
    // q0 = RN(x y), r = x - q0 s exactly by an fma, q = RN(q0 + r y) is RN(x / s) when
    // y = RN(1 / s) and nothing underflows). For s in [2^-90, 2^125] every quotient that can
    // reach a nonzero E4M3 code (|x / s| >= 2^-10) has a normal remainder; outside it the
    // quotients take the plain correctly rounded division.
    float scl[TBC], rcp[TBC];
    bool fast[TBC];
#pragma unroll
    for (int t = 0; t < TBC; ++t) {
      const uint32_t m = __reduce_max_sync(0xffffffffu, amax[t]);
      scl[t] = __fdiv_rn(__uint_as_float(m << 16), 448.0f);
      rcp[t] = __frcp_rn(scl[t]);
      fast[t] = scl[t] >= 0x1p-90f && scl[t] <= 0x1p125f;
      const int64_t tok = batch * TBC + t;
      if (lane == 0 && tok < g.N) scale_out[tok] = scl[t];
    }
    // codes, 8 per chunk (8 contiguous bytes of the token's row)
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const uint32_t c = lane + 32 * i;
      if (c >= static_cast<uint32_t>(TBC * PT)) continue;
      const uint32_t sidx = c / PT, cc = c - sidx * PT;
      const int64_t tok = batch * TBC + sidx;
      if (tok >= g.N) continue;
      const int t = TBC == 1 ? 0 : static_cast<int>((32 * i) / PT);
      const float sc = scl[t], y = rcp[t];
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      uint32_t out[2] = {0u, 0u};
      if (sc != 0.0f) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // the pair of elements in word q
          float2 z = make_float2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xFFFF0000u));
          if (fast[t]) {
            const float q0 = __fmul_rn(z.x, y), q1 = __fmul_rn(z.y, y);
            const float r0 = __fmaf_rn(-q0, sc, z.x), r1 = __fmaf_rn(-q1, sc, z.y);
            z.x = r0 == 0.0f ? q0 : __fmaf_rn(r0, y, q0);
            z.y = r1 == 0.0f ? q1 : __fmaf_rn(r1, y, q1);
          } else {
            z.x = __fdiv_rn(z.x, sc);
            z.y = __fdiv_rn(z.y, sc);
          }
          const uint32_t b2 = __nv_cvt_float2_to_fp8x2(z, __NV_SATFINITE, __NV_E4M3);  // z.x in the low byte
          out[q / 2] |= b2 << (16 * (q % 2));
        }
      }
      *reinterpret_cast<uint2*>(q_out + static_cast<uint64_t>(tok) * (PT * E) + cc * E) = make_uint2(out[0], out[1]);
    }
    __syncwarp();
    cur ^= 1;
  }
}

// ------------------------------------------------------------------ K2, NF4 rows

// A 34-byte NF4 row starts at an even byte offset o = 34 row mod 16, so it lies inside the
// three aligned 16-byte chunks [34 row - o, 34 row - o + 48). Each warp batch (tb tokens,
// tb * items <= 32 rows) copies those windows into the warp's shared-memory ring with
// cp.async (no registers held while the rows are in flight) kNf4Depth batches ahead, then
// dequantises from shared memory: the same task mapping and output stores as the bf16 path
// (one lane per 8 elements, 16 bytes of e_t per lane and 512 contiguous bytes per warp
// store).
// The IDs a batch hashes are loaded ahead too (window_raw_id two iterations before the
// batch is staged, window_canon_id one iteration before), so no load sits between a
// batch's dequantisation and the copies of the batch staged after it.
constexpr int kNf4Window = 48;
constexpr int kNf4Depth = 3;

struct Nf4Slot {
  uint8_t rows[32][kNf4Window];
  uint64_t sign[32];
  uint8_t off[32];
};

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int OUTT, int ITEMS>
__global__ void __launch_bounds__(kThreads, 4) gather_nf4_kernel(
    const __grid_constant__ HashParams P, uint64_t seed, const GatherGeom g, const int32_t* __restrict__ tokens,
    const uint32_t* __restrict__ canon_map, const uint8_t* __restrict__ table, uint8_t* __restrict__ e_out,
    int32_t* err) {
  constexpr int kWarps = kThreads / 32;
  constexpr int TBC = ITEMS > 0 ? batch_tokens(ITEMS * 8, ITEMS) : 1;
  static_assert(ITEMS == 0 || TBC <= kMaxBatchTokens, "the batch's ID window fits the lanes");
  const int items = ITEMS > 0 ? ITEMS : g.items;
  const int tb = ITEMS > 0 ? TBC : g.tb;  // <= kMaxBatchTokens (host)
  const int per_tok = items * 8;
  const int tasks = tb * per_tok;  // <= 32 * 8
  __shared__ ItemConst s_ic[kMaxItems];
  __shared__ float s_nf4[16];
  __shared__ __align__(16) Nf4Slot s_ring[kWarps][kNf4Depth];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < g.items) init_item_const(s_ic[threadIdx.x], P, seed, threadIdx.x);
  if (threadIdx.x < 16) s_nf4[threadIdx.x] = __uint_as_float(c_nf4_bits[threadIdx.x]);
  __syncthreads();

  auto raw_id = [&](int64_t batch) { return window_raw_id(g, tb, tokens, batch, lane); };
  auto canon_id = [&](int64_t batch, int32_t x) {
    return window_canon_id(g, tb, P.vocab, canon_map, batch, lane, x, err);
  };

  // a batch: lane p hashes row p from the window's canonical IDs `cid`, stores its sign
  // word and window offset, and starts the copy of its window
  auto stage = [&](int64_t batch, Nf4Slot& sl, uint32_t cid) {
    const int p = lane;
    const int s = p < tb * items ? p / items : 0;
    const int item = p - s * items;
    const int64_t tok = batch * tb + s;
    const bool valid = batch < g.nbatch && p < tb * items && tok < g.N;
    uint64_t hs;
    const uint32_t row = window_row(s_ic[valid ? item : 0], P.mode, g, tok, s, cid, valid, &hs);
    if (valid) {
      const uint64_t start = static_cast<uint64_t>(row) * 34u;
      const uint32_t off = static_cast<uint32_t>(start & 15u);
      sl.sign[p] = mix64(hs + kGolden);
      sl.off[p] = static_cast<uint8_t>(off);
      const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(sl.rows[p]));
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const uint64_t ch = start - off + 16u * k;
        if (ch < g.table_bytes) {
          const uint64_t left = g.table_bytes - ch;
          cp_async16_zfill(dst + 16 * k, table + ch, left < 16u ? static_cast<uint32_t>(left) : 16u);
        }
      }
    }
    cp_async_commit();
  };

  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  // prologue: IDs of the first kNf4Depth + 2 batches, canonical IDs of the first
  // kNf4Depth + 1, the first kNf4Depth batches staged
  int32_t raw[kNf4Depth + 2];
  uint32_t cid[kNf4Depth + 1];
#pragma unroll
  for (int d = 0; d < kNf4Depth + 2; ++d) raw[d] = raw_id(first + d * nwarps);
#pragma unroll
  for (int d = 0; d < kNf4Depth + 1; ++d) cid[d] = canon_id(first + d * nwarps, raw[d]);
#pragma unroll
  for (int d = 0; d < kNf4Depth; ++d) stage(first + d * nwarps, s_ring[warp][d], cid[d]);
  uint32_t cid_ahead = cid[kNf4Depth];      // canonical IDs of batch + kNf4Depth * nwarps
  int32_t raw_ahead = raw[kNf4Depth + 1];   // raw IDs of batch + (kNf4Depth + 1) * nwarps
  int slot = 0;
  for (int64_t batch = first; batch < g.nbatch; batch += nwarps) {
    // IDs for later batches, in flight during this batch's dequantisation
    const uint32_t cid_next = canon_id(batch + (kNf4Depth + 1) * nwarps, raw_ahead);
    raw_ahead = raw_id(batch + (kNf4Depth + 2) * nwarps);
    cp_async_wait<kNf4Depth - 1>();  // this lane's copies for `batch` have landed
    __syncwarp();                    // ... and every other lane's
    const Nf4Slot& sl = s_ring[warp][slot];
    const uint8_t* sign_bytes = reinterpret_cast<const uint8_t*>(sl.sign);  // byte j: bits 8 j .. 8 j + 7
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c >= tasks) continue;
      const int s = ITEMS > 0 ? c / (ITEMS * 8) : c / per_tok;
      const int cc = c - s * per_tok;
      const int64_t tok = batch * tb + s;
      if (tok >= g.N) continue;
      const int p = s * items + (cc >> 3), piece = cc & 7;
      const uint8_t* w = sl.rows[p] + sl.off[p];
      const uint32_t codes = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(w + 4 * piece)) |
                             (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(w + 4 * piece + 2)) << 16);
      const float scale = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(w + 32)));
      const uint32_t bits = sign_bytes[8 * p + piece];
      // level * scale in fp32 pairs; the sign goes on after rounding (round-to-nearest is
      // symmetric, so the result is the rounding of the signed product)
      const uint64_t sc2 = pk(scale, scale);
      float x[8];
#pragma unroll
      for (int q = 0; q < 8; q += 2)
        upk(mul2(pk(s_nf4[(codes >> (4 * q)) & 15u], s_nf4[(codes >> (4 * q + 4)) & 15u]), sc2), x[q], x[q + 1]);
      uint8_t* out_tok = e_out + static_cast<uint64_t>(tok) * g.e_bytes;
      if constexpr (OUTT == PG_F32) {
        uint8_t* dst = out_tok + cc * 32u;
        *reinterpret_cast<uint4*>(dst) = xor4(make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                                                         __float_as_uint(x[2]), __float_as_uint(x[3])),
                                              f32_sign_mask(bits & 15u));
        *reinterpret_cast<uint4*>(dst + 16) = xor4(make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]),
                                                              __float_as_uint(x[6]), __float_as_uint(x[7])),
                                                   f32_sign_mask(bits >> 4));
      } else {
        *reinterpret_cast<uint4*>(out_tok + cc * 16u) =
            xor4(make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7])),
                 bf16_sign_mask(bits));
      }
    }
    __syncwarp();  // every lane is done with the slot before it is refilled
    stage(batch + kNf4Depth * nwarps, s_ring[warp][slot], cid_ahead);
    cid_ahead = cid_next;
    slot = slot + 1 == kNf4Depth ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

using GatherFn = void (*)(const HashParams, uint64_t, const GatherGeom, const int32_t*, const uint32_t*,
                          const uint8_t*, uint8_t*, int32_t*);

template <int RC, int ITEMS>
GatherFn pick_layout(int row_dtype, int out_dtype, bool flat) {
  if (flat) {
    if (row_dtype == PG_F32 && out_dtype == PG_F32) return gather_kernel<PG_F32, PG_F32, true, RC, ITEMS>;
    if (row_dtype == PG_BF16 && out_dtype == PG_BF16) return gather_kernel<PG_BF16, PG_BF16, true, RC, ITEMS>;
    if (row_dtype == PG_BF16 && out_dtype == PG_F32) return gather_kernel<PG_BF16, PG_F32, true, RC, ITEMS>;
    return nullptr;
  }
  if (row_dtype == PG_F32 && out_dtype == PG_F32) return gather_kernel<PG_F32, PG_F32, false, RC, ITEMS>;
  if (row_dtype == PG_BF16 && out_dtype == PG_BF16) return gather_kernel<PG_BF16, PG_BF16, false, RC, ITEMS>;
  if (row_dtype == PG_BF16 && out_dtype == PG_F32) return gather_kernel<PG_BF16, PG_F32, false, RC, ITEMS>;
  if (row_dtype == PG_NF4 && out_dtype == PG_BF16) return gather_nf4_kernel<PG_BF16, 0>;
  if (row_dtype == PG_NF4 && out_dtype == PG_F32) return gather_nf4_kernel<PG_F32, 0>;
  return nullptr;
}

// Compile-time layouts: r = 64 rows (bf16 / NF4: 8 chunks; fp32: 16) and r = 80 bf16 (10)
// with 2 orders x 8 heads; flat d = 768 bf16 (96 chunks) and d = 256 fp32 (64).
GatherFn pick_gather(int row_dtype, int out_dtype, bool flat, uint32_t rc, int items) {
  const bool bb = row_dtype == PG_BF16 && out_dtype == PG_BF16;
  const bool bf = row_dtype == PG_BF16 && out_dtype == PG_F32;
  const bool ff = row_dtype == PG_F32 && out_dtype == PG_F32;
  if (!flat && items == 16) {
    if (rc == 8 && bb) return gather_kernel<PG_BF16, PG_BF16, false, 8, 16>;
    if (rc == 8 && bf) return gather_kernel<PG_BF16, PG_F32, false, 8, 16>;
    if (row_dtype == PG_NF4 && out_dtype == PG_BF16) return gather_nf4_kernel<PG_BF16, 16>;
    if (row_dtype == PG_NF4 && out_dtype == PG_F32) return gather_nf4_kernel<PG_F32, 16>;
    if (rc == 10 && bb) return gather_kernel<PG_BF16, PG_BF16, false, 10, 16>;
    if (rc == 16 && ff) return gather_kernel<PG_F32, PG_F32, false, 16, 16>;
  }
  if (flat && items == 2) {
    if (rc == 96 && bb) return gather_kernel<PG_BF16, PG_BF16, true, 96, 2>;
    if (rc == 64 && ff) return gather_kernel<PG_F32, PG_F32, true, 64, 2>;
  }
  return pick_layout<0, 0>(row_dtype, out_dtype, flat);
}

// ------------------------------------------------------------------ NF4 export

// NF4 export of 64-wide fp32 head rows into the 34-byte stored rows (PageGram report 3.3:
// 64 four-bit codes + one fp16 scale; QLoRA's absmax rule). One warp per row, lane l owns
// elements 2l and 2l+1 and writes byte l; lane 0 writes the scale. Scale = max |x| rounded
// to fp16 (nearest even), saturating at 65504; codes = the nearest level of x / scale
// (correctly rounded fp32 division, fp32 distances, the lowest code on ties); a zero scale
// gives the exact-zero level everywhere.
__global__ void __launch_bounds__(256) nf4_quantize_kernel(const float* __restrict__ x, int64_t n,
                                                           uint8_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t first = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  float lv[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) lv[k] = __uint_as_float(c_nf4_bits[k]);
  auto nearest = [&](float y) {
    int best = 0;
    float dbest = fabsf(y - lv[0]);
#pragma unroll
    for (int k = 1; k < 16; ++k) {
      const float dk = fabsf(y - lv[k]);
      if (dk < dbest) {
        dbest = dk;
        best = k;
      }
    }
    return best;
  };
  for (int64_t row = first; row < n; row += nwarps) {
    const float2 v = __ldg(reinterpret_cast<const float2*>(x + row * 64) + lane);
    float a = fmaxf(0.0f, fmaxf(fabsf(v.x), fabsf(v.y)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    __half h = __float2half_rn(a);
    if (__hisinf(h)) h = __ushort_as_half(static_cast<unsigned short>(0x7BFFu));
    const float s = __half2float(h);
    int c0 = 7, c1 = 7;
    if (s != 0.0f) {
      c0 = nearest(__fdiv_rn(v.x, s));
      c1 = nearest(__fdiv_rn(v.y, s));
    }
    uint8_t* o = out + row * 34;
    o[lane] = static_cast<uint8_t>(c0 | (c1 << 4));
    if (lane == 0) {
      const unsigned short sb = __half_as_ushort(h);
      o[32] = static_cast<uint8_t>(sb & 0xFFu);
      o[33] = static_cast<uint8_t>(sb >> 8);
    }
  }
}

// ------------------------------------------------------------------ streaming decode lookup

// One new token per sequence, a warp per sequence (decode_token_lookup); the ring slot of t
// and pos (t + 1) are written last, by lane 0, after every lane's reads (no other warp
// touches b).
constexpr int kDecodeWarps = 8;

template <int ROWT, int OUTT, bool FLAT>
__global__ void __launch_bounds__(kDecodeWarps * 32) decode_lookup_kernel(
    const __grid_constant__ HashParams P, uint64_t seed, const GatherGeom g, int B,
    const int32_t* __restrict__ tokens, const uint32_t* __restrict__ canon_map, const uint8_t* __restrict__ table,
    int32_t* __restrict__ pos, uint32_t* __restrict__ ids, uint8_t* __restrict__ e_out, int32_t* err,
    int* err_word) {
  __shared__ ItemConst s_ic[kMaxItems];
  __shared__ float s_nf4[16];
  __shared__ uint32_t s_rows[kDecodeWarps][kMaxItems];
  __shared__ uint64_t s_signs[kDecodeWarps][kMaxSignWords];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < g.items) init_item_const(s_ic[threadIdx.x], P, seed, threadIdx.x);
  if (threadIdx.x < 16) s_nf4[threadIdx.x] = __uint_as_float(c_nf4_bits[threadIdx.x]);
  __syncthreads();
  const int nw = gridDim.x * kDecodeWarps;
  for (int b = blockIdx.x * kDecodeWarps + warp; b < B; b += nw) {
    uint32_t c0;
    const int t = decode_token_lookup<ROWT, OUTT, FLAT>(P, g, s_ic, s_nf4, s_rows[warp], s_signs[warp], b, lane,
                                                        tokens, canon_map, table, pos, ids,
                                                        e_out + static_cast<uint64_t>(b) * g.e_bytes, err, err_word,
                                                        &c0);
    if (t >= 0 && lane == 0) {
      ids[4 * static_cast<int64_t>(b) + (t & 3)] = c0;
      pos[b] = t + 1;
    }
  }
}

using DecodeFn = void (*)(const HashParams, uint64_t, const GatherGeom, int, const int32_t*, const uint32_t*,
                          const uint8_t*, int32_t*, uint32_t*, uint8_t*, int32_t*, int*);

DecodeFn pick_decode(int row_dtype, int out_dtype, bool flat) {
  if (flat) {
    if (row_dtype == PG_F32 && out_dtype == PG_F32) return decode_lookup_kernel<PG_F32, PG_F32, true>;
    if (row_dtype == PG_BF16 && out_dtype == PG_BF16) return decode_lookup_kernel<PG_BF16, PG_BF16, true>;
    if (row_dtype == PG_BF16 && out_dtype == PG_F32) return decode_lookup_kernel<PG_BF16, PG_F32, true>;
    return nullptr;
  }
  if (row_dtype == PG_F32 && out_dtype == PG_F32) return decode_lookup_kernel<PG_F32, PG_F32, false>;
  if (row_dtype == PG_BF16 && out_dtype == PG_BF16) return decode_lookup_kernel<PG_BF16, PG_BF16, false>;
  if (row_dtype == PG_BF16 && out_dtype == PG_F32) return decode_lookup_kernel<PG_BF16, PG_F32, false>;
  if (row_dtype == PG_NF4 && out_dtype == PG_BF16) return decode_lookup_kernel<PG_NF4, PG_BF16, false>;
  if (row_dtype == PG_NF4 && out_dtype == PG_F32) return decode_lookup_kernel<PG_NF4, PG_F32, false>;
  return nullptr;
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
  Geometry geo;
  pg_status st = validate_desc(desc, &geo);
  if (st != PG_OK) return st;
  if (desc->hash_kind != PG_HASH_MULXOR) return PG_ERR_UNSUPPORTED;
  if (B < 0 || L < 0) return PG_ERR_SHAPE;
  const int64_t N = static_cast<int64_t>(B) * L;
  if (N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (N == 0) return PG_OK;
  if (!tokens || !table || !e_out) return PG_ERR_NULL;
  if (table_bytes < geo.rows * geo.row_bytes) return PG_ERR_RANGE;
  if (reinterpret_cast<uintptr_t>(table) % 16 || reinterpret_cast<uintptr_t>(e_out) % 16)
    return PG_ERR_ALIGN;
  if (out_dtype != PG_F32 && out_dtype != PG_BF16) return PG_ERR_DTYPE;
  const bool flat = desc->mode == PG_FLAT;
  const int items = geo.O * geo.H;
  if (items > kMaxItems || items * geo.W > kMaxSignWords) return PG_ERR_UNSUPPORTED;
  if (desc->row_dtype != PG_NF4 && geo.row_bytes % 16) return PG_ERR_UNSUPPORTED;
  const uint32_t rc_host = desc->row_dtype == PG_NF4 ? 8u : geo.row_bytes / 16u;
  GatherFn fn = pick_gather(desc->row_dtype, out_dtype, flat, rc_host, items);
  if (!fn) return desc->row_dtype == PG_F32 && out_dtype == PG_BF16 ? PG_ERR_DTYPE : PG_ERR_UNSUPPORTED;

  GatherGeom g;
  g.N = N;
  g.L = static_cast<uint32_t>(L);
  g.fm_L = fastmod_constant(g.L);
  g.items = items;
  g.W = geo.W;
  g.rc = desc->row_dtype == PG_NF4 ? 8u : geo.row_bytes / 16u;
  g.per_tok = flat ? static_cast<int>(g.rc) : items * static_cast<int>(g.rc);
  if (g.per_tok < 2) return PG_ERR_UNSUPPORTED;  // 16-byte flat rows: no workload uses them
  // a warp batch: tb tokens whose (token, item) pairs fit the 32 lanes and whose chunks
  // fit 8 per lane
  int tb = batch_tokens(g.per_tok, items);
  if (tb < 1) tb = 1;  // a token wider than one round: streamed in several rounds
  if (tb > kMaxBatchTokens) tb = kMaxBatchTokens;  // the batch's ID window fits the lanes
  g.tb = tb;
  // floor(x / n) = umulhi(x, floor(2^32 / n) + 1), exact while x * n < 2^32 (x, n < 2^16 here)
  g.tok_magic = static_cast<uint32_t>((1ull << 32) / static_cast<uint32_t>(g.per_tok) + 1ull);
  g.rc_magic = g.rc == 1u ? 0u : static_cast<uint32_t>((1ull << 32) / g.rc + 1ull);
  g.row_bytes = geo.row_bytes;
  g.e_bytes = geo.e_width * (out_dtype == PG_F32 ? 4u : 2u);
  g.nbatch = (N + tb - 1) / tb;
  g.table_bytes = table_bytes;

  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  st = prepare_err(err_index, stream);
  if (st != PG_OK) return st;
  HashParams P;
  fill_hash_params(desc, geo, &P);
  if (tb * items * geo.W > kMaxSignWords) return PG_ERR_UNSUPPORTED;
  const size_t dyn = 0;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void*>(fn),
                                                                kThreads, dyn);
  if (e != cudaSuccess) return cuda_fail(e);
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = static_cast<int64_t>(nsm) * per_sm;
  const int64_t want = (g.nbatch + kThreads / 32 - 1) / (kThreads / 32);
  const int blocks = static_cast<int>(want < cap ? want : cap);
  fn<<<blocks, kThreads, dyn, stream>>>(P, desc->hash_seed, g, tokens, canon_map,
                                        static_cast<const uint8_t*>(table), static_cast<uint8_t*>(e_out),
                                        err_index);
  return after_launch(1);
}

pg_status pg_gather_sign_concat_e4m3(const pg_table_desc* desc, const int32_t* tokens, int32_t B, int32_t L,
                                     const uint32_t* canon_map, const void* table, uint64_t table_bytes,
                                     uint8_t* q_out, float* scale_out, int32_t* err_index, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  Geometry geo;
  pg_status st = validate_desc(desc, &geo);
  if (st != PG_OK) return st;
  if (desc->hash_kind != PG_HASH_MULXOR) return PG_ERR_UNSUPPORTED;
  if (B < 0 || L < 0) return PG_ERR_SHAPE;
  const int64_t N = static_cast<int64_t>(B) * L;
  if (N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (N == 0) return PG_OK;
  if (!tokens || !table || !q_out || !scale_out) return PG_ERR_NULL;
  if (table_bytes < geo.rows * geo.row_bytes) return PG_ERR_RANGE;
  if (reinterpret_cast<uintptr_t>(table) % 16 || reinterpret_cast<uintptr_t>(q_out) % 16 ||
      reinterpret_cast<uintptr_t>(scale_out) % 4)
    return PG_ERR_ALIGN;
  if (desc->row_dtype != PG_BF16) return PG_ERR_DTYPE;
  const int items = geo.O * geo.H;
  const uint32_t rc = geo.row_bytes / 16u;
  using E4Fn = void (*)(const HashParams, uint64_t, const GatherGeom, const int32_t*, const uint32_t*,
                        const uint8_t*, uint8_t*, float*, int32_t*);
  E4Fn fn = nullptr;
  if (desc->mode != PG_FLAT && items == 16 && rc == 8) fn = gather_e4m3_kernel<8, 16>;
  if (desc->mode != PG_FLAT && items == 16 && rc == 10) fn = gather_e4m3_kernel<10, 16>;
  if (!fn) return PG_ERR_UNSUPPORTED;  // the layouts of the projected workloads (r = 64, 80; 16 heads)

  GatherGeom g{};
  g.N = N;
  g.L = static_cast<uint32_t>(L);
  g.fm_L = fastmod_constant(g.L);
  g.items = items;
  g.W = geo.W;
  g.rc = rc;
  g.per_tok = items * static_cast<int>(rc);
  g.tb = batch_tokens(g.per_tok, items);
  g.row_bytes = geo.row_bytes;
  g.e_bytes = geo.e_width;
  g.nbatch = (N + g.tb - 1) / g.tb;
  g.table_bytes = table_bytes;
  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  st = prepare_err(err_index, stream);
  if (st != PG_OK) return st;
  HashParams P;
  fill_hash_params(desc, geo, &P);
  if (g.tb * items * geo.W > kMaxSignWords) return PG_ERR_UNSUPPORTED;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void*>(fn),
                                                                kThreads, 0);
  if (e != cudaSuccess) return cuda_fail(e);
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = static_cast<int64_t>(nsm) * per_sm;
  const int64_t want = (g.nbatch + kThreads / 32 - 1) / (kThreads / 32);
  const int blocks = static_cast<int>(want < cap ? want : cap);
  fn<<<blocks, kThreads, 0, stream>>>(P, desc->hash_seed, g, tokens, canon_map, static_cast<const uint8_t*>(table),
                                      q_out, scale_out, err_index);
  return after_launch(1);
}

pg_status pg_nf4_quantize(const float* x, int64_t nrows, int32_t r, void* out, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (nrows < 0) return PG_ERR_SHAPE;
  if (r != 64) return PG_ERR_UNSUPPORTED;
  if (nrows == 0) return PG_OK;
  if (!x || !out) return PG_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(x) % 8) return PG_ERR_ALIGN;
  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  const int64_t want = (nrows + 7) / 8;  // 8 rows (warps) per block
  const int64_t cap = static_cast<int64_t>(nsm) * 8;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  nf4_quantize_kernel<<<blocks, 256, 0, stream>>>(x, nrows, static_cast<uint8_t*>(out));
  return after_launch(1);
}

pg_status pg_decode_lookup(const pg_table_desc* desc, const pg_decode_state* state, const int32_t* tokens,
                           const uint32_t* canon_map, const void* table, uint64_t table_bytes, void* e_out,
                           int32_t out_dtype, int32_t* err_index, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  Geometry geo;
  pg_status st = validate_desc(desc, &geo);
  if (st != PG_OK) return st;
  if (desc->hash_kind != PG_HASH_MULXOR) return PG_ERR_UNSUPPORTED;
  st = decode_state_check(state, false);
  if (st != PG_OK) return st;
  if (!tokens || !table || !e_out) return PG_ERR_NULL;
  if (table_bytes < geo.rows * geo.row_bytes) return PG_ERR_RANGE;
  if (reinterpret_cast<uintptr_t>(table) % 16 || reinterpret_cast<uintptr_t>(e_out) % 16) return PG_ERR_ALIGN;
  if (out_dtype != PG_F32 && out_dtype != PG_BF16) return PG_ERR_DTYPE;
  const bool flat = desc->mode == PG_FLAT;
  const int items = geo.O * geo.H;
  if (items > kMaxItems || items * geo.W > kMaxSignWords) return PG_ERR_UNSUPPORTED;
  if (desc->row_dtype != PG_NF4 && geo.row_bytes % 16) return PG_ERR_UNSUPPORTED;
  DecodeFn fn = pick_decode(desc->row_dtype, out_dtype, flat);
  if (!fn) return desc->row_dtype == PG_F32 && out_dtype == PG_BF16 ? PG_ERR_DTYPE : PG_ERR_UNSUPPORTED;

  GatherGeom g{};
  g.N = state->B;
  g.items = items;
  g.W = geo.W;
  g.rc = desc->row_dtype == PG_NF4 ? 8u : geo.row_bytes / 16u;
  g.per_tok = flat ? static_cast<int>(g.rc) : items * static_cast<int>(g.rc);
  g.row_bytes = geo.row_bytes;
  g.e_bytes = geo.e_width * (out_dtype == PG_F32 ? 4u : 2u);
  g.table_bytes = table_bytes;

  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  st = prepare_err(err_index, stream);
  if (st != PG_OK) return st;
  HashParams P;
  fill_hash_params(desc, geo, &P);
  const int64_t want = (static_cast<int64_t>(state->B) + kDecodeWarps - 1) / kDecodeWarps;
  const int64_t cap = static_cast<int64_t>(nsm) * 8;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  fn<<<blocks, kDecodeWarps * 32, 0, stream>>>(P, desc->hash_seed, g, state->B, tokens, canon_map,
                                               static_cast<const uint8_t*>(table), state->pos, state->ids,
                                               static_cast<uint8_t*>(e_out), err_index,
                                               device_error_word());
  return after_launch(1);
}

}  // extern "C"
