// One streaming decode step in one launch (sm_103a): lookup -> projection -> gate ->
// causal conv + residual for a few sequences (B <= 8), one new token each.
//
// A decode step over a handful of sequences is a few kernel latencies when its stages run
// as separate launches (lookup, the W-streaming projection, the alpha finalize, the decode
// conv), while its work is one pass over W (33 MB on the Engram-27B shapes) plus a few KB.
// Addressing depends on the token IDs alone (Engram notes, section 3.5), so every block can
// compute the step's e_t itself; the projection splits the model width d into one channel
// range per block, and each block then owns the same channels in the conv, which reads
// only those channels of v, H and the state's ring. The one grid-wide dependency is the
// context gate's RMSNorm sums over all d channels (alpha and mean(v^2) of the conv's
// RMSNorm): each block publishes its channels' partial sums, the grid meets once at a
// counter (bounded wait), and every block then reduces all partials in the same order.
//
// Per block (one per SM, 16 warps):
//   0  W streams from the first cycle: the block's W rows form 16-row tiles (row r of the
//      block is W row mat * d + c_lo + ch for r = mat * nch + ch); warp w owns k-steps
//      [w kq, w kq + kq) of every tile and copies that slice (16 rows x kq x 32 bytes) of
//      the next 4 tiles into its own shared-memory ring with cp.async, 16 bytes a lane;
//   1  warps b < B: the decode lookup of sequence b into shared memory (decode_token_lookup,
//      bit-identical to pg_decode_lookup's e_t); the other warps fetch the conv's operands
//      of the block's channels (H, the ring's earlier inputs and scalars, the gains);
//   2  the projection on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate):
//      a tile of 16 W rows times e_t^T (8 columns: the sequences), the K dimension split
//      over the 16 warps, each holding its k-steps of e_t as B fragments in registers and
//      refilling its ring slot with its slice of tile i + 4 once tile i is done (no
//      cross-warp waits); partial products are added over the warps in a fixed order
//      through shared memory (deterministic);
//   3  context gate: v rounded to bf16 and written; the block's partial sums
//      (sum gh gk h k, sum k^2, sum h^2 per branch, sum v^2) to the workspace; the grid
//      barrier; alpha, mean(v^2) and the tap factors; the conv + residual on the block's
//      channels, H and the ring updated; block 0 writes alpha, mean(v^2), the ring's
//      scalars, the ID ring and pos (every block has read them before the barrier).
//      Scalar / no gate: out = x + g v or v; the last block to arrive at the counter
//      writes the ID ring and pos.
// The grid barrier is one 32-bit counter: every block adds 1 except block 0, which adds
// 2^31 - (G - 1), so that one round adds exactly 2^31: bit 31 flips when the last block
// arrives and the low bits return to their value (0), ready for the next call.
// Sources: Engram notes (arXiv 2601.07372) sections 3.3 (gate, conv), 3.5 (decode);
// PageGram report sections 3.1, 3.3.
#include <cuda_bf16.h>

#include <algorithm>

#include "pg_conv_math.cuh"
#include "pg_gather.cuh"
#include "pg_internal.cuh"

namespace pg {
namespace {

constexpr int kStepThreads = 512;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kStepMaxB = 8;       // sequences per call (one n-tile of the MMA)
constexpr int kStepStages = 4;     // W tiles in flight
constexpr int kStepGroup = 2;      // tiles whose partial products are added per round
constexpr int kStepMaxDin = 4096;  // e_t width
constexpr int kStepMaxKq = kStepMaxDin / 16 / kStepWarps;  // k-steps per warp
constexpr int kStepMaxCh = 64;     // channels per block (d <= 64 x blocks)
constexpr int kStepTaps = 4;
constexpr int kErrStepWait = 32768;  // device error bit: a block gave up waiting at the grid barrier
constexpr int kErrStepCopy = 65536;  // device error bit: a tile of W did not land in time
constexpr uint64_t kStepWaitNs = 1000000000ull;  // bounded waits give up after ~1 s

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool bar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity`: false after the time limit.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  if (bar_try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (!bar_try_wait(bar, parity))
    if (now_ns() - t0 > kStepWaitNs) return false;
  return true;
}

// One arrival on `bar` that also makes its current phase expect `bytes` of copies.
__device__ __forceinline__ void bar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// `bytes` from global `src` into this CTA's shared `dst` (both 16-byte aligned, bytes % 16
// == 0), counted on `bar` when they land.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}


// Four 8x8 b16 matrices from shared memory; lane l gives the address of row l % 8 of
// matrix l / 8, and receives in r[i] the two elements (row l / 4, columns 2 (l % 4), +1)
// of matrix i.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row-major) B (16x8 bf16, column-major).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- parameters and layout

constexpr int kStepMaxM = 8;  // branches

enum StepRows : int { kRowsBf16 = 0, kRowsBf16Flat = 1, kRowsNf4 = 2 };

struct StepParams {
  ItemConst ic[kMaxItems];  // per-(order, head) hash constants, formed on the host
  GatherGeom g;
  int rows;        // StepRows
  int B, Din, d, M, nm, stages;
  int ks, dil, D;  // conv kernel size, dilation, ring depth
  float gs, eps;   // scalar gate g; RMSNorm epsilon
  const int32_t* tokens;
  const uint32_t* canon_map;
  const uint8_t* table;
  int32_t* pos;
  uint32_t* ids;
  const __nv_bfloat16* W;  // [nm d, Din]
  const __nv_bfloat16* x;  // scalar gate residual [B, d]
  __nv_bfloat16* H;        // context gate: [M, B, d]
  const float* gamma_h;
  const float* gamma_k;
  const float* gamma_c;
  const float* conv_w;
  __nv_bfloat16* ring_v;
  float* ring_a;
  float* ring_ms;
  __nv_bfloat16* e_out;    // optional [B, Din]
  __nv_bfloat16* out;      // [B, d]
  float* alpha_out;        // optional [M, B]
  float* v_ms_out;         // optional [B]
  float* partials;         // [B][3 M + 1][blocks]
  uint32_t* counter;       // the grid barrier's counter
  int32_t* err;
  int* err_word;
};

// Dynamic shared memory of a block (byte offsets, 16-byte aligned parts); nch = the
// largest channel count of a block. Rows of W tiles and of e_t are padded by 16 bytes.
struct StepSmem {
  uint32_t ring, e, red, res, h, x, v, gg, wg, total;
};

__host__ __device__ inline uint32_t step_take(uint32_t& o, uint32_t bytes) {
  const uint32_t r = o;
  o += (bytes + 15u) / 16u * 16u;
  return r;
}

// A W tile in shared memory is 8 parts of 2 consecutive rows of one matrix (one bulk copy
// each); part j starts 16 j bytes past a multiple of 128, so the 8 rows one ldmatrix reads
// (row 0 or row 1 of parts 0..7) fall in distinct banks.
__host__ __device__ inline uint32_t step_part_bytes(int Din) { return static_cast<uint32_t>(Din) * 4u + 16u; }

__host__ __device__ inline StepSmem step_smem(int B, int Din, int stages, int nm, int M, int nch) {
  const uint32_t rs = static_cast<uint32_t>(Din) * 2u + 16u;
  StepSmem s;
  uint32_t o = 0;
  s.ring = step_take(o, static_cast<uint32_t>(stages * 8) * step_part_bytes(Din));
  s.e = step_take(o, static_cast<uint32_t>(B) * rs);
  s.red = step_take(o, static_cast<uint32_t>(kStepWarps * kStepGroup * 32 * 16));
  s.res = step_take(o, static_cast<uint32_t>(nm * nch * kStepMaxB * 4));
  s.h = step_take(o, static_cast<uint32_t>(M * B * nch * 4));
  s.x = step_take(o, static_cast<uint32_t>((kStepTaps - 1) * B * nch * 4));
  s.v = step_take(o, static_cast<uint32_t>(B * nch * 4));
  s.gg = step_take(o, static_cast<uint32_t>(nch * 4));
  s.wg = step_take(o, static_cast<uint32_t>(kStepTaps * nch * 4));
  s.total = o;
  return s;
}

// ---------------------------------------------------------------- the kernel

template <int GATE>
__global__ void __launch_bounds__(kStepThreads, 1) decode_step_kernel(const __grid_constant__ HashParams P,
                                                                      const __grid_constant__ StepParams sp) {
  __shared__ ItemConst s_ic[kMaxItems];
  __shared__ float s_nf4[16];
  __shared__ uint32_t s_rows[kStepMaxB][kMaxItems];
  __shared__ uint64_t s_signs[kStepMaxB][kMaxSignWords];
  __shared__ __align__(8) uint64_t s_full[kStepStages];
  __shared__ int s_done[kStepStages];  // warps done with the stage's tile
  __shared__ int s_t[kStepMaxB];
  __shared__ uint32_t s_c0[kStepMaxB];
  __shared__ float s_tot[kStepMaxB][3 * kStepMaxM + 1];
  __shared__ float s_alpha[kStepMaxB][kStepMaxM];
  __shared__ float s_ms[kStepMaxB];
  __shared__ float s_f[kStepTaps][kStepMaxB][kStepMaxM];   // tap factors
  __shared__ float s_ra[kStepTaps][kStepMaxB][kStepMaxM];  // alpha of the earlier taps (ring)
  __shared__ float s_rms[kStepTaps][kStepMaxB];            // mean(v^2) of the earlier taps (ring)
  __shared__ int s_abort;
  extern __shared__ __align__(128) uint8_t s_dyn[];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = sp.B, Din = sp.Din, d = sp.d, M = sp.M, nm = sp.nm, stages = sp.stages;
  const int G = gridDim.x, blk = blockIdx.x;
  const int c_lo = static_cast<int>(static_cast<int64_t>(blk) * d / G);
  const int nch = static_cast<int>(static_cast<int64_t>(blk + 1) * d / G) - c_lo;
  const int nch_max = (d + G - 1) / G;
  // Block row r = mat * nch + ch is W row mat * d + c_lo + ch. Parts: pairs of rows (2 p,
  // 2 p + 1) of one matrix (the last of an odd nch alone), pps per matrix; tile i holds
  // parts 8 i .. 8 i + 7, its row j being row j / 8 of part 8 i + j % 8.
  const int pps = (nch + 1) / 2;
  const int nparts = nm * pps;
  const int ntiles = (nparts + 7) / 8;
  const uint32_t row_bytes = static_cast<uint32_t>(Din) * 2u;
  const uint32_t rs = row_bytes + 16u;  // padded row stride of W tiles and e_t in shared memory
  const StepSmem L = step_smem(B, Din, stages, nm, M, nch_max);
  uint8_t* s_ring = s_dyn + L.ring;
  uint8_t* s_e = s_dyn + L.e;                              // [b][rs]
  float4* s_red = reinterpret_cast<float4*>(s_dyn + L.red);   // [warp][tile of the group][lane]
  float* s_res = reinterpret_cast<float*>(s_dyn + L.res);  // [r][kStepMaxB]
  float* s_h = reinterpret_cast<float*>(s_dyn + L.h);      // [m][b][ch]
  float* s_x = reinterpret_cast<float*>(s_dyn + L.x);      // [j - 1][b][ch] (scalar gate: x [b][ch])
  float* s_v = reinterpret_cast<float*>(s_dyn + L.v);      // [b][ch]
  float* s_gg = reinterpret_cast<float*>(s_dyn + L.gg);    // [ch]
  float* s_wg = reinterpret_cast<float*>(s_dyn + L.wg);    // [j][ch]

  const uint32_t part_bytes = step_part_bytes(Din);
  const uint32_t stage_bytes = 8u * part_bytes;
  // Tile i into stage i % stages, by warp 0: lane 0 arms the stage's barrier with the tile's
  // bytes, then lane j copies part 8 i + j.
  auto issue_tile = [&](int i) {
    const int s = i % stages;
    const uint32_t bar = smem_addr(&s_full[s]);
    int rows = 0;  // rows of this lane's part
    const int pt = 8 * i + lane;
    int mat = 0, ch = 0;
    if (lane < 8 && pt < nparts) {
      mat = pt / pps;
      ch = 2 * (pt - mat * pps);
      rows = min(2, nch - ch);
    }
    int total = rows;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    if (lane == 0) bar_expect(bar, static_cast<uint32_t>(total) * row_bytes);
    __syncwarp();
    if (rows > 0)
      bulk_copy(smem_addr(s_ring + s * stage_bytes + lane * part_bytes),
                sp.W + (static_cast<int64_t>(mat) * d + c_lo + ch) * Din, static_cast<uint32_t>(rows) * row_bytes,
                bar);
  };

  // ---- 0: stage barriers, hash constants
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      bar_init(smem_addr(&s_full[s]), 1);
      s_done[s] = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_abort = 0;
  }
  if (threadIdx.x < sp.g.items) s_ic[threadIdx.x] = sp.ic[threadIdx.x];
  if (threadIdx.x < 16) s_nf4[threadIdx.x] = __uint_as_float(c_nf4_bits[threadIdx.x]);
  __syncthreads();

  // ---- 1: warp 0 starts the first tiles of W; warp 1 + b looks up sequence b; the other
  // warps fetch the conv's operands
  if (warp == 0) {
    for (int i = 0; i < stages && i < ntiles; ++i) issue_tile(i);
  } else if (warp <= B) {
    const int b = warp - 1;
    uint32_t c0 = 0;
    uint8_t* e_tok = s_e + static_cast<uint32_t>(b) * rs;
    int* ew = blk == 0 ? sp.err_word : nullptr;
    int t;
    if (sp.rows == kRowsNf4)
      t = decode_token_lookup<PG_NF4, PG_BF16, false>(P, sp.g, s_ic, s_nf4, s_rows[b], s_signs[b], b,
                                                      lane, sp.tokens, sp.canon_map, sp.table, sp.pos, sp.ids,
                                                      e_tok, sp.err, ew, &c0);
    else if (sp.rows == kRowsBf16Flat)
      t = decode_token_lookup<PG_BF16, PG_BF16, true>(P, sp.g, s_ic, s_nf4, s_rows[b], s_signs[b], b,
                                                      lane, sp.tokens, sp.canon_map, sp.table, sp.pos, sp.ids,
                                                      e_tok, sp.err, ew, &c0);
    else
      t = decode_token_lookup<PG_BF16, PG_BF16, false>(P, sp.g, s_ic, s_nf4, s_rows[b], s_signs[b], b,
                                                       lane, sp.tokens, sp.canon_map, sp.table, sp.pos, sp.ids,
                                                       e_tok, sp.err, ew, &c0);
    if (lane == 0) {
      s_t[b] = t;
      s_c0[b] = c0;
    }
  } else {
    const int tid = threadIdx.x - (B + 1) * 32, nthr = kStepThreads - (B + 1) * 32;
    if (GATE == PG_GATE_SCALAR) {
      for (int i = tid; i < B * nch; i += nthr) {
        const int b = i / nch, ch = i - b * nch;
        s_x[b * nch_max + ch] = __bfloat162float(sp.x[static_cast<int64_t>(b) * d + c_lo + ch]);
      }
    } else if (GATE == PG_GATE_CONTEXT) {
#pragma unroll 4
      for (int i = tid; i < M * B * nch; i += nthr) {
        const int mb = i / nch, ch = i - mb * nch;
        s_h[mb * nch_max + ch] = __bfloat162float(sp.H[static_cast<int64_t>(mb) * d + c_lo + ch]);
      }
      for (int i = tid; i < nch; i += nthr) {
        const int c = c_lo + i;
        const float gc = 0.5f * sp.gamma_c[c];
        float w[kStepTaps];
#pragma unroll
        for (int j = 0; j < kStepTaps; ++j) w[j] = j < sp.ks ? sp.conv_w[c * sp.ks + j] : 0.f;
        s_gg[i] = sp.gamma_h[c] * sp.gamma_k[c];
#pragma unroll
        for (int j = 0; j < kStepTaps; ++j) s_wg[j * nch_max + i] = w[j] * gc;
      }
      // the inputs and scalars of the earlier taps t - j dil (j = 1 .. 3) from the ring
#pragma unroll 2
      for (int i = tid; i < (kStepTaps - 1) * B * nch; i += nthr) {
        const int jb = i / nch, ch = i - jb * nch;
        const int j = 1 + jb / B, b = jb - (j - 1) * B;
        const int t = sp.pos[b], p = t - j * sp.dil;
        float xv = 0.f;
        if (t >= 0 && j < sp.ks && p >= 0)
          xv = __bfloat162float(sp.ring_v[(static_cast<int64_t>(b) * sp.D + p % sp.D) * d + c_lo + ch]);
        s_x[jb * nch_max + ch] = xv;
      }
      for (int i = tid; i < (kStepTaps - 1) * B * (M + 1); i += nthr) {
        const int jb = i / (M + 1), m = i - jb * (M + 1);
        const int j = 1 + jb / B, b = jb - (j - 1) * B;
        const int t = sp.pos[b], p = t - j * sp.dil;
        float val = 0.f;
        if (t >= 0 && j < sp.ks && p >= 0) {
          const int64_t slot = static_cast<int64_t>(b) * sp.D + p % sp.D;
          val = m < M ? sp.ring_a[slot * M + m] : sp.ring_ms[slot];
        }
        if (m < M) s_ra[j][b][m] = val;
        else s_rms[j][b] = val;
      }
    }
  }
  __syncthreads();
  if (blk == 0 && sp.e_out) {
    const int cpr = Din / 8;
    for (int i = threadIdx.x; i < B * cpr; i += kStepThreads) {
      const int b = i / cpr, c = i - b * cpr;
      if (s_t[b] >= 0)
        reinterpret_cast<uint4*>(sp.e_out)[i] = *reinterpret_cast<const uint4*>(s_e + b * rs + c * 16);
    }
  }

  // ---- 2: the projection. Warp w takes k-steps [q0, q0 + nq) of every tile; its B
  // fragments (e_t, 16 k x 8 sequences per step; sequences >= B read row 0) stay in registers.
  {
    const int ksteps = Din / 16;
    const int kq = (ksteps + kStepWarps - 1) / kStepWarps;
    const int q0 = warp * kq;
    const int nq = max(0, min(kq, ksteps - q0));
    uint32_t bf[kStepMaxKq][2];
    {
      const int n = lane & 7;
      const uint32_t erow = smem_addr(s_e + (n < B ? n : 0) * rs) + ((lane >> 3) & 1) * 16u;
#pragma unroll
      for (int q = 0; q < kStepMaxKq; ++q)
        if (q < nq) ldsm_x2(erow + (q0 + q) * 32u, bf[q][0], bf[q][1]);
    }
    // A fragments: lane l reads tile row (l % 8) + 8 ((l / 8) % 2) -- row (l / 8) % 2 of part
    // l % 8 -- at k-columns 8 (l / 16) of the k-step
    const uint32_t a_off = (lane & 7) * part_bytes + ((lane >> 3) & 1) * row_bytes + (lane >> 4) * 16u + q0 * 32u;
    for (int g0 = 0; g0 < ntiles; g0 += kStepGroup) {
      float acc[kStepGroup][4];
#pragma unroll
      for (int u = 0; u < kStepGroup; ++u) {
        acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
        const int i = g0 + u;
        if (i >= ntiles) break;
        const int s = i % stages;
        if (!bar_wait(smem_addr(&s_full[s]), static_cast<uint32_t>(i / stages) & 1u)) {
          if (lane == 0) {
            atomicOr(sp.err_word, kErrStepCopy);
            s_abort = 1;
          }
        }
        const uint32_t base = smem_addr(s_ring + s * stage_bytes) + a_off;
#pragma unroll
        for (int q = 0; q < kStepMaxKq; ++q) {
          if (q < nq) {
            uint32_t a[4];
            ldsm_x4(base + q * 32u, a);
            mma_bf16_16816(acc[u], a, bf[q][0], bf[q][1]);
          }
        }
        // the last warp done with the tile refills its stage with tile i + stages
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&s_done[s], 1) == kStepWarps - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          if (lane == 0) atomicExch(&s_done[s], 0);
          if (i + stages < ntiles) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_tile(i + stages);
          }
        }
      }
      // the group's partial products, added over the warps in warp order
#pragma unroll
      for (int u = 0; u < kStepGroup; ++u)
        s_red[(warp * kStepGroup + u) * 32 + lane] = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
      __syncthreads();
      if (threadIdx.x < kStepGroup * 128) {
        // output (tile row r, column n) of tile u is component (r / 8) * 2 + n % 2 of lane
        // (r % 8) * 4 + n / 2; tile row r is row r / 8 of part 8 (g0 + u) + r % 8
        const int u = threadIdx.x >> 7, e = threadIdx.x & 127;
        const int r = e >> 3, n = e & 7;
        const int ln = (r & 7) * 4 + (n >> 1), comp = (r >> 3) * 2 + (n & 1);
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kStepWarps; ++w) {
          const float4 v = s_red[(w * kStepGroup + u) * 32 + ln];
          sum += comp == 0 ? v.x : (comp == 1 ? v.y : (comp == 2 ? v.z : v.w));
        }
        const int pt = 8 * (g0 + u) + (r & 7);
        if (pt < nparts) {
          const int mat = pt / pps, ch = 2 * (pt - mat * pps) + (r >> 3);
          if (ch < nch) s_res[(mat * nch + ch) * kStepMaxB + n] = sum;
        }
      }
      __syncthreads();
    }
  }

  if constexpr (GATE != PG_GATE_CONTEXT) {
    // ---- 3: out = x + g v (scalar gate) or v
    for (int i = threadIdx.x; i < B * nch; i += kStepThreads) {
      const int b = i / nch, ch = i - b * nch;
      if (s_t[b] < 0) continue;
      const float a = s_res[ch * kStepMaxB + b];
      const float o = GATE == PG_GATE_SCALAR ? fmaf(sp.gs, a, s_x[b * nch_max + ch]) : a;
      sp.out[static_cast<int64_t>(b) * d + c_lo + ch] = __float2bfloat16_rn(o);
    }
    // the last block to arrive (every block has read pos and the ID ring) advances them
    if (threadIdx.x == 0) {
      const uint32_t add = blk == 0 ? 0x80000000u - static_cast<uint32_t>(G - 1) : 1u;
      const uint32_t old = atom_add_release_gpu(sp.counter, add);
      if (((old ^ (old + add)) & 0x80000000u) != 0u) {
        for (int b = 0; b < B; ++b) {
          const int t = s_t[b];
          if (t < 0) continue;
          sp.ids[4 * static_cast<int64_t>(b) + (t & 3)] = s_c0[b];
          sp.pos[b] = t + 1;
        }
      }
    }
  } else {
    const int Q = 3 * M + 1;
    // ---- 3a: v in bf16 (written, and the conv's x_t); the block's partial sums
    for (int i = threadIdx.x; i < B * nch; i += kStepThreads) {
      const int b = i / nch, ch = i - b * nch;
      const __nv_bfloat16 vb = __float2bfloat16_rn(s_res[ch * kStepMaxB + b]);
      if (s_t[b] >= 0) sp.out[static_cast<int64_t>(b) * d + c_lo + ch] = vb;
      s_v[b * nch_max + ch] = __bfloat162float(vb);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < B * Q; i += kStepThreads) {
      const int b = i / Q, q = i - b * Q;
      float s = 0.f;
      if (q < 3 * M) {
        const int kind = q / M, m = q - kind * M;
        const float* hrow = s_h + (m * B + b) * nch_max;
        for (int ch = 0; ch < nch; ++ch) {
          const float k = s_res[((1 + m) * nch + ch) * kStepMaxB + b];
          const float h = hrow[ch];
          s += kind == 0 ? s_gg[ch] * h * k : (kind == 1 ? k * k : h * h);
        }
      } else {
        for (int ch = 0; ch < nch; ++ch) {
          const float v = s_v[b * nch_max + ch];
          s += v * v;
        }
      }
      __stcg(sp.partials + static_cast<int64_t>(i) * G + blk, s);
    }
    // ---- 3b: the grid barrier (bounded): every block's partial sums are published
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t add = blk == 0 ? 0x80000000u - static_cast<uint32_t>(G - 1) : 1u;
      const uint32_t old = atom_add_release_gpu(sp.counter, add);
      if (((ld_acquire_u32(sp.counter) ^ old) & 0x80000000u) == 0u) {
        const uint64_t t0 = now_ns();
        while (((ld_acquire_u32(sp.counter) ^ old) & 0x80000000u) == 0u) {
          if (now_ns() - t0 > kStepWaitNs) {
            atomicOr(sp.err_word, kErrStepWait);
            s_abort = 1;
            break;
          }
        }
      }
    }
    __syncthreads();
    if (!s_abort) {
      // ---- 3c: the sums over all blocks: 8 lanes per (sequence, sum), each adding its
      // blocks j = lane8, lane8 + 8, ... (loads all in flight), then across the 8 lanes;
      // the same order in every block
      constexpr int kLoads = 24;  // up to 192 blocks
      for (int p0 = 0; p0 < B * Q; p0 += kStepThreads / 8) {
        const int p = p0 + (threadIdx.x >> 3), j0 = threadIdx.x & 7;
        float part[kLoads];
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
          const int j = j0 + 8 * u;
          part[u] = (p < B * Q && j < G) ? __ldcg(sp.partials + static_cast<int64_t>(p) * G + j) : 0.f;
        }
        float s = 0.f;
#pragma unroll
        for (int u = 0; u < kLoads; ++u) s += part[u];
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        if (j0 == 0 && p < B * Q) s_tot[p / Q][p % Q] = s;
      }
      __syncthreads();
      // alpha = sigmoid(RMSNorm(h) . RMSNorm(k) / sqrt(d)) and mean(v^2) of each sequence
      const float inv_d = 1.0f / static_cast<float>(d);
      if (threadIdx.x < B * (M + 1)) {
        const int b = threadIdx.x / (M + 1), m = threadIdx.x - b * (M + 1);
        if (m < M) {
          const float rh = sqrtf(__fmaf_rn(s_tot[b][2 * M + m], inv_d, sp.eps));
          const float rk = sqrtf(__fmaf_rn(s_tot[b][M + m], inv_d, sp.eps));
          const float z = s_tot[b][m] / (rh * rk * sqrtf(static_cast<float>(d)));
          s_alpha[b][m] = 1.0f / (1.0f + expf(-z));
        } else {
          s_ms[b] = s_tot[b][3 * M] / static_cast<float>(d);
        }
      }
      __syncthreads();
      // tap factors f = alpha / sqrt(alpha^2 mean(v^2) + eps) of t, t - dil, ... (0 where
      // the tap is past the kernel size or before the start of the sequence)
      if (threadIdx.x < kStepTaps * B * M) {
        const int j = threadIdx.x / (B * M), bm = threadIdx.x - j * (B * M);
        const int b = bm / M, m = bm - b * M;
        const int t = s_t[b];
        float f = 0.f;
        if (j == 0) f = tap_scale(s_alpha[b][m], s_ms[b], sp.eps);
        else if (t >= 0 && j < sp.ks && t - j * sp.dil >= 0) f = tap_scale(s_ra[j][b][m], s_rms[j][b], sp.eps);
        s_f[j][b][m] = f;
      }
      // block 0: alpha, mean(v^2), the ring's scalars of t, the ID ring and pos (every
      // block read pos and the rings before the barrier)
      if (blk == 0 && threadIdx.x < B * (M + 1)) {
        const int b = threadIdx.x / (M + 1), m = threadIdx.x - b * (M + 1);
        const int t = s_t[b];
        if (t >= 0) {
          const int64_t slot = static_cast<int64_t>(b) * sp.D + (sp.D > 0 ? t % sp.D : 0);
          if (m < M) {
            if (sp.alpha_out) sp.alpha_out[static_cast<int64_t>(m) * B + b] = s_alpha[b][m];
            if (sp.D > 0) sp.ring_a[slot * M + m] = s_alpha[b][m];
          } else {
            if (sp.v_ms_out) sp.v_ms_out[b] = s_ms[b];
            if (sp.D > 0) sp.ring_ms[slot] = s_ms[b];
            sp.ids[4 * static_cast<int64_t>(b) + (t & 3)] = s_c0[b];
            sp.pos[b] = t + 1;
          }
        }
      }
      __syncthreads();
      // ---- 3d: conv + SiLU + residual on the block's channels (the decode conv's arithmetic)
      for (int i = threadIdx.x; i < M * B * nch; i += kStepThreads) {
        const int mb = i / nch, ch = i - mb * nch;
        const int m = mb / B, b = mb - m * B;
        const int t = s_t[b];
        if (t < 0) continue;
        const float x0 = s_v[b * nch_max + ch];
        uint64_t prod[kStepTaps];
#pragma unroll
        for (int j = 0; j < kStepTaps; ++j) {
          const float xj = j == 0 ? x0 : s_x[((j - 1) * B + b) * nch_max + ch];
          prod[j] = mul2(pk(s_wg[j * nch_max + ch], 0.f), pk(xj, 0.f));
        }
        uint64_t c = mul2(pk(s_f[0][b][m], 0.f), prod[0]);  // c / 2
#pragma unroll
        for (int j = 1; j < kStepTaps; ++j) c = fma2(pk(s_f[j][b][m], 0.f), prod[j], c);
        const uint64_t acc = fma2(pk(s_alpha[b][m], 0.f), pk(x0, 0.f), pk(s_h[mb * nch_max + ch], 0.f));
        float y, unused;
        upk(silu2_add<__nv_bfloat16>(c, acc), y, unused);
        sp.H[static_cast<int64_t>(mb) * d + c_lo + ch] = __float2bfloat16_rn(y);
        if (m == 0 && sp.D > 0)
          sp.ring_v[(static_cast<int64_t>(b) * sp.D + t % sp.D) * d + c_lo + ch] = __float2bfloat16_rn(x0);
      }
    }
  }
}

// ---------------------------------------------------------------- host side

using StepFn = void (*)(const HashParams, const StepParams);

StepFn pick_step(int gate) {
  if (gate == PG_GATE_CONTEXT) return decode_step_kernel<PG_GATE_CONTEXT>;
  if (gate == PG_GATE_SCALAR) return decode_step_kernel<PG_GATE_SCALAR>;
  return decode_step_kernel<PG_GATE_NONE>;
}

// Blocks of a step: one per SM, at most one per channel.
int step_blocks(int d) { return std::min(sm_count(), d); }
constexpr int kStepMaxBlocks = 192;  // the partial-sum reduction's loads per lane x 8

constexpr uint64_t kStepCounterBytes = 256;

uint64_t step_workspace_bytes(int B, int M, int G) {
  return kStepCounterBytes + static_cast<uint64_t>(B) * (3 * M + 1) * G * 4u;
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace
}  // namespace pg

extern "C" {

pg_status pg_decode_step_workspace_size(int32_t B, int32_t d, int32_t M, uint64_t* bytes) {
  using namespace pg;
  if (!bytes) return PG_ERR_NULL;
  if (B < 1 || B > kStepMaxB || d < 1 || M < 0 || M > kStepMaxM) return PG_ERR_SHAPE;
  const int G = step_blocks(d);
  if (G < 1) return cuda_fail(cudaGetLastError());
  *bytes = step_workspace_bytes(B, M, G);
  return PG_OK;
}

pg_status pg_decode_step(const pg_table_desc* desc, const pg_decode_state* state, const int32_t* tokens,
                         const uint32_t* canon_map, const void* table, uint64_t table_bytes,
                         const pg_decode_step_args* a, void* workspace, uint64_t workspace_bytes,
                         int32_t* err_index, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!a) return PG_ERR_NULL;
  Geometry geo;
  pg_status st = validate_desc(desc, &geo);
  if (st != PG_OK) return st;
  if (desc->hash_kind != PG_HASH_MULXOR) return PG_ERR_UNSUPPORTED;
  const int gate = a->gate_kind;
  if (gate != PG_GATE_NONE && gate != PG_GATE_SCALAR && gate != PG_GATE_CONTEXT) return PG_ERR_UNSUPPORTED;
  const bool ctx = gate == PG_GATE_CONTEXT;
  st = decode_state_check(state, ctx);
  if (st != PG_OK) return st;
  if (!tokens || !table || !a->W || !a->out || !workspace) return PG_ERR_NULL;
  if (gate == PG_GATE_SCALAR && !a->x_resid) return PG_ERR_NULL;
  if (ctx && (!a->H || !a->gamma_h || !a->gamma_k || !a->gamma_c || !a->conv_w)) return PG_ERR_NULL;
  if (table_bytes < geo.rows * geo.row_bytes) return PG_ERR_RANGE;
  const bool flat = desc->mode == PG_FLAT;
  if (desc->row_dtype != PG_BF16 && !(desc->row_dtype == PG_NF4 && !flat)) return PG_ERR_DTYPE;
  const int items = geo.O * geo.H;
  if (items > kMaxItems || items * geo.W > kMaxSignWords) return PG_ERR_UNSUPPORTED;
  if (desc->row_dtype != PG_NF4 && geo.row_bytes % 16) return PG_ERR_UNSUPPORTED;
  const int B = state->B, d = a->d, Din = static_cast<int>(geo.e_width);
  const int M = ctx ? state->M : 0;
  if (B > kStepMaxB) return PG_ERR_UNSUPPORTED;
  if (device_cc() != 103 && device_cc() != 100) return PG_ERR_DEVICE;
  if (d < 1 || Din % 16 || Din > kStepMaxDin) return PG_ERR_SHAPE;
  if (ctx && (state->d != d || state->dtype != PG_BF16 || M > kStepMaxM)) return PG_ERR_SHAPE;
  if (!aligned16(table) || !aligned16(a->W) || !aligned16(workspace) || (a->e_out && !aligned16(a->e_out)))
    return PG_ERR_ALIGN;
  const int G = step_blocks(d);
  if (G < 1) return cuda_fail(cudaGetLastError());
  if (G > kStepMaxBlocks || (d + G - 1) / G > kStepMaxCh) return PG_ERR_UNSUPPORTED;
  if (workspace_bytes < step_workspace_bytes(B, M, G)) return PG_ERR_WORKSPACE;

  HashParams P;
  fill_hash_params(desc, geo, &P);
  StepParams sp{};
  for (int i = 0; i < items; ++i) init_item_const(sp.ic[i], P, desc->hash_seed, i);
  sp.g.N = B;
  sp.g.items = items;
  sp.g.W = geo.W;
  sp.g.rc = desc->row_dtype == PG_NF4 ? 8u : geo.row_bytes / 16u;
  sp.g.per_tok = flat ? static_cast<int>(sp.g.rc) : items * static_cast<int>(sp.g.rc);
  sp.g.row_bytes = geo.row_bytes;
  sp.g.e_bytes = geo.e_width * 2u;
  sp.g.table_bytes = table_bytes;
  sp.rows = desc->row_dtype == PG_NF4 ? kRowsNf4 : (flat ? kRowsBf16Flat : kRowsBf16);
  sp.B = B;
  sp.Din = Din;
  sp.d = d;
  sp.M = M;
  sp.nm = ctx ? 1 + M : 1;
  sp.ks = ctx ? state->kernel_size : 1;
  sp.dil = ctx ? state->dilation : 1;
  sp.D = ctx ? state->depth : 0;
  sp.gs = a->g;
  sp.eps = a->eps;
  sp.tokens = tokens;
  sp.canon_map = canon_map;
  sp.table = static_cast<const uint8_t*>(table);
  sp.pos = state->pos;
  sp.ids = state->ids;
  sp.W = static_cast<const __nv_bfloat16*>(a->W);
  sp.x = static_cast<const __nv_bfloat16*>(a->x_resid);
  sp.H = static_cast<__nv_bfloat16*>(a->H);
  sp.gamma_h = a->gamma_h;
  sp.gamma_k = a->gamma_k;
  sp.gamma_c = a->gamma_c;
  sp.conv_w = a->conv_w;
  sp.ring_v = static_cast<__nv_bfloat16*>(state->ring_v);
  sp.ring_a = state->ring_alpha;
  sp.ring_ms = state->ring_ms;
  sp.e_out = static_cast<__nv_bfloat16*>(a->e_out);
  sp.out = static_cast<__nv_bfloat16*>(a->out);
  sp.alpha_out = a->alpha_out;
  sp.v_ms_out = a->v_ms_out;
  sp.counter = static_cast<uint32_t*>(workspace);
  sp.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStepCounterBytes);
  sp.err = err_index;
  sp.err_word = device_error_word();

  // W tiles in flight: as many (up to 4) as fit beside the rest of shared memory
  const int nch_max = (d + G - 1) / G;
  StepFn fn = pick_step(gate);
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return cuda_fail(e);
  int dev = 0, optin = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const int budget = optin - static_cast<int>(fa.sharedSizeBytes);
  int stages = kStepStages;
  while (stages > 1 && static_cast<int>(step_smem(B, Din, stages, sp.nm, M, nch_max).total) > budget) --stages;
  const uint32_t smem = step_smem(B, Din, stages, sp.nm, M, nch_max).total;
  if (static_cast<int>(smem) > budget) return PG_ERR_UNSUPPORTED;
  sp.stages = stages;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e);
  // the grid barrier needs every block resident at once: one per SM must fit
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kStepThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  if (per_sm < 1 || G > per_sm * sm_count()) return PG_ERR_UNSUPPORTED;

  st = prepare_err(err_index, stream);
  if (st != PG_OK) return st;
  fn<<<static_cast<unsigned>(G), kStepThreads, smem, stream>>>(P, sp);
  return after_launch(1);
}

}  // extern "C"
