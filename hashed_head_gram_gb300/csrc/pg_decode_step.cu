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

#include "pg_async.cuh"
#include "pg_conv_math.cuh"
#include "pg_gather.cuh"
#include "pg_internal.cuh"

namespace pg {
namespace {

constexpr int kStepThreads = 512;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kStepMaxB = 8;       // sequences per call (one n-tile of the MMA)
constexpr int kStepBoxCols = 64;   // W columns per TMA box (one 128-byte swizzled row)
constexpr int kStepMaxTiles = 8;   // 16-row MMA tiles per block (W rows per block <= 128)
constexpr int kStepMaxDin = 4096;  // e_t width
constexpr int kStepMaxCh = 64;     // channels per block (d <= 64 x blocks)
constexpr int kStepTaps = 4;
constexpr int kErrStepWait = 32768;  // device error bit: a block gave up waiting at the grid barrier
constexpr int kErrStepCopy = 65536;  // device error bit: a tile of W did not land in time

// ---------------------------------------------------------------- PTX wrappers

// Box (x, y, z) of the 3-D tensor `map` into shared `dst`, counted on `bar` when it lands.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Programmatic dependent launch: wait until the grids this one depends on have completed
// and their writes are visible; let the next grid in the stream start being scheduled.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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
  CUtensorMap wmap;         // W as [nm][d][Din], boxes of 64 columns x nch_max rows x nm, 128-byte swizzle
  ItemConst ic[kMaxItems];  // per-(order, head) hash constants, formed on the host
  GatherGeom g;
  int rows;        // StepRows
  int split;       // 1: warp w owns W columns [80 w, 80 w + 80): a 64-column box + one k-step in registers
  int B, Din, d, M, nm;
  int ks, dil, D;  // conv kernel size, dilation, ring depth
  float gs, eps;   // scalar gate g; RMSNorm epsilon
  float inv_nm;    // 1 / nm
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

// Dynamic shared memory of a block (byte offsets from a 1024-byte aligned base; the
// allocation adds 1024 bytes for that alignment); nch = the largest channel count of a block.
// Every warp has one slot for a W box (nm x nch rows of 128 bytes, 128-byte swizzle), the
// slots 1024-byte aligned, 2 KB past the last one for the MMA tiles' rows past a box; the
// slots are reused for the cross-warp sums once every box is consumed. Rows of e_t are
// padded by 16 bytes (ldmatrix's 8 rows in distinct banks).
struct StepSmem {
  uint32_t slot, ring, e, res, h, x, v, gg, wg, total;
};

__host__ __device__ inline uint32_t step_take(uint32_t& o, uint32_t bytes) {
  const uint32_t r = o;
  o += (bytes + 15u) / 16u * 16u;
  return r;
}

__host__ __device__ inline StepSmem step_smem(int B, int Din, int nm, int M, int nch) {
  const uint32_t rs = static_cast<uint32_t>(Din) * 2u + 16u;
  const int ntiles = (nm * nch + 15) / 16;
  StepSmem s;
  s.slot = (static_cast<uint32_t>(nm * nch) * 128u + 1023u) / 1024u * 1024u;
  const uint32_t ring = kStepWarps * s.slot + 2048u;
  const uint32_t red = static_cast<uint32_t>(kStepWarps * ntiles * 32 * 16);
  uint32_t o = 0;
  s.ring = step_take(o, ring > red ? ring : red);
  s.e = step_take(o, static_cast<uint32_t>(B) * rs);
  s.res = step_take(o, static_cast<uint32_t>(nm * nch * kStepMaxB * 4));
  s.h = step_take(o, static_cast<uint32_t>(M * B * nch * 4));
  s.x = step_take(o, static_cast<uint32_t>((kStepTaps - 1) * B * nch * 4));
  s.v = step_take(o, static_cast<uint32_t>(B * nch * 4));
  s.gg = step_take(o, static_cast<uint32_t>(nch * 4));
  s.wg = step_take(o, static_cast<uint32_t>(kStepTaps * nch * 4));
  s.total = o + 1024u;
  return s;
}

// The per-block partial sums [pair][G] of every (sequence, sum) pair, added over the G
// blocks: LP lanes per pair, lane j0 adding blocks j0, j0 + LP, ... (all its loads in
// flight), then the LP lanes in an xor tree; the same order in every block.
constexpr int kStepMaxBlocks = 160;
template <int LP>
__device__ __forceinline__ void step_sum_partials(const float* partials, int PQ, int G, int Q,
                                                  float (*s_tot)[3 * kStepMaxM + 1]) {
  constexpr int kLoads = kStepMaxBlocks / LP;
  for (int p0 = 0; p0 < PQ; p0 += kStepThreads / LP) {
    const int p = p0 + static_cast<int>(threadIdx.x) / LP, j0 = static_cast<int>(threadIdx.x) % LP;
    float part[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int j = j0 + LP * u;
      part[u] = (p < PQ && j < G) ? __ldcg(partials + static_cast<int64_t>(p) * G + j) : 0.f;
    }
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < kLoads; ++u) s += part[u];
#pragma unroll
    for (int o = 1; o < LP; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (j0 == 0 && p < PQ) s_tot[p / Q][p % Q] = s;
  }
}

// ---------------------------------------------------------------- the kernel

template <int GATE, int ROWS>
__global__ void __launch_bounds__(kStepThreads, 1) decode_step_kernel(const __grid_constant__ HashParams P,
                                                                      const __grid_constant__ StepParams sp) {
  __shared__ ItemConst s_ic[kMaxItems];
  __shared__ float s_nf4[16];
  __shared__ uint32_t s_rows[kStepMaxB][kMaxItems];
  __shared__ uint64_t s_signs[kStepMaxB][kMaxSignWords];
  __shared__ __align__(8) uint64_t s_full[kStepWarps];  // each warp's W box
  __shared__ int s_t[kStepMaxB];
  __shared__ uint32_t s_c0[kStepMaxB];
  __shared__ float s_tot[kStepMaxB][3 * kStepMaxM + 1];
  __shared__ float s_alpha[kStepMaxB][kStepMaxM];
  __shared__ float s_f[kStepTaps][kStepMaxB][kStepMaxM];   // tap factors
  __shared__ float s_ra[kStepTaps][kStepMaxB][kStepMaxM];  // alpha of the earlier taps (ring)
  __shared__ float s_rms[kStepTaps][kStepMaxB];            // mean(v^2) of the earlier taps (ring)
  __shared__ int s_abort;
  __shared__ int16_t s_rowmap[16 * kStepMaxTiles];  // box row R -> block row mat * nch + y, or -1
  extern __shared__ __align__(128) uint8_t s_dyn[];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = sp.B, Din = sp.Din, d = sp.d, M = sp.M, nm = sp.nm;
  const int G = gridDim.x, blk = blockIdx.x;
  const int c_lo = static_cast<int>(static_cast<int64_t>(blk) * d / G);
  const int nch = static_cast<int>(static_cast<int64_t>(blk + 1) * d / G) - c_lo;
  const int nch_max = (d + G - 1) / G;
  // Block row r = mat * nch + ch is W row mat * d + c_lo + ch. A W box holds 64 columns of
  // the rows mat * d + c_lo + y, y < nch_max (rows of the next block's channels past nch, zeros
  // past d), for every mat: box row R = mat * nch_max + y; MMA tile t is box rows 16 t .. 16 t + 15.
  const int ntiles = (nm * nch_max + 15) / 16;
  const int nbox = Din / kStepBoxCols;
  const uint32_t row_bytes = static_cast<uint32_t>(Din) * 2u;
  const uint32_t rs = row_bytes + 16u;  // padded row stride of W tiles and e_t in shared memory
  const StepSmem L = step_smem(B, Din, nm, M, nch_max);
  uint8_t* s_base = s_dyn + ((1024u - (smem_addr(s_dyn) & 1023u)) & 1023u);
  uint8_t* s_ring = s_base + L.ring;
  uint8_t* s_e = s_base + L.e;                              // [b][rs]
  float4* s_red = reinterpret_cast<float4*>(s_ring);          // [warp][tile][lane], once the boxes are used
  float* s_res = reinterpret_cast<float*>(s_base + L.res);  // [r][kStepMaxB]
  float* s_h = reinterpret_cast<float*>(s_base + L.h);      // [m][b][ch]
  float* s_x = reinterpret_cast<float*>(s_base + L.x);      // [j - 1][b][ch] (scalar gate: x [b][ch])
  float* s_v = reinterpret_cast<float*>(s_base + L.v);      // [b][ch]
  float* s_gg = reinterpret_cast<float*>(s_base + L.gg);    // [ch]
  float* s_wg = reinterpret_cast<float*>(s_base + L.wg);    // [j][ch]

  // box j of this warp (j = warp, warp + 16, ...) into its slot, by lane 0
  const uint32_t box_bytes = static_cast<uint32_t>(nm * nch_max) * 128u;
  const uint32_t my_slot = smem_addr(s_ring) + static_cast<uint32_t>(warp) * L.slot;
  const uint32_t my_bar = smem_addr(&s_full[warp]);
  auto issue_box = [&](int x) {  // the box of columns [x, x + 64)
    bar_expect(my_bar, box_bytes);
    tma_load_3d(my_slot, &sp.wmap, my_bar, x, c_lo, 0);
  };
  // split layout (Din = 16 x 80): the warp's last k-step (columns 80 w + 64 .. 80 w + 79) of
  // every tile as mma A fragments in registers, loaded from W (L2) at once: lane (g, tq)
  // holds rows 16 t + g and + 8 at columns 2 tq, + 1 and 2 tq + 8, + 9 of the k-step
  uint32_t ra[kStepMaxTiles][4];
  if (sp.split) {
    const int g = lane >> 2, tq = lane & 3;
    const int col = warp * 80 + 64 + 2 * tq;
    auto w_pair = [&](int R, int c) -> uint32_t {  // two bf16 of box row R at column c
      const int mat = R / nch_max, y = R - mat * nch_max;
      if (mat >= nm || c_lo + y >= d) return 0u;
      return __ldg(reinterpret_cast<const uint32_t*>(sp.W + (static_cast<int64_t>(mat) * d + c_lo + y) * Din + c));
    };
#pragma unroll
    for (int t = 0; t < kStepMaxTiles; ++t) {
      if (t < ntiles) {
        ra[t][0] = w_pair(16 * t + g, col);
        ra[t][1] = w_pair(16 * t + g + 8, col);
        ra[t][2] = w_pair(16 * t + g, col + 8);
        ra[t][3] = w_pair(16 * t + g + 8, col + 8);
      }
    }
  }

  // ---- 0: each warp's W barrier and first box (W streams from the first instructions),
  // hash constants
  if (lane == 0) {
    bar_init(my_bar, 1);
    bar_init_fence();
    if (sp.split) issue_box(warp * 80);
    else if (warp < nbox) issue_box(warp * kStepBoxCols);
  }
  if (threadIdx.x == 0) s_abort = 0;
  // warp b < B: the window of sequence b's token (pos, the ID ring, the canonical ID), loads
  // only; meanwhile the other warps copy the hash constants, one item per warp and a word per
  // lane (uniform-address loads of the parameter space stay fast; items in one warp serialise)
  int t_b = 0;
  uint32_t c0_b = 0, slot_b = 0;
  // (W, the table, the maps and the gains are read-only; everything else that this step reads
  // may be written by the grid before it in the stream: read only after grid_dep_wait)
  if (warp < B) {
    grid_dep_wait();
    t_b = decode_token_window(P, warp, lane, sp.tokens, sp.canon_map, sp.pos, sp.ids, sp.err, &c0_b, &slot_b);
  } else {
    constexpr int kWords = static_cast<int>(sizeof(ItemConst) / 4);
    for (int it = warp - B; it < sp.g.items; it += kStepWarps - B) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(&sp.ic[it]);
      uint32_t* dst = reinterpret_cast<uint32_t*>(&s_ic[it]);
      for (int i = lane; i < kWords; i += 32) dst[i] = src[i];
    }
    if (warp == kStepWarps - 1 && lane < 16) s_nf4[lane] = __uint_as_float(c_nf4_bits[lane]);
    for (int R = threadIdx.x - B * 32; R < 16 * kStepMaxTiles; R += kStepThreads - B * 32) {
      const int mat = R / nch_max, y = R - mat * nch_max;
      s_rowmap[R] = static_cast<int16_t>(mat < nm && y < nch ? mat * nch + y : -1);
    }
    grid_dep_wait();
  }
  __syncthreads();

  // ---- 1: warp b looks up sequence b; the other warps fetch the conv's operands
  if (warp < B) {
    const int b = warp;
    uint8_t* e_tok = s_e + static_cast<uint32_t>(b) * rs;
    int* ew = blk == 0 ? sp.err_word : nullptr;
    if constexpr (ROWS == kRowsNf4)
      decode_token_gather<PG_NF4, PG_BF16, false>(P, sp.g, s_ic, s_nf4, s_rows[b], s_signs[b], lane, t_b, c0_b,
                                                  slot_b, sp.table, e_tok, ew);
    else if constexpr (ROWS == kRowsBf16Flat)
      decode_token_gather<PG_BF16, PG_BF16, true>(P, sp.g, s_ic, s_nf4, s_rows[b], s_signs[b], lane, t_b, c0_b,
                                                  slot_b, sp.table, e_tok, ew);
    else
      decode_token_gather<PG_BF16, PG_BF16, false>(P, sp.g, s_ic, s_nf4, s_rows[b], s_signs[b], lane, t_b, c0_b,
                                                   slot_b, sp.table, e_tok, ew);
    if (lane == 0) {
      s_t[b] = t_b;
      s_c0[b] = c0_b;
    }
  } else {
    const int tid = threadIdx.x - B * 32, nthr = kStepThreads - B * 32;
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

  // ---- 2: the projection. Warp w takes W boxes j = w, w + 16, ... (64 columns: k-steps
  // 4 j .. 4 j + 3) of every tile, or (split) its 80 columns; the B fragments (e_t, 16 k x 8
  // sequences per step; sequences >= B read row 0) come from e_t in shared memory.
  {
    float acc[kStepMaxTiles][4];
#pragma unroll
    for (int t = 0; t < kStepMaxTiles; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    const int n = lane & 7;
    const uint32_t erow = smem_addr(s_e + (n < B ? n : 0) * rs) + ((lane >> 3) & 1) * 16u;
    // A fragments: lane l reads box row 16 t + (l % 8) + 8 ((l / 8) % 2), 16-byte chunk
    // 2 q + l / 16 of the k-step, at its 128-byte swizzled place (chunk ^ (row % 8))
    const int ar = lane & 7;
    const uint32_t a_row = my_slot + static_cast<uint32_t>(ar + 8 * ((lane >> 3) & 1)) * 128u;
    const int a_hi = lane >> 4;
    // the k-steps of the box at column x (4 x 16 columns) of every tile
    auto box_mma = [&](int x) {
      uint32_t bf[4][2];
#pragma unroll
      for (int q = 0; q < 4; ++q) ldsm_x2(erow + static_cast<uint32_t>(x * 2 + q * 32), bf[q][0], bf[q][1]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t a_q = a_row + ((static_cast<uint32_t>(2 * q + a_hi) ^ ar) << 4);
#pragma unroll
        for (int t = 0; t < kStepMaxTiles; ++t) {
          if (t < ntiles) {
            uint32_t a[4];
            ldsm_x4(a_q + t * 2048u, a);
            mma_bf16_16816(acc[t], a, bf[q][0], bf[q][1]);
          }
        }
      }
    };
    auto box_wait = [&](int k) {
      if (!bar_wait(my_bar, static_cast<uint32_t>(k) & 1u)) {
        if (lane == 0) {
          atomicOr(sp.err_word, kErrStepCopy);
          s_abort = 1;
        }
      }
    };
    if (sp.split) {
      box_wait(0);
      box_mma(warp * 80);
      uint32_t b0, b1;
      ldsm_x2(erow + static_cast<uint32_t>((warp * 80 + 64) * 2), b0, b1);
#pragma unroll
      for (int t = 0; t < kStepMaxTiles; ++t)
        if (t < ntiles) mma_bf16_16816(acc[t], ra[t], b0, b1);
    } else {
      // boxes j = warp, warp + 16, ... through the warp's slot
      int k = 0;
      for (int j = warp; j < nbox; j += kStepWarps, ++k) {
        box_wait(k);
        box_mma(j * kStepBoxCols);
        __syncwarp();  // every lane is done with the slot: it takes the warp's next box
        if (lane == 0 && j + kStepWarps < nbox) {
          fence_async_smem();
          issue_box((j + kStepWarps) * kStepBoxCols);
        }
      }
    }
    // the partial products, added over the warps in warp order (the slots are free now)
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kStepMaxTiles; ++t)
      if (t < ntiles) s_red[(warp * ntiles + t) * 32 + lane] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
    __syncthreads();
    for (int o = threadIdx.x; o < ntiles * 32; o += kStepThreads) {
      // lane ln of tile t holds (tile row r, column n) for r = ln / 4 + 8 (c / 2),
      // n = 2 (ln % 4) + c % 2 in component c; tile row r is box row R = 16 t + r
      const int t = o >> 5, ln = o & 31;
      float4 v[kStepWarps];
#pragma unroll
      for (int w = 0; w < kStepWarps; ++w) v[w] = s_red[(w * ntiles + t) * 32 + ln];
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kStepWarps; ++w) {
        sum[0] += v[w].x;
        sum[1] += v[w].y;
        sum[2] += v[w].z;
        sum[3] += v[w].w;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int row = s_rowmap[16 * t + (ln >> 2) + 8 * (c >> 1)], nn = 2 * (ln & 3) + (c & 1);
        if (row >= 0) s_res[row * kStepMaxB + nn] = sum[c];
      }
    }
    __syncthreads();
  }

  if constexpr (GATE != PG_GATE_CONTEXT) {
    if (threadIdx.x == 0) grid_dep_launch();  // no grid barrier: the next step may be scheduled
    // ---- 3: out = x + g v (scalar gate) or v
    {  // thread (b, ch) = (threadIdx / 64, threadIdx % 64)
      const int b = threadIdx.x >> 6, ch = threadIdx.x & 63;
      if (b < B && ch < nch && s_t[b] >= 0) {
        const float a = s_res[ch * kStepMaxB + b];
        const float o = GATE == PG_GATE_SCALAR ? fmaf(sp.gs, a, s_x[b * nch_max + ch]) : a;
        sp.out[static_cast<int64_t>(b) * d + c_lo + ch] = __float2bfloat16_rn(o);
      }
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
    {  // thread (b, ch) = (threadIdx / 64, threadIdx % 64)
      const int b = threadIdx.x >> 6, ch = threadIdx.x & 63;
      if (b < B && ch < nch) {
        const __nv_bfloat16 vb = __float2bfloat16_rn(s_res[ch * kStepMaxB + b]);
        if (s_t[b] >= 0) sp.out[static_cast<int64_t>(b) * d + c_lo + ch] = vb;
        s_v[b * nch_max + ch] = __bfloat162float(vb);
      }
    }
    __syncthreads();
    // a warp per (sequence b, matrix mat), a lane per channel: mat 0 gives sum v^2, branch
    // m = mat - 1 the sums gh gk h k, k^2 and h^2; each added in an xor tree
    for (int task = warp; task < B * nm; task += kStepWarps) {
      const int b = __float2int_rz((static_cast<float>(task) + 0.5f) * sp.inv_nm), mat = task - b * nm;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f;
      for (int ch = lane; ch < nch; ch += 32) {
        if (mat == 0) {
          const float v = s_v[b * nch_max + ch];
          s0 += v * v;
        } else {
          const float k = s_res[(mat * nch + ch) * kStepMaxB + b];
          const float h = s_h[((mat - 1) * B + b) * nch_max + ch];
          s0 += s_gg[ch] * h * k;
          s1 += k * k;
          s2 += h * h;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      }
      if (lane == 0) {
        float* pb = sp.partials + static_cast<int64_t>(b) * Q * G + blk;
        if (mat == 0) {
          __stcg(pb + static_cast<int64_t>(3 * M) * G, s0);
        } else {
          const int m = mat - 1;
          __stcg(pb + static_cast<int64_t>(m) * G, s0);
          __stcg(pb + static_cast<int64_t>(M + m) * G, s1);
          __stcg(pb + static_cast<int64_t>(2 * M + m) * G, s2);
        }
      }
    }
    // ---- 3b: the grid barrier (bounded): every block's partial sums are published
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t add = blk == 0 ? 0x80000000u - static_cast<uint32_t>(G - 1) : 1u;
      const uint32_t old = atom_add_release_gpu(sp.counter, add);
      if (((ld_acquire_u32(sp.counter) ^ old) & 0x80000000u) == 0u) {
        const uint64_t t0 = now_ns();
        while (((ld_acquire_u32(sp.counter) ^ old) & 0x80000000u) == 0u) {
          if (now_ns() - t0 > kAsyncWaitNs) {
            atomicOr(sp.err_word, kErrStepWait);
            s_abort = 1;
            break;
          }
        }
      }
    }
    __syncthreads();
    // every block is resident (it reached the barrier): the next step may be scheduled
    if (threadIdx.x == 0) grid_dep_launch();
    if (!s_abort) {
      // ---- 3c: the sums over all blocks, the same order in every block; then alpha =
      // sigmoid(RMSNorm(h) . RMSNorm(k) / sqrt(d)), mean(v^2) and the tap factors
      // f = alpha / sqrt(alpha^2 mean(v^2) + eps) of t, t - dil, ... (0 where the tap is past
      // the kernel size or before the start of the sequence)
      if (B * Q <= kStepThreads / 8)
        step_sum_partials<8>(sp.partials, B * Q, G, Q, s_tot);
      else
        step_sum_partials<4>(sp.partials, B * Q, G, Q, s_tot);
      __syncthreads();
      if (threadIdx.x < B * M) {
        const int b = threadIdx.x / M, m = threadIdx.x - b * M;
        const float inv_d = 1.0f / static_cast<float>(d);
        const float rh = sqrtf(__fmaf_rn(s_tot[b][2 * M + m], inv_d, sp.eps));
        const float rk = sqrtf(__fmaf_rn(s_tot[b][M + m], inv_d, sp.eps));
        const float z = s_tot[b][m] / (rh * rk * sqrtf(static_cast<float>(d)));
        const float a = 1.0f / (1.0f + expf(-z));
        const float ms = s_tot[b][3 * M] / static_cast<float>(d);
        const int t = s_t[b];
        s_alpha[b][m] = a;
        s_f[0][b][m] = tap_scale(a, ms, sp.eps);
#pragma unroll
        for (int j = 1; j < kStepTaps; ++j)
          s_f[j][b][m] = (t >= 0 && j < sp.ks && t - j * sp.dil >= 0) ? tap_scale(s_ra[j][b][m], s_rms[j][b], sp.eps)
                                                                      : 0.f;
        // block 0: alpha, mean(v^2), the ring's scalars of t, the ID ring and pos (every
        // block read pos and the rings before the barrier)
        if (blk == 0 && t >= 0) {
          const int64_t slot = static_cast<int64_t>(b) * sp.D + (sp.D > 0 ? t % sp.D : 0);
          if (sp.alpha_out) sp.alpha_out[static_cast<int64_t>(m) * B + b] = a;
          if (sp.D > 0) sp.ring_a[slot * M + m] = a;
          if (m == 0) {
            if (sp.v_ms_out) sp.v_ms_out[b] = ms;
            if (sp.D > 0) sp.ring_ms[slot] = ms;
            sp.ids[4 * static_cast<int64_t>(b) + (t & 3)] = s_c0[b];
            sp.pos[b] = t + 1;
          }
        }
      }
      __syncthreads();
      // ---- 3d: conv + SiLU + residual on the block's channels (the decode conv's arithmetic)
      const int cb = threadIdx.x >> 6, ch = threadIdx.x & 63;  // thread (b, ch), the branches in turn
      if (cb < B && ch < nch && s_t[cb] >= 0) {
        const int b = cb, t = s_t[b];
        const float x0 = s_v[b * nch_max + ch];
        uint64_t prod[kStepTaps];
#pragma unroll
        for (int j = 0; j < kStepTaps; ++j) {
          const float xj = j == 0 ? x0 : s_x[((j - 1) * B + b) * nch_max + ch];
          prod[j] = mul2(pk(s_wg[j * nch_max + ch], 0.f), pk(xj, 0.f));
        }
        if (sp.D > 0)
          sp.ring_v[(static_cast<int64_t>(b) * sp.D + t % sp.D) * d + c_lo + ch] = __float2bfloat16_rn(x0);
        for (int m = 0; m < M; ++m) {
          const int mb = m * B + b;
          uint64_t c = mul2(pk(s_f[0][b][m], 0.f), prod[0]);  // c / 2
#pragma unroll
          for (int j = 1; j < kStepTaps; ++j) c = fma2(pk(s_f[j][b][m], 0.f), prod[j], c);
          const uint64_t acc = fma2(pk(s_alpha[b][m], 0.f), pk(x0, 0.f), pk(s_h[mb * nch_max + ch], 0.f));
          float y, unused;
          upk(silu2_add<__nv_bfloat16>(c, acc), y, unused);
          sp.H[static_cast<int64_t>(mb) * d + c_lo + ch] = __float2bfloat16_rn(y);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- host side

using StepFn = void (*)(const HashParams, const StepParams);

template <int ROWS>
StepFn pick_step_rows(int gate) {
  if (gate == PG_GATE_CONTEXT) return decode_step_kernel<PG_GATE_CONTEXT, ROWS>;
  if (gate == PG_GATE_SCALAR) return decode_step_kernel<PG_GATE_SCALAR, ROWS>;
  return decode_step_kernel<PG_GATE_NONE, ROWS>;
}

// One instantiation per (gate, row type): a kernel holds one lookup variant only (its code
// is read once per launch, so its size shows up as instruction-fetch stalls).
StepFn pick_step(int gate, int rows) {
  if (rows == kRowsNf4) return pick_step_rows<kRowsNf4>(gate);
  if (rows == kRowsBf16Flat) return pick_step_rows<kRowsBf16Flat>(gate);
  return pick_step_rows<kRowsBf16>(gate);
}

// Blocks of a step: one per SM, at most one per channel.
int step_blocks(int d) { return std::min(sm_count(), d); }

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
  if (d < 1 || Din % kStepBoxCols || Din > kStepMaxDin) return PG_ERR_SHAPE;
  if (ctx && (state->d != d || state->dtype != PG_BF16 || M > kStepMaxM)) return PG_ERR_SHAPE;
  if (!aligned16(table) || !aligned16(a->W) || !aligned16(workspace) || (a->e_out && !aligned16(a->e_out)))
    return PG_ERR_ALIGN;
  const int G = step_blocks(d);
  if (G < 1) return cuda_fail(cudaGetLastError());
  const int nm = ctx ? 1 + M : 1;
  const int nch_max = (d + G - 1) / G;
  if (G > kStepMaxBlocks || nch_max > kStepMaxCh || nm * nch_max > 16 * kStepMaxTiles) return PG_ERR_UNSUPPORTED;
  if (workspace_bytes < step_workspace_bytes(B, M, G)) return PG_ERR_WORKSPACE;

  HashParams P;
  fill_hash_params(desc, geo, &P);
  StepParams sp{};
  {  // W as [nm][d][Din]: boxes of 64 columns x nch_max rows x nm, 128-byte swizzle
    auto enc = tensor_map_encoder();
    if (!enc) return PG_ERR_UNSUPPORTED;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(Din), static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(nm)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(Din) * 2, static_cast<cuuint64_t>(d) * Din * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kStepBoxCols), static_cast<cuuint32_t>(nch_max),
                         static_cast<cuuint32_t>(nm)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&sp.wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a->W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PG_ERR_UNSUPPORTED;
  }
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
  sp.split = Din == kStepWarps * 80 ? 1 : 0;
  sp.B = B;
  sp.Din = Din;
  sp.d = d;
  sp.M = M;
  sp.nm = nm;
  sp.inv_nm = 1.0f / static_cast<float>(nm);
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

  StepFn fn = pick_step(gate, sp.rows);
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return cuda_fail(e);
  int dev = 0, optin = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const uint32_t smem = step_smem(B, Din, nm, M, nch_max).total;
  if (static_cast<int>(smem) > optin - static_cast<int>(fa.sharedSizeBytes)) return PG_ERR_UNSUPPORTED;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e);
  // the grid barrier needs every block resident at once: one per SM must fit
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kStepThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  if (per_sm < 1 || G > per_sm * sm_count()) return PG_ERR_UNSUPPORTED;

  st = prepare_err(err_index, stream);
  if (st != PG_OK) return st;
  // programmatic dependent launch: this step's W stream and constants start while the grid
  // before it in the stream finishes (the kernel waits for it before reading its outputs)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G));
  cfg.blockDim = dim3(kStepThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fn, P, sp);
  if (e != cudaSuccess) return cuda_fail(e);
  return after_launch(1);
}

}  // extern "C"
