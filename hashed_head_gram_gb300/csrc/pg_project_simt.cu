// Projections that do not use the tensor cores (sm_103a): the fp32 path of
// pg_project_gate, v = e W_V^T (+ the scalar gate x + g v) on the FP32 FMA pipes (the 1e-5
// fp32 tolerance rules out TF32), and W == NULL (a flat table's e_t is already d wide:
// v = e, or x + g e). PageGram report section 3.1 (scalar gate), Engram notes section 3.4.
#include <cuda_bf16.h>

#include "pg_internal.cuh"

namespace pg {
namespace {

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack_bf16x8(uint4 w, float* f) {
  f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xFFFF0000u);
  f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

// ---------------------------------------------------------------- fp32 SIMT GEMM

constexpr int kSimtTile = 64;   // 64 x 64 outputs per block
constexpr int kSimtK = 32;      // k-tile depth
constexpr int kSimtThreads = 128;

// Cluster rank and distributed shared memory (the split-K sums of a tile's CTAs).
__device__ __forceinline__ uint32_t simt_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void simt_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float4 ld_dsmem_f4(const void* local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(ra)
               : "memory");
  return v;
}

// out[N, Dout] = A[N, Din] B[Dout, Din]^T (+ gate). 128 threads, thread (ty, tx) owns rows
// ty*8 .. ty*8+7 and columns tx*4 .. tx*4+3 of the 64 x 64 tile (8 x 4 fp32 accumulators);
// per k step it reads 8 A values and 4 B values from shared memory (3 vector loads for 32
// FMAs). 32-deep k-tiles are double-buffered: the next tile's global loads are in registers while
// the current one is multiplied. Out-of-range rows, columns and k read as zero.
// KS > 1: a cluster of KS CTAs per tile splits K (CTA z takes k-tiles z, z + KS, ...); each
// writes its partial tile to its shared memory and CTA r adds rows 64 r / KS .. of all
// KS partials in rank order through distributed shared memory (deterministic) and stores
// them: KS times the CTAs of a 64 x 64 grid, so small problems fill the SMs.
template <int GATE, int KS>
__global__ void __launch_bounds__(kSimtThreads) simt_gemm_f32_kernel(const float* __restrict__ A,
                                                                    const float* __restrict__ Bw, int N,
                                                                    int Din, int Dout, const float* __restrict__ x,
                                                                    float g, float* __restrict__ out) {
  __shared__ __align__(16) float As[2][kSimtK][kSimtTile];
  __shared__ __align__(16) float Bs[2][kSimtK][kSimtTile];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * kSimtTile, n0 = blockIdx.x * kSimtTile;
  // global -> register staging: thread loads 8 consecutive k of one A row and of one B row
  const int lr = tid >> 1, lk = (tid & 1) * 16;
  const bool vec = (Din & 3) == 0 && reinterpret_cast<uintptr_t>(A) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(Bw) % 16 == 0;  // 16-byte loads of whole rows
  float ra[16], rb[16];
  auto load_tile = [&](int k0) {
    const int ar = m0 + lr, br = n0 + lr;
    const float* ap = A + static_cast<size_t>(ar) * Din + k0 + lk;
    const float* bp = Bw + static_cast<size_t>(br) * Din + k0 + lk;
    if (vec && k0 + lk + 16 <= Din) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a = ar < N ? __ldg(reinterpret_cast<const float4*>(ap) + q) : z;
        const float4 b = br < Dout ? __ldg(reinterpret_cast<const float4*>(bp) + q) : z;
        ra[4 * q] = a.x; ra[4 * q + 1] = a.y; ra[4 * q + 2] = a.z; ra[4 * q + 3] = a.w;
        rb[4 * q] = b.x; rb[4 * q + 1] = b.y; rb[4 * q + 2] = b.z; rb[4 * q + 3] = b.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int k = k0 + lk + i;
        ra[i] = (ar < N && k < Din) ? __ldg(ap + i) : 0.f;
        rb[i] = (br < Dout && k < Din) ? __ldg(bp + i) : 0.f;
      }
    }
  };
  auto store_tile = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      As[buf][lk + i][lr] = ra[i];
      Bs[buf][lk + i][lr] = rb[i];
    }
  };
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const int kz = KS > 1 ? static_cast<int>(simt_cluster_rank()) : 0;
  load_tile(kz * kSimtK);
  store_tile(0);
  __syncthreads();
  int buf = 0;
  for (int k0 = kz * kSimtK; k0 < Din; k0 += KS * kSimtK) {
    const bool more = k0 + KS * kSimtK < Din;
    if (more) load_tile(k0 + KS * kSimtK);
#pragma unroll
    for (int kk = 0; kk < kSimtK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 8 + 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
    }
    if (more) {
      store_tile(buf ^ 1);
      __syncthreads();
      buf ^= 1;
    }
  }
  if constexpr (KS == 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = m0 + ty * 8 + i;
      if (r >= N) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = n0 + tx * 4 + j;
        if (c < Dout) {
          const size_t off = static_cast<size_t>(r) * Dout + c;
          out[off] = GATE == PG_GATE_SCALAR ? fmaf(g, acc[i][j], x[off]) : acc[i][j];
        }
      }
    }
  } else {
    // the partial tile [64][64] in this CTA's shared memory (the A / B buffers are free)
    float* part = &As[0][0][0];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<float4*>(part + (ty * 8 + i) * kSimtTile + tx * 4) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    simt_cluster_sync();
    constexpr int kRows = kSimtTile / KS;  // rows this CTA adds and stores
    for (int q = threadIdx.x; q < kRows * (kSimtTile / 4); q += kSimtThreads) {
      const int rr = kz * kRows + q / (kSimtTile / 4), c4 = (q % (kSimtTile / 4)) * 4;
      float4 sum = ld_dsmem_f4(part + rr * kSimtTile + c4, 0);
#pragma unroll
      for (int z = 1; z < KS; ++z) {
        const float4 p4 = ld_dsmem_f4(part + rr * kSimtTile + c4, z);
        sum.x += p4.x;
        sum.y += p4.y;
        sum.z += p4.z;
        sum.w += p4.w;
      }
      const int r = m0 + rr;
      if (r < N) {
        const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = n0 + c4 + j;
          if (c < Dout) {
            const size_t off = static_cast<size_t>(r) * Dout + c;
            out[off] = GATE == PG_GATE_SCALAR ? fmaf(g, sv[j], x[off]) : sv[j];
          }
        }
      }
    }
    simt_cluster_sync();  // no CTA leaves while another reads its partial tile
  }
}

// The same product for 16-byte-aligned operands with Din % 4 == 0: 64 threads per 64 x 64
// tile, thread (ty, tx) = (tid / 8, tid % 8) owning rows ty*8 .. ty*8+7 and columns
// tx*8 .. tx*8+7 (8 x 8 fp32 accumulators). The A and B tiles, [64 rows][32 k] each, arrive
// through a kF32Stages-deep cp.async ring (no registers held in flight; rows and k past the
// matrix read as zeros); a 16-byte chunk c of row r sits at chunk c ^ ((r / 8) mod 8), so
// the 8 rows a warp reads at one chunk lie in 8 different bank groups. Per 4-deep k chunk a
// thread reads its 8 A rows and 8 B rows (16 vector loads) for 256 FMAs, each accumulator
// summed over k in increasing order. KS > 1: as above, CTA z of the cluster takes k-tiles
// z, z + KS, ... and CTA r adds rows 64 r / KS .. of the KS partial tiles in rank order.
constexpr int kF32Threads = 64;
constexpr int kF32Stages = 3;

__device__ __forceinline__ void f32_cp_async16(float* smem, const float* gmem, bool fill) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(
                   __cvta_generic_to_shared(smem))),
               "l"(gmem), "r"(fill ? 16 : 0)
               : "memory");
}

template <int GATE, int KS>
__global__ void __launch_bounds__(kF32Threads) simt_gemm_f32_tiled_kernel(const float* __restrict__ A,
                                                                          const float* __restrict__ Bw, int N,
                                                                          int Din, int Dout,
                                                                          const float* __restrict__ x, float g,
                                                                          float* __restrict__ out) {
  __shared__ __align__(16) float As[kF32Stages][kSimtTile][kSimtK];
  __shared__ __align__(16) float Bs[kF32Stages][kSimtTile][kSimtK];
  const int tid = threadIdx.x;
  const int ty = tid >> 3, tx = tid & 7;
  const int m0 = blockIdx.y * kSimtTile, n0 = blockIdx.x * kSimtTile;
  const int kz = KS > 1 ? static_cast<int>(simt_cluster_rank()) : 0;
  const int ntiles = (Din + kSimtK - 1) / kSimtK;
  const int my_tiles = ntiles > kz ? (ntiles - kz + KS - 1) / KS : 0;  // k-tiles kz, kz + KS, ...

  // k-tile `kt` (global index) into stage `st`: 64 rows x 8 chunks of A and of B, 8 + 8
  // chunks per thread (row tid / 8 + 8 q, chunk tid % 8)
  auto load = [&](int kt, int st) {
    const int k0 = kt * kSimtK;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int r = ty + 8 * q, c = tx, k = k0 + 4 * c;
      const int pc = c ^ (r >> 3 & 7);
      const bool ka = k < Din;  // Din % 4 == 0: a chunk is wholly inside K or outside it
      const bool va = ka && m0 + r < N, vb = ka && n0 + r < Dout;
      f32_cp_async16(&As[st][r][4 * pc], va ? A + static_cast<size_t>(m0 + r) * Din + k : A, va);
      f32_cp_async16(&Bs[st][r][4 * pc], vb ? Bw + static_cast<size_t>(n0 + r) * Din + k : Bw, vb);
    }
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

#pragma unroll
  for (int s = 0; s < kF32Stages - 1; ++s) {
    if (s < my_tiles) load(kz + s * KS, s);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int t = 0; t < my_tiles; ++t) {
    asm volatile("cp.async.wait_group %0;" ::"n"(kF32Stages - 2) : "memory");
    __syncthreads();  // stage t landed for every thread; stage t - 1 is no longer read
    if (t + kF32Stages - 1 < my_tiles) load(kz + (t + kF32Stages - 1) * KS, (t + kF32Stages - 1) % kF32Stages);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const int st = t % kF32Stages;
#pragma unroll
    for (int c = 0; c < kSimtK / 4; ++c) {
      float4 a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = *reinterpret_cast<const float4*>(&As[st][ty * 8 + i][4 * (c ^ ty)]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 b = *reinterpret_cast<const float4*>(&Bs[st][tx * 8 + j][4 * (c ^ tx)]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[i][j] = fmaf(a[i].x, b.x, acc[i][j]);
          acc[i][j] = fmaf(a[i].y, b.y, acc[i][j]);
          acc[i][j] = fmaf(a[i].z, b.z, acc[i][j]);
          acc[i][j] = fmaf(a[i].w, b.w, acc[i][j]);
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  if constexpr (KS == 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = m0 + ty * 8 + i;
      if (r >= N) continue;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = n0 + tx * 8 + j;
        if (c < Dout) {
          const size_t off = static_cast<size_t>(r) * Dout + c;
          out[off] = GATE == PG_GATE_SCALAR ? fmaf(g, acc[i][j], x[off]) : acc[i][j];
        }
      }
    }
  } else {
    // the partial tile [64][64] in this CTA's shared memory (the A ring is free)
    float* part = &As[0][0][0];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      *reinterpret_cast<float4*>(part + (ty * 8 + i) * kSimtTile + tx * 8) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4*>(part + (ty * 8 + i) * kSimtTile + tx * 8 + 4) =
          make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    simt_cluster_sync();
    constexpr int kRows = kSimtTile / KS;  // rows this CTA adds and stores
    for (int q = threadIdx.x; q < kRows * (kSimtTile / 4); q += kF32Threads) {
      const int rr = kz * kRows + q / (kSimtTile / 4), c4 = (q % (kSimtTile / 4)) * 4;
      float4 sum = ld_dsmem_f4(part + rr * kSimtTile + c4, 0);
#pragma unroll
      for (int z = 1; z < KS; ++z) {
        const float4 p4 = ld_dsmem_f4(part + rr * kSimtTile + c4, z);
        sum.x += p4.x;
        sum.y += p4.y;
        sum.z += p4.z;
        sum.w += p4.w;
      }
      const int r = m0 + rr;
      if (r < N) {
        const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = n0 + c4 + j;
          if (c < Dout) {
            const size_t off = static_cast<size_t>(r) * Dout + c;
            out[off] = GATE == PG_GATE_SCALAR ? fmaf(g, sv[j], x[off]) : sv[j];
          }
        }
      }
    }
    simt_cluster_sync();  // no CTA leaves while another reads its partial tile
  }
}

// ---------------------------------------------------------------- identity projection

// W == NULL (Din == d): v = e, or x + g e for the scalar gate; 8 elements per thread.
template <typename T, int GATE>
__global__ void __launch_bounds__(256) identity_gate_kernel(const T* __restrict__ e, const T* __restrict__ x,
                                                            float g, T* __restrict__ out, int64_t n) {
  for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * 8; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x * 8) {
    if constexpr (sizeof(T) == 2) {
      const uint4 ev = *reinterpret_cast<const uint4*>(e + i);
      float ef[8], o[8];
      unpack_bf16x8(ev, ef);
      if (GATE == PG_GATE_SCALAR) {
        float xf[8];
        unpack_bf16x8(*reinterpret_cast<const uint4*>(x + i), xf);
#pragma unroll
        for (int q = 0; q < 8; ++q) o[q] = fmaf(g, ef[q], xf[q]);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) o[q] = ef[q];
      }
      *reinterpret_cast<uint4*>(out + i) = make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]),
                                                      pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        out[i + q] = GATE == PG_GATE_SCALAR ? fmaf(g, e[i + q], x[i + q]) : e[i + q];
    }
  }
}

// ---------------------------------------------------------------- bf16, few rows (decode)

// pg_project_gate's bf16 path for N <= kSmallRows rows: out = e W^T over the (1+M) d
// columns is a matrix-vector product per row, bound by reading W once; tensor-core tiles
// of 128 / 256 rows would idle and leave W to a few dozen SMs. A block stages e [N, Din]
// in shared memory and owns `cpb` output columns (for the context gate one 64-column tile
// of the per-row sums); each warp takes CW of them at a time for all rows. Per 16-byte
// chunk of the K dimension a lane holds the chunk of each of its columns (streamed past
// L1, the next chunk's loads issued before the current one is used) and multiplies it
// with that chunk of every row of e, accumulating CW x NB fp32 dot products that a
// butterfly of shuffles completes. The gate is then applied to the block's results in
// shared memory; for the context gate each row's tile sums (sum gh gk h k, sum k^2,
// sum h^2, and sum v^2 of the stored v) are added in column order into the layout the
// alpha finalize pass reads.
template <int NB>
struct SmallCols {
  static constexpr int CW = NB <= 8 ? 4 : 2;  // columns per warp and pass
};

__device__ __forceinline__ uint4 ldg_stream16(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

template <int NB, int GATE>
__global__ void __launch_bounds__(512) small_rows_bf16_kernel(
    const __nv_bfloat16* __restrict__ e, const __nv_bfloat16* __restrict__ W, int N, int Din, int d, int cpb,
    float g, const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ h,
    const float* __restrict__ gamma_h, const float* __restrict__ gamma_k, __nv_bfloat16* __restrict__ out,
    float* __restrict__ partials, float* __restrict__ vpart) {
  constexpr int CW = SmallCols<NB>::CW;
  __shared__ float s_res[kSmallTile][NB];
  __shared__ float s_q[4][NB][kSmallTile];  // per column: h gh gk k, k^2, h^2; v^2
  extern __shared__ __align__(16) uint4 s_e[];  // e, [N][Din / 8] chunks of 8
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int c0 = blockIdx.x * cpb;
  const int chunks = Din >> 3;
  const bool is_k = GATE == PG_GATE_CONTEXT && c0 >= d;
  const int m_br = is_k ? c0 / d - 1 : 0;
  const int kc0 = is_k ? c0 - (m_br + 1) * d : 0;
  // the epilogue's own inputs (context gate, k tiles: h and the two gains of the thread's
  // first (column, row)) and the first K chunk of W are requested before e is staged
  float ep_h = 0.f, ep_g = 0.f;
  if (is_k && threadIdx.x < cpb * N) {
    const int c = threadIdx.x % cpb, n = threadIdx.x / cpb;
    ep_h = __bfloat162float(h[(static_cast<size_t>(m_br) * N + n) * d + kc0 + c]);
    ep_g = gamma_h[kc0 + c] * gamma_k[kc0 + c];
  }
  uint4 cur[CW], nxt[CW];
  int pc = warp * CW;
  if (pc < cpb && lane < chunks) {
#pragma unroll
    for (int c = 0; c < CW; ++c) cur[c] = ldg_stream16(W + static_cast<size_t>(c0 + pc + c) * Din + lane * 8);
  }
  for (int i = threadIdx.x; i < N * chunks; i += blockDim.x) s_e[i] = __ldg(reinterpret_cast<const uint4*>(e) + i);
  __syncthreads();
  for (bool first = true; pc < cpb; pc += nwarps * CW, first = false) {
    float acc[CW][NB];
#pragma unroll
    for (int c = 0; c < CW; ++c)
#pragma unroll
      for (int n = 0; n < NB; ++n) acc[c][n] = 0.f;
    const __nv_bfloat16* wrow = W + static_cast<size_t>(c0 + pc) * Din;
    int kc = lane;
    if (!first && kc < chunks) {
#pragma unroll
      for (int c = 0; c < CW; ++c) cur[c] = ldg_stream16(wrow + static_cast<size_t>(c) * Din + kc * 8);
    }
    while (kc < chunks) {
      const int kn = kc + 32;
      if (kn < chunks) {
#pragma unroll
        for (int c = 0; c < CW; ++c) nxt[c] = ldg_stream16(wrow + static_cast<size_t>(c) * Din + kn * 8);
      }
      float wf[CW][8];
#pragma unroll
      for (int c = 0; c < CW; ++c) unpack_bf16x8(cur[c], wf[c]);
#pragma unroll
      for (int n = 0; n < NB; ++n) {
        if (n >= N) break;
        float ef[8];
        unpack_bf16x8(s_e[n * chunks + kc], ef);
#pragma unroll
        for (int c = 0; c < CW; ++c)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[c][n] = fmaf(wf[c][i], ef[i], acc[c][n]);
      }
#pragma unroll
      for (int c = 0; c < CW; ++c) cur[c] = nxt[c];
      kc = kn;
    }
#pragma unroll
    for (int c = 0; c < CW; ++c)
#pragma unroll
      for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[c][n] += __shfl_xor_sync(0xffffffffu, acc[c][n], o);
    if (lane == 0) {
#pragma unroll
      for (int c = 0; c < CW; ++c)
#pragma unroll
        for (int n = 0; n < NB; ++n) s_res[pc + c][n] = acc[c][n];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < cpb * NB; idx += blockDim.x) {
    const int c = idx % cpb, n = idx / cpb;
    if (n >= N) continue;
    const float a = s_res[c][n];
    if (is_k) {
      const bool pre = idx == static_cast<int>(threadIdx.x);  // this (column, row) was prefetched
      const float hf = pre ? ep_h : __bfloat162float(h[(static_cast<size_t>(m_br) * N + n) * d + kc0 + c]);
      const float gg = pre ? ep_g : gamma_h[kc0 + c] * gamma_k[kc0 + c];
      s_q[0][n][c] = gg * hf * a;
      s_q[1][n][c] = a * a;
      s_q[2][n][c] = hf * hf;
    } else {
      float o = a;
      if (GATE == PG_GATE_SCALAR) o = fmaf(g, a, __bfloat162float(x[static_cast<size_t>(n) * d + c0 + c]));
      const __nv_bfloat16 ob = __float2bfloat16_rn(o);
      out[static_cast<size_t>(n) * d + c0 + c] = ob;
      if (GATE == PG_GATE_CONTEXT) {
        const float q = __bfloat162float(ob);
        s_q[3][n][c] = q * q;
      }
    }
  }
  if (GATE != PG_GATE_CONTEXT) return;
  __syncthreads();
  if (threadIdx.x < N) {
    const int n = threadIdx.x;
    const int tpb = d / kSmallTile;
    if (is_k) {
      float hk = 0.f, kk = 0.f, hh = 0.f;
      for (int c = 0; c < kSmallTile; ++c) {
        hk += s_q[0][n][c];
        kk += s_q[1][n][c];
        hh += s_q[2][n][c];
      }
      float* p = partials + (static_cast<size_t>(m_br * tpb + kc0 / kSmallTile) * 3) * N + n;
      p[0] = hk;
      p[N] = kk;
      p[2 * static_cast<size_t>(N)] = hh;
    } else if (vpart) {
      float vv = 0.f;
      for (int c = 0; c < kSmallTile; ++c) vv += s_q[3][n][c];
      vpart[static_cast<size_t>(c0 / kSmallTile) * N + n] = vv;
    }
  }
}

template <int NB>
pg_status launch_small_nb(int N, int Din, int d, int M, int gate_kind, const void* e, const void* W, float g,
                          const void* x, const void* h, const float* gamma_h, const float* gamma_k, void* out,
                          float* partials, float* vpart, cudaStream_t stream) {
  constexpr int CW = SmallCols<NB>::CW;
  const int dcols = (gate_kind == PG_GATE_CONTEXT ? 1 + M : 1) * d;
  // context: one 64-column tile of the per-row sums per block, a warp per CW columns (16
  // warps); otherwise as few columns per block as spread W over about every SM
  int warps = 16, cpb = kSmallTile;
  if (gate_kind != PG_GATE_CONTEXT) {
    const int want = dcols / (CW * sm_count());
    warps = want < 1 ? 1 : (want > 8 ? 8 : want);
    while (kSmallTile % (warps * CW)) --warps;
    cpb = warps * CW;
  }
  const unsigned blocks = static_cast<unsigned>(dcols / cpb);
  const size_t smem = static_cast<size_t>(N) * Din * sizeof(__nv_bfloat16);
  const auto* ep = static_cast<const __nv_bfloat16*>(e);
  const auto* wp = static_cast<const __nv_bfloat16*>(W);
  const auto* xp = static_cast<const __nv_bfloat16*>(x);
  const auto* hp = static_cast<const __nv_bfloat16*>(h);
  auto* op = static_cast<__nv_bfloat16*>(out);
  auto run = [&](auto kern) -> pg_status {
    // e may need more than the default 48 KB of dynamic shared memory next to the static part
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kSmallMaxE));
    if (err != cudaSuccess) return cuda_fail(err);
    kern<<<blocks, warps * 32, smem, stream>>>(ep, wp, N, Din, d, cpb, g, xp, hp, gamma_h, gamma_k, op, partials,
                                               vpart);
    return after_launch(1);
  };
  if (gate_kind == PG_GATE_CONTEXT) return run(small_rows_bf16_kernel<NB, PG_GATE_CONTEXT>);
  if (gate_kind == PG_GATE_SCALAR) return run(small_rows_bf16_kernel<NB, PG_GATE_SCALAR>);
  return run(small_rows_bf16_kernel<NB, PG_GATE_NONE>);
}

}  // namespace

pg_status launch_small_rows_bf16(int N, int Din, int d, int M, int gate_kind, const void* e, const void* W, float g,
                                 const void* x, const void* h, const float* gamma_h, const float* gamma_k, void* out,
                                 float* partials, float* vpart, cudaStream_t stream) {
  if (N < 1 || N > kSmallRows || d % kSmallTile || Din % 8) return PG_ERR_UNSUPPORTED;
  if (static_cast<size_t>(N) * Din * sizeof(__nv_bfloat16) > kSmallMaxE) return PG_ERR_UNSUPPORTED;
  if (N <= 1) return launch_small_nb<1>(N, Din, d, M, gate_kind, e, W, g, x, h, gamma_h, gamma_k, out, partials, vpart, stream);
  if (N <= 2) return launch_small_nb<2>(N, Din, d, M, gate_kind, e, W, g, x, h, gamma_h, gamma_k, out, partials, vpart, stream);
  if (N <= 4) return launch_small_nb<4>(N, Din, d, M, gate_kind, e, W, g, x, h, gamma_h, gamma_k, out, partials, vpart, stream);
  if (N <= 8) return launch_small_nb<8>(N, Din, d, M, gate_kind, e, W, g, x, h, gamma_h, gamma_k, out, partials, vpart, stream);
  return launch_small_nb<16>(N, Din, d, M, gate_kind, e, W, g, x, h, gamma_h, gamma_k, out, partials, vpart, stream);
}

namespace {

// The 8 x 8 kernel reads 16-byte chunks of rows: Din % 4 == 0 and 16-byte aligned operands.
inline bool f32_tiled_ok(int Din, const float* e, const float* W) {
  return Din % 4 == 0 && reinterpret_cast<uintptr_t>(e) % 16 == 0 && reinterpret_cast<uintptr_t>(W) % 16 == 0;
}

template <int GATE, int KS>
pg_status launch_simt_ks(int N, int Din, int d, const float* e, const float* W, float g, const float* x, float* out,
                         cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((d + kSimtTile - 1) / kSimtTile, (N + kSimtTile - 1) / kSimtTile, KS);
  cfg.blockDim = dim3(kSimtThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = KS;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool tiled = f32_tiled_ok(Din, e, W);
  if (tiled) cfg.blockDim = dim3(kF32Threads);
  const cudaError_t err =
      tiled ? cudaLaunchKernelEx(&cfg, simt_gemm_f32_tiled_kernel<GATE, KS>, e, W, N, Din, d, x, g, out)
            : cudaLaunchKernelEx(&cfg, simt_gemm_f32_kernel<GATE, KS>, e, W, N, Din, d, x, g, out);
  if (err != cudaSuccess) return cuda_fail(err);
  return after_launch(1);
}

}  // namespace

pg_status launch_simt_f32(int N, int Din, int d, int gate_kind, const float* e, const float* W, float g,
                          const float* x, float* out, cudaStream_t stream) {
  // split K over a cluster of 4 (or 2) CTAs per tile when the tiles alone leave SMs idle
  const int64_t tiles = static_cast<int64_t>((d + kSimtTile - 1) / kSimtTile) * ((N + kSimtTile - 1) / kSimtTile);
  const int64_t fill = 4ll * sm_count();
  if (f32_tiled_ok(Din, e, W)) {
    // 4 blocks per SM (registers): the largest split whose CTAs run in one wave (workload
    // 4096 x 1024 x 256: 2 -> 61 us, 4 -> 64 us)
    if (Din >= 4 * 2 * kSimtK && tiles * 4 <= fill)
      return gate_kind == PG_GATE_SCALAR ? launch_simt_ks<PG_GATE_SCALAR, 4>(N, Din, d, e, W, g, x, out, stream)
                                         : launch_simt_ks<PG_GATE_NONE, 4>(N, Din, d, e, W, g, x, out, stream);
    if (Din >= 2 * 2 * kSimtK && tiles * 2 <= fill)
      return gate_kind == PG_GATE_SCALAR ? launch_simt_ks<PG_GATE_SCALAR, 2>(N, Din, d, e, W, g, x, out, stream)
                                         : launch_simt_ks<PG_GATE_NONE, 2>(N, Din, d, e, W, g, x, out, stream);
  } else if (Din >= 4 * 2 * kSimtK && tiles * 2 < fill)
    return gate_kind == PG_GATE_SCALAR ? launch_simt_ks<PG_GATE_SCALAR, 4>(N, Din, d, e, W, g, x, out, stream)
                                       : launch_simt_ks<PG_GATE_NONE, 4>(N, Din, d, e, W, g, x, out, stream);
  else if (Din >= 2 * 2 * kSimtK && tiles < fill)
    return gate_kind == PG_GATE_SCALAR ? launch_simt_ks<PG_GATE_SCALAR, 2>(N, Din, d, e, W, g, x, out, stream)
                                       : launch_simt_ks<PG_GATE_NONE, 2>(N, Din, d, e, W, g, x, out, stream);
  dim3 grid((d + kSimtTile - 1) / kSimtTile, (N + kSimtTile - 1) / kSimtTile);
  if (f32_tiled_ok(Din, e, W)) {
    if (gate_kind == PG_GATE_SCALAR)
      simt_gemm_f32_tiled_kernel<PG_GATE_SCALAR, 1><<<grid, kF32Threads, 0, stream>>>(e, W, N, Din, d, x, g, out);
    else
      simt_gemm_f32_tiled_kernel<PG_GATE_NONE, 1><<<grid, kF32Threads, 0, stream>>>(e, W, N, Din, d, x, g, out);
  } else if (gate_kind == PG_GATE_SCALAR) {
    simt_gemm_f32_kernel<PG_GATE_SCALAR, 1><<<grid, kSimtThreads, 0, stream>>>(e, W, N, Din, d, x, g, out);
  } else {
    simt_gemm_f32_kernel<PG_GATE_NONE, 1><<<grid, kSimtThreads, 0, stream>>>(e, W, N, Din, d, x, g, out);
  }
  return after_launch(1);
}

pg_status launch_identity_gate(int64_t n, int dtype, int gate_kind, const void* e, const void* x, float g,
                               void* out, cudaStream_t stream) {
  const int64_t want = (n / 8 + 255) / 256;
  const int blocks = static_cast<int>(want < sm_count() * 8ll ? want : sm_count() * 8ll);
  if (dtype == PG_BF16) {
    auto* eb = static_cast<const __nv_bfloat16*>(e);
    auto* xb = static_cast<const __nv_bfloat16*>(x);
    auto* ob = static_cast<__nv_bfloat16*>(out);
    if (gate_kind == PG_GATE_SCALAR)
      identity_gate_kernel<__nv_bfloat16, PG_GATE_SCALAR><<<blocks, 256, 0, stream>>>(eb, xb, g, ob, n);
    else
      identity_gate_kernel<__nv_bfloat16, PG_GATE_NONE><<<blocks, 256, 0, stream>>>(eb, xb, g, ob, n);
  } else {
    auto* ef = static_cast<const float*>(e);
    auto* xf = static_cast<const float*>(x);
    auto* of = static_cast<float*>(out);
    if (gate_kind == PG_GATE_SCALAR)
      identity_gate_kernel<float, PG_GATE_SCALAR><<<blocks, 256, 0, stream>>>(ef, xf, g, of, n);
    else
      identity_gate_kernel<float, PG_GATE_NONE><<<blocks, 256, 0, stream>>>(ef, xf, g, of, n);
  }
  return after_launch(1);
}

}  // namespace pg
