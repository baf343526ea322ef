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

// out[N, Dout] = A[N, Din] B[Dout, Din]^T (+ gate). 128 threads, thread (ty, tx) owns rows
// ty*8 .. ty*8+7 and columns tx*4 .. tx*4+3 of the 64 x 64 tile (8 x 4 fp32 accumulators);
// per k step it reads 8 A values and 4 B values from shared memory (3 vector loads for 32
// FMAs). 32-deep k-tiles are double-buffered: the next tile's global loads are in registers while
// the current one is multiplied. Out-of-range rows, columns and k read as zero.
template <int GATE>
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
  const bool vec = (Din & 3) == 0;
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
  load_tile(0);
  store_tile(0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < Din; k0 += kSimtK) {
    const bool more = k0 + kSimtK < Din;
    if (more) load_tile(k0 + kSimtK);
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

}  // namespace

pg_status launch_simt_f32(int N, int Din, int d, int gate_kind, const float* e, const float* W, float g,
                          const float* x, float* out, cudaStream_t stream) {
  dim3 grid((d + kSimtTile - 1) / kSimtTile, (N + kSimtTile - 1) / kSimtTile);
  if (gate_kind == PG_GATE_SCALAR)
    simt_gemm_f32_kernel<PG_GATE_SCALAR><<<grid, kSimtThreads, 0, stream>>>(e, W, N, Din, d, x, g, out);
  else
    simt_gemm_f32_kernel<PG_GATE_NONE><<<grid, kSimtThreads, 0, stream>>>(e, W, N, Din, d, x, g, out);
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
