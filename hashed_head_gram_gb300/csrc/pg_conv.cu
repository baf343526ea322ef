// Causal depthwise conv + SiLU + residual into the branch states (sm_103a).
//
// Engram notes (arXiv 2601.07372) section 3.3: Y = SiLU(Conv1D(RMSNorm(V~))) + V~ with
// kernel 4 and dilation = max n-gram order; section 3.4: V~ = alpha^(m) v per branch;
// section 3.1: H^(m) <- H^(m) + Y. The explainer's "一次 lookup 经过哪些步骤？" requires
// the conv to be causal.
//
// One block per (sequence, run of kRun positions), d/8 threads: thread i owns channels
// [8i, 8i+8). Since u = alpha v, RMSNorm(u) = f v gamma with the per-(branch, position)
// scalar f = alpha / sqrt(alpha^2 mean(v^2) + eps), so the block first reduces sum(v^2)
// for its positions and their causal halo, then every thread walks its positions:
// c = sum_j w[:, j] f_{t-j dil} gamma v_{t-j dil};  H += SiLU(c) + alpha_t v_t.
#include <cuda_bf16.h>

#include "pg_internal.cuh"

namespace pg {
namespace {

constexpr int kRun = 16;        // positions per block
constexpr int kMaxHalo = 24;    // (kernel_size - 1) * dilation <= 3 * 8
constexpr int kMaxBranches = 8;
constexpr int kMaxPos = kRun + kMaxHalo;

template <typename T>
struct Vec8;

template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* f) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
    f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xFFFF0000u);
    f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xFFFF0000u);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 v = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const float* p, float* f) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
  static __device__ __forceinline__ void store(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
};

template <typename T>
__global__ void __launch_bounds__(1024) conv_residual_kernel(
    int B, int L, int d, int M, const T* __restrict__ v, const float* __restrict__ alpha,
    const float* __restrict__ gamma_c, const float* __restrict__ conv_w, int ks, int dil, float eps,
    T* __restrict__ H) {
  __shared__ float s_red[kMaxPos][32];
  __shared__ float s_f[kMaxBranches][kMaxPos];
  __shared__ float s_a[kMaxBranches][kMaxPos];

  const int runs = (L + kRun - 1) / kRun;
  const int b = blockIdx.x / runs;
  const int t0 = (blockIdx.x - b * runs) * kRun;
  const int t1 = min(t0 + kRun, L);
  const int halo = (ks - 1) * dil;
  const int p0 = max(0, t0 - halo);
  const int npos = t1 - p0;
  const int c0 = threadIdx.x * 8;
  const bool active = c0 < d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = (blockDim.x + 31) >> 5;
  const int64_t seq0 = static_cast<int64_t>(b) * L;
  const int64_t N = static_cast<int64_t>(B) * L;

  // ---- sum(v^2) per position (positions p0 .. t1-1)
  for (int i = 0; i < npos; ++i) {
    float s = 0.f;
    if (active) {
      float x[8];
      Vec8<T>::load(v + (seq0 + p0 + i) * d + c0, x);
#pragma unroll
      for (int q = 0; q < 8; ++q) s = fmaf(x[q], x[q], s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) s_red[i][warp] = s;
  }
  __syncthreads();
  const float inv_d = 1.0f / static_cast<float>(d);
  for (int idx = threadIdx.x; idx < M * npos; idx += blockDim.x) {
    const int m = idx / npos, i = idx - (idx / npos) * npos;
    float ms = 0.f;
    for (int w = 0; w < nwarps; ++w) ms += s_red[i][w];
    ms *= inv_d;
    const float a = alpha[static_cast<int64_t>(m) * N + seq0 + p0 + i];
    s_a[m][i] = a;
    s_f[m][i] = a / sqrtf(a * a * ms + eps);
  }
  __syncthreads();
  if (!active) return;

  float gam[8], w[4][8];
  {
    const float4 g0 = *reinterpret_cast<const float4*>(gamma_c + c0);
    const float4 g1 = *reinterpret_cast<const float4*>(gamma_c + c0 + 4);
    gam[0] = g0.x; gam[1] = g0.y; gam[2] = g0.z; gam[3] = g0.w;
    gam[4] = g1.x; gam[5] = g1.y; gam[6] = g1.z; gam[7] = g1.w;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < 8; ++q) w[j][q] = j < ks ? conv_w[(c0 + q) * ks + j] : 0.f;
  }

  for (int t = t0; t < t1; ++t) {
    float vt[4][8];  // v at t - j*dil (zeros before the start of the sequence)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int p = t - j * dil;
      if (j < ks && p >= 0) {
        Vec8<T>::load(v + (seq0 + p) * d + c0, vt[j]);
#pragma unroll
        for (int q = 0; q < 8; ++q) vt[j][q] *= gam[q];
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) vt[j][q] = 0.f;
      }
    }
    float vraw[8];
    Vec8<T>::load(v + (seq0 + t) * d + c0, vraw);
    for (int m = 0; m < M; ++m) {
      float conv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) conv[q] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = t - j * dil;
        if (j < ks && p >= 0) {
          const float f = s_f[m][p - p0];
#pragma unroll
          for (int q = 0; q < 8; ++q) conv[q] = fmaf(w[j][q] * f, vt[j][q], conv[q]);
        }
      }
      const float a = s_a[m][t - p0];
      T* hp = H + (static_cast<int64_t>(m) * N + seq0 + t) * d + c0;
      float hv[8];
      Vec8<T>::load(hp, hv);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float c = conv[q];
        const float silu = c / (1.0f + __expf(-c));
        hv[q] = hv[q] + (silu + a * vraw[q]);
      }
      Vec8<T>::store(hp, hv);
    }
  }
}

}  // namespace
}  // namespace pg

extern "C" pg_status pg_conv_residual(int32_t B, int32_t L, int32_t d, int32_t M, int32_t dtype,
                                      const void* v, const float* alpha, const float* gamma_c,
                                      const float* conv_w, int32_t kernel_size, int32_t dilation,
                                      float eps, void* H, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B < 0 || L < 0 || d < 8 || d % 8 || d > 8192 || M < 1 || M > kMaxBranches) return PG_ERR_SHAPE;
  if (kernel_size < 1 || kernel_size > 4 || dilation < 1 || dilation > 8) return PG_ERR_SHAPE;
  if (dtype != PG_BF16 && dtype != PG_F32) return PG_ERR_DTYPE;
  if (static_cast<int64_t>(B) * L == 0) return PG_OK;
  if (static_cast<int64_t>(B) * L >= (1ll << 31)) return PG_ERR_SHAPE;
  if (!v || !alpha || !gamma_c || !conv_w || !H) return PG_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(H) |
       reinterpret_cast<uintptr_t>(gamma_c)) & 15u)
    return PG_ERR_ALIGN;
  const int threads = ((d / 8) + 31) / 32 * 32;
  const int runs = (L + kRun - 1) / kRun;
  const int64_t blocks = static_cast<int64_t>(B) * runs;
  if (blocks >= (1ll << 31)) return PG_ERR_SHAPE;
  if (dtype == PG_BF16)
    conv_residual_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        B, L, d, M, static_cast<const __nv_bfloat16*>(v), alpha, gamma_c, conv_w, kernel_size, dilation,
        eps, static_cast<__nv_bfloat16*>(H));
  else
    conv_residual_kernel<float><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        B, L, d, M, static_cast<const float*>(v), alpha, gamma_c, conv_w, kernel_size, dilation, eps,
        static_cast<float*>(H));
  return after_launch(1);
}
