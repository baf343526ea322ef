// FP8 operands of the fused W_V + M W_K projection (sm_103a).
//
// Engram notes section 3.4: the fused projection of the table output and the per-branch
// keys runs in FP8. Each row x (a token's e_t, or an output channel of W) is stored as OCP
// E4M3 codes q_i = E4M3(x_i / s) with one fp32 scale s = max |x| / 448 per row (the
// largest element lands on +-448); the conversion rounds to nearest, ties to even, and
// saturates at +-448 (cvt.rn.satfinite); s = 0 stores zeros. pg_project_gate_fp8 then
// computes out[t, c] = s_e[t] s_w[c] sum_k q_e[t, k] q_w[c, k] on the tensor cores.
//
// One warp per row: pass 1 reduces max |x| over the row (16-byte loads, 8 elements per
// lane and step), pass 2 re-reads the row (from L1 / L2), divides (correctly rounded fp32)
// and converts, 8 codes per lane and step (one 8-byte store).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "pg_internal.cuh"

namespace pg {
namespace {

template <typename T>
struct Row8;

template <>
struct Row8<float> {
  static __device__ __forceinline__ void load(const float* p, float (&f)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

template <>
struct Row8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&f)[8]) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
    f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xFFFF0000u);
    f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xFFFF0000u);
  }
};

template <typename T>
__global__ void __launch_bounds__(256) fp8_quantize_kernel(const T* __restrict__ x, int64_t rows, int64_t cols,
                                                           uint8_t* __restrict__ q, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t first = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t chunks = cols / 8;
  for (int64_t row = first; row < rows; row += nwarps) {
    const T* xr = x + row * cols;
    float a = 0.0f;
    for (int64_t c = lane; c < chunks; c += 32) {
      float f[8];
      Row8<T>::load(xr + 8 * c, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    const float s = __fdiv_rn(a, 448.0f);
    if (lane == 0) scale[row] = s;
    uint8_t* qr = q + row * cols;
    for (int64_t c = lane; c < chunks; c += 32) {
      float f[8];
      Row8<T>::load(xr + 8 * c, f);
      uint32_t w[2] = {0u, 0u};
      if (s != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t b = __nv_cvt_float_to_fp8(__fdiv_rn(f[i], s), __NV_SATFINITE, __NV_E4M3);
          w[i / 4] |= b << (8 * (i % 4));
        }
      }
      *reinterpret_cast<uint2*>(qr + 8 * c) = make_uint2(w[0], w[1]);
    }
  }
}

}  // namespace
}  // namespace pg

extern "C" pg_status pg_fp8_quantize(const void* x, int32_t dtype, int64_t rows, int64_t cols, void* q,
                                     float* scale, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (rows < 0 || cols < 1) return PG_ERR_SHAPE;
  if (dtype != PG_F32 && dtype != PG_BF16) return PG_ERR_DTYPE;
  if (cols % 8) return PG_ERR_UNSUPPORTED;
  if (rows == 0) return PG_OK;
  if (!x || !q || !scale) return PG_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(q)) & 15u ||
      reinterpret_cast<uintptr_t>(scale) % 4)
    return PG_ERR_ALIGN;
  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  const int64_t want = (rows + 7) / 8;  // 8 rows (warps) per block
  const int64_t cap = static_cast<int64_t>(nsm) * 8;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  if (dtype == PG_F32)
    fp8_quantize_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<const float*>(x), rows, cols,
                                                          static_cast<uint8_t*>(q), scale);
  else
    fp8_quantize_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), rows,
                                                                  cols, static_cast<uint8_t*>(q), scale);
  return after_launch(1);
}
