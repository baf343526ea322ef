// Causal depthwise conv + SiLU + residual into the branch states (sm_103a).
//
// Engram notes (arXiv 2601.07372) section 3.3: Y = SiLU(Conv1D(RMSNorm(V~))) + V~ with
// kernel 4 and dilation = max n-gram order; section 3.4: V~ = alpha^(m) v per branch;
// section 3.1: H^(m) <- H^(m) + Y. The explainer's "一次 lookup 经过哪些步骤？" requires
// the conv to be causal.
//
// Since u = alpha v, RMSNorm(u) = f v gamma with the per-(branch, position) scalar
// f = alpha / sqrt(alpha^2 mean(v^2) + eps). A block owns runs of kRun positions of one
// sequence (persistent grid) and d/CPT threads, thread i owning channels [CPT i, CPT i + CPT)
// (CPT = 4 up to d = 3072, else 8):
//   1. one warp per position reduces sum(v^2) over the run and its causal halo;
//   2. f and alpha per (branch, position) go to shared memory;
//   3. every thread walks its positions by residue class mod dil (so the 4 taps form a
//      window sliding one row per step): c = sum_j f_{t-j dil} (w[:, j] gamma) v_{t-j dil},
//      H[m, t] += SiLU(c) + alpha_t v_t for all M branches, in packed fp32x2 arithmetic,
//      with H of the next positions prefetched into shared memory by cp.async.
// DRAM traffic per token: v once (2d bytes; the taps re-read it from L1/L2) and H read +
// written once per branch (2 * M * 2d bytes).
#include <cuda_bf16.h>

#include <type_traits>

#include "pg_internal.cuh"

namespace pg {
namespace {

constexpr int kRun = 32;        // positions per run
constexpr int kMaxHalo = 24;    // (kernel_size - 1) * dilation <= 3 * 8
constexpr int kMaxBranches = 8;
constexpr int kMaxPos = kRun + kMaxHalo;
constexpr int kTaps = 4;

// CPT consecutive channels of one row: load / unpack to fp32 / pack and store.
template <typename T, int CPT>
struct VecN;

template <>
struct VecN<__nv_bfloat16, 8> {
  using Raw = uint4;
  static __device__ __forceinline__ Raw zero() { return make_uint4(0, 0, 0, 0); }
  static __device__ __forceinline__ Raw load(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
  }
  static __device__ __forceinline__ void unpack(const Raw& w, float* f) {
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
struct VecN<__nv_bfloat16, 4> {
  using Raw = uint2;
  static __device__ __forceinline__ Raw zero() { return make_uint2(0, 0); }
  static __device__ __forceinline__ Raw load(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const uint2*>(p));
  }
  static __device__ __forceinline__ void unpack(const Raw& w, float* f) {
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* f) {
    __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]), b = __floats2bfloat162_rn(f[2], f[3]);
    *reinterpret_cast<uint2*>(p) = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
};

template <>
struct VecN<float, 8> {
  struct Raw {
    float4 a, b;
  };
  static __device__ __forceinline__ Raw zero() { return Raw{make_float4(0, 0, 0, 0), make_float4(0, 0, 0, 0)}; }
  static __device__ __forceinline__ Raw load(const float* p) {
    return Raw{__ldg(reinterpret_cast<const float4*>(p)), __ldg(reinterpret_cast<const float4*>(p + 4))};
  }
  static __device__ __forceinline__ void unpack(const Raw& r, float* f) {
    f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
    f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
  }
  static __device__ __forceinline__ void store(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
};

template <>
struct VecN<float, 4> {
  using Raw = float4;
  static __device__ __forceinline__ Raw zero() { return make_float4(0, 0, 0, 0); }
  static __device__ __forceinline__ Raw load(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
  static __device__ __forceinline__ void unpack(const Raw& r, float* f) {
    f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
  }
  static __device__ __forceinline__ void store(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

// Asynchronous 16-byte global -> shared copies of one thread (L1 bypassed); a thread
// waits only for its own copies, so no block-wide barrier is involved.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
// One thread's asynchronous copy of BYTES (8, 16 or 32) contiguous bytes.
template <int BYTES>
__device__ __forceinline__ void cp_async_bytes(void* smem, const void* gmem) {
  if constexpr (BYTES == 8) {
    cp_async8(smem, gmem);
  } else {
#pragma unroll
    for (int k = 0; k < BYTES / 16; ++k)
      cp_async16(static_cast<uint8_t*>(smem) + 16 * k, static_cast<const uint8_t*>(gmem) + 16 * k);
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Packed pairs of fp32 (Blackwell f32x2 arithmetic: two lanes per instruction).
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// SiLU(c) = c * sigmoid(c) with sigmoid(c) = (1 + tanh(c/2)) / 2 (one MUFU operation per
// element), on a packed pair.
__device__ __forceinline__ uint64_t silu2(uint64_t c) {
  float c0, c1, t0, t1;
  upk(mul2(c, pk(0.5f, 0.5f)), c0, c1);
  asm("tanh.approx.f32 %0, %1;" : "=f"(t0) : "f"(c0));
  asm("tanh.approx.f32 %0, %1;" : "=f"(t1) : "f"(c1));
  return mul2(c, fma2(pk(0.5f, 0.5f), pk(t0, t1), pk(0.5f, 0.5f)));
}

// PF: positions of H prefetched ahead of the one being computed (per thread, cp.async);
// CPT: channels per thread (4 gives twice the warps of 8 at half the registers each).
template <typename T, int MB, int PF, int CPT>
__global__ void __launch_bounds__(CPT == 4 ? 768 : 1024) conv_residual_kernel(
    int L, int d, int M_rt, int64_t N, const T* __restrict__ v, const float* __restrict__ alpha,
    const float* __restrict__ v_ms,
    const float* __restrict__ gamma_c, const float* __restrict__ conv_w, int ks, int dil, float eps,
    T* __restrict__ H, int runs_per_seq, int total_runs) {
  constexpr int MMAX = MB > 0 ? MB : kMaxBranches;
  const int M = MB > 0 ? MB : M_rt;
  __shared__ float s_ms[kMaxPos];  // sum(v^2) per position of the run
  __shared__ float s_f[MMAX][kMaxPos];
  __shared__ float s_a[MMAX][kMaxPos];
  // H prefetch ring: [PF][M][threads] chunks of CPT channels
  extern __shared__ __align__(16) uint8_t s_ring[];
  using Vec = VecN<T, CPT>;
  using Raw = typename Vec::Raw;
  Raw* ring = reinterpret_cast<Raw*>(s_ring);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  auto ring_at = [&](int slot, int m) -> Raw* { return ring + (slot * MMAX + m) * blockDim.x + threadIdx.x; };

  const int c0 = threadIdx.x * CPT;
  const bool active = c0 < d;
  const int chunks8 = d >> 3;
  const int halo = (ks - 1) * dil;
  const float inv_d = 1.0f / static_cast<float>(d);

  // conv taps with the RMSNorm gain folded in: wg[j][q] = w[c0+q, j] * gamma[c0+q]
  float wg[kTaps][CPT];
#pragma unroll
  for (int q = 0; q < CPT; ++q) {
    const float g = active ? gamma_c[c0 + q] : 0.f;
#pragma unroll
    for (int j = 0; j < kTaps; ++j) wg[j][q] = (active && j < ks) ? conv_w[(c0 + q) * ks + j] * g : 0.f;
  }

  for (int run = blockIdx.x; run < total_runs; run += gridDim.x) {
    const int b = run / runs_per_seq;
    const int t0 = (run - b * runs_per_seq) * kRun;
    const int t1 = min(t0 + kRun, L);
    const int p0 = max(0, t0 - halo);
    const int npos = t1 - p0;
    const int64_t seq0 = static_cast<int64_t>(b) * L;

    // 1. sum(v^2) per position: given (v_ms, the projection's mean(v^2)), or one warp per
    //    position (16-byte loads, unrolled so each lane has several of its row's loads in
    //    flight)
    if (v_ms)
      for (int i = threadIdx.x; i < npos; i += blockDim.x) s_ms[i] = v_ms[seq0 + p0 + i] * static_cast<float>(d);
    for (int i = warp; !v_ms && i < npos; i += nwarps) {
      const T* row = v + (seq0 + p0 + i) * d;
      float s = 0.f;
#pragma unroll 4
      for (int q = lane; q < chunks8; q += 32) {
        float x[8];
        VecN<T, 8>::unpack(VecN<T, 8>::load(row + 8 * q), x);
#pragma unroll
        for (int k = 0; k < 8; ++k) s = fmaf(x[k], x[k], s);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane == 0) s_ms[i] = s;
    }
    __syncthreads();

    // 2. alpha and f = alpha / sqrt(alpha^2 mean(v^2) + eps) per (branch, position)
    for (int idx = threadIdx.x; idx < M * npos; idx += blockDim.x) {
      const int m = idx / npos, i = idx - (idx / npos) * npos;
      const float a = alpha[m * N + seq0 + p0 + i];
      s_a[m][i] = a;
      s_f[m][i] = a * rsqrtf(a * a * (s_ms[i] * inv_d) + eps);
    }
    __syncthreads();

    // 3. conv + SiLU + residual. Positions are walked by residue class mod dil, so the taps
    //    of t (t, t - dil, t - 2 dil, t - 3 dil) form a window that slides by one row per
    //    step; H of the next PF positions in walking order is already on its way into this
    //    thread's ring slots (one cp.async group per position).
    int pr = 0, pi = 0, ps = 0;  // prefetch cursor: position t0 + pr + dil * pi, sequence ps
    auto prefetch_next = [&]() {
      if (pr < dil && t0 + pr < t1) {
        if (active) {
          const int t = t0 + pr + dil * pi;
          const int slot = ps % PF;
#pragma unroll
          for (int m = 0; m < MMAX; ++m) {
            if (m >= M) continue;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(H + (m * N + seq0 + t) * d + c0);
            uint8_t* dst = reinterpret_cast<uint8_t*>(ring_at(slot, m));
            cp_async_bytes<static_cast<int>(sizeof(Raw))>(dst, src);
          }
        }
        ++pi;
        if (t0 + pr + dil * pi >= t1) {
          ++pr;
          pi = 0;
        }
      }
      cp_async_commit();
      ++ps;
    };
#pragma unroll 1
    for (int i = 0; i < PF; ++i) prefetch_next();
    int s = 0;  // sequence index of the position being computed
    for (int r = 0; r < dil && t0 + r < t1; ++r) {
      float win[kTaps][CPT];  // v at t - j dil, zero before the start of the sequence
#pragma unroll
      for (int j = 0; j < kTaps; ++j) {
        const int p = t0 + r - j * dil;
        if (active && j < ks && p >= 0) {
          Vec::unpack(Vec::load(v + (seq0 + p) * d + c0), win[j]);
        } else {
#pragma unroll
          for (int q = 0; q < CPT; ++q) win[j][q] = 0.f;
        }
      }
      for (int t = t0 + r; t < t1; t += dil, ++s) {
        const bool has_next = active && t + dil < t1;
        Raw nxt = Vec::zero();
        if (has_next) nxt = Vec::load(v + (seq0 + t + dil) * d + c0);   // next window row, early
        cp_async_wait<PF - 1>();   // this thread's copies for position t have landed
        if (active) {
          const int slot = s % PF;
          constexpr int kPairs = CPT / 2;
          uint64_t prod[kTaps][kPairs];   // (w[:, j] gamma) * v_{t - j dil}, packed pairs
#pragma unroll
          for (int j = 0; j < kTaps; ++j)
#pragma unroll
            for (int q = 0; q < kPairs; ++q)
              prod[j][q] = mul2(pk(wg[j][2 * q], wg[j][2 * q + 1]), pk(win[j][2 * q], win[j][2 * q + 1]));
          uint64_t vt[kPairs];
#pragma unroll
          for (int q = 0; q < kPairs; ++q) vt[q] = pk(win[0][2 * q], win[0][2 * q + 1]);
#pragma unroll
          for (int m = 0; m < MMAX; ++m) {
            if (m >= M) continue;
            uint64_t fj[kTaps];
#pragma unroll
            for (int j = 0; j < kTaps; ++j) {
              const int p = t - j * dil;
              const float f = (j < ks && p >= 0) ? s_f[m][p - p0] : 0.f;
              fj[j] = pk(f, f);
            }
            const float a = s_a[m][t - p0];
            const uint64_t aa = pk(a, a);
            float h[CPT];
            Vec::unpack(*ring_at(slot, m), h);
#pragma unroll
            for (int q = 0; q < kPairs; ++q) {
              uint64_t c = mul2(fj[0], prod[0][q]);
#pragma unroll
              for (int j = 1; j < kTaps; ++j) c = fma2(fj[j], prod[j][q], c);
              const uint64_t y = fma2(aa, vt[q], silu2(c));           // SiLU(c) + alpha v_t
              upk(add2(pk(h[2 * q], h[2 * q + 1]), y), h[2 * q], h[2 * q + 1]);
            }
            Vec::store(H + (m * N + seq0 + t) * d + c0, h);
          }
        }
        prefetch_next();
        // slide the window by one row (t -> t + dil)
#pragma unroll
        for (int j = kTaps - 1; j > 0; --j)
#pragma unroll
          for (int q = 0; q < CPT; ++q) win[j][q] = win[j - 1][q];
        Vec::unpack(nxt, win[0]);
      }
    }
    cp_async_wait<0>();
    __syncthreads();
  }
}

template <typename T>
pg_status launch(int B, int L, int d, int M, const void* v, const float* alpha, const float* v_ms,
                 const float* gamma_c, const float* conv_w, int ks, int dil, float eps, void* H, cudaStream_t stream) {
  // 4 channels per thread up to d = 3072 (768 threads), else 8 (up to 1024 threads)
  const int cpt = d / 4 <= 768 ? 4 : 8;
  const int threads = ((d / cpt) + 31) / 32 * 32;
  const int runs_per_seq = (L + kRun - 1) / kRun;
  const int64_t total = static_cast<int64_t>(B) * runs_per_seq;
  if (total >= (1ll << 31)) return PG_ERR_SHAPE;
  const int64_t N = static_cast<int64_t>(B) * L;
  auto run = [&](auto kern, int mmax, int pf) -> pg_status {
    const size_t ring = static_cast<size_t>(pf) * mmax * threads * (sizeof(T) * cpt);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ring));
    if (e != cudaSuccess) return cuda_fail(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, ring);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm < 1) return PG_ERR_UNSUPPORTED;
    const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
    const int grid = static_cast<int>(total < cap ? total : cap);
    kern<<<grid, threads, ring, stream>>>(L, d, M, N, static_cast<const T*>(v), alpha, v_ms, gamma_c, conv_w, ks,
                                          dil, eps, static_cast<T*>(H), runs_per_seq, static_cast<int>(total));
    return after_launch(1);
  };
  // prefetch depth: 4 positions while the ring fits in 192 KB of shared memory, else 1
  const int mm = M == 1 || M == 2 || M == 4 ? M : kMaxBranches;
  const bool deep = 4ull * mm * threads * sizeof(T) * cpt <= (192u << 10);
  auto pick = [&](auto cpt_c) -> pg_status {
    constexpr int C = decltype(cpt_c)::value;
    switch (M) {
      case 1: return deep ? run(conv_residual_kernel<T, 1, 4, C>, 1, 4) : run(conv_residual_kernel<T, 1, 1, C>, 1, 1);
      case 2: return deep ? run(conv_residual_kernel<T, 2, 4, C>, 2, 4) : run(conv_residual_kernel<T, 2, 1, C>, 2, 1);
      case 4: return deep ? run(conv_residual_kernel<T, 4, 4, C>, 4, 4) : run(conv_residual_kernel<T, 4, 1, C>, 4, 1);
      default:
        return deep ? run(conv_residual_kernel<T, 0, 4, C>, kMaxBranches, 4)
                    : run(conv_residual_kernel<T, 0, 1, C>, kMaxBranches, 1);
    }
  };
  return cpt == 4 ? pick(std::integral_constant<int, 4>()) : pick(std::integral_constant<int, 8>());
}

}  // namespace
}  // namespace pg

extern "C" pg_status pg_conv_residual(int32_t B, int32_t L, int32_t d, int32_t M, int32_t dtype,
                                      const void* v, const float* alpha, const float* v_ms, const float* gamma_c,
                                      const float* conv_w, int32_t kernel_size, int32_t dilation,
                                      float eps, void* H, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B < 0 || L < 0 || d < 8 || d % 8 || d > 8192 || M < 1 || M > kMaxBranches) return PG_ERR_SHAPE;
  if (kernel_size < 1 || kernel_size > kTaps || dilation < 1 || dilation > 8) return PG_ERR_SHAPE;
  if (dtype != PG_BF16 && dtype != PG_F32) return PG_ERR_DTYPE;
  if (static_cast<int64_t>(B) * L == 0) return PG_OK;
  if (static_cast<int64_t>(B) * L >= (1ll << 31)) return PG_ERR_SHAPE;
  if (!v || !alpha || !gamma_c || !conv_w || !H) return PG_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(H)) & 15u) return PG_ERR_ALIGN;
  if (sm_count() == 0) return cuda_fail(cudaGetLastError());
  if (dtype == PG_BF16)
    return launch<__nv_bfloat16>(B, L, d, M, v, alpha, v_ms, gamma_c, conv_w, kernel_size, dilation, eps, H,
                                 stream);
  return launch<float>(B, L, d, M, v, alpha, v_ms, gamma_c, conv_w, kernel_size, dilation, eps, H, stream);
}
