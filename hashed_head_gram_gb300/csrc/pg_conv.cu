// Causal depthwise conv + SiLU + residual into the branch states (sm_103a).
//
// Engram notes (arXiv 2601.07372) section 3.3: Y = SiLU(Conv1D(RMSNorm(V~))) + V~ with
// kernel 4 and dilation = max n-gram order; section 3.4: V~ = alpha^(m) v per branch;
// section 3.1: H^(m) <- H^(m) + Y. The explainer's "一次 lookup 经过哪些步骤？" requires
// the conv to be causal.
//
// Since u = alpha v, RMSNorm(u) = f v gamma with the per-(branch, position) scalar
// f = alpha / sqrt(alpha^2 mean(v^2) + eps). A block owns one channel slice of runs of kRun
// positions of one sequence (persistent grid), thread i owning channels [4 i, 4 i + 4) of the
// slice. Slices are 512 channels (4 warps; six blocks fill an SM's 24 warp slots at 80
// registers) when mean(v^2) is handed over, else up to 3072 (every block then reads whole
// rows for its sums, so fewer and wider slices):
//   1. mean(v^2) per position of the run and its causal halo: handed over by the caller
//      (the projection's epilogue has it), else one warp per position reduces it;
//   2. per (branch, position) the four tap scalars f_{t - j dil} and alpha_t go to shared
//      memory as duplicated pairs, so one thread reads all of them with three vector loads;
//   3. every thread walks its positions by residue class mod dil (so the 4 taps form a
//      window of rows that rotates by one row per step, held in registers under a 4-way
//      unrolled walk), c = sum_j f_{t-j dil} (w[:, j] gamma) v_{t-j dil},
//      H[m, t] += SiLU(c) + alpha_t v_t for all M branches, in packed fp32x2 arithmetic,
//      with H and v of the next positions prefetched into shared memory by cp.async.
// DRAM traffic per token: v once (2d bytes; the taps re-read it from L1/L2) and H read +
// written once per branch (2 * M * 2d bytes).
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include "pg_conv_math.cuh"
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
  // coherent load, for memory the same kernel also writes
  static __device__ __forceinline__ Raw load_rw(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }
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
  static __device__ __forceinline__ Raw load_rw(const float* p) { return *reinterpret_cast<const float4*>(p); }
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

// mean(v^2) of one d-wide row by one warp: lane l sums the squares of 8-element groups
// l, l + 32, ... in order (one FMA each), then the lanes' sums are added in an xor tree.
template <typename T>
__device__ __forceinline__ float row_mean_square(const T* __restrict__ row, int chunks8, float inv_d, int lane) {
  float s = 0.f;
#pragma unroll 4
  for (int q = lane; q < chunks8; q += 32) {
    float x[8];
    VecN<T, 8>::unpack(VecN<T, 8>::load(row + 8 * q), x);
#pragma unroll
    for (int k = 0; k < 8; ++k) s = __fmaf_rn(x[k], x[k], s);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
  return __fmul_rn(s, inv_d);
}

constexpr int kCpt = 4;             // channels per thread
constexpr int kMaxThreads = 768;    // so a slice holds at most 3072 channels
constexpr int kSliceThreads = 128;  // slice width when mean(v^2) is given
constexpr int kPrefetch = 2;        // positions of H and v in flight per thread

// PF: positions of H prefetched ahead of the one being computed (per thread, cp.async).
// The grid is a multiple of `slices`; block b works on channel slice b mod slices.
template <typename T, int MB, int PF>
__global__ void __launch_bounds__(kMaxThreads) conv_residual_kernel(
    int L, int d, int M_rt, int64_t N, const T* __restrict__ v, const float* __restrict__ alpha,
    const float* __restrict__ v_ms,
    const float* __restrict__ gamma_c, const float* __restrict__ conv_w, int ks, int dil, float eps,
    T* __restrict__ H, int runs_per_seq, int total_runs, int slices) {
  constexpr int MMAX = MB > 0 ? MB : kMaxBranches;
  constexpr int CPT = kCpt;
  const int M = MB > 0 ? MB : M_rt;
  __shared__ float s_ms[kMaxPos];  // mean(v^2) per position of the run and its halo
  // per (branch, run position t): {f_t, f_t, f_{t-dil}, f_{t-dil}}, {f_{t-2dil} x2, f_{t-3dil} x2},
  // {alpha_t, alpha_t, -, -}; f is 0 before the start of the sequence and past the kernel size
  __shared__ __align__(16) float s_tap[MMAX][kRun][12];
  // operand ring: [PF][MMAX + 1][threads] chunks of CPT channels (H of each branch, then v)
  extern __shared__ __align__(16) uint8_t s_ring[];
  using Vec = VecN<T, CPT>;
  using Raw = typename Vec::Raw;
  constexpr int kPairs = CPT / 2;
  Raw* ring = reinterpret_cast<Raw*>(s_ring);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  auto ring_at = [&](int slot, int m) -> Raw* { return ring + (slot * (MMAX + 1) + m) * blockDim.x + threadIdx.x; };

  const int c0 = (blockIdx.x % slices) * blockDim.x * CPT + threadIdx.x * CPT;
  const bool active = c0 < d;
  const int chunks8 = d >> 3;
  const int halo = (ks - 1) * dil;
  const float inv_d = 1.0f / static_cast<float>(d);
  const int64_t branch_stride = N * d;

  // conv taps with the RMSNorm gain and SiLU's half-argument folded in, as packed pairs:
  // wg[j][q] = w[c, j] gamma[c] / 2 for c = c0 + 2q, c0 + 2q + 1
  uint64_t wg[kTaps][kPairs];
#pragma unroll
  for (int q = 0; q < kPairs; ++q) {
    float g[2], w[kTaps][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = c0 + 2 * q + e;
      g[e] = active ? 0.5f * gamma_c[c] : 0.f;
#pragma unroll
      for (int j = 0; j < kTaps; ++j) w[j][e] = (active && j < ks) ? conv_w[c * ks + j] * g[e] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kTaps; ++j) wg[j][q] = pk(w[j][0], w[j][1]);
  }

  for (int run = blockIdx.x / slices; run < total_runs; run += gridDim.x / slices) {
    const int b = run / runs_per_seq;
    const int t0 = (run - b * runs_per_seq) * kRun;
    const int t1 = min(t0 + kRun, L);
    const int p0 = max(0, t0 - halo);
    const int npos = t1 - p0;
    const int64_t seq0 = static_cast<int64_t>(b) * L;

    // 1. mean(v^2) per position: given (v_ms, the projection's), or one warp per position
    //    (16-byte loads, unrolled so each lane has several of its row's loads in flight)
    if (v_ms)
      for (int i = threadIdx.x; i < npos; i += blockDim.x) s_ms[i] = v_ms[seq0 + p0 + i];
    for (int i = warp; !v_ms && i < npos; i += nwarps) {
      const float s = row_mean_square(v + (seq0 + p0 + i) * d, chunks8, inv_d, lane);
      if (lane == 0) s_ms[i] = s;
    }
    __syncthreads();

    // 2. tap scalars: f = alpha / sqrt(alpha^2 mean(v^2) + eps) at t - j dil, and alpha_t
    for (int idx = threadIdx.x; idx < M * kRun * kTaps; idx += blockDim.x) {
      const int j = idx % kTaps, i = (idx / kTaps) % kRun, m = idx / (kTaps * kRun);
      const int t = t0 + i, p = t - j * dil;
      float a = 0.f, f = 0.f;
      if (t < t1 && j < ks && p >= 0) {
        a = alpha[m * N + seq0 + p];
        f = tap_scale(a, s_ms[p - p0], eps);
      }
      *reinterpret_cast<float2*>(&s_tap[m][i][2 * j]) = make_float2(f, f);
      if (j == 0) *reinterpret_cast<float2*>(&s_tap[m][i][8]) = make_float2(a, a);
    }
    __syncthreads();

    // 3. conv + SiLU + residual. Positions are walked by residue class mod dil, so the taps
    //    of t (t, t - dil, t - 2 dil, t - 3 dil) are the last four rows of the class: at the
    //    k-th step the row t - j dil sits in window slot (k - j) mod 4, and the walk is
    //    unrolled by 4 so every slot index is a constant. H and v of the next PF positions in
    //    walking order are already on their way into this thread's ring slots (one cp.async
    //    group per position); v_t enters the window from the ring at its step.
    int pr = 0, pi = 0, ps = 0;  // prefetch cursor: position t0 + pr + dil * pi, sequence ps
    auto prefetch_next = [&]() {
      if (pr < dil && t0 + pr < t1) {
        if (active) {
          const int t = t0 + pr + dil * pi;
          const int slot = ps % PF;
          const T* src = H + (seq0 + t) * d + c0;
#pragma unroll
          for (int m = 0; m < MMAX; ++m) {
            if (m >= M) continue;
            cp_async_bytes<static_cast<int>(sizeof(Raw))>(ring_at(slot, m), src + m * branch_stride);
          }
          cp_async_bytes<static_cast<int>(sizeof(Raw))>(ring_at(slot, MMAX), v + (seq0 + t) * d + c0);
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
      uint64_t win[kTaps][kPairs];  // v rows of this residue class, zero before the sequence start
#pragma unroll
      for (int j = 1; j < kTaps; ++j) {  // v_t itself comes from the ring at its step
        const int p = t0 + r - j * dil;
        float x[CPT];
        if (active && j < ks && p >= 0) {
          Vec::unpack(Vec::load(v + (seq0 + p) * d + c0), x);
        } else {
#pragma unroll
          for (int q = 0; q < CPT; ++q) x[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < kPairs; ++q) win[(kTaps - j) % kTaps][q] = pk(x[2 * q], x[2 * q + 1]);
      }
      int t = t0 + r;
      while (t < t1) {
#pragma unroll
        for (int k = 0; k < kTaps; ++k) {
          cp_async_wait<PF - 1>();  // this thread's copies for position t have landed
          if (active) {
            const Raw* hr = ring_at(s % PF, 0);
            {  // v_t into the window slot of v_{t - 4 dil}
              float x[CPT];
              Vec::unpack(hr[MMAX * blockDim.x], x);
#pragma unroll
              for (int q = 0; q < kPairs; ++q) win[k][q] = pk(x[2 * q], x[2 * q + 1]);
            }
            T* out = H + (seq0 + t) * d + c0;
            uint64_t prod[kTaps][kPairs];  // (w[:, j] gamma / 2) * v_{t - j dil}
#pragma unroll
            for (int j = 0; j < kTaps; ++j)
#pragma unroll
              for (int q = 0; q < kPairs; ++q) prod[j][q] = mul2(wg[j][q], win[(k - j + kTaps) % kTaps][q]);
#pragma unroll
            for (int m = 0; m < MMAX; ++m) {
              if (m >= M) continue;
              const ulonglong2 f01 = *reinterpret_cast<const ulonglong2*>(&s_tap[m][t - t0][0]);
              const ulonglong2 f23 = *reinterpret_cast<const ulonglong2*>(&s_tap[m][t - t0][4]);
              const uint64_t aa = *reinterpret_cast<const uint64_t*>(&s_tap[m][t - t0][8]);
              float h[CPT];
              Vec::unpack(hr[m * blockDim.x], h);
#pragma unroll
              for (int q = 0; q < kPairs; ++q) {
                uint64_t c = mul2(f01.x, prod[0][q]);  // c / 2
                c = fma2(f01.y, prod[1][q], c);
                c = fma2(f23.x, prod[2][q], c);
                c = fma2(f23.y, prod[3][q], c);
                const uint64_t acc = fma2(aa, win[k][q], pk(h[2 * q], h[2 * q + 1]));  // H + alpha v_t
                upk(silu2_add<T>(c, acc), h[2 * q], h[2 * q + 1]);
              }
              Vec::store(out + m * branch_stride, h);
            }
          }
          prefetch_next();
          t += dil;
          ++s;
          if (t >= t1) break;
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();
  }
}

// ------------------------------------------------------------------ streaming decode

// Position t = pos[b] - 1 of each sequence. A persistent grid of blocks, block i owning
// channel slice i mod slices (512 channels, thread j channels [4 j, 4 j + 4)) of every
// (gridDim / slices)-th sequence; the conv taps are loaded once per block. Operands go
// through a kStages-deep ring in shared memory filled by cp.async, kStages - 1 sequences
// ahead of the one being computed (no registers held while they are in flight): each
// thread copies its chunks of v_t, of H for the M branches and of the ring's earlier
// inputs (slot p mod D holds v_p, alpha_{:, p}, mean(v_p^2)), threads < 4 (M + 1) the raw
// tap scalars; the position of a sequence is read one fill earlier still. One barrier per
// sequence, once the thread's copies of this sequence and the next have landed: it makes
// both stages visible, frees the stage filled next and publishes this sequence's tap
// factors f, which threads < 4 M formed from the next-but-current stage's raw scalars in
// the previous iteration. Every product, FMA and the SiLU are the full-sequence kernel's,
// in its order, so H gets the same update.
// The ring has one slot more than the taps reach, so the slot of t, written here (v by
// each thread for its channels, the scalars by slice 0), is read by no block of this launch.
constexpr int kDecodeThreads = 128;
constexpr int kDecodeStages = 4;

__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}

template <typename T, int MMAX>
struct DecodeStage {
  using Raw = typename VecN<T, kCpt>::Raw;
  static constexpr int kOps = 1 + MMAX + (kTaps - 1);  // v_t, H of each branch, taps 1..3
  Raw ops[kOps][kDecodeThreads];
  float sc[kTaps][MMAX + 1];  // per tap j: alpha of each branch, then mean(v^2) (raw, copied)
  float f[kTaps][MMAX];       // tap factors f_{t - j dil} of each branch (formed from sc)
  float ms_t;                 // mean(v_t^2)
  int t;                      // position of the stage's sequence; < 0: nothing to do
};

template <typename T, int MB>
__global__ void __launch_bounds__(kDecodeThreads, 6) decode_conv_kernel(
    int B, int d, int M_rt, int slices, const T* __restrict__ v, const float* __restrict__ alpha,
    const float* __restrict__ v_ms, const float* __restrict__ gamma_c, const float* __restrict__ conv_w, int ks,
    int dil, float eps, const int32_t* __restrict__ pos, T* __restrict__ ring_v, float* __restrict__ ring_a,
    float* __restrict__ ring_ms, int D, T* __restrict__ H, int* err_word) {
  constexpr int MMAX = MB > 0 ? MB : kMaxBranches;
  const int M = MB > 0 ? MB : M_rt;
  using Vec = VecN<T, kCpt>;
  using Raw = typename Vec::Raw;
  using Stage = DecodeStage<T, MMAX>;
  constexpr int kPairs = kCpt / 2;
  extern __shared__ __align__(16) uint8_t s_raw[];
  Stage* stages = reinterpret_cast<Stage*>(s_raw);
  const int slice = blockIdx.x % slices;
  const int lane = threadIdx.x & 31;
  const int c0 = (slice * kDecodeThreads + threadIdx.x) * kCpt;
  const bool active = c0 < d;
  const int b0 = blockIdx.x / slices, bstride = gridDim.x / slices;

  // conv taps with the RMSNorm gain and SiLU's half-argument folded in (as the full kernel)
  uint64_t wg[kTaps][kPairs];
#pragma unroll
  for (int q = 0; q < kPairs; ++q) {
    float g[2], w[kTaps][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = c0 + 2 * q + e;
      g[e] = active ? 0.5f * gamma_c[c] : 0.f;
#pragma unroll
      for (int j = 0; j < kTaps; ++j) w[j][e] = (active && j < ks) ? conv_w[c * ks + j] * g[e] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kTaps; ++j) wg[j][q] = pk(w[j][0], w[j][1]);
  }

  // the k-th sequence of this block, at position t, into stage `st` (one commit group)
  auto fill = [&](int k, Stage& st, int t) {
    const int b = b0 + k * bstride;
    if (b < B && t >= 0) {
      if (active) {
        cp_async_bytes<static_cast<int>(sizeof(Raw))>(&st.ops[0][threadIdx.x], v + static_cast<int64_t>(b) * d + c0);
#pragma unroll
        for (int m = 0; m < MMAX; ++m)
          if (m < M)
            cp_async_bytes<static_cast<int>(sizeof(Raw))>(&st.ops[1 + m][threadIdx.x],
                                                          H + (static_cast<int64_t>(m) * B + b) * d + c0);
#pragma unroll
        for (int j = 1; j < kTaps; ++j) {
          const int p = t - j * dil;
          if (j < ks && p >= 0)
            cp_async_bytes<static_cast<int>(sizeof(Raw))>(&st.ops[MMAX + j][threadIdx.x],
                                                          ring_v + (static_cast<int64_t>(b) * D + p % D) * d + c0);
        }
      }
      if (threadIdx.x < kTaps * (M + 1)) {
        const int j = threadIdx.x / (M + 1), m = threadIdx.x - j * (M + 1);
        const int p = t - j * dil;
        if (j < ks && p >= 0) {
          if (j == 0) {
            if (m < M) cp_async4(&st.sc[0][m], alpha + static_cast<int64_t>(m) * B + b);
            else if (v_ms) cp_async4(&st.sc[0][MMAX], v_ms + b);
          } else {
            const int64_t slot = static_cast<int64_t>(b) * D + p % D;
            if (m < M) cp_async4(&st.sc[j][m], ring_a + slot * M + m);
            else cp_async4(&st.sc[j][MMAX], ring_ms + slot);
          }
        }
      }
    }
    if (threadIdx.x == 0) st.t = b < B ? t : -1;
    cp_async_commit();
  };
  auto pos_of = [&](int k) -> int {
    const int b = b0 + k * bstride;
    return b < B ? pos[b] - 1 : -1;
  };
  // tap factors of the k-th sequence from its stage's raw scalars (warp 0; the stage's
  // copies have landed and are visible): f = 0 before the start and past the kernel size
  auto prep = [&](int k, Stage& st) {
    const int b = b0 + k * bstride;
    const int t = st.t;
    if (threadIdx.x >= 32 || b >= B || t < 0) return;
    // mean(v_t^2): handed over, or reduced by this warp as the full kernel's warp does
    const float ms = v_ms ? st.sc[0][MMAX]
                          : row_mean_square(v + static_cast<int64_t>(b) * d, d >> 3, 1.0f / static_cast<float>(d),
                                            lane);
    if (threadIdx.x < kTaps * M) {
      const int j = threadIdx.x / M, m = threadIdx.x - j * M;
      const bool ok = j < ks && t - j * dil >= 0;
      st.f[j][m] = ok ? tap_scale(st.sc[j][m], j == 0 ? ms : st.sc[j][MMAX], eps) : 0.f;
    }
    if (threadIdx.x == 0) st.ms_t = ms;
  };

  int tp[kDecodeStages - 1];
#pragma unroll
  for (int k = 0; k < kDecodeStages - 1; ++k) tp[k] = pos_of(k);
#pragma unroll
  for (int k = 0; k < kDecodeStages - 1; ++k) fill(k, stages[k], tp[k]);
  int t_pf = pos_of(kDecodeStages - 1);
  cp_async_wait<kDecodeStages - 2>();  // sequence 0's copies
  __syncthreads();
  prep(0, stages[0]);

  for (int k = 0; b0 + k * bstride < B; ++k) {
    const int b = b0 + k * bstride;
    Stage& st = stages[k % kDecodeStages];
    cp_async_wait<kDecodeStages - 3>();  // this thread's copies of sequences k and k + 1 have landed
    __syncthreads();                     // everyone's; stage k's factors are out; stage k - 1 is free
    fill(k + kDecodeStages - 1, stages[(k + kDecodeStages - 1) % kDecodeStages], t_pf);
    t_pf = pos_of(k + kDecodeStages);
    prep(k + 1, stages[(k + 1) % kDecodeStages]);
    const int t = st.t;
    if (t < 0) {  // pos[b] < 1: no consumed token to apply the conv to (uniform in the block)
      if (threadIdx.x == 0 && slice == 0 && err_word) atomicOr(err_word, 512);
      continue;
    }
    if (active) {
      uint64_t x[kTaps][kPairs];
#pragma unroll
      for (int j = 0; j < kTaps; ++j) {
        const int p = t - j * dil;
        float xf[kCpt];
        if (j == 0) {
          Vec::unpack(st.ops[0][threadIdx.x], xf);
        } else if (j < ks && p >= 0) {
          Vec::unpack(st.ops[MMAX + j][threadIdx.x], xf);
        } else {
#pragma unroll
          for (int q = 0; q < kCpt; ++q) xf[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < kPairs; ++q) x[j][q] = pk(xf[2 * q], xf[2 * q + 1]);
      }
      uint64_t prod[kTaps][kPairs];
#pragma unroll
      for (int j = 0; j < kTaps; ++j)
#pragma unroll
        for (int q = 0; q < kPairs; ++q) prod[j][q] = mul2(wg[j][q], x[j][q]);
#pragma unroll
      for (int m = 0; m < MMAX; ++m) {
        if (m >= M) continue;
        const float a_t = st.sc[0][m];
        const uint64_t f0 = pk(st.f[0][m], st.f[0][m]), f1 = pk(st.f[1][m], st.f[1][m]);
        const uint64_t f2 = pk(st.f[2][m], st.f[2][m]), f3 = pk(st.f[3][m], st.f[3][m]);
        const uint64_t aa = pk(a_t, a_t);
        float h[kCpt];
        Vec::unpack(st.ops[1 + m][threadIdx.x], h);
#pragma unroll
        for (int q = 0; q < kPairs; ++q) {
          uint64_t c = mul2(f0, prod[0][q]);  // c / 2
          c = fma2(f1, prod[1][q], c);
          c = fma2(f2, prod[2][q], c);
          c = fma2(f3, prod[3][q], c);
          const uint64_t acc = fma2(aa, x[0][q], pk(h[2 * q], h[2 * q + 1]));  // H + alpha v_t
          upk(silu2_add<T>(c, acc), h[2 * q], h[2 * q + 1]);
        }
        Vec::store(H + (static_cast<int64_t>(m) * B + b) * d + c0, h);
      }
      if (D > 0) {
        float xf[kCpt];
        Vec::unpack(st.ops[0][threadIdx.x], xf);
        Vec::store(ring_v + (static_cast<int64_t>(b) * D + t % D) * d + c0, xf);
      }
    }
    // the scalars of position t into its slot
    if (D > 0 && slice == 0 && threadIdx.x < M) {
      const int64_t slot = static_cast<int64_t>(b) * D + t % D;
      ring_a[slot * M + threadIdx.x] = st.sc[0][threadIdx.x];
      if (threadIdx.x == 0) ring_ms[slot] = st.ms_t;
    }
  }
  cp_async_wait<0>();
}

template <typename T, int MB>
pg_status launch_decode(const pg_decode_state* st, const void* v, const float* alpha, const float* v_ms,
                        const float* gamma_c, const float* conv_w, float eps, void* H, cudaStream_t stream) {
  const int slices = (st->d + kDecodeThreads * kCpt - 1) / (kDecodeThreads * kCpt);
  auto kern = decode_conv_kernel<T, MB>;
  const size_t smem = sizeof(DecodeStage<T, (MB > 0 ? MB : kMaxBranches)>) * kDecodeStages;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e);
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  if (per_sm < 1) return PG_ERR_UNSUPPORTED;
  // sequences in flight: as many as fill the SMs' block slots, at most B
  const int64_t cap = std::max<int64_t>(1, static_cast<int64_t>(sm_count()) * per_sm / slices);
  const int64_t blocks = std::min<int64_t>(st->B, cap) * slices;
  kern<<<static_cast<unsigned>(blocks), kDecodeThreads, smem, stream>>>(
      st->B, st->d, st->M, slices, static_cast<const T*>(v), alpha, v_ms, gamma_c, conv_w, st->kernel_size,
      st->dilation, eps, st->pos, static_cast<T*>(st->ring_v), st->ring_alpha, st->ring_ms, st->depth,
      static_cast<T*>(H), device_error_word());
  return after_launch(1);
}

template <typename T>
pg_status dispatch_decode(const pg_decode_state* st, const void* v, const float* alpha, const float* v_ms,
                          const float* gamma_c, const float* conv_w, float eps, void* H, cudaStream_t stream) {
  switch (st->M) {
    case 1: return launch_decode<T, 1>(st, v, alpha, v_ms, gamma_c, conv_w, eps, H, stream);
    case 2: return launch_decode<T, 2>(st, v, alpha, v_ms, gamma_c, conv_w, eps, H, stream);
    case 4: return launch_decode<T, 4>(st, v, alpha, v_ms, gamma_c, conv_w, eps, H, stream);
    default: return launch_decode<T, 0>(st, v, alpha, v_ms, gamma_c, conv_w, eps, H, stream);
  }
}

template <typename T>
pg_status launch(int B, int L, int d, int M, const void* v, const float* alpha, const float* v_ms,
                 const float* gamma_c, const float* conv_w, int ks, int dil, float eps, void* H, cudaStream_t stream) {
  // channel slices of at most `width` threads * 4 channels, each a multiple of 128 (whole warps)
  const int width = v_ms ? kSliceThreads : kMaxThreads;
  const int slices = (d + width * kCpt - 1) / (width * kCpt);
  const int slice_ch = ((d + slices - 1) / slices + 32 * kCpt - 1) / (32 * kCpt) * (32 * kCpt);
  const int threads = slice_ch / kCpt;
  const int runs_per_seq = (L + kRun - 1) / kRun;
  const int64_t total = static_cast<int64_t>(B) * runs_per_seq;
  if (total >= (1ll << 31)) return PG_ERR_SHAPE;
  const int64_t N = static_cast<int64_t>(B) * L;
  auto run = [&](auto kern, int mmax, int pf) -> pg_status {
    const size_t ring = static_cast<size_t>(pf) * (mmax + 1) * threads * (sizeof(T) * kCpt);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ring));
    if (e != cudaSuccess) return cuda_fail(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, ring);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm < 1) return PG_ERR_UNSUPPORTED;
    const int64_t cap = std::max<int64_t>(1, static_cast<int64_t>(sm_count()) * per_sm / slices);  // runs in flight
    const int grid = static_cast<int>((total < cap ? total : cap) * slices);
    kern<<<grid, threads, ring, stream>>>(L, d, M, N, static_cast<const T*>(v), alpha, v_ms, gamma_c, conv_w, ks,
                                          dil, eps, static_cast<T*>(H), runs_per_seq, static_cast<int>(total),
                                          slices);
    return after_launch(1);
  };
  switch (M) {
    case 1: return run(conv_residual_kernel<T, 1, kPrefetch>, 1, kPrefetch);
    case 2: return run(conv_residual_kernel<T, 2, kPrefetch>, 2, kPrefetch);
    case 4: return run(conv_residual_kernel<T, 4, kPrefetch>, 4, kPrefetch);
    default: return run(conv_residual_kernel<T, 0, kPrefetch>, kMaxBranches, kPrefetch);
  }
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

extern "C" pg_status pg_decode_conv_residual(const pg_decode_state* state, const void* v, const float* alpha,
                                             const float* v_ms, const float* gamma_c, const float* conv_w, float eps,
                                             void* H, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const pg_status st = decode_state_check(state, true);
  if (st != PG_OK) return st;
  if (!v || !alpha || !gamma_c || !conv_w || !H) return PG_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(H)) & 15u) return PG_ERR_ALIGN;
  if (sm_count() == 0) return cuda_fail(cudaGetLastError());
  if (state->dtype == PG_BF16)
    return dispatch_decode<__nv_bfloat16>(state, v, alpha, v_ms, gamma_c, conv_w, eps, H, stream);
  return dispatch_decode<float>(state, v, alpha, v_ms, gamma_c, conv_w, eps, H, stream);
}
