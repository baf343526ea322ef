// Projection and gates (sm_103a).
//
//   v = W_V e_t, k^(m) = W_K^(m) e_t (one fused GEMM over [W_V; W_K^(1..M)], Engram notes
//   (arXiv 2601.07372) section 3.4), then
//   scalar gate   x + g v                                   PageGram report section 3.1
//   context gate  alpha = sigmoid(RMSNorm(h)^T RMSNorm(k) / sqrt(d))   Engram notes 3.3/3.4
//
// bf16: a persistent tcgen05 GEMM. One CTA per SM, 6 warps:
//   warp 0      TMA producer: 128x64 A (e) and BNx64 B (W) tiles, 128-byte swizzle,
//               into a 4-stage shared-memory ring (mbarrier full/empty pairs)
//   warp 1      allocates 2*BN TMEM columns (two fp32 accumulators) and issues
//               tcgen05.mma (M=128, N=BN, K=16) from one thread; tcgen05.commit
//               frees smem stages and publishes finished accumulators
//   warps 2..5  epilogue: tcgen05.ld 32x32b (thread = output row), gate math, stores;
//               context-gate tiles reduce per-row partial sums instead of storing
// The epilogue of tile i overlaps the MMAs of tile i+1 (double-buffered TMEM).
// fp32 and W == NULL: pg_project_simt.cu.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pg_conv_math.cuh"
#include "pg_hash.cuh"

namespace pg {
namespace {

// ==================================================================== PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Acquire at cluster scope: for barriers that threads of the peer CTA arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // a bounded wait gives up after ~1 s

template <bool CLUSTER>
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
  return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}

template <bool CLUSTER>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort) {
  const uint64_t t0 = globaltimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_poll<CLUSTER>(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
}

// Waits for the phase of `parity` to complete; false after the time limit or when
// another role of the CTA has already given up (`abort`). The first poll is inline: the
// MMA issuer runs one wait per 512 tensor-core cycles and a call costs it a large share.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  return mbar_poll<CLUSTER>(bar, parity) || mbar_wait_slow<CLUSTER>(bar, parity, abort);
}

// ---- CTA pairs (cluster of 2): rank 0 issues the M = 256 MMAs for both CTAs

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// All threads of both CTAs; release/acquire orders shared-memory work across the pair.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same shared-memory offset in CTA `rank` of the pair.
__device__ __forceinline__ uint32_t pair_addr(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Load into this CTA's shared memory; completion is counted on `bar_cluster`, which may be
// the barrier of the other CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

// Plain (non-tensor) bulk copy global -> this CTA's shared memory, counted on `bar`; both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// TMEM allocation: one warp of the CTA, or one warp of each CTA of a pair (PAIR).
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (PAIR)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) (+)= A(smem desc) x B(smem desc)^T, bf16 (FP8: E4M3) in, fp32 accumulate. PAIR:
// M = 256 rows over the two CTAs (each holds 128 rows of A and half of B's rows at the same
// offsets, and 128 rows of D in its TMEM). One instruction covers 32 bytes of K: 16 bf16
// or 32 E4M3 elements.
template <bool PAIR, bool FP8 = false>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  if constexpr (FP8 && PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else if constexpr (PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on `bar` when all previously issued tcgen05.mma of this thread complete;
// PAIR: on the barrier at that offset in both CTAs.
template <bool PAIR>
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  if constexpr (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// As umma_commit, on this CTA's barrier only.
template <bool PAIR>
__device__ __forceinline__ void umma_commit_local(uint32_t bar) {
  if constexpr (PAIR)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets row (lane base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// TMA store of a 2-D box from shared memory (bulk group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}

// 3-D tensor copies (the conv's branch-state tiles: [M, N, d] with rows clipped per branch).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until all but the most recent committed bulk store group have read shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Waits until the committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until the committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format) for a K-major operand tile written
// by TMA with 128-byte swizzle: rows of 64 bf16 (128 B), 8-row atoms of 1024 B.
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4 (unused here)
//   bits 32-45 stride byte offset >> 4 (1024 B between 8-row atoms)
//   bits 46-47 descriptor version 1    bits 61-63 layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9,
// 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B E4M3 (format 0 at bits 7-9, 10-12), both
// K-major, N >> 3 at bits 17-22, M >> 4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// the two bf16 of a 32-bit word as an fp32 pair (low half first)
__device__ __forceinline__ uint64_t bf16x2_as_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ void unpack_bf16x8(uint4 w, float* f) {
  f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xFFFF0000u);
  f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

// ==================================================================== tcgen05 GEMM

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kStages = 4;          // shared-memory ring of a single-CTA tile (48 KB per stage)
constexpr int kStagesPair = 6;      // of a CTA pair's tile (32 KB per stage and CTA)
constexpr int kGemmThreads = 224;   // 7 warps: A/B producer, MMA, operand producer, 4 x epilogue
constexpr int kFusedThreads = 480;  // + 8 gather warps producing the A operand
constexpr int kGatherWarp0 = 7;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kEpiCols = 32;        // columns per epilogue sub-tile
constexpr int kEpiStagesMax = 4;    // epilogue shared-memory ring (3 slots in the fused kernel)
constexpr int kEpiBytes = kBM * kEpiCols * 2;
constexpr int kFusedItems = 32;     // (order, head) items of the fused kernel
// Producing kernel (PRODUCE): 16 warps. Warps 0-2: A/B producer, MMA issuer, epilogue
// operand producer; warp 3: gather coordinator; warps 4-7: epilogue; warps 8-15: gather.
constexpr int kProduceThreads = 512;
constexpr int kProdCoordWarp = 3;
constexpr int kProdEpiWarp0 = 4;
constexpr int kProdGatherWarp0 = 8;
constexpr int kUnitSlots = 4;       // ring of gather units between the coordinator and the gather warps
constexpr int kCanonStride = 128 + 4;  // per slot: canonical IDs of the unit's tokens and the 3 before
constexpr int kUnitRows = 8 * 64;  // rows of a gather unit: 64 per gather warp

constexpr int kReadyTokens = kBM;   // tokens per ready counter (one A tile of one CTA)
// Projection + conv in one launch (CONV): GEMM operand stages (5: room for the conv ring),
// the lag of the conv items behind the GEMM tiles (in m-blocks), the largest causal halo
// (kernel_size - 1) * dilation, and the conv warps' ring: per stage a 16-column sub-tile of
// H and of v (128 rows each, 32-byte swizzle), v's halo rows before it and the packed taps
// of its 8 column pairs.
constexpr int kStagesConv = 5;
constexpr int kConvLag = 2;
constexpr int kConvMaxHalo = 24;
constexpr int kConvCols = 16;
constexpr int kConvTileBytes = kBM * kConvCols * 2;              // 4096
constexpr int kConvHaloBytes = kConvMaxHalo * kConvCols * 2;     // 768
constexpr int kConvTapBytes = (kConvCols / 2) * 4 * 8;           // 256
constexpr int kConvStageBytes = 2 * kConvTileBytes + kConvHaloBytes + kConvTapBytes;  // 9216
constexpr int kConvStages = 3;
constexpr int kConvRows = kBM + kConvMaxHalo;  // f and alpha rows of a conv item
constexpr int kConvWarp0 = 7;      // warps 7..14 compute the conv (row x 8-column chunk), warp 15 streams its operands
constexpr int kConvCompute = 256;  // conv compute threads
constexpr int kConvThreads = 512;
constexpr int kErrConvWait = 16384;

template <bool GATHER>
__host__ __device__ constexpr int epi_stages() { return GATHER ? 3 : 4; }

template <bool PAIR>
__host__ __device__ constexpr int gemm_stages() { return PAIR ? kStagesPair : kStages; }

// What the gather warps of the fused kernel need (empty in the plain GEMM).
struct FusedGather {
  HashParams P;
  uint64_t seed;
  const int32_t* tokens;
  const uint32_t* canon_map;
  const uint8_t* table;
  uint32_t L;
  uint64_t fm_L;
  int32_t* err;
  // producing kernel only: e_t [N, Din] written by the gather warps, per-128-token ready
  // counters (chunks done) and the chunk claim counter, both zeroed before the launch
  uint8_t* e_out;
  uint32_t* ready;
  uint32_t* claim;
  int unit_tokens;  // tokens per work unit: the largest power of two <= 128 with unit_tokens * items <= 8 x
                    // a gather warp's rows per unit
};
struct NoGather {};
template <bool GATHER>
struct GatherParam {
  using type = NoGather;
};
template <>
struct GatherParam<true> {
  using type = FusedGather;
};

struct GemmArgs {
  int N;          // rows of e (tokens)
  int Din;        // reduction length
  int Dcols;      // rows of W = output columns of the GEMM ((1+M)*d)
  int d;          // model width
  int M;          // branches (context gate)
  float g;        // scalar gate
  const float* gamma_h;      // [d]
  const float* gamma_k;      // [d]
  float* partials;           // [M, d/BN, 3, N] (context gate)
  float* vpart;              // [d/BN, N] row sums of v^2 per v tile (context gate, or null)
  const float* sa;           // FP8: per-row scales of e [N]
  const float* sw;           // FP8: per-row scales of W [Dcols]
  int* err_word;
  // CONV: the causal conv + residual behind the tiles
  uint32_t* done = nullptr;        // [m-blocks] CTA-tiles of each m-block finished and published
  const uint64_t* conv_taps = nullptr;  // [d / 2][4] fp32 pairs w[c, j] gamma_c[c] / 2, c = 2p, 2p + 1
  float* alpha_out = nullptr;      // [M, N]
  float* v_ms_out = nullptr;       // [N] or null
  float eps = 0.f;
  int L = 1;                       // sequence length
  int ks = 0;                      // conv kernel size (<= 4)
  int dil = 1;                     // dilation
  int halo = 0;                    // (ks - 1) * dil
};

template <int S>
struct GemmBarriers {
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t epi_full[kEpiStagesMax];   // operand sub-tile landed (or slot handed over)
  uint64_t epi_done[kEpiStagesMax];   // all 128 epilogue threads finished with the slot
  uint64_t epi_empty[kEpiStagesMax];  // slot free again (its TMA store finished reading)
  uint64_t mma_done;
  uint64_t unit_full[kUnitSlots];  // producing kernel: gather unit announced in its slot
  uint64_t unit_done[kUnitSlots];  // producing kernel: every gather warp stored its share of it
  uint64_t pub;                    // CONV: the 128 epilogue threads finished a GEMM tile
  uint64_t conv_sync;              // CONV: the conv threads wrote a conv item's f and alpha
  uint64_t cfull[kConvStages];     // CONV: a conv sub-tile's operands landed
  uint64_t cdone[kConvStages];     // CONV: the conv threads updated the stage's H
  uint32_t tmem_base;
  int abort;
};

// Per epilogue slot, the column vectors of its sub-tile staged beside the operand: gamma_h,
// gamma_k (context gate, k tiles) and FP8's per-column scales, 32 fp32 each.
constexpr int kVecBytes = kEpiStagesMax * 3 * kEpiCols * 4;

template <bool PAIR, bool CONV>
__host__ __device__ constexpr int stages_of() { return CONV ? kStagesConv : gemm_stages<PAIR>(); }

template <int BN, bool GATHER, bool PAIR, bool PRODUCE, bool VEC, bool CONV = false>
constexpr size_t gemm_smem_bytes() {
  return 1024 /* alignment slack */ + stages_of<PAIR, CONV>() * (kABytes + (PAIR ? BN / 2 : BN) * kBK * 2) +
         epi_stages<GATHER || PRODUCE>() * kEpiBytes + (VEC ? kVecBytes : 0) +
         (CONV ? 512 + kConvStages * kConvStageBytes + 2 * 2 * kConvRows * sizeof(float) : 0) +
         sizeof(GemmBarriers<stages_of<PAIR, CONV>()>) +
         (GATHER || PRODUCE ? kFusedItems * sizeof(ItemConst) : 0) +
         (PRODUCE ? kUnitSlots * kCanonStride * sizeof(uint32_t) : 0);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Wait (bounded) until the ready counter reaches `need`: false on abort or time-out.
__device__ __forceinline__ bool wait_ready(const uint32_t* flag, uint32_t need, volatile int* abort) {
  if (ld_acquire_gpu(flag) >= need) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(flag) >= need) return true;
    if (*abort || globaltimer() - t0 > kWaitLimitNs) return false;
  }
}

// Self-test of the two bounded waits every tcgen05 kernel here relies on: one thread
// waits on an mbarrier phase that nothing completes, then on a ready counter that nothing
// raises (the caller's zeroed word). Each wait must give up after its limit (~1 s) and the
// kernel reports it through the device error word (2048: the mbarrier wait, 4096: the
// counter wait) and returns; no copy, MMA or TMEM is involved.
constexpr int kErrSelftestBarrier = 2048;
constexpr int kErrSelftestCounter = 4096;

__global__ void __launch_bounds__(32) wait_selftest_kernel(const uint32_t* __restrict__ flag, int* err_word) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  volatile int* abort = &abort_flag;
  if (!mbar_wait(smem_u32(&bar), 0u, abort)) atomicOr(err_word, kErrSelftestBarrier);
  if (!wait_ready(flag, 1u, abort)) atomicOr(err_word, kErrSelftestCounter);
}

// The context gate of (branch m, row) from the per-tile partial sums of the projection's
// epilogue (sum gh gk h k, sum k^2, sum h^2 per 256-column tile), summed in tile order:
// alpha = sigmoid(RMSNorm(h) . RMSNorm(k) / sqrt(d)); and mean(v^2) from the per-tile sums
// of the stored v. Plain loads: the conv items read sums this launch wrote.
__device__ __forceinline__ float gate_alpha(const float* partials, int m, int tpb, int N, int d, float eps,
                                            int row) {
  float s_hk = 0.f, s_kk = 0.f, s_hh = 0.f;
  for (int t0 = 0; t0 < tpb; t0 += 16) {  // 16 tiles' loads in flight, then added in tile order
    float a[16], b[16], c[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      a[u] = b[u] = c[u] = 0.f;
      if (t0 + u < tpb) {
        const float* p = partials + (static_cast<size_t>(m * tpb + t0 + u) * 3) * N + row;
        a[u] = p[0];
        b[u] = p[N];
        c[u] = p[2 * static_cast<size_t>(N)];
      }
    }
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (t0 + u < tpb) {
        s_hk += a[u];
        s_kk += b[u];
        s_hh += c[u];
      }
  }
  const float inv_d = 1.0f / static_cast<float>(d);
  const float rh = sqrtf(__fmaf_rn(s_hh, inv_d, eps));
  const float rk = sqrtf(__fmaf_rn(s_kk, inv_d, eps));
  const float s = s_hk / (rh * rk * sqrtf(static_cast<float>(d)));
  return 1.0f / (1.0f + expf(-s));
}
__device__ __forceinline__ float row_mean_sq(const float* vpart, int tpb, int N, int d, int row) {
  float s_vv = 0.f;
  for (int t0 = 0; t0 < tpb; t0 += 16) {
    float a[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) a[u] = t0 + u < tpb ? vpart[static_cast<size_t>(t0 + u) * N + row] : 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (t0 + u < tpb) s_vv += a[u];
  }
  return s_vv / static_cast<float>(d);
}

// Epilogue operands and results move through 128 x 32 bf16 sub-tiles (64 bytes per row)
// written / read by TMA with 64-byte swizzle: 16-byte chunk c of row r sits at
// r * 64 + ((c ^ ((r >> 1) & 3)) * 16), so the 32 rows of a warp hit every bank.
__device__ __forceinline__ uint32_t epi_offset(int row, int chunk) {
  return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// GATHER: the A operand (e_t) is not read from global memory; 8 gather warps build each
// 128 x 64 A tile in shared memory from the table (k-block kb = head (o, k) of r = 64),
// exactly as pg_gather_sign_concat would have written it.
// PAIR: a cluster of two CTAs computes 256 x BN tiles. Each CTA stages its 128 rows of A
// and BN/2 rows of B; both CTAs' copies count on rank 0's `full` barrier, rank 0 issues
// M = 256 MMAs (rows 128 r .. 128 r + 127 accumulate in CTA r's TMEM) and its commits
// arrive on the barriers of both CTAs; each CTA runs the epilogue of its own 128 rows.
// PRODUCE: 8 more warps per CTA compute e_t itself (the lookup of pg_gather_sign_concat)
// into global memory while the tensor cores work: they claim chunks of 8 tokens from a
// global counter in the order the tiles are walked, write the chunk's e_t rows and count
// it on its 128-token block's ready counter (release); the A producer waits (acquire,
// bounded) for a block's count before its first TMA load of that block. Any resident CTA
// claims and finishes chunks without waiting on anything, so every wait ends.
//
// CONV: the same kernel (CTA pairs, context gate) also runs the causal conv + SiLU +
// residual of pg_conv_residual, as "conv items" interleaved with the GEMM tiles: the pair's
// work list walks the m-blocks in ascending order and, kConvLag m-blocks behind the GEMM
// tiles, takes for each m-block M * d / BN conv items (branch, 256-column block) of the same
// 256 x 256 shape. A conv item's branch-state tile was read as h by the k tiles of its
// m-block moments earlier, so its H comes mostly from L2. Each CTA's epilogue publishes a
// finished GEMM tile on its m-block's counter (release, after its v stores completed);
// a conv item waits (acquire, bounded) until the counters of its m-block and the one before
// (the causal halo) are full, forms alpha and the RMSNorm tap factors of its rows from the
// partial sums, and updates H with the arithmetic of pg_conv_residual (shared header), so
// H, alpha and mean(v^2) are bit-identical to pg_project_gate followed by pg_conv_residual.
// Every wait is on work that appears earlier in the list, which every pair walks in order:
// the earliest waiting item always depends on GEMM tiles only, so all waits end.
template <int BN, int GATE, bool GATHER, bool PAIR, bool PRODUCE = false, bool FP8 = false, bool CONV = false>
__global__ void __launch_bounds__(PRODUCE ? kProduceThreads : GATHER ? kFusedThreads : CONV ? kConvThreads : kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_h,
                   const __grid_constant__ CUtensorMap map_v, const GemmArgs args,
                   const __grid_constant__ typename GatherParam<GATHER || PRODUCE>::type gat,
                   const __grid_constant__ CUtensorMap map_h3, const __grid_constant__ CUtensorMap map_vh) {
  static_assert(!(GATHER && PAIR), "the fused gather runs on single-CTA tiles");
  static_assert(!(GATHER && PRODUCE), "one way of making A");
  static_assert(!FP8 || (PAIR && !GATHER && !PRODUCE), "FP8 operands: the plain CTA-pair kernel");
  static_assert(!CONV || (PAIR && GATE == PG_GATE_CONTEXT && !GATHER && !PRODUCE && BN == 256),
                "the conv behind the tiles: plain CTA pairs, context gate");
  constexpr int kKB = FP8 ? 2 * kBK : kBK;  // elements of a 128-byte k-block row
  // FP8: stages of two k-blocks (8 MMAs per barrier wait: an E4M3 k-block is half the tensor
  // time of a bf16 one, and the single issuing thread's per-wait overhead would set the pace)
  constexpr int kSubK = FP8 ? 2 : 1;
  constexpr int kSt = stages_of<PAIR, CONV>() / kSubK;
  constexpr int kEpiStages = epi_stages<GATHER || PRODUCE>();
  constexpr int kBRows = PAIR ? BN / 2 : BN;  // rows of W this CTA stages per k-block
  constexpr int kBBytes = kBRows * kBK * 2;
  constexpr int kAStage = kABytes * kSubK, kBStage = kBBytes * kSubK;
  constexpr int kTileM = PAIR ? 2 * kBM : kBM;  // output rows of a tile
  constexpr uint32_t kIdesc = FP8 ? idesc_e4m3(kTileM, BN) : idesc_bf16(kTileM, BN);
  constexpr uint32_t kTmemCols = 2 * BN;
  constexpr int kSub = BN / kEpiCols;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kSt * kAStage;
  uint8_t* sE = sB + kSt * kBStage;
  constexpr bool kVec = GATE == PG_GATE_CONTEXT || FP8;
  float* s_vec = reinterpret_cast<float*>(sE + kEpiStages * kEpiBytes);  // [slot][gamma_h, gamma_k, scale][32]
  // CONV: per pair of epilogue slots the halo rows of v, the taps and gamma_c; then f and
  // alpha of a conv item's rows, double-buffered by item
  uint8_t* s_conv = sE + kEpiStages * kEpiBytes + (kVec ? kVecBytes : 0) + (CONV ? 512 : 0);  // 1024-aligned
  float* s_cf = reinterpret_cast<float*>(s_conv + kConvStages * kConvStageBytes);  // [2][kConvRows]
  float* s_ca = s_cf + 2 * kConvRows;                                               // [2][kConvRows]
  GemmBarriers<kSt>* bars = reinterpret_cast<GemmBarriers<kSt>*>(
      CONV ? reinterpret_cast<uint8_t*>(s_ca + 2 * kConvRows) : s_conv);
  ItemConst* s_ic = reinterpret_cast<ItemConst*>(bars + 1);
  // producing kernel: slot u holds at [i] the canonical ID of flat position (unit start - 3 + i)
  uint32_t* s_canon = reinterpret_cast<uint32_t*>(s_ic + (GATHER || PRODUCE ? kFusedItems : 0));
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // work units: CTAs, or CTA pairs
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const int unit = PAIR ? static_cast<int>(cluster_index()) : static_cast<int>(blockIdx.x);
  const int units = PAIR ? static_cast<int>(cluster_count()) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      // the TMA expect-tx arrival, plus the 64 gather threads that build the A tile
      mbar_init(smem_u32(&bars->full[s]), GATHER ? 1 + 64 : 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&bars->tmem_full[a]), 1);
      mbar_init(smem_u32(&bars->tmem_empty[a]), (PAIR ? 2 : 1) * 4 * 32);  // every epilogue thread
    }
    for (int s = 0; s < kEpiStages; ++s) {
      mbar_init(smem_u32(&bars->epi_full[s]), 1);
      mbar_init(smem_u32(&bars->epi_done[s]), 4 * 32);
      mbar_init(smem_u32(&bars->epi_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->mma_done), 1);
    mbar_init(smem_u32(&bars->pub), 4 * 32);
    mbar_init(smem_u32(&bars->conv_sync), kConvCompute);
    for (int s = 0; s < kConvStages; ++s) {
      mbar_init(smem_u32(&bars->cfull[s]), 1);
      mbar_init(smem_u32(&bars->cdone[s]), kConvCompute);
    }
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(smem_u32(&bars->unit_full[s]), 1);
      mbar_init(smem_u32(&bars->unit_done[s]), kProduceThreads / 32 - kProdGatherWarp0);
    }
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc<PAIR>(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish<PAIR>();
  }
  if constexpr (GATHER || PRODUCE) {
    constexpr int t0 = 32 * (PRODUCE ? kProdGatherWarp0 : kGatherWarp0);
    if (threadIdx.x >= t0 && threadIdx.x - t0 < gat.P.O * gat.P.H)
      init_item_const(s_ic[threadIdx.x - t0], gat.P, gat.seed, threadIdx.x - t0);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers and TMEM exist before any remote use
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // Tiles are walked from the last m-block down: when the projection follows the gather,
  // the most recently written rows of e_t are the ones still in L2.
  const int num_m = (args.N + kTileM - 1) / kTileM;
  const int num_n = args.Dcols / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = args.Din / (kKB * kSubK);  // stages per tile
  // The pair's work list. CONV: stage s holds the GEMM tiles of m-block s (s < num_m) and
  // then the conv items of m-block s - lag (s >= lag); otherwise the GEMM tiles, last
  // m-block first.
  const int num_c = CONV ? args.M * (args.d / BN) : 0;  // conv items per m-block
  const int num_items = num_tiles + num_m * num_c;
  auto item_of = [&](int i, bool& conv, int& m_blk, int& n_blk) {
    if constexpr (!CONV) {
      const int rt = num_tiles - 1 - i;
      conv = false;
      m_blk = rt / num_n;
      n_blk = rt - m_blk * num_n;
    } else {
      const int lag = kConvLag < num_m ? kConvLag : num_m;
      const int a_end = lag * num_n;
      const int per = num_n + num_c;
      const int b_end = a_end + (num_m - lag) * per;
      if (i < a_end) {
        conv = false;
        m_blk = i / num_n;
        n_blk = i - m_blk * num_n;
      } else if (i < b_end) {
        const int r = i - a_end, st = r / per, o = r - st * per;
        conv = o >= num_n;
        m_blk = conv ? st : lag + st;
        n_blk = conv ? o - num_n : o;
      } else {
        const int r = i - b_end;
        conv = true;
        m_blk = num_m - lag + r / num_c;
        n_blk = r - (r / num_c) * num_c;
      }
    }
  };

  __shared__ int64_t s_unit[kUnitSlots];  // gather units handed out (producing kernel)
  if (warp == 0) {
    // ------------------------------------------------------------ A/B TMA producer
    if (lane == 0) {
      if (!GATHER) tma_prefetch_map(&map_a);
      tma_prefetch_map(&map_b);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t issued = 0;  // bit s: stage s holds a load nobody has consumed yet (error path)
      for (int tile = unit; tile < num_items && ok; tile += units) {
        bool conv_item;
        int m_blk, n_blk;
        item_of(tile, conv_item, m_blk, n_blk);
        if (conv_item) continue;  // no tensor-core operands
        if constexpr (PRODUCE) {
          // this CTA's 128 rows of A must have been written by the gather warps
          const int m0 = m_blk * kTileM + static_cast<int>(rank) * kBM;
          if (m0 < args.N) {
            const int rows = min(kBM, args.N - m0);
            if (!wait_ready(gat.ready + m0 / kReadyTokens,
                            static_cast<uint32_t>((rows + gat.unit_tokens - 1) / gat.unit_tokens), abort)) {
              atomicOr(args.err_word, 64);
              ok = false;
              break;
            }
            // their generic-proxy writes, now visible to this thread, ordered before its TMA reads
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1u, abort)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bars->full[stage]);
          if constexpr (PAIR) {
            if (rank == 0) mbar_expect_tx(full, 2 * (kAStage + kBStage));
            const uint32_t full0 = pair_addr(full, 0);
#pragma unroll
            for (int sb = 0; sb < kSubK; ++sb) {
              tma_load_2d_pair(smem_u32(sA + stage * kAStage + sb * kABytes), &map_a, full0, (kb * kSubK + sb) * kKB,
                               m_blk * kTileM + static_cast<int>(rank) * kBM);
              tma_load_2d_pair(smem_u32(sB + stage * kBStage + sb * kBBytes), &map_b, full0, (kb * kSubK + sb) * kKB,
                               n_blk * BN + static_cast<int>(rank) * kBRows);
            }
          } else {
            mbar_expect_tx(full, GATHER ? kBBytes : kABytes + kBBytes);
            if (!GATHER) tma_load_2d(smem_u32(sA + stage * kABytes), &map_a, full, kb * kBK, m_blk * kBM);
            tma_load_2d(smem_u32(sB + stage * kBBytes), &map_b, full, kb * kBK, n_blk * BN);
          }
          issued |= 1u << stage;
          if (++stage == kSt) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Tail: wait until the MMA has released the last fill of every stage. Its commits
      // arrive asynchronously (on the other CTA of a pair too); none may land after the
      // CTA has exited. (A stage never filled passes at once.)
      for (int i = 0; ok && i < kSt; ++i) {
        if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1u, abort)) {
          ok = false;
          break;
        }
        if (++stage == kSt) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        atomicOr(args.err_word, 1);
        *abort = 1;
        // Let copies already in flight land before the CTA can exit (bounded; a pair's
        // copies count on rank 0's barriers and are waited for at the end instead).
        for (int s = 0; s < kSt; ++s)
          if (!PAIR && (issued & (1u << s))) {
            const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&bars->full[s]), par) && globaltimer() - t0 < kWaitLimitNs) {
            }
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = unit; tile < num_items && ok; tile += units) {
        if constexpr (CONV) {
          bool conv_item;
          int mb_, nb_;
          item_of(tile, conv_item, mb_, nb_);
          if (conv_item) continue;
        }
        if (!mbar_wait<PAIR>(smem_u32(&bars->tmem_empty[acc]), acc_phase ^ 1u, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait<PAIR>(smem_u32(&bars->full[stage]), phase, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int sb = 0; sb < kSubK; ++sb) {
            const uint64_t a0 = sw128_desc(smem_u32(sA + stage * kAStage + sb * kABytes));
            const uint64_t b0 = sw128_desc(smem_u32(sB + stage * kBStage + sb * kBBytes));
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)  // advance 32 bytes = 2 units (16 bf16 or 32 E4M3)
              umma_bf16<PAIR, FP8>(d_tmem, a0 + 2u * k, b0 + 2u * k, kIdesc, (kb | sb | k) != 0);
          }
          umma_commit<PAIR>(smem_u32(&bars->empty[stage]));
          if (++stage == kSt) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit<PAIR>(smem_u32(&bars->tmem_full[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        atomicOr(args.err_word, 2);
        *abort = 1;
      }
      // Every MMA this thread issued has finished before TMEM can be released.
      umma_commit_local<PAIR>(smem_u32(&bars->mma_done));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&bars->mma_done), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ epilogue operand producer
    if (lane == 0) {
      if (GATE == PG_GATE_SCALAR) tma_prefetch_map(&map_x);
      if (GATE == PG_GATE_CONTEXT) tma_prefetch_map(&map_h);
      uint32_t seq = 0;
      bool ok = true;
      uint32_t issued = 0;
      for (int tile = unit; tile < num_items && ok; tile += units) {
        bool conv_item;
        int m_blk, n_blk;
        item_of(tile, conv_item, m_blk, n_blk);
        const int n0 = n_blk * BN, m0 = m_blk * kTileM + static_cast<int>(rank) * kBM;
        const bool is_k = GATE == PG_GATE_CONTEXT && n0 >= args.d;
        if (m0 >= args.N) continue;  // this CTA's rows of the tile lie past the last token
        if (conv_item) continue;  // conv items run on the conv warps
        for (int j = 0; j < kSub; ++j, ++seq) {
          const int slot = static_cast<int>(seq % kEpiStages);
          const uint32_t ph = (seq / kEpiStages) & 1u;
          if (!mbar_wait(smem_u32(&bars->epi_empty[slot]), ph ^ 1u, abort)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bars->epi_full[slot]);
          const uint32_t dst = smem_u32(sE + slot * kEpiBytes);
          float* vec = s_vec + slot * 3 * kEpiCols;
          const uint32_t tx = (GATE == PG_GATE_SCALAR || is_k ? kEpiBytes : 0) + (is_k ? 2 * kEpiCols * 4 : 0) +
                              (FP8 ? kEpiCols * 4 : 0);
          if (tx == 0) {
            mbar_arrive(full);   // output staging only: hand the free slot over
          } else {
            mbar_expect_tx(full, tx);
            if (GATE == PG_GATE_SCALAR) tma_load_2d(dst, &map_x, full, n0 + j * kEpiCols, m0);
            if (is_k) {
              const int m = n0 / args.d - 1;
              const int kc = n0 - (m + 1) * args.d;
              tma_load_2d(dst, &map_h, full, kc + j * kEpiCols, m * args.N + m0);
              bulk_load(smem_u32(vec), args.gamma_h + kc + j * kEpiCols, kEpiCols * 4, full);
              bulk_load(smem_u32(vec + kEpiCols), args.gamma_k + kc + j * kEpiCols, kEpiCols * 4, full);
            }
            if (FP8) bulk_load(smem_u32(vec + 2 * kEpiCols), args.sw + n0 + j * kEpiCols, kEpiCols * 4, full);
            issued |= 1u << slot;
          }
        }
      }
      if (!ok) {
        atomicOr(args.err_word, 8);
        *abort = 1;
        for (int s = 0; s < kEpiStages; ++s)
          if (issued & (1u << s)) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < kWaitLimitNs / 4 &&
                   !mbar_try_wait(smem_u32(&bars->epi_full[s]), ((seq - 1 - ((seq - 1 - s) % kEpiStages)) / kEpiStages) & 1u)) {
            }
          }
      }
    }
  } else if ((GATHER && warp >= kGatherWarp0) ||
             (PRODUCE && (warp == kProdCoordWarp || warp >= kProdGatherWarp0))) {
    if constexpr (PRODUCE) {
      // ---------------------------------------------------------- e_t producers (warps 3, 8..15)
      // Warps 8..15 gather units of T tokens x `items` heads = Hu <= 512 rows of 64 bf16
      // (128 bytes), T a power of two <= 128 (a unit never spans two ready counters). Warp
      // w takes rows [64 w, 64 w + 64) of every unit: lane l hashes rows 64 w + l + 32 j
      // (token p / items, head p mod items), then 8 lanes per row move its 16-byte pieces,
      // row 64 w + 4 i + (l >> 3) being lane ((4 i + (l >> 3)) mod 32)'s pair i / 8.
      // Warp 3 coordinates through a ring of kUnitSlots slots in shared memory: unit k goes
      // into slot k mod kUnitSlots (the claim order is the order the tiles are walked: last
      // m-block first) and is announced on unit_full[slot]; every gather warp arrives on
      // unit_done[slot] once its stores of the unit are issued, after which the
      // coordinator fences, counts the unit on its ready counter and reuses the slot. The
      // coordinator also stages each unit's canonical token IDs (and the 3 before it) in its
      // slot, so a gather warp hashes from shared memory. The gather warps never wait for one
      // another: each runs its own pipeline, hashing unit k while the loads of unit k - 1 are
      // in flight. Every wait is a bounded mbarrier wait.
      const int items = gat.P.O * gat.P.H;
      const int T = gat.unit_tokens;
      const uint32_t nunits = static_cast<uint32_t>((args.N + T - 1) / T);
      if (warp == kProdCoordWarp) {
        // lane 0 claims, waits and counts; all lanes stage the canonical IDs of each unit
        // (the reads of a token happen once, here, ahead of the gather warps)
        auto publish = [&](int64_t u) {
          if (u >= 0) {
            __threadfence();
            red_release_gpu_add(gat.ready + u / kReadyTokens, 1u);
          }
        };
        bool ok = true;
        int K = 0;  // units handed out (slot K holds -1)
        uint32_t pending = 0;
        if (lane == 0) pending = atomicAdd(gat.claim, 1u);
        for (int k = 0;; ++k) {
          const int s = k % kUnitSlots;
          int64_t val = -1;
          if (lane == 0) val = (pending >= nunits || *abort) ? -1 : static_cast<int64_t>(nunits - 1 - pending) * T;
          val = __shfl_sync(0xffffffffu, val, 0);
          // token IDs of positions val - 3 .. val + T - 1 (issued before the slot is free)
          constexpr int kStage = (kCanonStride + 31) / 32;
          int32_t x[kStage];
#pragma unroll
          for (int q = 0; q < kStage; ++q) {
            const int i = lane + 32 * q;
            const int64_t f = val - 3 + i;
            x[q] = 0;
            if (val >= 0 && i < T + 3 && f >= 0 && f < args.N) x[q] = __ldg(gat.tokens + f);
          }
          if (k >= kUnitSlots) {
            // unit k - kUnitSlots: stored by every gather warp, then counted; its slot is free
            bool waited = true;
            if (lane == 0) {
              waited = mbar_wait(smem_u32(&bars->unit_done[s]),
                                                    static_cast<uint32_t>((k / kUnitSlots - 1) & 1), abort);
              if (waited) publish(s_unit[s]);
            }
            if (!__shfl_sync(0xffffffffu, waited, 0)) {
              ok = false;
              break;
            }
          }
          // canonical IDs (an out-of-range ID reads as 0 and is reported by its own unit)
#pragma unroll
          for (int q = 0; q < kStage; ++q) {
            const int i = lane + 32 * q;
            const int64_t f = val - 3 + i;
            if (val >= 0 && i < T + 3 && f >= 0 && f < args.N) {
              int32_t id = x[q];
              if (id < 0 || static_cast<uint32_t>(id) >= gat.P.vocab) {
                if (i >= 3 && gat.err) atomicMin(reinterpret_cast<unsigned int*>(gat.err), static_cast<unsigned int>(f));
                id = 0;
              }
              s_canon[s * kCanonStride + i] = gat.canon_map ? __ldg(gat.canon_map + id) : static_cast<uint32_t>(id);
            }
          }
          __syncwarp();
          if (lane == 0) {
            s_unit[s] = val;
            mbar_arrive(smem_u32(&bars->unit_full[s]));
            if (val >= 0) pending = atomicAdd(gat.claim, 1u);  // needed one unit later
          }
          if (val < 0) {
            K = k;
            break;
          }
        }
        if (lane == 0) {
          for (int j = K - kUnitSlots + 1 < 0 ? 0 : K - kUnitSlots + 1; ok && j < K; ++j) {
            const int s = j % kUnitSlots;
            if (!mbar_wait(smem_u32(&bars->unit_done[s]),
                                              static_cast<uint32_t>((j / kUnitSlots) & 1), abort)) {
              ok = false;
              break;
            }
            publish(s_unit[s]);
          }
          if (!ok) {
            atomicOr(args.err_word, 128);
            *abort = 1;
          }
        }
        __syncwarp();
      } else {
        constexpr int kPairs = 2, kLoads = 16;      // 64 rows of this warp per unit
        const int gw = warp - kProdGatherWarp0;
        const int Hu = T * items;
        const uint32_t out_row = static_cast<uint32_t>(items) * 128u;
        const int piece = lane & 7, sub = lane >> 3;
        uint32_t r[kPairs], off[kPairs];            // unit being hashed and loaded
        uint64_t sw[kPairs];
        uint32_t offp[kPairs];                      // previous unit (loaded, to be stored)
        uint64_t swp[kPairs];
        int64_t prev = -1;
        int kprev = 0;
        uint4 vb[kLoads];
        auto hash = [&](int64_t tok0, const uint32_t* cs) {
#pragma unroll
          for (int j = 0; j < kPairs; ++j) {
            const int p = 64 * gw + lane + 32 * j;
            const int s = p / items;
            r[j] = 0;
            sw[j] = 0;
            off[j] = 0xFFFFFFFFu;  // no row
            if (p < Hu && tok0 + s < args.N) {
              const int it = p - s * items;
              const int64_t tok = tok0 + s;
              const uint32_t t = fastmod(static_cast<uint32_t>(tok), gat.fm_L, gat.L);
              const uint32_t* ids = cs + 3 + s;  // ids[-j]: position tok - j
              uint64_t c[4], hs;
#pragma unroll
              for (int jj = 0; jj < 4; ++jj)
                c[jj] = (jj < s_ic[it].n && t >= static_cast<uint32_t>(jj)) ? ids[-jj] : kPad;
              r[j] = item_row_ids(s_ic[it], gat.P.mode, c, &hs);
              sw[j] = mix64(hs + kGolden);
              off[j] = static_cast<uint32_t>(s) * out_row + static_cast<uint32_t>(it) * 128u;
            }
          }
        };
        auto issue_loads = [&]() {
#pragma unroll
          for (int i = 0; i < kLoads; ++i) {
            const int src = (4 * i + sub) & 31;
            const uint32_t row = __shfl_sync(0xffffffffu, r[i / 8], src);
            const uint32_t o = __shfl_sync(0xffffffffu, off[i / 8], src);
            vb[i] = make_uint4(0, 0, 0, 0);
            if (o != 0xFFFFFFFFu) vb[i] = ldg_stream(gat.table + static_cast<uint64_t>(row) * 128u + piece * 16);
          }
        };
        // sign-flip and store the previous unit, then report it to the coordinator
        auto store_prev = [&]() {
          if (prev < 0) return;
          uint8_t* out = gat.e_out + static_cast<uint64_t>(prev) * out_row + piece * 16;
#pragma unroll
          for (int q = 0; q < kLoads; ++q) {
            const int src = (4 * q + sub) & 31;
            const uint64_t w = __shfl_sync(0xffffffffu, swp[q / 8], src);
            const uint32_t o = __shfl_sync(0xffffffffu, offp[q / 8], src);
            const uint32_t bits = static_cast<uint32_t>(w >> (8 * piece)) & 0xFFu;
            if (o != 0xFFFFFFFFu) *reinterpret_cast<uint4*>(out + o) = xor4(vb[q], bf16_sign_mask(bits));
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->unit_done[kprev % kUnitSlots]));
        };
        // unit k: hashed under the previous unit's loads, then the previous unit is stored
        // and unit k's loads are issued
        bool ok = true;
        for (int k = 0;; ++k) {
          const int s = k % kUnitSlots;
          if (!mbar_wait(smem_u32(&bars->unit_full[s]), static_cast<uint32_t>((k / kUnitSlots) & 1), abort)) {
            ok = false;
            break;
          }
          const int64_t u = s_unit[s];
          if (u < 0) break;
          hash(u, s_canon + s * kCanonStride);
          store_prev();
          issue_loads();
          prev = u;
          kprev = k;
#pragma unroll
          for (int j = 0; j < kPairs; ++j) {
            offp[j] = off[j];
            swp[j] = sw[j];
          }
        }
        if (ok) {
          store_prev();  // the last unit
        } else {
          atomicOr(args.err_word, 128);
          *abort = 1;
        }
      }
    } else if constexpr (GATHER) {
      // ---------------------------------------------------------- A-operand gather (warps 7..14)
      // Pair p of warps builds every A tile of ring stage p; warp `half` of the pair covers
      // tokens [64 half, 64 half + 64) of the 128-token block. Lane l hashes tokens l and
      // l + 32 of its half for head kb, then 8 lanes per row move 16-byte chunks: chunk
      // (token, piece) -> A-tile row `token`, physical chunk piece ^ (row & 7) (128-byte
      // swizzle, the layout the TMA would have written).
      const int gw = warp - kGatherWarp0;
      const int pair = gw >> 1, half = gw & 1;
      const int piece = lane & 7, sub = lane >> 3;
      const int stage = pair;
      // rows and sign words of tokens (64 half + lane) and (+32) of one k-block
      auto hash_rows = [&](int tile, int kb, uint32_t& ra, uint32_t& rb, uint64_t& sa, uint64_t& sb) {
        const int m0 = ((num_tiles - 1 - tile) / num_n) * kBM;
        const ItemConst& it = s_ic[kb];
        const int64_t ta = static_cast<int64_t>(m0) + 64 * half + lane, tb = ta + 32;
        uint64_t hs;
        ra = rb = 0;
        sa = sb = 0;
        if (ta < args.N) {
          ra = item_row(it, gat.P.mode, gat.tokens, gat.canon_map, gat.P.vocab, ta,
                        fastmod(static_cast<uint32_t>(ta), gat.fm_L, gat.L), gat.err, &hs);
          sa = mix64(hs + kGolden);
        }
        if (tb < args.N) {
          rb = item_row(it, gat.P.mode, gat.tokens, gat.canon_map, gat.P.vocab, tb,
                        fastmod(static_cast<uint32_t>(tb), gat.fm_L, gat.L), gat.err, &hs);
          sb = mix64(hs + kGolden);
        }
      };
      // this pair's k-blocks: sequence numbers q = pair, pair + 4, ... over the CTA's tiles
      int tile = blockIdx.x, kb = pair;
      while (kb >= num_kb && tile < num_tiles) {
        kb -= num_kb;
        tile += gridDim.x;
      }
      uint32_t q = pair;
      uint32_t ra, rb;
      uint64_t sa, sb;
      if (tile < num_tiles) hash_rows(tile, kb, ra, rb, sa, sb);
      bool ok = true;
      while (tile < num_tiles) {
        // 1. loads of this k-block (they do not need the stage to be free)
        uint4 v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int src = 4 * (i & 7) + sub;
          const uint32_t r = __shfl_sync(0xffffffffu, i < 8 ? ra : rb, src);
          v[i] = __ldg(reinterpret_cast<const uint4*>(gat.table + static_cast<uint64_t>(r) * 128u + piece * 16));
        }
        // 2. hash the next k-block of this pair while the loads are in flight
        int ntile = tile, nkb = kb + 4;
        while (nkb >= num_kb && ntile < num_tiles) {
          nkb -= num_kb;
          ntile += gridDim.x;
        }
        uint32_t na = 0, nb = 0;
        uint64_t nsa = 0, nsb = 0;
        if (ntile < num_tiles) hash_rows(ntile, nkb, na, nb, nsa, nsb);
        // 3. wait for the stage, then sign-flip and store into the swizzled A tile
        if (!mbar_wait(smem_u32(&bars->empty[stage]), ((q >> 2) & 1u) ^ 1u, abort)) {
          ok = false;
          break;
        }
        uint8_t* a_tile = sA + stage * kAStage;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int src = 4 * (i & 7) + sub;
          const uint64_t sw = __shfl_sync(0xffffffffu, i < 8 ? sa : sb, src);
          const uint32_t bits = static_cast<uint32_t>(sw >> (8 * piece)) & 0xFFu;
          const int row = 64 * half + (i < 8 ? 0 : 32) + src;
          *reinterpret_cast<uint4*>(a_tile + row * 128 + ((piece ^ (row & 7)) << 4)) = xor4(v[i], bf16_sign_mask(bits));
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&bars->full[stage]));
        tile = ntile;
        kb = nkb;
        q += 4;
        ra = na;
        rb = nb;
        sa = nsa;
        sb = nsb;
      }
      if (!ok) {
        atomicOr(args.err_word, 16);
        *abort = 1;
      }
    }
  } else if (CONV && warp >= kConvWarp0) {
    if constexpr (CONV) {
      // ------------------------------------------------------------ conv warps (7..11)
      // The conv items of the pair's work list, in order. Warp 11's lane 0 streams each
      // item's 16 sub-tiles of 16 columns (H of the branch, v of the item's rows and of the
      // causal halo before them, the packed taps) through a kConvStages-deep ring once the
      // item's m-blocks are published, and writes every updated sub-tile of H back; warps
      // 7..10 (thread = row) first form the item's alpha and tap factors from the partial
      // sums, then update the sub-tiles in place with pg_conv_residual's arithmetic.
      const int tpbk = args.d / BN;
      constexpr int kSubs = BN / kConvCols;  // sub-tiles per conv item
      auto sw32 = [](int row, int chunk) -> uint32_t {  // 32-byte rows, 32-byte swizzle
        return static_cast<uint32_t>(row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4));
      };
      if (warp == kConvWarp0 + kConvCompute / 32) {
        if (lane == 0) {
          tma_prefetch_map(&map_h3);
          tma_prefetch_map(&map_x);
          if (args.halo > 0) tma_prefetch_map(&map_vh);
          uint32_t k = 0;  // conv sub-tiles issued
          bool ok = true;
          int st_r0[kConvStages], st_br[kConvStages], st_col[kConvStages];
          for (int tile = unit; tile < num_items && ok; tile += units) {
            bool cv;
            int m_blk, n_blk;
            item_of(tile, cv, m_blk, n_blk);
            if (!cv) continue;
            const int r0 = m_blk * kTileM + static_cast<int>(rank) * kBM;
            if (r0 >= args.N) continue;  // (the compute warps skip the same items)
            const int br = n_blk / tpbk, cb = n_blk - br * tpbk;
            // v of this m-block and of the one before is written by this launch's v tiles
            if (!wait_ready(args.done + m_blk, 2u * num_n, abort) ||
                (m_blk > 0 && !wait_ready(args.done + m_blk - 1, 2u * num_n, abort))) {
              atomicOr(args.err_word, kErrConvWait);
              ok = false;
              break;
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
            for (int j = 0; j < kSubs; ++j, ++k) {
              const int s = static_cast<int>(k % kConvStages);
              const uint32_t use = k / kConvStages;
              uint8_t* stg = s_conv + s * kConvStageBytes;
              if (use > 0) {
                // the compute warps are done with the sub-tile this stage held: write it back,
                // and let the store read the stage before it is refilled
                if (!mbar_wait(smem_u32(&bars->cdone[s]), (use - 1) & 1u, abort)) {
                  ok = false;
                  break;
                }
                tma_store_3d(&map_h3, smem_u32(stg), st_col[s], st_r0[s], st_br[s]);
                bulk_commit();
                bulk_wait_read_all();
              }
              const uint32_t full = smem_u32(&bars->cfull[s]);
              const int col = cb * BN + j * kConvCols;
              mbar_expect_tx(full, 2 * kConvTileBytes + args.halo * kConvCols * 2 + kConvTapBytes);
              tma_load_3d(smem_u32(stg), &map_h3, full, col, r0, br);
              tma_load_2d(smem_u32(stg + kConvTileBytes), &map_x, full, col, r0);
              if (args.halo > 0) tma_load_2d(smem_u32(stg + 2 * kConvTileBytes), &map_vh, full, col, r0 - args.halo);
              bulk_load(smem_u32(stg + 2 * kConvTileBytes + kConvHaloBytes), args.conv_taps + (col / 2) * 4,
                        kConvTapBytes, full);
              st_r0[s] = r0;
              st_br[s] = br;
              st_col[s] = col;
            }
          }
          // the last fills: written back once computed
          for (uint32_t q = k > kConvStages ? k - kConvStages : 0; ok && q < k; ++q) {
            const int s = static_cast<int>(q % kConvStages);
            if (!mbar_wait(smem_u32(&bars->cdone[s]), (q / kConvStages) & 1u, abort)) {
              ok = false;
              break;
            }
            tma_store_3d(&map_h3, smem_u32(s_conv + s * kConvStageBytes), st_col[s], st_r0[s], st_br[s]);
            bulk_commit();
          }
          bulk_wait_all();
          if (!ok) {
            atomicOr(args.err_word, 32);
            *abort = 1;
            // let the loads already issued land before the CTA can exit (bounded)
            for (uint32_t q = k > kConvStages ? k - kConvStages : 0; q < k; ++q) {
              const uint64_t t0 = globaltimer();
              while (!mbar_try_wait(smem_u32(&bars->cfull[q % kConvStages]), (q / kConvStages) & 1u) &&
                     globaltimer() - t0 < kWaitLimitNs / 4) {
              }
            }
          }
        }
      } else {
        const int cth = threadIdx.x - 32 * kConvWarp0;
        const int ct = cth & (kBM - 1);  // this thread's row of the item
        const int chunk = cth >> 7;      // and its 8 columns of every 16-column sub-tile
        const int halo = args.halo, dil = args.dil, ks = args.ks;
        uint32_t k = 0, sync_phase = 0;
        int cbuf = 0;
        bool ok = true;
        for (int tile = unit; tile < num_items && ok; tile += units) {
          bool cv;
          int m_blk, n_blk;
          item_of(tile, cv, m_blk, n_blk);
          if (!cv) continue;
          const int r0 = m_blk * kTileM + static_cast<int>(rank) * kBM;
          if (r0 >= args.N) continue;
          const int br = n_blk / tpbk;
          // the partial sums of this m-block and of the one before are complete
          if (!wait_ready(args.done + m_blk, 2u * num_n, abort) ||
              (m_blk > 0 && !wait_ready(args.done + m_blk - 1, 2u * num_n, abort))) {
            atomicOr(args.err_word, kErrConvWait);
            ok = false;
            break;
          }
          // alpha and the tap factor f = alpha / sqrt(alpha^2 mean(v^2) + eps) of the rows
          // [r0 - halo, r0 + 128), formed as the alpha finalize and pg_conv_residual form them;
          // the items of column block 0 also write alpha and mean(v^2) out
          const int cb = n_blk - br * tpbk;
          float* cf = s_cf + cbuf * kConvRows;
          float* ca = s_ca + cbuf * kConvRows;
          cbuf ^= 1;
          for (int i = cth; i < kBM + halo; i += kConvCompute) {
            const int p = r0 - halo + i;
            float a = 0.f, f = 0.f;
            if (p >= 0 && p < args.N) {
              a = gate_alpha(args.partials, br, tpbk, args.N, args.d, args.eps, p);
              const float ms = row_mean_sq(args.vpart, tpbk, args.N, args.d, p);
              f = tap_scale(a, ms, args.eps);
              if (cb == 0 && i >= halo) {
                args.alpha_out[static_cast<size_t>(br) * args.N + p] = a;
                if (br == 0 && args.v_ms_out) args.v_ms_out[p] = ms;
              }
            }
            cf[i] = f;
            ca[i] = a;
          }
          mbar_arrive(smem_u32(&bars->conv_sync));
          if (!mbar_wait(smem_u32(&bars->conv_sync), sync_phase, abort)) {
            ok = false;
            break;
          }
          sync_phase ^= 1u;
          // this thread's row t: its four tap factors (zero before the start of its sequence
          // and past the kernel size) and alpha_t
          const int tpos = (r0 + ct) % args.L;
          bool tap_ok[4];
          float fj[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            tap_ok[jj] = jj < ks && tpos >= jj * dil;
            fj[jj] = tap_ok[jj] ? cf[halo + ct - jj * dil] : 0.f;
          }
          const uint64_t f0 = pk(fj[0], fj[0]), f1 = pk(fj[1], fj[1]), f2 = pk(fj[2], fj[2]), f3 = pk(fj[3], fj[3]);
          const float at = ca[halo + ct];
          const uint64_t aa = pk(at, at);
          for (int j = 0; j < kSubs; ++j, ++k) {
            const int s = static_cast<int>(k % kConvStages);
            if (!mbar_wait(smem_u32(&bars->cfull[s]), (k / kConvStages) & 1u, abort)) {
              ok = false;
              break;
            }
            uint8_t* stg = s_conv + s * kConvStageBytes;  // H, overwritten by H + Y
            const uint8_t* vs = stg + kConvTileBytes;     // v of the item's rows
            const uint8_t* vh = stg + 2 * kConvTileBytes;  // v of the halo rows
            const uint64_t* taps = reinterpret_cast<const uint64_t*>(stg + 2 * kConvTileBytes + kConvHaloBytes);
            {
              const int c = chunk;  // 16-byte chunk c: columns 8c .. 8c + 7 of the sub-tile
              uint4 vr[4];
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int rr = ct - jj * dil;
                if (!tap_ok[jj])
                  vr[jj] = make_uint4(0, 0, 0, 0);
                else if (rr >= 0)
                  vr[jj] = *reinterpret_cast<const uint4*>(vs + sw32(rr, c));
                else
                  vr[jj] = *reinterpret_cast<const uint4*>(vh + (halo + rr) * (kConvCols * 2) + c * 16);
              }
              float h[8];
              unpack_bf16x8(*reinterpret_cast<const uint4*>(stg + sw32(ct, c)), h);
              const uint32_t vw[4][4] = {{vr[0].x, vr[0].y, vr[0].z, vr[0].w}, {vr[1].x, vr[1].y, vr[1].z, vr[1].w},
                                         {vr[2].x, vr[2].y, vr[2].z, vr[2].w}, {vr[3].x, vr[3].y, vr[3].z, vr[3].w}};
#pragma unroll
              for (int q = 0; q < 4; ++q) {  // columns 8c + 2q, 8c + 2q + 1
                const uint64_t* wq = taps + (4 * c + q) * 4;
                uint64_t prod[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) prod[jj] = mul2(wq[jj], bf16x2_as_f2(vw[jj][q]));
                uint64_t cc = mul2(f0, prod[0]);  // c / 2
                cc = fma2(f1, prod[1], cc);
                cc = fma2(f2, prod[2], cc);
                cc = fma2(f3, prod[3], cc);
                const uint64_t accv = fma2(aa, bf16x2_as_f2(vw[0][q]), pk(h[2 * q], h[2 * q + 1]));  // H + alpha v_t
                upk(silu2_add<__nv_bfloat16>(cc, accv), h[2 * q], h[2 * q + 1]);
              }
              *reinterpret_cast<uint4*>(stg + sw32(ct, c)) =
                  make_uint4(pack_bf16(h[0], h[1]), pack_bf16(h[2], h[3]), pack_bf16(h[4], h[5]), pack_bf16(h[6], h[7]));
            }
            fence_proxy_async_smem();  // the stage's H is read next by the TMA store
            mbar_arrive(smem_u32(&bars->cdone[s]));
          }
        }
        if (!ok) {
          atomicOr(args.err_word, 32);
          *abort = 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 3..6; 4..7 when PRODUCE)
    const int epi = threadIdx.x - 32 * (PRODUCE ? kProdEpiWarp0 : 3);
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row_in_tile = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t seq = 0;
    bool ok = true;
    int pending = -1;             // slot whose TMA store may still be reading (thread epi == 0)
    const int tpb = args.d / BN;  // tiles per branch (context gate)
    uint32_t pub_phase = 0;  // CONV: tile publication barrier
    for (int tile = unit; tile < num_items && ok; tile += units) {
      bool conv_item;
      int m_blk, n_blk;
      item_of(tile, conv_item, m_blk, n_blk);
      if (conv_item) continue;  // conv items run on the conv warps
      if (!mbar_wait(smem_u32(&bars->tmem_full[acc]), acc_phase, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int m0 = m_blk * kTileM + static_cast<int>(rank) * kBM;
      const bool rows_here = m0 < args.N;  // (the operand producer skips the same tiles)
      const int row = m0 + row_in_tile;
      const bool live = row < args.N;
      const int n0 = n_blk * BN;
      const bool is_k = GATE == PG_GATE_CONTEXT && n0 >= args.d;
      const int m_br = is_k ? n0 / args.d - 1 : 0;
      const int kc = is_k ? n0 - (m_br + 1) * args.d : 0;
      const uint32_t t_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
      // context gate, k tiles: sums over the row's columns of g h k, k^2 and h^2 (g = gamma_h
      // gamma_k), as fp32 pairs (even, odd column) in two interleaved sets; FP8: k without the
      // row scale s_e, which multiplies the sums once at the end
      uint64_t a_hk[2] = {0ull, 0ull}, a_kk[2] = {0ull, 0ull}, a_hh[2] = {0ull, 0ull};
      float s_vv = 0.f;  // context gate, v tiles: sum of the stored (bf16) v^2 of the row
      for (int j = 0; rows_here && j < kSub; ++j, ++seq) {
        const int slot = static_cast<int>(seq % kEpiStages);
        const uint32_t ph = (seq / kEpiStages) & 1u;
        if (!mbar_wait(smem_u32(&bars->epi_full[slot]), ph, abort)) {
          ok = false;
          break;
        }
        uint32_t r[32];
        tmem_ld32(t_base + static_cast<uint32_t>(j * kEpiCols), r);
        tmem_ld_wait();
        const float* vec = s_vec + slot * 3 * kEpiCols;
        if constexpr (FP8) {
          const float4* sc = reinterpret_cast<const float4*>(vec + 2 * kEpiCols);  // s_w of the columns
          if (is_k) {  // s_w[col] here, s_e[row] on the finished sums
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 c4 = sc[q];
              r[4 * q + 0] = __float_as_uint(__uint_as_float(r[4 * q + 0]) * c4.x);
              r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) * c4.y);
              r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) * c4.z);
              r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) * c4.w);
            }
          } else {
          // out = s_e[row] s_w[col] sum_k q_e q_w
          const float sr = live ? __ldg(args.sa + row) : 0.f;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 c4 = sc[q];
            r[4 * q + 0] = __float_as_uint(__uint_as_float(r[4 * q + 0]) * sr * c4.x);
            r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) * sr * c4.y);
            r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) * sr * c4.z);
            r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) * sr * c4.w);
          }
          }
        }
        uint8_t* slot_p = sE + slot * kEpiBytes;
        if (is_k) {
          const float4* gh = reinterpret_cast<const float4*>(vec);
          const float4* gk = reinterpret_cast<const float4*>(vec + kEpiCols);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 hw = *reinterpret_cast<const uint4*>(slot_p + epi_offset(row_in_tile, c));
            const float4 gh0 = gh[2 * c], gh1 = gh[2 * c + 1];
            const float4 gk0 = gk[2 * c], gk1 = gk[2 * c + 1];
            const uint64_t g2[4] = {f2_mul(f2_pack(gh0.x, gh0.y), f2_pack(gk0.x, gk0.y)),
                                    f2_mul(f2_pack(gh0.z, gh0.w), f2_pack(gk0.z, gk0.w)),
                                    f2_mul(f2_pack(gh1.x, gh1.y), f2_pack(gk1.x, gk1.y)),
                                    f2_mul(f2_pack(gh1.z, gh1.w), f2_pack(gk1.z, gk1.w))};
            const uint64_t h2[4] = {bf16x2_as_f2(hw.x), bf16x2_as_f2(hw.y), bf16x2_as_f2(hw.z), bf16x2_as_f2(hw.w)};
            const int set = c & 1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint64_t k2 = f2_pack(__uint_as_float(r[8 * c + 2 * i]), __uint_as_float(r[8 * c + 2 * i + 1]));
              a_kk[set] = f2_fma(k2, k2, a_kk[set]);
              a_hh[set] = f2_fma(h2[i], h2[i], a_hh[set]);
              a_hk[set] = f2_fma(f2_mul(g2[i], h2[i]), k2, a_hk[set]);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4* p = reinterpret_cast<uint4*>(slot_p + epi_offset(row_in_tile, c));
            float o[8];
            if (GATE == PG_GATE_SCALAR) {
              float xf[8];
              unpack_bf16x8(*p, xf);
#pragma unroll
              for (int i = 0; i < 8; ++i) o[i] = fmaf(args.g, __uint_as_float(r[8 * c + i]), xf[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) o[i] = __uint_as_float(r[8 * c + i]);
            }
            const uint4 packed = make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]),
                                            pack_bf16(o[6], o[7]));
            *p = packed;
            if (GATE == PG_GATE_CONTEXT) {
              float q[8];
              unpack_bf16x8(packed, q);
#pragma unroll
              for (int i = 0; i < 8; ++i) s_vv = fmaf(q[i], q[i], s_vv);
            }
          }
          fence_proxy_async_smem();
        }
        mbar_arrive(smem_u32(&bars->epi_done[slot]));
        if (epi == 0) {
          // the slot goes back to the producer once every thread is done with it and,
          // for outputs, once its TMA store has read it
          if (!mbar_wait(smem_u32(&bars->epi_done[slot]), ph, abort)) {
            ok = false;
            break;
          }
          if (!is_k) {
            tma_store_2d(&map_v, smem_u32(slot_p), n0 + j * kEpiCols, m0);
            bulk_commit();
            if (pending >= 0) {   // one store stays in flight; the one before it is done reading
              bulk_wait_read_all_but_one();
              mbar_arrive(smem_u32(&bars->epi_empty[pending]));
            }
            pending = slot;
          } else {
            if (pending >= 0) {
              bulk_wait_read_all();
              mbar_arrive(smem_u32(&bars->epi_empty[pending]));
              pending = -1;
            }
            mbar_arrive(smem_u32(&bars->epi_empty[slot]));
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      if constexpr (PAIR)
        mbar_arrive_cluster(pair_addr(smem_u32(&bars->tmem_empty[acc]), 0));
      else
        mbar_arrive(smem_u32(&bars->tmem_empty[acc]));
      if (is_k && live) {
        const float2 hk0 = f2_unpack(a_hk[0]), hk1 = f2_unpack(a_hk[1]);
        const float2 kk0 = f2_unpack(a_kk[0]), kk1 = f2_unpack(a_kk[1]);
        const float2 hh0 = f2_unpack(a_hh[0]), hh1 = f2_unpack(a_hh[1]);
        float s_hk = (hk0.x + hk0.y) + (hk1.x + hk1.y);
        float s_kk = (kk0.x + kk0.y) + (kk1.x + kk1.y);
        const float s_hh = (hh0.x + hh0.y) + (hh1.x + hh1.y);
        if constexpr (FP8) {
          const float sr = __ldg(args.sa + row);
          s_hk *= sr;
          s_kk *= sr * sr;
        }
        float* p = args.partials + (static_cast<size_t>(m_br * tpb + kc / BN) * 3) * args.N + row;
        p[0] = s_hk;
        p[args.N] = s_kk;
        p[2 * static_cast<size_t>(args.N)] = s_hh;
      }
      if (GATE == PG_GATE_CONTEXT && !is_k && live && args.vpart)
        args.vpart[static_cast<size_t>(n0 / BN) * args.N + row] = s_vv;
      if constexpr (CONV) {
        // publish this CTA's share of the tile on its m-block's counter once its partial
        // sums are visible and its v stores complete
        __threadfence();
        mbar_arrive(smem_u32(&bars->pub));
        if (epi == 0) {
          if (!mbar_wait(smem_u32(&bars->pub), pub_phase, abort)) {
            ok = false;
          } else {
            bulk_wait_all();
            if (pending >= 0) {
              mbar_arrive(smem_u32(&bars->epi_empty[pending]));
              pending = -1;
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
            red_release_gpu_add(args.done + m_blk, 1u);
          }
        }
        pub_phase ^= 1u;
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      atomicOr(args.err_word, 4);
      *abort = 1;
    }
    if (epi == 0) {
      bulk_wait_all();
      if (pending >= 0) mbar_arrive(smem_u32(&bars->epi_empty[pending]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // After an error, copies this CTA issued may still be landing: they count on rank 0's
    // barriers, so give them time (bounded) before the pair can leave.
    if (threadIdx.x == 0 && *abort) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 2000000ull) {
      }
    }
    __syncthreads();
    cluster_sync();  // no CTA leaves while the other may still reach its shared memory or TMEM
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem, kTmemCols);
  }
}

// The conv taps with the RMSNorm gain and SiLU's half-argument folded in, as pg_conv_residual
// forms them: out[p][j] = (w[c, j] gamma_c[c] / 2, w[c + 1, j] gamma_c[c + 1] / 2), c = 2p,
// zero for j >= kernel_size.
__global__ void __launch_bounds__(256) conv_taps_kernel(const float* __restrict__ conv_w,
                                                        const float* __restrict__ gamma_c, int d, int ks,
                                                        uint64_t* __restrict__ out) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (d / 2) * 4) return;
  const int p = idx >> 2, j = idx & 3;
  const int c0 = 2 * p, c1 = 2 * p + 1;
  const float g0 = 0.5f * gamma_c[c0], g1 = 0.5f * gamma_c[c1];
  const float w0 = j < ks ? conv_w[c0 * ks + j] * g0 : 0.f;
  const float w1 = j < ks ? conv_w[c1 * ks + j] * g1 : 0.f;
  out[idx] = pk(w0, w1);
}

// alpha[m, t] from the per-tile partial sums (summed in tile order: deterministic).
// With vpart, threads of branch 0 also write mean(v^2) of their row (tile order: deterministic).
__global__ void __launch_bounds__(256) alpha_finalize_kernel(const float* __restrict__ partials, int M,
                                                             int tpb, int N, int d, float eps,
                                                             float* __restrict__ alpha,
                                                             const float* __restrict__ vpart,
                                                             float* __restrict__ v_ms) {
  const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (idx >= static_cast<int64_t>(M) * N) return;
  const int m = static_cast<int>(idx / N);
  const int row = static_cast<int>(idx - static_cast<int64_t>(m) * N);
  if (vpart && m == 0) v_ms[row] = row_mean_sq(vpart, tpb, N, d, row);
  alpha[idx] = gate_alpha(partials, m, tpb, N, d, eps, row);
}

// The same for few rows (N <= kFinalizeWarpRows): one warp per (branch, row), lane l adding
// tiles l, l + 32, ... and an xor tree the lanes' sums (fixed order: deterministic), so the
// partials' round trips run side by side instead of one after another.
constexpr int kFinalizeWarpRows = 64;

__global__ void __launch_bounds__(256) alpha_finalize_warp_kernel(const float* __restrict__ partials, int M,
                                                                  int tpb, int N, int d, float eps,
                                                                  float* __restrict__ alpha,
                                                                  const float* __restrict__ vpart,
                                                                  float* __restrict__ v_ms) {
  const int64_t w = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<int64_t>(M) * N) return;  // whole warps
  const int m = static_cast<int>(w / N);
  const int row = static_cast<int>(w - static_cast<int64_t>(m) * N);
  const bool with_v = vpart && m == 0;
  float s_hk = 0.f, s_kk = 0.f, s_hh = 0.f, s_vv = 0.f;
  for (int tb = lane; tb < tpb; tb += 32) {
    const float* p = partials + (static_cast<size_t>(m * tpb + tb) * 3) * N + row;
    s_hk += p[0];
    s_kk += p[N];
    s_hh += p[2 * static_cast<size_t>(N)];
    if (with_v) s_vv += vpart[static_cast<size_t>(tb) * N + row];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s_hk += __shfl_xor_sync(0xffffffffu, s_hk, o);
    s_kk += __shfl_xor_sync(0xffffffffu, s_kk, o);
    s_hh += __shfl_xor_sync(0xffffffffu, s_hh, o);
    s_vv += __shfl_xor_sync(0xffffffffu, s_vv, o);
  }
  if (lane != 0) return;
  if (with_v) v_ms[row] = s_vv / static_cast<float>(d);
  const float inv_d = 1.0f / static_cast<float>(d);
  const float rh = sqrtf(s_hh * inv_d + eps);
  const float rk = sqrtf(s_kk * inv_d + eps);
  const float s = s_hk / (rh * rk * sqrtf(static_cast<float>(d)));
  alpha[w] = 1.0f / (1.0f + expf(-s));
}

// alpha (and mean(v^2)) from the per-tile sums: a thread per (branch, row), or a warp for few rows.
pg_status launch_alpha_finalize(const float* partials, int M, int tpb, int N, int d, float eps, float* alpha,
                                const float* vpart, float* v_ms, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(M) * N;
  if (N <= kFinalizeWarpRows)
    alpha_finalize_warp_kernel<<<static_cast<unsigned>((total * 32 + 255) / 256), 256, 0, stream>>>(
        partials, M, tpb, N, d, eps, alpha, vpart, v_ms);
  else
    alpha_finalize_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, stream>>>(
        partials, M, tpb, N, d, eps, alpha, vpart, v_ms);
  return after_launch(1);
}

// ==================================================================== host side

// 2-D bf16 (bytes1: 1-byte elements, E4M3) tensor [rows, cols] (row-major), box [box_rows, box_cols].
bool make_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swizzle, bool bytes1 = false) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (bytes1 ? 1 : 2)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, bytes1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor [z, rows, cols] (row-major), box [1, box_rows, box_cols]: rows clipped per z.
bool make_map_3d(CUtensorMap* map, const void* ptr, uint64_t zs, uint64_t rows, uint64_t cols, uint32_t box_cols,
                 uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, zs};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct GemmPtrs {
  const void* e;
  const void* W;
  const void* x;
  const void* h;
  void* v;
};

template <int BN, int GATE, bool GATHER = false, bool PAIR = false, bool PRODUCE = false, bool FP8 = false,
          bool CONV = false>
pg_status launch_tc(const GemmPtrs& ptr, const GemmArgs& a, cudaStream_t stream,
                    const typename GatherParam<GATHER || PRODUCE>::type& gat = {}) {
  CUtensorMap ma, mb, mx, mh, mv, mh3, mvh;
  constexpr uint32_t kBox = FP8 ? 2 * kBK : kBK;  // a 128-byte row of elements
  if ((!GATHER && !make_map(&ma, ptr.e, a.N, a.Din, kBox, kBM, CU_TENSOR_MAP_SWIZZLE_128B, FP8)) ||
      !make_map(&mb, ptr.W, a.Dcols, a.Din, kBox, PAIR ? BN / 2 : BN, CU_TENSOR_MAP_SWIZZLE_128B, FP8) ||
      !make_map(&mv, ptr.v, a.N, a.d, kEpiCols, kBM, CU_TENSOR_MAP_SWIZZLE_64B))
    return PG_ERR_UNSUPPORTED;
  // maps that this launch does not use alias the output map (never read)
  if (GATHER) ma = mv;
  mx = mv;
  mh = mv;
  if (GATE == PG_GATE_SCALAR && !make_map(&mx, ptr.x, a.N, a.d, kEpiCols, kBM, CU_TENSOR_MAP_SWIZZLE_64B))
    return PG_ERR_UNSUPPORTED;
  if (GATE == PG_GATE_CONTEXT &&
      !make_map(&mh, ptr.h, static_cast<uint64_t>(a.M) * a.N, a.d, kEpiCols, kBM, CU_TENSOR_MAP_SWIZZLE_64B))
    return PG_ERR_UNSUPPORTED;
  mh3 = mv;
  mvh = mv;
  if (CONV) {  // the conv warps' tiles: H per branch (stores clipped at each branch's last row), v, v's halo
    if (!make_map_3d(&mh3, ptr.h, a.M, a.N, a.d, kConvCols, kBM, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map(&mx, ptr.v, a.N, a.d, kConvCols, kBM, CU_TENSOR_MAP_SWIZZLE_32B))
      return PG_ERR_UNSUPPORTED;
    if (a.halo > 0 && !make_map(&mvh, ptr.v, a.N, a.d, kConvCols, a.halo, CU_TENSOR_MAP_SWIZZLE_NONE))
      return PG_ERR_UNSUPPORTED;
  }
  auto kern = tc_gemm_kernel<BN, GATE, GATHER, PAIR, PRODUCE, FP8, CONV>;
  constexpr size_t smem = gemm_smem_bytes<BN, GATHER, PAIR, PRODUCE, GATE == PG_GATE_CONTEXT || FP8, CONV>();
  static_assert(smem <= 232448, "dynamic shared memory above the 227 KB a CTA may hold");
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return cuda_fail(err);
  if constexpr (PAIR) {
    // persistent: one CTA pair per co-resident cluster slot, at most one per 256 x BN tile
    const int mblocks = (a.N + 2 * kBM - 1) / (2 * kBM);
    const int tiles = mblocks * (a.Dcols / BN) + (CONV ? mblocks * a.M * (a.d / BN) : 0);  // work items
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2u * static_cast<unsigned>(tiles));
    cfg.blockDim = dim3(PRODUCE ? kProduceThreads : CONV ? kConvThreads : kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int slots = 0;
    err = cudaOccupancyMaxActiveClusters(&slots, kern, &cfg);
    if (err != cudaSuccess) return cuda_fail(err);
    if (slots < 1) return PG_ERR_DEVICE;
    const int clusters = tiles < slots ? tiles : slots;
    cfg.gridDim = dim3(2u * static_cast<unsigned>(clusters));
    err = cudaLaunchKernelEx(&cfg, kern, ma, mb, mx, mh, mv, a, gat, mh3, mvh);
    if (err != cudaSuccess) return cuda_fail(err);
    return after_launch(1);
  }
  const int tiles = ((a.N + kBM - 1) / kBM) * (a.Dcols / BN);
  const int grid = tiles < sm_count() ? tiles : sm_count();
  kern<<<grid, GATHER ? kFusedThreads : kGemmThreads, smem, stream>>>(ma, mb, mx, mh, mv, a, gat, mh3, mvh);
  return after_launch(1);
}

template <int BN, bool PAIR>
pg_status dispatch_tc(int gate, const GemmPtrs& ptr, const GemmArgs& a, cudaStream_t stream) {
  if (gate == PG_GATE_NONE) return launch_tc<BN, PG_GATE_NONE, false, PAIR>(ptr, a, stream);
  if (gate == PG_GATE_SCALAR) return launch_tc<BN, PG_GATE_SCALAR, false, PAIR>(ptr, a, stream);
  return launch_tc<BN, PG_GATE_CONTEXT, false, PAIR>(ptr, a, stream);
}

pg_status dispatch_fp8(int gate, const GemmPtrs& ptr, const GemmArgs& a, cudaStream_t stream) {
  if (gate == PG_GATE_NONE) return launch_tc<256, PG_GATE_NONE, false, true, false, true>(ptr, a, stream);
  if (gate == PG_GATE_SCALAR) return launch_tc<256, PG_GATE_SCALAR, false, true, false, true>(ptr, a, stream);
  return launch_tc<256, PG_GATE_CONTEXT, false, true, false, true>(ptr, a, stream);
}

pg_status dispatch_produce(int gate, const GemmPtrs& ptr, const GemmArgs& a, const FusedGather& gat,
                           cudaStream_t stream) {
  if (gate == PG_GATE_NONE) return launch_tc<256, PG_GATE_NONE, false, true, true>(ptr, a, stream, gat);
  if (gate == PG_GATE_SCALAR) return launch_tc<256, PG_GATE_SCALAR, false, true, true>(ptr, a, stream, gat);
  return launch_tc<256, PG_GATE_CONTEXT, false, true, true>(ptr, a, stream, gat);
}

template <int BN>
pg_status dispatch_fused(int gate, const GemmPtrs& ptr, const GemmArgs& a, const FusedGather& gat,
                         cudaStream_t stream) {
  if (gate == PG_GATE_NONE) return launch_tc<BN, PG_GATE_NONE, true>(ptr, a, stream, gat);
  if (gate == PG_GATE_SCALAR) return launch_tc<BN, PG_GATE_SCALAR, true>(ptr, a, stream, gat);
  return launch_tc<BN, PG_GATE_CONTEXT, true>(ptr, a, stream, gat);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Context-gate workspace: per-(branch, tile) partial sums [M][d/BN][3][N], then, when
// mean(v^2) is requested, the v tiles' row sums of v^2 [d/BN][N].
// Scratch of the context gate's per-row tile sums: [M, d / BN, 3, N] (+ [d / BN, N] for
// v_ms). The tensor-core kernels sum per BN-column tile; the size query (query = true)
// also covers the few-rows kernel's 64-column tiles (up to kSmallRowsUsed rows).
size_t context_workspace(int64_t N, int d, int M, bool with_v_ms, bool query = false) {
  const int bn = (d % 256 == 0) ? 256 : 128;
  const size_t tiles = static_cast<size_t>(
      query && N <= kSmallRowsUsed && d % kSmallTile == 0 ? d / kSmallTile : d / bn);
  return (static_cast<size_t>(M) * tiles * 3 + (with_v_ms ? tiles : 0)) * static_cast<size_t>(N) * sizeof(float);
}

}  // namespace
}  // namespace pg

extern "C" {

pg_status pg_project_gate_workspace_size(int32_t N, int32_t Din, int32_t d, int32_t M, int32_t dtype,
                                         int32_t gate_kind, size_t* bytes) {
  if (!bytes) return PG_ERR_NULL;
  if (N < 0 || Din < 1 || d < 1 || M < 0) return PG_ERR_SHAPE;
  *bytes = 0;
  if (gate_kind == PG_GATE_CONTEXT && dtype == PG_BF16) *bytes = pg::context_workspace(N, d, M, true, true);
  return PG_OK;
}

pg_status pg_project_gate(int32_t N, int32_t Din, int32_t d, int32_t M, int32_t dtype, const void* e,
                          const void* W, int32_t gate_kind, float g, const void* x_resid, const void* h,
                          const float* gamma_h, const float* gamma_k, float eps, void* v_out,
                          float* alpha_out, float* v_ms_out, void* workspace, size_t workspace_bytes,
                          pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (N < 0 || Din < 1 || d < 1 || M < 0) return PG_ERR_SHAPE;
  if (gate_kind < PG_GATE_NONE || gate_kind > PG_GATE_CONTEXT) return PG_ERR_SHAPE;
  if (dtype != PG_F32 && dtype != PG_BF16) return PG_ERR_DTYPE;
  if (gate_kind != PG_GATE_CONTEXT && M != 0) return PG_ERR_SHAPE;
  if (gate_kind == PG_GATE_CONTEXT && M < 1) return PG_ERR_SHAPE;
  if (N == 0) return PG_OK;
  if (!e || !v_out) return PG_ERR_NULL;
  if (gate_kind == PG_GATE_SCALAR && !x_resid) return PG_ERR_NULL;
  if (gate_kind == PG_GATE_CONTEXT && (!W || !h || !gamma_h || !gamma_k || !alpha_out)) return PG_ERR_NULL;
  if (!aligned16(e) || !aligned16(v_out) || (x_resid && !aligned16(x_resid))) return PG_ERR_ALIGN;
  if (static_cast<int64_t>(N) * (d > Din ? d : Din) >= (1ll << 40)) return PG_ERR_SHAPE;
  if (sm_count() == 0) return cuda_fail(cudaGetLastError());

  if (!W) {  // identity projection: a flat table's e_t is already d wide
    if (Din != d) return PG_ERR_SHAPE;
    if (d % 8) return PG_ERR_UNSUPPORTED;
    return launch_identity_gate(static_cast<int64_t>(N) * d, dtype, gate_kind, e, x_resid, g, v_out, stream);
  }

  if (dtype == PG_F32) {
    if (gate_kind == PG_GATE_CONTEXT) return PG_ERR_UNSUPPORTED;
    return launch_simt_f32(N, Din, d, gate_kind, static_cast<const float*>(e), static_cast<const float*>(W), g,
                           static_cast<const float*>(x_resid), static_cast<float*>(v_out), stream);
  }

  // bf16 tensor-core path
  if (device_cc() != 103 && device_cc() != 100) return PG_ERR_DEVICE;
  if (Din % kBK != 0 || d % 128 != 0) return PG_ERR_UNSUPPORTED;
  if (!aligned16(W) || (h && !aligned16(h))) return PG_ERR_ALIGN;
  if (use_small_rows(N, Din)) {
    // a few rows (decode): W streamed over every SM by the SIMT kernel; the context gate
    // takes it when the workspace holds its 64-column tile sums (what the size query gives)
    if (gate_kind != PG_GATE_CONTEXT)
      return launch_small_rows_bf16(N, Din, d, M, gate_kind, e, W, g, x_resid, h, gamma_h, gamma_k, v_out, nullptr,
                                    nullptr, stream);
    const size_t tiles = static_cast<size_t>(d / kSmallTile);
    const size_t need = (static_cast<size_t>(M) * tiles * 3 + (v_ms_out ? tiles : 0)) * static_cast<size_t>(N) * 4;
    if (workspace && workspace_bytes >= need && aligned16(workspace) && aligned16(gamma_h) && aligned16(gamma_k)) {
      float* part = static_cast<float*>(workspace);
      float* vpart = v_ms_out ? part + static_cast<size_t>(M) * tiles * 3 * static_cast<size_t>(N) : nullptr;
      pg_status st = launch_small_rows_bf16(N, Din, d, M, gate_kind, e, W, g, x_resid, h, gamma_h, gamma_k, v_out,
                                            part, vpart, stream);
      if (st != PG_OK) return st;
      return launch_alpha_finalize(part, M, static_cast<int>(tiles), N, d, eps, alpha_out, vpart, v_ms_out, stream);
    }
  }
  const int bn = (d % 256 == 0) ? 256 : 128;
  GemmArgs a;
  a.N = N;
  a.Din = Din;
  a.Dcols = (gate_kind == PG_GATE_CONTEXT ? (1 + M) : 1) * d;
  a.d = d;
  a.M = M;
  a.g = g;
  a.gamma_h = gamma_h;
  a.gamma_k = gamma_k;
  a.partials = static_cast<float*>(workspace);
  a.vpart = (gate_kind == PG_GATE_CONTEXT && v_ms_out)
                ? static_cast<float*>(workspace) + static_cast<size_t>(M) * (d / bn) * 3 * static_cast<size_t>(N)
                : nullptr;
  if (gate_kind == PG_GATE_CONTEXT && static_cast<int64_t>(M) * N >= (1ll << 31)) return PG_ERR_SHAPE;
  const GemmPtrs ptrs{e, W, x_resid, h, v_out};
  a.err_word = device_error_word();
  a.sa = a.sw = nullptr;
  if (!a.err_word) return cuda_fail(cudaGetLastError());
  if (gate_kind == PG_GATE_CONTEXT) {
    const size_t need = context_workspace(N, d, M, v_ms_out != nullptr);
    if (!workspace || workspace_bytes < need) return PG_ERR_WORKSPACE;
    if (!aligned16(workspace) || !aligned16(gamma_h) || !aligned16(gamma_k)) return PG_ERR_ALIGN;
  }
  // 256-column tiles run on CTA pairs (256 x 256 per pair), 128-column ones on single CTAs
  pg_status st = bn == 256 ? dispatch_tc<256, true>(gate_kind, ptrs, a, stream)
                           : dispatch_tc<128, false>(gate_kind, ptrs, a, stream);
  if (st != PG_OK || gate_kind != PG_GATE_CONTEXT) return st;
  return launch_alpha_finalize(a.partials, M, d / bn, N, d, eps, alpha_out, a.vpart, v_ms_out, stream);
}


pg_status pg_project_gate_conv_workspace_size(int32_t N, int32_t d, int32_t M, size_t* bytes) {
  if (!bytes) return PG_ERR_NULL;
  if (N < 0 || d < 1 || M < 1) return PG_ERR_SHAPE;
  const size_t sync = (static_cast<size_t>((N + 255) / 256) * sizeof(uint32_t) + 255) / 256 * 256;
  const size_t taps = (static_cast<size_t>(d / 2) * 4 * sizeof(uint64_t) + 255) / 256 * 256;
  *bytes = sync + taps + pg::context_workspace(N, d, M, true);
  return PG_OK;
}

pg_status pg_project_gate_conv(int32_t B, int32_t L, int32_t Din, int32_t d, int32_t M, const void* e,
                               const void* W, void* H, const float* gamma_h, const float* gamma_k,
                               const float* gamma_c, const float* conv_w, int32_t kernel_size, int32_t dilation,
                               float eps, void* v_out, float* alpha_out, float* v_ms_out, void* workspace,
                               size_t workspace_bytes, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B < 0 || L < 1 || Din < 1 || d < 1 || M < 1) return PG_ERR_SHAPE;
  if (kernel_size < 1 || kernel_size > 4 || dilation < 1 || dilation > 8) return PG_ERR_SHAPE;
  const int64_t N64 = static_cast<int64_t>(B) * L;
  if (N64 >= (1ll << 31)) return PG_ERR_SHAPE;
  const int N = static_cast<int>(N64);
  if (N == 0) return PG_OK;
  if (!e || !W || !H || !gamma_h || !gamma_k || !gamma_c || !conv_w || !v_out || !alpha_out || !workspace)
    return PG_ERR_NULL;
  if (Din % kBK != 0 || d % 256 != 0) return PG_ERR_UNSUPPORTED;
  if (!aligned16(e) || !aligned16(W) || !aligned16(H) || !aligned16(v_out) || !aligned16(gamma_h) ||
      !aligned16(gamma_k) || !aligned16(gamma_c) || !aligned16(conv_w) || !aligned16(workspace) ||
      reinterpret_cast<uintptr_t>(alpha_out) % 4 || reinterpret_cast<uintptr_t>(v_ms_out) % 4)
    return PG_ERR_ALIGN;
  if (static_cast<int64_t>(N) * (d > Din ? d : Din) >= (1ll << 40)) return PG_ERR_SHAPE;
  if (static_cast<int64_t>(M) * N >= (1ll << 31)) return PG_ERR_SHAPE;
  size_t need = 0;
  pg_status st = pg_project_gate_conv_workspace_size(N, d, M, &need);
  if (st != PG_OK) return st;
  if (workspace_bytes < need) return PG_ERR_WORKSPACE;
  if (sm_count() == 0) return cuda_fail(cudaGetLastError());
  if (device_cc() != 103 && device_cc() != 100) return PG_ERR_DEVICE;
  constexpr int bn = 256;
  const size_t sync = (static_cast<size_t>((N + 255) / 256) * sizeof(uint32_t) + 255) / 256 * 256;
  const size_t taps_bytes = need - sync - context_workspace(N, d, M, true);
  GemmArgs a;
  a.N = N;
  a.Din = Din;
  a.Dcols = (1 + M) * d;
  a.d = d;
  a.M = M;
  a.g = 0.f;
  a.gamma_h = gamma_h;
  a.gamma_k = gamma_k;
  a.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + sync + taps_bytes);
  a.vpart = a.partials + static_cast<size_t>(M) * (d / bn) * 3 * static_cast<size_t>(N);
  a.sa = a.sw = nullptr;
  a.err_word = device_error_word();
  if (!a.err_word) return cuda_fail(cudaGetLastError());
  a.done = static_cast<uint32_t*>(workspace);
  uint64_t* taps = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(workspace) + sync);
  a.conv_taps = taps;
  a.alpha_out = alpha_out;
  a.v_ms_out = v_ms_out;
  a.eps = eps;
  a.L = L;
  a.ks = kernel_size;
  a.dil = dilation;
  a.halo = (kernel_size - 1) * dilation;
  if (a.halo > kConvMaxHalo) return PG_ERR_UNSUPPORTED;
  cudaError_t err = cudaMemsetAsync(workspace, 0, sync, stream);  // the m-blocks' counters
  if (err != cudaSuccess) return cuda_fail(err);
  const int ntaps = (d / 2) * 4;
  conv_taps_kernel<<<(ntaps + 255) / 256, 256, 0, stream>>>(conv_w, gamma_c, d, kernel_size, taps);
  st = after_launch(1);
  if (st != PG_OK) return st;
  const GemmPtrs ptrs{e, W, nullptr, H, v_out};
  return launch_tc<256, PG_GATE_CONTEXT, false, true, false, false, true>(ptrs, a, stream);
}

pg_status pg_project_gate_fp8(int32_t N, int32_t Din, int32_t d, int32_t M, const void* e_q, const float* e_scale,
                              const void* W_q, const float* W_scale, int32_t gate_kind, float g,
                              const void* x_resid, const void* h, const float* gamma_h, const float* gamma_k,
                              float eps, void* v_out, float* alpha_out, float* v_ms_out, void* workspace,
                              size_t workspace_bytes, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (N < 0 || Din < 1 || d < 1 || M < 0) return PG_ERR_SHAPE;
  if (gate_kind < PG_GATE_NONE || gate_kind > PG_GATE_CONTEXT) return PG_ERR_SHAPE;
  if (gate_kind != PG_GATE_CONTEXT && M != 0) return PG_ERR_SHAPE;
  if (gate_kind == PG_GATE_CONTEXT && M < 1) return PG_ERR_SHAPE;
  if (N == 0) return PG_OK;
  if (!e_q || !e_scale || !W_q || !W_scale || !v_out) return PG_ERR_NULL;
  if (gate_kind == PG_GATE_SCALAR && !x_resid) return PG_ERR_NULL;
  if (gate_kind == PG_GATE_CONTEXT && (!h || !gamma_h || !gamma_k || !alpha_out)) return PG_ERR_NULL;
  if (Din % (4 * kBK) != 0 || d % 256 != 0) return PG_ERR_UNSUPPORTED;  // stages of two 128-byte k-blocks
  if (!aligned16(e_q) || !aligned16(W_q) || !aligned16(v_out) || !aligned16(W_scale) ||
      (reinterpret_cast<uintptr_t>(e_scale) % 4) || (x_resid && !aligned16(x_resid)) || (h && !aligned16(h)))
    return PG_ERR_ALIGN;
  if (static_cast<int64_t>(N) * (d > Din ? d : Din) >= (1ll << 40)) return PG_ERR_SHAPE;
  if (gate_kind == PG_GATE_CONTEXT && static_cast<int64_t>(M) * N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (sm_count() == 0) return cuda_fail(cudaGetLastError());
  if (device_cc() != 103 && device_cc() != 100) return PG_ERR_DEVICE;
  constexpr int bn = 256;
  GemmArgs a;
  a.N = N;
  a.Din = Din;
  a.Dcols = (gate_kind == PG_GATE_CONTEXT ? (1 + M) : 1) * d;
  a.d = d;
  a.M = M;
  a.g = g;
  a.gamma_h = gamma_h;
  a.gamma_k = gamma_k;
  a.partials = static_cast<float*>(workspace);
  a.vpart = (gate_kind == PG_GATE_CONTEXT && v_ms_out)
                ? static_cast<float*>(workspace) + static_cast<size_t>(M) * (d / bn) * 3 * static_cast<size_t>(N)
                : nullptr;
  a.err_word = device_error_word();
  if (!a.err_word) return cuda_fail(cudaGetLastError());
  a.sa = e_scale;
  a.sw = W_scale;
  if (gate_kind == PG_GATE_CONTEXT) {
    const size_t need = context_workspace(N, d, M, v_ms_out != nullptr);
    if (!workspace || workspace_bytes < need) return PG_ERR_WORKSPACE;
    if (!aligned16(workspace) || !aligned16(gamma_h) || !aligned16(gamma_k)) return PG_ERR_ALIGN;
  }
  const GemmPtrs ptrs{e_q, W_q, x_resid, h, v_out};
  pg_status st = dispatch_fp8(gate_kind, ptrs, a, stream);
  if (st != PG_OK || gate_kind != PG_GATE_CONTEXT) return st;
  return launch_alpha_finalize(a.partials, M, d / bn, N, d, eps, alpha_out, a.vpart, v_ms_out, stream);
}

}  // extern "C"

// ==================================================================== fused lookup + projection

extern "C" pg_status pg_lookup_project_gate(const pg_table_desc* desc, const int32_t* tokens, int32_t B,
                                            int32_t L, const uint32_t* canon_map, const void* table,
                                            uint64_t table_bytes, int32_t d, int32_t M, const void* W,
                                            int32_t gate_kind, float g, const void* x_resid, const void* h,
                                            const float* gamma_h, const float* gamma_k, float eps, void* v_out,
                                            float* alpha_out, void* workspace, size_t workspace_bytes,
                                            int32_t* err_index, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  Geometry geo;
  pg_status st = validate_desc(desc, &geo);
  if (st != PG_OK) return st;
  if (desc->hash_kind != PG_HASH_MULXOR || desc->mode == PG_FLAT) return PG_ERR_UNSUPPORTED;
  if (desc->row_dtype != PG_BF16 || desc->r != kBK) return PG_ERR_UNSUPPORTED;
  const int items = geo.O * geo.H;
  if (items > kFusedItems) return PG_ERR_UNSUPPORTED;
  if (B < 0 || L < 0 || d < 1 || M < 0) return PG_ERR_SHAPE;
  if (gate_kind < PG_GATE_NONE || gate_kind > PG_GATE_CONTEXT) return PG_ERR_SHAPE;
  if (gate_kind != PG_GATE_CONTEXT && M != 0) return PG_ERR_SHAPE;
  if (gate_kind == PG_GATE_CONTEXT && M < 1) return PG_ERR_SHAPE;
  const int64_t N = static_cast<int64_t>(B) * L;
  if (N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (N == 0) return PG_OK;
  if (!tokens || !table || !W || !v_out) return PG_ERR_NULL;
  if (gate_kind == PG_GATE_SCALAR && !x_resid) return PG_ERR_NULL;
  if (gate_kind == PG_GATE_CONTEXT && (!h || !gamma_h || !gamma_k || !alpha_out)) return PG_ERR_NULL;
  if (table_bytes < geo.rows * geo.row_bytes) return PG_ERR_RANGE;
  if (!aligned16(table) || !aligned16(W) || !aligned16(v_out) || (x_resid && !aligned16(x_resid)) ||
      (h && !aligned16(h)))
    return PG_ERR_ALIGN;
  if (d % 128 != 0) return PG_ERR_UNSUPPORTED;
  if (gate_kind == PG_GATE_CONTEXT && static_cast<int64_t>(M) * N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (sm_count() == 0) return cuda_fail(cudaGetLastError());
  if (device_cc() != 103 && device_cc() != 100) return PG_ERR_DEVICE;
  const int din = items * kBK;
  if (gate_kind == PG_GATE_CONTEXT) {
    size_t need = 0;
    pg_project_gate_workspace_size(static_cast<int32_t>(N), din, d, M, PG_BF16, gate_kind, &need);
    if (!workspace || workspace_bytes < need) return PG_ERR_WORKSPACE;
    if (!aligned16(workspace) || !aligned16(gamma_h) || !aligned16(gamma_k)) return PG_ERR_ALIGN;
  }
  if (err_index) {
    if (reinterpret_cast<uintptr_t>(err_index) % 4) return PG_ERR_ALIGN;
    cudaError_t e = cudaMemsetAsync(err_index, 0xFF, sizeof(int32_t), stream);  // reads as -1
    if (e != cudaSuccess) return cuda_fail(e);
  }
  const int bn = (d % 256 == 0) ? 256 : 128;
  GemmArgs a;
  a.N = static_cast<int>(N);
  a.Din = din;
  a.Dcols = (gate_kind == PG_GATE_CONTEXT ? (1 + M) : 1) * d;
  a.d = d;
  a.M = M;
  a.g = g;
  a.gamma_h = gamma_h;
  a.gamma_k = gamma_k;
  a.partials = static_cast<float*>(workspace);
  a.vpart = nullptr;
  a.err_word = device_error_word();
  a.sa = a.sw = nullptr;
  if (!a.err_word) return cuda_fail(cudaGetLastError());
  FusedGather gat;
  fill_hash_params(desc, geo, &gat.P);
  gat.seed = desc->hash_seed;
  gat.tokens = tokens;
  gat.canon_map = canon_map;
  gat.table = static_cast<const uint8_t*>(table);
  gat.L = static_cast<uint32_t>(L);
  gat.fm_L = fastmod_constant(gat.L);
  gat.err = err_index;
  const GemmPtrs ptrs{nullptr, W, x_resid, h, v_out};
  st = bn == 256 ? dispatch_fused<256>(gate_kind, ptrs, a, gat, stream)
                 : dispatch_fused<128>(gate_kind, ptrs, a, gat, stream);
  if (st != PG_OK || gate_kind != PG_GATE_CONTEXT) return st;
  return launch_alpha_finalize(a.partials, M, d / bn, static_cast<int>(N), d, eps, alpha_out, nullptr, nullptr, stream);
}

// ==================================================================== lookup + projection, one launch

namespace pg {
namespace {

// Head of pg_gather_project_gate's workspace: the chunk claim counter, then one ready
// counter per 128-token block, zeroed by the call before its launch.
size_t produce_sync_bytes(int64_t N) {
  const size_t b = static_cast<size_t>(1 + (N + kReadyTokens - 1) / kReadyTokens) * sizeof(uint32_t);
  return (b + 255) / 256 * 256;
}

}  // namespace
}  // namespace pg

extern "C" pg_status pg_gather_project_gate_workspace_size(int32_t N, int32_t d, int32_t M, int32_t gate_kind,
                                                          size_t* bytes) {
  if (!bytes) return PG_ERR_NULL;
  if (N < 0 || d < 1 || M < 0) return PG_ERR_SHAPE;
  *bytes = pg::produce_sync_bytes(N) + (gate_kind == PG_GATE_CONTEXT ? pg::context_workspace(N, d, M, true, true) : 0);
  return PG_OK;
}

extern "C" pg_status pg_gather_project_gate(const pg_table_desc* desc, const int32_t* tokens, int32_t B,
                                            int32_t L, const uint32_t* canon_map, const void* table,
                                            uint64_t table_bytes, void* e_out, int32_t d, int32_t M,
                                            const void* W, int32_t gate_kind, float g, const void* x_resid,
                                            const void* h, const float* gamma_h, const float* gamma_k, float eps,
                                            void* v_out, float* alpha_out, float* v_ms_out, void* workspace,
                                            size_t workspace_bytes, int32_t* err_index, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  Geometry geo;
  pg_status st = validate_desc(desc, &geo);
  if (st != PG_OK) return st;
  if (desc->hash_kind != PG_HASH_MULXOR || desc->mode == PG_FLAT) return PG_ERR_UNSUPPORTED;
  if (desc->row_dtype != PG_BF16 || desc->r != kBK) return PG_ERR_UNSUPPORTED;
  const int items = geo.O * geo.H;
  if (items > kFusedItems) return PG_ERR_UNSUPPORTED;
  if (B < 0 || L < 0 || d < 1 || M < 0) return PG_ERR_SHAPE;
  if (gate_kind < PG_GATE_NONE || gate_kind > PG_GATE_CONTEXT) return PG_ERR_SHAPE;
  if (gate_kind != PG_GATE_CONTEXT && M != 0) return PG_ERR_SHAPE;
  if (gate_kind == PG_GATE_CONTEXT && M < 1) return PG_ERR_SHAPE;
  const int64_t N = static_cast<int64_t>(B) * L;
  if (N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (N == 0) return PG_OK;
  if (!tokens || !table || !W || !v_out || !e_out || !workspace) return PG_ERR_NULL;
  if (gate_kind == PG_GATE_SCALAR && !x_resid) return PG_ERR_NULL;
  if (gate_kind == PG_GATE_CONTEXT && (!h || !gamma_h || !gamma_k || !alpha_out)) return PG_ERR_NULL;
  if (table_bytes < geo.rows * geo.row_bytes) return PG_ERR_RANGE;
  if (!aligned16(table) || !aligned16(W) || !aligned16(v_out) || !aligned16(e_out) || !aligned16(workspace) ||
      (x_resid && !aligned16(x_resid)) || (h && !aligned16(h)))
    return PG_ERR_ALIGN;
  if (d % 256 != 0) return PG_ERR_UNSUPPORTED;
  if (gate_kind == PG_GATE_CONTEXT && static_cast<int64_t>(M) * N >= (1ll << 31)) return PG_ERR_SHAPE;
  if (sm_count() == 0) return cuda_fail(cudaGetLastError());
  if (device_cc() != 103 && device_cc() != 100) return PG_ERR_DEVICE;
  size_t need = 0;
  pg_gather_project_gate_workspace_size(static_cast<int32_t>(N), d, M, gate_kind, &need);
  if (workspace_bytes < need) return PG_ERR_WORKSPACE;
  if (gate_kind == PG_GATE_CONTEXT && (!aligned16(gamma_h) || !aligned16(gamma_k))) return PG_ERR_ALIGN;
  const size_t sync_bytes = produce_sync_bytes(N);
  if (use_small_rows(N, items * kBK)) {
    // a few rows (decode batches): the two calls themselves, whose projection then runs on
    // the few-rows kernel; the persistent producing grid would hold a tile of 256 rows
    st = pg_gather_sign_concat(desc, tokens, B, L, canon_map, table, table_bytes, e_out, PG_BF16, err_index,
                               stream_);
    if (st != PG_OK) return st;
    return pg_project_gate(static_cast<int32_t>(N), items * kBK, d, M, PG_BF16, e_out, W, gate_kind, g, x_resid, h,
                           gamma_h, gamma_k, eps, v_out, alpha_out, v_ms_out,
                           static_cast<uint8_t*>(workspace) + sync_bytes, workspace_bytes - sync_bytes, stream_);
  }
  if (err_index) {
    if (reinterpret_cast<uintptr_t>(err_index) % 4) return PG_ERR_ALIGN;
    cudaError_t e = cudaMemsetAsync(err_index, 0xFF, sizeof(int32_t), stream);  // reads as -1
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cudaError_t e = cudaMemsetAsync(workspace, 0, sync_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  constexpr int bn = 256;
  GemmArgs a;
  a.N = static_cast<int>(N);
  a.Din = items * kBK;
  a.Dcols = (gate_kind == PG_GATE_CONTEXT ? (1 + M) : 1) * d;
  a.d = d;
  a.M = M;
  a.g = g;
  a.gamma_h = gamma_h;
  a.gamma_k = gamma_k;
  a.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + sync_bytes);
  a.vpart = (gate_kind == PG_GATE_CONTEXT && v_ms_out)
                ? a.partials + static_cast<size_t>(M) * (d / bn) * 3 * static_cast<size_t>(N)
                : nullptr;
  a.err_word = device_error_word();
  a.sa = a.sw = nullptr;
  if (!a.err_word) return cuda_fail(cudaGetLastError());
  FusedGather gat;
  fill_hash_params(desc, geo, &gat.P);
  gat.seed = desc->hash_seed;
  gat.tokens = tokens;
  gat.canon_map = canon_map;
  gat.table = static_cast<const uint8_t*>(table);
  gat.L = static_cast<uint32_t>(L);
  gat.fm_L = fastmod_constant(gat.L);
  gat.err = err_index;
  gat.e_out = static_cast<uint8_t*>(e_out);
  gat.unit_tokens = 1;
  while (2 * gat.unit_tokens * items <= kUnitRows && 2 * gat.unit_tokens <= kReadyTokens) gat.unit_tokens *= 2;
  gat.claim = static_cast<uint32_t*>(workspace);
  gat.ready = static_cast<uint32_t*>(workspace) + 1;
  const GemmPtrs ptrs{e_out, W, x_resid, h, v_out};
  st = dispatch_produce(gate_kind, ptrs, a, gat, stream);
  if (st != PG_OK || gate_kind != PG_GATE_CONTEXT) return st;
  return launch_alpha_finalize(a.partials, M, d / bn, static_cast<int>(N), d, eps, alpha_out, a.vpart, v_ms_out, stream);
}

// ==================================================================== self-test of the bounded waits

extern "C" pg_status pg_selftest_bounded_waits(uint32_t* zero_word, pg_stream_t stream) {
  if (!zero_word) return PG_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(zero_word) % 4) return PG_ERR_ALIGN;
  int* err = pg::device_error_word();
  if (!err) return pg::cuda_fail(cudaGetLastError());
  cudaError_t e = cudaMemsetAsync(zero_word, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return pg::cuda_fail(e);
  pg::wait_selftest_kernel<<<1, 32, 0, stream>>>(zero_word, err);
  return pg::after_launch(1);
}

// ==================================================================== no-allocation variant

namespace pg {
namespace {

// Scratch of pg_project_gate_context_noalloc: per-row partial sums of the context
// gate. Device code never names it; host code passes its per-device address.
static __device__ __align__(256) float g_noalloc_scratch[PG_NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int kScratchDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kScratchDevices];

// Device address of the scratch array on the current device (looked up once per device).
pg_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= kScratchDevices) return PG_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (err != cudaSuccess) return cuda_fail(err);
    g_noalloc_addr[dev] = ptr;
  }
  *out = g_noalloc_addr[dev];
  return PG_OK;
}

}  // namespace
}  // namespace pg

extern "C" pg_status pg_project_gate_context_noalloc(int32_t N, int32_t Din, int32_t d, int32_t M,
                                                     const void* e, const void* W, const void* h,
                                                     const float* gamma_h, const float* gamma_k, float eps,
                                                     void* v_out, float* alpha_out, pg_stream_t stream) {
  size_t need = 0;
  pg_status st = pg_project_gate_workspace_size(N, Din, d, M, PG_BF16, PG_GATE_CONTEXT, &need);
  if (st != PG_OK) return st;
  need = pg::context_workspace(N, d, M, false);  // this entry point does not return mean(v^2)
  if (need > PG_NOALLOC_SCRATCH_BYTES) return PG_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  st = pg::noalloc_scratch(&scratch);
  if (st != PG_OK) return st;
  return pg_project_gate(N, Din, d, M, PG_BF16, e, W, PG_GATE_CONTEXT, 0.0f, nullptr, h, gamma_h, gamma_k,
                         eps, v_out, alpha_out, nullptr, scratch, PG_NOALLOC_SCRATCH_BYTES, stream);
}

namespace pg {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace pg
