// Correlated-collision counts over distinct n-grams (sm_103a).
//
// PageGram report 3.2: two n-grams hashed to one page collide on a given head with
// probability 1/S, so a pair colliding on head 0 shares (K - 1)/S further heads on average
// (0.467 at S = 15, measured in section 6.1), against about 1/M_{n,k} per head for
// independent Engram-style subtables. pg_collision_counts counts, over n distinct n-grams
// of one order, the unordered pairs sharing their head-0 row and, per head k, the pairs
// sharing head 0 and head k:
//   1. histogram of the head-0 rows (atomics);
//   2. exclusive scan of the histogram (tiles of 4096 counters: tile sums, one block scans
//      the sums, each tile then scans its counters from its offset) -> bucket offsets;
//   3. scatter of the n-gram indices into their buckets (atomic cursors);
//   4. per (head k, bucket): every pair of the bucket compared on head k; a warp holds 32
//      buckets of one head, sums its counts and adds them with one atomic.
// The counts are integers and do not depend on the order a bucket was filled in.
//
// pg_row_copy (diagnostic): the rows a lookup reads, moved and nothing else, to measure
// what that access pattern costs on its own.
#include <algorithm>

#include "pg_internal.cuh"

namespace pg {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kScanPer = 4;
constexpr int kScanTile = kScanThreads * kScanPer;  // counters per scan tile
constexpr uint32_t kGroupMax = 1024;                // largest head-0 group compared pairwise
constexpr uint64_t kAlign = 256;

uint64_t up(uint64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
  uint64_t cursor, off, tile_sum, tile_off, idx, total;
};

WsLayout ws_layout(int64_t n, uint32_t span) {
  const uint64_t tiles = (static_cast<uint64_t>(span) + kScanTile - 1) / kScanTile;
  WsLayout L;
  L.cursor = 0;
  L.off = L.cursor + up(4ull * span);
  L.tile_sum = L.off + up(4ull * (static_cast<uint64_t>(span) + 1));
  L.tile_off = L.tile_sum + up(4ull * tiles);
  L.idx = L.tile_off + up(4ull * tiles);
  L.total = L.idx + up(4ull * static_cast<uint64_t>(n));
  return L;
}

__global__ void hist_kernel(const uint32_t* __restrict__ rows, int64_t n, int64_t stride, uint32_t lo,
                            uint32_t span, uint32_t* __restrict__ cnt, int* err_word) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t r0 = rows[i * stride] - lo;  // below lo wraps to a value >= span
    if (r0 < span) atomicAdd(cnt + r0, 1u);
    else if (err_word) atomicOr(err_word, 1024);
  }
}

// Exclusive prefix of x over the block (blockDim.x == kScanThreads) and the block's total.
__device__ uint32_t block_exclusive_scan(uint32_t x, uint32_t* total) {
  __shared__ uint32_t s_warp[kScanThreads / 32];
  __shared__ uint32_t s_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = s_warp[lane];
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    s_warp[lane] = wi - w;
    if (lane == 31) s_total = wi;
  }
  __syncthreads();
  const uint32_t r = s_warp[warp] + incl - x;
  *total = s_total;
  __syncthreads();  // the shared words are reused by the caller's next scan
  return r;
}

__global__ void __launch_bounds__(kScanThreads) tile_sum_kernel(const uint32_t* __restrict__ cnt, uint32_t span,
                                                                 uint32_t* __restrict__ tile_sum) {
  const uint64_t base = static_cast<uint64_t>(blockIdx.x) * kScanTile + threadIdx.x * kScanPer;
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < kScanPer; ++i)
    if (base + i < span) s += cnt[base + i];
  uint32_t total;
  block_exclusive_scan(s, &total);
  if (threadIdx.x == 0) tile_sum[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads) tile_offset_kernel(const uint32_t* __restrict__ tile_sum,
                                                                    uint32_t tiles, uint32_t* __restrict__ tile_off,
                                                                    uint32_t* __restrict__ off, uint32_t span) {
  uint32_t carry = 0;
  for (uint32_t base = 0; base < tiles; base += kScanThreads) {
    const uint32_t i = base + threadIdx.x;
    const uint32_t x = i < tiles ? tile_sum[i] : 0u;
    uint32_t total;
    const uint32_t ex = block_exclusive_scan(x, &total);
    if (i < tiles) tile_off[i] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) off[span] = carry;
}

// off[r] = first slot of bucket r; the histogram's counters become the scatter cursors.
__global__ void __launch_bounds__(kScanThreads) tile_apply_kernel(uint32_t* __restrict__ cnt, uint32_t span,
                                                                   const uint32_t* __restrict__ tile_off,
                                                                   uint32_t* __restrict__ off) {
  const uint64_t base = static_cast<uint64_t>(blockIdx.x) * kScanTile + threadIdx.x * kScanPer;
  uint32_t c[kScanPer], s = 0;
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    c[i] = base + i < span ? cnt[base + i] : 0u;
    s += c[i];
  }
  uint32_t total;
  uint32_t at = tile_off[blockIdx.x] + block_exclusive_scan(s, &total);
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    if (base + i < span) {
      off[base + i] = at;
      cnt[base + i] = at;
    }
    at += c[i];
  }
}

__global__ void scatter_kernel(const uint32_t* __restrict__ rows, int64_t n, int64_t stride, uint32_t lo,
                               uint32_t span, uint32_t* __restrict__ cursor, uint32_t* __restrict__ idx) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t r0 = rows[i * stride] - lo;
    if (r0 < span) idx[atomicAdd(cursor + r0, 1u)] = static_cast<uint32_t>(i);
  }
}

// Item (k, r) = head k of bucket r, items k * span32 + r: the 32 items of a warp share k
// (span32 is a multiple of 32 and the grid stride a multiple of 32), so every lane of a
// warp runs the same number of loop trips and the warp's sum goes to counts[k] at once.
__global__ void pair_kernel(const uint32_t* __restrict__ rows, int64_t stride, int K, uint32_t span,
                            uint64_t span32, const uint32_t* __restrict__ off, const uint32_t* __restrict__ idx,
                            unsigned long long* __restrict__ counts, int* err_word) {
  const int lane = threadIdx.x & 31;
  const uint64_t items = static_cast<uint64_t>(K) * span32;
  for (uint64_t item = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; item < items;
       item += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(item / span32);
    const uint64_t r = item - static_cast<uint64_t>(k) * span32;
    unsigned long long c = 0;
    if (r < span) {
      const uint32_t s = off[r], e = off[r + 1];
      const uint32_t g = e - s;
      if (g > kGroupMax) {
        if (k == 0 && err_word) atomicOr(err_word, 1024);
      } else if (g >= 2) {
        if (k == 0) {
          c = static_cast<unsigned long long>(g) * (g - 1) / 2;
        } else {
          for (uint32_t a = s; a + 1 < e; ++a) {
            const uint32_t ra = rows[static_cast<int64_t>(idx[a]) * stride + k];
            for (uint32_t b2 = a + 1; b2 < e; ++b2) c += ra == rows[static_cast<int64_t>(idx[b2]) * stride + k];
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0 && c) atomicAdd(counts + k, c);
  }
}

// ---------------------------------------------------------------- row copy (diagnostic)

// Output row i holds ocpr 16-byte chunks: the first cpr are the 16-byte-aligned window that
// holds row rows[i] of the table, the rest zeros (so the written bytes can match a lookup's
// output row); window chunks not wholly inside the table are written as zeros.
// Consecutive threads take consecutive output chunks (a warp: 512 contiguous bytes, rows
// read with the lookup kernels' 16-byte non-L1-allocating loads); kCopyUnroll chunks per
// thread in flight. c / ocpr by Lemire's direct division (ocpr_div = ceil(2^64 / ocpr),
// exact for 32-bit c; ocpr == 1 takes c itself). chunks < 2^31, so base + kCopyUnroll
// threads' strides stays below 2^32.
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(256) row_copy_kernel(const uint8_t* __restrict__ table, uint64_t table_bytes,
                                                       uint32_t row_bytes, uint32_t cpr, uint32_t ocpr,
                                                       uint64_t ocpr_div, const uint32_t* __restrict__ rows,
                                                       uint32_t chunks, uint8_t* __restrict__ out) {
  const uint32_t nthreads = gridDim.x * blockDim.x;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < chunks; base += nthreads * kCopyUnroll) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const uint32_t c = base + u * nthreads;
      v[u] = make_uint4(0, 0, 0, 0);
      if (c < chunks) {
        const uint32_t i = ocpr == 1 ? c : static_cast<uint32_t>(__umul64hi(ocpr_div, c));  // c / ocpr
        const uint32_t piece = c - i * ocpr;
        if (piece < cpr) {
          const uint64_t at = (static_cast<uint64_t>(rows[i]) * row_bytes & ~15ull) + 16ull * piece;
          if (at + 16 <= table_bytes) {
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                         : "l"(table + at));
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const uint32_t c = base + u * nthreads;
      if (c < chunks) *reinterpret_cast<uint4*>(out + 16ull * c) = v[u];
    }
  }
}

}  // namespace
}  // namespace pg

extern "C" {

pg_status pg_row_copy_window(uint32_t row_bytes, uint32_t* window_bytes) {
  if (!window_bytes) return PG_ERR_NULL;
  if (row_bytes == 0 || row_bytes > 4096) return PG_ERR_SHAPE;
  // a row starts at a multiple of gcd(row_bytes, 16) within its first chunk
  uint32_t g = 16;
  while (row_bytes % g) g >>= 1;
  *window_bytes = (row_bytes + (16 - g) + 15) / 16 * 16;
  return PG_OK;
}

pg_status pg_row_copy(const void* table, uint64_t table_bytes, uint32_t row_bytes, const uint32_t* rows, int64_t n,
                      void* out, uint32_t out_row_bytes, pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint32_t wb = 0;
  pg_status st = pg_row_copy_window(row_bytes, &wb);
  if (st != PG_OK) return st;
  if (out_row_bytes == 0) out_row_bytes = wb;
  if (out_row_bytes < wb || out_row_bytes % 16 || out_row_bytes > 65536) return PG_ERR_SHAPE;
  const uint32_t cpr = wb / 16, ocpr = out_row_bytes / 16;
  if (n < 0 || static_cast<uint64_t>(n) * ocpr >= (1ull << 31)) return PG_ERR_SHAPE;
  if (n == 0) return PG_OK;
  if (!table || !rows || !out) return PG_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(table) % 16 || reinterpret_cast<uintptr_t>(out) % 16 ||
      reinterpret_cast<uintptr_t>(rows) % 4)
    return PG_ERR_ALIGN;
  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, row_copy_kernel, 256, 0);
  if (e != cudaSuccess) return cuda_fail(e);
  const uint32_t chunks = static_cast<uint32_t>(n * ocpr);
  const int64_t want = (static_cast<int64_t>(chunks) + 255) / 256;
  const int64_t cap = static_cast<int64_t>(nsm) * std::max(per_sm, 1);
  const int grid = static_cast<int>(std::min(want, cap));
  row_copy_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(table), table_bytes, row_bytes, cpr, ocpr,
                                            ~0ull / ocpr + 1ull, rows, chunks, static_cast<uint8_t*>(out));
  return after_launch(1);
}

pg_status pg_collision_counts_workspace_size(int64_t n, uint32_t row0_span, size_t* bytes) {
  if (!bytes) return PG_ERR_NULL;
  if (n < 0 || n >= (1ll << 31) || row0_span == 0) return PG_ERR_SHAPE;
  *bytes = static_cast<size_t>(pg::ws_layout(n, row0_span).total);
  return PG_OK;
}

pg_status pg_collision_counts(const uint32_t* rows, int64_t n, int32_t K, int64_t stride, uint32_t row0_lo,
                              uint32_t row0_span, uint64_t* counts_out, void* workspace, size_t workspace_bytes,
                              pg_stream_t stream_) {
  using namespace pg;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (n < 0 || n >= (1ll << 31) || K < 1 || K > PG_MAX_HEADS || stride < K || row0_span == 0) return PG_ERR_SHAPE;
  if (!counts_out) return PG_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(counts_out) % 8) return PG_ERR_ALIGN;
  const WsLayout L = ws_layout(n, row0_span);
  if (n > 0) {
    if (!rows || !workspace) return PG_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(rows) % 4 || reinterpret_cast<uintptr_t>(workspace) % kAlign) return PG_ERR_ALIGN;
    if (workspace_bytes < L.total) return PG_ERR_WORKSPACE;
  }
  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  cudaError_t e = cudaMemsetAsync(counts_out, 0, sizeof(uint64_t) * K, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (n == 0) return PG_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* cursor = reinterpret_cast<uint32_t*>(ws + L.cursor);
  uint32_t* off = reinterpret_cast<uint32_t*>(ws + L.off);
  uint32_t* tile_sum = reinterpret_cast<uint32_t*>(ws + L.tile_sum);
  uint32_t* tile_off = reinterpret_cast<uint32_t*>(ws + L.tile_off);
  uint32_t* idx = reinterpret_cast<uint32_t*>(ws + L.idx);
  e = cudaMemsetAsync(cursor, 0, 4ull * row0_span, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int* err = device_error_word();
  const uint32_t tiles = static_cast<uint32_t>((static_cast<uint64_t>(row0_span) + kScanTile - 1) / kScanTile);
  const int grid_n = static_cast<int>(std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(nsm) * 8));
  hist_kernel<<<grid_n, 256, 0, stream>>>(rows, n, stride, row0_lo, row0_span, cursor, err);
  tile_sum_kernel<<<tiles, kScanThreads, 0, stream>>>(cursor, row0_span, tile_sum);
  tile_offset_kernel<<<1, kScanThreads, 0, stream>>>(tile_sum, tiles, tile_off, off, row0_span);
  tile_apply_kernel<<<tiles, kScanThreads, 0, stream>>>(cursor, row0_span, tile_off, off);
  scatter_kernel<<<grid_n, 256, 0, stream>>>(rows, n, stride, row0_lo, row0_span, cursor, idx);
  const uint64_t span32 = (static_cast<uint64_t>(row0_span) + 31) / 32 * 32;
  const uint64_t items = static_cast<uint64_t>(K) * span32;
  const int grid_p = static_cast<int>(std::min<uint64_t>((items + 255) / 256, static_cast<uint64_t>(nsm) * 16));
  pair_kernel<<<grid_p, 256, 0, stream>>>(rows, stride, K, row0_span, span32, off, idx,
                                          reinterpret_cast<unsigned long long*>(counts_out), err);
  return after_launch(6);
}

}  // extern "C"
