// Internal declarations shared by the translation units of libpg.so.
#pragma once

#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pg.h"

namespace pg {

// ---------------------------------------------------------------- host helpers

// Remember a CUDA error for pg_last_cuda_error() and map it to PG_ERR_CUDA.
pg_status cuda_fail(cudaError_t err);

// Check the last launch; counts `n` launches on success.
pg_status after_launch(int n);

// Streaming multiprocessor count and compute capability of the current device.
int sm_count();
int device_cc();

// cuTensorMapEncodeTiled through the runtime's driver entry point (nullptr if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Device address of this library's device-side error word (current device).
int* device_error_word();

// Validated table geometry (what pg_table_geometry reports).
struct Geometry {
  uint64_t rows;
  uint32_t row_bytes;
  uint32_t e_width;
  int O;      // orders
  int H;      // heads per order (flat and toy: 1)
  int W;      // 64-bit sign words per (order, head)
};
pg_status validate_desc(const pg_table_desc* d, Geometry* g);

// ---------------------------------------------------------------- hashing

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;
constexpr uint32_t kPad = 0xFFFFFFFFu;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Flat index of multiplier (kind, o, k, j) in HashParams::mult.
__host__ __device__ __forceinline__ int mult_index(int kind, int o, int k, int j) {
  return ((kind * PG_MAX_ORDERS + o) * PG_MAX_HEADS + k) * 4 + j;
}
constexpr int kNumMult = 3 * PG_MAX_ORDERS * PG_MAX_HEADS * 4;

// Everything a hashing kernel needs, passed by value (kernel parameter space).
struct HashParams {
  uint64_t mult[kNumMult];                        // odd multipliers m_{kind,o,k,j}
  uint32_t divisor[PG_MAX_ORDERS][PG_MAX_HEADS];  // Engram M_{o,k}; flat R_o and PageGram P_o at [o][0]
  uint32_t base[PG_MAX_ORDERS][PG_MAX_HEADS];     // first row of (o,k) (Engram) or of order o at [o][0]
  int32_t order_n[PG_MAX_ORDERS];                 // n of order index o
  int32_t O, H, K, S, W, r;
  int32_t mode, hash_kind;
  uint32_t vocab;
  uint32_t toy_m;
};

void fill_hash_params(const pg_table_desc* d, const Geometry& g, HashParams* p);

// err_index (optional, device int32): set to -1 on `stream` before a lookup lowers it to
// the smallest offending index with an unsigned atomicMin (0xFFFFFFFF reads as -1).
inline pg_status prepare_err(int32_t* err_index, cudaStream_t stream) {
  if (!err_index) return PG_OK;
  if (reinterpret_cast<uintptr_t>(err_index) % 4) return PG_ERR_ALIGN;
  cudaError_t e = cudaMemsetAsync(err_index, 0xFF, sizeof(int32_t), stream);
  return e == cudaSuccess ? PG_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- streaming decode state

// PG_OK when `st` is a state pg_decode_state_init could have written (geometry in range,
// parts present and aligned); need_conv also requires the conv part (M >= 1).
pg_status decode_state_check(const pg_decode_state* st, bool need_conv);

// ---------------------------------------------------------------- projections without tensor cores

// fp32 out[N, d] = e[N, Din] W[d, Din]^T, plus x + g * out for the scalar gate
// (pg_project_simt.cu). One launch.
pg_status launch_simt_f32(int N, int Din, int d, int gate_kind, const float* e, const float* W, float g,
                          const float* x, float* out, cudaStream_t stream);

// bf16 pg_project_gate for N <= kSmallRows rows (decode batches): a W-streaming SIMT kernel
// over all SMs (pg_project_simt.cu). Context gate: per-row sums per 64-column tile go to
// partials [M, d / kSmallTile, 3, N] (and vpart [d / kSmallTile, N]) for the alpha finalize
// pass. Needs d % 64 == 0, Din % 8 == 0, 16-byte aligned e and W. One launch.
constexpr int kSmallRows = 16;
constexpr int kSmallTile = 64;
constexpr size_t kSmallMaxE = 48 * 1024;  // e staged in shared memory: N * Din * 2 bytes at most
// Whether pg_project_gate (bf16) takes the few-rows kernel: measured on GB300 against the
// tensor-core path (workloads 2 and 5), it is faster up to 4 rows, slower from 8.
constexpr int kSmallRowsUsed = 4;
inline bool use_small_rows(int64_t N, int Din) {
  return N >= 1 && N <= kSmallRowsUsed && static_cast<size_t>(N) * Din * 2 <= kSmallMaxE;
}
pg_status launch_small_rows_bf16(int N, int Din, int d, int M, int gate_kind, const void* e, const void* W, float g,
                                 const void* x, const void* h, const float* gamma_h, const float* gamma_k, void* out,
                                 float* partials, float* vpart, cudaStream_t stream);

// W == NULL: out = e, or x + g e for the scalar gate, over n elements of dtype (n % 8 == 0,
// 16-byte aligned). One launch.
pg_status launch_identity_gate(int64_t n, int dtype, int gate_kind, const void* e, const void* x, float g,
                               void* out, cudaStream_t stream);

}  // namespace pg
