// Streaming decode state: size, carving, reset (sm_103a).
//
// Per sequence the state holds what one more token's lookup and conv read (Engram notes
// 3.5 and PageGram report 3.3: addressing depends on the token IDs alone; Engram notes 3.3:
// the conv is causal with kernel 4 and dilation 3): the position, a 4-slot ring of
// canonical IDs, and a ring of the last (kernel_size - 1) * dilation conv inputs (plus the
// slot the current one is written to), stored factored as (v row, alpha per branch,
// mean(v^2)) from which RMSNorm(alpha v) follows.
// The kernels that read and advance it live beside the full-sequence kernels they match
// (decode_lookup_kernel in pg_lookup.cu, decode_conv_kernel in pg_conv.cu).
#include <algorithm>

#include "pg_internal.cuh"

namespace pg {
namespace {

constexpr uint64_t kPartAlign = 256;

uint64_t round_up(uint64_t x) { return (x + kPartAlign - 1) / kPartAlign * kPartAlign; }

struct Layout {
  uint64_t pos, ids, ring_v, ring_alpha, ring_ms, total;
  int depth;
};

pg_status layout_of(int32_t B, int32_t d, int32_t M, int32_t dtype, int32_t ks, int32_t dil, Layout* L) {
  if (B < 1) return PG_ERR_SHAPE;
  if (dtype != PG_BF16 && dtype != PG_F32) return PG_ERR_DTYPE;
  const bool conv = M != 0 || d != 0;
  if (conv) {
    if (M < 1 || M > 8 || d < 8 || d % 8 || d > 8192) return PG_ERR_SHAPE;
    if (ks < 1 || ks > 4 || dil < 1 || dil > 8) return PG_ERR_SHAPE;
  }
  const uint64_t b = static_cast<uint64_t>(B);
  L->depth = conv && ks > 1 ? (ks - 1) * dil + 1 : 0;
  const uint64_t R = static_cast<uint64_t>(L->depth);
  L->pos = 0;
  L->ids = L->pos + round_up(b * 4);
  L->ring_v = L->ids + round_up(b * 16);
  L->ring_alpha = L->ring_v + round_up(b * R * static_cast<uint64_t>(d) * (dtype == PG_F32 ? 4u : 2u));
  L->ring_ms = L->ring_alpha + round_up(b * R * static_cast<uint64_t>(M) * 4u);
  L->total = L->ring_ms + round_up(b * R * 4u);
  return PG_OK;
}

__global__ void decode_reset_kernel(int32_t* __restrict__ pos, int B, const int32_t* __restrict__ slots, int n,
                                    int* err_word) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int s = slots[i];
    if (s >= 0 && s < B) pos[s] = 0;
    else if (err_word) atomicOr(err_word, 256);
  }
}

}  // namespace

pg_status decode_state_check(const pg_decode_state* st, bool need_conv) {
  if (!st) return PG_ERR_NULL;
  Layout L;
  const pg_status s = layout_of(st->B, st->d, st->M, st->dtype, st->kernel_size, st->dilation, &L);
  if (s != PG_OK) return s;
  if (st->depth != L.depth) return PG_ERR_SHAPE;
  if (need_conv && st->M < 1) return PG_ERR_SHAPE;
  if (!st->pos || !st->ids) return PG_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(st->pos) % 4 || reinterpret_cast<uintptr_t>(st->ids) % 16) return PG_ERR_ALIGN;
  if (st->M >= 1 && L.depth > 0) {
    if (!st->ring_v || !st->ring_alpha || !st->ring_ms) return PG_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(st->ring_v) % 16 || reinterpret_cast<uintptr_t>(st->ring_alpha) % 4 ||
        reinterpret_cast<uintptr_t>(st->ring_ms) % 4)
      return PG_ERR_ALIGN;
  }
  return PG_OK;
}

}  // namespace pg

extern "C" {

pg_status pg_decode_state_size(int32_t B, int32_t d, int32_t M, int32_t dtype, int32_t kernel_size,
                               int32_t dilation, uint64_t* bytes) {
  if (!bytes) return PG_ERR_NULL;
  pg::Layout L;
  const pg_status s = pg::layout_of(B, d, M, dtype, kernel_size, dilation, &L);
  if (s != PG_OK) return s;
  *bytes = L.total;
  return PG_OK;
}

pg_status pg_decode_state_init(pg_decode_state* state, void* buffer, uint64_t buffer_bytes, int32_t B,
                               int32_t d, int32_t M, int32_t dtype, int32_t kernel_size, int32_t dilation,
                               pg_stream_t stream) {
  using namespace pg;
  if (!state || !buffer) return PG_ERR_NULL;
  Layout L;
  const pg_status s = layout_of(B, d, M, dtype, kernel_size, dilation, &L);
  if (s != PG_OK) return s;
  if (buffer_bytes < L.total) return PG_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(buffer) % kPartAlign) return PG_ERR_ALIGN;
  uint8_t* base = static_cast<uint8_t*>(buffer);
  const bool conv = M >= 1;
  pg_decode_state st{};
  st.B = B;
  st.d = conv ? d : 0;
  st.M = conv ? M : 0;
  st.dtype = dtype;
  st.kernel_size = kernel_size;
  st.dilation = dilation;
  st.depth = L.depth;
  st.pos = reinterpret_cast<int32_t*>(base + L.pos);
  st.ids = reinterpret_cast<uint32_t*>(base + L.ids);
  st.ring_v = conv && L.depth > 0 ? static_cast<void*>(base + L.ring_v) : nullptr;
  st.ring_alpha = conv && L.depth > 0 ? reinterpret_cast<float*>(base + L.ring_alpha) : nullptr;
  st.ring_ms = conv && L.depth > 0 ? reinterpret_cast<float*>(base + L.ring_ms) : nullptr;
  const cudaError_t e = cudaMemsetAsync(buffer, 0, L.total, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  *state = st;
  return PG_OK;
}

pg_status pg_decode_reset(const pg_decode_state* state, const int32_t* slots, int32_t n, pg_stream_t stream) {
  using namespace pg;
  const pg_status s = decode_state_check(state, false);
  if (s != PG_OK) return s;
  if (n < 0) return PG_ERR_SHAPE;
  if (n == 0) return PG_OK;
  if (!slots) return PG_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(slots) % 4) return PG_ERR_ALIGN;
  const int nsm = sm_count();
  if (nsm == 0) return cuda_fail(cudaGetLastError());
  const int blocks = static_cast<int>(std::min<int64_t>((static_cast<int64_t>(n) + 255) / 256, nsm));
  decode_reset_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(state->pos, state->B, slots, n,
                                                                                 device_error_word());
  return after_launch(1);
}

}  // extern "C"
