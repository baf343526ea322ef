// Host side of the C ABI: status strings, versions, descriptor validation, the
// device error word and the launch counter.
#include <atomic>
#include <mutex>

#include "pg_internal.cuh"

namespace {

thread_local int32_t t_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int g_sm_count[kMaxDevices];
int g_cc[kMaxDevices];
int* g_err_word[kMaxDevices];

// One error word per device: bounded device-side waits OR a code into it.
__device__ int pg_device_error_word;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

void init_device(int dev) {
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_sm_count[dev] != 0) return;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, pg_device_error_word) != cudaSuccess) return;
  g_err_word[dev] = static_cast<int*>(addr);
  g_cc[dev] = prop.major * 10 + prop.minor;
  g_sm_count[dev] = prop.multiProcessorCount;
}

}  // namespace

namespace pg {

pg_status cuda_fail(cudaError_t err) {
  t_last_cuda_error = static_cast<int32_t>(err);
  return PG_ERR_CUDA;
}

pg_status after_launch(int n) {
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err);
  g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed);
  return PG_OK;
}

int sm_count() {
  int dev = current_device();
  if (dev < 0) return 0;
  init_device(dev);
  return g_sm_count[dev];
}

int device_cc() {
  int dev = current_device();
  if (dev < 0) return 0;
  init_device(dev);
  return g_cc[dev];
}

int* device_error_word() {
  int dev = current_device();
  if (dev < 0) return nullptr;
  init_device(dev);
  return g_err_word[dev];
}

pg_status validate_desc(const pg_table_desc* d, Geometry* g) {
  if (!d) return PG_ERR_NULL;
  if (d->abi_version != PG_ABI_VERSION || d->hash_version != PG_HASH_VERSION) return PG_ERR_VERSION;
  if (d->mode < PG_FLAT || d->mode > PG_PAGEGRAM) return PG_ERR_SHAPE;
  if (d->hash_kind != PG_HASH_MULXOR && d->hash_kind != PG_HASH_TOY) return PG_ERR_SHAPE;
  if (d->num_orders < 1 || d->num_orders > PG_MAX_ORDERS) return PG_ERR_SHAPE;
  for (int o = 0; o < d->num_orders; ++o) {
    if (d->orders[o] < 1 || d->orders[o] > 4) return PG_ERR_SHAPE;
    if (o > 0 && d->orders[o] <= d->orders[o - 1]) return PG_ERR_SHAPE;
  }
  if (d->r < 1) return PG_ERR_SHAPE;
  if (d->row_dtype < PG_F32 || d->row_dtype > PG_NF4) return PG_ERR_DTYPE;
  if (d->row_dtype == PG_NF4 && d->r != 64) return PG_ERR_DTYPE;
  const int H = (d->mode == PG_FLAT) ? 1 : d->K;
  if (d->mode != PG_FLAT && (d->K < 1 || d->K > PG_MAX_HEADS)) return PG_ERR_SHAPE;
  if (d->mode == PG_FLAT && d->K != 1) return PG_ERR_SHAPE;
  if (d->hash_kind == PG_HASH_TOY &&
      (d->mode != PG_FLAT || d->num_orders != 1 || d->orders[0] != 2 || d->rows[0][0] == 0))
    return PG_ERR_SHAPE;
  if (d->vocab == 0) return PG_ERR_SHAPE;

  uint64_t rows = 0;
  if (d->mode == PG_PAGEGRAM) {
    if (d->S < 1) return PG_ERR_SHAPE;
    for (int o = 0; o < d->num_orders; ++o) {
      if (d->pages[o] == 0) return PG_ERR_SHAPE;
      rows += static_cast<uint64_t>(d->pages[o]) * d->K * d->S;
    }
  } else if (d->mode == PG_ENGRAM) {
    for (int o = 0; o < d->num_orders; ++o)
      for (int k = 0; k < d->K; ++k) {
        if (d->rows[o][k] == 0) return PG_ERR_SHAPE;
        rows += d->rows[o][k];
      }
  } else {
    for (int o = 0; o < d->num_orders; ++o) {
      if (d->rows[o][0] == 0) return PG_ERR_SHAPE;
      rows += d->rows[o][0];
    }
    if (d->hash_kind == PG_HASH_TOY) rows = d->rows[0][0];
  }
  if (rows >= 0xFFFFFFFFull) return PG_ERR_RANGE;  // row indices are uint32; 0xFFFFFFFF = no row

  const uint32_t esize = d->row_dtype == PG_F32 ? 4u : 2u;
  if (g) {
    g->rows = rows;
    g->row_bytes = d->row_dtype == PG_NF4 ? 34u : static_cast<uint32_t>(d->r) * esize;
    g->O = d->num_orders;
    g->H = H;
    g->W = (d->r + 63) / 64;
    g->e_width = d->mode == PG_FLAT ? static_cast<uint32_t>(d->r)
                                    : static_cast<uint32_t>(d->num_orders * H * d->r);
  }
  return PG_OK;
}

void fill_hash_params(const pg_table_desc* d, const Geometry& g, HashParams* p) {
  for (int kind = 0; kind < 3; ++kind)
    for (int o = 0; o < PG_MAX_ORDERS; ++o)
      for (int k = 0; k < PG_MAX_HEADS; ++k)
        for (int j = 0; j < 4; ++j) {
          // function id of hash_version 1: ((kind*4 + o)*64 + k)*4 + j
          const uint64_t fid = static_cast<uint64_t>(((kind * 4 + o) * 64 + k) * 4 + j);
          p->mult[mult_index(kind, o, k, j)] = mix64(d->hash_seed + kGolden * (1ull + fid)) | 1ull;
        }
  uint64_t base = 0;
  for (int o = 0; o < PG_MAX_ORDERS; ++o)
    for (int k = 0; k < PG_MAX_HEADS; ++k) {
      p->divisor[o][k] = 1;
      p->base[o][k] = 0;
    }
  for (int o = 0; o < g.O; ++o) {
    p->order_n[o] = d->orders[o];
    if (d->mode == PG_PAGEGRAM) {
      p->divisor[o][0] = d->pages[o];
      p->base[o][0] = static_cast<uint32_t>(base);
      base += static_cast<uint64_t>(d->pages[o]) * d->K * d->S;
    } else if (d->mode == PG_ENGRAM) {
      for (int k = 0; k < d->K; ++k) {
        p->divisor[o][k] = d->rows[o][k];
        p->base[o][k] = static_cast<uint32_t>(base);
        base += d->rows[o][k];
      }
    } else {
      p->divisor[o][0] = d->rows[o][0];
      p->base[o][0] = static_cast<uint32_t>(base);
      base += d->rows[o][0];
    }
  }
  p->O = g.O;
  p->H = g.H;
  p->K = d->K;
  p->S = d->S < 1 ? 1 : d->S;
  p->W = g.W;
  p->r = d->r;
  p->mode = d->mode;
  p->hash_kind = d->hash_kind;
  p->vocab = d->vocab;
  p->toy_m = d->rows[0][0];
}

}  // namespace pg

extern "C" {

const char* pg_status_str(pg_status s) {
  switch (s) {
    case PG_OK: return "ok";
    case PG_ERR_NULL: return "a required pointer is NULL";
    case PG_ERR_SHAPE: return "a size is out of range or inconsistent";
    case PG_ERR_DTYPE: return "unsupported dtype or dtype combination";
    case PG_ERR_RANGE: return "table smaller than the descriptor needs, or too many rows";
    case PG_ERR_ALIGN: return "a pointer is not aligned as required";
    case PG_ERR_UNSUPPORTED: return "request not supported by this build";
    case PG_ERR_VERSION: return "descriptor version not supported";
    case PG_ERR_WORKSPACE: return "workspace missing or too small";
    case PG_ERR_CUDA: return "a CUDA runtime call failed";
    case PG_ERR_DEVICE: return "the current device cannot run this kernel (needs sm_103a)";
    case PG_ERR_SCRATCH_LIMIT: return "request needs more scratch than the library's static scratch holds";
  }
  return "unknown status";
}

uint32_t pg_abi_version(void) { return PG_ABI_VERSION; }

int32_t pg_last_cuda_error(void) { return t_last_cuda_error; }

uint64_t pg_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

pg_status pg_device_error(int32_t* code, int32_t clear) {
  if (!code) return PG_ERR_NULL;
  int* word = pg::device_error_word();
  if (!word) return pg::cuda_fail(cudaGetLastError());
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return pg::cuda_fail(err);
  int value = 0;
  err = cudaMemcpy(&value, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return pg::cuda_fail(err);
  *code = value;
  if (clear) {
    err = cudaMemset(word, 0, sizeof(int));
    if (err != cudaSuccess) return pg::cuda_fail(err);
  }
  return PG_OK;
}

pg_status pg_table_geometry(const pg_table_desc* desc, uint64_t* rows, uint32_t* row_bytes,
                            uint32_t* e_width) {
  pg::Geometry g;
  pg_status st = pg::validate_desc(desc, &g);
  if (st != PG_OK) return st;
  if (rows) *rows = g.rows;
  if (row_bytes) *row_bytes = g.row_bytes;
  if (e_width) *e_width = g.e_width;
  return PG_OK;
}

}  // extern "C"
