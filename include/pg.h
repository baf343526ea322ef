/*
 * pg.h -- C ABI of libpg.so, the GB300 (sm_103a) hashed multi-head N-gram lookup.
 *
 * The lookup, per token t of a [B, L] batch (sources by page title and section):
 *   1. canonical IDs x'_t = P[x_t]            Engram notes (arXiv 2601.07372) 3.2
 *   2. suffix n-grams g_{t,n}, n in orders    PageGram report 2.1; Engram notes 3.2
 *   3. multiply-XOR hash per (order, head)    Engram notes 3.2
 *   4. row index in one of three layouts      PageGram report 2.1 (flat), 2.2 (multi-head,
 *                                             prime subtables), 3.1 (page-local row_{n,k})
 *   5. gather of the 2K head rows (f32, bf16 or NF4 34-byte rows, PageGram report 3.3)
 *   6. +-1 hash sign masks, concat e_t = ||_n ||_k s_{n,k} * row  (PageGram report 2.2, 3.1)
 *   7. projection W_V e_t (fused with M per-branch W_K, Engram notes 3.4), scalar gate
 *      x + g e (PageGram report 3.1) or RMSNorm-sigmoid gate alpha (Engram notes 3.3)
 *   8. causal depthwise conv + SiLU + residual into the branch states (Engram notes 3.3)
 *
 * Conventions for every call:
 *  - Pointers named as device memory must point to memory of the current CUDA
 *    device; all of it is owned by the caller. No call allocates memory that
 *    outlives the call, and no call frees anything.
 *  - Tensors are dense, row-major, with no padding between rows.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream): it returns after enqueueing its kernels. Host-side checks
 *    run first; when one fails the call returns its status and enqueues nothing.
 *  - Nothing traps or hangs on the device. Device-side waits are bounded; when one
 *    gives up the kernel records a code readable through pg_device_error().
 *  - Hash definition (hash_version 1; the pages name only "a multiply-XOR hash"):
 *      mix64 = splitmix64 output function (Steele, Lea & Flood 2014),
 *      G = 0x9E3779B97F4A7C15,
 *      multiplier m_{f,j} = mix64(seed + G*(1 + (((kind*4 + o)*64 + k)*4 + j))) | 1,
 *        kind 0 = page hash b_n, 1 = head hash (u_{n,k}, phi_{n,k}, flat h_n), 2 = sign,
 *      n-gram c_j = x'_{t-j} (j < n), or 0xFFFFFFFF before the start of the sequence,
 *      h_f = XOR_j c_j * m_{f,j} (mod 2^64), H_f = low 32 bits of h_f ^ (h_f >> 32),
 *      flat      row = base_n + H_{1,o,0} mod R_n
 *      Engram    row = base_{n,k} + H_{1,o,k} mod M_{n,k}   (subtables order-major, head-major)
 *      PageGram  row = base_n + ((H_{0,o,0} mod P_n) K + k) S + (H_{1,o,k} mod S)
 *      sign word q of (o,k) = mix64(h_{2,o,k} + G*(q+1)); element i of the head is
 *        negated iff bit i%64 of word i/64 is set (flat: k = 0 and i < d).
 */
#ifndef PG_H_
#define PG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without including the CUDA headers. */
typedef struct CUstream_st* pg_stream_t;

#define PG_ABI_VERSION 1u
#define PG_HASH_VERSION 1u
#define PG_MAX_ORDERS 4
#define PG_MAX_HEADS 16
#define PG_NO_ROW 0xFFFFFFFFu     /* rows_out entry for "no row" (toy hash at t = 0) */

typedef enum {
  PG_OK = 0,
  PG_ERR_NULL = 1,         /* a required pointer is NULL */
  PG_ERR_SHAPE = 2,        /* a size is out of range or inconsistent */
  PG_ERR_DTYPE = 3,        /* unsupported dtype or dtype combination */
  PG_ERR_RANGE = 4,        /* table smaller than its descriptor needs, or >= 2^32 rows */
  PG_ERR_ALIGN = 5,        /* a pointer is not aligned as the call requires */
  PG_ERR_UNSUPPORTED = 6,  /* well-formed request this build does not implement */
  PG_ERR_VERSION = 7,      /* descriptor abi_version / hash_version not supported */
  PG_ERR_WORKSPACE = 8,    /* workspace missing or smaller than the size query says */
  PG_ERR_CUDA = 9,         /* a CUDA runtime call failed; see pg_last_cuda_error() */
  PG_ERR_DEVICE = 10,      /* current device cannot run the kernel (needs sm_103a) */
  PG_ERR_SCRATCH_LIMIT = 11 /* request needs more than the library's static scratch */
} pg_status;

enum { PG_FLAT = 0, PG_ENGRAM = 1, PG_PAGEGRAM = 2 };
enum { PG_HASH_MULXOR = 0, PG_HASH_TOY = 1 };
enum { PG_F32 = 0, PG_BF16 = 1, PG_NF4 = 2 };
enum { PG_GATE_NONE = 0, PG_GATE_SCALAR = 1, PG_GATE_CONTEXT = 2 };

/*
 * Table descriptor (plain data; fill every field).
 *  abi_version, hash_version  PG_ABI_VERSION, PG_HASH_VERSION
 *  mode        PG_FLAT | PG_ENGRAM | PG_PAGEGRAM
 *  hash_kind   PG_HASH_MULXOR, or PG_HASH_TOY: the Engram explainer's teaching bucket
 *              (3a + b) mod m ("Hash 冲突是什么样？"), flat mode, one order n = 2,
 *              m = rows[0][0]; pg_canon_hash only.
 *  num_orders, orders[]  n-gram orders, strictly increasing, each in [1, 4]
 *  K           heads per order (multi-head modes), 1..16; flat: 1
 *  S           PageGram slots per head per page (>= 1); ignored otherwise
 *  r           head width (flat: the row width, = d)
 *  pages[o]    PageGram P_n for order index o
 *  rows[o][k]  Engram M_{n,k} for order index o, head k; flat R_n in rows[o][0]
 *  row_dtype   PG_F32 | PG_BF16 | PG_NF4 (NF4: r = 64, 34-byte rows: bytes 0..31
 *              hold codes, element 2i in the low nibble of byte i, 2i+1 in the high
 *              nibble; bytes 32..33 an fp16 scale, little-endian)
 *  hash_seed   seeds the hash family
 *  vocab       V: token IDs must lie in [0, V)
 *  canon_vocab V' (informational; the canonical map's values are used as given)
 */
typedef struct {
  uint32_t abi_version;
  uint32_t hash_version;
  int32_t mode;
  int32_t hash_kind;
  int32_t num_orders;
  int32_t orders[PG_MAX_ORDERS];
  int32_t K;
  int32_t S;
  int32_t r;
  uint32_t pages[PG_MAX_ORDERS];
  uint32_t rows[PG_MAX_ORDERS][PG_MAX_HEADS];
  int32_t row_dtype;
  int32_t reserved;
  uint64_t hash_seed;
  uint32_t vocab;
  uint32_t canon_vocab;
} pg_table_desc;

/* Message for a status code (static storage). */
const char* pg_status_str(pg_status status);

/* PG_ABI_VERSION of the loaded library. */
uint32_t pg_abi_version(void);

/* Last CUDA error code a pg_* call on this host thread met (0 if none). */
int32_t pg_last_cuda_error(void);

/* Number of kernels this library has launched in this process. */
uint64_t pg_launch_count(void);

/*
 * Device-side error word of the current device: 0, or the OR of codes of bounded
 * waits that gave up in the projection kernels (1 = TMA producer, 2 = MMA issuer,
 * 4 = epilogue, 8 = epilogue operand producer, 16 = gather warps of
 * pg_lookup_project_gate, 64 = a tile's wait for its rows of e_t in
 * pg_gather_project_gate, 128 = that call's gather warps or their coordinator), and
 * of decode-state checks (256 = pg_decode_reset met a slot outside [0, B), 512 = a
 * decode call met a position it cannot take; that sequence was skipped, left unchanged),
 * and of pg_collision_counts (1024 = a head-0 row outside the given span, or a head-0
 * group too large to compare pairwise; those n-grams or pairs were left out), and of
 * pg_selftest_bounded_waits (2048, 4096), and of pg_project_gate_conv (16384 = a conv item's wait
 * for the tiles of its m-blocks), and of pg_decode_step (32768 = a block's wait at the grid
 * barrier, 65536 = a wait for a row of W).
 * Synchronizes the device. With clear != 0 the word is reset to 0.
 */
pg_status pg_device_error(int32_t* code, int32_t clear);

/*
 * pg_selftest_bounded_waits -- checks, on the current device, that the bounded waits the
 * tensor-core kernels use give up and report instead of hanging. The pages have no
 * counterpart: this is failure handling of this library.
 *
 * One thread waits on an mbarrier phase that nothing completes, then on a ready counter
 * that nothing raises (*zero_word, set to 0 by the call on `stream`); each wait gives up
 * after about one second and ORs its code into the device error word (2048 = the mbarrier
 * wait, 4096 = the counter wait), so a correct run leaves 2048 | 4096 there after about
 * two seconds. No copy, tensor-core operation or TMEM is involved, and the device stays
 * usable. zero_word: caller-owned device memory, 4 bytes, 4-byte aligned.
 * PG_ERR_NULL / PG_ERR_ALIGN for a bad zero_word; PG_ERR_CUDA if the launch fails.
 */
pg_status pg_selftest_bounded_waits(uint32_t* zero_word, pg_stream_t stream);

/*
 * Table geometry of a descriptor: number of stored rows (the table's first
 * dimension), bytes per row, and the width of e_t (O*K*r, or r for flat).
 * Any out pointer may be NULL. Validates the descriptor (PG_ERR_VERSION,
 * PG_ERR_SHAPE, PG_ERR_DTYPE, PG_ERR_RANGE).
 */
pg_status pg_table_geometry(const pg_table_desc* desc, uint64_t* rows, uint32_t* row_bytes,
                            uint32_t* e_width);

/*
 * pg_canon_hash -- steps 1-4 plus sign words, written out (the addresses depend on
 * token IDs only, so they can be computed before the forward pass: PageGram report
 * 3.3 "prefetch"; Engram notes 3.5).
 *  tokens     device int32 [B, L]
 *  canon_map  device uint32 [vocab], or NULL for the identity map
 *  canon_out  device uint32 [B*L] (x'_t), or NULL
 *  rows_out   device uint32 [B*L, O, H], H = K (flat and toy: 1)
 *  sign_out   device uint64 [B*L, O, H, ceil(r/64)], or NULL (toy: all zero)
 *  err_index  device int32 [1], or NULL: set to the smallest flat index of a token
 *             outside [0, vocab) that the call read, else -1 (written on `stream`).
 *             Such a token is read as ID 0 and the call continues.
 * B, L >= 0 (B*L < 2^31); B*L == 0 enqueues nothing.
 */
pg_status pg_canon_hash(const pg_table_desc* desc, const int32_t* tokens, int32_t B, int32_t L,
                        const uint32_t* canon_map, uint32_t* canon_out, uint32_t* rows_out,
                        uint64_t* sign_out, int32_t* err_index, pg_stream_t stream);

/*
 * pg_gather_sign_concat -- steps 1-6 fused: hashes and row indices are computed in
 * registers, the rows gathered with 16-byte loads (PageGram: one warp serves a
 * token's K*S page blocks, one contiguous segment per order), NF4 rows dequantised
 * in registers (level[code] * float(scale), one fp32 multiply, round-to-nearest-even),
 * signs applied and the heads written concatenated.
 *  table      device memory, table_bytes long (>= rows * row_bytes), 16-byte aligned
 *  e_out      device [B*L, e_width] of out_dtype; multi-head column block
 *             (o*K + k)*r holds head (o, k); flat: e = s_0*T[row_0] + s_1*T[row_1] + ...
 *             summed in fp32 in order of increasing n, then rounded to out_dtype
 *  out_dtype  f32 rows -> PG_F32; bf16 rows -> PG_BF16 or PG_F32; NF4 -> PG_BF16 or PG_F32
 *  err_index  as in pg_canon_hash
 * PG_HASH_TOY is not accepted here (PG_ERR_UNSUPPORTED).
 */
pg_status pg_gather_sign_concat(const pg_table_desc* desc, const int32_t* tokens, int32_t B,
                                int32_t L, const uint32_t* canon_map, const void* table,
                                uint64_t table_bytes, void* e_out, int32_t out_dtype,
                                int32_t* err_index, pg_stream_t stream);

/*
 * pg_nf4_quantize -- NF4 export of head rows (PageGram report 3.3: deployed rows are 64
 * four-bit NormalFloat codes + one fp16 scale = 34 bytes; report 9.4, check 5: all-zero
 * rows stay exact and the error stays within the quantisation bound). Produces tables in
 * the PG_NF4 row layout that pg_gather_sign_concat reads.
 *  x      device fp32 [nrows, r], 8-byte aligned; r must be 64 (else PG_ERR_UNSUPPORTED)
 *  out    device [nrows, 34] bytes, any alignment (PG_NF4 layout: byte i = code of element
 *         2i | code of element 2i+1 << 4; bytes 32..33 the fp16 scale, little-endian)
 * Per row: scale = max |x_i| rounded to fp16 (nearest, ties to even; values that would
 * round past 65504 saturate to 65504); scale 0 gives the exact-zero level (code 7) for
 * every element; otherwise code_i = the NF4 level nearest to x_i / scale (fp32, correctly
 * rounded division, fp32 distances, the lowest code on ties). NaN elements do not count
 * towards the scale and get code 0. nrows == 0 enqueues nothing.
 */
pg_status pg_nf4_quantize(const float* x, int64_t nrows, int32_t r, void* out, pg_stream_t stream);

/*
 * Workspace bytes pg_project_gate needs for these arguments (0 when none).
 */
pg_status pg_project_gate_workspace_size(int32_t N, int32_t Din, int32_t d, int32_t M,
                                         int32_t dtype, int32_t gate_kind, size_t* bytes);

/*
 * pg_project_gate -- step 7 (PageGram report 2.2 and 3.1; Engram notes 3.3, 3.4).
 *  e      device [N, Din] (dtype)
 *  W      device [(1+M)*d, Din] (dtype): W_V rows, then W_K^(1..M) rows. May be NULL
 *         with Din == d and gate NONE or SCALAR: identity (a flat table's e_t is already
 *         d wide, PageGram report 2.1).
 *  gate_kind
 *    PG_GATE_NONE     v_out[N, d] = e W_V^T                       (M must be 0)
 *    PG_GATE_SCALAR   v_out[N, d] = x_resid + g * (e W_V^T)       (x_resid [N, d]; M = 0)
 *    PG_GATE_CONTEXT  v_out[N, d] = e W_V^T and, for each branch m,
 *                     alpha_out[m, t] = sigmoid(RMSNorm(h^(m)_t) . RMSNorm(W_K^(m) e_t) / sqrt(d))
 *                     with RMSNorm(z) = z / sqrt(mean(z^2) + eps) * gamma (gamma_h for h,
 *                     gamma_k for k; fp32 [d]); h device [M, N, d]; alpha_out fp32 [M, N]
 *  dtype  PG_F32: fp32 SIMT FFMA path (gates NONE and SCALAR).
 *         PG_BF16: tcgen05 tensor-core path, fp32 accumulation, bf16 results; requires
 *         Din % 64 == 0, d % 128 == 0, 16-byte aligned e and W. A few rows (decode
 *         batches of up to 4) run a SIMT kernel that streams W over every SM instead (a tensor-core tile's 128 / 256 rows would
 *         idle); the context gate takes it when the workspace is the size query's.
 *         Identity (W == NULL) works for both dtypes.
 *  v_ms_out  context gate, bf16 path only, optional (may be NULL): device fp32 [N],
 *             mean(v_t^2) over the d values of v_out as stored (bf16), the factor the
 *             RMSNorm of pg_conv_residual needs; computed in the projection's epilogue
 *             (per-tile sums added in tile order, deterministic).
 *  workspace  device, >= pg_project_gate_workspace_size() bytes, 16-byte aligned
 *             (only the context gate uses it; its contents are scratch). The query
 *             includes the room v_ms_out needs; without v_ms_out, M * (d / BN) * 3 * N * 4
 *             bytes suffice (BN = 256 if d % 256 == 0, else 128; the query uses BN = 64
 *             for N <= 4, which the few-rows kernel needs, and smaller workspaces send
 *             those calls to the tensor-core path).
 * N == 0 enqueues nothing. x_resid / h / v_out must not overlap e or W.
 */
pg_status pg_project_gate(int32_t N, int32_t Din, int32_t d, int32_t M, int32_t dtype,
                          const void* e, const void* W, int32_t gate_kind, float g,
                          const void* x_resid, const void* h, const float* gamma_h,
                          const float* gamma_k, float eps, void* v_out, float* alpha_out,
                          float* v_ms_out, void* workspace, size_t workspace_bytes, pg_stream_t stream);

/*
 * pg_conv_residual -- step 8 (Engram notes 3.3 and 3.1, explainer's causal conv):
 * for each branch m and position t of each sequence,
 *   u = alpha[m, t] * v_t;  z = RMSNorm(u) with gamma_c;
 *   c_t = sum_{j < kernel_size} conv_w[:, j] * z_{t - j*dilation}   (zero before t = 0)
 *   H[m, t] <- H[m, t] + SiLU(c_t) + u
 *  v      device [B*L, d] (dtype), alpha device fp32 [M, B*L]
 *  v_ms   optional (may be NULL): device fp32 [B*L], mean(v_t^2) (pg_project_gate's
 *         v_ms_out); when NULL the call computes it from v
 *  gamma_c, conv_w  device fp32 [d], [d, kernel_size] (shared by the branches)
 *  H      device [M, B*L, d] (dtype), updated in place
 *  dtype PG_BF16 or PG_F32; d % 8 == 0, d <= 8192; kernel_size in [1, 4];
 *  dilation in [1, 8]; v and H 16-byte aligned.
 */
pg_status pg_conv_residual(int32_t B, int32_t L, int32_t d, int32_t M, int32_t dtype,
                           const void* v, const float* alpha, const float* v_ms,
                           const float* gamma_c, const float* conv_w, int32_t kernel_size,
                           int32_t dilation, float eps, void* H, pg_stream_t stream);

/*
 * pg_project_gate_conv -- the context-gated projection and the causal conv + residual in one
 * launch: pg_project_gate(gate_kind = PG_GATE_CONTEXT, dtype = PG_BF16, h = H) followed by
 * pg_conv_residual(v, alpha, v_ms, gamma_c, conv_w, kernel_size, dilation, eps, H), with H
 * read as the gate's h and updated in place (Engram notes 3.3, 3.4, 3.1: alpha from
 * RMSNorm(h) . RMSNorm(k), then Y = SiLU(Conv1D(RMSNorm(alpha v))) + alpha v, H += Y).
 * The conv runs behind the projection's tiles in the same persistent kernel, so each
 * tile of H is read once from HBM for both steps. v_out, alpha_out, v_ms_out and H are
 * bit-identical to the two calls.
 *  e [B*L, Din], W [(1+M) d, Din], H [M, B*L, d]: device bf16, 16-byte aligned
 *  gamma_h, gamma_k, gamma_c [d], conv_w [d, kernel_size]: device fp32, 16-byte aligned
 *  v_out [B*L, d] bf16; alpha_out [M, B*L] fp32; v_ms_out [B*L] fp32 or NULL
 *  workspace: pg_project_gate_conv_workspace_size bytes, 16-byte aligned (the call zeroes
 *  its head, per-m-block counters, on `stream` before the launch)
 *  Din % 64 == 0, d % 256 == 0; kernel_size in [1, 4], dilation in [1, 8],
 *  (kernel_size - 1) * dilation <= 24. PG_ERR_WORKSPACE for a short workspace. A wait of a
 *  conv item for its m-blocks that gives up sets device error bit 16384.
 */
pg_status pg_project_gate_conv_workspace_size(int32_t N, int32_t d, int32_t M, size_t* bytes);
pg_status pg_project_gate_conv(int32_t B, int32_t L, int32_t Din, int32_t d, int32_t M, const void* e,
                               const void* W, void* H, const float* gamma_h, const float* gamma_k,
                               const float* gamma_c, const float* conv_w, int32_t kernel_size, int32_t dilation,
                               float eps, void* v_out, float* alpha_out, float* v_ms_out, void* workspace,
                               size_t workspace_bytes, pg_stream_t stream);

/*
 * FP8 operands of the fused projection (Engram notes 3.4: W_V and the M W_K run in FP8).
 *
 * pg_fp8_quantize -- rows of x [rows, cols] (dtype PG_F32 or PG_BF16, 16-byte aligned,
 * cols % 8 == 0) -> OCP E4M3 codes q [rows, cols] (1 byte each, 16-byte aligned) and one
 * fp32 scale per row (scale [rows], 4-byte aligned): scale = max |x| / 448 (fp32 division),
 * q_i = E4M3(x_i / scale) rounded to nearest, ties to even, saturating at +-448; a row
 * whose max |x| is 0 gets scale 0 and zero codes. NaN elements are outside the contract.
 */
pg_status pg_fp8_quantize(const void* x, int32_t dtype, int64_t rows, int64_t cols, void* q,
                          float* scale, pg_stream_t stream);

/*
 * pg_gather_sign_concat_e4m3 -- steps 1-7 of pg_gather_sign_concat with the FP8 projection's
 * operand as output: each token's e_t row (bf16 table rows, signed and concatenated exactly
 * as pg_gather_sign_concat writes it in bf16) quantised as pg_fp8_quantize does it, in the
 * same kernel (Engram notes 3.4: the fused projection runs in FP8, so e_t need not exist in
 * bf16). q_out and scale_out equal pg_gather_sign_concat(out_dtype = PG_BF16) followed by
 * pg_fp8_quantize(dtype = PG_BF16) bit for bit.
 *  q_out     device [B*L, O*K*r] E4M3 codes, 16-byte aligned
 *  scale_out device fp32 [B*L], 4-byte aligned
 *  other arguments, err_index and errors as pg_gather_sign_concat; PG_ERR_DTYPE unless the
 *  table holds bf16 rows; PG_ERR_UNSUPPORTED for layouts other than 16 (order, head) items
 *  of r = 64 or r = 80 (Engram or PageGram mode).
 */
pg_status pg_gather_sign_concat_e4m3(const pg_table_desc* desc, const int32_t* tokens, int32_t B, int32_t L,
                                     const uint32_t* canon_map, const void* table, uint64_t table_bytes,
                                     uint8_t* q_out, float* scale_out, int32_t* err_index, pg_stream_t stream);

/*
 * pg_project_gate_fp8 -- pg_project_gate (dtype PG_BF16 outputs and gates) on E4M3
 * operands: v = diag(e_scale) (e_q W_q^T) diag(W_scale) with e_q [N, Din] and W_q
 * [(1+M)*d, Din] from pg_fp8_quantize, fp32 accumulation on the tensor cores
 * (tcgen05.mma kind::f8f6f4, CTA pairs), then exactly pg_project_gate's gate epilogue.
 *  e_q, W_q     device E4M3 bytes, 16-byte aligned; Din % 256 == 0; d % 256 == 0
 *  e_scale      device fp32 [N] (4-byte aligned); W_scale device fp32 [(1+M)*d] (16-byte aligned)
 *  the rest     as pg_project_gate (workspace: pg_project_gate_workspace_size with PG_BF16)
 */
pg_status pg_project_gate_fp8(int32_t N, int32_t Din, int32_t d, int32_t M, const void* e_q,
                              const float* e_scale, const void* W_q, const float* W_scale,
                              int32_t gate_kind, float g, const void* x_resid, const void* h,
                              const float* gamma_h, const float* gamma_k, float eps, void* v_out,
                              float* alpha_out, float* v_ms_out, void* workspace,
                              size_t workspace_bytes, pg_stream_t stream);

/*
 * pg_lookup_project_gate -- steps 1-7 in one kernel: pg_gather_sign_concat followed by
 * pg_project_gate, without writing e_t to memory. The projection is the fused W_V (+ M
 * W_K) GEMM of the Engram notes section 3.4 fed straight by the lookup of section 3.2 /
 * PageGram report section 3.1: each 64-column k-block of e_t is one head (o, k) of 128
 * tokens, gathered, sign-flipped and laid out in shared memory by dedicated warps and
 * consumed there by the tensor cores.
 *  Tables: PG_ENGRAM or PG_PAGEGRAM mode, PG_BF16 rows, r = 64, O*K <= 32 (Din = O*K*64).
 *  desc .. table_bytes, err_index   as in pg_gather_sign_concat
 *  d .. workspace_bytes             as in pg_project_gate with dtype PG_BF16
 * Results are bit-identical to the two-call sequence (same values, same accumulation
 * order) except for the few tokens (up to 4) whose two-call
 * projection runs on the few-rows kernel, which this call matches within the
 * projection's tolerance. B*L == 0 enqueues nothing.
 */
pg_status pg_lookup_project_gate(const pg_table_desc* desc, const int32_t* tokens, int32_t B, int32_t L,
                                 const uint32_t* canon_map, const void* table, uint64_t table_bytes,
                                 int32_t d, int32_t M, const void* W, int32_t gate_kind, float g,
                                 const void* x_resid, const void* h, const float* gamma_h,
                                 const float* gamma_k, float eps, void* v_out, float* alpha_out,
                                 void* workspace, size_t workspace_bytes, int32_t* err_index,
                                 pg_stream_t stream);

/*
 * pg_gather_project_gate -- steps 1-7 in one launch that also writes e_t:
 * pg_gather_sign_concat(desc, tokens, ..., e_out, PG_BF16) followed by
 * pg_project_gate(e_out, W, ...), with the lookup of the Engram notes section 3.2 /
 * PageGram report section 3.1 running on extra warps of the projection's persistent CTA
 * pairs (Engram notes section 3.4), so that its random row reads overlap the tensor-core
 * work instead of preceding it. A coordinator warp per CTA claims units of e_t (the most
 * tokens, a power of two, whose rows number at most 512: 32 tokens at 16 rows per token) in
 * the order the projection's tiles consume them and hands them to the gather warps; each
 * finished unit is counted on its 128-token block's ready counter in the workspace, and a
 * tile's first load of its rows waits for that count (bounded: a wait that runs out sets
 * the device error word and the call's results are undefined).
 *  Tables: PG_ENGRAM or PG_PAGEGRAM mode, PG_BF16 rows, r = 64, O*K <= 32 (Din = O*K*64).
 *  desc .. table_bytes, err_index   as in pg_gather_sign_concat
 *  e_out  device [B*L, Din] bf16, 16-byte aligned: e_t, written (the projection's A operand)
 *  d .. v_ms_out                    as in pg_project_gate with dtype PG_BF16; d % 256 == 0
 *  workspace  device, 16-byte aligned, >= pg_gather_project_gate_workspace_size() bytes
 *         (always needed: the ready counters); zeroed in part by the call (one
 *         cudaMemsetAsync on `stream`) before its kernel.
 * e_out, v_out, alpha_out and v_ms_out are bit-identical to the two-call sequence (for
 * the few tokens that take the few-rows projection the call runs those two calls). Calls that share a workspace must be ordered
 * (same stream). B*L == 0 enqueues nothing.
 */
pg_status pg_gather_project_gate(const pg_table_desc* desc, const int32_t* tokens, int32_t B, int32_t L,
                                 const uint32_t* canon_map, const void* table, uint64_t table_bytes,
                                 void* e_out, int32_t d, int32_t M, const void* W, int32_t gate_kind,
                                 float g, const void* x_resid, const void* h, const float* gamma_h,
                                 const float* gamma_k, float eps, void* v_out, float* alpha_out,
                                 float* v_ms_out, void* workspace, size_t workspace_bytes,
                                 int32_t* err_index, pg_stream_t stream);

/* Workspace bytes pg_gather_project_gate needs for N = B*L tokens, d, M and gate_kind. */
pg_status pg_gather_project_gate_workspace_size(int32_t N, int32_t d, int32_t M, int32_t gate_kind,
                                                size_t* bytes);

/*
 * pg_project_gate_context_noalloc -- the context-gate projection of pg_project_gate
 * (gate PG_GATE_CONTEXT, dtype PG_BF16) for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point: it exists for the host side only.
 *
 * Some callers cannot call cudaMalloc: a serving runtime that hands all device memory
 * to its own pool at start-up, or a plug-in whose host gives it no allocator and does
 * not allow the device-wide synchronisation that cudaMalloc / cudaFree may cause. They
 * cannot provide the workspace pg_project_gate needs, so this call uses scratch held
 * by the library instead: a file-scope device array of PG_NOALLOC_SCRATCH_BYTES
 * (16 MiB) that every GPU which loads libpg.so keeps until the process exits.
 *
 * Arguments, results and errors are those of pg_project_gate with gate_kind =
 * PG_GATE_CONTEXT, dtype = PG_BF16, g and x_resid unused. In addition:
 *  - the call allocates nothing and frees nothing (no cudaMalloc, cudaFree or other
 *    allocating routine);
 *  - PG_ERR_SCRATCH_LIMIT when the scratch it needs, M * (d / BN) * 3 * N * 4 bytes with
 *    BN = 256 if d % 256 == 0 else 128, exceeds PG_NOALLOC_SCRATCH_BYTES (at d = 2560,
 *    M = 4: N <= 34,952 tokens); nothing is enqueued then;
 *  - the first call on a device looks up the scratch array's device address on that
 *    device (cudaGetSymbolAddress, with the device current). With lazy module loading
 *    (the CUDA default) that lookup may also be what loads the library's device code
 *    on that device, the 16 MiB array with it; so make the first call at start-up,
 *    before any stream capture, where a one-time load is acceptable;
 *  - devices with an ordinal of 64 or more are not served: PG_ERR_DEVICE;
 *  - every call on a device shares the one array and overwrites all of the scratch it
 *    uses before reading it (no part has to start at zero); calls whose kernels overlap
 *    on the GPU (other streams, other host threads) race on it and must be ordered by
 *    the caller.
 */
#define PG_NOALLOC_SCRATCH_BYTES (16u << 20)

pg_status pg_project_gate_context_noalloc(int32_t N, int32_t Din, int32_t d, int32_t M,
                                          const void* e, const void* W, const void* h,
                                          const float* gamma_h, const float* gamma_k, float eps,
                                          void* v_out, float* alpha_out, pg_stream_t stream);

/*
 * Streaming decode (one new token per sequence and call).
 *
 * Each sequence's lookup reads only its suffix n-gram (the last max(orders) - 1 canonical
 * IDs and the new one), and the causal conv reads only the inputs of the last
 * (kernel_size - 1) * dilation positions. Both are known before the step runs, since
 * addressing depends on the token IDs alone (Engram notes 3.5; PageGram report 3.3 on
 * prefetching). A decode state keeps exactly that per sequence, so a step over B
 * sequences costs B tokens' lookups, not a re-run of the prefix. A sequence's outputs at
 * position t equal those of the full-sequence calls at position t: pg_decode_lookup's e_t
 * is bit-identical to pg_gather_sign_concat's, and pg_decode_conv_residual's update of H
 * is bit-identical to pg_conv_residual's when given the same v, alpha and v_ms.
 *
 * State layout (device memory, carved from one caller-owned buffer by pg_decode_state_init):
 *   pos         int32  [B]        tokens of the sequence consumed so far
 *   ids         uint32 [B][4]     canonical ID of position p in slot p mod 4
 *   ring_v      dtype  [B][D][d]  v of position p in slot p mod D
 *   ring_alpha  fp32   [B][D][M]  alpha[m] of position p in slot p mod D
 *   ring_ms     fp32   [B][D]     mean(v_p^2) in slot p mod D
 * with D = (kernel_size - 1) * dilation + 1 (0 when kernel_size == 1): the conv inputs of
 * the last D - 1 positions, which the next output reads (9 for kernel 4, dilation 3), and
 * the slot the current position's input goes to, so that no block of a launch reads a
 * slot another block of it writes. Slots of positions before the start of a sequence are
 * never read, so an all-zero state (what pg_decode_state_init writes) is B empty
 * sequences, and setting pos[b] = 0 (pg_decode_reset) restarts sequence b. Sequences
 * advance independently: each reads its own pos, so a batch may hold sequences at
 * different positions.
 *
 * One decode step, on one stream:
 *   pg_decode_lookup                 -- consumes token b at t = pos[b]; pos[b] = t + 1
 *   pg_project_gate(N = B, ...)      -- the projection and gate of these tokens
 *   pg_decode_conv_residual          -- context-gate (multi-branch) path: position pos[b] - 1
 */
typedef struct {
  int32_t B;            /* sequences */
  int32_t d;            /* conv channels (model width); 0 when the state has no conv part */
  int32_t M;            /* branches; 0 when the state has no conv part */
  int32_t dtype;        /* PG_BF16 or PG_F32: dtype of v and ring_v */
  int32_t kernel_size;  /* 1..4 */
  int32_t dilation;     /* 1..8 */
  int32_t depth;        /* D above, filled in by pg_decode_state_init */
  int32_t reserved;
  int32_t* pos;
  uint32_t* ids;
  void* ring_v;
  float* ring_alpha;
  float* ring_ms;
} pg_decode_state;

/*
 * Bytes of the device buffer a decode state needs (host-only arithmetic; every part
 * starts on a 256-byte boundary). M == 0 (with d == 0) sizes a lookup-only state.
 * PG_ERR_SHAPE / PG_ERR_DTYPE for arguments outside the ranges above.
 */
pg_status pg_decode_state_size(int32_t B, int32_t d, int32_t M, int32_t dtype, int32_t kernel_size,
                               int32_t dilation, uint64_t* bytes);

/*
 * Fills *state with the geometry and the pointers of its parts inside `buffer` (device,
 * 256-byte aligned, >= pg_decode_state_size bytes, owned by the caller and used by the
 * state until the caller frees it) and zeroes the buffer on `stream` (B empty sequences).
 */
pg_status pg_decode_state_init(pg_decode_state* state, void* buffer, uint64_t buffer_bytes, int32_t B,
                               int32_t d, int32_t M, int32_t dtype, int32_t kernel_size, int32_t dilation,
                               pg_stream_t stream);

/*
 * Restarts the listed sequences: pos[slots[i]] = 0 for i < n (slots: device int32 [n]).
 * A slot outside [0, B) is skipped and reported as device error bit 256.
 */
pg_status pg_decode_reset(const pg_decode_state* state, const int32_t* slots, int32_t n, pg_stream_t stream);

/*
 * pg_decode_lookup -- steps 1-6 for one new token per sequence: tokens device int32 [B]
 * (token b continues sequence b at position t = pos[b]); e_out device [B, width] as
 * pg_gather_sign_concat's (out_dtype PG_F32 or PG_BF16; NF4 tables dequantised).
 * Writes ids[b][t mod 4] = the token's canonical ID and pos[b] = t + 1. Orders up to 4
 * (the ID ring holds the 3 IDs before t). Descriptor, table and err_index as in
 * pg_gather_sign_concat (err_index gets the smallest b whose token is out of range; that
 * token reads as ID 0). Multiply-XOR hashing only. A negative pos[b] is reported as
 * device error bit 512 and sequence b is skipped (e_out row, ids and pos left as they are).
 */
pg_status pg_decode_lookup(const pg_table_desc* desc, const pg_decode_state* state, const int32_t* tokens,
                           const uint32_t* canon_map, const void* table, uint64_t table_bytes, void* e_out,
                           int32_t out_dtype, int32_t* err_index, pg_stream_t stream);

/*
 * pg_decode_conv_residual -- step 8 for the position t = pos[b] - 1 of each sequence (the
 * token the step's pg_decode_lookup consumed):
 *   u = alpha[m, b] v_b;  z = RMSNorm(u) with gamma_c;
 *   c = sum_{j < kernel_size} conv_w[:, j] * z_{t - j*dilation}  (terms before t = 0 are 0;
 *       the earlier z come from the state's ring)
 *   H[m, b] <- H[m, b] + SiLU(c) + u
 * and stores v_b, alpha[:, b] and mean(v_b^2) in ring slot t mod D. pos is not changed.
 *  v  device [B, d] (state dtype, 16-byte aligned); alpha device fp32 [M, B];
 *  v_ms  optional device fp32 [B] (pg_project_gate's v_ms_out); computed from v when NULL
 *  gamma_c, conv_w  device fp32 [d], [d, kernel_size]; H device [M, B, d] (state dtype)
 *  The state must have a conv part (M >= 1, d % 8 == 0, d <= 8192). pos[b] < 1 is
 *  reported as device error bit 512 and sequence b is skipped (H and the ring unchanged).
 */
pg_status pg_decode_conv_residual(const pg_decode_state* state, const void* v, const float* alpha,
                                  const float* v_ms, const float* gamma_c, const float* conv_w, float eps,
                                  void* H, pg_stream_t stream);

/*
 * One decode step in one launch, for a few sequences (B <= 8): pg_decode_lookup, the
 * projection with its gate (pg_project_gate with N = B) and, for the context gate,
 * pg_decode_conv_residual, as one kernel. Addressing depends on the token IDs alone
 * (Engram notes 3.5), so every block computes the step's e_t; each block then owns a range
 * of the d channels, streams its rows of W and runs the conv on the same channels. The
 * context gate's sums over all d channels (alpha, mean(v^2)) meet once at a grid barrier:
 * every block publishes partial sums to the workspace and reduces all of them in one
 * order, so every block uses the same alpha.
 *
 * Results: e_t (e_out, optional) bit-identical to pg_decode_lookup's; out, alpha_out,
 * v_ms_out and the update of H equal the three calls' within rounding (the dot products
 * and the gate's sums are added in another order; given the same v, alpha and mean(v^2)
 * the conv rounds every step as pg_decode_conv_residual does). The state advances as in
 * pg_decode_lookup + pg_decode_conv_residual: ids, pos, and for the context gate the ring.
 * A sequence with pos[b] < 0 is skipped (device error bit 512): its rows of e_out, out,
 * alpha_out, H and the state are left as they are.
 */
typedef struct {
  const void* W;          /* bf16 [(1 + M) d, Din] (context gate; M = state->M) or [d, Din]:
                             pg_project_gate's W; 16-byte aligned; Din = the table's e_t width */
  int32_t d;              /* output width (context gate: state->d) */
  int32_t gate_kind;      /* PG_GATE_NONE, PG_GATE_SCALAR or PG_GATE_CONTEXT */
  float g;                /* scalar gate: out = x_resid + g (e W^T) */
  float eps;              /* context gate: RMSNorm epsilon (gate and conv) */
  const void* x_resid;    /* scalar gate: bf16 [B, d] */
  void* H;                /* context gate: bf16 [M, B, d], the gate's h and, updated in place,
                             the branch states the conv adds to */
  const float* gamma_h;   /* context gate: fp32 [d] each */
  const float* gamma_k;
  const float* gamma_c;   /* context gate: conv RMSNorm gain, fp32 [d] */
  const float* conv_w;    /* context gate: fp32 [d, kernel_size] */
  void* e_out;            /* optional bf16 [B, Din], 16-byte aligned */
  void* out;              /* bf16 [B, d]: v (context gate) or the gated output */
  float* alpha_out;       /* optional fp32 [M, B] (context gate) */
  float* v_ms_out;        /* optional fp32 [B]: mean(v^2) (context gate) */
} pg_decode_step_args;

/*
 * Workspace bytes of pg_decode_step for B sequences (1..8), width d and M branches (0 for
 * the scalar or no gate) on the current device (its SM count sets the block count).
 */
pg_status pg_decode_step_workspace_size(int32_t B, int32_t d, int32_t M, uint64_t* bytes);

/*
 * pg_decode_step -- desc, state, tokens, canon_map, table, table_bytes and err_index as in
 * pg_decode_lookup (rows bf16, or NF4 in the multi-head modes; e_t in bf16), B = state->B
 * <= 8; the context gate needs a bf16 state with a conv part (d and M as in args). The
 * workspace (device, 16-byte aligned, >= pg_decode_step_workspace_size bytes, owned by the
 * caller) must be zero before its first use (its first word is the grid barrier's counter:
 * every call flips its bit 31 and leaves the other bits as they were). Calls that share a
 * workspace must be ordered (one stream). Needs one block per SM resident at once (the grid barrier): PG_ERR_UNSUPPORTED
 * when the shapes leave no room for it (Din > 4096, more than 64 channels per SM). A block
 * that waits more than ~1 s at the grid barrier, or for a row of W, gives up and sets device
 * error bit 32768 or 65536; the step's outputs are then undefined. PG_ERR_WORKSPACE when it
 * is too small.
 */
pg_status pg_decode_step(const pg_table_desc* desc, const pg_decode_state* state, const int32_t* tokens,
                         const uint32_t* canon_map, const void* table, uint64_t table_bytes,
                         const pg_decode_step_args* args, void* workspace, uint64_t workspace_bytes,
                         int32_t* err_index, pg_stream_t stream);

/*
 * Correlated collisions (PageGram report 3.2, measured in 6.1): two n-grams that share a
 * page collide on each head with probability 1/S, so a pair colliding on head 0 shares
 * (K - 1)/S further heads on average; independent Engram-style subtables give about
 * 1/M_{n,k} per head.
 *
 * pg_collision_counts -- over n DISTINCT n-grams of one order, whose head rows are
 * rows[i * stride + k] (device uint32, k < K <= 16; e.g. pg_canon_hash's rows_out at one
 * position and order, stride = O * H times the positions per n-gram):
 *   counts_out[k] = number of unordered pairs {i, j} with equal head-0 rows and equal
 *   head-k rows (counts_out[0]: pairs colliding on head 0)   -- device uint64 [K]
 * so that sum_{k >= 1} counts_out[k] / counts_out[0] is the mean number of further shared
 * heads. Every head-0 row must lie in [row0_lo, row0_lo + row0_span) (the order's head-0
 * rows: PageGram base_n + [0, P_n K S), Engram the subtable of (n, 0)); one outside is
 * left out and reported as device error bit 1024, as is a head-0 group of more than 1024
 * n-grams (its pairs are left out). workspace: device, 256-byte aligned, at least
 * pg_collision_counts_workspace_size bytes. Counts are exact integers, independent of
 * scheduling. n == 0 writes zero counts.
 */
pg_status pg_collision_counts_workspace_size(int64_t n, uint32_t row0_span, size_t* bytes);

pg_status pg_collision_counts(const uint32_t* rows, int64_t n, int32_t K, int64_t stride, uint32_t row0_lo,
                              uint32_t row0_span, uint64_t* counts_out, void* workspace, size_t workspace_bytes,
                              pg_stream_t stream);

/*
 * Diagnostic, no counterpart on the pages: the memory access pattern of a lookup on its
 * own. pg_row_copy moves the rows a gather reads -- the same row indices, the same 16-byte
 * loads, a dense write -- without hashing, signs, dequantisation or concatenation, so the
 * time a gather takes can be set beside the time its rows alone take to move.
 *
 * pg_row_copy_window -- *window_bytes = the bytes copied per row: the 16-byte chunks that
 * hold a row of row_bytes bytes (row_bytes itself when it is a multiple of 16; 48 for the
 * 34-byte NF4 rows). row_bytes in [1, 4096], else PG_ERR_SHAPE.
 *
 * pg_row_copy -- output row i (out_row_bytes bytes at out + i * out_row_bytes; device,
 * 16-byte aligned) = the aligned window of `table` (device, 16-byte aligned, table_bytes
 * long) holding row rows[i] (device uint32 [n], 4-byte aligned; the row starts at byte
 * rows[i] * row_bytes), followed by zeros up to out_row_bytes: out_row_bytes = 0 takes the
 * window's size; otherwise a multiple of 16, at least the window and at most 65536 (a
 * lookup's output row, e.g. 128 bytes of bf16 e_t per 34-byte NF4 row), else PG_ERR_SHAPE.
 * A 16-byte chunk of a window that is not wholly inside the table (a row index past the
 * end) is written as zeros. n * out_row_bytes / 16 < 2^31, else PG_ERR_SHAPE; n == 0
 * enqueues nothing. One launch on `stream`.
 */
pg_status pg_row_copy_window(uint32_t row_bytes, uint32_t* window_bytes);

pg_status pg_row_copy(const void* table, uint64_t table_bytes, uint32_t row_bytes, const uint32_t* rows, int64_t n,
                      void* out, uint32_t out_row_bytes, pg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PG_H_ */
