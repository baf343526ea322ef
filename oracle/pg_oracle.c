/*
 * CPU ORACLE for the hashed multi-head N-gram lookup -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded C. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library; the product path never
 * does. It shares no code, header, table or constant generator with the CUDA
 * library: every constant below is written out here on its own.
 *
 * It computes, one token at a time and in the order the pages state them:
 *   canonical IDs -> suffix n-grams -> multiply-XOR hashes -> row indices
 *   (flat / Engram-style prime subtables / PageGram page-local slots)
 *   -> sign words -> signed rows concatenated into e_t (or summed, flat mode).
 * Row contents are passed in already fetched (rowdata), so the caller can feed
 * rows of a table of any size; the dense projection, gate and conv live in
 * oracle/dense.py (numpy, fp64).
 *
 * Sources (page title, section):
 *  - PageGram: Multi-Head N-gram Memory at the Read Cost of a Flat Table,
 *    section 2.1 (suffix n-grams of orders {2,3}; flat sum with hash sign
 *    vectors), 2.2 (multi-head addressing base_{n,k} + u_{n,k}(x) mod P_{n,k},
 *    concat of 2K heads), 3.1 (row_{n,k} = base_n + (p_n(x) K + k) S +
 *    (u_{n,k}(x) mod S), p_n = b_n mod P_n), 3.3 (NF4 row: 64 four-bit codes +
 *    one fp16 scale = 34 bytes).
 *  - Engram: conditional memory via scalable lookup (notes on arXiv 2601.07372),
 *    section 3.2 (canonical map P: V -> V'; g_{t,n} = (x'_{t-n+1},...,x'_t);
 *    z_{t,n,k} = phi_{n,k}(g_{t,n}) with a multiply-XOR hash; e_t = concat over
 *    n then k of E_{n,k}[z]).
 *  - Engram explainer ("Hash 冲突是什么样？"): teaching bucket (3a+b) mod m.
 *
 * Readings where the pages leave a step open (each one is also listed in the
 * design notes):
 *  R2  c_j = x'_{t-j}; a position before the start of its own sequence is the
 *      PAD id 0xFFFFFFFF, so every position gets all of its rows.
 *  R3  mix64 = the splitmix64 output function (Steele, Lea & Flood 2014).
 *      Multiplier m_{f,j} = mix64(seed + G*(1 + (((kind*4+o)*64+k)*4+j))) | 1
 *      with G = 0x9E3779B97F4A7C15, kind 0 = page hash b_n, 1 = head hash
 *      (u_{n,k} / phi_{n,k} / flat h_n), 2 = sign hash.
 *      h_f = XOR_j (c_j * m_{f,j}) mod 2^64; H_f = low32(h_f ^ (h_f >> 32));
 *      indices reduce H_f with '%' exactly as the formulas write it.
 *  R4  Engram subtables are stored order-major, then head-major.
 *  R5  sign word q of (o,k): mix64(h_{(2,o,k)} + G*(q+1)); element i of the head
 *      is negated iff bit (i mod 64) of word floor(i/64) is set.
 *  R6  NF4 row: byte i holds element 2i in its low nibble and 2i+1 in its high
 *      nibble; bytes 32..33 hold the fp16 scale, little-endian. value =
 *      level[code] * float(scale) in fp32, then round-to-nearest-even to bf16.
 *  R7  flat mode sums in fp32 in order of increasing n, starting from the first
 *      signed row (acc = s_0*T_0[..]; acc = acc + s_1*T_1[..]).
 *  R15 NF4 export (QLoRA's absmax quantisation of a 64-wide row): a = max |x_i|;
 *      scale = a rounded to fp16 (nearest, ties to even; a value that would round
 *      past 65504 saturates to 65504); s = float(scale). s = 0: every code is the
 *      exact-zero level (index 7). Otherwise y_i = x_i / s (fp32, correctly rounded)
 *      and code_i = the k minimising |y_i - level[k]| in fp32, the lowest k on ties.
 *  R16 FP8 projection operands (Engram notes 3.4: the fused W_V + M W_K GEMM runs in
 *      FP8): OCP E4M3 (bias 7, no infinities, max 448). A row x of e_t or of W is stored
 *      as q_i = E4M3(x_i / s) with s = max |x| / 448 (fp32 division; conversion rounds to
 *      nearest, ties to even, and saturates at +-448); s = 0 stores zeros. The product of
 *      two E4M3 values is exact in fp32, so the GEMM on the stored values is defined up to
 *      the order of its fp32 sums; out[t, c] = s_e[t] s_w[c] sum_k q_e[t,k] q_w[c,k].
 *  Toy: flat bigram only, row = (3a + b) mod m on canonical IDs, no row at t=0.
 */
#include <stdint.h>
#include <string.h>

#define ORC_PAD 0xFFFFFFFFu
#define ORC_NO_ROW 0xFFFFFFFFu
#define ORC_GOLDEN 0x9E3779B97F4A7C15ull

enum { ORC_FLAT = 0, ORC_ENGRAM = 1, ORC_PAGEGRAM = 2 };
enum { ORC_HASH_MULXOR = 0, ORC_HASH_TOY = 1 };
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_NF4 = 2 };

typedef struct {
  int32_t mode;
  int32_t hash_kind;
  int32_t num_orders;
  int32_t orders[4];
  int32_t K, S, r;
  uint32_t pages[4];
  uint32_t rows[4][16];
  int32_t row_dtype;
  int32_t pad_;
  uint64_t seed;
} orc_desc;

/* ------------------------------------------------------------ number formats */

/* NF4 levels: the 16 values of QLoRA's NormalFloat-4 data type as its paper prints
 * them (Dettmers et al. 2023, Appendix E), which the PageGram report (section 3.3) names
 * as the row format. They are normal quantiles at evenly spaced probabilities, 7
 * negative, an exact zero and 8 positive, outermost probability ~0.9677083, scaled so
 * the extremes are -1 and +1 (oracle/nf4_levels.py re-derives them to within 2 fp32
 * ulps). fp32 bit patterns. */
static const uint32_t ORC_NF4_BITS[16] = {
    0xbf800000u, 0xbf3239b1u, 0xbf066b30u, 0xbeca32a0u, 0xbe91a24du, 0xbe3d353fu,
    0xbdba7871u, 0x00000000u, 0x3da2faffu, 0x3e24cae3u, 0x3e7c04ddu, 0x3ead033au,
    0x3ee1a4b8u, 0x3f1007abu, 0x3f3913b3u, 0x3f800000u};

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

float orc_nf4_level(int code) { return bits_to_f32(ORC_NF4_BITS[code & 15]); }

/* IEEE binary16 -> binary32, from the format definition. */
float orc_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) << 31;
  uint32_t e = (h >> 10) & 0x1F, m = h & 0x3FF;
  if (e == 0) {
    /* zero or subnormal: m * 2^-24 (exact in fp32) */
    float v = (float)m * bits_to_f32(0x33800000u); /* 2^-24 */
    return sign ? -v : v;
  }
  if (e == 31) return bits_to_f32(sign | 0x7F800000u | (m << 13));
  return bits_to_f32(sign | ((e + 112u) << 23) | (m << 13));
}

/* binary32 -> binary16, round to nearest, ties to even, from the format definition;
 * finite values that would round past 65504 (and infinities) saturate to +-65504,
 * NaN stays NaN. */
uint16_t orc_f32_to_f16_sat(float f) {
  const uint32_t u = f32_to_bits(f);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);
  if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7BFFu);  /* >= 65520 would round to inf */
  const uint32_t e = a >> 23;
  if (e < 113u) {
    /* below 2^-14: a binary16 subnormal k * 2^-24, k = round(mantissa * 2^(e-126)) */
    const int sh = 126 - (int)e;
    if (sh > 24) return sign;
    const uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
    uint32_t k = mant >> sh;
    const uint32_t rem = mant & ((1u << sh) - 1u), half = 1u << (sh - 1);
    if (rem > half || (rem == half && (k & 1u))) k += 1u;  /* k = 0x400: smallest normal */
    return (uint16_t)(sign | k);
  }
  uint32_t h = (a >> 13) - ((127u - 15u) << 10);
  const uint32_t rem = a & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
  return (uint16_t)(sign | h);
}

/* binary32 -> bfloat16, round to nearest, ties to even (NaN stays NaN). */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u = f32_to_bits(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

float orc_bf16_to_f32(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* ------------------------------------------------------------------ hashing */

uint64_t orc_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t orc_multiplier(uint64_t seed, int kind, int o, int k, int j) {
  uint64_t fid = (uint64_t)((((kind * 4 + o) * 64 + k) * 4) + j);
  return orc_mix64(seed + ORC_GOLDEN * (1ull + fid)) | 1ull;
}

/* 64-bit multiply-XOR hash of the n-gram c[0..n-1] for function (kind, o, k). */
uint64_t orc_hash64(uint64_t seed, int kind, int o, int k, int n, const uint32_t* c) {
  uint64_t h = 0;
  for (int j = 0; j < n; ++j) h ^= (uint64_t)c[j] * orc_multiplier(seed, kind, o, k, j);
  return h;
}

uint32_t orc_fold32(uint64_t h) { return (uint32_t)(h ^ (h >> 32)); }

uint64_t orc_sign_word(uint64_t h_sign, int q) {
  return orc_mix64(h_sign + ORC_GOLDEN * (uint64_t)(q + 1));
}

/* The pages' teaching bucket: (3a + b) mod m. */
uint32_t orc_toy_bucket(uint32_t a, uint32_t b, uint32_t m) {
  return (uint32_t)((3ull * a + b) % m);
}

/* ------------------------------------------------------------- descriptors */

int orc_heads(const orc_desc* d) { return d->mode == ORC_FLAT ? 1 : d->K; }

/* Number of 64-bit sign words per (order, head). */
int orc_sign_words(const orc_desc* d) { return (d->r + 63) / 64; }

/* Start row of order o (flat, PageGram) or of subtable (o, k) (Engram). */
static uint64_t orc_base(const orc_desc* d, int o, int k) {
  uint64_t base = 0;
  if (d->mode == ORC_PAGEGRAM) {
    for (int i = 0; i < o; ++i) base += (uint64_t)d->pages[i] * d->K * d->S;
  } else if (d->mode == ORC_ENGRAM) {
    for (int i = 0; i < d->num_orders; ++i)
      for (int j = 0; j < d->K; ++j) {
        if (i == o && j == k) return base;
        base += d->rows[i][j];
      }
  } else {
    for (int i = 0; i < o; ++i) base += d->rows[i][0];
  }
  return base;
}

uint64_t orc_total_rows(const orc_desc* d) {
  uint64_t total = 0;
  if (d->mode == ORC_PAGEGRAM) {
    for (int i = 0; i < d->num_orders; ++i) total += (uint64_t)d->pages[i] * d->K * d->S;
  } else if (d->mode == ORC_ENGRAM) {
    for (int i = 0; i < d->num_orders; ++i)
      for (int j = 0; j < d->K; ++j) total += d->rows[i][j];
  } else {
    for (int i = 0; i < d->num_orders; ++i) total += d->rows[i][0];
  }
  return total;
}

/* -------------------------------------------------------------- addressing */

/*
 * Rows and sign words for the tokens listed in `which` (flat indices into the
 * [B, L] token array), or for all B*L tokens in order when which == NULL.
 * Outputs, per listed token i:
 *   canon_out[i]                      canonical ID x'_t            (may be NULL)
 *   rows_out[(i*O + o)*H + k]         table row of (order o, head k); H = K, or 1 flat
 *   sign_out[((i*O + o)*H + k)*W + q] sign word q                    (may be NULL)
 * canon_map == NULL means the identity map. Returns the smallest flat index of a
 * token outside [0, V) that any listed token's n-grams read, or -1.
 */
int64_t orc_index(const orc_desc* d, const int32_t* tokens, int64_t B, int64_t L,
                  const uint32_t* canon_map, uint32_t V, const int64_t* which,
                  int64_t n_which, uint32_t* canon_out, uint32_t* rows_out,
                  uint64_t* sign_out) {
  const int O = d->num_orders, H = orc_heads(d), W = orc_sign_words(d);
  const int64_t n = which ? n_which : B * L;
  int64_t bad = -1;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t flat = which ? which[i] : i;
    const int64_t b = flat / L, t = flat % L;
    /* canonical window c_j = x'_{t-j}, j = 0..3 */
    uint32_t c[4];
    for (int j = 0; j < 4; ++j) {
      if (t - j < 0) { c[j] = ORC_PAD; continue; }
      int64_t src = b * L + (t - j);
      int32_t x = tokens[src];
      if (x < 0 || (uint32_t)x >= V) {
        if (bad < 0 || src < bad) bad = src;
        x = 0;
      }
      c[j] = canon_map ? canon_map[x] : (uint32_t)x;
    }
    if (canon_out) canon_out[i] = c[0];
    for (int o = 0; o < O; ++o) {
      const int nord = d->orders[o];
      for (int k = 0; k < H; ++k) {
        uint32_t row;
        if (d->hash_kind == ORC_HASH_TOY) {
          row = (t >= 1) ? orc_toy_bucket(c[1], c[0], d->rows[0][0]) : ORC_NO_ROW;
        } else if (d->mode == ORC_PAGEGRAM) {
          uint32_t p = orc_fold32(orc_hash64(d->seed, 0, o, 0, nord, c)) % d->pages[o];
          uint32_t slot = orc_fold32(orc_hash64(d->seed, 1, o, k, nord, c)) % (uint32_t)d->S;
          row = (uint32_t)(orc_base(d, o, 0) + ((uint64_t)p * d->K + k) * d->S + slot);
        } else if (d->mode == ORC_ENGRAM) {
          uint32_t z = orc_fold32(orc_hash64(d->seed, 1, o, k, nord, c)) % d->rows[o][k];
          row = (uint32_t)(orc_base(d, o, k) + z);
        } else {
          uint32_t z = orc_fold32(orc_hash64(d->seed, 1, o, 0, nord, c)) % d->rows[o][0];
          row = (uint32_t)(orc_base(d, o, 0) + z);
        }
        rows_out[(i * O + o) * H + k] = row;
        if (sign_out) {
          uint64_t hs = orc_hash64(d->seed, 2, o, k, nord, c);
          for (int q = 0; q < W; ++q)
            sign_out[((i * O + o) * H + k) * W + q] =
                d->hash_kind == ORC_HASH_TOY ? 0ull : orc_sign_word(hs, q);
        }
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------ row assembly */

static int sign_bit(const uint64_t* words, int i) { return (int)((words[i / 64] >> (i % 64)) & 1ull); }

/* Element i of one stored row as fp32 (NF4: level * scale, one fp32 multiply). */
static float row_value(const orc_desc* d, const uint8_t* row, int i) {
  if (d->row_dtype == ORC_F32) {
    uint32_t u; memcpy(&u, row + 4 * i, 4); return bits_to_f32(u);
  }
  if (d->row_dtype == ORC_BF16) {
    uint16_t u; memcpy(&u, row + 2 * i, 2); return orc_bf16_to_f32(u);
  }
  uint8_t byte = row[i / 2];
  int code = (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
  uint16_t sbits = (uint16_t)(row[32] | ((uint16_t)row[33] << 8));
  return orc_nf4_level(code) * orc_f16_to_f32(sbits);
}

static int row_bytes(const orc_desc* d) {
  return d->row_dtype == ORC_NF4 ? 34 : d->r * (d->row_dtype == ORC_F32 ? 4 : 2);
}

static void store(void* e, int64_t idx, float v, int out_dtype) {
  if (out_dtype == ORC_F32) ((float*)e)[idx] = v;
  else ((uint16_t*)e)[idx] = orc_f32_to_bf16(v);
}

/*
 * e_t for n tokens from their fetched rows.
 *   rowdata [n, O, H, row_bytes]  the stored bytes of each addressed row
 *   signs   [n, O, H, W]          sign words from orc_index
 *   e_out   multi-head: [n, O*K*r], element (o*K + k)*r + i = s_{o,k,i} * row_{o,k}[i]
 *           flat: [n, r] (r = d), element i = sum over o of s_{o,i} * row_o[i]
 * A row index of ORC_NO_ROW (toy mode, t = 0) contributes zeros. out_dtype is
 * ORC_F32 or ORC_BF16. Returns 0, or -1 for an unsupported combination.
 */
int orc_assemble(const orc_desc* d, int64_t n, const uint32_t* rows, const uint8_t* rowdata,
                 const uint64_t* signs, int out_dtype, void* e_out) {
  const int O = d->num_orders, H = orc_heads(d), W = orc_sign_words(d), r = d->r;
  const int rb = row_bytes(d);
  if (out_dtype != ORC_F32 && out_dtype != ORC_BF16) return -1;
  if (d->row_dtype == ORC_F32 && out_dtype != ORC_F32) return -1;
  if (d->mode == ORC_FLAT && d->row_dtype == ORC_NF4) return -1;
  for (int64_t t = 0; t < n; ++t) {
    if (d->mode == ORC_FLAT) {
      for (int i = 0; i < r; ++i) {
        float acc = 0.0f;
        for (int o = 0; o < O; ++o) {
          const int64_t item = t * O + o;
          float v = 0.0f;
          if (rows[item] != ORC_NO_ROW) {
            v = row_value(d, rowdata + item * rb, i);
            if (sign_bit(signs + item * W, i)) v = -v;
          }
          acc = (o == 0) ? v : acc + v;
        }
        store(e_out, t * r + i, acc, out_dtype);
      }
    } else {
      const int64_t width = (int64_t)O * H * r;
      for (int o = 0; o < O; ++o)
        for (int k = 0; k < H; ++k) {
          const int64_t item = (t * O + o) * H + k;
          for (int i = 0; i < r; ++i) {
            float v = 0.0f;
            if (rows[item] != ORC_NO_ROW) {
              v = row_value(d, rowdata + item * rb, i);
              if (sign_bit(signs + item * W, i)) v = -v;
            }
            store(e_out, t * width + (int64_t)(o * H + k) * r + i, v, out_dtype);
          }
        }
    }
  }
  return 0;
}

/* NF4 export of n rows of 64 fp32 values into 34-byte rows (R6 layout, R15 rule). */
void orc_nf4_quantize(const float* x, int64_t n, uint8_t* out) {
  for (int64_t row = 0; row < n; ++row) {
    const float* xr = x + row * 64;
    uint8_t* o = out + row * 34;
    float a = 0.0f;
    for (int i = 0; i < 64; ++i) {
      const float v = xr[i] < 0.0f ? -xr[i] : xr[i];
      if (v > a) a = v;
    }
    const uint16_t sbits = orc_f32_to_f16_sat(a);
    const float s = orc_f16_to_f32(sbits);
    int code[64];
    for (int i = 0; i < 64; ++i) {
      if (s == 0.0f) {
        code[i] = 7;
        continue;
      }
      const float y = xr[i] / s;
      int best = 0;
      float dbest = y - orc_nf4_level(0);
      if (dbest < 0.0f) dbest = -dbest;
      for (int k = 1; k < 16; ++k) {
        float dk = y - orc_nf4_level(k);
        if (dk < 0.0f) dk = -dk;
        if (dk < dbest) {
          dbest = dk;
          best = k;
        }
      }
      code[i] = best;
    }
    for (int i = 0; i < 32; ++i) o[i] = (uint8_t)(code[2 * i] | (code[2 * i + 1] << 4));
    o[32] = (uint8_t)(sbits & 0xFFu);
    o[33] = (uint8_t)(sbits >> 8);
  }
}

/* binary32 -> OCP FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, S.1111.111 = NaN, max finite 448), round to nearest, ties to even, from the
 * format definition; values that would round past 448 saturate to +-448, NaN stays NaN. */
uint8_t orc_f32_to_e4m3_sat(float f) {
  const uint32_t u = f32_to_bits(f);
  const uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(sign | 0x7Fu);
  if (a > 0x43E80000u) return (uint8_t)(sign | 0x7Eu);  /* > 464: would round to 480 */
  const uint32_t e = a >> 23;
  if (e < 121u) {
    /* below 2^-6: a subnormal k * 2^-9, k = round(mantissa * 2^(e-141)) */
    const int sh = 141 - (int)e;
    if (sh > 24) return sign;
    const uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
    uint32_t k = mant >> sh;
    const uint32_t rem = mant & ((1u << sh) - 1u), half = 1u << (sh - 1);
    if (rem > half || (rem == half && (k & 1u))) k += 1u;  /* k = 8: smallest normal */
    return (uint8_t)(sign | k);
  }
  uint32_t h = (a >> 20) - ((127u - 7u) << 3);
  const uint32_t rem = a & 0xFFFFFu;
  if (rem > 0x80000u || (rem == 0x80000u && (h & 1u))) h += 1u;
  return (uint8_t)(sign | h);
}

/* OCP FP8 E4M3 -> binary32 (exact). */
float orc_e4m3_to_f32(uint8_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  float v;
  if (e == 15u && m == 7u) return bits_to_f32(0x7FC00000u);
  if (e == 0u) v = (float)m * bits_to_f32(0x3B000000u); /* m * 2^-9 */
  else v = bits_to_f32(((e + 120u) << 23) | (m << 20));
  return (b & 0x80u) ? -v : v;
}

/* FP8 rows (R16): n rows of `cols` fp32 values -> E4M3 bytes [n, cols] and scales [n]. */
void orc_fp8_quantize(const float* x, int64_t n, int64_t cols, uint8_t* q, float* scale) {
  for (int64_t row = 0; row < n; ++row) {
    const float* xr = x + row * cols;
    float a = 0.0f;
    for (int64_t i = 0; i < cols; ++i) {
      const float v = xr[i] < 0.0f ? -xr[i] : xr[i];
      if (v > a) a = v;
    }
    const float s = a / 448.0f;
    scale[row] = s;
    for (int64_t i = 0; i < cols; ++i) q[row * cols + i] = s == 0.0f ? 0u : orc_f32_to_e4m3_sat(xr[i] / s);
  }
}
