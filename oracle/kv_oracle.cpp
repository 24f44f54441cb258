// NVFP4 KV-cache oracle: a plain, slow CPU restatement of the method.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this file:
// only the test suite, the smoke check and the CPU-baseline leg of the benchmark use it.
// It shares no code, header, table or constant generator with the CUDA library.
//
// Sources (web pages, cited by address and section):
//   [NVFP4]  prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)":
//            K and V stored as 4-bit E2M1 codes with one E4M3 scale per 16 elements, scales
//            kept in natural row-major order, a Hadamard rotation applied to K (and Q) before
//            quantisation with V left unrotated, Q and K both quantised, V dequantised for P.V,
//            and 144 bytes per token per KV head (versus 264 for int8 and 512 for bf16).
//   [YaRN]   same page, section "YaRN context extension": theta = 1e7, 25 % of the head dims
//            rotary, linear position scaling (no NTK-by-parts) from 262k to 600k.
//
// Readings where the pages are silent (each one is listed in the design notes):
//   * RoPE pairs dimension i with i + rot_dim/2 (half-split), angle = (pos / f) * theta^(-2i/rot_dim),
//     cos/sin evaluated in double and rounded once to fp32; products rounded separately.
//   * The Hadamard rotation is the Sylvester-ordered 128-point Walsh-Hadamard transform, butterfly
//     stages h = 1, 2, 4, ..., 64 in that order, followed by one multiply by fp32 rn(2^-3.5), so
//     that the transform is orthonormal.
//   * Block scale = E4M3 round-to-nearest-even of (amax / 6), saturating at 448; no per-tensor
//     scale. Codes = E2M1 round-to-nearest-even of (x / decoded scale), saturating at 6, sign kept
//     (so -0 encodes as 0x8); a block whose scale decodes to 0 stores all-zero codes.
//   * Element 2j sits in the low nibble of byte j, element 2j+1 in the high nibble.
//   * Attention is softmax(q.k * scale) v over the dequantised values, computed here in double.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math: every fp32
// operation below must round exactly once, as written).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// ---------------------------------------------------------------------------------------------
// E2M1 (4-bit float: 1 sign, 2 exponent, 1 mantissa bit, exponent bias 1, no inf/nan).
// Magnitude codes 0..7 are the grid {0, 0.5, 1, 1.5, 2, 3, 4, 6}. [NVFP4]
// ---------------------------------------------------------------------------------------------
float orc_e2m1_decode(uint8_t code) {
  const int s = (code >> 3) & 1;
  const int e = (code >> 1) & 3;
  const int m = code & 1;
  double v;
  if (e == 0) {
    v = 0.5 * m;  // subnormal: m * 2^(1-bias) * 2^-1
  } else {
    v = std::ldexp(1.0 + 0.5 * m, e - 1);
  }
  return (float)(s ? -v : v);
}

// Nearest grid value, ties to the even magnitude code, saturating at 6; sign taken from x.
uint8_t orc_e2m1_encode(float x) {
  const double a = std::fabs((double)x);
  int best = 7;
  if (!(a >= 6.0)) {
    // Scan the grid upward. A tie can only be between two neighbouring codes, exactly one of
    // which is even, so on a tie the even candidate wins.
    best = 0;
    double best_err = a;
    for (int c = 1; c < 8; ++c) {
      const double err = std::fabs(a - (double)orc_e2m1_decode((uint8_t)c));
      if (err < best_err || (err == best_err && c % 2 == 0)) {
        best_err = err;
        best = c;
      }
    }
  }
  const uint8_t sign = std::signbit(x) ? 0x8 : 0x0;
  return (uint8_t)(sign | best);
}

// ---------------------------------------------------------------------------------------------
// E4M3 ("fn" variant: 1 sign, 4 exponent, 3 mantissa bits, bias 7, no inf, NaN = S.1111.111).
// ---------------------------------------------------------------------------------------------
float orc_e4m3_decode(uint8_t code) {
  const int s = code >> 7;
  const int e = (code >> 3) & 15;
  const int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) {
    v = std::ldexp((double)m, -9);  // subnormal: m/8 * 2^(1-7)
  } else {
    v = std::ldexp(1.0 + m / 8.0, e - 7);
  }
  return (float)(s ? -v : v);
}

// Round a non-negative value to the nearest finite E4M3 value, ties to the even code,
// saturating at 448 (code 0x7E). Codes 0x00..0x7E are increasing in value, so a binary search
// finds the pair that brackets t.
uint8_t orc_e4m3_encode(float t) {
  if (!(t > 0.0f)) return 0;  // zero (and -0) encode as +0; negative input is out of contract
  if (t >= 448.0f) return 0x7E;
  int lo = 0, hi = 0x7E;  // invariant: value(lo) <= t < value(hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if ((double)orc_e4m3_decode((uint8_t)mid) <= (double)t) lo = mid; else hi = mid;
  }
  const double dl = (double)t - (double)orc_e4m3_decode((uint8_t)lo);
  const double dh = (double)orc_e4m3_decode((uint8_t)hi) - (double)t;
  if (dl < dh) return (uint8_t)lo;
  if (dh < dl) return (uint8_t)hi;
  return (uint8_t)((lo % 2 == 0) ? lo : hi);
}

// ---------------------------------------------------------------------------------------------
// bf16 -> fp32 (exact widening).
// ---------------------------------------------------------------------------------------------
float orc_bf16_to_float(uint16_t h) {
  const uint32_t bits = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

// ---------------------------------------------------------------------------------------------
// RoPE table [YaRN]. Layout: table[pos * rot_dim + i] = cos, table[pos * rot_dim + rot_dim/2 + i]
// = sin, for i < rot_dim/2. inv_freq_i = theta^(-2i/rot_dim); angle = (pos / pos_scale) * inv_freq_i.
// ---------------------------------------------------------------------------------------------
void orc_rope_table(int32_t max_pos, int32_t rot_dim, double theta, double pos_scale, float* table) {
  const int half = rot_dim / 2;
  for (int32_t p = 0; p < max_pos; ++p) {
    for (int i = 0; i < half; ++i) {
      const double inv_freq = std::pow(theta, -(2.0 * i) / (double)rot_dim);
      const double angle = ((double)p / pos_scale) * inv_freq;
      table[(int64_t)p * rot_dim + i] = (float)std::cos(angle);
      table[(int64_t)p * rot_dim + half + i] = (float)std::sin(angle);
    }
  }
}

// Rotate the first rot_dim dims of one 128-dim row in place (fp32, each product rounded once).
void orc_rope_apply(float* x, const float* table, int32_t pos, int32_t rot_dim) {
  const int half = rot_dim / 2;
  const float* c = table + (int64_t)pos * rot_dim;
  const float* s = c + half;
  for (int i = 0; i < half; ++i) {
    const float a = x[i];
    const float b = x[i + half];
    const float ac = a * c[i];
    const float bs = b * s[i];
    const float bc = b * c[i];
    const float as = a * s[i];
    x[i] = ac - bs;
    x[i + half] = bc + as;
  }
}

// ---------------------------------------------------------------------------------------------
// Normalised 128-point Walsh-Hadamard transform [NVFP4 "Hadamard rotation"], in place.
// ---------------------------------------------------------------------------------------------
float orc_fwht_scale(void) { return (float)std::ldexp(std::sqrt(2.0), -4); }  // rn(2^-3.5)

void orc_fwht128(float* x) {
  for (int h = 1; h < 128; h *= 2) {
    for (int i = 0; i < 128; i += 2 * h) {
      for (int j = i; j < i + h; ++j) {
        const float a = x[j];
        const float b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
    }
  }
  const float c = orc_fwht_scale();
  for (int j = 0; j < 128; ++j) x[j] = x[j] * c;
}

// ---------------------------------------------------------------------------------------------
// NVFP4 quantisation of one 128-element row: 64 code bytes + 8 scale bytes [NVFP4].
// ---------------------------------------------------------------------------------------------
void orc_quantize_row(const float* x, uint8_t* codes, uint8_t* scales) {
  for (int b = 0; b < 8; ++b) {
    float amax = 0.0f;
    for (int j = 0; j < 16; ++j) {
      const float a = std::fabs(x[16 * b + j]);
      if (a > amax) amax = a;
    }
    const float t = amax / 6.0f;
    const uint8_t sc = orc_e4m3_encode(t);
    const float sd = orc_e4m3_decode(sc);
    scales[b] = sc;
    for (int j = 0; j < 16; j += 2) {
      uint8_t lo = 0, hi = 0;
      if (sd != 0.0f) {
        lo = orc_e2m1_encode(x[16 * b + j] / sd);
        hi = orc_e2m1_encode(x[16 * b + j + 1] / sd);
      }
      codes[8 * b + j / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

// The whole per-row pipeline for many rows: widen bf16, optionally RoPE + Hadamard, quantise.
//   rows:     bf16 bit patterns [n_rows][128]
//   pos:      position of each row (used only when rotate != 0)
//   rotate:   1 for Q and K rows (RoPE then Hadamard), 0 for V rows (quantise only)
//   codes:    out [n_rows][64]; scales: out [n_rows][8]
void orc_quantize_rows(const uint16_t* rows, int64_t n_rows, const int32_t* pos, int32_t rotate,
                       const float* rope_table, int32_t rot_dim, uint8_t* codes, uint8_t* scales,
                       int32_t nthreads) {
#ifdef _OPENMP
  const int nt_used = nthreads > 0 ? nthreads : omp_get_max_threads();  // global setting kept
#pragma omp parallel for num_threads(nt_used) schedule(static)
#endif
  for (int64_t r = 0; r < n_rows; ++r) {
    float x[128];
    for (int d = 0; d < 128; ++d) x[d] = orc_bf16_to_float(rows[r * 128 + d]);
    if (rotate) {
      if (rot_dim > 0) orc_rope_apply(x, rope_table, pos[r], rot_dim);
      orc_fwht128(x);
    }
    orc_quantize_row(x, codes + r * 64, scales + r * 8);
  }
}

// Dequantise one row exactly (every value e2m1 * e4m3 is exact in double).
static void dequant_row(const uint8_t* codes, const uint8_t* scales, double* out) {
  for (int d = 0; d < 128; ++d) {
    const uint8_t byte = codes[d / 2];
    const uint8_t code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    out[d] = (double)orc_e2m1_decode(code) * (double)orc_e4m3_decode(scales[d / 16]);
  }
}

void orc_dequant_rows(const uint8_t* codes, const uint8_t* scales, int64_t n_rows, double* out) {
  for (int64_t r = 0; r < n_rows; ++r) dequant_row(codes + r * 64, scales + r * 8, out + r * 128);
}

// ---------------------------------------------------------------------------------------------
// Paged layout. A pool is num_pages blocks of H * 9216 bytes (H = kv_heads), one block per page
// of 64 token slots holding every head: [K codes, H x 4096][K scales, H x 512][V codes, H x 4096]
// [V scales, H x 512]. K codes of head h are kept in 8-slot x 16-byte tiles: byte j of slot k is
// at h*4096 + (k/8)*512 + (j/16)*128 + (k%8)*16 + (j%16). K scale b of slot k of head h sits in
// the region of head pair h/2 (1024 bytes at H*4096 + (h/2)*1024): with c = b/4 (the 64-dim half)
// it is at c*512 + (k%32)*16 + (h%2)*8 + (k/32)*4 + b%4 for a full pair, and for a last head
// without a partner (odd H) at c*256 + (k%32)*8 + (k/32)*4 + b%4. V codes and V scales are
// row-major per slot. Token `pos` of sequence `seq` lives in page
// block_table[seq * max_pages + pos / 64], slot pos % 64. This gathers rows
// [n_tok][kv_heads][64 | 8] back out of a pool so that they can be compared with oracle arrays.
// Returns the number of rows whose page id was outside the pool.
// ---------------------------------------------------------------------------------------------
static int64_t blk_kscale_pair(int64_t H, int32_t h) { return H * 4096 + (int64_t)(h / 2) * 1024; }

int64_t orc_paged_gather(const uint8_t* pool, int32_t num_pages, int32_t kv_heads,
                         const int32_t* block_table, int32_t max_pages, int32_t seq,
                         int32_t pos0, int32_t n_tok, uint8_t* k_codes, uint8_t* k_scales,
                         uint8_t* v_codes, uint8_t* v_scales) {
  int64_t bad = 0;
  const int64_t H = kv_heads;
  for (int32_t i = 0; i < n_tok; ++i) {
    const int32_t pos = pos0 + i;
    const int32_t page = block_table[(int64_t)seq * max_pages + pos / 64];
    const int32_t k = pos % 64;
    for (int32_t h = 0; h < kv_heads; ++h) {
      const int64_t row = (int64_t)i * kv_heads + h;
      uint8_t* kc = k_codes + row * 64;
      uint8_t* ks = k_scales + row * 8;
      uint8_t* vc = v_codes + row * 64;
      uint8_t* vs = v_scales + row * 8;
      if (page < 0 || page >= num_pages) {
        std::memset(kc, 0, 64);
        std::memset(ks, 0, 8);
        std::memset(vc, 0, 64);
        std::memset(vs, 0, 8);
        ++bad;
        continue;
      }
      const uint8_t* blk = pool + (int64_t)page * H * 9216;
      for (int j = 0; j < 64; ++j)
        kc[j] = blk[h * 4096 + (k / 8) * 512 + (j / 16) * 128 + (k % 8) * 16 + (j % 16)];
      const int64_t pair = blk_kscale_pair(H, h);
      for (int b = 0; b < 8; ++b) {
        const int64_t c = b / 4, within = (h % 2 == 1 || h + 1 < H)
                                              ? c * 512 + (k % 32) * 16 + (h % 2) * 8 + (k / 32) * 4
                                              : c * 256 + (k % 32) * 8 + (k / 32) * 4;
        ks[b] = blk[pair + within + b % 4];
      }
      std::memcpy(vc, blk + H * 4608 + h * 4096 + k * 64, 64);
      std::memcpy(vs, blk + H * 8704 + h * 512 + k * 8, 8);
    }
  }
  return bad;
}

// ---------------------------------------------------------------------------------------------
// Attention over the dequantised cache, one output row per requested (seq, query token, q head).
//   Cache arrays are per token, contiguous per sequence: row index (tok_off[s] + pos) * kv_heads + h.
//   q rows: index (s * q_len + i) * q_heads + head. Query token i of sequence s sits at position
//   seq_lens[s] - q_len + i; with causal != 0 it sees keys at positions <= its own, otherwise all
//   seq_lens[s] keys. kv head = head / (q_heads / kv_heads).
//   Scores, softmax and the weighted sum are evaluated in double; the result is rounded to fp32.
// ---------------------------------------------------------------------------------------------
void orc_attention_rows(int32_t q_heads, int32_t kv_heads, int32_t q_len, int32_t causal,
                        double sm_scale, const int32_t* seq_lens, const int64_t* tok_off,
                        const uint8_t* q_codes, const uint8_t* q_scales, const uint8_t* k_codes,
                        const uint8_t* k_scales, const uint8_t* v_codes, const uint8_t* v_scales,
                        int64_t n_rows, const int32_t* row_seq, const int32_t* row_tok,
                        const int32_t* row_head, float* out, int32_t nthreads) {
  const int32_t group = q_heads / kv_heads;
#ifdef _OPENMP
  const int nt_used = nthreads > 0 ? nthreads : omp_get_max_threads();  // global setting kept
#pragma omp parallel for num_threads(nt_used) schedule(dynamic, 1)
#endif
  for (int64_t r = 0; r < n_rows; ++r) {
    const int32_t s = row_seq[r], i = row_tok[r], head = row_head[r];
    const int32_t kvh = head / group;
    const int32_t len = seq_lens[s];
    const int32_t n_vis = causal ? (len - q_len + i + 1) : len;
    double q[128], k[128], v[128];
    const int64_t qrow = ((int64_t)s * q_len + i) * q_heads + head;
    dequant_row(q_codes + qrow * 64, q_scales + qrow * 8, q);
    std::vector<double> score((size_t)n_vis);
    double mx = -INFINITY;
    for (int32_t t = 0; t < n_vis; ++t) {
      const int64_t krow = (tok_off[s] + t) * kv_heads + kvh;
      dequant_row(k_codes + krow * 64, k_scales + krow * 8, k);
      double dot = 0.0;
      for (int d = 0; d < 128; ++d) dot += q[d] * k[d];
      score[t] = dot * sm_scale;
      if (score[t] > mx) mx = score[t];
    }
    double acc[128] = {0.0};
    double denom = 0.0;
    for (int32_t t = 0; t < n_vis; ++t) {
      const double p = std::exp(score[t] - mx);
      denom += p;
      const int64_t vrow = (tok_off[s] + t) * kv_heads + kvh;
      dequant_row(v_codes + vrow * 64, v_scales + vrow * 8, v);
      for (int d = 0; d < 128; ++d) acc[d] += p * v[d];
    }
    for (int d = 0; d < 128; ++d) out[r * 128 + d] = (float)(acc[d] / denom);
  }
}

// Same attention on the unquantised inputs: bf16 q/k/v widened to fp32, RoPE applied to q and k
// in fp32 exactly as in the quantised path, no Hadamard rotation, no quantisation; the rest in
// double. Used only to report cosine similarity of the method against unquantised attention.
void orc_attention_ref_rows(int32_t q_heads, int32_t kv_heads, int32_t q_len, int32_t causal,
                            double sm_scale, const int32_t* seq_lens, const int64_t* tok_off,
                            const uint16_t* q_bf16, const uint16_t* k_bf16,
                            const uint16_t* v_bf16, const float* rope_table, int32_t rot_dim,
                            int64_t n_rows, const int32_t* row_seq, const int32_t* row_tok,
                            const int32_t* row_head, float* out, int32_t nthreads) {
  const int32_t group = q_heads / kv_heads;
#ifdef _OPENMP
  const int nt_used = nthreads > 0 ? nthreads : omp_get_max_threads();  // global setting kept
#pragma omp parallel for num_threads(nt_used) schedule(dynamic, 1)
#endif
  for (int64_t r = 0; r < n_rows; ++r) {
    const int32_t s = row_seq[r], i = row_tok[r], head = row_head[r];
    const int32_t kvh = head / group;
    const int32_t len = seq_lens[s];
    const int32_t qpos = len - q_len + i;
    const int32_t n_vis = causal ? (qpos + 1) : len;
    float qf[128], kf[128];
    const int64_t qrow = ((int64_t)s * q_len + i) * q_heads + head;
    for (int d = 0; d < 128; ++d) qf[d] = orc_bf16_to_float(q_bf16[qrow * 128 + d]);
    if (rot_dim > 0) orc_rope_apply(qf, rope_table, qpos, rot_dim);
    std::vector<double> score((size_t)n_vis);
    double mx = -INFINITY;
    for (int32_t t = 0; t < n_vis; ++t) {
      const int64_t krow = (tok_off[s] + t) * kv_heads + kvh;
      for (int d = 0; d < 128; ++d) kf[d] = orc_bf16_to_float(k_bf16[krow * 128 + d]);
      if (rot_dim > 0) orc_rope_apply(kf, rope_table, t, rot_dim);
      double dot = 0.0;
      for (int d = 0; d < 128; ++d) dot += (double)qf[d] * (double)kf[d];
      score[t] = dot * sm_scale;
      if (score[t] > mx) mx = score[t];
    }
    double acc[128] = {0.0};
    double denom = 0.0;
    for (int32_t t = 0; t < n_vis; ++t) {
      const double p = std::exp(score[t] - mx);
      denom += p;
      const int64_t vrow = (tok_off[s] + t) * kv_heads + kvh;
      for (int d = 0; d < 128; ++d) acc[d] += p * (double)orc_bf16_to_float(v_bf16[vrow * 128 + d]);
    }
    for (int d = 0; d < 128; ++d) out[r * 128 + d] = (float)(acc[d] / denom);
  }
}

// ---------------------------------------------------------------------------------------------
// Storage cost per token per KV head for head_dim 128 [NVFP4 "Result"]: NVFP4 = codes + E4M3
// scales for K and for V; int8 = 128 bytes + one fp32 scale, for K and V; bf16 = 2 bytes/elem.
// ---------------------------------------------------------------------------------------------
// ---------------------------------------------------------------------------------------------
// Page spill and restore (prismix.dev/news/833001997676, section "Multi-level prefix reuse with
// host-KV safety net": cache pages copied out to host memory and copied back when needed). A page
// block holds every KV head's K and V codes and scales for its 64 slots, so moving a page is a
// byte copy of the whole block: per head, 64 slots x (64 code bytes + 8 scale bytes) for K and the
// same for V.
//   spill:   arena slot i  <- pool page page_ids[i]
//   restore: pool page page_ids[i] <- arena slot i
// A page id outside [0, num_pages) is counted and its copy skipped (the destination is left as it
// was). Returns the number of skipped ids.
// ---------------------------------------------------------------------------------------------
static int64_t orc_page_block_bytes(int32_t kv_heads) {
  const int64_t slot_bytes = 128 / 2 + 128 / 16;  // E2M1 codes + E4M3 scales of one row
  return (int64_t)kv_heads * 2 * 64 * slot_bytes;
}

int64_t orc_spill_pages(const uint8_t* pool, int32_t num_pages, int32_t kv_heads,
                        const int32_t* page_ids, int32_t n, uint8_t* arena) {
  const int64_t pb = orc_page_block_bytes(kv_heads);
  int64_t bad = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = page_ids[i];
    if (id < 0 || id >= num_pages) {
      ++bad;
      continue;
    }
    std::memcpy(arena + (int64_t)i * pb, pool + (int64_t)id * pb, (size_t)pb);
  }
  return bad;
}

int64_t orc_restore_pages(uint8_t* pool, int32_t num_pages, int32_t kv_heads,
                          const int32_t* page_ids, int32_t n, const uint8_t* arena) {
  const int64_t pb = orc_page_block_bytes(kv_heads);
  int64_t bad = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = page_ids[i];
    if (id < 0 || id >= num_pages) {
      ++bad;
      continue;
    }
    std::memcpy(pool + (int64_t)id * pb, arena + (int64_t)i * pb, (size_t)pb);
  }
  return bad;
}

// ---------------------------------------------------------------------------------------------
// Comparator formats (prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)": the
// 144-byte NVFP4 row against 264 bytes for int8 and 512 for bf16, and the upstream variant with
// NVFP4 K and fp16 V, no Hadamard rotation). Readings, for the comparators only:
//   fmt 0 (bf16):  K = bf16(RoPE(k)), V = v (bf16 as given)                    512 B/token/head
//   fmt 1 (int8):  per row (K after RoPE, V raw) s = amax / 127 in fp32, codes = RNE(x / s)
//                  clamped to [-127, 127], s stored as fp32; an all-zero row has s = 0  264 B
//   fmt 2 (k4v16): K = NVFP4 of RoPE(k) (no Hadamard), V = fp16(v)              328 B
//   Q, every format: bf16(RoPE(q)), unquantised.
// Row bytes: Q, bf16 and fp16 rows 256; int8 rows 128 codes then the fp32 scale (132); NVFP4 K
// rows 64 codes then 8 scales (72).
// Page block: one chunk per KV head in head order; a chunk holds the 64 slots of K, then of V:
//   bf16:  [K 64 x 256][V 64 x 256]
//   int8:  [K codes 64 x 128][K scales 64 x 4][V codes 64 x 128][V scales 64 x 4]
//   k4v16: [K codes 64 x 64][K scales 64 x 8][V 64 x 256]
// Inside a row, 16-byte unit u of slot k is stored at unit u ^ sw(k) (a layout choice of the
// comparator kernels, for bank-conflict-free shared-memory reads): bf16 K and V rows and fp16 V
// rows sw = k & 7; int8 K rows sw = (k & 1) * 4; int8 V rows sw = ((k / 2) & 3) * 2; NVFP4 K
// codes and every scale are stored plainly.
// ---------------------------------------------------------------------------------------------
uint16_t orc_float_to_bf16(float x) {  // round to nearest even; finite x
  uint32_t b;
  std::memcpy(&b, &x, 4);
  const uint32_t lsb = (b >> 16) & 1u;
  return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

uint16_t orc_float_to_f16(float x) {  // IEEE binary16, round to nearest even, overflow to inf
  uint32_t b;
  std::memcpy(&b, &x, 4);
  const uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
  const double a = std::fabs((double)x);
  if (a == 0.0) return sign;
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);  // past half an ulp above 65504
  int e = 0;
  std::frexp(a, &e);
  int E = e - 1;  // a in [2^E, 2^(E+1))
  if (E < -14) {  // subnormal grid k * 2^-24 (k = 1024 is the smallest normal)
    const double k = std::nearbyint(std::ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)k);
  }
  double k = std::nearbyint(std::ldexp(a, 10 - E));  // 1024 .. 2048
  if (k == 2048.0) {
    k = 1024.0;
    ++E;
  }
  if (E > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(k - 1024.0));
}

double orc_f16_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1, E = (h >> 10) & 31, m = h & 1023;
  double v;
  if (E == 0) v = std::ldexp((double)m, -24);
  else if (E == 31) v = m ? NAN : INFINITY;
  else v = std::ldexp(1024.0 + m, E - 25);
  return sign ? -v : v;
}

void orc_int8_quantize_row(const float* x, int8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int d = 0; d < 128; ++d) amax = std::fmax(amax, std::fabs(x[d]));
  const float s = amax / 127.0f;
  *scale = s;
  for (int d = 0; d < 128; ++d) {
    if (s == 0.0f) {
      codes[d] = 0;
      continue;
    }
    const float q = x[d] / s;
    double c = std::nearbyint((double)q);  // ties to even (default rounding mode)
    if (c > 127.0) c = 127.0;
    if (c < -127.0) c = -127.0;
    codes[d] = (int8_t)c;
  }
}

int32_t orc_cmp_row_bytes(int32_t fmt, int32_t kind) {  // kind 0 = Q, 1 = K, 2 = V
  if (kind == 0) return 256;
  if (fmt == 0) return 256;
  if (fmt == 1) return 132;
  return kind == 1 ? 72 : 256;
}

void orc_cmp_encode_rows(int32_t fmt, int32_t kind, const uint16_t* rows, int64_t n_rows,
                         const int32_t* pos, const float* rope_table, int32_t rot_dim,
                         uint8_t* out) {
  const int32_t rb = orc_cmp_row_bytes(fmt, kind);
  for (int64_t r = 0; r < n_rows; ++r) {
    float x[128];
    for (int d = 0; d < 128; ++d) x[d] = orc_bf16_to_float(rows[r * 128 + d]);
    if (kind != 2 && rot_dim > 0) orc_rope_apply(x, rope_table, pos[r], rot_dim);
    uint8_t* o = out + r * rb;
    if (kind == 0 || (fmt == 0 && kind == 1)) {
      for (int d = 0; d < 128; ++d) {
        const uint16_t h = orc_float_to_bf16(x[d]);
        std::memcpy(o + 2 * d, &h, 2);
      }
    } else if (fmt == 0) {  // bf16 V: the row as given
      std::memcpy(o, rows + r * 128, 256);
    } else if (fmt == 1) {
      float sc;
      orc_int8_quantize_row(x, reinterpret_cast<int8_t*>(o), &sc);
      std::memcpy(o + 128, &sc, 4);
    } else if (kind == 1) {  // k4v16 K: NVFP4 without the Hadamard rotation
      orc_quantize_row(x, o, o + 64);
    } else {  // k4v16 V: fp16
      for (int d = 0; d < 128; ++d) {
        const uint16_t h = orc_float_to_f16(x[d]);
        std::memcpy(o + 2 * d, &h, 2);
      }
    }
  }
}

void orc_cmp_decode_rows(int32_t fmt, int32_t kind, const uint8_t* in, int64_t n_rows,
                         double* out) {
  const int32_t rb = orc_cmp_row_bytes(fmt, kind);
  for (int64_t r = 0; r < n_rows; ++r) {
    const uint8_t* row = in + r * rb;
    double* o = out + r * 128;
    if (kind == 0 || fmt == 0) {
      for (int d = 0; d < 128; ++d) {
        uint16_t h;
        std::memcpy(&h, row + 2 * d, 2);
        o[d] = (double)orc_bf16_to_float(h);
      }
    } else if (fmt == 1) {
      float sc;
      std::memcpy(&sc, row + 128, 4);
      for (int d = 0; d < 128; ++d) o[d] = (double)(int8_t)row[d] * (double)sc;
    } else if (kind == 1) {
      dequant_row(row, row + 64, o);
    } else {
      for (int d = 0; d < 128; ++d) {
        uint16_t h;
        std::memcpy(&h, row + 2 * d, 2);
        o[d] = orc_f16_to_double(h);
      }
    }
  }
}

// One row of `bytes` bytes out of a stored row whose 16-byte units are permuted by u ^ sw.
static void unswizzle_row(const uint8_t* stored, int32_t bytes, int32_t sw, uint8_t* out) {
  for (int32_t j = 0; j < bytes; ++j) out[j] = stored[(((j / 16) ^ sw) * 16) + j % 16];
}

// Rows [pos0, pos0 + n_tok) of one sequence out of a comparator pool (layout above):
// k_rows / v_rows [n_tok][kv_heads][row bytes]. Returns the number of rows on pages outside the
// pool (their bytes are zeroed).
int64_t orc_cmp_paged_gather(int32_t fmt, const uint8_t* pool, int32_t num_pages,
                             int32_t kv_heads, const int32_t* block_table, int32_t max_pages,
                             int32_t seq, int32_t pos0, int32_t n_tok, uint8_t* k_rows,
                             uint8_t* v_rows) {
  const int64_t kb = orc_cmp_row_bytes(fmt, 1), vb = orc_cmp_row_bytes(fmt, 2);
  const int64_t chunk = 64 * (kb + vb);
  int64_t bad = 0;
  for (int32_t i = 0; i < n_tok; ++i) {
    const int32_t pos = pos0 + i;
    const int32_t page = block_table[(int64_t)seq * max_pages + pos / 64];
    const int32_t k = pos % 64;
    for (int32_t h = 0; h < kv_heads; ++h) {
      uint8_t* ko = k_rows + ((int64_t)i * kv_heads + h) * kb;
      uint8_t* vo = v_rows + ((int64_t)i * kv_heads + h) * vb;
      if (page < 0 || page >= num_pages) {
        std::memset(ko, 0, (size_t)kb);
        std::memset(vo, 0, (size_t)vb);
        ++bad;
        continue;
      }
      const uint8_t* c = pool + ((int64_t)page * kv_heads + h) * chunk;
      if (fmt == 0) {
        unswizzle_row(c + k * 256, 256, k & 7, ko);
        unswizzle_row(c + 64 * 256 + k * 256, 256, k & 7, vo);
      } else if (fmt == 1) {
        unswizzle_row(c + k * 128, 128, (k & 1) * 4, ko);
        std::memcpy(ko + 128, c + 64 * 128 + k * 4, 4);
        unswizzle_row(c + 64 * 132 + k * 128, 128, ((k / 2) & 3) * 2, vo);
        std::memcpy(vo + 128, c + 64 * 132 + 64 * 128 + k * 4, 4);
      } else {
        std::memcpy(ko, c + k * 64, 64);
        std::memcpy(ko + 64, c + 64 * 64 + k * 8, 8);
        unswizzle_row(c + 64 * 72 + k * 256, 256, k & 7, vo);
      }
    }
  }
  return bad;
}

// fp64 attention over given (already decoded) rows, one output row per (seq, query token, q
// head): q [(s * q_len + i) * q_heads + head][128], k / v [(tok_off[s] + pos) * kv_heads + h][128].
// Same visibility and head mapping as orc_attention_rows; result rounded to fp32.
void orc_attention_f64_rows(int32_t q_heads, int32_t kv_heads, int32_t q_len, int32_t causal,
                            double sm_scale, const int32_t* seq_lens, const int64_t* tok_off,
                            const double* q, const double* k, const double* v, int64_t n_rows,
                            const int32_t* row_seq, const int32_t* row_tok,
                            const int32_t* row_head, float* out, int32_t nthreads) {
  const int32_t group = q_heads / kv_heads;
#ifdef _OPENMP
  const int nt_used = nthreads > 0 ? nthreads : omp_get_max_threads();  // global setting kept
#pragma omp parallel for num_threads(nt_used) schedule(dynamic, 1)
#endif
  for (int64_t r = 0; r < n_rows; ++r) {
    const int32_t s = row_seq[r], i = row_tok[r], head = row_head[r];
    const int32_t kvh = head / group;
    const int32_t len = seq_lens[s];
    const int32_t qpos = len - q_len + i;
    const int32_t n_vis = causal ? (qpos + 1) : len;
    const double* qr = q + (((int64_t)s * q_len + i) * q_heads + head) * 128;
    std::vector<double> score((size_t)n_vis);
    double mx = -INFINITY;
    for (int32_t t = 0; t < n_vis; ++t) {
      const double* kr = k + ((tok_off[s] + t) * kv_heads + kvh) * 128;
      double dot = 0.0;
      for (int d = 0; d < 128; ++d) dot += qr[d] * kr[d];
      score[t] = dot * sm_scale;
      if (score[t] > mx) mx = score[t];
    }
    double acc[128] = {0.0};
    double denom = 0.0;
    for (int32_t t = 0; t < n_vis; ++t) {
      const double p = std::exp(score[t] - mx);
      denom += p;
      const double* vr = v + ((tok_off[s] + t) * kv_heads + kvh) * 128;
      for (int d = 0; d < 128; ++d) acc[d] += p * vr[d];
    }
    for (int d = 0; d < 128; ++d) out[r * 128 + d] = (float)(acc[d] / denom);
  }
}

int32_t orc_bytes_per_token_head_nvfp4(int32_t head_dim) { return 2 * (head_dim / 2 + head_dim / 16); }
int32_t orc_bytes_per_token_head_int8(int32_t head_dim) { return 2 * (head_dim + 4); }
int32_t orc_bytes_per_token_head_bf16(int32_t head_dim) { return 2 * head_dim * 2; }

int32_t orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
