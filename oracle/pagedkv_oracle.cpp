// Oracle for paged decode attention over a blocked KV cache.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct CPU
// definition that the CUDA library is checked against. Only the test suite, the
// smoke check and the bench's CPU-baseline leg may load it; the product path
// never calls it and shares no code with it.
//
// What it follows (pages, by title and section):
//  * "AI大模型推理速度翻倍，Colossal-Inference开源发布", section 分块式KV缓存
//    (BlockedKeyValueCache): each sequence's keys/values live in fixed-size
//    blocks; a block table maps logical block i of a sequence to a physical
//    block anywhere in the pool.
//  * same page, section KV缓存量化 (KVCache Quant): the FP8 (E5M2) KV cache;
//    the writing kernel casts fp16 to fp8, the reading kernel casts back.
//  * same page, section 分页注意力算法 (PagedAttention): decode attention reads
//    the blocks through the block table.
//  * "AI 大模型推理优化技术详解", section 2.1.2 Paged Attention: block size 16.
//  * same page, section 2.2.2 GQA: G groups of query heads, each group shares
//    one key head and one value head.
//  * same page, section 2.7 / first page section 投机采样: several draft tokens
//    are verified at once, so a sequence may carry n > 1 query tokens.
//
// Readings where the pages are silent (each is also listed in the design notes):
//  * fp16 -> E5M2 rounds to nearest, ties to even; finite values beyond the
//    largest E5M2 magnitude (57344) and +-inf saturate to +-57344; NaN becomes
//    the quiet NaN 0x7E with the input's sign.
//  * context_lens[s] counts every cached token of sequence s, including the n
//    query tokens, which are its last n positions; query token j sees
//    positions p <= ctx - n + j (causal among the query tokens).
//  * query head hq uses KV head hq / G (contiguous groups).
//  * slot -1 in a slot mapping means "do not write".
//  * INT8 KV cache (the LMDeploy section of the inference-framework survey says
//    only "KV Cache INT8 量化"): symmetric codes per (token, KV head) row:
//    scale = max|x| / 127 and code = round-half-even(x / scale) clamped to
//    [-127, 127], both divisions in fp32 (the precision the kernel decides
//    the code in); an all-zero row has scale 0 and codes 0. A cached element's
//    value is code * scale.
//
// Arithmetic is fp64 throughout (products, sums, exp), with a single final
// rounding to the query dtype done by orc_round_from_f64.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

enum { ORC_FP16 = 0, ORC_BF16 = 1, ORC_E5M2 = 2, ORC_INT8 = 3 };

// ---- scalar decodes: bit pattern -> exact double --------------------------------

// IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits.
double fp16_value(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = std::ldexp((double)m, -24);  // subnormal: m * 2^-24
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = std::ldexp((double)(1024 + m), e - 25);  // (1 + m/1024) * 2^(e-15)
  }
  return sign ? -v : v;
}

// bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits.
double bf16_value(uint16_t b) {
  const int sign = (b >> 15) & 1;
  const int e = (b >> 7) & 0xFF;
  const int m = b & 0x7F;
  double v;
  if (e == 0) {
    v = std::ldexp((double)m, -133);  // subnormal: m * 2^-133
  } else if (e == 255) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = std::ldexp((double)(128 + m), e - 134);  // (1 + m/128) * 2^(e-127)
  }
  return sign ? -v : v;
}

// E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits.
double e5m2_value(uint8_t b) {
  const int sign = (b >> 7) & 1;
  const int e = (b >> 2) & 0x1F;
  const int m = b & 0x3;
  double v;
  if (e == 0) {
    v = std::ldexp((double)m, -16);  // subnormal: m * 2^-16
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = std::ldexp((double)(4 + m), e - 17);  // (1 + m/4) * 2^(e-15)
  }
  return sign ? -v : v;
}

// ---- round a double to a binary format with p significand bits --------------------
// Plain definition of round-to-nearest-even: find the quantum (spacing of
// representable values) at |x|'s binade, clamp it from below by the
// subnormal quantum, and round x/quantum to the nearest integer with ties to
// even (std::nearbyint in the default rounding mode). Scaling by a power of
// two is exact, so the only rounding is the one we want.
double round_to_format(double x, int sig_bits, int min_exp_normal, double max_finite,
                       bool saturate) {
  if (std::isnan(x)) return x;
  if (std::isinf(x)) return saturate ? std::copysign(max_finite, x) : x;
  if (x == 0.0) return x;
  int e;
  std::frexp(std::fabs(x), &e);      // |x| = f * 2^e with f in [0.5, 1)
  int exp_unbiased = e - 1;          // |x| in [2^(e-1), 2^e)
  if (exp_unbiased < min_exp_normal) exp_unbiased = min_exp_normal;
  const int quantum_exp = exp_unbiased - (sig_bits - 1);
  const double scaled = std::ldexp(x, -quantum_exp);
  const double r = std::ldexp(std::nearbyint(scaled), quantum_exp);
  if (std::fabs(r) > max_finite) {
    return saturate ? std::copysign(max_finite, x) : std::copysign(INFINITY, x);
  }
  return r;
}

uint16_t encode_fp16(double v) {  // v must be exactly representable (or inf/nan)
  uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  if (std::isnan(v)) return sign | 0x7E00;
  double a = std::fabs(v);
  if (std::isinf(a)) return sign | 0x7C00;
  if (a == 0.0) return sign;
  if (a < std::ldexp(1.0, -14)) {                      // subnormal
    return sign | (uint16_t)std::lrint(std::ldexp(a, 24));
  }
  int e;
  double f = std::frexp(a, &e);                        // a = f * 2^e, f in [0.5,1)
  int biased = (e - 1) + 15;
  uint16_t m = (uint16_t)std::lrint((f * 2.0 - 1.0) * 1024.0);
  return sign | (uint16_t)(biased << 10) | m;
}

uint16_t encode_bf16(double v) {
  uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  if (std::isnan(v)) return sign | 0x7FC0;
  double a = std::fabs(v);
  if (std::isinf(a)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  if (a < std::ldexp(1.0, -126)) {
    return sign | (uint16_t)std::lrint(std::ldexp(a, 133));
  }
  int e;
  double f = std::frexp(a, &e);
  int biased = (e - 1) + 127;
  uint16_t m = (uint16_t)std::lrint((f * 2.0 - 1.0) * 128.0);
  return sign | (uint16_t)(biased << 7) | m;
}

uint8_t encode_e5m2(double v) {
  uint8_t sign = std::signbit(v) ? 0x80 : 0;
  if (std::isnan(v)) return sign | 0x7E;
  double a = std::fabs(v);
  if (std::isinf(a)) return sign | 0x7C;
  if (a == 0.0) return sign;
  if (a < std::ldexp(1.0, -14)) {
    return sign | (uint8_t)std::lrint(std::ldexp(a, 16));
  }
  int e;
  double f = std::frexp(a, &e);
  int biased = (e - 1) + 15;
  uint8_t m = (uint8_t)std::lrint((f * 2.0 - 1.0) * 4.0);
  return sign | (uint8_t)(biased << 2) | m;
}

// fp16 -> E5M2: exact fp16 value, rounded to 3 significand bits (RNE), with
// E5M2's subnormal floor 2^-14 and saturation at 57344. NaN -> sign|0x7E.
uint8_t e5m2_from_fp16_bits(uint16_t h) {
  const double x = fp16_value(h);
  if (std::isnan(x)) return (uint8_t)(((h >> 8) & 0x80) | 0x7E);
  const double r = round_to_format(x, /*sig_bits=*/3, /*min_exp_normal=*/-14,
                                   /*max_finite=*/57344.0, /*saturate=*/true);
  return encode_e5m2(r);
}

// The smallest fp16 value >= v (v >= 0, below the fp16 maximum): the row scale
// of an INT8 row is max|x| / 127 rounded up this way.
float round_up_to_fp16(float v) {
  if (v == 0.0f) return 0.0f;
  const uint16_t h = encode_fp16(round_to_format((double)v, 11, -14, 65504.0, false));   // nearest
  const double r = fp16_value(h);
  return (float)(r < (double)v ? fp16_value((uint16_t)(h + 1)) : r);
}

// One INT8 code: fp32 division by the row's scale, round half to even, clamp.
int8_t int8_code(float x, float scale) {
  if (scale == 0.0f) return 0;
  float q = std::nearbyint(x / scale);
  q = std::fmax(q, -127.0f);
  q = std::fmin(q, 127.0f);
  return (int8_t)q;
}

// Element idx of a cache; INT8 elements are code * scale of their row
// (scales: one float per (slot, head) row of head_size elements).
double kv_value(const void* cache, int kv_dtype, int64_t idx, const float* scales = nullptr,
                int head_size = 1) {
  if (kv_dtype == ORC_INT8) return (double)((const int8_t*)cache)[idx] * (double)scales[idx / head_size];
  if (kv_dtype == ORC_E5M2) return e5m2_value(((const uint8_t*)cache)[idx]);
  const uint16_t bits = ((const uint16_t*)cache)[idx];
  return kv_dtype == ORC_BF16 ? bf16_value(bits) : fp16_value(bits);
}

double src_value(const uint16_t* p, int dtype, int64_t idx) {
  return dtype == ORC_BF16 ? bf16_value(p[idx]) : fp16_value(p[idx]);
}

}  // namespace

extern "C" {

// Version tag so callers can check they loaded this library.
int orc_version() { return 1; }

double orc_fp16_to_f64(uint16_t h) { return fp16_value(h); }
double orc_bf16_to_f64(uint16_t b) { return bf16_value(b); }
double orc_e5m2_to_f64(uint8_t b) { return e5m2_value(b); }
uint8_t orc_e5m2_from_fp16(uint16_t h) { return e5m2_from_fp16_bits(h); }

// E5M2 back to fp16: E5M2 shares fp16's sign, exponent width and bias, so the
// fp16 pattern is the byte followed by eight zero mantissa bits. The oracle
// gets it from the value instead of the bit identity.
uint16_t orc_fp16_from_e5m2(uint8_t b) { return encode_fp16(e5m2_value(b)); }

void orc_e5m2_from_fp16_array(const uint16_t* src, uint8_t* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = e5m2_from_fp16_bits(src[i]);
}

// Round fp64 values to fp16 (dtype 0) or bf16 (dtype 1), nearest-even,
// overflow to infinity (the IEEE default).
void orc_round_from_f64(const double* src, uint16_t* dst, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) {
    if (dtype == ORC_BF16) {
      dst[i] = encode_bf16(round_to_format(src[i], 8, -126, 3.3895313892515355e38, false));
    } else {
      dst[i] = encode_fp16(round_to_format(src[i], 11, -14, 65504.0, false));
    }
  }
}

// Decode an array of fp16/bf16/E5M2 patterns to fp64.
void orc_decode_to_f64(const void* src, double* dst, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; ++i) dst[i] = kv_value(src, dtype, i);
}

// Cache write. key/value: [num_tokens][num_kv_heads][head_size] in src_dtype
// (0 fp16, 1 bf16). Caches: [num_blocks][num_kv_heads][block_size][head_size]
// in kv_dtype (0 fp16, 1 bf16, 2 E5M2; one byte per element for E5M2).
// Token t goes to physical slot slot_mapping[t] = block * block_size + offset;
// slot -1 is skipped. Returns 0, or -1 if a slot is out of range (that token
// is skipped) or the dtype pair is not one the pages describe.
int orc_kv_cache_write(const uint16_t* key, const uint16_t* value, int src_dtype,
                       int num_tokens, const int32_t* slot_mapping, void* k_cache,
                       void* v_cache, int kv_dtype, int num_blocks, int block_size,
                       int num_kv_heads, int head_size) {
  const bool ok_pair = (src_dtype == ORC_FP16 && kv_dtype == ORC_FP16) ||
                       (src_dtype == ORC_BF16 && kv_dtype == ORC_BF16) ||
                       (src_dtype == ORC_FP16 && kv_dtype == ORC_E5M2);
  if (!ok_pair) return -1;
  int rc = 0;
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) { rc = -1; continue; }
    const int64_t block = slot / block_size;
    const int64_t offset = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int d = 0; d < head_size; ++d) {
        const int64_t src = ((int64_t)t * num_kv_heads + h) * head_size + d;
        const int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * head_size + d;
        if (kv_dtype == ORC_E5M2) {
          ((uint8_t*)k_cache)[dst] = e5m2_from_fp16_bits(key[src]);
          ((uint8_t*)v_cache)[dst] = e5m2_from_fp16_bits(value[src]);
        } else {
          ((uint16_t*)k_cache)[dst] = key[src];
          ((uint16_t*)v_cache)[dst] = value[src];
        }
      }
    }
  }
  return rc;
}

// INT8 cache write: key/value fp16 [num_tokens][num_kv_heads][head_size];
// caches int8 [num_blocks][num_kv_heads][block_size][head_size]; scales float
// [num_blocks][num_kv_heads][block_size]. Codes as in the file header.
int orc_kv_cache_write_int8(const uint16_t* key, const uint16_t* value, int num_tokens,
                            const int32_t* slot_mapping, int8_t* k_cache, int8_t* v_cache,
                            float* k_scale, float* v_scale, int num_blocks, int block_size,
                            int num_kv_heads, int head_size) {
  int rc = 0;
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) { rc = -1; continue; }
    const int64_t block = slot / block_size, offset = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const int64_t row = (block * num_kv_heads + h) * block_size + offset;
      for (int which = 0; which < 2; ++which) {
        const uint16_t* src = (which ? value : key) + ((int64_t)t * num_kv_heads + h) * head_size;
        float amax = 0.0f;
        for (int d = 0; d < head_size; ++d) amax = std::fmax(amax, std::fabs((float)fp16_value(src[d])));
        const float scale = round_up_to_fp16(amax / 127.0f);
        int8_t* dst = (which ? v_cache : k_cache) + row * head_size;
        for (int d = 0; d < head_size; ++d) dst[d] = int8_code((float)fp16_value(src[d]), scale);
        (which ? v_scale : k_scale)[row] = scale;
      }
    }
  }
  return rc;
}

// Paged decode attention, fp64.
//
// q: [rows][num_q_heads][head_size] in q_dtype (fp16/bf16). With cu_q_lens NULL,
//    sequence s has q_per_seq query tokens in rows s*q_per_seq + j; otherwise it
//    has cu_q_lens[s+1] - cu_q_lens[s] tokens in rows cu_q_lens[s] + j (the
//    unpadded mixed batch of the Colossal-Inference Continuous Batching section).
// out: same layout, fp64, unnormalised nothing: out = sum_p w_p V_p.
// weights (optional, may be NULL): [num_seqs*q_per_seq][num_q_heads][weights_stride],
//    w_p for p < limit, 0 elsewhere.
// seq_subset (optional): only these sequences are computed (others untouched).
// num_threads: rows (s, j, hq) are independent; they are split over threads
//    without changing any arithmetic.
// Returns 0, or -1 on an invalid argument / block id (computation stops for
// that row and its output is set to NaN).
int orc_paged_attention(double* out, double* weights, int64_t weights_stride,
                        const uint16_t* q, int q_dtype, int num_seqs, int num_q_heads,
                        int q_per_seq, const void* k_cache, const void* v_cache,
                        int kv_dtype, int num_blocks, int block_size, int num_kv_heads,
                        int head_size, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, double scale,
                        const int32_t* seq_subset, int n_subset, int num_threads,
                        const int32_t* cu_q_lens, const uint64_t* tree_masks,
                        const float* k_scale, const float* v_scale) {
  if (kv_dtype == ORC_INT8 && (!k_scale || !v_scale)) return -1;
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
  const int group = num_q_heads / num_kv_heads;
  // Query tokens and first query row of sequence s.
  auto tokens_of = [&](int s) { return cu_q_lens ? cu_q_lens[s + 1] - cu_q_lens[s] : q_per_seq; };
  auto first_row = [&](int s) { return cu_q_lens ? (int64_t)cu_q_lens[s] : (int64_t)s * q_per_seq; };

  std::vector<int32_t> seqs;
  if (seq_subset) {
    seqs.assign(seq_subset, seq_subset + n_subset);
  } else {
    for (int s = 0; s < num_seqs; ++s) seqs.push_back(s);
  }
  // Work items: (sequence, query token j, query head hq).
  struct Row { int s, j, hq; };
  std::vector<Row> rows;
  for (int s : seqs)
    for (int j = 0; j < tokens_of(s); ++j)
      for (int hq = 0; hq < num_q_heads; ++hq) rows.push_back({s, j, hq});

  std::vector<int> bad(std::max(1, num_threads), 0);
  auto work = [&](int tid, size_t begin, size_t end) {
    std::vector<double> logits;
    for (size_t ri = begin; ri < end; ++ri) {
      const Row r = rows[ri];
      const int s = r.s, j = r.j, hq = r.hq;
      const int h = hq / group;  // KV head of this query head
      const int ctx = context_lens[s];
      const int n = tokens_of(s);
      const int64_t qrow = (first_row(s) + j) * num_q_heads + hq;
      double* o = out + qrow * head_size;
      // Query token j is position ctx - n + j. The context before the n query
      // (draft) tokens is visible to all of them; draft token i (position
      // ctx - n + i) is visible to token j when bit i of j's tree mask is set —
      // without tree masks, when i <= j (causal among the query tokens, for any n).
      const int base = ctx - n;
      const uint64_t mask = tree_masks ? tree_masks[first_row(s) + j] : 0ull;
      auto visible = [&](int p) {
        if (p < base) return true;
        const int i = p - base;
        if (!tree_masks) return i <= j;
        return i < 64 && ((mask >> i) & 1ull) != 0;
      };
      const int limit = ctx;   // positions 0 .. ctx-1 exist
      if (base < 0 || ctx > max_blocks_per_seq * block_size) {
        for (int d = 0; d < head_size; ++d) o[d] = NAN;
        bad[tid] = 1;
        continue;
      }
      // Gather position p's key/value row through the block table.
      auto kv_index = [&](int p, int64_t* idx) -> bool {
        const int32_t blk = block_tables[(int64_t)s * max_blocks_per_seq + p / block_size];
        if (blk < 0 || blk >= num_blocks) return false;
        *idx = (((int64_t)blk * num_kv_heads + h) * block_size + p % block_size) * head_size;
        return true;
      };
      logits.assign(limit, 0.0);
      bool ok = true;
      for (int p = 0; p < limit && ok; ++p) {
        if (!visible(p)) continue;
        int64_t kbase;
        if (!kv_index(p, &kbase)) { ok = false; break; }
        double dot = 0.0;
        for (int d = 0; d < head_size; ++d) {
          dot += src_value(q, q_dtype, qrow * head_size + d) *
                 kv_value(k_cache, kv_dtype, kbase + d, k_scale, head_size);
        }
        logits[p] = scale * dot;
      }
      if (!ok) {
        for (int d = 0; d < head_size; ++d) o[d] = NAN;
        bad[tid] = 1;
        continue;
      }
      // softmax over the visible positions (a row that sees none gets output 0)
      double mx = -INFINITY;
      for (int p = 0; p < limit; ++p) if (visible(p)) mx = std::max(mx, logits[p]);
      double denom = 0.0;
      for (int p = 0; p < limit; ++p) if (visible(p)) denom += std::exp(logits[p] - mx);
      for (int d = 0; d < head_size; ++d) o[d] = 0.0;
      if (weights) {
        for (int64_t p = 0; p < weights_stride; ++p) weights[qrow * weights_stride + p] = 0.0;
      }
      for (int p = 0; p < limit; ++p) {
        if (!visible(p)) continue;
        const double w = std::exp(logits[p] - mx) / denom;
        if (weights) weights[qrow * weights_stride + p] = w;
        int64_t vbase;
        kv_index(p, &vbase);
        for (int d = 0; d < head_size; ++d) o[d] += w * kv_value(v_cache, kv_dtype, vbase + d, v_scale, head_size);
      }
    }
  };

  const int nt = std::max(1, num_threads);
  if (nt == 1 || rows.size() < 2) {
    work(0, 0, rows.size());
  } else {
    std::vector<std::thread> pool;
    const size_t per = (rows.size() + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
      const size_t b = std::min(rows.size(), (size_t)t * per);
      const size_t e = std::min(rows.size(), b + per);
      if (b < e) pool.emplace_back(work, t, b, e);
    }
    for (auto& th : pool) th.join();
  }
  for (int v : bad) if (v) return -1;
  return 0;
}

// Number of hardware threads the host offers (for the CPU baseline report).
int orc_hardware_threads() {
  unsigned n = std::thread::hardware_concurrency();
  return n ? (int)n : 1;
}

}  // extern "C"
