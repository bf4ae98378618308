// msa_oracle.cpp — plain, slow CPU reference of the MSA decode step over an NVFP4 cache.
//
// TEST INFRASTRUCTURE. Nothing in the product path may link, load or call this file:
// only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference leg use it.
// It shares no code, header, table or constant with the CUDA library; it is written from
// the number-format definitions (OCP 8-bit floating point E4M3; OCP MX/NV 4-bit E2M1) and
// from the algorithm steps described on the pages, in fp64 where the pages fix no precision.
//
// Sources (page title, section):
//  [P1] "vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash" — "MSA primer",
//       "NVIDIA Blackwell optimizado kernes MSA", "NVIDIA Rubin MSA optimizado",
//       "NVFP4 MSA kernel" (AMD section), "Indexador NVFP4 DCP".
//  [P4] "MiniMax M3 in vLLM: Day-0 Serving for 1M-Token Multimodal Reasoning" (Chinese
//       translation) — "MSA 机制详解" (MSA mechanism), "解码执行" (decode execution),
//       "解码内核中的推测解码" (speculative decoding inside the decode kernels).
//  [P5] "MiniMax-M3.1-Flash serving notes" — "How MSA reads memory", "The capacity numbers".
//
// Every function below is pinned by tests under tests/ (marked "not gpu") against values
// that do not come from this file: torch's float8_e4m3fn table, brute-force nearest-value
// searches, hand vectors, closed-form byte counts printed on the pages, and a numpy
// textbook softmax attention over the gathered keys.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <limits>
#include <thread>
#include <vector>

namespace {

// Fixed MSA geometry ([P5] "The architecture, in operator terms"; [P1] "MSA primer").
constexpr int kHeadDim = 128;      // head dim of Q, K, V and of the index query/key
constexpr int kGroups = 4;         // KV heads = GQA groups
constexpr int kHeadsPerGroup = 16; // 64 query heads / 4 KV heads
constexpr int kQHeads = kGroups * kHeadsPerGroup;
constexpr int kBlock = 128;        // tokens per KV block = cache page
constexpr int kSel = 16;           // selected blocks per (query token, group): local + 15

// ---------------------------------------------------------------------------------------
// Number formats.
// E4M3 (OCP "E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits. No infinity;
// S.1111.111 is NaN; largest finite magnitude 448; subnormals m * 2^-9.
double e4m3_decode(uint8_t b) {
  const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double mag = (e == 0) ? std::ldexp(double(m), -9) : std::ldexp(double(8 + m), e - 10);
  return s ? -mag : mag;
}

// Round to nearest, ties to even mantissa, saturating to +-448 ("satfinite").
// The sign of the input is kept, also for results that round to zero.
uint8_t e4m3_encode(double x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  if (std::isnan(x)) return sign | 0x7F;
  const double a = std::fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  // Spacing of representable values around a: the binade [2^E, 2^(E+1)) holds 8 values
  // 2^(E-3) apart; below 2^-6 the subnormals keep the spacing 2^-9 of the first binade.
  int ex = 0;
  std::frexp(a, &ex);            // a = f * 2^ex, f in [0.5, 1)
  int E = ex - 1;                // a in [2^E, 2^(E+1))
  if (E < -6) E = -6;
  const double q = std::ldexp(1.0, E - 3);
  const double n = std::nearbyint(a / q);  // a / q is exact; nearbyint rounds half to even
  const double v = n * q;                  // <= 448 because a < 448
  if (v == 0.0) return sign;
  // Encode the representable value v exactly.
  int ev = 0;
  std::frexp(v, &ev);
  const int biased = (ev - 1) + 7;
  if (biased <= 0) {  // subnormal: v = m * 2^-9, m in 1..7
    const int m = int(v / std::ldexp(1.0, -9));
    return sign | uint8_t(m);
  }
  const int m = int((v / std::ldexp(1.0, ev - 1) - 1.0) * 8.0);
  return sign | uint8_t(biased << 3) | uint8_t(m);
}

// E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. Magnitudes by code 0..7:
// 0, 0.5, 1, 1.5, 2, 3, 4, 6.
double e2m1_decode(uint8_t c) {
  const int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  const double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

// Nearest E2M1 magnitude, ties to the even code (even mantissa), saturating to 6.
// A result of magnitude zero is always the code +0 (0x0).
uint8_t e2m1_encode(float r) {
  const bool neg = std::signbit(r);
  double a = std::fabs(double(r));
  if (a > 6.0) a = 6.0;
  int best = 0;
  double best_err = std::numeric_limits<double>::infinity();
  for (int c = 0; c < 8; ++c) {
    const double err = std::fabs(a - e2m1_decode(uint8_t(c)));
    if (err < best_err || (err == best_err && (c % 2) == 0)) {
      best = c;
      best_err = err;
    }
  }
  if (best == 0) return 0;
  return uint8_t((neg ? 8 : 0) | best);
}

// ---------------------------------------------------------------------------------------
// NVFP4 row layout of this library (the pages fix no byte layout).
// A row of C elements (C % 16 == 0) has C/2 code bytes and C/16 scale bytes.
// Scale byte k (E4M3) covers elements 16k .. 16k+15.
// The code bytes are C/8 little-endian 32-bit words; word w holds elements 8w .. 8w+7.
// Element 8w+j keeps its three magnitude bits at bits 4j .. 4j+2 of the word and its sign
// bit at bit 4*sign_slot(j)+3, with sign_slot = (1, 3, 5, 7, 0, 2, 4, 6).
int sign_slot(int j) { return j < 4 ? 2 * j + 1 : 2 * (j - 4); }

uint32_t load_word(const uint8_t* p) {
  return uint32_t(p[0]) | (uint32_t(p[1]) << 8) | (uint32_t(p[2]) << 16) | (uint32_t(p[3]) << 24);
}

void store_word(uint8_t* p, uint32_t w) {
  p[0] = uint8_t(w);
  p[1] = uint8_t(w >> 8);
  p[2] = uint8_t(w >> 16);
  p[3] = uint8_t(w >> 24);
}

void unpack_row(const uint8_t* vals, int cols, uint8_t* codes) {
  for (int e = 0; e < cols; ++e) {
    const int w = e / 8, j = e % 8;
    const uint32_t word = load_word(vals + 4 * w);
    const uint32_t mag = (word >> (4 * j)) & 7u;
    const uint32_t sgn = (word >> (4 * sign_slot(j) + 3)) & 1u;
    codes[e] = uint8_t((sgn << 3) | mag);
  }
}

void pack_row(const uint8_t* codes, int cols, uint8_t* vals) {
  for (int w = 0; w < cols / 8; ++w) {
    uint32_t word = 0;
    for (int j = 0; j < 8; ++j) {
      const uint8_t c = codes[8 * w + j];
      word |= uint32_t(c & 7) << (4 * j);
      word |= uint32_t((c >> 3) & 1) << (4 * sign_slot(j) + 3);
    }
    store_word(vals + 4 * w, word);
  }
}

// NVFP4 quantisation of one row: per 16 elements, s = E4M3(amax / 6) and
// code_i = E2M1(x_i / S) with S the decoded scale ([P5] "The capacity numbers": 4-bit values
// plus one FP8 scale per 16 values; the amax/6 scale rule and RNE rounding are this
// library's reading, the pages leave them open).
void quantize_row(const float* x, int cols, uint8_t* vals, uint8_t* scales) {
  std::vector<uint8_t> codes(size_t(cols), 0);
  for (int k = 0; k < cols / 16; ++k) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(x[16 * k + i]));
    const float sf = amax / 6.0f;  // IEEE single-precision division, round to nearest
    const uint8_t s = e4m3_encode(double(sf));
    scales[k] = s;
    const float S = float(e4m3_decode(s));
    for (int i = 0; i < 16; ++i) {
      codes[16 * k + i] = (S == 0.0f) ? uint8_t(0) : e2m1_encode(x[16 * k + i] / S);
    }
  }
  pack_row(codes.data(), cols, vals);
}

// Dequantisation of one NVFP4 element to FP8 for the FP8 MMA ([P1] "NVIDIA Blackwell
// optimizado kernes MSA": the cache is dequantised to FP8; "NVIDIA Rubin MSA optimizado":
// the Blackwell scores carry this E4M3 re-rounding; "NVFP4 MSA kernel": the value is a pure
// function of (scale byte, magnitude), pre-rounded to FP8).
// v = E4M3_RNE_sat(E2M1(c) * E4M3(s)) with IEEE sign rules: |v| from |c| and |s|, and
// sign(v) = sign(c) xor sign(s). A NaN scale gives NaN (0x7F with that sign).
uint8_t dequant_fp8(uint8_t code, uint8_t scale) {
  const double mag = std::fabs(e2m1_decode(code & 7));
  const double S = std::fabs(e4m3_decode(scale & 0x7F));
  const uint8_t m = std::isnan(S) ? uint8_t(0x7F) : e4m3_encode(mag * S);
  const uint8_t sgn = uint8_t(((code >> 3) ^ (scale >> 7)) & 1);
  return uint8_t(m | (sgn << 7));
}

// v = E2M1(c) * E4M3(s) exactly, no re-rounding: the exact-score reading of an NVFP4 index key
// ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "NVIDIA Rubin MSA optimizado": the
// index key goes from NVFP4 straight to FP16, so the scores carry no E4M3 re-rounding). The
// product has at most 2 + 4 significant bits and is exact in double. A NaN scale gives NaN.
double dequant_exact(uint8_t code, uint8_t scale) {
  const double S = e4m3_decode(scale);
  if (std::isnan(S)) return std::numeric_limits<double>::quiet_NaN();
  return e2m1_decode(code) * S;
}

// Decode one NVFP4 row of kHeadDim elements to the FP8 values the MMA would see.
void dequant_row_values(const uint8_t* vals, const uint8_t* scales, double* out) {
  uint8_t codes[kHeadDim];
  unpack_row(vals, kHeadDim, codes);
  for (int d = 0; d < kHeadDim; ++d) out[d] = e4m3_decode(dequant_fp8(codes[d], scales[d / 16]));
}

void parallel_for(int64_t n, int nthreads, const std::function<void(int64_t)>& fn) {
  if (nthreads <= 0) nthreads = int(std::max(1u, std::thread::hardware_concurrency()));
  if (n <= 1 || nthreads == 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  const int nt = int(std::min<int64_t>(n, nthreads));
  std::vector<std::thread> pool;
  pool.reserve(size_t(nt));
  for (int w = 0; w < nt; ++w) {
    pool.emplace_back([&, w]() {
      for (int64_t i = w; i < n; i += nt) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

int32_t orc_version(void) { return 1; }
int32_t orc_hardware_threads(void) { return int32_t(std::thread::hardware_concurrency()); }

double orc_e4m3_decode(uint8_t b) { return e4m3_decode(b); }
uint8_t orc_e4m3_encode(double x) { return e4m3_encode(x); }
double orc_e2m1_decode(uint8_t c) { return e2m1_decode(c); }
uint8_t orc_e2m1_encode(float r) { return e2m1_encode(r); }
uint8_t orc_dequant_fp8(uint8_t code, uint8_t scale) { return dequant_fp8(code, scale); }

// FP8 (E4M3) cast of n fp32 values: queries, index queries and the FP8 index-key cache.
void orc_quantize_fp8(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(double(x[i]));
}

// NVFP4 quantisation of rows x[rows][cols] -> vals[rows][cols/2], scales[rows][cols/16].
void orc_quantize_nvfp4(const float* x, int64_t rows, int32_t cols, uint8_t* vals, uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    quantize_row(x + r * cols, cols, vals + r * (cols / 2), scales + r * (cols / 16));
  }
}

void orc_unpack_nvfp4(const uint8_t* vals, int64_t rows, int32_t cols, uint8_t* codes) {
  for (int64_t r = 0; r < rows; ++r) unpack_row(vals + r * (cols / 2), cols, codes + r * cols);
}

void orc_pack_nvfp4(const uint8_t* codes, int64_t rows, int32_t cols, uint8_t* vals) {
  for (int64_t r = 0; r < rows; ++r) pack_row(codes + r * cols, cols, vals + r * (cols / 2));
}

// NVFP4 rows -> FP8 bytes (the dequantised operand), out[rows][cols].
void orc_dequant_nvfp4(const uint8_t* vals, const uint8_t* scales, int64_t rows, int32_t cols, uint8_t* out) {
  std::vector<uint8_t> codes(static_cast<size_t>(cols), 0);
  for (int64_t r = 0; r < rows; ++r) {
    unpack_row(vals + r * (cols / 2), cols, codes.data());
    for (int d = 0; d < cols; ++d) out[r * cols + d] = dequant_fp8(codes[d], scales[r * (cols / 16) + d / 16]);
  }
}

// Indexer score and block max-pool for one sequence ([P1] "MSA primer": one index query per
// GQA group scored against the single shared index-key head, then the max over each
// 128-token block; [P4] "MSA 机制详解": the partial last block is masked and the causal
// boundary inside a block is respected; "解码内核中的推测解码": each of the q_len query
// tokens sits at its own causal position).
//   L        tokens in the cache for this sequence (query tokens included)
//   q_len    query tokens; token t sits at position p_t = L - q_len + t
//   iq       [q_len][4][128] E4M3 index queries
//   ik_vals  NVFP4: [L][64] code bytes, ik_scales [L][8];  FP8 (index_dtype 1): [L][128]
//   index_dtype 0: NVFP4 keys re-rounded to E4M3 (the FP8 score MMA); 1: FP8 keys; 2: NVFP4
//            keys taken exactly (dequant_exact, the exact-score variant)
//   out      [q_len][4][out_stride] block scores, fp64; blocks without a valid key get -inf
void orc_indexer_seq(int32_t L, int32_t q_len, int32_t index_dtype, const uint8_t* iq,
                     const uint8_t* ik_vals, const uint8_t* ik_scales, double* out,
                     int32_t out_stride, int32_t nthreads) {
  const int nb = (L + kBlock - 1) / kBlock;
  // Exact FP8 values of every index key (FP8 values are exact in float).
  std::vector<float> key(size_t(L) * kHeadDim);  // (exact NVFP4 products are exact in float too)
  parallel_for(L, nthreads, [&](int64_t j) {
    if (index_dtype == 0) {
      double row[kHeadDim];
      dequant_row_values(ik_vals + j * (kHeadDim / 2), ik_scales + j * (kHeadDim / 16), row);
      for (int d = 0; d < kHeadDim; ++d) key[size_t(j) * kHeadDim + d] = float(row[d]);
    } else if (index_dtype == 2) {
      uint8_t codes[kHeadDim];
      unpack_row(ik_vals + j * (kHeadDim / 2), kHeadDim, codes);
      const uint8_t* sc = ik_scales + j * (kHeadDim / 16);
      for (int d = 0; d < kHeadDim; ++d) key[size_t(j) * kHeadDim + d] = float(dequant_exact(codes[d], sc[d / 16]));
    } else {
      for (int d = 0; d < kHeadDim; ++d) key[size_t(j) * kHeadDim + d] = float(e4m3_decode(ik_vals[j * kHeadDim + d]));
    }
  });
  parallel_for(int64_t(q_len) * kGroups, nthreads, [&](int64_t tg) {
    const int t = int(tg / kGroups);
    const int64_t p = int64_t(L) - q_len + t;
    double q[kHeadDim];
    for (int d = 0; d < kHeadDim; ++d) q[d] = e4m3_decode(iq[tg * kHeadDim + d]);
    double* o = out + tg * out_stride;
    for (int k = 0; k < nb; ++k) {
      double best = -std::numeric_limits<double>::infinity();
      for (int64_t j = int64_t(k) * kBlock; j < std::min<int64_t>(int64_t(k + 1) * kBlock, L); ++j) {
        if (j > p) continue;
        double s = 0.0;
        for (int d = 0; d < kHeadDim; ++d) s += q[d] * double(key[size_t(j) * kHeadDim + d]);
        best = std::max(best, s);
      }
      o[k] = best;
    }
  });
}

// Block selection for one (query token, group) row ([P1] "MSA primer": the top blocks with
// the most recent block always kept, 16 in total, 2,048 keys at most; [P4] "MSA 机制详解":
// init_blocks = 0, local_blocks = 1, and a local block that also ranks in the top-k is not
// counted twice). local = floor(p / 128). Candidates are the blocks 0 .. local-1, ranked by
// a full stable sort on score, descending, so equal scores keep the lower block id first;
// NaN ranks as -inf. sel[0] = local, sel[1..15] = the 15 best candidates in rank order,
// -1 where there are fewer.
void orc_select_row(const double* scores, int32_t nb, int32_t local, int32_t* sel) {
  std::vector<int32_t> cand;
  for (int32_t k = 0; k < std::min(local, nb); ++k) cand.push_back(k);
  auto key = [&](int32_t k) {
    const double s = scores[k];
    return std::isnan(s) ? -std::numeric_limits<double>::infinity() : s;
  };
  std::stable_sort(cand.begin(), cand.end(), [&](int32_t a, int32_t b) { return key(a) > key(b); });
  sel[0] = local;
  for (int i = 1; i < kSel; ++i) sel[i] = (i - 1 < int(cand.size())) ? cand[size_t(i - 1)] : -1;
}

// Exact GQA attention over the selected blocks for one sequence ([P1] "MSA primer": main
// attention runs exactly, only over the selected blocks, and every query head of a GQA group
// uses its group's selection; [P4] "MSA 机制详解"/"预填充执行": the result equals dense
// attention restricted to the selected set; masking of the partial block and of keys after
// the query's causal position as in orc_indexer_seq). Head h belongs to group h / 16.
//   q        [q_len][64][128] E4M3
//   k_vals   [L][4][64], k_scales [L][4][8]; v_vals, v_scales likewise (NVFP4, this layout)
//   sel      [q_len][4][16] block ids (-1 = empty); the set of listed blocks is used
//   out      [q_len][64][128] fp64;  lse (nullable) [q_len][64] natural-log sum of exp
void orc_attention_seq(int32_t L, int32_t q_len, const uint8_t* q, const uint8_t* k_vals,
                       const uint8_t* k_scales, const uint8_t* v_vals, const uint8_t* v_scales,
                       const int32_t* sel, double softmax_scale, double* out, double* lse,
                       int32_t nthreads) {
  const int nb = (L + kBlock - 1) / kBlock;
  parallel_for(int64_t(q_len) * kGroups, nthreads, [&](int64_t tg) {
    const int t = int(tg / kGroups), g = int(tg % kGroups);
    const int64_t p = int64_t(L) - q_len + t;
    std::vector<int32_t> blocks;
    for (int i = 0; i < kSel; ++i) {
      const int32_t b = sel[tg * kSel + i];
      if (b >= 0 && b < nb) blocks.push_back(b);
    }
    std::sort(blocks.begin(), blocks.end());
    blocks.erase(std::unique(blocks.begin(), blocks.end()), blocks.end());
    std::vector<int64_t> keys;
    for (int32_t b : blocks) {
      for (int64_t j = int64_t(b) * kBlock; j < std::min<int64_t>(int64_t(b + 1) * kBlock, L); ++j) {
        if (j <= p) keys.push_back(j);
      }
    }
    const size_t n = keys.size();
    std::vector<double> K(n * kHeadDim), V(n * kHeadDim);
    for (size_t i = 0; i < n; ++i) {
      const int64_t row = keys[i] * kGroups + g;
      dequant_row_values(k_vals + row * (kHeadDim / 2), k_scales + row * (kHeadDim / 16), &K[i * kHeadDim]);
      dequant_row_values(v_vals + row * (kHeadDim / 2), v_scales + row * (kHeadDim / 16), &V[i * kHeadDim]);
    }
    std::vector<double> z(n);
    for (int hh = 0; hh < kHeadsPerGroup; ++hh) {
      const int h = g * kHeadsPerGroup + hh;
      const uint8_t* qh = q + (int64_t(t) * kQHeads + h) * kHeadDim;
      double qv[kHeadDim];
      for (int d = 0; d < kHeadDim; ++d) qv[d] = e4m3_decode(qh[d]);
      double m = -std::numeric_limits<double>::infinity();
      for (size_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int d = 0; d < kHeadDim; ++d) s += qv[d] * K[i * kHeadDim + d];
        z[i] = softmax_scale * s;
        m = std::max(m, z[i]);
      }
      double l = 0.0;
      double acc[kHeadDim] = {0.0};
      for (size_t i = 0; i < n; ++i) {
        const double w = std::exp(z[i] - m);
        l += w;
        for (int d = 0; d < kHeadDim; ++d) acc[d] += w * V[i * kHeadDim + d];
      }
      double* o = out + (int64_t(t) * kQHeads + h) * kHeadDim;
      for (int d = 0; d < kHeadDim; ++d) o[d] = (n > 0) ? acc[d] / l : 0.0;
      if (lse) lse[int64_t(t) * kQHeads + h] = (n > 0) ? m + std::log(l) : -std::numeric_limits<double>::infinity();
    }
  });
}

}  // extern "C"
