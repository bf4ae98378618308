// msa_device.cuh — device-side building blocks of the MSA decode kernels (sm_103a).
//
// PTX wrappers (mbarrier, 1-D bulk async copies, mma.sync, ldmatrix, FP8 converts), the
// bounded waits every kernel uses, and the NVFP4 -> E4M3 dequantiser: a 2 KB shared-memory
// table of pre-rounded FP8 values indexed by (scale byte, E2M1 magnitude) — the table idea
// of "vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", section "NVFP4 MSA kernel" —
// read with one byte-permute per four elements and a masked xor for the signs.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"

namespace msa {

// ------------------------------------------------------------------ fixed geometry ----
constexpr int kD = 128;          // head dim = index dim
constexpr int kGroups = 4;       // KV heads
constexpr int kHPG = 16;         // query heads per group
constexpr int kQHeads = 64;
constexpr int kBS = 128;         // tokens per block = page rows
constexpr int kSel = 16;         // selected blocks per (token, group)
constexpr int kMaxQLen = 8;
constexpr int kRowCodes = kD / 2;    // 64 B
constexpr int kRowScales = kD / 16;  // 8 B
constexpr int kRegion = kBS * (kRowCodes + kRowScales);  // 9,216 B: codes of 128 rows, scales
constexpr int kScaleOff = kBS * kRowCodes;               // 8,192: scales start in a region
constexpr int kIdxPageNv = kRegion;
constexpr int kIdxPageFp8 = kBS * kD;                    // 16,384 B
constexpr int kKvPage = kGroups * 2 * kRegion;           // 73,728 B
constexpr int kMaxSplits = 16;
constexpr int kMaxB = 4096;      // sequences per call (shared-memory prefix sums)

// Default budget of every device-side wait; a correct run never gets near it.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ void set_status(uint32_t* status, int code) {
  if (status != nullptr) atomicOr(status, 1u << code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier ----------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the hardware suspend the thread for up to ~65 us while the phase is
// still open, instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(0x10000u)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete. Gives up (returns false)
// after limit_ns of %globaltimer, or early when *abort becomes non-zero.
static __device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned long long limit_ns,
                                               volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// The same, with the already-complete case (the common one) decided inline.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return mbar_try_wait(bar, parity) || mbar_wait_bounded(bar, parity, kWaitLimitNs, abort);
}

// ------------------------------------------------------------------ tensor copies -----
// L2 policy for data read exactly once (evict first).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy for data that several CTAs read again soon (evict last).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tiled tensor copy global -> shared of the tensor map's box at element (x, y), completing
// its bytes on `bar`, with an L2 cache hint. x * element size must be a multiple of 16 B.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled tensor copy global -> shared of the tensor map's box at element (x, y, z),
// completing its bytes on `bar`. x * element size must be a multiple of 16 B.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Where byte o of a 128-byte-row tile lands when a 128-byte-swizzled tensor copy writes it to a
// 1024-B aligned buffer: its 16-byte chunk index is xor-ed with the row index mod 8.
__host__ __device__ constexpr uint32_t sw128_phys(uint32_t o) { return o ^ (((o >> 7) & 7u) << 4); }

// ------------------------------------------------------------------ loads -------------
// Shared-memory loads as plain C++ so the compiler orders them against barriers and can
// still schedule them freely around the (non-volatile) MMAs.
__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }

__device__ __forceinline__ uint32_t ldg_nc32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ------------------------------------------------------------------ MMAs --------------
// D(16x8, f32) += A(16x32, e4m3, row) * B(32x8, e4m3, col)
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D(16x8, f32) = A(16x32, e4m3, row) * B(32x8, e4m3, col)   (no accumulator input)
__device__ __forceinline__ void mma_e4m3_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p))
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p))
               : "memory");
}

// ------------------------------------------------------------------ conversions -------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two fp32 -> two E4M3 bytes (round to nearest even, saturating): lo in bits 0..7.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 bytes (bits 0..15) -> f16x2, exact.
__device__ __forceinline__ uint32_t cvt_f16x2_e4m3x2(uint32_t two_bytes) {
  uint32_t r;
  const uint16_t in = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
  return r;
}

// f16x2 -> two E4M3 bytes (round to nearest even, saturating): the low half in bits 0..7.
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t add_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 2^x of both halves of an f16x2 (-inf gives +0).
__device__ __forceinline__ uint32_t exp2_f16x2(uint32_t h2) {
  uint32_t r;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(r) : "r"(h2));
  return r;
}

// The two halves of an f16x2 added (in f16), as an fp32.
__device__ __forceinline__ float sum_f16x2(uint32_t h2) {
  float f;
  asm("{\n\t.reg .f16 lo, hi, s;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f16 s, lo, hi;\n\tcvt.f32.f16 %0, s;\n\t}"
      : "=f"(f) : "r"(h2));
  return f;
}

// a * b + c on two fp32 lanes in one instruction (the packed fp32 FMA of sm_100 and later).
__device__ __forceinline__ void fma_f32x2(float a0, float a1, float b0, float b1, float c0, float c1, float& d0,
                                          float& d1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  const uint32_t h2 = cvt_f16x2_e4m3x2(byte & 0xFFu);
  float f;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ NVFP4 codec -------
// E2M1 magnitudes by code 0..7 (the FP4 format definition).
__device__ __forceinline__ float e2m1_mag(int c) {
  return c < 4 ? 0.5f * static_cast<float>(c) : (c == 4 ? 2.0f : (c == 5 ? 3.0f : (c == 6 ? 4.0f : 6.0f)));
}

// E2M1 magnitude code of a >= 0: round to nearest, ties to the even code, saturating at 6.
__device__ __forceinline__ uint32_t e2m1_code(float a) {
  return static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) + static_cast<uint32_t>(a > 1.25f) +
         static_cast<uint32_t>(a >= 1.75f) + static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) +
         static_cast<uint32_t>(a > 5.0f);
}

// Sign slot of element j (0..7) inside its 32-bit code word.
__host__ __device__ constexpr int sign_slot(int j) { return j < 4 ? 2 * j + 1 : 2 * (j - 4); }

// Fill the 256-entry dequant table: lut[s] holds, for magnitudes 0..7, the E4M3 byte of
// |E2M1(m)| * |E4M3(s)| rounded to nearest even with saturation, with the sign of s in
// bit 7 (0x7F for a NaN scale). One 8-byte entry per scale byte: 2 KB.
__device__ __forceinline__ void build_dequant_lut(uint2* lut, int tid, int nthreads) {
  for (int s = tid; s < 256; s += nthreads) {
    const uint32_t mag = static_cast<uint32_t>(s) & 0x7Fu;
    const uint32_t sgn = (static_cast<uint32_t>(s) & 0x80u) ? 0x80808080u : 0u;
    uint32_t lo, hi;
    if (mag == 0x7Fu) {
      lo = hi = 0x7F7F7F7Fu;
    } else {
      const float S = e4m3_to_f32(mag);
      lo = cvt_e4m3x2(e2m1_mag(0) * S, e2m1_mag(1) * S) | (cvt_e4m3x2(e2m1_mag(2) * S, e2m1_mag(3) * S) << 16);
      hi = cvt_e4m3x2(e2m1_mag(4) * S, e2m1_mag(5) * S) | (cvt_e4m3x2(e2m1_mag(6) * S, e2m1_mag(7) * S) << 16);
    }
    lut[s] = make_uint2(lo | sgn, hi | sgn);
  }
}

// Fill the 256-entry exact f16 table: for scale byte s, the f16 values of E2M1(m) * E4M3(s)
// for magnitudes m = 0..7 (exact: at most 6 significant bits, inside the f16 range), the sign
// of s applied, a NaN scale giving NaN; stored as byte planes, low bytes of the eight values
// in .x/.y and high bytes in .z/.w, for byte-permute lookups. 4 KB.
__device__ __forceinline__ void build_exact_lut(uint4* lut, int tid, int nthreads) {
  for (int s = tid; s < 256; s += nthreads) {
    const uint32_t mag = static_cast<uint32_t>(s) & 0x7Fu;
    uint16_t h[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (mag == 0x7Fu) {
        h[m] = 0x7E00u;
      } else {
        const __half v = __float2half_rn(e2m1_mag(m) * e4m3_to_f32(mag));
        h[m] = static_cast<uint16_t>(__half_as_ushort(v) | ((s & 0x80) ? 0x8000u : 0u));
      }
    }
    uint32_t lo[2] = {0u, 0u}, hi[2] = {0u, 0u};
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      lo[m >> 2] |= static_cast<uint32_t>(h[m] & 0xFFu) << (8 * (m & 3));
      hi[m >> 2] |= static_cast<uint32_t>(h[m] >> 8) << (8 * (m & 3));
    }
    lut[s] = make_uint4(lo[0], lo[1], hi[0], hi[1]);
  }
}

// One code word (8 elements) to four f16x2 words with the exact table entry of its scale:
// o[i] = elements 2i, 2i + 1. The element signs flip the high bytes' top bits.
__device__ __forceinline__ void dq8_f16(uint32_t w, uint4 t, uint32_t (&o)[4]) {
  const uint32_t x = w & 0x77777777u;
  const uint32_t l03 = prmt(t.x, t.y, x), h03 = prmt(t.z, t.w, x) ^ (w & 0x80808080u);
  const uint32_t l47 = prmt(t.x, t.y, x >> 16), h47 = prmt(t.z, t.w, x >> 16) ^ ((w << 4) & 0x80808080u);
  o[0] = prmt(l03, h03, 0x5140u);
  o[1] = prmt(l03, h03, 0x7362u);
  o[2] = prmt(l47, h47, 0x5140u);
  o[3] = prmt(l47, h47, 0x7362u);
}

// Dequantise one code word (8 elements, this library's layout) with the table entry of
// its scale: lo = E4M3 bytes of elements 0..3, hi = elements 4..7, in element order.
__device__ __forceinline__ void dq8(uint32_t w, uint2 e, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w & 0x77777777u;
  lo = prmt(e.x, e.y, x) ^ (w & 0x80808080u);
  hi = prmt(e.x, e.y, x >> 16) ^ ((w << 4) & 0x80808080u);
}

// ------------------------------------------------------------------ tcgen05 ------------
// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle layout: rows
// of 128 bytes, 8-row groups 1024 B apart (atoms 1024-B aligned), 16-byte chunk c of row r
// stored at chunk c ^ (r & 7). Advancing the start address by 32 B selects the next K=32
// slice of 8-bit elements inside the atom.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset: 8-row groups
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}

// Byte offset of 16-byte chunk `chunk` of row `r` in a K-major 128-byte-swizzled operand.
__device__ __forceinline__ uint32_t sw128_chunk_off(int r, int chunk) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4));
}

// Shared-memory descriptor of an MN-major operand of 16-bit elements in the 128-byte swizzle
// layout: atoms of 8 K-rows x 64 MN-elements (128 B per row, 16-byte chunk c of row r stored at
// chunk c ^ (r & 7)); atoms `lbo` bytes apart along MN and `sbo` bytes apart along K.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: F16 x F16 -> F32, A K-major, B MN-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32_bmn(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (1u << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: E4M3 x E4M3 -> F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// TMEM allocation by one whole warp; the base address lands in *dst (shared memory).
// Programmatic dependent launch: wait until the previous kernel on the stream has completed
// and its writes are visible (returns at once when the kernel was launched the ordinary way).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, issued by one thread.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T: A (M = 128 rows, K = 32 E4M3 per MMA) held in TMEM,
// row m in lane m, four consecutive elements per 32-bit column.
__device__ __forceinline__ void tc_mma_f8_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]: kind::f16 (f16 operands, fp32 accumulator), issued
// by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16: F16 x F16 -> F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma kind::f16: F16 x F16 -> F32, A MN-major, B K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32_amn(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (1u << 15) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: E4M3 x E4M3 -> F32, A MN-major, B K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32_amn(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (1u << 15) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory descriptor of an MN-major operand of 8-bit elements whose MN extent is one
// 128-byte swizzle atom (128 elements): K-rows of 128 B, 16-byte chunk c of K-row r stored at
// chunk c ^ (r & 7), 8-row groups 1024 B apart along K.
__device__ __forceinline__ uint64_t sw128_mnmajor8_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (one atom along MN: unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: 8-row groups along K
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// 32 lanes x 32 consecutive 32-bit columns into registers: thread i gets lane (base lane + i).
// Completes at tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 16 lanes x 16 columns (shape 16x256b, two repeats): thread t gets, for o = 0..1 and e = 0..3,
// r[4o + e] = lane (base + t/4 + 8*(e/2)), column (8o + 2*(t%4) + e%2). Completes at tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16x256_x2(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

// 32 lanes x 4 consecutive 32-bit columns into / from registers: thread i, lane (base lane + i).
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns into registers: thread i gets lane (base lane + i).
// Completes at tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers: thread i writes lane (base lane + i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 8 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]: kind::f16 with f16 operands, fp32 accumulator; A (M = 128
// rows, K = 16 per MMA) in TMEM, two elements per 32-bit column, the even one in the low half.
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 lanes x 32 columns (shape 16x256b, four repeats): thread t gets, for o = 0..3 and e = 0..3,
// r[4o + e] = lane (base + t/4 + 8*(e/2)), column (8o + 2*(t%4) + e%2). Completes at
// tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// max(a, b, c); a NaN operand is ignored like fmaxf does.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Barrier over `nthreads` threads that also returns whether any of them passed pred = true:
// every participant gets the same answer, so branching on it keeps the group together.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ misc ---------------
__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace msa
