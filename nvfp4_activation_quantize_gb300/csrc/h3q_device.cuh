// h3q_device.cuh -- device building blocks of the NVFP4 producers (sm_103a).
//
// One lane owns one 16-element block: it loads the block's 32 bytes of bf16 with
// a single 256-bit load, computes the block's E4M3 scale and its eight bytes of
// packed E2M1 codes in registers, and stores the codes as one 8-byte write.
// Four neighbouring lanes own the four scale columns of one 128x4 swizzle atom
// row, so their scale bytes leave as one 4-byte word.
//
// Arithmetic is binary32 with one rounding per operation: explicit _rn
// intrinsics (never contracted into FMAs), paired f32x2 operations where two
// independent elements take the same step, and correctly rounded division,
// reciprocal and square root.  The library is built with -fmad=false and
// without fast-math, so no expression is fused behind these calls' back.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace h3q {

constexpr int kBlock = 16;          // elements per NVFP4 block
constexpr int kLanes = 32;

// ---------------------------------------------------------------------------
// Memory
// ---------------------------------------------------------------------------

// 32 bytes = 16 bf16 = one NVFP4 block.
struct Block16 {
  uint32_t w[8];
};

// Streaming read of data touched once (activations): bypasses L1 allocation.
__device__ __forceinline__ void load_stream(const void* p, Block16& b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(b.w[0]), "=r"(b.w[1]), "=r"(b.w[2]), "=r"(b.w[3]), "=r"(b.w[4]),
                 "=r"(b.w[5]), "=r"(b.w[6]), "=r"(b.w[7])
               : "l"(p));
}

// Read of data reused by many rows (gamma, modulation table): cached in L1.
__device__ __forceinline__ void load_reused(const void* p, Block16& b) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(b.w[0]), "=r"(b.w[1]), "=r"(b.w[2]), "=r"(b.w[3]), "=r"(b.w[4]),
                 "=r"(b.w[5]), "=r"(b.w[6]), "=r"(b.w[7])
               : "l"(p));
}

// 16-byte global accesses: streamed data read once (no L1 allocation), small
// read-only tables re-read across rows (L1-allocating), and a 16-byte store.
__device__ __forceinline__ uint4 load16_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 load16_reused(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void store16(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void store_codes(uint8_t* p, uint32_t lo, uint32_t hi) {
  asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(lo), "r"(hi) : "memory");
}

__device__ __forceinline__ void store_byte(uint8_t* p, uint32_t v) {
  asm volatile("st.global.b8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void store_word(uint8_t* p, uint32_t v) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// Paired binary32 arithmetic, each lane rounded to nearest even on its own.
// A paired multiply followed by a paired add of its result is contracted into a
// fused multiply-add by the code generator even with an explicit .rn and
// -fmad=false (a one-ulp difference from the separately rounded sequence, seen
// on rare elements of full-size outputs).  The kernels therefore never feed the
// result of mul2 into add2: such adds are done with scalar add.rn.f32 (or the
// mixed bf16 form below), which are not contracted.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// Paired fused multiply-add a * b + c with one rounding per lane.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// fl(b + c) for each half b of a bf16 pair and fp32 c (scalar add.rn, bf16
// operand taken as is): (lo + c.x, hi + c.y).
__device__ __forceinline__ float2 add_bf16x2_f32(uint32_t b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %4;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(b), "f"(c.x), "f"(c.y));
  return r;
}

// bf16(a + b) for each half of two bf16 pairs: add.rn.bf16x2 rounds the exact
// sum once.  That equals bf16(fl(a + b)), the sum formed in binary32 and then
// rounded to bf16: rounding first to 24 bits and then to 8 cannot differ from
// rounding once to 8 for the sum of two 8-bit operands, since 24 >= 2 * 8 + 2
// (S. A. Figueroa, "When is double rounding innocuous?", ACM SIGNUM Newsletter
// 30(3), 1995).  Checked for every pair of bf16 values by
// tests/device/identities.cu.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// fl(1 / d) for two d in [1, 2^126): a hardware reciprocal estimate refined by
// one Newton-Raphson step and Markstein's final correction (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor",
// IBM J. Res. Dev. 34(1), 1990): e = 1 - d*y, y' = y + y*e, twice, with fused
// multiply-adds; the last step rounds to the correctly rounded reciprocal.
// Equal to __frcp_rn for every binary32 d in [1, 2^126) (checked exhaustively
// on the GPU by tests/test_gpu_device_identities.py).
__device__ __forceinline__ float2 rcp_rn_ge1(float2 d) {
  float2 y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y.x) : "f"(d.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y.y) : "f"(d.y));
  const float2 nd = mul2(d, make_float2(-1.0f, -1.0f));
  float2 e = fma2(nd, y, make_float2(1.0f, 1.0f));
  y = fma2(y, e, y);
  e = fma2(nd, y, make_float2(1.0f, 1.0f));
  return fma2(y, e, y);
}

// bf16 pair (low half = element 2i, high half = element 2i+1) -> two fp32.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// bf16 pair -> two fp32 by a mixed-precision FMA per half (x * 1 + -0 = x,
// exact for every bf16 x, zeros keeping their sign): the same values as
// bf16x2_to_float2, computed on the FMA pipe instead of the integer pipe, which
// is the busier one in the SwiGLU and quantize kernels.
__device__ __forceinline__ float2 bf16x2_to_float2_fma(uint32_t w) {
  float2 r;
  asm("{\n\t.reg .b16 l, h, one;\n\tmov.b32 {l, h}, %2;\n\tmov.b16 one, 0x3F80;\n\t"
      "fma.rn.f32.bf16 %0, l, one, 0f80000000;\n\tfma.rn.f32.bf16 %1, h, one, 0f80000000;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(w));
  return r;
}

// Two fp32 -> bf16 pair, round to nearest even.
__device__ __forceinline__ uint32_t float2_to_bf16x2(float2 v) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(v.y), "f"(v.x));
  return r;
}

// E4M3 encode: round to nearest even, saturating at 448 (0x7E).
__device__ __forceinline__ uint32_t e4m3_encode(float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(s));
  return r & 0xffu;
}

// E4M3 decode of a non-negative finite code: exponent bias 7, three mantissa
// bits, subnormals m * 2^-9 (exact construction of the binary32 value).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 15u;
  const uint32_t m = code & 7u;
  return e == 0 ? __fmul_rn(static_cast<float>(m), 0x1p-9f)
                : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight fp32 values -> four bytes of E2M1 codes (round to nearest even,
// saturating at 6, sign kept).  Element 2i goes to the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1x8(float2 a, float2 b, float2 c, float2 d) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
  return r;
}

// ---------------------------------------------------------------------------
// Block quantize
// ---------------------------------------------------------------------------

// max(|a|, |b|) of each bf16 half (the sign bit of the result is the xor of the
// operands' signs; callers mask it off).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest magnitude held in the two halves of a bf16x2 word, as fp32 (exact).
__device__ __forceinline__ float halves_amax(uint32_t m) {
  m = absmax_bf16x2(m, __byte_perm(m, 0, 0x1032));
  return __uint_as_float((m << 16) & 0x7fff0000u);
}

// Largest |y| of a block of 16 bf16 values, exact.
__device__ __forceinline__ float block_amax(const Block16& y) {
  const uint32_t a = absmax_bf16x2(absmax_bf16x2(y.w[0], y.w[1]), absmax_bf16x2(y.w[2], y.w[3]));
  const uint32_t b = absmax_bf16x2(absmax_bf16x2(y.w[4], y.w[5]), absmax_bf16x2(y.w[6], y.w[7]));
  return halves_amax(absmax_bf16x2(a, b));
}

// fl(a / 6) for a bf16 value a >= 0 without a division: q0 = fl(a * fl(1/6)) is
// corrected once by its exact remainder.  Equal to the correctly rounded
// quotient for every finite such a (checked over all of them in exact
// arithmetic, and against the hardware division on the GPU); +inf (a bf16 overflow of y) is passed through as inf / 6 = inf.
__device__ __forceinline__ float amax_over_six(float a) {
  constexpr float kR6 = 0x1.555556p-3f;  // fl(1/6)
  const float q0 = __fmul_rn(a, kR6);
  const float rem = __fmaf_rn(-q0, 6.0f, a);
  const float t = __fmaf_rn(rem, kR6, q0);
  return a == __int_as_float(0x7f800000) ? a : t;
}

// Inverse block scale for each E4M3 code under the global scale gsf:
// inv[sf] = dec != 0 ? fl(1 / dec) : 0 with dec = fl(E4M3value(sf) / gsf).
// 128 entries in shared memory, filled once per CTA by threads 0..127 (code
// 0x7F never occurs: the encode saturates at 0x7E).  Call before a barrier.
__device__ __forceinline__ void fill_inverse_scales(float* inv, float gsf) {
  const int t = threadIdx.x;
  if (t < 128) {
    const float dec = t < 127 ? __fdiv_rn(e4m3_value(static_cast<uint32_t>(t)), gsf) : 0.0f;
    inv[t] = dec != 0.0f ? __frcp_rn(dec) : 0.0f;
  }
}

// E4M3 block scale of a block whose largest magnitude is amax:
// sf = E4M3(fl(gsf * fl(amax / 6))).
__device__ __forceinline__ uint32_t block_scale(float amax, float gsf) {
  return e4m3_encode(__fmul_rn(gsf, amax_over_six(amax)));
}

// Codes of eight bf16 values (four words) under the inverse scale inv.  FMA:
// unpack the bf16 values on the FMA pipe (kernels whose integer pipe is the
// busier one); the codes are the same either way.
template <bool FMA = false>
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
  return FMA ? bf16x2_to_float2_fma(w) : bf16x2_to_float2(w);
}
template <bool FMA = false>
__device__ __forceinline__ uint32_t codes8(const uint32_t* w, float inv) {
  const float2 inv2 = make_float2(inv, inv);
  return e2m1x8(mul2(unpack_bf16x2<FMA>(w[0]), inv2), mul2(unpack_bf16x2<FMA>(w[1]), inv2),
                mul2(unpack_bf16x2<FMA>(w[2]), inv2), mul2(unpack_bf16x2<FMA>(w[3]), inv2));
}

struct Quantized {
  uint32_t sf;        // E4M3 scale byte
  uint32_t codes_lo;  // codes of elements 0..7
  uint32_t codes_hi;  // codes of elements 8..15
};

// NVFP4 of one block of bf16 values y under the global scale gsf:
//   sf = E4M3(fl(gsf * fl(amax / 6))), inv = inv_table[sf], code_i = E2M1(fl(y_i * inv)).
template <bool FMA = false>
__device__ __forceinline__ Quantized quantize_block(const Block16& y, float gsf,
                                                    const float* inv_table) {
  Quantized q;
  q.sf = block_scale(block_amax(y), gsf);
  const float inv = inv_table[q.sf];
  q.codes_lo = codes8<FMA>(y.w, inv);
  q.codes_hi = codes8<FMA>(y.w + 4, inv);
  return q;
}

// ---------------------------------------------------------------------------
// Abs-max accumulation (dynamic and calibrated scales)
// ---------------------------------------------------------------------------

// Fold each thread's running maximum m >= 0 into *amax: a warp maximum, a CTA
// maximum through shared memory, one atomicMax per CTA on the binary32 bits
// (for values >= 0 -- +inf included -- the bit patterns order as the values
// do, so an integer maximum is the float maximum).  Every thread of the CTA
// calls this once, after its last use of the shared scratch it is given
// (32 floats).
__device__ __forceinline__ void commit_amax(float m, float* amax, float* scratch32) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) scratch32[warp] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int nwarps = (blockDim.x + 31) >> 5;
    float v = static_cast<int>(threadIdx.x) < nwarps ? scratch32[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(v));
  }
}

// ---------------------------------------------------------------------------
// 128x4 scale layout
// ---------------------------------------------------------------------------

// Byte offset, inside the scale matrix, of the 4-byte word that holds scale
// columns 4*quad .. 4*quad+3 of row `row`: atoms of 128 rows x 4 columns (512 B)
// laid out row-tile major; inside an atom, row r sits at (r%32)*16 + ((r/32)%4)*4.
__device__ __forceinline__ int64_t scale_word_offset(int64_t row, int64_t quad,
                                                     int64_t quads_per_row) {
  const int64_t atom = (row >> 7) * quads_per_row + quad;
  return atom * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

// Byte offset of row r's part of a scale word: everything of scale_word_offset
// but the scale-column quad (which adds quad * 512).
__device__ __forceinline__ int64_t scale_row_offset(int64_t r, int64_t quads) {
  return (r >> 7) * quads * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}

// Lanes 4a..4a+3 of a warp hold the scale bytes of four consecutive scale
// columns starting at a multiple of 4; lane 4a stores them as one word.
// All 32 lanes must call this (it shuffles); `active` masks the store.
__device__ __forceinline__ void store_scale_quad(uint8_t* scales, int64_t row, int64_t group,
                                                 int64_t quads_per_row, uint32_t sf, bool active) {
  const int lane = threadIdx.x & 31;
  uint32_t word = sf << (8 * (lane & 3));
  word |= __shfl_xor_sync(0xffffffffu, word, 1);
  word |= __shfl_xor_sync(0xffffffffu, word, 2);
  if (active && (lane & 3) == 0)
    store_word(scales + scale_word_offset(row, group >> 2, quads_per_row), word);
}

}  // namespace h3q
