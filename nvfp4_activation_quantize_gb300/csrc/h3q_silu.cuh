// h3q_silu.cuh -- the SwiGLU arithmetic of the library, shared by the SwiGLU
// producers (swiglu.cu) and the GEMM epilogue (gemm_swiglu.cu).
//
// Per element, in binary32 with one rounding per operation:
//   E = exp_c(-g), sigma = fl(1 / fl(1 + E)), s = fl(g * sigma), y = bf16(fl(s * u))
// exp_c is this library's fixed exponential: Cody-Waite additive reduction
// (W. J. Cody and W. Waite, "Software Manual for the Elementary Functions",
// 1980) by a two-part ln 2 applied with FMAs, and the degree-7 Taylor
// polynomial of e^r in Horner form:
//   z > 89 -> +inf, z < -104 -> +0, otherwise
//   t = fl(z * L2E), k = rint(t), r = fma(-k, C1, z), r = fma(-k, C2, r),
//   p = P7, p = fma(p, r, Pn) for n = 6..2, p = fma(p, r, 1), p = fma(p, r, 1),
//   result = p * 2^k rounded once.
//   L2E = fl(1/ln 2), C1 = fl(ln 2), C2 = fl(ln 2 - C1), Pn = fl(1/n!).
// rint uses the 1.5 * 2^23 addition: for |t| <= 2^22 the sum lands where the
// binary32 spacing is 1, so the addition itself rounds t half-to-even, and
// subtracting the constant again is exact.
//
// s = fl(g * sigma) depends on the bf16 gate alone, so -- as the pages' fused
// SwiGLU producer does with its SiLU table (FastVideo API page,
// swiglu_quantize) -- a CTA can tabulate s for every bf16 gate with
// 2^-25 <= |g| <= 127.5 (8,192 values, 32 KB of shared memory) and look it up
// for blocks whose gates all lie in that window; both give the same bits.
#pragma once

#include "h3q_device.cuh"

namespace h3q {

constexpr float kL2E = 0x1.715476p+0f;    // fl(1 / ln 2)
constexpr float kC1 = 0x1.62e430p-1f;     // fl(ln 2)
constexpr float kC2 = -0x1.05c610p-29f;   // fl(ln 2 - C1)
constexpr float kP2 = 0.5f;               // 1/2!
constexpr float kP3 = 0x1.555556p-3f;     // fl(1/3!)
constexpr float kP4 = 0x1.555556p-5f;     // fl(1/4!)
constexpr float kP5 = 0x1.111112p-7f;     // fl(1/5!)
constexpr float kP6 = 0x1.6c16c2p-10f;    // fl(1/6!)
constexpr float kP7 = 0x1.a01a02p-13f;    // fl(1/7!)
constexpr float kRound = 0x1.8p+23f;      // 1.5 * 2^23
constexpr float kFastLimit = 87.0f;       // |z| <= 87: k in [-126, 127]

// SiLU products s(g) = fl(g * sigma(g)) of the bf16 gates with magnitude bits in
// [kTabLo, kTabLo + 4095] (2^-25 <= |g| <= 127.5), both signs, tabulated per CTA
// in shared memory: entry sign * 4096 + (magnitude bits - kTabLo).  With exactly
// 4096 magnitudes a gate pair is inside the window iff w - (kTabLo, kTabLo) has
// bits 12..14 of both halves clear (a magnitude below kTabLo borrows into them,
// one above kTabLo + 4095 carries into them), so the window test is one AND per
// pair.
constexpr uint32_t kTabLo = 0x3300u;          // bf16 bits of 2^-25
constexpr uint32_t kTabWord = kTabLo | (kTabLo << 16);
constexpr uint32_t kTabOut = 0x70007000u;     // bits 12..14 of both halves
constexpr int kTabHalf = 4096;

__device__ __forceinline__ float2 splat(float v) { return make_float2(v, v); }

// exp_c(-g) for two gates g, with the negation folded away:
//   t  = fl(-g * L2E)        = fl(g * -L2E)
//   r1 = fma(-k, C1, -g)     = -fma(k, C1, g)       (so r' = fma(k, C1, g) = -r1)
//   r2 = fma(-k, C2, r1)     = -fma(k, C2, r')      (so r' = fma(k, C2, r') = -r2)
// and Horner in r = -r' run as Horner in r' with the coefficient of r^n
// multiplied by (-1)^n: every intermediate is the exact negation or copy of
// the one in the r form, because round-to-nearest is odd-symmetric.  The
// results are the bits exp_c defines.
// FAST: every |g| <= 87, so k lies in [-126, 127] and 2^k is normal.
template <bool FAST>
__device__ __forceinline__ float2 exp_neg2(float2 g) {
  float2 gc = g;
  if (!FAST) {  // z = -g clamped to [-104, 89]
    gc.x = fminf(fmaxf(g.x, -89.0f), 104.0f);
    gc.y = fminf(fmaxf(g.y, -89.0f), 104.0f);
  }
  const float2 t = mul2(gc, splat(-kL2E));
  // scalar adds: a paired add of a paired product would be contracted
  const float2 m = make_float2(__fadd_rn(t.x, kRound), __fadd_rn(t.y, kRound));
  const float2 k = add2(m, splat(-kRound));
  float2 r = fma2(k, splat(kC1), gc);
  r = fma2(k, splat(kC2), r);
  float2 p = splat(-kP7);
  p = fma2(p, r, splat(kP6));
  p = fma2(p, r, splat(-kP5));
  p = fma2(p, r, splat(kP4));
  p = fma2(p, r, splat(-kP3));
  p = fma2(p, r, splat(kP2));
  p = fma2(p, r, splat(-1.0f));
  p = fma2(p, r, splat(1.0f));
  if (FAST) {
    // 2^k is a normal binary32; its exponent field is k + 127, and k itself sits
    // in the low bits of m (spacing 1 around 1.5 * 2^23).
    const int kx = __float_as_int(m.x) - __float_as_int(kRound);
    const int ky = __float_as_int(m.y) - __float_as_int(kRound);
    const float2 s = make_float2(__int_as_float((kx + 127) << 23), __int_as_float((ky + 127) << 23));
    return mul2(p, s);
  }
  // k in [-150, 128]: ldexpf scales exactly and rounds once (into the subnormal
  // range or to infinity), which is fl(p * 2^k).
  float2 e = make_float2(ldexpf(p.x, __float2int_rn(k.x)), ldexpf(p.y, __float2int_rn(k.y)));
  if (g.x < -89.0f) e.x = __int_as_float(0x7f800000);  // z > 89
  if (g.y < -89.0f) e.y = __int_as_float(0x7f800000);
  if (g.x > 104.0f) e.x = 0.0f;                        // z < -104
  if (g.y > 104.0f) e.y = 0.0f;
  return e;
}

template <bool FAST>
__device__ __forceinline__ void swiglu_block(const Block16& g, const Block16& u, Block16& y) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 gv = bf16x2_to_float2(g.w[i]);
    const float2 uv = bf16x2_to_float2(u.w[i]);
    const float2 e = exp_neg2<FAST>(gv);
    // e = p * 2^k is exact except below 2^-126, where 1 + e rounds to 1 either
    // way, so even a fused form of this add would give the same d
    const float2 d = add2(splat(1.0f), e);
    // FAST: |g| <= 87, so d = 1 + e lies in [1, 2^126)
    const float2 sig = FAST ? rcp_rn_ge1(d) : make_float2(__frcp_rn(d.x), __frcp_rn(d.y));
    const float2 s = mul2(gv, sig);
    y.w[i] = float2_to_bf16x2(mul2(s, uv));
  }
}

// Byte offsets in the table of the gates in the low and high halves of a bf16 pair
// inside the window, from d = w - kTabWord = sign * 0x8000 + (magnitude - kTabLo)
// in each half (no borrow inside the window).
__device__ __forceinline__ void table_offsets(uint32_t d, uint32_t& lo, uint32_t& hi) {
  lo = ((d << 2) & 0x3ffcu) | ((d >> 1) & 0x4000u);
  hi = ((d >> 14) & 0x3ffcu) | ((d >> 17) & 0x4000u);
}

__device__ __forceinline__ void swiglu_block_table(const uint32_t (&d)[8], const Block16& u, Block16& y,
                                                   const char* table) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo, hi;
    table_offsets(d[i], lo, hi);
    const float2 sv = make_float2(*reinterpret_cast<const float*>(table + lo),
                                  *reinterpret_cast<const float*>(table + hi));
    y.w[i] = float2_to_bf16x2(mul2(sv, bf16x2_to_float2_fma(u.w[i])));
  }
}

// The block's table words d_i = w_i - kTabWord; true when every gate of the
// block lies inside the window.
__device__ __forceinline__ bool table_words(const Block16& g, uint32_t (&d)[8]) {
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    d[i] = g.w[i] - kTabWord;
    out |= d[i] & kTabOut;
  }
  return out == 0;
}

// Fill the table: entries i and i + kTabHalf hold the positive and negative gate
// of magnitude bits kTabLo + i, computed as a pair exactly as the direct path
// computes them: the FAST exponential up to |g| = 87, the general one above.
__device__ __forceinline__ void fill_silu_table(float* table) {
  constexpr uint32_t kFastHi = 0x42aeu;  // bf16 bits of 87 (kFastLimit)
  for (int i = threadIdx.x; i < kTabHalf; i += blockDim.x) {
    const uint32_t mag = kTabLo + static_cast<uint32_t>(i);
    const uint32_t pair = mag | ((mag | 0x8000u) << 16);  // (+g, -g)
    const float2 gv = bf16x2_to_float2(pair);
    float2 sv;
    if (mag <= kFastHi) {
      const float2 d = add2(splat(1.0f), exp_neg2<true>(gv));
      sv = mul2(gv, rcp_rn_ge1(d));
    } else {
      const float2 d = add2(splat(1.0f), exp_neg2<false>(gv));
      sv = mul2(gv, make_float2(__frcp_rn(d.x), __frcp_rn(d.y)));
    }
    table[i] = sv.x;
    table[i + kTabHalf] = sv.y;
  }
}

}  // namespace h3q
