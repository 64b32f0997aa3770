// Exhaustive checks of the library's division-free device routines against
// CUDA's correctly rounded operations (test program, built by
// tests/test_gpu_device_identities.py):
//   rcp_rn_ge1(d)   == __frcp_rn(d)    for every binary32 d in [1, 2^126)
//   amax_over_six(a) == __fdiv_rn(a, 6) for every bf16 value a >= 0, +inf included
//   add_bf16x2(a, b) == bf16(__fadd_rn(a, b)) for every pair of bf16 values a, b
//                      (two NaN results count as equal)
// and the hardware conversions the kernels use against integer formulations of
// the formats written here:
//   float2_to_bf16x2 (cvt.rn.bf16x2.f32)  every non-NaN binary32
//   e2m1x8 (cvt.rn.satfinite.e2m1x2.f32)  every non-NaN binary32
//   e4m3_encode (cvt.rn.satfinite.e4m3x2.f32)  every binary32 s >= 0, +inf included
// Prints the number of mismatches of each and exits non-zero if any.
#include <cstdint>
#include <cstdio>

#include "../../nvfp4_activation_quantize_gb300/csrc/h3q_device.cuh"

// Thread i checks the pair of values with bit patterns first + 2i, first + 2i + 1.
__global__ void check_rcp(uint32_t first, uint64_t pairs, unsigned long long* bad) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < pairs;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const float a = __uint_as_float(first + (uint32_t)(2 * i));
    const float b = __uint_as_float(first + (uint32_t)(2 * i + 1));
    const float2 r = h3q::rcp_rn_ge1(make_float2(a, b));
    if (__float_as_uint(r.x) != __float_as_uint(__frcp_rn(a))) atomicAdd(bad, 1ull);
    if (__float_as_uint(r.y) != __float_as_uint(__frcp_rn(b))) atomicAdd(bad, 1ull);
  }
}

__global__ void check_six(unsigned long long* bad) {
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i <= 0x7F80u; i += gridDim.x * blockDim.x) {
    const float a = __uint_as_float(i << 16);  // every bf16 >= 0 up to +inf
    if (__float_as_uint(h3q::amax_over_six(a)) != __float_as_uint(__fdiv_rn(a, 6.0f)))
      atomicAdd(bad, 1ull);
  }
}

__device__ __forceinline__ bool bf16_nan(uint32_t h) { return (h & 0x7f80u) == 0x7f80u && (h & 0x7fu) != 0; }

// Thread i checks a = i >> 15 against the bf16 pair b = 2(i & 0x7fff), 2(i & 0x7fff) + 1.
__global__ void check_add(unsigned long long* bad) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < (1ull << 31);
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t a = (uint32_t)(i >> 15);
    const uint32_t b0 = (uint32_t)(i & 0x7fffu) * 2;
    const uint32_t aw = a | (a << 16), bw = b0 | ((b0 + 1) << 16);
    const uint32_t got = h3q::add_bf16x2(aw, bw);
    const float fa = __uint_as_float(a << 16);
    const uint32_t want = h3q::float2_to_bf16x2(make_float2(__fadd_rn(fa, __uint_as_float(b0 << 16)),
                                                            __fadd_rn(fa, __uint_as_float((b0 + 1) << 16))));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t g = (got >> (16 * h)) & 0xffffu, w = (want >> (16 * h)) & 0xffffu;
      if (g != w && !(bf16_nan(g) && bf16_nan(w))) atomicAdd(bad, 1ull);
    }
  }
}

// bf16 bits of v: the top half of its pattern rounded to nearest, ties to even.
__device__ uint32_t bf16_int(uint32_t u) {
  const uint32_t kept = u >> 16, dropped = u & 0xffffu;
  return kept + ((dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) ? 1u : 0u);
}

// E2M1 code of v by the thresholds of its magnitude grid {0, .5, 1, 1.5, 2, 3, 4, 6}.
__device__ uint32_t e2m1_int(float v) {
  const float a = fabsf(v);
  const uint32_t idx = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
                       (a > 5.0f);
  return ((__float_as_uint(v) >> 31) << 3) | idx;
}

// E4M3 code of s >= 0: three mantissa bits rounded to nearest even in s's binade,
// m * 2^-9 below 2^-6, saturating at 448 (0x7E).
__device__ uint32_t e4m3_int(uint32_t u) {
  if (u >= 0x43e00000u) return 0x7eu;                    // s >= 448, +inf
  const int e = (int)(u >> 23) - 127;
  if (e < -6) {                                          // grid 2^-9: m = rne(s * 512), exact product
    const float m = rintf(__uint_as_float(u) * 512.0f);
    return (uint32_t)m;                                  // 8 is the code of 2^-6 as well
  }
  uint32_t mant = u & 0x7fffffu, m = mant >> 20, rem = mant & 0xfffffu;
  uint32_t code = ((uint32_t)(e + 7) << 3) | m;
  if (rem > 0x80000u || (rem == 0x80000u && (m & 1u))) ++code;  // a carry moves to the next binade
  return code > 0x7eu ? 0x7eu : code;
}

__global__ void check_conversions(unsigned long long* bad) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < (1ull << 29);
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t u0 = (uint32_t)(i * 8);
    float v[8];
    bool nan[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[k] = __uint_as_float(u0 + k);
      nan[k] = isnan(v[k]);
    }
    const uint32_t codes = h3q::e2m1x8(make_float2(v[0], v[1]), make_float2(v[2], v[3]),
                                       make_float2(v[4], v[5]), make_float2(v[6], v[7]));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (nan[k]) continue;
      if (((codes >> (4 * k)) & 15u) != e2m1_int(v[k])) atomicAdd(bad, 1ull);
    }
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const uint32_t b = h3q::float2_to_bf16x2(make_float2(v[k], v[k + 1]));
      if (!nan[k] && (b & 0xffffu) != bf16_int(u0 + k)) atomicAdd(bad + 1, 1ull);
      if (!nan[k + 1] && (b >> 16) != bf16_int(u0 + k + 1)) atomicAdd(bad + 1, 1ull);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t u = u0 + k;
      if (u <= 0x7f800000u && h3q::e4m3_encode(v[k]) != e4m3_int(u)) atomicAdd(bad + 2, 1ull);
    }
  }
}

int main() {
  unsigned long long* bad = nullptr;
  if (cudaMalloc(&bad, 6 * sizeof(unsigned long long)) != cudaSuccess) return 2;
  cudaMemset(bad, 0, 6 * sizeof(unsigned long long));
  const uint32_t first = 0x3F800000u, last = 0x7E800000u;  // [1, 2^126)
  check_rcp<<<152 * 8, 256>>>(first, (uint64_t)(last - first) / 2, bad);  // an even count
  check_six<<<32, 256>>>(bad + 1);
  check_add<<<152 * 8, 256>>>(bad + 2);
  check_conversions<<<152 * 8, 256>>>(bad + 3);
  const cudaError_t err = cudaDeviceSynchronize();
  unsigned long long host[6] = {0, 0, 0, 0, 0, 0};
  cudaMemcpy(host, bad, sizeof host, cudaMemcpyDeviceToHost);
  printf("cuda %d rcp_rn_ge1 mismatches %llu of %u; amax_over_six mismatches %llu of %u; "
         "add_bf16x2 mismatches %llu of 4294967296; e2m1 mismatches %llu; bf16 mismatches %llu; "
         "e4m3 mismatches %llu\n",
         (int)err, host[0], last - first, host[1], 0x7F81u, host[2], host[3], host[4], host[5]);
  bool ok = err == cudaSuccess;
  for (int k = 0; k < 6; ++k) ok = ok && host[k] == 0;
  return ok ? 0 : 1;
}
