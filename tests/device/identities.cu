// Exhaustive checks of the library's division-free device routines against
// CUDA's correctly rounded operations (test program, built by
// tests/test_gpu_device_identities.py):
//   rcp_rn_ge1(d)   == __frcp_rn(d)    for every binary32 d in [1, 2^126)
//   amax_over_six(a) == __fdiv_rn(a, 6) for every bf16 value a >= 0, +inf included
//   add_bf16x2(a, b) == bf16(__fadd_rn(a, b)) for every pair of bf16 values a, b
//                      (two NaN results count as equal)
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

int main() {
  unsigned long long* bad = nullptr;
  if (cudaMalloc(&bad, 3 * sizeof(unsigned long long)) != cudaSuccess) return 2;
  cudaMemset(bad, 0, 3 * sizeof(unsigned long long));
  const uint32_t first = 0x3F800000u, last = 0x7E800000u;  // [1, 2^126)
  check_rcp<<<152 * 8, 256>>>(first, (uint64_t)(last - first) / 2, bad);  // an even count
  check_six<<<32, 256>>>(bad + 1);
  check_add<<<152 * 8, 256>>>(bad + 2);
  const cudaError_t err = cudaDeviceSynchronize();
  unsigned long long host[3] = {0, 0, 0};
  cudaMemcpy(host, bad, sizeof host, cudaMemcpyDeviceToHost);
  printf("cuda %d rcp_rn_ge1 mismatches %llu of %u; amax_over_six mismatches %llu of %u; "
         "add_bf16x2 mismatches %llu of 4294967296\n",
         (int)err, host[0], last - first, host[1], 0x7F81u, host[2]);
  return (err != cudaSuccess || host[0] || host[1] || host[2]) ? 1 : 0;
}
