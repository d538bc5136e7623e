// Checks of device arithmetic identities the codec kernels rely on.
// Built and run by tests/test_gpu_device_identities.py on the GPU.
//
//  div_qmax<Q>(a) == __fdiv_rn(a, Q)   for every finite a >= 0, Q in {7, 127}
//                                      (exhaustive: all 2^31 bit patterns)
//  quantize8<Q>(x, make_scale<Q>(m)) == clamp(rint(__fdiv_rn(x, s)), -Q, Q)
//      for seeded random block maxima m (s = fl(m / Q) in the fast range) and
//      x drawn three ways: within 3 ulps of every (k + 1/2) s, |k| <= Q (the
//      rounding boundaries), uniform in [-m, m], and those values truncated to
//      bf16; 2^33 draws of 8 values each per divisor.
//  (float)(1.0 / (double)d) == __frcp_rn(d)   for every float d in [2^-40, 1]
//      (the host's reciprocal of the Adam bias corrections; exhaustive)
//  div2_bc(x, d, RN(1/d)) == __fdiv_rn(x, d)   for seeded d in [2^-40, 1] and x
//      drawn near the rounding boundaries of x/d, log-uniform over [2^-120, 2^100],
//      and zero; 2^32 draws of 2 values each.
//  dequant_acc_i4(w, i4_fma_scale(s), 1, acc) == acc + fl(q * s), each rounded,
//      for all 16 int4 codes q and every float s in [0, 2^-5) (exhaustive), with
//      acc a seeded value of the scale's magnitude (the one-FMA int4 dequantization)
//  dequant_acc_i8 likewise: all 256 int8 codes and every float s in [0, 2^-5)
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#include "zpp_device.cuh"

__device__ unsigned long long g_bad[8];
__device__ unsigned int g_first[8];

__global__ void check_div(uint32_t lo, uint32_t hi) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t b = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < hi; b += stride) {
    const float a = __uint_as_float((uint32_t)b);
    if (zpp::div_qmax<7>(a) != __fdiv_rn(a, 7.0f)) {
      if (atomicAdd(&g_bad[0], 1ull) == 0) g_first[0] = (uint32_t)b;
    }
    if (zpp::div_qmax<127>(a) != __fdiv_rn(a, 127.0f)) {
      if (atomicAdd(&g_bad[1], 1ull) == 0) g_first[1] = (uint32_t)b;
    }
  }
}

// lowbias32 (Chris Wellons' published integer hash)
__device__ __forceinline__ uint32_t mix(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

template <int Q>
__device__ void check_one(uint64_t t, int slot) {
  uint32_t h = mix((uint32_t)t ^ mix((uint32_t)(t >> 32) + 0x9e3779b9u + slot));
  // block maximum: log-uniform exponent over the fast scale range, random mantissa
  const int ex = (int)(h % 216u) - 96;  // 2^-96 .. 2^119
  h = mix(h);
  float m = ldexpf(1.0f + (float)(h >> 9) * (1.0f / 8388608.0f), ex);
  if (h & 1u) m = __uint_as_float(__float_as_uint(m) & 0xFFFF0000u);  // a bf16 maximum
  const zpp::Scale sc = zpp::make_scale<Q>(m);
  if (!sc.fast || sc.s == 0.0f) return;
  float x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h = mix(h + (uint32_t)i);
    const uint32_t kind = h & 3u;
    float v;
    if (kind <= 1) {  // next to a rounding boundary (k + 1/2) s
      const int k = (int)((h >> 2) % (uint32_t)(Q + 1)) - (int)((h >> 12) & 1u) * (Q + 1);
      const int j = (int)((h >> 13) % 7u) - 3;
      const float b = __fmul_rn((float)k + 0.5f, sc.s);
      v = __int_as_float(__float_as_int(b) + j);
    } else {  // uniform in [-m, m]
      const float u = (float)(int)(h >> 8) * (1.0f / 8388608.0f) - 1.0f;
      v = __fmul_rn(u, m);
    }
    if ((h >> 20) & 1u) v = __uint_as_float(__float_as_uint(v) & 0xFFFF0000u);  // bf16
    if (!(fabsf(v) <= m)) v = 0.0f;  // a block never holds more than its maximum
    x[i] = v;
  }
  uint32_t out[8];
  zpp::quantize8<Q>(x, sc, out);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float r = rintf(__fdiv_rn(x[i], sc.s));
    r = fminf(fmaxf(r, -(float)Q), (float)Q);
    const int want = (int)r;
    const int got = (int)out[i] - (int)zpp::kShiftBits;
    const int c = Q == 7 ? 2 : 3;
    if (got != want) {
      if (atomicAdd(&g_bad[c], 1ull) == 0) g_first[c] = __float_as_uint(x[i]);
    }
  }
}

__global__ void check_quant(uint64_t n) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += stride) {
    check_one<7>(t, 0);
    check_one<127>(t, 1);
  }
}

__global__ void check_rcp(uint32_t lo, uint32_t hi) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t b = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b <= hi; b += stride) {
    const float d = __uint_as_float((uint32_t)b);
    if ((float)(1.0 / (double)d) != __frcp_rn(d)) {
      if (atomicAdd(&g_bad[4], 1ull) == 0) g_first[4] = (uint32_t)b;
    }
  }
}

__global__ void check_bcdiv(uint64_t n) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += stride) {
    uint32_t h = mix((uint32_t)t ^ mix((uint32_t)(t >> 32) + 0x51ed270bu));
    const float d = ldexpf(1.0f + (float)(h >> 9) * (1.0f / 8388608.0f), -(int)(h % 41u));
    const float dd = d > 1.0f ? 1.0f : d;
    const float rd = (float)(1.0 / (double)dd);
    float x[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      h = mix(h + 0x9e3779b9u * (uint32_t)(i + 1));
      const uint32_t kind = h & 3u;
      float v;
      if (kind == 0) {  // next to a rounding boundary of x / d: x = RN(q d) +- a few ulps
        const float q = ldexpf(1.0f + (float)(h >> 9) * (1.0f / 8388608.0f),
                               (int)((h >> 2) % 200u) - 100);
        v = __int_as_float(__float_as_int(__fmul_rn(q, dd)) + (int)((h >> 27) % 7u) - 3);
      } else if (kind == 1) {
        v = ldexpf(1.0f + (float)(h >> 9) * (1.0f / 8388608.0f), (int)((h >> 2) % 220u) - 120);
      } else if (kind == 2) {
        v = 0.0f;
      } else {
        v = ldexpf(1.0f + (float)(h >> 9) * (1.0f / 8388608.0f), (int)((h >> 2) % 60u) - 40);
      }
      x[i] = (h >> 31) ? -v : v;
    }
    const float2 q = zpp::div2_bc(make_float2(x[0], x[1]), dd, rd);
    if (q.x != __fdiv_rn(x[0], dd) || q.y != __fdiv_rn(x[1], dd)) {
      if (atomicAdd(&g_bad[5], 1ull) == 0) g_first[5] = __float_as_uint(x[0]);
    }
  }
}

__global__ void check_i4fma(uint32_t lo, uint32_t hi) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t b = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < hi; b += stride) {
    const float s = __uint_as_float((uint32_t)b);
    const zpp::I4Fma k = zpp::i4_fma_scale(s);
    const uint32_t h = mix((uint32_t)b);
    // an accumulator of the scale's size, either sign
    const float a0 = __fmul_rn(s, (float)((int)(h >> 8) - (1 << 23)) * (1.0f / 1048576.0f));
    const float2 one2 = make_float2(1.0f, 1.0f);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      // codes q = -8..-1 (nibbles 8..15) then 0..7, element e in nibble e
      const uint32_t w = half == 0 ? 0xFEDCBA98u : 0x76543210u;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = a0;
      zpp::dequant_acc_i4(w, k, one2, acc);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int q = half == 0 ? e - 8 : e;
        if (acc[e] != __fadd_rn(a0, __fmul_rn((float)q, s))) {
          if (atomicAdd(&g_bad[6], 1ull) == 0) g_first[6] = (uint32_t)b;
        }
      }
    }
  }
}

__global__ void check_i8fma(uint32_t lo, uint32_t hi) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t b = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < hi; b += stride) {
    const float s = __uint_as_float((uint32_t)b);
    const zpp::I8Fma k = zpp::i8_fma_scale(s);
    const uint32_t h = mix((uint32_t)b ^ 0x5bd1e995u);
    const float a0 = __fmul_rn(s, (float)((int)(h >> 8) - (1 << 23)) * (1.0f / 1048576.0f));
    const float2 one2 = make_float2(1.0f, 1.0f);
    for (int g = 0; g < 32; ++g) {  // codes 8g .. 8g+7 as bytes, q = (int8_t)byte
      uint32_t lo8 = 0, hi8 = 0;
      for (int e = 0; e < 4; ++e) {
        lo8 |= (uint32_t)(8 * g + e) << (8 * e);
        hi8 |= (uint32_t)(8 * g + 4 + e) << (8 * e);
      }
      float acc[8];
      for (int e = 0; e < 8; ++e) acc[e] = a0;
      zpp::dequant_acc_i8(make_uint2(lo8, hi8), k, one2, acc);
      for (int e = 0; e < 8; ++e) {
        const int q = (int)(int8_t)(uint8_t)(8 * g + e);
        if (acc[e] != __fadd_rn(a0, __fmul_rn((float)q, s))) {
          if (atomicAdd(&g_bad[7], 1ull) == 0) g_first[7] = (uint32_t)b;
        }
      }
    }
  }
}

int main() {
  unsigned long long zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (cudaMemcpyToSymbol(g_bad, zero, sizeof zero) != cudaSuccess) return 2;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  check_div<<<sms * 8, 256>>>(0u, 0x7F800000u);  // +0 .. largest finite
  check_quant<<<sms * 8, 256>>>(1ull << 33);
  check_rcp<<<sms * 8, 256>>>(0x2B800000u, 0x3F800000u);  // 2^-40 .. 1
  check_bcdiv<<<sms * 8, 256>>>(1ull << 32);
  check_i4fma<<<sms * 8, 256>>>(0u, 0x3D000000u);  // +0 .. just below 2^-5
  check_i8fma<<<sms * 8, 256>>>(0u, 0x3D000000u);
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  unsigned long long bad[8];
  unsigned int first[8];
  cudaMemcpyFromSymbol(bad, g_bad, sizeof bad);
  cudaMemcpyFromSymbol(first, g_first, sizeof first);
  printf("div_qmax7 %llu %08x\n", bad[0], bad[0] ? first[0] : 0u);
  printf("div_qmax127 %llu %08x\n", bad[1], bad[1] ? first[1] : 0u);
  printf("quantize_q7 %llu %08x\n", bad[2], bad[2] ? first[2] : 0u);
  printf("quantize_q127 %llu %08x\n", bad[3], bad[3] ? first[3] : 0u);
  printf("bias_rcp %llu %08x\n", bad[4], bad[4] ? first[4] : 0u);
  printf("bias_div %llu %08x\n", bad[5], bad[5] ? first[5] : 0u);
  printf("i4_fma %llu %08x\n", bad[6], bad[6] ? first[6] : 0u);
  printf("i8_fma %llu %08x\n", bad[7], bad[7] ? first[7] : 0u);
  return 0;
}
