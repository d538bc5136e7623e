// adam.cu -- standalone sharded mixed-precision Adam step.
//
// ("ZeRO-1/2/3", Stage 1 steps 5-6 and Stage 2: each rank updates the fp32
// optimizer state and master of its own shard with the reduced gradient, then
// writes the 16-bit parameter copy; "ZeRO Stage 2: Gradient Partitioning":
// the gradient shard is fp32 at the optimizer step.)
//
// Pure streaming: 16 bytes read + 14 bytes written per parameter (fp32 g,
// master, m, v in; master, m, v, bf16 param out).
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {
namespace {

constexpr int kAdamRows = 2;                          // 8-element vectors per lane per unit
constexpr int kAdamUnit = 32 * 8 * kAdamRows;         // 512 parameters per warp unit

struct AdamArgs {
  const float* g;
  float* master;
  float* m;
  float* v;
  uint16_t* param;
  int64_t n;
  AdamConsts ac;
};

// WIDE: g, master, m, v all 32-byte aligned; one 256-bit access per lane.
template <bool WIDE>
__global__ void __launch_bounds__(kThreads) adam_kernel(const AdamArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t units = (a.n + kAdamUnit - 1) / kAdamUnit;
  for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units;
       u += (int64_t)gridDim.x * kWarps) {
    const int64_t base = u * kAdamUnit + lane * 8;
    if (base + (kAdamRows - 1) * 256 + 8 <= a.n) {
      float g[kAdamRows][8];
      AdamVec s[kAdamRows];
#pragma unroll
      for (int k = 0; k < kAdamRows; ++k) {
        ld8_cs(a.g + base + k * 256, WIDE, g[k]);
        s[k] = adam_load8(base + k * 256, a.master, a.m, a.v, WIDE);
      }
#pragma unroll
      for (int k = 0; k < kAdamRows; ++k)
        adam_apply8<true>(g[k], s[k], base + k * 256, a.master, a.m, a.v, a.param, a.ac, WIDE);
    } else {
#pragma unroll
      for (int k = 0; k < kAdamRows; ++k) {
        const int64_t idx = base + k * 256;
        for (int64_t i = idx; i < idx + 8 && i < a.n; ++i) {
          float p = a.master[i], m = a.m[i], v = a.v[i];
          adam_update(a.g[i], p, m, v, a.ac);
          a.master[i] = p;
          a.m[i] = m;
          a.v[i] = v;
          if (a.param) a.param[i] = bf16_bits(p);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_adam(const float* grad, int64_t n, const AdamConstsHost& ac, float* master,
                        float* m, float* v, uint16_t* param, cudaStream_t st) {
  AdamArgs a{grad, master, m, v, param, n,
             AdamConsts{ac.lr, ac.beta1, ac.beta2, ac.eps, ac.omb1, ac.omb2, ac.bc1, ac.bc2,
                        ac.rbc1, ac.rbc2, 1.0f}};
  const int64_t units = (n + kAdamUnit - 1) / kAdamUnit;
  const int64_t ctas = (units + kWarps - 1) / kWarps;
  if (aligned32(grad) && aligned32(master) && aligned32(m) && aligned32(v)) {
    const void* k = reinterpret_cast<const void*>(&adam_kernel<true>);
    adam_kernel<true><<<grid_for(k, ctas, 0, kStreamWaves), kThreads, 0, st>>>(a);
  } else {
    const void* k = reinterpret_cast<const void*>(&adam_kernel<false>);
    adam_kernel<false><<<grid_for(k, ctas, 0, kStreamWaves), kThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace zpp
