// quant.cu -- block quantization kernels: qwZ weight shards, qgZ one-shot
// quantization with the tensor-slice reorder folded into the store address,
// and the qwZ receiver-side dequantization.
//
// ("Quantized LLM Training at Scale with ZeRO++", "The Three Pillars of
// ZeRO++": 1 QWZ block quantization of the weights; 3 QGZ one-shot
// quantization on each GPU and tensor slice reordering before any
// communication.)
//
// HBM-bound streaming kernels: every element is read once (16-byte loads with
// the evict-first hint) and its code written once; one fp32 scale per block.
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {
namespace {

struct QuantArgs {
  const uint16_t* x;
  uint8_t* codes;
  float* scales;
  int64_t total_units;    // rows * units_per_row
  int64_t units_per_row;
  int64_t row_len;        // qwZ: shard; qgZ: slice length L
  int64_t row_blocks;     // qwZ: scales per shard
  int64_t bucket;         // qgZ: elements per rank
  int32_t nd, N, G;       // qgZ topology
  int32_t block;
};

// One row = one contiguous run that is quantized in blocks restarting at the
// row start: a qwZ shard, or one slice (rank r, slice j) of a qgZ bucket whose
// codes go to slice position p = (j % G) * N + j / G of rank r's message.
template <int BITS, bool REORDER>
__global__ void __launch_bounds__(kThreads) quant_kernel(const QuantArgs a) {
  __shared__ float red[2][kWarps];
  using CW = typename CodeVec<BITS>::T;
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.block;
  const int wpb = B > kWarpElems ? B / kWarpElems : 1;  // warps per unit
  const int gpc = kWarps / wpb;                         // units per CTA pass
  const int gid = warp / wpb, wsub = warp - gid * wpb;
  const int64_t U = (int64_t)wpb * kWarpElems;
  int parity = 0;

  for (int64_t u = (int64_t)blockIdx.x * gpc + gid; u < a.total_units;
       u += (int64_t)gridDim.x * gpc, parity ^= 1) {
    const int64_t row = u / a.units_per_row;
    const int64_t t = u - row * a.units_per_row;
    int64_t src_base, dst_base, scale_base;
    if constexpr (REORDER) {
      const int32_t r = (int32_t)(row / a.nd);
      const int32_t j = (int32_t)(row - (int64_t)r * a.nd);
      const int32_t p = (j % a.G) * a.N + j / a.G;
      src_base = (int64_t)r * a.bucket + (int64_t)j * a.row_len;
      dst_base = (int64_t)r * a.bucket + (int64_t)p * a.row_len;
      scale_base = dst_base / B;
    } else {
      src_base = row * a.row_len;
      dst_base = src_base;
      scale_base = row * a.row_blocks;
    }
    const int64_t e_warp = t * U + (int64_t)wsub * kWarpElems;  // first element (row-relative)
    const int64_t valid = a.row_len - e_warp;
    const bool aligned = ((src_base | dst_base) & 7) == 0;
    const bool full = aligned && valid >= kWarpElems;
    const uint16_t* xw = a.x + src_base + e_warp;

    float x[kRows][8];
    int nv[kRows];
    if (full) {
      uint4 w[kRows];
#pragma unroll
      for (int k = 0; k < kRows; ++k)
        w[k] = __ldcs(reinterpret_cast<const uint4*>(xw + (k * 32 + lane) * 8));
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        unpack_bf16x8(w[k], x[k]);
        nv[k] = 8;
      }
    } else {
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const int e = (k * 32 + lane) * 8;
        const int64_t rem = valid - e;
        nv[k] = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          x[k][i] = i < nv[k] ? __uint_as_float((uint32_t)xw[e + i] << 16) : 0.0f;
      }
    }

    float am[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      float m = fabsf(x[k][0]);
#pragma unroll
      for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(x[k][i]));
      am[k] = m;
    }
    warp_block_absmax(am, B);
    if (wpb > 1) {
      const float m = group_absmax(am[0], red, parity, warp, gid, wpb, lane);
#pragma unroll
      for (int k = 0; k < kRows; ++k) am[k] = m;
    }

    uint8_t* cw = a.codes + ((dst_base + e_warp) * BITS) / 8;
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      if (nv[k] == 0) continue;
      const int e = (k * 32 + lane) * 8;
      const Scale sc = make_scale(am[k], (float)qmax);
      uint32_t c[8];
      quantize8(x[k], sc, qmax, c);
      const CW w = pack8<BITS>(c);
      uint8_t* dst = cw + (e * BITS) / 8;
      if (nv[k] == 8 && aligned) {
        *reinterpret_cast<CW*>(dst) = w;
      } else {
        const int nbytes = (nv[k] * BITS + 7) / 8;
        const uint8_t* wb = reinterpret_cast<const uint8_t*>(&w);
        for (int i = 0; i < nbytes; ++i) dst[i] = wb[i];
      }
      if (((e_warp + e) & (B - 1)) == 0) a.scales[scale_base + (e_warp + e) / B] = sc.s;
    }
  }
}

struct DequantArgs {
  const uint8_t* codes;
  const float* scales;
  uint16_t* y;
  int64_t total_units, units_per_row;
  int64_t row_len, row_blocks;
  int32_t block;
};

// y = bf16_rn((float)q * s) for every element of every shard.
template <int BITS>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const DequantArgs a) {
  using CW = typename CodeVec<BITS>::T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < a.total_units;
       u += (int64_t)gridDim.x * kWarps) {
    const int64_t row = u / a.units_per_row;
    const int64_t t = u - row * a.units_per_row;
    const int64_t base = row * a.row_len;
    const int64_t e_warp = t * kWarpElems;
    const int64_t valid = a.row_len - e_warp;
    const bool aligned = (base & 7) == 0;
    const bool full = aligned && valid >= kWarpElems;
    const uint8_t* cw = a.codes + ((base + e_warp) * BITS) / 8;
    const float* sw = a.scales + row * a.row_blocks;
    uint16_t* yw = a.y + base + e_warp;
    if (full) {
      CW w[kRows];
      float s[kRows];
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const int e = (k * 32 + lane) * 8;
        w[k] = __ldcs(reinterpret_cast<const CW*>(cw + (e * BITS) / 8));
        s[k] = __ldg(sw + (e_warp + e) / a.block);
      }
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const int e = (k * 32 + lane) * 8;
        float q[8];
        decode8<BITS>(w[k], q);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(q[i], s[k]);
        __stcs(reinterpret_cast<uint4*>(yw + e),
               make_uint4(pack_bf16x2(q[0], q[1]), pack_bf16x2(q[2], q[3]),
                          pack_bf16x2(q[4], q[5]), pack_bf16x2(q[6], q[7])));
      }
    } else {
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const int e = (k * 32 + lane) * 8;
        for (int i = 0; i < 8; ++i) {
          const int64_t el = e_warp + e + i;
          if (el >= a.row_len) break;
          const int64_t pos = base + el;
          int q;
          if (BITS == 8) {
            q = (int8_t)a.codes[pos];
          } else {
            const uint8_t b = a.codes[pos >> 1];
            const int nib = (pos & 1) ? (b >> 4) : (b & 0xF);
            q = nib >= 8 ? nib - 16 : nib;
          }
          yw[e + i] = bf16_bits(__fmul_rn((float)q, sw[el / a.block]));
        }
      }
    }
  }
}

template <int BITS, bool REORDER>
cudaError_t run_quant(const QuantArgs& a, cudaStream_t st) {
  const void* k = reinterpret_cast<const void*>(&quant_kernel<BITS, REORDER>);
  const int wpb = a.block > kWarpElems ? a.block / kWarpElems : 1;
  const int64_t ctas = (a.total_units + (kWarps / wpb) - 1) / (kWarps / wpb);
  quant_kernel<BITS, REORDER><<<grid_for(k, ctas), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t run_dequant(const DequantArgs& a, cudaStream_t st) {
  const void* k = reinterpret_cast<const void*>(&dequant_kernel<BITS>);
  dequant_kernel<BITS><<<grid_for(k, (a.total_units + kWarps - 1) / kWarps), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

int64_t units_per(int64_t len, int32_t block) {
  const int64_t U = block > kWarpElems ? block : kWarpElems;
  return (len + U - 1) / U;
}

}  // namespace

cudaError_t launch_qwz_quant(const uint16_t* x, int64_t nranks, int64_t shard, int32_t block,
                             int32_t bits, void* codes, float* scales, cudaStream_t st) {
  QuantArgs a{};
  a.x = x;
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = scales;
  a.units_per_row = units_per(shard, block);
  a.total_units = nranks * a.units_per_row;
  a.row_len = shard;
  a.row_blocks = (shard + block - 1) / block;
  a.block = block;
  return bits == 8 ? run_quant<8, false>(a, st) : run_quant<4, false>(a, st);
}

cudaError_t launch_qgz_reorder_quant(const uint16_t* x, int32_t N, int32_t G, int64_t bucket,
                                     int32_t block, int32_t bits, void* codes, float* scales,
                                     cudaStream_t st) {
  QuantArgs a{};
  a.x = x;
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = scales;
  a.nd = N * G;
  a.N = N;
  a.G = G;
  a.bucket = bucket;
  a.row_len = bucket / a.nd;
  a.units_per_row = units_per(a.row_len, block);
  a.total_units = (int64_t)a.nd * a.nd * a.units_per_row;
  a.block = block;
  return bits == 8 ? run_quant<8, true>(a, st) : run_quant<4, true>(a, st);
}

cudaError_t launch_qwz_dequant(const void* codes, const float* scales, int64_t nranks,
                               int64_t shard, int32_t block, int32_t bits, uint16_t* y,
                               cudaStream_t st) {
  DequantArgs a{};
  a.codes = static_cast<const uint8_t*>(codes);
  a.scales = scales;
  a.y = y;
  a.units_per_row = (shard + kWarpElems - 1) / kWarpElems;
  a.total_units = nranks * a.units_per_row;
  a.row_len = shard;
  a.row_blocks = (shard + block - 1) / block;
  a.block = block;
  return bits == 8 ? run_dequant<8>(a, st) : run_dequant<4>(a, st);
}

}  // namespace zpp
