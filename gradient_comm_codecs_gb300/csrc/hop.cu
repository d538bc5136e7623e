// hop.cu -- the two hops of the qgZ hierarchical all-to-all with reduction.
//
// ("Quantized LLM Training at Scale with ZeRO++", "The Three Pillars of
// ZeRO++", 3 QGZ: an intra-node all-to-all and reduction, then an inter-node
// all-to-all; "ZeRO Stage 2: Gradient Partitioning": the reduce-scatter
// averages, GPU i ends with the averaged gradient of shard i, converted to
// fp32 for the optimizer step.)
//
// The simulated all-to-all is the addressing: destination rank d reads its
// chunk straight out of every peer's message in HBM.  One pass per hop fuses
// dequantize -> fp32 sum in rank order -> requantize (hop 1 of a two-hop
// topology) or -> x (1/N_d) -> fp32 gradient and/or the Adam step (final hop).
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {
namespace {

struct HopArgs {
  const uint8_t* codes_in;
  const float* scales_in;
  int64_t in_rank_elems;   // elements of one source message
  int32_t S;               // number of sources summed
  int32_t hop, N, G;
  int64_t R;               // output elements per destination rank
  int64_t units_per_row, total_units;
  int32_t block;
  uint8_t* codes_out;      // requant
  float* scales_out;
  float* grad_out;         // final
  float inv_nd;
  int32_t adam;
  AdamConsts ac;
  float* master;
  float* m;
  float* v;
  uint16_t* param;
};

constexpr int kSrcChunk = 4;  // sources whose loads are in flight together

// MODE 0: hop 1 of a two-hop topology (requantize); MODE 1: final hop.
template <int BITS, int MODE>
__global__ void __launch_bounds__(kThreads, 2) hop_kernel(const HopArgs a) {
  __shared__ float red[2][kWarps];
  using CW = typename CodeVec<BITS>::T;
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.block;
  const int wpb = (MODE == 0 && B > kWarpElems) ? B / kWarpElems : 1;
  const int gpc = kWarps / wpb;
  const int gid = warp / wpb, wsub = warp - gid * wpb;
  const int64_t U = (int64_t)wpb * kWarpElems;
  int parity = 0;

  for (int64_t u = (int64_t)blockIdx.x * gpc + gid; u < a.total_units;
       u += (int64_t)gridDim.x * gpc, parity ^= 1) {
    const int64_t d = u / a.units_per_row;
    const int64_t t = u - d * a.units_per_row;
    const int32_t dn = (int32_t)(d / a.G), dl = (int32_t)(d - (int64_t)dn * a.G);
    // hop 1: sources n*G + g, chunk l;  hop 2: sources n'*G + l, slot n
    const int64_t src0 = a.hop == 1 ? (int64_t)dn * a.G : dl;
    const int64_t sstride = a.hop == 1 ? 1 : a.G;
    const int64_t in_off = (a.hop == 1 ? (int64_t)dl : (int64_t)dn) * a.R;
    const int64_t e_warp = t * U + (int64_t)wsub * kWarpElems;
    const int64_t valid = a.R - e_warp;  // a multiple of 64 when positive

    bool on[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) on[k] = (int64_t)(k * 32 + lane) * 8 < valid;

    float acc[kRows][8];
#pragma unroll
    for (int k = 0; k < kRows; ++k)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[k][i] = 0.0f;

    for (int s0 = 0; s0 < a.S; s0 += kSrcChunk) {
      CW cw[kSrcChunk][kRows];
      float sc[kSrcChunk][kRows];
#pragma unroll
      for (int j = 0; j < kSrcChunk; ++j) {
        const int s = s0 + j;
        const int64_t pb = (src0 + (int64_t)s * sstride) * a.in_rank_elems + in_off + e_warp;
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
          const int64_t pos = pb + (k * 32 + lane) * 8;
          if (s < a.S && on[k]) {
            cw[j][k] = __ldcs(reinterpret_cast<const CW*>(a.codes_in + (pos * BITS) / 8));
            sc[j][k] = __ldg(a.scales_in + pos / B);
          } else {
            cw[j][k] = CW{};
            sc[j][k] = 0.0f;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kSrcChunk; ++j) {
        if (s0 + j >= a.S) break;
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
          float q[8];
          decode8<BITS>(cw[j][k], q);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[k][i] = __fadd_rn(acc[k][i], __fmul_rn(q[i], sc[j][k]));
        }
      }
    }

    const int64_t obase = d * a.R + e_warp;  // output element of this warp's first vector
    if constexpr (MODE == 0) {
      float am[kRows];
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        float m = fabsf(acc[k][0]);
#pragma unroll
        for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(acc[k][i]));
        am[k] = m;
      }
      warp_block_absmax(am, B);
      if (wpb > 1) {
        const float m = group_absmax(am[0], red, parity, warp, gid, wpb, lane);
#pragma unroll
        for (int k = 0; k < kRows; ++k) am[k] = m;
      }
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        if (!on[k]) continue;
        const int e = (k * 32 + lane) * 8;
        const Scale scl = make_scale(am[k], (float)qmax);
        uint32_t c[8];
        quantize8(acc[k], scl, qmax, c);
        *reinterpret_cast<CW*>(a.codes_out + ((obase + e) * BITS) / 8) = pack8<BITS>(c);
        if (((e_warp + e) & (B - 1)) == 0) a.scales_out[(obase + e) / B] = scl.s;
      }
    } else {
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        if (!on[k]) continue;
        const int64_t idx = obase + (k * 32 + lane) * 8;
        float g[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = __fmul_rn(acc[k][i], a.inv_nd);
        if (a.grad_out) {
          float4* go = reinterpret_cast<float4*>(a.grad_out + idx);
          __stcs(go, make_float4(g[0], g[1], g[2], g[3]));
          __stcs(go + 1, make_float4(g[4], g[5], g[6], g[7]));
        }
        if (a.adam) adam_update8(g, idx, a.master, a.m, a.v, a.param, a.ac);
      }
    }
  }
}

template <int BITS, int MODE>
cudaError_t run_hop(const HopArgs& a, cudaStream_t st) {
  const void* k = reinterpret_cast<const void*>(&hop_kernel<BITS, MODE>);
  const int wpb = (MODE == 0 && a.block > kWarpElems) ? a.block / kWarpElems : 1;
  const int gpc = kWarps / wpb;
  hop_kernel<BITS, MODE><<<grid_for(k, (a.total_units + gpc - 1) / gpc), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hop_reduce(const HopLaunch& h, cudaStream_t st) {
  HopArgs a{};
  const int32_t nd = h.N * h.G;
  const int64_t L = h.bucket / nd;
  const bool final_hop = (h.hop == 2) || (h.N == 1);
  a.codes_in = static_cast<const uint8_t*>(h.codes_in);
  a.scales_in = h.scales_in;
  a.hop = h.hop;
  a.N = h.N;
  a.G = h.G;
  a.S = h.hop == 1 ? h.G : h.N;
  a.in_rank_elems = h.hop == 1 ? h.bucket : (int64_t)h.N * L;
  a.R = (h.hop == 1 && h.N > 1) ? (int64_t)h.N * L : L;
  const int64_t U = (!final_hop && h.block > kWarpElems) ? h.block : kWarpElems;
  a.units_per_row = (a.R + U - 1) / U;
  a.total_units = (int64_t)nd * a.units_per_row;
  a.block = h.block;
  a.codes_out = static_cast<uint8_t*>(h.codes_out);
  a.scales_out = h.scales_out;
  a.grad_out = h.grad_out;
  a.inv_nd = h.inv_nd;
  a.adam = h.adam ? 1 : 0;
  a.ac = AdamConsts{h.ac.lr, h.ac.beta1, h.ac.beta2, h.ac.eps,
                    h.ac.omb1, h.ac.omb2, h.ac.bc1, h.ac.bc2};
  a.master = h.master;
  a.m = h.m;
  a.v = h.v;
  a.param = h.param;
  if (final_hop) return h.bits == 8 ? run_hop<8, 1>(a, st) : run_hop<4, 1>(a, st);
  return h.bits == 8 ? run_hop<8, 0>(a, st) : run_hop<4, 0>(a, st);
}

}  // namespace zpp
