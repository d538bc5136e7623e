// zpp_launch.h -- host-side launchers of the ZeRO++ codec kernels.  Called by
// the C ABI (zpp_abi.cu) after it has validated every argument; each launcher
// only shapes the grid and enqueues on `stream`.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace zpp {

constexpr int kThreads = 256;  // threads per CTA of every kernel

struct AdamConstsHost {
  float lr, beta1, beta2, eps, omb1, omb2, bc1, bc2;
  float rbc1, rbc2;  // RN(1 / bc) when bc is in [2^-40, 1], else 0
};

// Row-blocked quantization of bf16 rows.
//  qwZ   : rows = nranks, row r = x[r*shard .. +shard), codes/scales per rank.
//  qgZ   : rows = N_d * N_d (rank, slice); slice j of rank r goes to message
//          position p = (j % G) * N + j / G.
cudaError_t launch_qwz_quant(const uint16_t* x, int64_t nranks, int64_t shard, int32_t block,
                             int32_t bits, void* codes, float* scales, cudaStream_t st);
// hpZ backward gather: G sources of N rows (shards) each; bits 16 copies bf16.
constexpr int kMaxHpzSources = 64;
cudaError_t launch_hpz_gather(int32_t G, int32_t N, int64_t shard, int32_t block, int32_t bits,
                              const void* const* sec_codes, const float* const* sec_scales,
                              uint16_t* y, cudaStream_t st);
// acc: null, or the fp32 accumulator of earlier micro-batches (quantizes acc + x).
cudaError_t launch_qgz_reorder_quant(const uint16_t* x, const float* acc, int32_t N, int32_t G,
                                     int64_t bucket, int32_t block, int32_t bits, void* codes,
                                     float* scales, cudaStream_t st);
// acc = (first ? 0 : acc) + (float)g, elementwise in fp32.
cudaError_t launch_grad_accumulate(const uint16_t* g, float* acc, int64_t n, int first,
                                   cudaStream_t st);
cudaError_t launch_qwz_dequant(const void* codes, const float* scales, int64_t nranks,
                               int64_t shard, int32_t block, int32_t bits, uint16_t* y,
                               cudaStream_t st);

// One hop of the hierarchical reduce (see zpp_qgz_hop_reduce).
struct HopLaunch {
  int32_t hop;            // 1 or 2
  const void* codes_in;
  const float* scales_in;
  int32_t N, G;
  int64_t bucket;
  int32_t block, bits;
  void* codes_out;        // non-final hop
  float* scales_out;
  float* grad_out;        // final hop, optional
  float inv_nd;
  bool adam;              // final hop: fused Adam
  AdamConstsHost ac;
  float* master;
  float* m;
  float* v;
  uint16_t* param;
  void* qwz_codes;        // fused int8 qwZ of the new parameters (final hop + Adam), optional
  float* qwz_scales;
};
cudaError_t launch_hop_reduce(const HopLaunch& h, cudaStream_t st);

// One step of the quantized ring reduce-scatter for all N_d ranks.
cudaError_t launch_ring_rs_step(int32_t step, int32_t nd, int64_t bucket, int32_t block,
                                int32_t bits, const uint16_t* x, const void* codes_in,
                                const float* scales_in, void* codes_out, float* scales_out,
                                float* grad_out, cudaStream_t st);

cudaError_t launch_adam(const float* grad, int64_t n, const AdamConstsHost& ac, float* master,
                        float* m, float* v, uint16_t* param, cudaStream_t st);

// Grid size for a kernel: min(work CTAs, waves * SMs * resident CTAs per SM).
// waves = 1: a persistent grid, every CTA resident at once, each warp group
// walking a fixed contiguous range of units.  waves > 1: up to that many
// rounds of resident CTAs, each CTA taking a smaller range; the hardware
// hands the next CTA to whichever SM frees a slot first, so SMs that stream
// faster take more of the work and the grid ends together instead of waiting
// on the slowest fixed range.
int grid_for(const void* kernel, int64_t work_ctas, size_t smem = 0, int waves = 1);

// Rounds of resident CTAs for the streaming kernels (quantize, dequantize,
// standalone Adam, accumulation), measured on GB300 over 1, 8, 16, 24, 32 and
// 64 rounds: with 8, in the 7B step the qwZ quantizer went from 0.82 to 0.95
// of the copy peak, the dequantizer 0.91 -> 0.99, the reorder quantizer
// 0.94 -> 1.00 and Adam 0.97 -> 0.99; from 24 rounds on the quantizers lose
// again (a warp group then gets one or two units, and each CTA's start-up --
// its first copies in flight -- is no longer amortised).  The register-chunk
// hop kernels (two CTAs an SM, heavy per-CTA set-up) stay persistent: no round
// count changed them.  The staged int4 hop 1 and the ring step pick their own
// round counts (four each).
constexpr int kStreamWaves = 8;

// Raises the kernel's dynamic shared-memory limit to `smem` bytes on the
// current device, once per (kernel, device); a failure is returned and not
// remembered, so a later call tries again.
cudaError_t smem_opt_in(const void* kernel, size_t smem);

}  // namespace zpp
