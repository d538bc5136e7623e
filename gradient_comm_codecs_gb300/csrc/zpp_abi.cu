// zpp_abi.cu -- the extern "C" entry points declared in include/zpp.h:
// argument validation, host-side constants, and dispatch to the launchers.
// Nothing here touches the device until every argument has been checked.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "zpp.h"
#include "zpp_launch.h"

namespace zpp {

namespace {

thread_local char g_last_cuda_error[256] = "";

zpp_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ZPP_OK;
  std::strncpy(g_last_cuda_error, cudaGetErrorString(e), sizeof g_last_cuda_error - 1);
  g_last_cuda_error[sizeof g_last_cuda_error - 1] = '\0';
  return ZPP_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_bits(int32_t b) { return b == 4 || b == 8; }
bool valid_block(int32_t b) { return b >= 64 && b <= 4096 && (b & (b - 1)) == 0; }

// Largest element count any one call accepts: keeps every byte offset inside
// int64 with room to spare.
constexpr int64_t kMaxElems = int64_t(1) << 52;
constexpr int32_t kMaxRanks = 1 << 16;

double pow_by_squaring(double b, int64_t t) {
  double r = 1.0;
  while (t > 0) {
    if (t & 1) r *= b;
    b *= b;
    t >>= 1;
  }
  return r;
}

zpp_status adam_consts(const zpp_adam_hparams* hp, AdamConstsHost* ac) {
  if (!hp || hp->step < 1) return ZPP_ERR_INVALID_ARG;
  ac->lr = hp->lr;
  ac->beta1 = hp->beta1;
  ac->beta2 = hp->beta2;
  ac->eps = hp->eps;
  ac->bc1 = (float)(1.0 - pow_by_squaring((double)hp->beta1, hp->step));
  ac->bc2 = (float)(1.0 - pow_by_squaring((double)hp->beta2, hp->step));
  ac->omb1 = (float)(1.0 - (double)hp->beta1);
  ac->omb2 = (float)(1.0 - (double)hp->beta2);
  // RN(1/bc): the double quotient rounded to float is the correctly rounded
  // float reciprocal, double rounding being innocuous for a quotient when the
  // wider format has at least 2p + 2 bits (53 >= 2*24 + 2).
  auto rcp = [](float bc) {
    return (bc >= 0x1p-40f && bc <= 1.0f) ? (float)(1.0 / (double)bc) : 0.0f;
  };
  ac->rbc1 = rcp(ac->bc1);
  ac->rbc2 = rcp(ac->bc2);
  return ZPP_OK;
}

zpp_status check_state(const zpp_adam_state* st) {
  if (!st || !st->master || !st->m || !st->v) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(st->master) || !aligned16(st->m) || !aligned16(st->v) ||
      (st->param_bf16 && !aligned16(st->param_bf16)))
    return ZPP_ERR_MISALIGNED;
  return ZPP_OK;
}

zpp_status check_topology(int32_t nodes, int32_t gpn, int64_t bucket, int32_t block,
                          int32_t bits) {
  if (nodes < 1 || gpn < 1 || (int64_t)nodes * gpn > kMaxRanks) return ZPP_ERR_INVALID_ARG;
  if (!valid_bits(bits) || !valid_block(block)) return ZPP_ERR_INVALID_ARG;
  const int64_t nd = (int64_t)nodes * gpn;
  if (bucket < 0 || bucket > kMaxElems / nd) return ZPP_ERR_INVALID_ARG;
  if (bucket % (nd * block) != 0) return ZPP_ERR_INVALID_ARG;
  return ZPP_OK;
}

}  // namespace

int grid_for(const void* kernel, int64_t work_ctas, size_t smem, int waves) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> cache;  // (kernel, device) -> resident CTAs
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t key = reinterpret_cast<uintptr_t>(kernel) * 131u + (uint64_t)dev;
  int total = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) total = it->second;
  }
  if (total == 0) {
    int sms = 1, per_sm = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    total = (sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = total;
  }
  const int64_t cap = (int64_t)total * (waves > 1 ? waves : 1);
  int64_t g = work_ctas < cap ? work_ctas : cap;
  return g < 1 ? 1 : (int)g;
}

cudaError_t smem_opt_in(const void* kernel, size_t smem) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, size_t> done;  // (kernel, device) -> bytes opted in
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t key = reinterpret_cast<uintptr_t>(kernel) * 131u + (uint64_t)dev;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= smem) return cudaSuccess;
  }
  const cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
  if (r == cudaSuccess) {
    std::lock_guard<std::mutex> lock(mu);
    done[key] = smem;
  }
  return r;
}

}  // namespace zpp

using namespace zpp;

extern "C" {

int64_t zpp_codes_bytes(int64_t n, int32_t bits) {
  if (n < 0 || !valid_bits(bits) || n > kMaxElems) return -1;
  return (n * bits + 7) / 8;
}

int64_t zpp_num_blocks(int64_t n, int32_t block) {
  if (n < 0 || block <= 0 || n > kMaxElems) return -1;
  return (n + block - 1) / block;
}

zpp_status zpp_qgz_slice_perm(int32_t nodes, int32_t gpus_per_node, int32_t* perm_host) {
  if (nodes < 1 || gpus_per_node < 1 || (int64_t)nodes * gpus_per_node > kMaxRanks || !perm_host)
    return ZPP_ERR_INVALID_ARG;
  for (int32_t n = 0; n < nodes; ++n)
    for (int32_t l = 0; l < gpus_per_node; ++l) perm_host[l * nodes + n] = n * gpus_per_node + l;
  return ZPP_OK;
}

const char* zpp_status_string(zpp_status s) {
  switch (s) {
    case ZPP_OK: return "ok";
    case ZPP_ERR_INVALID_ARG: return "invalid argument";
    case ZPP_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case ZPP_ERR_UNSUPPORTED: return "unsupported";
    case ZPP_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* zpp_last_cuda_error(void) { return g_last_cuda_error; }

int32_t zpp_abi_version(void) { return (1 << 16) | 2; }

zpp_status zpp_qwz_quant(const uint16_t* x_bf16, int64_t nranks, int64_t shard_elems,
                         int32_t block, int32_t bits, void* codes, float* scales,
                         void* stream) {
  if (nranks < 0 || shard_elems < 0 || !valid_bits(bits) || !valid_block(block))
    return ZPP_ERR_INVALID_ARG;
  if (bits == 4 && (shard_elems & 1)) return ZPP_ERR_INVALID_ARG;
  if (shard_elems > 0 && nranks > kMaxElems / shard_elems) return ZPP_ERR_INVALID_ARG;
  if (nranks == 0 || shard_elems == 0) return ZPP_OK;
  if (!x_bf16 || !codes || !scales) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(codes) || !aligned16(scales)) return ZPP_ERR_MISALIGNED;
  return cuda_status(launch_qwz_quant(x_bf16, nranks, shard_elems, block, bits, codes, scales,
                                      static_cast<cudaStream_t>(stream)));
}

zpp_status zpp_qwz_dequant(const void* codes, const float* scales, int64_t nranks,
                           int64_t shard_elems, int32_t block, int32_t bits, uint16_t* y_bf16,
                           void* stream) {
  if (nranks < 0 || shard_elems < 0 || !valid_bits(bits) || !valid_block(block))
    return ZPP_ERR_INVALID_ARG;
  if (bits == 4 && (shard_elems & 1)) return ZPP_ERR_INVALID_ARG;
  if (shard_elems > 0 && nranks > kMaxElems / shard_elems) return ZPP_ERR_INVALID_ARG;
  if (nranks == 0 || shard_elems == 0) return ZPP_OK;
  if (!codes || !scales || !y_bf16) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(y_bf16)) return ZPP_ERR_MISALIGNED;
  return cuda_status(launch_qwz_dequant(codes, scales, nranks, shard_elems, block, bits, y_bf16,
                                        static_cast<cudaStream_t>(stream)));
}

zpp_status zpp_qgz_reorder_quant(const uint16_t* grads_bf16, int32_t nodes,
                                 int32_t gpus_per_node, int64_t bucket_elems, int32_t block,
                                 int32_t bits, void* codes, float* scales, void* stream) {
  zpp_status s = check_topology(nodes, gpus_per_node, bucket_elems, block, bits);
  if (s != ZPP_OK) return s;
  if (bucket_elems == 0) return ZPP_OK;
  if (!grads_bf16 || !codes || !scales) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(grads_bf16) || !aligned16(codes) || !aligned16(scales))
    return ZPP_ERR_MISALIGNED;
  return cuda_status(launch_qgz_reorder_quant(grads_bf16, nullptr, nodes, gpus_per_node,
                                              bucket_elems, block, bits, codes, scales,
                                              static_cast<cudaStream_t>(stream)));
}

zpp_status zpp_ring_rs_step(int32_t step, int32_t nranks, int64_t bucket_elems, int32_t block,
                            int32_t bits, const uint16_t* grads_bf16, const void* codes_in,
                            const float* scales_in, void* codes_out, float* scales_out,
                            float* grad_out, void* stream) {
  zpp_status s = check_topology(1, nranks, bucket_elems, block, bits);
  if (s != ZPP_OK) return s;
  if (step < 0 || step >= nranks) return ZPP_ERR_INVALID_ARG;
  if (bucket_elems == 0) return ZPP_OK;
  const bool first = step == 0, last = step == nranks - 1;
  if (!grads_bf16 || (!first && (!codes_in || !scales_in)) ||
      (!last && (!codes_out || !scales_out)) || (last && !grad_out))
    return ZPP_ERR_INVALID_ARG;
  if (!aligned16(grads_bf16) || (!first && (!aligned16(codes_in) || !aligned16(scales_in))) ||
      (!last && (!aligned16(codes_out) || !aligned16(scales_out))) ||
      (last && !aligned16(grad_out)))
    return ZPP_ERR_MISALIGNED;
  return cuda_status(launch_ring_rs_step(step, nranks, bucket_elems, block, bits, grads_bf16,
                                         codes_in, scales_in, codes_out, scales_out, grad_out,
                                         static_cast<cudaStream_t>(stream)));
}

zpp_status zpp_hpz_gather(int32_t gpus_per_node, int32_t shards_per_rank, int64_t shard_elems,
                          int32_t block, int32_t bits, const void* const* sec_codes,
                          const float* const* sec_scales, uint16_t* y_bf16, void* stream) {
  if (gpus_per_node < 1 || gpus_per_node > kMaxHpzSources || shards_per_rank < 1 ||
      shard_elems < 0 || !valid_block(block) || !(bits == 16 || valid_bits(bits)))
    return ZPP_ERR_INVALID_ARG;
  if (bits == 4 && (shard_elems & 1)) return ZPP_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)gpus_per_node * shards_per_rank;
  if (shard_elems > 0 && rows > kMaxElems / shard_elems) return ZPP_ERR_INVALID_ARG;
  if (shard_elems == 0) return ZPP_OK;
  if (!sec_codes || !y_bf16 || (bits != 16 && !sec_scales)) return ZPP_ERR_INVALID_ARG;
  for (int l = 0; l < gpus_per_node; ++l) {
    if (!sec_codes[l] || (bits != 16 && !sec_scales[l])) return ZPP_ERR_INVALID_ARG;
    if (!aligned16(sec_codes[l]) || (bits != 16 && !aligned16(sec_scales[l])))
      return ZPP_ERR_MISALIGNED;
  }
  if (!aligned16(y_bf16)) return ZPP_ERR_MISALIGNED;
  return cuda_status(launch_hpz_gather(gpus_per_node, shards_per_rank, shard_elems, block, bits,
                                       sec_codes, sec_scales, y_bf16,
                                       static_cast<cudaStream_t>(stream)));
}

int64_t zpp_hpz_secondary_bytes(int32_t shards_per_rank, int64_t shard_elems, int32_t block,
                                int32_t bits) {
  if (shards_per_rank < 1 || shard_elems < 0 || !valid_block(block)) return -1;
  if (shard_elems > kMaxElems / shards_per_rank) return -1;
  if (bits == 16) return (int64_t)shards_per_rank * 2 * shard_elems;
  if (!valid_bits(bits)) return -1;
  return (int64_t)shards_per_rank *
         (zpp_codes_bytes(shard_elems, bits) + 4 * zpp_num_blocks(shard_elems, block));
}

zpp_status zpp_grad_accumulate(const uint16_t* grads_bf16, float* acc, int64_t n, int32_t first,
                               void* stream) {
  if (n < 0 || n > kMaxElems || (first != 0 && first != 1)) return ZPP_ERR_INVALID_ARG;
  if (n == 0) return ZPP_OK;
  if (!grads_bf16 || !acc) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(grads_bf16) || !aligned16(acc)) return ZPP_ERR_MISALIGNED;
  return cuda_status(launch_grad_accumulate(grads_bf16, acc, n, first,
                                            static_cast<cudaStream_t>(stream)));
}

zpp_status zpp_qgz_reorder_quant_acc(const uint16_t* grads_bf16, const float* acc, int32_t nodes,
                                     int32_t gpus_per_node, int64_t bucket_elems, int32_t block,
                                     int32_t bits, void* codes, float* scales, void* stream) {
  zpp_status s = check_topology(nodes, gpus_per_node, bucket_elems, block, bits);
  if (s != ZPP_OK) return s;
  if (bucket_elems == 0) return ZPP_OK;
  if (!grads_bf16 || !acc || !codes || !scales) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(grads_bf16) || !aligned16(acc) || !aligned16(codes) || !aligned16(scales))
    return ZPP_ERR_MISALIGNED;
  return cuda_status(launch_qgz_reorder_quant(grads_bf16, acc, nodes, gpus_per_node, bucket_elems,
                                              block, bits, codes, scales,
                                              static_cast<cudaStream_t>(stream)));
}

zpp_status zpp_qgz_hop_reduce(int32_t hop, const void* codes_in, const float* scales_in,
                              int32_t nodes, int32_t gpus_per_node, int64_t bucket_elems,
                              int32_t block, int32_t bits, void* codes_out,
                              float* scales_out, float* grad_out,
                              const zpp_adam_hparams* adam, const zpp_adam_state* state,
                              void* stream) {
  zpp_status s = check_topology(nodes, gpus_per_node, bucket_elems, block, bits);
  if (s != ZPP_OK) return s;
  if (hop != 1 && hop != 2) return ZPP_ERR_INVALID_ARG;
  if (hop == 2 && nodes < 2) return ZPP_ERR_INVALID_ARG;  // with one node hop 1 is final
  const bool final_hop = (hop == 2) || (nodes == 1);
  if (final_hop) {
    if (codes_out || scales_out) return ZPP_ERR_INVALID_ARG;
    if (!grad_out && !adam) return ZPP_ERR_INVALID_ARG;
    if (adam && !state) return ZPP_ERR_INVALID_ARG;
  } else {
    if (!codes_out || !scales_out || grad_out || adam || state) return ZPP_ERR_INVALID_ARG;
  }
  HopLaunch h{};
  if (adam) {
    s = adam_consts(adam, &h.ac);
    if (s != ZPP_OK) return s;
    s = check_state(state);
    if (s != ZPP_OK) return s;
  }
  if (bucket_elems == 0) return ZPP_OK;
  if (!codes_in || !scales_in) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(codes_in) || !aligned16(scales_in) || (codes_out && !aligned16(codes_out)) ||
      (scales_out && !aligned16(scales_out)) || (grad_out && !aligned16(grad_out)))
    return ZPP_ERR_MISALIGNED;
  h.hop = hop;
  h.codes_in = codes_in;
  h.scales_in = scales_in;
  h.N = nodes;
  h.G = gpus_per_node;
  h.bucket = bucket_elems;
  h.block = block;
  h.bits = bits;
  h.codes_out = codes_out;
  h.scales_out = scales_out;
  h.grad_out = grad_out;
  h.inv_nd = 1.0f / (float)((int64_t)nodes * gpus_per_node);
  h.adam = adam != nullptr;
  if (adam) {
    h.master = state->master;
    h.m = state->m;
    h.v = state->v;
    h.param = state->param_bf16;
  }
  return cuda_status(launch_hop_reduce(h, static_cast<cudaStream_t>(stream)));
}

zpp_status zpp_qgz_final_hop_adam_qwz(int32_t hop, const void* codes_in, const float* scales_in,
                                      int32_t nodes, int32_t gpus_per_node,
                                      int64_t bucket_elems, int32_t block, int32_t bits,
                                      float* grad_out, const zpp_adam_hparams* adam,
                                      const zpp_adam_state* state, int32_t qwz_bits,
                                      void* qwz_codes, float* qwz_scales, void* stream) {
  zpp_status s = check_topology(nodes, gpus_per_node, bucket_elems, block, bits);
  if (s != ZPP_OK) return s;
  if (hop != 1 && hop != 2) return ZPP_ERR_INVALID_ARG;
  if ((hop == 2) != (nodes > 1)) return ZPP_ERR_INVALID_ARG;  // must be the final hop
  if (!adam || !state) return ZPP_ERR_INVALID_ARG;
  if (qwz_bits != 8) return qwz_bits == 4 ? ZPP_ERR_UNSUPPORTED : ZPP_ERR_INVALID_ARG;
  HopLaunch h{};
  s = adam_consts(adam, &h.ac);
  if (s != ZPP_OK) return s;
  s = check_state(state);
  if (s != ZPP_OK) return s;
  const int64_t nd = (int64_t)nodes * gpus_per_node;
  const int64_t L = bucket_elems / nd;
  const int64_t unit = block > 512 ? block : 512;
  if (L % unit != 0) return ZPP_ERR_UNSUPPORTED;
  if (bucket_elems == 0) return ZPP_OK;
  if (!codes_in || !scales_in || !qwz_codes || !qwz_scales) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(codes_in) || !aligned16(scales_in) || !aligned16(qwz_codes) ||
      !aligned16(qwz_scales) || (grad_out && !aligned16(grad_out)))
    return ZPP_ERR_MISALIGNED;
  h.hop = hop;
  h.codes_in = codes_in;
  h.scales_in = scales_in;
  h.N = nodes;
  h.G = gpus_per_node;
  h.bucket = bucket_elems;
  h.block = block;
  h.bits = bits;
  h.grad_out = grad_out;
  h.inv_nd = 1.0f / (float)nd;
  h.adam = true;
  h.master = state->master;
  h.m = state->m;
  h.v = state->v;
  h.param = state->param_bf16;
  h.qwz_codes = qwz_codes;
  h.qwz_scales = qwz_scales;
  return cuda_status(launch_hop_reduce(h, static_cast<cudaStream_t>(stream)));
}

zpp_status zpp_shard_adam_step(const float* grad, int64_t n, const zpp_adam_hparams* hp,
                               const zpp_adam_state* st, void* stream) {
  if (n < 0 || n > kMaxElems) return ZPP_ERR_INVALID_ARG;
  AdamConstsHost ac{};
  zpp_status s = adam_consts(hp, &ac);
  if (s != ZPP_OK) return s;
  s = check_state(st);
  if (s != ZPP_OK) return s;
  if (n == 0) return ZPP_OK;
  if (!grad) return ZPP_ERR_INVALID_ARG;
  if (!aligned16(grad)) return ZPP_ERR_MISALIGNED;
  return cuda_status(launch_adam(grad, n, ac, st->master, st->m, st->v, st->param_bf16,
                                 static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
