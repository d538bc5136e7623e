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

constexpr int kQRows = 4;  // rows of 256 elements per warp slab

struct QuantArgs {
  const uint16_t* x;
  const float* acc;       // accumulated micro-batch gradients (fp32), or null
  uint8_t* codes;
  float* scales;
  int64_t total_units;    // rows * units_per_row
  int64_t units_per_row;
  int64_t row_len;        // qwZ: shard; qgZ: slice length L
  int64_t row_blocks;     // qwZ: scales per shard
  int64_t bucket;         // qgZ: elements per rank
  int32_t nd, N, G;       // qgZ topology
};

// A warp unit is q_rows rows of 256 elements; each warp keeps q_stages units
// (a power of two) in a shared-memory prefetch ring.  bf16 input: 4 rows,
// 4 stages (2 KiB a unit).  With the fp32 accumulator riding along (6 B an
// element): 2 rows, 4 stages, so three 3 KiB units stay in flight per warp.
template <bool ACC>
__host__ __device__ constexpr int q_rows() { return ACC ? 2 : kQRows; }
template <bool ACC>
__host__ __device__ constexpr int q_stages() { return ACC ? 2 : 4; }
template <bool ACC>
__host__ __device__ constexpr size_t q_smem() {
  return (size_t)kWarps * q_stages<ACC>() * q_rows<ACC>() * 32 *
         (sizeof(uint4) + (ACC ? 2 * sizeof(float4) : 0));
}

// Tiled layout: every row is a whole number of units, so unit u's input is the
// contiguous run x[u*U + ...] (qwZ shards and qgZ slices follow one another in
// memory).  Each warp keeps its next q_stages-1 units in flight with cp.async
// into its own slice of shared memory: the loads never wait behind the
// arithmetic and cost no registers.
//
// One row = one contiguous run quantized in blocks restarting at the row
// start: a qwZ shard, or slice j of rank r's qgZ bucket, whose codes go to
// slice position p = l'*N + n' (j = n'*G + l') of rank r's message.
//
// ACC: the quantized value is acc + x, the fp32 accumulator of the earlier
// micro-batches plus the last micro-batch's bf16 gradient (one fp32 add).
template <int BITS, bool REORDER, int LOGB, bool ACC>
__global__ void __launch_bounds__(kThreads) quant_tiled_kernel(const QuantArgs a) {
  constexpr int K = q_rows<ACC>(), S = q_stages<ACC>();
  using G = Geo<LOGB, K>;
  constexpr int GPC = kWarps / G::WPB;
  __shared__ float red[2][kWarps];
  extern __shared__ uint4 qsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = warp / G::WPB, wsub = warp - gid * G::WPB;
  uint4* ring = qsm + (size_t)warp * S * K * 32;  // [S][K][32]
  float4* aring = reinterpret_cast<float4*>(qsm + (size_t)kWarps * S * K * 32) +
                  (size_t)warp * S * K * 64;      // [S][K][64]: rows of 256 floats

  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * GPC + gid, (int64_t)gridDim.x * GPC, u, uend);
  if (u >= uend) return;  // the whole group shares the range
  const uint16_t* xg = a.x + (int64_t)wsub * G::kWarpElems + lane * 8;
  const float* ag = ACC ? a.acc + (int64_t)wsub * G::kWarpElems + lane * 4 : nullptr;
  auto issue = [&](int64_t v) {
    if (v < uend) {
      const uint16_t* src = xg + v * G::U;
      uint4* slot = ring + (size_t)(v & (S - 1)) * K * 32 + lane;
#pragma unroll
      for (int k = 0; k < K; ++k) cp_async16(slot + k * 32, src + k * 256);
      if constexpr (ACC) {  // whole rows, 512 contiguous bytes per instruction
        const float* asrc = ag + v * G::U;
        float4* aslot = aring + (size_t)(v & (S - 1)) * K * 64 + lane;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          cp_async16(aslot + k * 64, asrc + k * 256);
          cp_async16(aslot + k * 64 + 32, asrc + k * 256 + 128);
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < S - 1; ++i) issue(u + i);

  // destination of the current unit: row = u / units_per_row, tile t
  int64_t row = u / a.units_per_row;
  int64_t t = u - row * a.units_per_row;
  int32_t r = 0, j = 0, np = 0, lp = 0;
  if constexpr (REORDER) {
    r = (int32_t)(row / a.nd);
    j = (int32_t)(row - (int64_t)r * a.nd);
    np = j / a.G;
    lp = j - np * a.G;
  }
  auto row_dst = [&]() -> int64_t {
    if constexpr (REORDER)
      return (int64_t)r * a.bucket + ((int64_t)lp * a.N + np) * a.row_len;
    else
      return row * a.row_len;
  };
  int64_t dst_row = row_dst();
  int nv[K];
#pragma unroll
  for (int k = 0; k < K; ++k) nv[k] = 8;
  int parity = 0;

  for (; u < uend; ++u, parity ^= 1) {
    if constexpr (ACC) __syncwarp();  // every lane is done with the slot refilled next
    issue(u + S - 1);
    cp_async_wait<S - 1>();  // this unit's copies have landed
    if constexpr (ACC) __syncwarp();  // ... the other lanes' accumulator copies too
    float x[K][8];
    const uint4* slot = ring + (size_t)(u & (S - 1)) * K * 32 + lane;
#pragma unroll
    for (int k = 0; k < K; ++k) unpack_bf16x8(slot[k * 32], x[k]);
    if constexpr (ACC) {
      const float4* aslot = aring + (size_t)(u & (S - 1)) * K * 64 + 2 * lane;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const float4 p0 = aslot[k * 64], p1 = aslot[k * 64 + 1];
        const float av[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) x[k][i] = __fadd_rn(av[i], x[k][i]);
      }
    }
    const int64_t e_warp = t * G::U + (int64_t)wsub * G::kWarpElems;
    quantize_unit<BITS, LOGB, G>(x, nv, true, dst_row, dst_row >> LOGB, e_warp, a.codes, a.scales,
                                 red, parity, warp, gid, lane);
    if (++t == a.units_per_row) {
      t = 0;
      ++row;
      if constexpr (REORDER) {
        ++j;
        if (++lp == a.G) {
          lp = 0;
          ++np;
        }
        if (j == a.nd) {
          j = np = lp = 0;
          ++r;
        }
      }
      dst_row = row_dst();
    }
  }
  cp_async_wait<0>();  // no copy outlives the warp
}

// General layout (a row tail shorter than a unit, or shards whose starts are
// not 16-byte aligned): direct loads, element loads with zero fill where needed.
template <int BITS, bool REORDER, int LOGB, bool ACC>
__global__ void __launch_bounds__(kThreads) quant_kernel(const QuantArgs a) {
  constexpr int K = q_rows<ACC>();
  using G = Geo<LOGB, K>;
  constexpr int GPC = kWarps / G::WPB;
  __shared__ float red[2][kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = warp / G::WPB, wsub = warp - gid * G::WPB;
  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * GPC + gid, (int64_t)gridDim.x * GPC, u, uend);
  if (u >= uend) return;
  int64_t row = u / a.units_per_row;
  int64_t t = u - row * a.units_per_row;
  int32_t r = 0, j = 0, np = 0, lp = 0;
  if constexpr (REORDER) {
    r = (int32_t)(row / a.nd);
    j = (int32_t)(row - (int64_t)r * a.nd);
    np = j / a.G;
    lp = j - np * a.G;
  }
  int parity = 0;
  for (; u < uend; ++u, parity ^= 1) {
    const int64_t src_base = row * a.row_len;
    int64_t dst_base, scale_base;
    if constexpr (REORDER) {
      dst_base = (int64_t)r * a.bucket + ((int64_t)lp * a.N + np) * a.row_len;
      scale_base = dst_base >> LOGB;
    } else {
      dst_base = src_base;
      scale_base = row * a.row_blocks;
    }
    const int64_t e_warp = t * G::U + (int64_t)wsub * G::kWarpElems;
    const int64_t valid = a.row_len - e_warp;
    const bool aligned = ((src_base | dst_base) & 7) == 0;
    const uint16_t* xw = a.x + src_base + e_warp;
    float x[K][8];
    int nv[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int e = k * 256 + lane * 8;
      const int64_t rem = valid - e;
      nv[k] = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
      if (nv[k] == 8 && aligned) {
        unpack_bf16x8(__ldcs(reinterpret_cast<const uint4*>(xw + e)), x[k]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          x[k][i] = i < nv[k] ? __uint_as_float((uint32_t)xw[e + i] << 16) : 0.0f;
      }
      if constexpr (ACC) {
        const float* aw = a.acc + src_base + e_warp + e;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < nv[k]) x[k][i] = __fadd_rn(aw[i], x[k][i]);
      }
    }
    quantize_unit<BITS, LOGB, G>(x, nv, aligned, dst_base, scale_base, e_warp, a.codes, a.scales,
                                 red, parity, warp, gid, lane);
    if (++t == a.units_per_row) {
      t = 0;
      ++row;
      if constexpr (REORDER) {
        ++j;
        if (++lp == a.G) {
          lp = 0;
          ++np;
        }
        if (j == a.nd) {
          j = np = lp = 0;
          ++r;
        }
      }
    }
  }
}

// Rows (shards) come from up to kMaxSources separate buffers: source s holds
// rows s*rows_per_src .. s*rows_per_src + rows_per_src - 1, back to back
// (row_code_bytes of codes and row_blocks scales each).  The qwZ receiver is
// the one-source case; the hpZ backward gather reads the G secondary
// partitions of a node.
constexpr int kMaxSources = kMaxHpzSources;

struct DequantArgs {
  const uint8_t* codes[kMaxSources];
  const float* scales[kMaxSources];
  uint16_t* y;
  int64_t total_units, units_per_row;
  int64_t row_len, row_blocks, row_code_bytes, rows_per_src;
};

template <int BITS>
struct RowWord {  // the 8-element load of one lane: codes, or bf16 values when BITS == 16
  using T = typename CodeVec<BITS>::T;
};
template <>
struct RowWord<16> {
  using T = uint4;
};

// y = bf16_rn((float)q * s) for every element of every row; BITS == 16
// copies bf16 rows unchanged.  The next unit's codes and scales are loaded
// before the current unit is converted.
template <int BITS, int LOGB>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const DequantArgs a) {
  constexpr int K = kQRows;
  constexpr int WE = 256 * K;
  using CW = typename RowWord<BITS>::T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * kWarps + warp, (int64_t)gridDim.x * kWarps, u, uend);
  if (u >= uend) return;
  struct Row {
    const uint8_t* c;
    const float* s;
    uint16_t* y;
    bool aligned;
  };
  auto row_of = [&](int64_t rw) -> Row {
    const int64_t src = rw / a.rows_per_src, j = rw - src * a.rows_per_src;
    Row r;
    r.c = a.codes[src] + j * a.row_code_bytes;
    r.s = BITS == 16 ? nullptr : a.scales[src] + j * a.row_blocks;
    r.y = a.y + rw * a.row_len;
    r.aligned = ((reinterpret_cast<uintptr_t>(r.c) % sizeof(CW)) |
                 (reinterpret_cast<uintptr_t>(r.y) & 15)) == 0;
    return r;
  };
  struct Loads {
    CW w[K];
    float s[K];
  };
  // lane-invariant offsets: the lane's code bytes and each row's scale within a unit
  constexpr int ROWB = 256 * BITS / 8;
  const int lane_code = lane * 8 * BITS / 8;
  int soff[K];
#pragma unroll
  for (int k = 0; k < K; ++k) soff[k] = (k * 256 + lane * 8) >> LOGB;
  auto load = [&](Loads& l, const Row& r, int64_t e_warp) {
    const uint8_t* cw = r.c + ((e_warp * BITS) >> 3) + lane_code;
    const float* sw = r.s + (e_warp >> LOGB);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      l.w[k] = __ldcs(reinterpret_cast<const CW*>(cw + k * ROWB));
      if constexpr (BITS != 16) l.s[k] = __ldg(sw + soff[k]);
    }
  };
  int64_t row = u / a.units_per_row;
  int64_t t = u - row * a.units_per_row;
  Row cur_row = row_of(row), nxt_row = cur_row;
  bool cur_full = cur_row.aligned && a.row_len - t * WE >= WE;
  Loads cur, nxt;
  if (cur_full) load(cur, cur_row, t * WE);
  for (; u < uend; ++u) {
    int64_t rown = row, tn = t + 1;
    if (tn == a.units_per_row) {
      tn = 0;
      ++rown;
      if (u + 1 < uend) nxt_row = row_of(rown);
    }
    const bool nxt_full = u + 1 < uend && nxt_row.aligned && a.row_len - tn * WE >= WE;
    if (nxt_full) load(nxt, nxt_row, tn * WE);
    const int64_t e_warp = t * WE;
    uint16_t* yw = cur_row.y + e_warp;
    if (cur_full) {
      uint16_t* yl = yw + lane * 8;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if constexpr (BITS == 16) {
          __stcs(reinterpret_cast<uint4*>(yl + k * 256), cur.w[k]);
        } else {
          float q[8];
          decode8<BITS>(cur.w[k], q);
          const float2 s2 = make_float2(cur.s[k], cur.s[k]);
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const float2 v = mul2(make_float2(q[i], q[i + 1]), s2);
            q[i] = v.x;
            q[i + 1] = v.y;
          }
          __stcs(reinterpret_cast<uint4*>(yl + k * 256),
                 make_uint4(pack_bf16x2(q[0], q[1]), pack_bf16x2(q[2], q[3]),
                            pack_bf16x2(q[4], q[5]), pack_bf16x2(q[6], q[7])));
        }
      }
    } else {
      const uint8_t* crow = cur_row.c;
      const float* srow = cur_row.s;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int e = k * 256 + lane * 8;
        for (int i = 0; i < 8; ++i) {
          const int64_t el = e_warp + e + i;  // element within the row
          if (el >= a.row_len) break;
          if constexpr (BITS == 16) {
            yw[e + i] = reinterpret_cast<const uint16_t*>(crow)[el];
          } else {
            int q;
            if constexpr (BITS == 8) {
              q = (int8_t)crow[el];
            } else {
              const uint8_t b = crow[el >> 1];
              const int nib = (el & 1) ? (b >> 4) : (b & 0xF);
              q = nib >= 8 ? nib - 16 : nib;
            }
            yw[e + i] = bf16_bits(__fmul_rn((float)q, srow[el >> LOGB]));
          }
        }
      }
    }
    row = rown;
    t = tn;
    cur_row = nxt_row;
    cur_full = nxt_full;
    cur = nxt;
  }
}

template <int BITS, bool REORDER, bool ACC>
cudaError_t run_quant(const QuantArgs& a0, int block, cudaStream_t st) {
  return dispatch_logb(block, [&](auto lb) -> cudaError_t {
    constexpr int LOGB = decltype(lb)::value;
    using G = Geo<LOGB, q_rows<ACC>()>;
    QuantArgs a = a0;
    a.units_per_row = (a.row_len + G::U - 1) / G::U;
    a.total_units = a.total_units * a.units_per_row;  // caller passes the row count
    const int64_t groups = kWarps / G::WPB;
    const int64_t ctas = (a.total_units + groups - 1) / groups;
    if (a.row_len % G::U == 0) {  // tiled: every unit full, 16-byte aligned
      constexpr size_t smem = q_smem<ACC>();
      const void* k = reinterpret_cast<const void*>(&quant_tiled_kernel<BITS, REORDER, LOGB, ACC>);
      const cudaError_t attr = smem_opt_in(k, smem);
      if (attr != cudaSuccess) return attr;
      quant_tiled_kernel<BITS, REORDER, LOGB, ACC>
          <<<grid_for(k, ctas, smem, kStreamWaves), kThreads, smem, st>>>(a);
    } else {
      const void* k = reinterpret_cast<const void*>(&quant_kernel<BITS, REORDER, LOGB, ACC>);
      quant_kernel<BITS, REORDER, LOGB, ACC><<<grid_for(k, ctas), kThreads, 0, st>>>(a);
    }
    return cudaGetLastError();
  });
}

template <int BITS>
cudaError_t run_dequant(const DequantArgs& a0, int block, cudaStream_t st) {
  if constexpr (BITS == 16) {  // a copy: the block size plays no part
    const void* k = reinterpret_cast<const void*>(&dequant_kernel<16, 12>);
    dequant_kernel<16, 12>
        <<<grid_for(k, (a0.total_units + kWarps - 1) / kWarps, 0, kStreamWaves), kThreads, 0, st>>>(a0);
    return cudaGetLastError();
  } else {
    return dispatch_logb(block, [&](auto lb) -> cudaError_t {
      constexpr int LOGB = decltype(lb)::value;
      const void* k = reinterpret_cast<const void*>(&dequant_kernel<BITS, LOGB>);
      dequant_kernel<BITS, LOGB>
          <<<grid_for(k, (a0.total_units + kWarps - 1) / kWarps, 0, kStreamWaves), kThreads, 0, st>>>(a0);
      return cudaGetLastError();
    });
  }
}

// acc = (first ? 0 : acc) + (float)g for n elements; 8 per lane per step
// (`wide`: acc 32-byte aligned, one 256-bit access per lane).
__global__ void __launch_bounds__(kThreads) accumulate_kernel(const uint16_t* __restrict__ g,
                                                              float* __restrict__ acc, int64_t n,
                                                              int first, bool wide) {
  const int64_t stride = (int64_t)gridDim.x * kThreads * 8;
  for (int64_t i = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * 8; i < n; i += stride) {
    if (i + 8 <= n) {
      float x[8];
      unpack_bf16x8(__ldcs(reinterpret_cast<const uint4*>(g + i)), x);
      if (!first) {
        float av[8];
        ld8_cs(acc + i, wide, av);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = __fadd_rn(av[k], x[k]);
      }
      st8_cs(acc + i, wide, x);
    } else {
      for (int64_t k = i; k < n; ++k) {
        const float x = __uint_as_float((uint32_t)g[k] << 16);
        acc[k] = first ? x : __fadd_rn(acc[k], x);
      }
    }
  }
}

}  // namespace

cudaError_t launch_grad_accumulate(const uint16_t* g, float* acc, int64_t n, int first,
                                   cudaStream_t st) {
  const void* k = reinterpret_cast<const void*>(&accumulate_kernel);
  const int64_t ctas = (n + (int64_t)kThreads * 8 - 1) / ((int64_t)kThreads * 8);
  accumulate_kernel<<<grid_for(k, ctas, 0, kStreamWaves), kThreads, 0, st>>>(g, acc, n, first,
                                                                         aligned32(acc));
  return cudaGetLastError();
}

cudaError_t launch_qwz_quant(const uint16_t* x, int64_t nranks, int64_t shard, int32_t block,
                             int32_t bits, void* codes, float* scales, cudaStream_t st) {
  QuantArgs a{};
  a.x = x;
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = scales;
  a.total_units = nranks;  // rows; scaled by units per row in run_quant
  a.row_len = shard;
  a.row_blocks = (shard + block - 1) / block;
  return bits == 8 ? run_quant<8, false, false>(a, block, st) : run_quant<4, false, false>(a, block, st);
}

cudaError_t launch_qgz_reorder_quant(const uint16_t* x, const float* acc, int32_t N, int32_t G,
                                     int64_t bucket, int32_t block, int32_t bits, void* codes,
                                     float* scales, cudaStream_t st) {
  QuantArgs a{};
  a.x = x;
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = scales;
  a.nd = N * G;
  a.N = N;
  a.G = G;
  a.bucket = bucket;
  a.row_len = bucket / a.nd;
  a.total_units = (int64_t)a.nd * a.nd;  // rows (rank, slice)
  a.acc = acc;
  if (acc) return bits == 8 ? run_quant<8, true, true>(a, block, st) : run_quant<4, true, true>(a, block, st);
  return bits == 8 ? run_quant<8, true, false>(a, block, st) : run_quant<4, true, false>(a, block, st);
}

namespace {
cudaError_t run_gather(DequantArgs& a, int64_t rows, int64_t shard, int32_t block, int32_t bits,
                       cudaStream_t st) {
  a.units_per_row = (shard + 256 * kQRows - 1) / (256 * kQRows);
  a.total_units = rows * a.units_per_row;
  a.row_len = shard;
  a.row_blocks = (shard + block - 1) / block;
  a.row_code_bytes = shard * bits / 8;
  if (bits == 16) return run_dequant<16>(a, block, st);
  return bits == 8 ? run_dequant<8>(a, block, st) : run_dequant<4>(a, block, st);
}
}  // namespace

cudaError_t launch_qwz_dequant(const void* codes, const float* scales, int64_t nranks,
                               int64_t shard, int32_t block, int32_t bits, uint16_t* y,
                               cudaStream_t st) {
  DequantArgs a{};
  a.codes[0] = static_cast<const uint8_t*>(codes);
  a.scales[0] = scales;
  a.y = y;
  a.rows_per_src = nranks;
  return run_gather(a, nranks, shard, block, bits, st);
}

cudaError_t launch_hpz_gather(int32_t G, int32_t N, int64_t shard, int32_t block, int32_t bits,
                              const void* const* sec_codes, const float* const* sec_scales,
                              uint16_t* y, cudaStream_t st) {
  if (G > kMaxSources) return cudaErrorInvalidValue;
  DequantArgs a{};
  for (int l = 0; l < G; ++l) {
    a.codes[l] = static_cast<const uint8_t*>(sec_codes[l]);
    a.scales[l] = bits == 16 ? nullptr : sec_scales[l];
  }
  a.y = y;
  a.rows_per_src = N;
  return run_gather(a, (int64_t)G * N, shard, block, bits, st);
}

}  // namespace zpp
