// ring.cu -- one step of a ring reduce-scatter of quantized gradients, for
// every simulated rank at once: the precision (and time) comparator of qgZ.
//
// ("Quantized LLM Training at Scale with ZeRO++", 3 QGZ, the challenge of
// sequential quantization: in a ring reduce-scatter every GPU dequantizes the
// partial sum it receives, adds its own gradient chunk and requantizes it for
// the next GPU, N sequential quantizations where qgZ's one-shot scheme has one.)
//
// Ring r -> r + 1 (mod N_d); chunk c = elements [c*L, (c+1)*L) of a rank's
// bucket; at step s rank r works on chunk c = (r - 1 - s) mod N_d:
//   s = 0            msg_r = Q(x_r[c])
//   0 < s < N_d - 1  msg_r = Q(D(msg_{r-1}) + x_r[c])
//   s = N_d - 1      g_r   = (D(msg_{r-1}) + x_r[r]) * (1.0f / N_d)
// Q is the block quantization of the other codecs (blocks restart at the chunk
// start), D = (float)q * s, + one rounded fp32 add.
//
// Streaming, like the one-shot quantizer: 2 B of own gradient in, plus the
// incoming message (bits/8 + 4/B B) after the first step, and the outgoing
// message (or 4 B of fp32 gradient at the last step) out, per element.
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {
namespace {

constexpr int kRingRows = 4;  // rows of 256 elements per warp slab

struct RingArgs {
  const uint16_t* x;          // [N_d][bucket] bf16
  const uint8_t* codes_in;    // [N_d][cb]: the message each rank received
  const float* scales_in;     // [N_d][nb]
  uint8_t* codes_out;         // [N_d][cb]
  float* scales_out;          // [N_d][nb]
  float* grad_out;            // [N_d][L] (last step)
  int64_t bucket, L, cb, nb;
  int64_t units_per_row, total_units;
  int32_t nd, step;
  float inv_nd;
  float one;  // 1.0f, read at run time (see accumulate8)
};

enum { kRingFirst = 0, kRingMiddle = 1, kRingLast = 2 };

template <int BITS, int LOGB, int MODE>
__global__ void __launch_bounds__(kThreads) ring_kernel(const RingArgs a) {
  using G = Geo<LOGB, kRingRows>;
  constexpr int K = kRingRows;
  constexpr int GPC = kWarps / G::WPB;
  using CW = typename CodeVec<BITS>::T;
  __shared__ float red[2][kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = warp / G::WPB, wsub = warp - gid * G::WPB;
  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * GPC + gid, (int64_t)gridDim.x * GPC, u, uend);
  if (u >= uend) return;  // the whole group shares the range
  int64_t r = u / a.units_per_row;
  int64_t t = u - r * a.units_per_row;
  const bool has_input = MODE == kRingMiddle || (MODE == kRingLast && a.step > 0);
  int parity = 0;
  // A rank's row pointers: its own chunk c = (r - 1 - step) mod N_d and the
  // message of rank r - 1 (r - 1 - step lies in [-N_d, N_d - 2], one wrap).
  struct Row {
    const uint16_t* x;
    const uint8_t* c;
    const float* s;
  };
  auto row_of = [&](int64_t rr) -> Row {
    const int32_t ri = (int32_t)rr;
    int32_t c = ri - 1 - a.step;
    if (c < 0) c += a.nd;
    const int32_t prev = ri == 0 ? a.nd - 1 : ri - 1;
    if (!has_input) return {a.x + rr * a.bucket + (int64_t)c * a.L, nullptr, nullptr};
    return {a.x + rr * a.bucket + (int64_t)c * a.L, a.codes_in + (int64_t)prev * a.cb,
            a.scales_in + (int64_t)prev * a.nb};
  };
  // The next unit's loads are issued before the current unit is computed.
  struct Loads {
    uint4 x[K];
    CW c[K];
    float s[K];
  };
  auto load = [&](Loads& l, const Row& row, int64_t tt) {
    const int64_t ew = tt * G::U + (int64_t)wsub * G::kWarpElems;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t e = ew + k * 256 + lane * 8;
      if (e < a.L) {
        l.x[k] = __ldcs(reinterpret_cast<const uint4*>(row.x + e));
        if (has_input) {
          l.c[k] = __ldcs(reinterpret_cast<const CW*>(row.c + ((e * BITS) >> 3)));
          l.s[k] = __ldg(row.s + (e >> LOGB));
        }
      }
    }
  };
  Row cur_row = row_of(r), nxt_row = cur_row;
  Loads cur, nxt;
  load(cur, cur_row, t);
  for (; u < uend; ++u, parity ^= 1) {
    int64_t rn = r, tn = t + 1;
    if (tn == a.units_per_row) {
      tn = 0;
      ++rn;
      if (u + 1 < uend) nxt_row = row_of(rn);
    }
    if (u + 1 < uend) load(nxt, nxt_row, tn);
    const int64_t e_warp = t * G::U + (int64_t)wsub * G::kWarpElems;
    const int64_t valid = a.L - e_warp;  // a multiple of 64 when positive
    float v[K][8];
    int nv[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int e = k * 256 + lane * 8;
      nv[k] = (int64_t)e < valid ? 8 : 0;
      if (nv[k]) {
        unpack_bf16x8(cur.x[k], v[k]);
        if (has_input) {
          float q[8];
          decode8<BITS>(cur.c[k], q);
          accumulate8(v[k], q, cur.s[k], a.one);  // own + D(msg), each rounded
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[k][i] = 0.0f;
      }
    }
    if constexpr (MODE == kRingLast) {
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if (!nv[k]) continue;
        float g[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = __fmul_rn(v[k][i], a.inv_nd);
        st8_cs(a.grad_out + r * a.L + e_warp + k * 256 + lane * 8, false, g);
      }
    } else {
      const int64_t dst = r * a.L;  // rank r's message starts at element r*L
      quantize_unit<BITS, LOGB, G>(v, nv, true, dst, dst >> LOGB, e_warp, a.codes_out,
                                   a.scales_out, red, parity, warp, gid, lane);
    }
    r = rn;
    t = tn;
    cur = nxt;
    cur_row = nxt_row;
  }
}

// Whole-unit chunks (L a multiple of the unit): a lane owns 32 consecutive
// elements of its warp's 1024, as in the hop-1 kernel.  Per unit it loads 64
// bytes of its own bf16 chunk (two 32-byte vectors when WIDE: whole sectors per
// request), one code vector (16 bytes int4, 32 int8) and one scale of the
// incoming message; a block of B <= 1024 elements is B/32 neighbouring lanes.
// The next unit's loads are in flight while the current one is computed.
//
// Units whose incoming scales are all below 2^-5 (a warp vote) are
// dequantized by one FMA a code (dequant_acc_i4 / dequant_acc_i8); others by
// the magic-number decode.  WIDE: x and grad_out 32-byte aligned.
//
// Three CTAs an SM (80 registers, a few values spilled to L1): the kernel waits
// on memory, and the extra warps hide more of it than the spills cost
// (measured on GB300: 0.69 -> 0.76 of the copy peak against two CTAs an SM).
template <int BITS, int LOGB, int MODE, bool WIDE>
__global__ void __launch_bounds__(kThreads, 3) ring1_kernel(const RingArgs a) {
  using G = Geo<LOGB, kRingRows>;
  constexpr int WPB = G::WPB, GPC = kWarps / WPB;
  constexpr int QMAX = (1 << (BITS - 1)) - 1;
  constexpr int CV = BITS / 4;                       // 16-byte code vectors of a lane
  constexpr unsigned kAll = 0xffffffffu;
  __shared__ float red[2][kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = warp / WPB, wsub = warp - gid * WPB;
  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * GPC + gid, (int64_t)gridDim.x * GPC, u, uend);
  if (u >= uend) return;  // the whole group shares the range
  int64_t r = u / a.units_per_row;
  int64_t t = u - r * a.units_per_row;
  const bool has_input = MODE == kRingMiddle || (MODE == kRingLast && a.step > 0);
  const int64_t e_lane = (int64_t)wsub * G::kWarpElems + 32 * lane;  // lane's element in tile 0
  // rank rr's pointers at tile 0: its own chunk c = (rr - 1 - step) mod N_d and the
  // message of rank rr - 1
  struct Row {
    const float* x;  // bf16 pairs, read as 32-bit words
    const uint8_t* c;
    const float* s;
  };
  auto row_of = [&](int64_t rr) -> Row {
    const int32_t ri = (int32_t)rr;
    int32_t c = ri - 1 - a.step;
    if (c < 0) c += a.nd;
    const int32_t prev = ri == 0 ? a.nd - 1 : ri - 1;
    Row w;
    w.x = reinterpret_cast<const float*>(a.x + rr * a.bucket + (int64_t)c * a.L + e_lane);
    w.c = has_input ? a.codes_in + (int64_t)prev * a.cb + ((e_lane * BITS) >> 3) : nullptr;
    w.s = has_input ? a.scales_in + (int64_t)prev * a.nb + (e_lane >> LOGB) : nullptr;
    return w;
  };
  struct Loads {
    float x[16];  // 32 bf16
    uint32_t c[BITS];
    float s;
  };
  auto load = [&](Loads& l, const Row& w, int64_t tt) {
    const int64_t eo = tt * G::U;
    float (&x0)[8] = *reinterpret_cast<float(*)[8]>(&l.x[0]);
    float (&x1)[8] = *reinterpret_cast<float(*)[8]>(&l.x[8]);
    ld8_cs(w.x + eo / 2, WIDE, x0);
    ld8_cs(w.x + eo / 2 + 8, WIDE, x1);
    if (has_input) {
      const uint4* cp = reinterpret_cast<const uint4*>(w.c + ((eo * BITS) >> 3));
#pragma unroll
      for (int h = 0; h < CV; ++h) {
        const uint4 v = __ldcs(cp + h);
        l.c[4 * h] = v.x;
        l.c[4 * h + 1] = v.y;
        l.c[4 * h + 2] = v.z;
        l.c[4 * h + 3] = v.w;
      }
      l.s = __ldg(w.s + (eo >> LOGB));
    }
  };

  Row cur_row = row_of(r), nxt_row = cur_row;
  Loads cur, nxt;
  load(cur, cur_row, t);
  int parity = 0;
  for (; u < uend; ++u, parity ^= 1) {
    int64_t rn = r, tn = t + 1;
    if (tn == a.units_per_row) {
      tn = 0;
      ++rn;
      if (u + 1 < uend) nxt_row = row_of(rn);
    }
    if (u + 1 < uend) load(nxt, nxt_row, tn);

    float v[4][8];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w = __float_as_uint(cur.x[4 * m + i]);
        v[m][2 * i] = bf16_lo(w);
        v[m][2 * i + 1] = bf16_hi(w);
      }
    if (has_input) {  // own + D(msg), each rounded
      const bool fma_path = __all_sync(kAll, cur.s < kFmaDequantMaxScale);
      lane32_dequant_acc<BITS>(cur.c, cur.s, fma_path, a.one, v);
    }
    const int64_t e = t * G::U + e_lane;  // the lane's first element within the chunk
    if constexpr (MODE == kRingLast) {
      float* go = a.grad_out + r * a.L + e;
      const float2 inv = make_float2(a.inv_nd, a.inv_nd);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float g[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float2 p = mul2(make_float2(v[m][i], v[m][i + 1]), inv);
          g[i] = p.x;
          g[i + 1] = p.y;
        }
        st8_cs(go + 8 * m, WIDE, g);
      }
    } else {  // requantize the lane's 32 values with its block's scale
      const Scale sc = lane32_block_scale<QMAX, LOGB, WPB>(v, red, parity, warp, gid, lane);
      lane32_quantize_store<BITS>(v, sc, a.codes_out + r * a.cb + ((e * BITS) >> 3));
      if ((e & (G::B - 1)) == 0) a.scales_out[r * a.nb + (e >> LOGB)] = sc.s;
    }
    r = rn;
    t = tn;
    cur = nxt;
    cur_row = nxt_row;
  }
}

template <int BITS, int MODE>
cudaError_t run_ring(RingArgs a, int block, cudaStream_t st) {
  return dispatch_logb(block, [&](auto lb) -> cudaError_t {
    constexpr int LOGB = decltype(lb)::value;
    using G = Geo<LOGB, kRingRows>;
    a.units_per_row = (a.L + G::U - 1) / G::U;
    a.total_units = (int64_t)a.nd * a.units_per_row;
    const int64_t groups = kWarps / G::WPB;
    const int64_t ctas = (a.total_units + groups - 1) / groups;
    if (a.L % G::U == 0) {  // whole-unit chunks
      auto launch1 = [&](auto w) {
        constexpr bool W = decltype(w)::value;
        const void* k = reinterpret_cast<const void*>(&ring1_kernel<BITS, LOGB, MODE, W>);
        // four rounds of CTAs: measured on GB300 (two-hop buckets, a middle step) 0.726 of
        // the copy peak with one persistent round, 0.748 with four, 0.742 with eight, 0.678
        // with sixteen
        ring1_kernel<BITS, LOGB, MODE, W><<<grid_for(k, ctas, 0, 4), kThreads, 0, st>>>(a);
      };
      if (aligned32(a.x) && (!a.grad_out || aligned32(a.grad_out)))
        launch1(std::integral_constant<bool, true>{});
      else
        launch1(std::integral_constant<bool, false>{});
      return cudaGetLastError();
    }
    const void* k = reinterpret_cast<const void*>(&ring_kernel<BITS, LOGB, MODE>);
    ring_kernel<BITS, LOGB, MODE><<<grid_for(k, ctas), kThreads, 0, st>>>(a);
    return cudaGetLastError();
  });
}

template <int BITS>
cudaError_t run_ring_mode(const RingArgs& a, int block, cudaStream_t st) {
  if (a.step == a.nd - 1) return run_ring<BITS, kRingLast>(a, block, st);
  if (a.step == 0) return run_ring<BITS, kRingFirst>(a, block, st);
  return run_ring<BITS, kRingMiddle>(a, block, st);
}

}  // namespace

cudaError_t launch_ring_rs_step(int32_t step, int32_t nd, int64_t bucket, int32_t block,
                                int32_t bits, const uint16_t* x, const void* codes_in,
                                const float* scales_in, void* codes_out, float* scales_out,
                                float* grad_out, cudaStream_t st) {
  RingArgs a{};
  a.x = x;
  a.codes_in = static_cast<const uint8_t*>(codes_in);
  a.scales_in = scales_in;
  a.codes_out = static_cast<uint8_t*>(codes_out);
  a.scales_out = scales_out;
  a.grad_out = grad_out;
  a.bucket = bucket;
  a.L = bucket / nd;
  a.cb = a.L * bits / 8;
  a.nb = a.L / block;
  a.nd = nd;
  a.step = step;
  a.inv_nd = 1.0f / (float)nd;
  a.one = 1.0f;
  return bits == 8 ? run_ring_mode<8>(a, block, st) : run_ring_mode<4>(a, block, st);
}

}  // namespace zpp
