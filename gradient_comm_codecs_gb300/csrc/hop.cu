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
//
// Memory-level parallelism: the sources are read in chunks whose loads are
// all issued before the chunk is summed, and the next chunk's loads are in
// flight while the current one is summed (two register buffers); in the Adam
// mode the optimizer state of the unit is loaded before the sum starts.
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
  uint8_t* codes_out;      // requant
  float* scales_out;
  float* grad_out;         // final
  float inv_nd;
  AdamConsts ac;
  float* master;
  float* m;
  float* v;
  uint16_t* param;
  uint8_t* qwz_codes;      // final hop + Adam + qwZ: next step's weight message
  float* qwz_scales;
  bool wide;               // grad_out, master, m, v (those given) 32-byte aligned
  float one;               // 1.0f, read at run time (see accumulate8)
};

// kFinalAdamQwz: the final hop, the Adam step, and the int8 block
// quantization of the new bf16 parameters (the next forward all-gather's qwZ
// message, blocks restarting at every rank's owned shard) in one pass.
enum { kRequant = 0, kFinal = 1, kFinalAdam = 2, kFinalAdamQwz = 3 };

template <int MODE>
constexpr int hop_rows() { return MODE >= kFinalAdam ? 2 : 4; }

template <int BITS, int MODE, int LOGB>
struct HopCfg {
  static constexpr int K = hop_rows<MODE>();
  using G = Geo<LOGB, K>;
  // the requantizing modes need whole blocks per warp group; plain final hops do not
  static constexpr int WPB = (MODE == kRequant || MODE == kFinalAdamQwz) ? G::WPB : 1;
  static constexpr int U = WPB * G::kWarpElems;
  static constexpr int SCH = (BITS == 4 && G::NSC == 1) ? 4 : 2;  // sources per load chunk
};

template <int BITS, int K, int NSC, int SCH>
struct Chunk {
  typename CodeVec<BITS>::T c[SCH][K];
  float s[SCH][NSC];
};

template <int BITS, int MODE, int LOGB>
__global__ void __launch_bounds__(kThreads, 2) hop_kernel(const HopArgs a) {
  using C = HopCfg<BITS, MODE, LOGB>;
  using G = typename C::G;
  constexpr int K = C::K, WPB = C::WPB, SCH = C::SCH, NSC = G::NSC, RPB = G::RPB;
  constexpr int QMAX = (1 << (BITS - 1)) - 1;
  constexpr int GPC = kWarps / WPB;
  using CW = typename CodeVec<BITS>::T;
  using CH = Chunk<BITS, K, NSC, SCH>;
  __shared__ float red[2][kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = warp / WPB, wsub = warp - gid * WPB;

  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * GPC + gid, (int64_t)gridDim.x * GPC, u, uend);
  if (u >= uend) return;
  int64_t d = u / a.units_per_row;
  int64_t t = u - d * a.units_per_row;
  int32_t dn = (int32_t)(d / a.G), dl = (int32_t)(d - (int64_t)dn * a.G);
  int parity = 0;

  for (; u < uend; ++u, parity ^= 1) {
    // hop 1: sources n*G + g, chunk l;  hop 2: sources n'*G + l, slot n
    const int64_t src0 = a.hop == 1 ? (int64_t)dn * a.G : dl;
    const int64_t sstride = a.hop == 1 ? 1 : a.G;
    const int64_t in_off = (a.hop == 1 ? (int64_t)dl : (int64_t)dn) * a.R;
    const int64_t e_warp = t * C::U + (int64_t)wsub * G::kWarpElems;
    const int64_t valid = a.R - e_warp;  // a multiple of 64 when positive
    const int64_t obase = d * a.R + e_warp;
    bool on[K];
#pragma unroll
    for (int k = 0; k < K; ++k) on[k] = (int64_t)(k * 256 + lane * 8) < valid;

    AdamVec st[MODE == kFinalAdam ? K : 1];
    if constexpr (MODE == kFinalAdam) {
#pragma unroll
      for (int k = 0; k < K; ++k)
        if (on[k]) st[k] = adam_load8(obase + k * 256 + lane * 8, a.master, a.m, a.v, a.wide);
    }

    auto load = [&](CH& ch, int s0) {
#pragma unroll
      for (int j = 0; j < SCH; ++j) {
        const int s = s0 + j;
        const int64_t pb = (src0 + (int64_t)s * sstride) * a.in_rank_elems + in_off + e_warp;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const int64_t pos = pb + k * 256 + lane * 8;
          ch.c[j][k] = (s < a.S && on[k])
                           ? __ldcs(reinterpret_cast<const CW*>(a.codes_in + ((pos * BITS) >> 3)))
                           : CW{};
        }
#pragma unroll
        for (int i = 0; i < NSC; ++i) {
          const int64_t pos = pb + i * RPB * 256 + lane * 8;
          ch.s[j][i] = (s < a.S && on[i * RPB]) ? __ldg(a.scales_in + (pos >> LOGB)) : 0.0f;
        }
      }
    };
    float acc[K][8];
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[k][i] = 0.0f;
    auto sum = [&](const CH& ch, int s0) {
#pragma unroll
      for (int j = 0; j < SCH; ++j) {
        if (s0 + j >= a.S) break;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          float q[8];
          decode8<BITS>(ch.c[j][k], q);
          accumulate8(acc[k], q, ch.s[j][k / RPB], a.one);
        }
      }
    };

    CH ca, cb;
    load(ca, 0);
    for (int c = 0; c < a.S; c += 2 * SCH) {
      if (c + SCH < a.S) load(cb, c + SCH);
      sum(ca, c);
      if (c + SCH >= a.S) break;
      if (c + 2 * SCH < a.S) load(ca, c + 2 * SCH);
      sum(cb, c + SCH);
    }

    if constexpr (MODE == kRequant) {
      float am[K];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        float m = fabsf(acc[k][0]);
#pragma unroll
        for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(acc[k][i]));
        am[k] = m;
      }
      Scale sc[NSC];
      block_scales<G, QMAX>(am, sc, red, parity, warp, gid, lane);
      // R is a multiple of B, so obase mod B = e_warp mod B
      const int ew_mod = (int)(e_warp & (G::B - 1));
      float* so = a.scales_out + (obase >> LOGB);
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int e = k * 256 + lane * 8;
        uint32_t c[8];
        quantize8<QMAX>(acc[k], sc[k / RPB], c);
        if (!on[k]) continue;
        *reinterpret_cast<CW*>(a.codes_out + (((obase + e) * BITS) >> 3)) = pack8<BITS>(c);
        if (((ew_mod + e) & (G::B - 1)) == 0) so[(ew_mod + e) >> LOGB] = sc[k / RPB].s;
      }
    } else {
#pragma unroll
      for (int k = 0; k < K; ++k) {
        if (!on[k]) continue;
        const int64_t idx = obase + k * 256 + lane * 8;
        float g[8];
        const float2 inv = make_float2(a.inv_nd, a.inv_nd);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float2 v = mul2(make_float2(acc[k][i], acc[k][i + 1]), inv);
          g[i] = v.x;
          g[i + 1] = v.y;
        }
        if (a.grad_out) st8_cs(a.grad_out + idx, a.wide, g);
        if constexpr (MODE == kFinalAdam)
          adam_apply8(g, st[k], idx, a.master, a.m, a.v, a.param, a.ac, a.wide);
      }
    }

    if (++t == a.units_per_row) {
      t = 0;
      ++d;
      if (++dl == a.G) {
        dl = 0;
        ++dn;
      }
    }
  }
}

// Tiled layout (every destination row a whole number of units, true whenever
// the slice length is a multiple of 1024): per-row source base pointers, no
// per-element 64-bit address arithmetic and no tail predication.  Sources are
// read two at a time, the next pair's loads in flight while the current pair
// is summed.
//
// WIDE (fixed at compile time, so the loads of the next chunk schedule
// freely around the state accesses): grad_out and the Adam state move as one
// 256-bit access per lane; the launcher picks it when they are 32-byte aligned.
//
// SCH: sources per load chunk (two chunks in flight).  Four for the final
// modes of int4 messages with more than two sources, else two; the launcher
// picks it from the source count.
template <int BITS, int MODE, int LOGB, bool WIDE, int SCH>
__global__ void __launch_bounds__(kThreads, 2) hop_tiled_kernel(const HopArgs a) {
  using C = HopCfg<BITS, MODE, LOGB>;
  using G = typename C::G;
  constexpr int K = C::K, WPB = C::WPB, NSC = G::NSC, RPB = G::RPB;
  constexpr int QMAX = (1 << (BITS - 1)) - 1;
  constexpr int GPC = kWarps / WPB;
  constexpr int ROWB = 256 * BITS / 8;  // code bytes of one 256-element row
  using CW = typename CodeVec<BITS>::T;
  using CH = Chunk<BITS, K, NSC, SCH>;
  __shared__ float red[2][kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = warp / WPB, wsub = warp - gid * WPB;

  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * GPC + gid, (int64_t)gridDim.x * GPC, u, uend);
  if (u >= uend) return;
  int64_t d = u / a.units_per_row;
  int64_t t = u - d * a.units_per_row;
  int32_t dn = (int32_t)(d / a.G), dl = (int32_t)(d - (int64_t)dn * a.G);
  // source s of destination d starts at element (src0 + s*sstride)*in_rank_elems + in_off
  const int64_t sstep = (a.hop == 1 ? 1 : (int64_t)a.G) * a.in_rank_elems;
  const int64_t cstep = (sstep * BITS) >> 3;   // bytes between consecutive sources
  const int64_t fstep = sstep >> LOGB;         // scales between consecutive sources
  const uint8_t* crow;
  const float* srow;
  auto row_bases = [&]() {
    const int64_t src0 = a.hop == 1 ? (int64_t)dn * a.G : dl;
    const int64_t e0 = src0 * a.in_rank_elems + (a.hop == 1 ? (int64_t)dl : (int64_t)dn) * a.R;
    crow = a.codes_in + ((e0 * BITS) >> 3) + lane * (8 * BITS / 8);
    srow = a.scales_in + (e0 >> LOGB);
  };
  row_bases();
  // scale of row k's block for this lane, relative to the unit's first scale
  int soff[NSC];
#pragma unroll
  for (int i = 0; i < NSC; ++i) soff[i] = (i * RPB * 256 + lane * 8) >> LOGB;
  int parity = 0;

  for (; u < uend; ++u, parity ^= 1) {
    const int64_t e_warp = t * C::U + (int64_t)wsub * G::kWarpElems;
    const int64_t obase = d * a.R + e_warp;
    const uint8_t* cu = crow + ((e_warp * BITS) >> 3);
    const float* su = srow + (e_warp >> LOGB);

    AdamVec st[MODE >= kFinalAdam ? K : 1];
    if constexpr (MODE >= kFinalAdam) {
#pragma unroll
      for (int k = 0; k < K; ++k) st[k] = adam_load8(obase + k * 256 + lane * 8, a.master, a.m, a.v, WIDE);
    }
    auto load = [&](CH& ch, int s0) {
#pragma unroll
      for (int j = 0; j < SCH; ++j) {
        const int s = s0 + j;
        if (s < a.S) {
          const uint8_t* cs = cu + (int64_t)s * cstep;
          const float* ss = su + (int64_t)s * fstep;
#pragma unroll
          for (int k = 0; k < K; ++k) ch.c[j][k] = __ldcs(reinterpret_cast<const CW*>(cs + k * ROWB));
#pragma unroll
          for (int i = 0; i < NSC; ++i) ch.s[j][i] = __ldg(ss + soff[i]);
        }
      }
    };
    float acc[K][8];
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[k][i] = 0.0f;
    auto sum = [&](const CH& ch, int s0) {
#pragma unroll
      for (int j = 0; j < SCH; ++j) {
        if (s0 + j >= a.S) break;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          float q[8];
          decode8<BITS>(ch.c[j][k], q);
          accumulate8(acc[k], q, ch.s[j][k / RPB], a.one);
        }
      }
    };
    CH ca, cb;
    load(ca, 0);
    for (int c = 0; c < a.S; c += 2 * SCH) {
      if (c + SCH < a.S) load(cb, c + SCH);
      sum(ca, c);
      if (c + SCH >= a.S) break;
      if (c + 2 * SCH < a.S) load(ca, c + 2 * SCH);
      sum(cb, c + SCH);
    }

    if constexpr (MODE == kRequant) {
      float am[K];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const float m0 = fmaxf(fabsf(acc[k][0]), fabsf(acc[k][1]));
        const float m1 = fmaxf(fabsf(acc[k][2]), fabsf(acc[k][3]));
        const float m2 = fmaxf(fabsf(acc[k][4]), fabsf(acc[k][5]));
        const float m3 = fmaxf(fabsf(acc[k][6]), fabsf(acc[k][7]));
        am[k] = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
      }
      Scale sc[NSC];
      block_scales<G, QMAX>(am, sc, red, parity, warp, gid, lane);
      uint8_t* co = a.codes_out + ((obase * BITS) >> 3) + lane * (8 * BITS / 8);
      // R is a multiple of B, so obase mod B = e_warp mod B
      const int ew_mod = (int)(e_warp & (G::B - 1));
      float* so = a.scales_out + (obase >> LOGB);
#pragma unroll
      for (int k = 0; k < K; ++k) {
        uint32_t c[8];
        quantize8<QMAX>(acc[k], sc[k / RPB], c);
        *reinterpret_cast<CW*>(co + k * ROWB) = pack8<BITS>(c);
        const int e = k * 256 + lane * 8;
        if (((ew_mod + e) & (G::B - 1)) == 0) so[(ew_mod + e) >> LOGB] = sc[k / RPB].s;
      }
    } else {
      const float2 inv = make_float2(a.inv_nd, a.inv_nd);
      float pq[MODE == kFinalAdamQwz ? K : 1][8];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int64_t idx = obase + k * 256 + lane * 8;
        float g[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float2 v = mul2(make_float2(acc[k][i], acc[k][i + 1]), inv);
          g[i] = v.x;
          g[i + 1] = v.y;
        }
        if (a.grad_out) st8_cs(a.grad_out + idx, WIDE, g);
        if constexpr (MODE == kFinalAdam)
          adam_apply8(g, st[k], idx, a.master, a.m, a.v, a.param, a.ac, WIDE);
        if constexpr (MODE == kFinalAdamQwz)
          adam_apply8(g, st[k], idx, a.master, a.m, a.v, a.param, a.ac, WIDE, pq[k]);
      }
      if constexpr (MODE == kFinalAdamQwz) {
        float am[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const float m0 = fmaxf(fabsf(pq[k][0]), fabsf(pq[k][1]));
          const float m1 = fmaxf(fabsf(pq[k][2]), fabsf(pq[k][3]));
          const float m2 = fmaxf(fabsf(pq[k][4]), fabsf(pq[k][5]));
          const float m3 = fmaxf(fabsf(pq[k][6]), fabsf(pq[k][7]));
          am[k] = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        }
        Scale sc[NSC];
        block_scales<G, 127>(am, sc, red, parity, warp, gid, lane);
        const int ew_mod = (int)(e_warp & (G::B - 1));  // = obase mod B
        float* qs = a.qwz_scales + (obase >> LOGB);
#pragma unroll
        for (int k = 0; k < K; ++k) {
          uint32_t c[8];
          quantize8<127>(pq[k], sc[k / RPB], c);
          const int e = k * 256 + lane * 8;
          *reinterpret_cast<uint2*>(a.qwz_codes + obase + e) = pack_i8x8(c);
          if (((ew_mod + e) & (G::B - 1)) == 0) qs[(ew_mod + e) >> LOGB] = sc[k / RPB].s;
        }
      }
    }

    if (++t == a.units_per_row) {
      t = 0;
      ++d;
      if (++dl == a.G) {
        dl = 0;
        ++dn;
      }
      row_bases();
    }
  }
}

// Hop 1 of a two-hop topology (dequantize, sum the G sources of the node in
// rank order, requantize), laid out for the sum: a lane owns 32 consecutive
// elements of the warp's 1024, so one source costs it one 16-byte code load
// (int4; two for int8) and one scale load, and a block of B <= 1024 elements
// is B/32 neighbouring lanes.  (Messages start 16-byte aligned and every
// source, row and unit offset is a multiple of 1024 elements, so each lane's
// code vector is 16-byte aligned.)
//
// Sources are read SCH at a time in two register chunks, the next chunk in
// flight while the current one is summed; the next unit's first chunk is
// loaded while the last chunk of this unit is summed, so the loads never
// drain between units.  Requires S to be a multiple of 2*SCH.
//
// Chunks whose scales are all below 2^-5 (a warp vote) are dequantized by one
// FMA a code (dequant_acc_i4 / dequant_acc_i8); others by the magic-number
// decode.  int4 with eight sources takes hop1_staged_kernel below instead; this
// kernel serves int8 (whose stages would leave one CTA an SM) and other source
// counts.
template <int BITS, int LOGB, int SCH>
__global__ void __launch_bounds__(kThreads, 2) hop1_kernel(const HopArgs a) {
  using G = Geo<LOGB, 4>;
  constexpr int WPB = G::WPB, GPC = kWarps / WPB;
  constexpr int QMAX = (1 << (BITS - 1)) - 1;
  constexpr int LCB = 32 * BITS / 8;                 // code bytes of a lane's 32 elements
  constexpr unsigned kAll = 0xffffffffu;
  struct Chunk {
    uint32_t w[SCH][BITS];  // 32 codes a source
    float s[SCH];
  };
  __shared__ float red[2][kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = warp / WPB, wsub = warp - gid * WPB;

  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * GPC + gid, (int64_t)gridDim.x * GPC, u, uend);
  if (u >= uend) return;
  const int64_t d0 = u / a.units_per_row;
  int64_t t = u - d0 * a.units_per_row;
  int32_t dn = (int32_t)(d0 / a.G), dl = (int32_t)(d0 - (int64_t)dn * a.G);
  const int64_t cstep = (a.in_rank_elems * BITS) >> 3;  // bytes between consecutive sources
  const int64_t fstep = a.in_rank_elems >> LOGB;        // scales between consecutive sources
  const int lane_e = 32 * lane;                         // the lane's first element in the slab
  // lane's code and scale pointers of unit (dn, dl, t), source 0 (node dn's first rank)
  auto bases = [&](int32_t n, int32_t l, int64_t tt, const uint8_t*& cp, const float*& sp) {
    const int64_t e0 = (int64_t)n * a.G * a.in_rank_elems + (int64_t)l * a.R + tt * G::U +
                       (int64_t)wsub * G::kWarpElems;
    cp = a.codes_in + ((e0 * BITS) >> 3) + lane * LCB;
    sp = a.scales_in + ((e0 + lane_e) >> LOGB);
  };
  auto load = [&](Chunk& ch, const uint8_t* cp, const float* sp, int s0) {
#pragma unroll
    for (int j = 0; j < SCH; ++j) {
      const uint4* src = reinterpret_cast<const uint4*>(cp + (int64_t)(s0 + j) * cstep);
#pragma unroll
      for (int h = 0; h < BITS / 4; ++h) {
        const uint4 v = __ldcs(src + h);
        ch.w[j][4 * h] = v.x;
        ch.w[j][4 * h + 1] = v.y;
        ch.w[j][4 * h + 2] = v.z;
        ch.w[j][4 * h + 3] = v.w;
      }
      ch.s[j] = __ldg(sp + (int64_t)(s0 + j) * fstep);
    }
  };
  float acc[4][8];
  const float2 one2 = make_float2(a.one, a.one);
  auto sum = [&](const Chunk& ch) {
    float smax = ch.s[0];
#pragma unroll
    for (int j = 1; j < SCH; ++j) smax = fmaxf(smax, ch.s[j]);
    const bool fma_path = __all_sync(kAll, smax < kFmaDequantMaxScale);
    if (fma_path) {
#pragma unroll
      for (int j = 0; j < SCH; ++j) {
        if constexpr (BITS == 4) {
          const I4Fma k = i4_fma_scale(ch.s[j]);
#pragma unroll
          for (int m = 0; m < 4; ++m) dequant_acc_i4(ch.w[j][m], k, one2, acc[m]);
        } else {
          const I8Fma k = i8_fma_scale(ch.s[j]);
#pragma unroll
          for (int m = 0; m < 4; ++m)
            dequant_acc_i8(make_uint2(ch.w[j][2 * m], ch.w[j][2 * m + 1]), k, one2, acc[m]);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < SCH; ++j) lane32_dequant_acc<BITS>(ch.w[j], ch.s[j], false, a.one, acc);
    }
  };

  const uint8_t* cp;
  const float* sp;
  bases(dn, dl, t, cp, sp);
  Chunk ca, cb;
  load(ca, cp, sp, 0);
  int parity = 0;
  for (; u < uend; ++u, parity ^= 1) {
    int64_t tn = t + 1;
    int32_t dnn = dn, dln = dl;
    if (tn == a.units_per_row) {
      tn = 0;
      if (++dln == a.G) {
        dln = 0;
        ++dnn;
      }
    }
    const bool more = u + 1 < uend;
    const uint8_t* cpn;
    const float* spn;
    bases(dnn, dln, tn, cpn, spn);
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[m][i] = 0.0f;
    for (int c = 0; c < a.S; c += 2 * SCH) {
      load(cb, cp, sp, c + SCH);
      sum(ca);
      if (c + 2 * SCH < a.S) load(ca, cp, sp, c + 2 * SCH);
      else if (more) load(ca, cpn, spn, 0);
      sum(cb);
    }

    // requantize the lane's 32 sums with its block's scale
    const Scale sc = lane32_block_scale<QMAX, LOGB, WPB>(acc, red, parity, warp, gid, lane);
    const int64_t e_warp = t * G::U + (int64_t)wsub * G::kWarpElems;
    const int64_t obase = ((int64_t)dn * a.G + dl) * a.R + e_warp;
    lane32_quantize_store<BITS>(acc, sc, a.codes_out + ((obase * BITS) >> 3) + lane * LCB);
    // R is a multiple of B, so obase mod B = e_warp mod B
    const int eb = (int)(e_warp & (G::B - 1)) + lane_e;
    if ((eb & (G::B - 1)) == 0) a.scales_out[(obase >> LOGB) + (eb >> LOGB)] = sc.s;

    t = tn;
    dn = dnn;
    dl = dln;
    cp = cpn;
    sp = spn;
  }
}

// Hop 1 for int4 with eight sources, the codes staged in shared memory.  Same
// lane layout and arithmetic as hop1_kernel (a lane owns 32 consecutive
// elements of its warp's 1024; sources summed in rank order), but the sources
// of the next unit are brought in by cp.async while this unit is summed:
//  - each lane copies its own 16-byte code vector of every source into a
//    slot it alone reads back, so the codes need no cross-lane sync;
//  - the warp slab's 1024/B scales of a source (at least one) are copied by
//    the first lanes and read by all, behind a __syncwarp;
//  - two stages a warp: unit u+1 is copied while unit u is summed, and a
//    stage is refilled only after every lane has read it (the __syncwarp at
//    the end of a unit).
// With no code registers held across units the kernel needs 80 registers, so
// three CTAs (24 warps) fit an SM next to their 3 x 66 KB of stages, and
// cp.async.wait_group is a hardware wait: on GB300 the long-scoreboard stalls
// per issue fall from about 1.2 to 0.07-0.25 against hop1_kernel and issue
// goes from 62-64% to 68-72% active, for 5% more instructions (the copies, the
// shared-memory reads and the start-up of four times as many CTAs); what is
// left is the decode's ALU work.  The first source of a unit is written
// straight into the accumulator (dequant_set_i4).
// acc[i] = RN(q_i s), i = 0..7: the first source of a sum written straight
// into the accumulator instead of added to a zero one.  The two differ only
// where RN(q s) is -0 (0 + -0 is +0), and a requantizing sum cannot tell: the
// block absmax takes |x| and a zero quantizes to code 0 either way.  Requires
// s < 2^-5, like dequant_acc_i4.
__device__ __forceinline__ void dequant_set_i4(uint32_t w, const I4Fma& k, float* acc) {
  const uint32_t x = w ^ 0x88888888u;
  const uint32_t ev = x & 0x0F0F0F0Fu, od = (x >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 dq = __ffma2_rn(i4_subnormal_pair(ev, od, j), k.sp, k.c);
    acc[2 * j] = dq.x;
    acc[2 * j + 1] = dq.y;
  }
}

constexpr int kStagedSources = 8;
constexpr int kHop1StagedRounds = 4;  // CTA rounds (grid_for): 0.576 / 0.589 / 0.593 of the
                                      // copy peak for 1 / 2 / 4 on the two-hop bucket

template <int LOGB>
__host__ __device__ constexpr int hop1_scale_slot() {  // a warp's scales of one source, padded
  return LOGB <= 8 ? 16 << (8 - LOGB) : 16;
}
template <int LOGB>
__host__ __device__ constexpr int hop1_stage_bytes() {  // one warp's stage
  return kStagedSources * (32 * 16 + hop1_scale_slot<LOGB>());
}

template <int LOGB>
__global__ void __launch_bounds__(kThreads, 3) hop1_staged_kernel(const HopArgs a) {
  constexpr int BITS = 4, S = kStagedSources;
  using G = Geo<LOGB, 4>;
  constexpr int WPB = G::WPB, GPC = kWarps / WPB;
  constexpr int QMAX = 7;
  constexpr int LCB = 16;                              // a lane's code bytes of one source
  constexpr int SRC = 32 * LCB + hop1_scale_slot<LOGB>();  // one source in a stage
  constexpr int STAGE = hop1_stage_bytes<LOGB>();
  constexpr int NSC = LOGB <= 10 ? (1024 >> LOGB) : 1;  // scales of a warp slab (at least one)
  constexpr unsigned kAll = 0xffffffffu;
  extern __shared__ __align__(128) uint8_t stages[];
  __shared__ float red[2][kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = warp / WPB, wsub = warp - gid * WPB;

  int64_t u, uend;
  unit_range(a.total_units, (int64_t)blockIdx.x * GPC + gid, (int64_t)gridDim.x * GPC, u, uend);
  if (u >= uend) return;
  uint8_t* const wstage = stages + (size_t)warp * 2 * STAGE;
  const int64_t d0 = u / a.units_per_row;
  int64_t t = u - d0 * a.units_per_row;
  int32_t dn = (int32_t)(d0 / a.G), dl = (int32_t)(d0 - (int64_t)dn * a.G);
  const int64_t cstep = (a.in_rank_elems * BITS) >> 3;  // bytes between consecutive sources
  const int64_t fstep = a.in_rank_elems >> LOGB;        // scales between consecutive sources
  const int lane_e = 32 * lane;
  const int my_sc = LOGB <= 10 ? (lane_e >> LOGB) : 0;  // the lane's scale in its slab's
  // copies of unit (n, l, tt), all S sources, into stage `st`
  auto issue = [&](int st, int32_t n, int32_t l, int64_t tt) {
    const int64_t e0 = (int64_t)n * a.G * a.in_rank_elems + (int64_t)l * a.R + tt * G::U +
                       (int64_t)wsub * G::kWarpElems;
    const uint8_t* cw = a.codes_in + ((e0 * BITS) >> 3) + lane * LCB;
    const float* sw = a.scales_in + (e0 >> LOGB);  // 16-byte aligned: e0 is a multiple of 1024
    uint8_t* dst = wstage + st * STAGE;
#pragma unroll
    for (int j = 0; j < S; ++j) {
      cp_async16(dst + j * SRC + lane * LCB, cw + (int64_t)j * cstep);
      uint8_t* sdst = dst + j * SRC + 32 * LCB;
      const float* ssrc = sw + (int64_t)j * fstep;
      if constexpr (NSC >= 4) {
        if (lane < NSC / 4) cp_async16(sdst + 16 * lane, ssrc + 4 * lane);
      } else if (lane == 0) {
        if constexpr (NSC == 2)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(sdst)), "l"(ssrc)
                       : "memory");
        else
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(sdst)), "l"(ssrc)
                       : "memory");
      }
    }
  };
  auto next_unit = [&](int64_t& tt, int32_t& n, int32_t& l) {
    if (++tt == a.units_per_row) {
      tt = 0;
      if (++l == a.G) {
        l = 0;
        ++n;
      }
    }
  };

  issue(0, dn, dl, t);
  cp_async_commit();
  int64_t t1 = t;  // (t1, dn1, dl1): the unit after the current one
  int32_t dn1 = dn, dl1 = dl;
  next_unit(t1, dn1, dl1);
  float acc[4][8];
  const float2 one2 = make_float2(a.one, a.one);
  for (int64_t q = 0; u < uend; ++u, ++q) {
    const int st = (int)(q & 1), parity = st;
    if (u + 1 < uend) issue(st ^ 1, dn1, dl1, t1);  // read during the unit before this one
    cp_async_commit();
    cp_async_wait<1>();  // this unit's copies have landed
    __syncwarp();        // and so have the other lanes' scale copies
    const uint8_t* src = wstage + st * STAGE;
    float sc[S];
#pragma unroll
    for (int j = 0; j < S; ++j) sc[j] = reinterpret_cast<const float*>(src + j * SRC + 32 * LCB)[my_sc];
    float smax = sc[0];
#pragma unroll
    for (int j = 1; j < S; ++j) smax = fmaxf(smax, sc[j]);
    if (__all_sync(kAll, smax < kFmaDequantMaxScale)) {
#pragma unroll
      for (int j = 0; j < S; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + j * SRC + lane * LCB);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const I4Fma k = i4_fma_scale(sc[j]);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if (j == 0) dequant_set_i4(w[m], k, acc[m]);
          else dequant_acc_i4(w[m], k, one2, acc[m]);
        }
      }
    } else {
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[m][i] = 0.0f;
#pragma unroll
      for (int j = 0; j < S; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + j * SRC + lane * LCB);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        lane32_dequant_acc<BITS>(w, sc[j], false, a.one, acc);
      }
    }
    // requantize the lane's 32 sums with its block's scale
    const Scale sco = lane32_block_scale<QMAX, LOGB, WPB>(acc, red, parity, warp, gid, lane);
    const int64_t e_warp = t * G::U + (int64_t)wsub * G::kWarpElems;
    const int64_t obase = ((int64_t)dn * a.G + dl) * a.R + e_warp;
    lane32_quantize_store<BITS>(acc, sco, a.codes_out + ((obase * BITS) >> 3) + lane * LCB);
    const int eb = (int)(e_warp & (G::B - 1)) + lane_e;
    if ((eb & (G::B - 1)) == 0) a.scales_out[(obase >> LOGB) + (eb >> LOGB)] = sco.s;
    __syncwarp();  // every lane has read its scales before the stage is refilled
    next_unit(t, dn, dl);
    next_unit(t1, dn1, dl1);
  }
  cp_async_wait<0>();  // no copy outlives the warp
}

template <int BITS, int MODE>
cudaError_t run_hop(const HopArgs& a0, int block, cudaStream_t st) {
  return dispatch_logb(block, [&](auto lb) -> cudaError_t {
    constexpr int LOGB = decltype(lb)::value;
    using C = HopCfg<BITS, MODE, LOGB>;
    HopArgs a = a0;
    a.units_per_row = (a.R + C::U - 1) / C::U;
    a.total_units = (int64_t)a.N * a.G * a.units_per_row;
    const int64_t groups = kWarps / C::WPB;
    const int64_t ctas = (a.total_units + groups - 1) / groups;
    const bool tiled = a.R % C::U == 0;
    // four sources a chunk pays off for int4 final hops with many sources
    constexpr bool kWideChunk = MODE != kRequant && BITS == 4;
    const bool wide_chunk = kWideChunk && a.S > 2;
    auto launch_tiled = [&](auto w, auto sch) {
      constexpr bool W = decltype(w)::value;
      constexpr int S = decltype(sch)::value;
      const void* k = reinterpret_cast<const void*>(&hop_tiled_kernel<BITS, MODE, LOGB, W, S>);
      hop_tiled_kernel<BITS, MODE, LOGB, W, S><<<grid_for(k, ctas), kThreads, 0, st>>>(a);
    };
    if constexpr (MODE == kRequant) {
      if (tiled && a.S % 4 == 0) {  // sources in pairs of chunks of 2 or 4
        auto launch1 = [&](auto sch) {
          constexpr int S = decltype(sch)::value;
          const void* k = reinterpret_cast<const void*>(&hop1_kernel<BITS, LOGB, S>);
          hop1_kernel<BITS, LOGB, S><<<grid_for(k, ctas), kThreads, 0, st>>>(a);
        };
        if constexpr (BITS == 4) {
          if (a.S == kStagedSources) {
            constexpr size_t smem = (size_t)kWarps * 2 * hop1_stage_bytes<LOGB>();
            const void* k = reinterpret_cast<const void*>(&hop1_staged_kernel<LOGB>);
            const cudaError_t e = smem_opt_in(k, smem);
            if (e != cudaSuccess) return e;
            hop1_staged_kernel<LOGB>
                <<<grid_for(k, ctas, smem, kHop1StagedRounds), kThreads, smem, st>>>(a);
            return cudaGetLastError();
          }
        }
        if (BITS == 4 && a.S % 8 == 0) launch1(std::integral_constant<int, BITS == 4 ? 4 : 2>{});
        else launch1(std::integral_constant<int, 2>{});
        return cudaGetLastError();
      }
    }
    using Two = std::integral_constant<int, 2>;
    using Four = std::integral_constant<int, kWideChunk ? 4 : 2>;
    if (tiled && (MODE == kRequant || a.wide)) {
      using W = std::integral_constant<bool, MODE != kRequant>;
      if (wide_chunk) launch_tiled(W{}, Four{});
      else launch_tiled(W{}, Two{});
    } else if constexpr (MODE == kFinalAdamQwz) {
      if (!tiled) return cudaErrorNotSupported;
      using W = std::integral_constant<bool, false>;
      if (wide_chunk) launch_tiled(W{}, Four{});
      else launch_tiled(W{}, Two{});
    } else {  // ragged rows, or fp32 arrays only 16-byte aligned
      const void* k = reinterpret_cast<const void*>(&hop_kernel<BITS, MODE, LOGB>);
      hop_kernel<BITS, MODE, LOGB><<<grid_for(k, ctas), kThreads, 0, st>>>(a);
    }
    return cudaGetLastError();
  });
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
  a.codes_out = static_cast<uint8_t*>(h.codes_out);
  a.scales_out = h.scales_out;
  a.grad_out = h.grad_out;
  a.inv_nd = h.inv_nd;
  a.ac = AdamConsts{h.ac.lr,   h.ac.beta1, h.ac.beta2, h.ac.eps, h.ac.omb1, h.ac.omb2,
                    h.ac.bc1,  h.ac.bc2,   h.ac.rbc1,  h.ac.rbc2, 1.0f};
  a.master = h.master;
  a.m = h.m;
  a.v = h.v;
  a.param = h.param;
  a.qwz_codes = static_cast<uint8_t*>(h.qwz_codes);
  a.qwz_scales = h.qwz_scales;
  a.one = 1.0f;
  a.wide = (!a.grad_out || aligned32(a.grad_out)) &&
           (!h.adam || (aligned32(a.master) && aligned32(a.m) && aligned32(a.v)));
  const int b = h.block;
  if (!final_hop) return h.bits == 8 ? run_hop<8, kRequant>(a, b, st) : run_hop<4, kRequant>(a, b, st);
  if (h.adam && h.qwz_codes)
    return h.bits == 8 ? run_hop<8, kFinalAdamQwz>(a, b, st) : run_hop<4, kFinalAdamQwz>(a, b, st);
  if (h.adam) return h.bits == 8 ? run_hop<8, kFinalAdam>(a, b, st) : run_hop<4, kFinalAdam>(a, b, st);
  return h.bits == 8 ? run_hop<8, kFinal>(a, b, st) : run_hop<4, kFinal>(a, b, st);
}

}  // namespace zpp
