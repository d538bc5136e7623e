/*
 * zpp_oracle.c -- plain, slow, single-threaded CPU oracle of the ZeRO++
 * data-parallel codec path (qwZ, qgZ two-hop reduce, sharded mixed-precision
 * Adam).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call it: only the
 * tests, the entry point's smoke check and the bench's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Pins: each function here is checked by the test suite against something
 * other than itself (brute force, closed forms, exact sums, the pages'
 * numbers).  The two-hop chain with a real int4/int8 codec is parity
 * unpinned beyond an error bound: its pieces (the block codec, the summation
 * order, the slice placement) are pinned one by one, and the composed values
 * only by the sum of the half-scales they went through.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * Every floating-point operation below is a separately rounded IEEE fp32
 * operation (no FMA contraction), in the order written.
 *
 * Sources (page title, then section):
 *  [P1] "Quantized LLM Training at Scale with ZeRO++", section "The Three
 *       Pillars of ZeRO++": 1 (QWZ, block quantization, 8-bit weights),
 *       3 (QGZ: one-shot quantization, two-hop all-to-all with reduction,
 *       tensor slice reordering).
 *  [P2] "ZeRO-1/2/3 (Zero Redundancy Optimizer)", section "Stage 1" steps
 *       4-6 (reduce-scatter, fp32 update, write back 16-bit params) and the
 *       ZeRO++ note (qwZ int8/int4).
 *  [P3] "ZeRO Stage 2: Gradient Partitioning": reduce-scatter averages, so
 *       GPU i ends with the averaged gradient of shard i; the optimizer step
 *       converts the gradient shard to fp32 and updates fp32 master and state.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - qmax = 2^(bits-1) - 1 (127 for int8, 7 for int4; code -8 unused).
 *  - s = absmax / qmax (fp32 divide); q = clamp(rint(x / s), -qmax, qmax),
 *    rint = round half to even, fp32 divide per element.
 *  - s == 0 (all-zero block, or a scale that underflows) -> every code is 0.
 *  - A tail block covers only the remaining elements; its scale is taken over
 *    them; no padding codes are written.
 *  - int4 codes are two's-complement nibbles, element 2i in the low nibble of
 *    byte i.
 *  - Dequant: (float)q * s, one rounded multiply; qwZ output bf16 = round to
 *    nearest even of that.
 *  - Hop sums: acc = 0; acc = acc + deq(source) for sources in rank order.
 *  - Slice reorder: slice j = n'G + l' is stored at position p = l'N + n'.
 *  - Final hop output: g = sum * (1.0f / N_d).  When N == 1, hop 1 is final.
 *  - Adam: Kingma & Ba with bias correction, eps outside the square root, no
 *    weight decay.  bc = 1 - beta^t with beta^t by repeated squaring in
 *    double, rounded to float once; (1 - beta) rounded from double.
 *  - Master -> 16-bit write-back: bf16 round to nearest even.
 *  - bits == 32 is an oracle-only identity codec (fp32 payload, no scale) used
 *    to pin the placement of the reorder and the two hops with exact sums.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1

/* ---- bf16 <-> fp32 (definitions) -------------------------------------- */

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round to nearest, ties to even, keeping the upper 16 bits of the fp32 word. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN: keep it a quiet NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* ---- sizes ------------------------------------------------------------ */

int64_t orc_codes_bytes(int64_t n, int bits)
{
    if (bits == 32) return 4 * n;
    return (n * bits + 7) / 8;
}

int64_t orc_num_blocks(int64_t n, int64_t block)
{
    return (n + block - 1) / block;
}

static int valid_bits(int bits) { return bits == 4 || bits == 8 || bits == 32; }

/* ---- O1: quantize one block ------------------------------------------- */

static int qmax_of(int bits) { return (1 << (bits - 1)) - 1; }

/* Store code q of element `pos` of a code stream. */
static void put_code(void* codes, int64_t pos, int bits, int q, float xf)
{
    if (bits == 8) {
        ((int8_t*)codes)[pos] = (int8_t)q;
    } else if (bits == 4) {
        uint8_t* b = (uint8_t*)codes + pos / 2;
        uint8_t nib = (uint8_t)(q & 0xf);
        if (pos % 2 == 0) *b = (uint8_t)((*b & 0xf0u) | nib);
        else              *b = (uint8_t)((*b & 0x0fu) | (uint8_t)(nib << 4));
    } else { /* identity codec */
        ((float*)codes)[pos] = xf;
    }
}

static int get_code(const void* codes, int64_t pos, int bits)
{
    if (bits == 8) return ((const int8_t*)codes)[pos];
    uint8_t b = ((const uint8_t*)codes)[pos / 2];
    int nib = (pos % 2 == 0) ? (b & 0xf) : (b >> 4);
    return nib >= 8 ? nib - 16 : nib; /* two's complement nibble */
}

/* O2: dequantized fp32 value of element `pos`. */
static float deq(const void* codes, const float* scales, int64_t pos,
                 int64_t block, int bits)
{
    if (bits == 32) return ((const float*)codes)[pos];
    float s = scales[pos / block];
    float q = (float)get_code(codes, pos, bits);
    return q * s;
}

/* Quantize n fp32 values x[0..n) as one block.  Codes go to element
 * positions code_pos .. code_pos+n of `codes`; the scale to *scale. */
static void quant_one_block(const float* x, int64_t n, int bits,
                            void* codes, int64_t code_pos, float* scale)
{
    if (bits == 32) {
        for (int64_t i = 0; i < n; ++i) put_code(codes, code_pos + i, 32, 0, x[i]);
        if (scale) *scale = 1.0f;
        return;
    }
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    const float qmax = (float)qmax_of(bits);
    const float s = amax / qmax;
    *scale = s;
    for (int64_t i = 0; i < n; ++i) {
        int q = 0;
        if (s != 0.0f) {
            float y = x[i] / s;
            float r = rintf(y);
            if (r > qmax) r = qmax;
            if (r < -qmax) r = -qmax;
            q = (int)r;
        }
        put_code(codes, code_pos + i, bits, q, 0.0f);
    }
}

/* Block-quantize a run of n fp32 values in blocks of `block` (tail allowed).
 * Used for qwZ, for the qgZ one-shot quantization, for the hop-1 requant and,
 * with block >= n, for global quantization. */
int orc_block_quant(const float* x, int64_t n, int64_t block, int bits,
                    void* codes, float* scales)
{
    if (n < 0 || block <= 0 || !valid_bits(bits)) return ORC_EINVAL;
    int64_t nb = orc_num_blocks(n, block);
    for (int64_t b = 0; b < nb; ++b) {
        int64_t lo = b * block;
        int64_t len = (n - lo < block) ? (n - lo) : block;
        quant_one_block(x + lo, len, bits, codes, lo, scales ? scales + b : NULL);
    }
    return ORC_OK;
}

int orc_block_dequant(const void* codes, const float* scales, int64_t n,
                      int64_t block, int bits, float* y)
{
    if (n < 0 || block <= 0 || !valid_bits(bits)) return ORC_EINVAL;
    for (int64_t i = 0; i < n; ++i) y[i] = deq(codes, scales, i, block, bits);
    return ORC_OK;
}

/* ---- a1/a2: qwZ --------------------------------------------------------- */

/* x_bf16 [nranks][shard] -> codes [nranks][codes_bytes(shard)],
 * scales [nranks][num_blocks(shard)]; blocks restart at every shard. */
int orc_qwz_quant(const uint16_t* x, int64_t nranks, int64_t shard, int64_t block,
                  int bits, void* codes, float* scales)
{
    if (nranks < 0 || shard < 0 || block <= 0 || (bits != 4 && bits != 8))
        return ORC_EINVAL;
    if (bits == 4 && shard % 2) return ORC_EINVAL;
    float* tmp = (float*)malloc((size_t)(shard > 0 ? shard : 1) * sizeof(float));
    if (!tmp) return ORC_EINVAL;
    int64_t cb = orc_codes_bytes(shard, bits), nb = orc_num_blocks(shard, block);
    for (int64_t r = 0; r < nranks; ++r) {
        for (int64_t i = 0; i < shard; ++i) tmp[i] = bf16_to_f32(x[r * shard + i]);
        orc_block_quant(tmp, shard, block, bits, (uint8_t*)codes + r * cb, scales + r * nb);
    }
    free(tmp);
    return ORC_OK;
}

/* All-gather receiver: codes/scales of every shard -> the full bf16 tensor. */
int orc_qwz_dequant(const void* codes, const float* scales, int64_t nranks,
                    int64_t shard, int64_t block, int bits, uint16_t* y)
{
    if (nranks < 0 || shard < 0 || block <= 0 || (bits != 4 && bits != 8))
        return ORC_EINVAL;
    if (bits == 4 && shard % 2) return ORC_EINVAL;
    int64_t cb = orc_codes_bytes(shard, bits), nb = orc_num_blocks(shard, block);
    for (int64_t r = 0; r < nranks; ++r)
        for (int64_t i = 0; i < shard; ++i)
            y[r * shard + i] = orc_f32_to_bf16(
                deq((const uint8_t*)codes + r * cb, scales + r * nb, i, block, bits));
    return ORC_OK;
}

/* ---- a3: slice reorder + one-shot quantization -------------------------- */

/* perm[p] = source slice j stored at message position p.
 * Slice j = n*G + l belongs to rank (node n, local l); it goes to p = l*N + n,
 * so that local peer l receives one contiguous chunk of N slots in hop 1 and
 * node n receives slot n in hop 2. */
int orc_qgz_slice_perm(int N, int G, int32_t* perm)
{
    if (N <= 0 || G <= 0) return ORC_EINVAL;
    for (int n = 0; n < N; ++n)
        for (int l = 0; l < G; ++l)
            perm[l * N + n] = n * G + l;
    return ORC_OK;
}

static int qgz_check(int N, int G, int64_t bucket, int64_t block, int bits)
{
    if (N <= 0 || G <= 0 || bucket < 0 || block <= 0 || !valid_bits(bits))
        return ORC_EINVAL;
    if (bucket % ((int64_t)N * G * block)) return ORC_EINVAL;
    return ORC_OK;
}

/* Shared body: source element (r, i) read through either a bf16 or an fp32
 * array (exactly one of g16 / g32 is non-NULL). */
static int reorder_quant_src(const uint16_t* g16, const float* g32, int N, int G, int64_t bucket,
                             int64_t block, int bits, const int32_t* perm, void* codes,
                             float* scales)
{
    if (qgz_check(N, G, bucket, block, bits)) return ORC_EINVAL;
    const int64_t Nd = (int64_t)N * G, L = bucket / Nd;
    const int64_t cb = orc_codes_bytes(bucket, bits), nb = bucket / block;
    float* tmp = (float*)malloc((size_t)(L > 0 ? L : 1) * sizeof(float));
    if (!tmp) return ORC_EINVAL;
    for (int64_t r = 0; r < Nd; ++r) {
        uint8_t* rc = (uint8_t*)codes + r * cb;
        float* rs = scales ? scales + r * nb : NULL;
        for (int64_t p = 0; p < Nd; ++p) {
            int64_t j = perm[p];
            for (int64_t i = 0; i < L; ++i) {
                const int64_t k = r * bucket + j * L + i;
                tmp[i] = g16 ? bf16_to_f32(g16[k]) : g32[k];
            }
            /* blocks of slice j restart at the slice start (L % block == 0) */
            for (int64_t b = 0; b < L / block; ++b)
                quant_one_block(tmp + b * block, block, bits, rc, p * L + b * block,
                                rs ? rs + (p * L + b * block) / block : NULL);
        }
    }
    free(tmp);
    return ORC_OK;
}

/* Same as orc_qgz_reorder_quant with an explicit permutation (perm[p] = j). */
int orc_qgz_reorder_quant_perm(const uint16_t* grads, int N, int G, int64_t bucket,
                               int64_t block, int bits, const int32_t* perm,
                               void* codes, float* scales)
{
    return reorder_quant_src(grads, NULL, N, G, bucket, block, bits, perm, codes, scales);
}

int orc_qgz_reorder_quant(const uint16_t* grads, int N, int G, int64_t bucket,
                          int64_t block, int bits, void* codes, float* scales)
{
    if (N <= 0 || G <= 0) return ORC_EINVAL;
    int32_t* perm = (int32_t*)malloc((size_t)N * G * sizeof(int32_t));
    if (!perm) return ORC_EINVAL;
    orc_qgz_slice_perm(N, G, perm);
    int rc = orc_qgz_reorder_quant_perm(grads, N, G, bucket, block, bits, perm,
                                        codes, scales);
    free(perm);
    return rc;
}

/* ---- a4: hop 1, intra-node dequant -> sum -> requant --------------------- */

/* Destination rank d = n*G + l receives chunk l (N slots of L elements) of
 * each local peer n*G + g, g = 0..G-1, and sums them in that order.
 * N > 1: the sum is requantized (same block and bits) into
 *        codes_out [N_d][codes_bytes(N*L)], scales_out [N_d][N*L/block].
 * N == 1: hop 1 is the final hop; grad_out[d*L + i] = sum * (1/N_d). */
int orc_qgz_hop1(const void* codes_in, const float* scales_in, int N, int G,
                 int64_t bucket, int64_t block, int bits, void* codes_out,
                 float* scales_out, float* grad_out)
{
    if (qgz_check(N, G, bucket, block, bits)) return ORC_EINVAL;
    const int64_t Nd = (int64_t)N * G, L = bucket / Nd, NL = (int64_t)N * L;
    const int64_t cb_in = orc_codes_bytes(bucket, bits), nb_in = bucket / block;
    const int64_t cb_out = orc_codes_bytes(NL, bits), nb_out = NL / block;
    const float inv_nd = 1.0f / (float)Nd;
    if (N > 1 && !codes_out) return ORC_EINVAL;
    if (N == 1 && !grad_out) return ORC_EINVAL;
    float* acc = (float*)malloc((size_t)(NL > 0 ? NL : 1) * sizeof(float));
    if (!acc) return ORC_EINVAL;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t l = 0; l < G; ++l) {
            const int64_t d = n * G + l;
            for (int64_t e = 0; e < NL; ++e) acc[e] = 0.0f;
            for (int64_t g = 0; g < G; ++g) {
                const int64_t src = n * G + g;
                const uint8_t* c = (const uint8_t*)codes_in + src * cb_in;
                const float* s = scales_in ? scales_in + src * nb_in : NULL;
                for (int64_t e = 0; e < NL; ++e)
                    acc[e] = acc[e] + deq(c, s, l * NL + e, block, bits);
            }
            if (N == 1) {
                for (int64_t e = 0; e < L; ++e) grad_out[d * L + e] = acc[e] * inv_nd;
            } else {
                orc_block_quant(acc, NL, block, bits, (uint8_t*)codes_out + d * cb_out,
                                scales_out ? scales_out + d * nb_out : NULL);
            }
        }
    }
    free(acc);
    return ORC_OK;
}

/* ---- a5: hop 2, inter-node dequant -> sum -> average ---------------------- */

/* Destination rank d = n*G + l receives slot n of rank n'*G + l for
 * n' = 0..N-1 (hop-1 messages), sums in that order and scales by 1/N_d:
 * grad_out[d*L + i] is rank d's averaged gradient slice. */
int orc_qgz_hop2(const void* codes_in, const float* scales_in, int N, int G,
                 int64_t bucket, int64_t block, int bits, float* grad_out)
{
    if (qgz_check(N, G, bucket, block, bits) || N < 2 || !grad_out) return ORC_EINVAL;
    const int64_t Nd = (int64_t)N * G, L = bucket / Nd, NL = (int64_t)N * L;
    const int64_t cb_in = orc_codes_bytes(NL, bits), nb_in = NL / block;
    const float inv_nd = 1.0f / (float)Nd;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t l = 0; l < G; ++l) {
            const int64_t d = n * G + l;
            for (int64_t i = 0; i < L; ++i) {
                float acc = 0.0f;
                for (int64_t np = 0; np < N; ++np) {
                    const int64_t src = np * G + l;
                    acc = acc + deq((const uint8_t*)codes_in + src * cb_in,
                                    scales_in ? scales_in + src * nb_in : NULL,
                                    n * L + i, block, bits);
                }
                grad_out[d * L + i] = acc * inv_nd;
            }
        }
    }
    return ORC_OK;
}

/* ---- a6: sharded mixed-precision Adam ----------------------------------- */

static double pow_by_squaring(double b, int64_t t)
{
    double r = 1.0;
    while (t > 0) {
        if (t & 1) r = r * b;
        b = b * b;
        t >>= 1;
    }
    return r;
}

/* Bias corrections and (1 - beta) as the Adam step uses them. */
void orc_adam_consts(float beta1, float beta2, int32_t t, float* bc1, float* bc2,
                     float* omb1, float* omb2)
{
    *bc1 = (float)(1.0 - pow_by_squaring((double)beta1, t));
    *bc2 = (float)(1.0 - pow_by_squaring((double)beta2, t));
    *omb1 = (float)(1.0 - (double)beta1);
    *omb2 = (float)(1.0 - (double)beta2);
}

/* One Adam step on n owned parameters with fp32 gradient g:
 *   m <- b1*m + (1-b1)*g ;  v <- b2*v + (1-b2)*(g*g)
 *   p <- p - (lr * (m/bc1)) / (sqrt(v/bc2) + eps)
 *   param_bf16 <- bf16_rne(p)                                              */
int orc_adam_step(const float* g, int64_t n, float lr, float beta1, float beta2,
                  float eps, int32_t t, float* master, float* m, float* v,
                  uint16_t* param)
{
    if (n < 0 || t < 1) return ORC_EINVAL;
    float bc1, bc2, omb1, omb2;
    orc_adam_consts(beta1, beta2, t, &bc1, &bc2, &omb1, &omb2);
    for (int64_t i = 0; i < n; ++i) {
        const float gi = g[i];
        const float mi = beta1 * m[i] + omb1 * gi;
        const float vi = beta2 * v[i] + omb2 * (gi * gi);
        const float mhat = mi / bc1;
        const float vhat = vi / bc2;
        const float denom = sqrtf(vhat) + eps;
        const float p = master[i] - (lr * mhat) / denom;
        m[i] = mi;
        v[i] = vi;
        master[i] = p;
        if (param) param[i] = orc_f32_to_bf16(p);
    }
    return ORC_OK;
}

/* ---- next row: gradient accumulation ---------------------------------------------
 *
 * ("ZeRO Stage 2: Gradient Partitioning", gradient accumulation: the partial
 * gradients of several micro-batches are accumulated locally and the
 * reduce-scatter fires once, when the accumulation is complete; the optimizer
 * side holds them in fp32.)  Micro-batch gradients arrive in bf16 and are
 * summed in fp32 in arrival order: acc = g_1; acc = acc + g_k.  The one-shot
 * quantization of the accumulated bucket reads acc + g_last (one more fp32
 * add) and is otherwise orc_qgz_reorder_quant on fp32 values. */

int orc_grad_accumulate(const uint16_t* g, float* acc, int64_t n, int first)
{
    if (n < 0) return ORC_EINVAL;
    for (int64_t i = 0; i < n; ++i)
        acc[i] = first ? bf16_to_f32(g[i]) : acc[i] + bf16_to_f32(g[i]);
    return ORC_OK;
}

int orc_qgz_reorder_quant_f32(const float* grads, int N, int G, int64_t bucket,
                              int64_t block, int bits, void* codes, float* scales)
{
    if (N <= 0 || G <= 0) return ORC_EINVAL;
    int32_t* perm = (int32_t*)malloc((size_t)N * G * sizeof(int32_t));
    if (!perm) return ORC_EINVAL;
    orc_qgz_slice_perm(N, G, perm);
    int rc = reorder_quant_src(NULL, grads, N, G, bucket, block, bits, perm, codes, scales);
    free(perm);
    return rc;
}

/* ---- hpZ: secondary partition and the node-local backward gather --------
 * [P1] section 2 (HPZ): each node holds a secondary replica of the model
 * partitions, so the backward weight gather reads only the node's own GPUs
 * and its cross-node volume drops to zero.
 * Reading: the secondary partition of rank (node n, local l) is slice l of
 * the G-way split of the weights = the N consecutive primary shards
 * l*N .. l*N + N - 1, kept in the form the forward all-gather delivered them
 * (qwZ codes + scales; bf16 values when bits == 16).  The backward gather of
 * node n concatenates the G secondary slices in local rank order
 * l = 0..G-1 and dequantizes each shard as the forward receiver does. */

int orc_hpz_gather(int G, int N, int64_t shard, int64_t block, int bits,
                   const void* const* sec_codes, const float* const* sec_scales, uint16_t* y)
{
    if (G <= 0 || N <= 0 || shard < 0 || block <= 0) return ORC_EINVAL;
    if (bits != 16 && bits != 8 && bits != 4) return ORC_EINVAL;
    for (int l = 0; l < G; ++l) {
        uint16_t* yl = y + (int64_t)l * N * shard;
        if (bits == 16) {
            const uint16_t* src = (const uint16_t*)sec_codes[l];
            for (int64_t i = 0; i < (int64_t)N * shard; ++i) yl[i] = src[i];
        } else {
            int rc = orc_qwz_dequant(sec_codes[l], sec_scales[l], N, shard, block, bits, yl);
            if (rc != ORC_OK) return rc;
        }
    }
    return ORC_OK;
}

/* Bytes one rank holds for its secondary partition: N shards' codes and
 * scales (bits 4/8), or N shards of bf16 (bits 16). */
int64_t orc_hpz_secondary_bytes(int N, int64_t shard, int64_t block, int bits)
{
    if (N <= 0 || shard < 0 || block <= 0) return -1;
    if (bits == 16) return (int64_t)N * 2 * shard;
    if (bits != 8 && bits != 4) return -1;
    return (int64_t)N * (orc_codes_bytes(shard, bits) + 4 * orc_num_blocks(shard, block));
}

/* ---- ring reduce-scatter with a requantization at every hop (comparator) --
 * [P1] section 3 (QGZ), challenge "sequential quantization overhead": in a
 * ring reduce-scatter of quantized gradients every GPU on the ring
 * dequantizes, adds and requantizes, N sequential quantizations where qgZ
 * does one.  This is the comparator for that precision loss.
 * Reading: ring r -> r + 1 (mod N_d); chunk c = elements [c*L, (c+1)*L) of a
 * rank's bucket, L = bucket / N_d; at step s = 0..N_d-1 rank r works on chunk
 * c = (r - 1 - s) mod N_d:
 *   s = 0            msg_r = Q(x_r[c])
 *   0 < s < N_d - 1  msg_r = Q(D(msg_{r-1}) + x_r[c])
 *   s = N_d - 1      g_r   = (D(msg_{r-1}) + x_r[c]) * (1.0f / N_d),  c = r
 * so chunk c is summed in the ring order c+1, c+2, ..., c and rank r ends with
 * the average of its own chunk, as the reduce-scatter of qgZ delivers it.
 * Q is the block quantization (blocks restart at the chunk start), D its
 * dequantization, + one rounded fp32 add.  With N_d == 1 the only step is the
 * last one and g = x. */

static int64_t ring_chunk(int r, int s, int nd)
{
    return (((int64_t)r - 1 - s) % nd + nd) % nd;
}

int orc_ring_rs_step(int step, int nd, int64_t bucket, int64_t block, int bits,
                     const uint16_t* x, const void* codes_in, const float* scales_in,
                     void* codes_out, float* scales_out, float* grad_out)
{
    if (nd <= 0 || step < 0 || step >= nd || bucket < 0 || block <= 0 || !valid_bits(bits))
        return ORC_EINVAL;
    if (bucket % ((int64_t)nd * block)) return ORC_EINVAL;
    const int64_t L = bucket / nd;
    const int64_t cb = orc_codes_bytes(L, bits), nb = orc_num_blocks(L, block);
    float* v = (float*)malloc((size_t)(L > 0 ? L : 1) * sizeof(float));
    if (!v) return ORC_EINVAL;
    const int last = (step == nd - 1);
    for (int r = 0; r < nd; ++r) {
        const int64_t c = ring_chunk(r, step, nd);
        const uint16_t* xr = x + (int64_t)r * bucket + c * L;
        const int prev = (r - 1 + nd) % nd;
        for (int64_t i = 0; i < L; ++i) {
            float own = bf16_to_f32(xr[i]);
            if (step == 0) {
                v[i] = own;
            } else {
                float d = deq((const uint8_t*)codes_in + prev * cb, scales_in + prev * nb, i,
                              block, bits);
                v[i] = d + own;
            }
        }
        if (last) {
            const float inv = 1.0f / (float)nd;
            for (int64_t i = 0; i < L; ++i) grad_out[(int64_t)r * L + i] = v[i] * inv;
        } else {
            orc_block_quant(v, L, block, bits, (uint8_t*)codes_out + r * cb, scales_out + r * nb);
        }
    }
    free(v);
    return ORC_OK;
}

/* The whole ring: N_d steps, messages passed between two buffers. */
int orc_ring_reduce_scatter(int nd, int64_t bucket, int64_t block, int bits,
                            const uint16_t* x, float* grad_out)
{
    if (nd <= 0 || bucket < 0 || block <= 0 || !valid_bits(bits)) return ORC_EINVAL;
    if (bucket % ((int64_t)nd * block)) return ORC_EINVAL;
    const int64_t L = bucket / nd;
    const int64_t cb = orc_codes_bytes(L, bits), nb = orc_num_blocks(L, block);
    uint8_t* c[2];
    float* s[2];
    for (int k = 0; k < 2; ++k) {
        c[k] = (uint8_t*)calloc((size_t)(nd * cb > 0 ? nd * cb : 1), 1);
        s[k] = (float*)calloc((size_t)(nd * nb > 0 ? nd * nb : 1), sizeof(float));
    }
    int rc = ORC_OK;
    for (int step = 0; step < nd && rc == ORC_OK; ++step)
        rc = orc_ring_rs_step(step, nd, bucket, block, bits, x, c[(step + 1) & 1],
                              s[(step + 1) & 1], c[step & 1], s[step & 1], grad_out);
    for (int k = 0; k < 2; ++k) {
        free(c[k]);
        free(s[k]);
    }
    return rc;
}
