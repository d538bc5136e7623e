/*
 * _gen.c -- host fast path of the counter-based synthetic generator.
 *
 * Computes exactly what the tensor path of synth/__init__.py computes, one
 * element at a time in 32-bit unsigned arithmetic (the tensor path splits the
 * same products into 16-bit halves inside int64 tensors): the lowbias32 hash
 * (C. Wellons, "Prospecting for Hash Functions", 2018) of the element index,
 * whose top 20 bits index a table of bf16 quantiles, and the optional
 * per-block outlier.  No codec or optimizer arithmetic lives here.  Plain C,
 * single-threaded per call; callers run several calls side by side.
 */
#include <stdint.h>
#include <string.h>

static inline uint32_t lowbias32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

/* h = H(H(lo(i) ^ k1) ^ (hi(i) + k2 mod 2^32)) */
static inline uint32_t hash_index(uint64_t i, uint32_t k1, uint32_t k2) {
    uint32_t x = lowbias32((uint32_t)i ^ k1);
    x ^= (uint32_t)(i >> 32) + k2;
    return lowbias32(x);
}

static inline uint16_t bf16_scale_rne(uint16_t b, float factor) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    f = f * factor;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u); /* round to nearest even (finite values) */
    return (uint16_t)(u >> 16);
}

/* Outlier description: block size B (0 = none); a block is picked when its
 * hash under (p1, p2) is below thr; the picked element is the hash under
 * (e1, e2) modulo B; it is multiplied by `factor` and rounded to bf16. */
typedef struct {
    int64_t block;
    uint64_t thr;
    uint32_t p1, p2, e1, e2;
    float factor;
} synth_outliers;

/* out[j] = value of global index start + j, j < count. */
void synth_fill(uint16_t* out, const uint16_t* table, int32_t table_shift, uint32_t k1,
                uint32_t k2, int64_t start, int64_t count, const synth_outliers* o) {
    for (int64_t j = 0; j < count; ++j)
        out[j] = table[hash_index((uint64_t)(start + j), k1, k2) >> table_shift];
    if (!o || o->block <= 0 || count <= 0) return;
    const int64_t B = o->block;
    const int64_t b0 = start / B, b1 = (start + count - 1) / B;
    for (int64_t b = b0; b <= b1; ++b) {
        if ((uint64_t)hash_index((uint64_t)b, o->p1, o->p2) >= o->thr) continue;
        const int64_t e = b * B + (int64_t)(hash_index((uint64_t)b, o->e1, o->e2) % (uint64_t)B);
        if (e >= start && e < start + count) out[e - start] = bf16_scale_rne(out[e - start], o->factor);
    }
}

/* out[j] = value of global index idx[j]. */
void synth_at(uint16_t* out, const uint16_t* table, int32_t table_shift, uint32_t k1, uint32_t k2,
              const int64_t* idx, int64_t count, const synth_outliers* o) {
    for (int64_t j = 0; j < count; ++j) {
        const uint64_t i = (uint64_t)idx[j];
        uint16_t v = table[hash_index(i, k1, k2) >> table_shift];
        if (o && o->block > 0) {
            const int64_t b = idx[j] / o->block;
            if ((uint64_t)hash_index((uint64_t)b, o->p1, o->p2) < o->thr &&
                b * o->block + (int64_t)(hash_index((uint64_t)b, o->e1, o->e2) % (uint64_t)o->block) ==
                    idx[j])
                v = bf16_scale_rne(v, o->factor);
        }
        out[j] = v;
    }
}
