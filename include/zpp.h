/*
 * zpp.h -- C ABI of the GB300 ZeRO++ data-parallel codec path.
 *
 * Three parts, all on one GPU, with the N_d data-parallel ranks simulated as
 * separate buffers in device memory (a "message" is an HBM buffer written by
 * one call and read by the next):
 *
 *   qwZ  block-wise int8/int4 quantization of 16-bit weight shards before the
 *        forward all-gather, and the receiver-side dequantization
 *        ("Quantized LLM Training at Scale with ZeRO++", section "The Three
 *        Pillars of ZeRO++", 1 QWZ; "ZeRO-1/2/3", ZeRO++ note: qwZ int8/int4).
 *   qgZ  tensor-slice reordering plus one-shot block quantization of every
 *        rank's gradient bucket, then the two-hop hierarchical reduce: hop 1 an
 *        intra-node all-to-all with reduction, hop 2 an inter-node all-to-all
 *        with reduction ("Quantized LLM Training at Scale with ZeRO++", 3 QGZ,
 *        the three challenge/solution pairs).
 *   Adam the Stage-2/3 sharded mixed-precision Adam step on the owned shard:
 *        fp32 gradient, fp32 master/m/v, 16-bit parameter written back
 *        ("ZeRO-1/2/3", Stage 1 steps 4-6 and Stage 2; "ZeRO Stage 2:
 *        Gradient Partitioning", last paragraph on mixed precision).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named *_dev / device buffers are CUDA device pointers owned and
 *   allocated by the caller; the library never allocates, frees or
 *   synchronises.  Every device pointer must be 16-byte aligned
 *   (ZPP_ERR_MISALIGNED otherwise).  `stream` is a cudaStream_t passed as
 *   void* (NULL = the legacy default stream); work is enqueued on it and the
 *   call returns without waiting.
 * - bf16 values are passed as their raw 16-bit patterns (uint16_t).
 * - Block quantization (a "block" is `block` consecutive elements):
 *     qmax = 2^(bits-1) - 1                     (127 for int8, 7 for int4)
 *     s    = absmax(block) / qmax               (fp32 IEEE divide)
 *     q    = clamp(rint(x / s), -qmax, qmax)    (fp32 divide, ties to even)
 *     s == 0 gives q == 0 for the whole block.
 *   Codes are int8, or int4 two's-complement nibbles with element 2i in the
 *   low nibble of byte i.  Scales are fp32, one per block.  Dequantization is
 *   the single rounded product (float)q * s.  `block` is a power of two in
 *   [64, 4096]; `bits` is 4 or 8.
 * - Topology: N_d = nodes * gpus_per_node ranks; rank r = n*G + l is GPU l of
 *   node n.  A gradient bucket of `bucket_elems` elements is cut into N_d
 *   slices of L = bucket_elems / N_d; slice j belongs to rank j.
 * - Errors: arguments are validated on the host before anything is
 *   launched; a failed check returns its code and enqueues nothing.  Launch
 *   failures return ZPP_ERR_CUDA (the CUDA error is cleared and its text is
 *   available from zpp_last_cuda_error()).  Faults during execution surface
 *   at the caller's next synchronisation.  Zero-sized work returns ZPP_OK
 *   without launching.
 * - Results are bit-identical from run to run (no atomics, fixed summation
 *   order).  Calls on different streams may run concurrently as long as they
 *   do not write the same buffers.
 */
#ifndef ZPP_H
#define ZPP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t zpp_status;
#define ZPP_OK 0
#define ZPP_ERR_INVALID_ARG 1 /* a size, bit width, block, topology or pointer is invalid */
#define ZPP_ERR_MISALIGNED 2  /* a device pointer is not 16-byte aligned                 */
#define ZPP_ERR_UNSUPPORTED 3 /* valid request this build does not implement            */
#define ZPP_ERR_CUDA 4        /* a CUDA runtime call or kernel launch failed             */

/* Adam hyper-parameters of one step.  `step` is t >= 1; bias corrections are
 * bc = 1 - beta^t (beta^t in double, rounded to float once) and (1 - beta) is
 * rounded to float from double. */
typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    int32_t step;
} zpp_adam_hparams;

/* Adam state of the owned parameters (device pointers, fp32 except the bf16
 * parameter copy); element i is global parameter i of the bucket / shard. */
typedef struct {
    float* master;
    float* m;
    float* v;
    uint16_t* param_bf16; /* may be NULL: then no 16-bit copy is written */
} zpp_adam_state;

/* ---- qwZ ------------------------------------------------------------------ */

/* zpp_qwz_quant -- quantize nranks weight shards for the forward all-gather.
 * ("Quantized LLM Training at Scale with ZeRO++", Three Pillars, 1 QWZ: the
 * weight tensor is cut into chunks, each quantized with its own scale.)
 *   x_bf16  [nranks][shard_elems] bf16 (device, read).
 *   codes   [nranks][zpp_codes_bytes(shard_elems, bits)] bytes (device, written).
 *   scales  [nranks][zpp_num_blocks(shard_elems, block)] fp32 (device, written).
 * Blocks restart at the start of every shard; the last block of a shard may
 * be short and its scale covers only its own elements.  int4 needs an even
 * shard_elems.  Errors: ZPP_ERR_INVALID_ARG (bits, block, negative sizes,
 * odd int4 shard, NULL pointer with nonzero work), ZPP_ERR_MISALIGNED. */
zpp_status zpp_qwz_quant(const uint16_t* x_bf16, int64_t nranks, int64_t shard_elems,
                         int32_t block, int32_t bits, void* codes, float* scales,
                         void* stream);

/* zpp_qwz_dequant -- receiver side of the quantized all-gather: the codes and
 * scales of all nranks shards become one full bf16 tensor
 * y[r*shard_elems + i] = bf16_rn((float)q * s) (round to nearest even).
 * ("Quantized LLM Training at Scale with ZeRO++", 1 QWZ: weights travel in
 * 8-bit and are used in 16-bit.)  Layouts as in zpp_qwz_quant; y_bf16 is
 * [nranks][shard_elems] (device, written).  Errors as zpp_qwz_quant. */
zpp_status zpp_qwz_dequant(const void* codes, const float* scales, int64_t nranks,
                           int64_t shard_elems, int32_t block, int32_t bits,
                           uint16_t* y_bf16, void* stream);

/* ---- qgZ ------------------------------------------------------------------ */

/* zpp_qgz_reorder_quant -- tensor-slice reordering fused with the one-shot
 * block quantization of every rank's gradient bucket.
 * ("Quantized LLM Training at Scale with ZeRO++", 3 QGZ: one-shot
 * quantization on each GPU; slices swapped before any communication so they
 * land on the right GPU after the two hops.)
 *   grads_bf16  [N_d][bucket_elems] bf16 (device, read).
 *   codes       [N_d][zpp_codes_bytes(bucket_elems, bits)] (device, written).
 *   scales      [N_d][bucket_elems / block] fp32 (device, written).
 * Slice j = n'*G + l' of rank r's bucket is stored at slice position
 * p = l'*N + n' of rank r's message (zpp_qgz_slice_perm), so chunk l of the
 * message (N consecutive slices) is what rank r sends to local peer l in hop 1.
 * Requires bucket_elems % (N_d * block) == 0 (blocks never straddle slices).
 * Errors: ZPP_ERR_INVALID_ARG, ZPP_ERR_MISALIGNED. */
zpp_status zpp_qgz_reorder_quant(const uint16_t* grads_bf16, int32_t nodes,
                                 int32_t gpus_per_node, int64_t bucket_elems, int32_t block,
                                 int32_t bits, void* codes, float* scales, void* stream);

/* zpp_grad_accumulate -- fp32 accumulation of one micro-batch's gradients.
 * ("ZeRO Stage 2: Gradient Partitioning", compatibility with gradient
 * accumulation: micro-batch gradients are summed on each GPU with no
 * communication; the reduce-scatter runs once, after the last micro-batch.)
 *   grads_bf16  [n] bf16 (device, read): this micro-batch's gradients.
 *   acc         [n] fp32 (device, read unless first, written):
 *               acc <- (first ? 0 : acc) + (float)grads, one fp32 add each.
 *   first       1 for the first micro-batch (acc is not read), else 0.
 * For the last micro-batch use zpp_qgz_reorder_quant_acc instead, which adds
 * it while quantizing and never writes the sum back.
 * Errors: ZPP_ERR_INVALID_ARG (n < 0, first not 0/1, NULL), ZPP_ERR_MISALIGNED. */
zpp_status zpp_grad_accumulate(const uint16_t* grads_bf16, float* acc, int64_t n, int32_t first,
                               void* stream);

/* zpp_qgz_reorder_quant_acc -- zpp_qgz_reorder_quant of the accumulated
 * gradient: element e of rank r's bucket is acc[r][e] + (float)grads[r][e]
 * (one fp32 add, the last micro-batch's contribution), quantized from fp32.
 * ("ZeRO Stage 2: Gradient Partitioning", gradient accumulation: the
 * reduce-scatter fires once the accumulation is complete.)
 *   grads_bf16  [N_d][bucket_elems] bf16 (device, read): the last micro-batch.
 *   acc         [N_d][bucket_elems] fp32 (device, read): the earlier ones,
 *               as zpp_grad_accumulate left them.
 *   other arguments, layout and errors as zpp_qgz_reorder_quant. */
zpp_status zpp_qgz_reorder_quant_acc(const uint16_t* grads_bf16, const float* acc, int32_t nodes,
                                     int32_t gpus_per_node, int64_t bucket_elems, int32_t block,
                                     int32_t bits, void* codes, float* scales, void* stream);

/* zpp_qgz_hop_reduce -- one hop of the hierarchical all-to-all with reduction.
 * ("Quantized LLM Training at Scale with ZeRO++", 3 QGZ: first an intra-node
 * all-to-all and reduction, then an inter-node all-to-all; "ZeRO Stage 2:
 * Gradient Partitioning": the reduce-scatter averages, GPU i ends with the
 * averaged gradient of shard i.)
 *
 * hop == 1 (intra-node).  codes_in/scales_in: the one-shot messages of
 *   zpp_qgz_reorder_quant.  Rank d = n*G + l sums, elementwise in fp32 and in
 *   the order g = 0..G-1, the dequantized chunk l of ranks n*G + g.
 *   - N > 1: the sum (N*L elements, slot k = partial sum of slice k*G + l over
 *     node n) is requantized with the same block and bits into
 *     codes_out [N_d][zpp_codes_bytes(N*L, bits)], scales_out [N_d][N*L/block].
 *   - N == 1: hop 1 is the final hop (see below).
 * hop == 2 (inter-node, requires N > 1).  codes_in/scales_in: the hop-1
 *   messages.  Rank d = n*G + l sums, in the order n' = 0..N-1, the
 *   dequantized slot n of ranks n'*G + l; this is the final hop.
 * Final hop: g = sum * (1.0f / N_d) for rank d's own slice, element i of which
 *   is global parameter d*L + i.  Optional outputs (at least one required):
 *   - grad_out [N_d][L] fp32 (device, written);
 *   - adam/state: the Adam step of zpp_shard_adam_step applied to g in the same
 *     pass (state indexed d*L + i, updated in place).
 *   codes_out/scales_out must be NULL.
 * Requires bucket_elems % (N_d * block) == 0.
 * Errors: ZPP_ERR_INVALID_ARG (hop/topology mismatch, missing or extra
 * outputs, sizes), ZPP_ERR_MISALIGNED. */
zpp_status zpp_qgz_hop_reduce(int32_t hop, const void* codes_in, const float* scales_in,
                              int32_t nodes, int32_t gpus_per_node, int64_t bucket_elems,
                              int32_t block, int32_t bits, void* codes_out,
                              float* scales_out, float* grad_out,
                              const zpp_adam_hparams* adam, const zpp_adam_state* state,
                              void* stream);

/* zpp_qgz_final_hop_adam_qwz -- the final hop of zpp_qgz_hop_reduce with the
 * Adam step, fused with the int8 block quantization of the updated 16-bit
 * parameters: the qwZ message of the next step's forward all-gather, produced
 * without reading the parameters again.
 * ("ZeRO-1/2/3", Stage 1 steps 6-7: the updated fp32 master is written back as
 * 16-bit parameters, which the next all-gather distributes; "Quantized LLM
 * Training at Scale with ZeRO++", 1 QWZ: that all-gather travels as blocks of
 * 8-bit codes with one scale each.)
 *   hop, codes_in .. grad_out, adam, state: as zpp_qgz_hop_reduce's final hop
 *     (hop 1 with nodes == 1, else hop 2); adam and state are required,
 *     state->param_bf16 may be NULL.
 *   qwz_bits: 8.  The quantization block is `block`, restarting at every
 *     rank's owned shard:
 *   qwz_codes  [N_d][L] int8 (device, written), qwz_scales [N_d][L / block]
 *     fp32 (device, written) -- exactly zpp_qwz_quant(param_bf16, N_d, L,
 *     block, 8) of the new parameters.
 * Requires L = bucket_elems / N_d to be a multiple of max(block, 512)
 * (ZPP_ERR_UNSUPPORTED otherwise) and qwz_bits == 8 (ZPP_ERR_UNSUPPORTED for
 * 4).  Other errors as zpp_qgz_hop_reduce. */
zpp_status zpp_qgz_final_hop_adam_qwz(int32_t hop, const void* codes_in, const float* scales_in,
                                      int32_t nodes, int32_t gpus_per_node,
                                      int64_t bucket_elems, int32_t block, int32_t bits,
                                      float* grad_out, const zpp_adam_hparams* adam,
                                      const zpp_adam_state* state, int32_t qwz_bits,
                                      void* qwz_codes, float* qwz_scales, void* stream);

/* zpp_ring_rs_step -- one step of a ring reduce-scatter of quantized
 * gradients, for every rank at once: the comparator of the one-shot scheme.
 * ("Quantized LLM Training at Scale with ZeRO++", 3 QGZ: a ring reduce-scatter
 * of quantized gradients dequantizes and requantizes once per GPU on the
 * ring -- N sequential quantizations, with their latency and precision loss
 * -- where qgZ quantizes once.)
 * Ring r -> r+1 (mod N_d); chunk c = elements [c*L, (c+1)*L) of a bucket,
 * L = bucket_elems / N_d; at step s (0..N_d-1) rank r works on chunk
 * c = (r - 1 - s) mod N_d:
 *   s = 0            out_r = Q(x_r[c])
 *   0 < s < N_d - 1  out_r = Q(D(in_{r-1}) + x_r[c])
 *   s = N_d - 1      g_r   = (D(in_{r-1}) + x_r[r]) * (1.0f / N_d)
 * Q: block quantization as zpp_qwz_quant (blocks restart at the chunk start),
 * D: (float)q * s, +: one rounded fp32 add.  Chunk c is summed in the ring
 * order c+1, c+2, ..., c; rank r ends with the average of chunk r, the
 * element ownership of zpp_qgz_hop_reduce's final hop.
 *   grads_bf16  [N_d][bucket_elems] bf16 (device, read).
 *   codes_in    [N_d][zpp_codes_bytes(L, bits)], scales_in [N_d][L / block]:
 *               the previous step's codes_out/scales_out (device, read;
 *               unused, may be NULL, at step 0).
 *   codes_out, scales_out: same shapes (device, written) for s < N_d - 1;
 *               grad_out [N_d][L] fp32 (device, written) at s = N_d - 1.
 * Requires bucket_elems % (N_d * block) == 0.  With N_d == 1 the only step is
 * the last: g = x.
 * Errors: ZPP_ERR_INVALID_ARG (step outside 0..N_d-1, sizes, missing
 * buffers), ZPP_ERR_MISALIGNED. */
zpp_status zpp_ring_rs_step(int32_t step, int32_t nranks, int64_t bucket_elems, int32_t block,
                            int32_t bits, const uint16_t* grads_bf16, const void* codes_in,
                            const float* scales_in, void* codes_out, float* scales_out,
                            float* grad_out, void* stream);

/* ---- hpZ ------------------------------------------------------------------ */

/* zpp_hpz_gather -- the backward weight all-gather of one node under hpZ,
 * read from the node's secondary partitions.
 * ("Quantized LLM Training at Scale with ZeRO++", 2 HPZ: every node keeps a
 * secondary replica of the model partitions, so the backward all-gather
 * reads only the node's own GPUs and moves nothing across nodes.)
 *   gpus_per_node    G, 1..64: one secondary partition per local rank.
 *   shards_per_rank  N (the number of nodes): local rank l's secondary
 *                    partition is slice l of the G-way split of the weights,
 *                    the N primary shards l*N .. l*N + N - 1, kept in the form
 *                    the forward all-gather delivered them.
 *   shard_elems      elements of one primary shard (even for bits 4).
 *   bits 8 or 4      sec_codes[l] [N][zpp_codes_bytes(shard, bits)] and
 *                    sec_scales[l] [N][zpp_num_blocks(shard, block)] (device,
 *                    read): the qwZ messages of those shards.
 *   bits 16          sec_codes[l] [N][shard] bf16 values; sec_scales unused
 *                    (may be NULL); block must still be valid.
 *   sec_codes, sec_scales: host arrays of G device pointers.
 *   y_bf16           [G*N][shard] bf16 (device, written): the full weights;
 *                    shard d = l*N + j is the j-th shard of sec_codes[l],
 *                    dequantized exactly as zpp_qwz_dequant does.
 * Errors: ZPP_ERR_INVALID_ARG (G outside 1..64, N < 1, sizes, bits, block,
 * NULL pointers), ZPP_ERR_MISALIGNED (a pointer not 16-byte aligned). */
zpp_status zpp_hpz_gather(int32_t gpus_per_node, int32_t shards_per_rank, int64_t shard_elems,
                          int32_t block, int32_t bits, const void* const* sec_codes,
                          const float* const* sec_scales, uint16_t* y_bf16, void* stream);

/* Bytes of one rank's secondary partition under hpZ: N shards of codes and
 * scales (bits 4/8) or of bf16 values (bits 16); -1 on bad args.  The G ranks
 * of a node together hold one full replica of the weights. */
int64_t zpp_hpz_secondary_bytes(int32_t shards_per_rank, int64_t shard_elems, int32_t block,
                                int32_t bits);

/* ---- sharded mixed-precision Adam ------------------------------------------ */

/* zpp_shard_adam_step -- one Adam step on n owned parameters.
 * ("ZeRO-1/2/3", Stage 1 steps 5-6: update the fp32 optimizer state and master
 * with the reduced gradient, then write the 16-bit parameter; "ZeRO Stage 2:
 * Gradient Partitioning": the gradient shard is converted to fp32 first.)
 *   grad   [n] fp32 (device, read).  hp: host pointer.  st: host pointer to a
 *   struct of device pointers, each [n], updated in place:
 *     m <- b1*m + (1-b1)*g ;  v <- b2*v + (1-b2)*(g*g)
 *     master <- master - (lr * (m/bc1)) / (sqrt(v/bc2) + eps)
 *     param_bf16 <- bf16_rn(master)
 *   every operation a separately rounded fp32 IEEE operation in that order.
 * Errors: ZPP_ERR_INVALID_ARG (step < 1, NULL state pointers), ZPP_ERR_MISALIGNED. */
zpp_status zpp_shard_adam_step(const float* grad, int64_t n, const zpp_adam_hparams* hp,
                               const zpp_adam_state* st, void* stream);

/* ---- host-only helpers (no device work) ------------------------------------ */

/* Bytes of the code array of n elements: ceil(n * bits / 8); -1 on bad args. */
int64_t zpp_codes_bytes(int64_t n, int32_t bits);

/* Number of blocks of n elements: ceil(n / block); -1 on bad args. */
int64_t zpp_num_blocks(int64_t n, int32_t block);

/* Slice permutation of the qgZ message: perm_host[p] = source slice stored at
 * position p, p = l*N + n holds slice n*G + l.  perm_host: host array [N_d]. */
zpp_status zpp_qgz_slice_perm(int32_t nodes, int32_t gpus_per_node, int32_t* perm_host);

/* Static text of a status code. */
const char* zpp_status_string(zpp_status s);

/* Text of the last CUDA error this library saw on the calling thread
 * ("" if none). */
const char* zpp_last_cuda_error(void);

/* ABI version of this header: (major << 16) | minor. */
int32_t zpp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZPP_H */
