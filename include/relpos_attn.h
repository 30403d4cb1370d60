/*
 * relpos_attn.h -- C ABI of the GB300 (sm_103a) relative-position attention
 * library (librelpos_attn.so): the forward pass (also over right-padded
 * batches), the T5 cached decode and the T5, Shaw, DeBERTa and ALiBi
 * backward passes (relpos_t5_attn_bwd, relpos_shaw_attn_bwd,
 * relpos_deberta_attn_bwd, relpos_alibi_attn_bwd, at the end of this header).
 *
 * One forward call computes multi-head attention whose logits carry a relative-
 * position term that is formed inside the kernel and never written to
 * device memory as an L x L (or L x L x d) tensor:
 *
 *   RELPOS_T5      per-head scalar bias looked up by bucket of the offset
 *                  key - query ("Relative Position Embeddings, in depth",
 *                  section "T5: one scalar per head, looked up by bucket";
 *                  "T5 Relative-Position Bias", bucket definition and the
 *                  cached-decoder example).
 *                  logit = q.k / sqrt(d) + bias[bucket(j - p)][h]
 *   RELPOS_SHAW    clipped relative key and value vectors ("Relative
 *                  Position Embeddings, in depth", section "Shaw et al.").
 *                  logit = q.(k_j + a_K[clip(j - p, -k, k) + k]) / sqrt(d)
 *                  out   = sum_j softmax_j * (v_j + a_V[clip(j - p, -k, k) + k])
 *   RELPOS_DEBERTA disentangled content/position attention ("Relative
 *                  Position Embeddings, in depth", section "DeBERTa:
 *                  disentangled content and position"; "DeBERTa > Relative
 *                  Position Encoding", section "The Relative Position
 *                  Formula" for delta).
 *                  logit = (q_i.k_j + q_i.Pk[delta(p, j)] + k_j.Pq[delta(j, p)])
 *                          / sqrt(3d),  delta(a, b) = clip(a - b, -k, k - 1) + k
 *   RELPOS_ALIBI   a fixed slope per head times the distance, no table and
 *                  no maximum distance ("Relative Position Embeddings, in
 *                  depth", section "ALiBi and RoPE: the two endpoints").
 *                  logit = q.k / sqrt(d) - slope[h] * |j - p|
 *   RELPOS_TXL     Transformer-XL: content and position keys with their own
 *                  projections and two global biases u, v ("Relative
 *                  Position Embeddings, in depth", section "Transformer-XL:
 *                  four terms and two global biases").
 *                  logit = ((q + u[h]).k_j + (q + v[h]).W[h] R(p - j)) / sqrt(d)
 *                  with R(t) the fixed sinusoidal encoding of the offset
 *                  t = query - key position: R[2m] = sin(w_m t),
 *                  R[2m+1] = cos(w_m t), w_m = 10000^(-2m/d).
 *
 * Positions: query row i sits at absolute position p = i + q_offset; key
 * row j at position j. With causal = 1 keys j > p are masked out (and T5
 * uses its causal bucket mapping). A query row with no visible key gets a
 * zero output row.
 *
 * Conventions shared by every entry point:
 *  - Pointers marked "device" are CUDA device pointers owned by the caller;
 *    the library keeps no reference to them after the call returns.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous on that stream unless stated otherwise.
 *  - Return value: RELPOS_OK (0) or a negative RELPOS_ERR_* code; argument
 *    errors are reported before anything is launched. relpos_strerror()
 *    names a code. No entry point falls back to a CPU path.
 */
#ifndef RELPOS_ATTN_H_
#define RELPOS_ATTN_H_

#ifdef __cplusplus
extern "C" {
#endif

/* modes */
#define RELPOS_T5 0
#define RELPOS_SHAW 1
#define RELPOS_DEBERTA 2
#define RELPOS_ALIBI 3
#define RELPOS_TXL 4

/* element types of Q, K, V and out */
#define RELPOS_BF16 0
#define RELPOS_FP32 1

/* return codes */
#define RELPOS_OK 0
#define RELPOS_ERR_INVALID_ARG (-1)    /* null pointer, bad size or parameter */
#define RELPOS_ERR_UNSUPPORTED (-2)    /* valid request this build does not run (d = 128 Shaw, ...) */
#define RELPOS_ERR_CUDA (-3)           /* a CUDA runtime call or launch failed */
#define RELPOS_ERR_DEVICE_TIMEOUT (-4) /* a kernel gave up on a bounded wait */
#define RELPOS_ERR_SCRATCH_LIMIT (-5)  /* request needs more than the fixed scratch of
                                          relpos_t5_decode_noalloc */

/*
 * relpos_attn_fwd -- attention forward with an in-kernel relative term.
 *
 *   mode        RELPOS_T5, RELPOS_SHAW, RELPOS_DEBERTA, RELPOS_ALIBI or RELPOS_TXL.
 *   dtype       RELPOS_BF16 or RELPOS_FP32: element type of Q, K, V and out.
 *               FP32 inputs are rounded to bf16 on the device before the
 *               tensor-core products (fp32 accumulation); out is fp32.
 *   Q           device, [B, H, Lq, d] row-major.
 *   K, V        device, [B, H, Lk, d] row-major.
 *   table0/1    device tables, row-major:
 *                 T5:      table0 = bias [num_buckets, H] fp32; table1 unused.
 *                 Shaw:    table0 = a_K, table1 = a_V, each [2k+1, d] bf16,
 *                          shared by all heads.
 *                 DeBERTa: table0 = Pk, table1 = Pq, each [2k, H, d] bf16
 *                          (already projected per head).
 *                 ALiBi:   table0 = slopes [H] fp32 (any values the caller
 *                          chooses); table1 unused.
 *                 TXL:     table0 = W [H, d, d] fp32, the key projection of
 *                          the sinusoid per head, output index first
 *                          (r[e] = sum_f W[h][e][f] R[f]); table1 = [2, H, d]
 *                          fp32, u then v. Memory (cached keys of the
 *                          previous segment) is ordinary keys at positions
 *                          0 .. mem - 1 with q_offset = mem.
 *   B, H        batch and heads (>= 0; 0 makes the call a no-op).
 *   Lq, Lk      query and key lengths (Lq >= 0, Lk >= 0). Lk == 0 writes
 *               zeros.
 *   d           head dimension: 64 for every mode; also 128 for T5 and
 *               ALiBi with dtype BF16 (other modes and FP32 inputs at
 *               d = 128 return RELPOS_ERR_UNSUPPORTED). At d = 128 a few
 *               query rows take the prefill kernel, not the split-key
 *               decode path, and T5 keeps a single table copy when its
 *               four shifted copies do not fit beside the larger tiles.
 *   num_buckets T5 only: even, 4 <= num_buckets <= 128 (ignored otherwise).
 *   rel_param   T5: max_distance (> num_buckets/4 bidirectional, > num_buckets/2
 *               causal); Shaw: clip k (1 <= k <= 64); DeBERTa: k (1 <= k <= 4096);
 *               ALiBi, TXL: ignored.
 *               Shaw's per-row tables and T5's bias-by-offset table live in
 *               shared memory: this build runs Shaw k <= 27, and T5 as long as
 *               the distance at which the last bucket starts (about
 *               max_distance, or the longest offset of the call if shorter)
 *               is at most about 2500 (beyond about 480 through a slower
 *               single-copy table); beyond, the call returns
 *               RELPOS_ERR_UNSUPPORTED.
 *   causal      0 or 1.
 *   q_offset    absolute position of query row 0 (>= 0), for cached decoding.
 *   out         device, [B, H, Lq, d], element type per dtype; written fully.
 *   stream      cudaStream_t.
 *
 * Scratch: calls with dtype FP32, with DeBERTa or TXL (the rows
 * [q + u | W^T (q + v) rotated by the query's angles], 256 bytes per query
 * row, and the keys' sinusoid table), or that take the split-key
 * decode path (few query rows) draw temporary device memory with
 * cudaMallocAsync on `stream` and release it with cudaFreeAsync before
 * returning. Nothing persists between calls.
 * Errors: RELPOS_ERR_INVALID_ARG / _UNSUPPORTED before launch;
 * RELPOS_ERR_CUDA if a launch or allocation fails. Device-side bounded-wait
 * failures are reported by relpos_check_status().
 */
int relpos_attn_fwd(int mode, int dtype, const void* Q, const void* K, const void* V,
                    const void* table0, const void* table1, int B, int H, int Lq, int Lk,
                    int d, int num_buckets, int rel_param, int causal, int q_offset,
                    void* out, void* stream);

/*
 * relpos_attn_fwd_padded -- relpos_attn_fwd over a right-padded batch of
 * sequences of different lengths. The pages do not treat padding; the
 * reading here: batch element b holds lengths[b] valid query rows and keys
 * (its first rows of Q, K and V), so its output equals that sequence
 * computed alone, and its rows from lengths[b] on are written as zeros.
 * Keys from lengths[b] on are masked for every row of element b; the rows and
 * keys in the padding may hold anything. Positions and q_offset are as for
 * relpos_attn_fwd (the relative offsets are the unpadded ones).
 *
 *   lengths     device, int32 [B], 4-byte aligned: read by the kernels, so
 *               the host does not check its values; a negative length counts
 *               as 0 (all rows zero), one beyond Lq / Lk as no padding.
 *   all other arguments as for relpos_attn_fwd. Calls with T5 and Lq <= 8
 *   run the fused kernel, not the split-key decode.
 * Errors: as relpos_attn_fwd; RELPOS_ERR_INVALID_ARG for a null or
 * misaligned lengths.
 */
int relpos_attn_fwd_padded(int mode, int dtype, const void* Q, const void* K, const void* V,
                           const void* table0, const void* table1, const int* lengths, int B,
                           int H, int Lq, int Lk, int d, int num_buckets, int rel_param, int causal,
                           int q_offset, void* out, void* stream);

/*
 * relpos_index_ids -- test hook: the device index generator the kernels use,
 * run over n consecutive offsets rel_first .. rel_first + n - 1.
 *
 *   T5:      offsets are key - query; ids are buckets ("T5: one scalar per
 *            head, looked up by bucket"); causal selects the causal mapping.
 *   Shaw:    offsets are key - query; ids are clip(rel, -k, k) + k.
 *   DeBERTa: offsets are query - key; ids are delta = clip(rel, -k, k-1) + k.
 *   ALiBi:   offsets are key - query; ids are the distances |rel|.
 *   TXL:     offsets are key - query; ids are t = query - key = -rel, the
 *            argument of the sinusoidal encoding R(t).
 *   out_dev  device int32[n], written asynchronously on `stream`.
 * Parameter checks are those of relpos_attn_fwd.
 */
int relpos_index_ids(int mode, int n, int rel_first, int num_buckets, int rel_param,
                     int causal, int* out_dev, void* stream);

/*
 * relpos_check_status -- synchronize `stream` and report whether any kernel
 * of this library hit a bounded-wait limit since the last check
 * (RELPOS_ERR_DEVICE_TIMEOUT), or a CUDA error (RELPOS_ERR_CUDA). Clears the
 * recorded device status. Blocking.
 */
int relpos_check_status(void* stream);

/* relpos_strerror -- static description of a return code; never NULL. */
const char* relpos_strerror(int code);

/*
 * relpos_selftest_wait_timeout -- runs one tiny kernel that waits, with a
 * limit of `timeout_us` microseconds (1 .. 1000000), on a barrier that
 * nothing completes, exactly as the attention kernels' waits do. It records
 * RELPOS_ERR_DEVICE_TIMEOUT in the device status word and returns; the
 * context stays usable. Used to test the failure path without faulting or
 * hanging the GPU. Asynchronous; read the result with relpos_check_status().
 */
int relpos_selftest_wait_timeout(int timeout_us, void* stream);

/*
 * relpos_t5_decode_noalloc -- T5-bias cached decoding that allocates nothing.
 *
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory while they run -- code working inside a
 * memory budget planned ahead, or a serving loop that must keep the
 * allocator (cudaMallocAsync can synchronize or fail once the pool is
 * exhausted) off its hot path. It computes exactly what relpos_attn_fwd
 * computes for mode RELPOS_T5, dtype RELPOS_BF16 and Lq <= 8 (the split-key
 * decode path), but keeps the per-chunk partial results in one static
 * device array of 4 MiB built into the library, which every GPU that loads
 * the library holds until the process exits.
 *
 *   Q, K, V, bias, out, B, H, Lq, Lk, num_buckets, max_distance, causal,
 *   q_offset, stream: as for relpos_attn_fwd (bf16 Q/K/V/out, d = 64, fp32
 *   bias [num_buckets, H]); Lq must be <= 8 (RELPOS_ERR_UNSUPPORTED otherwise).
 * Limit: B * H * Lq * ceil(Lk / 256) * 264 bytes must fit in the 4 MiB array
 *   (for example B * H = 512 single-row queries over 4096 keys take 2.2 MiB);
 *   larger requests return RELPOS_ERR_SCRATCH_LIMIT before anything launches.
 * No cudaMalloc, cudaFree or allocating library routine is called. The first
 * call on each device looks up the array's device address (with that device
 * current); make that first call before any stream capture. Every call
 * shares the one array, so calls whose kernels overlap on the GPU (other
 * streams, other host threads) race and corrupt each other's results; order
 * them on one stream. Each call overwrites every partial it reads, so nothing
 * has to be cleared between calls. Asynchronous on `stream`.
 */
int relpos_t5_decode_noalloc(const void* Q, const void* K, const void* V, const void* bias, int B,
                             int H, int Lq, int Lk, int num_buckets, int max_distance, int causal,
                             int q_offset, void* out, void* stream);

/*
 * relpos_t5_decode_positions -- T5-bias cached decoding over keys at explicit
 * positions: a cache that evicted tokens keeps each remaining key at its
 * original position, and since the bias depends only on the offset nothing
 * stored needs rewriting ("Relative Position Embeddings, in depth", section
 * "Kernels and the KV cache").
 *
 *   key_pos     device, int32 [B, H, Lk]: the position of each key row, in
 *               any order, each in [0, 2^28]. The offset of key j to query
 *               row i is key_pos[b, h, j] - (i + q_offset); with causal = 1 a
 *               key whose position lies after the query's is masked out. A
 *               query row with no visible key gets a zero row.
 *   Q, K, V, bias, out, B, H, Lq, Lk, num_buckets, max_distance, causal,
 *   q_offset, stream: as for relpos_attn_fwd with mode RELPOS_T5 and dtype
 *   RELPOS_BF16 (d = 64), any Lq: up to 8 query rows run the split-key
 *   decode kernels, more rows (a chunk of new tokens against the cache) the
 *   fused prefill kernel, which then visits every key tile (a key's index
 *   says nothing about its position) and takes the bias per element from
 *   the positions on tiles that are neither wholly beyond the saturation
 *   distance nor free of masked keys.
 * Scratch: for Lq <= 8 the per-chunk partials (B * H * Lq * ceil(Lk / 256) *
 * 264 bytes) come from cudaMallocAsync on `stream` and go back with
 * cudaFreeAsync before the call returns; none otherwise. Asynchronous on
 * `stream`.
 */
int relpos_t5_decode_positions(const void* Q, const void* K, const void* V, const void* bias,
                               const int* key_pos, int B, int H, int Lq, int Lk, int num_buckets,
                               int max_distance, int causal, int q_offset, void* out, void* stream);

/*
 * relpos_alibi_decode_positions -- ALiBi cached decoding over keys at
 * explicit positions ("Relative Position Embeddings, in depth", sections
 * "ALiBi and RoPE: the two endpoints" and "Kernels and the KV cache"): the
 * logit of query row i and key j is q_i . k_j / sqrt(64) - slope_h *
 * |key_pos[b, h, j] - (i + q_offset)|.
 *
 *   slopes      device, fp32 [H], 4-byte aligned: the heads' slopes.
 *   key_pos, causal, q_offset, out, B, H, Lk, stream: as for
 *               relpos_t5_decode_positions (bf16 Q, K, V, out; d = 64).
 *   Lq          0 .. 8 query rows (RELPOS_ERR_UNSUPPORTED beyond).
 * The split-key decode kernels, with each key's bias formed from its
 * position. Scratch and asynchrony as relpos_t5_decode_positions for
 * Lq <= 8.
 */
int relpos_alibi_decode_positions(const void* Q, const void* K, const void* V, const void* slopes,
                                  const int* key_pos, int B, int H, int Lq, int Lk, int causal,
                                  int q_offset, void* out, void* stream);

/*
 * relpos_t5_attn_bwd -- gradients of the T5-bias attention forward
 * (relpos_attn_fwd with mode RELPOS_T5, dtype RELPOS_BF16). The bias is a
 * learned table ("Relative Position Embeddings, in depth", section "T5: one
 * scalar per head, looked up by bucket"; "T5 Relative-Position Bias": every
 * offset of a bucket shares the bucket's value), so its gradient gathers the
 * logit gradients dS_ij = P_ij (dP_ij - sum_l P_il dP_il) of every (batch, i, j)
 * whose offset falls in the bucket. The pages print no backward pass; the
 * other gradients follow from the chain rule through the forward:
 * dV = P^T dO, dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d). The row term
 * sum_j P_ij dP_ij is formed from P and dP themselves (not from the forward's
 * output), so no output of the forward is needed.
 *
 *   Q, K, V, bias, B, H, Lq, Lk, d, num_buckets, max_distance, causal,
 *   q_offset, stream: the forward call's arguments (bf16 Q [B,H,Lq,64], K, V
 *               [B,H,Lk,64]; fp32 bias [num_buckets, H]; d must be 64).
 *   dO          device, bf16 [B,H,Lq,64]: gradient of the loss w.r.t. O.
 *   dQ          device, bf16 [B,H,Lq,64], written.
 *   dK, dV      device, bf16 [B,H,Lk,64], written (rows no query sees: zero).
 *   dbias       device, fp32 [num_buckets, H], overwritten with the sum over
 *               the whole batch (the table is shared by it).
 * All pointers 16-byte aligned and caller-owned; the outputs must not overlap
 * the inputs. Limits: the distance R at which the last bucket starts (or the
 * largest offset present, if smaller) must be <= 1024
 * (RELPOS_ERR_UNSUPPORTED otherwise; max_distance 128 gives R = 91
 * bidirectional, 113 causal). Scratch: about 264 * B * H * Lq bytes (an
 * fp32 dQ accumulator and the row statistics, padded to 128-row tiles) from cudaMallocAsync on `stream`,
 * freed with cudaFreeAsync before the call returns. dQ and dbias are
 * accumulated with floating-point atomics, so their last bits may differ
 * between runs. Asynchronous on `stream`; device timeouts surface through
 * relpos_check_status().
 */
int relpos_t5_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                       const void* bias, int B, int H, int Lq, int Lk, int d, int num_buckets,
                       int max_distance, int causal, int q_offset, void* dQ, void* dK, void* dV,
                       void* dbias, void* stream);

/*
 * relpos_alibi_attn_bwd -- gradients of the ALiBi attention forward
 * (relpos_attn_fwd with mode RELPOS_ALIBI, dtype RELPOS_BF16; "Relative
 * Position Embeddings, in depth", section "ALiBi and RoPE: the two
 * endpoints"). The pages treat the slopes as fixed; their gradient is still
 * returned, dslope_h = -sum_{b,i,j} dS_ij |j - p_i|, with dS, dQ, dK, dV as
 * for relpos_t5_attn_bwd.
 *
 *   Q, K, V, dO, B, H, Lq, Lk, d, causal, q_offset, dQ, dK, dV, stream: as for
 *               relpos_t5_attn_bwd.
 *   slopes      device, fp32 [H]: the forward call's slopes.
 *   dslopes     device, fp32 [H], overwritten with the sum over the batch.
 * Scratch, limits and errors as relpos_t5_attn_bwd (no saturation-distance
 * limit). dslopes is accumulated with floating-point atomics.
 */
int relpos_alibi_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                          const void* slopes, int B, int H, int Lq, int Lk, int d, int causal,
                          int q_offset, void* dQ, void* dK, void* dV, void* dslopes, void* stream);

/*
 * relpos_shaw_attn_bwd -- gradients of the Shaw attention forward
 * (relpos_attn_fwd with mode RELPOS_SHAW, dtype RELPOS_BF16; "Relative
 * Position Embeddings, in depth", section "Shaw et al."). With r_ij =
 * clip(j - p_i, -k, k) + k the logit is q_i . (k_j + a_K[r_ij]) / sqrt(d) and
 * the value of key j for query i is v_j + a_V[r_ij]. The chain rule gives
 *   dP_ij = dO_i . (v_j + a_V[r_ij]),  dS_ij = P_ij (dP_ij - sum_l P_il dP_il),
 *   dQ_i = sum_j dS_ij (k_j + a_K[r_ij]) / sqrt(d),  dK_j = sum_i dS_ij q_i / sqrt(d),
 *   dV_j = sum_i P_ij dO_i,
 *   da_K[r] = sum of dS_ij q_i / sqrt(d) and da_V[r] = sum of P_ij dO_i over
 *   every (batch, head, i, j) with r_ij = r (the tables are shared by the
 *   batch and the heads).
 *
 *   Q, K, V, dO, B, H, Lq, Lk, d, causal, q_offset, dQ, dK, dV, stream: as for
 *               relpos_t5_attn_bwd.
 *   aK, aV      device, bf16 [2k + 1, 64]: the forward call's tables.
 *   clip_k      k, the forward call's rel_param; 1 <= k <= 16
 *               (RELPOS_ERR_INVALID_ARG below 1, RELPOS_ERR_UNSUPPORTED above 16).
 *   daK, daV    device, fp32 [2k + 1, 64], overwritten with the sums over the
 *               batch and the heads.
 * Scratch: about (264 + 16 (2k + 2) + 4) * B * H * Lq bytes plus
 * 2 (2k + 1) * 256 bytes per 128-row query tile and head, from cudaMallocAsync on `stream`,
 * freed with cudaFreeAsync before the call returns. daK and daV are summed in
 * a fixed order (the same bits every run); dQ, dK and dV as for
 * relpos_t5_attn_bwd. Errors and asynchrony as relpos_t5_attn_bwd.
 */
int relpos_shaw_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                         const void* aK, const void* aV, int B, int H, int Lq, int Lk, int d,
                         int clip_k, int causal, int q_offset, void* dQ, void* dK, void* dV,
                         void* daK, void* daV, void* stream);

/*
 * relpos_deberta_attn_bwd -- gradients of the DeBERTa attention forward
 * (relpos_attn_fwd with mode RELPOS_DEBERTA, dtype RELPOS_BF16; "Relative
 * Position Embeddings, in depth", section "DeBERTa: disentangled content and
 * position"; "DeBERTa > Relative Position", the relative-position formula).
 * With delta(i, j) = clip(p_i - j, -k, k - 1) + k and s = 1 / sqrt(3 d) the
 * logit is s (q_i . k_j + q_i . Pk[delta(i, j), h] + k_j . Pq[delta(j, i), h]);
 * the chain rule gives, with dS as for relpos_t5_attn_bwd,
 *   dQ_i = s sum_j dS_ij (k_j + Pk[delta(i, j), h]),
 *   dK_j = s sum_i dS_ij (q_i + Pq[delta(j, i), h]),  dV = P^T dO,
 *   dPk[r, h] = s sum of dS_ij q_i over every (batch, i, j) of head h with
 *   delta(i, j) = r, and dPq[r, h] = s sum of dS_ij k_j over delta(j, i) = r.
 *
 *   Q, K, V, dO, B, H, Lq, Lk, d, causal, q_offset, dQ, dK, dV, stream: as for
 *               relpos_t5_attn_bwd.
 *   Pk, Pq      device, bf16 [2k, H, 64]: the forward call's tables.
 *   k           the forward call's rel_param; 1 <= k <= 4096
 *               (RELPOS_ERR_INVALID_ARG below 1, RELPOS_ERR_UNSUPPORTED above).
 *   dPk, dPq    device, fp32 [2k, H, 64], overwritten with the sums over the
 *               batch.
 * The logits' relative part comes from the forward's band pre-pass (c2p +
 * p2c inside the band, rounded to bf16 as in the forward). Scratch, from
 * cudaMallocAsync on `stream` and freed before the call returns: about
 * (300 + 8k) * B * H * Lq bytes plus (280 + 4k) * B * H * Lk bytes (the
 * band, dS gathered by table row query- and key-major, fp32 dQ and dK).
 * The table products run as cuBLAS GEMMs (bf16 operands, fp32 accumulation;
 * the library is loaded with this one). Errors and asynchrony as
 * relpos_t5_attn_bwd.
 */
int relpos_deberta_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                            const void* Pk, const void* Pq, int B, int H, int Lq, int Lk, int d, int k,
                            int causal, int q_offset, void* dQ, void* dK, void* dV, void* dPk, void* dPq,
                            void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RELPOS_ATTN_H_ */
