/*
 * entropycache.h — C ABI of the EntropyCache denoising-step library (GB300, sm_103a).
 *
 * One denoising step of EntropyCache, the training-free KV-cache policy for diffusion
 * language models described in "EntropyCache: Decoded Token Entropy Guided KV Caching for
 * Diffusion Language Models" (Cheong, Son, Lim, Yoo; summaries at gist.science, zh and pt):
 *
 *   (a) softmax + greedy decode + Shannon entropy over the V-wide logits of each masked
 *       candidate position                         -> ec_entropy_decode
 *   (b) commit the decoded tokens, take the maximum entropy E of the newly decoded tokens
 *       and compare it with tau (full recompute iff E > tau)
 *   (c) push the new tokens onto the decode history and build the recompute set
 *       (still-masked positions plus the last k decoded ones; every position on a full
 *       step)                                      -> ec_select_recompute (b + c)
 *       then write the fresh K/V rows of that set into the layer's cache
 *                                                  -> ec_kv_scatter
 *   (d) bidirectional attention of the recompute rows against all L cached rows
 *                                                  -> ec_partial_attention
 *       (or, for a step known to be full, of every row: ec_dense_attention)
 *   ec_step runs (a)(b)(c) once and then (c-scatter)(d) for every layer.
 *
 * Beyond the step: ec_layer_forward runs the partial (or full) forward of one transformer layer
 * for the recompute set; ec_lm_head_entropy computes (a) from the candidates' hidden states (the
 * output projection fused with the decode, so the logits are never stored); ec_candidates builds
 * a step's candidates for block-wise or sliding-window decoding;
 * ec_entropy_decode_noalloc is (a) for callers that cannot allocate a workspace; and
 * ec_selftest_bounded_wait exercises the kernels' timeout path.
 *
 * Conventions shared by every entry point
 *   - Every call returns an ec_status and never throws or aborts.
 *   - Every data pointer is a DEVICE pointer owned by the caller (allocated by any means,
 *     e.g. PyTorch). The library allocates and frees no memory: scratch space is a
 *     caller-provided workspace whose size the matching *_workspace_size() call returns.
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL = legacy default
 *     stream). Outputs are valid once the stream has synchronised.
 *   - Arguments are validated on the host before any launch. On a validation error
 *     nothing is launched and EC_ERR_INVALID_ARG / EC_ERR_UNSUPPORTED is returned.
 *   - Data the host cannot see (positions, indices) is checked on the device. A bad
 *     element is skipped and a bit is OR-ed into the caller's device error word
 *     (`dev_err`, one int32, may be NULL); ec_read_device_error() reports it.
 *   - Shapes are in elements, tensors are dense row-major in the order written, and every
 *     base pointer must be 16-byte aligned.
 *   - bf16 means IEEE-754 binary32 truncated to its upper 16 bits (round-to-nearest-even
 *     when produced); fp32 is IEEE binary32. Entropies are in nats (natural logarithm).
 */
#ifndef ENTROPYCACHE_H_
#define ENTROPYCACHE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------------------- */
typedef int32_t ec_status;
#define EC_OK 0
#define EC_ERR_INVALID_ARG 1   /* a null pointer, a bad size, a misaligned pointer       */
#define EC_ERR_UNSUPPORTED 2   /* a valid request the library does not implement          */
#define EC_ERR_CUDA 3          /* a CUDA runtime/driver call failed                      */
#define EC_ERR_DEVICE_CHECK 4  /* a device-side bounds/consistency check fired           */
#define EC_ERR_TIMEOUT 5       /* a bounded device-side wait gave up                     */

/* Bits of the device error word. */
#define EC_DEVERR_BAD_CAND_POS 0x1  /* candidate position outside [0, L) or not masked   */
#define EC_DEVERR_BAD_IDX 0x2       /* recompute index outside [0, L)                    */
#define EC_DEVERR_BAD_R 0x4         /* recompute-set size outside [0, L]                 */
#define EC_DEVERR_TIMEOUT 0x8       /* a bounded pipeline wait ran out                   */

/* ---- logits element types ------------------------------------------------------------ */
#define EC_F32 0
#define EC_BF16 1

typedef void* ec_stream_t; /* a cudaStream_t */

/* ---- step parameters ------------------------------------------------------------------
 * B      sequences in the batch (1 <= B <= 4096)
 * L      positions per sequence, prompt + generation (1 <= L <= 1048576)
 * Hq     query heads; Hkv key/value heads; Hq % Hkv == 0 and Hq / Hkv <= 128
 *        (grouped-query attention: query head h reads key/value head h / (Hq / Hkv))
 * D      head dimension, 64 or 128
 * V      vocabulary size (1 <= V <= 2^30)
 * C_max  candidate rows per sequence: the masked positions of the current block whose
 *        logits the step receives (1 <= C_max <= min(L, 1024))
 * k      decode-history length: how many of the most recently decoded positions a
 *        partial step recomputes (1 <= k <= L)
 * n_dec  tokens committed per sequence per step (1 <= n_dec <= C_max): the n_dec most
 *        confident candidates
 * tau    entropy threshold in nats: a step whose decoded tokens' maximum entropy is
 *        strictly above tau triggers a full recompute
 * logits_dtype  EC_F32 or EC_BF16
 * conf_threshold  0 (or less): commit the n_dec most confident candidates. Greater than 0
 *        (at most 1): a confidence-threshold commit, a decoding variant that the pages leave
 *        open — of those n_dec, only the candidates whose decode confidence p(id) is at least
 *        conf_threshold are committed, and the single most confident one when none is. A
 *        zero-initialised struct gets the fixed-count commit.
 * scope_lo, scope_hi  the gate's scope, the same for every sequence of the call. Both 0: the
 *        whole sequence [0, L) (the EntropyCache step as the pages state it). Otherwise
 *        0 <= scope_lo < scope_hi <= L: block-by-block decoding (block diffusion) with the
 *        gate as a sub-block recompute signal, a use the pages name for the gate (zh summary
 *        §5 "通用性潜力"; pt summary §5 "Generalidade"). The block being decoded is
 *        [scope_lo, scope_hi) and the blocks after it do not exist yet, so:
 *          - candidates must lie in the scope (others are dropped, EC_DEVERR_BAD_CAND_POS);
 *          - a full step recomputes the scope: idx = scope_lo .. scope_hi - 1;
 *          - a partial step recomputes the scope's masked positions and those of the last
 *            min(k, count) history entries that lie in the scope;
 *          - attention reads the keys [0, scope_hi) only (block-causal: the block and every
 *            block before it).
 *        A zero-initialised struct gets the whole-sequence gate.
 */
typedef struct ec_params {
  int32_t B, L, Hq, Hkv, D, V, C_max, k, n_dec;
  float tau;
  int32_t logits_dtype;
  float conf_threshold;
  int32_t scope_lo, scope_hi;
} ec_params;

/* ---- per-sequence decode state (all device arrays, caller-owned) ----------------------
 * tokens     int32 [B, L]   committed token id per position (untouched where masked)
 * mask       uint8 [B, L]   1 = position still masked, 0 = decoded
 * ring       int32 [B, k]   decode history: ring[b, (head - 1 - t) mod k] is the t-th
 *                           most recently decoded position, for t < count
 * ring_head  int32 [B]      next ring slot to write
 * ring_count int32 [B]      entries held, saturating at k
 * dec_pos    int32 [B, n_dec]  positions committed by the last step, ascending, -1 padded
 * E          fp32  [B]      max entropy over the tokens committed by the last step
 * flag       uint8 [B]      1 = full recompute (E > tau or E is NaN), 0 = partial
 * idx        int32 [B, L]   recompute set in ascending position order; first R[b] valid
 * R          int32 [B]      recompute-set size
 * dev_err    int32 [1]      device error word (EC_DEVERR_* bits OR-ed in), may be NULL
 */
typedef struct ec_state {
  int32_t* tokens;
  uint8_t* mask;
  int32_t* ring;
  int32_t* ring_head;
  int32_t* ring_count;
  int32_t* dec_pos;
  float* E;
  uint8_t* flag;
  int32_t* idx;
  int32_t* R;
  int32_t* dev_err;
} ec_state;

/* ---- error reporting ------------------------------------------------------------------ */

/* Human-readable name of a status code; never NULL. */
const char* ec_status_string(ec_status st);

/* Synchronises `stream`, copies the device error word to *host_word (if non-NULL) and
 * returns EC_OK when it is zero, EC_ERR_TIMEOUT when the EC_DEVERR_TIMEOUT bit is set,
 * else EC_ERR_DEVICE_CHECK. Does not clear the word. */
ec_status ec_read_device_error(const int32_t* dev_err, int32_t* host_word, ec_stream_t stream);

/* Self-test of the failure path (the pages have no counterpart: it checks the library's own
 * timeout handling). Launches one CTA that waits, through the same bounded mbarrier wait every
 * kernel of the library uses, for a barrier phase that nothing completes. After limit_ns
 * nanoseconds (1 .. 10^10) the wait gives up, ORs EC_DEVERR_TIMEOUT into *dev_err and the
 * kernel returns normally; no asynchronous copy or tensor-core work is in flight, so the
 * context stays usable. ec_read_device_error() then reports EC_ERR_TIMEOUT.
 * EC_ERR_INVALID_ARG for a NULL dev_err or a limit out of range. */
ec_status ec_selftest_bounded_wait(int32_t* dev_err, uint64_t limit_ns, ec_stream_t stream);

/* A measurement aid with no counterpart in the pages: reads `bytes` bytes of the device buffer
 * `buf` in the launch shape of the entropy decode's split launch (one 256-thread CTA per 16 KB,
 * four 16-byte streaming loads per thread, all in flight at once) and nothing else, so that its
 * time is the floor for the decode's read of the same bytes. sink: one device word, written
 * only in the practically impossible case that the folded words equal a fixed constant (it
 * keeps the loads). buf 16-byte aligned, bytes a multiple of 16. */
ec_status ec_read_floor(const void* buf, size_t bytes, uint32_t* sink, ec_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
int32_t ec_version(void);

/* ---- (a) fused softmax / argmax decode / entropy ---------------------------------------
 * Follows the decode-and-entropy stage of the EntropyCache workflow (zh summary §2.2: the
 * new tokens are decoded from the logits and the entropy -sum_j p_ij log p_ij of each is
 * evaluated; pt summary §2 "Fluxo de Funcionamento"), per row i:
 *   m_i = max_j x_ij, ids[i] = the LOWEST j with x_ij == m_i (greedy decode),
 *   p_ij = exp(x_ij - m_i) / sum_j exp(x_ij - m_i)   (softmax at temperature 1),
 *   entropy[i]  = -sum_j p_ij ln p_ij  (0 ln 0 = 0),
 *   log_conf[i] = ln p_{i, ids[i]}     (log-probability of the decoded token).
 * logits     [n_rows, row_stride] of `dtype` (EC_F32 / EC_BF16); the first V entries of
 *            each row are read. row_stride >= V and row_stride * elem_size % 16 == 0.
 * ids        int32 [n_rows]; entropy, log_conf fp32 [n_rows].
 * ws         workspace of at least ec_entropy_decode_workspace_size(n_rows, V, dtype)
 *            bytes (16-byte aligned); no initial contents are needed. Calls that share a
 *            workspace must not overlap in time.
 * Accumulation is fp32; argmax compares the raw stored values, so ids are exact. -inf
 * logits contribute zero probability. NaN logits are not supported (results undefined).
 * n_rows == 0 is a valid no-op. */
size_t ec_entropy_decode_workspace_size(int32_t n_rows, int32_t V, int32_t dtype);
ec_status ec_entropy_decode(const void* logits, int64_t row_stride, int32_t n_rows, int32_t V,
                            int32_t dtype, int32_t* ids, float* entropy, float* log_conf,
                            void* ws, size_t ws_bytes, ec_stream_t stream);

/* ---- (a) without a workspace, for callers that cannot allocate -------------------------
 * The paper has no counterpart to this entry point: it is a deployment convenience.
 * Same computation, arguments and results as ec_entropy_decode, minus the workspace. It is
 * for callers that hold only their input and output buffers and cannot allocate device
 * memory: a plugin or custom-op interface of a serving runtime that passes an op its tensors
 * but no allocator, or latency-critical code that must not call cudaMalloc because it
 * synchronises the whole device.
 * Scratch lives in a library-owned static device array of EC_NOALLOC_SCRATCH_BYTES (1 MiB)
 * that every GPU which loads the library holds until the process exits. A request that
 * needs more (ec_entropy_decode_workspace_size(n_rows, V, dtype) > EC_NOALLOC_SCRATCH_BYTES,
 * e.g. more than about 4000 rows of a 126464-entry bf16 vocabulary) returns
 * EC_ERR_UNSUPPORTED and launches nothing.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current): make that first call before any stream capture. The address is
 * kept for the life of the process; cudaDeviceReset() on a device invalidates it, so do not
 * call this entry point on a device after resetting it.
 * Every call shares the one array, which keeps the last call's contents; no call needs it to
 * start in any particular state (every partial result a call reads is one it wrote first).
 * Calls whose executions overlap on the GPU (other streams, other host threads) race and give
 * wrong results: order them. No cudaMalloc, cudaFree or allocating library routine is called. */
#define EC_NOALLOC_SCRATCH_BYTES (1u << 20)
ec_status ec_entropy_decode_noalloc(const void* logits, int64_t row_stride, int32_t n_rows, int32_t V,
                                    int32_t dtype, int32_t* ids, float* entropy, float* log_conf,
                                    ec_stream_t stream);

/* ---- (a) from the hidden states: output projection fused with the decode ---------------
 * Stage (a) of the step (EntropyCache, gist.science zh summary §2.2: decode each masked
 * candidate and take the entropy of its softmax) applied to logits that are computed here
 * and never stored: logits[r, v] = sum_k hidden[r, k] * weight[v, k], accumulated in fp32
 * from bf16 products on the tensor cores. The pages leave this product to the model (its
 * output projection); fusing it with the decode has no counterpart in the pages.
 *   hidden  [n_rows, d_model] bf16, row-major, contiguous, 16-byte aligned (device).
 *   weight  [V, d_model] bf16, row-major, contiguous, 16-byte aligned (device).
 *   ids, entropy, log_conf [n_rows]: as ec_entropy_decode (greedy id, lowest index on ties;
 *            entropy in nats; ln of the decoded token's probability).
 *   ws       device workspace of ec_lm_head_entropy_workspace_size(n_rows) bytes, 16-byte
 *            aligned; no initial contents needed. Calls sharing a workspace must not overlap.
 * 1 <= n_rows <= 256; d_model a multiple of 64 (64 .. 65536); 1 <= V <= 2^30.
 * EC_ERR_INVALID_ARG for a bad argument (nothing launched). A wait inside the kernel that
 * gives up (never expected) makes the affected rows' entropy NaN. */
size_t ec_lm_head_entropy_workspace_size(int32_t n_rows);
ec_status ec_lm_head_entropy(const void* hidden, const void* weight, int32_t n_rows, int32_t d_model, int32_t V,
                             int32_t* ids, float* entropy, float* log_conf, void* ws, size_t ws_bytes,
                             ec_stream_t stream);

/* ---- (b)+(c) commit, max-entropy gate, decode history, recompute set -------------------
 * Follows the skip decision and selection stage of the workflow (zh summary §2.2: full
 * recompute iff E_{t+1} = max over newly decoded tokens of their entropy exceeds tau,
 * else reuse the cache except the current masked tokens and the k most recently decoded
 * tokens, taken from a decode history; §2.3: O(k) memory for the history; pt summary §2
 * "Decisão de Pulo", "Histórico de Decodificação"). Per sequence b:
 *   1. D = the n_dec candidates i < cand_count[b] with the largest log_conf (a NaN
 *      log_conf ranks lowest; ties go to the smaller position cand_pos[b, i]).
 *   2. tokens[b, cand_pos] = ids, mask[b, cand_pos] = 0 for i in D; dec_pos[b] = the
 *      positions of D ascending, -1 padded.
 *   3. E[b] = max over D of entropy (0 when D is empty); flag[b] = E[b] > tau, or 1 when
 *      E[b] is NaN.
 *   4. The positions of D are pushed onto the ring in ascending order (count saturates
 *      at k).
 *   5. flag = 1: idx[b] = 0..L-1, R[b] = L. flag = 0: idx[b] = the ascending list of
 *      positions p with mask[b, p] = 1 (after step 2) or p among the last min(k, count)
 *      ring entries; R[b] = its length.
 * cand_pos   int32 [B, C_max]; cand_count int32 [B] (0 <= count <= C_max).
 * ids, entropy, log_conf  as produced by ec_entropy_decode for the B*C_max rows
 *            (row b*C_max + i belongs to cand_pos[b, i]).
 * A candidate position outside [0, L) or not masked sets EC_DEVERR_BAD_CAND_POS and is
 * dropped from the candidate list; a bad cand_count is clamped to [0, C_max] and sets
 * EC_DEVERR_BAD_R. */
ec_status ec_select_recompute(const ec_params* p, const ec_state* st, const int32_t* cand_pos,
                              const int32_t* cand_count, const int32_t* ids,
                              const float* entropy, const float* log_conf, ec_stream_t stream);

/* ---- candidates for block-wise and sliding-window decoding -------------------------------
 * The pages note that the entropy gate carries over to other decoding strategies, such as
 * sliding-window and block decoding (pt summary §5 "Generalidade"; zh summary §5). A step's
 * candidates (the rows whose logits it decodes: cand_pos / cand_count of ec_step) are the
 * masked positions of the window being decoded; this builds them on the device from
 * st->mask, so that a multi-step decoding loop needs no host round trip. Per sequence b:
 *   EC_CAND_BLOCK    window [start, start + width): the block starting at `start`;
 *   EC_CAND_SLIDING  window [f, f + width), f = the first masked position at or after
 *                    `start` (L if none): a window that slides forward as its earliest
 *                    position is decoded;
 *   cand_pos[b, 0 .. n-1] = the masked positions of the window (clipped to [0, L)),
 *   ascending; cand_pos[b, n .. C_max-1] = -1; cand_count[b] = n.
 * 0 <= start < L, 1 <= width <= C_max. cand_pos int32 [B, C_max], cand_count int32 [B]
 * (device). Only st->mask is read. */
#define EC_CAND_BLOCK 0
#define EC_CAND_SLIDING 1
ec_status ec_candidates(const ec_params* p, const ec_state* st, int32_t mode, int32_t start, int32_t width,
                        int32_t* cand_pos, int32_t* cand_count, ec_stream_t stream);

/* ---- (c) K/V cache refresh ---------------------------------------------------------------
 * Recomputed positions receive fresh K/V, all other positions keep their cached rows
 * (zh summary §2.2, partial forward: only the recompute set is recomputed, the rest is
 * read from the cache; a full forward refreshes every row). For r < R[b]:
 *   k_cache[b, idx[b, r], :, :] = k_new[b, src_row, :, :]   (same for v)
 * where src_row = r when src_by_position == 0 (k_new holds the fresh rows in recompute
 * order) and src_row = idx[b, r] when src_by_position == 1 (k_new is indexed by position).
 * k_cache, v_cache  bf16 [B, L, Hkv, D]; k_new, v_new bf16 [B, L, Hkv, D].
 * idx int32 [B, L], R int32 [B] on the device. An idx outside [0, L) sets
 * EC_DEVERR_BAD_IDX and that row is skipped; R outside [0, L] sets EC_DEVERR_BAD_R and
 * that sequence is skipped. k_new/v_new must not overlap the caches, nor the two caches
 * each other (checked on the host over the [B, L, Hkv, D] extents: EC_ERR_INVALID_ARG). */
ec_status ec_kv_scatter(const ec_params* p, void* k_cache, void* v_cache, const void* k_new,
                        const void* v_new, int32_t src_by_position, const int32_t* idx,
                        const int32_t* R, int32_t* dev_err, ec_stream_t stream);

/* ---- (d) partial (or full) bidirectional attention ---------------------------------------
 * Attention of the recompute rows against every cached row, with no causal mask (dLLMs
 * attend bidirectionally: zh summary §1; pt summary §1 "Atenção Bidirecional"). For
 * b < B, r < R[b], query head h (g = Hq / Hkv, kv head = h / g):
 *   s_j = scale * <q[b, r, h, :], k_cache[b, j, h/g, :]>   for j < L
 *   out[b, r, h, :] = sum_j softmax(s)_j * v_cache[b, j, h/g, :]
 * With R[b] = L and q in position order this is dense bidirectional attention (the full
 * recompute of the pt summary §2 "Decisão de Pulo").
 * q, out  bf16 [B, L, Hq, D] (rows in recompute order, first R[b] valid; rows >= R[b]
 *         of out are not written); k_cache, v_cache bf16 [B, L, Hkv, D].
 * R       int32 [B] on the device (read by the kernel: no host synchronisation).
 * scale   softmax scale, normally 1/sqrt(D).
 * ws      at least ec_partial_attention_workspace_size(p) bytes (reserved: the key-split
 *         merge runs in on-chip shared memory of a 4-CTA cluster).
 * Products run on bf16 tensor cores with fp32 accumulation; probabilities are rounded to
 * bf16 before the PV product. A pipeline wait that exceeds its limit sets
 * EC_DEVERR_TIMEOUT in dev_err (if given) and leaves that tile unwritten. out must not
 * overlap q, k_cache or v_cache (checked on the host over the extents above:
 * EC_ERR_INVALID_ARG). */
size_t ec_partial_attention_workspace_size(const ec_params* p);
ec_status ec_partial_attention(const ec_params* p, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* R, float scale, void* out,
                               void* ws, size_t ws_bytes, int32_t* dev_err, ec_stream_t stream);

/* ---- (d) dense attention for a step known to be full --------------------------------------
 * Every position attends to every cached key (the full recompute of the pt summary §2
 * "Decisão de Pulo"; no mask, zh summary §1). The same result as ec_partial_attention with
 * R[b] = L and q in position order, for the steps a caller knows are full before they run
 * (the first forward of each generation block is full by definition): each CTA takes two
 * 128-row query tiles that share every K/V block, with a softmax warpgroup per tile, so one
 * tile's softmax overlaps the other's tensor-core products. For b < B, position r < L, query
 * head h (kv head h / (Hq / Hkv)):
 *   out[b, r, h, :] = sum_j softmax_j(scale * <q[b, r, h, :], k_cache[b, j, h/g, :]>) v_cache[b, j, h/g, :]
 * q, out bf16 [B, L, Hq, D]; k_cache, v_cache bf16 [B, L, Hkv, D]; D = 128 (other head
 * sizes return EC_ERR_UNSUPPORTED). No workspace. Rounding as ec_partial_attention. A
 * pipeline wait that exceeds its limit sets EC_DEVERR_TIMEOUT in dev_err (if given). out
 * must not overlap q, k_cache or v_cache (EC_ERR_INVALID_ARG). */
ec_status ec_dense_attention(const ec_params* p, const void* q, const void* k_cache, const void* v_cache,
                             float scale, void* out, int32_t* dev_err, ec_stream_t stream);

/* ---- the partial forward of one transformer layer ------------------------------------------
 * The forward pass the step's flag selects (EntropyCache, gist.science zh summary §2.2,
 * "前向传播 / 部分传播"): a partial forward recomputes only the recompute set (idx, R as
 * built by ec_select_recompute) and reads every other position from the K/V cache; with the
 * full set (R = L) it is the full forward. The layer is the LLaMA-style block of the models the
 * pages evaluate (LLaDA-8B, Dream-7B; the pages name the models, not their layers). For each
 * sequence b and recompute row r < R[b] at position p = idx[b, r]:
 *   x = x_src[b, p];  h = RMSNorm(x) * gamma1           (x / sqrt(mean(x^2) + eps))
 *   q = h wq^T, k = h wk^T, v = h wv^T; q and k rotated by RoPE at position p (rotate-half:
 *       feature i and i + D/2 of a head turn by the angle p * theta^(-2i/D), from rope_cos /
 *       rope_sin, see ec_rope_table)
 *   k_cache[b, p] = k, v_cache[b, p] = v                 (the K/V refresh of the recompute set)
 *   o = attention of q against the whole cache (as ec_partial_attention, scale 1/sqrt(D); with
 *       a gate scope, the keys [0, scope_hi))
 *   x2 = x + o wo^T;  h2 = RMSNorm(x2) * gamma2;  y[b, r] = x2 + (SiLU(h2 wg^T) * (h2 wu^T)) wd^T
 * Shapes (params p: B, L, Hq, Hkv, D; d = Hq * D is the model width):
 *   wq [Hq D, d], wk and wv [Hkv D, d], wo [d, Hq D], wg and wu [d_ff, d], wd [d, d_ff],
 *   gamma1 and gamma2 [d]: bf16, row-major (out, in), 16-byte aligned;
 *   rope_cos, rope_sin fp32 [L, D / 2];  x_src bf16 [B, L, d] (position-indexed layer input);
 *   k_cache, v_cache bf16 [B, L, Hkv, D];  y bf16 [B, L, d] (rows in recompute order, the
 *   first R[b] written);  idx int32 [B, L], R int32 [B] on the device (no host synchronisation).
 * d % 128 == 0, d <= 8192, (Hkv D) % 128 == 0, d_ff % 64 == 0; eps > 0.
 * Products on bf16 tensor cores with fp32 accumulation; every intermediate (h, q, k, v, o, x2,
 * h2, the SwiGLU output) is rounded to bf16. ws: ec_layer_forward_workspace_size(p, d_ff)
 * bytes, no initial contents needed. */
typedef struct ec_layer {
  int32_t d_ff;
  float eps;
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  const void *gamma1, *gamma2;
  const float *rope_cos, *rope_sin;
} ec_layer;

size_t ec_layer_forward_workspace_size(const ec_params* p, int32_t d_ff);
ec_status ec_layer_forward(const ec_params* p, const ec_layer* w, const int32_t* idx, const int32_t* R,
                           const void* x_src, void* k_cache, void* v_cache, void* y, void* ws, size_t ws_bytes,
                           int32_t* dev_err, ec_stream_t stream);

/* The RoPE table of ec_layer_forward: cos and sin of pos * theta^(-2i / D) for pos < L and
 * i < D / 2, computed on the device in double precision and stored as fp32 [L, D / 2].
 * 1 <= L, D even (2 .. 256), theta > 0. */
ec_status ec_rope_table(int32_t L, int32_t D, float theta, float* rope_cos, float* rope_sin, ec_stream_t stream);

/* ---- one whole denoising step ---------------------------------------------------------------
 * Runs the three stages of the workflow in order (zh summary §2.2): (a) decode and
 * entropy over the B*C_max candidate rows of `logits` ([B, C_max, V], row stride V);
 * (b)+(c) the gate and recompute set, updating `st`; then, for each of n_layers layers,
 * the K/V refresh of the recompute set from the position-indexed fresh rows k_src[l],
 * v_src[l] (bf16 [B, L, Hkv, D]) into k_cache[l], v_cache[l], the gather of the recompute
 * rows' queries from q_src[l] (bf16 [B, L, Hq, D], position-indexed) and the attention of
 * those rows against the refreshed cache into out[l] (bf16 [B, L, Hq, D], recompute
 * order). One flag and one recompute set serve every layer (zh summary §2.3: the decision
 * is independent of depth). The flag computed from this step's logits governs this
 * call's attention stage, which stands for the next forward pass of the workflow.
 * The pointer arrays k_cache ... out are HOST arrays of n_layers device pointers. Within a
 * layer, out must not overlap q_src, k_cache or v_cache, and neither cache may overlap the
 * other or the fresh rows (EC_ERR_INVALID_ARG).
 * cand_pos, cand_count: as for ec_select_recompute.
 * ws at least ec_step_workspace_size(p) bytes (16-byte aligned, no initial contents needed).
 * scale as for ec_partial_attention. With tau < 0, no scope and D = 128 every step is full
 * (entropies are non-negative), so the attention runs on the kernel of ec_dense_attention,
 * reading q_src[l] in place (the recompute order is the position order); otherwise on the
 * kernel of ec_partial_attention, from the gathered queries. */
size_t ec_step_workspace_size(const ec_params* p);
ec_status ec_step(const ec_params* p, const ec_state* st, const void* logits,
                  const int32_t* cand_pos, const int32_t* cand_count, int32_t n_layers,
                  void* const* k_cache, void* const* v_cache, const void* const* k_src,
                  const void* const* v_src, const void* const* q_src, void* const* out,
                  float scale, void* ws, size_t ws_bytes, ec_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* ENTROPYCACHE_H_ */
