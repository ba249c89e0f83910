/*
 * moe.h -- C ABI of libmoe: one routed Mixture-of-Experts layer over MLX-style
 * affine group-quantised weights, on one B300 (sm_103a).
 *
 * The operation (from the pages of the TurboFieldfare write-ups; pages are named
 * by title and section):
 *   - weights are affine 4-bit, group 64, w = scale * q + bias with fp16 scale and
 *     bias; the router is 8-bit ("TurboFieldfare esegue Mac Gemma 4 26B in 2 GB...",
 *     section "L'affermazione dei 2 GB trasforma la larghezza di banda dell'SSD nel
 *     nuovo vincolo"; "Correr un modelo de 26.000 millones...", section "Detalles
 *     tecnicos y rendimiento");
 *   - per token the router picks 8 experts; an always-on shared expert runs beside
 *     them and both branches are combined ("Come eseguire un modello da 26
 *     miliardi...", section "Qual e il trucco principale dell'architettura";
 *     remio.ai page, section "Mac Gemma 4 26B entra nello spazio disponibile...");
 *   - prefill runs in chunks of up to 128 tokens so that one expert load serves
 *     many rows (devtrends page, section "Prestazioni nel mondo reale");
 *   - a 16-slot least-frequently-used expert cache per layer, refilled while the
 *     shared expert computes (devtrends page, "Qual e il trucco principale...").
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented as "device" are CUDA device pointers owned
 *     by the caller; the library never frees them.  Host pointers are named h_*.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are stream-ordered and return before the GPU finishes, except where a
 *     call says it synchronises.
 *   - Every call returns an int status (MOE_OK = 0).  Arguments are checked on the
 *     host before anything is launched; a rejected call launches nothing.  No C++
 *     exception crosses this boundary.
 *   - Matrices are row-major.  A 4-bit matrix [N][K] is stored as
 *       q     uint32 [N][K/8]   element j of a row = bits 4*(j%8) of word j/8
 *       scale fp16   [N][K/64]  (raw IEEE binary16 bits in uint16_t)
 *       bias  fp16   [N][K/64]
 *     An 8-bit matrix is the same with q uint32 [N][K/4], element j = byte j%4 of
 *     word j/4.  K must be a multiple of 64.
 *   - All fp32 outputs are accumulated in fp32; results are deterministic (no
 *     floating-point atomics).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
#define MOE_OK 0
#define MOE_EINVAL 1     /* bad shape, size, flag or NULL pointer */
#define MOE_ECUDA 2      /* a CUDA runtime call failed */
#define MOE_ECAPACITY 3  /* more distinct experts requested than cache slots */
#define MOE_ETIMEOUT 4   /* a bounded device-side wait gave up */
#define MOE_EWORKSPACE 5 /* workspace missing or smaller than moe_workspace_bytes */
#define MOE_ENOTREADY 6  /* handle not initialised for this use */

MOE_API const char *moe_status_string(int status);

/* flags for moe_layer_decode / moe_layer_prefill_chunk */
#define MOE_RESIDUAL 1 /* y = x + MoE(x) instead of y = MoE(x) */
#define MOE_PRENORM 2  /* the layer reads RMSNorm(x) (layer->norm_w, norm_eps) instead of x;
                          with MOE_RESIDUAL: y = x + MoE(RMSNorm(x)), the pre-norm block */

#define MOE_GROUP 64
#define MOE_MAX_TOPK 8
#define MOE_MAX_EXPERTS 256
#define MOE_MAX_DECODE_TOKENS 16
#define MOE_MAX_PREFILL_TOKENS 128
#define MOE_MAX_CACHE_SLOTS 64

/* ---------------------------------------------------------------- layout */

/*
 * MLX layout of one expert (the interchange form; what affine_quantise writes):
 * one contiguous blob
 *   gu_q [2I][H/8] u32 | gu_s [2I][H/64] f16 | gu_b [2I][H/64] f16 |
 *   d_q  [H][I/8]  u32 | d_s  [H][I/64]  f16 | d_b  [H][I/64]  f16
 * The gate/up matrix holds the I gate rows first, then the I up rows.  Every
 * part starts on a 256-byte boundary; the blob size is a multiple of 256.
 * moe_expert_blob_offsets writes the six byte offsets.  Returns 0 for bad shapes.
 */
MOE_API size_t moe_expert_blob_bytes(int H, int I);
MOE_API int moe_expert_blob_offsets(int H, int I, size_t offsets_out[6]);

/*
 * Tile layout of one expert (the form the layer kernels read, and the unit a
 * cache slot holds).  The same codes, scales and biases in another order; the
 * pages give no storage layout, this one is the library's own.  A tile is 16
 * matrix rows by one group of 64 columns, 576 bytes (4.5 bits per weight):
 *   bytes 16L..16L+15, lane L = 4r + c (r = 0..7, c = 0..3): words 2c and 2c+1
 *     of the group in row a(r), then the same two words of row b(r);
 *   bytes 512+8r..512+8r+7: fp16 scale, bias of row a(r), scale, bias of row b(r).
 * Gate/up part at byte 0: tile (it, g) at 576 (it H/64 + g) for it < I/8,
 *   g < H/64, with a(r) = gate row 8it + r and b(r) = up row 8it + r.
 * Down part at byte 576 (I/8)(H/64): tile (rt, g) at 576 (rt I/64 + g) from
 *   its start, rt < H/16, g < I/64, with a(r) = row 16rt + r, b(r) = row 16rt+8+r.
 * moe_tile_blob_bytes: the blob size (a multiple of 256), 0 for bad shapes
 * (H must be a multiple of 128, I of 64).
 * moe_expert_tile: converts one expert from the MLX layout (device, at least
 * moe_expert_blob_bytes(H, I) bytes) to the tile layout (device, at least
 * moe_tile_blob_bytes(H, I) bytes, not overlapping the source); stream-ordered.
 */
MOE_API size_t moe_tile_blob_bytes(int H, int I);
MOE_API int moe_expert_tile(const void *mlx_blob, int H, int I, void *tile_blob, void *stream);

/*
 * A layer.  All pointers are device pointers owned by the caller.
 *   H hidden size, E experts (<= MOE_MAX_EXPERTS), topk (1..MOE_MAX_TOPK),
 *   I routed-expert intermediate size, Is shared-expert intermediate size;
 *   H a multiple of 128 (at most 4096 for the layer calls), I and Is multiples
 *   of 64.
 *   r_q/r_s/r_b: 8-bit router matrix [E][H] (MLX layout, 16-byte aligned).
 *   experts: E tile-layout blobs of shape (H, I), blob e at experts + e * expert_stride
 *     (256-byte aligned; expert_stride a multiple of 256 and >= moe_tile_blob_bytes(H, I)).
 *     May be NULL when a cache supplies the experts.
 *   shared: one tile-layout blob of shape (H, Is), 256-byte aligned.
 *   logit_bias: optional fp32 [E] added to the router logits (NULL = none).
 *   norm_w, norm_eps: the RMSNorm in front of the layer (used with MOE_PRENORM):
 *     RMSNorm(x)[j] = x[j] * norm_w[j] / sqrt(mean over j of x[j]^2 + norm_eps).
 */
typedef struct moe_layer {
    int H, E, topk, I, Is;
    const uint32_t *r_q;
    const uint16_t *r_s, *r_b;
    const void *experts;
    size_t expert_stride;
    const void *shared;
    const float *logit_bias;
    const float *norm_w; /* RMSNorm weight, fp32 [H], device; read with MOE_PRENORM only */
    float norm_eps;      /* RMSNorm epsilon (>= 0) */
} moe_layer_t;

/* ---------------------------------------------------------------- workspace */

/*
 * Scratch for moe_route / moe_layer_decode / moe_layer_prefill_chunk on up to
 * T_max tokens (T_max <= MOE_MAX_PREFILL_TOKENS).  The caller allocates it on the
 * device (256-byte aligned) and must zero it once with moe_workspace_init before
 * first use; every call leaves it ready for the next one, whatever the layer, so
 * one workspace sized for the largest layer and T_max can serve several layers
 * in turn.  One workspace serves one call at a time: calls that overlap on the
 * GPU must use different workspaces.  Returns 0 for an invalid layer or T_max.
 */
MOE_API size_t moe_workspace_bytes(const moe_layer_t *layer, int T_max);
MOE_API int moe_workspace_init(void *d_ws, size_t ws_bytes, void *stream);

/*
 * Synchronises `stream`, then reports whether a device-side wait of an earlier
 * call on this workspace gave up (MOE_ETIMEOUT) and re-initialises the workspace
 * in that case (zeroes it and waits for the device).  MOE_OK otherwise.  Outputs
 * of a call whose wait gave up are undefined.
 */
MOE_API int moe_workspace_status(void *d_ws, size_t ws_bytes, void *stream);

/*
 * The part of the workspace that moe_route and moe_layer_decode use for up to
 * T_max tokens (1..MOE_MAX_DECODE_TOKENS): a caller that never runs a prefill
 * chunk may allocate only this many bytes.  Returns 0 for an invalid layer or
 * T_max.  (moe_workspace_bytes covers the prefill chunk as well.)
 */
MOE_API size_t moe_decode_workspace_bytes(const moe_layer_t *layer, int T_max);

/* ---------------------------------------------------------------- kernels */

/*
 * Affine quantiser (encoding used to build packed weights): for each row and
 * group of 64, s = fp16((max-min)/(2^bits-1)), b = fp16(min),
 * q = clamp(rint((w - b)/s), 0, 2^bits-1) in fp32 (q = 0 when s == 0).
 * w: device fp32 [N][K]; q/s/b: device outputs in the layout above.
 * bits is 4 or 8.  The MLX affine format is named by the remio.ai page, section
 * "L'affermazione dei 2 GB...".
 */
MOE_API int affine_quantise(const float *w, int N, int K, int bits, uint32_t *q, uint16_t *s, uint16_t *b,
                    void *stream);

/*
 * One 4-bit quantised GEMV, y[n] = sum_j (s[n][j/64] q[n][j] + b[n][j/64]) x[j]
 * (the "quantised GEMV" kernel of the devtrends page, section "Senza dipendenze
 * da llama.cpp e MLX").  q/s/b device [N][K] 4-bit; x device fp32 [K];
 * y device fp32 [N].  N >= 1, K a multiple of 64; q and x 16-byte aligned.
 * With N a multiple of 16, K <= 8192 and s, b, y 16-byte aligned as well, the
 * rows are read by bulk copies into shared memory, 16 rows per CTA; otherwise by
 * plain loads.  fp16 x as the tensor-core operand, fp32 accumulation.
 */
MOE_API int qgemv_affine4(const uint32_t *q, const uint16_t *s, const uint16_t *b, int N, int K,
                  const float *x, float *y, void *stream);

/*
 * RMSNorm of T rows (T >= 1) of H values (H a multiple of 4):
 *   y[t][j] = x[t][j] * w[j] / sqrt(mean over j of x[t][j]^2 + eps)
 * The pages list an RMSNorm kernel among the engine's own kernels (devtrends page
 * "Come eseguire un modello da 26 miliardi...", section "Senza dipendenze da
 * llama.cpp e MLX"; iitog.ru page "TurboFieldfare: движок с открытым кодом...");
 * this is the plain root-mean-square normalisation.  x, w, y: device fp32 (x and y
 * [T][H], w [H]); y may alias x.  fp32 arithmetic.  The layer calls apply the same
 * normalisation inside their kernels with the MOE_PRENORM flag.
 */
MOE_API int moe_rmsnorm(const float *x, const float *w, float eps, int T, int H, float *y, void *stream);

/*
 * One token per row of vocabulary logits (the engine samples with temperature,
 * top-K and top-P, defaults 0.2, 64 and 0.95: elsolitario.org "Correr un modelo de
 * 26.000 millones...", section "Como empezar"; the pages give the parameters, the
 * order of the steps is this library's plain reading):
 *   1. keep the top_k largest logits, larger first, equal -> lower index (top_k <= 0
 *      or >= V keeps all V);
 *   2. softmax of the kept logits at the temperature;
 *   3. keep the shortest prefix, in that order, whose probability reaches top_p
 *      (at least one token; top_p = 1 keeps all);
 *   4. return the first kept token whose cumulative weight exceeds u[t] times the
 *      prefix's total.
 * temperature <= 0 is greedy (the largest logit, equal -> lower index).
 * logits: device fp32 [T][V]; u: device fp32 [T], uniform numbers in [0, 1) that
 * the caller draws (the library has no random state); tokens: device int32 [T].
 * T >= 1, V >= 1, 0 < top_p <= 1; with temperature > 0 at most 1024 tokens may
 * survive top-K (MOE_EINVAL otherwise).  fp32 arithmetic, deterministic.
 */
#define MOE_SAMPLE_MAX_K 1024
MOE_API int moe_sample(const float *logits, int T, int V, float temperature, int top_k, float top_p,
                       const float *u, int32_t *tokens, void *stream);

/*
 * Router on T tokens (1..MOE_MAX_PREFILL_TOKENS): logits = deq(Wr) x (+ bias),
 * idx = the topk largest logits, larger first, equal -> lower expert index;
 * gate = softmax over the chosen logits.  x device fp32 [T][H]; idx device int32
 * [T][topk]; gate device fp32 [T][topk]; logits (optional, NULL = not written)
 * device fp32 [T][E].  (devtrends page, "Qual e il trucco principale..."; remio.ai
 * page, "L'affermazione dei 2 GB...".)
 */
MOE_API int moe_route(const moe_layer_t *layer, const float *x, int T, int32_t *idx, float *gate,
              float *logits, void *d_ws, size_t ws_bytes, void *stream);

typedef struct moe_cache moe_cache_t;

/*
 * Decode step on T = 1..MOE_MAX_DECODE_TOKENS independent tokens (the per-token
 * MoE layer the pages describe: an 8-bit router choosing 8 experts per token, an
 * always-on shared expert, both branches summed -- devtrends page "Come eseguire
 * un modello da 26 miliardi...", section "Qual e il trucco principale
 * dell'architettura"; remio.ai page "TurboFieldfare esegue Mac Gemma 4 26B in
 * 2 GB...", sections "Mac Gemma 4 26B entra nello spazio disponibile..." and
 * "L'affermazione dei 2 GB trasforma la larghezza di banda dell'SSD nel nuovo
 * vincolo"; 4-bit affine group-64 weights per elsolitario.org "Correr un modelo
 * de 26.000 millones...", section "Detalles tecnicos y rendimiento"):
 *   y_t = sum_k gate_tk * expert_{idx_tk}(x_t) + shared(x_t)   (+ x_t with MOE_RESIDUAL)
 * expert(x) = Wd (gelu_tanh(Wg x) * (Wu x)).  With MOE_PRENORM the router and the
 * experts read RMSNorm(x) (see moe_rmsnorm) while MOE_RESIDUAL adds the raw x.  Every
 * distinct expert is read once
 * for all the tokens that chose it.  x, y: device fp32 [T][H] (y must not alias
 * x).  idx_out / gate_out: optional device outputs [T][topk].
 * cache == NULL: experts come from layer->experts; the call does not synchronise.
 * cache != NULL: experts come from the cache's device slots; the router writes the
 *   routing into page-locked host memory mapped for the device and the call waits
 *   for it (polling; MOE_ETIMEOUT after 5 s), runs the LFU policy, issues the
 *   missing experts' host->device copies on the cache's side stream while the
 *   shared expert runs on `stream`, and then computes the routed experts.  It
 *   returns once all work is enqueued (not finished).  MOE_ECAPACITY if the
 *   tokens request more distinct experts than the cache has slots.
 */
MOE_API int moe_layer_decode(const moe_layer_t *layer, const float *x, int T, int flags, float *y,
                     int32_t *idx_out, float *gate_out, moe_cache_t *cache, void *d_ws,
                     size_t ws_bytes, void *stream);

/*
 * Prefill chunk of T = 1..MOE_MAX_PREFILL_TOKENS tokens (the pages' prefill in
 * chunks of 128 tokens, so that one loaded expert serves many rows: devtrends
 * page "Come eseguire un modello da 26 miliardi...", section "Prestazioni nel
 * mondo reale"; remio.ai page, section "L'affermazione dei 2 GB..."; iitog.ru
 * page "TurboFieldfare: движок с открытым кодом..."): the same result as T
 * independent decodes (chunking only lets one expert load serve many rows).  The
 * tokens routed to each expert are gathered, multiplied on the tensor cores with
 * fp16 operands and fp32 accumulation, and scattered back through the gates.
 * Arguments as moe_layer_decode (no cache).
 */
MOE_API int moe_layer_prefill_chunk(const moe_layer_t *layer, const float *x, int T, int flags, float *y,
                            int32_t *idx_out, float *gate_out, void *d_ws, size_t ws_bytes,
                            void *stream);

/*
 * moe_layer_decode_host -- moe_layer_decode on HOST buffers: x_host (T x H fp32),
 * y_host (T x H fp32) and the optional idx_host / gate_host (T x topk) are host
 * memory; page-locked memory makes the copies asynchronous, pageable memory also
 * works.  The call copies x into the workspace (which holds device staging for x,
 * y and the routing), runs the decode step on `stream` (through `cache` when it is
 * non-null), copies y and the requested routing back, and waits for `stream`
 * (polling it, so the calling thread stays busy meanwhile) before it returns: the
 * outputs are ready on return.  Page-locked buffers that are mapped into the
 * device's address space (cudaHostAlloc memory, a pinned PyTorch tensor) skip the
 * DMA copies: a small kernel reads x from host memory and, without a cache, the
 * decode kernel writes y and the routing straight into host memory.  x_host and
 * y_host must not overlap.  Same workspace (moe_workspace_bytes) and error codes as
 * moe_layer_decode; MOE_ECUDA if a copy or the stream wait fails.
 */
MOE_API int moe_layer_decode_host(const moe_layer_t *layer, const float *x_host, int T, int flags,
                                  float *y_host, int32_t *idx_host, float *gate_host, moe_cache_t *cache,
                                  void *d_ws, size_t ws_bytes, void *stream);

/*
 * moe_host_call -- a prepared moe_layer_decode_host for a decode loop: the same
 * decode step (the routed MoE layer of moe_layer_decode; devtrends page, section
 * "Qual è il trucco principale dell'architettura") for one layer, workspace,
 * token count T (1..MOE_MAX_DECODE_TOKENS), flags and stream, all fixed when the
 * handle is created.  Creation allocates page-locked, device-mapped staging rows
 * for x and y (T x H fp32 each) and a completion word, and records the step -- x
 * read from its staging row into the workspace, the decode kernel writing y into
 * its staging row, the completion word set -- as a CUDA graph.
 *
 * moe_host_call_run copies x_host (T x H fp32, host memory) into the x row,
 * launches the graph on the stream, waits for the completion word (polling host
 * memory, the calling thread stays busy) and copies the y row to y_host: one
 * driver call per step.  moe_host_call_rows returns the two staging rows; a caller
 * may write x into the x row and read y from the y row and pass those rows to
 * moe_host_call_run, which then skips the copies.  Outputs are ready on return.
 *
 * The layer's weights, the workspace and the stream must stay valid while the
 * handle lives; a handle serves one thread at a time; a failed device wait is
 * reported by moe_workspace_status as for moe_layer_decode.  Errors: MOE_EINVAL
 * (arguments as moe_layer_decode, NULL handle or buffers), MOE_EWORKSPACE,
 * MOE_ECUDA (allocation, capture or launch failed, or the step ended without its
 * completion word), MOE_ETIMEOUT (no completion within 5 s).
 * moe_host_call_destroy waits for the stream and frees the handle (NULL is fine).
 */
typedef struct moe_host_call moe_host_call_t;
MOE_API int moe_host_call_create(moe_host_call_t **out, const moe_layer_t *layer, int T, int flags, void *d_ws,
                                 size_t ws_bytes, void *stream);
MOE_API int moe_host_call_run(moe_host_call_t *c, const float *x_host, float *y_host);
MOE_API int moe_host_call_rows(moe_host_call_t *c, float **x_row, float **y_row);
MOE_API int moe_host_call_destroy(moe_host_call_t *c);

/*
 * moe_layer_decode_noalloc -- the same decode step as moe_layer_decode (no cache),
 * for callers that cannot allocate device memory: for example a plug-in running
 * inside a host framework that reserves the GPU's memory through its own allocator
 * and forbids other cudaMalloc calls, or a latency-critical loop that may not
 * risk cudaMalloc's implicit device synchronisation.  The pages have no
 * counterpart to this call; it only changes where the scratch memory lives.
 *
 * It allocates nothing: its scratch is one file-scope device array of
 * MOE_NOALLOC_SCRATCH_BYTES inside libmoe, present on every GPU that loads the
 * library until the process exits.  The caller still supplies x, y and the
 * optional idx/gate outputs (device pointers, as in moe_layer_decode).
 *   - The first call on a device does a one-time set-up with that device
 *     current: it looks up the array's device address and zeroes the array
 *     (this synchronises the device).  Make that first call before any stream
 *     capture.  The set-up belongs to the device's primary context: it does not
 *     survive a reset of that context (cudaDeviceReset), after which this call
 *     must not be used again in the process.
 *   - Every call shares the one array, so calls that overlap on the GPU (two
 *     streams, or two host threads) race and give wrong results; serialise them.
 *     The array carries state from call to call: the decode's cumulative
 *     counters (each call starts from the values the previous call left) and
 *     the output-tile tickets, which each call returns to zero.
 *   - A device-side wait that gives up (a lost signal) raises an error word in
 *     the array; that call's outputs, and those of every later call, are
 *     undefined until moe_noalloc_status has seen it.  moe_noalloc_status
 *     synchronises `stream`, returns MOE_ETIMEOUT and zeroes the array if a wait
 *     gave up, and MOE_OK otherwise.  A caller that must know its result is good
 *     checks it after the call.
 *   - Returns MOE_EWORKSPACE when the layer at T tokens needs more scratch than
 *     MOE_NOALLOC_SCRATCH_BYTES; moe_decode_workspace_bytes tells how much it
 *     needs (the full-size layer, hidden 2816 with 128 experts, top-8, expert
 *     inter 704, shared inter 2112, needs 2,602,240 bytes at T = 16).  Other
 *     errors as moe_layer_decode.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)
MOE_API int moe_layer_decode_noalloc(const moe_layer_t *layer, const float *x, int T, int flags,
                                     float *y, int32_t *idx_out, float *gate_out, void *stream);
MOE_API int moe_noalloc_status(void *stream);

/* ---------------------------------------------------------------- LFU cache */

/*
 * The cache policy (the pages give "16 slots, LFU, per layer": devtrends page,
 * section "Qual e il trucco principale dell'architettura"; remio.ai page,
 * section "Mac Gemma 4 26B entra nello spazio disponibile..."; the tie rules are
 * this library's reading).  A step brings a request list R: the distinct
 * experts of the step in first-appearance order (token-major over the router's
 * choices).  Every resident expert in R is a hit (use count += 1, last use =
 * step).  Then every missing expert of R, in order, takes the lowest empty slot,
 * or else evicts the slot not holding a member of R with the smallest
 * (count, last use, slot); it starts at count 1, last use = step.  Counts are
 * forgotten on eviction.  More distinct experts than slots: MOE_ECAPACITY and no
 * change.  A repeated or out-of-range expert in R: MOE_EINVAL and no change.
 *
 * moe_lfu_*: the policy alone, on the host (no GPU needed).  slots <= 64,
 * E <= MOE_MAX_EXPERTS.  moe_lfu_step writes, per request, the slot now holding
 * it (slot_out) and whether it was a hit (hit_out); either may be NULL.
 * moe_lfu_state: expert per slot (-1 = empty), use counts, last-use steps,
 * running hit and miss totals; any output may be NULL.
 */
typedef struct moe_lfu moe_lfu_t;
MOE_API int moe_lfu_create(moe_lfu_t **out, int slots, int E);
MOE_API int moe_lfu_destroy(moe_lfu_t *lfu);
MOE_API int moe_lfu_step(moe_lfu_t *lfu, const int32_t *req, int n, int32_t *slot_out, uint8_t *hit_out);
MOE_API int moe_lfu_state(const moe_lfu_t *lfu, int32_t *expert_of_slot, uint32_t *counts, int64_t *last,
                          uint64_t *hits, uint64_t *misses);

/*
 * Per-layer expert cache on the current device: `slots` (<= 64) device slots of
 * moe_tile_blob_bytes(H, I) bytes, run by the policy above, filled from the E
 * tile-layout expert blobs the caller keeps in host memory at
 * h_experts + e * host_stride (page-locked memory is needed for the copies to
 * overlap compute; the library neither copies nor frees it).  The library
 * allocates the slot pool, a non-blocking side stream and two events, all
 * released by moe_cache_destroy (which first waits for the side stream).
 * Use one cache with calls issued in order on one stream.
 * moe_cache_slots: expert per slot (-1 = empty) and use counts.
 * moe_cache_stats: hits, misses and bytes copied host -> device so far.
 */
MOE_API int moe_cache_create(moe_cache_t **out, int H, int E, int I, const void *h_experts,
                             size_t host_stride, int slots);
MOE_API int moe_cache_destroy(moe_cache_t *cache);
MOE_API int moe_cache_slots(const moe_cache_t *cache, int32_t *expert_of_slot, uint32_t *counts);
MOE_API int moe_cache_stats(const moe_cache_t *cache, uint64_t *hits, uint64_t *misses,
                            uint64_t *h2d_bytes);

/*
 * Device-resident policy (enable = 1) or host policy (0, the default).  The pages
 * have the CPU schedule the expert reads while the GPU computes; with the policy on
 * the device a cached decode needs no host round trip:
 *   - the router's ranking CTA runs the policy step above on the device;
 *   - a fetch kernel copies the missing experts from the host blobs (read by the SMs
 *     through the blobs' device mapping) into their slots;
 *   - the decode kernel reads each expert's slot from device memory.
 * The call then returns without waiting for the GPU, like an uncached decode.  The
 * policy, its tie rules and its statistics are the same in both modes, and
 * switching carries the state over.
 * Enabling needs h_experts to be page-locked and mapped into the device's address
 * space (cudaHostGetDevicePointer succeeds on it; memory from cudaHostAlloc or a
 * pinned PyTorch tensor is), else MOE_EINVAL.  With the device policy a call needs
 * T * topk <= slots (the request list then always fits; MOE_ECAPACITY otherwise).
 * moe_cache_slots and moe_cache_stats wait for the device (cudaDeviceSynchronize)
 * before they read a device-resident state.  Switching waits as well.
 */
MOE_API int moe_cache_set_device_policy(moe_cache_t *cache, int enable);

/* ---------------------------------------------------------------- tests */

/*
 * Fault injection for tests of the error paths (the pages have no counterpart).
 * The next eligible call consumes the injection:
 *   MOE_INJECT_WAIT  the next moe_layer_decode / moe_layer_decode_noalloc without
 *                    a cache makes its routing wait expect one router row more
 *                    than exist, with a 2 ms limit: the wait gives up, the kernel
 *                    drains without computing, and moe_workspace_status (or
 *                    moe_noalloc_status) reports MOE_ETIMEOUT.
 *   MOE_INJECT_COPY  the next host -> device expert copy of a cached decode fails
 *                    as if cudaMemcpyAsync had returned an error: the call returns
 *                    MOE_ECUDA and the cache's policy state is as before the call.
 *   MOE_INJECT_ATTN_WAIT  the next moe_attn_step makes its attention CTAs expect
 *                    16 bytes more than their copies bring, with a 2 ms limit:
 *                    the waits give up, the CTAs drain, and
 *                    moe_attn_workspace_status reports MOE_ETIMEOUT (the keys
 *                    and values of the call are stored; its outputs are not valid).
 *   MOE_INJECT_NONE  clears a pending injection.
 * No GPU fault is involved.  Returns MOE_EINVAL for an unknown value.
 */
#define MOE_INJECT_NONE 0
#define MOE_INJECT_WAIT 1
#define MOE_INJECT_COPY 2
#define MOE_INJECT_ATTN_WAIT 3
MOE_API int moe_debug_inject(int what);

/* ---------------------------------------------------------------- attention */

/*
 * One attention block of a decoder layer over a binary16 key/value cache.  The
 * pages list attention and RoPE among the engine's own kernels, quantise the
 * attention weights in the same 4-bit affine format as the experts and keep the
 * key/value cache in FP16: a bounded ring for the 25 sliding-window layers, a
 * linear store for the 5 full-attention layers, 4096 tokens in the measured setup
 * (iitog.ru page "TurboFieldfare: движок с открытым кодом...", main technical
 * paragraph; remio.ai page, section "Mac Gemma 4 26B entra nello spazio
 * disponibile...").  They give no shapes or formulas; this library's readings:
 *   xn = RMSNorm(x) with MOE_PRENORM (norm_w, norm_eps as in moe_layer_t), else x;
 *   [q; k; v] = Wqkv xn: nq query heads, then nkv key heads, then nkv value heads,
 *     d rows each;
 *   RoPE on every query and key head at the token's position p, rotate-half
 *     pairing: for i < d/2, a = p * theta^(-2i/d),
 *     (u_i, u_{i+d/2}) -> (u_i cos a - u_{i+d/2} sin a, u_{i+d/2} cos a + u_i sin a);
 *   the rotated key and the value are stored in binary16 at slot p mod kv_len (a
 *     sliding-window layer, window > 0) or slot p (a full layer, window == 0);
 *   query head h attends, with key/value head h / (nq / nkv), to positions
 *     max(0, p - window + 1) .. p (sliding) or 0 .. p (full), the token's own
 *     included: o_h = sum_j softmax_j(scale q_h . k_j) v_j;
 *   y = Wo o, plus x with MOE_RESIDUAL.
 * The shapes:
 *   H hidden size, a multiple of 64, at most MOE_ATTN_MAX_HIDDEN;
 *   nq query heads, nkv key/value heads, nq a multiple of nkv; d in {64, 128, 256,
 *   512}; nq * d at most MOE_ATTN_MAX_HIDDEN;
 *   window >= 0; kv_len entries per key/value head (1 .. MOE_ATTN_MAX_KV);
 *   theta > 0 the RoPE base; scale the score scale (1/sqrt(d) is the usual one).
 * All pointers are device pointers owned by the caller, 16-byte aligned:
 *   wqkv_q/s/b 4-bit [(nq + 2 nkv) d][H], wo_q/s/b 4-bit [H][nq d] (MLX layout);
 *   k_cache, v_cache binary16 [nkv][kv_len][d], 16-byte aligned, read and updated.
 */
#define MOE_ATTN_MAX_HIDDEN 8192
#define MOE_ATTN_MAX_KV 65536

typedef struct moe_attn {
    int H, nq, nkv, d;
    int window, kv_len;
    float theta, scale;
    const uint32_t *wqkv_q;
    const uint16_t *wqkv_s, *wqkv_b;
    const uint32_t *wo_q;
    const uint16_t *wo_s, *wo_b;
    const float *norm_w;
    float norm_eps;
    uint16_t *k_cache, *v_cache;
} moe_attn_t;

/*
 * Workspace for moe_attn_step calls of up to T tokens (0 for bad shapes or T out
 * of 1..MOE_MAX_PREFILL_TOKENS).  The workspace is device memory the caller owns,
 * 256-byte aligned, zero-filled once before its first use (cudaMemset); every call
 * leaves its control words zero again.  One workspace serves one stream at a time.
 */
MOE_API size_t moe_attn_workspace_bytes(const moe_attn_t *attn, int T);

/*
 * T consecutive tokens (1..MOE_MAX_PREFILL_TOKENS) of one sequence at positions
 * pos .. pos+T-1: their keys and values are written into the cache, then each
 * token attends as above (so a chunk equals T one-token calls in order).
 * x, y: device fp32 [T][H]; y may alias x.  attn_out: optional device fp32
 * [T][nq d], the attention output o before Wo.  flags: MOE_RESIDUAL, MOE_PRENORM.
 * MOE_ECAPACITY when the positions do not fit the cache: a full layer needs
 * pos + T <= kv_len; a sliding layer needs kv_len >= window + T - 1, so that the new
 * entries overwrite no position the chunk still attends to (window + 0 suffices for
 * one token).  fp16 activations as tensor-core operands in the projections, fp32
 * everywhere else; deterministic.  Three kernel launches, stream-ordered.
 */
MOE_API int moe_attn_step(const moe_attn_t *attn, const float *x, int T, int pos, int flags, float *y,
                          float *attn_out, void *d_ws, size_t ws_bytes, void *stream);

/*
 * Synchronises `stream` and reports whether a bounded device-side wait of an
 * attention call on this workspace gave up since the last status call
 * (MOE_ETIMEOUT; the outputs of that call are not valid) and clears the report.
 * MOE_OK otherwise.
 */
MOE_API int moe_attn_workspace_status(void *d_ws, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
