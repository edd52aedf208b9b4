/*
 * mk.h — C ABI of the persistent MoE decode megakernel for GB300 (sm_103a).
 *
 * The library runs the token-generation decode step of a Flint-shaped
 * mixture-of-experts transformer as ONE cooperative CUDA launch per step
 * (one block per SM, grid-wide barriers only where data crosses blocks),
 * as described for Apple's Metal in "rec Megakernel and Tempo9 Compared",
 * §2 "Where Does rec's Single-Stream Advantage Come From?": input RMSNorm,
 * QKV projection fused with RoPE and the KV write, split attention with a
 * merge, output projection + residual, post-attention RMSNorm, router and
 * top-k, expert gate/up -> SiLU -> down (dense MLP in the first layers), and
 * after the last layer final norm, lm_head and argmax — all in one launch.
 *
 * Conventions shared by every call:
 *  - Every function returns an int status (MK_OK == 0, else an MK_ERR_*
 *    code) and never aborts the process.  mk_last_error() gives a message
 *    for the calling thread's last failure.
 *  - "device pointer" means memory on the context's CUDA device; "host
 *    pointer" means ordinary (pageable or pinned) host memory.  No call
 *    takes ownership of caller memory.
 *  - Streams are passed as `void*` holding a cudaStream_t (NULL = legacy
 *    default stream).  Launching calls are asynchronous on that stream and
 *    return before the GPU work finishes; device-side failures (a grid
 *    barrier that timed out, an index out of range) are reported by the next
 *    mk_sync().
 *  - A context is not thread-safe: calls on one context must be serialised
 *    by the caller, and all launches of one context must be ordered on the
 *    GPU (one stream, or explicit events between streams).
 */
#ifndef MK_H_
#define MK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MK_API __attribute__((visibility("default")))
#else
#define MK_API
#endif

/* ---- status codes ---- */
#define MK_OK 0
#define MK_ERR_INVALID_ARG 1      /* a null pointer, bad size or index, misaligned weight */
#define MK_ERR_NO_PAGES 2         /* the KV page pool has no free page */
#define MK_ERR_STATE 3            /* call out of order (e.g. no KV pool, position mismatch) */
#define MK_ERR_CUDA 4             /* a CUDA runtime call failed (message has the CUDA error) */
#define MK_ERR_UNSUPPORTED 5      /* shape / dtype not compiled in, device not sm_103, no co-residency */
#define MK_ERR_BARRIER_TIMEOUT 6  /* a grid barrier gave up waiting (reported by mk_sync) */
#define MK_ERR_DEVICE_INDEX 7     /* the kernel's own bounds check refused an index (mk_sync) */

/* ---- weight storage formats ---- */
#define MK_F32 0        /* float32, row-major [rows, K] */
#define MK_BF16 1       /* bfloat16, row-major [rows, K] */
#define MK_INT4_G64 2   /* symmetric int4: codes [rows, K/2] uint8, two's-complement
                           nibbles with the even k in the low nibble; scales
                           [rows, K/64] bfloat16; w[r,k] = q[r,k] * s[r,k/64] */
#define MK_INT3_G64 3   /* symmetric int3 (expert matrices only): codes [rows, 3K/8]
                           uint8, each 3 bytes one little-endian 24-bit word of 8
                           consecutive k, the 3-bit two's-complement code of k at
                           bits 3(k%8) .. 3(k%8)+2; scales [rows, K/64] bfloat16;
                           w[r,k] = q[r,k] * s[r,k/64] */

/* Model description.  The library compiles the decode step for fixed layer
 * shapes; mk_create() answers MK_ERR_UNSUPPORTED for others.  Compiled shapes:
 *   Flint: hidden 2048, 16 q / 4 kv heads of 128, 64 experts top-6 of FFN 768,
 *          dense FFN 6144;
 *   tiny:  hidden 256, 4 q / 2 kv heads of 64, 8 experts top-2 of FFN 128,
 *          dense FFN 512.
 * n_layers, n_dense, vocab, rope_theta and rms_eps are free.  page_tokens
 * must be 128 and max_batch at most 16. */
typedef struct mk_model_desc {
  int32_t n_layers;
  int32_t hidden;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t vocab;
  int32_t n_dense;      /* layers [0, n_dense) use the dense SwiGLU MLP */
  int32_t dense_ffn;
  int32_t n_experts;
  int32_t top_k;
  int32_t expert_ffn;
  float rope_theta;
  float rms_eps;
  int32_t wdtype;       /* MK_F32 | MK_BF16 | MK_INT4_G64: the linear layers */
  int32_t page_tokens;  /* must be 128 */
  int32_t max_batch;    /* rows per launch, 1..16 */
  int32_t max_ctx;      /* largest position + 1 any sequence may reach, 1..1048576 */
  int32_t max_seqs;     /* sequence ids are 0 .. max_seqs-1; 1..65536 */
  int32_t expert_wdtype;  /* format of exp_gate / exp_up / exp_down: equal to wdtype, or
                             MK_INT3_G64 with wdtype MK_INT4_G64 (int3 experts, int4
                             elsewhere); anything else is MK_ERR_INVALID_ARG */
} mk_model_desc;

/* A linear weight: `w` points at the codes / values; `scales` only for int4 / int3. */
typedef struct mk_linear {
  const void* w;
  const void* scales;
} mk_linear;

/* One layer's weights (device pointers, logical layouts above).  The
 * "aux" tensors (norms, router, embedding) are float32 when wdtype is MK_F32
 * and bfloat16 otherwise.
 *   attn_norm, ffn_norm [hidden]
 *   wq [n_heads*head_dim, hidden], wk / wv [n_kv_heads*head_dim, hidden],
 *   wo [hidden, n_heads*head_dim]
 *   dense layers (index < n_dense): gate, up [dense_ffn, hidden], down [hidden, dense_ffn]
 *   MoE layers: router [n_experts, hidden]; exp_gate, exp_up
 *   [n_experts, expert_ffn, hidden]; exp_down [n_experts, hidden, expert_ffn]
 *   (int4 / int3 scales stacked the same way).  Unused fields may be NULL. */
typedef struct mk_layer_weights {
  const void* attn_norm;
  mk_linear wq, wk, wv, wo;
  const void* ffn_norm;
  mk_linear gate, up, down;
  const void* router;
  mk_linear exp_gate, exp_up, exp_down;
} mk_layer_weights;

typedef struct mk_weights {
  const void* embed;              /* [vocab, hidden] aux dtype */
  const void* final_norm;         /* [hidden] aux dtype */
  mk_linear lm_head;              /* [vocab, hidden] wdtype */
  const mk_layer_weights* layers; /* HOST array of n_layers entries */
} mk_weights;

typedef struct mk_ctx mk_ctx;

/* Information about a context (filled by mk_get_info). */
typedef struct mk_info {
  int32_t device;
  int32_t num_sms;
  int32_t grid;              /* blocks per launch (one per SM) */
  int32_t block_threads;
  int32_t smem_bytes;        /* dynamic shared memory per block of a launch of 2+ rows (one-row
                                launches ask for less, leaving more of the SM's storage as L1) */
  int32_t n_pages;           /* KV pages in the pool (0 before mk_kv_alloc) */
  int32_t free_pages;
  int64_t scratch_bytes;     /* library-owned device scratch */
  int64_t kv_bytes;          /* KV pool bytes */
  int32_t last_chunk;        /* attention split size (tokens) of the last launch */
  int32_t last_units;        /* attention work units of the last launch */
} mk_info;

/* Create a context on the current CUDA device.
 * d: model description (copied).  w: weight pointers in the logical layouts
 * above; every pointer must be 16-byte aligned.  The linear layers (wq, wk,
 * wv, wo, gate/up/down, the experts and lm_head) are COPIED during the call
 * into a library-owned packed buffer (the layout of mk_pack_weights); the
 * embedding, the norms and the routers are BORROWED: the library reads them
 * in place and they must stay valid and unchanged until mk_destroy.  The host
 * array w->layers is copied and may be freed after the call.  Allocates the
 * packed weights, library-owned scratch and the RoPE table (computed on the
 * host in double precision).  *out receives the context.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
MK_API int mk_create(const mk_model_desc* d, const mk_weights* w, mk_ctx** out);

/* Bytes of the packed linear weights of a model (0 if d is invalid).  The
 * packed layout is the library's own: one 16-byte aligned record per output
 * row (codes, then the int4 / int3 group scales), the rows a decode task
 * reads together adjacent (the two RoPE rows of a q/k/v pair, the gate and up
 * rows of an FFN row).  An int3 record holds, per 32-value chunk, two words of
 * 2-bit fields and one word of 1-bit fields (the codes plus 4), in the byte
 * order of the kernel's dot products.  The method itself has no such call: it
 * exists so that the allocation-free entry point can run on weights its caller
 * packed. */
MK_API size_t mk_packed_bytes(const mk_model_desc* d);

/* Pack the linear weights of w (logical layouts above) into dst_dev, a
 * caller-owned device buffer of at least mk_packed_bytes(d) bytes, 256-byte
 * aligned.  Runs kernels on `stream` and returns without waiting; w must stay
 * valid until they finish.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
MK_API int mk_pack_weights(const mk_model_desc* d, const mk_weights* w, void* dst_dev, size_t dst_bytes,
                           void* stream);

/* Allocate the KV cache: a pool of n_pages pages of page_tokens (128)
 * positions for every layer, bf16, laid out
 * [layer][page][K|V][kv_head][slot][head_dim], owned by the library.
 * Call once per context; a second call returns MK_ERR_STATE.
 * Errors: INVALID_ARG, STATE, CUDA. */
MK_API int mk_kv_alloc(mk_ctx* ctx, int32_t n_pages);

/* Prefill: run n (1..4096) prompt tokens of sequence seq_id at positions
 * start_pos .. start_pos+n-1 through the model, writing their K/V into
 * pages taken from the pool.  The chunk limit follows "rec Megakernel and
 * Tempo9 Compared", §1 (Prefill), where the megakernel engine splits long
 * prompts into pieces of 4096 tokens.  start_pos must
 * equal the sequence's current length (0 starts a new sequence).
 * tokens_dev: device int32[n].  out_token_dev: device int32[1] that receives
 * the greedy next token after the last position (may be NULL).
 * A chunk of up to 16 positions runs as one launch of the decode kernel.  A
 * longer chunk runs the model over all of its positions at once, layer by
 * layer: the projections as tensor-core GEMMs over the chunk's rows (cuBLAS,
 * fp32 accumulation; activations split into two 16-bit parts; int4 and int3
 * weights widened exactly to fp16, bf16 weights used in place), attention, norms,
 * routing, the grouping of rows by expert and the residuals as the library's
 * kernels.  This path takes its pages up front, makes a workspace of about
 * 1.2 GB (Flint shape; kept by the context) on its first use, and waits for
 * the stream once per MoE layer (the expert GEMMs are sized on the host from
 * the routing counts), so the call returns only when the chunk's last layer
 * is enqueued.
 * Errors: INVALID_ARG, STATE, NO_PAGES (nothing is launched then), CUDA. */
MK_API int mk_prefill_chunk(mk_ctx* ctx, int32_t seq_id, const int32_t* tokens_dev,
                            int32_t n, int32_t start_pos, int32_t* out_token_dev,
                            void* stream);

/* One decode step for n (1..max_batch) sequences in ONE launch (continuous
 * batching: any set of open sequences, each at its own position).
 * seq_ids_host, positions_host: host int32[n]; positions[i] must equal the
 * length of sequence seq_ids[i] (ids distinct).  tokens_dev: device int32[n]
 * input tokens; out_tokens_dev: device int32[n] greedy next tokens.
 * tokens_dev may alias out_tokens_dev, so steps chain on the GPU with no host
 * synchronisation.  On success every sequence's length grows by one.
 * Errors: INVALID_ARG, STATE, NO_PAGES (nothing is launched then), CUDA. */
MK_API int mk_decode_step(mk_ctx* ctx, const int32_t* seq_ids_host, const int32_t* tokens_dev,
                          const int32_t* positions_host, int32_t n, int32_t* out_tokens_dev,
                          void* stream);

/* Close a sequence and return its pages to the pool (a page shared with a
 * forked sequence stays held until its last holder is released).  Pages
 * become reusable by launches enqueued after this call on the context's
 * stream.
 * Errors: INVALID_ARG (bad id), STATE (sequence not open). */
MK_API int mk_seq_release(mk_ctx* ctx, int32_t seq_id);

/* Copy K/V between a sequence's pages and a caller buffer.  Buffer layout:
 * device bf16 [n_layers][n][2 (K, V)][n_kv_heads][head_dim], 16-byte
 * aligned, owned by the caller.  Both calls run a kernel on `stream` and
 * return without waiting; the buffer must stay valid until it finishes.
 *
 * mk_kv_write stores positions start_pos .. start_pos+n-1 of seq_id.
 * start_pos must lie in [0, length]: positions below the length are
 * overwritten, positions at or past it extend the sequence (pages are taken
 * from the pool, the length becomes start_pos + n, a closed sequence is
 * opened).  The KV written this way is what later launches attend to, as if
 * the model had computed it: a prefix restored from elsewhere, or (in tests)
 * a reference computation's cache.  "rec Megakernel and Tempo9 Compared",
 * §1 (Prefix cache), measures the value of not recomputing a known prefix.
 * Errors: INVALID_ARG, STATE (start_pos past the length, or a position in a
 * page shared with another sequence), NO_PAGES (nothing written), CUDA.
 *
 * mk_kv_read copies positions start_pos .. start_pos+n-1 (all below the
 * length) into dst_dev.  Errors: INVALID_ARG, STATE, CUDA. */
MK_API int mk_kv_write(mk_ctx* ctx, int32_t seq_id, int32_t start_pos, int32_t n, const void* src_dev,
                       void* stream);
MK_API int mk_kv_read(mk_ctx* ctx, int32_t seq_id, int32_t start_pos, int32_t n, void* dst_dev,
                      void* stream);

/* Open sequence dst_seq as a copy of the first n_tokens positions of src_seq
 * by SHARING their pages (no K/V is copied): n_tokens must be a positive
 * multiple of 128 (whole pages, so neither sequence ever writes a shared
 * page again) and at most src_seq's length; dst_seq must be closed.  Pages
 * are reference-counted: mk_seq_release of either sequence keeps the pages
 * the other still holds.  This is the page-pool form of the prefix reuse that
 * "rec Megakernel and Tempo9 Compared", §1 (Prefix cache) measures (a turn
 * reusing 7,936 of 8,022 prompt tokens in 128-token spans).  Sets dst_seq's
 * block-table entries with a kernel on `stream`.
 * Errors: INVALID_ARG, STATE, CUDA. */
MK_API int mk_seq_fork(mk_ctx* ctx, int32_t src_seq, int32_t dst_seq, int32_t n_tokens, void* stream);

/* Current length (positions written) of a sequence; -1 if it is not open. */
MK_API int32_t mk_seq_length(mk_ctx* ctx, int32_t seq_id);

/* Wait for the stream, then read and clear the device error word.
 * Returns MK_OK, MK_ERR_BARRIER_TIMEOUT, MK_ERR_DEVICE_INDEX or MK_ERR_CUDA. */
MK_API int mk_sync(mk_ctx* ctx, void* stream);

/* Debugging.  flags: MK_DBG_TRACE makes every launch write its trace into
 * trace_dev (device float buffer of trace_bytes, laid out as documented for
 * mk_trace_bytes).  MK_DBG_SKIP_ARRIVAL makes block `arg & 0xffff` skip its
 * arrival at grid barrier number `arg >> 16` of the next launch, so that the
 * other blocks' bounded waits run out (a test of the timeout path).
 * spin_limit_us bounds every grid-barrier wait (0 keeps the default, 1 s).
 * Errors: INVALID_ARG. */
#define MK_DBG_TRACE 1u
#define MK_DBG_SKIP_ARRIVAL 2u
#define MK_DBG_SPLIT 8u    /* each decode / prefill launch runs as 4 * n_layers + 1 launches of the
                              same kernel, one per phase group of a layer (QKV | attention |
                              o_proj | routing + gate/up + down) and one for lm_head: the kernel
                              boundary takes the place of the grid barrier between groups.
                              Results are the same bits; it exists to measure a launch
                              boundary against a grid barrier on the same device code. */
#define MK_DBG_TIMING 4u   /* trace_dev receives uint64 %globaltimer stamps (ns) of
                              every block: block b's record of R = 16 * n_layers + 2
                              stamps starts at [b * R]; in it [0] block start; for
                              layer l and phase p (0 qkv, 1 attention, 2 o_proj,
                              3 routing and gate/up, 4 down) [1 + 16*l + 3*p + k]
                              with k = 0 staging done, 1 phase work done, 2 grid
                              barrier released; [1 + 16*l + 15] the routing of MoE
                              layer l ready; then [1 + 16*n_layers] lm_head done.
                              After the grid's records, each block's ring log of
                              3072 stamps at [grid * R + b * 3072]: for its k-th
                              weight / KV tile (k < 1024) [3k] issued, [3k + 1]
                              found landed by the compute warps, [3k + 2] released
                              by warp 0.  Size: 8 * grid * (R + 3072) bytes (grid:
                              mk_get_info).
                              Not combinable with MK_DBG_TRACE. */
MK_API int mk_set_debug(mk_ctx* ctx, uint32_t flags, uint32_t arg, void* trace_dev,
                        size_t trace_bytes, uint32_t spin_limit_us);

/* Size of the trace for one launch of `rows` rows.  Layout (float32):
 *   x      [n_layers][rows][hidden]     residual after each layer
 *   attn   [n_layers][rows][n_heads*head_dim]  attention output (merged)
 *   logits [n_layers][rows][n_experts]  router logits (0 for dense layers)
 *   topk   [n_layers][rows][2*top_k]    expert ids (as float) then weights
 *   final  [rows][vocab]                lm_head logits (rows with an output) */
MK_API size_t mk_trace_bytes(const mk_model_desc* d, int32_t rows);

/* The attention split a decode launch uses for rows whose new positions are
 * positions_host[0..n) (host int32, each >= 0; n in 1..16): every (row, kv
 * head) is cut into chunks of *chunk_out cached positions (a whole number of
 * tile_tokens, the kernel's cached positions per ring tile: mk_info
 * tile_tokens), giving *units_out (row, kv head, chunk) units over `grid`
 * blocks.  The chunk minimises ceil(units / grid) x (chunk + 1.5 tiles of fixed
 * cost per unit), the larger chunk on a tie, with at most 64 chunks per row,
 * 4 units per block and grid + 16 x n_kv_heads units.  Host only, no device
 * work.  Errors: INVALID_ARG. */
MK_API int mk_attention_plan(int32_t n_kv_heads, int32_t grid, int32_t tile_tokens, const int32_t* positions_host,
                             int32_t n, int32_t* chunk_out, int32_t* units_out);

MK_API int mk_get_info(mk_ctx* ctx, mk_info* info);

/* Release every resource of the context (waits for its device work). */
MK_API int mk_destroy(mk_ctx* ctx);

/* Decode step that allocates no device memory.  The method itself has no
 * such call.  It is for callers that cannot call cudaMalloc: a host that
 * gives the library a fixed memory budget carved by its own allocator (and
 * so must not see allocations it did not plan), or a loop that must not take
 * the device-wide synchronisation that cudaMalloc / cudaFree can bring.
 * It launches the same kernel as mk_decode_step without a context: the
 * per-layer pointer table, the RoPE table and the kernel's scratch live in a
 * file-scope device array of 8 MiB that every GPU loading the library holds
 * until the process exits.  Positions must be below 8192 (the size of that
 * RoPE table); a model whose scratch does not fit in the array is rejected
 * with MK_ERR_UNSUPPORTED.
 * d, w: as for mk_create (weights borrowed for the duration of the call;
 *   the linear layers are read from packed_dev instead).
 * packed_dev: the caller's packed linear weights (mk_pack_weights), 256-byte
 *   aligned.
 * kv_dev: caller-owned KV pool of n_pages pages in the layout of mk_kv_alloc.
 * block_table_dev: caller-owned int32 [max_seqs][max_pages_per_seq]; entry
 *   [slot][p / 128] must hold the page of every cached position p < position;
 *   the call itself writes the entry of each row's new position.
 * slots_host, positions_host, pages_host: host int32[n]: the block-table row
 *   of each sequence (distinct), its position (= its current length) and the
 *   pool page that holds that position.
 * tokens_dev / out_tokens_dev: device int32[n] inputs / greedy next tokens.
 * status_dev: optional device int32[1] that receives the kernel's error word
 *   (0, MK_ERR_BARRIER_TIMEOUT or MK_ERR_DEVICE_INDEX) after the launch.
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address and uploads the RoPE and layer tables with
 * synchronous copies; make that first call before any stream capture.  A
 * later call whose model differs (weights, n_layers, rope_theta, head_dim)
 * first waits for the whole device to go idle (cudaDeviceSynchronize: an
 * earlier call on any stream may still read the tables), then rewrites the
 * tables the same way and clears the kernel scratch (synchronous memset, then
 * another wait).  A call with the same model as the previous one only
 * enqueues on `stream`: four memsets that clear the counters (all but the
 * launch epoch) and the error word (the array keeps the last call's
 * contents), the launch and the optional status copy.
 * Every call shares the one array: calls that overlap on the GPU, on any
 * stream, race, and so does a call that changes the model while another
 * thread's call is being enqueued.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
MK_API int mk_decode_step_static(const mk_model_desc* d, const mk_weights* w, const void* packed_dev,
                                 void* kv_dev, int32_t n_pages, int32_t* block_table_dev,
                                 int32_t max_pages_per_seq, const int32_t* slots_host,
                                 const int32_t* positions_host, const int32_t* pages_host,
                                 int32_t n, const int32_t* tokens_dev, int32_t* out_tokens_dev,
                                 int32_t* status_dev, void* stream);

/* Bytes of the static array that mk_decode_step_static needs for model d on
 * a device of `grid` SMs (the launch takes one block per SM): the RoPE table,
 * the layer table and the kernel scratch, each 256-byte aligned
 * (*need_out), and the array's size (*capacity_out, 8 MiB).  A model with
 * *need_out > *capacity_out is one that mk_decode_step_static rejects with
 * MK_ERR_UNSUPPORTED.  Host only, no device work.
 * Errors: INVALID_ARG, UNSUPPORTED (as mk_create's description checks). */
MK_API int mk_static_bytes(const mk_model_desc* d, int32_t grid, int64_t* need_out, int64_t* capacity_out);

/* Message of the calling thread's last failure ("" if none). */
MK_API const char* mk_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MK_H_ */
