// Internal types shared by the host library (mk_host.cpp) and the decode
// kernel (mk_kernel.cu).  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "mk.h"

namespace mk {

constexpr int kMaxBatch = 16;        // rows per launch
constexpr int kPageTokens = 128;     // KV positions per page
// 15 compute warps + 1 weight-streaming warp: 16 warps keep 4 per scheduler
// partition, so each thread may hold 128 registers (a 17th warp would cut
// that to 96)
constexpr int kThreads = 480;        // compute threads per block (15 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kBlockThreads = kThreads + 32;  // plus one weight-streaming warp
constexpr int kMaxStages = 16;       // shared-memory ring stages
constexpr int kRlogitGroups = 8;     // copies of the router-logit sums (less atomic contention)
// Router-logit partials are summed as 64-bit fixed-point integers (units of
// 2^-32): integer addition is associative, so the sum, and with it the expert
// selection, is the same bits whatever order the blocks' atomics land in.
// Range: |sum| < 2^31.
constexpr float kFixScale = 4294967296.f;       // 2^32
constexpr float kFixUnit = 2.3283064365386963e-10f;  // 2^-32
constexpr int kRingLog = 1024;      // ring items per block whose issue / arrival times MK_DBG_TIMING logs
constexpr int kMaxUpd = 64;          // block-table updates carried by one launch
constexpr int kMaxRowsPerBlock = 32; // hidden rows owned by one block (hidden / grid)
constexpr int kMaxOwnUnits = 4;     // attention units one block may take in a launch
constexpr int kMaxChunks = 64;       // attention chunks per (row, kv head): one per lane-pair of a warp
constexpr int kSmemBytes = 227 * 1024;  // dynamic shared memory per block (the sm_100 family maximum)
// A launch of one row asks for less (its staging area and a ring of a few
// stages), so that more of the SM's 256 KB of L1/shared storage stays L1 for
// local memory and cached loads (the full size leaves 28 KB); 128 KB is the
// most that the 132 KB carve-out holds.
constexpr int kSmemSingleRow = 128 * 1024;

// Linear-weight slots of a layer.
enum Lin { WQ = 0, WK, WV, WO, GATE, UP, DOWN, EGATE, EUP, EDOWN, NLIN };

// Blocks of the packed linear weights of a layer (see mk_pack.cu).
enum PackBlock { PK_QKV = 0, PK_O, PK_GU, PK_DN, NPK };
constexpr int kMaxLayers = 128;

// Device-side copy of one layer's weight pointers.
struct LayerW {
  const void* attn_norm;
  const void* ffn_norm;
  const void* router;
  const void* w[NLIN];
  const void* s[NLIN];   // int4 scales (null otherwise)
  const uint8_t* pk[NPK];  // packed records (QKV pairs, o_proj, gate/up pairs, down)
};

// Byte offsets of the packed blocks inside one packed buffer.
struct PackLayout {
  size_t layer[kMaxLayers][NPK];
  size_t lm;
};

struct PageUpd {
  int32_t slot;   // sequence id
  int32_t index;  // page index within the sequence
  int32_t page;   // pool page
};

// Library-owned device scratch (one allocation, carved on the host).
struct Scratch {
  float* x;          // [kMaxBatch][H] residual stream
  float* h;          // [kMaxBatch][H] residual after attention
  float* q;          // [kMaxBatch][n_heads*hd] roped queries
  float* attn;       // [kMaxBatch][n_heads*hd] merged attention output
  float* part;       // [max_units][gqa][hd + 2] attention partials (m, l, o[hd])
  long long* rlogit; // [kRlogitGroups][kMaxBatch][E] router logits before the RMS scale, fixed
                     // point: block partials summed into one of kRlogitGroups
                     // copies (block id mod groups)
  float* act;        // [kMaxBatch][top_k][Fe] expert activations
  float* dact;       // [kMaxBatch][Fd] dense-MLP activations
  float* amax_v;     // [grid][kMaxBatch] per-block best logit
  int32_t* amax_i;   // [grid][kMaxBatch] per-block best token
  int32_t* merge_cnt;   // [kMaxBatch][n_kv] attention merge arrivals
  uint32_t* sync;       // counters, one per 128-byte line: [0] barrier, [32] exit,
                        // [64] launch epoch (advanced by every launch), [96] argmax reduce
  uint64_t* xll;        // [2][kMaxBatch][H] the residual as flagged words (value, tag),
                        // double-buffered by layer parity
  int32_t* err;         // [0] status, [1] site, [2] detail
};

struct StepArgs {
  const LayerW* layers;
  const void* embed;
  const void* final_norm;
  const void* lm_head;
  const void* lm_head_s;
  const uint8_t* lm_pk;      // packed lm_head records
  const float2* rope;        // [max_ctx][hd/2] (cos, sin)
  uint16_t* kv;              // bf16 pool
  int32_t* block_table;      // [max_seqs][max_pages_per_seq]
  Scratch sc;
  const int32_t* tokens;     // [n] (device)
  int32_t* out_tokens;       // written for rows >= out_first at out_tokens[row - out_first]
  float* trace;              // debug trace or null
  uint64_t* timing;          // per-phase timestamps (block 0) or null
  int32_t n_pages;
  int32_t max_pages_per_seq;
  int32_t n;                 // rows in this launch
  int32_t n_layers;
  int32_t n_dense;
  int32_t vocab;
  float eps;
  int32_t chunk;             // attention split size (tokens)
  int32_t n_units;           // attention work units
  int32_t out_first;         // first row that gets an lm_head output (n = none)
  int32_t max_units;         // capacity of sc.part
  int32_t n_upd;
  uint32_t dbg_flags;
  uint32_t dbg_arg;
  // the phase groups this launch runs: group s is layer s / 4, part s % 4
  // (0 QKV, 1 attention, 2 o_proj, 3 routing + gate/up + down); a step is
  // groups [0, 4 * n_layers) and then lm_head (run_lm)
  int32_t slice_lo, slice_hi, run_lm;
  uint64_t spin_limit_ns;
  int32_t slot[kMaxBatch];
  int32_t pos[kMaxBatch];
  int32_t new0[kMaxBatch];   // first position of the row's sequence written by this launch
  int32_t cur_page[kMaxBatch];
  PageUpd upd[kMaxUpd];
};

// One KV transfer (mk_kv.cu): block-table entries to set, then the K/V of
// positions [start, start + n) of sequence `slot` copied from src into the
// pool (src != null) or from the pool into dst.  Caller buffer layout: bf16
// [n_layers][n][K|V][n_kv_heads][head_dim].  upd[i] sets page index
// upd_index0 + i of sequence `slot` (fork calls may set other sequences'
// entries with n == 0).
struct KvXfer {
  uint16_t* kv;
  int32_t* block_table;
  const uint16_t* src;
  uint16_t* dst;
  int32_t n_pages, max_pages_per_seq, n_layers, n_kv_heads, head_dim;
  int32_t slot, start, n;
  int32_t n_upd, upd_index0;
  PageUpd upd[kMaxUpd];
};
int launch_kv_xfer(const KvXfer& a, cudaStream_t st);

// Chunked prefill (mk_prefill.cu): chunks of more than kMaxBatch positions
// run as per-layer GEMMs over all rows of the chunk.
constexpr int kMaxPrefill = 4096;
struct PrefillWork;  // workspace kept by a context (made on first use)
struct PrefillArgs {
  mk_model_desc d;
  const LayerW* layers;        // host copy of the layer table (packed record pointers)
  const void* embed;
  const void* final_norm;
  const uint8_t* lm_pk;
  const float2* rope;          // device RoPE table [max_ctx][hd/2]
  uint16_t* kv;
  int32_t* block_table;        // holds the pages of every position of the chunk
  int32_t n_pages, max_pages_per_seq, slot, start, n;
  const int32_t* tokens;       // device [n]
  int32_t* out_token;          // device [1] or null
  float* trace;                // trace of the chunk's last trace_rows rows, or null
  size_t trace_bytes;
  int32_t trace_rows;
  int32_t* err;                // device error word
};
int prefill_run(PrefillWork** work, const PrefillArgs& a, cudaStream_t st);
void prefill_free(PrefillWork* w);
int prefill_setup_attributes(const mk_model_desc& m);

// Error sites recorded in err[1].
enum ErrSite {
  SITE_BARRIER = 1, SITE_PAGE = 2, SITE_UNIT = 3, SITE_TOKEN = 4, SITE_RING = 5, SITE_SMEM = 6, SITE_FLAG = 7
};

// Kernel variants compiled into the library.
enum ShapeId { SHAPE_FLINT = 0, SHAPE_TINY = 1, NSHAPE };

struct KernelInfo {
  const void* fn;
  int smem_bytes;
  int tile_tokens;  // cached positions per ring stage (attention chunks are multiples)
  int smem_single;  // dynamic shared memory of a one-row launch
};
inline int launch_smem_bytes(const KernelInfo& k, int rows) { return rows == 1 ? k.smem_single : k.smem_bytes; }

// The kernel variants, by translation unit (mk_kernel.cu is compiled once per
// part); each returns fn == nullptr for the variants it does not hold.
KernelInfo get_kernel_part0(int shape, int wdtype, int xdtype);
KernelInfo get_kernel_part1(int shape, int wdtype, int xdtype);
KernelInfo get_kernel_part2(int shape, int wdtype, int xdtype);
KernelInfo get_kernel_part3(int shape, int wdtype, int xdtype);
// Returns the kernel for (shape, linear-layer format, expert format) or
// fn == nullptr if not compiled.
inline KernelInfo get_kernel(int shape, int wdtype, int xdtype) {
  KernelInfo (*const parts[4])(int, int, int) = {get_kernel_part0, get_kernel_part1, get_kernel_part2,
                                                 get_kernel_part3};
  for (auto f : parts) {
    const KernelInfo k = f(shape, wdtype, xdtype);
    if (k.fn) return k;
  }
  return {nullptr, 0, 0, 0};
}

// Host helpers of mk_host.cpp shared with the allocation-free entry point.
// host_check_model: validates the description and weight pointers and fills
// the per-layer pointer table (status code; message via mk_last_error).
int host_check_model(const mk_model_desc* d, const mk_weights* w, int* shape, LayerW* layers);
size_t host_carve_scratch(const mk_model_desc& d, int grid, int max_units, char* base, Scratch* sc);
void host_attention_split(int n_kv_heads, int grid, int tile_tokens, const int32_t* pos, int n, int* chunk,
                          int* units);
int host_fail(int code, const char* msg);
void host_clear_error();
int host_validate_desc(const mk_model_desc* d, int* shape);

// Packed weights (mk_pack.cu): record sizes, the layout (returns the total
// bytes; pl may be null) and the pack itself (kernels on stream st).
int pack_row_bytes(int wdtype, int K);
int pack_scale_bytes(int wdtype, int K);
int pack_rec_bytes(int wdtype, int K);
size_t host_pack_layout(const mk_model_desc& d, PackLayout* pl);
int host_pack(const mk_model_desc& d, const mk_weights& w, uint8_t* dst, cudaStream_t st);

}  // namespace mk
