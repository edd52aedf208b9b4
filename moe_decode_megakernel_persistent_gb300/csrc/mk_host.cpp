// Host side of the C ABI declared in include/mk.h: context and weight-table
// set-up, the KV page pool and per-sequence page lists, per-launch argument
// building (positions, pages, attention split) and the cooperative launch.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "mk_internal.h"

using namespace mk;

namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

#define MK_CUDA(call)                                                                       \
  do {                                                                                      \
    cudaError_t e_ = (call);                                                                \
    if (e_ != cudaSuccess)                                                                  \
      return fail(MK_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_));        \
  } while (0)

struct Seq {
  bool open = false;
  int32_t len = 0;
  std::vector<int32_t> pages;
};

struct ShapeRow {
  int id, hidden, heads, kv_heads, head_dim, experts, top_k, expert_ffn, dense_ffn;
};
constexpr ShapeRow kShapes[] = {
    {SHAPE_FLINT, 2048, 16, 4, 128, 64, 6, 768, 6144},
    {SHAPE_TINY, 256, 4, 2, 64, 8, 2, 128, 512},
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Host tables sized by the description (the RoPE table, max_ctx x head_dim / 2
// pairs; the sequence table) stay bounded: 512 MiB and 64 Ki entries at most.
constexpr int32_t kMaxCtx = 1 << 20;
constexpr int32_t kMaxSeqs = 1 << 16;

}  // namespace

struct mk_ctx {
  mk_model_desc d{};
  int shape = -1;
  KernelInfo kern{};
  int device = 0, num_sms = 0, grid = 0;
  LayerW* layers_dev = nullptr;
  const void* embed = nullptr;
  const void* final_norm = nullptr;
  const void* lm_head = nullptr;
  const void* lm_head_s = nullptr;
  uint8_t* packed_dev = nullptr;   // the library's packed copy of the linear weights
  size_t packed_bytes = 0;
  const uint8_t* lm_pk = nullptr;
  float2* rope_dev = nullptr;
  void* scratch_dev = nullptr;
  size_t scratch_bytes = 0;
  Scratch sc{};
  int max_units = 0;
  uint16_t* kv_dev = nullptr;
  int32_t n_pages = 0;
  size_t kv_bytes = 0;
  std::vector<int32_t> free_pages;  // stack; back() is handed out next
  std::vector<int32_t> page_ref;    // sequences holding each page (forked sequences share pages)
  int32_t* block_table_dev = nullptr;
  int32_t max_pages_per_seq = 0;
  std::vector<Seq> seqs;
  uint32_t dbg_flags = 0, dbg_arg = 0;
  float* trace = nullptr;
  size_t trace_bytes = 0;
  uint64_t spin_limit_ns = 1000000000ull;
  int last_chunk = 0, last_units = 0;
  std::vector<LayerW> layers_host;   // the layer table (for the chunked prefill)
  PrefillWork* prefill = nullptr;    // chunked-prefill workspace, made on first use
};

namespace {

int validate_desc(const mk_model_desc* d, int* shape) {
  if (!d) return fail(MK_ERR_INVALID_ARG, "model description is NULL");
  if (d->n_layers < 1 || d->n_layers > kMaxLayers || d->vocab < 1 || d->n_dense < 0 || d->n_dense > d->n_layers)
    return fail(MK_ERR_INVALID_ARG, "n_layers (1..128) / vocab / n_dense out of range");
  if (d->wdtype == MK_INT4_G64 && d->vocab % 8 != 0)
    return fail(MK_ERR_UNSUPPORTED, "int4 lm_head needs a vocabulary that is a multiple of 8 rows");
  if (d->page_tokens != kPageTokens) return fail(MK_ERR_UNSUPPORTED, "page_tokens must be 128");
  if (d->max_batch < 1 || d->max_batch > kMaxBatch)
    return fail(MK_ERR_INVALID_ARG, "max_batch must be in [1, 16]");
  if (d->max_ctx < 1 || d->max_ctx > kMaxCtx || d->max_seqs < 1 || d->max_seqs > kMaxSeqs)
    return fail(MK_ERR_INVALID_ARG, "max_ctx must be in [1, 1048576] and max_seqs in [1, 65536]");
  if (d->wdtype != MK_F32 && d->wdtype != MK_BF16 && d->wdtype != MK_INT4_G64)
    return fail(MK_ERR_INVALID_ARG, "unknown wdtype");
  if (d->expert_wdtype != d->wdtype && !(d->wdtype == MK_INT4_G64 && d->expert_wdtype == MK_INT3_G64))
    return fail(MK_ERR_INVALID_ARG, "expert_wdtype must equal wdtype, or be MK_INT3_G64 with MK_INT4_G64");
  if (!(d->rms_eps >= 0.f) || !(d->rope_theta > 0.f))
    return fail(MK_ERR_INVALID_ARG, "rms_eps must be >= 0 and rope_theta > 0");
  for (const ShapeRow& s : kShapes)
    if (d->hidden == s.hidden && d->n_heads == s.heads && d->n_kv_heads == s.kv_heads &&
        d->head_dim == s.head_dim && d->n_experts == s.experts && d->top_k == s.top_k &&
        d->expert_ffn == s.expert_ffn && d->dense_ffn == s.dense_ffn) {
      *shape = s.id;
      return MK_OK;
    }
  return fail(MK_ERR_UNSUPPORTED, "layer shape is not compiled into this library");
}

bool quantised(int fmt) { return fmt == MK_INT4_G64 || fmt == MK_INT3_G64; }

int check_lin(const mk_linear& l, bool scaled, const char* what, int layer) {
  if (!l.w || !aligned16(l.w) || (scaled && (!l.scales || !aligned16(l.scales))))
    return fail(MK_ERR_INVALID_ARG, std::string("weight ") + what + " of layer " +
                                        std::to_string(layer) + " is NULL or not 16-byte aligned");
  return MK_OK;
}

int check_aux(const void* p, const char* what, int layer) {
  if (!p || !aligned16(p))
    return fail(MK_ERR_INVALID_ARG, std::string("tensor ") + what + " of layer " +
                                        std::to_string(layer) + " is NULL or not 16-byte aligned");
  return MK_OK;
}

// Scratch layout: sub-buffers of the one allocation, 256-byte aligned.
size_t carve_scratch(const mk_model_desc& d, int grid, int max_units, char* base, Scratch* sc) {
  const int H = d.hidden, QD = d.n_heads * d.head_dim, GQA = d.n_heads / d.n_kv_heads;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off = round_up(off + bytes, 256);
    return p;
  };
  Scratch s{};
  s.x = (float*)take(sizeof(float) * kMaxBatch * H);
  s.h = (float*)take(sizeof(float) * kMaxBatch * H);
  s.q = (float*)take(sizeof(float) * kMaxBatch * QD);
  s.attn = (float*)take(sizeof(float) * kMaxBatch * QD);
  s.part = (float*)take(sizeof(float) * (size_t)max_units * GQA * (d.head_dim + 4));
  s.rlogit = (long long*)take(sizeof(long long) * kRlogitGroups * kMaxBatch * d.n_experts);
  s.act = (float*)take(sizeof(float) * kMaxBatch * d.top_k * d.expert_ffn);
  s.dact = (float*)take(sizeof(float) * kMaxBatch * d.dense_ffn);
  s.amax_v = (float*)take(sizeof(float) * (size_t)grid * kMaxBatch);
  s.amax_i = (int32_t*)take(sizeof(int32_t) * (size_t)grid * kMaxBatch);
  s.merge_cnt = (int32_t*)take(sizeof(int32_t) * kMaxBatch * d.n_kv_heads);
  s.sync = (uint32_t*)take(sizeof(uint32_t) * 128);
  s.xll = (uint64_t*)take(sizeof(uint64_t) * 2 * kMaxBatch * H);
  s.err = (int32_t*)take(sizeof(int32_t) * 4);
  if (sc) *sc = s;
  return off;
}

// Split of the attention work into (row, kv head, chunk of positions) units,
// with chunks a whole number of ring tiles (tile_tokens cached positions
// each) and at most kMaxChunks chunks per row.
void host_attention_split_impl(int n_kv_heads, int grid, int tile_tokens, const int32_t* pos, int n, int* chunk,
                               int* units) {
  long long total = 0, longest = 0;
  for (int i = 0; i < n; ++i) {
    total += pos[i] + 1;
    longest = std::max<long long>(longest, pos[i] + 1);
  }
  (void)total;
  const long long tt = std::max(1, tile_tokens);
  // chunks are whole ring tiles, at most kMaxChunks per row
  const long long lo = std::max(tt, ((longest + kMaxChunks - 1) / kMaxChunks + tt - 1) / tt * tt);
  // Blocks take units round-robin, so the attention phase lasts about
  // ceil(units / grid) x (chunk + a unit's fixed cost, about 1.5 ring tiles:
  // the query staging, the partial written, the merge share).  Take the chunk
  // that minimises it; on a tie the larger chunk (fewer units and merges).
  // A block takes at most kMaxOwnUnits units, and the partials' buffer holds
  // grid + n_kv_heads * kMaxBatch units.
  const long long ovh = tt + tt / 2;
  const long long cap = std::min<long long>((long long)kMaxOwnUnits * grid, (long long)grid + n_kv_heads * kMaxBatch);
  long long best_ch = -1, best_u = 0, best_cost = 0;
  for (long long ch = lo;; ch += tt) {
    long long u = 0;
    for (int i = 0; i < n; ++i) u += n_kv_heads * ((pos[i] + 1 + ch - 1) / ch);
    if (u <= cap) {
      const long long cost = (u + grid - 1) / grid * (ch + ovh);
      if (best_ch < 0 || cost <= best_cost) {
        best_ch = ch;
        best_u = u;
        best_cost = cost;
      }
    }
    if (ch >= longest) break;
  }
  if (best_ch < 0) {  // not reachable: one chunk per row gives n * n_kv_heads units
    best_ch = std::max(lo, (longest + tt - 1) / tt * tt);
    best_u = (long long)n * n_kv_heads;
  }
  *chunk = (int)best_ch;
  *units = (int)best_u;
}

void attention_split(const mk_ctx* c, const int32_t* pos, int n, int* chunk, int* units) {
  host_attention_split_impl(c->d.n_kv_heads, c->grid, c->kern.tile_tokens, pos, n, chunk, units);
}

// One launch over `n` rows.  Pages for positions that start a new page are
// taken from the pool here (rolled back if the pool runs dry).
int launch(mk_ctx* c, const int32_t* slots, const int32_t* positions, int n,
           const int32_t* tokens_dev, int32_t* out_dev, int out_first, cudaStream_t st) {
  if (!c->kv_dev) return fail(MK_ERR_STATE, "mk_kv_alloc has not been called");
  if ((c->dbg_flags & MK_DBG_TRACE) && c->trace_bytes < mk_trace_bytes(&c->d, n))
    return fail(MK_ERR_INVALID_ARG, "trace buffer is smaller than mk_trace_bytes(rows)");
  if ((c->dbg_flags & MK_DBG_TIMING) &&
      c->trace_bytes < sizeof(uint64_t) * (size_t)c->grid * (16 * (size_t)c->d.n_layers + 2 + 3 * kRingLog))
    return fail(MK_ERR_INVALID_ARG, "timing buffer is smaller than 8 * grid * (16 * n_layers + 2 + 3072) bytes");
  StepArgs a;
  std::memset(&a, 0, sizeof(a));
  std::vector<std::pair<int, int32_t>> taken;  // (slot, page) handed out by this call
  auto rollback = [&]() {
    for (auto it = taken.rbegin(); it != taken.rend(); ++it) {
      c->seqs[it->first].pages.pop_back();
      c->page_ref[it->second] = 0;
      c->free_pages.push_back(it->second);
    }
  };
  for (int i = 0; i < n; ++i) {
    const int s = slots[i], p = positions[i];
    Seq& q = c->seqs[s];
    const int pi = p / kPageTokens;
    if (pi == (int)q.pages.size()) {
      if (c->free_pages.empty()) {
        rollback();
        return fail(MK_ERR_NO_PAGES, "KV page pool exhausted");
      }
      const int32_t pg = c->free_pages.back();
      c->free_pages.pop_back();
      c->page_ref[pg] = 1;
      q.pages.push_back(pg);
      taken.emplace_back(s, pg);
      a.upd[a.n_upd++] = PageUpd{s, pi, pg};
    } else if (pi > (int)q.pages.size()) {
      rollback();
      return fail(MK_ERR_STATE, "position skips a page");
    }
    a.slot[i] = s;
    a.pos[i] = p;
    a.cur_page[i] = q.pages[pi];
  }
  // first position of each row's sequence that this launch writes: earlier
  // positions are in the cache before the launch starts
  for (int i = 0; i < n; ++i) {
    a.new0[i] = a.pos[i];
    for (int j = 0; j < n; ++j)
      if (a.slot[j] == a.slot[i] && a.pos[j] < a.new0[i]) a.new0[i] = a.pos[j];
  }
  attention_split(c, positions, n, &a.chunk, &a.n_units);
  if (a.n_units > kMaxOwnUnits * c->grid) {
    rollback();
    return fail(MK_ERR_INVALID_ARG, "more attention units than the grid can merge");
  }
  if (a.n_units > c->max_units) {
    rollback();
    return fail(MK_ERR_INVALID_ARG, "attention split exceeds the partials buffer");
  }
  a.layers = c->layers_dev;
  a.embed = c->embed;
  a.final_norm = c->final_norm;
  a.lm_head = c->lm_head;
  a.lm_head_s = c->lm_head_s;
  a.lm_pk = c->lm_pk;
  a.rope = c->rope_dev;
  a.kv = c->kv_dev;
  a.block_table = c->block_table_dev;
  a.sc = c->sc;
  a.tokens = tokens_dev;
  a.out_tokens = out_dev;
  a.trace = (c->dbg_flags & MK_DBG_TRACE) ? c->trace : nullptr;
  a.timing = (c->dbg_flags & MK_DBG_TIMING) ? reinterpret_cast<uint64_t*>(c->trace) : nullptr;
  a.n_pages = c->n_pages;
  a.max_pages_per_seq = c->max_pages_per_seq;
  a.n = n;
  a.n_layers = c->d.n_layers;
  a.n_dense = c->d.n_dense;
  a.vocab = c->d.vocab;
  a.eps = c->d.rms_eps;
  a.out_first = out_first;
  a.max_units = c->max_units;
  a.dbg_flags = c->dbg_flags;
  a.dbg_arg = c->dbg_arg;
  a.spin_limit_ns = c->spin_limit_ns;
  // a skipped arrival is a one-shot request
  c->dbg_flags &= ~MK_DBG_SKIP_ARRIVAL;
  auto go = [&](int lo, int hi, int lm) {
    a.slice_lo = lo;
    a.slice_hi = hi;
    a.run_lm = lm;
    void* args[] = {&a};
    return cudaLaunchCooperativeKernel(c->kern.fn, dim3(c->grid), dim3(kBlockThreads), args,
                                       (size_t)launch_smem_bytes(c->kern, n), st);
  };
  const int groups = 4 * c->d.n_layers;
  cudaError_t e = cudaSuccess;
  if (c->dbg_flags & MK_DBG_SPLIT) {
    // one launch per phase group, then lm_head: kernel boundaries in place of
    // the grid barriers between groups
    for (int s = 0; s < groups && e == cudaSuccess; ++s) {
      e = go(s, s + 1, 0);
      a.n_upd = 0;  // the first launch entered the new pages
    }
    if (e == cudaSuccess) e = go(groups, groups, 1);
  } else {
    e = go(0, groups, 1);
  }
  if (e != cudaSuccess) {
    rollback();
    return fail(MK_ERR_CUDA, std::string("cudaLaunchCooperativeKernel: ") + cudaGetErrorString(e));
  }
  c->last_chunk = a.chunk;
  c->last_units = a.n_units;
  return MK_OK;
}

}  // namespace

namespace mk {

int host_fail(int code, const char* msg) { return fail(code, msg); }
int host_validate_desc(const mk_model_desc* d, int* shape) { return validate_desc(d, shape); }
void host_clear_error() { g_err.clear(); }

size_t host_carve_scratch(const mk_model_desc& d, int grid, int max_units, char* base, Scratch* sc) {
  return carve_scratch(d, grid, max_units, base, sc);
}

void host_attention_split(int n_kv_heads, int grid, int tile_tokens, const int32_t* pos, int n, int* chunk,
                          int* units) {
  host_attention_split_impl(n_kv_heads, grid, tile_tokens, pos, n, chunk, units);
}

int host_check_model(const mk_model_desc* d, const mk_weights* w, int* shape, LayerW* lw) {
  if (int r = validate_desc(d, shape)) return r;
  if (!w || !w->layers) return fail(MK_ERR_INVALID_ARG, "weights or weights->layers is NULL");
  const bool int4 = d->wdtype == MK_INT4_G64;
  if (int r = check_aux(w->embed, "embed", -1)) return r;
  if (int r = check_aux(w->final_norm, "final_norm", -1)) return r;
  if (int r = check_lin(w->lm_head, int4, "lm_head", -1)) return r;
  for (int l = 0; l < d->n_layers; ++l) {
    const mk_layer_weights& L = w->layers[l];
    LayerW& o = lw[l];
    std::memset(&o, 0, sizeof(o));
    if (int r = check_aux(L.attn_norm, "attn_norm", l)) return r;
    if (int r = check_aux(L.ffn_norm, "ffn_norm", l)) return r;
    const mk_linear* lin[NLIN] = {&L.wq, &L.wk, &L.wv, &L.wo, &L.gate, &L.up, &L.down,
                                  &L.exp_gate, &L.exp_up, &L.exp_down};
    static const char* names[NLIN] = {"wq", "wk", "wv", "wo", "gate", "up", "down",
                                      "exp_gate", "exp_up", "exp_down"};
    const bool dense = l < d->n_dense;
    for (int k = 0; k < NLIN; ++k) {
      const bool used = k <= WO || (dense ? (k >= GATE && k <= DOWN) : k >= EGATE);
      if (!used) continue;
      const bool scaled = quantised(k >= EGATE ? d->expert_wdtype : d->wdtype);
      if (int r = check_lin(*lin[k], scaled, names[k], l)) return r;
      o.w[k] = lin[k]->w;
      o.s[k] = scaled ? lin[k]->scales : nullptr;
    }
    if (!dense) {
      if (int r = check_aux(L.router, "router", l)) return r;
      o.router = L.router;
    }
    o.attn_norm = L.attn_norm;
    o.ffn_norm = L.ffn_norm;
  }
  return MK_OK;
}

}  // namespace mk

extern "C" {

MK_API const char* mk_last_error(void) { return g_err.c_str(); }

MK_API size_t mk_trace_bytes(const mk_model_desc* d, int32_t rows) {
  if (!d || rows < 0) return 0;
  const size_t L = d->n_layers, R = rows;
  return sizeof(float) * (L * R * ((size_t)d->hidden + (size_t)d->n_heads * d->head_dim +
                                   d->n_experts + 2 * (size_t)d->top_k) +
                          R * (size_t)d->vocab);
}

MK_API int mk_create(const mk_model_desc* d, const mk_weights* w, mk_ctx** out) {
  g_err.clear();
  if (!out) return fail(MK_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int shape = -1;
  if (int r = validate_desc(d, &shape)) return r;
  std::vector<LayerW> lw(d->n_layers);
  if (int r = host_check_model(d, w, &shape, lw.data())) return r;
  const bool int4 = d->wdtype == MK_INT4_G64;

  mk_ctx* c = new mk_ctx();
  c->d = *d;
  c->shape = shape;
  c->kern = get_kernel(shape, d->wdtype, d->expert_wdtype);
  auto bail = [&](int code) {
    mk_destroy(c);
    return code;
  };
  if (!c->kern.fn) {
    delete c;
    return fail(MK_ERR_UNSUPPORTED, "no kernel for this shape and dtype");
  }
  cudaError_t e = cudaGetDevice(&c->device);
  if (e != cudaSuccess) {
    delete c;
    return fail(MK_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  }
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, c->device);
  if (e != cudaSuccess) {
    delete c;
    return fail(MK_ERR_CUDA, std::string("cudaGetDeviceProperties: ") + cudaGetErrorString(e));
  }
  if (prop.major != 10 || prop.minor != 3) {
    delete c;
    return fail(MK_ERR_UNSUPPORTED, "the library is built for sm_103a (GB300) only");
  }
  if (!prop.cooperativeLaunch) {
    delete c;
    return fail(MK_ERR_UNSUPPORTED, "device does not support cooperative launch");
  }
  c->num_sms = prop.multiProcessorCount;
  c->grid = c->num_sms;
  if ((d->hidden / 4 + c->grid - 1) / c->grid * 4 > kMaxRowsPerBlock) {
    delete c;
    return fail(MK_ERR_UNSUPPORTED, "too few SMs for the compiled per-block row budget");
  }
  e = cudaFuncSetAttribute(c->kern.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, c->kern.smem_bytes);
  // prefer L1: each launch then gets the smallest shared-memory carve-out its
  // dynamic size needs
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(c->kern.fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxL1);
  if (e != cudaSuccess) {
    delete c;
    return fail(MK_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
  }
  int nb = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, c->kern.fn, kBlockThreads, c->kern.smem_bytes);
  if (e != cudaSuccess || nb < 1) {
    delete c;
    return fail(MK_ERR_UNSUPPORTED, "one block per SM cannot be resident (occupancy check)");
  }

  // weights: the linear layers are copied into the packed layout (mk_pack.cu);
  // embedding, norms and router stay borrowed
  c->embed = w->embed;
  c->final_norm = w->final_norm;
  c->lm_head = w->lm_head.w;
  c->lm_head_s = int4 ? w->lm_head.scales : nullptr;
  {
    PackLayout pl;
    c->packed_bytes = host_pack_layout(*d, &pl);
    e = cudaMalloc(&c->packed_dev, c->packed_bytes);
    if (e != cudaSuccess)
      return bail(fail(MK_ERR_CUDA, std::string("cudaMalloc(packed weights): ") + cudaGetErrorString(e)));
    if (int r = host_pack(*d, *w, c->packed_dev, 0)) return bail(r);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return bail(fail(MK_ERR_CUDA, std::string("weight pack: ") + cudaGetErrorString(e)));
    for (int l = 0; l < d->n_layers; ++l)
      for (int k = 0; k < NPK; ++k) lw[l].pk[k] = c->packed_dev + pl.layer[l][k];
    c->lm_pk = c->packed_dev + pl.lm;
  }
  c->layers_host = lw;
  if (int r = prefill_setup_attributes(*d)) return bail(r);
  e = cudaMalloc(&c->layers_dev, sizeof(LayerW) * d->n_layers);
  if (e != cudaSuccess) return bail(fail(MK_ERR_CUDA, std::string("cudaMalloc(layers): ") + cudaGetErrorString(e)));
  e = cudaMemcpy(c->layers_dev, lw.data(), sizeof(LayerW) * d->n_layers, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return bail(fail(MK_ERR_CUDA, std::string("cudaMemcpy(layers): ") + cudaGetErrorString(e)));

  // RoPE table in double precision: angle = pos * theta^(-2i/d)
  const int half = d->head_dim / 2;
  std::vector<float2> rope((size_t)d->max_ctx * half);
  for (int p = 0; p < d->max_ctx; ++p)
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow((double)d->rope_theta, -2.0 * i / d->head_dim);
      const double ang = (double)p * inv;
      rope[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
  e = cudaMalloc(&c->rope_dev, sizeof(float2) * rope.size());
  if (e != cudaSuccess) return bail(fail(MK_ERR_CUDA, std::string("cudaMalloc(rope): ") + cudaGetErrorString(e)));
  e = cudaMemcpy(c->rope_dev, rope.data(), sizeof(float2) * rope.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return bail(fail(MK_ERR_CUDA, std::string("cudaMemcpy(rope): ") + cudaGetErrorString(e)));

  // scratch
  c->max_units = c->grid + d->n_kv_heads * kMaxBatch;
  c->scratch_bytes = carve_scratch(*d, c->grid, c->max_units, nullptr, nullptr);
  e = cudaMalloc(&c->scratch_dev, c->scratch_bytes);
  if (e != cudaSuccess) return bail(fail(MK_ERR_CUDA, std::string("cudaMalloc(scratch): ") + cudaGetErrorString(e)));
  e = cudaMemset(c->scratch_dev, 0, c->scratch_bytes);
  if (e != cudaSuccess) return bail(fail(MK_ERR_CUDA, std::string("cudaMemset(scratch): ") + cudaGetErrorString(e)));
  carve_scratch(*d, c->grid, c->max_units, (char*)c->scratch_dev, &c->sc);

  c->max_pages_per_seq = (d->max_ctx + kPageTokens - 1) / kPageTokens;
  c->seqs.assign(d->max_seqs, Seq{});
  *out = c;
  return MK_OK;
}

MK_API int mk_kv_alloc(mk_ctx* c, int32_t n_pages) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (n_pages < 1) return fail(MK_ERR_INVALID_ARG, "n_pages must be >= 1");
  if (c->kv_dev) return fail(MK_ERR_STATE, "the KV pool is already allocated");
  const mk_model_desc& d = c->d;
  c->kv_bytes = sizeof(uint16_t) * (size_t)d.n_layers * n_pages * 2 * d.n_kv_heads * kPageTokens * d.head_dim;
  MK_CUDA(cudaMalloc(&c->kv_dev, c->kv_bytes));
  const size_t bt = sizeof(int32_t) * (size_t)d.max_seqs * c->max_pages_per_seq;
  cudaError_t e = cudaMalloc(&c->block_table_dev, bt);
  if (e == cudaSuccess) e = cudaMemset(c->block_table_dev, 0xFF, bt);
  if (e != cudaSuccess) {
    cudaFree(c->kv_dev);
    cudaFree(c->block_table_dev);
    c->kv_dev = nullptr;
    c->block_table_dev = nullptr;
    return fail(MK_ERR_CUDA, std::string("block table: ") + cudaGetErrorString(e));
  }
  c->n_pages = n_pages;
  c->page_ref.assign(n_pages, 0);
  c->free_pages.clear();
  for (int32_t p = n_pages - 1; p >= 0; --p) c->free_pages.push_back(p);
  return MK_OK;
}

// A chunk of more than kMaxBatch positions: pages for all of it are taken
// and entered in the block table, then mk_prefill.cu runs the model over the
// chunk's rows layer by layer.
static int prefill_gemm_chunk(mk_ctx* c, int32_t seq_id, const int32_t* tokens_dev, int32_t n, int32_t start_pos,
                              int32_t* out_token_dev, cudaStream_t st) {
  Seq& q = c->seqs[seq_id];
  const int rows_traced = n - ((n - 1) / kMaxBatch) * kMaxBatch;  // what a launch-by-launch prefill leaves
  if ((c->dbg_flags & MK_DBG_TRACE) && c->trace_bytes < mk_trace_bytes(&c->d, rows_traced))
    return fail(MK_ERR_INVALID_ARG, "trace buffer is smaller than mk_trace_bytes(rows)");
  const int have = (int)q.pages.size();
  const int end_page = (start_pos + n + kPageTokens - 1) / kPageTokens;
  std::vector<int32_t> taken;
  for (int pi = have; pi < end_page; ++pi) {
    const int32_t pg = c->free_pages.back();  // availability was checked by the caller
    c->free_pages.pop_back();
    c->page_ref[pg] = 1;
    q.pages.push_back(pg);
    taken.push_back(pg);
  }
  auto rollback = [&]() {
    for (auto it = taken.rbegin(); it != taken.rend(); ++it) {
      q.pages.pop_back();
      c->page_ref[*it] = 0;
      c->free_pages.push_back(*it);
    }
    if (q.len == 0 && q.pages.empty()) q.open = false;
  };
  for (size_t i0 = 0; i0 < taken.size(); i0 += kMaxUpd) {
    KvXfer x;
    std::memset(&x, 0, sizeof(x));
    x.kv = c->kv_dev;
    x.block_table = c->block_table_dev;
    x.n_pages = c->n_pages;
    x.max_pages_per_seq = c->max_pages_per_seq;
    x.n_layers = c->d.n_layers;
    x.n_kv_heads = c->d.n_kv_heads;
    x.head_dim = c->d.head_dim;
    x.slot = seq_id;
    x.upd_index0 = have + (int)i0;
    for (size_t i = i0; i < std::min(taken.size(), i0 + kMaxUpd); ++i)
      x.upd[x.n_upd++] = PageUpd{seq_id, have + (int32_t)i, taken[i]};
    if (int r = launch_kv_xfer(x, st)) {
      rollback();
      return r;
    }
  }
  PrefillArgs a;
  std::memset(&a, 0, sizeof(a));
  a.d = c->d;
  a.layers = c->layers_host.data();
  a.embed = c->embed;
  a.final_norm = c->final_norm;
  a.lm_pk = c->lm_pk;
  a.rope = c->rope_dev;
  a.kv = c->kv_dev;
  a.block_table = c->block_table_dev;
  a.n_pages = c->n_pages;
  a.max_pages_per_seq = c->max_pages_per_seq;
  a.slot = seq_id;
  a.start = start_pos;
  a.n = n;
  a.tokens = tokens_dev;
  a.out_token = out_token_dev;
  if (c->dbg_flags & MK_DBG_TRACE) {
    a.trace = c->trace;
    a.trace_bytes = mk_trace_bytes(&c->d, rows_traced);
    a.trace_rows = rows_traced;
  }
  a.err = c->sc.err;
  if (int r = prefill_run(&c->prefill, a, st)) {
    rollback();
    return r;
  }
  q.len = start_pos + n;
  return MK_OK;
}

MK_API int mk_prefill_chunk(mk_ctx* c, int32_t seq_id, const int32_t* tokens_dev, int32_t n,
                            int32_t start_pos, int32_t* out_token_dev, void* stream) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (!tokens_dev) return fail(MK_ERR_INVALID_ARG, "tokens_dev is NULL");
  if (n < 1 || n > 4096) return fail(MK_ERR_INVALID_ARG, "n must be in [1, 4096]");
  if (seq_id < 0 || seq_id >= c->d.max_seqs) return fail(MK_ERR_INVALID_ARG, "seq_id out of range");
  if (!c->kv_dev) return fail(MK_ERR_STATE, "mk_kv_alloc has not been called");
  Seq& q = c->seqs[seq_id];
  const int len = q.open ? q.len : 0;
  if (start_pos != len) return fail(MK_ERR_STATE, "start_pos must equal the sequence length");
  if ((long long)start_pos + n > c->d.max_ctx) return fail(MK_ERR_INVALID_ARG, "positions exceed max_ctx");
  // pages this chunk needs, checked before anything is launched
  const int have = (int)q.pages.size();
  const int need = (start_pos + n + kPageTokens - 1) / kPageTokens - have;
  if (need > (int)c->free_pages.size()) return fail(MK_ERR_NO_PAGES, "KV page pool exhausted");
  q.open = true;
  cudaStream_t st = (cudaStream_t)stream;
  if (n > kMaxBatch) return prefill_gemm_chunk(c, seq_id, tokens_dev, n, start_pos, out_token_dev, st);
  const int B = c->d.max_batch;
  int32_t slots[kMaxBatch], pos[kMaxBatch];
  for (int off = 0; off < n; off += B) {
    const int rows = std::min(B, n - off);
    for (int i = 0; i < rows; ++i) {
      slots[i] = seq_id;
      pos[i] = start_pos + off + i;
    }
    const bool last = off + rows == n;
    const int out_first = (last && out_token_dev) ? rows - 1 : rows;
    if (int r = launch(c, slots, pos, rows, tokens_dev + off, out_token_dev, out_first, st)) {
      if (q.len == 0 && q.pages.empty()) q.open = false;
      return r;
    }
    q.len = start_pos + off + rows;
  }
  return MK_OK;
}

MK_API int mk_decode_step(mk_ctx* c, const int32_t* seq_ids, const int32_t* tokens_dev,
                          const int32_t* positions, int32_t n, int32_t* out_tokens_dev, void* stream) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (!seq_ids || !positions || !tokens_dev || !out_tokens_dev)
    return fail(MK_ERR_INVALID_ARG, "NULL argument");
  if (n < 1 || n > c->d.max_batch) return fail(MK_ERR_INVALID_ARG, "n must be in [1, max_batch]");
  if (!c->kv_dev) return fail(MK_ERR_STATE, "mk_kv_alloc has not been called");
  int need = 0;
  for (int i = 0; i < n; ++i) {
    const int s = seq_ids[i];
    if (s < 0 || s >= c->d.max_seqs) return fail(MK_ERR_INVALID_ARG, "seq_id out of range");
    for (int j = 0; j < i; ++j)
      if (seq_ids[j] == s) return fail(MK_ERR_INVALID_ARG, "seq_ids must be distinct");
    const Seq& q = c->seqs[s];
    const int len = q.open ? q.len : 0;
    if (positions[i] != len) return fail(MK_ERR_STATE, "position must equal the sequence length");
    if (positions[i] >= c->d.max_ctx) return fail(MK_ERR_INVALID_ARG, "position exceeds max_ctx");
    need += positions[i] % kPageTokens == 0;
  }
  if (need > (int)c->free_pages.size()) return fail(MK_ERR_NO_PAGES, "KV page pool exhausted");
  if (int r = launch(c, seq_ids, positions, n, tokens_dev, out_tokens_dev, 0, (cudaStream_t)stream))
    return r;
  for (int i = 0; i < n; ++i) {
    Seq& q = c->seqs[seq_ids[i]];
    q.open = true;
    q.len = positions[i] + 1;
  }
  return MK_OK;
}

MK_API int mk_seq_release(mk_ctx* c, int32_t seq_id) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (seq_id < 0 || seq_id >= c->d.max_seqs) return fail(MK_ERR_INVALID_ARG, "seq_id out of range");
  Seq& q = c->seqs[seq_id];
  if (!q.open) return fail(MK_ERR_STATE, "sequence is not open");
  for (auto it = q.pages.rbegin(); it != q.pages.rend(); ++it)
    if (--c->page_ref[*it] == 0) c->free_pages.push_back(*it);
  q = Seq{};
  return MK_OK;
}

// Common part of the KV transfers: a KvXfer with the context's pool.
static KvXfer xfer_base(const mk_ctx* c, int32_t seq_id) {
  KvXfer x;
  std::memset(&x, 0, sizeof(x));
  x.kv = c->kv_dev;
  x.block_table = c->block_table_dev;
  x.n_pages = c->n_pages;
  x.max_pages_per_seq = c->max_pages_per_seq;
  x.n_layers = c->d.n_layers;
  x.n_kv_heads = c->d.n_kv_heads;
  x.head_dim = c->d.head_dim;
  x.slot = seq_id;
  return x;
}

MK_API int mk_kv_write(mk_ctx* c, int32_t seq_id, int32_t start_pos, int32_t n, const void* src_dev,
                       void* stream) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (!src_dev || !aligned16(src_dev)) return fail(MK_ERR_INVALID_ARG, "src_dev is NULL or not 16-byte aligned");
  if (n < 1) return fail(MK_ERR_INVALID_ARG, "n must be >= 1");
  if (seq_id < 0 || seq_id >= c->d.max_seqs) return fail(MK_ERR_INVALID_ARG, "seq_id out of range");
  if (!c->kv_dev) return fail(MK_ERR_STATE, "mk_kv_alloc has not been called");
  Seq& q = c->seqs[seq_id];
  const int len = q.open ? q.len : 0;
  if (start_pos < 0 || start_pos > len) return fail(MK_ERR_STATE, "start_pos must be in [0, sequence length]");
  if ((long long)start_pos + n > c->d.max_ctx) return fail(MK_ERR_INVALID_ARG, "positions exceed max_ctx");
  // positions already held may be overwritten only in pages of this sequence alone
  for (int pi = start_pos / kPageTokens; pi < (int)q.pages.size() && pi * kPageTokens < start_pos + n; ++pi)
    if (c->page_ref[q.pages[pi]] > 1) return fail(MK_ERR_STATE, "position lies in a page shared with another sequence");
  const int have = (int)q.pages.size();
  const int need = (start_pos + n + kPageTokens - 1) / kPageTokens - have;
  if (need > (int)c->free_pages.size()) return fail(MK_ERR_NO_PAGES, "KV page pool exhausted");
  // segments of at most kMaxUpd - 1 pages, so one launch carries every new page it touches
  const int seg = (kMaxUpd - 1) * kPageTokens;
  const uint16_t* src = static_cast<const uint16_t*>(src_dev);
  // pages taken by a segment whose launch fails go back to the pool (the
  // block-table entries they were given are rewritten when next handed out)
  auto give_back = [&](const KvXfer& x) {
    for (int i = x.n_upd - 1; i >= 0; --i) {
      q.pages.pop_back();
      c->page_ref[x.upd[i].page] = 0;
      c->free_pages.push_back(x.upd[i].page);
    }
  };
  const size_t per_pos = (size_t)2 * c->d.n_kv_heads * c->d.head_dim;  // bf16 values of one position, one layer
  for (int off = 0; off < n; off += seg) {
    const int m = std::min(seg, n - off);
    KvXfer x = xfer_base(c, seq_id);
    x.start = start_pos + off;
    x.n = m;
    x.upd_index0 = (int)q.pages.size();
    const int end_page = (x.start + m + kPageTokens - 1) / kPageTokens;
    while ((int)q.pages.size() < end_page) {
      const int32_t pg = c->free_pages.back();
      c->free_pages.pop_back();
      c->page_ref[pg] = 1;
      x.upd[x.n_upd++] = PageUpd{seq_id, (int32_t)q.pages.size(), pg};
      q.pages.push_back(pg);
    }
    // the caller buffer holds all n positions per layer: copy layer by layer
    // when the call is split, else in one launch
    if (m == n) {
      x.src = src;
      if (int r = launch_kv_xfer(x, (cudaStream_t)stream)) {
        give_back(x);
        return r;
      }
    } else {
      for (int l = 0; l < c->d.n_layers; ++l) {
        KvXfer y = x;
        y.n_layers = 1;
        y.src = src + ((size_t)l * n + off) * per_pos;
        y.kv = c->kv_dev + (size_t)l * c->n_pages * 2 * c->d.n_kv_heads * kPageTokens * c->d.head_dim;
        if (l > 0) y.n_upd = 0;  // the entries are set by the first launch; reads use the list
        if (int r = launch_kv_xfer(y, (cudaStream_t)stream)) {
          give_back(x);
          return r;
        }
      }
    }
    q.open = true;
    q.len = std::max(q.len, x.start + m);
  }
  return MK_OK;
}

MK_API int mk_kv_read(mk_ctx* c, int32_t seq_id, int32_t start_pos, int32_t n, void* dst_dev, void* stream) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (!dst_dev || !aligned16(dst_dev)) return fail(MK_ERR_INVALID_ARG, "dst_dev is NULL or not 16-byte aligned");
  if (n < 1) return fail(MK_ERR_INVALID_ARG, "n must be >= 1");
  if (seq_id < 0 || seq_id >= c->d.max_seqs) return fail(MK_ERR_INVALID_ARG, "seq_id out of range");
  if (!c->kv_dev) return fail(MK_ERR_STATE, "mk_kv_alloc has not been called");
  const Seq& q = c->seqs[seq_id];
  if (!q.open || start_pos < 0 || (long long)start_pos + n > q.len)
    return fail(MK_ERR_STATE, "positions must lie within the open sequence");
  KvXfer x = xfer_base(c, seq_id);
  x.start = start_pos;
  x.n = n;
  x.dst = static_cast<uint16_t*>(dst_dev);
  x.upd_index0 = INT32_MAX;
  return launch_kv_xfer(x, (cudaStream_t)stream);
}

MK_API int mk_seq_fork(mk_ctx* c, int32_t src_seq, int32_t dst_seq, int32_t n_tokens, void* stream) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (src_seq < 0 || src_seq >= c->d.max_seqs || dst_seq < 0 || dst_seq >= c->d.max_seqs || src_seq == dst_seq)
    return fail(MK_ERR_INVALID_ARG, "sequence ids out of range or equal");
  if (!c->kv_dev) return fail(MK_ERR_STATE, "mk_kv_alloc has not been called");
  const Seq& a = c->seqs[src_seq];
  Seq& b = c->seqs[dst_seq];
  if (!a.open) return fail(MK_ERR_STATE, "source sequence is not open");
  if (b.open) return fail(MK_ERR_STATE, "destination sequence is already open");
  if (n_tokens < kPageTokens || n_tokens % kPageTokens != 0 || n_tokens > a.len)
    return fail(MK_ERR_INVALID_ARG, "n_tokens must be a positive multiple of 128 within the source's length");
  const int np = n_tokens / kPageTokens;
  for (int i0 = 0; i0 < np; i0 += kMaxUpd) {
    KvXfer x = xfer_base(c, dst_seq);
    x.upd_index0 = i0;
    for (int i = i0; i < std::min(np, i0 + kMaxUpd); ++i) x.upd[x.n_upd++] = PageUpd{dst_seq, i, a.pages[i]};
    if (int r = launch_kv_xfer(x, (cudaStream_t)stream)) return r;
  }
  b.pages.assign(a.pages.begin(), a.pages.begin() + np);
  for (int32_t pg : b.pages) ++c->page_ref[pg];
  b.open = true;
  b.len = n_tokens;
  return MK_OK;
}

MK_API int32_t mk_seq_length(mk_ctx* c, int32_t seq_id) {
  if (!c || seq_id < 0 || seq_id >= c->d.max_seqs || !c->seqs[seq_id].open) return -1;
  return c->seqs[seq_id].len;
}

MK_API int mk_sync(mk_ctx* c, void* stream) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  MK_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  int32_t err[4] = {0, 0, 0, 0};
  MK_CUDA(cudaMemcpy(err, c->sc.err, sizeof(err), cudaMemcpyDeviceToHost));
  if (err[0] != 0) {
    MK_CUDA(cudaMemset(c->sc.err, 0, sizeof(err)));
    static const char* sites[] = {"?", "grid barrier", "page table", "attention unit", "token id",
                                  "weight ring", "shared-memory plan", "flagged residual word"};
    const int site = err[1] >= 1 && err[1] <= SITE_FLAG ? err[1] : 0;
    return fail(err[0], std::string("device reported error ") + std::to_string(err[0]) + " at " +
                            sites[site] + " (site " + std::to_string(err[1]) + ", detail " +
                            std::to_string(err[2]) + ", " + std::to_string(err[3]) + ")");
  }
  return MK_OK;
}

MK_API int mk_set_debug(mk_ctx* c, uint32_t flags, uint32_t arg, void* trace_dev, size_t trace_bytes,
                        uint32_t spin_limit_us) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if ((flags & (MK_DBG_TRACE | MK_DBG_TIMING)) && (!trace_dev || trace_bytes == 0))
    return fail(MK_ERR_INVALID_ARG, "MK_DBG_TRACE / MK_DBG_TIMING need a buffer");
  if ((flags & MK_DBG_TRACE) && (flags & MK_DBG_TIMING))
    return fail(MK_ERR_INVALID_ARG, "MK_DBG_TRACE and MK_DBG_TIMING share the buffer: pick one");
  if ((flags & MK_DBG_SKIP_ARRIVAL) && (int)(arg & 0xffffu) >= c->grid)
    return fail(MK_ERR_INVALID_ARG, "MK_DBG_SKIP_ARRIVAL block index out of range");
  c->dbg_flags = flags;
  c->dbg_arg = arg;
  c->trace = (float*)trace_dev;
  c->trace_bytes = trace_bytes;
  c->spin_limit_ns = spin_limit_us ? (uint64_t)spin_limit_us * 1000ull : 1000000000ull;
  return MK_OK;
}

MK_API int mk_attention_plan(int32_t n_kv_heads, int32_t grid, int32_t tile_tokens, const int32_t* positions_host,
                             int32_t n, int32_t* chunk_out, int32_t* units_out) {
  g_err.clear();
  if (!positions_host || !chunk_out || !units_out) return fail(MK_ERR_INVALID_ARG, "NULL argument");
  if (n_kv_heads < 1 || grid < 1 || tile_tokens < 1 || n < 1 || n > kMaxBatch)
    return fail(MK_ERR_INVALID_ARG, "n_kv_heads, grid, tile_tokens >= 1 and n in 1..16");
  for (int i = 0; i < n; ++i)
    if (positions_host[i] < 0) return fail(MK_ERR_INVALID_ARG, "negative position");
  int ch = 0, u = 0;
  host_attention_split_impl(n_kv_heads, grid, tile_tokens, positions_host, n, &ch, &u);
  *chunk_out = ch;
  *units_out = u;
  return MK_OK;
}

MK_API int mk_get_info(mk_ctx* c, mk_info* info) {
  g_err.clear();
  if (!c || !info) return fail(MK_ERR_INVALID_ARG, "NULL argument");
  info->device = c->device;
  info->num_sms = c->num_sms;
  info->grid = c->grid;
  info->block_threads = kBlockThreads;
  info->smem_bytes = c->kern.smem_bytes;
  info->n_pages = c->n_pages;
  info->free_pages = (int32_t)c->free_pages.size();
  info->scratch_bytes = (int64_t)c->scratch_bytes;
  info->kv_bytes = (int64_t)c->kv_bytes;
  info->last_chunk = c->last_chunk;
  info->last_units = c->last_units;
  return MK_OK;
}

MK_API int mk_destroy(mk_ctx* c) {
  g_err.clear();
  if (!c) return MK_OK;
  cudaError_t e = cudaDeviceSynchronize();
  cudaFree(c->layers_dev);
  cudaFree(c->packed_dev);
  cudaFree(c->rope_dev);
  cudaFree(c->scratch_dev);
  cudaFree(c->kv_dev);
  cudaFree(c->block_table_dev);
  prefill_free(c->prefill);
  delete c;
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, std::string("cudaDeviceSynchronize: ") + cudaGetErrorString(e));
  return MK_OK;
}

}  // extern "C"
