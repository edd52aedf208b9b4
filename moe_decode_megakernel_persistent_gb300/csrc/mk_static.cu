// mk_decode_step_static: the decode step for callers that cannot allocate
// device memory -- a host that hands the library a fixed memory budget from
// its own allocator, or a loop that must not take the device-wide
// synchronisation a cudaMalloc / cudaFree can bring.  It launches the same
// decode kernel as mk_decode_step, but everything the library would
// otherwise cudaMalloc (the per-layer pointer table, the RoPE table and the
// kernel's scratch: residual stream, attention partials, router partials,
// expert activations, argmax candidates, barrier counters and the error
// word) lives in one file-scope device array of kStaticBytes bytes.  Every
// GPU that loads the library holds that array until the process exits.
// Weights (the logical tensors for embedding, norms and router, and the
// packed copy of the linear layers made by mk_pack_weights), the KV cache
// and its block table, tokens and outputs are the caller's memory.
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "mk_internal.h"

namespace mk {
namespace {

constexpr size_t kStaticBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kStaticRopePositions = 8192;         // positions the RoPE table covers
constexpr int kMaxDevices = 64;
constexpr int kMaxStaticLayers = 128;
constexpr int kMaxStaticHalf = 64;                 // head_dim / 2 of the compiled shapes

static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

// Set-up state per device: the array's device address and the RoPE table
// (theta, head_dim) and layer table it currently holds.  Host copies live in
// static storage, so a call allocates no memory on the host either.
struct DeviceState {
  bool ready = false;
  char* base = nullptr;
  float rope_theta = 0.f;
  int head_dim = 0;
  int n_layers = 0;
  size_t off_layers = 0;
  LayerW table[kMaxStaticLayers];
};
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
float2 g_rope_host[(size_t)kStaticRopePositions * kMaxStaticHalf];  // guarded by g_mu

size_t rope_bytes(int head_dim) {
  return sizeof(float2) * (size_t)kStaticRopePositions * (head_dim / 2);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Layout of the static array for a launch of `grid` blocks: RoPE table |
// layer table | kernel scratch.  Returns the bytes the model needs.
size_t static_need(const mk_model_desc& d, int grid, size_t* off_layers, size_t* off_scratch) {
  const int max_units = grid + d.n_kv_heads * kMaxBatch;
  const size_t ol = align256(rope_bytes(d.head_dim));
  const size_t os = align256(ol + sizeof(LayerW) * d.n_layers);
  if (off_layers) *off_layers = ol;
  if (off_scratch) *off_scratch = os;
  return os + host_carve_scratch(d, grid, max_units, nullptr, nullptr);
}

// With device `dev` current: the first call resolves the array's device
// address.  When the RoPE parameters or the layer table differ from what the
// array holds, the device is first drained (an earlier call, on any stream,
// may still be reading them), the tables are rewritten with synchronous
// copies, and the kernel scratch [off_scratch, off_scratch + scratch_bytes)
// is cleared: another model's scratch may have left, where this model keeps
// its flagged residual words, bytes whose tag half could match a current tag.
// Calls with the same model reach none of these steps.
int setup(int dev, const mk_model_desc& d, const LayerW* layers, size_t off_layers, size_t off_scratch,
          size_t scratch_bytes, char** base) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess)
      return host_fail(MK_ERR_CUDA, (std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e)).c_str());
    s.base = static_cast<char*>(ptr);
    s.ready = true;
  }
  const bool rope_changed = s.rope_theta != d.rope_theta || s.head_dim != d.head_dim;
  const bool table_changed = rope_changed || s.n_layers != d.n_layers || s.off_layers != off_layers ||
                             std::memcmp(s.table, layers, sizeof(LayerW) * d.n_layers) != 0;
  if (table_changed) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
      return host_fail(MK_ERR_CUDA, (std::string("waiting for earlier calls: ") + cudaGetErrorString(e)).c_str());
    if (rope_changed) {
      const int half = d.head_dim / 2;
      for (int p = 0; p < kStaticRopePositions; ++p)
        for (int i = 0; i < half; ++i) {
          const double ang = (double)p * std::pow((double)d.rope_theta, -2.0 * i / d.head_dim);
          g_rope_host[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
      e = cudaMemcpy(s.base, g_rope_host, rope_bytes(d.head_dim), cudaMemcpyHostToDevice);
      if (e != cudaSuccess) {
        s.rope_theta = 0.f;  // unknown contents: rebuilt by the next call
        return host_fail(MK_ERR_CUDA, (std::string("RoPE table upload: ") + cudaGetErrorString(e)).c_str());
      }
      s.rope_theta = d.rope_theta;
      s.head_dim = d.head_dim;
    }
    std::memcpy(s.table, layers, sizeof(LayerW) * d.n_layers);
    e = cudaMemcpy(s.base + off_layers, s.table, sizeof(LayerW) * d.n_layers, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      s.n_layers = 0;
      return host_fail(MK_ERR_CUDA, (std::string("layer table upload: ") + cudaGetErrorString(e)).c_str());
    }
    e = cudaMemset(s.base + off_scratch, 0, scratch_bytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      s.n_layers = 0;
      return host_fail(MK_ERR_CUDA, (std::string("scratch clear: ") + cudaGetErrorString(e)).c_str());
    }
    s.n_layers = d.n_layers;
    s.off_layers = off_layers;
  }
  *base = s.base;
  return MK_OK;
}

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" MK_API int mk_decode_step_static(
    const mk_model_desc* d, const mk_weights* w, const void* packed_dev, void* kv_dev, int32_t n_pages,
    int32_t* block_table_dev, int32_t max_pages_per_seq, const int32_t* slots_host,
    const int32_t* positions_host, const int32_t* pages_host, int32_t n,
    const int32_t* tokens_dev, int32_t* out_tokens_dev, int32_t* status_dev, void* stream) {
  host_clear_error();
  int shape = -1;
  if (!d || !w) return host_fail(MK_ERR_INVALID_ARG, "model description or weights is NULL");
  if (d->n_layers > kMaxStaticLayers)
    return host_fail(MK_ERR_INVALID_ARG, "more layers than the static layer table holds (128)");
  LayerW layers[kMaxStaticLayers];
  if (int r = host_check_model(d, w, &shape, layers)) return r;
  if (!packed_dev || (reinterpret_cast<uintptr_t>(packed_dev) & 255u) != 0)
    return host_fail(MK_ERR_INVALID_ARG, "packed weights (mk_pack_weights) missing or not 256-byte aligned");
  PackLayout pl;
  host_pack_layout(*d, &pl);
  const uint8_t* pk = static_cast<const uint8_t*>(packed_dev);
  for (int l = 0; l < d->n_layers; ++l)
    for (int k = 0; k < NPK; ++k) layers[l].pk[k] = pk + pl.layer[l][k];
  if (!kv_dev || !block_table_dev || !slots_host || !positions_host || !pages_host || !tokens_dev ||
      !out_tokens_dev)
    return host_fail(MK_ERR_INVALID_ARG, "NULL argument");
  if (n < 1 || n > d->max_batch) return host_fail(MK_ERR_INVALID_ARG, "n must be in [1, max_batch]");
  if (n_pages < 1 || max_pages_per_seq < 1)
    return host_fail(MK_ERR_INVALID_ARG, "n_pages and max_pages_per_seq must be >= 1");
  for (int i = 0; i < n; ++i) {
    if (slots_host[i] < 0 || slots_host[i] >= d->max_seqs)
      return host_fail(MK_ERR_INVALID_ARG, "slot out of range [0, max_seqs)");
    for (int j = 0; j < i; ++j)
      if (slots_host[j] == slots_host[i]) return host_fail(MK_ERR_INVALID_ARG, "slots must be distinct");
    const int p = positions_host[i];
    if (p < 0 || p >= d->max_ctx || p >= kStaticRopePositions)
      return host_fail(MK_ERR_INVALID_ARG,
                       "position out of range (the static RoPE table covers positions < 8192)");
    if (p / kPageTokens >= max_pages_per_seq)
      return host_fail(MK_ERR_INVALID_ARG, "position beyond max_pages_per_seq pages");
    if (pages_host[i] < 0 || pages_host[i] >= n_pages)
      return host_fail(MK_ERR_INVALID_ARG, "page out of range [0, n_pages)");
  }
  const KernelInfo kern = get_kernel(shape, d->wdtype, d->expert_wdtype);
  if (!kern.fn) return host_fail(MK_ERR_UNSUPPORTED, "no kernel for this shape and dtype");

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return host_fail(MK_ERR_CUDA, cudaGetErrorString(e));
  if (dev >= kMaxDevices) return host_fail(MK_ERR_UNSUPPORTED, "device ordinal >= 64");
  if ((d->hidden / 4 + sms - 1) / sms * 4 > kMaxRowsPerBlock)
    return host_fail(MK_ERR_UNSUPPORTED, "too few SMs for the compiled per-block row budget");

  const int grid = sms;
  const int max_units = grid + d->n_kv_heads * kMaxBatch;
  size_t off_layers = 0, off_scratch = 0;
  const size_t need = static_need(*d, grid, &off_layers, &off_scratch);
  if (need > kStaticBytes)
    return host_fail(MK_ERR_UNSUPPORTED,
                     ("model needs " + std::to_string(need) + " bytes of static scratch; the array holds " +
                      std::to_string(kStaticBytes)).c_str());

  if (d->head_dim / 2 > kMaxStaticHalf) return host_fail(MK_ERR_UNSUPPORTED, "head_dim above 128");
  char* base = nullptr;
  if (int r = setup(dev, *d, layers, off_layers, off_scratch, need - off_scratch, &base)) return r;
  e = cudaFuncSetAttribute(kern.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kern.smem_bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern.fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxL1);
  if (e != cudaSuccess) return host_fail(MK_ERR_CUDA, cudaGetErrorString(e));

  StepArgs a;
  std::memset(&a, 0, sizeof(a));
  host_carve_scratch(*d, grid, max_units, base + off_scratch, &a.sc);
  host_attention_split(d->n_kv_heads, grid, kern.tile_tokens, positions_host, n, &a.chunk, &a.n_units);
  if (a.n_units > max_units) return host_fail(MK_ERR_INVALID_ARG, "attention split exceeds its buffer");
  if (a.n_units > kMaxOwnUnits * grid) return host_fail(MK_ERR_INVALID_ARG, "more attention units than the grid can merge");
  for (int i = 0; i < n; ++i) {
    a.slot[i] = slots_host[i];
    a.pos[i] = positions_host[i];
    a.new0[i] = positions_host[i];  // one row per sequence
    a.cur_page[i] = pages_host[i];
    a.upd[a.n_upd++] = PageUpd{slots_host[i], positions_host[i] / kPageTokens, pages_host[i]};
  }
  a.layers = reinterpret_cast<const LayerW*>(base + off_layers);
  a.embed = w->embed;
  a.final_norm = w->final_norm;
  a.lm_head = w->lm_head.w;
  a.lm_head_s = d->wdtype == MK_INT4_G64 ? w->lm_head.scales : nullptr;
  a.lm_pk = pk + pl.lm;
  a.rope = reinterpret_cast<const float2*>(base);
  a.kv = static_cast<uint16_t*>(kv_dev);
  a.block_table = block_table_dev;
  a.tokens = tokens_dev;
  a.out_tokens = out_tokens_dev;
  a.n_pages = n_pages;
  a.max_pages_per_seq = max_pages_per_seq;
  a.n = n;
  a.n_layers = d->n_layers;
  a.n_dense = d->n_dense;
  a.vocab = d->vocab;
  a.eps = d->rms_eps;
  a.out_first = 0;
  a.max_units = max_units;
  a.spin_limit_ns = 1000000000ull;
  a.slice_lo = 0;
  a.slice_hi = 4 * d->n_layers;
  a.run_lm = 1;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: counters, merge counts and
  // the error word must start at zero; the launch epoch (sync[64], the tag of
  // the flagged residual words) must not, or a stale word would match
  e = cudaMemsetAsync(a.sc.merge_cnt, 0, sizeof(int32_t) * kMaxBatch * d->n_kv_heads, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.sc.sync, 0, sizeof(uint32_t) * 64, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.sc.sync + 96, 0, sizeof(uint32_t) * 32, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.sc.err, 0, sizeof(int32_t) * 4, st);
  if (e != cudaSuccess) return host_fail(MK_ERR_CUDA, cudaGetErrorString(e));
  void* args[] = {&a};
  e = cudaLaunchCooperativeKernel(kern.fn, dim3(grid), dim3(kBlockThreads), args,
                                  (size_t)launch_smem_bytes(kern, n), st);
  if (e != cudaSuccess)
    return host_fail(MK_ERR_CUDA, (std::string("cudaLaunchCooperativeKernel: ") + cudaGetErrorString(e)).c_str());
  if (status_dev) {
    e = cudaMemcpyAsync(status_dev, a.sc.err, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return host_fail(MK_ERR_CUDA, cudaGetErrorString(e));
  }
  return MK_OK;
}

extern "C" MK_API int mk_static_bytes(const mk_model_desc* d, int32_t grid, int64_t* need_out,
                                      int64_t* capacity_out) {
  host_clear_error();
  if (!need_out || !capacity_out) return host_fail(MK_ERR_INVALID_ARG, "NULL argument");
  int shape = -1;
  if (int r = host_validate_desc(d, &shape)) return r;
  if (grid < 1) return host_fail(MK_ERR_INVALID_ARG, "grid must be >= 1");
  if (d->n_layers > kMaxStaticLayers)
    return host_fail(MK_ERR_INVALID_ARG, "more layers than the static layer table holds (128)");
  *need_out = (int64_t)static_need(*d, grid, nullptr, nullptr);
  *capacity_out = (int64_t)kStaticBytes;
  return MK_OK;
}
