// Chunked prefill: mk_prefill_chunk for chunks of more than 16 positions runs
// the model over all positions of the chunk at once, layer by layer, instead
// of as one-launch decode steps of up to 16 rows.  "rec Megakernel and Tempo9
// Compared", §1 (Prefill), splits long prompts into 4096-token pieces; a
// piece is M <= 4096 rows here.
//
// The linear layers are dense contractions over the chunk's rows and run as
// tensor-core GEMMs (cuBLAS, fp32 accumulation).  bf16 weights are used in
// place with bf16 activation operands.  int4 and int3 weights are widened, per layer,
// from the library's packed records to fp16, which holds code * group scale
// exactly (a 3-bit code times an 8-bit bf16 scale needs at most 11 significant
// bits), with fp16 activation operands.  Every activation is split into two
// parts, hi + lo, so a projection is two GEMMs into one fp32 result (16
// significant bits of the activation with bf16, 22 with fp16); fp32 models
// use fp32 GEMMs.  Router logits are computed in fp32 by a kernel of this file.  Everything between the GEMMs is
// this file's kernels: embedding, RMSNorm and the split, RoPE and the paged K/V
// write, causal attention over the pages (fp32), residuals, the router's top-k,
// the grouping of rows by expert (in a fixed order), SiLU, the weighted expert
// sum in slot order, and for the last position the final norm, lm_head and
// argmax.
//
// GEMM outputs follow the packed record order of mk_pack.cu: QKV record 2p + r
// is RoPE pair task p, row i (r = 0) or i + hd/2 (r = 1); gate/up record 2t + r
// is gate (r = 0) / up (r = 1) of FFN row t; o_proj and down records are output
// rows.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cfloat>
#include <climits>
#include <string>
#include <vector>

#include "mk_internal.h"

namespace mk {

struct PrefillWork {
  cublasHandle_t blas = nullptr;
  int max_m = 0;
  size_t a_elems = 0, c_elems = 0, wb_elems = 0;
  float* X = nullptr;        // [M][H] residual
  float* Hr = nullptr;       // [M][H] residual after attention
  float* Q = nullptr;        // [M][QD] roped queries
  float* O = nullptr;        // [M][QD] attention output
  void* A = nullptr;         // activations: fp32 [rows][K], or bf16 hi then bf16 lo
  float* C = nullptr;        // GEMM output
  float* D = nullptr;        // expert down outputs [entries][H]
  uint16_t* Wb = nullptr;    // fp16 weights widened from int4
  float* Z = nullptr;        // [M][H] normalised FFN input (fp32, for the router)
  float* logits = nullptr;   // [M][E]
  int32_t* ids = nullptr;    // [M][TOPK]
  float* wts = nullptr;      // [M][TOPK]
  int32_t* cnt = nullptr;    // [E] counts, then [E + 1] offsets
  int32_t* ent = nullptr;    // [M * TOPK] row of the entry at each expert-sorted position
  int32_t* pos_of = nullptr; // [M * TOPK] expert-sorted position of entry (row, slot)
  float* lm_v = nullptr;     // lm_head per-block best logit
  int32_t* lm_i = nullptr;   // and token
  std::vector<int32_t> cnt_host;
};

namespace {

constexpr int kLmBlocks = 608;  // lm_head blocks (4 per SM of the GB300)

// activation operand formats
enum { ACT_F32 = 0, ACT_BF16 = 1, ACT_F16 = 2 };

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ float aux_val(const void* p, size_t i, bool f32) {
  return f32 ? reinterpret_cast<const float*>(p)[i] : bf2f(reinterpret_cast<const uint16_t*>(p)[i]);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];  // fixed order: every block gets the same bits
  return t;
}

// Store row values as the GEMM operand: fp32, or hi / lo parts (bf16 or fp16).
__device__ __forceinline__ void put_act(void* A, size_t lo_off, size_t idx, float v, int fmt) {
  if (fmt == ACT_F32) {
    reinterpret_cast<float*>(A)[idx] = v;
  } else if (fmt == ACT_BF16) {
    const uint16_t h = f2bf(v);
    reinterpret_cast<uint16_t*>(A)[idx] = h;
    reinterpret_cast<uint16_t*>(A)[lo_off + idx] = f2bf(v - bf2f(h));
  } else {
    const uint16_t h = f2h(v);
    reinterpret_cast<uint16_t*>(A)[idx] = h;
    reinterpret_cast<uint16_t*>(A)[lo_off + idx] = f2h(v - h2f(h));
  }
}

__global__ void k_embed(const int32_t* tok, const void* embed, bool f32, int H, int V, int M, float* X,
                        int32_t* err) {
  const int i = blockIdx.x;
  int t = tok[i];
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0 && atomicCAS(err, 0, MK_ERR_DEVICE_INDEX) == 0) {
      err[1] = SITE_TOKEN;
      err[2] = t;
    }
    t = 0;
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) X[(size_t)i * H + h] = aux_val(embed, (size_t)t * H + h, f32);
}

// out = split(rmsnorm(in) * w) (w null: no norm); with `add`, in = in + add
// is formed first and kept in `sum`; z (if not null) receives the fp32 values.
__global__ void k_norm_act(const float* in, const float* add, float* sum, const void* w, bool aux_f32, float eps,
                           int K, void* A, size_t lo_off, int fmt, float* z) {
  __shared__ float red[32];
  const int i = blockIdx.x;
  const float* x = in + (size_t)i * K;
  float ss = 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float v = x[k];
    if (add) {
      v += add[(size_t)i * K + k];
      sum[(size_t)i * K + k] = v;
    }
    ss += v * v;
  }
  float r = 1.f;
  if (w) r = rsqrtf(block_sum(ss, red) / K + eps);
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float v = add ? sum[(size_t)i * K + k] : x[k];
    if (w) v = v * r * aux_val(w, k, aux_f32);
    if (z) z[(size_t)i * K + k] = v;
    put_act(A, lo_off, (size_t)i * K + k, v, fmt);
  }
}

// int4 records (codes, then bf16 group scales) -> fp16 rows [rows][K]: exact
// (a code of at most 3 significant bits times an 8-bit scale fits fp16's 11;
// the model's scales are far above fp16's subnormal range).
__global__ void k_widen_int4(const uint8_t* rec, int rec_bytes, int K, long long rows, uint16_t* out) {
  const long long total = rows * (K / 2);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / (K / 2);
    const int j = (int)(i % (K / 2));
    const uint8_t* p = rec + (size_t)r * rec_bytes;
    const uint8_t b = p[j];
    const float s = bf2f(reinterpret_cast<const uint16_t*>(p + K / 2)[(2 * j) / 64]);
    const int q0 = (int)(b & 0xF) - ((b & 0x8) ? 16 : 0);
    const int q1 = (int)(b >> 4) - ((b & 0x80) ? 16 : 0);
    out[(size_t)r * K + 2 * j] = f2h((float)q0 * s);
    out[(size_t)r * K + 2 * j + 1] = f2h((float)q1 * s);
  }
}

// int3 records (the kernel's bit planes, then bf16 group scales; see
// mk_pack.cu) -> fp16 rows [rows][K]: exact as for int4 (|q| <= 4).
__global__ void k_widen_int3(const uint8_t* rec, int rec_bytes, int K, long long rows, uint16_t* out) {
  const int nch = K / 32;
  const long long total = rows * K;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / K;
    const int k = (int)(i % K), c = k / 32, v = k % 32;
    const int t = v / 8, bi = (v % 8) / 2, e = v % 2;
    const uint8_t* p = rec + (size_t)r * rec_bytes;
    const uint32_t lw = reinterpret_cast<const uint32_t*>(p + 8 * c)[t / 2];
    const uint32_t hw = reinterpret_cast<const uint32_t*>(p + 8 * nch)[c];
    const int u = (int)(((lw >> (8 * bi + 2 * (2 * (t % 2) + e))) & 3u) | (((hw >> (8 * bi + 2 * t + e)) & 1u) << 2));
    const float s = bf2f(reinterpret_cast<const uint16_t*>(p + 3 * K / 8)[k / 64]);
    out[(size_t)r * K + k] = f2h((float)(u - 4) * s);
  }
}

// QKV records -> roped q (fp32) and K / V (bf16) into the pages.
__global__ void k_qkv_epi(const float* C, int NQKV, int NH, int NKV, int HD, const float2* rope, int start, int M,
                          float* Q, uint16_t* kv, const int32_t* bt, int slot, int mpps, int n_pages, int layer,
                          int32_t* err) {
  const int HALF = HD / 2, NQP = NH * HALF, NKP = NKV * HALF, QD = NH * HD;
  const long long total = (long long)M * (NQP + 2 * NKP);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(idx / (NQP + 2 * NKP)), p = (int)(idx % (NQP + 2 * NKP));
    const float v0 = C[(size_t)i * NQKV + 2 * p], v1 = C[(size_t)i * NQKV + 2 * p + 1];
    const int pos = start + i;
    if (p < NQP + NKP) {
      const int q = p < NQP ? p : p - NQP;
      const int hh = q / HALF, ii = q % HALF;
      const float2 cs = rope[(size_t)pos * HALF + ii];
      const float e0 = v0 * cs.x - v1 * cs.y, e1 = v1 * cs.x + v0 * cs.y;
      if (p < NQP) {
        Q[(size_t)i * QD + hh * HD + ii] = e0;
        Q[(size_t)i * QD + hh * HD + ii + HALF] = e1;
        continue;
      }
      const int page = bt[slot * mpps + pos / kPageTokens];
      if (page < 0 || page >= n_pages) {
        if (atomicCAS(err, 0, MK_ERR_DEVICE_INDEX) == 0) { err[1] = SITE_PAGE; err[2] = pos; }
        continue;
      }
      uint16_t* dst = kv + ((((size_t)layer * n_pages + page) * 2 + 0) * NKV + hh) * (size_t)(kPageTokens * HD) +
                      (size_t)(pos % kPageTokens) * HD;
      dst[ii] = f2bf(e0);
      dst[ii + HALF] = f2bf(e1);
    } else {
      const int q = p - NQP - NKP, g = q / HALF, ii = q % HALF;
      const int page = bt[slot * mpps + pos / kPageTokens];
      if (page < 0 || page >= n_pages) continue;
      uint16_t* dst = kv + ((((size_t)layer * n_pages + page) * 2 + 1) * NKV + g) * (size_t)(kPageTokens * HD) +
                      (size_t)(pos % kPageTokens) * HD;
      dst[ii] = f2bf(v0);
      dst[ii + HALF] = f2bf(v1);
    }
  }
}

// Causal attention of the chunk's rows over every cached position up to
// their own, paged, grouped-query.  One block per (16 rows, kv head): the
// GQA q heads x 16 rows = VPB query vectors; keys in tiles of 64 positions
// (K and V, bf16, in shared memory).  Warp w owns query vectors w*VPW ..; a
// lane owns keys 2 lane, 2 lane + 1 of a tile for the scores and dims
// DPL*lane .. of the output.  Online softmax in fp32.
template <int HD, int GQA>
__global__ void __launch_bounds__(256) k_attention(const float* Q, const uint16_t* kv, const int32_t* bt, int slot,
                                                   int mpps, int n_pages, int layer, int NKV, int start, int M,
                                                   float scale, float* O) {
  constexpr int RT = 16, VPB = GQA * RT, NW = 8, VPW = VPB / NW, DPL = HD / 32, KT = 64, KS = HD + 2;
  static_assert(VPB % NW == 0 && HD % 32 == 0, "shape");
  extern __shared__ __align__(16) uint8_t smp[];
  float* qs = reinterpret_cast<float*>(smp);                   // [VPB][HD]
  uint16_t* ks = reinterpret_cast<uint16_t*>(qs + VPB * HD);   // [KT][KS]
  uint16_t* vs = ks + KT * KS;                                 // [KT][HD]
  float* ps = reinterpret_cast<float*>(vs + KT * HD);          // [NW][VPW][KT]
  const int g = blockIdx.y, i0 = blockIdx.x * RT;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int NH = NKV * GQA, QD = NH * HD;
  // query vector v = hl * RT + r: head g * GQA + hl, row i0 + r
  for (int e = threadIdx.x; e < VPB * HD; e += blockDim.x) {
    const int v = e / HD, d = e % HD, r = v % RT, hl = v / RT;
    qs[e] = (i0 + r < M) ? Q[(size_t)(i0 + r) * QD + (g * GQA + hl) * HD + d] * scale : 0.f;
  }
  float m[VPW], l[VPW], o[VPW][DPL];
#pragma unroll
  for (int j = 0; j < VPW; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int dd = 0; dd < DPL; ++dd) o[j][dd] = 0.f;
  }
  const int last = start + min(M, i0 + RT) - 1;  // the block's last query position
  for (int t0 = 0; t0 <= last; t0 += KT) {
    __syncthreads();
    for (int e = threadIdx.x; e < KT * HD / 8; e += blockDim.x) {  // 16-byte words of K and V rows
      const int kk = e / (HD / 8), wd = e % (HD / 8), t = t0 + kk;
      uint4 kw = make_uint4(0u, 0u, 0u, 0u), vw = kw;
      if (t <= last) {
        const int page = bt[slot * mpps + t / kPageTokens];
        if (page >= 0 && page < n_pages) {
          const size_t base = (((size_t)layer * n_pages + page) * 2 * NKV + g) * (size_t)(kPageTokens * HD) +
                              (size_t)(t % kPageTokens) * HD + 8 * wd;
          kw = *reinterpret_cast<const uint4*>(kv + base);
          vw = *reinterpret_cast<const uint4*>(kv + base + (size_t)NKV * kPageTokens * HD);
        }
      }
      const uint32_t kk4[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) *reinterpret_cast<uint32_t*>(ks + kk * KS + 8 * wd + 2 * u) = kk4[u];
      *reinterpret_cast<uint4*>(vs + kk * HD + 8 * wd) = vw;
    }
    __syncthreads();
    // scores of this lane's two keys for the warp's vectors
    float s[VPW][2];
#pragma unroll
    for (int j = 0; j < VPW; ++j) s[j][0] = s[j][1] = 0.f;
    const uint16_t* k0 = ks + (2 * lane) * KS;
    const uint16_t* k1 = k0 + KS;
#pragma unroll 4
    for (int d = 0; d < HD; d += 2) {
      const uint32_t a = *reinterpret_cast<const uint32_t*>(k0 + d), b = *reinterpret_cast<const uint32_t*>(k1 + d);
      const float a0 = __uint_as_float(a << 16), a1 = __uint_as_float(a & 0xFFFF0000u);
      const float b0 = __uint_as_float(b << 16), b1 = __uint_as_float(b & 0xFFFF0000u);
#pragma unroll
      for (int j = 0; j < VPW; ++j) {
        const float2 q = *reinterpret_cast<const float2*>(qs + (w * VPW + j) * HD + d);
        s[j][0] = fmaf(q.x, a0, fmaf(q.y, a1, s[j][0]));
        s[j][1] = fmaf(q.x, b0, fmaf(q.y, b1, s[j][1]));
      }
    }
    float* pw = ps + (size_t)w * VPW * KT;
#pragma unroll
    for (int j = 0; j < VPW; ++j) {
      const int v = w * VPW + j, qpos = start + i0 + v % RT;
      const int ta = t0 + 2 * lane, tb = ta + 1;
      const float sa = ta <= qpos ? s[j][0] : -INFINITY, sb = tb <= qpos ? s[j][1] : -INFINITY;
      float mx = fmaxf(sa, sb);
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[j], mx);
      const float corr = mn == -INFINITY ? 1.f : expf(m[j] - mn);
      const float pa = sa == -INFINITY ? 0.f : expf(sa - mn), pb = sb == -INFINITY ? 0.f : expf(sb - mn);
      float ls = pa + pb;
      for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      l[j] = l[j] * corr + ls;
      m[j] = mn;
#pragma unroll
      for (int dd = 0; dd < DPL; ++dd) o[j][dd] *= corr;
      pw[j * KT + 2 * lane] = pa;
      pw[j * KT + 2 * lane + 1] = pb;
    }
    __syncwarp();
    for (int kk = 0; kk < KT; ++kk) {
      float vv[DPL];
#pragma unroll
      for (int dd = 0; dd < DPL; ++dd) vv[dd] = bf2f(vs[kk * HD + DPL * lane + dd]);
#pragma unroll
      for (int j = 0; j < VPW; ++j) {
        const float p = pw[j * KT + kk];
#pragma unroll
        for (int dd = 0; dd < DPL; ++dd) o[j][dd] = fmaf(p, vv[dd], o[j][dd]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < VPW; ++j) {
    const int v = w * VPW + j, r = v % RT, hl = v / RT;
    if (i0 + r >= M) continue;
    const float inv = 1.f / l[j];
#pragma unroll
    for (int dd = 0; dd < DPL; ++dd)
      O[(size_t)(i0 + r) * QD + (g * GQA + hl) * HD + DPL * lane + dd] = o[j][dd] * inv;
  }
}

// act = silu(gate) * up from interleaved gate/up columns; split for the down GEMM.
__global__ void k_silu_act(const float* C, int rows, int F, void* A, size_t lo_off, int fmt) {
  const long long total = (long long)rows * F;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long i = idx / F;
    const int f = (int)(idx % F);
    const float g = C[(size_t)i * 2 * F + 2 * f], u = C[(size_t)i * 2 * F + 2 * f + 1];
    put_act(A, lo_off, (size_t)idx, g / (1.f + expf(-g)) * u, fmt);
  }
}

__global__ void k_add(const float* a, const float* b, float* out, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    out[i] = a[i] + b[i];
}

// Router logits in fp32: logits[i][e] = z[i] . router[e]; one warp per
// (row, expert), lanes over K in a fixed order.
__global__ void k_router(const float* z, const void* router, bool aux_f32, int M, int E, int H, float* logits) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long wi = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); wi < (long long)M * E;
       wi += nwarps) {
    const int i = (int)(wi / E), e = (int)(wi % E);
    float acc = 0.f;
    for (int k = lane; k < H; k += 32) acc = fmaf(z[(size_t)i * H + k], aux_val(router, (size_t)e * H + k, aux_f32), acc);
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) logits[wi] = acc;
  }
}

// Softmax over the experts, top-k (ties to the lower id), weights renormalised
// over the selection.  One warp per row; E <= 64.
__global__ void k_route(const float* logits, int M, int E, int K, int32_t* ids, float* wts) {
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= M) return;
  const float* lg = logits + (size_t)i * E;
  float v[2];
  int rank[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int e = lane + 32 * u;
    v[u] = e < E ? lg[e] : -INFINITY;
    rank[u] = 0;
    if (e < E)
      for (int e2 = 0; e2 < E; ++e2) {
        const float w2 = lg[e2];
        rank[u] += (w2 > v[u]) || (w2 == v[u] && e2 < e);
      }
  }
  float mx = fmaxf(v[0], v[1]);
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sel = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u)
    if (lane + 32 * u < E && rank[u] < K) sel += expf(v[u] - mx);
  for (int off = 16; off > 0; off >>= 1) sel += __shfl_xor_sync(0xffffffffu, sel, off);
#pragma unroll
  for (int u = 0; u < 2; ++u)
    if (lane + 32 * u < E && rank[u] < K) {
      ids[(size_t)i * K + rank[u]] = lane + 32 * u;
      wts[(size_t)i * K + rank[u]] = expf(v[u] - mx) / sel;
    }
}

// Entries (row, slot) grouped by expert, in row-then-slot order within an
// expert: counts, offsets, the row of every sorted position and the sorted
// position of every entry.  One thread per expert scans the entries in order.
__global__ void k_group(const int32_t* ids, int n_ent, int E, int K, int32_t* cnt, int32_t* ent, int32_t* pos_of) {
  __shared__ int off[65];
  const int e = threadIdx.x;
  int c = 0;
  if (e < E)
    for (int j = 0; j < n_ent; ++j) c += ids[j] == e;
  if (e < E) cnt[e] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int x = 0; x < E; ++x) {
      off[x] = acc;
      acc += cnt[x];
    }
    off[E] = acc;
    for (int x = 0; x <= E; ++x) cnt[E + x] = off[x];
  }
  __syncthreads();
  if (e < E) {
    int p = off[e];
    for (int j = 0; j < n_ent; ++j)
      if (ids[j] == e) {
        ent[p] = j / K;
        pos_of[j] = p;
        ++p;
      }
  }
}

// Rows of the activation matrix gathered into expert-sorted order.
__global__ void k_gather(const void* A, size_t lo_in, void* G, size_t lo_out, const int32_t* ent, int n_ent, int K,
                         int fmt) {
  const long long total = (long long)n_ent * K;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long p = idx / K;
    const int k = (int)(idx % K);
    const size_t src = (size_t)ent[p] * K + k;
    if (fmt == ACT_F32) {
      reinterpret_cast<float*>(G)[idx] = reinterpret_cast<const float*>(A)[src];
    } else {
      reinterpret_cast<uint16_t*>(G)[idx] = reinterpret_cast<const uint16_t*>(A)[src];
      reinterpret_cast<uint16_t*>(G)[lo_out + idx] = reinterpret_cast<const uint16_t*>(A)[lo_in + src];
    }
  }
}

// x = h + sum over the slots, in slot order, of weight * expert output.
__global__ void k_combine(const float* Hr, const float* D, const float* wts, const int32_t* pos_of, int M, int H,
                          int K, float* X) {
  const long long total = (long long)M * H;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long i = idx / H;
    const int h = (int)(idx % H);
    float s = 0.f;
    for (int k = 0; k < K; ++k) s = fmaf(wts[i * K + k], D[(size_t)pos_of[i * K + k] * H + h], s);
    X[idx] = Hr[idx] + s;
  }
}

// Trace of the chunk's last rows (the layout of mk_trace_bytes).
__global__ void k_trace_rows(const float* src, int ld, int r0, int rows, int width, float* dst) {
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < rows * width; idx += gridDim.x * blockDim.x)
    dst[idx] = src[(size_t)(r0 + idx / width) * ld + idx % width];
}
__global__ void k_trace_topk(const int32_t* ids, const float* wts, int r0, int rows, int K, float* dst) {
  for (int idx = threadIdx.x; idx < rows * K; idx += blockDim.x) {
    const int r = idx / K, k = idx % K;
    dst[r * 2 * K + k] = (float)ids[(size_t)(r0 + r) * K + k];
    dst[r * 2 * K + K + k] = wts[(size_t)(r0 + r) * K + k];
  }
}

// Final norm of one row, lm_head over the vocabulary, argmax (larger logit,
// then the lower id): per-block candidates, then one block reduces them in
// block order.
__global__ void k_lm_head(const float* x, const void* fnorm, bool aux_f32, float eps, int H, const uint8_t* lm,
                          int rec, int wdtype, int V, float* cand_v, int32_t* cand_i, float* trace_logits) {
  extern __shared__ float ys[];
  __shared__ float red[32];
  __shared__ float bv[32];
  __shared__ int bi[32];
  float ss = 0.f;
  for (int k = threadIdx.x; k < H; k += blockDim.x) ss += x[k] * x[k];
  const float r = rsqrtf(block_sum(ss, red) / H + eps);
  for (int k = threadIdx.x; k < H; k += blockDim.x) ys[k] = x[k] * r * aux_val(fnorm, k, aux_f32);
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float best = -INFINITY;
  int bid = INT_MAX;
  for (int row = blockIdx.x * nw + w; row < V; row += gridDim.x * nw) {
    const uint8_t* p = lm + (size_t)row * rec;
    float acc = 0.f;
    if (wdtype == MK_INT4_G64) {
      for (int j = lane; j < H / 2; j += 32) {
        const uint8_t b = p[j];
        const float s = bf2f(reinterpret_cast<const uint16_t*>(p + H / 2)[(2 * j) / 64]);
        const int q0 = (int)(b & 0xF) - ((b & 0x8) ? 16 : 0), q1 = (int)(b >> 4) - ((b & 0x80) ? 16 : 0);
        acc = fmaf((float)q0 * s, ys[2 * j], fmaf((float)q1 * s, ys[2 * j + 1], acc));
      }
    } else if (wdtype == MK_BF16) {
      for (int k = lane; k < H; k += 32) acc = fmaf(bf2f(reinterpret_cast<const uint16_t*>(p)[k]), ys[k], acc);
    } else {
      for (int k = lane; k < H; k += 32) acc = fmaf(reinterpret_cast<const float*>(p)[k], ys[k], acc);
    }
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (trace_logits && lane == 0) trace_logits[row] = acc;
    if (acc > best || (acc == best && row < bid)) {
      best = acc;
      bid = row;
    }
  }
  if (lane == 0) {
    bv[w] = best;
    bi[w] = bid;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < nw; ++i)
      if (bv[i] > best || (bv[i] == best && bi[i] < bid)) {
        best = bv[i];
        bid = bi[i];
      }
    cand_v[blockIdx.x] = best;
    cand_i[blockIdx.x] = bid;
  }
}
__global__ void k_lm_reduce(const float* cand_v, const int32_t* cand_i, int n, int32_t* out) {
  if (threadIdx.x != 0) return;
  float best = -INFINITY;
  int bid = INT_MAX;
  for (int i = 0; i < n; ++i)
    if (cand_v[i] > best || (cand_v[i] == best && cand_i[i] < bid)) {
      best = cand_v[i];
      bid = cand_i[i];
    }
  *out = bid == INT_MAX ? 0 : bid;
}

int grid_for(long long n) { return (int)std::max(1ll, std::min(8192ll, (n + 255) / 256)); }

int cuda_err(const char* what) {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MK_OK : host_fail(MK_ERR_CUDA, (std::string(what) + ": " + cudaGetErrorString(e)).c_str());
}

int blas_err(cublasStatus_t s, const char* what) {
  return s == CUBLAS_STATUS_SUCCESS ? MK_OK
                                    : host_fail(MK_ERR_CUDA, (std::string(what) + ": cuBLAS status " + std::to_string((int)s)).c_str());
}

struct Dims {
  int H, NH, NKV, HD, QD, KD, NQKV, E, K, FE, FD, V;
  bool aux_f32;
  int wdtype;
  int xdtype;  // the expert matrices' format
  int fmt;    // activation operand format
  int esz;    // bytes of one operand element (4 fp32, 2 bf16 / fp16)
};

// C[M][N] (fp32, row-major, ldc) = A[M][Kd] . W[N][Kd]^T with W rows of ldw
// elements; fp32 operands, or hi then lo parts of A (lo at lo_off elements)
// against bf16 / fp16 W.
int gemm(PrefillWork& w, const Dims& d, int M, int N, int Kd, const void* W, int ldw, const void* A, size_t lo_off,
         float* C, int ldc) {
  if (M == 0) return MK_OK;
  const float one = 1.f, zero = 0.f;
  if (d.fmt == ACT_F32)
    return blas_err(cublasGemmEx(w.blas, CUBLAS_OP_T, CUBLAS_OP_N, N, M, Kd, &one, W, CUDA_R_32F, ldw, A, CUDA_R_32F,
                                 Kd, &zero, C, CUDA_R_32F, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT),
                    "cublasGemmEx");
  const cudaDataType_t t = d.fmt == ACT_BF16 ? CUDA_R_16BF : CUDA_R_16F;
  const uint16_t* Ah = static_cast<const uint16_t*>(A);
  if (int r = blas_err(cublasGemmEx(w.blas, CUBLAS_OP_T, CUBLAS_OP_N, N, M, Kd, &one, W, t, ldw, Ah, t, Kd, &zero, C,
                                    CUDA_R_32F, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT),
                       "cublasGemmEx"))
    return r;
  return blas_err(cublasGemmEx(w.blas, CUBLAS_OP_T, CUBLAS_OP_N, N, M, Kd, &one, W, t, ldw, Ah + lo_off, t, Kd, &one,
                               C, CUDA_R_32F, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT),
                  "cublasGemmEx");
}

// The operand of `rows` packed records of width Kd in format fmt: int4 /
// int3 widened into the scratch, bf16 / fp32 records used in place (a record
// is exactly one row).
const void* weight_rows(PrefillWork& w, int fmt, const uint8_t* rec, long long rows, int Kd, cudaStream_t st) {
  if (fmt == MK_INT4_G64) {
    k_widen_int4<<<grid_for(rows * Kd / 2), 256, 0, st>>>(rec, pack_rec_bytes(fmt, Kd), Kd, rows, w.Wb);
    return w.Wb;
  }
  if (fmt == MK_INT3_G64) {
    k_widen_int3<<<grid_for(rows * Kd), 256, 0, st>>>(rec, pack_rec_bytes(fmt, Kd), Kd, rows, w.Wb);
    return w.Wb;
  }
  return rec;
}

}  // namespace

void prefill_free(PrefillWork* w) {
  if (!w) return;
  if (w->blas) cublasDestroy(w->blas);
  void* bufs[] = {w->X, w->Hr, w->Q, w->O, w->A, w->C, w->D, w->Wb, w->Z, w->logits, w->ids, w->wts, w->cnt,
                  w->ent, w->pos_of, w->lm_v, w->lm_i};
  for (void* p : bufs) cudaFree(p);
  delete w;
}

int prefill_run(PrefillWork** pw, const PrefillArgs& a, cudaStream_t st) {
  const mk_model_desc& m = a.d;
  Dims d;
  d.H = m.hidden; d.NH = m.n_heads; d.NKV = m.n_kv_heads; d.HD = m.head_dim; d.QD = m.n_heads * m.head_dim;
  d.KD = m.n_kv_heads * m.head_dim; d.NQKV = d.QD + 2 * d.KD; d.E = m.n_experts; d.K = m.top_k;
  d.FE = m.expert_ffn; d.FD = m.dense_ffn; d.V = m.vocab; d.wdtype = m.wdtype;
  d.xdtype = m.expert_wdtype;
  d.aux_f32 = m.wdtype == MK_F32;
  d.fmt = m.wdtype == MK_F32 ? ACT_F32 : (m.wdtype == MK_BF16 ? ACT_BF16 : ACT_F16);
  d.esz = d.fmt == ACT_F32 ? 4 : 2;
  const int M = a.n;
  if (M < 1 || M > kMaxPrefill) return host_fail(MK_ERR_INVALID_ARG, "prefill chunk of 1..4096 positions");
  // ---- workspace, made on first use and kept by the context
  if (!*pw) {
    PrefillWork* w = new PrefillWork();
    *pw = w;
    if (cublasCreate(&w->blas) != CUBLAS_STATUS_SUCCESS) {
      w->blas = nullptr;
      return host_fail(MK_ERR_CUDA, "cublasCreate failed");
    }
    const size_t MM = kMaxPrefill, H = d.H, QD = d.QD, E = d.E, K = d.K, ent = MM * K;
    const size_t kmax = std::max({H, QD, (size_t)d.FD, (size_t)d.FE});
    w->a_elems = std::max({ent * H, MM * kmax, ent * (size_t)d.FE});
    w->c_elems = std::max({MM * d.NQKV, MM * 2 * (size_t)d.FD, ent * 2 * (size_t)d.FE, MM * H, MM * E});
    w->wb_elems = d.wdtype == MK_INT4_G64 || d.xdtype == MK_INT3_G64
                      ? std::max({E * 2 * d.FE * H, E * H * d.FE, 2 * (size_t)d.FD * H, H * (size_t)d.FD,
                                  (size_t)d.NQKV * H, H * QD})
                      : 0;
    cudaError_t e = cudaSuccess;
    auto alloc = [&](void** p, size_t bytes) {
      if (e == cudaSuccess && bytes) e = cudaMalloc(p, bytes);
    };
    alloc((void**)&w->X, 4 * MM * H);
    alloc((void**)&w->Hr, 4 * MM * H);
    alloc((void**)&w->Q, 4 * MM * QD);
    alloc((void**)&w->O, 4 * MM * QD);
    alloc(&w->A, 4 * w->a_elems);
    alloc((void**)&w->C, 4 * w->c_elems);
    alloc((void**)&w->D, 4 * ent * H);
    alloc((void**)&w->Wb, 2 * w->wb_elems);
    alloc((void**)&w->Z, 4 * MM * H);
    alloc((void**)&w->logits, 4 * MM * E);
    alloc((void**)&w->ids, 4 * ent);
    alloc((void**)&w->wts, 4 * ent);
    alloc((void**)&w->cnt, 4 * (2 * E + 1));
    alloc((void**)&w->ent, 4 * ent);
    alloc((void**)&w->pos_of, 4 * ent);
    alloc((void**)&w->lm_v, 4 * kLmBlocks);
    alloc((void**)&w->lm_i, 4 * kLmBlocks);
    if (e != cudaSuccess) return host_fail(MK_ERR_CUDA, (std::string("prefill workspace: ") + cudaGetErrorString(e)).c_str());
    w->max_m = kMaxPrefill;
    w->cnt_host.resize(2 * E + 1);
  }
  PrefillWork& w = **pw;
  if (int r = blas_err(cublasSetStream(w.blas, st), "cublasSetStream")) return r;
  const size_t lo = w.a_elems;  // bf16 lo parts follow the hi parts (the buffer holds 4 bytes per element)
  const int TB = 256;
  const int tr_rows = a.trace ? a.trace_rows : 0, tr0 = M - tr_rows;
  float* tr_x = a.trace;
  float* tr_attn = a.trace ? tr_x + (size_t)m.n_layers * tr_rows * d.H : nullptr;
  float* tr_lg = a.trace ? tr_attn + (size_t)m.n_layers * tr_rows * d.QD : nullptr;
  float* tr_tk = a.trace ? tr_lg + (size_t)m.n_layers * tr_rows * d.E : nullptr;
  float* tr_fin = a.trace ? tr_tk + (size_t)m.n_layers * tr_rows * 2 * d.K : nullptr;
  if (a.trace) cudaMemsetAsync(a.trace, 0, a.trace_bytes, st);

  k_embed<<<M, TB, 0, st>>>(a.tokens, a.embed, d.aux_f32, d.H, d.V, M, w.X, a.err);
  if (int r = cuda_err("prefill embed")) return r;
  const size_t att_smem =
      sizeof(float) * (size_t)d.NH / d.NKV * 16 * d.HD + 2 * 64 * (d.HD + 2) + 2 * 64 * d.HD + 4 * 16 * 64 * (d.NH / d.NKV);
  for (int l = 0; l < m.n_layers; ++l) {
    const LayerW& Lw = a.layers[l];
    const bool dense = l < m.n_dense;
    // attention block
    k_norm_act<<<M, TB, 0, st>>>(w.X, nullptr, nullptr, Lw.attn_norm, d.aux_f32, m.rms_eps, d.H, w.A, lo, d.fmt,
                                 nullptr);
    const void* W = weight_rows(w, d.wdtype, Lw.pk[PK_QKV], d.NQKV, d.H, st);
    if (int r = gemm(w, d, M, d.NQKV, d.H, W, d.H, w.A, lo, w.C, d.NQKV)) return r;
    k_qkv_epi<<<grid_for((long long)M * d.NQKV / 2), TB, 0, st>>>(w.C, d.NQKV, d.NH, d.NKV, d.HD, a.rope, a.start, M,
                                                                   w.Q, a.kv, a.block_table, a.slot,
                                                                   a.max_pages_per_seq, a.n_pages, l, a.err);
    dim3 ag((M + 15) / 16, d.NKV);
    const float scale = 1.f / sqrtf((float)d.HD);
    if (d.HD == 128 && d.NH == 4 * d.NKV) {
      k_attention<128, 4><<<ag, 256, att_smem, st>>>(w.Q, a.kv, a.block_table, a.slot, a.max_pages_per_seq,
                                                     a.n_pages, l, d.NKV, a.start, M, scale, w.O);
    } else if (d.HD == 64 && d.NH == 2 * d.NKV) {
      k_attention<64, 2><<<ag, 256, att_smem, st>>>(w.Q, a.kv, a.block_table, a.slot, a.max_pages_per_seq,
                                                    a.n_pages, l, d.NKV, a.start, M, scale, w.O);
    } else {
      return host_fail(MK_ERR_UNSUPPORTED, "prefill attention not compiled for this head shape");
    }
    if (int r = cuda_err("prefill attention")) return r;
    if (a.trace)
      k_trace_rows<<<32, TB, 0, st>>>(w.O, d.QD, tr0, tr_rows, d.QD, tr_attn + (size_t)l * tr_rows * d.QD);
    k_norm_act<<<M, TB, 0, st>>>(w.O, nullptr, nullptr, nullptr, d.aux_f32, 0.f, d.QD, w.A, lo, d.fmt, nullptr);
    W = weight_rows(w, d.wdtype, Lw.pk[PK_O], d.H, d.QD, st);
    if (int r = gemm(w, d, M, d.H, d.QD, W, d.QD, w.A, lo, w.C, d.H)) return r;
    // h = x + attention; the FFN input
    k_norm_act<<<M, TB, 0, st>>>(w.X, w.C, w.Hr, Lw.ffn_norm, d.aux_f32, m.rms_eps, d.H, w.A, lo, d.fmt,
                                 dense ? nullptr : w.Z);
    if (dense) {
      W = weight_rows(w, d.wdtype, Lw.pk[PK_GU], 2LL * d.FD, d.H, st);
      if (int r = gemm(w, d, M, 2 * d.FD, d.H, W, d.H, w.A, lo, w.C, 2 * d.FD)) return r;
      k_silu_act<<<grid_for((long long)M * d.FD), TB, 0, st>>>(w.C, M, d.FD, w.A, lo, d.fmt);
      W = weight_rows(w, d.wdtype, Lw.pk[PK_DN], d.H, d.FD, st);
      if (int r = gemm(w, d, M, d.H, d.FD, W, d.FD, w.A, lo, w.C, d.H)) return r;
      k_add<<<grid_for((long long)M * d.H), TB, 0, st>>>(w.Hr, w.C, w.X, (long long)M * d.H);
    } else {
      k_router<<<grid_for((long long)M * d.E * 32), 256, 0, st>>>(w.Z, Lw.router, d.aux_f32, M, d.E, d.H, w.logits);
      k_route<<<(M + 7) / 8, 256, 0, st>>>(w.logits, M, d.E, d.K, w.ids, w.wts);
      if (a.trace) {
        k_trace_rows<<<8, TB, 0, st>>>(w.logits, d.E, tr0, tr_rows, d.E, tr_lg + (size_t)l * tr_rows * d.E);
        k_trace_topk<<<1, TB, 0, st>>>(w.ids, w.wts, tr0, tr_rows, d.K, tr_tk + (size_t)l * tr_rows * 2 * d.K);
      }
      const int n_ent = M * d.K;
      k_group<<<1, 64, 0, st>>>(w.ids, n_ent, d.E, d.K, w.cnt, w.ent, w.pos_of);
      if (int r = cuda_err("prefill routing")) return r;
      cudaError_t e = cudaMemcpyAsync(w.cnt_host.data(), w.cnt, sizeof(int32_t) * (2 * d.E + 1),
                                      cudaMemcpyDeviceToHost, st);
      if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // the expert GEMMs are sized on the host
      if (e != cudaSuccess) return host_fail(MK_ERR_CUDA, (std::string("prefill routing counts: ") + cudaGetErrorString(e)).c_str());
      const int32_t* off = w.cnt_host.data() + d.E;
      // the FFN inputs gathered into expert-sorted order, in A; the M rows of
      // A are first copied to D (free until the down GEMMs) and gathered from there
      void* G = w.A;
      const size_t a_bytes = (size_t)d.esz * M * d.H;
      cudaMemcpyAsync(w.D, w.A, a_bytes, cudaMemcpyDeviceToDevice, st);
      if (d.fmt != ACT_F32)
        cudaMemcpyAsync(reinterpret_cast<uint8_t*>(w.D) + a_bytes, static_cast<uint16_t*>(w.A) + lo, a_bytes,
                        cudaMemcpyDeviceToDevice, st);
      k_gather<<<grid_for((long long)n_ent * d.H), TB, 0, st>>>(w.D, (size_t)M * d.H, G, lo, w.ent, n_ent, d.H, d.fmt);
      // gate/up of every expert, then SiLU
      W = weight_rows(w, d.xdtype, Lw.pk[PK_GU], 2LL * d.E * d.FE, d.H, st);
      const size_t wrow = d.esz;
      for (int x = 0; x < d.E; ++x) {
        const int mx = off[x + 1] - off[x];
        if (!mx) continue;
        const uint8_t* We = static_cast<const uint8_t*>(W) + (size_t)x * 2 * d.FE * d.H * wrow;
        const void* Ge = static_cast<const uint8_t*>(G) + (size_t)off[x] * d.H * d.esz;
        if (int r = gemm(w, d, mx, 2 * d.FE, d.H, We, d.H, Ge, lo, w.C + (size_t)off[x] * 2 * d.FE, 2 * d.FE))
          return r;
      }
      k_silu_act<<<grid_for((long long)n_ent * d.FE), TB, 0, st>>>(w.C, n_ent, d.FE, w.A, lo, d.fmt);
      W = weight_rows(w, d.xdtype, Lw.pk[PK_DN], (long long)d.E * d.H, d.FE, st);
      for (int x = 0; x < d.E; ++x) {
        const int mx = off[x + 1] - off[x];
        if (!mx) continue;
        const uint8_t* We = static_cast<const uint8_t*>(W) + (size_t)x * d.H * d.FE * wrow;
        const void* Ae = static_cast<const uint8_t*>(w.A) + (size_t)off[x] * d.FE * d.esz;
        if (int r = gemm(w, d, mx, d.H, d.FE, We, d.FE, Ae, lo, w.D + (size_t)off[x] * d.H, d.H)) return r;
      }
      k_combine<<<grid_for((long long)M * d.H), TB, 0, st>>>(w.Hr, w.D, w.wts, w.pos_of, M, d.H, d.K, w.X);
    }
    if (int r = cuda_err("prefill layer")) return r;
    if (a.trace) k_trace_rows<<<32, TB, 0, st>>>(w.X, d.H, tr0, tr_rows, d.H, tr_x + (size_t)l * tr_rows * d.H);
  }
  if (a.out_token) {
    k_lm_head<<<kLmBlocks, 256, sizeof(float) * d.H, st>>>(w.X + (size_t)(M - 1) * d.H, a.final_norm, d.aux_f32,
                                                           m.rms_eps, d.H, a.lm_pk, pack_rec_bytes(d.wdtype, d.H),
                                                           d.wdtype, d.V, w.lm_v, w.lm_i,
                                                           a.trace ? tr_fin + (size_t)(tr_rows - 1) * d.V : nullptr);
    k_lm_reduce<<<1, 32, 0, st>>>(w.lm_v, w.lm_i, kLmBlocks, a.out_token);
  }
  return cuda_err("prefill lm_head");
}

int prefill_setup_attributes(const mk_model_desc& m) {
  const size_t att_smem = sizeof(float) * (size_t)m.n_heads / m.n_kv_heads * 16 * m.head_dim +
                          2 * 64 * (m.head_dim + 2) + 2 * 64 * m.head_dim + 4 * 16 * 64 * (m.n_heads / m.n_kv_heads);
  cudaError_t e = cudaSuccess;
  if (m.head_dim == 128)
    e = cudaFuncSetAttribute(k_attention<128, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)att_smem);
  else if (m.head_dim == 64)
    e = cudaFuncSetAttribute(k_attention<64, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)att_smem);
  return e == cudaSuccess ? MK_OK : host_fail(MK_ERR_CUDA, cudaGetErrorString(e));
}

}  // namespace mk
