// The library's packed copy of the linear weights.  Every output row becomes
// one record of its codes followed by its group scales (int4, int3), padded
// to 16 bytes, and rows a task reads together are adjacent:
//   QKV   record 2p + r: RoPE pair task p (q heads, then k heads, then v
//         heads; p = head * hd/2 + i) and its row i (r = 0) or i + hd/2 (r = 1)
//   O     record = output row
//   GU    record 2t + r: gate (r = 0) / up (r = 1) row t (t = expert * F + f
//         for expert layers, t = f for the dense layers)
//   DOWN  record = output row (expert layers: expert * hidden + row)
//   LM    record = vocabulary row
// so each tile the decode kernel streams is one contiguous range (or one per
// expert).  int4 and bf16 / fp32 rows are copied as they are; int3 rows are
// recoded from 24-bit words into the kernel's bit planes (pack_rows_int3).  The pack runs once (mk_create, or mk_pack_weights for the
// allocation-free entry point).
#include <string>
#include <vector>

#include "mk_internal.h"

namespace mk {
namespace {

__global__ void pack_rows(const uint8_t* codes, const uint8_t* scales, int rb, int sb, int rec, int nrows,
                          uint8_t* dst, int mode, int p0, int half, int hd) {
  for (int row = blockIdx.x; row < nrows; row += gridDim.x) {
    long long d;
    if (mode == 0) {
      d = row;
    } else if (mode == 1) {
      d = 2LL * row + p0;
    } else {
      const int h = row / hd, i = row % hd, r = i / half, ii = i % half;
      d = 2LL * (p0 + h * half + ii) + r;
    }
    uint8_t* o = dst + d * rec;
    const uint4* src = reinterpret_cast<const uint4*>(codes + (size_t)row * rb);
    for (int c = threadIdx.x; c < rb / 16; c += blockDim.x) reinterpret_cast<uint4*>(o)[c] = src[c];
    if (sb) {
      const uint16_t* ss = reinterpret_cast<const uint16_t*>(scales + (size_t)row * sb);
      for (int c = threadIdx.x; c < sb / 2; c += blockDim.x) reinterpret_cast<uint16_t*>(o + rb)[c] = ss[c];
    }
    for (int c = threadIdx.x; c < rec - rb - sb; c += blockDim.x) o[rb + sb + c] = 0;
  }
}

// int3 rows: logical codes (8 per little-endian 24-bit word, two's
// complement) -> per 32-value chunk c, the low-plane words L0, L1 at 8c and
// the high-plane word at 8 NCH + 4c, holding the offset code u = q + 4 of
// value v = 8t + 2i + e of the chunk: its low bits in byte i of L[t / 2] at
// bit 2 (2 (t % 2) + e), its high bit in byte i of the high word at bit
// 2t + e.  The scales follow the 3K/8 code bytes.  One thread per chunk.
__global__ void pack_rows_int3(const uint8_t* codes, const uint8_t* scales, int K, int rec, int nrows,
                               uint8_t* dst, int mode, int p0) {
  const int nch = K / 32, rb = 3 * K / 8, sb = K / 32;
  for (int row = blockIdx.x; row < nrows; row += gridDim.x) {
    const long long d = mode == 0 ? row : 2LL * row + p0;
    uint8_t* o = dst + d * rec;
    const uint8_t* src = codes + (size_t)row * rb;
    for (int c = threadIdx.x; c < nch; c += blockDim.x) {
      uint32_t L[2] = {0u, 0u}, hh = 0u;
      for (int wd = 0; wd < 4; ++wd) {  // the chunk's four 24-bit words: values 8 wd .. 8 wd + 7
        const uint8_t* b = src + 12 * c + 3 * wd;
        const uint32_t word = (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16);
        for (int j = 0; j < 8; ++j) {
          const uint32_t u = ((word >> (3 * j)) & 7u) ^ 4u;  // two's complement -> q + 4
          const int t = wd, i = j >> 1, e = j & 1;
          L[t >> 1] |= (u & 3u) << (8 * i + 2 * (2 * (t & 1) + e));
          hh |= (u >> 2) << (8 * i + 2 * t + e);
        }
      }
      reinterpret_cast<uint32_t*>(o + 8 * c)[0] = L[0];
      reinterpret_cast<uint32_t*>(o + 8 * c)[1] = L[1];
      reinterpret_cast<uint32_t*>(o + 8 * nch)[c] = hh;
    }
    const uint16_t* ss = reinterpret_cast<const uint16_t*>(scales + (size_t)row * sb);
    for (int c = threadIdx.x; c < sb / 2; c += blockDim.x) reinterpret_cast<uint16_t*>(o + rb)[c] = ss[c];
    for (int c = threadIdx.x; c < rec - rb - sb; c += blockDim.x) o[rb + sb + c] = 0;
  }
}

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

int pack_row_bytes(int wdtype, int K) {
  return wdtype == MK_INT4_G64 ? K / 2 : (wdtype == MK_INT3_G64 ? 3 * K / 8 : (wdtype == MK_BF16 ? 2 * K : 4 * K));
}
int pack_scale_bytes(int wdtype, int K) {
  return wdtype == MK_INT4_G64 || wdtype == MK_INT3_G64 ? K / 64 * 2 : 0;
}
int pack_rec_bytes(int wdtype, int K) {
  return (pack_row_bytes(wdtype, K) + pack_scale_bytes(wdtype, K) + 15) / 16 * 16;
}

size_t host_pack_layout(const mk_model_desc& d, PackLayout* pl) {
  const int H = d.hidden, QD = d.n_heads * d.head_dim, KD = d.n_kv_heads * d.head_dim;
  const int w = d.wdtype;
  size_t off = 0;
  for (int l = 0; l < d.n_layers; ++l) {
    const bool dense = l < d.n_dense;
    const int f = dense ? w : d.expert_wdtype;  // the FFN matrices' format
    size_t o[4];
    o[PK_QKV] = off;
    off = a256(off + (size_t)(QD + 2 * KD) * pack_rec_bytes(w, H));
    o[PK_O] = off;
    off = a256(off + (size_t)H * pack_rec_bytes(w, QD));
    o[PK_GU] = off;
    off = a256(off + 2 * (size_t)(dense ? d.dense_ffn : (size_t)d.n_experts * d.expert_ffn) * pack_rec_bytes(f, H));
    o[PK_DN] = off;
    off = a256(off + (size_t)(dense ? H : (size_t)d.n_experts * H) *
                         pack_rec_bytes(f, dense ? d.dense_ffn : d.expert_ffn));
    if (pl)
      for (int k = 0; k < 4; ++k) pl->layer[l][k] = o[k];
  }
  if (pl) pl->lm = off;
  off = a256(off + (size_t)d.vocab * pack_rec_bytes(w, H));
  return off;
}

int host_pack(const mk_model_desc& d, const mk_weights& wts, uint8_t* dst, cudaStream_t st) {
  const int H = d.hidden, HD = d.head_dim, HALF = d.head_dim / 2, w = d.wdtype;
  const int QD = d.n_heads * HD;
  PackLayout pl;
  host_pack_layout(d, &pl);
  auto launch = [&](const mk_linear& lin, int K, int nrows, size_t off, int mode, int p0, int f = -1) -> int {
    if (f < 0) f = w;
    const int rb = pack_row_bytes(f, K), sb = pack_scale_bytes(f, K), rec = pack_rec_bytes(f, K);
    const int grid = nrows < 8192 ? nrows : 8192;
    if (f == MK_INT3_G64)
      pack_rows_int3<<<grid, 128, 0, st>>>(static_cast<const uint8_t*>(lin.w),
                                          static_cast<const uint8_t*>(lin.scales), K, rec, nrows, dst + off, mode, p0);
    else
      pack_rows<<<grid, 128, 0, st>>>(static_cast<const uint8_t*>(lin.w), static_cast<const uint8_t*>(lin.scales),
                                     rb, sb, rec, nrows, dst + off, mode, p0, HALF, HD);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return host_fail(MK_ERR_CUDA, (std::string("pack: ") + cudaGetErrorString(e)).c_str());
    return MK_OK;
  };
  for (int l = 0; l < d.n_layers; ++l) {
    const mk_layer_weights& L = wts.layers[l];
    const bool dense = l < d.n_dense;
    const size_t* o = pl.layer[l];
    int r;
    if ((r = launch(L.wq, H, QD, o[PK_QKV], 2, 0))) return r;
    if ((r = launch(L.wk, H, d.n_kv_heads * HD, o[PK_QKV], 2, d.n_heads * HALF))) return r;
    if ((r = launch(L.wv, H, d.n_kv_heads * HD, o[PK_QKV], 2, (d.n_heads + d.n_kv_heads) * HALF))) return r;
    if ((r = launch(L.wo, QD, H, o[PK_O], 0, 0))) return r;
    if (dense) {
      if ((r = launch(L.gate, H, d.dense_ffn, o[PK_GU], 1, 0))) return r;
      if ((r = launch(L.up, H, d.dense_ffn, o[PK_GU], 1, 1))) return r;
      if ((r = launch(L.down, d.dense_ffn, H, o[PK_DN], 0, 0))) return r;
    } else {
      const int rows = d.n_experts * d.expert_ffn, x = d.expert_wdtype;
      if ((r = launch(L.exp_gate, H, rows, o[PK_GU], 1, 0, x))) return r;
      if ((r = launch(L.exp_up, H, rows, o[PK_GU], 1, 1, x))) return r;
      if ((r = launch(L.exp_down, d.expert_ffn, d.n_experts * H, o[PK_DN], 0, 0, x))) return r;
    }
  }
  return launch(wts.lm_head, H, d.vocab, pl.lm, 0, 0);
}

}  // namespace mk

using namespace mk;

extern "C" MK_API size_t mk_packed_bytes(const mk_model_desc* d) {
  int shape = -1;
  if (!d || host_validate_desc(d, &shape) != MK_OK) return 0;
  return host_pack_layout(*d, nullptr);
}

extern "C" MK_API int mk_pack_weights(const mk_model_desc* d, const mk_weights* w, void* dst_dev,
                                      size_t dst_bytes, void* stream) {
  host_clear_error();
  int shape = -1;
  if (!d || !w || !dst_dev) return host_fail(MK_ERR_INVALID_ARG, "NULL argument");
  if (int r = host_validate_desc(d, &shape)) return r;
  std::vector<LayerW> layers(d->n_layers);
  if (int r = host_check_model(d, w, &shape, layers.data())) return r;
  if (dst_bytes < host_pack_layout(*d, nullptr))
    return host_fail(MK_ERR_INVALID_ARG, "destination is smaller than mk_packed_bytes");
  if ((reinterpret_cast<uintptr_t>(dst_dev) & 255u) != 0)
    return host_fail(MK_ERR_INVALID_ARG, "destination must be 256-byte aligned");
  return host_pack(*d, *w, static_cast<uint8_t*>(dst_dev), static_cast<cudaStream_t>(stream));
}
