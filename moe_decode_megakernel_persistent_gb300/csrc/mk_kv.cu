// KV-cache transfers of the C ABI: a sequence's K/V copied between the paged
// pool and a caller buffer (mk_kv_write / mk_kv_read), and block-table entries
// set for pages that a forked sequence shares (mk_seq_fork).  One kernel does
// both: it first writes the block-table entries the call carries, then copies
// 16-byte words between the caller buffer and the pages.
#include <algorithm>

#include "mk_internal.h"

namespace mk {

namespace {

__global__ void __launch_bounds__(256) kv_xfer_kernel(const __grid_constant__ KvXfer a) {
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < a.n_upd; i += blockDim.x)
      a.block_table[a.upd[i].slot * a.max_pages_per_seq + a.upd[i].index] = a.upd[i].page;
  if (a.n == 0) return;
  const int W = a.head_dim / 8;  // 16-byte words of one head's row
  const long long total = (long long)a.n_layers * a.n * 2 * a.n_kv_heads * W;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    long long r = i;
    const int w = (int)(r % W);
    r /= W;
    const int h = (int)(r % a.n_kv_heads);
    r /= a.n_kv_heads;
    const int kvsel = (int)(r % 2);
    r /= 2;
    const int p = (int)(r % a.n);
    const int l = (int)(r / a.n);
    const int t = a.start + p, pi = t / kPageTokens;
    // pages of indices the call sets itself come from its own list: the
    // block-table writes above are not ordered before other blocks' reads
    int page;
    if (pi >= a.upd_index0 && pi < a.upd_index0 + a.n_upd) page = a.upd[pi - a.upd_index0].page;
    else page = a.block_table[a.slot * a.max_pages_per_seq + pi];
    if (page < 0 || page >= a.n_pages) continue;  // the host checked every index
    const size_t pool = ((((size_t)l * a.n_pages + page) * 2 + kvsel) * a.n_kv_heads + h) *
                            (size_t)(kPageTokens * a.head_dim) +
                        (size_t)(t % kPageTokens) * a.head_dim + 8 * w;
    const size_t buf = ((((size_t)l * a.n + p) * 2 + kvsel) * a.n_kv_heads + h) * (size_t)a.head_dim + 8 * w;
    if (a.src) *reinterpret_cast<uint4*>(a.kv + pool) = *reinterpret_cast<const uint4*>(a.src + buf);
    else *reinterpret_cast<uint4*>(a.dst + buf) = *reinterpret_cast<const uint4*>(a.kv + pool);
  }
}

}  // namespace

int launch_kv_xfer(const KvXfer& a, cudaStream_t st) {
  const long long words = (long long)a.n_layers * a.n * 2 * a.n_kv_heads * (a.head_dim / 8);
  const int blocks = (int)std::max(1ll, std::min(4096ll, (words + 255) / 256));
  kv_xfer_kernel<<<blocks, 256, 0, st>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MK_OK : host_fail(MK_ERR_CUDA, cudaGetErrorString(e));
}

}  // namespace mk
