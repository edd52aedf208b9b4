// The persistent decode kernel: one cooperative launch runs a whole decode
// step (all layers, then lm_head + argmax) for up to 16 rows.
//
// Structure of one layer (after "rec Megakernel and Tempo9 Compared", §2:
// every operator of the layer inside one dispatch; grid-wide barriers only
// where data crosses blocks; each block recomputes RMSNorm itself):
//   P1  RMSNorm (every block, redundantly) -> QKV projection of this block's
//       rows, RoPE on q/k, the new K/V written into the paged cache      | barrier
//   P2  split attention: (row, kv head, chunk of positions) units, the last
//       unit of a (row, kv head) merges all chunks (log-sum-exp)          | barrier
//   P3  o_proj rows + residual; MoE layers also form this block's partial
//       router logits, reduced by the last block to arrive                | barrier
//   P4  RMSNorm + softmax/top-k (every block), expert gate/up -> SiLU
//       (dense layers: the SwiGLU gate/up)                                | barrier
//   P5  down projection rows, weighted sum over the selected experts, residual
//                                                                          | barrier
// After the last layer: final RMSNorm, lm_head rows, per-block argmax, and
// the last block to arrive reduces the argmax (no barrier needed).
#include <cfloat>
#include <climits>
#include <type_traits>
#include "mk_device.cuh"

namespace mk {

constexpr int kMaxEnt = kMaxBatch * 8; // (row, expert slot) entries

// Per-launch, per-block context shared by the phases; it lives in shared
// memory (inside Fixed) so the phases read it with shared-memory loads.
struct Ctx {
  uint8_t* act;    // staging area in shared memory
  int G, bid, n;
  int r0, nr;      // hidden rows owned by this block
  float *tr_x, *tr_attn, *tr_rl, *tr_tk, *tr_fin;
  uint64_t* tm;    // timing stamps (block 0, thread 0 only) or null
};

struct Fixed {
  StepArgs args;   // copy of the launch arguments
  LayerW lw;       // the current layer's weight pointers
  Ctx ctx;
  int tok[kMaxBatch];
  int topk_id[kMaxBatch][8];
  float topk_w[kMaxBatch][8];
  float dots[kMaxEnt][kMaxRowsPerBlock];
  float hs[kMaxBatch][kMaxRowsPerBlock];
  float red[kThreads];
  float best_v[kWarps][kMaxBatch];
  int best_i[kWarps][kMaxBatch];
  int unit_start[kMaxBatch + 1];
  int upages[2][64];   // pool pages of this block's attention units (same for every layer)
  float rnorm[kMaxBatch];
  int16_t ue_expert[64], ue_start[64], ue_len[64];
  int16_t run_start[kMaxEnt], run_len[kMaxEnt], run_mat[kMaxEnt];
  uint8_t ent_b[kMaxEnt], ent_j[kMaxEnt];
  uint8_t ent_of[kMaxBatch][8];
  int n_ue, n_runs, flag;
};
constexpr int kActOffset = (sizeof(Fixed) + 127) / 128 * 128;
constexpr int kActBytes = kSmemBytes - kActOffset;

__device__ __forceinline__ Fixed& fixed() {
  extern __shared__ __align__(128) uint8_t smem_dyn[];
  return *reinterpret_cast<Fixed*>(smem_dyn);
}

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

template <class S>
struct Kv {
  __device__ static __forceinline__ size_t offset(int l, int n_pages, int page, int kvsel, int g,
                                                  int slot) {
    return ((((size_t)l * n_pages + page) * 2 + kvsel) * S::NKV + g) * (size_t)(kPageTokens * S::HD) +
           (size_t)slot * S::HD;
  }
};

// Timing record layout (uint64 ns): [0] start; per layer l and phase p:
// [1 + 16 l + 3 p + k], k = 0 staging done, 1 work done, 2 barrier released;
// [1 + 16 L] lm_head done.
#define MK_STAMP(c, l, p, k) \
  if ((c).tm && threadIdx.x == 0) (c).tm[1 + 16 * (l) + 3 * (p) + (k)] = globaltimer()

template <class S, int WDT>
struct Model {
  static constexpr int AUX = WDT == WF32 ? WF32 : WBF16;
  static constexpr int H = S::H, NH = S::NH, NKV = S::NKV, HD = S::HD, E = S::E, TOPK = S::TOPK;
  static constexpr int FE = S::FE, FD = S::FD, QD = NH * HD, GQA = NH / NKV, HALF = HD / 2;
  static constexpr int DPL = HD / 32;
  static constexpr int KSD = FD <= 2048 ? FD : (WDT == WBF16 ? 1024 : 2048);  // dense-down segment
  static constexpr int NSEG = FD / KSD;
  static_assert(FD % KSD == 0, "dense FFN splits into segments");
  using GH = Gemv<WDT, H>;
  using GQ = Gemv<WDT, QD>;
  using GE = Gemv<WDT, FE>;
  using GS = Gemv<WDT, KSD>;
  static_assert(kMaxBatch * GH::ACT_BYTES <= kActBytes, "staging area holds a full batch");
  static_assert(kMaxBatch * GQ::ACT_BYTES <= kActBytes, "staging area holds a full batch");
  static_assert((kWarps * GQA * (HD + 2) + GQA * HD) * 4 <= kActBytes, "attention combine + query buffers");
  static_assert(TOPK <= 8 && E <= 64, "router tables");



  static constexpr int PR = HD + 4;  // partial row: m, l, pad, pad, o[HD] (16-byte rows)
  static constexpr int TU = 4;

  __device__ static __forceinline__ void unit_of(const StepArgs& a, const int* unit_start, int u, int n,
                                                 int& b, int& g, int& ci, int& nch) {
    b = 0;
    while (b + 1 < n && unit_start[b + 1] <= u) ++b;
    nch = (a.pos[b] + 1 + a.chunk - 1) / a.chunk;
    const int rem = u - unit_start[b];
    g = rem / nch;
    ci = rem % nch;
  }

  static constexpr int NQP = NH * HALF, NKP = NKV * HALF, NP = NQP + 2 * NKP;

  // Weight rows of QKV task p (a RoPE pair of q or k rows, or two v rows).
  __device__ static __forceinline__ RowRef qkv_row(const LayerW& Lw, int p, int r) {
    int m, row;
    if (p < NQP) { m = WQ; row = (p / HALF) * HD + p % HALF + r * HALF; }
    else if (p < NQP + NKP) { const int q = p - NQP; m = WK; row = (q / HALF) * HD + q % HALF + r * HALF; }
    else { const int q = p - NQP - NKP; m = WV; row = (q / HALF) * HD + 2 * (q % HALF) + r; }
    return {(const uint8_t*)Lw.w[m] + (size_t)row * GH::ROW_BYTES,
            (const uint16_t*)Lw.s[m] + (size_t)row * (H / 64)};
  }

  // --- L2 warm-up (all threads of the block): bytes a block reads in a
  // later phase are requested from HBM early, so that phase's loads find
  // them in L2.
  __device__ static void prefetch_rows(const void* w, const void* s, size_t row0, int rows, int row_bytes,
                                       int scale_bytes) {
    if (rows <= 0) return;
    prefetch_l2_block((const uint8_t*)w + row0 * row_bytes, (size_t)rows * row_bytes);
    if (WDT == WINT4) prefetch_l2_block((const uint8_t*)s + row0 * scale_bytes, (size_t)rows * scale_bytes);
  }

  // QKV rows and o_proj rows of layer l owned by this block.
  __device__ static void prefetch_attn_weights(int l) {
    const Ctx& c = fixed().ctx;
    const LayerW& Lw = fixed().args.layers[l];  // (a later layer: read from global)
    int p0, p1;
    split_range(NP, c.G, c.bid, p0, p1);
    // rows of consecutive tasks are consecutive within a head: merge them
    for (int r = 0; r < 2; ++r) {
      const uint8_t* run_w = nullptr; const uint16_t* run_s = nullptr;
      int run_n = 0;
      for (int p = p0; p <= p1; ++p) {
        const uint8_t* w = nullptr; const uint16_t* s = nullptr;
        if (p < p1) { const RowRef rr = qkv_row(Lw, p, r); w = rr.w; s = rr.s; }
        if (run_n && p < p1 && w == run_w + (size_t)run_n * GH::ROW_BYTES) { ++run_n; continue; }
        if (run_n) prefetch_rows(run_w, run_s, 0, run_n, GH::ROW_BYTES, H / 64 * 2);
        run_w = w; run_s = s; run_n = p < p1 ? 1 : 0;
      }
    }
    prefetch_rows(Lw.w[WO], Lw.s[WO], c.r0, c.nr, GQ::ROW_BYTES, QD / 64 * 2);
  }

  // Cached K/V of this block's attention units at layer l.  Pages come from
  // the block table, or for a row's newest page from the launch arguments;
  // out-of-range entries are skipped.
  __device__ static void prefetch_kv(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    for (int u = c.bid; u < a.n_units; u += c.G) {
      int b, g, ci, nch;
      unit_of(a, fixed().unit_start, u, c.n, b, g, ci, nch);
      const int t0 = ci * a.chunk, t1 = min(a.pos[b] + 1, t0 + a.chunk);
      for (int pi = t0 / kPageTokens; pi <= (t1 - 1) / kPageTokens; ++pi) {
        int page = pi == a.pos[b] / kPageTokens ? a.cur_page[b]
                 : (pi < a.max_pages_per_seq ? __ldcg(a.block_table + a.slot[b] * a.max_pages_per_seq + pi) : -1);
        if (page < 0 || page >= a.n_pages) continue;
        const int s0 = max(t0, pi * kPageTokens) % kPageTokens;
        const int s1 = (min(t1, (pi + 1) * kPageTokens) - 1) % kPageTokens + 1;
        for (int kv = 0; kv < 2; ++kv)
          prefetch_l2_block(a.kv + Kv<S>::offset(l, a.n_pages, page, kv, g, s0), (size_t)(s1 - s0) * HD * 2);
      }
    }
  }

  // ---------------------------------------------------------------- P1
  // RMSNorm of the residual (every block, redundantly) -> this block's rows of
  // the QKV projection.  A task is a RoPE pair of q or k rows (i, i + HD/2)
  // of one head, or two adjacent v rows, so the warp that forms a pair also
  // rotates it and writes it: q to scratch, k and v as bf16 into the page.
  __device__ static __noinline__ void qkv(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    const LayerW& Lw = F.lw;
    const int n = c.n;
    if (l == 0 && c.bid == 0)
      for (int i = tid; i < a.n_upd; i += kThreads)
        a.block_table[a.upd[i].slot * a.max_pages_per_seq + a.upd[i].index] = a.upd[i].page;
    if (c.bid == 0 && l >= a.n_dense)  // router logits are accumulated in P3
      for (int i = tid; i < n * E; i += kThreads) a.sc.rlogit[i] = 0.f;
    {
      const void* nw = Lw.attn_norm;
      const void* embed = a.embed;
      const float* x = a.sc.x;
      const int* tok = F.tok;
      const bool first = l == 0;
      stage_block<WDT, H>(
          c.act, n,
          [&](int r, int f4) -> float4 {
            return first ? ld_aux4<AUX>(embed, (size_t)tok[r] * (H / 4) + f4)
                         : __ldcg(reinterpret_cast<const float4*>(x + r * H) + f4);
          },
          true, a.eps, [&](int f4) { return ld_aux4<AUX>(nw, f4); }, F.red, nullptr);
    }
    if (l == 0)  // residual rows this block reads back in P3
      for (int i = tid; i < n * c.nr; i += kThreads) {
        const int b = i / c.nr, r = c.r0 + i % c.nr;
        a.sc.x[b * H + r] = ld_aux<AUX>(a.embed, (size_t)F.tok[b] * H + r);
      }
    __syncthreads();
    MK_STAMP(c, l, 0, 0);

    int p0, p1;
    split_range(NP, c.G, c.bid, p0, p1);
    struct {
      const StepArgs* a; const LayerW* Lw; int p0, l, lane;
      __device__ __forceinline__ RowRef row(int t, int r) const {
        return qkv_row(*Lw, p0 + t, r);
      }
      __device__ __forceinline__ ActRange acts(int) const {
        return {nullptr, 0, a->n};
      }
      __device__ __forceinline__ void out(int t, int b, int, float v0, float v1) const {
        if (lane != 0) return;
        const int p = p0 + t;
        const int pos = a->pos[b];
        if (p < NQP + NKP) {
          const int q = p < NQP ? p : p - NQP;
          const int hh = q / HALF, i = q % HALF;
          const float2 cs = __ldg(a->rope + (size_t)pos * HALF + i);
          const float e0 = v0 * cs.x - v1 * cs.y;
          const float e1 = v1 * cs.x + v0 * cs.y;
          if (p < NQP) {
            a->sc.q[b * QD + hh * HD + i] = e0;
            a->sc.q[b * QD + hh * HD + i + HALF] = e1;
          } else {
            uint16_t* dst = a->kv + Kv<S>::offset(l, a->n_pages, a->cur_page[b], 0, hh, pos % kPageTokens);
            dst[i] = f_to_bf16(e0);
            dst[i + HALF] = f_to_bf16(e1);
          }
        } else {
          const int q = p - NQP - NKP;
          const int g = q / HALF, i2 = 2 * (q % HALF);
          uint16_t* dst = a->kv + Kv<S>::offset(l, a->n_pages, a->cur_page[b], 1, g, pos % kPageTokens);
          dst[i2] = f_to_bf16(v0);
          dst[i2 + 1] = f_to_bf16(v1);
        }
      }
    } task{&a, &Lw, p0, l, lane};
    run_tasks<WDT, H, 2>(p1 - p0, c.act, task);
  }

  // ---------------------------------------------------------------- P2
  // Split attention over the paged cache.  Unit = (row, kv head, chunk of
  // positions); each warp takes TU positions at a time (their K and V rows
  // loaded together), keeps a running max, sum and weighted value (online
  // softmax) for the GQA heads of the kv head; the warps are combined and
  // the unit's partial (m, l, o) written.  The last unit of a (row, kv head)
  // to finish copies all its chunk partials into shared memory and merges
  // them in chunk order (log-sum-exp).
  __device__ static __noinline__ void attention(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    const int n = c.n;
    float* comb = reinterpret_cast<float*>(c.act);  // [warp][GQA][HD + 2]
    float* qs = comb + kWarps * GQA * (HD + 2);     // [GQA][HD] this unit's queries
    const float qscale = rsqrtf((float)HD);
    if (l == 0) {
      // the pool pages of this block's units, read once per launch (after the
      // block table got this launch's new pages): every warp of every unit
      // reading the table itself would queue on the same L2 lines
      int k = 0;
      for (int u = c.bid; u < a.n_units; u += c.G, ++k) {
        int b, g, ci, nch;
        unit_of(a, F.unit_start, u, n, b, g, ci, nch);
        const int t0 = ci * a.chunk, t1 = min(a.pos[b] + 1, t0 + a.chunk);
        const int p0 = t0 / kPageTokens, np = (t1 - 1) / kPageTokens - p0 + 1;
        if (k >= 2 || np > 64) {
          if (tid == 0) set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_UNIT, u);
          continue;
        }
        for (int j = tid; j < np; j += kThreads) {
          const int pi = p0 + j;
          int page = pi < a.max_pages_per_seq ? __ldcg(a.block_table + a.slot[b] * a.max_pages_per_seq + pi) : -1;
          if (page < 0 || page >= a.n_pages) {
            set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_PAGE, pi);
            page = 0;
          }
          F.upages[k][j] = page;
        }
      }
      __syncthreads();
    }
    int k_unit = 0;
    for (int u = c.bid; u < a.n_units; u += c.G, ++k_unit) {
      int b, g, ci, nch;
      unit_of(a, F.unit_start, u, n, b, g, ci, nch);
      const int ctx = a.pos[b] + 1;
      const int t0 = ci * a.chunk, t1 = min(ctx, t0 + a.chunk);
      const int pbase = t0 / kPageTokens;
      const int* upg = F.upages[min(k_unit, 1)];
      // this unit's queries into shared memory once (coalesced), not per warp
      for (int v = tid; v < GQA * HD / 4; v += kThreads)
        reinterpret_cast<float4*>(qs)[v] =
            __ldcg(reinterpret_cast<const float4*>(a.sc.q + b * QD + g * GQA * HD) + v);
      __syncthreads();

      float q[GQA][DPL];
#pragma unroll
      for (int i = 0; i < GQA; ++i)
#pragma unroll
        for (int d = 0; d < DPL; ++d) q[i][d] = qs[i * HD + lane * DPL + d] * qscale;
      float m[GQA], lsum[GQA], o[GQA][DPL];
#pragma unroll
      for (int i = 0; i < GQA; ++i) {
        m[i] = -INFINITY; lsum[i] = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[i][d] = 0.f;
      }
      for (int tb = t0 + wid; tb < t1; tb += kWarps * TU) {
        // TU positions per warp: all K/V loads issued before any is used;
        // positions past the chunk are predicated off (no break: the loops
        // stay fully unrolled and the arrays stay in registers)
        float kf[TU][DPL], vf[TU][DPL];
        bool ok[TU];
#pragma unroll
        for (int k = 0; k < TU; ++k) {
          const int t = tb + k * kWarps;
          ok[k] = t < t1;
          const int tt = ok[k] ? t : t0;
          const int page = upg[tt / kPageTokens - pbase];
          const int slot = tt % kPageTokens;
          const uint16_t* kp = a.kv + Kv<S>::offset(l, a.n_pages, page, 0, g, slot) + lane * DPL;
          const uint16_t* vp = a.kv + Kv<S>::offset(l, a.n_pages, page, 1, g, slot) + lane * DPL;
          if constexpr (DPL == 4) {
            const uint2 kr = __ldcg(reinterpret_cast<const uint2*>(kp));
            const uint2 vr = __ldcg(reinterpret_cast<const uint2*>(vp));
            kf[k][0] = bf16_to_f(kr.x & 0xffff); kf[k][1] = bf16_to_f(kr.x >> 16);
            kf[k][2] = bf16_to_f(kr.y & 0xffff); kf[k][3] = bf16_to_f(kr.y >> 16);
            vf[k][0] = bf16_to_f(vr.x & 0xffff); vf[k][1] = bf16_to_f(vr.x >> 16);
            vf[k][2] = bf16_to_f(vr.y & 0xffff); vf[k][3] = bf16_to_f(vr.y >> 16);
          } else {
            const uint32_t kr = __ldcg(reinterpret_cast<const unsigned int*>(kp));
            const uint32_t vr = __ldcg(reinterpret_cast<const unsigned int*>(vp));
            kf[k][0] = bf16_to_f(kr & 0xffff); kf[k][1] = bf16_to_f(kr >> 16);
            vf[k][0] = bf16_to_f(vr & 0xffff); vf[k][1] = bf16_to_f(vr >> 16);
          }
        }
        // scores of the TU positions for the GQA heads: lane partials, one
        // transposing reduction for all of them, then broadcast back
        constexpr int NV = TU * GQA;
        constexpr int NB = NV == 32 ? 5 : NV == 16 ? 4 : NV == 8 ? 3 : NV == 4 ? 2 : NV == 2 ? 1 : 0;
        float sv[NV];
#pragma unroll
        for (int k = 0; k < TU; ++k)
#pragma unroll
          for (int i = 0; i < GQA; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc = fmaf(q[i][d], kf[k][d], acc);
            sv[k * GQA + i] = acc;
          }
        const float mine = warp_reduce_scatter<NV>(sv, lane);
        float sc[TU][GQA];
#pragma unroll
        for (int idx = 0; idx < NV; ++idx)
          sc[idx / GQA][idx % GQA] = __shfl_sync(0xffffffffu, mine, bitrev<NB>(idx));
        // one online-softmax update per head for the whole batch
#pragma unroll
        for (int i = 0; i < GQA; ++i) {
          float mn = m[i];
#pragma unroll
          for (int k = 0; k < TU; ++k) mn = ok[k] ? fmaxf(mn, sc[k][i]) : mn;
          const float corr = __expf(m[i] - mn);
          float psum = 0.f, p[TU];
#pragma unroll
          for (int k = 0; k < TU; ++k) {
            p[k] = ok[k] ? __expf(sc[k][i] - mn) : 0.f;
            psum += p[k];
          }
          lsum[i] = fmaf(lsum[i], corr, psum);
#pragma unroll
          for (int d = 0; d < DPL; ++d) {
            float acc = o[i][d] * corr;
#pragma unroll
            for (int k = 0; k < TU; ++k) acc = fmaf(p[k], vf[k][d], acc);
            o[i][d] = acc;
          }
          m[i] = mn;
        }
      }
#pragma unroll
      for (int i = 0; i < GQA; ++i) {
        float* cw = comb + (wid * GQA + i) * (HD + 2);
        if (lane == 0) { cw[0] = m[i]; cw[1] = lsum[i]; }
#pragma unroll
        for (int d = 0; d < DPL; ++d) cw[2 + lane * DPL + d] = o[i][d];
      }
      __syncthreads();
      if (u >= a.max_units) set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_UNIT, u);
      float* pu = a.sc.part + (size_t)min(u, a.max_units - 1) * GQA * PR;
      // factors exp(m_w - M) once per (warp, head), then a weighted sum per dim
      float* fac = F.red;                 // [kWarps][GQA], then M[GQA]
      float* Ms = F.red + kWarps * GQA;
      if (tid < GQA) {
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, comb[(w * GQA + tid) * (HD + 2)]);
        Ms[tid] = M;
      }
      __syncthreads();
      if (tid < kWarps * GQA) {
        const int w = tid / GQA, i = tid % GQA;
        const float mw = comb[(w * GQA + i) * (HD + 2)];
        fac[tid] = mw == -INFINITY ? 0.f : __expf(mw - Ms[i]);
      }
      __syncthreads();
      for (int idx = tid; idx < GQA * HD; idx += kThreads) {
        const int i = idx / HD, d = idx % HD;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float* cw = comb + (w * GQA + i) * (HD + 2);
          L = fmaf(cw[1], fac[w * GQA + i], L);
          O = fmaf(cw[2 + d], fac[w * GQA + i], O);
        }
        if (d == 0) { pu[i * PR] = Ms[i]; pu[i * PR + 1] = L; }
        pu[i * PR + 4 + d] = O;
      }
      __syncthreads();
      if (tid == 0) {
        // release this unit's partial, acquire the others' if it is the last
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(old) : "l"(a.sc.merge_cnt + b * NKV + g) : "memory");
        F.flag = old == nch - 1;
      }
      __syncthreads();
      if (F.flag) {  // last unit of (b, g): log-sum-exp merge of its chunks
        if (nch > kMaxChunks || nch * GQA > kThreads) {
          if (tid == 0) set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_UNIT, nch);
          __syncthreads();
          continue;
        }
        const float* pb = a.sc.part + (size_t)(F.unit_start[b] + g * nch) * GQA * PR;
        // one warp per head: M = max_c m_c, L = sum_c l_c exp(m_c - M), and the
        // chunk factors exp(m_c - M) / L into shared memory
        float* mfac = F.red;  // [nch][GQA]
        if (wid < GQA) {
          const int i = wid;
          float mv[2], lv[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int cc = lane + 32 * r;
            mv[r] = cc < nch ? __ldcg(pb + (cc * GQA + i) * PR) : -INFINITY;
            lv[r] = cc < nch ? __ldcg(pb + (cc * GQA + i) * PR + 1) : 0.f;
          }
          const float M = warp_max(fmaxf(mv[0], mv[1]));
          float f[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) f[r] = mv[r] == -INFINITY ? 0.f : __expf(mv[r] - M);
          const float Linv = 1.f / warp_sum(fmaf(lv[0], f[0], lv[1] * f[1]));
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int cc = lane + 32 * r;
            if (cc < nch) mfac[cc * GQA + i] = f[r] * Linv;
          }
        }
        __syncthreads();
        // weighted sum of the chunk outputs, read from L2 eight chunks at a time
        for (int idx = tid; idx < GQA * HD; idx += kThreads) {
          const int i = idx / HD, d = idx % HD;
          float O = 0.f;
          for (int c0 = 0; c0 < nch; c0 += 8) {
            float ov[8];
#pragma unroll
            for (int u2 = 0; u2 < 8; ++u2)
              ov[u2] = c0 + u2 < nch ? __ldcg(pb + ((c0 + u2) * GQA + i) * PR + 4 + d) : 0.f;
#pragma unroll
            for (int u2 = 0; u2 < 8; ++u2)
              if (c0 + u2 < nch) O = fmaf(ov[u2], mfac[(c0 + u2) * GQA + i], O);
          }
          a.sc.attn[b * QD + (g * GQA + i) * HD + d] = O;
          if (c.tr_attn) c.tr_attn[((size_t)l * n + b) * QD + (g * GQA + i) * HD + d] = O;
        }
        if (tid == 0) a.sc.merge_cnt[b * NKV + g] = 0;
      }
      __syncthreads();
    }
  }

  // ---------------------------------------------------------------- P3
  // o_proj rows of this block + residual.  In MoE layers the block also forms
  // its partial router logits: the post-attention RMSNorm is one scalar per
  // row times w2, so logits = rsqrt(mean(h^2) + eps) * sum_blocks(partials);
  // the scalar is applied in P4.  The last block to finish adds the
  // partials in block order (deterministic).
  __device__ static __noinline__ void oproj(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    const LayerW& Lw = F.lw;
    const int n = c.n;
    {
      const float* at = a.sc.attn;
      stage_block<WDT, QD>(
          c.act, n, [&](int r, int f4) { return __ldcg(reinterpret_cast<const float4*>(at + r * QD) + f4); },
          false, 0.f, [&](int) { return make_float4(1.f, 1.f, 1.f, 1.f); }, F.red, nullptr);
    }
    __syncthreads();
    MK_STAMP(c, l, 2, 0);
    struct {
      const StepArgs* a; const LayerW* Lw; Fixed* F; int r0, lane;
      __device__ __forceinline__ RowRef row(int t, int) const {
        return {(const uint8_t*)Lw->w[WO] + (size_t)(r0 + t) * GQ::ROW_BYTES,
                (const uint16_t*)Lw->s[WO] + (size_t)(r0 + t) * (QD / 64)};
      }
      __device__ __forceinline__ ActRange acts(int) const {
        return {nullptr, 0, a->n};
      }
      __device__ __forceinline__ void out(int t, int b, int, float v0, float v1) const {
        if (lane != 0) return;
        const float hv = __ldcg(a->sc.x + b * H + r0 + t) + v0;
        a->sc.h[b * H + r0 + t] = hv;
        F->hs[b][t] = hv;
      }
    } task{&a, &Lw, &F, c.r0, lane};
    run_tasks<WDT, QD, 1>(c.nr, c.act, task);
    if (l < a.n_dense) return;
    __syncthreads();
    for (int idx = tid; idx < n * E; idx += kThreads) {
      const int b = idx / E, e = idx % E;
      float s = 0.f;
      for (int t = 0; t < c.nr; ++t)
        s = fmaf(F.hs[b][t] * ld_aux<AUX>(Lw.ffn_norm, c.r0 + t), ld_aux<AUX>(Lw.router, e * H + c.r0 + t), s);
      // every block adds its partial; after the grid barrier all blocks read
      // the same totals (the order of the additions may differ run to run)
      atomicAdd(a.sc.rlogit + b * E + e, s);
    }
  }

  // ---------------------------------------------------------------- P4a
  // Routing, then the post-attention RMSNorm.  The router logits of a row are
  // rsqrt(mean(h^2) + eps) times the block-summed partials of P3; that factor
  // is positive and common to the row, so the top-k selection (ties -> lower
  // expert id) is made from the partials before the norm is known.  The
  // selected experts' weights are then requested from HBM while the norm is
  // computed, and the softmax weights (renormalised over the selection) are
  // formed from the scaled logits.  Dense layers only norm.
  __device__ static __noinline__ void route(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    const LayerW& Lw = F.lw;
    const bool moe = l >= a.n_dense;
    const int n = c.n;
    constexpr int EJ = (E + 31) / 32;
    if (moe) {
      for (int b = wid; b < n; b += kWarps) {
        float lg[EJ];
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
          const int e = lane + 32 * j;
          lg[j] = e < E ? __ldcg(a.sc.rlogit + b * E + e) : -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < TOPK; ++k) {
          float bv = -INFINITY;
          int be = INT_MAX;
#pragma unroll
          for (int j = 0; j < EJ; ++j) {
            const int e = lane + 32 * j;
            if (e < E && (lg[j] > bv || (lg[j] == bv && e < be))) { bv = lg[j]; be = e; }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
          }
          if (lane == 0) { F.topk_id[b][k] = be; F.topk_w[b][k] = bv; }  // partial logit for now
#pragma unroll
          for (int j = 0; j < EJ; ++j)
            if (lane + 32 * j == be) lg[j] = -INFINITY;
        }
      }
      __syncthreads();
      if (wid == 0) {
        // entries sorted by (expert, row, slot); one run of rows per distinct expert
        int base = 0, nue = 0;
#pragma unroll
        for (int j = 0; j < EJ; ++j) {
          const int e = lane + 32 * j;
          int cnt = 0;
          for (int b = 0; b < n; ++b)
            for (int k = 0; k < TOPK; ++k) cnt += F.topk_id[b][k] == e;
          const int has = cnt > 0;
          int incl = cnt, hincl = has;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            const int hy = __shfl_up_sync(0xffffffffu, hincl, o);
            if (lane >= o) { incl += y; hincl += hy; }
          }
          const int start = base + incl - cnt;
          const int ue = nue + hincl - has;
          if (has) {
            F.ue_expert[ue] = (int16_t)e;
            F.ue_start[ue] = (int16_t)start;
            F.ue_len[ue] = (int16_t)cnt;
            int pos = start;
            for (int b = 0; b < n; ++b)
              for (int k = 0; k < TOPK; ++k)
                if (F.topk_id[b][k] == e) {
                  F.ent_b[pos] = (uint8_t)b;
                  F.ent_j[pos] = (uint8_t)k;
                  F.ent_of[b][k] = (uint8_t)pos;
                  ++pos;
                }
          }
          base += __shfl_sync(0xffffffffu, incl, 31);
          nue += __shfl_sync(0xffffffffu, hincl, 31);
        }
        if (lane == 0) F.n_ue = nue;
      }
      __syncthreads();
    }
    {
      const void* nw = Lw.ffn_norm;
      const float* hp = a.sc.h;
      stage_block<WDT, H>(
          c.act, n, [&](int r, int f4) { return __ldcg(reinterpret_cast<const float4*>(hp + r * H) + f4); },
          true, a.eps, [&](int f4) { return ld_aux4<AUX>(nw, f4); }, F.red, F.rnorm);
    }
    __syncthreads();
    MK_STAMP(c, l, 3, 0);
    if (!moe) return;
    for (int b = wid; b < n; b += kWarps) {
      const float r = F.rnorm[b];
      if (c.tr_rl && c.bid == 0)
        for (int e = lane; e < E; e += 32)
          c.tr_rl[((size_t)l * n + b) * E + e] = r * __ldcg(a.sc.rlogit + b * E + e);
      if (lane == 0) {
        // softmax over the selection = softmax over all experts renormalised
        const float top = r * F.topk_w[b][0];
        float wk[TOPK], wsum = 0.f;
#pragma unroll
        for (int k = 0; k < TOPK; ++k) {
          wk[k] = expf(r * F.topk_w[b][k] - top);
          wsum += wk[k];
        }
#pragma unroll
        for (int k = 0; k < TOPK; ++k) {
          F.topk_w[b][k] = wk[k] / wsum;
          if (c.tr_tk && c.bid == 0) {
            c.tr_tk[((size_t)l * n + b) * 2 * TOPK + k] = (float)F.topk_id[b][k];
            c.tr_tk[((size_t)l * n + b) * 2 * TOPK + TOPK + k] = wk[k] / wsum;
          }
        }
      }
    }
  }

  // After routing (all threads): this block's gate/up and down rows of layer l,
  // then the attention weights and cached K/V of layer l + 1 (or the start of
  // its lm_head rows after the last layer).
  __device__ static void prefetch_ffn_and_next(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    const LayerW& Lw = F.lw;
    if (l >= a.n_dense) {
      int u0, u1;
      split_range(F.n_ue * FE, c.G, c.bid, u0, u1);
      for (int ue = u0 / FE; ue < F.n_ue && ue * FE < u1; ++ue) {
        const int e = F.ue_expert[ue];
        const int f0 = max(u0, ue * FE) - ue * FE, f1 = min(u1, (ue + 1) * FE) - ue * FE;
        for (int m = EGATE; m <= EUP; ++m)
          prefetch_rows(Lw.w[m], Lw.s[m], (size_t)e * FE + f0, f1 - f0, GH::ROW_BYTES, H / 64 * 2);
      }
      for (int ue = 0; ue < F.n_ue; ++ue)
        prefetch_rows(Lw.w[EDOWN], Lw.s[EDOWN], (size_t)F.ue_expert[ue] * H + c.r0, c.nr, GE::ROW_BYTES,
                      FE / 64 * 2);
    } else {
      int f0, f1;
      split_range(FD, c.G, c.bid, f0, f1);
      for (int m = GATE; m <= UP; ++m) prefetch_rows(Lw.w[m], Lw.s[m], f0, f1 - f0, GH::ROW_BYTES, H / 64 * 2);
      prefetch_rows(Lw.w[DOWN], Lw.s[DOWN], c.r0, c.nr, NSEG * GS::ROW_BYTES, FD / 64 * 2);
    }
    if (l + 1 < a.n_layers) {
      prefetch_attn_weights(l + 1);
      prefetch_kv(l + 1);
    } else if (a.out_first < c.n) {
      int v0, v1;
      split_range(a.vocab, c.G, c.bid, v0, v1);
      prefetch_rows(a.lm_head, a.lm_head_s, v0, min(v1 - v0, 128), GH::ROW_BYTES, H / 64 * 2);
    }
  }

  // ---------------------------------------------------------------- P4b
  // Gate/up rows -> silu(gate) * up.  MoE: units (distinct expert, ffn row),
  // each computed for every row routed to that expert.  Dense: ffn rows.
  __device__ static __noinline__ void gateup(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    const LayerW& Lw = F.lw;
    if (l >= a.n_dense) {
      int u0, u1;
      split_range(F.n_ue * FE, c.G, c.bid, u0, u1);
      struct {
        const StepArgs* a; const LayerW* Lw; Fixed* F; int u0, lane;
        __device__ __forceinline__ RowRef row(int t, int r) const {
          const int u = u0 + t, e = F->ue_expert[u / FE], f = u % FE;
          const size_t rr = (size_t)e * FE + f;
          return {(const uint8_t*)Lw->w[r ? EUP : EGATE] + rr * GH::ROW_BYTES,
                  (const uint16_t*)Lw->s[r ? EUP : EGATE] + rr * (H / 64)};
        }
        __device__ __forceinline__ ActRange acts(int t) const {
          const int ue = (u0 + t) / FE;
          return {F->ent_b, F->ue_start[ue], F->ue_len[ue]};
        }
        __device__ __forceinline__ void out(int t, int b, int i, float v0, float v1) const {
          if (lane != 0) return;
          const int u = u0 + t, f = u % FE;
          const int j = F->ent_j[F->ue_start[u / FE] + i];
          a->sc.act[(b * TOPK + j) * FE + f] = silu(v0) * v1;
        }
      } task{&a, &Lw, &F, u0, lane};
      run_tasks<WDT, H, 2>(u1 - u0, c.act, task);
    } else {
      int f0, f1;
      split_range(FD, c.G, c.bid, f0, f1);
      struct {
        const StepArgs* a; const LayerW* Lw; int f0, lane;
        __device__ __forceinline__ RowRef row(int t, int r) const {
          return {(const uint8_t*)Lw->w[r ? UP : GATE] + (size_t)(f0 + t) * GH::ROW_BYTES,
                  (const uint16_t*)Lw->s[r ? UP : GATE] + (size_t)(f0 + t) * (H / 64)};
        }
        __device__ __forceinline__ ActRange acts(int) const {
          return {nullptr, 0, a->n};
        }
        __device__ __forceinline__ void out(int t, int b, int, float v0, float v1) const {
          if (lane == 0) a->sc.dact[b * FD + f0 + t] = silu(v0) * v1;
        }
      } task{&a, &Lw, f0, lane};
      run_tasks<WDT, H, 2>(f1 - f0, c.act, task);
    }
  }

  // ---------------------------------------------------------------- P5
  // Down projection of this block's hidden rows.  Activation vectors
  // ("entries": (row, expert slot) in MoE layers, (segment, row) in dense
  // layers) are staged in rounds that fit the staging area; entries sharing
  // one weight matrix form a run, so each weight row is read once per run.
  // The weighted sum over experts is taken in slot order, then the residual.
  template <bool MOE>
  __device__ static __noinline__ void down(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    const LayerW& Lw = F.lw;
    using GD = typename std::conditional<MOE, GE, GS>::type;
    const int n = c.n, nr = c.nr;
    const int nent = MOE ? n * TOPK : n * NSEG;
    const int cap = kActBytes / GD::ACT_BYTES;
    for (int base = 0; base < nent; base += cap) {
      const int cnt = min(cap, nent - base);
      {
        const float* act = a.sc.act;
        const float* dact = a.sc.dact;
        const Fixed* Fp = &F;
        stage_block<WDT, MOE ? FE : KSD>(
            c.act, cnt,
            [&](int r, int f4) -> float4 {
              const int en = base + r;
              const float* src = MOE ? act + (Fp->ent_b[en] * TOPK + Fp->ent_j[en]) * FE
                                     : dact + (en % n) * FD + (en / n) * KSD;
              return __ldcg(reinterpret_cast<const float4*>(src) + f4);
            },
            false, 0.f, [&](int) { return make_float4(1.f, 1.f, 1.f, 1.f); }, F.red, nullptr);
      }
      if (tid == 0) {
        int nrun = 0;
        for (int en = base; en < base + cnt; ++en) {
          const int mat = MOE ? F.topk_id[F.ent_b[en]][F.ent_j[en]] : en / n;
          if (nrun == 0 || F.run_mat[nrun - 1] != mat) {
            F.run_mat[nrun] = (int16_t)mat;
            F.run_start[nrun] = (int16_t)(en - base);
            F.run_len[nrun] = 0;
            ++nrun;
          }
          ++F.run_len[nrun - 1];
        }
        F.n_runs = nrun;
      }
      __syncthreads();
      MK_STAMP(c, l, 4, 0);
      struct {
        const LayerW* Lw; Fixed* F; int r0, nr, base, lane;
        __device__ __forceinline__ RowRef row(int t, int) const {
          const int run = t / nr, rr = t % nr, mat = F->run_mat[run];
          if (MOE) {
            const size_t row = (size_t)mat * H + r0 + rr;
            return {(const uint8_t*)Lw->w[EDOWN] + row * GD::ROW_BYTES,
                    (const uint16_t*)Lw->s[EDOWN] + row * (FE / 64)};
          } else {
            const size_t row = (size_t)(r0 + rr);
            return {(const uint8_t*)Lw->w[DOWN] + (row * NSEG + mat) * GD::ROW_BYTES,
                    (const uint16_t*)Lw->s[DOWN] + row * (FD / 64) + mat * (KSD / 64)};
          }
        }
        __device__ __forceinline__ ActRange acts(int t) const {
          const int run = t / nr;
          return {nullptr, F->run_start[run], F->run_len[run]};
        }
        __device__ __forceinline__ void out(int t, int ai, int, float v0, float v1) const {
          if (lane == 0) F->dots[base + ai][t % nr] = v0;
        }
      } task{&Lw, &F, c.r0, nr, base, lane};
      run_tasks<WDT, MOE ? FE : KSD, 1>(F.n_runs * nr, c.act, task);
      __syncthreads();
    }
    for (int idx = tid; idx < n * nr; idx += kThreads) {
      const int b = idx / nr, rr = idx % nr;
      float s = 0.f;
      if (MOE)
        for (int k = 0; k < TOPK; ++k) s = fmaf(F.topk_w[b][k], F.dots[F.ent_of[b][k]][rr], s);
      else
        for (int sg = 0; sg < NSEG; ++sg) s += F.dots[sg * n + b][rr];
      const float xv = __ldcg(a.sc.h + b * H + c.r0 + rr) + s;
      a.sc.x[b * H + c.r0 + rr] = xv;
      if (c.tr_x) c.tr_x[((size_t)l * n + b) * H + c.r0 + rr] = xv;
    }
  }

  // ---------------------------------------------------------------- lm_head
  // Final RMSNorm, this block's vocabulary rows, argmax per row of the batch
  // (ties -> lowest token id); the last block to finish reduces the blocks'
  // candidates in block order and writes the tokens.
  __device__ static __noinline__ void lm_head() {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    (void)tid; (void)lane; (void)wid;
    const int n = c.n;
    {
      const void* nw = a.final_norm;
      const float* x = a.sc.x + a.out_first * H;
      stage_block<WDT, H>(
          c.act + a.out_first * GH::ACT_BYTES, n - a.out_first,
          [&](int r, int f4) { return __ldcg(reinterpret_cast<const float4*>(x + r * H) + f4); },
          true, a.eps, [&](int f4) { return ld_aux4<AUX>(nw, f4); }, F.red, nullptr);
    }
    for (int i = tid; i < kWarps * kMaxBatch; i += kThreads) {
      F.best_v[i / kMaxBatch][i % kMaxBatch] = -INFINITY;
      F.best_i[i / kMaxBatch][i % kMaxBatch] = INT_MAX;
    }
    __syncthreads();
    int v0, v1;
    split_range(a.vocab, c.G, c.bid, v0, v1);
    struct {
      const StepArgs* a; Fixed* F; float* tr; int vr0, lane, wid;
      __device__ __forceinline__ RowRef row(int t, int) const {
        return {(const uint8_t*)a->lm_head + (size_t)(vr0 + t) * GH::ROW_BYTES,
                (const uint16_t*)a->lm_head_s + (size_t)(vr0 + t) * (H / 64)};
      }
      __device__ __forceinline__ ActRange acts(int) const {
        return {nullptr, a->out_first, a->n - a->out_first};
      }
      __device__ __forceinline__ void out(int t, int b, int, float v0, float v1) const {
        if (lane != 0) return;
        const int tok = vr0 + t;
        // a warp visits its rows in increasing order: '>' keeps the lowest id
        if (v0 > F->best_v[wid][b]) { F->best_v[wid][b] = v0; F->best_i[wid][b] = tok; }
        if (tr) tr[(size_t)b * a->vocab + tok] = v0;
      }
    } task{&a, &F, c.tr_fin, v0, lane, wid};
    run_tasks<WDT, H, 1>(v1 - v0, c.act, task);
    __syncthreads();
    if (tid < n) {
      float bv = -INFINITY;
      int bi = INT_MAX;
      for (int w = 0; w < kWarps; ++w) {
        const float v = F.best_v[w][tid];
        const int i = F.best_i[w][tid];
        if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
      }
      a.sc.amax_v[c.bid * kMaxBatch + tid] = bv;
      a.sc.amax_i[c.bid * kMaxBatch + tid] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      F.flag = atomicAdd(a.sc.sync + 96, 1u) == (uint32_t)(c.G - 1);
    }
    __syncthreads();
    if (!F.flag) return;
    __threadfence();
    for (int b = a.out_first + wid; b < n; b += kWarps) {
      float bv = -INFINITY;
      int bi = INT_MAX;
      for (int g = lane; g < c.G; g += 32) {
        const float v = __ldcg(a.sc.amax_v + g * kMaxBatch + b);
        const int i = __ldcg(a.sc.amax_i + g * kMaxBatch + b);
        if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) a.out_tokens[b - a.out_first] = bi == INT_MAX ? 0 : bi;
    }
    if (tid == 0) a.sc.sync[96] = 0;
  }
};

template <class S, int WDT>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepArgs a) {
  using M = Model<S, WDT>;
  extern __shared__ __align__(128) uint8_t smem[];
  Fixed& F = *reinterpret_cast<Fixed*>(smem);
  const int tid = threadIdx.x;
  // launch arguments into shared memory: the phases read them from there
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&a);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&F.args);
    static_assert(sizeof(StepArgs) % 4 == 0, "word copy");
    for (int i = tid; i < (int)(sizeof(StepArgs) / 4); i += kThreads) dst[i] = src[i];
  }
  const int n = a.n;
  if (tid == 0) {
    Ctx& c = F.ctx;
    c.act = smem + kActOffset;
    c.G = gridDim.x;
    c.bid = blockIdx.x;
    c.n = n;
    int r0, r1;
    split_range(S::H, c.G, c.bid, r0, r1);
    c.r0 = r0;
    c.nr = r1 - r0;
    c.tr_x = a.trace;
    c.tr_attn = a.trace ? c.tr_x + (size_t)a.n_layers * n * S::H : nullptr;
    c.tr_rl = a.trace ? c.tr_attn + (size_t)a.n_layers * n * M::QD : nullptr;
    c.tr_tk = a.trace ? c.tr_rl + (size_t)a.n_layers * n * S::E : nullptr;
    c.tr_fin = a.trace ? c.tr_tk + (size_t)a.n_layers * n * 2 * S::TOPK : nullptr;
    c.tm = (a.timing && blockIdx.x == 0) ? a.timing : nullptr;
    // attention work units: (row, kv head, chunk), row-major
    int acc = 0;
    for (int b = 0; b < n; ++b) {
      F.unit_start[b] = acc;
      acc += S::NKV * ((a.pos[b] + 1 + a.chunk - 1) / a.chunk);
    }
    F.unit_start[n] = acc;
  }
  // token ids (device memory; may be the previous step's output)
  if (tid < n) {
    int t = a.tokens[tid];
    if (t < 0 || t >= a.vocab) {
      set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_TOKEN, t);
      t = 0;
    }
    F.tok[tid] = t;
  }
  __syncthreads();
  const Ctx& c = F.ctx;

  uint32_t nbar = 0;
  if (c.tm && tid == 0) c.tm[0] = globaltimer();
  for (int l = 0; l < a.n_layers; ++l) {
    {  // this layer's weight pointers into shared memory (read by every task)
      const uint32_t* src = reinterpret_cast<const uint32_t*>(a.layers + l);
      uint32_t* dst = reinterpret_cast<uint32_t*>(&F.lw);
      for (int i = tid; i < (int)(sizeof(LayerW) / 4); i += kThreads) dst[i] = __ldg(src + i);
      __syncthreads();
    }
    M::qkv(l);
    MK_STAMP(c, l, 0, 1);
    if (!grid_barrier(a, nbar)) goto done;
    MK_STAMP(c, l, 0, 2);
    M::attention(l);
    MK_STAMP(c, l, 1, 1);
    if (!grid_barrier(a, nbar)) goto done;
    MK_STAMP(c, l, 1, 2);
    M::oproj(l);
    MK_STAMP(c, l, 2, 1);
    if (!grid_barrier(a, nbar)) goto done;
    MK_STAMP(c, l, 2, 2);
    M::route(l);
    __syncthreads();
    M::gateup(l);
    MK_STAMP(c, l, 3, 1);
    if (!grid_barrier(a, nbar)) goto done;
    MK_STAMP(c, l, 3, 2);
    if (l >= a.n_dense) M::template down<true>(l);
    else M::template down<false>(l);
    MK_STAMP(c, l, 4, 1);
    if (!grid_barrier(a, nbar)) goto done;
    MK_STAMP(c, l, 4, 2);
  }
  if (a.out_first < n) M::lm_head();
  if (c.tm && tid == 0) c.tm[1 + 16 * a.n_layers] = globaltimer();

done:
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.sc.sync + 32, 1u) == (uint32_t)(c.G - 1)) {
      // every block has left its work: reset the launch-scoped counters
      a.sc.sync[0] = 0;
      a.sc.sync[96] = 0;
      for (int i = 0; i < kMaxBatch * S::NKV; ++i) a.sc.merge_cnt[i] = 0;
      __threadfence();
      a.sc.sync[32] = 0;
    }
  }
}

template <class S, int WDT>
static KernelInfo make() {
  return {reinterpret_cast<const void*>(&step_kernel<S, WDT>), kSmemBytes};
}

KernelInfo get_kernel(int shape, int wdtype) {
  if (shape == SHAPE_FLINT) {
    if (wdtype == MK_INT4_G64) return make<ShapeFlint, WINT4>();
    if (wdtype == MK_BF16) return make<ShapeFlint, WBF16>();
  } else if (shape == SHAPE_TINY) {
    if (wdtype == MK_INT4_G64) return make<ShapeTiny, WINT4>();
    if (wdtype == MK_BF16) return make<ShapeTiny, WBF16>();
    if (wdtype == MK_F32) return make<ShapeTiny, WF32>();
  }
  return {nullptr, 0};
}

}  // namespace mk
