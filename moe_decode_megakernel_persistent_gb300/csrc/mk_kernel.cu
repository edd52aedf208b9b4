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

struct Fixed {
  int topk_id[kMaxBatch][8];
  float topk_w[kMaxBatch][8];
  float dots[kMaxEnt][kMaxRowsPerBlock];
  float hs[kMaxBatch][kMaxRowsPerBlock];
  float red[kThreads];
  float best_v[kWarps][kMaxBatch];
  int best_i[kWarps][kMaxBatch];
  int unit_start[kMaxBatch + 1];
  int16_t ue_expert[64], ue_start[64], ue_len[64];
  int16_t run_start[kMaxEnt], run_len[kMaxEnt], run_mat[kMaxEnt];
  uint8_t ent_b[kMaxEnt], ent_j[kMaxEnt];
  uint8_t ent_of[kMaxBatch][8];
  int n_ue, n_runs, flag;
};
constexpr int kActOffset = (sizeof(Fixed) + 127) / 128 * 128;
constexpr int kActBytes = kSmemBytes - kActOffset;

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

template <class S>
struct Kv {
  __device__ static __forceinline__ size_t offset(int l, int n_pages, int page, int kvsel, int g,
                                                  int slot) {
    return ((((size_t)l * n_pages + page) * 2 + kvsel) * S::NKV + g) * (size_t)(kPageTokens * S::HD) +
           (size_t)slot * S::HD;
  }
};

// Per-launch context shared by the phases (one per block, in registers of
// the caller and passed by reference).
struct Ctx {
  const StepArgs* a;
  Fixed* F;
  uint8_t* act;    // staging area in shared memory
  const int* tok;  // token ids of the rows (shared memory)
  int tid, lane, wid, G, bid, n;
  int r0, nr;      // hidden rows owned by this block
  float *tr_x, *tr_attn, *tr_rl, *tr_tk, *tr_fin;
};

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
  static_assert(kWarps * GQA * (HD + 2) * 4 <= kActBytes, "attention combine buffer");
  static_assert(TOPK <= 8 && E <= 64, "router tables");

  __device__ static __forceinline__ float emb(const Ctx& c, int b, int k) {
    return ld_aux<AUX>(c.a->embed, c.tok[b] * H + k);
  }

  // ---------------------------------------------------------------- P1
  // RMSNorm of the residual (every block, redundantly) -> this block's rows of
  // the QKV projection.  A task is a RoPE pair of q or k rows (i, i + HD/2)
  // of one head, or two adjacent v rows, so the warp that forms a pair also
  // rotates it and writes it: q to scratch, k and v as bf16 into the page.
  __device__ static __noinline__ void qkv(const Ctx& c, int l) {
    const StepArgs& a = *c.a;
    const LayerW& Lw = a.layers[l];
    const int n = c.n, lane = c.lane;
    if (l == 0 && c.bid == 0)
      for (int i = c.tid; i < a.n_upd; i += kThreads)
        a.block_table[a.upd[i].slot * a.max_pages_per_seq + a.upd[i].index] = a.upd[i].page;
    for (int b = c.wid; b < n; b += kWarps) {
      const float* xb = a.sc.x + b * H;
      auto xv = [&](int k) -> float { return l == 0 ? emb(c, b, k) : __ldcg(xb + k); };
      const float r = rsqrtf(warp_sumsq<H>(lane, xv) / H + a.eps);
      GH::stage(c.act + b * GH::ACT_BYTES, lane,
                [&](int k) { return xv(k) * r * ld_aux<AUX>(Lw.attn_norm, k); });
    }
    if (l == 0)  // residual rows this block reads back in P3
      for (int i = c.tid; i < n * c.nr; i += kThreads) {
        const int b = i / c.nr, r = c.r0 + i % c.nr;
        a.sc.x[b * H + r] = emb(c, b, r);
      }
    __syncthreads();

    constexpr int NQP = NH * HALF, NKP = NKV * HALF, NP = NQP + 2 * NKP;
    int p0, p1;
    split_range(NP, c.G, c.bid, p0, p1);
    struct {
      const StepArgs* a; const LayerW* Lw; int p0, l, lane;
      __device__ void row(int t, int r, const uint8_t** w, const uint16_t** s) const {
        const int p = p0 + t;
        int m, row;
        if (p < NQP) { m = WQ; row = (p / HALF) * HD + p % HALF + r * HALF; }
        else if (p < NQP + NKP) { const int q = p - NQP; m = WK; row = (q / HALF) * HD + q % HALF + r * HALF; }
        else { const int q = p - NQP - NKP; m = WV; row = (q / HALF) * HD + 2 * (q % HALF) + r; }
        *w = (const uint8_t*)Lw->w[m] + (size_t)row * GH::ROW_BYTES;
        *s = (const uint16_t*)Lw->s[m] + (size_t)row * (H / 64);
      }
      __device__ int acts(int, const uint8_t** list, int* start) const {
        *list = nullptr; *start = 0; return a->n;
      }
      __device__ void out(int t, int b, int, const float* v) const {
        if (lane != 0) return;
        const int p = p0 + t;
        const int pos = a->pos[b];
        if (p < NQP + NKP) {
          const int q = p < NQP ? p : p - NQP;
          const int hh = q / HALF, i = q % HALF;
          const float2 cs = __ldg(a->rope + (size_t)pos * HALF + i);
          const float e0 = v[0] * cs.x - v[1] * cs.y;
          const float e1 = v[1] * cs.x + v[0] * cs.y;
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
          dst[i2] = f_to_bf16(v[0]);
          dst[i2 + 1] = f_to_bf16(v[1]);
        }
      }
    } task{&a, &Lw, p0, l, lane};
    run_tasks<WDT, H, 2>(p1 - p0, c.act, task);
  }

  // ---------------------------------------------------------------- P2
  // Split attention over the paged cache.  Unit = (row, kv head, chunk of
  // positions); warps take positions of the chunk, keep a running max, sum
  // and weighted value (online softmax) for the GQA heads of the kv head,
  // combine across warps, and write the unit's partial (m, l, o).  The last
  // unit of a (row, kv head) to finish merges all its chunks in chunk order.
  __device__ static __noinline__ void attention(const Ctx& c, int l) {
    const StepArgs& a = *c.a;
    Fixed& F = *c.F;
    const int n = c.n, tid = c.tid, lane = c.lane, wid = c.wid;
    if (tid == 0) {
      int acc = 0;
      for (int b = 0; b < n; ++b) {
        F.unit_start[b] = acc;
        acc += NKV * ((a.pos[b] + 1 + a.chunk - 1) / a.chunk);
      }
      F.unit_start[n] = acc;
    }
    __syncthreads();
    float* comb = reinterpret_cast<float*>(c.act);  // [warp][GQA][HD + 2]
    const float qscale = rsqrtf((float)HD);
    for (int u = c.bid; u < a.n_units; u += c.G) {
      int b = 0;
      while (b + 1 < n && F.unit_start[b + 1] <= u) ++b;
      const int ctx = a.pos[b] + 1;
      const int nch = (ctx + a.chunk - 1) / a.chunk;
      const int rem = u - F.unit_start[b];
      const int g = rem / nch, ci = rem % nch;
      const int t0 = ci * a.chunk, t1 = min(ctx, t0 + a.chunk);
      const int* bt = a.block_table + a.slot[b] * a.max_pages_per_seq;

      float q[GQA][DPL];
#pragma unroll
      for (int i = 0; i < GQA; ++i)
#pragma unroll
        for (int d = 0; d < DPL; ++d)
          q[i][d] = __ldcg(a.sc.q + b * QD + (g * GQA + i) * HD + lane * DPL + d) * qscale;
      float m[GQA], lsum[GQA], o[GQA][DPL];
#pragma unroll
      for (int i = 0; i < GQA; ++i) {
        m[i] = -INFINITY; lsum[i] = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[i][d] = 0.f;
      }
      for (int t = t0 + wid; t < t1; t += kWarps) {
        const int pi = t / kPageTokens;
        int page = pi < a.max_pages_per_seq ? __ldcg(bt + pi) : -1;
        if (page < 0 || page >= a.n_pages) {
          set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_PAGE, t);
          page = 0;
        }
        const int slot = t % kPageTokens;
        const uint16_t* kp = a.kv + Kv<S>::offset(l, a.n_pages, page, 0, g, slot) + lane * DPL;
        const uint16_t* vp = a.kv + Kv<S>::offset(l, a.n_pages, page, 1, g, slot) + lane * DPL;
        float kf[DPL], vf[DPL];
        if constexpr (DPL == 4) {
          const uint2 kr = __ldcg(reinterpret_cast<const uint2*>(kp));
          const uint2 vr = __ldcg(reinterpret_cast<const uint2*>(vp));
          kf[0] = bf16_to_f(kr.x & 0xffff); kf[1] = bf16_to_f(kr.x >> 16);
          kf[2] = bf16_to_f(kr.y & 0xffff); kf[3] = bf16_to_f(kr.y >> 16);
          vf[0] = bf16_to_f(vr.x & 0xffff); vf[1] = bf16_to_f(vr.x >> 16);
          vf[2] = bf16_to_f(vr.y & 0xffff); vf[3] = bf16_to_f(vr.y >> 16);
        } else {
          const uint32_t kr = __ldcg(reinterpret_cast<const unsigned int*>(kp));
          const uint32_t vr = __ldcg(reinterpret_cast<const unsigned int*>(vp));
          kf[0] = bf16_to_f(kr & 0xffff); kf[1] = bf16_to_f(kr >> 16);
          vf[0] = bf16_to_f(vr & 0xffff); vf[1] = bf16_to_f(vr >> 16);
        }
#pragma unroll
        for (int i = 0; i < GQA; ++i) {
          float s = 0.f;
#pragma unroll
          for (int d = 0; d < DPL; ++d) s = fmaf(q[i][d], kf[d], s);
          s = warp_sum(s);
          const float mn = fmaxf(m[i], s);
          const float corr = expf(m[i] - mn);
          const float p = expf(s - mn);
          lsum[i] = lsum[i] * corr + p;
#pragma unroll
          for (int d = 0; d < DPL; ++d) o[i][d] = fmaf(o[i][d], corr, p * vf[d]);
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
      float* pu = a.sc.part + (size_t)min(u, a.max_units - 1) * GQA * (HD + 2);
      for (int idx = tid; idx < GQA * HD; idx += kThreads) {
        const int i = idx / HD, d = idx % HD;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, comb[(w * GQA + i) * (HD + 2)]);
        float L = 0.f, O = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          const float* cw = comb + (w * GQA + i) * (HD + 2);
          const float f = cw[0] == -INFINITY ? 0.f : expf(cw[0] - M);
          L = fmaf(cw[1], f, L);
          O = fmaf(cw[2 + d], f, O);
        }
        if (d == 0) { pu[i * (HD + 2)] = M; pu[i * (HD + 2) + 1] = L; }
        pu[i * (HD + 2) + 2 + d] = O;
      }
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        const int old = atomicAdd(a.sc.merge_cnt + b * NKV + g, 1);
        F.flag = old == nch - 1;
      }
      __syncthreads();
      if (F.flag) {  // last unit of (b, g): log-sum-exp merge of its chunks
        __threadfence();
        const float* pb = a.sc.part + (size_t)(F.unit_start[b] + g * nch) * GQA * (HD + 2);
        for (int idx = tid; idx < GQA * HD; idx += kThreads) {
          const int i = idx / HD, d = idx % HD;
          float M = -INFINITY;
          for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(pb + (cc * GQA + i) * (HD + 2)));
          float L = 0.f, O = 0.f;
          for (int cc = 0; cc < nch; ++cc) {
            const float* pc = pb + (cc * GQA + i) * (HD + 2);
            const float f = expf(__ldcg(pc) - M);
            L = fmaf(__ldcg(pc + 1), f, L);
            O = fmaf(__ldcg(pc + 2 + d), f, O);
          }
          const float val = O / L;
          a.sc.attn[b * QD + (g * GQA + i) * HD + d] = val;
          if (c.tr_attn) c.tr_attn[((size_t)l * n + b) * QD + (g * GQA + i) * HD + d] = val;
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
  __device__ static __noinline__ void oproj(const Ctx& c, int l) {
    const StepArgs& a = *c.a;
    Fixed& F = *c.F;
    const LayerW& Lw = a.layers[l];
    const int n = c.n, tid = c.tid, lane = c.lane;
    for (int b = c.wid; b < n; b += kWarps) {
      const float* ab = a.sc.attn + b * QD;
      GQ::stage(c.act + b * GQ::ACT_BYTES, lane, [&](int k) { return __ldcg(ab + k); });
    }
    __syncthreads();
    struct {
      const StepArgs* a; const LayerW* Lw; Fixed* F; int r0, lane;
      __device__ void row(int t, int, const uint8_t** w, const uint16_t** s) const {
        *w = (const uint8_t*)Lw->w[WO] + (size_t)(r0 + t) * GQ::ROW_BYTES;
        *s = (const uint16_t*)Lw->s[WO] + (size_t)(r0 + t) * (QD / 64);
      }
      __device__ int acts(int, const uint8_t** list, int* start) const {
        *list = nullptr; *start = 0; return a->n;
      }
      __device__ void out(int t, int b, int, const float* v) const {
        if (lane != 0) return;
        const float hv = __ldcg(a->sc.x + b * H + r0 + t) + v[0];
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
      a.sc.rpart[((size_t)c.bid * kMaxBatch + b) * E + e] = s;
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      F.flag = atomicAdd(a.sc.sync + 64, 1u) == (uint32_t)(c.G - 1);
    }
    __syncthreads();
    if (F.flag) {
      __threadfence();
      const int P = n * E;
      const int NS = max(1, kThreads / P);
      for (int idx = tid; idx < P * NS; idx += kThreads) {
        const int p = idx % P, sp = idx / P;
        const int b = p / E, e = p % E;
        int g0, g1;
        split_range(c.G, NS, sp, g0, g1);
        float s = 0.f;
        for (int g = g0; g < g1; ++g) s += __ldcg(a.sc.rpart + ((size_t)g * kMaxBatch + b) * E + e);
        if (NS == 1) a.sc.rlogit[b * E + e] = s;
        else F.red[idx] = s;
      }
      if (NS > 1) {
        __syncthreads();
        for (int p = tid; p < P; p += kThreads) {
          float s = 0.f;
          for (int sp = 0; sp < NS; ++sp) s += F.red[sp * P + p];
          a.sc.rlogit[p] = s;
        }
      }
      if (tid == 0) a.sc.sync[64] = 0;
    }
  }

  // ---------------------------------------------------------------- P4a
  // RMSNorm of h (every block) and, in MoE layers, softmax over the experts,
  // top-k (ties -> lower expert id) and renormalised weights, then the
  // selections grouped by expert.
  __device__ static __noinline__ void route(const Ctx& c, int l) {
    const StepArgs& a = *c.a;
    Fixed& F = *c.F;
    const LayerW& Lw = a.layers[l];
    const bool moe = l >= a.n_dense;
    const int n = c.n, lane = c.lane, wid = c.wid;
    constexpr int EJ = (E + 31) / 32;
    for (int b = wid; b < n; b += kWarps) {
      const float* hb = a.sc.h + b * H;
      auto hv = [&](int k) -> float { return __ldcg(hb + k); };
      const float r = rsqrtf(warp_sumsq<H>(lane, hv) / H + a.eps);
      GH::stage(c.act + b * GH::ACT_BYTES, lane,
                [&](int k) { return hv(k) * r * ld_aux<AUX>(Lw.ffn_norm, k); });
      if (!moe) continue;
      float lg[EJ];
#pragma unroll
      for (int j = 0; j < EJ; ++j) {
        const int e = lane + 32 * j;
        lg[j] = e < E ? r * __ldcg(a.sc.rlogit + b * E + e) : -INFINITY;
        if (c.tr_rl && c.bid == 0 && e < E) c.tr_rl[((size_t)l * n + b) * E + e] = lg[j];
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < EJ; ++j) mx = fmaxf(mx, lg[j]);
      mx = warp_max(mx);
      float wsum = 0.f, wk[TOPK];
      int ids[TOPK];
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
        ids[k] = be;
        wk[k] = expf(bv - mx);
        wsum += wk[k];
#pragma unroll
        for (int j = 0; j < EJ; ++j)
          if (lane + 32 * j == be) lg[j] = -INFINITY;
      }
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < TOPK; ++k) {
          F.topk_id[b][k] = ids[k];
          F.topk_w[b][k] = wk[k] / wsum;
          if (c.tr_tk && c.bid == 0) {
            c.tr_tk[((size_t)l * n + b) * 2 * TOPK + k] = (float)ids[k];
            c.tr_tk[((size_t)l * n + b) * 2 * TOPK + TOPK + k] = wk[k] / wsum;
          }
        }
      }
    }
    __syncthreads();
    if (!moe || wid != 0) return;
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

  // ---------------------------------------------------------------- P4b
  // Gate/up rows -> silu(gate) * up.  MoE: units (distinct expert, ffn row),
  // each computed for every row routed to that expert.  Dense: ffn rows.
  __device__ static __noinline__ void gateup(const Ctx& c, int l) {
    const StepArgs& a = *c.a;
    Fixed& F = *c.F;
    const LayerW& Lw = a.layers[l];
    if (c.tid == 0) {  // warm L2 with this block's down-projection rows
      if (l >= a.n_dense) {
        for (int ue = 0; ue < F.n_ue; ++ue)
          prefetch_l2((const uint8_t*)Lw.w[EDOWN] + ((size_t)F.ue_expert[ue] * H + c.r0) * GE::ROW_BYTES,
                      c.nr * GE::ROW_BYTES);
      } else {
        prefetch_l2((const uint8_t*)Lw.w[DOWN] + (size_t)c.r0 * NSEG * GS::ROW_BYTES, c.nr * NSEG * GS::ROW_BYTES);
      }
    }
    if (l >= a.n_dense) {
      int u0, u1;
      split_range(F.n_ue * FE, c.G, c.bid, u0, u1);
      struct {
        const StepArgs* a; const LayerW* Lw; Fixed* F; int u0, lane;
        __device__ void row(int t, int r, const uint8_t** w, const uint16_t** s) const {
          const int u = u0 + t, e = F->ue_expert[u / FE], f = u % FE;
          const size_t rr = (size_t)e * FE + f;
          *w = (const uint8_t*)Lw->w[r ? EUP : EGATE] + rr * GH::ROW_BYTES;
          *s = (const uint16_t*)Lw->s[r ? EUP : EGATE] + rr * (H / 64);
        }
        __device__ int acts(int t, const uint8_t** list, int* start) const {
          const int ue = (u0 + t) / FE;
          *list = F->ent_b; *start = F->ue_start[ue]; return F->ue_len[ue];
        }
        __device__ void out(int t, int b, int i, const float* v) const {
          if (lane != 0) return;
          const int u = u0 + t, f = u % FE;
          const int j = F->ent_j[F->ue_start[u / FE] + i];
          a->sc.act[(b * TOPK + j) * FE + f] = silu(v[0]) * v[1];
        }
      } task{&a, &Lw, &F, u0, c.lane};
      run_tasks<WDT, H, 2>(u1 - u0, c.act, task);
    } else {
      int f0, f1;
      split_range(FD, c.G, c.bid, f0, f1);
      struct {
        const StepArgs* a; const LayerW* Lw; int f0, lane;
        __device__ void row(int t, int r, const uint8_t** w, const uint16_t** s) const {
          *w = (const uint8_t*)Lw->w[r ? UP : GATE] + (size_t)(f0 + t) * GH::ROW_BYTES;
          *s = (const uint16_t*)Lw->s[r ? UP : GATE] + (size_t)(f0 + t) * (H / 64);
        }
        __device__ int acts(int, const uint8_t** list, int* start) const {
          *list = nullptr; *start = 0; return a->n;
        }
        __device__ void out(int t, int b, int, const float* v) const {
          if (lane == 0) a->sc.dact[b * FD + f0 + t] = silu(v[0]) * v[1];
        }
      } task{&a, &Lw, f0, c.lane};
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
  __device__ static __noinline__ void down(const Ctx& c, int l) {
    const StepArgs& a = *c.a;
    Fixed& F = *c.F;
    const LayerW& Lw = a.layers[l];
    using GD = typename std::conditional<MOE, GE, GS>::type;
    const int n = c.n, tid = c.tid, lane = c.lane, nr = c.nr;
    const int nent = MOE ? n * TOPK : n * NSEG;
    const int cap = kActBytes / GD::ACT_BYTES;
    for (int base = 0; base < nent; base += cap) {
      const int cnt = min(cap, nent - base);
      for (int en = base + c.wid; en < base + cnt; en += kWarps) {
        const float* src = MOE ? a.sc.act + (F.ent_b[en] * TOPK + F.ent_j[en]) * FE
                               : a.sc.dact + (en % n) * FD + (en / n) * KSD;
        GD::stage(c.act + (en - base) * GD::ACT_BYTES, lane, [&](int k) { return __ldcg(src + k); });
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
      struct {
        const LayerW* Lw; Fixed* F; int r0, nr, base, lane;
        __device__ void row(int t, int, const uint8_t** w, const uint16_t** s) const {
          const int run = t / nr, rr = t % nr, mat = F->run_mat[run];
          if (MOE) {
            const size_t row = (size_t)mat * H + r0 + rr;
            *w = (const uint8_t*)Lw->w[EDOWN] + row * GD::ROW_BYTES;
            *s = (const uint16_t*)Lw->s[EDOWN] + row * (FE / 64);
          } else {
            const size_t row = (size_t)(r0 + rr);
            *w = (const uint8_t*)Lw->w[DOWN] + (row * NSEG + mat) * GD::ROW_BYTES;
            *s = (const uint16_t*)Lw->s[DOWN] + row * (FD / 64) + mat * (KSD / 64);
          }
        }
        __device__ int acts(int t, const uint8_t** list, int* start) const {
          const int run = t / nr;
          *list = nullptr; *start = F->run_start[run]; return F->run_len[run];
        }
        __device__ void out(int t, int ai, int, const float* v) const {
          if (lane == 0) F->dots[base + ai][t % nr] = v[0];
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
  __device__ static __noinline__ void lm_head(const Ctx& c) {
    const StepArgs& a = *c.a;
    Fixed& F = *c.F;
    const int n = c.n, tid = c.tid, lane = c.lane, wid = c.wid;
    for (int b = a.out_first + wid; b < n; b += kWarps) {
      const float* xb = a.sc.x + b * H;
      auto xv = [&](int k) -> float { return __ldcg(xb + k); };
      const float r = rsqrtf(warp_sumsq<H>(lane, xv) / H + a.eps);
      GH::stage(c.act + b * GH::ACT_BYTES, lane,
                [&](int k) { return xv(k) * r * ld_aux<AUX>(a.final_norm, k); });
    }
    for (int i = tid; i < kWarps * kMaxBatch; i += kThreads) {
      F.best_v[i / kMaxBatch][i % kMaxBatch] = -INFINITY;
      F.best_i[i / kMaxBatch][i % kMaxBatch] = INT_MAX;
    }
    __syncthreads();
    int v0, v1;
    split_range(a.vocab, c.G, c.bid, v0, v1);
    struct {
      const StepArgs* a; Fixed* F; float* tr; int v0, lane, wid;
      __device__ void row(int t, int, const uint8_t** w, const uint16_t** s) const {
        *w = (const uint8_t*)a->lm_head + (size_t)(v0 + t) * GH::ROW_BYTES;
        *s = (const uint16_t*)a->lm_head_s + (size_t)(v0 + t) * (H / 64);
      }
      __device__ int acts(int, const uint8_t** list, int* start) const {
        *list = nullptr; *start = a->out_first; return a->n - a->out_first;
      }
      __device__ void out(int t, int b, int, const float* v) const {
        if (lane != 0) return;
        const int tok = v0 + t;
        // a warp visits its rows in increasing order: '>' keeps the lowest id
        if (v[0] > F->best_v[wid][b]) { F->best_v[wid][b] = v[0]; F->best_i[wid][b] = tok; }
        if (tr) tr[(size_t)b * a->vocab + tok] = v[0];
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
    const int b = wid;
    if (b >= a.out_first && b < n) {
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
  __shared__ int s_tok[kMaxBatch];
  Ctx c;
  c.a = &a;
  c.F = reinterpret_cast<Fixed*>(smem);
  c.act = smem + kActOffset;
  c.tok = s_tok;
  c.tid = threadIdx.x;
  c.lane = c.tid & 31;
  c.wid = c.tid >> 5;
  c.G = gridDim.x;
  c.bid = blockIdx.x;
  c.n = a.n;
  int r1;
  split_range(S::H, c.G, c.bid, c.r0, r1);
  c.nr = r1 - c.r0;
  const int n = a.n;
  c.tr_x = a.trace;
  c.tr_attn = a.trace ? c.tr_x + (size_t)a.n_layers * n * S::H : nullptr;
  c.tr_rl = a.trace ? c.tr_attn + (size_t)a.n_layers * n * M::QD : nullptr;
  c.tr_tk = a.trace ? c.tr_rl + (size_t)a.n_layers * n * S::E : nullptr;
  c.tr_fin = a.trace ? c.tr_tk + (size_t)a.n_layers * n * 2 * S::TOPK : nullptr;

  // token ids (device memory; may be the previous step's output)
  if (c.tid < n) {
    int t = a.tokens[c.tid];
    if (t < 0 || t >= a.vocab) {
      set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_TOKEN, t);
      t = 0;
    }
    s_tok[c.tid] = t;
  }
  __syncthreads();

  uint32_t nbar = 0;
  for (int l = 0; l < a.n_layers; ++l) {
    M::qkv(c, l);
    if (!grid_barrier(a, nbar)) goto done;
    M::attention(c, l);
    if (!grid_barrier(a, nbar)) goto done;
    M::oproj(c, l);
    if (!grid_barrier(a, nbar)) goto done;
    M::route(c, l);
    __syncthreads();
    M::gateup(c, l);
    if (!grid_barrier(a, nbar)) goto done;
    if (l >= a.n_dense) M::template down<true>(c, l);
    else M::template down<false>(c, l);
    if (!grid_barrier(a, nbar)) goto done;
  }
  if (a.out_first < n) M::lm_head(c);

done:
  __syncthreads();
  if (c.tid == 0) {
    __threadfence();
    if (atomicAdd(a.sc.sync + 32, 1u) == (uint32_t)(c.G - 1)) {
      // every block has left its work: reset the launch-scoped counters
      a.sc.sync[0] = 0;
      a.sc.sync[64] = 0;
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
