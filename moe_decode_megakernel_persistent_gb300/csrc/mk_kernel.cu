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
//       router logits                                                     | barrier
//   P4  RMSNorm + softmax/top-k (every block), expert gate/up -> SiLU
//       (dense layers: the SwiGLU gate/up)                                | barrier
//   P5  down projection rows, weighted sum over the selected experts, residual
//                                                                          | barrier
// After the last layer: final RMSNorm, lm_head rows, per-block argmax, and
// the last block to arrive reduces the argmax (no barrier needed).
//
// Data movement.  A block is 15 compute warps plus one streaming warp.  Every
// weight row and every cached K/V row a block reads goes through a ring of
// shared-memory stages filled by bulk copies (cp.async.bulk): the streaming
// warp walks the block's whole schedule for the launch (layer by layer, phase
// by phase, in the order the compute warps consume it) and issues each tile
// as soon as a stage is free, so the next phase's weights are already in
// shared memory when a grid barrier releases.  Only expert tiles wait, for
// the layer's routing.  The compute warps wait on a stage's "full" mbarrier,
// form their dot products from shared memory and release the stage.
#include <cfloat>
#include <cstddef>
#include <climits>
#include <type_traits>
#include "mk_device.cuh"

namespace mk {

constexpr int kMaxEnt = kMaxBatch * 8;  // (row, expert slot) entries
constexpr int kMmaUnits = 2;            // tensor-core units per pass (a dense tile has at most 2)

// Per-launch, per-block context shared by the phases (in shared memory).
struct Ctx {
  uint8_t* act;    // activation staging area
  uint8_t* ring;   // weight ring stages
  int ns;          // ring stages
  int act_bytes;   // size of the staging area
  int G, bid, n;
  int r0, nr;      // hidden rows owned by this block
  bool tc;         // tensor-core GEMV (plain fp32 staging) for this launch
  bool flagged;    // one-row launch of a whole step: the residual reaches the next
                   // layer's QKV as flagged words, with no grid barrier
  uint32_t tag0;   // this launch's epoch * 256: the tag of layer l's words is tag0 + l + 1
  float *tr_x, *tr_attn, *tr_rl, *tr_tk, *tr_fin;
  uint64_t* tm;    // this block's timing stamps (thread 0 writes them) or null
  uint64_t* ring_log;  // this block's ring log: [3k] item k issued, [3k + 1] landed (thread 0 saw it),
                       // [3k + 2] released by warp 0 (or null)
};

struct Fixed {
  StepArgs args;   // copy of the launch arguments
  LayerW lw;       // the current layer's weight pointers
  Ctx ctx;
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint32_t kc;            // ring items consumed so far by the compute warps
  uint32_t prod_k;        // ring items issued by the streaming warp (for the exit drain)
  volatile int route_gen; // l + 1 once layer l's routing tables are ready
  volatile int abort;     // compute warps left the step early
  volatile int ok_word;   // grid barrier outcome broadcast
  int tok[kMaxBatch];
  int topk_id[kMaxBatch][8];
  float topk_w[kMaxBatch][8];
  float dots[kMaxEnt][kMaxRowsPerBlock];
  float hs[kMaxBatch][kMaxRowsPerBlock];
  uint32_t nslw[kMaxRowsPerBlock];  // raw slice of the post-attention norm weights
  float red[kThreads];
  unsigned long long best_key[kMaxBatch];  // lm_head argmax per row (argmax_key)
  // tensor-core path: each warp's partial of its unit, read and written as
  // float4 (16-byte aligned whatever precedes it)
  alignas(16) float mma_part[kWarps * 128];
  int unit_start[kMaxBatch + 1];
  int upages[2][64];      // pool pages of this block's attention units (streaming warp)
  float rnorm[kMaxBatch];
  int16_t ue_expert[64], ue_start[64], ue_len[64];
  uint8_t ent_b[kMaxEnt], ent_j[kMaxEnt];
  uint8_t ent_of[kMaxBatch][8];
  uint8_t efirst[kMaxEnt];
  int n_ue, flag;
  int n_merge, merge_job[kMaxOwnUnits][4];  // attention merges this block owes: (b, g, h0, h1)
};
constexpr int kActOffset = (sizeof(Fixed) + 127) / 128 * 128;
static_assert(offsetof(Fixed, mma_part) % 16 == 0, "float4 access to the tensor-core partials");

__device__ __forceinline__ Fixed& fixed() {
  extern __shared__ __align__(128) uint8_t smem_dyn[];
  return *reinterpret_cast<Fixed*>(smem_dyn);
}

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

// Argmax as one 64-bit maximum: the logit's bits mapped to an unsigned order
// (negative values flipped) above the complemented token id, so the larger
// logit wins and, on equal logits, the lower token id.  Key 0 = no candidate.
__device__ __forceinline__ unsigned long long argmax_key(float v, int tok) {
  const uint32_t b = __float_as_uint(v);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)ord << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)tok);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
  const uint32_t ord = (uint32_t)(k >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
__device__ __forceinline__ int key_token(unsigned long long k) { return (int)(0xFFFFFFFFu - (uint32_t)k); }

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
// [1 + 16 l + 15] the layer's routing tables ready (MoE layers);
// [1 + 16 L] lm_head done.
#define MK_STAMP(c, l, p, k) \
  if ((c).tm && threadIdx.x == 0) (c).tm[1 + 16 * (l) + 3 * (p) + (k)] = globaltimer()

// ---------------------------------------------------------------- ring, consumer side
// Every compute thread calls acquire/release for every item, in order.
template <int STAGE>
__device__ __forceinline__ const uint8_t* ring_acquire(uint32_t k) {
  Fixed& F = fixed();
  const int s = (int)(k % (uint32_t)F.ctx.ns);
  const uint32_t par = (k / (uint32_t)F.ctx.ns) & 1u;
  mbar_wait(&F.full[s], par, &F.abort, F.args.sc.err, F.args.spin_limit_ns, (int)k);
  if (F.ctx.ring_log && threadIdx.x == 0 && k < (uint32_t)kRingLog) F.ctx.ring_log[3 * k + 1] = globaltimer();
  return F.ctx.ring + (size_t)s * STAGE;
}
__device__ __forceinline__ void ring_release(uint32_t k) {
  Fixed& F = fixed();
  __syncwarp();
  if (F.ctx.ring_log && threadIdx.x == 0 && k < (uint32_t)kRingLog) F.ctx.ring_log[3 * k + 2] = globaltimer();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&F.empty[k % (uint32_t)F.ctx.ns]);
}

// ---------------------------------------------------------------- ring, producer side
// Lane 0 of the streaming warp.  Item k goes to stage k % NS once the compute
// warps released the stage's previous item (and that item's copies landed);
// each run of contiguous bytes is one bulk copy counted on the stage's full
// mbarrier, and the producer's own arrival closes the item.
struct Producer {
  uint32_t k = 0;
  bool dead = false;
  uint8_t* stage = nullptr;
  uint64_t* bar = nullptr;

  template <int STAGE>
  __device__ __forceinline__ bool begin() {
    Fixed& F = fixed();
    if (dead) return false;
    // the shared abort flag only: a global error-word read here would cost an
    // L2 round trip per item (the waits below poll it while they spin)
    if (F.abort) { dead = true; return false; }
    const uint32_t ns = (uint32_t)F.ctx.ns;
    const int s = (int)(k % ns);
    const uint32_t round = k / ns;
    if (round > 0) {
      if (!mbar_wait(&F.empty[s], (round & 1u) ^ 1u, &F.abort, F.args.sc.err, F.args.spin_limit_ns, (int)k) ||
          !mbar_wait(&F.full[s], (round - 1) & 1u, &F.abort, F.args.sc.err, F.args.spin_limit_ns, (int)k)) {
        dead = true;
        return false;
      }
    }
    stage = F.ctx.ring + (size_t)s * STAGE;
    bar = &F.full[s];
    if (F.ctx.ring_log && k < (uint32_t)kRingLog) F.ctx.ring_log[3 * k] = globaltimer();
    return true;
  }
  __device__ __forceinline__ void copy(uint32_t off, const void* src, uint32_t bytes) {
    mbar_expect_tx(bar, bytes);
    bulk_g2s(stage + off, src, bytes, bar);
  }
  __device__ __forceinline__ void end() {
    mbar_arrive(bar);
    ++k;
  }
  // Before the block exits: the last item of every stage has landed.
  __device__ void drain() {
    Fixed& F = fixed();
    const uint32_t ns = (uint32_t)F.ctx.ns;
    for (uint32_t s = 0; s < ns && s < k; ++s) {
      const uint32_t last = s + ((k - 1 - s) / ns) * ns;
      mbar_wait_drain(&F.full[s], (last / ns) & 1u, 100000000ull);
    }
  }
};


struct ActRange {
  const uint8_t* list;   // staged index of the i-th activation: list ? list[start + i] : start + i
  int start, count;
};

// WDT: the format of the linear layers; XDT: the format of the expert
// matrices (WDT, or int3 experts in an int4 model)
template <class S, int WDT, int XDT = WDT>
struct Model {
  static constexpr int AUX = WDT == WF32 ? WF32 : WBF16;
  static constexpr int H = S::H, NH = S::NH, NKV = S::NKV, HD = S::HD, E = S::E, TOPK = S::TOPK;
  static constexpr int FE = S::FE, FD = S::FD, QD = NH * HD, GQA = NH / NKV, HALF = HD / 2;
  static constexpr int DPL = HD / 32;
  using GH = Gemv<WDT, H>;
  using GQ = Gemv<WDT, QD>;
  using GE = Gemv<WDT, FE>;
  using GD = Gemv<WDT, FD>;
  using GXH = Gemv<XDT, H>;   // expert gate / up rows
  using GXE = Gemv<XDT, FE>;  // expert down rows
  static_assert(XDT == WDT || (WDT == WINT4 && XDT == WINT3), "int3 experts come with int4 layers");
  static_assert(GXH::ACT_BYTES == GH::ACT_BYTES && GXE::ACT_BYTES == GE::ACT_BYTES,
                "expert rows read the layers' staged activations");

  // ring stage: 17 KB for int4 (16 KB of codes + their scales), 32 KB for
  // bf16 and 16 KB for fp32 weights
  static constexpr int STAGE = WDT == WINT4 ? 17408 : (WDT == WBF16 ? 32768 : 16384);
  __host__ __device__ static constexpr int cmax(int a, int b) { return a > b ? a : b; }
  // a packed weight record: one row's codes, then its scales, 16-byte aligned
  template <int K, int FMT = WDT>
  __host__ __device__ static constexpr int rec() {
    return (Gemv<FMT, K>::ROW_BYTES + Gemv<FMT, K>::SCALE_BYTES + 15) / 16 * 16;
  }
  static constexpr int REC_H = rec<H>(), REC_Q = rec<QD>(), REC_E = rec<FE>(), REC_D = rec<FD>();
  static constexpr int REC_XH = rec<H, XDT>(), REC_XE = rec<FE, XDT>();
  // hidden rows go to blocks in groups of 2, so a block's slice of a bf16 row
  // (router, norm) starts and ends on a 4-byte boundary
  static constexpr int A_Q = 1;
  static constexpr int A_H = 2;
  // tasks per tile (RP records each)
  static constexpr int T_QKV = STAGE / (2 * REC_H);
  static constexpr int T_O = STAGE / REC_Q;
  static constexpr int T_GU = STAGE / (2 * REC_H);   // dense gate / up
  static constexpr int T_XGU = STAGE / (2 * REC_XH); // expert gate / up
  static constexpr int T_XDN = STAGE / REC_XE;       // expert down
  static constexpr int T_DD = STAGE / REC_D;
  static constexpr int T_LM = STAGE / REC_H;
  static_assert(T_QKV >= 1 && T_O >= 1 && T_GU >= 1 && T_XGU >= 1 && T_XDN >= 1 && T_DD >= 1 && T_LM >= 1,
                "tile sizes");
  static constexpr int TU = STAGE / (4 * HD) / kWarps;  // positions per warp per stage
  static constexpr int TT = TU * kWarps;              // cached positions per stage (K and V rows, bf16)
  static_assert(TU >= 1, "a stage holds a position per warp");
  // attention: tiles of TT positions, MTS m-tiles of 16
  static constexpr int MTS = (TT + 15) / 16;  // position m-tiles of a tile (score warps) = PV k-steps
  static constexpr int TTP = MTS * 16;        // padded positions of a tile
  static constexpr int NDT = HD / 16;         // dim m-tiles (value warps)
  static constexpr int KST = HD / 16;         // score k-steps
  static constexpr int W_SC = NDT;            // first score warp
  static constexpr int W_SM = kWarps - GQA;   // first softmax warp
  static_assert(GQA <= 8 && HD % 16 == 0, "one n-tile of heads, whole k-steps");
  static_assert(NDT + MTS <= kWarps && GQA <= kWarps, "warp roles");
  // attention scratch in the staging area (byte offsets)
  static constexpr int AO_QS = 0;                                 // float [GQA][HD] scaled queries
  static constexpr int AO_QF = AO_QS + GQA * HD * 4;              // uint4 [KST][32] q fragments (hi b0 b1, lo b0 b1)
  static constexpr int AO_SC = AO_QF + KST * 32 * 16;             // float [TTP][8] scores
  static constexpr int AO_PB = AO_SC + TTP * 8 * 4;               // bf16 [2][8][TTP] P hi, lo
  static constexpr int AO_ML = AO_PB + 2 * 8 * TTP * 2;           // float [3][8] m, l, corr
  static constexpr int AO_NT = (AO_ML + 3 * 8 * 4 + 127) / 128 * 128;  // bf16 [2][TT][HD] new-position tile
  // (the value warps read V rows up to TTP - 1: the padding rows stay inside)
  static constexpr int ATT_SMEM = AO_NT + (TT + TTP) * HD * 2;
  static constexpr int SPL = (TTP + 31) / 32;  // positions per softmax lane
  static_assert(STAGE >= (TT + TTP) * HD * 2, "padding rows of a ring tile stay inside the stage");
  static_assert(H % A_H == 0, "aligned row groups");
  static_assert(TOPK <= 8 && E <= 64, "router tables");

  static constexpr int NQP = NH * HALF, NKP = NKV * HALF, NP = NQP + 2 * NKP;
  static constexpr int PR = HD + 4;  // partial row: m, l, pad, pad, o[HD] (16-byte rows)

  // Staging area for n rows: every phase's activations fit; the MoE down
  // entries take what is left above 3 ring stages (rounds if they do not fit).
  static constexpr bool TC = WDT != WF32;  // the tensor-core path serves launches of 2+ rows
  // (the tensor-core path stages plain fp32 rows for the dense projections;
  // the expert phases keep the GEMV engine's staged form)
  __host__ __device__ static constexpr int act_base_bytes(int n, bool tc) {
    return cmax(tc ? cmax(cmax(n * plain_stride(H), n * plain_stride(QD)), plain_stride(FD)) : 0,
                cmax(cmax(n * GH::ACT_BYTES, n * GQ::ACT_BYTES),
                     cmax(cmax(ATT_SMEM, GD::ACT_BYTES), n * GE::ACT_BYTES)));
  }
  static_assert(kActOffset + act_base_bytes(kMaxBatch, TC) + 2 * STAGE <= kSmemBytes,
                "a full batch leaves at least two ring stages");
  // dynamic shared memory of a one-row launch: the staging area and three
  // ring stages, at least kSmemSingleRow (the most that the 132 KB
  // L1/shared carve-out holds), at most the full size
  static constexpr int SMEM1 =
      cmax(kSmemSingleRow,
           (kActOffset + (cmax(act_base_bytes(1, false), TOPK * GE::ACT_BYTES) + 127) / 128 * 128 + 3 * STAGE + 1023) /
               1024 * 1024);
  static constexpr int SMEM_SINGLE = SMEM1 < kSmemBytes ? SMEM1 : kSmemBytes;

  __device__ static __forceinline__ void unit_of(const StepArgs& a, const int* unit_start, int u, int n,
                                                 int& b, int& g, int& ci, int& nch) {
    b = 0;
    while (b + 1 < n && unit_start[b + 1] <= u) ++b;
    nch = (a.pos[b] + 1 + a.chunk - 1) / a.chunk;
    const int rem = u - unit_start[b];
    g = rem / nch;
    ci = rem % nch;
  }

  // ---- the block's task ranges (identical for the streaming warp and the
  // compute warps)
  __device__ static __forceinline__ void qkv_range(const Ctx& c, int& p0, int& p1) {
    split_range(NP / A_Q, c.G, c.bid, p0, p1);
    p0 *= A_Q;
    p1 *= A_Q;
  }
  __device__ static __forceinline__ void gu_range(const Ctx& c, int total, int& u0, int& u1) {
    split_range(total / A_Q, c.G, c.bid, u0, u1);
    u0 *= A_Q;
    u1 *= A_Q;
  }
  // rounds of the MoE down projection: distinct experts [ua, ub) whose
  // entries fit the staging area together
  // staged bytes per MoE down entry / per dense down row in this launch
  __device__ static __forceinline__ int moe_entry_bytes(const Ctx&) { return GE::ACT_BYTES; }
  __device__ static __forceinline__ int dense_entry_bytes(const Ctx& c) {
    return c.tc ? plain_stride(FD) : GD::ACT_BYTES;
  }
  __device__ static __forceinline__ int moe_round_end(const Fixed& F, int ua, int cap) {
    int ub = ua, cnt = 0;
    while (ub < F.n_ue && cnt + F.ue_len[ub] <= cap) cnt += F.ue_len[ub++];
    return ub > ua ? ub : ua + 1;
  }
  // ring positions of unit u: cached positions [t0, rt1) come through the
  // ring, the ones this launch writes, [rt1, t1), are read from global memory
  __device__ static __forceinline__ void unit_span(const StepArgs& a, int b, int ci, int& t0, int& rt1,
                                                   int& t1) {
    t0 = ci * a.chunk;
    t1 = min(a.pos[b] + 1, t0 + a.chunk);
    rt1 = min(t1, max(t0, a.new0[b]));
  }

  static __device__ __forceinline__ bool same_acts(const ActRange& x, const ActRange& y) {
    return x.list == y.list && x.start == y.start && x.count == y.count;
  }

  // ---- generic GEMV over ring tiles.  Tasks [0, ntask) of the phase, T per
  // ring item; task t runs on warp t % kWarps, or (CONTIG) each warp takes a
  // contiguous block of a tile's tasks (tasks sharing an activation stay on
  // one warp, whose activation registers then reload rarely).  TK provides
  //   ActRange acts(t) and void put(t, ai, i, v0, v1) (one lane writes the
  //   results of task t for activation ai, the i-th of the task's list).
  template <int K, int RP, int T, bool REGS, bool CONTIG, bool MMA, int FMT = WDT, class TK>
  __device__ static __forceinline__ void run_gemv(int ntask, const uint8_t* act_base, const TK& task) {
    if constexpr (TC && MMA) {
      if (fixed().ctx.tc) {
        run_mma<K, RP, T>(ntask, act_base, task);
        return;
      }
    }
    using Gv = Gemv<FMT, K>;
    Fixed& F = fixed();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t k = F.kc;
    typename Gv::Act a;
    int loaded = -1;
#pragma unroll 1
    for (int t0 = 0; t0 < ntask; t0 += T, ++k) {
      const uint8_t* st = ring_acquire<STAGE>(k);
      const int tn = min(T, ntask - t0);
      const int per = (tn + kWarps - 1) / kWarps;
      const int j_first = CONTIG ? wid * per : ((wid - t0) % kWarps + kWarps) % kWarps;
      const int j_end = CONTIG ? min(tn, j_first + per) : tn;
#pragma unroll 1
      for (int j = j_first; j < j_end;) {
        const int t = t0 + j;
        constexpr int RC = rec<K, FMT>();
        const ActRange ar = task.acts(t);
        // one-row tasks of a contiguous block: two consecutive rows that share
        // an activation list are dotted together (two independent chains)
        bool pair = false;
        if constexpr (RP == 1 && CONTIG) pair = j + 1 < j_end && same_acts(task.acts(t + 1), ar);
        const uint8_t* wr[2];
        const uint8_t* sr[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int rowi = RP == 2 ? j * 2 + r : j + (pair ? r : 0);
          wr[r] = st + (size_t)rowi * RC;
          sr[r] = wr[r] + Gv::ROW_BYTES;
        }
#pragma unroll 1
        for (int i = 0; i < ar.count; ++i) {
          const int ai = ar.list ? ar.list[ar.start + i] : ar.start + i;
          const uint8_t* ab = act_base + ai * Gv::ACT_BYTES;
          if constexpr (REGS) {
            if (ai != loaded) { Gv::load_act(a, ab, lane); loaded = ai; }
          }
          float v0, v1;
          if (RP == 2 || pair) {
            Gv::template dots<2, REGS>(wr, sr, a, ab, lane, v0, v1);
            if (lane == 0) {
              if (RP == 2) task.put(t, ai, i, v0, v1);
              else { task.put(t, ai, i, v0, 0.f); task.put(t + 1, ai, i, v1, 0.f); }
            }
          } else {
            Gv::template dots<1, REGS>(wr, sr, a, ab, lane, v0, v1);
            if (lane == 0) task.put(t, ai, i, v0, v1);
          }
        }
        j += CONTIG ? (pair ? 2 : 1) : kWarps;
      }
      ring_release(k);
    }
    csync();
    if (threadIdx.x == 0) F.kc = k;
    csync();
  }

  // This block's slice of the layer's router weights (E rows x nr columns)
  // and of its post-attention norm, copied into shared memory with
  // asynchronous 4-byte copies (F.dots holds the router slice: it is free
  // from P1 to P3).  The slices are 4-byte aligned: r0 and nr are multiples
  // of A_H >= 2.
  __device__ static __forceinline__ void fetch_router_slice(const LayerW& Lw) {
    Fixed& F = fixed();
    const Ctx& c = F.ctx;
    constexpr int VPW = AUX == WF32 ? 1 : 2;  // values per 4-byte word
    const int words = c.nr / VPW;
    uint32_t* rs = reinterpret_cast<uint32_t*>(&F.dots[0][0]);
    const uint8_t* rb = reinterpret_cast<const uint8_t*>(Lw.router);
    constexpr int VB = AUX == WF32 ? 4 : 2;
    for (int idx = threadIdx.x; idx < (E + 1) * words; idx += kThreads) {
      const int e = idx / words, w = idx % words;
      const uint8_t* src = e < E ? rb + ((size_t)e * H + c.r0) * VB + 4 * w
                                 : reinterpret_cast<const uint8_t*>(Lw.ffn_norm) + (size_t)c.r0 * VB + 4 * w;
      uint32_t* dst = e < E ? rs + e * kMaxRowsPerBlock + w : F.nslw + w;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  // value t of a raw slice row (bf16 pairs or fp32 words)
  __device__ static __forceinline__ float slice_val(const uint32_t* row, int t) {
    if constexpr (AUX == WF32) return __uint_as_float(row[t]);
    else return bf16_to_f((row[t >> 1] >> (16 * (t & 1))) & 0xFFFFu);
  }

  // ---- tensor-core GEMV (launches of 2+ rows).  A ring tile is cut into
  // m-tiles of 16 weight rows (RP == 2: 8 tasks, rows g and g + 8 are the two
  // rows of task g; RP == 1: 16 tasks) and, per run of tasks sharing one
  // activation list, n-tiles of 8 activations.  mma.sync m16n8k16, bf16 in,
  // fp32 accumulate: int4 codes are widened to bf16 exactly in registers; each
  // activation (plain fp32 staging) is split into three bf16 parts
  // hi + mid + lo (24 significant bits), all multiplied into one accumulator.
  // K is split over the warps in 64-value groups (the int4 scale group: a
  // group's sum is scaled before it is added); the warps' partials meet in
  // shared memory.  Within a group, thread q of a quad takes the values
  // 16q .. 16q+15 of weights and activations alike (the order of k inside an
  // mma is free as long as A and B agree on it).
  __device__ static __forceinline__ uint32_t nib_pair_bf16(uint32_t E, uint32_t O, int i) {
    // byte i of E / O (codes q + 8) -> bf16x2 {q_lo, q_hi}: (128 + c) - 136
    uint32_t r;
    const uint32_t sel = (uint32_t)i | ((uint32_t)i << 4) | ((uint32_t)(4 + i) << 8) | ((uint32_t)(4 + i) << 12);
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(E), "r"(O), "r"(sel));
    r = (r & 0x00FF00FFu) | 0x43004300u;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(r), "r"(0x3F803F80u), "r"(0xC308C308u));
    return r;
  }
  __device__ static __forceinline__ void split3(float x0, float x1, uint32_t& h, uint32_t& m, uint32_t& l) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(x1), "f"(x0));
    const float r0 = x0 - __uint_as_float(h << 16), r1 = x1 - __uint_as_float(h & 0xFFFF0000u);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(m) : "f"(r1), "f"(r0));
    const float s0 = r0 - __uint_as_float(m << 16), s1 = r1 - __uint_as_float(m & 0xFFFF0000u);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(s1), "f"(s0));
  }
  __device__ static __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                  uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }

  // Walk the units of one ring tile in order: (m-tile, run of tasks sharing
  // one activation list, n-tile of 8 activations); f(u, ta, tb, sa, sb, ar, c0).
  template <int RP, class TK, class F_>
  __device__ static __forceinline__ int for_units(int t0, int tn, const TK& task, F_ f) {
    constexpr int MT = RP == 2 ? 8 : 16;
    int u = 0;
#pragma unroll 1
    for (int ta = 0; ta < tn; ta += MT) {
      const int tb = min(tn, ta + MT);
#pragma unroll 1
      for (int sa = ta; sa < tb;) {
        const ActRange ar = task.acts(t0 + sa);
        int sb = sa + 1;
        while (sb < tb && same_acts(task.acts(t0 + sb), ar)) ++sb;
#pragma unroll 1
        for (int c0 = 0; c0 < ar.count; c0 += 8, ++u) f(u, ta, tb, sa, sb, ar, c0);
        sa = sb;
      }
    }
    return u;
  }

  template <int K, int RP, int T, class TK>
  __device__ static __noinline__ void run_mma(int ntask, const uint8_t* act_base, const TK& task) {
    using Gv = Gemv<WDT, K>;
    constexpr int NGR = K / 64;
    constexpr int RB = Gv::ROW_BYTES, AS = plain_stride(K);
    static_assert(K % 64 == 0, "whole 64-value groups");
    Fixed& F = fixed();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, g = lane >> 2, q = lane & 3;
    uint32_t k = F.kc;
#pragma unroll 1
    for (int t0 = 0; t0 < ntask; t0 += T, ++k) {
      const uint8_t* st = ring_acquire<STAGE>(k);
      const int tn = min(T, ntask - t0);
      const int n_units = for_units<RP>(t0, tn, task, [](int, int, int, int, int, const ActRange&, int) {});
#pragma unroll 1
      for (int base = 0; base < n_units; base += kMmaUnits) {
        // units [base, base + U) are computed in this pass: warp w works on
        // unit base + w % U, over the 64-value groups w / U, w / U + nw, ...
        // (nw = warps on that unit), and writes its partial to its own slot;
        // the slots of a unit are then summed in warp order, so the result
        // does not depend on timing
        const int U = min(kMmaUnits, n_units - base);
        const int my_u = base + wid % U, kw = wid / U, nw = (kWarps - wid % U + U - 1) / U;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for_units<RP>(t0, tn, task, [&](int u, int ta, int tb, int, int, const ActRange& ar, int c0) {
          if (u != my_u) return;
          // rows of this lane: task rows rho0 = g, rho1 = g + 8 of the m-tile
          int j0, j1, seg1;
          if (RP == 2) { j0 = ta + g; j1 = j0; seg1 = 1; }
          else { j0 = ta + g; j1 = ta + 8 + g; seg1 = 0; }
          j0 = j0 < tb ? j0 : ta;
          j1 = j1 < tb ? j1 : ta;
          constexpr int RC = rec<K>();
          const uint8_t* w0 = st + (size_t)(j0 * RP) * RC;
          const uint8_t* w1 = st + (size_t)(j1 * RP + seg1) * RC;
          const uint8_t* s0p = w0 + RB;
          const uint8_t* s1p = w1 + RB;
          // this lane's activation column
          const int col = c0 + g;
          const bool cv = col < ar.count;
          const int ai = cv ? (ar.list ? ar.list[ar.start + col] : ar.start + col) : 0;
          const uint8_t* xa = act_base + (size_t)ai * AS;
#pragma unroll 1
          for (int G = kw; G < NGR; G += nw) {
            float xv[16];
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const uint4 r = cv ? lds128(xa + (64 * G + 16 * q + 4 * v4) * 4) : make_uint4(0u, 0u, 0u, 0u);
              xv[4 * v4] = __uint_as_float(r.x); xv[4 * v4 + 1] = __uint_as_float(r.y);
              xv[4 * v4 + 2] = __uint_as_float(r.z); xv[4 * v4 + 3] = __uint_as_float(r.w);
            }
            uint32_t aw[2][8];  // per row: bf16x2 words for steps 0..3 (2 per step)
            if constexpr (WDT == WINT4) {
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const uint2 wv = lds64((r ? w1 : w0) + 32 * G + 8 * q);
                const uint32_t x2[2] = {wv.x, wv.y};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint32_t y = x2[h] ^ 0x88888888u;
                  const uint32_t E = y & 0x0F0F0F0Fu, O = (y >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                  for (int bi = 0; bi < 4; ++bi) aw[r][4 * h + bi] = nib_pair_bf16(E, O, bi);
                }
              }
            } else {
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const uint4 lo = lds128((r ? w1 : w0) + 128 * G + 32 * q);
                const uint4 hi = lds128((r ? w1 : w0) + 128 * G + 32 * q + 16);
                aw[r][0] = lo.x; aw[r][1] = lo.y; aw[r][2] = lo.z; aw[r][3] = lo.w;
                aw[r][4] = hi.x; aw[r][5] = hi.y; aw[r][6] = hi.z; aw[r][7] = hi.w;
              }
            }
            float cg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int sstep = 0; sstep < 4; ++sstep) {
              uint32_t bh0, bm0, bl0, bh1, bm1, bl1;
              split3(xv[4 * sstep], xv[4 * sstep + 1], bh0, bm0, bl0);
              split3(xv[4 * sstep + 2], xv[4 * sstep + 3], bh1, bm1, bl1);
              const uint32_t a0 = aw[0][2 * sstep], a2 = aw[0][2 * sstep + 1];
              const uint32_t a1 = aw[1][2 * sstep], a3 = aw[1][2 * sstep + 1];
              mma16816(cg, a0, a1, a2, a3, bh0, bh1);
              mma16816(cg, a0, a1, a2, a3, bm0, bm1);
              mma16816(cg, a0, a1, a2, a3, bl0, bl1);
            }
            if constexpr (WDT == WINT4) {
              const float sc0 = bf16_to_f(lds16(s0p + 2 * G)), sc1 = bf16_to_f(lds16(s1p + 2 * G));
              acc[0] = fmaf(cg[0], sc0, acc[0]);
              acc[1] = fmaf(cg[1], sc0, acc[1]);
              acc[2] = fmaf(cg[2], sc1, acc[2]);
              acc[3] = fmaf(cg[3], sc1, acc[3]);
            } else {
#pragma unroll
              for (int r = 0; r < 4; ++r) acc[r] += cg[r];
            }
          }
        });
        *reinterpret_cast<float4*>(&F.mma_part[(wid * 32 + lane) * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        csync();
        // results: warp j < U writes unit base + j (lane: rows g / g + 8,
        // columns 2q, 2q + 1), summing the slots of warps j, j + U, ... in order
        if (wid < U) {
          const int my_out = base + wid;
          for_units<RP>(t0, tn, task, [&](int u, int ta, int tb, int sa, int sb, const ActRange& ar, int c0) {
            if (u != my_out) return;
            float r4[4] = {0.f, 0.f, 0.f, 0.f};
            for (int w = wid; w < kWarps; w += U) {
              const float4 v = *reinterpret_cast<const float4*>(&F.mma_part[(w * 32 + lane) * 4]);
              r4[0] += v.x; r4[1] += v.y; r4[2] += v.z; r4[3] += v.w;
            }
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int col = c0 + 2 * q + cc;
              if (col >= ar.count) continue;
              const int ai = ar.list ? ar.list[ar.start + col] : ar.start + col;
              if (RP == 2) {
                const int j = ta + g;
                if (j >= sa && j < sb) task.put(t0 + j, ai, col, r4[cc], r4[2 + cc]);
              } else {
                const int ja = ta + g, jb = ta + 8 + g;
                if (ja >= sa && ja < sb) task.put(t0 + ja, ai, col, r4[cc], 0.f);
                if (jb >= sa && jb < sb) task.put(t0 + jb, ai, col, r4[2 + cc], 0.f);
              }
            }
          });
        }
        csync();  // the slots are free for the next pass
      }
      ring_release(k);
    }
    csync();
    if (threadIdx.x == 0) F.kc = k;
    csync();
  }

  // ---------------------------------------------------------------- P1
  // RMSNorm of the residual (every block, redundantly) -> this block's QKV
  // tasks.  A task is a RoPE pair of rows (i, i + HD/2) of one q, k or v head,
  // so the warp that forms a pair also rotates it and writes it: q to
  // scratch, k and v as bf16 into the page.
  // Staging runs in functions of its own, called from the layer loop where
  // few values are live: a call from inside a phase would save and restore
  // the phase's registers through local memory, which the small L1 left
  // beside 227 KB of shared memory mostly misses.
  template <int MODE>
  __device__ static __noinline__ void qkv_stage(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x;
    const LayerW& Lw = F.lw;
    const int n = c.n;
    if (l == 0 && c.bid == 0)
      for (int i = tid; i < a.n_upd; i += kThreads)
        a.block_table[a.upd[i].slot * a.max_pages_per_seq + a.upd[i].index] = a.upd[i].page;
    if (c.bid == 0 && l >= a.n_dense)  // router logits are accumulated in P3
      for (int i = tid; i < kRlogitGroups * n * E; i += kThreads)
        a.sc.rlogit[(i / (n * E)) * kMaxBatch * E + i % (n * E)] = 0ll;
    if (l >= a.n_dense) fetch_router_slice(Lw);
    {
      const void* nw = Lw.attn_norm;
      const void* embed = a.embed;
      const float* x = a.sc.x;
      const int* tok = F.tok;
      const bool first = l == 0;
      // the previous layer's residual: flagged words (one-row step), else
      // plain rows behind the grid barrier
      const uint64_t* xw = c.flagged && !first ? a.sc.xll + (size_t)((l - 1) & 1) * kMaxBatch * H : nullptr;
      const uint32_t tag = c.tag0 + l;
      if (MODE == 2 && !first)  // plain rows of x: one round of asynchronous copies
        stage_plain_async<AUX, H, true>(c.act, n, x, H, a.eps, nw, F.red, nullptr);
      else
        stage_block<MODE, WDT, H, true>(
            c.act, n,
            [&](int r, int f4) -> float4 {
              return first ? ld_aux4<AUX>(embed, (size_t)tok[r] * (H / 4) + f4)
                     : xw  ? flag_get4(xw + (size_t)r * H + 4 * f4, tag, a)
                           : __ldcg(reinterpret_cast<const float4*>(x + r * H) + f4);
            },
            a.eps, [&](int f4) { return ld_aux4<AUX>(nw, f4); }, F.red, nullptr);
    }
    if (l == 0)  // residual rows this block reads back in P3
      for (int i = tid; i < n * c.nr; i += kThreads) {
        const int b = i / c.nr, r = c.r0 + i % c.nr;
        a.sc.x[b * H + r] = ld_aux<AUX>(a.embed, (size_t)F.tok[b] * H + r);
      }
    csync();
    MK_STAMP(c, l, 0, 0);
  }
  __device__ static __noinline__ void qkv(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int lane = threadIdx.x & 31;
    int p0, p1;
    qkv_range(c, p0, p1);
    struct {
      const StepArgs* a; int p0, l, lane;
      __device__ __forceinline__ ActRange acts(int) const { return {nullptr, 0, a->n}; }
      __device__ __forceinline__ void put(int t, int b, int, float v0, float v1) const {
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
          const int g = q / HALF, i = q % HALF;
          uint16_t* dst = a->kv + Kv<S>::offset(l, a->n_pages, a->cur_page[b], 1, g, pos % kPageTokens);
          dst[i] = f_to_bf16(v0);
          dst[i + HALF] = f_to_bf16(v1);
        }
      }
    } task{&a, p0, l, lane};
    run_gemv<H, 2, T_QKV, false, false, true>(p1 - p0, c.act, task);
  }

  // ---------------------------------------------------------------- P2
  // Split attention over the paged cache.  Unit = (row, kv head, chunk of
  // positions).  Cached positions arrive through the ring, TT per stage (K
  // rows, then V rows, bf16); positions this launch wrote are copied from
  // global memory into a tile of the same layout.  The whole block works on
  // one tile at a time with mma.sync m16n8k16 (bf16 in, fp32 accumulate):
  //   scores  S^T = K q^T     (m = 16 positions, n = the GQA heads, k = 16
  //           dims), by the score warps, one m-tile each; q is split into
  //           bf16 hi + lo (16 significant bits; K is bf16 exactly);
  //   softmax one warp per head: running max m, sum l, correction factor
  //           exp(m_old - m_new) and P = exp(S - m_new), split hi + lo;
  //   values  O^T = O^T corr + V^T P^T (m = 16 dims, n = heads, k = 16
  //           positions), by the value warps, one m-tile of dims each, the
  //           accumulators kept in registers across the unit's tiles.
  // Padding positions of a tile get P = 0 and their V operand is zeroed.
  // The unit's partial (m, l, o) is written straight from those registers;
  // the last units of a (row, kv head) merge all its chunks in chunk order
  // (log-sum-exp).

  __device__ static __forceinline__ void split2(float x0, float x1, uint32_t& h, uint32_t& l) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(x1), "f"(x0));
    const float r0 = x0 - __uint_as_float(h << 16), r1 = x1 - __uint_as_float(h & 0xFFFF0000u);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(r1), "f"(r0));
  }
  __device__ static __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                 uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
  }
  __device__ static __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                   uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
  }

  // One tile of nt positions (K rows at kv, V rows at kv + TT * HD * 2,
  // 32-bit shared addresses): scores, softmax, values.  `o` is the value
  // warps' accumulator (rows g, g + 8 = dims, columns 2q, 2q + 1 = heads).
  __device__ static __noinline__ float4 att_tile(uint32_t kv, int nt, uint8_t* att, float4 ov) {
    float o[4] = {ov.x, ov.y, ov.z, ov.w};
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, g = lane >> 2, q = lane & 3;
    float* sc = reinterpret_cast<float*>(att + AO_SC);
    uint16_t* pb = reinterpret_cast<uint16_t*>(att + AO_PB);
    float* ml = reinterpret_cast<float*>(att + AO_ML);
    if (wid >= W_SC && wid < W_SC + MTS) {
      // S^T rows 16 mt .. 16 mt + 15 (positions), all heads
      const int mt = wid - W_SC;
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      const uint4* qf = reinterpret_cast<const uint4*>(att + AO_QF);
      // ldmatrix rows: lanes 0-7 / 8-15 positions 0-7 / 8-15 at dims +0,
      // lanes 16-31 the same positions at dims +8
      const uint32_t ra = kv + (uint32_t)(16 * mt + (lane & 15)) * HD * 2 + (uint32_t)(lane >> 4) * 16;
#pragma unroll
      for (int ks = 0; ks < KST; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ra + ks * 32, a0, a1, a2, a3);
        const uint4 b = qf[ks * 32 + lane];
        mma16816(s, a0, a1, a2, a3, b.x, b.y);
        mma16816(s, a0, a1, a2, a3, b.z, b.w);
      }
      const int p0 = 16 * mt + g;
      sc[p0 * 8 + 2 * q] = s[0];
      sc[p0 * 8 + 2 * q + 1] = s[1];
      sc[(p0 + 8) * 8 + 2 * q] = s[2];
      sc[(p0 + 8) * 8 + 2 * q + 1] = s[3];
    }
    csync();
    if (wid >= W_SM) {
      // head i: positions lane + 32 j
      const int i = wid - W_SM;
      float v[SPL];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < SPL; ++j) {
        const int p = lane + 32 * j;
        v[j] = p < nt ? sc[p * 8 + i] : -INFINITY;
        mx = fmaxf(mx, v[j]);
      }
      const float mold = ml[i];
      const float mn = fmaxf(mold, warp_max(mx));
      const float corr = mold == -INFINITY ? 0.f : __expf(mold - mn);
      float ps = 0.f;
#pragma unroll
      for (int j = 0; j < SPL; ++j) {
        const int p = lane + 32 * j;
        const float e = p < nt ? __expf(v[j] - mn) : 0.f;
        ps += e;
        // P = hi + lo, two bf16
        const __nv_bfloat16 h = __float2bfloat16_rn(e);
        const __nv_bfloat16 lo = __float2bfloat16_rn(e - __bfloat162float(h));
        if (p < TTP) {
          pb[i * TTP + p] = __bfloat16_as_ushort(h);
          pb[8 * TTP + i * TTP + p] = __bfloat16_as_ushort(lo);
        }
      }
      ps = warp_sum(ps);
      if (lane == 0) {
        ml[i] = mn;
        ml[8 + i] = ml[8 + i] * corr + ps;
        ml[16 + i] = corr;
      }
    }
    csync();
    if (wid < NDT) {
      const float c0 = ml[16 + 2 * q], c1 = ml[16 + 2 * q + 1];  // heads >= GQA: 0 (never used)
      o[0] *= c0; o[1] *= c1; o[2] *= c0; o[3] *= c1;
      // V^T via transposed ldmatrix: matrices (dims +0, positions +0),
      // (dims +8, +0), (dims +0, +8), (dims +8, +8)
      const int mi = lane >> 3;
      const uint32_t ra = kv + (uint32_t)TT * HD * 2 +
                          (uint32_t)((mi >> 1) * 8 + (lane & 7)) * HD * 2 + (uint32_t)(16 * wid + (mi & 1) * 8) * 2;
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(pb);
#pragma unroll
      for (int kt = 0; kt < MTS; ++kt) {
        uint32_t a0, a1, a2, a3;
        // rows past the tile's TT positions are never read: clamp the
        // address (their P is 0 and the operand is zeroed below)
        ldsm_x4_t(ra + (uint32_t)kt * 16 * HD * 2, a0, a1, a2, a3);
        const int pa = 16 * kt + 2 * q, pbp = pa + 8;
        if (pa >= nt) { a0 = 0u; a1 = 0u; } else if (pa + 1 >= nt) { a0 &= 0xFFFFu; a1 &= 0xFFFFu; }
        if (pbp >= nt) { a2 = 0u; a3 = 0u; } else if (pbp + 1 >= nt) { a2 &= 0xFFFFu; a3 &= 0xFFFFu; }
        const uint32_t bh0 = pw[(g * TTP + pa) >> 1], bh1 = pw[(g * TTP + pbp) >> 1];
        const uint32_t bl0 = pw[(8 * TTP + g * TTP + pa) >> 1], bl1 = pw[(8 * TTP + g * TTP + pbp) >> 1];
        mma16816(o, a0, a1, a2, a3, bh0, bh1);
        mma16816(o, a0, a1, a2, a3, bl0, bl1);
      }
    }
    return make_float4(o[0], o[1], o[2], o[3]);
  }

  __device__ static __noinline__ void attention(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n = c.n;
    uint8_t* att = c.act;
    float* qs = reinterpret_cast<float*>(att + AO_QS);
    float* ml = reinterpret_cast<float*>(att + AO_ML);
    uint16_t* pb = reinterpret_cast<uint16_t*>(att + AO_PB);
    const uint32_t nt_base = smem_u32(att + AO_NT);
    const float qscale = rsqrtf((float)HD);
    uint32_t k = F.kc;
#pragma unroll 1
    for (int u = c.bid; u < a.n_units; u += c.G) {
      int b, g, ci, nch;
      unit_of(a, F.unit_start, u, n, b, g, ci, nch);
      int t0, rt1, t1;
      unit_span(a, b, ci, t0, rt1, t1);
      // this unit's queries (scaled), the softmax state, P of the padding
      // heads (never written by the softmax warps) zero
      for (int v = tid; v < GQA * HD / 4; v += kThreads) {
        float4 x = __ldcg(reinterpret_cast<const float4*>(a.sc.q + b * QD + g * GQA * HD) + v);
        x.x *= qscale; x.y *= qscale; x.z *= qscale; x.w *= qscale;
        reinterpret_cast<float4*>(qs)[v] = x;
      }
      if (tid < 8) {
        ml[tid] = -INFINITY;
        ml[8 + tid] = 0.f;
        ml[16 + tid] = 0.f;
      }
      for (int v = tid; v < 2 * (8 - GQA) * TTP; v += kThreads) {
        const int hl = v / ((8 - GQA) * TTP), r = v % ((8 - GQA) * TTP);
        pb[hl * 8 * TTP + GQA * TTP + r] = 0;
      }
      csync();
      // B fragments of q^T for the score warps: thread (g, q) of k-step ks
      // holds head g, dims 16 ks + 2q, +1 (b0) and + 8 (b1), hi then lo
      for (int v = tid; v < KST * 32; v += kThreads) {
        const int ks = v >> 5, ln = v & 31, hg = ln >> 2, qq = ln & 3;
        uint4 f = make_uint4(0u, 0u, 0u, 0u);
        if (hg < GQA) {
          const float* qr = qs + hg * HD + 16 * ks + 2 * qq;
          split2(qr[0], qr[1], f.x, f.z);
          split2(qr[8], qr[9], f.y, f.w);
        }
        reinterpret_cast<uint4*>(att + AO_QF)[v] = f;
      }
      csync();
      // positions this launch wrote (at L2, written before the grid barrier)
      // are copied into the new-position tile with cp.async; the first such
      // tile is requested now and lands while the ring tiles are processed
      auto stage_new = [&](int tb, int nt) {
        constexpr int RW = HD * 2 / 16;  // 16-byte words per row
        for (int v = tid; v < 2 * nt * RW; v += kThreads) {
          const int kvh = v / (nt * RW), r = (v / RW) % nt, w = v % RW;
          const int t = tb + r, pi = t / kPageTokens;
          int page = pi == a.pos[b] / kPageTokens
                         ? a.cur_page[b]
                         : (pi < a.max_pages_per_seq ? __ldcg(a.block_table + a.slot[b] * a.max_pages_per_seq + pi)
                                                     : -1);
          if (page < 0 || page >= a.n_pages) {
            set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_PAGE, pi);
            page = 0;
          }
          const uint4* src =
              reinterpret_cast<const uint4*>(a.kv + Kv<S>::offset(l, a.n_pages, page, kvh, g, t % kPageTokens)) + w;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(nt_base + (uint32_t)((kvh * TT + r) * RW + w) * 16),
                       "l"(src)
                       : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      };
      if (rt1 < t1) stage_new(rt1, min(TT, t1 - rt1));
      float4 ov = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
      for (int tb = t0; tb < rt1; tb += TT, ++k) {
        const uint32_t st = smem_u32(ring_acquire<STAGE>(k));
        ov = att_tile(st, min(TT, rt1 - tb), att, ov);
        ring_release(k);
      }
#pragma unroll 1
      for (int tb = rt1; tb < t1; tb += TT) {
        const int nt = min(TT, t1 - tb);
        if (tb != rt1) {
          csync();  // the previous tile's readers are done with the new-position tile
          stage_new(tb, nt);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        csync();
        ov = att_tile(nt_base, nt, att, ov);
      }
      const float o[4] = {ov.x, ov.y, ov.z, ov.w};
      csync();
      if (u >= a.max_units) set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_UNIT, u);
      float* pu = a.sc.part + (size_t)min(u, a.max_units - 1) * GQA * PR;
      if (wid < NDT) {
        const int gg = lane >> 2, qq = lane & 3, d0 = 16 * wid + gg;
        if (2 * qq < GQA) {
          pu[(2 * qq) * PR + 4 + d0] = o[0];
          pu[(2 * qq) * PR + 4 + d0 + 8] = o[2];
        }
        if (2 * qq + 1 < GQA) {
          pu[(2 * qq + 1) * PR + 4 + d0] = o[1];
          pu[(2 * qq + 1) * PR + 4 + d0 + 8] = o[3];
        }
      }
      if (tid < GQA) {
        pu[tid * PR] = ml[tid];
        pu[tid * PR + 1] = ml[8 + tid];
      }
      csync();
      // release this unit's partial; the last MG units of (b, g) to arrive
      // (MG = min(GQA, nch)) each merge a share of the GQA heads once every
      // unit of the layer has arrived (the counter grows by nch per layer
      // and is cleared when the launch ends)
      // (a merge waits for other blocks' units, so it runs only after this
      // block has finished all of its own units: no two blocks wait on each
      // other)
      const int MG = min(GQA, nch);
      if (tid == 0) {
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(old) : "l"(a.sc.merge_cnt + b * NKV + g) : "memory");
        const int arr = old - (l - F.args.slice_lo / 4) * nch;
        if (arr >= nch - MG) {
          const int r = arr - (nch - MG);
          if (F.n_merge >= kMaxOwnUnits) {  // the host bounds units per block
            set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_UNIT, u);
            F.n_merge = kMaxOwnUnits - 1;
          }
          F.merge_job[F.n_merge][0] = b;
          F.merge_job[F.n_merge][1] = g;
          F.merge_job[F.n_merge][2] = r * GQA / MG;
          F.merge_job[F.n_merge][3] = (r + 1) * GQA / MG;
          ++F.n_merge;
        }
      }
      csync();
    }
#pragma unroll 1
    for (int jm = 0; jm < F.n_merge; ++jm) {
      const int b = F.merge_job[jm][0], g = F.merge_job[jm][1];
      const int nch = (a.pos[b] + 1 + a.chunk - 1) / a.chunk;
      if (tid == 0) {
        const int target = (l + 1 - a.slice_lo / 4) * nch;
        WaitClock wc;
        wc.start();
        F.flag = 1;
        for (;;) {
          int v;
          asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(a.sc.merge_cnt + b * NKV + g) : "memory");
          if (v >= target) break;
          if (wc.check(a.sc.err, a.spin_limit_ns)) {
            set_error(a.sc.err, MK_ERR_BARRIER_TIMEOUT, SITE_UNIT, b * NKV + g);
            F.flag = 0;
            break;
          }
        }
      }
      csync();
      if (F.flag) merge(l, b, g, nch, F.merge_job[jm][2], F.merge_job[jm][3]);
      csync();
    }
    if (tid == 0) {
      F.kc = k;
      F.n_merge = 0;
    }
    csync();
  }

  // Heads [h0, h1) of (b, g): log-sum-exp merge of the chunk partials into
  // the attention output, in chunk order.
  __device__ static __noinline__ void merge(int l, int b, int g, int nch, int h0, int h1) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n = c.n;
    if (nch > kMaxChunks) {
      if (tid == 0) set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_UNIT, nch);
      return;
    }
    const float* pb = a.sc.part + (size_t)(F.unit_start[b] + g * nch) * GQA * PR;
    // float4 output o = (head h0 + o / (HD/4), 4 dims) is summed by NG thread
    // groups over chunks grp, grp + NG, ...; the first batch of chunk outputs
    // is requested together with the (m, l) pairs: one L2 round trip
    constexpr int BATCH = 5;
    const int nout4 = (h1 - h0) * (HD / 4);
    const int NG = kThreads / nout4;
    const bool sum_thread = tid < NG * nout4;
    const int grp = tid / nout4, o4 = tid % nout4, hi = h0 + o4 / (HD / 4), d4 = o4 % (HD / 4);
    float4 ov[BATCH];
    if (sum_thread) {
#pragma unroll
      for (int u2 = 0; u2 < BATCH; ++u2) {
        const int cc = grp + u2 * NG;
        ov[u2] = cc < nch ? __ldcg(reinterpret_cast<const float4*>(pb + (cc * GQA + hi) * PR + 4) + d4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    // one warp per head: M = max_c m_c, L = sum_c l_c exp(m_c - M), and the
    // chunk factors exp(m_c - M) / L into shared memory
    float* mfac = F.red;  // [nch][GQA]
    if (wid < h1 - h0) {
      const int i = h0 + wid;
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
    csync();
    float4* gsum = reinterpret_cast<float4*>(c.act);  // [NG][nout4] (the combine area is free now)
    if (sum_thread) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c0 = grp;; c0 += NG * BATCH) {
#pragma unroll
        for (int u2 = 0; u2 < BATCH; ++u2) {
          const int cc = c0 + u2 * NG;
          const float f = cc < nch ? mfac[cc * GQA + hi] : 0.f;
          acc.x = fmaf(ov[u2].x, f, acc.x);
          acc.y = fmaf(ov[u2].y, f, acc.y);
          acc.z = fmaf(ov[u2].z, f, acc.z);
          acc.w = fmaf(ov[u2].w, f, acc.w);
        }
        if (c0 + NG * BATCH >= nch) break;
#pragma unroll
        for (int u2 = 0; u2 < BATCH; ++u2) {  // further chunks (long contexts)
          const int cc = c0 + NG * BATCH + u2 * NG;
          ov[u2] = cc < nch ? __ldcg(reinterpret_cast<const float4*>(pb + (cc * GQA + hi) * PR + 4) + d4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      gsum[grp * nout4 + o4] = acc;
    }
    csync();
    if (tid < nout4) {
      const int i = h0 + tid / (HD / 4), dd = tid % (HD / 4);
      float4 o = gsum[tid];
      for (int gg = 1; gg < NG; ++gg) {
        const float4 v = gsum[gg * nout4 + tid];
        o.x += v.x; o.y += v.y; o.z += v.z; o.w += v.w;
      }
      const size_t off = (size_t)(g * GQA + i) * HD + 4 * dd;
      *reinterpret_cast<float4*>(a.sc.attn + b * QD + off) = o;
      if (c.tr_attn) *reinterpret_cast<float4*>(c.tr_attn + ((size_t)l * n + b) * QD + off) = o;
    }
  }

  // ---------------------------------------------------------------- P3
  // o_proj rows of this block + residual.  In MoE layers the block also forms
  // its partial router logits: the post-attention RMSNorm is one scalar per
  // row times w2, so logits = rsqrt(mean(h^2) + eps) * sum_blocks(partials);
  // the scalar is applied in P4.
  template <int MODE>
  __device__ static __noinline__ void oproj_stage(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    // the residual rows this block adds to (its own rows of x), loaded in
    // the same round trip as the attention output
    for (int i = threadIdx.x; i < c.n * c.nr; i += kThreads) {
      const int b = i / c.nr, t = i % c.nr;
      F.hs[b][t] = __ldcg(a.sc.x + b * H + c.r0 + t);
    }
    {
      const float* at = a.sc.attn;
      if constexpr (MODE == 2)
        stage_plain_async<AUX, QD, false>(c.act, c.n, at, QD, 0.f, nullptr, F.red, nullptr);
      else
        stage_block<MODE, WDT, QD, false>(
            c.act, c.n, [&](int r, int f4) { return __ldcg(reinterpret_cast<const float4*>(at + r * QD) + f4); },
            0.f, [&](int) { return make_float4(1.f, 1.f, 1.f, 1.f); }, F.red, nullptr);
    }
    csync();
    MK_STAMP(c, l, 2, 0);
  }
  __device__ static __noinline__ void oproj(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31;
    const int n = c.n;
    struct {
      const StepArgs* a; Fixed* F; int r0, lane;
      __device__ __forceinline__ ActRange acts(int) const { return {nullptr, 0, a->n}; }
      __device__ __forceinline__ void put(int t, int b, int, float v0, float) const {
        const float hv = F->hs[b][t] + v0;   // residual row staged with the attention output
        a->sc.h[b * H + r0 + t] = hv;
        F->hs[b][t] = hv;
      }
    } task{&a, &F, c.r0, lane};
    run_gemv<QD, 1, T_O, false, false, true>(c.nr, c.act, task);
    if (l < a.n_dense) return;
    // the router / norm slices requested in P1 have landed
    asm volatile("cp.async.wait_all;" ::: "memory");
    csync();
    const uint32_t* rs = reinterpret_cast<const uint32_t*>(&F.dots[0][0]);
    for (int idx = tid; idx < n * E; idx += kThreads) {
      const int b = idx / E, e = idx % E;
      float s = 0.f;
      for (int t = 0; t < c.nr; ++t)
        s = fmaf(F.hs[b][t] * slice_val(F.nslw, t), slice_val(rs + e * kMaxRowsPerBlock, t), s);
      // every block adds its partial, as a 64-bit fixed-point integer, into
      // one of kRlogitGroups copies (fewer atomics queue on one address);
      // after the grid barrier every block sums the copies.  Integer sums do
      // not depend on the order of the additions, so every run and every
      // block get the same logits bit for bit.
      const long long q = to_fixed(s);
      atomicAdd(reinterpret_cast<unsigned long long*>(a.sc.rlogit + (c.bid % kRlogitGroups) * kMaxBatch * E + b * E + e),
                (unsigned long long)q);
    }
  }

  // ---------------------------------------------------------------- P4a
  // Routing, then the post-attention RMSNorm.  The router logits of a row are
  // rsqrt(mean(h^2) + eps) times the block-summed partials of P3; that factor
  // is positive and common to the row, so the top-k selection (ties -> lower
  // expert id) is made from the partials before the norm is known, and the
  // streaming warp is told at once so the experts' weights start moving while
  // the norm is computed.  The softmax weights (renormalised over the
  // selection) are formed from the scaled logits.  Dense layers only norm.
  // Routing of a one-row launch by warp 0 alone, with no block barrier: the
  // logit sums, the top-k (ranks, ties to the lower id) and the entry tables,
  // then the streaming warp is signalled.  The other warps go straight on to
  // the post-attention staging, whose block barriers publish the tables.
  __device__ static __forceinline__ void route_one(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const int lane = threadIdx.x & 31;
    float* lg = &F.dots[0][0];
    // every lane's loads in one round trip: experts lane and lane + 32
    constexpr int EPL = (E + 31) / 32;
    float v[EPL];
    {
      long long q[EPL][kRlogitGroups];
#pragma unroll
      for (int j = 0; j < EPL; ++j)
#pragma unroll
        for (int gr = 0; gr < kRlogitGroups; ++gr)
          q[j][gr] = lane + 32 * j < E ? __ldcg(a.sc.rlogit + gr * kMaxBatch * E + lane + 32 * j) : 0ll;
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        unsigned long long s = 0ull;  // wrapping two's-complement sum
#pragma unroll
        for (int gr = 0; gr < kRlogitGroups; ++gr) s += (unsigned long long)q[j][gr];
        v[j] = from_fixed((long long)s);
        if (lane + 32 * j < E) lg[lane + 32 * j] = v[j];
      }
    }
    // rank of each expert = experts with a larger logit, ties to the lower id,
    // counted over register values passed round the warp
    int rank[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) rank[j] = 0;
#pragma unroll
    for (int src = 0; src < 32; ++src)
#pragma unroll
      for (int j2 = 0; j2 < EPL; ++j2) {
        const float w = __shfl_sync(0xffffffffu, v[j2], src);
        const int e2 = src + 32 * j2;
        if (e2 < E)
#pragma unroll
          for (int j = 0; j < EPL; ++j) rank[j] += (w > v[j]) || (w == v[j] && e2 < lane + 32 * j);
      }
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (lane + 32 * j < E && rank[j] < TOPK) {
        F.topk_id[0][rank[j]] = lane + 32 * j;
        F.topk_w[0][rank[j]] = v[j];  // partial logit for now
      }
    __syncwarp();
    // one entry per slot, the distinct experts in increasing id order
    if (lane < TOPK) {
      const int my_e = F.topk_id[0][lane];
      int pos = 0;
#pragma unroll
      for (int j = 0; j < TOPK; ++j) pos += F.topk_id[0][j] < my_e;
      F.ent_b[pos] = 0;
      F.ent_j[pos] = (uint8_t)lane;
      F.ent_of[0][lane] = (uint8_t)pos;
      F.ue_expert[pos] = (int16_t)my_e;
      F.ue_start[pos] = (int16_t)pos;
      F.ue_len[pos] = 1;
    }
    __syncwarp();
    if (lane == 0) {
      F.n_ue = TOPK;
      __threadfence_block();
      F.route_gen = l + 1;
    }
    MK_STAMP(F.ctx, l, 5, 0);
  }

  __device__ static __noinline__ void route(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x;
    const bool moe = l >= a.n_dense;
    const int n = c.n;
    if (moe && n == 1) {
      if (tid < 32) route_one(l);
      return;
    }
    if (moe) {
      // partial logits into shared memory (F.dots is free between P3 and P5)
      float* lg = &F.dots[0][0];
      for (int i = tid; i < n * E; i += kThreads) {
        unsigned long long v = 0ull;  // wrapping two's-complement sum
#pragma unroll
        for (int gr = 0; gr < kRlogitGroups; ++gr)
          v += (unsigned long long)__ldcg(a.sc.rlogit + gr * kMaxBatch * E + i);
        lg[i] = from_fixed((long long)v);
      }
      for (int i = tid; i < n * TOPK; i += kThreads) F.topk_id[i / TOPK][i % TOPK] = i % TOPK;  // valid ids
      if (tid == 0) F.n_ue = 0;
      csync();
      // rank of each (row, expert) = experts with a larger partial logit, ties
      // to the lower id; the selection is the ranks below k (the same set and
      // order as k rounds of argmax)
      for (int i = tid; i < n * E; i += kThreads) {
        const int b = i / E, e = i % E;
        const float v = lg[i];
        int rank = 0;
#pragma unroll 8
        for (int e2 = 0; e2 < E; ++e2) {
          const float w = lg[b * E + e2];
          rank += (w > v) || (w == v && e2 < e);
        }
        if (rank < TOPK) {
          F.topk_id[b][rank] = e;
          F.topk_w[b][rank] = v;  // partial logit for now
        }
      }
      csync();
      // entries (row, slot) sorted by (expert, row, slot); one run of entries
      // per distinct expert
      const int N = n * TOPK;
      int my_e = 0, my_pos = 0;
      bool my_first = false;
      if (tid < N) {
        const int b = tid / TOPK, k = tid % TOPK;
        my_e = F.topk_id[b][k];
        int pos = 0;
        bool first = true;
        for (int j = 0; j < N; ++j) {
          const int e2 = F.topk_id[j / TOPK][j % TOPK];
          pos += (e2 < my_e) || (e2 == my_e && j < tid);
          first = first && !(e2 == my_e && j < tid);
        }
        F.ent_b[pos] = (uint8_t)b;
        F.ent_j[pos] = (uint8_t)k;
        F.ent_of[b][k] = (uint8_t)pos;
        F.efirst[tid] = first;
        my_pos = pos;
        my_first = first;
      }
      csync();
      if (my_first) {
        int ue = 0, len = 0;
        for (int j = 0; j < N; ++j) {
          const int e2 = F.topk_id[j / TOPK][j % TOPK];
          ue += F.efirst[j] && e2 < my_e;
          len += e2 == my_e;
        }
        F.ue_expert[ue] = (int16_t)my_e;
        F.ue_start[ue] = (int16_t)my_pos;
        F.ue_len[ue] = (int16_t)len;
        atomicMax(&F.n_ue, ue + 1);
      }
      csync();
      if (tid == 0) {
        __threadfence_block();
        F.route_gen = l + 1;
      }
      MK_STAMP(c, l, 5, 0);
    }
  }
  template <int MODE>
  __device__ static __noinline__ void ffn_stage(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    {
      const void* nw = F.lw.ffn_norm;
      const float* hp = a.sc.h;
      if constexpr (MODE == 2)
        stage_plain_async<AUX, H, true>(c.act, c.n, hp, H, a.eps, nw, F.red, F.rnorm);
      else
        stage_block<MODE, WDT, H, true>(
            c.act, c.n, [&](int r, int f4) { return __ldcg(reinterpret_cast<const float4*>(hp + r * H) + f4); },
            a.eps, [&](int f4) { return ld_aux4<AUX>(nw, f4); }, F.red, F.rnorm);
    }
    csync();
    MK_STAMP(c, l, 3, 0);
  }
  // Softmax weights of the selection, once the norm factor is known.
  __device__ static __noinline__ void route_weights(int l) {
    Fixed& F = fixed();
    const Ctx& c = F.ctx;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int n = c.n;
    for (int b = wid; b < n; b += kWarps) {
      const float r = F.rnorm[b];
      if (c.tr_rl && c.bid == 0)
        for (int e = lane; e < E; e += 32)
          c.tr_rl[((size_t)l * n + b) * E + e] = r * (&F.dots[0][0])[b * E + e];
      if (lane == 0) {
        // softmax over the selection = softmax over all experts renormalised
        const float top = r * F.topk_w[b][0];
        float wk[TOPK], wsum = 0.f;
#pragma unroll
        for (int kk = 0; kk < TOPK; ++kk) {
          wk[kk] = expf(r * F.topk_w[b][kk] - top);
          wsum += wk[kk];
        }
#pragma unroll
        for (int kk = 0; kk < TOPK; ++kk) {
          F.topk_w[b][kk] = wk[kk] / wsum;
          if (c.tr_tk && c.bid == 0) {
            c.tr_tk[((size_t)l * n + b) * 2 * TOPK + kk] = (float)F.topk_id[b][kk];
            c.tr_tk[((size_t)l * n + b) * 2 * TOPK + TOPK + kk] = wk[kk] / wsum;
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- P4b
  // Gate/up rows -> silu(gate) * up.  MoE: tasks (distinct expert, ffn row),
  // each computed for every row routed to that expert.  Dense: ffn rows.
  __device__ static __noinline__ void gateup(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int lane = threadIdx.x & 31;
    if (l >= a.n_dense) {
      route_weights(l);
      int u0, u1;
      gu_range(c, F.n_ue * FE, u0, u1);
      struct {
        const StepArgs* a; Fixed* F; int u0, lane;
        __device__ __forceinline__ ActRange acts(int t) const {
          const int ue = (u0 + t) / FE;
          return {F->ent_b, F->ue_start[ue], F->ue_len[ue]};
        }
        __device__ __forceinline__ void put(int t, int b, int i, float v0, float v1) const {
          const int u = u0 + t, f = u % FE;
          const int j = F->ent_j[F->ue_start[u / FE] + i];
          a->sc.act[(b * TOPK + j) * FE + f] = silu(v0) * v1;
        }
      } task{&a, &F, u0, lane};
      run_gemv<H, 2, T_XGU, false, false, false, XDT>(u1 - u0, c.act, task);
    } else {
      int f0, f1;
      gu_range(c, FD, f0, f1);
      struct {
        const StepArgs* a; int f0, lane;
        __device__ __forceinline__ ActRange acts(int) const { return {nullptr, 0, a->n}; }
        __device__ __forceinline__ void put(int t, int b, int, float v0, float v1) const {
          a->sc.dact[b * FD + f0 + t] = silu(v0) * v1;
        }
      } task{&a, f0, lane};
      run_gemv<H, 2, T_GU, false, false, true>(f1 - f0, c.act, task);
    }
  }

  // ---------------------------------------------------------------- P5
  // Down projection of this block's hidden rows.  MoE: the (row, expert slot)
  // activation vectors are staged in rounds of whole experts that fit the
  // staging area; a tile holds this block's rows of one or more experts'
  // matrices, each row is dotted with every entry of its expert.  Dense: the
  // batch rows are staged in rounds, the full-width rows of the block are
  // streamed once per round.  Then the weighted sum over experts in slot
  // order and the residual.
  // A round is the expert entries (MoE) or batch rows (dense) that fit the
  // staging area; `u` is the round's first distinct expert / row.
  template <bool MOE>
  __device__ static __forceinline__ int down_next(int u) {
    const Fixed& F = fixed();
    if constexpr (MOE) return moe_round_end(F, u, F.ctx.act_bytes / moe_entry_bytes(F.ctx));
    else return u + F.ctx.act_bytes / dense_entry_bytes(F.ctx);
  }
  template <bool MOE, int MODE>
  __device__ static __noinline__ void down_stage(int l, int u) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int ub = down_next<MOE>(u);
    if constexpr (MOE) {
      const int e0 = F.ue_start[u], ecnt = F.ue_start[ub - 1] + F.ue_len[ub - 1] - e0;
      const float* act = a.sc.act;
      const Fixed* Fp = &F;
      stage_block<MODE, WDT, FE, false>(
          c.act, ecnt,
          [&](int r, int f4) -> float4 {
            const int en = e0 + r;
            const float* src = act + (Fp->ent_b[en] * TOPK + Fp->ent_j[en]) * FE;
            return __ldcg(reinterpret_cast<const float4*>(src) + f4);
          },
          0.f, [&](int) { return make_float4(1.f, 1.f, 1.f, 1.f); }, F.red, nullptr);
    } else {
      const int cnt = min(ub, c.n) - u;
      const float* dact = a.sc.dact;
      if constexpr (MODE == 2)
        stage_plain_async<AUX, FD, false>(c.act, cnt, dact + (size_t)u * FD, FD, 0.f, nullptr, F.red, nullptr);
      else
        stage_block<MODE, WDT, FD, false>(
            c.act, cnt,
            [&](int r, int f4) { return __ldcg(reinterpret_cast<const float4*>(dact + (u + r) * FD) + f4); },
            0.f, [&](int) { return make_float4(1.f, 1.f, 1.f, 1.f); }, F.red, nullptr);
    }
    csync();
    MK_STAMP(c, l, 4, 0);
  }
  template <bool MOE>
  __device__ static __noinline__ void down_gemv(int l, int u) {
    Fixed& F = fixed();
    const Ctx& c = F.ctx;
    const int lane = threadIdx.x & 31;
    const int nr = c.nr;
    const int ub = down_next<MOE>(u);
    if constexpr (MOE) {
      const int e0 = F.ue_start[u];
      struct {
        Fixed* F; int ua, nr, e0, lane;
        __device__ __forceinline__ ActRange acts(int t) const {
          const int ue = ua + t / nr;
          return {nullptr, F->ue_start[ue] - e0, F->ue_len[ue]};
        }
        __device__ __forceinline__ void put(int t, int ai, int, float v0, float) const {
          F->dots[e0 + ai][t % nr] = v0;
        }
      } task{&F, u, nr, e0, lane};
      run_gemv<FE, 1, T_XDN, GXE::ACT_REGS, true, false, XDT>((ub - u) * nr, c.act, task);
    } else {
      const int cnt = min(ub, c.n) - u;
      struct {
        Fixed* F; int ba, cnt, lane;
        __device__ __forceinline__ ActRange acts(int) const { return {nullptr, 0, cnt}; }
        __device__ __forceinline__ void put(int t, int ai, int, float v0, float) const {
          F->dots[ba + ai][t] = v0;
        }
      } task{&F, u, cnt, lane};
      run_gemv<FD, 1, T_DD, false, false, true>(nr, c.act, task);
    }
  }
  // The weighted sum over the experts in slot order, plus the residual.
  // (The next layer's pointers, requested during gate/up, land here: the
  // grid barrier that follows publishes them to the whole block.)
  template <bool MOE>
  __device__ static __noinline__ void down_finish(int l) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x;
    asm volatile("cp.async.wait_all;" ::: "memory");
    const int n = c.n, nr = c.nr;
    for (int idx = tid; idx < n * nr; idx += kThreads) {
      const int b = idx / nr, rr = idx % nr;
      float s = 0.f;
      if (MOE)
        for (int kk = 0; kk < TOPK; ++kk) s = fmaf(F.topk_w[b][kk], F.dots[F.ent_of[b][kk]][rr], s);
      else
        s = F.dots[b][rr];
      const float xv = F.hs[b][rr] + s;   // this block's rows of h, kept since o_proj
      a.sc.x[b * H + c.r0 + rr] = xv;
      if (c.flagged) flag_put(a.sc.xll + ((size_t)(l & 1) * kMaxBatch + b) * H + c.r0 + rr, xv, c.tag0 + l + 1);
      if (c.tr_x) c.tr_x[((size_t)l * n + b) * H + c.r0 + rr] = xv;
    }
  }
  template <bool MOE>
  __device__ static __forceinline__ void down(int l) {
    const Fixed& F = fixed();
    const int end = MOE ? F.n_ue : F.ctx.n;
    // MoE rounds hold several entries (the experts of a row); dense rounds
    // are batch rows
    const int mode = MOE ? 1 : stage_mode(F.ctx, true);
#pragma unroll 1
    for (int u = 0; u < end; u = down_next<MOE>(u)) {
      if (mode == 0) down_stage<MOE, 0>(l, u);
      else if (mode == 1) down_stage<MOE, 1>(l, u);
      else down_stage<MOE, 2>(l, u);
      down_gemv<MOE>(l, u);
    }
    down_finish<MOE>(l);
  }
  // staging variant of a launch: plain rows for the tensor-core path, one
  // row, or several
  __device__ static __forceinline__ int stage_mode(const Ctx& c, bool tc_ok) {
    return (c.tc && tc_ok) ? 2 : (c.n == 1 ? 0 : 1);
  }

  // ---------------------------------------------------------------- lm_head
  // Final RMSNorm, this block's vocabulary rows, argmax per row of the batch
  // (ties -> lowest token id); the last block to finish reduces the blocks'
  // candidates in block order and writes the tokens.
  template <int MODE>
  __device__ static __noinline__ void lm_stage() {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    {
      const void* nw = a.final_norm;
      const float* x = a.sc.x + a.out_first * H;
      if constexpr (MODE == 2)
        stage_plain_async<AUX, H, true>(c.act + a.out_first * plain_stride(H), c.n - a.out_first, x, H, a.eps, nw,
                                        F.red, nullptr);
      else
        stage_block<MODE, WDT, H, true>(
            c.act + a.out_first * (MODE == 2 ? plain_stride(H) : GH::ACT_BYTES), c.n - a.out_first,
            [&](int r, int f4) { return __ldcg(reinterpret_cast<const float4*>(x + r * H) + f4); },
            a.eps, [&](int f4) { return ld_aux4<AUX>(nw, f4); }, F.red, nullptr);
    }
    if (threadIdx.x < kMaxBatch) F.best_key[threadIdx.x] = 0ull;
    csync();
  }
  __device__ static __noinline__ void lm_head() {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n = c.n;
    int v0, v1;
    gu_range(c, a.vocab, v0, v1);
    struct {
      const StepArgs* a; Fixed* F; float* tr; int vr0, lane, wid;
      __device__ __forceinline__ ActRange acts(int) const { return {nullptr, a->out_first, a->n - a->out_first}; }
      __device__ __forceinline__ void put(int t, int b, int, float v0, float) const {
        const int tok = vr0 + t;
        // one 64-bit key per row: larger logit first, then the lower token id
        atomicMax(&F->best_key[b], argmax_key(v0, tok));
        if (tr) tr[(size_t)b * a->vocab + tok] = v0;
      }
    } task{&a, &F, c.tr_fin, v0, lane, wid};
    run_gemv<H, 1, T_LM, GH::ACT_REGS, false, true>(v1 - v0, c.act, task);
    if (tid < n) {
      const unsigned long long key = F.best_key[tid];
      a.sc.amax_v[c.bid * kMaxBatch + tid] = key ? key_value(key) : -INFINITY;
      a.sc.amax_i[c.bid * kMaxBatch + tid] = key ? key_token(key) : INT_MAX;
    }
    csync();
    if (tid == 0) {
      __threadfence();
      F.flag = atomicAdd(a.sc.sync + 96, 1u) == (uint32_t)(c.G - 1);
    }
    csync();
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

  // ---------------------------------------------------------------- streaming warp
  // One run of `cnt` consecutive packed records into the stage at record j.
  __device__ static __forceinline__ void put_recs(Producer& p, int j, int cnt, const uint8_t* src, int rc) {
    p.copy((uint32_t)(j * rc), src, (uint32_t)(cnt * rc));
  }

  // Pool pages of this block's attention units (positions before new0 only,
  // the same for every layer), read once per launch by the whole streaming
  // warp.
  __device__ static __forceinline__ void load_unit_pages() {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int lane = threadIdx.x & 31;
    int k = 0;
    for (int u = c.bid; u < a.n_units; u += c.G, ++k) {
      int b, g, ci, nch;
      unit_of(a, F.unit_start, u, c.n, b, g, ci, nch);
      int t0, rt1, t1;
      unit_span(a, b, ci, t0, rt1, t1);
      if (rt1 <= t0) continue;
      const int p0 = t0 / kPageTokens, np = (rt1 - 1) / kPageTokens - p0 + 1;
      if (k >= 2 || np > 64) {
        if (lane == 0) set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_UNIT, u);
        continue;
      }
      for (int j = lane; j < np; j += 32) {
        const int pi = p0 + j;
        int page = pi < a.max_pages_per_seq ? __ldcg(a.block_table + a.slot[b] * a.max_pages_per_seq + pi) : -1;
        if (page < 0 || page >= a.n_pages) {
          set_error(a.sc.err, MK_ERR_DEVICE_INDEX, SITE_PAGE, pi);
          page = 0;
        }
        F.upages[k][j] = page;
      }
    }
    __syncwarp();
  }

  // The block's schedule of ring items for the whole launch, in the order the
  // compute warps consume them (lane 0 of the streaming warp).  Every tile is
  // one run of packed records, or one run per expert.
  __device__ static __noinline__ void produce() {
    Producer p;  // registers of the streaming lane; the item count goes to F.prod_k
    run_schedule(p);
    fixed().prod_k = p.k;
  }
  __device__ static __forceinline__ void run_schedule(Producer& p) {
    Fixed& F = fixed();
    const StepArgs& a = F.args;
    const Ctx& c = F.ctx;
    const int n = c.n;
#pragma unroll 1
    for (int s = a.slice_lo; s < a.slice_hi; s += 4 - s % 4) {  // one pass per layer touched
      const int l = s / 4;
      const int part_lo = s % 4, part_hi = min(4, a.slice_hi - 4 * l);  // parts [part_lo, part_hi) of layer l
      const LayerW Lg = a.layers[l];  // one batch of loads per layer
      if (part_lo <= 0 && part_hi > 0) {  // P1: RoPE pair tasks [p0, p1): records 2p, 2p + 1
        int p0, p1;
        qkv_range(c, p0, p1);
#pragma unroll 1
        for (int ta = p0; ta < p1; ta += T_QKV) {
          if (!p.template begin<STAGE>()) return;
          put_recs(p, 0, 2 * min(T_QKV, p1 - ta), Lg.pk[PK_QKV] + (size_t)2 * ta * REC_H, REC_H);
          p.end();
        }
      }
      if (part_lo <= 1 && part_hi > 1) {  // P2: cached K/V of this block's units
        int k = 0;
#pragma unroll 1
        for (int u = c.bid; u < a.n_units; u += c.G, ++k) {
          int b, g, ci, nch;
          unit_of(a, F.unit_start, u, n, b, g, ci, nch);
          int t0, rt1, t1;
          unit_span(a, b, ci, t0, rt1, t1);
          const int pbase = t0 / kPageTokens;
#pragma unroll 1
          for (int tb = t0; tb < rt1; tb += TT) {
            if (!p.template begin<STAGE>()) return;
            const int nt = min(TT, rt1 - tb);
#pragma unroll 1
            for (int j = 0; j < nt;) {
              const int t = tb + j, slot = t % kPageTokens;
              const int run = min(nt - j, kPageTokens - slot);
              const int page = F.upages[min(k, 1)][t / kPageTokens - pbase];
#pragma unroll
              for (int kv = 0; kv < 2; ++kv)
                p.copy((uint32_t)((kv * TT + j) * HD * 2), a.kv + Kv<S>::offset(l, a.n_pages, page, kv, g, slot),
                       (uint32_t)(run * HD * 2));
              j += run;
            }
            p.end();
          }
        }
      }
      // P3: o_proj rows [r0, r0 + nr)
      if (part_lo <= 2 && part_hi > 2) {
#pragma unroll 1
        for (int t0 = 0; t0 < c.nr; t0 += T_O) {
          if (!p.template begin<STAGE>()) return;
          put_recs(p, 0, min(T_O, c.nr - t0), Lg.pk[PK_O] + (size_t)(c.r0 + t0) * REC_Q, REC_Q);
          p.end();
        }
      }
      if (part_hi <= 3) continue;
      if (l >= a.n_dense) {
        // P4/P5 need the layer's routing
        {
          WaitClock wc;
          wc.start();
          uint32_t i = 0;
          while (F.route_gen < l + 1) {
            if ((++i & 15u) == 0) {
              if (F.abort) return;
              const int r = wc.check(a.sc.err, a.spin_limit_ns);
              if (r == 2) set_error(a.sc.err, MK_ERR_BARRIER_TIMEOUT, SITE_RING, l);
              if (r) return;
            }
          }
          __threadfence_block();
        }
        int u0, u1;
        gu_range(c, F.n_ue * FE, u0, u1);
#pragma unroll 1
        for (int ta = u0; ta < u1; ta += T_XGU) {
          if (!p.template begin<STAGE>()) return;
          const int tb = min(u1, ta + T_XGU);
#pragma unroll 1
          for (int q0 = ta; q0 < tb;) {  // a run stays inside one expert: records 2t, 2t + 1
            const int q1 = min(tb, (q0 / FE + 1) * FE);
            const size_t t = (size_t)F.ue_expert[q0 / FE] * FE + q0 % FE;
            put_recs(p, 2 * (q0 - ta), 2 * (q1 - q0), Lg.pk[PK_GU] + 2 * t * REC_XH, REC_XH);
            q0 = q1;
          }
          p.end();
        }
        const int cap = c.act_bytes / moe_entry_bytes(c);
        const int nr = c.nr;
#pragma unroll 1
        for (int ua = 0; ua < F.n_ue;) {
          const int ub = moe_round_end(F, ua, cap);
          const int ntask = (ub - ua) * nr;
#pragma unroll 1
          for (int ta = 0; ta < ntask; ta += T_XDN) {
            if (!p.template begin<STAGE>()) return;
            const int tb = min(ntask, ta + T_XDN);
#pragma unroll 1
            for (int q0 = ta; q0 < tb;) {  // a run stays inside one expert
              const int q1 = min(tb, (q0 / nr + 1) * nr);
              const size_t row = (size_t)F.ue_expert[ua + q0 / nr] * H + c.r0 + q0 % nr;
              put_recs(p, q0 - ta, q1 - q0, Lg.pk[PK_DN] + row * REC_XE, REC_XE);
              q0 = q1;
            }
            p.end();
          }
          ua = ub;
        }
      } else {
        int f0, f1;
        gu_range(c, FD, f0, f1);
#pragma unroll 1
        for (int t0 = f0; t0 < f1; t0 += T_GU) {
          if (!p.template begin<STAGE>()) return;
          put_recs(p, 0, 2 * min(T_GU, f1 - t0), Lg.pk[PK_GU] + (size_t)2 * t0 * REC_H, REC_H);
          p.end();
        }
        const int cap = c.act_bytes / dense_entry_bytes(c);
#pragma unroll 1
        for (int ba = 0; ba < n; ba += cap) {
#pragma unroll 1
          for (int t0 = 0; t0 < c.nr; t0 += T_DD) {
            if (!p.template begin<STAGE>()) return;
            put_recs(p, 0, min(T_DD, c.nr - t0), Lg.pk[PK_DN] + (size_t)(c.r0 + t0) * REC_D, REC_D);
            p.end();
          }
        }
      }
    }
    if (a.run_lm && a.out_first < n) {
      int v0, v1;
      gu_range(c, a.vocab, v0, v1);
#pragma unroll 1
      for (int t0 = v0; t0 < v1; t0 += T_LM) {
        if (!p.template begin<STAGE>()) return;
        put_recs(p, 0, min(T_LM, v1 - t0), a.lm_pk + (size_t)t0 * REC_H, REC_H);
        p.end();
      }
    }
  }
};

template <class S, int WDT, int XDT>
__global__ void __launch_bounds__(kBlockThreads, 1) step_kernel(const __grid_constant__ StepArgs a) {
  using M = Model<S, WDT, XDT>;
  extern __shared__ __align__(128) uint8_t smem[];
  Fixed& F = *reinterpret_cast<Fixed*>(smem);
  const int tid = threadIdx.x;
  // launch arguments into shared memory: the phases read them from there
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&a);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&F.args);
    static_assert(sizeof(StepArgs) % 4 == 0, "word copy");
    for (int i = tid; i < (int)(sizeof(StepArgs) / 4); i += kBlockThreads) dst[i] = src[i];
  }
  const int n = a.n;
  if (tid == 0) {
    Ctx& c = F.ctx;
    c.act = smem + kActOffset;
    c.G = gridDim.x;
    c.bid = blockIdx.x;
    c.n = n;
    int r0, r1;
    split_range(S::H / M::A_H, c.G, c.bid, r0, r1);
    c.r0 = r0 * M::A_H;
    c.nr = (r1 - r0) * M::A_H;
    // staging area, then the ring in what is left
    // the launch's dynamic shared memory (less for one row: more L1)
    uint32_t dsz;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dsz));
    const int avail = (int)dsz - kActOffset;
    c.tc = M::TC && n >= 2;
    c.flagged = n == 1 && a.slice_lo == 0 && a.slice_hi == 4 * a.n_layers;
    c.tag0 = *(volatile uint32_t*)(a.sc.sync + 64) * 256u;
    int act = M::act_base_bytes(n, c.tc);
    const int want = n * S::TOPK * M::moe_entry_bytes(c);
    if (want > act) act = max(act, min(want, avail - 3 * M::STAGE));
    act = (act + 127) / 128 * 128;
    c.act_bytes = act;
    c.ring = smem + kActOffset + act;
    c.ns = min(kMaxStages, (avail - act) / M::STAGE);
    c.tr_x = a.trace;
    c.tr_attn = a.trace ? c.tr_x + (size_t)a.n_layers * n * S::H : nullptr;
    c.tr_rl = a.trace ? c.tr_attn + (size_t)a.n_layers * n * M::QD : nullptr;
    c.tr_tk = a.trace ? c.tr_rl + (size_t)a.n_layers * n * S::E : nullptr;
    c.tr_fin = a.trace ? c.tr_tk + (size_t)a.n_layers * n * 2 * S::TOPK : nullptr;
    c.tm = a.timing ? a.timing + (size_t)blockIdx.x * (16 * a.n_layers + 2) : nullptr;
    c.ring_log = a.timing ? a.timing + (size_t)c.G * (16 * a.n_layers + 2) + (size_t)blockIdx.x * 3 * kRingLog
                          : nullptr;
    // attention work units: (row, kv head, chunk), row-major
    int acc = 0;
    for (int b = 0; b < n; ++b) {
      F.unit_start[b] = acc;
      acc += S::NKV * ((a.pos[b] + 1 + a.chunk - 1) / a.chunk);
    }
    F.unit_start[n] = acc;
    F.kc = 0;
    F.prod_k = 0;
    F.route_gen = 0;
    F.n_merge = 0;
    F.abort = 0;
    for (int s = 0; s < c.ns; ++s) {
      mbar_init(&F.full[s], 1);
      mbar_init(&F.empty[s], kWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (c.ns < 2) set_error(a.sc.err, MK_ERR_UNSUPPORTED, SITE_SMEM, c.ns);
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

  if (tid >= kThreads) {
    // streaming warp
    if (c.ns >= 2) {
      M::load_unit_pages();
      if (tid == kThreads) M::produce();
    }
    __syncwarp();
  } else {
    bool ok = c.ns >= 2;
    uint32_t nbar = 0;
    if (c.tm && tid == 0) c.tm[0] = globaltimer();
    // the layer's norm / router pointers in shared memory; layer l + 1's are
    // requested (cp.async, nothing waits on them) once layer l's staging has
    // used them, and have landed by the end of the layer (down_finish waits)
    auto load_lw = [&](int l) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(a.layers + l);
      for (int i = tid; i < (int)(sizeof(LayerW) / 4); i += kThreads)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(reinterpret_cast<uint32_t*>(&F.lw) + i)),
                     "l"(src + i)
                     : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    load_lw(a.slice_lo / 4 < a.n_layers ? a.slice_lo / 4 : 0);
    asm volatile("cp.async.wait_all;" ::: "memory");
    csync();
    // phase groups [slice_lo, slice_hi): a whole step, or one group per launch
    // (MK_DBG_SPLIT), where state a group keeps in shared memory for a later
    // group is reloaded from global memory at the start of the launch
    for (int s = a.slice_lo; ok && s < a.slice_hi; ++s) {
      const int l = s / 4, part = s % 4;
      // a later group, or lm_head (which reads every block's rows of x),
      // follows in this launch: the group ends with a grid barrier
      const bool more = s + 1 < a.slice_hi || (a.run_lm && a.out_first < n);
      const bool first = s == a.slice_lo;
      const int sm = M::stage_mode(c, true);
      if (part == 0) {
        if (sm == 0) M::template qkv_stage<0>(l);
        else if (sm == 1) M::template qkv_stage<1>(l);
        else M::template qkv_stage<2>(l);
        M::qkv(l);
        MK_STAMP(c, l, 0, 1);
        if (more && !(ok = grid_barrier(a, nbar, &F.ok_word))) break;
        MK_STAMP(c, l, 0, 2);
      } else if (part == 1) {
        M::attention(l);
        MK_STAMP(c, l, 1, 1);
        if (more && !(ok = grid_barrier(a, nbar, &F.ok_word))) break;
        MK_STAMP(c, l, 1, 2);
      } else if (part == 2) {
        if (first && l >= a.n_dense) M::fetch_router_slice(F.lw);  // fetched by the QKV group otherwise
        if (sm == 0) M::template oproj_stage<0>(l);
        else if (sm == 1) M::template oproj_stage<1>(l);
        else M::template oproj_stage<2>(l);
        M::oproj(l);
        MK_STAMP(c, l, 2, 1);
        if (more && !(ok = grid_barrier(a, nbar, &F.ok_word))) break;
        MK_STAMP(c, l, 2, 2);
      } else {
        if (first)  // this block's rows of h, kept by the o_proj group otherwise
          for (int i = tid; i < n * c.nr; i += kThreads)
            F.hs[i / c.nr][i % c.nr] = __ldcg(a.sc.h + (i / c.nr) * S::H + c.r0 + i % c.nr);
        M::route(l);
        {
          const int fm = M::stage_mode(c, l < a.n_dense);
          if (fm == 0) M::template ffn_stage<0>(l);
          else if (fm == 1) M::template ffn_stage<1>(l);
          else M::template ffn_stage<2>(l);
        }
        if (l + 1 < a.n_layers) load_lw(l + 1);
        M::gateup(l);
        MK_STAMP(c, l, 3, 1);
        if (!(ok = grid_barrier(a, nbar, &F.ok_word))) break;
        MK_STAMP(c, l, 3, 2);
        if (l >= a.n_dense) M::template down<true>(l);
        else M::template down<false>(l);
        MK_STAMP(c, l, 4, 1);
        // the next layer's QKV waits for the flagged residual words instead
        const bool by_flags = c.flagged && s + 1 < a.slice_hi;
        if (more && !by_flags && !(ok = grid_barrier(a, nbar, &F.ok_word))) break;
        MK_STAMP(c, l, 4, 2);
      }
    }
    if (ok && a.run_lm && a.out_first < n) {
      // rows from out_first on: one row alone takes the one-row variant
      const int lm = c.tc ? 2 : (n - a.out_first == 1 ? 0 : 1);
      if (lm == 0) M::template lm_stage<0>();
      else if (lm == 1) M::template lm_stage<1>();
      else M::template lm_stage<2>();
      M::lm_head();
    }
    if (c.tm && tid == 0) c.tm[1 + 16 * a.n_layers] = globaltimer();
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy into shared memory outlives the block
    csync();
    if (tid == 0 && !ok) F.abort = 1;
  }
  __syncthreads();
  // every copy the streaming warp issued has landed before the block ends
  if (tid >= kThreads) {
    if (tid == kThreads) {
      Producer prod;
      prod.k = F.prod_k;
      prod.drain();
    }
    __syncwarp();
  }
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.sc.sync + 32, 1u) == (uint32_t)(c.G - 1)) {
      // every block has left its work: reset the launch-scoped counters
      a.sc.sync[0] = 0;
      a.sc.sync[96] = 0;
      a.sc.sync[64] += 1;  // the next launch's epoch
      for (int i = 0; i < kMaxBatch * S::NKV; ++i) a.sc.merge_cnt[i] = 0;
      __threadfence();
      a.sc.sync[32] = 0;
    }
  }
}

template <class S, int WDT, int XDT = WDT>
static KernelInfo make() {
  return {reinterpret_cast<const void*>(&step_kernel<S, WDT, XDT>), kSmemBytes, Model<S, WDT, XDT>::TT,
          Model<S, WDT, XDT>::SMEM_SINGLE};
}

// The instantiations are spread over translation units (this file compiled
// once per value of MK_KERNEL_PART), which build in parallel.
#if MK_KERNEL_PART == 0
KernelInfo get_kernel_part0(int shape, int wdtype, int xdtype) {
  if (shape == SHAPE_FLINT && wdtype == MK_INT4_G64 && xdtype == wdtype) return make<ShapeFlint, WINT4>();
  return {nullptr, 0, 0, 0};
}
#elif MK_KERNEL_PART == 1
KernelInfo get_kernel_part1(int shape, int wdtype, int xdtype) {
  if (shape == SHAPE_FLINT && wdtype == MK_BF16 && xdtype == wdtype) return make<ShapeFlint, WBF16>();
  return {nullptr, 0, 0, 0};
}
#elif MK_KERNEL_PART == 2
KernelInfo get_kernel_part2(int shape, int wdtype, int xdtype) {
  if (shape == SHAPE_FLINT && wdtype == MK_INT4_G64 && xdtype == MK_INT3_G64) return make<ShapeFlint, WINT4, WINT3>();
  return {nullptr, 0, 0, 0};
}
#else
KernelInfo get_kernel_part3(int shape, int wdtype, int xdtype) {
  if (shape == SHAPE_TINY) {
    if (wdtype == MK_INT4_G64 && xdtype == wdtype) return make<ShapeTiny, WINT4>();
    if (wdtype == MK_INT4_G64 && xdtype == MK_INT3_G64) return make<ShapeTiny, WINT4, WINT3>();
    if (wdtype == MK_BF16 && xdtype == wdtype) return make<ShapeTiny, WBF16>();
    if (wdtype == MK_F32 && xdtype == wdtype) return make<ShapeTiny, WF32>();
  }
  return {nullptr, 0, 0, 0};
}
#endif

}  // namespace mk
