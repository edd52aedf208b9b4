// Device building blocks of the decode megakernel: memory access helpers,
// the grid barrier, the shared-memory weight ring (mbarriers + bulk copies),
// activation staging and the warp-level GEMV engine.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include "mk_internal.h"

namespace mk {

enum { WF32 = 0, WBF16 = 1, WINT4 = 2, WINT3 = 3 };

// ------------------------------------------------------------------ shapes
// The layer shapes the kernel is compiled for.  Flint: the model of "rec
// Megakernel and Tempo9 Compared", §2 (2048-wide residual, 49 layers, top-6
// experts, dense MLP in layers 0-1) with the remaining sizes fixed by the
// workload; tiny: a small model of the same family for fast parity runs.
struct ShapeFlint {
  static constexpr int H = 2048, NH = 16, NKV = 4, HD = 128, E = 64, TOPK = 6, FE = 768,
                       FD = 6144;
};
struct ShapeTiny {
  static constexpr int H = 256, NH = 4, NKV = 2, HD = 64, E = 8, TOPK = 2, FE = 128, FD = 512;
};

// ------------------------------------------------------------------ memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint32_t lds32(const void* p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint32_t lds16(const void* p) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ float bf16_to_f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ uint16_t f_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int AUX>  // aux dtype: WF32 or WBF16
__device__ __forceinline__ float ld_aux(const void* p, int i) {
  if constexpr (AUX == WF32) return __ldg(reinterpret_cast<const float*>(p) + i);
  else return bf16_to_f(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
}

// Four consecutive aux values (elements 4*i4 .. 4*i4+3) as float4.
template <int AUX>
__device__ __forceinline__ float4 ld_aux4(const void* p, size_t i4) {
  if constexpr (AUX == WF32) return __ldg(reinterpret_cast<const float4*>(p) + i4);
  else {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p) + i4);
    return make_float4(bf16_to_f(u.x & 0xffff), bf16_to_f(u.x >> 16), bf16_to_f(u.y & 0xffff),
                       bf16_to_f(u.y >> 16));
  }
}

// Fixed-point values (units of 2^-32) of the router sums; the scale is a
// power of two, so the conversions round only once.
__device__ __forceinline__ long long to_fixed(float v) { return __float2ll_rn(v * kFixScale); }
__device__ __forceinline__ float from_fixed(long long q) { return __ll2float_rn(q) * kFixUnit; }
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Transposing butterfly: reduce NV (a power of two <= 32) per-lane partial
// values across the warp with NV - 1 + log2(32 / NV) shuffles instead of
// 5 * NV.  Returns, in every lane, the full sum of value number
// bitrev(lane mod NV) (bit-reversed over log2(NV) bits).
template <int NV>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NV], int lane) {
  static_assert(NV >= 1 && NV <= 32 && (NV & (NV - 1)) == 0, "power of two");
  int m = 1;
#pragma unroll
  for (int h = NV / 2; h >= 1; h >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < h; ++j) {
      const float keep = up ? v[j + h] : v[j];
      const float send = up ? v[j] : v[j + h];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
    m <<= 1;
  }
#pragma unroll
  for (int mm = NV; mm < 32; mm <<= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], mm);
  return v[0];
}

template <int BITS>
__device__ __forceinline__ constexpr int bitrev(int x) {
  int r = 0;
  for (int i = 0; i < BITS; ++i) r |= ((x >> i) & 1) << (BITS - 1 - i);
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_error(int32_t* err, int code, int site, int detail) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = site;
    err[2] = detail;
  }
}

// Barrier among the compute warps only (the streaming warp never joins).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// ------------------------------------------------------------------ grid barrier
// One monotonically increasing arrival counter per launch: barrier k of the
// launch completes when the counter reaches k * gridDim.x.  The arrive is a
// release reduction (cumulative over the block's writes ordered before it by
// the block barrier), the wait an acquire load, so every write before the
// barrier is visible to every block after it.  The wait is bounded: it gives
// up when another block has recorded an error, or after spin_limit_ns, and
// then records MK_ERR_BARRIER_TIMEOUT; the caller skips to the exit path.
// `ok` is a shared-memory word used to broadcast the outcome.
// Every bounded wait polls its own condition and, while it waits, the global
// error word (another block gave up).  Reading the error word is an L2 round
// trip during which the condition goes unseen, so a wait reads it only after
// kErrPollNs of waiting and then once per kErrPollNs: a wait that ends within
// that time never reads it.
constexpr uint64_t kErrPollNs = 8000;
struct WaitClock {
  uint64_t t0, next;
  __device__ __forceinline__ void start() {
    t0 = globaltimer();
    next = t0 + kErrPollNs;
  }
  // 0 keep waiting, 1 an error is recorded, 2 this wait ran past limit_ns
  __device__ __forceinline__ int check(const int32_t* err, uint64_t limit_ns) {
    const uint64_t now = globaltimer();
    if (now < next) return 0;
    next = now + kErrPollNs;
    if (*(const volatile int32_t*)err != 0) return 1;
    return now - t0 > limit_ns ? 2 : 0;
  }
};

// ------------------------------------------------------------------ flagged words
// A value exchanged between blocks without a grid barrier travels with its
// tag in one 64-bit word (value bits low, tag high), written by one 64-bit
// store, which is single-copy atomic: a reader that sees the tag it expects
// sees the value that came with it.  Tags are unique per launch and layer, so
// a word left from an earlier layer or launch never matches.
__device__ __forceinline__ void flag_put(uint64_t* p, float v, uint32_t tag) {
  const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// The four values at p (32-byte aligned) once all four carry `tag`.  The wait
// is bounded like the others: on an error or a timeout it records the error
// and returns zeros (the step is then reported failed).
__device__ __forceinline__ float4 flag_get4(const uint64_t* p, uint32_t tag, const StepArgs& a);

static __device__ __noinline__ bool grid_barrier(const StepArgs& a, uint32_t& k, volatile int* ok_word) {
  csync();
  if (threadIdx.x == 0) {
    ++k;
    uint32_t* ctr = a.sc.sync;
    bool skip = (a.dbg_flags & MK_DBG_SKIP_ARRIVAL) && (a.dbg_arg >> 16) == k &&
                (a.dbg_arg & 0xffffu) == blockIdx.x;
    if (!skip) asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(1u) : "memory");
    const uint32_t target = k * gridDim.x;
    int ok = 1;
    WaitClock wc;
    wc.start();
    for (;;) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      const int r = wc.check(a.sc.err, a.spin_limit_ns);
      if (r) {
        if (r == 2) set_error(a.sc.err, MK_ERR_BARRIER_TIMEOUT, SITE_BARRIER, (int)k);
        ok = 0;
        break;
      }
    }
    *ok_word = ok;
  }
  csync();
  return *ok_word != 0;
}

__device__ __forceinline__ float4 flag_get4(const uint64_t* p, uint32_t tag, const StepArgs& a) {
  uint64_t w0, w1, w2, w3;
  WaitClock wc;
  bool waited = false;
  for (;;) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p) : "memory");
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(w2), "=l"(w3) : "l"(p + 2) : "memory");
    if ((uint32_t)(w0 >> 32) == tag && (uint32_t)(w1 >> 32) == tag && (uint32_t)(w2 >> 32) == tag &&
        (uint32_t)(w3 >> 32) == tag)
      break;
    if (!waited) {
      wc.start();
      waited = true;
    }
    if (const int r = wc.check(a.sc.err, a.spin_limit_ns)) {
      if (r == 2) set_error(a.sc.err, MK_ERR_BARRIER_TIMEOUT, SITE_FLAG, (int)(tag & 0xFFu));
      return make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  return make_float4(__uint_as_float((uint32_t)w0), __uint_as_float((uint32_t)w1), __uint_as_float((uint32_t)w2),
                     __uint_as_float((uint32_t)w3));
}

// ------------------------------------------------------------------ weight ring
// Shared-memory stages filled by bulk copies (cp.async.bulk, the TMA unit)
// and tracked by mbarriers: full[s] completes when the bytes of stage s have
// landed (one arrival by the streaming warp plus the copies' transaction
// bytes), empty[s] when all compute warps have released it.  Item k of the
// launch's stream uses stage k % NS in round k / NS; the parity of the round
// selects the mbarrier phase.
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the given phase parity: gives up (returns false) when
// `abort` is set, an error is recorded, or after limit_ns.  The first test is
// inline; the spin loop is one out-of-line copy for every call site (the
// kernel's code per layer is kept small: it is fetched again every layer).
static __device__ __noinline__ bool mbar_wait_loop(uint64_t* b, uint32_t parity, const volatile int* abort, int32_t* err,
                                            uint64_t limit_ns, int site_detail) {
  WaitClock wc;
  wc.start();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(b, parity)) return true;
    if ((i & 3u) == 0) {
      if (*abort) return false;
      const int r = wc.check(err, limit_ns);
      if (r == 1) return false;
      if (r == 2) {
        set_error(err, MK_ERR_BARRIER_TIMEOUT, SITE_RING, site_detail);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, const volatile int* abort,
                                          int32_t* err, uint64_t limit_ns, int site_detail) {
  if (mbar_try(b, parity)) return true;
  return mbar_wait_loop(b, parity, abort, err, limit_ns, site_detail);
}
// Bounded wait that ignores abort and errors: used on the exit path, where
// copies still in flight into shared memory must land before the block ends.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* b, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(b, parity)) return true;
    if ((i & 15u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
}
// Global -> shared bulk copy completing on mbarrier `b` (addresses and size
// multiples of 16 bytes).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(b))
      : "memory");
}

// ------------------------------------------------------------------ GEMV engine
// A row of K weights is read as 16-byte chunks; lane l of a warp owns chunks
// l, l+32, l+64, ...  The rows come from the weight ring in shared memory; the
// activation vector is staged once per block in shared memory in the same
// chunk order, and (for short rows) each warp keeps the chunks of its lanes in
// registers, so a row costs one pass over its bytes.
//
// int4 weights: chunk = 32 codes.  The activation chunk is held as 24-bit
// fixed point (scale max|y| / (2^23 - 1), float32 precision) in three byte
// planes: low and middle bytes unsigned, high byte signed.  Each plane's dot
// product with the codes is formed exactly with dp4a (four codes per
// instruction, the codes read as q + 8 and corrected with the plane sum), the
// planes combine as 65536 * high + 256 * middle + low, and each chunk's dot
// is scaled to float32 (group scale x activation scale) and accumulated in
// float32.  bf16 / fp32 weights: chunk = 8 / 4 values, float32 activations,
// float32 FMA.
//
// Staged int4 chunk: six 16-byte pieces, piece 2p + e of plane p holds, in
// word t, the plane's bytes of values 8t + {0, 2, 4, 6} (e = 0) or
// 8t + {1, 3, 5, 7} (e = 1) -- the order in which a code word splits into
// even and odd nibbles -- followed by {scale, 8 sum high, 8 sum middle,
// 8 sum low}.
__device__ __forceinline__ float int4_chunk_dot(const uint4 w4, const uint4 (&p)[6], const int4 m) {
  const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
  const uint32_t p0[4] = {p[0].x, p[0].y, p[0].z, p[0].w}, p1[4] = {p[1].x, p[1].y, p[1].z, p[1].w};
  const uint32_t p2[4] = {p[2].x, p[2].y, p[2].z, p[2].w}, p3[4] = {p[3].x, p[3].y, p[3].z, p[3].w};
  const uint32_t p4[4] = {p[4].x, p[4].y, p[4].z, p[4].w}, p5[4] = {p[5].x, p[5].y, p[5].z, p[5].w};
  uint32_t d0 = 0, d1 = 0;
  int d2 = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t x = wv[t] ^ 0x88888888u;      // two's complement -> q + 8
    const uint32_t be = x & 0x0F0F0F0Fu;          // codes of values 8t + 0, 2, 4, 6
    const uint32_t bo = (x >> 4) & 0x0F0F0F0Fu;   // codes of values 8t + 1, 3, 5, 7
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(d0) : "r"(p0[t]), "r"(be));
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(d0) : "r"(p1[t]), "r"(bo));
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(d1) : "r"(p2[t]), "r"(be));
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(d1) : "r"(p3[t]), "r"(bo));
    asm("dp4a.s32.u32 %0, %1, %2, %0;" : "+r"(d2) : "r"(p4[t]), "r"(be));
    asm("dp4a.s32.u32 %0, %1, %2, %0;" : "+r"(d2) : "r"(p5[t]), "r"(bo));
  }
  // sum y (q + 8) - 8 sum y = sum y q per plane, exactly in int32
  const int lowmid = ((int)d1 - m.z) * 256 + ((int)d0 - m.w);
  return fmaf((float)(d2 - m.y), 65536.f, (float)lowmid);
}

// int3 weights: chunk = 32 codes in 12 bytes of a row's two planes.  The
// row's low plane holds, per chunk, two words L0, L1 of 2-bit fields; its
// high plane one word Hh of 1-bit fields.  Value 8t + 2i + e of the chunk
// (t = 0..3, i = 0..3, e = 0..1, as in the staged activation's pieces) has
// the offset code u = q + 4 in [0, 7]: its low two bits in byte i of
// L[t / 2] at bit 2 (2 (t % 2) + e), its high bit in byte i of Hh at bit
// 2t + e.  So one shift and mask of each plane gives the four codes of a
// staged activation word, and the dot product is formed with dp4a as for
// int4, corrected with 4 (not 8) times the plane sums.
__device__ __forceinline__ float int3_chunk_dot(const uint4 w, const uint4 (&p)[6], const int4 m) {
  const uint32_t L[2] = {w.x, w.y}, hh = w.z;
  const uint32_t p0[4] = {p[0].x, p[0].y, p[0].z, p[0].w}, p1[4] = {p[1].x, p[1].y, p[1].z, p[1].w};
  const uint32_t p2[4] = {p[2].x, p[2].y, p[2].z, p[2].w}, p3[4] = {p[3].x, p[3].y, p[3].z, p[3].w};
  const uint32_t p4[4] = {p[4].x, p[4].y, p[4].z, p[4].w}, p5[4] = {p[5].x, p[5].y, p[5].z, p[5].w};
  uint32_t d0 = 0, d1 = 0;
  int d2 = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    uint32_t u[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int fl = 2 * (2 * (t & 1) + e), fh = 2 * t + e;
      const uint32_t hi = fh >= 2 ? (hh >> (fh - 2)) : (hh << (2 - fh));
      u[e] = ((L[t >> 1] >> fl) & 0x03030303u) | (hi & 0x04040404u);
    }
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(d0) : "r"(p0[t]), "r"(u[0]));
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(d0) : "r"(p1[t]), "r"(u[1]));
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(d1) : "r"(p2[t]), "r"(u[0]));
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(d1) : "r"(p3[t]), "r"(u[1]));
    asm("dp4a.s32.u32 %0, %1, %2, %0;" : "+r"(d2) : "r"(p4[t]), "r"(u[0]));
    asm("dp4a.s32.u32 %0, %1, %2, %0;" : "+r"(d2) : "r"(p5[t]), "r"(u[1]));
  }
  // sum y (q + 4) - 4 sum y = sum y q per plane (the metadata holds 8 sum y)
  const int lowmid = ((int)d1 - (m.z >> 1)) * 256 + ((int)d0 - (m.w >> 1));
  return fmaf((float)(d2 - (m.y >> 1)), 65536.f, (float)lowmid);
}

template <int WDT, int K>
struct Gemv {
  // int4 and int3 rows share the 32-value chunk and the staged fixed-point
  // activation (a model with int3 experts stages one form for both)
  static constexpr bool QNT = WDT == WINT4 || WDT == WINT3;
  static constexpr int VPC = QNT ? 32 : (WDT == WBF16 ? 8 : 4);
  static constexpr int NCH = K / VPC;
  static constexpr int CPL = (NCH + 31) / 32;
  static constexpr int SUBS = QNT ? 6 : VPC / 4;  // 16-byte pieces of a staged chunk
  static constexpr int META = QNT ? 16 : 0;
  static constexpr int ACT_BYTES = NCH * SUBS * 16 + NCH * META;
  static constexpr int ROW_BYTES = WDT == WINT4 ? K / 2 : (WDT == WINT3 ? 3 * K / 8 : (WDT == WBF16 ? 2 * K : 4 * K));
  static constexpr int SCALE_BYTES = QNT ? K / 64 * 2 : 0;
  // rows per aligned group: A rows of scales are a multiple of 16 bytes
  static constexpr int A = SCALE_BYTES == 0 ? 1
                         : (SCALE_BYTES % 16 == 0 ? 1 : (SCALE_BYTES % 8 == 0 ? 2 : (SCALE_BYTES % 4 == 0 ? 4 : 8)));
  // short rows may keep the activation chunks in registers (worth it when a
  // warp dots many rows with one activation); otherwise they are read from
  // shared memory per chunk
  static constexpr bool ACT_REGS = CPL <= 2;
  static constexpr int AR = ACT_REGS ? CPL : 1;
  static_assert(K % VPC == 0, "K must be a multiple of the chunk");
  static_assert(!QNT || K % 64 == 0, "int4 / int3 rows are whole scale groups");
  static_assert(ACT_BYTES % 16 == 0 && ROW_BYTES % 16 == 0, "16-byte aligned rows and vectors");

  struct Act {
    uint4 v[AR][SUBS];
    int4 m[AR];
  };

  __device__ static __forceinline__ void load_act(Act& a, const uint8_t* base, int lane) {
    if constexpr (ACT_REGS) {
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = lane + 32 * j;
        if (NCH % 32 == 0 || c < NCH) {
#pragma unroll
          for (int t = 0; t < SUBS; ++t) a.v[j][t] = lds128(base + (t * NCH + c) * 16);
          if constexpr (QNT) {
            const uint4 m = lds128(base + NCH * SUBS * 16 + c * 16);
            a.m[j] = make_int4((int)m.x, (int)m.y, (int)m.z, (int)m.w);
          }
        }
      }
    }
  }

  // lane-partial dot product of one weight chunk (16 bytes, group scale sc)
  // with an activation chunk (pieces p, int4 metadata m)
  __device__ static __forceinline__ float chunk(const uint4 w, float sc, const uint4 (&p)[SUBS], const int4 m,
                                                float acc) {
    if constexpr (WDT == WINT4) {
      return fmaf(int4_chunk_dot(w, p, m), __int_as_float(m.x) * sc, acc);
    } else if constexpr (WDT == WINT3) {
      return fmaf(int3_chunk_dot(w, p, m), __int_as_float(m.x) * sc, acc);
    } else if constexpr (WDT == WBF16) {
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
      const float av[8] = {__uint_as_float(p[0].x), __uint_as_float(p[0].y), __uint_as_float(p[0].z),
                           __uint_as_float(p[0].w), __uint_as_float(p[1].x), __uint_as_float(p[1].y),
                           __uint_as_float(p[1].z), __uint_as_float(p[1].w)};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        acc = fmaf(__uint_as_float(wv[t] << 16), av[2 * t], acc);
        acc = fmaf(__uint_as_float(wv[t] & 0xFFFF0000u), av[2 * t + 1], acc);
      }
      return acc;
    } else {
      acc = fmaf(__uint_as_float(w.x), __uint_as_float(p[0].x), acc);
      acc = fmaf(__uint_as_float(w.y), __uint_as_float(p[0].y), acc);
      acc = fmaf(__uint_as_float(w.z), __uint_as_float(p[0].z), acc);
      acc = fmaf(__uint_as_float(w.w), __uint_as_float(p[0].w), acc);
      return acc;
    }
  }

  // Full dot products (warp-reduced, in every lane) of RP rows (codes at
  // w[r], scales at s[r], shared memory) with one staged activation: from
  // registers (REGS, after load_act) or read chunk by chunk from shared
  // memory at `base`.  Each weight chunk is read where it is used.
  template <int RP, bool REGS>
  __device__ static __forceinline__ void dots(const uint8_t* const (&w)[2], const uint8_t* const (&s)[2],
                                              const Act& a, const uint8_t* base, int lane, float& v0,
                                              float& v1) {
    static_assert(!REGS || ACT_REGS, "activation registers only for short rows");
    float acc[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      if (NCH % 32 == 0 || c < NCH) {
        uint4 wv[2];
        float sc[2] = {1.f, 1.f};
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          if constexpr (WDT == WINT3) {
            const uint2 lo = lds64(w[r] + 8 * c);
            wv[r] = make_uint4(lo.x, lo.y, lds32(w[r] + 8 * NCH + 4 * c), 0u);
          } else {
            wv[r] = lds128(w[r] + 16 * c);
          }
          if constexpr (QNT) sc[r] = bf16_to_f(lds16(s[r] + 2 * (c >> 1)));
        }
        if constexpr (REGS) {
#pragma unroll
          for (int r = 0; r < RP; ++r) acc[r] = chunk(wv[r], sc[r], a.v[j], a.m[j], acc[r]);
        } else {
          uint4 p[SUBS];
#pragma unroll
          for (int t = 0; t < SUBS; ++t) p[t] = lds128(base + (t * NCH + c) * 16);
          int4 m = make_int4(0, 0, 0, 0);
          if constexpr (QNT) {
            const uint4 mm = lds128(base + NCH * SUBS * 16 + c * 16);
            m = make_int4((int)mm.x, (int)mm.y, (int)mm.z, (int)mm.w);
          }
#pragma unroll
          for (int r = 0; r < RP; ++r) acc[r] = chunk(wv[r], sc[r], p, m, acc[r]);
        }
      }
    }
    v0 = warp_sum(acc[0]);
    v1 = RP > 1 ? warp_sum(acc[1]) : 0.f;
  }
};

// Block-cooperative staging (the compute warps) of `rows` activation
// vectors of K floats into the staged form of Gemv<WDT, K> (vector r at
// dst + r * ACT_BYTES).  A thread takes one 8-value word of a vector (two
// float4, coalesced: the block reads each vector as one contiguous stream)
// and, with norm, the matching norm weights in the same round trip;
// optionally RMS-normalises the row (block reduction in a fixed order, so
// every block gets the same scale), then writes its part of the staged
// chunk.  For int4 the 4 threads holding one 32-value chunk agree on its
// scale and plane sums with shuffles.
//   LD(row, f4) -> float4 values 4*f4 .. 4*f4+3 of vector `row`
//   WT(f4)      -> float4 weights (only with norm)
//   red         -> shared scratch of kWarps * 4 floats
//   rscale      -> if non-null, receives each row's RMS scale (shared memory)
// Row stride of the plain fp32 staging used by the tensor-core path (16
// bytes of padding keep the rows of 8 columns on distinct banks).
__host__ __device__ constexpr int plain_stride(int K) { return K * 4 + 16; }

template <int WDT, int K, bool NORM, int RG, bool PLAIN, class LD, class WT>
__device__ __forceinline__ void stage_rows(uint8_t* dst, int rows, LD ld, float eps, WT wt, float* red,
                                           float* rscale) {
  using Gv = Gemv<WDT, K>;
  constexpr int NW = K / 8;                      // 8-value words per vector
  static_assert(K % 32 == 0, "vectors are whole chunks");
  const bool norm = NORM;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int PER = (RG * NW + kThreads - 1) / kThreads;  // RG rows per pass
  for (int r0 = 0; r0 < rows; r0 += RG) {
    const int nrg = min(RG, rows - r0);
    float4 va[PER], vb[PER], wa[NORM ? PER : 1], wb[NORM ? PER : 1];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int it = tid + i * kThreads;
      if (it < nrg * NW) {
        const int row = it / NW, w = it % NW;
        va[i] = ld(r0 + row, 2 * w);
        vb[i] = ld(r0 + row, 2 * w + 1);
        if constexpr (NORM) {
          wa[i] = wt(2 * w);
          wb[i] = wt(2 * w + 1);
        }
      }
    }
    float rs[RG];
#pragma unroll
    for (int g = 0; g < RG; ++g) rs[g] = 1.f;
    if (norm) {
      float ss[RG];
#pragma unroll
      for (int g = 0; g < RG; ++g) ss[g] = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int it = tid + i * kThreads;
        if (it < nrg * NW) {
          const float q = va[i].x * va[i].x + va[i].y * va[i].y + va[i].z * va[i].z + va[i].w * va[i].w +
                          vb[i].x * vb[i].x + vb[i].y * vb[i].y + vb[i].z * vb[i].z + vb[i].w * vb[i].w;
#pragma unroll
          for (int g = 0; g < RG; ++g) ss[g] += (it / NW == g) ? q : 0.f;
        }
      }
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        ss[g] = warp_sum(ss[g]);
        if (lane == 0) red[wid * RG + g] = ss[g];
      }
      csync();
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        float t = 0.f;
        for (int w = 0; w < kWarps; ++w) t += red[w * RG + g];
        rs[g] = rsqrtf(t / K + eps);
      }
      if (rscale && tid < nrg) rscale[r0 + tid] = rs[tid];
      csync();
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int it = tid + i * kThreads;
      // int4 chunks span 4 consecutive threads, so the whole warp takes part
      // in the shuffles; threads past the end are predicated off (no
      // continue: the loop stays unrolled and the arrays stay in registers)
      const bool live = it < nrg * NW;
      const bool warp_live = (WDT == WINT4 && !PLAIN) ? __any_sync(0xffffffffu, live) : live;
      if (warp_live) {
        const int row = live ? it / NW : 0, w = live ? it % NW : 0;
        float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (live) {
          float r = rs[0];
#pragma unroll
          for (int g = 1; g < RG; ++g) r = row == g ? rs[g] : r;
          float4 ma = make_float4(1.f, 1.f, 1.f, 1.f), mb = ma;
          if constexpr (NORM) {
            ma = make_float4(r * wa[i].x, r * wa[i].y, r * wa[i].z, r * wa[i].w);
            mb = make_float4(r * wb[i].x, r * wb[i].y, r * wb[i].z, r * wb[i].w);
          }
          y[0] = va[i].x * ma.x; y[1] = va[i].y * ma.y; y[2] = va[i].z * ma.z; y[3] = va[i].w * ma.w;
          y[4] = vb[i].x * mb.x; y[5] = vb[i].y * mb.y; y[6] = vb[i].z * mb.z; y[7] = vb[i].w * mb.w;
        }
        uint8_t* base = dst + (r0 + row) * (PLAIN ? plain_stride(K) : Gv::ACT_BYTES);
        if constexpr (PLAIN) {
          if (live) {
            *reinterpret_cast<float4*>(base + 32 * w) = make_float4(y[0], y[1], y[2], y[3]);
            *reinterpret_cast<float4*>(base + 32 * w + 16) = make_float4(y[4], y[5], y[6], y[7]);
          }
        } else if constexpr (WDT == WINT4) {
          // chunk c = w / 4 (32 values) lives in threads 4j .. 4j+3; word t of
          // the chunk holds values 8t .. 8t+7
          float amax = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(y[e]));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          // 24-bit fixed point, |q| <= 2^23 - 1, split into byte planes
          const float inv = amax > 0.f ? __fdividef(8388607.f, amax) : 0.f;
          int q[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) q[e] = max(-8388607, min(8388607, __float2int_rn(y[e] * inv)));
          int s01 = 0, s2 = 0;  // low + (middle << 16), high
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            s01 += (q[e] & 0xFF) + (((q[e] >> 8) & 0xFF) << 16);
            s2 += q[e] >> 16;
          }
          s01 += __shfl_xor_sync(0xffffffffu, s01, 1);
          s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
          s01 += __shfl_xor_sync(0xffffffffu, s01, 2);
          s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
          const int c = w >> 2, t = w & 3;
          if (live) {
#pragma unroll
            for (int pl = 0; pl < 3; ++pl) {
              uint32_t b[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) b[e] = (uint32_t)(q[e] >> (8 * pl)) & 0xFFu;
              const uint32_t ev = b[0] | (b[2] << 8) | (b[4] << 16) | (b[6] << 24);
              const uint32_t od = b[1] | (b[3] << 8) | (b[5] << 16) | (b[7] << 24);
              *reinterpret_cast<uint32_t*>(base + ((2 * pl) * Gv::NCH + c) * 16 + 4 * t) = ev;
              *reinterpret_cast<uint32_t*>(base + ((2 * pl + 1) * Gv::NCH + c) * 16 + 4 * t) = od;
            }
            if (t == 0)
              *reinterpret_cast<int4*>(base + Gv::NCH * Gv::SUBS * 16 + c * 16) =
                  make_int4(__float_as_int(amax * (1.f / 8388607.f)), 8 * s2, 8 * (s01 >> 16), 8 * (s01 & 0xFFFF));
          }
        } else if (live) {
          // chunk c holds VPC values = VPC/4 float4; sub t of chunk c at (t*NCH + c)*16
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int f4 = 2 * w + h;
            const int c = f4 / (Gv::VPC / 4), t = f4 % (Gv::VPC / 4);
            *reinterpret_cast<float4*>(base + (t * Gv::NCH + c) * 16) =
                make_float4(y[4 * h], y[4 * h + 1], y[4 * h + 2], y[4 * h + 3]);
          }
        }
      }
    }
  }
}

// Staging entry.  MODE 2: the plain fp32 rows of the tensor-core path;
// otherwise the GEMV engine's staged form, MODE 0 one row per pass (fewest
// registers), MODE 1 several rows per pass: four with a norm (one load round
// trip and one norm reduction for four rows), as many as two words per
// thread cover without one.  The mode is a template argument so that a
// staging function holds one variant and its registers are allocated for it
// alone.
template <int MODE, int WDT, int K, bool NORM, class LD, class WT>
__device__ __forceinline__ void stage_block(uint8_t* dst, int rows, LD ld, float eps, WT wt, float* red,
                                            float* rscale) {
  constexpr int RGM = NORM ? 4 : ((2 * kThreads) / (K / 8) > 1 ? (2 * kThreads) / (K / 8) : 1);
  if constexpr (MODE == 2) stage_rows<WDT, K, NORM, RGM, true>(dst, rows, ld, eps, wt, red, rscale);
  else if constexpr (MODE == 0) stage_rows<WDT, K, NORM, 1, false>(dst, rows, ld, eps, wt, red, rscale);
  else stage_rows<WDT, K, NORM, RGM, false>(dst, rows, ld, eps, wt, red, rscale);
}

// Plain fp32 rows for the tensor-core path (rows of `ld` floats at src),
// staged with one round of 16-byte asynchronous copies: the plain layout is
// the rows' own values plus padding, so the bytes land as they are, in one L2
// round trip for all rows.  With NORM they are then RMS-normalised in place:
// one warp per row sums the squares in a fixed order (every block gets the
// same scale), then every value is multiplied by scale x norm weight.
// red: shared scratch of at least `rows` floats; rscale as in stage_rows.
template <int AUX, int K, bool NORM>
__device__ __forceinline__ void stage_plain_async(uint8_t* dst, int rows, const float* src, int ld, float eps,
                                                  const void* w, float* red, float* rscale) {
  constexpr int C4 = K / 4;  // 16-byte pieces of a row
  constexpr int PS = plain_stride(K);
  static_assert(K % 4 == 0, "whole 16-byte pieces");
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int idx = tid; idx < rows * C4; idx += kThreads) {
    const int r = idx / C4, c = idx % C4;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + r * PS + 16 * c)),
                 "l"(src + (size_t)r * ld + 4 * c)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  csync();
  if constexpr (NORM) {
    for (int r = wid; r < rows; r += kWarps) {
      float s = 0.f;
      for (int c = lane; c < C4; c += 32) {
        const float4 v = *reinterpret_cast<const float4*>(dst + r * PS + 16 * c);
        s += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
      s = warp_sum(s);
      if (lane == 0) {
        const float rs = rsqrtf(s / K + eps);
        red[r] = rs;
        if (rscale) rscale[r] = rs;
      }
    }
    csync();
    for (int idx = tid; idx < rows * C4; idx += kThreads) {
      const int r = idx / C4, c = idx % C4;
      float4* p = reinterpret_cast<float4*>(dst + r * PS + 16 * c);
      const float4 v = *p, wv = ld_aux4<AUX>(w, c);
      const float rs = red[r];
      *p = make_float4(v.x * (rs * wv.x), v.y * (rs * wv.y), v.z * (rs * wv.z), v.w * (rs * wv.w));
    }
    csync();
  }
}

__device__ __forceinline__ void split_range(int n, int parts, int idx, int& lo, int& hi) {
  lo = (int)(((long long)n * idx) / parts);
  hi = (int)(((long long)n * (idx + 1)) / parts);
}

}  // namespace mk
