// Device building blocks of the decode megakernel: memory access helpers,
// the grid barrier, activation staging and the warp-level GEMV engine.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include "mk_internal.h"

namespace mk {

enum { WF32 = 0, WBF16 = 1, WINT4 = 2 };

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
__device__ __forceinline__ uint4 ld_weight16(const void* p) {
  // weights are read-only for the launch and read once: no L1 allocation
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ld_weight2(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
// Data written by other blocks during the launch: read at L2, never from a
// (non-coherent) L1 line.
__device__ __forceinline__ float ld_shared_f(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ld_shared_f4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ int ld_shared_i(const int* p) { return __ldcg(p); }

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  // bulk L2 prefetch (TMA unit); addresses and sizes rounded to 16 bytes
  uintptr_t a = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15);
  uintptr_t e = (reinterpret_cast<uintptr_t>(p) + bytes + 15) & ~uintptr_t(15);
  while (a < e) {
    const uintptr_t left = e - a;
    uint32_t n = (uint32_t)(left < 32768 ? left : 32768);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(n) : "memory");
    a += n;
  }
}

// L2 warm-up of a byte range by the whole block: each thread requests every
// kThreads-th 128-byte line (cheap to issue, no registers held).
__device__ __forceinline__ void prefetch_l2_block(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(127);
  const uintptr_t e = reinterpret_cast<uintptr_t>(p) + bytes;
  for (uintptr_t q = a + (uintptr_t)threadIdx.x * 128; q < e; q += (uintptr_t)kThreads * 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
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

// ------------------------------------------------------------------ grid barrier
// One monotonically increasing arrival counter per launch: barrier k of the
// launch completes when the counter reaches k * gridDim.x.  The arrive is a
// release reduction, the wait an acquire load, so every write before the
// barrier is visible to every block after it.  The wait is bounded: it gives
// up when another block has recorded an error, or after spin_limit_ns, and
// then records MK_ERR_BARRIER_TIMEOUT; the caller skips to the exit path.
__device__ __forceinline__ bool grid_barrier(const StepArgs& a, uint32_t& k) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    ++k;
    uint32_t* ctr = a.sc.sync;
    bool skip = (a.dbg_flags & MK_DBG_SKIP_ARRIVAL) && (a.dbg_arg >> 16) == k &&
                (a.dbg_arg & 0xffffu) == blockIdx.x;
    if (!skip) {
      __threadfence();
      asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(1u) : "memory");
    }
    const uint32_t target = k * gridDim.x;
    int ok = 1;
    uint64_t t0 = 0;
    for (uint32_t spins = 0;; ++spins) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if ((spins & 31u) == 0) {
        if (*(volatile int32_t*)a.sc.err != 0) { ok = 0; break; }
        uint64_t now = globaltimer();
        if (spins == 0) t0 = now;
        else if (now - t0 > a.spin_limit_ns) {
          set_error(a.sc.err, MK_ERR_BARRIER_TIMEOUT, SITE_BARRIER, (int)k);
          ok = 0;
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// ------------------------------------------------------------------ GEMV engine
// A row of K weights is read as 16-byte chunks; lane l of a warp owns chunks
// l, l+32, l+64, ...  (coalesced: each warp load instruction reads 512
// contiguous bytes of the row).  The activation vector is staged once per
// block in shared memory in the same chunk order, and each warp holds the
// chunks of its lanes in registers, so a row costs one pass over its bytes.
//
// int4 weights: chunk = 32 codes.  The activation chunk is held as 30-bit
// fixed point (scale max|y| / 2^30, i.e. float32 precision), split into a
// signed high half and an unsigned low half of 16 bits each; the products
// with the 4-bit codes are formed exactly with dp2a (two halves x two codes
// per instruction, two passes) in int32, combined as 65536 * high + low, and
// each chunk's dot is scaled to float32 (weight scale x activation scale) and
// accumulated in float32.  bf16 / fp32 weights: chunk = 8 / 4 values, float32
// activations, float32 FMA.
// Dot product of one 16-byte chunk of int4 codes (32 values) with a staged
// activation chunk: pieces p[0..3] hold the high halves, p[4..7] the low
// halves, each as (0,2) (4,6) (1,3) (5,7) pairs of every 8-value word.
// Returns sum_k y_k * q_k in units of the activation scale (exact integer
// parts, one float rounding at the end).
__device__ __forceinline__ float int4_chunk_dot(const uint4 w4, const uint4* p, int ch, int cl) {
  const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
  int ih = 0;
  uint32_t il = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t x = wv[t] ^ 0x88888888u;      // two's complement -> q + 8
    const uint32_t be = x & 0x0F0F0F0Fu;          // codes of k+0, k+2, k+4, k+6
    const uint32_t bo = (x >> 4) & 0x0F0F0F0Fu;   // codes of k+1, k+3, k+5, k+7
    const uint32_t h[4] = {p[t].x, p[t].y, p[t].z, p[t].w};
    const uint32_t lo[4] = {p[4 + t].x, p[4 + t].y, p[4 + t].z, p[4 + t].w};
    asm("dp2a.lo.s32.u32 %0, %1, %2, %0;" : "+r"(ih) : "r"(h[0]), "r"(be));
    asm("dp2a.hi.s32.u32 %0, %1, %2, %0;" : "+r"(ih) : "r"(h[1]), "r"(be));
    asm("dp2a.lo.s32.u32 %0, %1, %2, %0;" : "+r"(ih) : "r"(h[2]), "r"(bo));
    asm("dp2a.hi.s32.u32 %0, %1, %2, %0;" : "+r"(ih) : "r"(h[3]), "r"(bo));
    asm("dp2a.lo.u32.u32 %0, %1, %2, %0;" : "+r"(il) : "r"(lo[0]), "r"(be));
    asm("dp2a.hi.u32.u32 %0, %1, %2, %0;" : "+r"(il) : "r"(lo[1]), "r"(be));
    asm("dp2a.lo.u32.u32 %0, %1, %2, %0;" : "+r"(il) : "r"(lo[2]), "r"(bo));
    asm("dp2a.hi.u32.u32 %0, %1, %2, %0;" : "+r"(il) : "r"(lo[3]), "r"(bo));
  }
  // sum y (q + 8) - 8 sum y = sum y q, per half, exactly in int32
  return fmaf((float)(ih - ch), 65536.f, (float)((int)il - cl));
}

template <int WDT, int K>
struct Gemv {
  static constexpr int VPC = WDT == WINT4 ? 32 : (WDT == WBF16 ? 8 : 4);
  static constexpr int NCH = K / VPC;
  static constexpr int CPL = (NCH + 31) / 32;
  static constexpr int SUBS = WDT == WINT4 ? 8 : VPC / 4;  // 16-byte pieces of a staged chunk
  // int4 chunk metadata: activation scale, 8 * sum of high halves, 8 * sum of
  // low halves (the nibbles are read as q + 8), padding
  static constexpr int META = WDT == WINT4 ? 16 : 0;
  static constexpr int ACT_BYTES = NCH * SUBS * 16 + NCH * META;
  static constexpr int ROW_BYTES = WDT == WINT4 ? K / 2 : (WDT == WBF16 ? 2 * K : 4 * K);
  static constexpr bool PIPE = CPL <= 2;  // registers allow loading the next task early
  // int4 (and short rows) keep the activation in registers; long bf16/fp32
  // rows read the staged chunk from shared memory per row instead (2 bytes
  // of shared memory per weight byte, well inside its bandwidth)
  static constexpr bool ACT_REGS = WDT == WINT4 || CPL <= 2;
  static constexpr int AR = ACT_REGS ? CPL : 1;
  static_assert(K % VPC == 0, "K must be a multiple of the chunk");
  static_assert(ACT_BYTES % 16 == 0, "staged vectors stay 16-byte aligned");

  struct Act {
    uint4 v[AR][SUBS];
    float s[AR];
    int ch[AR], cl[AR];
    const uint8_t* base;
  };
  struct Row {
    uint4 w[CPL];
    float s[CPL];
  };

  __device__ static __forceinline__ void load_row(Row& r, const uint8_t* w, const uint16_t* s,
                                                  int lane) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      if (NCH % 32 == 0 || c < NCH) {
        r.w[j] = ld_weight16(w + 16 * c);
        if constexpr (WDT == WINT4) r.s[j] = bf16_to_f(ld_weight2(s + (c >> 1)));
      }
    }
  }

  __device__ static __forceinline__ void load_act(Act& a, const uint8_t* base, int lane) {
    a.base = base;
    if constexpr (ACT_REGS) {
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = lane + 32 * j;
        if (NCH % 32 == 0 || c < NCH) {
#pragma unroll
          for (int t = 0; t < SUBS; ++t)
            a.v[j][t] = *reinterpret_cast<const uint4*>(base + (t * NCH + c) * 16);
          if constexpr (WDT == WINT4) {
            const int4 m = *reinterpret_cast<const int4*>(base + NCH * SUBS * 16 + c * 16);
            a.s[j] = __int_as_float(m.x);
            a.ch[j] = m.y;
            a.cl[j] = m.z;
          }
        }
      }
    }
  }

  __device__ static __forceinline__ uint4 act_piece(const Act& a, int j, int t, int c) {
    if constexpr (ACT_REGS) return a.v[j][t];
    else return *reinterpret_cast<const uint4*>(a.base + (t * NCH + c) * 16);
  }

  // lane-partial dot product (sum over the lane's chunks)
  __device__ static __forceinline__ float dot(const Row& r, const Act& a, int lane) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      if (NCH % 32 == 0 || c < NCH) {
        if constexpr (WDT == WINT4) {
          acc = fmaf(int4_chunk_dot(r.w[j], a.v[j], a.ch[j], a.cl[j]), a.s[j] * r.s[j], acc);
        } else if constexpr (WDT == WBF16) {
          const uint32_t wv[4] = {r.w[j].x, r.w[j].y, r.w[j].z, r.w[j].w};
          const uint4 a0 = act_piece(a, j, 0, c), a1 = act_piece(a, j, 1, c);
          const float av[8] = {__uint_as_float(a0.x), __uint_as_float(a0.y), __uint_as_float(a0.z),
                               __uint_as_float(a0.w), __uint_as_float(a1.x), __uint_as_float(a1.y),
                               __uint_as_float(a1.z), __uint_as_float(a1.w)};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            acc = fmaf(__uint_as_float(wv[t] << 16), av[2 * t], acc);
            acc = fmaf(__uint_as_float(wv[t] & 0xFFFF0000u), av[2 * t + 1], acc);
          }
        } else {
          const uint4 a0 = act_piece(a, j, 0, c);
          acc = fmaf(__uint_as_float(r.w[j].x), __uint_as_float(a0.x), acc);
          acc = fmaf(__uint_as_float(r.w[j].y), __uint_as_float(a0.y), acc);
          acc = fmaf(__uint_as_float(r.w[j].z), __uint_as_float(a0.z), acc);
          acc = fmaf(__uint_as_float(r.w[j].w), __uint_as_float(a0.w), acc);
        }
      }
    }
    return acc;
  }

  // Dot products of two rows with one staged activation, the activation read
  // chunk by chunk from shared memory (fewer live registers than load_act).
  __device__ static __forceinline__ void dot2_smem(const Row& r0, const Row& r1, const uint8_t* base,
                                                   int lane, float& v0, float& v1) {
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      if (NCH % 32 == 0 || c < NCH) {
        if constexpr (WDT == WINT4) {
          uint4 p[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) p[t] = *reinterpret_cast<const uint4*>(base + (t * NCH + c) * 16);
          const int4 m = *reinterpret_cast<const int4*>(base + NCH * SUBS * 16 + c * 16);
          const float sa = __int_as_float(m.x);
          acc0 = fmaf(int4_chunk_dot(r0.w[j], p, m.y, m.z), sa * r0.s[j], acc0);
          acc1 = fmaf(int4_chunk_dot(r1.w[j], p, m.y, m.z), sa * r1.s[j], acc1);
        } else {
#pragma unroll
          for (int t = 0; t < SUBS; ++t) {
            const uint4 ap = *reinterpret_cast<const uint4*>(base + (t * NCH + c) * 16);
            const float av[4] = {__uint_as_float(ap.x), __uint_as_float(ap.y), __uint_as_float(ap.z),
                                 __uint_as_float(ap.w)};
            if constexpr (WDT == WBF16) {
              const uint32_t a0 = t == 0 ? r0.w[j].x : r0.w[j].z, b0 = t == 0 ? r0.w[j].y : r0.w[j].w;
              const uint32_t a1 = t == 0 ? r1.w[j].x : r1.w[j].z, b1 = t == 0 ? r1.w[j].y : r1.w[j].w;
              acc0 = fmaf(__uint_as_float(a0 << 16), av[0], acc0);
              acc0 = fmaf(__uint_as_float(a0 & 0xFFFF0000u), av[1], acc0);
              acc0 = fmaf(__uint_as_float(b0 << 16), av[2], acc0);
              acc0 = fmaf(__uint_as_float(b0 & 0xFFFF0000u), av[3], acc0);
              acc1 = fmaf(__uint_as_float(a1 << 16), av[0], acc1);
              acc1 = fmaf(__uint_as_float(a1 & 0xFFFF0000u), av[1], acc1);
              acc1 = fmaf(__uint_as_float(b1 << 16), av[2], acc1);
              acc1 = fmaf(__uint_as_float(b1 & 0xFFFF0000u), av[3], acc1);
            } else {
              acc0 = fmaf(__uint_as_float(r0.w[j].x), av[0], acc0);
              acc0 = fmaf(__uint_as_float(r0.w[j].y), av[1], acc0);
              acc0 = fmaf(__uint_as_float(r0.w[j].z), av[2], acc0);
              acc0 = fmaf(__uint_as_float(r0.w[j].w), av[3], acc0);
              acc1 = fmaf(__uint_as_float(r1.w[j].x), av[0], acc1);
              acc1 = fmaf(__uint_as_float(r1.w[j].y), av[1], acc1);
              acc1 = fmaf(__uint_as_float(r1.w[j].z), av[2], acc1);
              acc1 = fmaf(__uint_as_float(r1.w[j].w), av[3], acc1);
            }
          }
        }
      }
    }
    v0 = warp_sum(acc0);
    v1 = warp_sum(acc1);
  }

};

// Block-cooperative staging of `rows` activation vectors of K floats into the
// staged form of Gemv<WDT, K> (vector r at dst + r * ACT_BYTES).  Thread t
// loads float4 number t (coalesced: the block reads each vector as one
// contiguous stream), optionally RMS-normalises the row (block reduction in a
// fixed order, so every block gets the same scale) and multiplies by a
// weight, then writes its part of the staged chunk; for int4 the 8 lanes
// holding one 32-value chunk agree on its scale with shuffles.
//   LD(row, f4) -> float4 values 4*f4 .. 4*f4+3 of vector `row`
//   WT(f4)      -> float4 weights (only with norm)
//   red         -> shared scratch of kWarps * 4 floats
//   rscale      -> if non-null, receives each row's RMS scale (shared memory)
template <int WDT, int K, class LD, class WT>
__device__ __forceinline__ void stage_block(uint8_t* dst, int rows, LD ld, bool norm, float eps, WT wt,
                                            float* red, float* rscale) {
  using Gv = Gemv<WDT, K>;
  constexpr int NF4 = K / 4;
  static_assert(K % 32 == 0, "vectors are whole chunks");
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int RG = 4;                          // rows per pass
  constexpr int PER = (RG * NF4 + kThreads - 1) / kThreads;
  for (int r0 = 0; r0 < rows; r0 += RG) {
    const int nrg = min(RG, rows - r0);
    float4 v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int it = tid + i * kThreads;
      if (it < nrg * NF4) v[i] = ld(r0 + it / NF4, it % NF4);
    }
    float rs[RG] = {1.f, 1.f, 1.f, 1.f};
    if (norm) {
      float ss[RG] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int it = tid + i * kThreads;
        if (it < nrg * NF4) {
          const float q = v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
#pragma unroll
          for (int g = 0; g < RG; ++g) ss[g] += (it / NF4 == g) ? q : 0.f;
        }
      }
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        ss[g] = warp_sum(ss[g]);
        if (lane == 0) red[wid * RG + g] = ss[g];
      }
      __syncthreads();
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        float t = 0.f;
        for (int w = 0; w < kWarps; ++w) t += red[w * RG + g];
        rs[g] = rsqrtf(t / K + eps);
      }
      if (rscale && tid < nrg) rscale[r0 + tid] = rs[tid];
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int it = tid + i * kThreads;
      // int4 chunks span 8 consecutive lanes, so the whole warp takes part in
      // the shuffles; lanes past the end are predicated off (no continue: the
      // loop stays unrolled and v[] stays in registers)
      const bool live = it < nrg * NF4;
      const bool warp_live = WDT == WINT4 ? __any_sync(0xffffffffu, live) : live;
      if (warp_live) {
      const int row = live ? it / NF4 : 0, f4 = live ? it % NF4 : 0;
      float4 y = v[i];
      if (norm && live) {
        const float4 w = wt(f4);
        float r = rs[0];
#pragma unroll
        for (int g = 1; g < RG; ++g) r = row == g ? rs[g] : r;
        y = make_float4(y.x * r * w.x, y.y * r * w.y, y.z * r * w.z, y.w * r * w.w);
      }
      uint8_t* base = dst + (r0 + row) * Gv::ACT_BYTES;
      if constexpr (WDT == WINT4) {
        // chunk c = f4 / 8 (32 values) lives in lanes 8j .. 8j+7
        float amax = live ? fmaxf(fmaxf(fabsf(y.x), fabsf(y.y)), fmaxf(fabsf(y.z), fabsf(y.w))) : 0.f;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        // 30-bit fixed point: |q| <= 2^30, split q = 65536 * hi + lo
        const float inv = amax > 0.f ? 1073741824.f / amax : 0.f;
        const int q0 = __float2int_rn(y.x * inv), q1 = __float2int_rn(y.y * inv);
        const int q2 = __float2int_rn(y.z * inv), q3 = __float2int_rn(y.w * inv);
        const int h0 = q0 >> 16, h1 = q1 >> 16, h2 = q2 >> 16, h3 = q3 >> 16;
        const int l0 = q0 & 0xFFFF, l1 = q1 & 0xFFFF, l2 = q2 & 0xFFFF, l3 = q3 & 0xFFFF;
        int sh = h0 + h1 + h2 + h3, sl = l0 + l1 + l2 + l3;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          sh += __shfl_xor_sync(0xffffffffu, sh, o);
          sl += __shfl_xor_sync(0xffffffffu, sl, o);
        }
        // word group t = (f4 % 8) / 2 holds values 8t .. 8t+7 of the chunk:
        // dp2a operand order (0,2) (4,6) (1,3) (5,7); the even lane of the
        // pair holds values 0-3, the odd lane 4-7
        const uint32_t ha = (uint32_t)(h0 & 0xFFFF) | ((uint32_t)h2 << 16);
        const uint32_t hb = (uint32_t)(h1 & 0xFFFF) | ((uint32_t)h3 << 16);
        const uint32_t la = (uint32_t)l0 | ((uint32_t)l2 << 16);
        const uint32_t lb = (uint32_t)l1 | ((uint32_t)l3 << 16);
        const uint32_t oha = __shfl_xor_sync(0xffffffffu, ha, 1);
        const uint32_t ohb = __shfl_xor_sync(0xffffffffu, hb, 1);
        const uint32_t ola = __shfl_xor_sync(0xffffffffu, la, 1);
        const uint32_t olb = __shfl_xor_sync(0xffffffffu, lb, 1);
        const int c = f4 >> 3, t = (f4 & 7) >> 1;
        if (live && (f4 & 1) == 0) {
          *reinterpret_cast<uint4*>(base + (t * Gv::NCH + c) * 16) = make_uint4(ha, oha, hb, ohb);
          *reinterpret_cast<uint4*>(base + ((4 + t) * Gv::NCH + c) * 16) = make_uint4(la, ola, lb, olb);
          if (t == 0)
            *reinterpret_cast<int4*>(base + Gv::NCH * Gv::SUBS * 16 + c * 16) =
                make_int4(__float_as_int(amax * 9.3132257461547852e-10f), 8 * sh, 8 * sl, 0);
        }
      } else {
        // chunk c holds VPC values = VPC/4 float4; sub t of chunk c at (t*NCH + c)*16
        const int c = f4 / (Gv::VPC / 4), t = f4 % (Gv::VPC / 4);
        *reinterpret_cast<float4*>(base + (t * Gv::NCH + c) * 16) = y;
      }
      }
    }
  }
}

// Block-level task runner.  Tasks t = warp, warp + 16, ... ; each task has RP
// weight rows and a list of staged activations; the warp loads each row once
// and forms its dot product with every activation of the task.  A task
// object provides (all inlined, results returned by value):
//   RowRef row(t, r)        row pointers of row r of task t
//   ActRange acts(t)        activations: i-th is list ? list[start+i] : start+i
//   void out(t, ai, i, v0, v1)  results for activation ai (i-th of the task), all lanes
struct RowRef {
  const uint8_t* w;
  const uint16_t* s;
};
struct ActRange {
  const uint8_t* list;
  int start, count;
};

template <int WDT, int K, int RP, class T>
__device__ __forceinline__ void run_tasks(int ntasks, const uint8_t* act_base, const T& task) {
  using Gv = Gemv<WDT, K>;
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  typename Gv::Act a;
  int loaded = -1;
  auto prefetch_rows_l2 = [&](int tf) {
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      const RowRef rr = task.row(tf, r);
#pragma unroll
      for (int j = 0; j < Gv::CPL; ++j) {
        const int c = lane + 32 * j;
        if (Gv::NCH % 32 == 0 || c < Gv::NCH) asm volatile("prefetch.global.L2 [%0];" ::"l"(rr.w + 16 * c));
      }
    }
  };
  if constexpr (Gv::PIPE && RP == 1) {
    typename Gv::Row cur, nxt;
    int t = wid;
    if (t < ntasks) {
      const RowRef rr = task.row(t, 0);
      Gv::load_row(cur, rr.w, rr.s, lane);
    }
    for (; t < ntasks; t += kWarps) {
      const int tn = t + kWarps;
      if (tn < ntasks) {
        const RowRef rr = task.row(tn, 0);
        Gv::load_row(nxt, rr.w, rr.s, lane);
      }
      if (t + 4 * kWarps < ntasks) prefetch_rows_l2(t + 4 * kWarps);  // keep HBM busy further ahead
      const ActRange ar = task.acts(t);
      for (int i = 0; i < ar.count; ++i) {
        const int ai = ar.list ? ar.list[ar.start + i] : ar.start + i;
        if (ai != loaded) { Gv::load_act(a, act_base + ai * Gv::ACT_BYTES, lane); loaded = ai; }
        const float v0 = warp_sum(Gv::dot(cur, a, lane));
        task.out(t, ai, i, v0, 0.f);
      }
      cur = nxt;
    }
  } else {
    // activations read from shared memory per chunk: no activation registers
    // live across the task loop
    typename Gv::Row row[2];
    for (int t = wid; t < ntasks; t += kWarps) {
      if (t + kWarps < ntasks) prefetch_rows_l2(t + kWarps);  // warm L2 for this warp's next task
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const RowRef rr = task.row(t, r);
        Gv::load_row(row[r], rr.w, rr.s, lane);
      }
      if (RP == 1) row[1] = row[0];
      const ActRange ar = task.acts(t);
      for (int i = 0; i < ar.count; ++i) {
        const int ai = ar.list ? ar.list[ar.start + i] : ar.start + i;
        float v0, v1;
        Gv::dot2_smem(row[0], row[1], act_base + ai * Gv::ACT_BYTES, lane, v0, v1);
        task.out(t, ai, i, v0, v1);
      }
    }
  }
}

__device__ __forceinline__ void split_range(int n, int parts, int idx, int& lo, int& hi) {
  lo = (int)(((long long)n * idx) / parts);
  hi = (int)(((long long)n * (idx + 1)) / parts);
}

}  // namespace mk
