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

__device__ __forceinline__ float bf16_to_f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ uint16_t f_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int AUX>  // aux dtype: WF32 or WBF16
__device__ __forceinline__ float ld_aux(const void* p, int i) {
  if constexpr (AUX == WF32) return __ldg(reinterpret_cast<const float*>(p) + i);
  else return bf16_to_f(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
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
// int4 weights: chunk = 32 codes.  The activation chunk is quantised to
// int16 with its own scale (max |y| / 32767, relative error <= 1.5e-5 of the
// chunk maximum); products are formed exactly with dp2a (two int16 x two
// 4-bit codes per instruction) in int32, and each chunk's integer dot is
// scaled to float32 (weight scale x activation scale) and accumulated in
// float32.  bf16 / fp32 weights: chunk = 8 / 4 values, float32 activations,
// float32 FMA.
template <int WDT, int K>
struct Gemv {
  static constexpr int VPC = WDT == WINT4 ? 32 : (WDT == WBF16 ? 8 : 4);
  static constexpr int NCH = K / VPC;
  static constexpr int CPL = (NCH + 31) / 32;
  static constexpr int SUBS = WDT == WINT4 ? 4 : VPC / 4;  // 16-byte pieces of a staged chunk
  static constexpr int META = WDT == WINT4 ? 8 : 0;        // (scale, offset correction)
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
    int corr[AR];
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
            const int2 m = *reinterpret_cast<const int2*>(base + NCH * SUBS * 16 + c * 8);
            a.s[j] = __int_as_float(m.x);
            a.corr[j] = m.y;
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
          const uint32_t wv[4] = {r.w[j].x, r.w[j].y, r.w[j].z, r.w[j].w};
          const uint32_t av[16] = {a.v[j][0].x, a.v[j][0].y, a.v[j][0].z, a.v[j][0].w,
                                   a.v[j][1].x, a.v[j][1].y, a.v[j][1].z, a.v[j][1].w,
                                   a.v[j][2].x, a.v[j][2].y, a.v[j][2].z, a.v[j][2].w,
                                   a.v[j][3].x, a.v[j][3].y, a.v[j][3].z, a.v[j][3].w};
          int ia = 0;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t x = wv[t] ^ 0x88888888u;          // two's complement -> q + 8
            const uint32_t be = x & 0x0F0F0F0Fu;              // codes of k+0, k+2, k+4, k+6
            const uint32_t bo = (x >> 4) & 0x0F0F0F0Fu;       // codes of k+1, k+3, k+5, k+7
            asm("dp2a.lo.s32.u32 %0, %1, %2, %0;" : "+r"(ia) : "r"(av[4 * t + 0]), "r"(be));
            asm("dp2a.hi.s32.u32 %0, %1, %2, %0;" : "+r"(ia) : "r"(av[4 * t + 1]), "r"(be));
            asm("dp2a.lo.s32.u32 %0, %1, %2, %0;" : "+r"(ia) : "r"(av[4 * t + 2]), "r"(bo));
            asm("dp2a.hi.s32.u32 %0, %1, %2, %0;" : "+r"(ia) : "r"(av[4 * t + 3]), "r"(bo));
          }
          acc = fmaf((float)(ia - a.corr[j]), a.s[j] * r.s[j], acc);
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

  // Stage y[k] = f(k) (k < K) into shared memory at `dst` (one warp).
  template <class F>
  __device__ static __forceinline__ void stage(uint8_t* dst, int lane, F f) {
    for (int c = lane; c < NCH; c += 32) {
      float y[VPC];
#pragma unroll
      for (int i = 0; i < VPC; ++i) y[i] = f(c * VPC + i);
      if constexpr (WDT == WINT4) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(y[i]));
        const float inv = amax > 0.f ? 32767.f / amax : 0.f;
        int sum = 0;
        // dp2a operand order per 8-value word t: (0,2) (4,6) (1,3) (5,7)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          int v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[i] = __float2int_rn(y[8 * t + i] * inv);
            sum += v[i];
          }
          *reinterpret_cast<uint4*>(dst + (t * NCH + c) * 16) =
              make_uint4((uint32_t)(v[0] & 0xFFFF) | ((uint32_t)v[2] << 16),
                         (uint32_t)(v[4] & 0xFFFF) | ((uint32_t)v[6] << 16),
                         (uint32_t)(v[1] & 0xFFFF) | ((uint32_t)v[3] << 16),
                         (uint32_t)(v[5] & 0xFFFF) | ((uint32_t)v[7] << 16));
        }
        *reinterpret_cast<int2*>(dst + NCH * SUBS * 16 + c * 8) =
            make_int2(__float_as_int(amax / 32767.f), 8 * sum);
      } else {
#pragma unroll
        for (int t = 0; t < SUBS; ++t)
          *reinterpret_cast<float4*>(dst + (t * NCH + c) * 16) =
              make_float4(y[4 * t], y[4 * t + 1], y[4 * t + 2], y[4 * t + 3]);
      }
    }
  }
};

// Sum of squares of a K-vector from a value function (one warp, all lanes get it).
template <int K, class F>
__device__ __forceinline__ float warp_sumsq(int lane, F f) {
  float s = 0.f;
  for (int k = lane; k < K; k += 32) {
    const float v = f(k);
    s = fmaf(v, v, s);
  }
  return warp_sum(s);
}

// Block-level task runner.  Tasks t = warp, warp + 16, ... ; each task has RP
// weight rows and a list of staged activations; the warp loads each row once
// and forms its dot product with every activation of the task.
//   T::row(t, r, &w, &s)       row pointers of row r of task t
//   T::acts(t, &list, &start)  -> count; activation i is list ? list[start+i] : start+i
//   T::out(t, ai, i, v[RP])    result for activation ai (i-th of the task), all lanes
template <int WDT, int K, int RP, class T>
__device__ __forceinline__ void run_tasks(int ntasks, const uint8_t* act_base, T& task) {
  using Gv = Gemv<WDT, K>;
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  typename Gv::Act a;
  int loaded = -1;
  if constexpr (Gv::PIPE && RP == 1) {
    typename Gv::Row cur[RP], nxt[RP];
    int t = wid;
    if (t < ntasks) {
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const uint8_t* w; const uint16_t* s;
        task.row(t, r, &w, &s);
        Gv::load_row(cur[r], w, s, lane);
      }
    }
    for (; t < ntasks; t += kWarps) {
      const int tn = t + kWarps;
      if (tn < ntasks) {
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const uint8_t* w; const uint16_t* s;
          task.row(tn, r, &w, &s);
          Gv::load_row(nxt[r], w, s, lane);
        }
      }
      const uint8_t* list; int start;
      const int cnt = task.acts(t, &list, &start);
      for (int i = 0; i < cnt; ++i) {
        const int ai = list ? list[start + i] : start + i;
        if (ai != loaded) { Gv::load_act(a, act_base + ai * Gv::ACT_BYTES, lane); loaded = ai; }
        float v[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) v[r] = warp_sum(Gv::dot(cur[r], a, lane));
        task.out(t, ai, i, v);
      }
#pragma unroll
      for (int r = 0; r < RP; ++r) cur[r] = nxt[r];
    }
  } else {
    typename Gv::Row row;
    for (int t = wid; t < ntasks; t += kWarps) {
      const uint8_t* list; int start;
      const int cnt = task.acts(t, &list, &start);
      for (int i = 0; i < cnt; ++i) {
        const int ai = list ? list[start + i] : start + i;
        if (ai != loaded) { Gv::load_act(a, act_base + ai * Gv::ACT_BYTES, lane); loaded = ai; }
        float v[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const uint8_t* w; const uint16_t* s;
          task.row(t, r, &w, &s);
          Gv::load_row(row, w, s, lane);
          v[r] = warp_sum(Gv::dot(row, a, lane));
        }
        task.out(t, ai, i, v);
      }
    }
  }
}

__device__ __forceinline__ void split_range(int n, int parts, int idx, int& lo, int& hi) {
  lo = (int)(((long long)n * idx) / parts);
  hi = (int)(((long long)n * (idx + 1)) / parts);
}

}  // namespace mk
