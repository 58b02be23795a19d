// ar_device.cuh -- device-side building blocks shared by the all-reduce kernels:
// 16-byte vector lanes per data type, the combine operators, the fused
// scale / narrowing epilogue, streaming load / store wrappers and the two
// binary trees as compile-time functions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ar {

enum : int { kF32 = 0, kBF16 = 1, kI32 = 2 };
enum : int { kSum = 0, kMin = 1, kMax = 2 };
enum : int { kRing = 1, kTree = 2, kHier = 4 };

// A 16-byte vector of each data type and the type it is accumulated in:
// fp32 and bf16 accumulate in fp32, int32 in int32 with wrap-around adds.
template <int DT> struct Lanes;
template <> struct Lanes<kF32> { static constexpr int N = 4; using T = float; static constexpr int kBytes = 4; };
template <> struct Lanes<kBF16> { static constexpr int N = 8; using T = float; static constexpr int kBytes = 2; };
template <> struct Lanes<kI32> { static constexpr int N = 4; using T = int32_t; static constexpr int kBytes = 4; };

template <int DT> struct Acc {
  typename Lanes<DT>::T v[Lanes<DT>::N];
};

// ----------------------------------------------------------------- launch order

// Every kernel starts here.  Launched with programmatic dependent launch
// (launch_kernel), a kernel may be scheduled while the kernel before it on the
// stream is still draining; it first lets its own successor be scheduled the
// same way, then waits until its predecessor has completed and that kernel's
// writes are visible, before it touches memory.  Launched plainly, or with no
// kernel before it, the wait returns at once.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ----------------------------------------------------------------- memory

// Cache hints of the streaming accesses (compile-time tunables).
#ifndef AR_LD_HINT
#define AR_LD_HINT 0
#endif
#ifndef AR_ST_HINT
#define AR_ST_HINT 0
#endif
#if AR_LD_HINT == 0
#define AR_LD_OP "ld.global.L1::no_allocate.v4.u32"
#elif AR_LD_HINT == 1
#define AR_LD_OP "ld.global.nc.L1::no_allocate.v4.u32"
#elif AR_LD_HINT == 2
#define AR_LD_OP "ld.global.cs.v4.u32"
#else
#define AR_LD_OP "ld.global.L1::no_allocate.L2::256B.v4.u32"
#endif
#if AR_ST_HINT == 0
#define AR_ST_OP "st.global.cs.v4.u32"
#elif AR_ST_HINT == 1
#define AR_ST_OP "st.global.v4.u32"
#else
#define AR_ST_OP "st.global.L1::no_allocate.v4.u32"
#endif

// Streaming 16-byte load: each input element is read exactly once, so it
// is not kept in L1.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm(AR_LD_OP " {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Streaming 16-byte store: outputs are not re-read by this kernel.
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile(AR_ST_OP " [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w));
}

// 8-byte accesses used by the LL protocol.  A naturally aligned 64-bit access
// is single-copy atomic, so a reader that sees the flag half of a word also
// sees the payload half written with it -- no fence is needed.
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ------------------------------------------------------------ arithmetic

template <int DT, int OP>
__device__ __forceinline__ typename Lanes<DT>::T combine(typename Lanes<DT>::T acc,
                                                         typename Lanes<DT>::T x) {
  if constexpr (OP == kSum) {
    if constexpr (DT == kI32) {
      return (int32_t)((uint32_t)acc + (uint32_t)x);  // two's-complement wrap
    } else {
      return __fadd_rn(acc, x);                        // never contracted into an FMA
    }
  } else if constexpr (OP == kMin) {
    return (x < acc) ? x : acc;                        // a tie keeps the earlier operand
  } else {
    return (x > acc) ? x : acc;
  }
}

template <int DT, int OP>
__device__ __forceinline__ void fold(Acc<DT>& acc, const Acc<DT>& x) {
#pragma unroll
  for (int i = 0; i < Lanes<DT>::N; ++i) acc.v[i] = combine<DT, OP>(acc.v[i], x.v[i]);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 values to a bf16 pair, each rounded to nearest even (the
// hardware conversion instruction); `hi` lands in the upper half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

template <int DT>
__device__ __forceinline__ Acc<DT> widen(uint4 r) {
  Acc<DT> a;
  if constexpr (DT == kF32) {
    a.v[0] = __uint_as_float(r.x); a.v[1] = __uint_as_float(r.y);
    a.v[2] = __uint_as_float(r.z); a.v[3] = __uint_as_float(r.w);
  } else if constexpr (DT == kBF16) {
    a.v[0] = bf16_lo(r.x); a.v[1] = bf16_hi(r.x); a.v[2] = bf16_lo(r.y); a.v[3] = bf16_hi(r.y);
    a.v[4] = bf16_lo(r.z); a.v[5] = bf16_hi(r.z); a.v[6] = bf16_lo(r.w); a.v[7] = bf16_hi(r.w);
  } else {
    a.v[0] = (int32_t)r.x; a.v[1] = (int32_t)r.y; a.v[2] = (int32_t)r.z; a.v[3] = (int32_t)r.w;
  }
  return a;
}

// Epilogue: y = narrow(acc * scale); the multiply only when do_scale.
template <int DT>
__device__ __forceinline__ uint4 narrow(Acc<DT> a, float scale, bool do_scale) {
  uint4 r;
  if constexpr (DT == kI32) {
    r.x = (uint32_t)a.v[0]; r.y = (uint32_t)a.v[1]; r.z = (uint32_t)a.v[2]; r.w = (uint32_t)a.v[3];
  } else {
    if (do_scale) {
#pragma unroll
      for (int i = 0; i < Lanes<DT>::N; ++i) a.v[i] = __fmul_rn(a.v[i], scale);
    }
    if constexpr (DT == kF32) {
      r.x = __float_as_uint(a.v[0]); r.y = __float_as_uint(a.v[1]);
      r.z = __float_as_uint(a.v[2]); r.w = __float_as_uint(a.v[3]);
    } else {
      r.x = pack_bf16x2(a.v[0], a.v[1]); r.y = pack_bf16x2(a.v[2], a.v[3]);
      r.z = pack_bf16x2(a.v[4], a.v[5]); r.w = pack_bf16x2(a.v[6], a.v[7]);
    }
  }
  return r;
}

// The last, partial vector of a rank (n < lanes valid elements): loaded and
// stored element by element, the missing lanes read as zero and not stored.
template <int DT>
__device__ __forceinline__ uint4 load_partial(const uint4* p, int n) {
  // unrolled over the vector's lanes with a predicate per lane, so the
  // words stay in registers
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if constexpr (Lanes<DT>::kBytes == 4) {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < n) w[i] = q[i];
  } else {
    const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < n) w[i >> 1] |= (uint32_t)q[i] << (16 * (i & 1));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT>
__device__ __forceinline__ void store_partial(uint4* p, uint4 v, int n) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (Lanes<DT>::kBytes == 4) {
    uint32_t* q = reinterpret_cast<uint32_t*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < n) q[i] = w[i];
  } else {
    uint16_t* q = reinterpret_cast<uint16_t*>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < n) q[i] = (uint16_t)(w[i >> 1] >> (16 * (i & 1)));
  }
}

// ------------------------------------------------------ double binary tree
// In-order binary tree on labels 1..P ("NCCL and NVSHMEM -- two GPU
// communication models, side by side", section "double binary tree").

__host__ __device__ constexpr int tree_root(int P) {
  int r = 1;
  while (r * 2 <= P) r *= 2;
  return r;
}
__host__ __device__ constexpr int tree_lowbit(int v) { return v & -v; }
__host__ __device__ constexpr int tree_left(int v) {
  return tree_lowbit(v) >= 2 ? v - tree_lowbit(v) / 2 : 0;
}
__host__ __device__ constexpr int tree_right(int v, int P) {
  int b = tree_lowbit(v);
  if (b < 2) return 0;
  for (int h = b / 2; h >= 1; h /= 2)
    if (v + h <= P) return v + h;
  return 0;
}
// Tree 0: label v belongs to rank v-1; tree 1 shifts ranks by one: rank v mod P.
__host__ __device__ constexpr int tree_owner(int v, int P, int t) { return t == 0 ? v - 1 : v % P; }

}  // namespace ar
