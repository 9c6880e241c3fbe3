// reduce_ops.cuh -- MAX / MIN combiners of the AllReduce and ReduceScatter.
//
// The MSCCL++ pages speak of sum reductions only.  MAX and MIN here are the
// IEEE 754-2019 maximum / minimum operations applied in rank order: a NaN
// operand gives NaN, written as the type's canonical quiet NaN (positive, top
// mantissa bit set); -0 orders below +0; otherwise the larger / smaller
// operand is the result.  int32 takes the signed maximum / minimum.
//
// The result is always one of the operands' bit patterns (or that NaN), so the
// kernels combine raw storage bits: nothing is widened or rounded, and every
// algorithm returns the same bits.  Order key: the bits of an IEEE value read
// as a sign-magnitude integer; flipping the magnitude bits of negative values
// turns it into two's complement, where signed integer order is numeric order
// with -0 (key -1) just below +0 (key 0).  Equal keys mean equal bits.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "memory_channel.cuh"

namespace dcc {

enum RedOp { kOpSum = 0, kOpMax = 1, kOpMin = 2 };

template <typename T>
struct IeeeBits;

template <>
struct IeeeBits<float> {
  static constexpr uint32_t kNaN = 0x7fc00000u;
  static constexpr uint32_t kInf = 0x7f800000u;
  __device__ static bool is_nan(uint32_t b) { return (b & 0x7fffffffu) > kInf; }
  __device__ static int32_t key(uint32_t b) {
    const int32_t s = (int32_t)b;
    return s ^ ((s >> 31) & 0x7fffffff);
  }
};

// 16-bit formats: the value sits in the low 16 bits of b
template <uint32_t kInfBits, uint32_t kNaNBits>
struct Ieee16Bits {
  static constexpr uint32_t kNaN = kNaNBits;
  static constexpr uint32_t kInf = kInfBits;
  __device__ static bool is_nan(uint32_t b) { return (b & 0x7fffu) > kInfBits; }
  __device__ static int32_t key(uint32_t b) {
    const int32_t s = (int16_t)(uint16_t)b;  // sign-extended
    return s ^ ((s >> 31) & 0x7fff);
  }
};
template <>
struct IeeeBits<__half> : Ieee16Bits<0x7c00u, 0x7e00u> {};
template <>
struct IeeeBits<__nv_bfloat16> : Ieee16Bits<0x7f80u, 0x7fc0u> {};

// a OP b for one element held in the low bits of a 32-bit word (the
// element-by-element tail)
template <typename T, int OP>
__device__ __forceinline__ uint32_t pick1(uint32_t a, uint32_t b) {
  if constexpr (std::is_same<T, int32_t>::value) {
    const int32_t x = (int32_t)a, y = (int32_t)b;
    return (uint32_t)(OP == kOpMax ? (y > x ? y : x) : (y < x ? y : x));
  } else {
    using F = IeeeBits<T>;
    if (F::is_nan(a) || F::is_nan(b)) return F::kNaN;
    const int32_t ka = F::key(a), kb = F::key(b);
    return (OP == kOpMax ? kb > ka : kb < ka) ? b : a;
  }
}

// ---------------------------------------------------------------- vectors
// The vector path keeps its running result in key space (the key map is its
// own inverse: it never changes the sign bit) and, per lane, the largest
// magnitude seen; a lane whose largest magnitude lies above infinity has seen
// a NaN.  Per 32-bit word and rank that is one key map, one signed max / min
// and one unsigned max, with the 16-bit formats done two lanes at a time
// (PTX max/min.s16x2, max.u16x2).  Same results as pick1 lane by lane.
__device__ __forceinline__ uint32_t max_s16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t min_s16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <typename T, int OP>
struct PickWord {
  uint32_t k;    // running MAX / MIN as order keys (int32: the value itself)
  uint32_t mag;  // largest magnitude per lane (IEEE formats)

  __device__ static uint32_t key(uint32_t w) {
    if constexpr (sizeof(T) == 2) return w ^ (((w >> 15) & 0x00010001u) * 0x7fffu);  // both lanes
    else return w ^ ((uint32_t)((int32_t)w >> 31) & 0x7fffffffu);
  }
  __device__ void init(uint32_t w) {
    if constexpr (std::is_same<T, int32_t>::value) {
      k = w;
    } else {
      k = key(w);
      mag = w & (sizeof(T) == 2 ? 0x7fff7fffu : 0x7fffffffu);
    }
  }
  __device__ void add(uint32_t w) {
    if constexpr (std::is_same<T, int32_t>::value) {
      const int32_t a = (int32_t)k, b = (int32_t)w;
      k = (uint32_t)(OP == kOpMax ? max(a, b) : min(a, b));
    } else if constexpr (sizeof(T) == 2) {
      k = OP == kOpMax ? max_s16x2(k, key(w)) : min_s16x2(k, key(w));
      mag = max_u16x2(mag, w & 0x7fff7fffu);
    } else {
      const int32_t a = (int32_t)k, b = (int32_t)key(w);
      k = (uint32_t)(OP == kOpMax ? max(a, b) : min(a, b));
      mag = max(mag, w & 0x7fffffffu);
    }
  }
  __device__ uint32_t result() const {
    if constexpr (std::is_same<T, int32_t>::value) {
      return k;
    } else if constexpr (sizeof(T) == 2) {
      using F = IeeeBits<T>;
      // bit 15 of a lane set where its largest magnitude is above infinity
      // (no carry between lanes: the sum stays below 0x10000)
      const uint32_t nan = (mag + (0x7fffu - F::kInf) * 0x00010001u) & 0x80008000u;
      const uint32_t lanes = (nan >> 15) * 0xffffu;
      return (key(k) & ~lanes) | (F::kNaN * 0x00010001u & lanes);
    } else {
      return mag > IeeeBits<float>::kInf ? IeeeBits<float>::kNaN : key(k);
    }
  }
};

template <typename T, int OP>
struct PickVec {
  PickWord<T, OP> w[4];
  __device__ void init(uint4 x) { w[0].init(x.x); w[1].init(x.y); w[2].init(x.z); w[3].init(x.w); }
  __device__ void add(uint4 x) { w[0].add(x.x); w[1].add(x.y); w[2].add(x.z); w[3].add(x.w); }
  __device__ uint4 result() const { return make_uint4(w[0].result(), w[1].result(), w[2].result(), w[3].result()); }
};

// MAX / MIN of vector v over the N ranks' buffers, rank order; with a
// compile-time N all N gets are issued before the first combine.  A NaN is
// canonical for every N, one rank included.
template <typename T, int NT, int OP>
__device__ __forceinline__ uint4 pick_ranks_vec(const DevComm& dc, const CollArgs& a, int n, size_t v) {
  PickVec<T, OP> acc;
  auto get = [&](int p) {
    return in_bounds(dc, a, kBufSend, p, v * 16, 16) ? ld_vec(static_cast<const uint4*>(a.send[p]) + v)
                                                     : make_uint4(0, 0, 0, 0);
  };
  if constexpr (NT > 0) {
    uint4 x[NT];
#pragma unroll
    for (int p = 0; p < NT; ++p) x[p] = get(p);
    acc.init(x[0]);
#pragma unroll
    for (int p = 1; p < NT; ++p) acc.add(x[p]);
  } else {
    acc.init(get(0));
    for (int p = 1; p < n; ++p) acc.add(get(p));
  }
  return acc.result();
}

// one element i; S is the element's storage type (int32_t, float, uint16_t)
template <typename T, int OP, typename S>
__device__ __forceinline__ S pick_ranks_scalar(const DevComm& dc, const CollArgs& a, int n, size_t i) {
  static_assert(sizeof(S) == sizeof(T), "storage type");
  auto bits = [&](int p) {
    S x = in_bounds(dc, a, kBufSend, p, i * sizeof(S), sizeof(S)) ? static_cast<const S*>(a.send[p])[i] : S{};
    uint32_t b = 0;
    memcpy(&b, &x, sizeof(S));
    return b;
  };
  uint32_t acc = bits(0);
  if (n == 1) acc = pick1<T, OP>(acc, acc);
  for (int p = 1; p < n; ++p) acc = pick1<T, OP>(acc, bits(p));
  S out;
  memcpy(&out, &acc, sizeof(S));  // little-endian: the low bytes hold the element
  return out;
}

}  // namespace dcc
