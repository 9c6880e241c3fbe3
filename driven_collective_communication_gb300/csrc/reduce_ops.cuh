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
  __device__ static bool is_nan(uint32_t b) { return (b & 0x7fffffffu) > 0x7f800000u; }
  __device__ static int32_t key(uint32_t b) {
    const int32_t s = (int32_t)b;
    return s ^ ((s >> 31) & 0x7fffffff);
  }
};

// 16-bit formats: the value sits in the low 16 bits of b
template <uint32_t kInfBits, uint32_t kNaNBits>
struct Ieee16Bits {
  static constexpr uint32_t kNaN = kNaNBits;
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

// a OP b for one element held in the low bits of a 32-bit word
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

// a OP b for every element of a 32-bit word (one 32-bit or two 16-bit lanes)
template <typename T, int OP>
__device__ __forceinline__ uint32_t pick_word(uint32_t a, uint32_t b) {
  if constexpr (sizeof(T) == 4) {
    return pick1<T, OP>(a, b);
  } else {
    const uint32_t lo = pick1<T, OP>(a & 0xffffu, b & 0xffffu);
    const uint32_t hi = pick1<T, OP>(a >> 16, b >> 16);
    return lo | (hi << 16);
  }
}

template <typename T, int OP>
__device__ __forceinline__ uint4 pick_vec(uint4 a, uint4 b) {
  return make_uint4(pick_word<T, OP>(a.x, b.x), pick_word<T, OP>(a.y, b.y), pick_word<T, OP>(a.z, b.z),
                    pick_word<T, OP>(a.w, b.w));
}

// MAX / MIN of vector v over the N ranks' buffers, rank order; with a
// compile-time N all N gets are issued before the first combine.  A NaN is
// canonical for every N: with one rank the value is combined with itself.
template <typename T, int NT, int OP>
__device__ __forceinline__ uint4 pick_ranks_vec(void* const* src, int n, size_t v) {
  if constexpr (NT > 0) {
    uint4 x[NT];
#pragma unroll
    for (int p = 0; p < NT; ++p) x[p] = ld_vec(static_cast<const uint4*>(src[p]) + v);
    uint4 acc = x[0];
    if constexpr (NT == 1) acc = pick_vec<T, OP>(acc, acc);
#pragma unroll
    for (int p = 1; p < NT; ++p) acc = pick_vec<T, OP>(acc, x[p]);
    return acc;
  } else {
    uint4 acc = ld_vec(static_cast<const uint4*>(src[0]) + v);
    if (n == 1) acc = pick_vec<T, OP>(acc, acc);
    for (int p = 1; p < n; ++p) acc = pick_vec<T, OP>(acc, ld_vec(static_cast<const uint4*>(src[p]) + v));
    return acc;
  }
}

// one element i; S is the element's storage type (int32_t, float, uint16_t)
template <typename T, int OP, typename S>
__device__ __forceinline__ S pick_ranks_scalar(void* const* src, int n, size_t i) {
  static_assert(sizeof(S) == sizeof(T), "storage type");
  auto bits = [&](int p) {
    S x = static_cast<const S*>(src[p])[i];
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
