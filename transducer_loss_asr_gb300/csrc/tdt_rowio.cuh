// tdt_rowio.cuh -- 16-byte vector access to one logits / gradient row.
//
// A row of V+D elements may start at any element-aligned address (rows of
// [..., 8198] fp32 are 8-byte aligned, a bf16 slice of a [..., 8205] tensor
// only 2-byte aligned), so a warp walks a row as: a scalar head up to the
// first 16-byte boundary, a body of 16-byte vectors, a scalar tail.  This
// keeps every body load a full 16-byte access whatever the row stride is
// ("Vectorized Memory Access", "cuda-kernels" skill page, re-derived for
// rows that are not 16-byte aligned).
#pragma once

#include "tdt_common.cuh"

namespace tdt {

template <int DT> struct Vec {
  static constexpr int N = 16 / (int)sizeof(typename Elem<DT>::T);  // elements per vector
};

// 16-byte streaming load that does not allocate in L1 (each logits byte is
// read once per pass).  With COH = false it takes the non-coherent read-only
// path (the row is not written while the kernel runs); with COH = true a
// plain global load, for the gradient pass writing over its own input.
template <bool COH> __device__ __forceinline__ uint4 ld_row16(const uint4 *p) {
  uint4 v;
  if (COH)
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
  else
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
  return v;
}

// 16-byte load that allocates in L1: for vectors that neighbouring lanes
// read twice (the realigned gradient path).  Read-only path unless COH.
template <bool COH> __device__ __forceinline__ uint4 ld_row16_l1(const void *p) {
  uint4 v;
  if (COH)
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
  else
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
  return v;
}

// The 16 bytes that start `qw` words plus `rb` bits into the 32-byte pair
// (lo, hi), qw in [0, 3], rb in {0, 8, 16, 24}.
__device__ __forceinline__ uint4 funnel16(uint4 lo, uint4 hi, int qw, int rb) {
  // shift by whole words: 2 then 1
  unsigned w0 = lo.x, w1 = lo.y, w2 = lo.z, w3 = lo.w, w4 = hi.x, w5 = hi.y, w6 = hi.z,
           w7 = hi.w;
  if (qw & 2) {
    w0 = w2; w1 = w3; w2 = w4; w3 = w5; w4 = w6; w5 = w7;
  }
  if (qw & 1) {
    w0 = w1; w1 = w2; w2 = w3; w3 = w4; w4 = w5;
  }
  return make_uint4(__funnelshift_r(w0, w1, rb), __funnelshift_r(w1, w2, rb),
                    __funnelshift_r(w2, w3, rb), __funnelshift_r(w3, w4, rb));
}

// One element as float, read-only path unless COH.
template <int DT, bool COH>
__device__ __forceinline__ float ld_elem(const typename Elem<DT>::T *p) {
  if (COH) return Elem<DT>::to_float(*p);
  return Elem<DT>::load(p);
}

// Streaming 16-byte load through the read-only path.
__device__ __forceinline__ uint4 ld_vec(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

template <int DT> __device__ __forceinline__ void unpack(uint4 v, float *x);
template <> __device__ __forceinline__ void unpack<kF32>(uint4 v, float *x) {
  x[0] = __uint_as_float(v.x);
  x[1] = __uint_as_float(v.y);
  x[2] = __uint_as_float(v.z);
  x[3] = __uint_as_float(v.w);
}
template <> __device__ __forceinline__ void unpack<kBF16>(uint4 v, float *x) {
  const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <> __device__ __forceinline__ void unpack<kF16>(uint4 v, float *x) {
  const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
    float2 f = __half22float2(h);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

template <int DT> __device__ __forceinline__ uint4 pack(const float *x);
template <> __device__ __forceinline__ uint4 pack<kF32>(const float *x) {
  return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                    __float_as_uint(x[3]));
}
template <> __device__ __forceinline__ uint4 pack<kBF16>(const float *x) {
  unsigned w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    w[i] = *reinterpret_cast<unsigned *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <> __device__ __forceinline__ uint4 pack<kF16>(const float *x) {
  unsigned w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
    w[i] = *reinterpret_cast<unsigned *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Elements before the first 16-byte boundary of a row starting at p.
template <int DT> __device__ __forceinline__ int head_elems(const void *p) {
  const int mis = (int)(reinterpret_cast<uintptr_t>(p) & 15);
  return ((16 - mis) & 15) / (int)sizeof(typename Elem<DT>::T);
}

}  // namespace tdt

namespace tdt {

// Threads per row group for a row of row_bytes: the smallest power of two in
// [8, 256] whose `batch` 16-byte loads per thread cover the row's vector
// body.  The body holds at most row_bytes / 16 whole vectors (the head and
// tail around it are scalar accesses).
inline int row_group_threads(long long row_bytes, int batch) {
  int t = 8;
  while (t < 256 && (long long)t * batch < row_bytes / 16) t <<= 1;
  return t;
}

}  // namespace tdt
