// dsc_common.cuh -- element types, 16-byte vector access and small helpers
// shared by the DSC kernels.  Device code only; no host logic here.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsc {

// ---------------------------------------------------------------- types ----

// Elements carried by one 16-byte vector.
template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// ------------------------------------------------- 16-byte vector access ----

// Unpack one 16-byte vector of T into fp32 lanes.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float (&f)[Vec<T>::N]);

template <>
__device__ __forceinline__ void unpack16<float>(const uint4& u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float (&f)[Vec<T>::N]);

template <>
__device__ __forceinline__ uint4 pack16<float>(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                    __float_as_uint(f[2]), __float_as_uint(f[3]));
}

template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Streaming 16-byte load through the read-only path.
__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte store with the evict-first (streaming) cache hint.
__device__ __forceinline__ void stcs16(void* p, const uint4& v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// --------------------------------------------- loads of a few filter taps ----

// Load `n` consecutive elements of T starting at `p` into fp32, using the
// widest aligned vector access the byte count allows.  `p` must be aligned
// to that width, which holds whenever every thread's chunk starts at a
// multiple of the chunk size (the callers guarantee it).
template <typename T, int n>
__device__ __forceinline__ void load_chunk(const T* __restrict__ p, float (&out)[n]) {
  constexpr int bytes = n * (int)sizeof(T);
  constexpr int vb = (bytes % 16 == 0) ? 16 : (bytes % 8 == 0) ? 8
                   : (bytes % 4 == 0) ? 4 : (int)sizeof(T);
  constexpr int per = vb / (int)sizeof(T);   // elements per access
#pragma unroll
  for (int i = 0; i < n / per; ++i) {
    const T* q = p + i * per;
    if constexpr (vb == 16) {
      uint4 u = __ldg(reinterpret_cast<const uint4*>(q));
      float f[Vec<T>::N];
      unpack16<T>(u, f);
#pragma unroll
      for (int e = 0; e < per; ++e) out[i * per + e] = f[e];
    } else if constexpr (vb == 8) {
      uint2 u = __ldg(reinterpret_cast<const uint2*>(q));
      const uint32_t w2[2] = {u.x, u.y};
      if constexpr (sizeof(T) == 4) {
        out[i * per + 0] = __uint_as_float(w2[0]);
        out[i * per + 1] = __uint_as_float(w2[1]);
      } else {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          out[i * per + 2 * e] = __uint_as_float(w2[e] << 16);
          out[i * per + 2 * e + 1] = __uint_as_float(w2[e] & 0xffff0000u);
        }
      }
    } else if constexpr (vb == 4) {
      uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(q));
      if constexpr (sizeof(T) == 4) {
        out[i * per] = __uint_as_float(u);
      } else {
        out[i * per] = __uint_as_float(u << 16);
        out[i * per + 1] = __uint_as_float(u & 0xffff0000u);
      }
    } else {
      out[i] = to_f32(__ldg(q));
    }
  }
}

// The same `n` elements held as raw bits, so a load can be issued early
// (prefetched) and decoded to fp32 later.  Same alignment rule as above.
template <typename T, int n>
struct RawChunk {
  static constexpr int bytes = n * (int)sizeof(T);
  static constexpr int vb = (bytes % 16 == 0) ? 16 : (bytes % 8 == 0) ? 8
                          : (bytes % 4 == 0) ? 4 : (int)sizeof(T);
  static constexpr int per = vb / (int)sizeof(T);   // elements per access
  static constexpr int cnt = n / per;                // accesses
  static constexpr int words = vb >= 4 ? vb / 4 : 1; // 32-bit words per access
  uint32_t w[cnt][words];

  __device__ __forceinline__ void load(const T* __restrict__ p) {
#pragma unroll
    for (int i = 0; i < cnt; ++i) {
      const T* q = p + i * per;
      if constexpr (vb == 16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(q));
        w[i][0] = u.x; w[i][1] = u.y; w[i][2] = u.z; w[i][3] = u.w;
      } else if constexpr (vb == 8) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(q));
        w[i][0] = u.x; w[i][1] = u.y;
      } else if constexpr (vb == 4) {
        w[i][0] = __ldg(reinterpret_cast<const unsigned int*>(q));
      } else {
        w[i][0] = __ldg(reinterpret_cast<const unsigned short*>(q));
      }
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < cnt; ++i)
#pragma unroll
      for (int j = 0; j < words; ++j) w[i][j] = 0u;
  }
  __device__ __forceinline__ void unpack(float (&out)[n]) const {
#pragma unroll
    for (int i = 0; i < cnt; ++i) {
      if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < per; ++e) out[i * per + e] = __uint_as_float(w[i][e]);
      } else if constexpr (vb >= 4) {
#pragma unroll
        for (int e = 0; e < per / 2; ++e) {
          out[i * per + 2 * e] = __uint_as_float(w[i][e] << 16);
          out[i * per + 2 * e + 1] = __uint_as_float(w[i][e] & 0xffff0000u);
        }
      } else {
        out[i] = __uint_as_float(w[i][0] << 16);
      }
    }
  }
};

// Store `n` consecutive fp32 values as T, widest aligned access (see above).
template <typename T, int n>
__device__ __forceinline__ void store_chunk(T* __restrict__ p, const float (&v)[n]) {
  constexpr int bytes = n * (int)sizeof(T);
  constexpr int vb = (bytes % 16 == 0) ? 16 : (bytes % 8 == 0) ? 8
                   : (bytes % 4 == 0) ? 4 : (int)sizeof(T);
  constexpr int per = vb / (int)sizeof(T);
#pragma unroll
  for (int i = 0; i < n / per; ++i) {
    T* q = p + i * per;
    if constexpr (vb == 16) {
      float f[Vec<T>::N];
#pragma unroll
      for (int e = 0; e < per; ++e) f[e] = v[i * per + e];
      *reinterpret_cast<uint4*>(q) = pack16<T>(f);
    } else if constexpr (vb == 8) {
      if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<uint2*>(q) =
            make_uint2(__float_as_uint(v[i * per]), __float_as_uint(v[i * per + 1]));
      } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(v[i * per], v[i * per + 1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(v[i * per + 2], v[i * per + 3]);
        *reinterpret_cast<uint2*>(q) = make_uint2(*reinterpret_cast<uint32_t*>(&a),
                                                  *reinterpret_cast<uint32_t*>(&b));
      }
    } else if constexpr (vb == 4) {
      if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float*>(q) = v[i * per];
      } else {
        *reinterpret_cast<__nv_bfloat162*>(q) =
            __floats2bfloat162_rn(v[i * per], v[i * per + 1]);
      }
    } else {
      *q = from_f32<T>(v[i]);
    }
  }
}

}  // namespace dsc
