// Device helpers shared by the AttnRes kernels: 16-byte vector I/O, bf16 <-> fp32
// conversion, cp.async staging and block reductions.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

using bf16 = __nv_bfloat16;

// Elements per 16-byte vector.
template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<bf16> { static constexpr int N = 8; };

// ---- global memory ------------------------------------------------------------------------
// Streaming load of data read once by this kernel (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_global(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ---- conversions -------------------------------------------------------------------------
// bf16 is the top half of an fp32: widening is a shift (low element) or a mask (high).
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}

// A row vector of VE elements (VE = elements per 16 bytes of the I/O type) stored as TO, which
// is the I/O type or fp32: NW = VE * sizeof(TO) / 16 words of 16 bytes.
template <typename TO, int VE> struct OWords {
  static constexpr int N = VE * int(sizeof(TO)) / 16;
};

template <typename TO, int VE>
__device__ __forceinline__ void ld_stream_w(const TO* p, uint4 (&r)[OWords<TO, VE>::N]) {
#pragma unroll
  for (int i = 0; i < OWords<TO, VE>::N; ++i)
    r[i] = ld_stream(reinterpret_cast<const char*>(p) + 16 * i);
}

template <typename TO, int VE>
__device__ __forceinline__ void unpack_w(const uint4 (&r)[OWords<TO, VE>::N], float (&f)[VE]) {
  if constexpr (sizeof(TO) == 2) {
    unpack(r[0], f);
  } else {
#pragma unroll
    for (int i = 0; i < OWords<TO, VE>::N; ++i) {
      f[4 * i] = __uint_as_float(r[i].x);
      f[4 * i + 1] = __uint_as_float(r[i].y);
      f[4 * i + 2] = __uint_as_float(r[i].z);
      f[4 * i + 3] = __uint_as_float(r[i].w);
    }
  }
}

// Stores VE elements as TO (bf16 rounded to nearest even, or fp32 as computed).
template <typename TO, int VE>
__device__ __forceinline__ void st_vec(TO* p, const float (&f)[VE]) {
  if constexpr (sizeof(TO) == 2) {
    st_global(p, pack(f));
  } else {
#pragma unroll
    for (int i = 0; i < VE / 4; ++i)
      st_global(reinterpret_cast<char*>(p) + 16 * i,
                make_uint4(__float_as_uint(f[4 * i]), __float_as_uint(f[4 * i + 1]),
                           __float_as_uint(f[4 * i + 2]), __float_as_uint(f[4 * i + 3])));
  }
}

// Eight consecutive elements starting at a 16-byte aligned address (generic or shared).
template <typename T> __device__ __forceinline__ void load8(const void* p, float (&f)[8]);
template <> __device__ __forceinline__ void load8<bf16>(const void* p, float (&f)[8]) {
  unpack(*reinterpret_cast<const uint4*>(p), f);
}
template <> __device__ __forceinline__ void load8<float>(const void* p, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

template <typename T> __device__ __forceinline__ void store8(void* p, const float (&f)[8]);
template <> __device__ __forceinline__ void store8<bf16>(void* p, const float (&f)[8]) {
  st_global(p, pack(f));
}
template <> __device__ __forceinline__ void store8<float>(void* p, const float (&f)[8]) {
  st_global(p, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3])));
  st_global(static_cast<char*>(p) + 16,
            make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                       __float_as_uint(f[7])));
}

// ---- cp.async (global -> shared, 16 bytes, zero-filled when !valid) ------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const int bytes = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- programmatic dependent launch -----------------------------------------------------------
// Every kernel of the library is launched with programmatic stream serialisation (launch_pdl
// below), so it may be scheduled while the kernel before it on the stream is still finishing.
// pdl_enter() first lets this kernel's own successor be scheduled (once every CTA of this grid
// has started), then waits until the predecessor has completed and its memory is visible.  All
// threads call it before their first global read or write.  Without a programmatic predecessor
// both instructions return at once.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Only the wait: the kernel's successor is scheduled when this grid's CTAs have exited.  Used by
// the kernels whose CTAs fill the SMs for many waves and whose successor gains nothing from
// waiting beside their last waves: with the tensor-core phase 1 entering through pdl_enter(),
// the long-context step (8 chunks of 16384 tokens, no events between the launches) took 71.0
// instead of 58.5 ms; the block backward's kernels gain 1 %.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch `kern` on stream `s` with programmatic stream serialisation allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ---- reductions ------------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of two values over the whole CTA; every thread gets the totals.  `scratch` holds at
// least 2 * 33 floats of shared memory and is reused across calls (the trailing barrier
// protects it).
__device__ __forceinline__ void block_sum2(float& a, float& b, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) {
    scratch[warp] = a;
    scratch[33 + warp] = b;
  }
  __syncthreads();
  if (warp == 0) {
    float x = lane < nw ? scratch[lane] : 0.f;
    float y = lane < nw ? scratch[33 + lane] : 0.f;
    x = warp_sum(x);
    y = warp_sum(y);
    if (lane == 0) {
      scratch[32] = x;
      scratch[65] = y;
    }
  }
  __syncthreads();
  a = scratch[32];
  b = scratch[65];
  __syncthreads();
}

// Sum of N values over the whole CTA with one set of barriers; every thread gets the totals.
// `scratch` holds at least N * 33 floats of shared memory.
template <int N>
__device__ __forceinline__ void block_sum_n(float (&v)[N], float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = warp_sum(v[i]);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) scratch[i * 33 + warp] = v[i];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      float x = lane < nw ? scratch[i * 33 + lane] : 0.f;
      x = warp_sum(x);
      if (lane == 0) scratch[i * 33 + 32] = x;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = scratch[i * 33 + 32];
  __syncthreads();
}

}  // namespace attnres
