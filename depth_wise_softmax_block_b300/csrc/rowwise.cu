// Row-wise AttnRes kernels: one CTA owns one token row of d features, held in registers.
//
//   phase2_kernel  phase 2 of the two-phase schedule for one sublayer ("Attention Residuals"
//                  note §10 step 2): forms the partial-sum source p = partial + v_prev (the
//                  fused block-sum update of §8), scores it (RMS + dot in one pass), merges it
//                  with the phase-1 result by online softmax ("Attention Residuals 阅读补充",
//                  merge of two partitions) and applies the sublayer's input RMSNorm.
//   full_kernel    the direct single-pass aggregation over an explicit source list (§7),
//                  online softmax over the sources, then the input RMSNorm; optionally seeded
//                  with an earlier partition (o, lse), which makes it the phase 2 of the
//                  grouped Full AttnRes schedule ("Attention Residuals 阅读补充", section
//                  "静态 Query 与两阶段计算").
// Both take the Table 4 variant flags (sigmoid weights, no key RMSNorm; "Attention
// Residuals" note, result 4).
//   add_kernel     partial-sum update / block close: out = partial + v.
//   prep_kernel    query preparation u = w ⊙ gamma_key (and its bf16 hi/lo split).
//
// Each thread owns VPT 16-byte vectors of the row (vector v = threadIdx.x + k * blockDim.x).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace attnres {
namespace {

constexpr int kRowThreads = 256;    // full path: at most 256 threads per row
// phase 2: at most 256 threads per row (224 x 4 vectors at d = 7168 measured faster than
// 448 x 2: 0.219 ms against 0.239 ms for a 16384-row fused call)
constexpr int kMergeThreads = 256;

// Phase 2 of one row from the vectors this thread holds (vector v = threadIdx.x + k *
// blockDim.x of the row): o_l in ro, the stored partial in rp, v_prev in rv (each used only if
// the corresponding input is present).  Ends with the row's stores; `scratch` is the CTA's
// reduction buffer (the block reductions synchronise the CTA).
template <typename T, int VPT>
__device__ __forceinline__ void merge_row(const Phase2Args& a, int64_t row, const uint4 (&ro)[VPT],
                                          const uint4 (&rp)[VPT], const uint4 (&rv)[VPT],
                                          float* scratch) {
  constexpr int VE = Vec<T>::N;
  const int nv = a.d / VE;
  const int64_t base = row * a.d;
  const bool has_p = a.partial != nullptr || a.v_prev != nullptr;

  float h[VPT][VE];
  float p[VPT][VE];
  float ssp = 0.f, dot = 0.f;
  if (has_p) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        float x[VE], y[VE];
        if (a.partial) {
          unpack(rp[k], x);
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) x[e] = 0.f;
        }
        if (a.v_prev) {
          unpack(rv[k], y);
#pragma unroll
          for (int e = 0; e < VE; ++e) x[e] += y[e];
        }
        // The source is the exact fp32 sum; only the stored copy for the next sublayer is
        // rounded to the io type.
        if (a.partial_out) st_global(static_cast<T*>(a.partial_out) + base + v * VE, pack(x));
#pragma unroll
        for (int e = 0; e < VE; ++e) p[k][e] = x[e];
        const float4* u4 = reinterpret_cast<const float4*>(a.u + v * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
          const float4 uu = __ldg(u4 + e / 4);
          dot = fmaf(uu.x, p[k][e], dot);
          dot = fmaf(uu.y, p[k][e + 1], dot);
          dot = fmaf(uu.z, p[k][e + 2], dot);
          dot = fmaf(uu.w, p[k][e + 3], dot);
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) ssp = fmaf(p[k][e], p[k][e], ssp);
      }
    }
    block_sum2(ssp, dot, scratch);
  }

  // Online-softmax merge of the phase-1 partition (lse) with the partial source (z_p); with
  // sigmoid weights the two partitions simply add, h = o + sigmoid(z_p) p.
  float wa = 1.f, wc = 0.f;
  if (has_p) {
    const float z = (a.flags & kNoKeyNorm)
                        ? dot
                        : dot / sqrtf(ssp / static_cast<float>(a.d) + a.eps_key);
    if (a.flags & kSigmoid) {
      wc = 1.f / (1.f + expf(-z));
    } else {
      const float L = a.lse[row];
      const float M = fmaxf(L, z);
      const float ea = expf(L - M), ec = expf(z - M);
      wa = ea / (ea + ec);
      wc = ec / (ea + ec);
    }
    if (a.alpha_p != nullptr && threadIdx.x == 0) a.alpha_p[row] = wc;
  }

  float ssh = 0.f, unused = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      unpack(ro[k], h[k]);
      if (has_p) {
#pragma unroll
        for (int e = 0; e < VE; ++e) h[k][e] = fmaf(wa, h[k][e], wc * p[k][e]);
      }
#pragma unroll
      for (int e = 0; e < VE; ++e) ssh = fmaf(h[k][e], h[k][e], ssh);
    }
  }
  block_sum2(ssh, unused, scratch);
  const float inv = 1.f / sqrtf(ssh / static_cast<float>(a.d) + a.eps_in);

#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      if (a.h) st_global(static_cast<T*>(a.h) + base + v * VE, pack(h[k]));
      float y[VE];
      if (a.gamma_in) {
        const float4* g4 = reinterpret_cast<const float4*>(a.gamma_in + v * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
          const float4 gg = __ldg(g4 + e / 4);
          y[e] = gg.x * (h[k][e] * inv);
          y[e + 1] = gg.y * (h[k][e + 1] * inv);
          y[e + 2] = gg.z * (h[k][e + 2] * inv);
          y[e + 3] = gg.w * (h[k][e + 3] * inv);
        }
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) y[e] = h[k][e] * inv;
      }
      st_global(static_cast<T*>(a.y) + base + v * VE, pack(y));
    }
  }
}

// One CTA per row; every load of the row is issued before any arithmetic.
template <typename T, int VPT>
__global__ void __launch_bounds__(kMergeThreads) phase2_kernel(const Phase2Args a) {
  constexpr int VE = Vec<T>::N;
  __shared__ float scratch[66];
  const int64_t row = blockIdx.x;
  const int nv = a.d / VE;
  const int64_t base = row * a.d;
  uint4 ro[VPT], rp[VPT], rv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      ro[k] = ld_stream(static_cast<const T*>(a.o) + base + v * VE);
      if (a.partial) rp[k] = ld_stream(static_cast<const T*>(a.partial) + base + v * VE);
      if (a.v_prev) rv[k] = ld_stream(static_cast<const T*>(a.v_prev) + base + v * VE);
    }
  }
  merge_row<T, VPT>(a, row, ro, rp, rv, scratch);
}

// Online softmax over the sources, one source per step, with the rows of the next two sources
// already in flight (two register buffers; the source loop is unrolled by two).
template <typename T, int VPT>
__global__ void __launch_bounds__(kRowThreads) full_kernel(const FullArgs a) {
  constexpr int VE = Vec<T>::N;
  __shared__ float scratch[66];
  __shared__ float zs[kMaxSources];
  const int64_t row = blockIdx.x;
  const int nv = a.d / VE;
  const int64_t base = row * a.d;
  const float fd = static_cast<float>(a.d);

  float acc[VPT][VE];
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < VE; ++e) acc[k][e] = 0.f;
  float mrun = -INFINITY, lrun = 0.f;
  // An earlier partition of the sources (phase 1 of a group: normalised o0 and its lse) starts
  // the online softmax: with the running max at lse0 it contributes o0 with exp-sum 1.
  if (a.o0 != nullptr) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) unpack(ld_stream(static_cast<const T*>(a.o0) + base + v * VE), acc[k]);
    }
    if ((a.flags & kSigmoid) == 0) {
      mrun = a.lse0[row];
      lrun = 1.f;
    }
  }

  auto load = [&](uint4 (&r)[VPT], int j) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      r[k] = make_uint4(0u, 0u, 0u, 0u);  // zeros are bf16 and fp32 zeros
      if (v < nv) r[k] = ld_stream(static_cast<const T*>(a.srcs[j]) + base + v * VE);
    }
  };
  // Score source j (held in x), then fold it into the running max, sum and accumulator.
  auto fold = [&](const float (&x)[VPT][VE], int j) {
    float ss = 0.f, dot = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        const float4* u4 = reinterpret_cast<const float4*>(a.u + v * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
          const float4 uu = __ldg(u4 + e / 4);
          dot = fmaf(uu.x, x[k][e], dot);
          dot = fmaf(uu.y, x[k][e + 1], dot);
          dot = fmaf(uu.z, x[k][e + 2], dot);
          dot = fmaf(uu.w, x[k][e + 3], dot);
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) ss = fmaf(x[k][e], x[k][e], ss);
      }
    }
    block_sum2(ss, dot, scratch);
    const float z = (a.flags & kNoKeyNorm) ? dot : dot / sqrtf(ss / fd + a.eps_key);
    if (threadIdx.x == 0) zs[j] = z;
    float sc, ez;
    if (a.flags & kSigmoid) {  // independent weights: no running max, no rescaling
      sc = 1.f;
      ez = 1.f / (1.f + expf(-z));
      mrun = fmaxf(mrun, z);
    } else {
      const float mnew = fmaxf(mrun, z);
      sc = expf(mrun - mnew);  // 0 for the first source (mrun = -inf)
      ez = expf(z - mnew);
      lrun = lrun * sc + ez;
      mrun = mnew;
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[k][e] = fmaf(acc[k][e], sc, ez * x[k][e]);
  };

  uint4 bufA[VPT], bufB[VPT];
  if (a.n > 0) load(bufA, 0);
  if (a.n > 1) load(bufB, 1);
  for (int j = 0; j < a.n; j += 2) {
    float x[VPT][VE];
#pragma unroll
    for (int k = 0; k < VPT; ++k) unpack(bufA[k], x[k]);
    if (j + 2 < a.n) load(bufA, j + 2);
    fold(x, j);
    if (j + 1 < a.n) {  // uniform over the CTA
#pragma unroll
      for (int k = 0; k < VPT; ++k) unpack(bufB[k], x[k]);
      if (j + 3 < a.n) load(bufB, j + 3);
      fold(x, j + 1);
    }
  }

  const bool sigmoid = (a.flags & kSigmoid) != 0;
  const float rl = sigmoid ? 1.f : 1.f / lrun;
  float ssh = 0.f, unused = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      acc[k][e] *= rl;
      ssh = fmaf(acc[k][e], acc[k][e], ssh);
    }
  float inv = 0.f;
  if (a.y != nullptr) {  // uniform over the CTA
    block_sum2(ssh, unused, scratch);  // its barriers also publish zs[]
    inv = 1.f / sqrtf(ssh / fd + a.eps_in);
  } else {
    __syncthreads();  // publish zs[]
  }

  const float lse = mrun + logf(lrun);
  if (threadIdx.x == 0) {
    if (a.m != nullptr) a.m[row] = mrun;
    if (a.lse != nullptr && !sigmoid) a.lse[row] = lse;
  }
  if (a.alpha != nullptr) {
    for (int j = threadIdx.x; j < a.n; j += blockDim.x)
      a.alpha[row * a.n + j] = sigmoid ? 1.f / (1.f + expf(-zs[j])) : expf(zs[j] - lse);
  }
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      if (a.h) st_global(static_cast<T*>(a.h) + base + v * VE, pack(acc[k]));
      if (a.y) {
        float y[VE];
#pragma unroll
        for (int e = 0; e < VE; ++e) y[e] = acc[k][e] * inv;
        if (a.gamma_in) {
          const float4* g4 = reinterpret_cast<const float4*>(a.gamma_in + v * VE);
#pragma unroll
          for (int e = 0; e < VE; e += 4) {
            const float4 gg = __ldg(g4 + e / 4);
            y[e] *= gg.x;
            y[e + 1] *= gg.y;
            y[e + 2] *= gg.z;
            y[e + 3] *= gg.w;
          }
        }
        st_global(static_cast<T*>(a.y) + base + v * VE, pack(y));
      }
    }
  }
}

template <typename T>
__global__ void add_kernel(const T* __restrict__ pa, const T* __restrict__ pb, T* out,
                           int64_t nvec) {
  constexpr int VE = Vec<T>::N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float x[VE], y[VE];
    unpack(ld_stream(pa + i * VE), x);
    unpack(ld_stream(pb + i * VE), y);
#pragma unroll
    for (int e = 0; e < VE; ++e) x[e] += y[e];
    st_global(out + i * VE, pack(x));
  }
}

// u = w * g; with `split`, also rows 2r (hi) and 2r + 1 (lo) of the bf16 split of u:
// hi = bf16(u), lo = bf16(u - hi), both rounded to nearest even.
__global__ void prep_kernel(const float* w, const float* g, float* u, uint16_t* split, int d,
                            int64_t n4) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 x = reinterpret_cast<const float4*>(w)[i];
    if (g != nullptr) {
      const float4 y = reinterpret_cast<const float4*>(g)[i];
      x.x *= y.x;
      x.y *= y.y;
      x.z *= y.z;
      x.w *= y.w;
    }
    reinterpret_cast<float4*>(u)[i] = x;
    if (split != nullptr) {
      const int64_t e = i * 4, r = e / d, c = e - r * d;
      const uint32_t h0 = pack_bf16x2(x.x, x.y), h1 = pack_bf16x2(x.z, x.w);
      const uint32_t l0 = pack_bf16x2(x.x - __uint_as_float(h0 << 16),
                                      x.y - __uint_as_float(h0 & 0xffff0000u));
      const uint32_t l1 = pack_bf16x2(x.z - __uint_as_float(h1 << 16),
                                      x.w - __uint_as_float(h1 & 0xffff0000u));
      *reinterpret_cast<uint2*>(split + (2 * r) * d + c) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(split + (2 * r + 1) * d + c) = make_uint2(l0, l1);
    }
  }
}

// Vectors per thread and threads per CTA for a row of nv 16-byte vectors.
inline void row_geometry(int nv, int& vpt, int& threads, int max_threads = kRowThreads) {
  vpt = 1;
  while ((nv + vpt - 1) / vpt > max_threads) vpt *= 2;
  threads = ((nv + vpt - 1) / vpt + 31) / 32 * 32;
}

template <typename T>
cudaError_t phase2_io(const Phase2Args& a, cudaStream_t s) {
  int vpt, threads;
  row_geometry(a.d / Vec<T>::N, vpt, threads, kMergeThreads);
  const unsigned grid = static_cast<unsigned>(a.T);
  switch (vpt) {
    case 1: phase2_kernel<T, 1><<<grid, threads, 0, s>>>(a); break;
    case 2: phase2_kernel<T, 2><<<grid, threads, 0, s>>>(a); break;
    case 4: phase2_kernel<T, 4><<<grid, threads, 0, s>>>(a); break;
    case 8: phase2_kernel<T, 8><<<grid, threads, 0, s>>>(a); break;
    case 16: phase2_kernel<T, 16><<<grid, threads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t full_io(const FullArgs& a, cudaStream_t s) {
  int vpt, threads;
  row_geometry(a.d / Vec<T>::N, vpt, threads);
  const unsigned grid = static_cast<unsigned>(a.T);
  switch (vpt) {
    case 1: full_kernel<T, 1><<<grid, threads, 0, s>>>(a); break;
    case 2: full_kernel<T, 2><<<grid, threads, 0, s>>>(a); break;
    case 4: full_kernel<T, 4><<<grid, threads, 0, s>>>(a); break;
    case 8: full_kernel<T, 8><<<grid, threads, 0, s>>>(a); break;
    case 16: full_kernel<T, 16><<<grid, threads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

inline unsigned grid_for(int64_t work, int threads) {
  int64_t b = (work + threads - 1) / threads;
  const int64_t cap = 148 * 16;
  return static_cast<unsigned>(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

cudaError_t launch_phase2(IO io, const Phase2Args& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  return io == IO::BF16 ? phase2_io<bf16>(a, s) : phase2_io<float>(a, s);
}


cudaError_t launch_full(IO io, const FullArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  return io == IO::BF16 ? full_io<bf16>(a, s) : full_io<float>(a, s);
}

cudaError_t launch_partial_update(IO io, const void* pa, const void* pb, void* out,
                                  int64_t n_elems, cudaStream_t s) {
  if (n_elems == 0) return cudaSuccess;
  constexpr int threads = 256;
  if (io == IO::BF16) {
    const int64_t nvec = n_elems / 8;
    add_kernel<bf16><<<grid_for(nvec, threads), threads, 0, s>>>(
        static_cast<const bf16*>(pa), static_cast<const bf16*>(pb), static_cast<bf16*>(out), nvec);
  } else {
    const int64_t nvec = n_elems / 4;
    add_kernel<float><<<grid_for(nvec, threads), threads, 0, s>>>(
        static_cast<const float*>(pa), static_cast<const float*>(pb), static_cast<float*>(out),
        nvec);
  }
  return cudaGetLastError();
}

cudaError_t launch_query_prep(const float* w, const float* g, float* u, void* u_split, int rows,
                              int d, cudaStream_t s) {
  const int64_t n_elems = static_cast<int64_t>(rows) * d;
  if (n_elems == 0) return cudaSuccess;
  constexpr int threads = 256;
  prep_kernel<<<grid_for(n_elems / 4, threads), threads, 0, s>>>(
      w, g, u, static_cast<uint16_t*>(u_split), d, n_elems / 4);
  return cudaGetLastError();
}

}  // namespace attnres
