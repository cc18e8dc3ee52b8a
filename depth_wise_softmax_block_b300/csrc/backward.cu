// Backward of one sublayer's depth aggregation over an explicit source list, with the key and
// input RMSNorms ("Attention Residuals" note §7: the logit gradient
// dL/dz_i = alpha_i g_h^T (v_i - h); "Attention Residuals 阅读补充", section "梯度沿切向传播":
// the RMSNorm input gradient (1/r)(g' - yhat (yhat^T g') / d) with g' = gamma ⊙ g).
//
// Forward, per token:  r_i = rms(v_i), z_i = u . v_i / r_i (u = w ⊙ gamma_key folded),
// alpha = softmax(z), h = sum_i alpha_i v_i, y = gamma_in ⊙ h / r_h.
// Backward, given g_y = dL/dy:
//   g_h   = (gamma_in ⊙ g_y) / r_h - h (sum gamma_in g_y h) / (d r_h^3)
//   dz_i  = alpha_i (g_h . v_i - g_h . h),   with g_h . h = sum_j alpha_j (g_h . v_j)
//   dv_i  = alpha_i g_h + (dz_i / r_i) u - (dz_i z_i / (d r_i^2)) v_i
//   du   += sum_i (dz_i / r_i) v_i          dgamma_in += g_y ⊙ h / r_h       (over tokens)
//
// Persistent CTAs (two per SM) walk token rows.  Per row, four passes over the row's sources
// (the first from HBM, the others mostly from L1/L2):
//   A  one warp per quarter of a source row: its sum of squares and u . v_i (warp reductions),
//      the quarters added in shared memory, so r_i and z_i;
//   B  one thread per column (the same columns for every row): h, the input norm (one CTA
//      reduction of two values) and g_h, which goes to shared memory;
//   C  one warp per quarter of a source row: g_h . v_i;
//   D  one thread per column: dv_i for every source and the row's du contribution, summed over
//      the sources in registers and added to the CTA's du partial sums.
// The partial sums of du and dgamma_in live in shared memory with column (v, e) at e * nv + v,
// so the threads of a warp touch consecutive words; one atomic per element at the end.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace attnres {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBatch = 8;  // 16-byte vectors per lane in flight in the per-source passes
constexpr int kParts = 4;  // a source row is split into this many column ranges, one warp each

// Warp-wide sums over one source row: sum of squares and dot product with a second vector,
// `other(v, f)` filling the 8 (bf16) or 4 (fp32) floats of the second vector at vector v.
template <typename T, typename Other>
__device__ __forceinline__ void row_dots(const T* p, int nv, int lane, Other other, float& ss,
                                         float& dot) {
  constexpr int VE = Vec<T>::N;
  ss = 0.f;
  dot = 0.f;
  for (int v0 = lane; v0 < nv; v0 += 32 * kBatch) {
    uint4 raw[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int v = v0 + 32 * b;
      raw[b] = v < nv ? __ldg(reinterpret_cast<const uint4*>(p + v * VE)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int v = v0 + 32 * b;
      if (v < nv) {
        float x[VE], o[VE];
        unpack(raw[b], x);
        other(v, o);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          ss = fmaf(x[e], x[e], ss);
          dot = fmaf(o[e], x[e], dot);
        }
      }
    }
  }
  ss = warp_sum(ss);
  dot = warp_sum(dot);
}

template <typename T, int VPT>
__global__ void __launch_bounds__(kBwdThreads, 2) backward_kernel(const BwdArgs a) {
  constexpr int VE = Vec<T>::N;
  constexpr int NM = kBwdMaxSources;
  extern __shared__ float sm[];
  const int d = a.d, nv = d / VE, n = a.n;
  float* acc_du = sm;         // [VE][nv]: this CTA's du partial sums
  float* acc_dg = sm + d;     // [VE][nv]: its dgamma_in partial sums
  float* ghs = sm + 2 * d;    // [nv][VE]: g_h of the current row
  __shared__ float st_r[NM], st_z[NM], st_pq[NM];  // per source: r_i, z_i, g_h . v_i
  __shared__ float cf_u[NM], cf_v[NM];             // per source: dz_i / r_i, dz_i z_i / (d r_i^2)
  __shared__ float st_hs[kParts * NM], st_hd[kParts * NM];  // per row part: sum of squares, dot
  __shared__ float scratch[66];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float fd = static_cast<float>(d);
  for (int i = tid; i < 2 * d; i += blockDim.x) sm[i] = 0.f;
  __syncthreads();
  pdl_enter();  // the prologue above touches no global memory

  const float4* u4 = reinterpret_cast<const float4*>(a.u);
  const float4* g4 = reinterpret_cast<const float4*>(a.gamma_in);  // may be null
  auto load = [&](const void* p, int64_t off, float (&x)[VE]) {
    unpack(__ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p) + off)), x);
  };
  auto load4s = [&](const float4* p, int v, float (&f)[VE]) {  // VE floats of a float4 array
#pragma unroll
    for (int e = 0; e < VE; e += 4) {
      const float4 q = __ldg(p + (v * VE + e) / 4);
      f[e] = q.x;
      f[e + 1] = q.y;
      f[e + 2] = q.z;
      f[e + 3] = q.w;
    }
  };

  for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
    const int64_t base = row * d;
    // ---- pass A: r_i and z_i, one warp per quarter of a source row ----
    for (int t = warp; t < kParts * n; t += kBwdWarps) {
      const int j = t / kParts, q = t - j * kParts;
      const int vb = q * nv / kParts, vc = (q + 1) * nv / kParts - vb;
      float ss, dot;
      row_dots<T>(static_cast<const T*>(a.srcs[j]) + base + vb * VE, vc, lane,
                  [&](int v, float (&f)[VE]) { load4s(u4, v + vb, f); }, ss, dot);
      if (lane == 0) {
        st_hs[t] = ss;
        st_hd[t] = dot;
      }
    }
    __syncthreads();
    if (tid < n) {
      float ss = 0.f, dot = 0.f;
#pragma unroll
      for (int q = 0; q < kParts; ++q) {
        ss += st_hs[kParts * tid + q];
        dot += st_hd[kParts * tid + q];
      }
      const float r = sqrtf(ss / fd + a.eps_key);
      st_r[tid] = r;
      st_z[tid] = dot / r;
    }
    __syncthreads();
    float al[NM];
    {
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < NM; ++j)
        if (j < n) m = fmaxf(m, st_z[j]);
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < NM; ++j) {
        al[j] = j < n ? expf(st_z[j] - m) : 0.f;
        l += al[j];
      }
      const float rl = 1.f / l;
#pragma unroll
      for (int j = 0; j < NM; ++j) al[j] *= rl;
    }

    // ---- pass B: h, the input norm and g_h, one thread per column ----
    float h[VPT][VE], gh[VPT][VE];
    float ssh = 0.f, s1 = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * blockDim.x;
#pragma unroll
      for (int e = 0; e < VE; ++e) h[k][e] = gh[k][e] = 0.f;
      if (v < nv) {
#pragma unroll
        for (int j = 0; j < NM; ++j) {
          if (j < n) {
            float x[VE];
            load(a.srcs[j], base + v * VE, x);
#pragma unroll
            for (int e = 0; e < VE; ++e) h[k][e] = fmaf(al[j], x[e], h[k][e]);
          }
        }
        float g[VE], gi[VE];
        load(a.g_y, base + v * VE, g);
        if (g4) {
          load4s(g4, v, gi);
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) gi[e] = 1.f;
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          gh[k][e] = gi[e] * g[e];  // gamma_in ⊙ g_y for now
          ssh = fmaf(h[k][e], h[k][e], ssh);
          s1 = fmaf(gh[k][e], h[k][e], s1);
        }
      }
    }
    block_sum2(ssh, s1, scratch);
    const float rh = sqrtf(ssh / fd + a.eps_in);
    const float c1 = 1.f / rh, c2 = s1 / (fd * rh * rh * rh);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * blockDim.x;
      if (v < nv) {
        float g[VE];
        load(a.g_y, base + v * VE, g);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          acc_dg[e * nv + v] = fmaf(g[e] * h[k][e], c1, acc_dg[e * nv + v]);
          gh[k][e] = gh[k][e] * c1 - h[k][e] * c2;
        }
        float4* gs = reinterpret_cast<float4*>(ghs + v * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4)
          gs[e / 4] = make_float4(gh[k][e], gh[k][e + 1], gh[k][e + 2], gh[k][e + 3]);
      }
    }
    __syncthreads();

    // ---- pass C: g_h . v_i, one warp per quarter of a source row ----
    for (int t = warp; t < kParts * n; t += kBwdWarps) {
      const int j = t / kParts, q = t - j * kParts;
      const int vb = q * nv / kParts, vc = (q + 1) * nv / kParts - vb;
      float ss, dot;
      row_dots<T>(static_cast<const T*>(a.srcs[j]) + base + vb * VE, vc, lane,
                  [&](int v, float (&f)[VE]) {
                    const float4* gs = reinterpret_cast<const float4*>(ghs + (v + vb) * VE);
#pragma unroll
                    for (int e = 0; e < VE; e += 4) {
                      const float4 q = gs[e / 4];
                      f[e] = q.x;
                      f[e + 1] = q.y;
                      f[e + 2] = q.z;
                      f[e + 3] = q.w;
                    }
                  },
                  ss, dot);
      if (lane == 0) st_hd[t] = dot;
    }
    __syncthreads();
    if (tid < n) {
      float dot = 0.f;
#pragma unroll
      for (int q = 0; q < kParts; ++q) dot += st_hd[kParts * tid + q];
      st_pq[tid] = dot;
    }
    __syncthreads();
    if (tid < n) {  // coefficients of dv_i; g_h . h = sum_j alpha_j (g_h . v_j)
      float ghh = 0.f;
#pragma unroll
      for (int j = 0; j < NM; ++j)
        if (j < n) ghh = fmaf(al[j], st_pq[j], ghh);
      const int j = tid;
      const float r = st_r[j], z = st_z[j];
      float aj = 0.f;
#pragma unroll
      for (int i = 0; i < NM; ++i)
        if (i == j) aj = al[i];
      const float dz = aj * (st_pq[j] - ghh);
      cf_u[j] = dz / r;
      cf_v[j] = dz * z / (fd * r * r);
    }
    __syncthreads();

    // ---- pass D: dv_i and du, one thread per column ----
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * blockDim.x;
      if (v < nv) {
        float uu[VE], dacc[VE];
        load4s(u4, v, uu);
#pragma unroll
        for (int e = 0; e < VE; ++e) dacc[e] = 0.f;
#pragma unroll
        for (int j = 0; j < NM; ++j) {
          if (j < n) {
            float x[VE], o[VE];
            load(a.srcs[j], base + v * VE, x);
            const float cu = cf_u[j], cv = cf_v[j];
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              o[e] = fmaf(al[j], gh[k][e], fmaf(cu, uu[e], -cv * x[e]));
              dacc[e] = fmaf(cu, x[e], dacc[e]);
            }
            st_global(static_cast<T*>(a.dsrcs[j]) + base + v * VE, pack(o));
          }
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) acc_du[e * nv + v] += dacc[e];
      }
    }
  }
  __syncthreads();
  for (int c = tid; c < d; c += blockDim.x) {
    const int v = c / VE, e = c - v * VE;
    atomicAdd(a.du + c, acc_du[e * nv + v]);
    if (a.dgamma_in != nullptr) atomicAdd(a.dgamma_in + c, acc_dg[e * nv + v]);
  }
}

template <typename T>
cudaError_t backward_io(const BwdArgs& a, cudaStream_t s) {
  const int nv = a.d / Vec<T>::N;
  const int vpt = (nv + kBwdThreads - 1) / kBwdThreads;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(a.T, 2 * sms));
  const int smem = 3 * a.d * static_cast<int>(sizeof(float));
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r != cudaSuccess) return r;
    return launch_pdl(kern, grid, kBwdThreads, smem, s, a);
  };
  switch (vpt) {
    case 1: return launch(backward_kernel<T, 1>);
    case 2: return launch(backward_kernel<T, 2>);
    case 3: return launch(backward_kernel<T, 3>);
    case 4: return launch(backward_kernel<T, 4>);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_backward(IO io, const BwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  return io == IO::BF16 ? backward_io<bf16>(a, s) : backward_io<float>(a, s);
}

}  // namespace attnres
