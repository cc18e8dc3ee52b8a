// Backward of one sublayer's depth aggregation over an explicit source list, with the key and
// input RMSNorms ("Attention Residuals" note §7: the logit gradient
// dL/dz_i = alpha_i g_h^T (v_i - h); "Attention Residuals 阅读补充", section "梯度沿切向传播":
// the RMSNorm input gradient (1/r)(g' - yhat (yhat^T g') / d) with g' = gamma ⊙ g).
//
// Forward, per token:  r_i = rms(v_i), z_i = u . v_i / r_i (u = w ⊙ gamma_key folded),
// alpha = softmax(z), h = sum_i alpha_i v_i, y = gamma_in ⊙ h / r_h.
// Backward, given g_y = dL/dy:
//   g_h   = (gamma_in ⊙ g_y) / r_h - h (sum gamma_in g_y h) / (d r_h^3)
//   dz_i  = alpha_i (g_h . v_i - g_h . h)
//   dv_i  = alpha_i g_h + (dz_i / r_i) u - (dz_i z_i / (d r_i^2)) v_i
//   du   += sum_i (dz_i / r_i) v_i          dgamma_in += g_y ⊙ h / r_h       (over tokens)
//
// A persistent CTA walks token rows; each thread owns the same columns of every row, so the
// CTA's partial sums of du and dgamma_in accumulate in shared memory without conflicts and are
// added to the outputs with one atomic per element at the end.  Per row, four passes over the
// n source rows (the first from HBM, the others from L1, where a row's sources fit): logits,
// h and the norm, the logit gradients, the outputs.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace attnres {
namespace {

constexpr int kBwdThreads = 256;

template <typename T, int VPT>
__global__ void __launch_bounds__(kBwdThreads, 1) backward_kernel(const BwdArgs a) {
  constexpr int VE = Vec<T>::N;
  constexpr int NM = kBwdMaxSources;
  extern __shared__ float acc_s[];  // [2][d]: this CTA's du and dgamma_in partial sums
  __shared__ float scratch[2 * NM * 33];
  const int nv = a.d / VE, n = a.n, d = a.d;
  const float fd = static_cast<float>(d);
  for (int i = threadIdx.x; i < 2 * d; i += blockDim.x) acc_s[i] = 0.f;
  __syncthreads();

  // Cached loads: the four passes over a row's sources re-read them from L1.
  auto load = [&](const void* p, int64_t base, int v, float (&x)[VE]) {
    unpack(__ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p) + base + v * VE)), x);
  };

  for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
    const int64_t base = row * d;
    // ---- pass A: sums of squares and logit numerators of every source ----
    float part[2 * NM];
#pragma unroll
    for (int j = 0; j < 2 * NM; ++j) part[j] = 0.f;
#pragma unroll
    for (int j = 0; j < NM; ++j) {
      if (j < n) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int v = threadIdx.x + k * blockDim.x;
          if (v < nv) {
            float x[VE];
            load(a.srcs[j], base, v, x);
            const float* up = a.u + v * VE;
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              part[2 * j] = fmaf(x[e], x[e], part[2 * j]);
              part[2 * j + 1] = fmaf(__ldg(up + e), x[e], part[2 * j + 1]);
            }
          }
        }
      }
    }
    block_sum_n<2 * NM>(part, scratch);
    float r[NM], z[NM], al[NM];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NM; ++j) {
      r[j] = sqrtf(part[2 * j] / fd + a.eps_key);
      z[j] = j < n ? part[2 * j + 1] / r[j] : -INFINITY;
      m = fmaxf(m, z[j]);
    }
    float l = 0.f;
#pragma unroll
    for (int j = 0; j < NM; ++j) {
      al[j] = j < n ? expf(z[j] - m) : 0.f;
      l += al[j];
    }
#pragma unroll
    for (int j = 0; j < NM; ++j) al[j] /= l;

    // ---- pass B: h, the input norm and its input gradient g_h ----
    float h[VPT][VE], gh[VPT][VE];
    float ssh = 0.f, s1 = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
#pragma unroll
      for (int e = 0; e < VE; ++e) h[k][e] = 0.f;
      if (v < nv) {
#pragma unroll
        for (int j = 0; j < NM; ++j) {
          if (j < n) {
            float x[VE];
            load(a.srcs[j], base, v, x);
#pragma unroll
            for (int e = 0; e < VE; ++e) h[k][e] = fmaf(al[j], x[e], h[k][e]);
          }
        }
        float g[VE];
        load(a.g_y, base, v, g);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float gi = a.gamma_in ? __ldg(a.gamma_in + v * VE + e) : 1.f;
          gh[k][e] = gi * g[e];  // gamma_in ⊙ g_y for now
          ssh = fmaf(h[k][e], h[k][e], ssh);
          s1 = fmaf(gh[k][e], h[k][e], s1);
        }
      }
    }
    block_sum2(ssh, s1, scratch);
    const float rh = sqrtf(ssh / fd + a.eps_in);
    const float c1 = 1.f / rh, c2 = s1 / (fd * rh * rh * rh);
    float pq[NM + 1];
#pragma unroll
    for (int j = 0; j <= NM; ++j) pq[j] = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        float g[VE];
        load(a.g_y, base, v, g);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          acc_s[d + v * VE + e] += g[e] * h[k][e] * c1;  // dgamma_in
          gh[k][e] = gh[k][e] * c1 - h[k][e] * c2;
          pq[NM] = fmaf(gh[k][e], h[k][e], pq[NM]);
        }
      }
    }

    // ---- pass C: g_h . v_i for the logit gradients ----
#pragma unroll
    for (int j = 0; j < NM; ++j) {
      if (j < n) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int v = threadIdx.x + k * blockDim.x;
          if (v < nv) {
            float x[VE];
            load(a.srcs[j], base, v, x);
#pragma unroll
            for (int e = 0; e < VE; ++e) pq[j] = fmaf(gh[k][e], x[e], pq[j]);
          }
        }
      }
    }
    block_sum_n<NM + 1>(pq, scratch);

    // ---- pass D: source gradients and the du partial sums ----
#pragma unroll
    for (int j = 0; j < NM; ++j) {
      if (j < n) {
        const float dz = al[j] * (pq[j] - pq[NM]);
        const float cu = dz / r[j];
        const float cv = dz * z[j] / (fd * r[j] * r[j]);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int v = threadIdx.x + k * blockDim.x;
          if (v < nv) {
            float x[VE], o[VE];
            load(a.srcs[j], base, v, x);
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              const float uu = __ldg(a.u + v * VE + e);
              o[e] = fmaf(al[j], gh[k][e], fmaf(cu, uu, -cv * x[e]));
              acc_s[v * VE + e] = fmaf(cu, x[e], acc_s[v * VE + e]);
            }
            st_global(static_cast<T*>(a.dsrcs[j]) + base + v * VE, pack(o));
          }
        }
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    atomicAdd(a.du + i, acc_s[i]);
    if (a.dgamma_in != nullptr) atomicAdd(a.dgamma_in + i, acc_s[d + i]);
  }
}

template <typename T>
cudaError_t backward_io(const BwdArgs& a, cudaStream_t s) {
  const int nv = a.d / Vec<T>::N;
  int vpt = 1;
  while ((nv + vpt - 1) / vpt > kBwdThreads) vpt *= 2;
  const int threads = ((nv + vpt - 1) / vpt + 31) / 32 * 32;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(a.T, sms));
  const int smem = 2 * a.d * static_cast<int>(sizeof(float));
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r != cudaSuccess) return r;
    kern<<<grid, threads, smem, s>>>(a);
    return cudaGetLastError();
  };
  switch (vpt) {
    case 1: return launch(backward_kernel<T, 1>);
    case 2: return launch(backward_kernel<T, 2>);
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
