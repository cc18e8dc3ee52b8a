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
// Both take the Table 4 variants ("Attention Residuals" note, result 4): the flags (sigmoid
// weights, no key RMSNorm) and depth-attention heads (H contiguous feature slices, each with its
// own key RMS, logit and softmax; the input RMSNorm over the whole row).
//   phase2_heads_kernel, full_heads_kernel
//                  the same two with H <= 16 heads of at most 128 vectors: one warp per head,
//                  so every per-head sum is a warp reduction (the other head counts go through
//                  the generic kernels' per-head reduction in shared memory).
//   add_kernel     partial-sum update / block close: out = partial + v.
//   prep_kernel    query preparation u = w ⊙ gamma_key (and its bf16 hi/lo split).
//
// In the generic kernels each thread owns VPT 16-byte vectors of the row (vector v =
// threadIdx.x + k * blockDim.x).  Every kernel is launched with programmatic stream
// serialisation and enters through pdl_enter() (common.cuh).
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

// Per-head sums of two per-vector partials (depth-attention heads: the row's nv 16-byte vectors
// split into H heads of nvh consecutive vectors).  Thread-owned vector v = threadIdx.x + k *
// blockDim.x contributes pa[k], pb[k].  `red` holds 2 * nv floats of shared memory; on return
// hs[h] and hs[H + h] hold head h's two sums, summed in a fixed order, for every thread.
template <int VPT>
__device__ __forceinline__ void head_sum2(const float (&pa)[VPT], const float (&pb)[VPT], int nv,
                                          int nvh, int H, float* red, float* hs) {
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      red[v] = pa[k];
      red[nv + v] = pb[k];
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int h = warp; h < H; h += nw) {
    float sa = 0.f, sb = 0.f;
    for (int i = lane; i < nvh; i += 32) {
      sa += red[h * nvh + i];
      sb += red[nv + h * nvh + i];
    }
    sa = warp_sum(sa);
    sb = warp_sum(sb);
    if (lane == 0) {
      hs[h] = sa;
      hs[H + h] = sb;
    }
  }
  __syncthreads();
}

// Phase 2 of one row from the vectors this thread holds (vector v = threadIdx.x + k *
// blockDim.x of the row): o_l in ro, the stored partial in rp, v_prev in rv (each used only if
// the corresponding input is present).  Ends with the row's stores; `scratch` is the CTA's
// reduction buffer (the block reductions synchronise the CTA).  kHeads: H > 1 depth-attention
// heads, each merging its slice with its own z_p and lse; `red` is then 2 * nv + 2 * H floats of
// shared memory.
template <typename T, typename TO, int VPT, bool kHeads>
__device__ __forceinline__ void merge_row(const Phase2Args& a, int64_t row,
                                          const uint4 (&ro)[VPT][OWords<TO, Vec<T>::N>::N],
                                          const uint4 (&rp)[VPT], const uint4 (&rv)[VPT],
                                          float* scratch, float* red) {
  constexpr int VE = Vec<T>::N;
  const int nv = a.d / VE;
  const int H = kHeads ? a.heads : 1;
  const int nvh = nv / H;
  const int64_t base = row * a.d;
  const bool has_p = a.partial != nullptr || a.v_prev != nullptr;

  float h[VPT][VE];
  float p[VPT][VE];
  float wa[VPT], wc[VPT];  // weights of o_l and of p for the head of each vector
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    wa[k] = 1.f;
    wc[k] = 0.f;
  }
  if (has_p) {
    // per-vector partial sums with heads; everything in slot 0 without
    float ssv[VPT], dtv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) ssv[k] = dtv[k] = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      const int kq = kHeads ? k : 0;
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
          dtv[kq] = fmaf(uu.x, p[k][e], dtv[kq]);
          dtv[kq] = fmaf(uu.y, p[k][e + 1], dtv[kq]);
          dtv[kq] = fmaf(uu.z, p[k][e + 2], dtv[kq]);
          dtv[kq] = fmaf(uu.w, p[k][e + 3], dtv[kq]);
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) ssv[kq] = fmaf(p[k][e], p[k][e], ssv[kq]);
      }
    }
    // Online-softmax merge of the phase-1 partition (lse) with the partial source (z_p); with
    // sigmoid weights the two partitions simply add, h = o + sigmoid(z_p) p.
    const float fdh = static_cast<float>(a.d / H);
    auto weights = [&](float ssp, float dot, int hd, float& w_o, float& w_p) {
      const float z = (a.flags & kNoKeyNorm) ? dot : dot / sqrtf(ssp / fdh + a.eps_key);
      if (a.flags & kSigmoid) {
        w_o = 1.f;
        w_p = 1.f / (1.f + expf(-z));
      } else {
        const float L = a.lse[static_cast<int64_t>(hd) * a.T + row];
        const float M = fmaxf(L, z);
        const float ea = expf(L - M), ec = expf(z - M);
        w_o = ea / (ea + ec);
        w_p = ec / (ea + ec);
      }
    };
    if constexpr (!kHeads) {
      block_sum2(ssv[0], dtv[0], scratch);
      float w_o, w_p;
      weights(ssv[0], dtv[0], 0, w_o, w_p);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        wa[k] = w_o;
        wc[k] = w_p;
      }
      if (a.alpha_p != nullptr && threadIdx.x == 0) a.alpha_p[row] = w_p;
    } else {
      float* hsum = red + 2 * nv;
      head_sum2(ssv, dtv, nv, nvh, H, red, hsum);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
        const int hd = v < nv ? v / nvh : 0;
        weights(hsum[hd], hsum[H + hd], hd, wa[k], wc[k]);
      }
      if (a.alpha_p != nullptr) {
        for (int hd = threadIdx.x; hd < H; hd += blockDim.x) {
          float w_o, w_p;
          weights(hsum[hd], hsum[H + hd], hd, w_o, w_p);
          a.alpha_p[static_cast<int64_t>(hd) * a.T + row] = w_p;
        }
      }
    }
  }

  float ssh = 0.f, unused = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      unpack_w<TO, VE>(ro[k], h[k]);
      if (has_p) {
#pragma unroll
        for (int e = 0; e < VE; ++e) h[k][e] = fmaf(wa[k], h[k][e], wc[k] * p[k][e]);
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

// One CTA per row; every load of the row is issued before any arithmetic.  TO: the type o_l is
// stored in (the I/O type, or fp32 with kOF32).
template <typename T, typename TO, int VPT, bool kHeads>
__global__ void __launch_bounds__(kMergeThreads) phase2_kernel(const Phase2Args a) {
  constexpr int VE = Vec<T>::N;
  __shared__ float scratch[66];
  extern __shared__ float red[];  // kHeads: [2 * nv + 2 * H]
  pdl_enter();
  const int64_t row = blockIdx.x;
  const int nv = a.d / VE;
  const int64_t base = row * a.d;
  uint4 ro[VPT][OWords<TO, VE>::N], rp[VPT], rv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      ld_stream_w<TO, VE>(static_cast<const TO*>(a.o) + base + v * VE, ro[k]);
      if (a.partial) rp[k] = ld_stream(static_cast<const T*>(a.partial) + base + v * VE);
      if (a.v_prev) rv[k] = ld_stream(static_cast<const T*>(a.v_prev) + base + v * VE);
    }
  }
  merge_row<T, TO, VPT, kHeads>(a, row, ro, rp, rv, scratch, red);
}

// Online softmax over the sources, one source per step, with the rows of the next two sources
// already in flight (two register buffers; the source loop is unrolled by two).  kHeads: H > 1
// depth-attention heads, each with its own running max and sum (kept per vector: a thread's
// vectors may lie in different heads); dynamic shared memory then holds
// [2 * nv reduction | 2 * H head sums | n * H logits | H log-sum-exps] floats.
template <typename T, int VPT, bool kHeads>
__global__ void __launch_bounds__(kRowThreads) full_kernel(const FullArgs a) {
  constexpr int VE = Vec<T>::N;
  constexpr int KS = kHeads ? VPT : 1;  // online-softmax states
  __shared__ float scratch[66];
  __shared__ float zs[kHeads ? 1 : kMaxSources];
  extern __shared__ float dyn[];
  pdl_enter();
  const int64_t row = blockIdx.x;
  const int nv = a.d / VE;
  const int H = kHeads ? a.heads : 1;
  const int nvh = nv / H;
  const int64_t base = row * a.d;
  const float fd = static_cast<float>(a.d);
  const float fdh = static_cast<float>(a.d / H);
  float* red = dyn;
  float* hsum = dyn + 2 * nv;
  float* zsh = hsum + 2 * H;   // [n][H]
  float* hl = zsh + a.n * H;   // [H]
  int hv[VPT];                 // head of each of the thread's vectors
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    hv[k] = (kHeads && v < nv) ? v / nvh : 0;
  }

  float acc[VPT][VE];
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < VE; ++e) acc[k][e] = 0.f;
  float mrun[KS], lrun[KS];
#pragma unroll
  for (int k = 0; k < KS; ++k) {
    mrun[k] = -INFINITY;
    lrun[k] = 0.f;
  }
  // An earlier partition of the sources (phase 1 of a group: normalised o0 and its lse) starts
  // the online softmax: with the running max at lse0 it contributes o0 with exp-sum 1.
  if (a.o0 != nullptr) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        if (a.o0_f32) {
          uint4 r[OWords<float, VE>::N];
          ld_stream_w<float, VE>(static_cast<const float*>(a.o0) + base + v * VE, r);
          unpack_w<float, VE>(r, acc[k]);
        } else {
          unpack(ld_stream(static_cast<const T*>(a.o0) + base + v * VE), acc[k]);
        }
      }
    }
    if ((a.flags & kSigmoid) == 0) {
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        mrun[k] = a.lse0[static_cast<int64_t>(hv[k]) * a.T + row];
        lrun[k] = 1.f;
      }
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
  auto logit = [&](float ss, float dot) {
    return (a.flags & kNoKeyNorm) ? dot : dot / sqrtf(ss / fdh + a.eps_key);
  };
  // Score source j (held in x), then fold it into the running max, sum and accumulator.
  auto fold = [&](const float (&x)[VPT][VE], int j) {
    float ss[KS], dot[KS];
#pragma unroll
    for (int k = 0; k < KS; ++k) ss[k] = dot[k] = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      const int kq = kHeads ? k : 0;
      if (v < nv) {
        const float4* u4 = reinterpret_cast<const float4*>(a.u + v * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
          const float4 uu = __ldg(u4 + e / 4);
          dot[kq] = fmaf(uu.x, x[k][e], dot[kq]);
          dot[kq] = fmaf(uu.y, x[k][e + 1], dot[kq]);
          dot[kq] = fmaf(uu.z, x[k][e + 2], dot[kq]);
          dot[kq] = fmaf(uu.w, x[k][e + 3], dot[kq]);
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) ss[kq] = fmaf(x[k][e], x[k][e], ss[kq]);
      }
    }
    float z[KS];
    if constexpr (!kHeads) {
      block_sum2(ss[0], dot[0], scratch);
      z[0] = logit(ss[0], dot[0]);
      if (threadIdx.x == 0) zs[j] = z[0];
    } else {
      head_sum2(ss, dot, nv, nvh, H, red, hsum);
#pragma unroll
      for (int k = 0; k < KS; ++k) z[k] = logit(hsum[hv[k]], hsum[H + hv[k]]);
      for (int hd = threadIdx.x; hd < H; hd += blockDim.x)
        zsh[j * H + hd] = logit(hsum[hd], hsum[H + hd]);
    }
    float sc[KS], ez[KS];
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      if (a.flags & kSigmoid) {  // independent weights: no running max, no rescaling
        sc[k] = 1.f;
        ez[k] = 1.f / (1.f + expf(-z[k]));
        mrun[k] = fmaxf(mrun[k], z[k]);
      } else {
        const float mnew = fmaxf(mrun[k], z[k]);
        sc[k] = expf(mrun[k] - mnew);  // 0 for the first source (mrun = -inf)
        ez[k] = expf(z[k] - mnew);
        lrun[k] = lrun[k] * sc[k] + ez[k];
        mrun[k] = mnew;
      }
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int kq = kHeads ? k : 0;
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[k][e] = fmaf(acc[k][e], sc[kq], ez[kq] * x[k][e]);
    }
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
  float ssh = 0.f, unused = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int kq = kHeads ? k : 0;
    const float rl = sigmoid ? 1.f : 1.f / lrun[kq];
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      acc[k][e] *= rl;
      ssh = fmaf(acc[k][e], acc[k][e], ssh);
    }
  }
  // Statistics: one writer per head (thread 0, or the owner of the head's first vector).
  float lse0 = 0.f;
  if constexpr (!kHeads) {
    lse0 = mrun[0] + logf(lrun[0]);
    if (threadIdx.x == 0) {
      if (a.m != nullptr) a.m[row] = mrun[0];
      if (a.lse != nullptr && !sigmoid) a.lse[row] = lse0;
    }
  } else {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv && v % nvh == 0) {
        const float l = mrun[k] + logf(lrun[k]);
        const int64_t at = static_cast<int64_t>(hv[k]) * a.T + row;
        if (a.m != nullptr) a.m[at] = mrun[k];
        if (a.lse != nullptr && !sigmoid) a.lse[at] = l;
        hl[hv[k]] = l;
      }
    }
  }
  float inv = 0.f;
  if (a.y != nullptr) {  // uniform over the CTA
    block_sum2(ssh, unused, scratch);  // its barriers also publish zs[] and hl[]
    inv = 1.f / sqrtf(ssh / fd + a.eps_in);
  } else {
    __syncthreads();  // publish zs[] and hl[]
  }

  if (a.alpha != nullptr) {
    if constexpr (!kHeads) {
      for (int j = threadIdx.x; j < a.n; j += blockDim.x)
        a.alpha[row * a.n + j] = sigmoid ? 1.f / (1.f + expf(-zs[j])) : expf(zs[j] - lse0);
    } else {
      for (int i = threadIdx.x; i < H * a.n; i += blockDim.x) {
        const int hd = i / a.n, j = i - hd * a.n;
        const float zj = zsh[j * H + hd];
        a.alpha[(static_cast<int64_t>(hd) * a.T + row) * a.n + j] =
            sigmoid ? 1.f / (1.f + expf(-zj)) : expf(zj - hl[hd]);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      if (a.h) {
        if (a.h_f32)
          st_vec<float, VE>(static_cast<float*>(a.h) + base + v * VE, acc[k]);
        else
          st_global(static_cast<T*>(a.h) + base + v * VE, pack(acc[k]));
      }
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

// ---- depth-attention heads, head-aligned: one warp per head ------------------------------
// For H <= 16 heads of at most 32 * VH vectors: warp w owns head w and lane l the vectors
// l + 32 q (q < VH) of it, so every per-head sum is a warp reduction (no shared memory, no
// CTA barrier); only the input RMSNorm over the whole row takes one CTA reduction.
constexpr int kHeadWarpsMax = 16;

// Resident CTAs per SM asked of the compiler (registers), for enough loads in flight.
template <int VH> constexpr int heads_min_blocks() { return VH <= 2 ? 2 : 1; }

template <typename T, typename TO, int VH>
__global__ void __launch_bounds__(kHeadWarpsMax * 32, heads_min_blocks<VH>())
    phase2_heads_kernel(const Phase2Args a) {
  constexpr int VE = Vec<T>::N;
  __shared__ float scratch[66];
  pdl_enter();
  const int64_t row = blockIdx.x;
  const int hd = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvh = a.d / VE / a.heads;
  const int64_t base = row * a.d + static_cast<int64_t>(hd) * nvh * VE;  // the head's slice
  const bool has_p = a.partial != nullptr || a.v_prev != nullptr;
  uint4 ro[VH][OWords<TO, VE>::N], rp[VH], rv[VH];
#pragma unroll
  for (int q = 0; q < VH; ++q) {
    const int i = lane + 32 * q;
    if (i < nvh) {
      ld_stream_w<TO, VE>(static_cast<const TO*>(a.o) + base + i * VE, ro[q]);
      if (a.partial) rp[q] = ld_stream(static_cast<const T*>(a.partial) + base + i * VE);
      if (a.v_prev) rv[q] = ld_stream(static_cast<const T*>(a.v_prev) + base + i * VE);
    }
  }
  const float* u = a.u + static_cast<int64_t>(hd) * nvh * VE;
  float p[VH][VE];
  float wa = 1.f, wc = 0.f;
  if (has_p) {
    float ss = 0.f, dot = 0.f;
#pragma unroll
    for (int q = 0; q < VH; ++q) {
      const int i = lane + 32 * q;
#pragma unroll
      for (int e = 0; e < VE; ++e) p[q][e] = 0.f;
      if (i < nvh) {
        float y[VE];
        if (a.partial) unpack(rp[q], p[q]);
        if (a.v_prev) {
          unpack(rv[q], y);
#pragma unroll
          for (int e = 0; e < VE; ++e) p[q][e] += y[e];
        }
        if (a.partial_out)
          st_global(static_cast<T*>(a.partial_out) + base + i * VE, pack(p[q]));
        const float4* u4 = reinterpret_cast<const float4*>(u + i * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
          const float4 uu = __ldg(u4 + e / 4);
          dot = fmaf(uu.x, p[q][e], dot);
          dot = fmaf(uu.y, p[q][e + 1], dot);
          dot = fmaf(uu.z, p[q][e + 2], dot);
          dot = fmaf(uu.w, p[q][e + 3], dot);
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) ss = fmaf(p[q][e], p[q][e], ss);
      }
    }
    ss = warp_sum(ss);
    dot = warp_sum(dot);
    const float fdh = static_cast<float>(nvh * VE);
    const float z = (a.flags & kNoKeyNorm) ? dot : dot / sqrtf(ss / fdh + a.eps_key);
    if (a.flags & kSigmoid) {
      wc = 1.f / (1.f + expf(-z));
    } else {
      const float L = a.lse[static_cast<int64_t>(hd) * a.T + row];
      const float M = fmaxf(L, z);
      const float ea = expf(L - M), ec = expf(z - M);
      wa = ea / (ea + ec);
      wc = ec / (ea + ec);
    }
    if (a.alpha_p != nullptr && lane == 0) a.alpha_p[static_cast<int64_t>(hd) * a.T + row] = wc;
  }
  float h[VH][VE];
  float ssh = 0.f, unused = 0.f;
#pragma unroll
  for (int q = 0; q < VH; ++q) {
    const int i = lane + 32 * q;
#pragma unroll
    for (int e = 0; e < VE; ++e) h[q][e] = 0.f;
    if (i < nvh) {
      unpack_w<TO, VE>(ro[q], h[q]);
      if (has_p) {
#pragma unroll
        for (int e = 0; e < VE; ++e) h[q][e] = fmaf(wa, h[q][e], wc * p[q][e]);
      }
#pragma unroll
      for (int e = 0; e < VE; ++e) ssh = fmaf(h[q][e], h[q][e], ssh);
    }
  }
  block_sum2(ssh, unused, scratch);
  const float inv = 1.f / sqrtf(ssh / static_cast<float>(a.d) + a.eps_in);
  const float* g = a.gamma_in ? a.gamma_in + static_cast<int64_t>(hd) * nvh * VE : nullptr;
#pragma unroll
  for (int q = 0; q < VH; ++q) {
    const int i = lane + 32 * q;
    if (i < nvh) {
      if (a.h) st_global(static_cast<T*>(a.h) + base + i * VE, pack(h[q]));
      float y[VE];
#pragma unroll
      for (int e = 0; e < VE; ++e) y[e] = h[q][e] * inv;
      if (g) {
        const float4* g4 = reinterpret_cast<const float4*>(g + i * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
          const float4 gg = __ldg(g4 + e / 4);
          y[e] *= gg.x;
          y[e + 1] *= gg.y;
          y[e + 2] *= gg.z;
          y[e + 3] *= gg.w;
        }
      }
      st_global(static_cast<T*>(a.y) + base + i * VE, pack(y));
    }
  }
}

// Online softmax over the sources per head (warp), the next two sources' rows in flight.
template <typename T, int VH>
__global__ void __launch_bounds__(kHeadWarpsMax * 32, VH <= 2 ? 2 : 1)
    full_heads_kernel(const FullArgs a) {
  constexpr int VE = Vec<T>::N;
  __shared__ float scratch[66];
  __shared__ float zsh[kMaxSources * kHeadWarpsMax];  // [source][head] logits
  __shared__ float hl[kHeadWarpsMax];                 // per-head log-sum-exp
  pdl_enter();
  const int64_t row = blockIdx.x;
  const int H = a.heads;
  const int hd = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvh = a.d / VE / H;
  const int64_t off = static_cast<int64_t>(hd) * nvh * VE;  // the head's first column
  const int64_t base = row * a.d + off;
  const float fdh = static_cast<float>(nvh * VE);
  const bool sigmoid = (a.flags & kSigmoid) != 0;
  const float* u = a.u + off;

  float acc[VH][VE];
#pragma unroll
  for (int q = 0; q < VH; ++q)
#pragma unroll
    for (int e = 0; e < VE; ++e) acc[q][e] = 0.f;
  float mrun = -INFINITY, lrun = 0.f;
  if (a.o0 != nullptr) {  // an earlier partition (normalised o0, lse0) seeds the softmax
#pragma unroll
    for (int q = 0; q < VH; ++q) {
      const int i = lane + 32 * q;
      if (i < nvh) {
        if (a.o0_f32) {
          uint4 r[OWords<float, VE>::N];
          ld_stream_w<float, VE>(static_cast<const float*>(a.o0) + base + i * VE, r);
          unpack_w<float, VE>(r, acc[q]);
        } else {
          unpack(ld_stream(static_cast<const T*>(a.o0) + base + i * VE), acc[q]);
        }
      }
    }
    if (!sigmoid) {
      mrun = a.lse0[static_cast<int64_t>(hd) * a.T + row];
      lrun = 1.f;
    }
  }
  auto load = [&](uint4 (&r)[VH], int j) {
#pragma unroll
    for (int q = 0; q < VH; ++q) {
      const int i = lane + 32 * q;
      r[q] = make_uint4(0u, 0u, 0u, 0u);
      if (i < nvh) r[q] = ld_stream(static_cast<const T*>(a.srcs[j]) + base + i * VE);
    }
  };
  auto fold = [&](const float (&x)[VH][VE], int j) {
    float ss = 0.f, dot = 0.f;
#pragma unroll
    for (int q = 0; q < VH; ++q) {
      const int i = lane + 32 * q;
      if (i < nvh) {
        const float4* u4 = reinterpret_cast<const float4*>(u + i * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
          const float4 uu = __ldg(u4 + e / 4);
          dot = fmaf(uu.x, x[q][e], dot);
          dot = fmaf(uu.y, x[q][e + 1], dot);
          dot = fmaf(uu.z, x[q][e + 2], dot);
          dot = fmaf(uu.w, x[q][e + 3], dot);
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) ss = fmaf(x[q][e], x[q][e], ss);
      }
    }
    ss = warp_sum(ss);
    dot = warp_sum(dot);
    const float z = (a.flags & kNoKeyNorm) ? dot : dot / sqrtf(ss / fdh + a.eps_key);
    if (lane == 0) zsh[j * H + hd] = z;
    float sc, ez;
    if (sigmoid) {
      sc = 1.f;
      ez = 1.f / (1.f + expf(-z));
      mrun = fmaxf(mrun, z);
    } else {
      const float mnew = fmaxf(mrun, z);
      sc = expf(mrun - mnew);
      ez = expf(z - mnew);
      lrun = lrun * sc + ez;
      mrun = mnew;
    }
#pragma unroll
    for (int q = 0; q < VH; ++q)
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[q][e] = fmaf(acc[q][e], sc, ez * x[q][e]);
  };

  uint4 bufA[VH], bufB[VH];
  if (a.n > 0) load(bufA, 0);
  if (a.n > 1) load(bufB, 1);
  for (int j = 0; j < a.n; j += 2) {
    float x[VH][VE];
#pragma unroll
    for (int q = 0; q < VH; ++q) unpack(bufA[q], x[q]);
    if (j + 2 < a.n) load(bufA, j + 2);
    fold(x, j);
    if (j + 1 < a.n) {
#pragma unroll
      for (int q = 0; q < VH; ++q) unpack(bufB[q], x[q]);
      if (j + 3 < a.n) load(bufB, j + 3);
      fold(x, j + 1);
    }
  }

  const float rl = sigmoid ? 1.f : 1.f / lrun;
  float ssh = 0.f, unused = 0.f;
#pragma unroll
  for (int q = 0; q < VH; ++q)
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      acc[q][e] *= rl;
      ssh = fmaf(acc[q][e], acc[q][e], ssh);
    }
  const float lse = mrun + logf(lrun);
  if (lane == 0) {
    const int64_t at = static_cast<int64_t>(hd) * a.T + row;
    if (a.m != nullptr) a.m[at] = mrun;
    if (a.lse != nullptr && !sigmoid) a.lse[at] = lse;
    hl[hd] = lse;
  }
  float inv = 0.f;
  if (a.y != nullptr) {
    block_sum2(ssh, unused, scratch);  // its barriers also publish zsh[] and hl[]
    inv = 1.f / sqrtf(ssh / static_cast<float>(a.d) + a.eps_in);
  } else {
    __syncthreads();
  }
  if (a.alpha != nullptr) {
    for (int i = threadIdx.x; i < H * a.n; i += blockDim.x) {
      const int h2 = i / a.n, j = i - h2 * a.n;
      const float zj = zsh[j * H + h2];
      a.alpha[(static_cast<int64_t>(h2) * a.T + row) * a.n + j] =
          sigmoid ? 1.f / (1.f + expf(-zj)) : expf(zj - hl[h2]);
    }
  }
  const float* g = a.gamma_in ? a.gamma_in + off : nullptr;
#pragma unroll
  for (int q = 0; q < VH; ++q) {
    const int i = lane + 32 * q;
    if (i < nvh) {
      if (a.h) {
        if (a.h_f32)
          st_vec<float, VE>(static_cast<float*>(a.h) + base + i * VE, acc[q]);
        else
          st_global(static_cast<T*>(a.h) + base + i * VE, pack(acc[q]));
      }
      if (a.y) {
        float y[VE];
#pragma unroll
        for (int e = 0; e < VE; ++e) y[e] = acc[q][e] * inv;
        if (g) {
          const float4* g4 = reinterpret_cast<const float4*>(g + i * VE);
#pragma unroll
          for (int e = 0; e < VE; e += 4) {
            const float4 gg = __ldg(g4 + e / 4);
            y[e] *= gg.x;
            y[e + 1] *= gg.y;
            y[e + 2] *= gg.z;
            y[e + 3] *= gg.w;
          }
        }
        st_global(static_cast<T*>(a.y) + base + i * VE, pack(y));
      }
    }
  }
}

// Vectors per lane of the head-aligned kernels (1, 2 or 4), 0 if the shape does not fit them.
inline int head_vh(int d, int VE, int H) {
  if (H < 2 || H > kHeadWarpsMax) return 0;
  const int nvh = d / VE / H;
  for (int vh = 1; vh <= 4; vh *= 2)
    if (nvh <= 32 * vh) return vh;
  return 0;
}

template <typename T>
__global__ void add_kernel(const T* __restrict__ pa, const T* __restrict__ pb, T* out,
                           int64_t nvec) {
  constexpr int VE = Vec<T>::N;
  pdl_enter();
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
  pdl_enter();
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

template <typename T, typename TO>
cudaError_t phase2_heads(const Phase2Args& a, int vh, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(a.T);
  const int threads = 32 * a.heads;
  switch (vh) {
    case 1: return launch_pdl(phase2_heads_kernel<T, TO, 1>, grid, threads, 0, s, a);
    case 2: return launch_pdl(phase2_heads_kernel<T, TO, 2>, grid, threads, 0, s, a);
    case 4: return launch_pdl(phase2_heads_kernel<T, TO, 4>, grid, threads, 0, s, a);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t full_heads(const FullArgs& a, int vh, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>(a.T);
  const int threads = 32 * a.heads;
  switch (vh) {
    case 1: return launch_pdl(full_heads_kernel<T, 1>, grid, threads, 0, s, a);
    case 2: return launch_pdl(full_heads_kernel<T, 2>, grid, threads, 0, s, a);
    case 4: return launch_pdl(full_heads_kernel<T, 4>, grid, threads, 0, s, a);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, typename TO, int VPT>
cudaError_t phase2_vpt(const Phase2Args& a, unsigned grid, int threads, cudaStream_t s) {
  if (a.heads == 1) return launch_pdl(phase2_kernel<T, TO, VPT, false>, grid, threads, 0, s, a);
  const int smem = (2 * (a.d / Vec<T>::N) + 2 * a.heads) * static_cast<int>(sizeof(float));
  return launch_pdl(phase2_kernel<T, TO, VPT, true>, grid, threads, smem, s, a);
}

// TO: the type phase 1's output o_l is stored in (T, or fp32 with kOF32).
template <typename T, typename TO>
cudaError_t phase2_io(const Phase2Args& a, cudaStream_t s) {
  const int vh = head_vh(a.d, Vec<T>::N, a.heads);
  if (vh) return phase2_heads<T, TO>(a, vh, s);
  int vpt, threads;
  row_geometry(a.d / Vec<T>::N, vpt, threads, kMergeThreads);
  const unsigned grid = static_cast<unsigned>(a.T);
  switch (vpt) {
    case 1: return phase2_vpt<T, TO, 1>(a, grid, threads, s);
    case 2: return phase2_vpt<T, TO, 2>(a, grid, threads, s);
    case 4: return phase2_vpt<T, TO, 4>(a, grid, threads, s);
    case 8: return phase2_vpt<T, TO, 8>(a, grid, threads, s);
    case 16: return phase2_vpt<T, TO, 16>(a, grid, threads, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int VPT>
cudaError_t full_vpt(const FullArgs& a, unsigned grid, int threads, cudaStream_t s) {
  if (a.heads == 1) return launch_pdl(full_kernel<T, VPT, false>, grid, threads, 0, s, a);
  const int H = a.heads;
  const int smem =
      (2 * (a.d / Vec<T>::N) + 2 * H + a.n * H + H) * static_cast<int>(sizeof(float));
  return launch_pdl(full_kernel<T, VPT, true>, grid, threads, smem, s, a);
}

template <typename T>
cudaError_t full_io(const FullArgs& a, cudaStream_t s) {
  const int vh = head_vh(a.d, Vec<T>::N, a.heads);
  if (vh) return full_heads<T>(a, vh, s);
  int vpt, threads;
  row_geometry(a.d / Vec<T>::N, vpt, threads);
  const unsigned grid = static_cast<unsigned>(a.T);
  switch (vpt) {
    case 1: return full_vpt<T, 1>(a, grid, threads, s);
    case 2: return full_vpt<T, 2>(a, grid, threads, s);
    case 4: return full_vpt<T, 4>(a, grid, threads, s);
    case 8: return full_vpt<T, 8>(a, grid, threads, s);
    case 16: return full_vpt<T, 16>(a, grid, threads, s);
    default: return cudaErrorInvalidValue;
  }
}

inline unsigned grid_for(int64_t work, int threads) {
  int64_t b = (work + threads - 1) / threads;
  const int64_t cap = 148 * 16;
  return static_cast<unsigned>(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

cudaError_t launch_phase2(IO io, const Phase2Args& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (io == IO::F32) return phase2_io<float, float>(a, s);
  return (a.flags & kOF32) ? phase2_io<bf16, float>(a, s) : phase2_io<bf16, bf16>(a, s);
}


cudaError_t launch_full(IO io, const FullArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (full_ring_supported(io, a)) return launch_full_ring(io, a, s);
  return io == IO::BF16 ? full_io<bf16>(a, s) : full_io<float>(a, s);
}

cudaError_t launch_partial_update(IO io, const void* pa, const void* pb, void* out,
                                  int64_t n_elems, cudaStream_t s) {
  if (n_elems == 0) return cudaSuccess;
  constexpr int threads = 256;
  if (io == IO::BF16) {
    const int64_t nvec = n_elems / 8;
    return launch_pdl(add_kernel<bf16>, grid_for(nvec, threads), threads, 0, s,
                      static_cast<const bf16*>(pa), static_cast<const bf16*>(pb),
                      static_cast<bf16*>(out), nvec);
  }
  const int64_t nvec = n_elems / 4;
  return launch_pdl(add_kernel<float>, grid_for(nvec, threads), threads, 0, s,
                    static_cast<const float*>(pa), static_cast<const float*>(pb),
                    static_cast<float*>(out), nvec);
}

cudaError_t launch_query_prep(const float* w, const float* g, float* u, void* u_split, int rows,
                              int d, cudaStream_t s) {
  const int64_t n_elems = static_cast<int64_t>(rows) * d;
  if (n_elems == 0) return cudaSuccess;
  constexpr int threads = 256;
  return launch_pdl(prep_kernel, grid_for(n_elems / 4, threads), threads, 0, s, w, g, u,
                    static_cast<uint16_t*>(u_split), d, n_elems / 4);
}

}  // namespace attnres
