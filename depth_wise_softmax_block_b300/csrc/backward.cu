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
//
// bf16 rows of 512 to 896 vectors over at most 10 sources (d = 7168 and below) go to
// backward_ring_kernel instead: one CTA per SM, a copy warp streaming the row's n sources and
// g_y into a ring of shared-memory row slots (bulk copies), 14 compute warps with two vectors a
// thread, and the same four passes read from the slots:
//   1  sum of squares and u . v_j (a 4-value reduce-scatter over the warp per pair of sources);
//      one barrier; r_j, z_j and alpha_j on lane j of every warp
//   2  h = sum alpha_j v_j, t = gamma_in ⊙ g_y, |h|^2 and t . h; one barrier; g_h kept in
//      registers; g_y's slot released
//   3  g_h . v_j (one reduce-scatter per four sources); one barrier; dz_j and the coefficients
//   4  dL/dv_j stored from registers, du += (dz_j / r_j) v_j, slot j released
// Element pairs go through packed fp32 FMAs; du and dgamma_in are summed in registers (16 + 16
// a thread) and added atomically when the CTA ends.  Every wait is bounded (tma.cuh).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

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

constexpr int kBrWarps = 14;
constexpr int kBrCompute = kBrWarps * 32;
constexpr int kBrThreads = kBrCompute + 32;
constexpr int kBrVPT = 2;
constexpr int kBrVectors = kBrVPT * kBrCompute;  // 896
constexpr int kBrMaxN = 10;
constexpr int kBrSlotBytes = 216 * 1024;

__device__ __forceinline__ void br_bulk_load(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Reduce-scatter of four values over the warp: afterwards lane L holds the warp's total of value
// 2 (L >> 4 & 1) + (L >> 3 & 1); lanes 0, 8, 16, 24 hold values 0, 1, 2, 3.
__device__ __forceinline__ float rs4(const float (&v4)[4], int lane) {
  const bool up16 = (lane & 16) != 0, up8 = (lane & 8) != 0;
  const float k0 =
      (up16 ? v4[2] : v4[0]) + __shfl_xor_sync(0xffffffffu, up16 ? v4[0] : v4[2], 16);
  const float k1 =
      (up16 ? v4[3] : v4[1]) + __shfl_xor_sync(0xffffffffu, up16 ? v4[1] : v4[3], 16);
  float t = (up8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, up8 ? k0 : k1, 8);
  t += __shfl_xor_sync(0xffffffffu, t, 4);
  t += __shfl_xor_sync(0xffffffffu, t, 2);
  t += __shfl_xor_sync(0xffffffffu, t, 1);
  return t;
}

__device__ __forceinline__ float2 lohi(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <bool kFullRow>
__global__ void __launch_bounds__(kBrThreads, 1) backward_ring_kernel(const BwdArgs a, int SB) {
  using T = bf16;
  constexpr int VE = 8;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  const int d = a.d, n = a.n;
  const int rowbytes = d * 2;
  const int nv = kFullRow ? kBrVectors : d / VE;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + SB * rowbytes);
  uint64_t* empty = full + SB;
  float* pw1 = reinterpret_cast<float*>(empty + SB);  // [2][14][32]: ss, dot of the sources
  float* pw2 = pw1 + 2 * kBrWarps * 32;               // [2][14][2]: |h|^2, t . h
  float* pw3 = pw2 + 2 * kBrWarps * 2;                // [2][14][32]: g_h . v_j
  int* abort_flag = reinterpret_cast<int*>(pw3 + 2 * kBrWarps * 32);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float fd = static_cast<float>(d);

  if (tid == 0) {
    for (int s = 0; s < SB; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kBrCompute);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_enter();
  volatile int* abort_v = abort_flag;

  // ---- copy warp: per row the n sources, then g_y ----
  if (warp == kBrWarps) {
    if (lane == 0) {
      int it = 0, bs = 0, ph = 0;
      for (int64_t r = blockIdx.x; r < a.T && !*abort_v; r += gridDim.x) {
        for (int j = 0; j <= n; ++j) {
          if (it >= SB && !mbar_wait(&empty[bs], ph ^ 1)) {
            *abort_v = 1;
            break;
          }
          if (*abort_v) break;
          const void* src = j < n ? a.srcs[j] : a.g_y;
          mbar_arrive_expect_tx(&full[bs], static_cast<uint32_t>(rowbytes));
          br_bulk_load(ring + bs * rowbytes,
                       static_cast<const char*>(src) + r * static_cast<int64_t>(rowbytes),
                       static_cast<uint32_t>(rowbytes), &full[bs]);
          ++it;
          if (++bs == SB) {
            bs = 0;
            ph ^= 1;
          }
        }
      }
      for (int s = 0; s < SB && s < it; ++s) {
        const int last = it - 1 - ((it - 1 - s) % SB);
        mbar_wait_drain(&full[s], (last / SB) & 1);
      }
    }
    return;
  }

  // ---- compute warps ----
  float2 uq[kBrVPT][4], du[kBrVPT][4], dg[kBrVPT][4];
#pragma unroll
  for (int k = 0; k < kBrVPT; ++k) {
    const int v = tid + k * kBrCompute;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uq[k][i] = kFullRow || v < nv
                     ? make_float2(__ldg(a.u + v * VE + 2 * i), __ldg(a.u + v * VE + 2 * i + 1))
                     : make_float2(0.f, 0.f);
      du[k][i] = dg[k][i] = make_float2(0.f, 0.f);
    }
  }
  auto slot_vec = [&](int slot, int k) -> uint4 {
    const int v = tid + k * kBrCompute;
    return kFullRow || v < nv ? reinterpret_cast<const uint4*>(ring + slot * rowbytes)[v]
                              : make_uint4(0u, 0u, 0u, 0u);
  };

  int bs = 0, ph = 0;
  int par = 0;
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x, par ^= 1) {
    bool ab = *abort_v;
    const int b0 = bs;  // slot of source 0; source j at (b0 + j) mod SB, g_y at (b0 + n) mod SB
    auto slot = [&](int j) { const int s = b0 + j; return s >= SB ? s - SB : s; };
    float* p1 = pw1 + par * kBrWarps * 32;
    float* p2 = pw2 + par * kBrWarps * 2;
    float* p3 = pw3 + par * kBrWarps * 32;

    // ---- pass 1: ss_j, u . v_j ----
#pragma unroll
    for (int j0 = 0; j0 < kBrMaxN; j0 += 2) {
      if (j0 < n) {
        float v4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int j = j0 + q;
          if (j < n) {
            if (!ab && !mbar_wait(&full[bs], static_cast<uint32_t>(ph))) {
              ab = true;
              *abort_v = 1;
            }
            float2 ss = make_float2(0.f, 0.f), dot = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kBrVPT; ++k) {
              const uint4 x = slot_vec(bs, k);
              const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 e = lohi(w[i]);
                ss = __ffma2_rn(e, e, ss);
                dot = __ffma2_rn(uq[k][i], e, dot);
              }
            }
            v4[2 * q] = ss.x + ss.y;
            v4[2 * q + 1] = dot.x + dot.y;
            if (++bs == SB) {
              bs = 0;
              ph ^= 1;
            }
          }
        }
        const float t = rs4(v4, lane);
        if ((lane & 7) == 0) p1[warp * 32 + 2 * j0 + (lane >> 3)] = t;
      }
    }
    // g_y's slot (waited for in pass 2)
    const int gslot = bs;
    const int gph = ph;
    if (++bs == SB) {
      bs = 0;
      ph ^= 1;
    }
    named_barrier(1, kBrCompute);
    // statistics on lane j (every warp the same)
    float rj = 1.f, zj = -INFINITY, al = 0.f;
    {
      if (lane < n) {
        float ss = 0.f, dot = 0.f;
#pragma unroll
        for (int w = 0; w < kBrWarps; ++w) {
          ss += p1[w * 32 + 2 * lane];
          dot += p1[w * 32 + 2 * lane + 1];
        }
        rj = sqrtf(ss / fd + a.eps_key);
        zj = dot / rj;
      }
      float m = zj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float ez = lane < n ? expf(zj - m) : 0.f;
      al = ez / warp_sum(ez);
    }

    // ---- pass 2: h, t = gamma_in * g_y, the input-norm sums ----
    float2 h[kBrVPT][4];
#pragma unroll
    for (int k = 0; k < kBrVPT; ++k)
#pragma unroll
      for (int i = 0; i < 4; ++i) h[k][i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kBrMaxN; ++j) {
      if (j < n) {
        const float aj = __shfl_sync(0xffffffffu, al, j);
        const float2 a2 = make_float2(aj, aj);
#pragma unroll
        for (int k = 0; k < kBrVPT; ++k) {
          const uint4 x = slot_vec(slot(j), k);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) h[k][i] = __ffma2_rn(a2, lohi(w[i]), h[k][i]);
        }
      }
    }
    if (!ab && !mbar_wait(&full[gslot], static_cast<uint32_t>(gph))) {
      ab = true;
      *abort_v = 1;
    }
    float2 gh[kBrVPT][4];  // t = gamma_in * g_y for now
    uint4 gyv[kBrVPT];
    float2 sh = make_float2(0.f, 0.f), st = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kBrVPT; ++k) {
      const int v = tid + k * kBrCompute;
      gyv[k] = slot_vec(gslot, k);
      const uint32_t w[4] = {gyv[k].x, gyv[k].y, gyv[k].z, gyv[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 gi = make_float2(1.f, 1.f);
        if (a.gamma_in != nullptr && (kFullRow || v < nv))
          gi = make_float2(__ldg(a.gamma_in + v * VE + 2 * i),
                           __ldg(a.gamma_in + v * VE + 2 * i + 1));
        gh[k][i] = __fmul2_rn(gi, lohi(w[i]));
        sh = __ffma2_rn(h[k][i], h[k][i], sh);
        st = __ffma2_rn(gh[k][i], h[k][i], st);
      }
    }
    mbar_arrive(&empty[gslot]);  // g_y consumed (kept packed in gyv)
    {
      float v4[4] = {sh.x + sh.y, st.x + st.y, 0.f, 0.f};
      const float t = rs4(v4, lane);
      if (lane == 0 || lane == 8) p2[warp * 2 + (lane >> 3)] = t;
    }
    named_barrier(1, kBrCompute);
    float ssh = 0.f, s1 = 0.f;
#pragma unroll
    for (int w = 0; w < kBrWarps; ++w) {
      ssh += p2[w * 2];
      s1 += p2[w * 2 + 1];
    }
    const float rh = sqrtf(ssh / fd + a.eps_in);
    const float c1 = 1.f / rh, c2 = s1 / (fd * rh * rh * rh);
    const float2 c1v = make_float2(c1, c1), c2n = make_float2(-c2, -c2);
#pragma unroll
    for (int k = 0; k < kBrVPT; ++k) {
      const uint32_t w[4] = {gyv[k].x, gyv[k].y, gyv[k].z, gyv[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dg[k][i] = __ffma2_rn(__fmul2_rn(lohi(w[i]), h[k][i]), c1v, dg[k][i]);
        gh[k][i] = __ffma2_rn(h[k][i], c2n, __fmul2_rn(gh[k][i], c1v));
      }
    }

    // ---- pass 3: g_h . v_j, quads of sources ----
#pragma unroll
    for (int j0 = 0; j0 < kBrMaxN; j0 += 4) {
      if (j0 < n) {
        float v4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = j0 + q;
          if (j < n) {
            float2 dot = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kBrVPT; ++k) {
              const uint4 x = slot_vec(slot(j), k);
              const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) dot = __ffma2_rn(gh[k][i], lohi(w[i]), dot);
            }
            v4[q] = dot.x + dot.y;
          }
        }
        const float t = rs4(v4, lane);
        if ((lane & 7) == 0) p3[warp * 32 + j0 + (lane >> 3)] = t;
      }
    }
    named_barrier(1, kBrCompute);
    float cu = 0.f, cv = 0.f;
    {
      float pq = 0.f;
      if (lane < n) {
#pragma unroll
        for (int w = 0; w < kBrWarps; ++w) pq += p3[w * 32 + lane];
      }
      const float ghh = warp_sum(al * pq);  // g_h . h = sum_j alpha_j (g_h . v_j)
      const float dz = al * (pq - ghh);
      if (lane < n) {
        cu = dz / rj;
        cv = dz * zj / (fd * rj * rj);
      }
    }

    // ---- pass 4: dv_j, du; slot j released ----
#pragma unroll
    for (int j = 0; j < kBrMaxN; ++j) {
      if (j < n) {
        const float aj = __shfl_sync(0xffffffffu, al, j);
        const float cuj = __shfl_sync(0xffffffffu, cu, j);
        const float cvj = __shfl_sync(0xffffffffu, cv, j);
        const float2 a2 = make_float2(aj, aj), cu2 = make_float2(cuj, cuj),
                     cvn = make_float2(-cvj, -cvj);
        const int sj = slot(j);
#pragma unroll
        for (int k = 0; k < kBrVPT; ++k) {
          const int v = tid + k * kBrCompute;
          const uint4 x = slot_vec(sj, k);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
          float o[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 e = lohi(w[i]);
            const float2 dv =
                __ffma2_rn(a2, gh[k][i], __ffma2_rn(cu2, uq[k][i], __fmul2_rn(cvn, e)));
            o[2 * i] = dv.x;
            o[2 * i + 1] = dv.y;
            du[k][i] = __ffma2_rn(cu2, e, du[k][i]);
          }
          if (kFullRow || v < nv)
            st_global(static_cast<T*>(a.dsrcs[j]) + r * d + v * VE, pack(o));
        }
        mbar_arrive(&empty[sj]);  // the stores consumed every register read from the slot
      }
    }
  }

  // ---- this CTA's du and dgamma_in partial sums ----
#pragma unroll
  for (int k = 0; k < kBrVPT; ++k) {
    const int v = tid + k * kBrCompute;
    if (kFullRow || v < nv) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        atomicAdd(a.du + v * VE + 2 * i, du[k][i].x);
        atomicAdd(a.du + v * VE + 2 * i + 1, du[k][i].y);
        if (a.dgamma_in != nullptr) {
          atomicAdd(a.dgamma_in + v * VE + 2 * i, dg[k][i].x);
          atomicAdd(a.dgamma_in + v * VE + 2 * i + 1, dg[k][i].y);
        }
      }
    }
  }
}

bool backward_ring_supported(const BwdArgs& a) {
  const int nv = a.d / 8;
  return a.n >= 1 && a.n <= kBrMaxN && a.d % 8 == 0 && nv >= 512 && nv <= kBrVectors &&
         kBrSlotBytes / (a.d * 2) >= a.n + 3;
}

cudaError_t launch_backward_ring(const BwdArgs& a, cudaStream_t s) {
  if (!backward_ring_supported(a)) return cudaErrorInvalidValue;
  if (a.T == 0) return cudaSuccess;
  const int rowbytes = a.d * 2;
  const int SB = std::min(64, kBrSlotBytes / rowbytes);
  // slots | full, empty barriers | reduction buffers [2][14][32], [2][14][2], [2][14][32] | flag
  const int smem = 128 + SB * rowbytes + 2 * SB * 8 +
                   (2 * kBrWarps * 32 * 2 + 2 * kBrWarps * 2) * 4 + 16;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  auto kern = a.d / 8 == kBrVectors ? backward_ring_kernel<true> : backward_ring_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = a.T < sms ? a.T : sms;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kBrThreads),
                    static_cast<size_t>(smem), s, a, SB);
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
  if (io == IO::BF16 && backward_ring_supported(a)) return launch_backward_ring(a, s);
  return io == IO::BF16 ? backward_io<bf16>(a, s) : backward_io<float>(a, s);
}

unsigned int backward_poll_timeouts() {
  return take_wait_timeouts();
}

}  // namespace attnres
