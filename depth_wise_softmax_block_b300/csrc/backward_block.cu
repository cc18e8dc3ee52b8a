// Backward of one block of Block AttnRes, structured by the two-phase schedule ("Attention
// Residuals" note §8 block definition, §10 two-phase computation; the logit gradient of §7;
// "Attention Residuals 阅读补充", section "梯度沿切向传播" for the RMSNorm gradients, and the
// Block AttnRes training section: the inter-block attention is recomputed in the backward
// pass, not stored).
//
// Forward of the block (n completed sources b_0 .. b_{n-1}, S sublayers, partial sums
// p_i = v_1 + ... + v_{i-1} for i >= 2): sublayer i attends over A = {b_j} (phase 1: o_i, lse_i,
// alpha_ij over A) and the partial p_i (phase 2: w_A = e^{lse}/(e^{lse} + e^{z_p}), w_p = 1 - w_A,
// h_i = w_A o_i + w_p p_i), then y_i = gamma_in,i ⊙ h_i / r(h_i).
//
// Backward, given g_i = dL/dy_i.  With g_h = RMSNorm backward of g_i at h_i, the direct logit
// gradient alpha_full (g_h . x - g_h . h) splits by partition:
//   partial      dz_p = w_p (g_h . p - g_h . h)
//                dL/dp_i = w_p g_h + (dz_p / r_p) u_i - (dz_p z_p / (d r_p^2)) p_i
//   sources      dz_ij = alpha_ij (q_i . b_j + c_i),  q_i = w_A g_h  (= dL/do_i),
//                c_i = -w_A g_h . o_i + w_A w_p (g_h . o_i - g_h . p_i)
//                dL/db_j = sum_i alpha_ij q_i + sum_i (dz_ij / r_j) u_i - b_j sum_i dz_ij z_ij / (d r_j^2)
//   parameters   du_i = sum_t [(dz_p / r_p) p_i + sum_j (dz_ij / r_j) b_j],
//                dgamma_in,i = sum_t g_i ⊙ h_i / r(h_i)
//   outputs      dL/dv_k = sum_{i > k} dL/dp_i   (v_k enters the partial of every later sublayer)
//
// Four launches, each source row of the block read a bounded number of times (not once per
// sublayer):
//   1. phase 1 recomputed (the forward's own kernel) over the n sources for the S queries:
//      o_i (fp32), lse_i, alpha_ij into the workspace;
//   2. bwd_merge_kernel, one CTA per token row, the S sublayers in reverse order with the
//      partial sum and the dL/dv running sums in registers: per sublayer one CTA reduction of
//      six sums (|p|^2, u.p, |o|^2, o.p, gamma g.o, gamma g.p) gives every scalar of the merge
//      and of both norms' backward; writes q_i (fp32) and dL/dv_{i-1};
//   3. bwd_sources_kernel, one CTA per token row: q_i . b_j for all (i, j) and |b_j|^2 (eight
//      warps, three queries each), the coefficients dz_ij / r_j and sum_i dz_ij z_ij / (d r_j^2),
//      then dL/db_j per element in a second pass (q_i again, from L2); the coefficients the
//      parameter sums need go to a per-token record;
//   4. bwd_params_kernel, one thread per column and a range of tokens: du_i and dgamma_in,i
//      summed over the CTA's tokens in registers (one atomic per element and CTA at the end).
// Softmax weights, key RMSNorm, one head (the method as defined).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace attnres {
namespace {

constexpr int kRowThreads = 512;    // merge kernel: at most 512 threads per row
constexpr int kDotThreads = 256;    // sources kernel: 8 warps
constexpr int kDotQ = 3;            // queries per warp in the sources kernel's dots (8 x 3 = 24)
constexpr int kDbGroup = 8;         // sources whose gradients a thread accumulates at once
constexpr int kColThreads = 256;    // columns per CTA of the parameter kernel
constexpr int kColBatch = 16;       // token records staged in shared memory at a time

inline int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

// Per-token record written by the sources kernel for the parameter kernel (floats):
// [E = dz_ij / r_j: S*n][a = w_A / r_h: S][b = w_p / r_h: S][e = dz_p / r_p: S], padded to 4.
inline int record_floats(int n, int S) { return (S * n + 3 * S + 3) / 4 * 4; }

// VE consecutive fp32 values from a 16-byte aligned address through the read-only path.
template <int VE>
__device__ __forceinline__ void ldg_f32(const float* p, float (&f)[VE]) {
#pragma unroll
  for (int e = 0; e < VE; e += 4) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(p + e));
    f[e] = x.x;
    f[e + 1] = x.y;
    f[e + 2] = x.z;
    f[e + 3] = x.w;
  }
}

// ------------------------------------------------------------------------------------------
// 2. merge backward: one CTA per token row, sublayers S .. 1; the rows of sublayer i - 1 (o, g)
// and v_{i-1} are loaded while sublayer i is reduced and written.
template <typename IOT, int VPT>
__global__ void __launch_bounds__(kRowThreads) bwd_merge_kernel(const BwdBlockArgs a) {
  constexpr int VE = Vec<IOT>::N;
  constexpr int NW = OWords<float, VE>::N;
  __shared__ float scratch[6 * 33];
  pdl_enter();
  const int64_t t = blockIdx.x, T = a.T;
  const int d = a.d, nv = d / VE, S = a.S;
  const float fd = static_cast<float>(d);
  const int64_t row = t * d;

  float P[VPT][VE], A[VPT][VE];  // running partial sum p_i and running sum of dL/dp
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int e = 0; e < VE; ++e) P[k][e] = A[k][e] = 0.f;
#pragma unroll 4
  for (int kv = 1; kv < S; ++kv) {  // p_S = v_1 + ... + v_{S-1}
    const IOT* vk = static_cast<const IOT*>(a.v) + (kv - 1) * a.v_stride + row;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        float x[VE];
        unpack(ld_stream(vk + v * VE), x);
#pragma unroll
        for (int e = 0; e < VE; ++e) P[k][e] += x[e];
      }
    }
  }
  auto load_og = [&](int i, uint4 (&ro)[VPT][NW], uint4 (&rg)[VPT]) {
    const int64_t ri = static_cast<int64_t>(i - 1) * T + t;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        ld_stream_w<float, VE>(a.o + ri * d + v * VE, ro[k]);
        rg[k] = ld_stream(static_cast<const IOT*>(a.g_y) + ri * d + v * VE);
      }
    }
  };
  uint4 ro[VPT][NW], rg[VPT];
  load_og(S, ro, rg);

  for (int i = S; i >= 1; --i) {
    const bool has_p = i >= 2;
    const int64_t ri = static_cast<int64_t>(i - 1) * T + t;
    const float* ui = a.u + static_cast<int64_t>(i - 1) * d;
    const float* gam = a.gamma_in ? a.gamma_in + static_cast<int64_t>(i - 1) * d : nullptr;
    uint4 no[VPT][NW], ng[VPT], rv[VPT];  // sublayer i - 1 and v_{i-1}, in flight
    if (has_p) {
      load_og(i - 1, no, ng);
      const IOT* vk = static_cast<const IOT*>(a.v) + (i - 2) * a.v_stride + row;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
        if (v < nv) rv[k] = ld_stream(vk + v * VE);
      }
    }
    // |p|^2, u.p, |o|^2, o.p, (gamma g).o, (gamma g).p
    float s[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        float o[VE], g[VE], uu[VE], gg[VE];
        unpack_w<float, VE>(ro[k], o);
        unpack(rg[k], g);
        ldg_f32<VE>(ui + v * VE, uu);
        if (gam) {
          ldg_f32<VE>(gam + v * VE, gg);
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) gg[e] = 1.f;
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float ge = gg[e] * g[e];
          const float p = P[k][e];
          s[0] = fmaf(p, p, s[0]);
          s[1] = fmaf(uu[e], p, s[1]);
          s[2] = fmaf(o[e], o[e], s[2]);
          s[3] = fmaf(o[e], p, s[3]);
          s[4] = fmaf(ge, o[e], s[4]);
          s[5] = fmaf(ge, p, s[5]);
        }
      }
    }
    block_sum_n<6>(s, scratch);
    // the merge (page 2 §10) and both norms' backward, from the six sums
    float wA = 1.f, wP = 0.f, rp = 1.f, zp = 0.f;
    if (has_p) {
      rp = sqrtf(s[0] / fd + a.eps_key);
      zp = s[1] / rp;
      const float L = a.lse[ri];
      const float M = fmaxf(L, zp);
      const float ea = expf(L - M), ec = expf(zp - M);
      wA = ea / (ea + ec);
      wP = ec / (ea + ec);
    }
    const float shh = wA * wA * s[2] + 2.f * wA * wP * s[3] + wP * wP * s[0];
    const float rh = sqrtf(shh / fd + a.eps_in);
    const float sgh = wA * s[4] + wP * s[5];
    const float kap = sgh / (fd * rh * rh * rh);
    const float hp = wA * s[3] + wP * s[0], ho = wA * s[2] + wP * s[3];
    const float ghp = s[5] / rh - kap * hp, gho = s[4] / rh - kap * ho;
    const float ghh = wA * gho + wP * ghp;
    const float dzp = has_p ? wP * (ghp - ghh) : 0.f;
    const float coefu = has_p ? dzp / rp : 0.f;
    const float coefp = has_p ? dzp * zp / (fd * rp * rp) : 0.f;
    const float c = -wA * gho + wA * wP * (gho - ghp);
    const float inv_rh = 1.f / rh;

    float* qi = a.q + ri * d;
    IOT* dvi = has_p ? static_cast<IOT*>(a.d_v) + static_cast<int64_t>(i - 2) * a.dv_stride + row
                     : nullptr;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        float o[VE], g[VE], q[VE], uu[VE], gg[VE];
        unpack_w<float, VE>(ro[k], o);
        unpack(rg[k], g);
        ldg_f32<VE>(ui + v * VE, uu);
        if (gam) {
          ldg_f32<VE>(gam + v * VE, gg);
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) gg[e] = 1.f;
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float h = wA * o[e] + wP * P[k][e];
          const float gh = gg[e] * g[e] * inv_rh - kap * h;
          q[e] = wA * gh;
          if (has_p) A[k][e] += wP * gh + coefu * uu[e] - coefp * P[k][e];
        }
        st_vec<float, VE>(qi + v * VE, q);
        if (has_p) st_vec<IOT, VE>(dvi + v * VE, A[k]);
      }
    }
    if (threadIdx.x == 0)
      *reinterpret_cast<float4*>(a.sc2 + ri * 4) = make_float4(c, wA * inv_rh, wP * inv_rh, coefu);
    if (has_p) {  // p_{i-1} = p_i - v_{i-1}; the next sublayer's rows are already loaded
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
        if (v < nv) {
          float x[VE];
          unpack(rv[k], x);
#pragma unroll
          for (int e = 0; e < VE; ++e) P[k][e] -= x[e];
#pragma unroll
          for (int w = 0; w < NW; ++w) ro[k][w] = no[k][w];
          rg[k] = ng[k];
        }
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// 3. sources: per token, q_i . b_j for all (i, j) and |b_j|^2 (pass 1), the coefficients, then
// dL/db_j = sum_i alpha_ij q_i + sum_i E_ij u_i - F_j b_j per element (pass 2, q_i again from
// L2), with E_ij = dz_ij / r_j and F_j = sum_i dz_ij z_ij / (d r_j^2).
template <typename IOT>
__global__ void __launch_bounds__(kDotThreads) bwd_sources_kernel(const BwdBlockArgs a) {
  constexpr int VE = Vec<IOT>::N;
  constexpr int NJ = kBlkMaxN;
  constexpr int NW = OWords<float, VE>::N;
  __shared__ float Ds[kBlkMaxS * NJ];   // D_ij, then E_ij
  __shared__ float As[kBlkMaxS * NJ];   // alpha_ij
  __shared__ float dzz[kBlkMaxS * NJ];
  __shared__ float ssj[NJ], Fs[NJ];
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = blockIdx.x, T = a.T;
  const int d = a.d, nv = d / VE, S = a.S, n = a.n;
  const float fd = static_cast<float>(d);
  const IOT* b0 = static_cast<const IOT*>(a.reps) + t * d;   // source j at b0 + j * src_stride
  const float* qb = a.q;

  // ---- pass 1: dot products ----
  float acc[kDotQ][NJ], ss[2] = {0.f, 0.f};
#pragma unroll
  for (int r = 0; r < kDotQ; ++r)
#pragma unroll
    for (int j = 0; j < NJ; ++j) acc[r][j] = 0.f;
  for (int v = lane; v < nv; v += 32) {
    float qv[kDotQ][VE];
#pragma unroll
    for (int r = 0; r < kDotQ; ++r) {
      const int i = warp + 8 * r;
      if (i < S) {
        uint4 w[NW];
        ld_stream_w<float, VE>(qb + (static_cast<int64_t>(i) * T + t) * d + v * VE, w);
        unpack_w<float, VE>(w, qv[r]);
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) qv[r][e] = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < n) {
        float x[VE];
        unpack(*reinterpret_cast<const uint4*>(b0 + j * a.src_stride + v * VE), x);
#pragma unroll
        for (int r = 0; r < kDotQ; ++r)
#pragma unroll
          for (int e = 0; e < VE; ++e) acc[r][j] = fmaf(qv[r][e], x[e], acc[r][j]);
        if (j == warp || j == warp + 8) {
#pragma unroll
          for (int e = 0; e < VE; ++e)
            ss[j == warp ? 0 : 1] = fmaf(x[e], x[e], ss[j == warp ? 0 : 1]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kDotQ; ++r)
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < n) {
        const float x = warp_sum(acc[r][j]);
        const int i = warp + 8 * r;
        if (lane == 0 && i < S) Ds[i * NJ + j] = x;
      }
    }
  const float s0 = warp_sum(ss[0]), s1 = warp_sum(ss[1]);
  if (lane == 0) {
    if (warp < n) ssj[warp] = s0;
    if (warp + 8 < n) ssj[warp + 8] = s1;
  }
  __syncthreads();

  // ---- coefficients ----
  const int R = a.rec_floats;
  float* rec = a.rec + t * R;
  for (int k = threadIdx.x; k < S * n; k += blockDim.x) {
    const int i = k / n, j = k - i * n;
    const int64_t ri = static_cast<int64_t>(i) * T + t;
    const float al = a.alpha[ri * n + j];
    const float c = a.sc2[ri * 4];
    const float rj = sqrtf(ssj[j] / fd + a.eps_key);
    const float dz = al * (Ds[i * NJ + j] + c);
    // z_ij = lse_i + ln alpha_ij (alpha = exp(z - lse)); a zero weight carries no gradient
    dzz[i * NJ + j] = al > 0.f ? dz * (a.lse[ri] + logf(al)) : 0.f;
    As[i * NJ + j] = al;
    Ds[i * NJ + j] = dz / rj;   // E_ij (this thread alone reads and writes entry k)
    rec[k] = dz / rj;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    float f = 0.f;
    for (int i = 0; i < S; ++i) f += dzz[i * NJ + j];
    Fs[j] = f / (fd * (ssj[j] / fd + a.eps_key));
  }
  for (int i = threadIdx.x; i < S; i += blockDim.x) {
    const float4 sc =
        *reinterpret_cast<const float4*>(a.sc2 + (static_cast<int64_t>(i) * T + t) * 4);
    rec[S * n + i] = sc.y;
    rec[S * n + S + i] = sc.z;
    rec[S * n + 2 * S + i] = sc.w;
  }
  __syncthreads();

  // ---- pass 2: dL/db_j, up to kDbGroup sources at a time ----
  IOT* dr = static_cast<IOT*>(a.d_reps);
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    for (int jg = 0; jg < n; jg += kDbGroup) {
      float db[kDbGroup][VE];
#pragma unroll
      for (int jj = 0; jj < kDbGroup; ++jj)
#pragma unroll
        for (int e = 0; e < VE; ++e) db[jj][e] = 0.f;
#pragma unroll 2
      for (int i = 0; i < S; ++i) {
        float q[VE], uu[VE];
        ldg_f32<VE>(qb + (static_cast<int64_t>(i) * T + t) * d + v * VE, q);
        ldg_f32<VE>(a.u + static_cast<int64_t>(i) * d + v * VE, uu);
#pragma unroll
        for (int jj = 0; jj < kDbGroup; ++jj) {
          const int j = jg + jj;
          if (j < n) {
            const float al = As[i * NJ + j], E = Ds[i * NJ + j];
#pragma unroll
            for (int e = 0; e < VE; ++e) db[jj][e] = fmaf(al, q[e], fmaf(E, uu[e], db[jj][e]));
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < kDbGroup; ++jj) {
        const int j = jg + jj;
        if (j < n) {
          float x[VE];
          unpack(*reinterpret_cast<const uint4*>(b0 + j * a.src_stride + v * VE), x);
#pragma unroll
          for (int e = 0; e < VE; ++e) db[jj][e] = fmaf(-Fs[j], x[e], db[jj][e]);
          st_vec<IOT, VE>(dr + (static_cast<int64_t>(j) * T + t) * d + v * VE, db[jj]);
        }
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// 4. per column: du_i and dgamma_in,i summed over a range of tokens in registers.
template <typename IOT>
__device__ __forceinline__ float ld1(const IOT* p) {
  if constexpr (sizeof(IOT) == 2) {
    return __bfloat162float(*reinterpret_cast<const bf16*>(p));
  } else {
    return *reinterpret_cast<const float*>(p);
  }
}

template <typename IOT>
__global__ void __launch_bounds__(kColThreads) bwd_params_kernel(const BwdBlockArgs a,
                                                                 int tokens_per_cta) {
  constexpr int NJ = kBlkMaxN, NS = kBlkMaxS;
  extern __shared__ float srec[];  // [kColBatch][R]
  pdl_enter();
  const int d = a.d, S = a.S, n = a.n, R = a.rec_floats;
  const int64_t T = a.T;
  const int c = blockIdx.x * kColThreads + threadIdx.x;
  const bool valid = c < d;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * tokens_per_cta;
  const int64_t t1 = t0 + tokens_per_cta < T ? t0 + tokens_per_cta : T;
  const IOT* reps = static_cast<const IOT*>(a.reps);
  const IOT* vb = static_cast<const IOT*>(a.v);
  const IOT* gb = static_cast<const IOT*>(a.g_y);

  float du[NS], dg[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) du[i] = dg[i] = 0.f;
  const int oE = 0, oa = S * n, ob = oa + S, oe = ob + S;

  for (int64_t tb0 = t0; tb0 < t1; tb0 += kColBatch) {
    const int nb = static_cast<int>(t1 - tb0 < kColBatch ? t1 - tb0 : kColBatch);
    __syncthreads();  // the previous batch's records are no longer read
    for (int k = threadIdx.x; k < nb * R / 4; k += blockDim.x)
      reinterpret_cast<float4*>(srec)[k] = reinterpret_cast<const float4*>(a.rec + tb0 * R)[k];
    __syncthreads();
    if (!valid) continue;
    for (int tb = 0; tb < nb; ++tb) {
      const int64_t t = tb0 + tb;
      const float* rr = srec + tb * R;
      float b[NJ];
#pragma unroll
      for (int j = 0; j < NJ; ++j) b[j] = j < n ? ld1(reps + j * a.src_stride + t * d + c) : 0.f;
      float P = 0.f;  // partial sum of sublayer i + 1
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        if (i < S) {
          if (i >= 1) P += ld1(vb + (i - 1) * a.v_stride + t * d + c);
          const int64_t at = (static_cast<int64_t>(i) * T + t) * d + c;
          const float o = a.o[at], g = ld1(gb + at);
          dg[i] = fmaf(g, rr[oa + i] * o + rr[ob + i] * P, dg[i]);
          float dui = rr[oe + i] * P;
#pragma unroll
          for (int j = 0; j < NJ; ++j)
            if (j < n) dui = fmaf(rr[oE + i * n + j], b[j], dui);
          du[i] += dui;
        }
      }
    }
  }
  if (valid) {
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      if (i < S) {
        atomicAdd(a.du + static_cast<int64_t>(i) * d + c, du[i]);
        if (a.dgamma_in != nullptr) atomicAdd(a.dgamma_in + static_cast<int64_t>(i) * d + c, dg[i]);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
template <typename IOT>
cudaError_t launch_merge(const BwdBlockArgs& a, cudaStream_t s) {
  constexpr int VE = Vec<IOT>::N;
  const int nv = a.d / VE;
  int vpt = 1;
  while ((nv + vpt - 1) / vpt > kRowThreads) vpt *= 2;
  const int threads = ((nv + vpt - 1) / vpt + 31) / 32 * 32;
  const unsigned grid = static_cast<unsigned>(a.T);
  switch (vpt) {
    case 1: return launch_pdl(bwd_merge_kernel<IOT, 1>, grid, threads, 0, s, a);
    case 2: return launch_pdl(bwd_merge_kernel<IOT, 2>, grid, threads, 0, s, a);
    default: return cudaErrorInvalidValue;
  }
}

template <typename IOT>
cudaError_t launch_rest(const BwdBlockArgs& a, cudaStream_t s) {
  cudaError_t e = launch_pdl(bwd_sources_kernel<IOT>, dim3(static_cast<unsigned>(a.T)),
                             dim3(kDotThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int gx = (a.d + kColThreads - 1) / kColThreads;
  int64_t gy = (8LL * sms + gx - 1) / gx;   // about eight CTAs per SM
  if (gy > a.T) gy = a.T;
  const int tpc = static_cast<int>((a.T + gy - 1) / gy);
  gy = (a.T + tpc - 1) / tpc;
  const size_t smem = static_cast<size_t>(kColBatch) * a.rec_floats * sizeof(float);
  auto kern = bwd_params_kernel<IOT>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                    dim3(kColThreads), smem, s, a, tpc);
}

}  // namespace

int64_t backward_block_workspace_bytes(IO io, int n, int S, int64_t T, int d) {
  (void)io;
  const int64_t SR = static_cast<int64_t>(S) * T;
  return align256(SR * d * 4) + align256(SR * 4) + align256(SR * n * 4) + align256(SR * d * 4) +
         align256(SR * 16) + align256(T * record_floats(n, S) * 4);
}

bool backward_block_supported(IO io, int n, int S, int d) {
  const int VE = io == IO::BF16 ? 8 : 4;
  return n >= 1 && n <= kBlkMaxN && S >= 1 && S <= kBlkMaxS && d % VE == 0 &&
         d / VE <= 2 * kRowThreads;   // the merge kernel keeps two vectors per thread
}

cudaError_t launch_backward_block(IO io, BwdBlockArgs a, void* workspace, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int64_t SR = static_cast<int64_t>(a.S) * a.T;
  char* w = static_cast<char*>(workspace);
  a.o = reinterpret_cast<float*>(w);
  w += align256(SR * a.d * 4);
  a.lse = reinterpret_cast<float*>(w);
  w += align256(SR * 4);
  a.alpha = reinterpret_cast<float*>(w);
  w += align256(SR * a.n * 4);
  a.q = reinterpret_cast<float*>(w);
  w += align256(SR * a.d * 4);
  a.sc2 = reinterpret_cast<float*>(w);
  w += align256(SR * 16);
  a.rec = reinterpret_cast<float*>(w);
  a.rec_floats = record_floats(a.n, a.S);
  // 1. phase 1 recomputed: o (fp32), lse, alpha over the completed sources
  Phase1Args p1{a.reps, a.src_stride, a.n, a.T, a.d, a.u, a.u_split, a.S, a.eps_key,
                a.o, nullptr, a.lse, a.alpha, kOF32, 1};
  cudaError_t e = launch_phase1(io, p1, s);
  if (e != cudaSuccess) return e;
  // 2. merge backward per token row
  e = io == IO::BF16 ? launch_merge<bf16>(a, s) : launch_merge<float>(a, s);
  if (e != cudaSuccess) return e;
  // 3, 4. the source and parameter gradients
  return io == IO::BF16 ? launch_rest<bf16>(a, s) : launch_rest<float>(a, s);
}

}  // namespace attnres
