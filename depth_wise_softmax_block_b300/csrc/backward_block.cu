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
// Five launches, each source row of the block read a bounded number of times (not once per
// sublayer):
//   1. phase 1 recomputed (the forward's own kernel) over the n sources for the S queries:
//      o_i (fp32), lse_i, alpha_ij into the workspace;
//   2. bwd_merge_kernel, one CTA per token row, the S sublayers in reverse order with the
//      partial sum and the dL/dv running sums in shared memory: per sublayer one CTA reduction of
//      six sums (|p|^2, u.p, |o|^2, o.p, gamma g.o, gamma g.p) gives every scalar of the merge
//      and of both norms' backward; writes q_i (fp32) and dL/dv_{i-1};
//   3. bwd_sources_kernel, one CTA per token row: q_i . b_j for all (i, j) and |b_j|^2 (eight
//      warps, three queries each), the coefficients dz_ij / r_j and sum_i dz_ij z_ij / (d r_j^2),
//      then dL/db_j per element in a second pass (q_i again, from L2); the coefficients the
//      parameter sums need go to a per-token record;
//   4. bwd_params_kernel, two columns per thread and 32 tokens per CTA: the partial sums' part
//      of du_i and dgamma_in,i, summed over the CTA's tokens (one atomic per element, CTA and
//      sublayer);
//   5. bwd_du_kernel: the sources' part of du_i, sum over tokens and sources of E_ij b_j, as a
//      register-blocked product (six sublayers x four columns per thread).
// Softmax weights, key RMSNorm, one head (the method as defined).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace attnres {
namespace {

constexpr int kRowThreads = 256;    // merge kernel: at most 256 threads per row
constexpr int kDotThreads = 256;    // sources kernel: 8 warps
constexpr int kDotQ = 3;            // queries per warp in the sources kernel's dots (8 x 3 = 24)
constexpr int kDbGroup = 8;         // sources whose gradients a thread accumulates at once

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
// 2. merge backward: one CTA per token row, sublayers S .. 1.  The running partial sum p_i and
// the running sum of dL/dp live in shared memory (element (v, e) of the row at e * nv + v, so
// the threads of a warp touch consecutive words), which keeps the registers low enough for
// three rows per SM; the rows of o_i, g_i and v_{i-1} are all requested at the start of a
// sublayer.
template <typename IOT, int VPT>
__global__ void __launch_bounds__(kRowThreads, 2) bwd_merge_kernel(const BwdBlockArgs a) {
  constexpr int VE = Vec<IOT>::N;
  constexpr int NW = OWords<float, VE>::N;
  __shared__ float scratch[6 * 33];
  extern __shared__ float pa[];   // P [VE][nv], then A [VE][nv]
  pdl_wait();
  const int64_t t = blockIdx.x, T = a.T;
  const int d = a.d, nv = d / VE, S = a.S;
  const float fd = static_cast<float>(d);
  const int64_t row = t * d;
  float* Ps = pa;
  float* As = pa + d;

#pragma unroll
  for (int k = 0; k < VPT; ++k) {  // p_S = v_1 + ... + v_{S-1}, and A = 0
    const int v = threadIdx.x + k * blockDim.x;
    if (v < nv) {
      float acc[VE];
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[e] = 0.f;
#pragma unroll 4
      for (int kv = 1; kv < S; ++kv) {
        float x[VE];
        unpack(ld_stream(static_cast<const IOT*>(a.v) + (kv - 1) * a.v_stride + row + v * VE), x);
#pragma unroll
        for (int e = 0; e < VE; ++e) acc[e] += x[e];
      }
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        Ps[e * nv + v] = acc[e];
        As[e * nv + v] = 0.f;
      }
    }
  }

  for (int i = S; i >= 1; --i) {
    const bool has_p = i >= 2;
    const int64_t ri = static_cast<int64_t>(i - 1) * T + t;
    const float* ui = a.u + static_cast<int64_t>(i - 1) * d;
    const float* gam = a.gamma_in ? a.gamma_in + static_cast<int64_t>(i - 1) * d : nullptr;
    uint4 ro[VPT][NW], rg[VPT], rv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = threadIdx.x + k * blockDim.x;
      if (v < nv) {
        ld_stream_w<float, VE>(a.o + ri * d + v * VE, ro[k]);
        rg[k] = ld_stream(static_cast<const IOT*>(a.g_y) + ri * d + v * VE);
        if (has_p)
          rv[k] = ld_stream(static_cast<const IOT*>(a.v) + (i - 2) * a.v_stride + row + v * VE);
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
          const float p = Ps[e * nv + v];
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
        float o[VE], g[VE], q[VE], uu[VE], gg[VE], dv[VE], x[VE];
        unpack_w<float, VE>(ro[k], o);
        unpack(rg[k], g);
        ldg_f32<VE>(ui + v * VE, uu);
        if (gam) {
          ldg_f32<VE>(gam + v * VE, gg);
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) gg[e] = 1.f;
        }
        if (has_p) unpack(rv[k], x);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float p = Ps[e * nv + v];
          const float h = wA * o[e] + wP * p;
          const float gh = gg[e] * g[e] * inv_rh - kap * h;
          q[e] = wA * gh;
          if (has_p) {
            dv[e] = As[e * nv + v] + wP * gh + coefu * uu[e] - coefp * p;
            As[e * nv + v] = dv[e];
            Ps[e * nv + v] = p - x[e];   // p_{i-1} = p_i - v_{i-1}
          }
        }
        st_vec<float, VE>(qi + v * VE, q);
        if (has_p) st_vec<IOT, VE>(dvi + v * VE, dv);
      }
    }
    if (threadIdx.x == 0)
      *reinterpret_cast<float4*>(a.sc2 + ri * 4) = make_float4(c, wA * inv_rh, wP * inv_rh, coefu);
  }
}

// ------------------------------------------------------------------------------------------
// 3. sources: per token, q_i . b_j for all (i, j) and |b_j|^2 (pass 1), the coefficients, then
// dL/db_j = sum_i alpha_ij q_i + sum_i E_ij u_i - F_j b_j per element (pass 2, q_i again from
// L2), with E_ij = dz_ij / r_j and F_j = sum_i dz_ij z_ij / (d r_j^2).
template <typename IOT>
__global__ void __launch_bounds__(kDotThreads, 3) bwd_sources_kernel(const BwdBlockArgs a) {
  constexpr int VE = Vec<IOT>::N;
  constexpr int NJ = kBlkMaxN;
  constexpr int NW = OWords<float, VE>::N;
  __shared__ float Ds[kBlkMaxS * NJ];   // D_ij, then E_ij
  __shared__ float As[kBlkMaxS * NJ];   // alpha_ij
  __shared__ float dzz[kBlkMaxS * NJ];
  __shared__ float ssj[NJ], Fs[NJ];
  pdl_wait();
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
__device__ __forceinline__ void ld2(const IOT* p, float& x, float& y) {
  if constexpr (sizeof(IOT) == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    x = __uint_as_float(w << 16);
    y = __uint_as_float(w & 0xffff0000u);
  } else {
    const float2 f = *reinterpret_cast<const float2*>(p);
    x = f.x;
    y = f.y;
  }
}

// The CTA owns kParCols columns (two per thread) and kParTok consecutive tokens.  Sublayers run
// in the outer loop, tokens in the inner one, so all loads of a sublayer over the CTA's tokens
// are independent: the partial sums p_i of the CTA's tokens live in shared memory
// ([token][column], updated with v_{i-1} before sublayer i), and the per-token scalars
// (w_A / r_h, w_p / r_h, dz_p / r_p of every sublayer) are staged once.
constexpr int kParThreads = 128;
constexpr int kParCols = 2 * kParThreads;
constexpr int kParTok = 32;

template <typename IOT>
__global__ void __launch_bounds__(kParThreads) bwd_params_kernel(const BwdBlockArgs a) {
  extern __shared__ float psm[];   // P [kParTok][kParCols], then scalars [kParTok][3S]
  pdl_wait();
  const int d = a.d, S = a.S, n = a.n, R = a.rec_floats;
  const int64_t T = a.T;
  const int cl = 2 * threadIdx.x;                 // local column pair
  const int c = blockIdx.x * kParCols + cl;
  const bool valid = c < d;                       // d is even
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kParTok;
  const int nt = static_cast<int>(T - t0 < kParTok ? T - t0 : kParTok);
  float* Ps = psm;
  float* sc = psm + kParTok * kParCols;
  for (int k = threadIdx.x; k < nt * 3 * S; k += blockDim.x) {
    const int tt = k / (3 * S), r = k - tt * 3 * S;
    sc[k] = a.rec[(t0 + tt) * R + S * n + r];      // a [S], b [S], e [S] of token t0 + tt
  }
  for (int tt = 0; tt < nt; ++tt) {
    Ps[tt * kParCols + cl] = 0.f;
    Ps[tt * kParCols + cl + 1] = 0.f;
  }
  __syncthreads();
  if (!valid) return;
  const IOT* vb = static_cast<const IOT*>(a.v);
  const IOT* gb = static_cast<const IOT*>(a.g_y);
  for (int i = 0; i < S; ++i) {                   // sublayer i + 1
    float du0 = 0.f, du1 = 0.f, dg0 = 0.f, dg1 = 0.f;
#pragma unroll 8
    for (int tt = 0; tt < nt; ++tt) {
      const int64_t t = t0 + tt;
      float p0 = Ps[tt * kParCols + cl], p1 = Ps[tt * kParCols + cl + 1];
      if (i >= 1) {
        float x0, x1;
        ld2(vb + (i - 1) * a.v_stride + t * d + c, x0, x1);
        p0 += x0;
        p1 += x1;
        Ps[tt * kParCols + cl] = p0;
        Ps[tt * kParCols + cl + 1] = p1;
      }
      const int64_t at = (static_cast<int64_t>(i) * T + t) * d + c;
      const float2 o = *reinterpret_cast<const float2*>(a.o + at);
      float g0, g1;
      ld2(gb + at, g0, g1);
      const float* st = sc + tt * 3 * S;
      const float wa = st[i], wb = st[S + i], we = st[2 * S + i];
      dg0 = fmaf(g0, wa * o.x + wb * p0, dg0);
      dg1 = fmaf(g1, wa * o.y + wb * p1, dg1);
      du0 = fmaf(we, p0, du0);
      du1 = fmaf(we, p1, du1);
    }
    atomicAdd(a.du + static_cast<int64_t>(i) * d + c, du0);
    atomicAdd(a.du + static_cast<int64_t>(i) * d + c + 1, du1);
    if (a.dgamma_in != nullptr) {
      atomicAdd(a.dgamma_in + static_cast<int64_t>(i) * d + c, dg0);
      atomicAdd(a.dgamma_in + static_cast<int64_t>(i) * d + c + 1, dg1);
    }
  }
}

// ------------------------------------------------------------------------------------------
// 5. the sources' part of the query gradients, du_i += sum_t sum_j E_ij(t) b_j(t): a product of
// the [S x (tokens x sources)] coefficients and the [(tokens x sources) x d] source rows, summed
// over a range of tokens per CTA.  Warp w owns sublayers 6w .. 6w + 5, lane l four columns; the
// CTA stages its tokens' coefficients in shared memory as [token][source][sublayer].
constexpr int kDuThreads = 128;   // 4 warps x 6 sublayers = 24
constexpr int kDuCols = 128;      // columns per CTA (4 per lane)
constexpr int kDuRows = 6;        // sublayers per warp
constexpr int kDuBatch = 32;      // tokens staged at a time

template <typename IOT>
__device__ __forceinline__ void ld4(const IOT* p, float (&f)[4]) {
  if constexpr (sizeof(IOT) == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
  } else {
    const float4 x = *reinterpret_cast<const float4*>(p);
    f[0] = x.x;
    f[1] = x.y;
    f[2] = x.z;
    f[3] = x.w;
  }
}

template <typename IOT>
__global__ void __launch_bounds__(kDuThreads) bwd_du_kernel(const BwdBlockArgs a,
                                                            int tokens_per_cta) {
  constexpr int SP = 24;                      // padded sublayer stride of the staged tile
  extern __shared__ float ce[];               // [kDuBatch][n][SP]
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, S = a.S, n = a.n, R = a.rec_floats;
  const int64_t T = a.T;
  const int c = blockIdx.x * kDuCols + 4 * lane;
  const bool valid = c < d;                   // d is a multiple of 4
  const int i0 = warp * kDuRows;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * tokens_per_cta;
  const int64_t t1 = t0 + tokens_per_cta < T ? t0 + tokens_per_cta : T;
  const IOT* reps = static_cast<const IOT*>(a.reps);
  float acc[kDuRows][4];
#pragma unroll
  for (int r = 0; r < kDuRows; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[r][e] = 0.f;
  for (int64_t tb0 = t0; tb0 < t1; tb0 += kDuBatch) {
    const int nb = static_cast<int>(t1 - tb0 < kDuBatch ? t1 - tb0 : kDuBatch);
    __syncthreads();
    for (int k = threadIdx.x; k < nb * S * n; k += blockDim.x) {  // record [i][j] -> [j][i]
      const int tb = k / (S * n), rem = k - tb * S * n, i = rem / n, j = rem - i * n;
      ce[(tb * n + j) * SP + i] = a.rec[(tb0 + tb) * R + rem];
    }
    __syncthreads();
    if (!valid || i0 >= S) continue;
    for (int tb = 0; tb < nb; ++tb) {
      const IOT* bt = reps + (tb0 + tb) * d + c;
#pragma unroll 3
      for (int j = 0; j < n; ++j) {
        float b[4];
        ld4(bt + j * a.src_stride, b);
        const float* e = ce + (tb * n + j) * SP + i0;
#pragma unroll
        for (int r = 0; r < kDuRows; ++r) {
          const float er = e[r];
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(er, b[q], acc[r][q]);
        }
      }
    }
  }
  if (valid) {
#pragma unroll
    for (int r = 0; r < kDuRows; ++r)
      if (i0 + r < S)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          atomicAdd(a.du + static_cast<int64_t>(i0 + r) * d + c + q, acc[r][q]);
  }
}

// ------------------------------------------------------------------------------------------
template <typename IOT, int VPT>
cudaError_t launch_merge_vpt(const BwdBlockArgs& a, int threads, cudaStream_t s) {
  const size_t smem = 2 * static_cast<size_t>(a.d) * sizeof(float);
  auto kern = bwd_merge_kernel<IOT, VPT>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(static_cast<unsigned>(a.T)), dim3(threads), smem, s, a);
}

template <typename IOT>
cudaError_t launch_merge(const BwdBlockArgs& a, cudaStream_t s) {
  constexpr int VE = Vec<IOT>::N;
  const int nv = a.d / VE;
  int vpt = 1;
  while ((nv + vpt - 1) / vpt > kRowThreads) vpt *= 2;
  const int threads = ((nv + vpt - 1) / vpt + 31) / 32 * 32;
  switch (vpt) {
    case 1: return launch_merge_vpt<IOT, 1>(a, threads, s);
    case 2: return launch_merge_vpt<IOT, 2>(a, threads, s);
    case 4: return launch_merge_vpt<IOT, 4>(a, threads, s);
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
  const int gx = (a.d + kParCols - 1) / kParCols;
  const int64_t gy = (a.T + kParTok - 1) / kParTok;
  const size_t smem = (static_cast<size_t>(kParTok) * kParCols + kParTok * 3 * a.S) * sizeof(float);
  auto kern = bwd_params_kernel<IOT>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                 dim3(kParThreads), smem, s, a);
  if (e != cudaSuccess) return e;
  // the sources' part of du
  const int dx = (a.d + kDuCols - 1) / kDuCols;
  int64_t dy = (6LL * sms + dx - 1) / dx;
  if (dy > a.T) dy = a.T;
  const int dtpc = static_cast<int>((a.T + dy - 1) / dy);
  dy = (a.T + dtpc - 1) / dtpc;
  const size_t dsmem = static_cast<size_t>(kDuBatch) * a.n * 24 * sizeof(float);
  auto dkern = bwd_du_kernel<IOT>;
  e = cudaFuncSetAttribute(dkern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(dsmem));
  if (e != cudaSuccess) return e;
  return launch_pdl(dkern, dim3(static_cast<unsigned>(dx), static_cast<unsigned>(dy)),
                    dim3(kDuThreads), dsmem, s, a, dtpc);
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
         d / VE <= 4 * kRowThreads;   // the merge kernel keeps four vectors per thread
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
