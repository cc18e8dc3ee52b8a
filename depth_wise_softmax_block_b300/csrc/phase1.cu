// Phase 1 of the two-phase Block AttnRes schedule: all S pseudo-queries of a block scored
// against the n completed sources in one kernel ("Attention Residuals" note, §10 step 1;
// "Attention Residuals 阅读补充", section "静态 Query 与两阶段计算": stacking the static
// queries turns S matrix-vector products into one pass over the history).
//
// One CTA owns a tile of TT tokens and runs two sweeps over the hidden dimension d:
//   sweep 1  streams the tile's source rows [n][TT][64 columns] and the query slice [S][64]
//            through a 3-stage cp.async pipeline in shared memory.  Each warp takes one
//            8-column octet of every stage; each lane accumulates the logit numerators
//            u_s . b_j[t] of (NS sources x NQ queries) of one token and the sums of squares,
//            with packed fp32 FMAs over column pairs (even and odd columns are summed
//            separately and added at the end).
//   reduce   the 8 warps' partial sums are added in a fixed order (deterministic), then one
//            thread per (token, query) forms r_j, z_j, m, lse and alpha.
//   sweep 2  streams the same source rows again (from L2 when they are still there) and
//            writes o[s,t,:] = sum_j alpha_j b_j[t,:] with 16-byte streaming stores.
// Arithmetic is fp32 throughout; o is rounded once to the I/O type.  A single query (S = 1,
// the final aggregation) has no logits to share across queries and runs on the row-wise
// single-pass kernel instead.
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace attnres {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int KC = 64;        // columns per pipeline stage (one 8-column octet per warp)
constexpr int kStages = 3;
constexpr int kUnit = 16;     // cp.async granule in bytes
constexpr int kMaxSmem = 227 * 1024;

struct P1Plan {
  int SG, QG, TT;       // source groups, query groups, tokens per CTA
  int ttShift;          // log2(TT): TT is a power of two
  int rowB, uRowB;      // bytes per staged (source, token) row / query row
  int bBytes, stageBytes;
  int RS;               // floats per thread in the cross-warp reduction buffer (odd)
  int offDots, offAlpha;
  int smem;
};

inline int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}
inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Register-tile shape (NS sources x NQ queries per lane) for S >= 2.
inline void tile_shape(int S, int& NS, int& NQ) {
  if (S <= 4) { NS = 9; NQ = 4; }
  else if (S <= 24) { NS = 9; NQ = 6; }
  else { NS = 4; NQ = 8; }
}

bool make_plan(int n, int S, int E, P1Plan& p) {
  int NS, NQ;
  tile_shape(S, NS, NQ);
  p.SG = next_pow2((n + NS - 1) / NS);
  p.QG = next_pow2((S + NQ - 1) / NQ);
  if (p.SG * p.QG > 32) return false;
  p.rowB = KC * E + 16;
  p.uRowB = KC * 4 + 16;
  p.RS = NS * NQ + NS;
  if ((p.RS & 1) == 0) p.RS += 1;
  for (p.TT = 32 / (p.SG * p.QG); p.TT >= 1; p.TT /= 2) {
    p.bBytes = n * p.TT * p.rowB;
    const int uBytes = S * p.uRowB + p.QG * kUnit;
    p.stageBytes = align_up(p.bBytes + uBytes, 128);
    const int area0 = std::max(kStages * p.stageBytes, kThreads * p.RS * 4);
    p.offDots = align_up(area0, 16);
    p.offAlpha = align_up(p.offDots + p.TT * n * (S + 1) * 4, 16);
    p.smem = p.offAlpha + p.TT * n * p.QG * NQ * 2 * 4;
    p.ttShift = 0;
    while ((1 << p.ttShift) < p.TT) ++p.ttShift;
    if (p.smem <= kMaxSmem) return true;
  }
  return false;
}

// Streaming (evict-first) store of the phase-1 output, which phase 2 reads once much later.
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// Eight consecutive elements as four (even, odd) column pairs.
template <typename T> __device__ __forceinline__ void load_pairs(const void* p, float2 (&f)[4]);
template <> __device__ __forceinline__ void load_pairs<bf16>(const void* p, float2 (&f)[4]) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}
template <> __device__ __forceinline__ void load_pairs<float>(const void* p, float2 (&f)[4]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  f[0] = make_float2(a.x, a.y);
  f[1] = make_float2(a.z, a.w);
  f[2] = make_float2(b.x, b.y);
  f[3] = make_float2(b.z, b.w);
}

template <typename T> __device__ __forceinline__ void store_pairs(void* p, const float2 (&f)[4]);
template <> __device__ __forceinline__ void store_pairs<bf16>(void* p, const float2 (&f)[4]) {
  st_stream(p, make_uint4(pack_bf16x2(f[0].x, f[0].y), pack_bf16x2(f[1].x, f[1].y),
                          pack_bf16x2(f[2].x, f[2].y), pack_bf16x2(f[3].x, f[3].y)));
}
template <> __device__ __forceinline__ void store_pairs<float>(void* p, const float2 (&f)[4]) {
  st_stream(p, make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                          __float_as_uint(f[1].x), __float_as_uint(f[1].y)));
  st_stream(static_cast<char*>(p) + 16,
            make_uint4(__float_as_uint(f[2].x), __float_as_uint(f[2].y),
                       __float_as_uint(f[3].x), __float_as_uint(f[3].y)));
}

template <typename IOT, int NS, int NQ>
__global__ void __launch_bounds__(kThreads, 1)
phase1_kernel(const Phase1Args a, const P1Plan pl) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = sizeof(IOT);
  constexpr int UPR = KC * E / kUnit;  // 16-byte units per staged source row
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = a.n, S = a.S, d = a.d;
  const int TT = pl.TT, QG = pl.QG, SG = pl.SG;
  const int64_t T = a.T;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * TT;
  const int nchunks = (d + KC - 1) / KC;
  const char* reps = static_cast<const char*>(a.reps);

  // Stage chunk c (columns c*KC ..) into pipeline slot `slot`; zero-fill past T and d.
  auto issue = [&](int c, int slot, bool with_u) {
    unsigned char* st = smem + slot * pl.stageBytes;
    const int k0 = c * KC;
    const int nb = n * TT * UPR;
    for (int i = tid; i < nb; i += kThreads) {
      const int unit = i % UPR, row = i / UPR;  // row = j * TT + t (TT a power of two)
      const int t = row & (TT - 1), j = row >> pl.ttShift;
      const int k = k0 + unit * (kUnit / E);
      const bool ok = (t0 + t < T) && (k < d);
      const char* src =
          ok ? reps + (static_cast<int64_t>(j) * a.src_stride + (t0 + t) * d + k) * E : reps;
      cp_async16(st + row * pl.rowB + unit * kUnit, src, ok);
    }
    if (with_u) {
      unsigned char* ut = st + pl.bBytes;
      const int nu = S * (KC * 4 / kUnit);
      for (int i = tid; i < nu; i += kThreads) {
        const int unit = i % (KC * 4 / kUnit), q = i / (KC * 4 / kUnit);
        const int k = k0 + unit * 4;
        const bool ok = k < d;
        const float* src = ok ? a.u + static_cast<int64_t>(q) * d + k : a.u;
        // query groups are offset by one granule so the QG groups hit distinct banks
        cp_async16(ut + q * pl.uRowB + (q / NQ) * kUnit + unit * kUnit, src, ok);
      }
    }
  };

  // ---------------- sweep 1: logit numerators and sums of squares ----------------
  const bool active1 = lane < TT * SG * QG;
  const int g = lane % QG;
  const int sg = (lane / QG) % SG;
  const int tl = lane / (QG * SG);
  float2 acc[NS][NQ];
  float2 ss[NS];
#pragma unroll
  for (int jj = 0; jj < NS; ++jj) {
    ss[jj] = make_float2(0.f, 0.f);
#pragma unroll
    for (int qq = 0; qq < NQ; ++qq) acc[jj][qq] = make_float2(0.f, 0.f);
  }

#pragma unroll
  for (int c = 0; c < kStages - 1; ++c) {
    if (c < nchunks) issue(c, c, true);
    cp_async_commit();
  }
  for (int c = 0; c < nchunks; ++c) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    if (c + kStages - 1 < nchunks) issue(c + kStages - 1, (c + kStages - 1) % kStages, true);
    cp_async_commit();
    if (active1) {
      const unsigned char* st = smem + (c % kStages) * pl.stageBytes;
      const unsigned char* ut = st + pl.bBytes + g * kUnit + warp * 32;
      float2 uv[NQ][4];
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq) {
        if (g * NQ + qq < S) {  // padded queries of the last group read nothing
          load_pairs<float>(ut + (g * NQ + qq) * pl.uRowB, uv[qq]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) uv[qq][i] = make_float2(0.f, 0.f);
        }
      }
      const unsigned char* bt = st + tl * pl.rowB + warp * 8 * E;
#pragma unroll
      for (int jj = 0; jj < NS; ++jj) {
        const int j = sg * NS + jj;
        if (j < n) {
          float2 bv[4];
          load_pairs<IOT>(bt + j * TT * pl.rowB, bv);
          // the sum-of-squares chain is spread between independent dot-product updates
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            ss[jj] = __ffma2_rn(bv[i], bv[i], ss[jj]);
#pragma unroll
            for (int qq = 0; qq < NQ; ++qq) acc[jj][qq] = __ffma2_rn(uv[qq][i], bv[i], acc[jj][qq]);
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---------------- reduce the 8 warps' partial sums (fixed order) ----------------
  float* red = reinterpret_cast<float*>(smem);  // reuses the pipeline slots
  if (active1) {
    float* r = red + tid * pl.RS;
#pragma unroll
    for (int jj = 0; jj < NS; ++jj) {
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq) r[jj * NQ + qq] = acc[jj][qq].x + acc[jj][qq].y;
      r[NS * NQ + jj] = ss[jj].x + ss[jj].y;
    }
  }
  __syncthreads();
  float* dots = reinterpret_cast<float*>(smem + pl.offDots);  // [TT][n][S + 1]
  const int S1 = S + 1;
  for (int i = tid; i < TT * n * S1; i += kThreads) {
    const int s = i % S1, j = (i / S1) % n, t = i / (S1 * n);
    const int gg = s < S ? s / NQ : 0;
    const int ln = (t * SG + j / NS) * QG + gg;
    const int idx = s < S ? (j % NS) * NQ + (s - gg * NQ) : NS * NQ + (j % NS);
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) sum += red[(w * 32 + ln) * pl.RS + idx];
    dots[i] = sum;
  }
  __syncthreads();

  // The pipeline slots are free again: start staging sweep 2 while the softmax runs.
#pragma unroll
  for (int c = 0; c < kStages - 1; ++c) {
    if (c < nchunks) issue(c, c, false);
    cp_async_commit();
  }

  // ---------------- softmax statistics, one thread per (token, query) ----------------
  // alpha is stored twice, (a, a), so sweep 2 reads ready-made pairs: [TT][n][QG][NQ][2]
  float* alph = reinterpret_cast<float*>(smem + pl.offAlpha);
  const float fd = static_cast<float>(d);
  for (int i = tid; i < TT * S; i += kThreads) {
    const int t = i / S, s = i % S;
    const int64_t tok = t0 + t;
    const float* dt = dots + t * n * S1;
    float m = -INFINITY;
    for (int j = 0; j < n; ++j) {
      const float z = dt[j * S1 + s] / sqrtf(dt[j * S1 + S] / fd + a.eps);
      m = fmaxf(m, z);
    }
    float l = 0.f;
    for (int j = 0; j < n; ++j) {
      const float z = dt[j * S1 + s] / sqrtf(dt[j * S1 + S] / fd + a.eps);
      l += expf(z - m);
    }
    const float lse = m + logf(l);
    for (int j = 0; j < n; ++j) {
      const float z = dt[j * S1 + s] / sqrtf(dt[j * S1 + S] / fd + a.eps);
      const float al = expf(z - m) / l;
      float* ap = alph + (((t * n + j) * QG + s / NQ) * NQ + s % NQ) * 2;
      ap[0] = al;
      ap[1] = al;
      if (a.alpha != nullptr && tok < T) a.alpha[(static_cast<int64_t>(s) * T + tok) * n + j] = al;
    }
    if (tok < T) {
      if (a.m != nullptr) a.m[static_cast<int64_t>(s) * T + tok] = m;
      if (a.lse != nullptr) a.lse[static_cast<int64_t>(s) * T + tok] = lse;
    }
  }

  // ---------------- sweep 2: o[s,t,:] = sum_j alpha[s,t,j] b_j[t,:] ----------------
  const bool active2 = tid < TT * QG * 8;
  const int kg = tid % 8, g2 = (tid / 8) % QG, t2 = tid / (8 * QG);
  const int64_t tok2 = t0 + t2;
  char* o = static_cast<char*>(a.o);
  for (int c = 0; c < nchunks; ++c) {
    cp_async_wait<kStages - 2>();
    __syncthreads();  // also orders the softmax's alpha writes before the first use
    if (c + kStages - 1 < nchunks) issue(c + kStages - 1, (c + kStages - 1) % kStages, false);
    cp_async_commit();
    if (active2) {
      const unsigned char* bt = smem + (c % kStages) * pl.stageBytes + t2 * pl.rowB + kg * 8 * E;
      const float* at = alph + (t2 * n * QG + g2) * NQ * 2;
      float2 acc2[NQ][4];
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc2[qq][i] = make_float2(0.f, 0.f);
      // The next source's octet and alpha pairs are read from shared memory while the
      // current source is accumulated (the trip count n is a runtime value).
      float2 bv[4], bn[4];
      float4 af[NQ / 2], an[NQ / 2];
      load_pairs<IOT>(bt, bn);
#pragma unroll
      for (int h = 0; h < NQ / 2; ++h) an[h] = reinterpret_cast<const float4*>(at)[h];
      for (int j = 0; j < n; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) bv[i] = bn[i];
#pragma unroll
        for (int h = 0; h < NQ / 2; ++h) af[h] = an[h];
        if (j + 1 < n) {
          load_pairs<IOT>(bt + (j + 1) * TT * pl.rowB, bn);
          const float4* ap = reinterpret_cast<const float4*>(at + (j + 1) * QG * NQ * 2);
#pragma unroll
          for (int h = 0; h < NQ / 2; ++h) an[h] = ap[h];
        }
        float2 al[NQ];
#pragma unroll
        for (int h = 0; h < NQ / 2; ++h) {
          al[2 * h] = make_float2(af[h].x, af[h].y);
          al[2 * h + 1] = make_float2(af[h].z, af[h].w);
        }
#pragma unroll
        for (int qq = 0; qq < NQ; ++qq)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc2[qq][i] = __ffma2_rn(al[qq], bv[i], acc2[qq][i]);
      }
      const int k = c * KC + kg * 8;
      if (tok2 < T && k < d) {
#pragma unroll
        for (int qq = 0; qq < NQ; ++qq) {
          const int q = g2 * NQ + qq;
          if (q < S)
            store_pairs<IOT>(o + ((static_cast<int64_t>(q) * T + tok2) * d + k) * E, acc2[qq]);
        }
      }
    }
  }
  cp_async_wait<0>();
}

template <typename T, int NS, int NQ>
cudaError_t launch_t(const Phase1Args& a, const P1Plan& pl, cudaStream_t s) {
  auto kern = phase1_kernel<T, NS, NQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (a.T + pl.TT - 1) / pl.TT;
  kern<<<static_cast<unsigned>(blocks), kThreads, pl.smem, s>>>(a, pl);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_io(const Phase1Args& a, cudaStream_t s) {
  P1Plan pl;
  if (!make_plan(a.n, a.S, sizeof(T), pl)) return cudaErrorInvalidValue;
  int NS, NQ;
  tile_shape(a.S, NS, NQ);
  if (NQ == 4) return launch_t<T, 9, 4>(a, pl, s);
  if (NQ == 6) return launch_t<T, 9, 6>(a, pl, s);
  return launch_t<T, 4, 8>(a, pl, s);
}

}  // namespace

bool phase1_supported(int n, int S) {
  if (S == 1) return n >= 1 && n <= kMaxSources;
  P1Plan pl;
  return make_plan(n, S, 4, pl) && make_plan(n, S, 2, pl);
}

cudaError_t launch_phase1(IO io, const Phase1Args& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.S == 1) {  // one query: the row-wise single-pass kernel, sources at base + j * stride
    FullArgs f;
    memset(&f, 0, sizeof(f));
    const int64_t E = io == IO::BF16 ? 2 : 4;
    for (int j = 0; j < a.n; ++j)
      f.srcs[j] = static_cast<const char*>(a.reps) + j * a.src_stride * E;
    f.n = a.n;
    f.T = a.T;
    f.d = a.d;
    f.u = a.u;
    f.eps_key = a.eps;
    f.h = a.o;
    f.alpha = a.alpha;
    f.m = a.m;
    f.lse = a.lse;
    return launch_full(io, f, s);
  }
  return io == IO::BF16 ? launch_io<bf16>(a, s) : launch_io<float>(a, s);
}

}  // namespace attnres
