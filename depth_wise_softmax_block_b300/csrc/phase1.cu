// Phase 1 of the two-phase Block AttnRes schedule: all S pseudo-queries of a block scored
// against the n completed sources in one kernel ("Attention Residuals" note, §10 step 1;
// "Attention Residuals 阅读补充", section "静态 Query 与两阶段计算": stacking the static
// queries turns S matrix-vector products into one pass over the history).
//
// One CTA of 8 warps owns a tile of TT tokens.  Thread 0 streams the tile through a ring of
// shared-memory stages with tensor (TMA) copies: a stage is the 128-byte column slice
// (64 bf16 or 32 fp32 columns) of all n x TT source rows, plus, during the first sweep, the
// same columns of the S queries.  Copies use the 128-byte swizzle, so 16-byte reads of eight
// different rows hit eight different bank groups.  The warps run:
//   sweep 1  each warp takes one 16-byte column chunk of every stage; each lane accumulates
//            the logit numerators u_s . b_j[t] of (NS sources x NQ queries) of one token and
//            the sums of squares, with packed fp32 FMAs over column pairs;
//   reduce   the 8 warps' partial sums are added in a fixed order (deterministic); then
//            r_j, z_j = u_s . b_j / r_j, m, lse and alpha for every (token, query);
//   sweep 2  the same source rows stream through the ring again (its first stages are already
//            in flight while the reduction runs) and o[s,t,:] = sum_j alpha_j b_j[t,:] is
//            written with 16-byte streaming stores.
// Stage hand-off uses "full" (copy landed) and "empty" (all warps done) mbarriers;
// every wait is bounded (tma.cuh).  Arithmetic is fp32; o is rounded once to the I/O type.
// A single query (S = 1, the final aggregation) has nothing to share across queries and runs
// on the row-wise single-pass kernel instead.
// Depth-attention heads (multi-head variant of Table 4, "Attention Residuals" note, result 4):
// grid.y walks the H heads and a CTA covers its head's columns k*dh .. k*dh + dh - 1 only
// (dh = d / H); a stage's column chunks past the head's end hold the next head's columns and
// are skipped.  Statistics are per (query, head).
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace attnres {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSmem = 227 * 1024;
constexpr int kMaxStages = 8;
constexpr int kRow = 128;                     // bytes per staged row (one swizzle span)

struct P1Plan {
  int SG, QG, TT;       // source groups, query groups, tokens per CTA
  int KC;               // columns per stage (kRow bytes of a row)
  int nUBox;            // query boxes per stage (32 fp32 columns each)
  int bBytes, bSpan;    // bytes of the source box as copied / rounded up to 1024
  int uBox, uSpan;      // bytes of one query box as copied / rounded up to 1024
  int stageBytes, ST;   // bytes per stage, number of stages
  int RS;               // floats per thread in the cross-warp reduction (odd)
  int offRed, offDots, offBar;
  int smem;             // dynamic shared memory to request (includes 1024 alignment slack)
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
  p.KC = kRow / E;
  p.nUBox = p.KC * 4 / kRow;
  p.RS = NS * NQ + NS;
  if ((p.RS & 1) == 0) p.RS += 1;
  p.uBox = S * kRow;
  p.uSpan = align_up(p.uBox, 1024);
  for (p.TT = 32 / (p.SG * p.QG); p.TT >= 1; p.TT /= 2) {
    p.bBytes = n * p.TT * kRow;
    p.bSpan = align_up(p.bBytes, 1024);
    p.stageBytes = p.bSpan + p.nUBox * p.uSpan;
    const int red = std::max(kThreads * p.RS * 4, p.TT * n * p.QG * NQ * 2 * 4);
    const int dots = p.TT * n * (S + 1) * 4;
    const int fixed = align_up(red, 16) + align_up(dots, 16) + (2 * kMaxStages + 2) * 8;
    const int room = kMaxSmem - 1024 - fixed;
    p.ST = std::min(kMaxStages, room / p.stageBytes);
    if (p.ST < 2) continue;
    p.offRed = p.ST * p.stageBytes;
    p.offDots = p.offRed + align_up(red, 16);
    p.offBar = p.offDots + align_up(dots, 16);
    p.smem = 1024 + p.offBar + (2 * p.ST + 2) * 8;
    return true;
  }
  return false;
}

// Streaming (evict-first) store of the phase-1 output, which phase 2 reads once much later.
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// One 16-byte chunk as (even, odd) column pairs: 4 pairs of bf16, 2 pairs of fp32.
template <typename T> struct Chunk;
template <> struct Chunk<bf16> {
  static constexpr int PR = 4;
  // The same pairs stored as fp32 (phase 1's o with kOF32): two 16-byte words.
  static __device__ __forceinline__ void store_f32(void* p, const float2 (&f)[PR]) {
    st_stream(p, make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                            __float_as_uint(f[1].x), __float_as_uint(f[1].y)));
    st_stream(static_cast<char*>(p) + 16,
              make_uint4(__float_as_uint(f[2].x), __float_as_uint(f[2].y),
                         __float_as_uint(f[3].x), __float_as_uint(f[3].y)));
  }
  static __device__ __forceinline__ void load(const void* p, float2 (&f)[PR]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
  static __device__ __forceinline__ void store(void* p, const float2 (&f)[PR]) {
    st_stream(p, make_uint4(pack_bf16x2(f[0].x, f[0].y), pack_bf16x2(f[1].x, f[1].y),
                            pack_bf16x2(f[2].x, f[2].y), pack_bf16x2(f[3].x, f[3].y)));
  }
};
template <> struct Chunk<float> {
  static constexpr int PR = 2;
  static __device__ __forceinline__ void store_f32(void* p, const float2 (&f)[PR]) {
    store(p, f);
  }
  static __device__ __forceinline__ void load(const void* p, float2 (&f)[PR]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    f[0] = make_float2(a.x, a.y);
    f[1] = make_float2(a.z, a.w);
  }
  static __device__ __forceinline__ void store(void* p, const float2 (&f)[PR]) {
    st_stream(p, make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                            __float_as_uint(f[1].x), __float_as_uint(f[1].y)));
  }
};

template <typename IOT, int NS, int NQ>
__global__ void __launch_bounds__(kThreads, 1)
phase1_kernel(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_u,
              const Phase1Args a, const P1Plan pl) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  constexpr int E = sizeof(IOT);
  constexpr int VE = 16 / E;                 // elements per 16-byte chunk
  constexpr int PR = Chunk<IOT>::PR;         // column pairs per chunk
  constexpr int NUC = VE / 4;                // 16-byte query chunks per column chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = a.n, S = a.S, d = a.d, H = a.heads;
  const int TT = pl.TT, QG = pl.QG, SG = pl.SG, ST = pl.ST, KC = pl.KC;
  const int64_t T = a.T;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * TT;
  const int head = static_cast<int>(blockIdx.y);
  const int dh = d / H;          // this CTA's columns: cw .. cw + dh - 1
  const int cw = head * dh;
  const int nch = (dh + KC - 1) / KC;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.offBar);
  uint64_t* empty = full + ST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + ST);

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // the prologue above touches no global memory; the successor waits for the exit

  // The ring runs 2 * nch iterations: sweep 1 (sources + queries), then sweep 2 (sources).
  // Thread 0 issues the copies: the first ST iterations up front, then, at every iteration,
  // the refill of the slot used one iteration earlier once all warps have released it.
  const int total = 2 * nch;
  auto issue = [&](int i) {
    const int slot = i % ST;
    const bool first = i < nch;
    const int c = first ? i : i - nch;
    unsigned char* st = smem + slot * pl.stageBytes;
    mbar_arrive_expect_tx(&full[slot], pl.bBytes + (first ? pl.nUBox * pl.uBox : 0));
    tma_load_3d(st, &tm_b, cw + c * KC, static_cast<int>(t0), 0, &full[slot]);
    if (first) {
      for (int h = 0; h < pl.nUBox; ++h)
        tma_load_2d(st + pl.bSpan + h * pl.uSpan, &tm_u, cw + c * KC + 32 * h, 0, &full[slot]);
    }
  };
  int issued = 0;  // meaningful in thread 0 only
  if (tid == 0) {
    tma_prefetch_map(&tm_b);
    tma_prefetch_map(&tm_u);
    issued = ST < total ? ST : total;
    for (int i = 0; i < issued; ++i) issue(i);
  }

  int it = 0;  // ring position, shared by both sweeps
  auto acquire = [&](int slot) {
    if (!*abort_flag && !mbar_wait(&full[slot], (it / ST) & 1)) *abort_flag = 1;
  };
  auto release = [&](int slot) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (warp == 0) {  // the whole warp waits, lane 0 issues
      const int prev = it - 1;
      if (prev >= 0 && prev + ST < total) {
        const int ps = prev % ST;
        if (!*abort_flag && !mbar_wait(&empty[ps], (prev / ST) & 1)) *abort_flag = 1;
        __syncwarp();
        if (lane == 0 && !*abort_flag) {
          issue(prev + ST);
          issued = prev + ST + 1;
        }
      }
    }
  };

  // ---------------- sweep 1: logit numerators and sums of squares ----------------
  const bool active1 = lane < TT * SG * QG;
  const int g = lane % QG;
  const int sg = (lane / QG) % SG;
  const int tl = lane / (QG * SG);
  int boff[NS];
#pragma unroll
  for (int jj = 0; jj < NS; ++jj) boff[jj] = sw128((sg * NS + jj) * TT + tl, warp);
  int uoff[NQ][NUC];
#pragma unroll
  for (int qq = 0; qq < NQ; ++qq) {
    const int q = g * NQ + qq;
#pragma unroll
    for (int h = 0; h < NUC; ++h)  // bf16: chunks 2(w%4), 2(w%4)+1 of box w/4; fp32: chunk w
      uoff[qq][h] = pl.bSpan + (NUC == 2 ? (warp >> 2) * pl.uSpan : 0) +
                    sw128(q, NUC == 2 ? 2 * (warp & 3) + h : warp);
  }

  float2 acc[NS][NQ];
  float2 ss[NS];
#pragma unroll
  for (int jj = 0; jj < NS; ++jj) {
    ss[jj] = make_float2(0.f, 0.f);
#pragma unroll
    for (int qq = 0; qq < NQ; ++qq) acc[jj][qq] = make_float2(0.f, 0.f);
  }

  for (int c = 0; c < nch; ++c, ++it) {
    const int slot = it % ST;
    acquire(slot);
    if (active1 && c * KC + warp * VE < dh) {  // the warp's chunk lies in the head
      const unsigned char* st = smem + slot * pl.stageBytes;
      float2 uv[NQ][PR];
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq) {
        if (g * NQ + qq < S) {  // padded queries of the last group read nothing
#pragma unroll
          for (int h = 0; h < NUC; ++h) {
            const float4 x = *reinterpret_cast<const float4*>(st + uoff[qq][h]);
            uv[qq][2 * h] = make_float2(x.x, x.y);
            uv[qq][2 * h + 1] = make_float2(x.z, x.w);
          }
        } else {
#pragma unroll
          for (int i = 0; i < PR; ++i) uv[qq][i] = make_float2(0.f, 0.f);
        }
      }
#pragma unroll
      for (int jj = 0; jj < NS; ++jj) {
        if (sg * NS + jj < n) {
          float2 bv[PR];
          Chunk<IOT>::load(st + boff[jj], bv);
#pragma unroll
          for (int i = 0; i < PR; ++i) {
            ss[jj] = __ffma2_rn(bv[i], bv[i], ss[jj]);
#pragma unroll
            for (int qq = 0; qq < NQ; ++qq) acc[jj][qq] = __ffma2_rn(uv[qq][i], bv[i], acc[jj][qq]);
          }
        }
      }
    }
    release(slot);
  }

  // ---------------- reduce the 8 warps' partial sums (fixed order) ----------------
  float* red = reinterpret_cast<float*>(smem + pl.offRed);
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
  // 1 / r_j (1 without the key RMSNorm) in place of the sum of squares
  const float fd = static_cast<float>(dh);
  const bool key_norm = (a.flags & kNoKeyNorm) == 0;
  const bool sigmoid = (a.flags & kSigmoid) != 0;
  for (int i = tid; i < TT * n; i += kThreads) {
    float* p = dots + i * S1 + S;
    *p = key_norm ? 1.f / sqrtf(*p / fd + a.eps) : 1.f;
  }
  __syncthreads();

  // ---------------- softmax statistics, one thread per (token, query) ----------------
  // alpha is stored twice, (a, a), so sweep 2 reads ready-made pairs: [TT][n][QG][NQ][2].
  // It reuses the reduction buffer, which is dead once `dots` is complete.
  float* alph = red;
  for (int i = tid; i < TT * S; i += kThreads) {
    const int t = i / S, s = i % S;
    const int64_t tok = t0 + t;
    const int64_t sh = static_cast<int64_t>(s) * H + head;  // row of the [S][H] statistics
    const float* dt = dots + t * n * S1;
    float m = -INFINITY;
    for (int j = 0; j < n; ++j) m = fmaxf(m, dt[j * S1 + s] * dt[j * S1 + S]);
    float l = 0.f;
    if (!sigmoid)
      for (int j = 0; j < n; ++j) l += expf(dt[j * S1 + s] * dt[j * S1 + S] - m);
    const float lse = m + logf(l);
    const float rl = 1.f / l;
    for (int j = 0; j < n; ++j) {
      const float zj = dt[j * S1 + s] * dt[j * S1 + S];
      const float al = sigmoid ? 1.f / (1.f + expf(-zj)) : expf(zj - m) * rl;
      float* ap = alph + (((t * n + j) * QG + s / NQ) * NQ + s % NQ) * 2;
      ap[0] = al;
      ap[1] = al;
      if (a.alpha != nullptr && tok < T) a.alpha[(sh * T + tok) * n + j] = al;
    }
    if (tok < T) {
      if (a.m != nullptr) a.m[sh * T + tok] = m;
      if (a.lse != nullptr && !sigmoid) a.lse[sh * T + tok] = lse;
    }
  }
  __syncthreads();

  // ---------------- sweep 2: o[s,t,:] = sum_j alpha[s,t,j] b_j[t,:] ----------------
  const bool active2 = tid < TT * QG * 8;
  const int kg = tid & 7, g2 = (tid >> 3) % QG, t2 = tid / (8 * QG);
  const int64_t tok2 = t0 + t2;
  const float* at = alph + (t2 * n * QG + g2) * NQ * 2;
  char* o = static_cast<char*>(a.o);
  const bool of32 = (a.flags & kOF32) != 0;  // o stored in fp32 whatever the I/O type
  for (int c = 0; c < nch; ++c, ++it) {
    const int slot = it % ST;
    acquire(slot);
    if (active2) {
      const unsigned char* st = smem + slot * pl.stageBytes;
      float2 acc2[NQ][PR];
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq)
#pragma unroll
        for (int i = 0; i < PR; ++i) acc2[qq][i] = make_float2(0.f, 0.f);
      // The next source's chunk and alpha pairs are read from shared memory while the
      // current source is accumulated (the trip count n is a runtime value).
      float2 bv[PR], bn[PR];
      float4 af[NQ / 2], an[NQ / 2];
      Chunk<IOT>::load(st + sw128(t2, kg), bn);
#pragma unroll
      for (int h = 0; h < NQ / 2; ++h) an[h] = reinterpret_cast<const float4*>(at)[h];
      for (int j = 0; j < n; ++j) {
#pragma unroll
        for (int i = 0; i < PR; ++i) bv[i] = bn[i];
#pragma unroll
        for (int h = 0; h < NQ / 2; ++h) af[h] = an[h];
        if (j + 1 < n) {
          Chunk<IOT>::load(st + sw128((j + 1) * TT + t2, kg), bn);
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
          for (int i = 0; i < PR; ++i) acc2[qq][i] = __ffma2_rn(al[qq], bv[i], acc2[qq][i]);
      }
      const int k = c * KC + kg * VE;  // column in the head
      if (tok2 < T && k < dh) {
#pragma unroll
        for (int qq = 0; qq < NQ; ++qq) {
          const int q = g2 * NQ + qq;
          const int64_t at = (static_cast<int64_t>(q) * T + tok2) * d + cw + k;
          if (q < S) {
            if (of32)
              Chunk<IOT>::store_f32(o + at * 4, acc2[qq]);
            else
              Chunk<IOT>::store(o + at * E, acc2[qq]);
          }
        }
      }
    }
    release(slot);
  }
  // Drain: the last copy issued into every slot has landed before the CTA may exit (only
  // an aborted run can leave one in flight).
  if (tid == 0) {
    for (int s = 0; s < ST && s < issued; ++s) {
      const int last = issued - 1 - ((issued - 1 - s) % ST);
      mbar_wait_drain(&full[s], (last / ST) & 1);
    }
  }
}

// ---------------------------------- host side ----------------------------------
template <typename T, int NS, int NQ>
cudaError_t launch_t(const Phase1Args& a, const P1Plan& pl, cudaStream_t s) {
  CUtensorMap mb, mu;
  cudaError_t e = encode_source_map(&mb, a.reps, a.src_stride, a.n, a.T, a.d, sizeof(T), pl.KC,
                                    pl.TT);
  if (e == cudaSuccess) e = encode_query_map(&mu, a.u, a.S, a.d);
  if (e != cudaSuccess) return e;
  auto kern = phase1_kernel<T, NS, NQ>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (a.T + pl.TT - 1) / pl.TT;
  const dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(a.heads));
  return launch_pdl(kern, grid, kThreads, pl.smem, s, mb, mu, a, pl);
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
    f.flags = a.flags;
    f.heads = a.heads;
    f.h_f32 = io == IO::BF16 && (a.flags & kOF32) != 0;
    return launch_full(io, f, s);
  }
  if (io == IO::BF16 && a.u_split != nullptr && phase1_tc_supported(a.n, a.S, a.d, a.heads))
    return launch_phase1_tc(a, s);
  return io == IO::BF16 ? launch_io<bf16>(a, s) : launch_io<float>(a, s);
}

unsigned int phase1_poll_timeouts() {
  return take_wait_timeouts();
}

}  // namespace attnres
