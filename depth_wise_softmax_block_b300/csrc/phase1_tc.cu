// Phase 1 of the two-phase Block AttnRes schedule with the logits on the tensor cores
// ("Attention Residuals" note, §10 step 1; "Attention Residuals 阅读补充", section
// "静态 Query 与两阶段计算": the S static queries of a block stacked into one matrix turn the
// block's scoring into one product Q K^T over the history).
//
// The logit numerators of all tokens form one dense product: U [S x d] (the block's queries,
// shared by every token) times the source rows b_j[t] [d] of every (source, token) pair.  This
// kernel computes it with tcgen05 MMAs (bf16 x bf16 -> fp32 in tensor memory).  U is fp32; each
// query row is split exactly enough into two bf16 rows, u = hi + lo with |u - hi - lo| <=
// 2^-16 |u|, and both rows enter the product, so the logits keep fp32-level accuracy (the
// sources are bf16 already).  Everything else runs on the CUDA cores:
//   sweep 1  a copy-issuing warp streams 64-column stages of the tile (n sources x 8 tokens,
//            128-byte swizzled rows) through a ring of up to 12 slots, and the same columns of
//            U (fp32) through a ring of 4; the 16 compute warps split U into the hi/lo bf16
//            operand tile and accumulate each source row's sum of squares; thread 0 issues the
//            four K=16 MMAs of the stage, D[row, 2s + {hi,lo}] += b_row . u_s, with the tile's
//            n*8 rows as M (= 128, unused rows ignored);
//   softmax  warps 0-3 read D from tensor memory (one row per thread), form
//            z = (hi + lo) / r_j, and one thread per (token, query) computes m, lse, alpha;
//   sweep 2  the tile streams through the ring again, columns in reverse order so that the
//            chunks read last in sweep 1 are still in L2, and the 16 warps write
//            o[s,t,:] = sum_j alpha_j b_j[t,:] (packed fp32 FMAs, 16-byte streaming stores).
// Stage hand-off uses mbarriers ("full": copy landed; "conv": split queries written; "empty":
// all warps and the stage's MMAs done); every wait is bounded (tma.cuh).  The tensor-memory
// allocation is released on every path before the CTA exits.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tma.cuh"

namespace attnres {
namespace {

constexpr int kCompute = 512;              // 16 compute warps
constexpr int kWarps = kCompute / 32;
constexpr int kThreads = kCompute + 32;    // + 1 copy-issuing warp
constexpr int kTT = 8;              // tokens per CTA tile
constexpr int kKC = 64;             // bf16 columns per stage (one 128-byte row slice)
constexpr int kM = 128;             // MMA rows (tile rows n * 8 <= 128)
constexpr int kMaxS = 24;           // sweep 2 covers 8 groups of 3 queries
constexpr int kMaxN = kM / kTT;     // 16 sources
constexpr int kTmemCols = 64;       // D uses at most 2 * 24 = 48 columns
constexpr int kMaxB = 12;           // source-ring slots
constexpr int kQStages = 4;         // query-ring slots (sweep 1 only)
constexpr int kMaxSmem = 227 * 1024;

struct TcPlan {
  int Npad;           // MMA N: 2S rounded up to 16
  int bBytes;         // source box bytes as copied (n * 8 * 128)
  int bSlot, SB;      // source-ring slot bytes (1024-aligned), slots
  int uBox, uSpan;    // one fp32 query box (S rows x 128 bytes) / rounded up to 1024
  int qSlot;          // query-ring slot: two fp32 boxes + the split operand tile
  int offQ;           // query ring (after the source ring and its MMA read-over slack)
  int offZ, offAlph, offSs, offBar, offTmem;
  int smem;
};

inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

bool make_tc_plan(int n, int S, TcPlan& p) {
  if (n < 1 || n > kMaxN || S < 2 || S > kMaxS) return false;
  p.Npad = align_up(2 * S, 16);
  p.bBytes = n * kTT * 128;
  p.bSlot = align_up(p.bBytes, 1024);
  p.uBox = S * 128;
  p.uSpan = align_up(p.uBox, 1024);
  p.qSlot = 2 * p.uSpan + align_up(p.Npad * 128, 1024);
  // The MMA reads 128 rows (16 KB) from a source slot's base; rows past the tile's n * 8 are
  // ignored but must lie inside the allocation, hence the slack after the last slot.
  const int slack = kM * 128 - p.bSlot;
  const int zb = kM * S * 4;
  const int ab = kTT * n * 8 * 8 * 4;
  const int fixed = slack + kQStages * p.qSlot + align_up(zb, 16) + align_up(ab, 16) + kM * 4 +
                    (2 * kMaxB + 3 * kQStages + 2) * 8 + 16;
  p.SB = std::min(kMaxB, (kMaxSmem - 1024 - fixed) / p.bSlot);
  if (p.SB < 3) return false;
  p.offQ = p.SB * p.bSlot + slack;
  p.offZ = p.offQ + kQStages * p.qSlot;
  p.offAlph = p.offZ + align_up(zb, 16);
  p.offSs = p.offAlph + align_up(ab, 16);
  p.offBar = p.offSs + kM * 4;
  p.offTmem = p.offBar + (2 * p.SB + 3 * kQStages + 2) * 8;
  p.smem = 1024 + p.offTmem + 16;
  return true;
}

__device__ __forceinline__ void unpack_pairs(const uint4& v, float2 (&f)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

__global__ void __launch_bounds__(kThreads, 1)
phase1_tc_kernel(const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_u, const Phase1Args a, const TcPlan pl) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = a.n, S = a.S, d = a.d, SB = pl.SB;
  const int64_t T = a.T;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTT;
  const int nch = (d + kKC - 1) / kKC;
  const int total = 2 * nch;  // source-ring iterations: sweep 1, then sweep 2

  uint64_t* full_b = reinterpret_cast<uint64_t*>(smem + pl.offBar);
  uint64_t* empty_b = full_b + SB;
  uint64_t* full_q = empty_b + SB;
  uint64_t* conv = full_q + kQStages;
  uint64_t* empty_q = conv + kQStages;
  uint64_t* dready = empty_q + kQStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(dready + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + pl.offTmem);
  float* zbuf = reinterpret_cast<float*>(smem + pl.offZ);     // [128 rows][S]
  float* alph = reinterpret_cast<float*>(smem + pl.offAlph);  // [8][n][8 groups][4 pairs][2]
  float* ssbuf = reinterpret_cast<float*>(smem + pl.offSs);   // [128 rows]

  if (tid == 0) {
    for (int s = 0; s < SB; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_b[s], kWarps + 1);  // every compute warp + the stage's MMAs (or thread 0)
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&full_q[s], 1);
      mbar_init(&conv[s], kWarps);         // split queries written
      mbar_init(&empty_q[s], 1);           // the stage's MMAs completed
    }
    mbar_init(dready, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  // Rows [2S, Npad) of every split-query tile stay zero for the whole kernel.
  {
    const int zrows = pl.Npad - 2 * S;
    for (int i = tid; i < kQStages * zrows * 8; i += kThreads) {
      const int s = i / (zrows * 8), rr = 2 * S + (i / 8) % zrows, ch = i % 8;
      *reinterpret_cast<uint4*>(smem + pl.offQ + s * pl.qSlot + 2 * pl.uSpan + sw128(rr, ch)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ------------------------------ copy-issuing warp ------------------------------
  if (warp == kWarps) {
    if (lane == 0) {
      tma_prefetch_map(&tm_b);
      tma_prefetch_map(&tm_u);
      int ib = 0, iq = 0;  // copies issued into each ring
      for (; ib < total; ++ib) {
        if (ib < nch) {  // the stage's query columns first: the MMAs need both
          const int qs = ib % kQStages;
          if (ib >= kQStages && !mbar_wait(&empty_q[qs], ((ib / kQStages) - 1) & 1)) {
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          unsigned char* q = smem + pl.offQ + qs * pl.qSlot;
          mbar_arrive_expect_tx(&full_q[qs], 2 * pl.uBox);
          tma_load_2d(q, &tm_u, ib * kKC, 0, &full_q[qs]);
          tma_load_2d(q + pl.uSpan, &tm_u, ib * kKC + 32, 0, &full_q[qs]);
          iq = ib + 1;
        }
        const int bs = ib % SB;
        if (ib >= SB && !mbar_wait(&empty_b[bs], ((ib / SB) - 1) & 1)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        // sweep 2 walks the columns backwards: the chunks read last come back first, from L2
        const int c = ib < nch ? ib : total - 1 - ib;
        mbar_arrive_expect_tx(&full_b[bs], pl.bBytes);
        tma_load_3d(smem + bs * pl.bSlot, &tm_b, c * kKC, static_cast<int>(t0), 0, &full_b[bs]);
      }
      // Drain: the last copy issued into every slot has landed before the CTA may exit.
      for (int s = 0; s < SB && s < ib; ++s) {
        const int last = ib - 1 - ((ib - 1 - s) % SB);
        mbar_wait(&full_b[s], (last / SB) & 1);
      }
      for (int s = 0; s < kQStages && s < iq; ++s) {
        const int last = iq - 1 - ((iq - 1 - s) % kQStages);
        mbar_wait(&full_q[s], (last / kQStages) & 1);
      }
    }
    return;
  }

  // -------------------------------- compute warps --------------------------------
  const uint32_t tmem = *tmem_slot;
  const uint32_t idesc = idesc_bf16_f32(kM, pl.Npad);
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (!*abort_flag && !mbar_wait(bar, parity)) *abort_flag = 1;
  };
  auto release_b = [&](int bs, bool substitute_mma) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_b[bs]);
    if (substitute_mma && tid == 0) mbar_arrive(&empty_b[bs]);
  };

  // ------------------------------------ sweep 1 ------------------------------------
  const int nrows = n * kTT;  // tile rows: row j * 8 + t
  float2 ssa[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  for (int c = 0; c < nch; ++c) {
    const int bs = c % SB, qs = c % kQStages;
    unsigned char* st = smem + bs * pl.bSlot;
    unsigned char* qb = smem + pl.offQ + qs * pl.qSlot;
    // split the stage's queries: operand rows 2s (hi) and 2s + 1 (lo), bf16, swizzled
    wait(&full_q[qs], (c / kQStages) & 1);
    if (tid < S * 8) {
      const int q = tid >> 3, g8 = tid & 7;
      const unsigned char* ub = qb + (g8 >> 2) * pl.uSpan;
      const float4 x0 = *reinterpret_cast<const float4*>(ub + sw128(q, 2 * (g8 & 3)));
      const float4 x1 = *reinterpret_cast<const float4*>(ub + sw128(q, 2 * (g8 & 3) + 1));
      const float u[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = pack_bf16x2(u[2 * e], u[2 * e + 1]);
        lo[e] = pack_bf16x2(u[2 * e] - __uint_as_float(hi[e] << 16),
                            u[2 * e + 1] - __uint_as_float(hi[e] & 0xffff0000u));
      }
      unsigned char* bt = qb + 2 * pl.uSpan;
      *reinterpret_cast<uint4*>(bt + sw128(2 * q, g8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(bt + sw128(2 * q + 1, g8)) =
          make_uint4(lo[0], lo[1], lo[2], lo[3]);
      fence_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&conv[qs]);
    // sums of squares: (row, 16-byte chunk) pairs tid and tid + 512
    wait(&full_b[bs], (c / SB) & 1);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = tid + k * kCompute;
      if (i < nrows * 8) {
        float2 f[4];
        unpack_pairs(*reinterpret_cast<const uint4*>(st + sw128(i >> 3, i & 7)), f);
#pragma unroll
        for (int e = 0; e < 4; ++e) ssa[k] = __ffma2_rn(f[e], f[e], ssa[k]);
      }
    }
    // the stage's four K = 16 MMAs, issued by thread 0 once the split queries are in place
    if (warp == 0) {
      wait(&conv[qs], (c / kQStages) & 1);
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a0 = smem_addr(st), b0 = smem_addr(qb + 2 * pl.uSpan);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(tmem, desc_kmajor_sw128(a0 + 32 * kk), desc_kmajor_sw128(b0 + 32 * kk),
                      idesc, (c | kk) != 0 ? 1u : 0u);
        tc_commit(&empty_b[bs]);
        tc_commit(&empty_q[qs]);
        if (c == nch - 1) tc_commit(dready);
      }
    }
    release_b(bs, false);
  }

  // row sums of squares: the 8 chunks of a row sit in 8 consecutive lanes
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = tid + k * kCompute;
    float x = ssa[k].x + ssa[k].y;
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    if (i < nrows * 8 && (i & 7) == 0) ssbuf[i >> 3] = x;
  }
  named_barrier(1, kCompute);

  // ------------------------- logits from tensor memory -------------------------------
  const float fd = static_cast<float>(d);
  if (warp < 4) {
    wait(dready, 0);
    tc_fence_after();
    const int r = warp * 32 + lane;
    const float rinv = r < nrows ? 1.f / sqrtf(ssbuf[r] / fd + a.eps) : 0.f;
    for (int cc = 0; cc < pl.Npad / 16; ++cc) {
      uint32_t v[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc * 16, v);
      tmem_ld_wait();
      if (r < nrows) {
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const int s = cc * 8 + e / 2;
          if (s < S) zbuf[r * S + s] = (__uint_as_float(v[e]) + __uint_as_float(v[e + 1])) * rinv;
        }
      }
    }
  }
  named_barrier(1, kCompute);

  // ---------------- softmax statistics, one thread per (token, query) ----------------
  for (int i = tid; i < kTT * S; i += kCompute) {
    const int t = i / S, s = i % S;
    const int64_t tok = t0 + t;
    float m = -INFINITY;
    for (int j = 0; j < n; ++j) m = fmaxf(m, zbuf[(j * kTT + t) * S + s]);
    float l = 0.f;
    for (int j = 0; j < n; ++j) l += expf(zbuf[(j * kTT + t) * S + s] - m);
    const float lse = m + logf(l);
    const float rl = 1.f / l;
    const int g = s / 3, pp = s % 3;
    for (int j = 0; j < n; ++j) {
      const float al = expf(zbuf[(j * kTT + t) * S + s] - m) * rl;
      float* ap = alph + (((t * n + j) * 8 + g) * 4 + pp) * 2;
      ap[0] = al;
      ap[1] = al;
      if (a.alpha != nullptr && tok < T) a.alpha[(static_cast<int64_t>(s) * T + tok) * n + j] = al;
    }
    if (tok < T) {
      if (a.m != nullptr) a.m[static_cast<int64_t>(s) * T + tok] = m;
      if (a.lse != nullptr) a.lse[static_cast<int64_t>(s) * T + tok] = lse;
    }
  }
  named_barrier(1, kCompute);

  // ------------------------------------ sweep 2 ------------------------------------
  // warp w: token w / 2, queries (w % 2) * 12 + [0, 12); lane: group of 3 queries, chunk
  const int t2 = warp >> 1;
  const int grp = (warp & 1) * 4 + (lane >> 3);
  const int kg = lane & 7;
  const int64_t tok2 = t0 + t2;
  const bool active2 = grp * 3 < S;
  const float* at = alph + ((t2 * n) * 8 + grp) * 8;
  char* o = static_cast<char*>(a.o);
  for (int ib = nch; ib < total; ++ib) {
    const int bs = ib % SB;
    const int c = total - 1 - ib;  // columns in reverse
    wait(&full_b[bs], (ib / SB) & 1);
    if (active2) {
      const unsigned char* st = smem + bs * pl.bSlot;
      float2 acc[3][4];
#pragma unroll
      for (int qq = 0; qq < 3; ++qq)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[qq][e] = make_float2(0.f, 0.f);
      for (int j = 0; j < n; ++j) {
        float2 bv[4];
        unpack_pairs(*reinterpret_cast<const uint4*>(st + sw128(j * kTT + t2, kg)), bv);
        const float4 a01 = *reinterpret_cast<const float4*>(at + j * 64);
        const float2 a2 = *reinterpret_cast<const float2*>(at + j * 64 + 4);
        const float2 al[3] = {make_float2(a01.x, a01.y), make_float2(a01.z, a01.w), a2};
#pragma unroll
        for (int qq = 0; qq < 3; ++qq)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[qq][e] = __ffma2_rn(al[qq], bv[e], acc[qq][e]);
      }
      const int k = c * kKC + kg * 8;
      if (tok2 < T && k < d) {
#pragma unroll
        for (int qq = 0; qq < 3; ++qq) {
          const int q = grp * 3 + qq;
          if (q < S)
            __stcs(reinterpret_cast<uint4*>(o + ((static_cast<int64_t>(q) * T + tok2) * d + k) * 2),
                   make_uint4(pack_bf16x2(acc[qq][0].x, acc[qq][0].y),
                              pack_bf16x2(acc[qq][1].x, acc[qq][1].y),
                              pack_bf16x2(acc[qq][2].x, acc[qq][2].y),
                              pack_bf16x2(acc[qq][3].x, acc[qq][3].y)));
        }
      }
    }
    release_b(bs, true);
  }

  // ------------------------------------ teardown ------------------------------------
  tc_fence_before();
  named_barrier(1, kCompute);
  tc_fence_after();
  if (warp == 0) {
    if (lane == 0 && *abort_flag) mbar_wait(dready, 0);  // MMAs of an aborted run may still run
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool phase1_tc_supported(int n, int S) {
  TcPlan p;
  return make_tc_plan(n, S, p);
}

cudaError_t launch_phase1_tc(const Phase1Args& a, cudaStream_t s) {
  TcPlan pl;
  if (!make_tc_plan(a.n, a.S, pl)) return cudaErrorInvalidValue;
  CUtensorMap mb, mu;
  cudaError_t e = encode_source_map(&mb, a.reps, a.src_stride, a.n, a.T, a.d, 2, kKC, kTT);
  if (e == cudaSuccess) e = encode_query_map(&mu, a.u, a.S, a.d);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(phase1_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (a.T + kTT - 1) / kTT;
  phase1_tc_kernel<<<static_cast<unsigned>(blocks), kThreads, pl.smem, s>>>(mb, mu, a, pl);
  return cudaGetLastError();
}

unsigned int phase1_tc_poll_timeouts() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v != 0) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_wait_timeouts, &z, sizeof(z));
  }
  return v;
}

}  // namespace attnres
