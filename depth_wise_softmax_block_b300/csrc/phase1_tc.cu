// Phase 1 of the two-phase Block AttnRes schedule with the logits on the tensor cores
// ("Attention Residuals" note, §10 step 1; "Attention Residuals 阅读补充", section
// "静态 Query 与两阶段计算": the S static queries of a block stacked into one matrix turn the
// block's scoring into one product Q K^T over the history).
//
// The logit numerators of all tokens form one dense product: U [S x d] (the block's queries,
// shared by every token) times the source rows b_j[t] [d] of every (source, token) pair.  This
// kernel computes it with tcgen05 MMAs (bf16 x bf16 -> fp32 in tensor memory).  U is fp32; the
// caller passes it also as split bf16 rows (attnres_query_prep): row 2s = hi(u_s), row 2s + 1 =
// lo(u_s), with |u - hi - lo| <= 2^-16 |u|, so the logits keep fp32-level accuracy (the sources
// are bf16 already).
//   sweep 1  a copy-issuing warp streams 64-column stages of the tile (n sources x 8 tokens,
//            128-byte swizzled rows) and of the split queries through a ring of up to 12 slots
//            (an even number); an MMA-issuing warp issues the stage's four K=16 MMAs,
//            D[row, 2s + {hi,lo}] += b_row . u_s, with the tile's n*8 rows as M (= 128, unused
//            rows ignored), while the 16 compute warps, in two halves that take alternate
//            stages, accumulate each source row's sum of squares;
//   softmax  warps 0-3 read D from tensor memory (one row per thread), form
//            z = (hi + lo) / r_j, and one thread per (token, query) computes m, lse, alpha;
//   sweep 2  the tile streams again, columns in reverse order so that the chunks read last in
//            sweep 1 are still in L2, and o[s,t,:] = sum_j alpha_j b_j[t,:] is formed
//            - with one head and 3 to 9 sources, on the tensor cores: per 128-column stage
//              D[column][s*8 + t] = sum over (j, t') of b[j,t'][column] W[(j,t'), (s,t)], W
//              zero off the token diagonal and alpha on it (bf16 hi and lo halves, two MMAs per
//              K step), through a ring of its own; the compute warps read D in the fragment
//              layout, write it transposed to shared memory (stmatrix, 128-byte swizzle) and
//              store it with tensor stores of [6 queries][8 tokens][64 columns] tiles;
//            - otherwise on the CUDA cores: the two halves of the compute warps take alternate
//              stages of the ring (one half's loads and stores overlap the other half's
//              arithmetic), packed fp32 FMAs and 16-byte streaming stores.
// Depth-attention heads (the multi-head variant of Table 4, "Attention Residuals" note,
// result 4): head k owns the contiguous columns k*dh .. k*dh + dh - 1 (dh = d / H, a multiple of
// 64 so that every stage lies in one head).  A CTA covers a window of Hs whole heads (grid.y
// walks the windows): the MMAs of a head accumulate into its own block of tensor-memory columns,
// the sums of squares, logits and softmax statistics are kept per head, and sweep 2 weights a
// stage with its head's alpha.  Hs is the largest divisor of H whose columns fit the 512
// tensor-memory columns (H = 1: one window, the whole row).
// Few token tiles (decode-sized T, one head, n <= 16): a cluster of 2 or 4 CTAs along grid.y
// splits each tile's columns; after sweep 1 the CTAs add their partial logit numerators and sums
// of squares through distributed shared memory (xready / xdone mbarriers), then each runs the
// softmax and sweep 2 on its own columns (rank 0 alone writes the statistics).
// Stage hand-off uses mbarriers ("full": copy landed; "empty": all compute warps and the
// stage's MMAs done; on the tensor-core sweep 2 also "dfull" / "dempty" for its two tensor-memory
// accumulators); every wait is bounded (tma.cuh).  The tensor-memory allocation is released on
// every path before the CTA exits.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tma.cuh"

namespace attnres {
namespace {

constexpr int kCompute = 512;              // 16 compute warps
constexpr int kWarps = kCompute / 32;
constexpr int kThreads = kCompute + 64;    // + a copy-issuing warp and an MMA-issuing warp
constexpr int kTT = 8;              // tokens per CTA tile
constexpr int kKC = 64;             // bf16 columns per stage (one 128-byte row slice)
constexpr int kM = 128;             // rows per MMA (M-tile); a tile has n * 8 rows
constexpr int kMaxS = 24;           // sweep 2 covers 4 groups of 6 queries
constexpr int kMaxN = 64;           // sources (up to 4 M-tiles)
constexpr int kSmallN = 9;          // up to here the sweep-2 weights are stored as ready pairs
constexpr int kTmemMax = 512;       // tensor-memory columns of an SM
constexpr int kMaxSlots = 12;       // ring slots
constexpr int kMaxSmem = 227 * 1024;
constexpr int kTc2Col0 = 128;       // first tensor-memory column of the sweep-2 accumulators
// The tensor-core weighted sum writes o at about the same cost whatever n is; with one or two
// sources the CUDA-core sum is cheaper (16384 tokens, S = 24, CUDA cores against tensor cores:
// 1.37 / 1.46 ms at n = 1, 1.43 / 1.46 at n = 2, 1.46 / 1.44 at n = 3, 1.74 / 1.54 at n = 6,
// 2.02 / 1.60 at n = 9).
constexpr int kTc2MinN = 3;
constexpr int kGrpQ = 6;                          // sweep 2: queries per group of 4 warps
// A group's staged o tile: two halves [6 queries][8 tokens][64 columns] bf16 with the 128-byte
// swizzle, each 1024-byte aligned (6 KB)
constexpr int kStgHalf = kGrpQ * kTT * 64 * 2;

struct TcPlan {
  int Hs, windows;    // heads per CTA window, windows (= H / Hs, or csplit)
  int csplit;         // > 1: a cluster of csplit CTAs splits one head's columns (few tiles)
  int tcols;          // tensor-memory columns allocated: nMT * Hs * Npad rounded up to 2^k >= 32
  int R;              // rows of a per-head sum-of-squares buffer (nMT * 128)
  int Npad;           // MMA N: 2S rounded up to 16
  int rows, nMT;      // tile rows (n * 8) and M-tiles (ceil(rows / 128))
  int bBytes;         // source box bytes as copied (rows * 128)
  int bSpan;          // rounded up to 1024
  int qBytes;         // split-query box bytes (Npad rows x 128 bytes, rows >= 2S zero-filled)
  int qOff;           // offset of the split-query box in a slot
  int slot, SB;       // ring slot bytes ([sources][split queries]), slots (even: see below)
  // sweep 2 on the tensor cores (tc2) has a ring of its own over the same memory: SB2 slots of
  // two 64-column source boxes `region` bytes apart (rows padded to a multiple of 16 with
  // zeros), then the weights as the MMA's B operand, [Nb / 8 row groups][KC chunks of 8 rows]
  // core matrices, once as hi and once as lo halves
  int tc2, region, KC, Nb, abBytes, slot2, SB2;
  int offAB, offZ, offAlph, offSs, offBar, offTmem;
  int smem;
};

inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Layout for n sources, S queries and a window of Hs heads, with sweep 2 on the tensor cores
// (tc2: one head, n <= 9) or on the CUDA cores; false if it does not fit.
bool make_tc_window(int n, int S, int H, int Hs, bool tc2, TcPlan& p) {
  p.Hs = Hs;
  p.windows = H / Hs;
  p.csplit = 1;
  p.tc2 = tc2 ? 1 : 0;
  p.Npad = align_up(2 * S, 16);
  p.rows = n * kTT;
  p.nMT = (p.rows + kM - 1) / kM;
  p.R = p.nMT * kM;
  int cols = p.nMT * Hs * p.Npad;
  if (tc2) {
    if (H != 1 || n > kSmallN || cols > kTc2Col0) return false;
    p.Nb = align_up(kTT * S, 16);            // sweep-2 MMA N: (query, token) pairs
    p.KC = align_up(p.rows, 16) / 8;         // sweep-2 K chunks: (source, token) rows / 8
    cols = kTc2Col0 + 2 * p.Nb;              // two accumulators, alternate 128-column stages
  }
  if (cols > kTmemMax) return false;
  for (p.tcols = 32; p.tcols < cols; p.tcols *= 2) {
  }
  p.bBytes = p.rows * 128;
  p.qBytes = p.Npad * 128;
  p.bSpan = align_up(p.bBytes, 1024);
  p.qOff = p.bSpan;
  p.slot = p.bSpan + align_up(p.qBytes, 1024);
  // The MMAs read nMT * 128 rows from a slot's base; rows past the tile's n * 8 are ignored but
  // must lie inside the allocation, hence the slack after the last slot.
  const int slack = std::max(0, p.nMT * kM * 128 - p.slot);
  // logits [rows][Hs][SZ] (SZ = S rounded up to even, for 8-byte loads), then (unless the
  // small layout) the weights in their place; 8 floats of padding for the last query group's
  // 6-wide read
  const int zb = (p.rows * Hs * ((S + 1) & ~1) + 8) * 4;
  const bool small = H == 1 && n <= kSmallN && !tc2;
  const int ab = small ? kTT * n * 4 * 12 * 4 : 0;  // [token][source][4][6 pairs][2]
  const int sb = 2 * Hs * p.R * 4;                  // per-half, per-head row sums of squares
  // tc2: sweep 2 stages its output tiles where the logits and sums of squares were (dead by then)
  const int zone = std::max(align_up(zb, 16) + align_up(ab, 16) + sb,
                            tc2 ? 4 * 2 * kStgHalf : 0);
  const int avail = kMaxSmem - 1024 - zone - (4 * kMaxSlots + 10) * 8 - 16;
  // The two halves of the compute warps take alternate stages of the sweep-1 ring, each
  // waiting on the "full" barriers of its own stages only.  With an odd number of slots
  // consecutive users of a slot belong to different halves, and a half running a ring ahead
  // could see the completion two phases back (same parity) as its own stage's: the slot count
  // is even, so a slot's successive stages always belong to the same half.
  if (tc2) {
    p.region = p.KC * 8 * 128;  // a multiple of 2048: both boxes stay 1024-byte aligned
    p.slot2 = 2 * p.region;
    p.abBytes = (p.Nb / 8) * p.KC * 128;
    p.SB2 = std::min(kMaxSlots, (avail - 2 * p.abBytes) / p.slot2);  // one in-order consumer
    if (p.SB2 < 2) return false;
    p.offAB = p.SB2 * p.slot2;
    p.offZ = p.offAB + 2 * p.abBytes;  // the sweep-1 ring spans [0, offZ): both rings, weights
    p.SB = std::min(kMaxSlots, (p.offZ - slack) / p.slot) & ~1;
  } else {
    p.region = p.KC = p.Nb = p.abBytes = p.slot2 = p.SB2 = 0;
    p.SB = std::min(kMaxSlots, (avail - slack) / p.slot) & ~1;
    p.offAB = p.SB * p.slot + slack;
    p.offZ = p.offAB;
  }
  if (p.SB < 2) return false;
  p.offAlph = p.offZ + align_up(zb, 16);
  p.offSs = p.offAlph + align_up(ab, 16);
  p.offBar = p.offZ + zone;
  // full[SB], empty[SB], dready, abort, xready, xdone, dfull[2], dempty[2], aready, mdone,
  // full2[SB2], empty2[SB2]
  p.offTmem = p.offBar + (2 * p.SB + 10 + 2 * p.SB2) * 8;
  p.smem = 1024 + p.offTmem + 16;
  return true;
}

// The widest window (most heads per CTA) that fits; false if none does.
bool make_tc_plan(int n, int S, int d, int H, bool tc2, TcPlan& p) {
  if (n < 1 || n > kMaxN || S < 2 || S > kMaxS || H < 1 || d % H != 0) return false;
  if (H > 1 && (d / H) % kKC != 0) return false;
  for (int Hs = H; Hs >= 1; --Hs)
    if (H % Hs == 0 && make_tc_window(n, S, H, Hs, tc2, p)) return true;
  return false;
}

__device__ __forceinline__ void unpack_pairs(const uint4& v, float2 (&f)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

// Slot and phase parity of ring position `it` (it % SB, (it / SB) & 1), advanced without
// divisions (a step of at most SB positions).
struct RingPos {
  int bs, ph;
  __device__ __forceinline__ RingPos(int it, int SB) : bs(it % SB), ph((it / SB) & 1) {}
  __device__ __forceinline__ void advance(int step, int SB) {
    bs += step;
    if (bs >= SB) {
      bs -= SB;
      ph ^= 1;
    }
  }
};

// kN = n in 1 .. 9 with one head: the small layout (one M-tile, sweep-2 weights as ready-made
// pairs, sums of squares in registers) with the source count known at compile time, so every
// loop over the sources is unrolled without guards; kN = 0: any n (runtime).  kSplit: the
// cluster column split for few token tiles (compiled out of the other instantiations).  kTc:
// sweep 2 on the tensor cores (one head, kN >= kTc2MinN, no split).
template <int kN, bool kSplit, bool kTc>
__global__ void __launch_bounds__(kThreads, 1)
phase1_tc_kernel(const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_o, const Phase1Args a, const TcPlan pl) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr bool kSmall = kN > 0;
  constexpr bool kTc2 = kTc;
  static_assert(!kTc || (kN >= kTc2MinN && !kSplit), "tensor-core sweep 2: 3 to 9 sources");
  const int n = kSmall ? kN : a.n;
  const int S = a.S, d = a.d, SB = pl.SB, SB2 = pl.SB2;
  const int H = a.heads, Hs = pl.Hs, R = pl.R;
  const int64_t T = a.T;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTT;
  const int dh = d / H;                       // columns per head
  const int W = kSplit ? pl.csplit : 1;       // > 1: the cluster's CTAs split the columns
  const int wcols = W > 1 ? dh / W : Hs * dh;  // columns of this CTA's window
  const int cw = static_cast<int>(blockIdx.y) * wcols;  // its first column
  const int h0 = W > 1 ? 0 : static_cast<int>(blockIdx.y) * Hs;  // its first head
  const int cph = (W > 1 ? wcols : dh) / kKC + ((W > 1 ? wcols : dh) % kKC != 0);  // stages per head
  const bool writer = W == 1 || blockIdx.y == 0;  // writes the statistics of the tile
  const int nch = (wcols + kKC - 1) / kKC;
  const int nch2 = kTc2 ? (wcols + 2 * kKC - 1) / (2 * kKC) : nch;  // sweep-2 stages
  const int total = nch + nch2;  // source-ring iterations: sweep 1, then sweep 2

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.offBar);
  uint64_t* empty = full + SB;
  uint64_t* dready = empty + SB;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(dready + 1);
  uint64_t* xready = dready + 2;  // split: the peers' partial sums are ready to be read
  uint64_t* xdone = dready + 3;   // split: the peers have read this CTA's partial sums
  uint64_t* dfull = dready + 4;   // tc2: accumulator b holds a finished stage
  uint64_t* dempty = dready + 6;  // tc2: every compute warp has read accumulator b
  uint64_t* aready = dready + 8;  // tc2: the weights are in place as the B operand
  uint64_t* mdone = dready + 9;   // tc2: every MMA has completed
  uint64_t* full2 = dready + 10;  // tc2: the sweep-2 ring's barriers
  uint64_t* empty2 = full2 + SB2;
  unsigned char* abuf = smem + pl.offAB;  // tc2: weights, hi halves then lo halves
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + pl.offTmem);
  float* zbuf = reinterpret_cast<float*>(smem + pl.offZ);     // [n * 8 rows][Hs][SZ]
  const int SZ = (S + 1) & ~1;
  const int ZR = Hs * SZ;                                      // zbuf row stride
  float* alph = reinterpret_cast<float*>(smem + pl.offAlph);  // small: [8][n][4][6 pairs][2]
  float* ssbuf = reinterpret_cast<float*>(smem + pl.offSs);   // [2 halves][Hs][R rows]

  if (tid == 0) {
    for (int s = 0; s < SB; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps / 2 + 1);  // the consuming half + the stage's MMAs (or a stand-in)
    }
    mbar_init(dready, 1);
    if (W > 1) {
      mbar_init(xready, W - 1);
      mbar_init(xdone, W - 1);
    }
    if (kTc2) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&dfull[b], 1);
        mbar_init(&dempty[b], kWarps);
      }
      mbar_init(aready, kWarps);
      mbar_init(mdone, 1);
      for (int s = 0; s < SB2; ++s) {
        mbar_init(&full2[s], 1);
        mbar_init(&empty2[s], 1);  // the stage's MMAs
      }
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (kTc2) {
    // Zeros in the rows that pad each sweep-2 box to a multiple of 16 (the weights there are
    // zero too, but a stale non-finite value times zero would not be).  Sweep 1's copies may
    // overwrite some of them with source rows, which are finite as well.  Made visible to the
    // async proxy before the barrier below.
    const int pad16 = (pl.region - pl.bBytes) / 16;  // 16-byte words of padding per box
    if (pad16 > 0)
      for (int i = tid; i < SB2 * 2 * pad16; i += kThreads) {
        const int box = i / pad16, k = i - box * pad16;
        *reinterpret_cast<uint4*>(smem + (box >> 1) * pl.slot2 + (box & 1) * pl.region +
                                  pl.bBytes + k * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    fence_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, pl.tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (W > 1) cluster_sync();  // the peers' barriers are initialised before any remote arrival
  pdl_wait();  // the prologue above touches no global memory; the successor waits for the exit

  // ------------------------------ copy-issuing warp ------------------------------
  if (warp == kWarps) {
    if (lane == 0) {
      tma_prefetch_map(&tm_b);
      tma_prefetch_map(&tm_q);
      const int n1 = kTc2 ? nch : total;  // iterations of the first ring
      int ib = 0;  // ring iterations issued
      for (RingPos rp(0, SB); ib < n1; ++ib, rp.advance(1, SB)) {
        const int bs = rp.bs;
        if (ib >= SB && !mbar_wait(&empty[bs], rp.ph ^ 1)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        // sweep 2 walks the columns backwards: the chunks read last come back first, from L2
        const bool first = ib < nch;
        unsigned char* st = smem + bs * pl.slot;
        if (first) {
          mbar_arrive_expect_tx(&full[bs], pl.bBytes + pl.qBytes);
          tma_load_3d(st, &tm_b, cw + ib * kKC, static_cast<int>(t0), 0, &full[bs]);
          tma_load_2d(st + pl.qOff, &tm_q, cw + ib * kKC, 0, &full[bs]);
        } else {
          const int c = total - 1 - ib;
          mbar_arrive_expect_tx(&full[bs], pl.bBytes);
          tma_load_3d(st, &tm_b, cw + c * kKC, static_cast<int>(t0), 0, &full[bs]);
        }
      }
      // Drain: the last copy issued into every slot has landed before the CTA may exit.
      for (int s = 0; s < SB && s < ib; ++s) {
        const int last = ib - 1 - ((ib - 1 - s) % SB);
        mbar_wait_drain(&full[s], (last / SB) & 1);
      }
      if (kTc2 && !*abort_flag) {
        // Sweep 2's ring reuses the first ring's memory: every sweep-1 stage is consumed first.
        for (int s = 0; s < SB && s < nch; ++s) {
          const int last = nch - 1 - ((nch - 1 - s) % SB);
          if (!*abort_flag && !mbar_wait(&empty[s], (last / SB) & 1)) *abort_flag = 1;
        }
        // 128-column stages, columns in reverse (the chunks read last in sweep 1 come back
        // first, from L2): two boxes, the second only if it starts in the row.
        int q = 0;
        for (RingPos r2(0, SB2); q < nch2 && !*abort_flag; ++q, r2.advance(1, SB2)) {
          if (q >= SB2 && !mbar_wait(&empty2[r2.bs], r2.ph ^ 1)) {
            *abort_flag = 1;
            break;
          }
          unsigned char* st = smem + r2.bs * pl.slot2;
          const int c2 = (nch2 - 1 - q) * 2 * kKC;
          const bool second = c2 + kKC < wcols;
          mbar_arrive_expect_tx(&full2[r2.bs], pl.bBytes * (second ? 2 : 1));
          tma_load_3d(st, &tm_b, cw + c2, static_cast<int>(t0), 0, &full2[r2.bs]);
          if (second)
            tma_load_3d(st + pl.region, &tm_b, cw + c2 + kKC, static_cast<int>(t0), 0,
                        &full2[r2.bs]);
        }
        for (int s = 0; s < SB2 && s < q; ++s) {
          const int last = q - 1 - ((q - 1 - s) % SB2);
          mbar_wait_drain(&full2[s], (last / SB2) & 1);
        }
      }
    }
    return;
  }

  // ------------------------------- MMA-issuing warp -------------------------------
  // The stage's K = 16 MMAs (four per M-tile), D[row, 2s + {hi, lo}] += b_row . u_s into the
  // columns of the stage's head, as soon as its copies land; completion arrives on the stage's "empty" barrier (and, after the last stage, on
  // "dready").  An MMA costs about the same for every N up to 128, so issuing from a warp of
  // its own keeps the tensor core off the compute warps' critical path.
  if (warp == kWarps + 1) {
    const uint32_t tmem = *tmem_slot;
    const uint32_t idesc = idesc_bf16_f32(kM, pl.Npad);
    int hs = 0, ch = 0;  // head in the window and stage in the head of stage c
    RingPos rp(0, SB);
    for (int c = 0; c < nch; ++c, rp.advance(1, SB)) {
      const int bs = rp.bs;
      if (!*abort_flag && !mbar_wait(&full[bs], rp.ph)) *abort_flag = 1;
      tc_fence_after();
      if (lane == 0) {
        const unsigned char* st = smem + bs * pl.slot;
        const uint32_t b0 = smem_addr(st + pl.qOff);
        for (int mt = 0; mt < (kSmall ? 1 : pl.nMT); ++mt) {  // M-tile mt: rows mt * 128 ..
          const uint32_t a0 = smem_addr(st + mt * kM * 128);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(tmem + (mt * Hs + hs) * pl.Npad, desc_kmajor_sw128(a0 + 32 * kk),
                        desc_kmajor_sw128(b0 + 32 * kk), idesc, (ch | kk) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[bs]);
        if (c == nch - 1) tc_commit(dready);
      }
      __syncwarp();
      if (++ch == cph) {
        ch = 0;
        ++hs;
      }
    }
    if constexpr (kTc2) {
      // Sweep 2: o^T of a 128-column stage, D[column][query * 8 + token] =
      // sum over (source, token') of b[source, token'][column] * w[(query, token), (source,
      // token')], with w zero unless token' = token (alpha on the diagonal of every 8 x 8 core
      // matrix), once with the weights' bf16 hi halves and once with their lo halves.  A is the
      // stage's two boxes as copied (MN-major); the accumulators alternate between two blocks
      // of tensor-memory columns.
      const uint32_t idesc2 = idesc_bf16_f32_amn(kM, pl.Nb);
      const uint32_t ab0 = smem_addr(abuf);
      if (!*abort_flag && !mbar_wait(aready, 0)) *abort_flag = 1;
      tc_fence_after();
      RingPos r2(0, SB2);
      for (int q = 0; q < nch2; ++q, r2.advance(1, SB2)) {
        const int bs = r2.bs, b = q & 1, use = q >> 1;
        if (!*abort_flag && !mbar_wait(&full2[bs], r2.ph)) *abort_flag = 1;
        if (use > 0 && !*abort_flag && !mbar_wait(&dempty[b], (use - 1) & 1)) *abort_flag = 1;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_addr(smem + bs * pl.slot2);
          const uint32_t dcol = tmem + kTc2Col0 + b * pl.Nb;
          for (int kk = 0; kk < pl.KC / 2; ++kk)
#pragma unroll
            for (int hl = 0; hl < 2; ++hl)
              tc_mma_bf16(dcol, desc_mnmajor_sw128(a0 + 2048 * kk, pl.region),
                          desc_kmajor_plain(ab0 + hl * pl.abBytes + 256 * kk, 128, pl.KC * 128),
                          idesc2, (kk | hl) != 0 ? 1u : 0u);
          tc_commit(&empty2[bs]);  // the slot may be refilled
          tc_commit(&dfull[b]);
        }
        __syncwarp();
      }
      if (lane == 0) tc_commit(mdone);
    }
    return;
  }

  // -------------------------------- compute warps --------------------------------
  const uint32_t tmem = *tmem_slot;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (!*abort_flag && !mbar_wait(bar, parity)) *abort_flag = 1;
  };
  // Stage `it` of the ring is consumed by half (it & 1) of the compute warps: warps 0-7 take the
  // even stages, warps 8-15 the odd ones, so the two halves work on different stages at once.
  const int half = warp >> 3, hw = warp & 7, ht = tid & 255;
  auto release = [&](int bs, bool substitute_mma) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[bs]);
    if (substitute_mma && ht == 0) mbar_arrive(&empty[bs]);
  };

  // ------------------------------------ sweep 1 ------------------------------------
  const int nrows = n * kTT;  // tile rows: row j * 8 + t
  const bool key_norm = (a.flags & kNoKeyNorm) == 0;
  const bool sigmoid = (a.flags & kSigmoid) != 0;
  // sums of squares: the half's thread ht takes the (row, 16-byte chunk) pairs ht + 256 k, and
  // each half sums its stages into its own per-head row buffer.  Up to 4 pairs per thread
  // (n <= 16) the sums stay in registers until the half's last stage of the head; beyond that
  // the 8 chunks of a row (8 consecutive lanes) are summed with shuffles every stage and added
  // to the buffer (one owner per row within a half: no race).
  const int ntask = (nrows * 8 + 255) / 256;
  const bool reg_ss = kSmall || ntask <= 4;
  float* ssh = ssbuf + half * (Hs * R);
  for (int i = tid; i < 2 * Hs * R; i += kCompute) ssbuf[i] = 0.f;
  named_barrier(1, kCompute);
  float2 ssa[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                   make_float2(0.f, 0.f)};
  auto flush = [&](int hs) {  // register sums of head hs into the half's buffer
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = ht + k * 256;
      float x = ssa[k].x + ssa[k].y;
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      if (i < nrows * 8 && (i & 7) == 0) ssh[hs * R + (i >> 3)] += x;
      ssa[k] = make_float2(0.f, 0.f);
    }
  };
  int cur = -1;          // head whose sums the registers hold
  int hs = 0, hend = cph;  // head of stage c and the first stage past it
  RingPos rp1(half, SB);
  for (int c = half; c < nch; c += 2, rp1.advance(2, SB)) {
    const int bs = rp1.bs;
    const unsigned char* st = smem + bs * pl.slot;
    while (c >= hend) {
      ++hs;
      hend += cph;
    }
    wait(&full[bs], rp1.ph);
    if (key_norm && reg_ss) {
      if (hs != cur) {
        if (cur >= 0) flush(cur);
        cur = hs;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = ht + k * 256;
        if (i < nrows * 8) {
          float2 f[4];
          unpack_pairs(*reinterpret_cast<const uint4*>(st + sw128(i >> 3, i & 7)), f);
#pragma unroll
          for (int e = 0; e < 4; ++e) ssa[k] = __ffma2_rn(f[e], f[e], ssa[k]);
        }
      }
    } else if (!kSmall && key_norm) {
      for (int k = 0; k < ntask; ++k) {
        const int i = ht + k * 256;
        float x = 0.f;
        if (i < nrows * 8) {
          float2 f[4];
          unpack_pairs(*reinterpret_cast<const uint4*>(st + sw128(i >> 3, i & 7)), f);
          float2 sq = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 4; ++e) sq = __ffma2_rn(f[e], f[e], sq);
          x = sq.x + sq.y;
        }
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        if (i < nrows * 8 && (i & 7) == 0) ssh[hs * R + (i >> 3)] += x;
      }
    }
    release(bs, false);
  }
  if (key_norm && reg_ss && cur >= 0) flush(cur);
  named_barrier(1, kCompute);

  // ------------------------- logits from tensor memory -------------------------------
  const float fd = static_cast<float>(dh);
  if (warp < 4 * pl.nMT) {  // warp w reads TMEM lanes 32 (w % 4) .. of M-tile w / 4
    wait(dready, 0);
    tc_fence_after();
    const int mt = warp >> 2, sub = warp & 3;
    const int r = mt * kM + sub * 32 + lane;
    for (int hs = 0; hs < Hs; ++hs) {
      const float ss = r < nrows ? ssbuf[hs * R + r] + ssbuf[(Hs + hs) * R + r] : 0.f;
      // split: raw dot products here; scaled once the cluster's sums are known
      const float rinv =
          r >= nrows ? 0.f : (key_norm && W == 1) ? 1.f / sqrtf(ss / fd + a.eps) : 1.f;
      for (int cc = 0; cc < pl.Npad / 16; ++cc) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(sub * 32) << 16) + (mt * Hs + hs) * pl.Npad +
                      cc * 16,
                  v);
        tmem_ld_wait();
        if (r < nrows) {
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const int s = cc * 8 + e / 2;
            if (s < S)
              zbuf[r * ZR + hs * SZ + s] =
                  (__uint_as_float(v[e]) + __uint_as_float(v[e + 1])) * rinv;
          }
        }
      }
    }
  }
  named_barrier(1, kCompute);

  // ---------- split: sum the logit numerators and sums of squares over the cluster ----------
  if (W > 1) {
    const uint32_t rank = cluster_rank();
    if (tid == 0)
      for (int q = 0; q < W; ++q)
        if (q != static_cast<int>(rank)) mbar_arrive_cluster(mapa_shared(smem_addr(xready), q));
    if (!*abort_flag && !mbar_wait_cluster(xready, 0)) *abort_flag = 1;
    // entry i: logit numerator (row i / S, query i % S), then the row sums of squares
    const int ne = nrows * S + nrows;
    constexpr int kMaxE = (kM * (kMaxS + 1) + kCompute - 1) / kCompute;  // split: n * 8 <= 128
    float acc[kMaxE];
    auto entry = [&](int i) -> float* {
      return i < nrows * S ? zbuf + (i / S) * ZR + i % S : ssbuf + (i - nrows * S);
    };
#pragma unroll
    for (int k = 0; k < kMaxE; ++k) {
      const int i = tid + k * kCompute;
      acc[k] = 0.f;
      if (i < ne) {
        float* e = entry(i);
        const bool ssrow = i >= nrows * S;
        for (int q = 0; q < W; ++q) {
          if (q == static_cast<int>(rank)) {
            acc[k] += e[0] + (ssrow ? e[R] : 0.f);
          } else {
            const uint32_t ra = mapa_shared(smem_addr(e), q);
            acc[k] += ld_cluster_f32(ra) + (ssrow ? ld_cluster_f32(ra + R * 4) : 0.f);
          }
        }
      }
    }
    named_barrier(1, kCompute);  // every read of the peers is done
    if (tid == 0)
      for (int q = 0; q < W; ++q)
        if (q != static_cast<int>(rank)) mbar_arrive_cluster(mapa_shared(smem_addr(xdone), q));
    if (!*abort_flag && !mbar_wait_cluster(xdone, 0)) *abort_flag = 1;  // mine are read
#pragma unroll
    for (int k = 0; k < kMaxE; ++k) {
      const int i = tid + k * kCompute;
      if (i < ne) {
        float* e = entry(i);
        e[0] = acc[k];
        if (i >= nrows * S) e[R] = 0.f;
      }
    }
    named_barrier(1, kCompute);
    // z = numerator / r with the row's full sum of squares
    for (int i = tid; i < nrows * S; i += kCompute) {
      const int r = i / S;
      if (key_norm) zbuf[r * ZR + i % S] *= 1.f / sqrtf(ssbuf[r] / fd + a.eps);
    }
    named_barrier(1, kCompute);
  }

  if (kTc2) {
    // The weight operand lies in the sweep-1 ring's memory, free now (every sweep-1 copy has
    // been consumed and every sweep-1 MMA has completed): zero it, then the softmax below
    // writes the diagonals.
    for (int i = tid; i < 2 * pl.abBytes / 16; i += kCompute)
      *reinterpret_cast<uint4*>(abuf + i * 16) = make_uint4(0u, 0u, 0u, 0u);
    named_barrier(1, kCompute);
  }

  // ------------- softmax statistics, one thread per (token, head, query) -------------
  for (int i = tid; i < kTT * Hs * S; i += kCompute) {
    const int t = i / (Hs * S), hs = (i / S) % Hs, s = i % S;
    const int64_t tok = t0 + t;
    const int64_t sh = static_cast<int64_t>(s) * H + h0 + hs;  // row of the [S][H] statistics
    const float* zc = zbuf + t * ZR + hs * SZ + s;             // source j at zc + j * 8 * ZR
    float m = -INFINITY;
    for (int j = 0; j < n; ++j) m = fmaxf(m, zc[j * kTT * ZR]);
    float l = 0.f;
    if (!sigmoid)
      for (int j = 0; j < n; ++j) l += expf(zc[j * kTT * ZR] - m);
    const float lse = m + logf(l);
    const float rl = 1.f / l;
    const int g = s / 6, pp = s % 6;
    for (int j = 0; j < n; ++j) {
      float* zp = zbuf + (j * kTT + t) * ZR + hs * SZ + s;
      const float zj = *zp;
      const float al = sigmoid ? 1.f / (1.f + expf(-zj)) : expf(zj - m) * rl;
      if (kTc2) {  // diagonal entry (t, t) of core matrix (query s, source j), hi and lo halves
        const __nv_bfloat16 hi = __float2bfloat16_rn(al);
        const __nv_bfloat16 lo = __float2bfloat16_rn(al - __bfloat162float(hi));
        const int off = (s * pl.KC + j) * 128 + t * 18;
        *reinterpret_cast<__nv_bfloat16*>(abuf + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(abuf + pl.abBytes + off) = lo;
      } else if (kSmall) {  // ready-made (a, a) pairs
        float* ap = alph + (((t * n + j) * 4 + g) * 6 + pp) * 2;
        ap[0] = al;
        ap[1] = al;
      } else {             // in place of the logit, which this thread alone reads
        *zp = al;
      }
      if (a.alpha != nullptr && tok < T && writer) a.alpha[(sh * T + tok) * n + j] = al;
    }
    if (tok < T && writer) {
      if (a.m != nullptr) a.m[sh * T + tok] = m;
      if (a.lse != nullptr && !sigmoid) a.lse[sh * T + tok] = lse;
    }
  }
  if (kTc2) {  // the weights, written through the generic proxy, go to the tensor core
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(aready);
  }
  named_barrier(1, kCompute);

  // ------------------------------------ sweep 2 ------------------------------------
  if constexpr (kTc2) {
    // The MMA warp leaves o^T of 128 columns in accumulator b = stage & 1: tensor-memory lane
    // = column, column query * 8 + token.  Warp w reads lanes 32 (w % 4) .. + 31 (its columns)
    // of the queries s = 6 (w / 4) .. 6 (w / 4) + 5 and frees the accumulator.  bf16 o: each
    // 16-lane x 8-token block comes in the accumulator-fragment layout (16x256b loads), is packed
    // to bf16 and written transposed (stmatrix) into the group's [6 queries][8 tokens][128
    // columns] tile, as two 64-column halves with the 128-byte swizzle (16-byte chunk c of row r
    // at c ^ (r % 8): conflict-free); after a group barrier one thread writes the halves out with
    // two tensor stores (rows past T, columns past d and queries past S clipped).  fp32 o: 32x32b
    // loads (lane = column) and direct stores, 128-byte row pieces.
    const int quarter = warp & 3, grp = warp >> 2;
    const int sg = grp * kGrpQ;                         // the group's first query
    const int nq = min(kGrpQ, S - sg);                  // its queries (<= 0: none)
    const bool of32 = (a.flags & kOF32) != 0;
    char* o = static_cast<char*>(a.o);
    unsigned char* gstg = smem + pl.offZ + grp * 2 * kStgHalf;
    const bool issuer = quarter == 0 && lane == 0;
    // stmatrix row address of thread `lane` for query 0: row t = lane % 8 of the half holding
    // this warp's columns, 16-byte chunk (quarter % 2) * 4 + lane / 8, swizzled by t
    const int t8 = lane & 7;
    const uint32_t stg_row = smem_addr(gstg) + (quarter >> 1) * kStgHalf + t8 * 128 +
                             ((((quarter & 1) * 4 + (lane >> 3)) ^ t8) << 4);
    const uint32_t tq = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kTc2Col0;
    for (int q = 0; q < nch2; ++q) {
      const int b = q & 1;
      wait(&dfull[b], (q >> 1) & 1);
      tc_fence_after();
      const int c2 = (nch2 - 1 - q) * 2 * kKC;  // the stage's first column in the window
      uint32_t v[kGrpQ][8];
      if (!of32) {
#pragma unroll
        for (int k = 0; k < kGrpQ; ++k)
          if (k < nq) {
            uint32_t(&lo)[4] = *reinterpret_cast<uint32_t(*)[4]>(&v[k][0]);
            uint32_t(&hi)[4] = *reinterpret_cast<uint32_t(*)[4]>(&v[k][4]);
            const uint32_t col = b * pl.Nb + (sg + k) * kTT;
            tmem_ld_16x256b(tq + col, lo);
            tmem_ld_16x256b(tq + (16u << 16) + col, hi);
          }
      } else {
#pragma unroll
        for (int k = 0; k < kGrpQ; ++k)
          if (k < nq) tmem_ld8(tq + b * pl.Nb + (sg + k) * kTT, v[k]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[b]);
      if (nq <= 0) continue;
      if (!of32) {
        if (issuer) bulk_wait_read<0>();  // the previous stage's stores have read the tile
        named_barrier(2 + grp, 128);
#pragma unroll
        for (int k = 0; k < kGrpQ; ++k)
          if (k < nq)
            stmatrix_x4_trans(stg_row + k * kTT * 128,
                              pack_bf16x2(__uint_as_float(v[k][0]), __uint_as_float(v[k][1])),
                              pack_bf16x2(__uint_as_float(v[k][2]), __uint_as_float(v[k][3])),
                              pack_bf16x2(__uint_as_float(v[k][4]), __uint_as_float(v[k][5])),
                              pack_bf16x2(__uint_as_float(v[k][6]), __uint_as_float(v[k][7])));
        fence_async_smem();
        named_barrier(2 + grp, 128);
        if (issuer) {
          tma_store_3d(&tm_o, gstg, cw + c2, static_cast<int>(t0), sg);
          if (c2 + kKC < wcols)
            tma_store_3d(&tm_o, gstg + kStgHalf, cw + c2 + kKC, static_cast<int>(t0), sg);
          bulk_commit();
        }
      } else {
        const int tc = quarter * 32 + lane;  // this thread's column in the stage
        if (c2 + tc < wcols) {
#pragma unroll
          for (int k = 0; k < kGrpQ; ++k)
            if (k < nq)
#pragma unroll
              for (int t = 0; t < kTT; ++t) {
                const int64_t tok = t0 + t;
                if (tok < T)
                  __stcs(reinterpret_cast<float*>(
                             o + ((static_cast<int64_t>(sg + k) * T + tok) * d + cw + c2 + tc) * 4),
                         __uint_as_float(v[k][t]));
              }
        }
      }
    }
    if (issuer) bulk_wait_all();  // o written before the CTA exits
  } else {
  // Half h takes the ring's stages of parity h.  Within a half, warp hw is token hw; lane:
  // group of 6 queries (lane / 8) and 16-byte chunk (lane % 8).  The weights come from shared
  // memory as ready-made (a, a) pairs, 3 x 16 bytes per source.
  const int t2 = hw;
  const int grp = lane >> 3;
  const int kg = lane & 7;
  const int64_t tok2 = t0 + t2;
  const bool active2 = grp * 6 < S;
  const float* at = alph + (t2 * n * 4 + grp) * 12;     // n <= 9
  const float* zt = zbuf + t2 * ZR + grp * 6;  // weights of (j, t2, head, 6 queries)
  // source j's chunk: row j * 8 + t2, swizzled chunk kg ^ t2 (independent of j)
  const int boff = t2 * 128 + ((kg ^ t2) << 4);
  char* o = static_cast<char*>(a.o);
  const bool of32 = (a.flags & kOF32) != 0;  // o stored in fp32 instead of bf16
  const int first2 = nch + (((nch & 1) != half) ? 1 : 0);
  RingPos rp2(first2, SB);
  for (int ib = first2; ib < total; ib += 2, rp2.advance(2, SB)) {
    const int bs = rp2.bs;
    const int c = total - 1 - ib;  // columns in reverse
    wait(&full[bs], rp2.ph);
    if (active2) {
      const unsigned char* st = smem + bs * pl.slot + boff;
      float2 acc[6][4];
#pragma unroll
      for (int qq = 0; qq < 6; ++qq)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[qq][e] = make_float2(0.f, 0.f);
      if (kSmall) {
#pragma unroll
        for (int j = 0; j < kSmallN; ++j) {
          if (j < n) {
            float2 bv[4];
            unpack_pairs(*reinterpret_cast<const uint4*>(st + j * 1024), bv);
            const float4* ap = reinterpret_cast<const float4*>(at + j * 48);
            const float4 a0 = ap[0], a1 = ap[1], a2 = ap[2];
            const float2 al[6] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w),
                                  make_float2(a1.x, a1.y), make_float2(a1.z, a1.w),
                                  make_float2(a2.x, a2.y), make_float2(a2.z, a2.w)};
#pragma unroll
            for (int qq = 0; qq < 6; ++qq)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[qq][e] = __ffma2_rn(al[qq], bv[e], acc[qq][e]);
          }
        }
      } else {
        const float* zh = zt + (c / cph) * SZ;  // the stage's head
        for (int j = 0; j < n; ++j) {
          float2 bv[4];
          unpack_pairs(*reinterpret_cast<const uint4*>(st + j * 1024), bv);
          const float2* zp = reinterpret_cast<const float2*>(zh + j * kTT * ZR);
          const float2 w01 = zp[0], w23 = zp[1], w45 = zp[2];
          const float2 al[6] = {make_float2(w01.x, w01.x), make_float2(w01.y, w01.y),
                                make_float2(w23.x, w23.x), make_float2(w23.y, w23.y),
                                make_float2(w45.x, w45.x), make_float2(w45.y, w45.y)};
#pragma unroll
          for (int qq = 0; qq < 6; ++qq)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[qq][e] = __ffma2_rn(al[qq], bv[e], acc[qq][e]);
        }
      }
      const int k = c * kKC + kg * 8;  // column in the window
      if (tok2 < T && k < wcols && !of32) {
        char* op = o + ((static_cast<int64_t>(grp * 6) * T + tok2) * d + cw + k) * 2;
        const int64_t qstride = T * d * 2;
#pragma unroll
        for (int qq = 0; qq < 6; ++qq) {
          if (grp * 6 + qq < S)
            __stcs(reinterpret_cast<uint4*>(op + qq * qstride),
                   make_uint4(pack_bf16x2(acc[qq][0].x, acc[qq][0].y),
                              pack_bf16x2(acc[qq][1].x, acc[qq][1].y),
                              pack_bf16x2(acc[qq][2].x, acc[qq][2].y),
                              pack_bf16x2(acc[qq][3].x, acc[qq][3].y)));
        }
      } else if (tok2 < T && k < wcols) {  // o in fp32: two 16-byte words per chunk
        char* op = o + ((static_cast<int64_t>(grp * 6) * T + tok2) * d + cw + k) * 4;
        const int64_t qstride = T * d * 4;
#pragma unroll
        for (int qq = 0; qq < 6; ++qq) {
          if (grp * 6 + qq < S) {
            uint4* q4 = reinterpret_cast<uint4*>(op + qq * qstride);
            __stcs(q4, make_uint4(__float_as_uint(acc[qq][0].x), __float_as_uint(acc[qq][0].y),
                                  __float_as_uint(acc[qq][1].x), __float_as_uint(acc[qq][1].y)));
            __stcs(q4 + 1,
                   make_uint4(__float_as_uint(acc[qq][2].x), __float_as_uint(acc[qq][2].y),
                              __float_as_uint(acc[qq][3].x), __float_as_uint(acc[qq][3].y)));
          }
        }
      }
    }
    release(bs, true);
  }
  }

  // ------------------------------------ teardown ------------------------------------
  tc_fence_before();
  named_barrier(1, kCompute);
  tc_fence_after();
  if (warp == 0) {
    // the MMAs of an aborted run may still be running
    if (lane == 0 && *abort_flag) mbar_wait_drain(dready, 0);
    // every MMA (and its completion signals) done before the columns are freed
    if (kTc2 && lane == 0) mbar_wait_drain(mdone, 0);
    __syncwarp();
    tmem_dealloc(tmem, pl.tcols);
  }
}

}  // namespace

using Phase1TcKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap,
                                const Phase1Args, const TcPlan);

// The kernel instantiation for kn sources (1 .. 9: compile-time count; 0: any), sweep 2 on the
// CUDA cores.
template <bool kSplit>
Phase1TcKernel phase1_tc_instance(int kn) {
  switch (kn) {
    case 1: return phase1_tc_kernel<1, kSplit, false>;
    case 2: return phase1_tc_kernel<2, kSplit, false>;
    case 3: return phase1_tc_kernel<3, kSplit, false>;
    case 4: return phase1_tc_kernel<4, kSplit, false>;
    case 5: return phase1_tc_kernel<5, kSplit, false>;
    case 6: return phase1_tc_kernel<6, kSplit, false>;
    case 7: return phase1_tc_kernel<7, kSplit, false>;
    case 8: return phase1_tc_kernel<8, kSplit, false>;
    case 9: return phase1_tc_kernel<9, kSplit, false>;
    default: return phase1_tc_kernel<0, kSplit, false>;
  }
}

// Sweep 2 on the tensor cores, kn in kTc2MinN .. 9.
Phase1TcKernel phase1_tc2_instance(int kn) {
  switch (kn) {
    case 3: return phase1_tc_kernel<3, false, true>;
    case 4: return phase1_tc_kernel<4, false, true>;
    case 5: return phase1_tc_kernel<5, false, true>;
    case 6: return phase1_tc_kernel<6, false, true>;
    case 7: return phase1_tc_kernel<7, false, true>;
    case 8: return phase1_tc_kernel<8, false, true>;
    default: return phase1_tc_kernel<9, false, true>;
  }
}

// One head and kTc2MinN .. 9 sources: the weighted sum on the tensor cores.
bool use_tc2(int n, int heads) { return heads == 1 && n >= kTc2MinN && n <= kSmallN; }

bool phase1_tc_supported(int n, int S, int d, int heads) {
  TcPlan p;
  return make_tc_plan(n, S, d, heads, use_tc2(n, heads), p);
}

cudaError_t launch_phase1_tc(const Phase1Args& a, cudaStream_t s) {
  TcPlan pl;
  const bool small = a.heads == 1 && a.n <= kSmallN;  // compile-time source count
  const bool tc2 = use_tc2(a.n, a.heads);
  if (a.u_split == nullptr || !make_tc_plan(a.n, a.S, a.d, a.heads, tc2, pl))
    return cudaErrorInvalidValue;
  CUtensorMap mb, mq, mo;
  cudaError_t e = encode_source_map(&mb, a.reps, a.src_stride, a.n, a.T, a.d, 2, kKC, kTT);
  if (e == cudaSuccess) e = encode_split_query_map(&mq, a.u_split, a.S, a.d, pl.Npad);
  // bf16 o of the tensor-core sweep 2 leaves through tensor stores; otherwise unused
  if (e == cudaSuccess)
    e = tc2 && (a.flags & kOF32) == 0
            ? encode_output_map(&mo, a.o, a.S, a.T, a.d, kKC, kTT, kGrpQ, true)
            : (mo = mb, cudaSuccess);
  if (e != cudaSuccess) return e;
  const int kn = small ? a.n : 0;  // compile-time source count
  auto kern = tc2 ? phase1_tc2_instance(kn) : phase1_tc_instance<false>(kn);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (a.T + kTT - 1) / kTT;
  // Few token tiles (decode-sized T, one head, at most 16 sources): a cluster of W CTAs splits
  // each tile's columns, if W tiles' worth of CTAs still fit one wave and such clusters can be
  // resident; the CTAs add their partial sums through distributed shared memory.
  TcPlan psplit;  // the split kernels keep sweep 2 on the CUDA cores
  if (a.heads == 1 && a.n * kTT <= kM && make_tc_plan(a.n, a.S, a.d, 1, false, psplit)) {
    int sms = 0, dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    auto ksplit = phase1_tc_instance<true>(kn);
    e = cudaFuncSetAttribute(ksplit, cudaFuncAttributeMaxDynamicSharedMemorySize, psplit.smem);
    if (e != cudaSuccess) return e;
    for (int W = 4; W >= 2; W /= 2) {
      if (a.d % (W * kKC) != 0 || blocks * W > sms) continue;
      TcPlan ps = psplit;
      ps.csplit = W;
      ps.windows = W;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(W));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = ps.smem;
      cfg.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = static_cast<unsigned>(W);
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, ksplit, &cfg) != cudaSuccess || clusters < 1) {
        cudaGetLastError();  // not launchable with this cluster size: try the next
        continue;
      }
      return cudaLaunchKernelEx(&cfg, ksplit, mb, mq, mo, a, ps);
    }
  }
  const dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(pl.windows));
  return launch_pdl(kern, grid, kThreads, pl.smem, s, mb, mq, mo, a, pl);
}

namespace {
// A wait that cannot succeed: an mbarrier that expects one arrival and gets none.  Thread 0 polls
// it `polls` times, then counts the timeout like any bounded wait of the library and returns.
__global__ void wait_selftest_kernel(uint32_t polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t addr = smem_addr(&bar);
    bool done = false;
    for (uint32_t i = 0; i < polls && !done; ++i) done = mbar_try_wait(addr, 0);
    if (!done) atomicAdd(&g_wait_timeouts, 1u);
  }
}
}  // namespace

cudaError_t launch_wait_selftest(unsigned int polls, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(polls);
  return cudaGetLastError();
}

unsigned int phase1_tc_poll_timeouts() {
  return take_wait_timeouts();
}

}  // namespace attnres
