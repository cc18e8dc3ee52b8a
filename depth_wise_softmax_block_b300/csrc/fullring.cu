// The direct single-pass aggregation over an explicit source list ("Attention Residuals" note,
// §7: softmax over the sources of w . RMSNorm(v_i), h = sum_i alpha_i v_i, then the sublayer's
// input RMSNorm), as a persistent kernel that streams whole source rows through a ring of
// shared-memory row slots.  Used for one head without a seeded partition, n <= 16 sources and
// rows of 512 to 1024 16-byte vectors (the final aggregation over the block representations is
// the case it is built for: n = 10 rows of 14 KB per token).
//
// One CTA per SM walks the rows blockIdx.x, blockIdx.x + gridDim.x, ...  A copy warp issues one
// bulk copy per (row, source) into the next ring slot, as soon as the slot is free, so the copies
// of the next row stream in while the current one is computed.  The 16 compute warps take a
// row in two passes over its n resident slots:
//   pass 1  each thread sums its vectors' squares and query products for every source in
//           registers (no reduction between sources); one butterfly reduce-scatter over the
//           warp (31 shuffles) leaves lane L with the warp's total of value L (source L / 2,
//           square sum or product); one barrier; lane j of every warp then adds the 16 warps'
//           totals of source j, forms z_j and, with warp shuffles, the softmax statistics, so
//           each lane holds alpha_j for the sources j = lane;
//   pass 2  h = sum_j alpha_j v_j from the same slots (alpha_j by one shuffle per source); each
//           slot is released as soon as the 16 warps are done with it.
// Against the row-per-CTA kernel (an online softmax whose every source costs a CTA-wide
// reduction, with two sources in flight in registers) a row costs one barrier (two with the
// input RMSNorm) and the copy engine keeps the next row's sources in flight.
//
// Rows held in registers (full_hold_kernel: bf16, n <= 10 sources, rows of up to 896 vectors,
// which is the final aggregation at d = 7168).  Holding a row's n slots through both passes
// leaves only SB - n slots to prefetch the next row (5 of 15 at that shape), and the copies of
// the rest start only as pass 2 frees its slots.  Here 14 compute warps (two vectors a thread)
// copy the first eight sources' vectors into registers in pass 1 (64 registers of packed
// bf16), release those slots at once, and run pass 2 from the registers (and from the slots
// of sources 9 and 10, released after it): 13 of the 15 slots prefetch while a row is reduced,
// weighted and stored.  With fewer instructions per element (packed FMAs, one reduce-scatter
// per pair of sources, no per-vector guards for 7168-wide rows) this takes 0.477 ms per
// 16384-row launch at n = 10, against 0.616 ms for the kernel that holds the slots.
// Every wait is bounded (tma.cuh); after a wait gives up the CTA stops issuing copies, skips the
// remaining waits and exits once its copies in flight have landed.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace attnres {
namespace {

constexpr int kRingCompute = 512;                  // 16 compute warps
constexpr int kRingWarps = kRingCompute / 32;
constexpr int kRingThreads = kRingCompute + 32;    // + the copy-issuing warp
constexpr int kRingVPT = 2;                        // vectors per compute thread: nv <= 1024
// Shorter rows leave most of the 16 warps idle and the per-row reductions dominate; there the
// row-per-CTA kernel is faster (measured at 256 vectors: a direct Full AttnRes walk at d = 2048
// took 21.1 ms through this kernel against 18.0 ms).
constexpr int kRingMinVectors = 512;
constexpr int kRingMaxN = 16;                      // 2 sums per source: one lane each
constexpr int kRingSlotBytes = 216 * 1024;         // shared memory for the slots
constexpr int kRingMaxSlots = 64;
// Rows held in registers: 14 compute warps + the copy warp = 480 threads.  Four of the 15 warps
// share one of the SM's four register-file partitions, so a thread may keep 128 registers (a
// 136-register build is refused at launch); the sources held take 2 x 4 of them each.
constexpr int kHoldWarps = 14;
constexpr int kHoldCompute = kHoldWarps * 32;
constexpr int kHoldThreads = kHoldCompute + 32;
constexpr int kHoldMaxN = 10;
// Sources a row keeps in registers (64 registers); sources 9 and 10 stay in their slot until
// pass 2.  Holding all ten spills (0.546 against 0.505 ms per 16384-row launch at n = 10).
constexpr int kHoldRegSrc = 8;
constexpr int kHoldVectors = kRingVPT * kHoldCompute;  // 896: d = 7168 in bf16

// Row slots for rows of `rowbytes` bytes; 0 if the ring cannot hold n sources plus two slots.
int ring_slots(int rowbytes, int n) {
  const int sb = std::min(kRingMaxSlots, kRingSlotBytes / rowbytes);
  return sb >= n + 2 ? sb : 0;
}

// The register-held kernel takes bf16 rows of at most kHoldVectors vectors and kHoldMaxN sources.
bool held_in_registers(size_t elem, const FullArgs& a) {
  return elem == 2 && a.n <= kHoldMaxN && a.d / 8 <= kHoldVectors;
}

int ring_smem(int rowbytes, int SB) {
  // slots | full, empty barriers | per-warp totals [2 rows][16 warps][32] | y sums [2][16]
  return 128 + SB * rowbytes + 2 * SB * 8 + 2 * kRingWarps * 32 * 4 + 2 * kRingWarps * 4 + 16;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// The copy-issuing thread: one bulk copy per (row, source) of the CTA's rows into the ring, each
// slot reused once its consumers have released it (`empty`), then a drain of the copies in flight.
__device__ __forceinline__ void copy_rows(const FullArgs& a, unsigned char* ring, uint64_t* full,
                                          uint64_t* empty, int SB, int rowbytes,
                                          volatile int* abort_v) {
  int it = 0, bs = 0, ph = 0;  // copies issued; slot and phase parity of the next one
  for (int64_t r = blockIdx.x; r < a.T && !*abort_v; r += gridDim.x) {
    for (int j = 0; j < a.n; ++j) {
      if (it >= SB && !mbar_wait(&empty[bs], ph ^ 1)) {
        *abort_v = 1;
        break;
      }
      if (*abort_v) break;
      mbar_arrive_expect_tx(&full[bs], static_cast<uint32_t>(rowbytes));
      bulk_load(ring + bs * rowbytes,
                static_cast<const char*>(a.srcs[j]) + r * static_cast<int64_t>(rowbytes),
                static_cast<uint32_t>(rowbytes), &full[bs]);
      ++it;
      if (++bs == SB) {
        bs = 0;
        ph ^= 1;
      }
    }
  }
  // Drain: the last copy issued into every slot has landed before the CTA may exit.
  for (int s = 0; s < SB && s < it; ++s) {
    const int last = it - 1 - ((it - 1 - s) % SB);
    mbar_wait_drain(&full[s], (last / SB) & 1);
  }
}

// Softmax (or sigmoid) weights of row r from the per-warp totals `pw` ([kWarps][32]: value 2j the
// sum of squares of source j, 2j + 1 its query product).  Every warp computes the same values;
// lane j returns alpha_j (0 for lanes j >= n).  Warp 0 stores alpha, m and lse.
template <int kWarps>
__device__ __forceinline__ float row_weights(const FullArgs& a, const float* pw, int64_t r,
                                             int warp, int lane) {
  const int n = a.n;
  const bool sigmoid = (a.flags & kSigmoid) != 0;
  const bool key_norm = (a.flags & kNoKeyNorm) == 0;
  float z = -INFINITY;
  if (lane < n) {
    float ss = 0.f, dot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      ss += pw[w * 32 + 2 * lane];
      dot += pw[w * 32 + 2 * lane + 1];
    }
    z = key_norm ? dot / sqrtf(ss / static_cast<float>(a.d) + a.eps_key) : dot;
  }
  float m = z;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float al, lse = 0.f;
  if (sigmoid) {
    al = lane < n ? 1.f / (1.f + expf(-z)) : 0.f;
  } else {
    const float ez = lane < n ? expf(z - m) : 0.f;
    const float l = warp_sum(ez);
    al = ez / l;
    lse = m + logf(l);
  }
  if (warp == 0) {
    if (a.alpha != nullptr && lane < n) a.alpha[r * n + lane] = al;
    if (lane == 0) {
      if (a.m != nullptr) a.m[r] = m;
      if (a.lse != nullptr && !sigmoid) a.lse[r] = lse;
    }
  }
  return al;
}

// Stores row r of h (this thread's vectors tid, tid + kWarps * 32) and, when requested, of
// y = gamma_in * h / r(h); `ysum` holds [kWarps] partial sums of |h|^2 for this row (the caller
// alternates two of them between rows, so one barrier suffices).
template <typename T, int kWarps>
__device__ __forceinline__ void store_row(const FullArgs& a, const float (&acc)[kRingVPT][Vec<T>::N],
                                          int64_t r, float* ysum, int tid, int warp, int lane,
                                          int nv) {
  constexpr int VE = Vec<T>::N;
  constexpr int kCompute = kWarps * 32;
  const int64_t base = r * a.d;
  float inv = 0.f;
  if (a.y != nullptr) {  // uniform over the CTA
    float s2 = 0.f;
#pragma unroll
    for (int k = 0; k < kRingVPT; ++k)
#pragma unroll
      for (int e = 0; e < VE; ++e) s2 = fmaf(acc[k][e], acc[k][e], s2);
    s2 = warp_sum(s2);
    if (lane == 0) ysum[warp] = s2;
    named_barrier(1, kCompute);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += ysum[w];
    inv = 1.f / sqrtf(tot / static_cast<float>(a.d) + a.eps_in);
  }
#pragma unroll
  for (int k = 0; k < kRingVPT; ++k) {
    const int v = tid + k * kCompute;
    if (v < nv) {
      if (a.h != nullptr) {
        if (a.h_f32)
          st_vec<float, VE>(static_cast<float*>(a.h) + base + v * VE, acc[k]);
        else
          st_global(static_cast<T*>(a.h) + base + v * VE, pack(acc[k]));
      }
      if (a.y != nullptr) {
        float y[VE];
#pragma unroll
        for (int e = 0; e < VE; ++e)
          y[e] = acc[k][e] * inv * (a.gamma_in != nullptr ? __ldg(a.gamma_in + v * VE + e) : 1.f);
        st_global(static_cast<T*>(a.y) + base + v * VE, pack(y));
      }
    }
  }
}

// Butterfly reduce-scatter over the warp: at the step of width o a lane keeps the half of its
// values selected by its lane bit o and adds the partner's copy of that half; after the five
// steps ps[0] of lane L is the warp's total of value L.
__device__ __forceinline__ void warp_reduce_scatter(float (&ps)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? ps[i] : ps[i + o];
      const float keep = upper ? ps[i + o] : ps[i];
      ps[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kRingThreads, 1) full_ring_kernel(const FullArgs a, int SB) {
  constexpr int VE = Vec<T>::N;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  const int rowbytes = a.d * static_cast<int>(sizeof(T));
  const int nv = a.d / VE;
  const int n = a.n;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + SB * rowbytes);
  uint64_t* empty = full + SB;
  float* part = reinterpret_cast<float*>(empty + SB);  // [2][16 warps][32]: value 2j + {ss, dot}
  float* ysum = part + 2 * kRingWarps * 32;             // [2][16 warps]
  int* abort_flag = reinterpret_cast<int*>(ysum + 2 * kRingWarps);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < SB; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kRingWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_enter();  // nothing above touches global memory
  volatile int* abort_v = abort_flag;

  // ------------------------------ copy-issuing warp ------------------------------
  if (warp == kRingWarps) {
    if (lane == 0) copy_rows(a, ring, full, empty, SB, rowbytes, abort_v);
    return;
  }

  // ------------------------------- compute warps --------------------------------
  auto wait = [&](uint64_t* bar, int parity) {
    if (!*abort_v && !mbar_wait(bar, static_cast<uint32_t>(parity))) *abort_v = 1;
  };
  // The query for this thread's vectors, kept for the CTA's life.
  float uq[kRingVPT][VE];
#pragma unroll
  for (int k = 0; k < kRingVPT; ++k) {
    const int v = tid + k * kRingCompute;
#pragma unroll
    for (int e = 0; e < VE; ++e) uq[k][e] = v < nv ? __ldg(a.u + v * VE + e) : 0.f;
  }

  int bs = 0, ph = 0;  // ring position of the row's first source
  int par = 0;         // row parity: which half of the partial buffers
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x, par ^= 1) {
    float* pw = part + par * (kRingWarps * 32);
    // ---- pass 1: this thread's sums of squares and query products of every source ----
    float ps[2 * kRingMaxN];  // value 2j: sum of squares of source j; 2j + 1: query product
    {
      int b = bs, p = ph;
#pragma unroll
      for (int j = 0; j < kRingMaxN; ++j) {
        ps[2 * j] = ps[2 * j + 1] = 0.f;
        if (j < n) {
          wait(&full[b], p);
          const uint4* sl = reinterpret_cast<const uint4*>(ring + b * rowbytes);
#pragma unroll
          for (int k = 0; k < kRingVPT; ++k) {
            const int v = tid + k * kRingCompute;
            if (v < nv) {
              float x[VE];
              unpack(sl[v], x);
#pragma unroll
              for (int e = 0; e < VE; ++e) {
                ps[2 * j] = fmaf(x[e], x[e], ps[2 * j]);
                ps[2 * j + 1] = fmaf(uq[k][e], x[e], ps[2 * j + 1]);
              }
            }
          }
          if (++b == SB) {
            b = 0;
            p ^= 1;
          }
        }
      }
    }
    warp_reduce_scatter(ps, lane);
    pw[warp * 32 + lane] = ps[0];
    named_barrier(1, kRingCompute);
    const float al = row_weights<kRingWarps>(a, pw, r, warp, lane);
    // ---- pass 2: h = sum_j alpha_j v_j; each slot is released after its use ----
    float acc[kRingVPT][VE];
#pragma unroll
    for (int k = 0; k < kRingVPT; ++k)
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[k][e] = 0.f;
    for (int j = 0; j < n; ++j) {
      const float aj = __shfl_sync(0xffffffffu, al, j);
      const uint4* sl = reinterpret_cast<const uint4*>(ring + bs * rowbytes);
#pragma unroll
      for (int k = 0; k < kRingVPT; ++k) {
        const int v = tid + k * kRingCompute;
        if (v < nv) {
          float x[VE];
          unpack(sl[v], x);
#pragma unroll
          for (int e = 0; e < VE; ++e) acc[k][e] = fmaf(aj, x[e], acc[k][e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[bs]);
      if (++bs == SB) {
        bs = 0;
        ph ^= 1;
      }
    }
    store_row<T, kRingWarps>(a, acc, r, ysum + par * kRingWarps, tid, warp, lane, nv);
  }
}


// Rows held in registers (bf16, n <= kHoldMaxN, nv <= kHoldVectors): the same ring, the same
// copy warp and statistics; pass 1 keeps each source's vectors in registers and releases the
// slot once they are consumed, pass 2 weights the registers.  The 15 warps place four on some
// of the SM's four register-file partitions, which caps a thread at 128 registers: the first
// kHoldRegSrc sources take 64, and the sums are reduced over the warp a pair of sources at a
// time instead of being held for one reduce-scatter at the end of the pass.  The kernel is
// bound by instruction issue (the copies keep up): element pairs go through packed fp32 FMAs
// (two independent round-to-nearest FMAs per instruction) and a thread releases a slot with
// its own arrival.
// kFullRow: the row has exactly kHoldVectors vectors (d = 7168), so no vector guard; with the
// abort flag kept in a register (one shared-memory read per row instead of one per source) this
// takes the launch from 0.505 to 0.477 ms (16384 rows, n = 10; identical outputs).
template <bool kFullRow>
__global__ void __launch_bounds__(kHoldThreads, 1) full_hold_kernel(const FullArgs a, int SB) {
  using T = bf16;
  constexpr int VE = Vec<T>::N;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  const int rowbytes = a.d * static_cast<int>(sizeof(T));
  const int nv = kFullRow ? kHoldVectors : a.d / VE;
  const int n = a.n;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + SB * rowbytes);
  uint64_t* empty = full + SB;
  float* part = reinterpret_cast<float*>(empty + SB);  // [2][14 warps][32]
  float* ysum = part + 2 * kRingWarps * 32;             // [2][14 warps]
  int* abort_flag = reinterpret_cast<int*>(ysum + 2 * kRingWarps);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < SB; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kHoldCompute);  // every compute thread releases the slot
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_enter();  // nothing above touches global memory
  volatile int* abort_v = abort_flag;

  if (warp == kHoldWarps) {
    if (lane == 0) copy_rows(a, ring, full, empty, SB, rowbytes, abort_v);
    return;
  }

  // The query for this thread's vectors as (low, high) element pairs, kept for the CTA's life.
  float2 uq[kRingVPT][VE / 2];
#pragma unroll
  for (int k = 0; k < kRingVPT; ++k) {
    const int v = tid + k * kHoldCompute;
#pragma unroll
    for (int i = 0; i < VE / 2; ++i)
      uq[k][i] = v < nv ? make_float2(__ldg(a.u + v * VE + 2 * i), __ldg(a.u + v * VE + 2 * i + 1))
                        : make_float2(0.f, 0.f);
  }

  int bs = 0, ph = 0;  // ring position of the next source
  int par = 0;
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x, par ^= 1) {
    float* pw = part + par * (kHoldWarps * 32);
    bool ab = *abort_v;  // a wait of this CTA gave up: skip the remaining waits
    uint4 xv[kHoldRegSrc][kRingVPT];          // the row's first kHoldRegSrc sources, packed
    int slot_of[kHoldMaxN - kHoldRegSrc + 1];  // ring slots of the others
    // ---- pass 1: copy every source's vectors into registers, release the slot, sum ----
    // Sources go in pairs: the pair's four warp totals (square sum and query product of each)
    // come from one reduce-scatter over the warp, six shuffles.  (Waiting for and reading both
    // sources of a pair before summing either was measured slower: 0.515 against 0.506 ms.)
#pragma unroll
    for (int j0 = 0; j0 < kHoldMaxN; j0 += 2) {
      if (j0 < n) {
        float v4[4] = {0.f, 0.f, 0.f, 0.f};  // ss, dot of source j0; ss, dot of source j0 + 1
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int j = j0 + q;
          if (j < n) {
            if (!ab && !mbar_wait(&full[bs], static_cast<uint32_t>(ph))) {
              ab = true;
              *abort_v = 1;
            }
            const uint4* sl = reinterpret_cast<const uint4*>(ring + bs * rowbytes);
            uint4 xt[kRingVPT];
#pragma unroll
            for (int k = 0; k < kRingVPT; ++k) {
              const int v = tid + k * kHoldCompute;
              xt[k] = kFullRow || v < nv ? sl[v] : make_uint4(0u, 0u, 0u, 0u);
              if (j < kHoldRegSrc) xv[j][k] = xt[k];
            }
            float2 ss = make_float2(0.f, 0.f), dot = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kRingVPT; ++k) {
              const uint32_t w[4] = {xt[k].x, xt[k].y, xt[k].z, xt[k].w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 x = make_float2(__uint_as_float(w[i] << 16),
                                             __uint_as_float(w[i] & 0xffff0000u));
                ss = __ffma2_rn(x, x, ss);
                dot = __ffma2_rn(uq[k][i], x, dot);
              }
            }
            // The sums consumed every register this thread loaded from the slot, so its reads
            // are complete: each thread releases the slot for itself (a source not held in
            // registers keeps its slot until pass 2).
            if (j < kHoldRegSrc)
              mbar_arrive(&empty[bs]);
            else
              slot_of[j - kHoldRegSrc] = bs;
            if (++bs == SB) {
              bs = 0;
              ph ^= 1;
            }
            v4[2 * q] = ss.x + ss.y;
            v4[2 * q + 1] = dot.x + dot.y;
          }
        }
        // Reduce-scatter of the four values: lane bit 4 picks the source of the pair, lane
        // bit 3 the sum, the last three steps add over the remaining lanes.
        const bool up16 = (lane & 16) != 0, up8 = (lane & 8) != 0;
        const float k0 =
            (up16 ? v4[2] : v4[0]) + __shfl_xor_sync(0xffffffffu, up16 ? v4[0] : v4[2], 16);
        const float k1 =
            (up16 ? v4[3] : v4[1]) + __shfl_xor_sync(0xffffffffu, up16 ? v4[1] : v4[3], 16);
        float t = (up8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, up8 ? k0 : k1, 8);
        t += __shfl_xor_sync(0xffffffffu, t, 4);
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        t += __shfl_xor_sync(0xffffffffu, t, 1);
        if ((lane & 7) == 0) pw[warp * 32 + 2 * j0 + (lane >> 3)] = t;
      }
    }
    named_barrier(1, kHoldCompute);
    const float al = row_weights<kHoldWarps>(a, pw, r, warp, lane);
    // ---- pass 2: h = sum_j alpha_j v_j from the registers ----
    float2 acc2[kRingVPT][VE / 2];
#pragma unroll
    for (int k = 0; k < kRingVPT; ++k)
#pragma unroll
      for (int i = 0; i < VE / 2; ++i) acc2[k][i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kHoldMaxN; ++j) {
      if (j < n) {
        const float aj = __shfl_sync(0xffffffffu, al, j);
        const float2 a2 = make_float2(aj, aj);
        uint4 xt[kRingVPT];
        const int slot = j < kHoldRegSrc ? 0 : slot_of[j - kHoldRegSrc];
#pragma unroll
        for (int k = 0; k < kRingVPT; ++k) {
          if (j < kHoldRegSrc) {
            xt[k] = xv[j][k];
          } else {
            const int v = tid + k * kHoldCompute;
            xt[k] = kFullRow || v < nv ? reinterpret_cast<const uint4*>(ring + slot * rowbytes)[v]
                                       : make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int k = 0; k < kRingVPT; ++k) {
          const uint32_t w[4] = {xt[k].x, xt[k].y, xt[k].z, xt[k].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 x = make_float2(__uint_as_float(w[i] << 16),
                                         __uint_as_float(w[i] & 0xffff0000u));
            acc2[k][i] = __ffma2_rn(a2, x, acc2[k][i]);
          }
        }
        if (j >= kHoldRegSrc) mbar_arrive(&empty[slot]);  // the FMAs consumed the slot's reads
      }
    }
    float acc[kRingVPT][VE];
#pragma unroll
    for (int k = 0; k < kRingVPT; ++k)
#pragma unroll
      for (int i = 0; i < VE / 2; ++i) {
        acc[k][2 * i] = acc2[k][i].x;
        acc[k][2 * i + 1] = acc2[k][i].y;
      }
    store_row<T, kHoldWarps>(a, acc, r, ysum + par * kRingWarps, tid, warp, lane, nv);
  }
}

template <typename T>
cudaError_t launch_ring(const FullArgs& a, int SB, cudaStream_t s) {
  const int rowbytes = a.d * static_cast<int>(sizeof(T));
  const int smem = ring_smem(rowbytes, SB);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool hold = held_in_registers(sizeof(T), a);
  auto kern = !hold                         ? full_ring_kernel<T>
              : a.d / 8 == kHoldVectors ? full_hold_kernel<true>
                                        : full_hold_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = a.T < sms ? a.T : sms;
  const int threads = hold ? kHoldThreads : kRingThreads;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(threads),
                    static_cast<size_t>(smem), s, a, SB);
}

}  // namespace

bool full_ring_supported(IO io, const FullArgs& a) {
  const int E = io == IO::BF16 ? 2 : 4;
  const int VE = 16 / E;
  if (a.heads != 1 || a.o0 != nullptr || a.n < 1 || a.n > kRingMaxN) return false;
  if (a.d % VE != 0 || a.d / VE < kRingMinVectors || a.d / VE > kRingVPT * kRingCompute)
    return false;
  return ring_slots(a.d * E, a.n) > 0;
}

cudaError_t launch_full_ring(IO io, const FullArgs& a, cudaStream_t s) {
  if (!full_ring_supported(io, a)) return cudaErrorInvalidValue;
  if (a.T == 0) return cudaSuccess;
  const int E = io == IO::BF16 ? 2 : 4;
  const int SB = ring_slots(a.d * E, a.n);
  return io == IO::BF16 ? launch_ring<bf16>(a, SB, s) : launch_ring<float>(a, SB, s);
}

unsigned int full_ring_poll_timeouts() {
  return take_wait_timeouts();
}

}  // namespace attnres
