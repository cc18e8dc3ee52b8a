// Internal launch interface between the C ABI (attnres_abi.cu) and the kernels.
// Arguments arrive here already validated.
#pragma once

#include <cuda.h>  // CUtensorMap (type only)
#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

enum class IO { F32 = 0, BF16 = 1 };

// Variant flags (values of ATTNRES_SIGMOID_WEIGHTS / ATTNRES_NO_KEY_NORM in attnres.h).
constexpr unsigned kSigmoid = 1u;    // alpha_i = sigmoid(z_i), no normalisation over sources
constexpr unsigned kNoKeyNorm = 2u;  // z_i = u . v_i, no RMS division
// Phase 1's output o is stored in fp32 whatever the I/O type (value of ATTNRES_O_F32); phase 2
// and the grouped merge then read o_l in fp32.
constexpr unsigned kOF32 = 4u;

struct Phase1Args {
  const void* reps;
  int64_t src_stride;  // elements between sources
  int n;               // sources
  int64_t T;
  int d;
  const float* u;      // [S, d]
  const void* u_split; // [2S, d] bf16 (hi, lo row pairs) or null
  int S;
  float eps;
  void* o;             // [S, T, d]
  float* m;            // [S, H, T] or null
  float* lse;          // [S, H, T] or null
  float* alpha;        // [S, H, T, n] or null
  unsigned flags;      // kSigmoid | kNoKeyNorm
  int heads;           // depth-attention heads H: m, lse [S][H][T], alpha [S][H][T][n]
};

struct Phase2Args {
  const void* o;
  const float* lse;
  const void* partial;
  const void* v_prev;
  void* partial_out;
  int64_t T;
  int d;
  const float* u;
  float eps_key;
  const float* gamma_in;
  float eps_in;
  void* h;
  void* y;
  float* alpha_p;      // [H][T] or null
  unsigned flags;
  int heads;           // lse [H][T]
};

constexpr int kMaxSources = 64;

struct FullArgs {
  const void* srcs[kMaxSources];
  int n;
  int64_t T;
  int d;
  const float* u;
  float eps_key;
  const float* gamma_in;
  float eps_in;
  void* h;
  void* y;
  float* alpha;     // [H][T][n] or null
  float* m;         // [H][T] or null: max logit
  float* lse;       // [H][T] or null: log-sum-exp of the logits
  unsigned flags;
  const void* o0;   // [T, d] or null: normalised output of an earlier source partition
  const float* lse0;  // [H][T]: its log-sum-exp (required with o0 unless sigmoid weights)
  int heads;          // alpha [H][T][n], m and lse [H][T]
  bool h_f32;         // h is stored in fp32 (phase 1 with one query and kOF32)
  bool o0_f32;        // o0 is stored in fp32 (the grouped merge with kOF32)
};

// Backward of one sublayer's aggregation (backward.cu).
constexpr int kBwdMaxSources = 16;
struct BwdArgs {
  const void* srcs[kBwdMaxSources];   // [T, d] each
  void* dsrcs[kBwdMaxSources];        // [T, d] each: dL/dv_i
  int n;
  int64_t T;
  int d;
  const float* u;         // [d] folded query
  float eps_key;
  const float* gamma_in;  // [d] or null
  float eps_in;
  const void* g_y;        // [T, d] dL/dy
  float* du;              // [d] accumulated
  float* dgamma_in;       // [d] accumulated, or null
};
// Row-vector limit of the backward kernel: d / (elements per 16 bytes) <= 4 * 256.
constexpr int kBwdMaxVectors = 1024;
cudaError_t launch_backward(IO io, const BwdArgs& a, cudaStream_t s);
// Bounded waits of the ring backward that gave up since the last call (synchronises the device).
unsigned int backward_poll_timeouts();

// Backward of one block of Block AttnRes (backward_block.cu).
constexpr int kBlkMaxN = 16;   // completed sources
constexpr int kBlkMaxS = 24;   // sublayers of the block
struct BwdBlockArgs {
  const void* reps;       // [n][T][d]: source j at reps + j * src_stride elements
  int64_t src_stride;
  int n;
  int64_t T;
  int d;
  const void* v;          // v_1 .. v_{S-1}: v_k at v + (k - 1) * v_stride elements ([T, d] each)
  int64_t v_stride;
  int S;
  const float* u;         // [S][d] folded queries
  const void* u_split;    // [2S][d] bf16 or null (tensor-core phase 1)
  float eps_key;
  const float* gamma_in;  // [S][d] or null
  float eps_in;
  const void* g_y;        // [S][T][d] dL/dy_i
  void* d_reps;           // [n][T][d] dL/db_j (written)
  void* d_v;              // dL/dv_k at d_v + (k - 1) * dv_stride, k = 1 .. S-1 (written)
  int64_t dv_stride;
  float* du;              // [S][d] added
  float* dgamma_in;       // [S][d] added, or null
  // workspace (set by the launcher)
  float* o;               // [S][T][d] phase 1 recomputed, fp32
  float* lse;             // [S][T]
  float* alpha;           // [S][T][n]
  float* q;               // [S][T][d] dL/do_i, fp32
  float* sc2;             // [S][T][4]: c_i, w_A / r_h, w_p / r_h, dz_p / r_p
  float* rec;             // [T][rec_floats] per-token coefficients of the column kernel
  int rec_floats;
};
int64_t backward_block_workspace_bytes(IO io, int n, int S, int64_t T, int d);
bool backward_block_supported(IO io, int n, int S, int d);
cudaError_t launch_backward_block(IO io, BwdBlockArgs a, void* workspace, cudaStream_t s);

// Each launcher returns cudaSuccess or the launch error.
cudaError_t launch_phase1(IO io, const Phase1Args& a, cudaStream_t s);
// Returns false when the (n, S) combination does not fit the phase-1 kernel.
bool phase1_supported(int n, int S);
cudaError_t launch_phase2(IO io, const Phase2Args& a, cudaStream_t s);
cudaError_t launch_full(IO io, const FullArgs& a, cudaStream_t s);
// The same aggregation by the persistent row-ring kernel (fullring.cu): one head, no seeded
// partition, n <= 16 sources, rows of 512 to 1024 16-byte vectors that fit the ring.
bool full_ring_supported(IO io, const FullArgs& a);
cudaError_t launch_full_ring(IO io, const FullArgs& a, cudaStream_t s);
unsigned int full_ring_poll_timeouts();
cudaError_t launch_partial_update(IO io, const void* a, const void* b, void* out, int64_t n_elems,
                                  cudaStream_t s);
// u = w * g (g null: copy); u_split (null: not written) receives rows 2r, 2r + 1 = the bf16
// hi and lo parts of row r of u.
cudaError_t launch_query_prep(const float* w, const float* g, float* u, void* u_split, int rows,
                              int d, cudaStream_t s);
// Tensor-copy descriptors (tmap.cu).  Sources: dims (column, token, source) of a [n][T][d]
// tensor whose sources are src_stride elements apart, box (box_k, box_t, n), 128-byte swizzle.
// Queries: dims (column, query) of an fp32 [S][d] tensor, box (32, S), 128-byte swizzle.
cudaError_t encode_source_map(CUtensorMap* map, const void* reps, int64_t src_stride, int n,
                              int64_t T, int d, int E, int box_k, int box_t);
cudaError_t encode_query_map(CUtensorMap* map, const float* u, int S, int d);
// Split queries: dims (column, row) of a bf16 [2S][d] tensor, box (64, rows_box) with rows past
// 2S zero-filled, 128-byte swizzle.
cudaError_t encode_split_query_map(CUtensorMap* map, const void* u_split, int S, int d,
                                   int rows_box);
// bf16 [S][T][d] output (phase 1's o) for tensor stores of [box_s queries][box_t rows][box_k
// columns] tiles, unswizzled or with the 128-byte swizzle (box_k = 64).
cudaError_t encode_output_map(CUtensorMap* map, void* o, int S, int64_t T, int d, int box_k,
                              int box_t, int box_s, bool swizzle128);

// Tensor-core phase 1 (phase1_tc.cu): bf16 I/O, 2 <= S <= 24, n <= 64, split queries given;
// with H > 1 heads, d / H a multiple of 64.
bool phase1_tc_supported(int n, int S, int d, int heads);
cudaError_t launch_phase1_tc(const Phase1Args& a, cudaStream_t s);
unsigned int phase1_tc_poll_timeouts();
// One CTA whose bounded wait cannot succeed: gives up after `polls` polls and counts a timeout
// (read by phase1_tc_poll_timeouts).
cudaError_t launch_wait_selftest(unsigned int polls, cudaStream_t s);

// Number of bounded waits in the phase-1 kernel that gave up since the last call (read and
// cleared; synchronous).  0xffffffff if the device word could not be read.
unsigned int phase1_poll_timeouts();

}  // namespace attnres
