// Block backward without any allocation: attnres_backward_block_noalloc.
//
// attnres_backward_block needs scratch memory (phase 1 recomputed, dL/do, per-token
// coefficients), which its caller passes in.  Some callers cannot allocate device memory when
// they run this: code that works inside a framework whose allocator owns every device byte and
// hands out no extra buffers during execution, or code on a latency-critical path that must not
// pay for cudaMalloc's implicit synchronisation.  This entry point runs the same kernels with the
// scratch taken from a fixed array that lives in this library's own device memory.
//
// The array is a file-scope __device__ variable: the driver reserves it on every GPU that loads
// this file's kernels and keeps it there until the process exits.  Its size is
// ATTNRES_NOALLOC_SCRATCH_BYTES; larger blocks are rejected before anything runs.
// Host code cannot use the array's name as a device address (on the host it only stands for
// the symbol), so the first call on each device, with that device current, asks the runtime for
// the array's device address (cudaGetSymbolAddress) and keeps it for later calls.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/attnres.h"
#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTNRES_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool opt_aligned16(const void* p) { return p == nullptr || aligned16(p); }

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" attnres_status attnres_backward_block_noalloc(
    const void* reps, int64_t src_stride, int n_src, const void* v, int64_t v_stride, int S,
    int64_t T, int d, attnres_dtype io, const float* u, const void* u_split, float eps_key,
    const float* gamma_in, float eps_in, const void* g_y, void* d_reps, void* d_v,
    int64_t dv_stride, float* du, float* dgamma_in, void* stream) {
  if (io != ATTNRES_F32 && io != ATTNRES_BF16) return ATTNRES_ERR_INVALID_ARG;
  uint64_t need = 0;
  const attnres_status st = attnres_backward_block_workspace_size(n_src, S, T, d, io, &need);
  if (st != ATTNRES_OK) return st;
  if (need > ATTNRES_NOALLOC_SCRATCH_BYTES) return ATTNRES_ERR_UNSUPPORTED;  // too many tokens
  if (!(eps_key >= 0.f) || !(eps_in >= 0.f)) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (reps == nullptr || u == nullptr || g_y == nullptr || d_reps == nullptr || du == nullptr)
    return ATTNRES_ERR_INVALID_ARG;
  if (S > 1 && (v == nullptr || d_v == nullptr)) return ATTNRES_ERR_INVALID_ARG;
  if (n_src > 1 && src_stride < T * d) return ATTNRES_ERR_INVALID_ARG;
  if (S > 2 && (v_stride < T * d || dv_stride < T * d)) return ATTNRES_ERR_INVALID_ARG;
  if (src_stride < 0 || v_stride < 0 || dv_stride < 0) return ATTNRES_ERR_INVALID_ARG;
  if (!aligned16(reps) || !aligned16(u) || !aligned16(g_y) || !aligned16(d_reps) ||
      !aligned16(du) || !opt_aligned16(v) || !opt_aligned16(d_v) || !opt_aligned16(u_split) ||
      !opt_aligned16(gamma_in) || !opt_aligned16(dgamma_in) || src_stride % 8 != 0 ||
      v_stride % 8 != 0 || dv_stride % 8 != 0)
    return ATTNRES_ERR_MISALIGNED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return ATTNRES_ERR_CUDA;
  attnres::BwdBlockArgs a;
  memset(&a, 0, sizeof(a));
  a.reps = reps;
  a.src_stride = src_stride;
  a.n = n_src;
  a.T = T;
  a.d = d;
  a.v = v;
  a.v_stride = v_stride;
  a.S = S;
  a.u = u;
  a.u_split = u_split;
  a.eps_key = eps_key;
  a.gamma_in = gamma_in;
  a.eps_in = eps_in;
  a.g_y = g_y;
  a.d_reps = d_reps;
  a.d_v = d_v;
  a.dv_stride = dv_stride;
  a.du = du;
  a.dgamma_in = dgamma_in;
  // Every region of the scratch is written before it is read within one call, so nothing in
  // it has to start at zero and the previous call's contents do no harm.
  const cudaError_t e = attnres::launch_backward_block(static_cast<attnres::IO>(io), a, scratch,
                                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTNRES_OK : ATTNRES_ERR_CUDA;
}
