// The C ABI of include/attnres.h: host-side argument validation, then dispatch to the
// kernels.  Nothing is launched unless every check passes; no exception crosses the ABI.
#include <stdint.h>
#include <string.h>

#include <string>

#include "../../include/attnres.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_cuda_error;

using attnres::IO;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool opt_aligned16(const void* p) { return p == nullptr || aligned16(p); }
bool valid_io(attnres_dtype io) { return io == ATTNRES_F32 || io == ATTNRES_BF16; }
bool valid_flags(unsigned flags) {
  return (flags & ~(ATTNRES_SIGMOID_WEIGHTS | ATTNRES_NO_KEY_NORM)) == 0;
}
// The entry points that pass phase 1's output on also take its storage flag.
bool valid_o_flags(unsigned flags) { return valid_flags(flags & ~ATTNRES_O_F32); }

attnres_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ATTNRES_OK;
  g_last_cuda_error = cudaGetErrorString(e);
  return ATTNRES_ERR_CUDA;
}

// Shared checks on T and d.
attnres_status check_shape(int64_t T, int d) {
  if (T < 0 || d <= 0) return ATTNRES_ERR_INVALID_ARG;
  if (d % 8 != 0) return ATTNRES_ERR_INVALID_ARG;
  if (d > ATTNRES_MAX_D) return ATTNRES_ERR_UNSUPPORTED;
  if (T > INT32_MAX) return ATTNRES_ERR_UNSUPPORTED;  // one CTA (or tile) per row in x
  return ATTNRES_OK;
}

// Depth-attention heads: d splits into `heads` slices whose width is a multiple of 8.
attnres_status check_heads(int d, int heads) {
  if (heads < 1) return ATTNRES_ERR_INVALID_ARG;
  if (heads > ATTNRES_MAX_HEADS) return ATTNRES_ERR_UNSUPPORTED;
  if (d % heads != 0 || (d / heads) % 8 != 0) return ATTNRES_ERR_INVALID_ARG;
  return ATTNRES_OK;
}

}  // namespace

extern "C" {

int attnres_abi_version(void) { return ATTNRES_ABI_VERSION; }

const char* attnres_status_string(attnres_status s) {
  switch (s) {
    case ATTNRES_OK: return "ATTNRES_OK";
    case ATTNRES_ERR_INVALID_ARG: return "ATTNRES_ERR_INVALID_ARG";
    case ATTNRES_ERR_UNSUPPORTED: return "ATTNRES_ERR_UNSUPPORTED";
    case ATTNRES_ERR_MISALIGNED: return "ATTNRES_ERR_MISALIGNED";
    case ATTNRES_ERR_CUDA: return "ATTNRES_ERR_CUDA";
    case ATTNRES_ERR_TIMEOUT: return "ATTNRES_ERR_TIMEOUT";
  }
  return "ATTNRES_ERR_UNKNOWN";
}

const char* attnres_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

attnres_status attnres_poll_device_errors(void) {
  const unsigned int n1 = attnres::phase1_poll_timeouts();
  const unsigned int n2 = attnres::phase1_tc_poll_timeouts();
  const unsigned int n3 = attnres::full_ring_poll_timeouts();
  const unsigned int n4 = attnres::backward_poll_timeouts();
  const unsigned int n =
      (n1 == 0xffffffffu || n2 == 0xffffffffu || n3 == 0xffffffffu || n4 == 0xffffffffu)
          ? 0xffffffffu
          : n1 + n2 + n3 + n4;
  if (n == 0xffffffffu) {
    g_last_cuda_error = "could not read the device wait-timeout counter";
    return ATTNRES_ERR_CUDA;
  }
  return n == 0 ? ATTNRES_OK : ATTNRES_ERR_TIMEOUT;
}

attnres_status attnres_selftest_wait_timeout(unsigned int polls, void* stream) {
  if (polls > (1u << 20)) return ATTNRES_ERR_INVALID_ARG;
  return cuda_status(attnres::launch_wait_selftest(polls, static_cast<cudaStream_t>(stream)));
}

attnres_status attnres_query_prep(const float* w, const float* gamma_key, float* u_out,
                                  void* u_split_out, int rows, int d, void* stream) {
  if (rows < 0) return ATTNRES_ERR_INVALID_ARG;
  const attnres_status sh = check_shape(rows, d);
  if (sh != ATTNRES_OK) return sh;
  if (rows == 0) return ATTNRES_OK;
  if (w == nullptr || u_out == nullptr) return ATTNRES_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(u_out) || !opt_aligned16(gamma_key) ||
      !opt_aligned16(u_split_out))
    return ATTNRES_ERR_MISALIGNED;
  return cuda_status(attnres::launch_query_prep(w, gamma_key, u_out, u_split_out, rows, d,
                                                static_cast<cudaStream_t>(stream)));
}

attnres_status attnres_phase1(const void* reps, int64_t src_stride, int n_src, int64_t T, int d,
                              attnres_dtype io, const float* u, const void* u_split, int S,
                              float eps, void* o_out, float* m_out, float* lse_out,
                              float* alpha_out, unsigned int flags, int heads, void* stream) {
  if (!valid_io(io) || !valid_o_flags(flags)) return ATTNRES_ERR_INVALID_ARG;
  attnres_status sh = check_shape(T, d);
  if (sh == ATTNRES_OK) sh = check_heads(d, heads);
  if (sh != ATTNRES_OK) return sh;
  if (n_src < 1 || S < 1 || !(eps >= 0.f)) return ATTNRES_ERR_INVALID_ARG;
  if (n_src > ATTNRES_MAX_SOURCES || S > ATTNRES_MAX_QUERIES) return ATTNRES_ERR_UNSUPPORTED;
  if (!attnres::phase1_supported(n_src, S)) return ATTNRES_ERR_UNSUPPORTED;
  if (T == 0) return ATTNRES_OK;
  if (reps == nullptr || u == nullptr || o_out == nullptr) return ATTNRES_ERR_INVALID_ARG;
  if (n_src > 1 && src_stride < T * d) return ATTNRES_ERR_INVALID_ARG;
  if (src_stride < 0) return ATTNRES_ERR_INVALID_ARG;
  if (!aligned16(reps) || !aligned16(u) || !aligned16(o_out) || !opt_aligned16(u_split) ||
      src_stride % 8 != 0)
    return ATTNRES_ERR_MISALIGNED;
  attnres::Phase1Args a{reps,  src_stride, n_src, T,      d,       u,        u_split,
                        S,     eps,        o_out, m_out, lse_out, alpha_out, flags, heads};
  return cuda_status(attnres::launch_phase1(static_cast<IO>(io), a,
                                            static_cast<cudaStream_t>(stream)));
}

attnres_status attnres_phase2_merge(const void* o_l, const float* lse_l, const void* partial,
                                    const void* v_prev, void* partial_out, int64_t T, int d,
                                    attnres_dtype io, const float* u_l, float eps_key,
                                    const float* gamma_in, float eps_in, void* h_out, void* y_out,
                                    float* alpha_p_out, unsigned int flags, int heads,
                                    void* stream) {
  if (!valid_io(io) || !valid_o_flags(flags)) return ATTNRES_ERR_INVALID_ARG;
  attnres_status sh = check_shape(T, d);
  if (sh == ATTNRES_OK) sh = check_heads(d, heads);
  if (sh != ATTNRES_OK) return sh;
  if (!(eps_key >= 0.f) || !(eps_in >= 0.f)) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (o_l == nullptr || y_out == nullptr) return ATTNRES_ERR_INVALID_ARG;
  const bool has_p = partial != nullptr || v_prev != nullptr;
  if (has_p && u_l == nullptr) return ATTNRES_ERR_INVALID_ARG;
  if (has_p && lse_l == nullptr && !(flags & ATTNRES_SIGMOID_WEIGHTS))
    return ATTNRES_ERR_INVALID_ARG;
  if (partial_out != nullptr && !has_p) return ATTNRES_ERR_INVALID_ARG;
  if (!(eps_key >= 0.f) || !(eps_in >= 0.f)) return ATTNRES_ERR_INVALID_ARG;
  if (!aligned16(o_l) || !aligned16(y_out) || !opt_aligned16(partial) || !opt_aligned16(v_prev) ||
      !opt_aligned16(partial_out) || !opt_aligned16(u_l) || !opt_aligned16(gamma_in) ||
      !opt_aligned16(h_out))
    return ATTNRES_ERR_MISALIGNED;
  attnres::Phase2Args a{o_l, lse_l, partial, v_prev, partial_out, T, d, u_l, eps_key, gamma_in,
                        eps_in, h_out, y_out, alpha_p_out, flags, heads};
  return cuda_status(attnres::launch_phase2(static_cast<IO>(io), a,
                                            static_cast<cudaStream_t>(stream)));
}

attnres_status attnres_partial_update(const void* partial, const void* v, void* out, int64_t T,
                                      int d, attnres_dtype io, void* stream) {
  if (!valid_io(io)) return ATTNRES_ERR_INVALID_ARG;
  const attnres_status sh = check_shape(T, d);
  if (sh != ATTNRES_OK) return sh;
  if (T == 0) return ATTNRES_OK;
  if (partial == nullptr || v == nullptr || out == nullptr) return ATTNRES_ERR_INVALID_ARG;
  if (!aligned16(partial) || !aligned16(v) || !aligned16(out)) return ATTNRES_ERR_MISALIGNED;
  return cuda_status(attnres::launch_partial_update(static_cast<IO>(io), partial, v, out, T * d,
                                                    static_cast<cudaStream_t>(stream)));
}

attnres_status attnres_full_reference_path(const void* const* srcs, int n_src, int64_t T, int d,
                                           attnres_dtype io, const float* u_l, float eps_key,
                                           const float* gamma_in, float eps_in, void* h_out,
                                           void* y_out, float* alpha_out, unsigned int flags,
                                           int heads, void* stream) {
  if (!valid_io(io) || !valid_flags(flags)) return ATTNRES_ERR_INVALID_ARG;
  attnres_status sh = check_shape(T, d);
  if (sh == ATTNRES_OK) sh = check_heads(d, heads);
  if (sh != ATTNRES_OK) return sh;
  if (n_src < 1) return ATTNRES_ERR_INVALID_ARG;
  if (n_src > ATTNRES_MAX_SOURCES) return ATTNRES_ERR_UNSUPPORTED;
  if (!(eps_key >= 0.f) || !(eps_in >= 0.f)) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (srcs == nullptr || u_l == nullptr) return ATTNRES_ERR_INVALID_ARG;
  if (h_out == nullptr && y_out == nullptr) return ATTNRES_ERR_INVALID_ARG;
  attnres::FullArgs a;
  memset(&a, 0, sizeof(a));
  for (int j = 0; j < n_src; ++j) {
    if (srcs[j] == nullptr) return ATTNRES_ERR_INVALID_ARG;
    if (!aligned16(srcs[j])) return ATTNRES_ERR_MISALIGNED;
    a.srcs[j] = srcs[j];
  }
  if (!aligned16(u_l) || !opt_aligned16(gamma_in) || !opt_aligned16(h_out) ||
      !opt_aligned16(y_out))
    return ATTNRES_ERR_MISALIGNED;
  a.n = n_src;
  a.T = T;
  a.d = d;
  a.u = u_l;
  a.eps_key = eps_key;
  a.gamma_in = gamma_in;
  a.eps_in = eps_in;
  a.h = h_out;
  a.y = y_out;
  a.alpha = alpha_out;
  a.flags = flags;
  a.heads = heads;
  return cuda_status(attnres::launch_full(static_cast<IO>(io), a,
                                          static_cast<cudaStream_t>(stream)));
}

attnres_status attnres_phase2_merge_sources(const void* o_l, const float* lse_l,
                                            const void* const* srcs, int k, int64_t T, int d,
                                            attnres_dtype io, const float* u_l, float eps_key,
                                            const float* gamma_in, float eps_in, void* h_out,
                                            void* y_out, float* alpha_out, unsigned int flags,
                                            int heads, void* stream) {
  if (!valid_io(io) || !valid_o_flags(flags)) return ATTNRES_ERR_INVALID_ARG;
  attnres_status sh = check_shape(T, d);
  if (sh == ATTNRES_OK) sh = check_heads(d, heads);
  if (sh != ATTNRES_OK) return sh;
  if (k < 0) return ATTNRES_ERR_INVALID_ARG;
  if (k > ATTNRES_MAX_SOURCES) return ATTNRES_ERR_UNSUPPORTED;
  if (!(eps_key >= 0.f) || !(eps_in >= 0.f)) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (o_l == nullptr || (h_out == nullptr && y_out == nullptr)) return ATTNRES_ERR_INVALID_ARG;
  if (lse_l == nullptr && !(flags & ATTNRES_SIGMOID_WEIGHTS)) return ATTNRES_ERR_INVALID_ARG;
  if (k > 0 && (srcs == nullptr || u_l == nullptr)) return ATTNRES_ERR_INVALID_ARG;
  attnres::FullArgs a;
  memset(&a, 0, sizeof(a));
  for (int j = 0; j < k; ++j) {
    if (srcs[j] == nullptr) return ATTNRES_ERR_INVALID_ARG;
    if (!aligned16(srcs[j])) return ATTNRES_ERR_MISALIGNED;
    a.srcs[j] = srcs[j];
  }
  if (!aligned16(o_l) || !opt_aligned16(u_l) || !opt_aligned16(gamma_in) ||
      !opt_aligned16(h_out) || !opt_aligned16(y_out))
    return ATTNRES_ERR_MISALIGNED;
  a.n = k;
  a.T = T;
  a.d = d;
  a.u = u_l;
  a.eps_key = eps_key;
  a.gamma_in = gamma_in;
  a.eps_in = eps_in;
  a.h = h_out;
  a.y = y_out;
  a.alpha = alpha_out;
  a.flags = flags;
  a.heads = heads;
  a.o0 = o_l;
  a.lse0 = lse_l;
  a.o0_f32 = io == ATTNRES_BF16 && (flags & ATTNRES_O_F32) != 0;
  return cuda_status(attnres::launch_full(static_cast<IO>(io), a,
                                          static_cast<cudaStream_t>(stream)));
}

attnres_status attnres_backward(const void* const* srcs, int n_src, int64_t T, int d,
                                attnres_dtype io, const float* u, float eps_key,
                                const float* gamma_in, float eps_in, const void* g_y,
                                void* const* dsrcs, float* du, float* dgamma_in, void* stream) {
  if (!valid_io(io)) return ATTNRES_ERR_INVALID_ARG;
  const attnres_status sh = check_shape(T, d);
  if (sh != ATTNRES_OK) return sh;
  if (n_src < 1) return ATTNRES_ERR_INVALID_ARG;
  if (n_src > attnres::kBwdMaxSources) return ATTNRES_ERR_UNSUPPORTED;
  if (d / (io == ATTNRES_BF16 ? 8 : 4) > attnres::kBwdMaxVectors) return ATTNRES_ERR_UNSUPPORTED;
  if (!(eps_key >= 0.f) || !(eps_in >= 0.f)) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (srcs == nullptr || dsrcs == nullptr || u == nullptr || g_y == nullptr || du == nullptr)
    return ATTNRES_ERR_INVALID_ARG;
  attnres::BwdArgs a;
  memset(&a, 0, sizeof(a));
  for (int j = 0; j < n_src; ++j) {
    if (srcs[j] == nullptr || dsrcs[j] == nullptr) return ATTNRES_ERR_INVALID_ARG;
    if (!aligned16(srcs[j]) || !aligned16(dsrcs[j])) return ATTNRES_ERR_MISALIGNED;
    a.srcs[j] = srcs[j];
    a.dsrcs[j] = dsrcs[j];
  }
  if (!aligned16(u) || !aligned16(g_y) || !opt_aligned16(gamma_in) || !aligned16(du) ||
      !opt_aligned16(dgamma_in))
    return ATTNRES_ERR_MISALIGNED;
  a.n = n_src;
  a.T = T;
  a.d = d;
  a.u = u;
  a.eps_key = eps_key;
  a.gamma_in = gamma_in;
  a.eps_in = eps_in;
  a.g_y = g_y;
  a.du = du;
  a.dgamma_in = dgamma_in;
  return cuda_status(attnres::launch_backward(static_cast<IO>(io), a,
                                              static_cast<cudaStream_t>(stream)));
}

attnres_status attnres_backward_block_workspace_size(int n_src, int S, int64_t T, int d,
                                                     attnres_dtype io, uint64_t* bytes) {
  if (!valid_io(io) || bytes == nullptr) return ATTNRES_ERR_INVALID_ARG;
  const attnres_status sh = check_shape(T, d);
  if (sh != ATTNRES_OK) return sh;
  if (n_src < 1 || S < 1) return ATTNRES_ERR_INVALID_ARG;
  if (!attnres::backward_block_supported(static_cast<IO>(io), n_src, S, d))
    return ATTNRES_ERR_UNSUPPORTED;
  *bytes = static_cast<uint64_t>(
      attnres::backward_block_workspace_bytes(static_cast<IO>(io), n_src, S, T, d));
  return ATTNRES_OK;
}

attnres_status attnres_backward_block(const void* reps, int64_t src_stride, int n_src,
                                      const void* v, int64_t v_stride, int S, int64_t T, int d,
                                      attnres_dtype io, const float* u, const void* u_split,
                                      float eps_key, const float* gamma_in, float eps_in,
                                      const void* g_y, void* d_reps, void* d_v,
                                      int64_t dv_stride, float* du, float* dgamma_in,
                                      void* workspace, uint64_t workspace_bytes, void* stream) {
  uint64_t need = 0;
  const attnres_status st = attnres_backward_block_workspace_size(n_src, S, T, d, io, &need);
  if (st != ATTNRES_OK) return st;
  if (!(eps_key >= 0.f) || !(eps_in >= 0.f)) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (reps == nullptr || u == nullptr || g_y == nullptr || d_reps == nullptr || du == nullptr ||
      workspace == nullptr)
    return ATTNRES_ERR_INVALID_ARG;
  if (S > 1 && (v == nullptr || d_v == nullptr)) return ATTNRES_ERR_INVALID_ARG;
  if (workspace_bytes < need) return ATTNRES_ERR_INVALID_ARG;
  if (n_src > 1 && src_stride < T * d) return ATTNRES_ERR_INVALID_ARG;
  if (S > 2 && (v_stride < T * d || dv_stride < T * d)) return ATTNRES_ERR_INVALID_ARG;
  if (src_stride < 0 || v_stride < 0 || dv_stride < 0) return ATTNRES_ERR_INVALID_ARG;
  if (!aligned16(reps) || !aligned16(u) || !aligned16(g_y) || !aligned16(d_reps) ||
      !aligned16(du) || !opt_aligned16(v) || !opt_aligned16(d_v) || !opt_aligned16(u_split) ||
      !opt_aligned16(gamma_in) || !opt_aligned16(dgamma_in) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || src_stride % 8 != 0 ||
      v_stride % 8 != 0 || dv_stride % 8 != 0)
    return ATTNRES_ERR_MISALIGNED;
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
  return cuda_status(attnres::launch_backward_block(static_cast<IO>(io), a, workspace,
                                                    static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
