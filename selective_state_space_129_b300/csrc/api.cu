// C ABI of libm3scan.so: argument validation and kernel dispatch.
// The declarations, layouts and error behaviour are documented in m3scan.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "launch.h"
#include "m3scan.h"

namespace {

constexpr int64_t kMaxElems = int64_t(1) << 40;

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > kMaxElems / a) return false;
  *out = a * b;
  return true;
}

bool count(std::initializer_list<int64_t> dims, int64_t* out) {
  int64_t c = 1;
  for (int64_t d : dims)
    if (!mul_ok(c, d, &c)) return false;
  *out = c;
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A pointer may be NULL only when the tensor it points to is empty.
bool ptr_ok(const void* p, int64_t elems, size_t align) {
  if (elems == 0) return true;
  return p != nullptr && aligned(p, align);
}

m3_status check_dims(const m3_dims* d, int R) {
  if (d == nullptr) return M3_ERR_INVALID_ARG;
  if (d->batch < 0 || d->heads < 1 || d->groups < 1 || d->headdim < 1 || d->dstate < 2)
    return M3_ERR_INVALID_ARG;
  if (d->dstate % 2 != 0 || d->heads % d->groups != 0) return M3_ERR_INVALID_ARG;
  if ((d->flags & ~M3_FLAG_BC_NORM) != 0 || R < 1) return M3_ERR_INVALID_ARG;
  if (d->act_dtype != M3_F32 && d->act_dtype != M3_BF16) return M3_ERR_UNSUPPORTED;
  if (d->heads > (1 << 20) || d->headdim > (1 << 20) || d->dstate > (1 << 20) || R > 1024)
    return M3_ERR_UNSUPPORTED;
  return M3_OK;
}

m3_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return M3_ERR_CUDA;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return M3_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return M3_ERR_UNSUPPORTED;
  return M3_OK;
}

m3_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return M3_OK;
  cudaGetLastError();
  return M3_ERR_CUDA;
}

// Fault injection, for tests of the error paths, from the environment
// variable M3_FAULT (read at every call; unset or any other value: none):
//   arg      every valid compute call returns M3_ERR_INVALID_ARG before any
//            device work;
//   launch   the call returns M3_ERR_CUDA in place of its launches;
//   alloc    the library's own scratch allocation (a segmented prefill
//            without a caller workspace) fails: M3_ERR_CUDA before any launch;
//   timeout  the work is replaced by a kernel whose bounded device wait runs
//            out (1 ms), so that m3_device_status reports M3_ERR_TIMEOUT.
// In every mode the call's outputs (and a decode's state) are left untouched.
enum class Fault { kNone, kArg, kLaunch, kAlloc, kTimeout };

Fault fault_mode() {
  const char* v = getenv("M3_FAULT");
  if (v == nullptr) return Fault::kNone;
  if (strcmp(v, "arg") == 0) return Fault::kArg;
  if (strcmp(v, "launch") == 0) return Fault::kLaunch;
  if (strcmp(v, "alloc") == 0) return Fault::kAlloc;
  if (strcmp(v, "timeout") == 0) return Fault::kTimeout;
  return Fault::kNone;
}

constexpr uint64_t kInjectedWaitNs = 1000000ull;  // 1 ms

// The launch-time faults: M3_OK to go on with the real work, else the status
// to return (the timeout fault has launched its expiring wait by then).
m3_status injected_launch_fault(Fault f, cudaStream_t s) {
  if (f == Fault::kLaunch) return M3_ERR_CUDA;
  if (f == Fault::kTimeout) {
    const m3_status st = from_cuda(m3::launch_expired_wait(kInjectedWaitNs, s));
    return st == M3_OK ? M3_ERR_TIMEOUT : st;
  }
  return M3_OK;
}

}  // namespace

extern "C" {

int m3_version(void) { return 200; }  // 0.2.0: m3_decode_tokens, m3_scan_fwd_state

const char* m3_status_string(m3_status s) {
  switch (s) {
    case M3_OK: return "M3_OK";
    case M3_ERR_INVALID_ARG: return "M3_ERR_INVALID_ARG";
    case M3_ERR_UNSUPPORTED: return "M3_ERR_UNSUPPORTED";
    case M3_ERR_CUDA: return "M3_ERR_CUDA";
    case M3_ERR_TIMEOUT: return "M3_ERR_TIMEOUT";
  }
  return "M3_ERR_UNKNOWN";
}

size_t m3_scan_bwd_workspace_bytes(const m3_dims* dims, int R) {
  if (check_dims(dims, R) == M3_ERR_INVALID_ARG || dims->seqlen < 0) return (size_t)-1;
  m3::BwdArgs a = {};
  a.batch = dims->batch; a.L = dims->seqlen; a.H = dims->heads; a.G = dims->groups;
  a.P = dims->headdim; a.N = dims->dstate; a.R = R;
  return m3::scan_bwd_workspace_bytes(a, dims->act_dtype == M3_BF16);
}

size_t m3_scan_workspace_bytes(const m3_dims* dims, int R, int chunk) {
  if (check_dims(dims, R) == M3_ERR_INVALID_ARG || chunk < 1 || dims->seqlen < 0)
    return (size_t)-1;
  m3::ScanArgs a = {};
  a.batch = dims->batch; a.L = dims->seqlen; a.H = dims->heads; a.G = dims->groups;
  a.P = dims->headdim; a.N = dims->dstate; a.R = R; a.Q = chunk;
  if (a.L == 0 || a.batch == 0) return 0;
  return m3::scan_tc_workspace_bytes(a);
}

}  // extern "C"

namespace {

// Prefill from a given entering state (continuation) or from zero. With
// `state` (the m3_scan_fwd_state form) final_state is `state` itself: it is
// read as the entering state, has the pending beta term of B_prev / x_prev
// added first, and receives the state after the block.
m3_status scan_impl(const void* x, const float* dt, const float* A, const float* lambda,
                    const void* B, const void* C, const float* theta, const m3_dims* dims, int R,
                    int chunk, void* out, float* final_state, bool continue_state,
                    const void* B_prev, const void* x_prev, void* stream) {
  m3_status st = check_dims(dims, R);
  if (st != M3_OK) return st;
  if (chunk < 1 || dims->seqlen < 0) return M3_ERR_INVALID_ARG;
  const int64_t b = dims->batch, L = dims->seqlen, H = dims->heads, G = dims->groups,
                P = dims->headdim, N = dims->dstate;
  const size_t act = dims->act_dtype == M3_BF16 ? 2 : 4;
  int64_t n_x, n_t, n_bc, n_th, n_st, n_bias;
  if (!count({b, L, H, P, R}, &n_x) || !count({b, L, H}, &n_t) ||
      !count({b, L, G, N, R}, &n_bc) || !count({b, L, G, N / 2}, &n_th) ||
      !count({b, H, N, P}, &n_st) || !count({H, N, R}, &n_bias))
    return M3_ERR_INVALID_ARG;
  if (!ptr_ok(x, n_x, act) || !ptr_ok(out, n_x, act) || !ptr_ok(dt, n_t, 4) ||
      !ptr_ok(lambda, n_t, 4) || !ptr_ok(A, H, 4) || !ptr_ok(B, n_bc, act) ||
      !ptr_ok(C, n_bc, act) || !ptr_ok(theta, n_th, 4))
    return M3_ERR_INVALID_ARG;
  if (final_state && !aligned(final_state, 4)) return M3_ERR_INVALID_ARG;
  if ((dims->B_bias && !aligned(dims->B_bias, 4)) || (dims->C_bias && !aligned(dims->C_bias, 4)))
    return M3_ERR_INVALID_ARG;
  if (continue_state) {
    int64_t n_bp, n_xp;
    if (!count({b, G, N, R}, &n_bp) || !count({b, H, P, R}, &n_xp)) return M3_ERR_INVALID_ARG;
    if (!ptr_ok(final_state, n_st, 4)) return M3_ERR_INVALID_ARG;
    if ((B_prev == nullptr) != (x_prev == nullptr)) return M3_ERR_INVALID_ARG;
    if (B_prev && (!ptr_ok(B_prev, n_bp, act) || !ptr_ok(x_prev, n_xp, act)))
      return M3_ERR_INVALID_ARG;
    if (!(R == 1 || R == 2 || R == 4)) return M3_ERR_UNSUPPORTED;
  }
  if ((int64_t)chunk * R > 4096 || chunk > 4096) return M3_ERR_UNSUPPORTED;

  const bool bf16 = dims->act_dtype == M3_BF16;
  // The tensor-core path moves tiles with TMA and 128-bit accesses: it takes
  // 16-byte-aligned activations, biases and final state and 8-byte-aligned
  // theta; other calls use the CUDA cores.
  // (fp32 activations take the split-fp16 tensor-core mode when the shape and
  // alignment allow, with the same conditions)
  const bool use_tc = m3::scan_tc_supported(N, P, R, chunk) && aligned(x, 16) &&
                      aligned(out, 16) && aligned(B, 16) && aligned(C, 16) &&
                      aligned(theta, 8) &&
                      (dims->B_bias == nullptr || aligned(dims->B_bias, 16)) &&
                      (dims->C_bias == nullptr || aligned(dims->C_bias, 16)) &&
                      (final_state == nullptr || aligned(final_state, 16));
  const bool bc_norm = (dims->flags & M3_FLAG_BC_NORM) != 0;
  if (bc_norm && (!use_tc || !bf16 || continue_state)) return M3_ERR_UNSUPPORTED;
  if (!use_tc) {
    const size_t smem = m3::scan_simt_smem_bytes(N, P, R, chunk);
    if (smem > 227 * 1024) return M3_ERR_UNSUPPORTED;
  }
  if (b * H > 0x7fffffff) return M3_ERR_UNSUPPORTED;
  const Fault fault = fault_mode();
  if (fault == Fault::kArg) return M3_ERR_INVALID_ARG;

  st = check_device();
  if (st != M3_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n_st == 0) return M3_OK;
  {
    const m3_status f = injected_launch_fault(fault, s);
    if (f == M3_ERR_TIMEOUT) return M3_OK;  // reported by m3_device_status
    if (f != M3_OK) return f;
  }
  if (L == 0) {
    if (continue_state) return M3_OK;  // no token: the state stays as it is
    if (final_state)
      return from_cuda(cudaMemsetAsync(final_state, 0, sizeof(float) * (size_t)n_st, s));
    return M3_OK;
  }
  if (fault == Fault::kAlloc && use_tc && dims->workspace == nullptr) {
    m3::ScanArgs q = {};
    q.batch = b; q.L = L; q.H = H; q.G = G; q.P = P; q.N = N; q.R = R; q.Q = chunk;
    if (m3::scan_tc_workspace_bytes(q) > 0) return M3_ERR_CUDA;  // the allocation "failed"
  }
  if (continue_state && B_prev) {
    st = from_cuda(m3::launch_entry_state(final_state, B_prev, x_prev, dt, lambda, dims->B_bias,
                                          b, L, H, G, P, N, R, bf16, s));
    if (st != M3_OK) return st;
  }
  m3::ScanArgs a;
  a.x = x; a.dt = dt; a.A = A; a.lam = lambda; a.B = B; a.C = C; a.theta = theta;
  a.B_bias = dims->B_bias; a.C_bias = dims->C_bias; a.out = out; a.final_state = final_state;
  a.h_init = continue_state ? final_state : nullptr;
  a.workspace = dims->workspace; a.workspace_bytes = dims->workspace_bytes;
  a.batch = b; a.L = L; a.H = H; a.G = G; a.P = P; a.N = N; a.R = R; a.Q = chunk;
  a.bc_norm = bc_norm;
  a.f32 = !bf16;
  if (use_tc) {
    // a caller-provided workspace must be large enough; NULL means the
    // library allocates (stream-ordered) what it needs
    if (dims->workspace != nullptr) {
      if (!aligned(dims->workspace, 16)) return M3_ERR_INVALID_ARG;
      if (dims->workspace_bytes < m3::scan_tc_workspace_bytes(a)) return M3_ERR_INVALID_ARG;
    }
    unsigned int* status = nullptr;
    st = from_cuda(m3::status_word(&status));
    if (st != M3_OK) return st;
    return from_cuda(m3::launch_scan_tc(a, status, s));
  }
  return from_cuda(m3::launch_scan_simt(a, bf16, s));
}

}  // namespace

extern "C" {

m3_status m3_scan_fwd(const void* x, const float* dt, const float* A, const float* lambda,
                      const void* B, const void* C, const float* theta, const m3_dims* dims,
                      int R, int chunk, void* out, float* final_state, void* stream) {
  return scan_impl(x, dt, A, lambda, B, C, theta, dims, R, chunk, out, final_state, false,
                   nullptr, nullptr, stream);
}

m3_status m3_scan_fwd_state(const void* x, const float* dt, const float* A, const float* lambda,
                            const void* B, const void* C, const float* theta,
                            const void* B_prev, const void* x_prev, const m3_dims* dims, int R,
                            int chunk, void* out, float* state, void* stream) {
  return scan_impl(x, dt, A, lambda, B, C, theta, dims, R, chunk, out, state, true, B_prev,
                   x_prev, stream);
}

m3_status m3_decode_step(float* state, const void* x, const float* dt, const float* A,
                         const float* lambda, const void* B_prev, const void* x_prev,
                         const void* B, const void* C, const float* theta, const m3_dims* dims,
                         int R, void* out, void* stream) {
  m3_status st = check_dims(dims, R);
  if (st != M3_OK) return st;
  if (dims->flags & M3_FLAG_BC_NORM) return M3_ERR_UNSUPPORTED;
  if ((B_prev == nullptr) != (x_prev == nullptr)) return M3_ERR_INVALID_ARG;
  const int64_t b = dims->batch, H = dims->heads, G = dims->groups, P = dims->headdim,
                N = dims->dstate;
  const size_t act = dims->act_dtype == M3_BF16 ? 2 : 4;
  int64_t n_x, n_t, n_bc, n_th, n_st;
  if (!count({b, H, P, R}, &n_x) || !count({b, H}, &n_t) || !count({b, G, N, R}, &n_bc) ||
      !count({b, G, N / 2}, &n_th) || !count({b, H, N, P}, &n_st))
    return M3_ERR_INVALID_ARG;
  if (!ptr_ok(state, n_st, 16) || !ptr_ok(x, n_x, act) || !ptr_ok(out, n_x, act) ||
      !ptr_ok(dt, n_t, 4) || !ptr_ok(lambda, n_t, 4) || !ptr_ok(A, H, 4) ||
      !ptr_ok(B, n_bc, act) || !ptr_ok(C, n_bc, act) || !ptr_ok(theta, n_th, 4))
    return M3_ERR_INVALID_ARG;
  if (B_prev && (!ptr_ok(B_prev, n_bc, act) || !ptr_ok(x_prev, n_x, act)))
    return M3_ERR_INVALID_ARG;
  if ((dims->B_bias && !aligned(dims->B_bias, 4)) || (dims->C_bias && !aligned(dims->C_bias, 4)))
    return M3_ERR_INVALID_ARG;
  if (!m3::decode_supported(N, P, R)) return M3_ERR_UNSUPPORTED;
  if (b * H > 0x7fffffff) return M3_ERR_UNSUPPORTED;
  const Fault fault = fault_mode();
  if (fault == Fault::kArg) return M3_ERR_INVALID_ARG;

  st = check_device();
  if (st != M3_OK) return st;
  if (n_st == 0) return M3_OK;
  {
    const m3_status f = injected_launch_fault(fault, static_cast<cudaStream_t>(stream));
    if (f == M3_ERR_TIMEOUT) return M3_OK;
    if (f != M3_OK) return f;
  }
  m3::DecodeArgs a;
  a.state = state; a.x = x; a.dt = dt; a.A = A; a.lam = lambda; a.B_prev = B_prev;
  a.x_prev = x_prev; a.B = B; a.C = C; a.theta = theta; a.B_bias = dims->B_bias;
  a.C_bias = dims->C_bias; a.out = out; a.batch = b; a.H = H; a.G = G; a.P = P; a.N = N; a.R = R;
  a.status = nullptr;
  st = from_cuda(m3::status_word(&a.status));
  if (st != M3_OK) return st;
  return from_cuda(m3::launch_decode(a, dims->act_dtype == M3_BF16,
                                     static_cast<cudaStream_t>(stream)));
}

m3_status m3_decode_tokens(float* state, const void* x, const float* dt, const float* A,
                           const float* lambda, const void* B_prev, const void* x_prev,
                           const void* B, const void* C, const float* theta,
                           const m3_dims* dims, int R, void* out, void* stream) {
  m3_status st = check_dims(dims, R);
  if (st != M3_OK) return st;
  if (dims->flags & M3_FLAG_BC_NORM) return M3_ERR_UNSUPPORTED;
  if (dims->seqlen < 0) return M3_ERR_INVALID_ARG;
  if ((B_prev == nullptr) != (x_prev == nullptr)) return M3_ERR_INVALID_ARG;
  const int64_t b = dims->batch, K = dims->seqlen, H = dims->heads, G = dims->groups,
                P = dims->headdim, N = dims->dstate;
  const size_t act = dims->act_dtype == M3_BF16 ? 2 : 4;
  int64_t n_x, n_t, n_bc, n_th, n_st, n_xp, n_bp;
  if (!count({b, K, H, P, R}, &n_x) || !count({b, K, H}, &n_t) || !count({b, K, G, N, R}, &n_bc) ||
      !count({b, K, G, N / 2}, &n_th) || !count({b, H, N, P}, &n_st) ||
      !count({b, H, P, R}, &n_xp) || !count({b, G, N, R}, &n_bp))
    return M3_ERR_INVALID_ARG;
  if (!ptr_ok(state, n_st, 16) || !ptr_ok(x, n_x, act) || !ptr_ok(out, n_x, act) ||
      !ptr_ok(dt, n_t, 4) || !ptr_ok(lambda, n_t, 4) || !ptr_ok(A, H, 4) ||
      !ptr_ok(B, n_bc, act) || !ptr_ok(C, n_bc, act) || !ptr_ok(theta, n_th, 4))
    return M3_ERR_INVALID_ARG;
  if (B_prev && (!ptr_ok(B_prev, n_bp, act) || !ptr_ok(x_prev, n_xp, act)))
    return M3_ERR_INVALID_ARG;
  if ((dims->B_bias && !aligned(dims->B_bias, 4)) || (dims->C_bias && !aligned(dims->C_bias, 4)))
    return M3_ERR_INVALID_ARG;
  m3::TokensArgs a;
  a.state = state; a.x = x; a.dt = dt; a.A = A; a.lam = lambda; a.B_prev = B_prev;
  a.x_prev = x_prev; a.B = B; a.C = C; a.theta = theta; a.B_bias = dims->B_bias;
  a.C_bias = dims->C_bias; a.out = out; a.status = nullptr; a.batch = b; a.K = K; a.H = H;
  a.G = G; a.P = P; a.N = N; a.R = R;
  // the kernel moves every per-token block with 16-byte vectors
  const void* vec[] = {x, B, C, theta, B_prev, x_prev, dims->B_bias, dims->C_bias};
  for (const void* p : vec)
    if (p != nullptr && !aligned(p, 16)) return M3_ERR_UNSUPPORTED;
  if (K == 0 || n_st == 0) return M3_OK;  // nothing to compute
  if (!m3::tokens_supported(a, (int)act)) return M3_ERR_UNSUPPORTED;
  if (b * H > 0x7fffffff) return M3_ERR_UNSUPPORTED;
  const Fault fault = fault_mode();
  if (fault == Fault::kArg) return M3_ERR_INVALID_ARG;

  st = check_device();
  if (st != M3_OK) return st;
  {
    const m3_status f = injected_launch_fault(fault, static_cast<cudaStream_t>(stream));
    if (f == M3_ERR_TIMEOUT) return M3_OK;
    if (f != M3_OK) return f;
  }
  a.status = nullptr;
  st = from_cuda(m3::status_word(&a.status));
  if (st != M3_OK) return st;
  return from_cuda(m3::launch_decode_tokens(a, dims->act_dtype == M3_BF16,
                                            static_cast<cudaStream_t>(stream)));
}

m3_status m3_scan_bwd(const void* x, const float* dt, const float* A, const float* lambda,
                      const void* B, const void* C, const float* theta, const void* dy,
                      const float* d_final, const m3_dims* dims, int R, float* dx, float* ddt,
                      float* dA, float* dlambda, float* dB, float* dC, float* dtheta,
                      float* dB_bias, float* dC_bias, void* stream) {
  m3_status st = check_dims(dims, R);
  if (st != M3_OK) return st;
  if (dims->flags & M3_FLAG_BC_NORM) return M3_ERR_UNSUPPORTED;
  if (dims->seqlen < 0) return M3_ERR_INVALID_ARG;
  const int64_t b = dims->batch, L = dims->seqlen, H = dims->heads, G = dims->groups,
                P = dims->headdim, N = dims->dstate;
  const size_t act = dims->act_dtype == M3_BF16 ? 2 : 4;
  int64_t n_x, n_t, n_bc, n_th, n_st, n_bias;
  if (!count({b, L, H, P, R}, &n_x) || !count({b, L, H}, &n_t) ||
      !count({b, L, G, N, R}, &n_bc) || !count({b, L, G, N / 2}, &n_th) ||
      !count({b, H, N, P}, &n_st) || !count({H, N, R}, &n_bias))
    return M3_ERR_INVALID_ARG;
  if (!ptr_ok(x, n_x, act) || !ptr_ok(dy, n_x, act) || !ptr_ok(dt, n_t, 4) ||
      !ptr_ok(lambda, n_t, 4) || !ptr_ok(A, H, 4) || !ptr_ok(B, n_bc, act) ||
      !ptr_ok(C, n_bc, act) || !ptr_ok(theta, n_th, 4) || !ptr_ok(dx, n_x, 4) ||
      !ptr_ok(ddt, n_t, 4) || !ptr_ok(dlambda, n_t, 4) || !ptr_ok(dA, H, 4) ||
      !ptr_ok(dB, n_bc, 4) || !ptr_ok(dC, n_bc, 4) || !ptr_ok(dtheta, n_th, 4))
    return M3_ERR_INVALID_ARG;
  if ((d_final && !aligned(d_final, 16)) || (dB_bias && !aligned(dB_bias, 4)) ||
      (dC_bias && !aligned(dC_bias, 4)))
    return M3_ERR_INVALID_ARG;
  if ((dims->B_bias && !aligned(dims->B_bias, 4)) || (dims->C_bias && !aligned(dims->C_bias, 4)))
    return M3_ERR_INVALID_ARG;
  if (!m3::scan_bwd_supported(N, P, R)) return M3_ERR_UNSUPPORTED;
  if (b * H > 0x7fffffff) return M3_ERR_UNSUPPORTED;
  m3::BwdArgs a;
  a.x = x; a.dt = dt; a.A = A; a.lam = lambda; a.B = B; a.C = C; a.theta = theta;
  a.B_bias = dims->B_bias; a.C_bias = dims->C_bias; a.dy = dy; a.d_final = d_final;
  a.dx = dx; a.ddt = ddt; a.dA = dA; a.dlam = dlambda; a.dB = dB; a.dC = dC; a.dtheta = dtheta;
  a.dB_bias = dB_bias; a.dC_bias = dC_bias;
  a.batch = b; a.L = L; a.H = H; a.G = G; a.P = P; a.N = N; a.R = R;
  const bool bf16 = dims->act_dtype == M3_BF16;
  if (dims->workspace != nullptr &&
      (!aligned(dims->workspace, 16) ||
       dims->workspace_bytes < m3::scan_bwd_workspace_bytes(a, bf16)))
    return M3_ERR_INVALID_ARG;
  const Fault fault = fault_mode();
  if (fault == Fault::kArg) return M3_ERR_INVALID_ARG;

  st = check_device();
  if (st != M3_OK) return st;
  {
    const m3_status f = injected_launch_fault(fault, static_cast<cudaStream_t>(stream));
    if (f == M3_ERR_TIMEOUT) return M3_OK;
    if (f != M3_OK) return f;
  }
  return from_cuda(m3::launch_scan_bwd(a, bf16, dims->workspace,
                                       static_cast<cudaStream_t>(stream)));
}

m3_status m3_device_status(void* stream) {
  unsigned int v = 0;
  if (m3::read_clear_status(&v, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return M3_ERR_CUDA;
  }
  return v ? M3_ERR_TIMEOUT : M3_OK;
}

}  // extern "C"
