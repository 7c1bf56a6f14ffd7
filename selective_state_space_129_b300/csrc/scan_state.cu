// Entering state of a prefill that continues a sequence.
//
// The recurrence (Prop. 1, sec. 4.1 of
// "MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc)) carries, besides the state
// h_{-1}, the previous token's B_{-1} x_{-1}^T into the first token through
// its beta term: h_0 = alpha_0 R_0 (h_{-1} + beta_hat_0 B_{-1} x_{-1}^T) +
// gamma_0 B_0 x_0^T. Both prefill kernels take the state entering their first
// chunk in the explicit frame with that pending term included, so a
// continuation first forms, in place,
//   state[b,h] += beta_hat_0 (B_prev + B_bias[h]) x_prev^T,
//   beta_hat_0 = (1 - lambda[b,0,h]) dt[b,0,h].
// One thread per state element; the call is HBM-bound (the state read and
// written once) and runs once per prefill call.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace m3 {
namespace {

template <typename T, int R>
__global__ void __launch_bounds__(256)
    entry_state_kernel(float* __restrict__ state, const T* __restrict__ Bp,
                       const T* __restrict__ xp, const float* __restrict__ dt,
                       const float* __restrict__ lam, const float* __restrict__ B_bias,
                       int64_t total, int64_t L, int64_t H, int64_t G, int P, int N) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t bh = i / ((int64_t)N * P);
  const int n = (int)((i / P) % N), p = (int)(i % P);
  const int64_t b = bh / H, h = bh % H, g = h / (H / G);
  const float bhat = (1.f - lam[b * L * H + h]) * dt[b * L * H + h];
  const T* brow = Bp + ((b * G + g) * N + n) * R;
  const T* xrow = xp + (bh * P + p) * R;
  float acc = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float bb = B_bias ? B_bias[(h * N + n) * R + r] : 0.f;
    acc = fmaf(ld_act(brow + r) + bb, ld_act(xrow + r), acc);
  }
  state[i] = fmaf(bhat, acc, state[i]);
}

template <typename T>
cudaError_t launch_t(float* state, const void* B_prev, const void* x_prev, const float* dt,
                     const float* lam, const float* B_bias, int64_t batch, int64_t L, int64_t H,
                     int64_t G, int64_t P, int64_t N, int R, cudaStream_t s) {
  const int64_t total = batch * H * N * P;
  const unsigned grid = (unsigned)((total + 255) / 256);
  const T* Bp = static_cast<const T*>(B_prev);
  const T* xp = static_cast<const T*>(x_prev);
  switch (R) {
#define M3_ENTRY(RR)                                                                      \
  case RR:                                                                                \
    entry_state_kernel<T, RR><<<grid, 256, 0, s>>>(state, Bp, xp, dt, lam, B_bias, total, L, \
                                                   H, G, (int)P, (int)N);                 \
    break;
    M3_ENTRY(1)
    M3_ENTRY(2)
    M3_ENTRY(4)
#undef M3_ENTRY
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_entry_state(float* state, const void* B_prev, const void* x_prev,
                               const float* dt, const float* lam, const float* B_bias,
                               int64_t batch, int64_t L, int64_t H, int64_t G, int64_t P,
                               int64_t N, int R, bool bf16, cudaStream_t s) {
  if (batch * H * N * P == 0) return cudaSuccess;
  return bf16 ? launch_t<__nv_bfloat16>(state, B_prev, x_prev, dt, lam, B_bias, batch, L, H, G, P,
                                        N, R, s)
              : launch_t<float>(state, B_prev, x_prev, dt, lam, B_bias, batch, L, H, G, P, N, R, s);
}

}  // namespace m3
