// One decode token of the Mamba-3 scan, state streamed once.
//
// For every (batch, head):
//   G   = h + beta_hat (B_prev + bias) x_prev^T
//   h' = alpha Rot(Delta theta) G + gamma (B + bias) x^T
//   y   = (C + bias)^T h'                                   (P x R, stored [P][R])
// which is the recurrence of Prop. 1 (aipaper.cc sec. 4.1) with the state
// rotation of the complex-valued SSM (sec. 4.2; rotation matrix from the
// metaphor-xennon blog sec. 2.2), MIMO rank R (papernotes.org sec. 3).
//
// The step is bound by HBM traffic: the fp32 state (N x P per head) is read
// and written once, everything else is a few KB per head. The rank-R
// products are formed on the CUDA cores in registers while the state streams;
// at R <= 4 they are a handful of FMAs per state element, far below the FMA
// roof, so moving them to the tensor pipe would not shorten the step.
//
// Layout of work: one CTA per (batch, head), 256 threads. A work item is one
// rotating row pair (2k, 2k+1) times four consecutive columns, loaded as two
// 16-byte vectors, so that a warp reads 2 x 256 contiguous bytes per
// instruction. Each thread keeps a fixed column quad, so its x / x_prev values
// and its partial y stay in registers. The first items' state loads are issued
// before the per-head coefficients are prepared, so that they are in flight
// during that set-up; the partial y are reduced with warp shuffles and one
// shared-memory pass, without atomics.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace m3 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 4;  // items per thread per pass

// Shared memory: coefficient rows [N][R] (gamma B, beta_hat B_prev, C),
// rotation [N/2] (alpha cos, alpha sin), partial y [kWarps][P][R].
__host__ __device__ inline size_t decode_smem_floats(int N, int P, int R) {
  return (size_t)3 * N * R + N + (size_t)kWarps * P * R;
}

template <int R>
__device__ __forceinline__ void ld_row(const float* p, float (&v)[R]) {
  if constexpr (R == 4) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  } else if constexpr (R == 2) {
    const float2 q = *reinterpret_cast<const float2*>(p);
    v[0] = q.x; v[1] = q.y;
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = p[r];
  }
}

template <typename T, int R>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float sm[];
  const int N = (int)a.N, P = (int)a.P, K2 = N / 2, PQ = P / 4;
  const int64_t H = a.H, G = a.G;
  const int64_t bh = blockIdx.x, b = bh / H, h = bh % H, g = h / (H / G);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* bg = sm;              // gamma (B + bias)          [N][R]
  float* bp = bg + N * R;      // beta_hat (B_prev + bias)  [N][R]
  float* cc = bp + N * R;      // C + bias                  [N][R]
  float* rc = cc + N * R;      // alpha cos                 [K2]
  float* rs = rc + K2;         // alpha sin                 [K2]
  float* yred = rs + K2;       // partial y per warp        [kWarps][P][R]
  const T* x = static_cast<const T*>(a.x);
  const T* xprev = static_cast<const T*>(a.x_prev);
  const T* Bm = static_cast<const T*>(a.B);
  const T* Bprev = static_cast<const T*>(a.B_prev);
  const T* Cm = static_cast<const T*>(a.C);
  const bool has_prev = (Bprev != nullptr);
  float* st = a.state + bh * (int64_t)N * P;

  // this thread's column quad is fixed: PQ divides kThreads
  const int q = tid % PQ;
  const int items = K2 * PQ;

  // the token's B, C, B_prev (raw) first: they are small and needed first
  const float d = a.dt[b * H + h];
  const float lm = a.lam[b * H + h];
  const float A_h = a.A[h];
  const int64_t bc_base = (b * G + g) * (int64_t)N * R;
  constexpr int kPre = 4;  // coefficients per thread held in registers
  float rb[kPre], rp[kPre], rcv[kPre], rbb[kPre], rcb[kPre];
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const int i = tid + j * kThreads;
    rb[j] = rp[j] = rcv[j] = rbb[j] = rcb[j] = 0.f;
    if (i < N * R) {
      rb[j] = ld_act(Bm + bc_base + i);
      rp[j] = has_prev ? ld_act(Bprev + bc_base + i) : 0.f;
      rcv[j] = ld_act(Cm + bc_base + i);
      rbb[j] = a.B_bias ? a.B_bias[h * N * R + i] : 0.f;
      rcb[j] = a.C_bias ? a.C_bias[h * N * R + i] : 0.f;
    }
  }

  // the first pass's state, in flight while the coefficients are prepared
  float4 h0[kItems], h1[kItems];
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int it = tid + j * kThreads;
    if (it < items) {
      const int k = it / PQ;
      h0[j] = *reinterpret_cast<const float4*>(st + (2 * k) * P + 4 * q);
      h1[j] = *reinterpret_cast<const float4*>(st + (2 * k + 1) * P + 4 * q);
    }
  }

  const float alpha = expf(d * A_h);
  const float gamma = lm * d, bhat = (1.f - lm) * d;
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const int i = tid + j * kThreads;
    if (i < N * R) {
      bg[i] = gamma * (rb[j] + rbb[j]);
      bp[i] = has_prev ? bhat * (rp[j] + rbb[j]) : 0.f;
      cc[i] = rcv[j] + rcb[j];
    }
  }
  for (int i = tid + kPre * kThreads; i < N * R; i += kThreads) {
    const float bb = a.B_bias ? a.B_bias[h * N * R + i] : 0.f;
    const float cb = a.C_bias ? a.C_bias[h * N * R + i] : 0.f;
    bg[i] = gamma * (ld_act(Bm + bc_base + i) + bb);
    bp[i] = has_prev ? bhat * (ld_act(Bprev + bc_base + i) + bb) : 0.f;
    cc[i] = ld_act(Cm + bc_base + i) + cb;
  }
  // a warp holds partials only for the column quads of its lanes
  for (int i = tid; i < kWarps * P * R; i += kThreads) yred[i] = 0.f;
  for (int k = tid; k < K2; k += kThreads) {
    float sn, cs;
    sincosf(d * a.theta[(b * G + g) * K2 + k], &sn, &cs);
    rc[k] = alpha * cs;
    rs[k] = alpha * sn;
  }
  const int64_t x_base = bh * (int64_t)P * R;
  float xr[4][R], xpr[4][R];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      xr[c][r] = ld_act(x + x_base + (4 * q + c) * R + r);
      xpr[c][r] = has_prev ? ld_act(xprev + x_base + (4 * q + c) * R + r) : 0.f;
    }
  float yp[4][R];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int r = 0; r < R; ++r) yp[c][r] = 0.f;
  __syncthreads();

  for (int base = 0; base < items; base += kItems * kThreads) {
    if (base > 0) {
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int it = base + tid + j * kThreads;
        if (it < items) {
          const int k = it / PQ;
          h0[j] = *reinterpret_cast<const float4*>(st + (2 * k) * P + 4 * q);
          h1[j] = *reinterpret_cast<const float4*>(st + (2 * k + 1) * P + 4 * q);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      const int it = base + tid + j * kThreads;
      if (it < items) {
        const int k = it / PQ;
        float bp0[R], bp1[R], bg0[R], bg1[R], c0[R], c1[R];
        ld_row<R>(bp + (2 * k) * R, bp0);
        ld_row<R>(bp + (2 * k + 1) * R, bp1);
        ld_row<R>(bg + (2 * k) * R, bg0);
        ld_row<R>(bg + (2 * k + 1) * R, bg1);
        ld_row<R>(cc + (2 * k) * R, c0);
        ld_row<R>(cc + (2 * k + 1) * R, c1);
        const float ac = rc[k], as = rs[k];
        float* v0 = reinterpret_cast<float*>(&h0[j]);
        float* v1 = reinterpret_cast<float*>(&h1[j]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float g0 = v0[c], g1 = v1[c], u0 = 0.f, u1 = 0.f;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            g0 = fmaf(bp0[r], xpr[c][r], g0);
            g1 = fmaf(bp1[r], xpr[c][r], g1);
            u0 = fmaf(bg0[r], xr[c][r], u0);
            u1 = fmaf(bg1[r], xr[c][r], u1);
          }
          const float n0 = fmaf(ac, g0, fmaf(-as, g1, u0));
          const float n1 = fmaf(as, g0, fmaf(ac, g1, u1));
          v0[c] = n0;
          v1[c] = n1;
#pragma unroll
          for (int r = 0; r < R; ++r) yp[c][r] = fmaf(c0[r], n0, fmaf(c1[r], n1, yp[c][r]));
        }
        *reinterpret_cast<float4*>(st + (2 * k) * P + 4 * q) = h0[j];
        *reinterpret_cast<float4*>(st + (2 * k + 1) * P + 4 * q) = h1[j];
      }
    }
  }
  // y: lanes of a warp with the same column quad fold by shuffles, then the
  // warps' partials are summed through shared memory
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int r = 0; r < R; ++r)
      for (int o = PQ; o < 32; o <<= 1) yp[c][r] += __shfl_xor_sync(0xffffffffu, yp[c][r], o);
  if (lane < PQ) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int r = 0; r < R; ++r) yred[(warp * P + 4 * q + c) * R + r] = yp[c][r];
  }
  __syncthreads();
  T* out = static_cast<T*>(a.out);
  for (int i = tid; i < P * R; i += kThreads) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) acc += yred[w * P * R + i];
    st_act(out + x_base + i, acc);
  }
}

template <typename T>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t s) {
  const int N = (int)a.N, P = (int)a.P, R = a.R;
  const size_t smem = sizeof(float) * decode_smem_floats(N, P, R);
  const dim3 grid((unsigned)(a.batch * a.H));
  switch (R) {
    case 1: decode_kernel<T, 1><<<grid, kThreads, smem, s>>>(a); break;
    case 2: decode_kernel<T, 2><<<grid, kThreads, smem, s>>>(a); break;
    case 4: decode_kernel<T, 4><<<grid, kThreads, smem, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(int64_t N, int64_t P, int R) {
  if (!(R == 1 || R == 2 || R == 4)) return false;
  if (P % 4 != 0 || P < 4 || P > 1024) return false;
  if (kThreads % (P / 4) != 0) return false;
  if (N < 2 || N % 2 != 0 || N > 1024) return false;
  return sizeof(float) * decode_smem_floats((int)N, (int)P, R) <= 48 * 1024;
}

cudaError_t launch_decode(const DecodeArgs& a, bool bf16, cudaStream_t s) {
  return bf16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace m3
