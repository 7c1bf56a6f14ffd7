// CUDA-core chunked prefill of the Mamba-3 scan (fp32 arithmetic).
//
// One CTA walks one (batch, head) sequence chunk by chunk. Within a chunk of
// Q tokens starting at t0 (chunk-local cumulative sums, state carried between
// chunks in the explicit frame):
//   Lam_t = sum_{u=t0..t} dt_u A                       (decay exponent)
//   Phi_t = sum_{u=t0..t} dt_u theta_u (per pair)      (rotation angle)
//   Bt_s = Rot(-Phi_s)(B_s + bias), Ct_t = Rot(-Phi_t)(C_t + bias)
//        -- the rotation folded into B and C (Prop. 3, sec. 4.2 of "MAMBA-3:
//           IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc))
//   S[(t,r'),(s,r)] = Ct_t[:,r'] . Bt_s[:,r]  masked by
//   M[t,s] = exp(Lam_t - Lam_s) (gamma_s + [s<t] beta_hat_{s+1}), s <= t
//        -- decay (1-semiseparable) times the 2-band trapezoid mask
//           (sec. 1 of "Mamba-3: Improved Sequence Modeling using State Space
//           Principles" (papernotes.org); SSD form Y = (L o C B^T) X)
//   y_t = sum_s S M x_s + exp(Lam_t) Ct_t^T H_in
//   H_out = Rot(Phi_end)(exp(Lam_end) H_in + sum_s exp(Lam_end-Lam_s) w_s Bt_s x_s^T)
//   w_s = gamma_s + beta_hat_{s+1}   (beta_hat of the token after s; 0 at the end)
// H_in of the first chunk is zero, or the caller's entering state. This is
// the path for the fp32 precision mode and for bf16 shapes that the
// tensor-core kernel does not take.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace m3 {
namespace {

constexpr int kThreads = 256;

struct SmemLayout {
  int ldn, ldp, ldq;
  size_t off_Bt, off_Ct, off_X, off_H, off_S, off_Phi, off_lam, off_w, off_gam, off_bnx, off_dt,
      total;  // in floats
};

__host__ __device__ inline SmemLayout make_layout(int N, int P, int R, int Q) {
  SmemLayout l;
  const int QR = Q * R;
  l.ldn = N + 1;
  l.ldp = P + 1;
  l.ldq = QR + 1;
  size_t o = 0;
  l.off_Bt = o; o += (size_t)QR * l.ldn;
  l.off_Ct = o; o += (size_t)QR * l.ldn;
  l.off_X = o; o += (size_t)QR * l.ldp;
  l.off_H = o; o += (size_t)N * l.ldp;
  l.off_S = o; o += (size_t)QR * l.ldq;
  l.off_Phi = o; o += (size_t)Q * (N / 2);
  l.off_lam = o; o += Q;
  l.off_w = o; o += Q;
  l.off_gam = o; o += Q;
  l.off_bnx = o; o += Q;
  l.off_dt = o; o += Q;
  l.total = o;
  return l;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) scan_simt_kernel(ScanArgs a) {
  extern __shared__ float sm[];
  const int64_t L = a.L, H = a.H, G = a.G;
  const int N = (int)a.N, P = (int)a.P, R = a.R, Q = a.Q, QR = Q * R, K2 = N / 2;
  const int64_t bh = blockIdx.x;
  const int64_t b = bh / H, h = bh % H, g = h / (H / G);
  const int tid = threadIdx.x;
  const SmemLayout l = make_layout(N, P, R, Q);
  float* Bt = sm + l.off_Bt;
  float* Ct = sm + l.off_Ct;
  float* Xs = sm + l.off_X;
  float* Hs = sm + l.off_H;
  float* S = sm + l.off_S;
  float* Phi = sm + l.off_Phi;
  float* lamc = sm + l.off_lam;
  float* wv = sm + l.off_w;
  float* gam = sm + l.off_gam;
  float* bnx = sm + l.off_bnx;
  float* dtv = sm + l.off_dt;
  const int ldn = l.ldn, ldp = l.ldp, ldq = l.ldq;
  const T* x = static_cast<const T*>(a.x);
  const T* Bm = static_cast<const T*>(a.B);
  const T* Cm = static_cast<const T*>(a.C);
  T* out = static_cast<T*>(a.out);
  const float A_h = a.A[h];

  // the entering state (explicit frame, pending beta term included), or zero
  if (a.h_init) {
    const float* hi = a.h_init + bh * (int64_t)N * P;
    for (int i = tid; i < N * P; i += kThreads) Hs[(i / P) * ldp + i % P] = hi[i];
  } else {
    for (int i = tid; i < N * ldp; i += kThreads) Hs[i] = 0.f;
  }

  for (int64_t t0 = 0; t0 < L; t0 += Q) {
    const int q = (int)((L - t0 < Q) ? (L - t0) : Q);
    __syncthreads();  // previous chunk fully consumed
    for (int i = tid; i < Q; i += kThreads) {
      const int64_t t = t0 + i;
      float d = 0.f, lm = 0.f, bn = 0.f;
      if (i < q) {
        d = a.dt[(b * L + t) * H + h];
        lm = a.lam[(b * L + t) * H + h];
        if (t + 1 < L) bn = (1.f - a.lam[(b * L + t + 1) * H + h]) * a.dt[(b * L + t + 1) * H + h];
      }
      dtv[i] = d;
      gam[i] = lm * d;
      bnx[i] = bn;
    }
    __syncthreads();
    if (tid == 0) {
      float acc = 0.f;
      for (int i = 0; i < Q; ++i) {
        acc += dtv[i] * A_h;
        lamc[i] = acc;
      }
    }
    for (int k = tid; k < K2; k += kThreads) {
      float phi = 0.f;
      const float* th = a.theta + ((b * L + t0) * G + g) * K2 + k;
      for (int i = 0; i < Q; ++i) {
        const float inc = (i < q) ? dtv[i] * th[(int64_t)i * G * K2] : 0.f;
        phi = wrap_angle(phi + inc);
        Phi[i * K2 + k] = phi;
      }
    }
    __syncthreads();
    for (int i = tid; i < Q; i += kThreads) wv[i] = expf(lamc[Q - 1] - lamc[i]) * (gam[i] + bnx[i]);
    for (int idx = tid; idx < Q * K2 * R; idx += kThreads) {
      const int i = idx / (K2 * R), rem = idx % (K2 * R), k = rem / R, r = rem % R;
      float b0 = 0.f, b1 = 0.f, c0 = 0.f, c1 = 0.f;
      if (i < q) {
        const int64_t base = ((b * L + t0 + i) * G + g) * (int64_t)N * R;
        b0 = ld_act(Bm + base + (2 * k) * R + r);
        b1 = ld_act(Bm + base + (2 * k + 1) * R + r);
        c0 = ld_act(Cm + base + (2 * k) * R + r);
        c1 = ld_act(Cm + base + (2 * k + 1) * R + r);
        if (a.B_bias) {
          b0 += a.B_bias[(h * N + 2 * k) * R + r];
          b1 += a.B_bias[(h * N + 2 * k + 1) * R + r];
        }
        if (a.C_bias) {
          c0 += a.C_bias[(h * N + 2 * k) * R + r];
          c1 += a.C_bias[(h * N + 2 * k + 1) * R + r];
        }
      }
      float sn, cs;
      sincosf(Phi[i * K2 + k], &sn, &cs);
      float* brow = Bt + (i * R + r) * ldn;
      float* crow = Ct + (i * R + r) * ldn;
      brow[2 * k] = cs * b0 + sn * b1;  // Rot(-Phi) = [[c, s], [-s, c]]
      brow[2 * k + 1] = -sn * b0 + cs * b1;
      crow[2 * k] = cs * c0 + sn * c1;
      crow[2 * k + 1] = -sn * c0 + cs * c1;
    }
    for (int idx = tid; idx < Q * R * P; idx += kThreads) {
      const int i = idx / (R * P), rem = idx % (R * P), p = rem / R, r = rem % R;
      Xs[(i * R + r) * ldp + p] =
          (i < q) ? ld_act(x + ((b * L + t0 + i) * H + h) * (int64_t)P * R + rem) : 0.f;
    }
    __syncthreads();
    // masked scores over the flattened (token, rank) index
    for (int idx = tid; idx < QR * QR; idx += kThreads) {
      const int ar = idx / QR, cr = idx % QR, ti = ar / R, si = cr / R;
      float m;
      if (si > ti) m = 0.f;
      else if (si == ti) m = gam[si];
      else m = expf(lamc[ti] - lamc[si]) * (gam[si] + bnx[si]);
      float acc = 0.f;
      if (m != 0.f) {
        const float* cr_ = Ct + ar * ldn;
        const float* br_ = Bt + cr * ldn;
        for (int n = 0; n < N; ++n) acc = fmaf(cr_[n], br_[n], acc);
      }
      S[ar * ldq + cr] = m * acc;
    }
    __syncthreads();
    // outputs: intra-chunk part plus the entering state's contribution
    for (int idx = tid; idx < QR * P; idx += kThreads) {
      const int ar = idx / P, p = idx % P, ti = ar / R, r = ar % R;
      if (ti >= q) continue;
      float acc = 0.f;
      const int cmax = (ti + 1) * R;
      for (int cr = 0; cr < cmax; ++cr) acc = fmaf(S[ar * ldq + cr], Xs[cr * ldp + p], acc);
      float off = 0.f;
      const float* crow = Ct + ar * ldn;
      for (int n = 0; n < N; ++n) off = fmaf(crow[n], Hs[n * ldp + p], off);
      const float yv = fmaf(expf(lamc[ti]), off, acc);
      st_act(out + ((b * L + t0 + ti) * H + h) * (int64_t)P * R + (int64_t)p * R + r, yv);
    }
    __syncthreads();
    // chunk state, then back to the explicit frame
    const float e_end = expf(lamc[Q - 1]);
    for (int idx = tid; idx < K2 * P; idx += kThreads) {
      const int k = idx / P, p = idx % P;
      float h0 = e_end * Hs[(2 * k) * ldp + p];
      float h1 = e_end * Hs[(2 * k + 1) * ldp + p];
      for (int cr = 0; cr < QR; ++cr) {
        const float xw = wv[cr / R] * Xs[cr * ldp + p];
        h0 = fmaf(Bt[cr * ldn + 2 * k], xw, h0);
        h1 = fmaf(Bt[cr * ldn + 2 * k + 1], xw, h1);
      }
      float sn, cs;
      sincosf(Phi[(Q - 1) * K2 + k], &sn, &cs);
      Hs[(2 * k) * ldp + p] = cs * h0 - sn * h1;
      Hs[(2 * k + 1) * ldp + p] = sn * h0 + cs * h1;
    }
  }
  __syncthreads();
  if (a.final_state) {
    float* fs = a.final_state + bh * (int64_t)N * P;
    for (int i = tid; i < N * P; i += kThreads) fs[i] = Hs[(i / P) * ldp + (i % P)];
  }
}

}  // namespace

size_t scan_simt_smem_bytes(int64_t N, int64_t P, int R, int Q) {
  if (N > 4096 || P > 4096 || R > 64 || Q > 4096) return (size_t)-1;
  return make_layout((int)N, (int)P, R, Q).total * sizeof(float);
}

cudaError_t launch_scan_simt(const ScanArgs& a, bool bf16, cudaStream_t s) {
  const size_t smem = scan_simt_smem_bytes(a.N, a.P, a.R, a.Q);
  const dim3 grid((unsigned)(a.batch * a.H));
  cudaError_t e;
  if (bf16) {
    e = cudaFuncSetAttribute(scan_simt_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    scan_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(scan_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    scan_simt_kernel<float><<<grid, kThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace m3
