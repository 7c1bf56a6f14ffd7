// Backward pass of the Mamba-3 scan: the gradients of <y, dy> + <h_final,
// d_final> for a prefill that starts from a zero state, on the CUDA cores.
//
// Forward (Prop. 1 and the rotation, sec. 4.1 and 4.2 of
// "MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc); MIMO
// rank R, sec. 3 of "Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org)),
// per (batch, head), with Bb = B + B_bias and Cb = C + C_bias:
//   U_t = Bb_t x_t^T,  G_t = h_{t-1} + beta_hat_t U_{t-1},
//   h_t = alpha_t Rot(phi_t) G_t + gamma_t U_t,  y_t = Cb_t^T h_t,
//   phi_t = dt_t theta_t,  alpha = exp(dt A),  gamma = lambda dt,  beta_hat = (1 - lambda) dt.
// Reverse recurrence with g_t = dL/dh_t (carried from t+1 as q_{t+1}):
//   g_t += Cb_t dy_t^T                   dCb_t = h_t dy_t
//   r = Rot(phi_t) G_t                    dalpha_t = <g_t, r>
//   dphi_t[k] = alpha_t sum_p (g_{2k+1} r_{2k} - g_{2k} r_{2k+1})
//   q_t = alpha_t Rot(phi_t)^T g_t        (= dL/dG_t = dL/dh_{t-1})
//   dgamma_t = <g_t, U_t>,  dbeta_hat_t = <q_t, U_{t-1}>
//   dU_t = gamma_t g_t + beta_hat_{t+1} q_{t+1}
//   dBb_t = dU_t x_t,  dx_t = dU_t^T Bb_t
//   ddt_t = A alpha dalpha + lambda dgamma + (1 - lambda) dbeta_hat + sum_k theta_k dphi_k
//   dlambda_t = dt (dgamma - dbeta_hat),  dA += dt alpha dalpha,  dtheta_t = dt dphi_t.
//
// One CTA per (batch, head), 256 threads; a work item is a rotating row pair
// times four columns and a thread owns items tid + 256 m (m < 4), so N P <=
// 8192. The states h_t are needed in reverse order: a forward sweep stores the
// state entering every chunk of kBChunk tokens (checkpoints); the reverse
// sweep recomputes each chunk's states from its checkpoint into a per-CTA
// scratch and walks the chunk backwards. g and the carried beta_hat q stay in
// registers. Reductions: over the 16 (P/4) lanes of a row pair by warp
// shuffles, over row pairs through shared-memory atomics, and into the
// gradients shared by heads, batches or tokens (dB, dC, dtheta, dA, the bias
// gradients) by global atomics. The order in which those atomics land varies
// from run to run, so these gradients vary in their last bits between runs
// (they are not bit-reproducible); the others are.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace m3 {
namespace {

constexpr int kBThreads = 256;
constexpr int kBItems = 4;
constexpr int kBChunk = 64;  // tokens between state checkpoints

template <typename T, int R>
__device__ __forceinline__ void ld_quad_g(const T* p, float (&v)[4][R]) {
#pragma unroll
  for (int i = 0; i < 4 * R; ++i) v[i / R][i % R] = ld_act(p + i);
}

template <typename T, int R>
__global__ void __launch_bounds__(kBThreads)
    scan_bwd_kernel(BwdArgs a, float* __restrict__ ckpt, float* __restrict__ scr) {
  extern __shared__ float smb[];
  const int N = (int)a.N, P = (int)a.P, K2 = N / 2, PQ = P / 4;
  const int64_t L = a.L, H = a.H, G = a.G;
  const int64_t bh = blockIdx.x, b = bh / H, h = bh % H, g = h / (H / G);
  const int tid = threadIdx.x, lane = tid & 31;
  const int q = tid % PQ;  // column quad (PQ divides 32)
  const int items = K2 * PQ;
  const int nC = (int)((L + kBChunk - 1) / kBChunk);
  const int64_t NP = (int64_t)N * P, NR = (int64_t)N * R, PR = (int64_t)P * R;
  float* ck = ckpt + bh * (int64_t)nC * NP;   // [nC][N][P]
  float* sc = scr + bh * (int64_t)kBChunk * NP;  // [kBChunk][N][P]
  // shared tables of one token
  float* t_bg = smb;              // gamma Bb_t        [N][R] (forward)
  float* t_bp = t_bg + NR;        // beta_hat Bb_{t-1} [N][R] (forward)
  float* t_bb = t_bp + NR;        // Bb_t              [N][R]
  float* t_bq = t_bb + NR;        // Bb_{t-1} (0 at t = 0) [N][R]
  float* t_cb = t_bq + NR;        // Cb_t              [N][R]
  float* t_c = t_cb + NR;         // cos phi           [K2]
  float* t_s = t_c + K2;          // sin phi           [K2]
  float* dxs = t_s + K2;          // dx accumulator    [P][R]
  float* scal = dxs + PR;         // dalpha, dgamma, dbeta_hat, sum theta dphi, alpha, gamma, bhat, dt
  const T* x = static_cast<const T*>(a.x);
  const T* Bm = static_cast<const T*>(a.B);
  const T* Cm = static_cast<const T*>(a.C);
  const T* dy = static_cast<const T*>(a.dy);
  const float A_h = a.A[h];

  int kqs[kBItems];
#pragma unroll
  for (int m = 0; m < kBItems; ++m) {
    const int it = tid + kBThreads * m;
    kqs[m] = it < items ? it / PQ : -1;
  }
  auto x_at = [&](int64_t t) { return x + ((b * L + t) * H + h) * PR + 4 * q * R; };

  // token t's tables: the forward products gamma Bb_t and beta_hat Bb_{t-1},
  // the plain rows Bb_t, Bb_{t-1}, Cb_t for the reverse step, cos / sin phi_t,
  // and alpha, gamma, beta_hat, dt of the token
  auto prep = [&](int64_t t) {
    const float d = a.dt[(b * L + t) * H + h], lm = a.lam[(b * L + t) * H + h];
    const float alpha = expf(d * A_h), gamma = lm * d, bhat = (1.f - lm) * d;
    const int64_t bc = ((b * L + t) * G + g) * NR, bcp = bc - G * NR;  // token t-1: one L step back
    for (int i = tid; i < NR; i += kBThreads) {
      const float bias_b = a.B_bias ? a.B_bias[h * NR + i] : 0.f;
      const float bias_c = a.C_bias ? a.C_bias[h * NR + i] : 0.f;
      const float bb = ld_act(Bm + bc + i) + bias_b;
      const float bq = t > 0 ? ld_act(Bm + bcp + i) + bias_b : 0.f;
      t_bb[i] = bb;
      t_bq[i] = bq;
      t_bg[i] = gamma * bb;
      t_bp[i] = bhat * bq;
      t_cb[i] = ld_act(Cm + bc + i) + bias_c;
    }
    const float* th = a.theta + ((b * L + t) * G + g) * K2;
    for (int k = tid; k < K2; k += kBThreads) {
      float sn, cs;
      sincosf(d * th[k], &sn, &cs);
      t_c[k] = cs;
      t_s[k] = sn;
    }
    if (tid == 0) {
      scal[4] = alpha;
      scal[5] = gamma;
      scal[6] = bhat;
      scal[7] = d;
    }
  };

  // one forward token on the thread's items (tables of token t prepared)
  auto fwd_token = [&](int64_t t, float4 (&h0)[kBItems], float4 (&h1)[kBItems]) {
    float xr[4][R], xp[4][R];
    ld_quad_g<T, R>(x_at(t), xr);
    if (t > 0) {
      ld_quad_g<T, R>(x_at(t - 1), xp);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int r = 0; r < R; ++r) xp[c][r] = 0.f;
    }
    const float alpha = scal[4];
#pragma unroll
    for (int m = 0; m < kBItems; ++m) {
      const int kq = kqs[m];
      if (kq < 0) continue;
      const float ac = alpha * t_c[kq], as = alpha * t_s[kq];
      float* v0 = reinterpret_cast<float*>(&h0[m]);
      float* v1 = reinterpret_cast<float*>(&h1[m]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float g0 = v0[c], g1 = v1[c], u0 = 0.f, u1 = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          g0 = fmaf(t_bp[(2 * kq) * R + r], xp[c][r], g0);
          g1 = fmaf(t_bp[(2 * kq + 1) * R + r], xp[c][r], g1);
          u0 = fmaf(t_bg[(2 * kq) * R + r], xr[c][r], u0);
          u1 = fmaf(t_bg[(2 * kq + 1) * R + r], xr[c][r], u1);
        }
        v0[c] = fmaf(ac, g0, fmaf(-as, g1, u0));
        v1[c] = fmaf(as, g0, fmaf(ac, g1, u1));
      }
    }
  };
  auto store_state = [&](float* dst, const float4 (&h0)[kBItems], const float4 (&h1)[kBItems]) {
#pragma unroll
    for (int m = 0; m < kBItems; ++m) {
      const int kq = kqs[m];
      if (kq < 0) continue;
      *reinterpret_cast<float4*>(dst + (2 * kq) * P + 4 * q) = h0[m];
      *reinterpret_cast<float4*>(dst + (2 * kq + 1) * P + 4 * q) = h1[m];
    }
  };
  auto load_state = [&](const float* src, float4 (&h0)[kBItems], float4 (&h1)[kBItems]) {
#pragma unroll
    for (int m = 0; m < kBItems; ++m) {
      const int kq = kqs[m];
      if (kq < 0) {
        h0[m] = h1[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      h0[m] = *reinterpret_cast<const float4*>(src + (2 * kq) * P + 4 * q);
      h1[m] = *reinterpret_cast<const float4*>(src + (2 * kq + 1) * P + 4 * q);
    }
  };

  // 1. forward sweep: the state entering every chunk
  {
    float4 h0[kBItems], h1[kBItems];
#pragma unroll
    for (int m = 0; m < kBItems; ++m) h0[m] = h1[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t t = 0; t < L; ++t) {
      if (t % kBChunk == 0) store_state(ck + (t / kBChunk) * NP, h0, h1);
      prep(t);
      __syncthreads();
      fwd_token(t, h0, h1);
      __syncthreads();
    }
  }

  // 2. reverse sweep, chunk by chunk
  float4 g0r[kBItems], g1r[kBItems], u0r[kBItems], u1r[kBItems];  // g, carried beta_hat q
#pragma unroll
  for (int m = 0; m < kBItems; ++m) {
    g0r[m] = g1r[m] = u0r[m] = u1r[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int kq = kqs[m];
    if (kq >= 0 && a.d_final) {
      const float* df = a.d_final + bh * NP;
      g0r[m] = *reinterpret_cast<const float4*>(df + (2 * kq) * P + 4 * q);
      g1r[m] = *reinterpret_cast<const float4*>(df + (2 * kq + 1) * P + 4 * q);
    }
  }
  for (int i = tid; i < PR + 8; i += kBThreads) dxs[i] = 0.f;  // dx accumulator and scalars
  float dA_acc = 0.f;  // thread 0
  __syncthreads();
  for (int c = nC - 1; c >= 0; --c) {
    const int64_t t0 = (int64_t)c * kBChunk;
    const int64_t t1 = (t0 + kBChunk < L) ? t0 + kBChunk : L;
    // 2a. the chunk's states h_t into the scratch
    {
      float4 h0[kBItems], h1[kBItems];
      load_state(ck + c * NP, h0, h1);
      for (int64_t t = t0; t < t1; ++t) {
        prep(t);
        __syncthreads();
        fwd_token(t, h0, h1);
        store_state(sc + (t - t0) * NP, h0, h1);
        __syncthreads();
      }
    }
    // 2b. the chunk's tokens in reverse
    for (int64_t t = t1 - 1; t >= t0; --t) {
      prep(t);
      __syncthreads();
      const float alpha = scal[4], gamma = scal[5], bhat = scal[6], d = scal[7];
      float xr[4][R], xp[4][R], dyv[4][R];
      ld_quad_g<T, R>(x_at(t), xr);
      if (t > 0) {
        ld_quad_g<T, R>(x_at(t - 1), xp);
      } else {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int r = 0; r < R; ++r) xp[cc][r] = 0.f;
      }
      ld_quad_g<T, R>(dy + ((b * L + t) * H + h) * PR + 4 * q * R, dyv);
      const float* hcur = sc + (t - t0) * NP;
      const float* hprv = t > t0 ? sc + (t - 1 - t0) * NP : ck + c * NP;
      float s_alpha = 0.f, s_gamma = 0.f, s_bhat = 0.f;
      float dxp[4][R];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int r = 0; r < R; ++r) dxp[cc][r] = 0.f;
#pragma unroll
      for (int m = 0; m < kBItems; ++m) {
        const int kq = kqs[m];
        // every lane of a row pair's 16-lane group runs the shuffles below,
        // so the item loop stays uniform within each group (kq is -1 for a
        // whole group or for none of it)
        const bool live = kq >= 0;
        const int n0 = 2 * (live ? kq : 0), n1 = n0 + 1;
        const float ck_ = live ? t_c[n0 / 2] : 0.f, sk_ = live ? t_s[n0 / 2] : 0.f;
        float4 hc0 = make_float4(0.f, 0.f, 0.f, 0.f), hc1 = hc0, hp0 = hc0, hp1 = hc0;
        if (live) {
          hc0 = *reinterpret_cast<const float4*>(hcur + n0 * P + 4 * q);
          hc1 = *reinterpret_cast<const float4*>(hcur + n1 * P + 4 * q);
          hp0 = *reinterpret_cast<const float4*>(hprv + n0 * P + 4 * q);
          hp1 = *reinterpret_cast<const float4*>(hprv + n1 * P + 4 * q);
        }
        const float* vc0 = reinterpret_cast<const float*>(&hc0);
        const float* vc1 = reinterpret_cast<const float*>(&hc1);
        const float* vp0 = reinterpret_cast<const float*>(&hp0);
        const float* vp1 = reinterpret_cast<const float*>(&hp1);
        float* g0 = reinterpret_cast<float*>(&g0r[m]);
        float* g1 = reinterpret_cast<float*>(&g1r[m]);
        float* w0 = reinterpret_cast<float*>(&u0r[m]);
        float* w1 = reinterpret_cast<float*>(&u1r[m]);
        float dC0[R], dC1[R], dB0[R], dB1[R];
#pragma unroll
        for (int r = 0; r < R; ++r) dC0[r] = dC1[r] = dB0[r] = dB1[r] = 0.f;
        float dphi = 0.f;
        if (live) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            float ut0 = 0.f, ut1 = 0.f, up0 = 0.f, up1 = 0.f, gy0 = 0.f, gy1 = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
              ut0 = fmaf(t_bb[n0 * R + r], xr[cc][r], ut0);
              ut1 = fmaf(t_bb[n1 * R + r], xr[cc][r], ut1);
              up0 = fmaf(t_bq[n0 * R + r], xp[cc][r], up0);
              up1 = fmaf(t_bq[n1 * R + r], xp[cc][r], up1);
              gy0 = fmaf(t_cb[n0 * R + r], dyv[cc][r], gy0);
              gy1 = fmaf(t_cb[n1 * R + r], dyv[cc][r], gy1);
              dC0[r] = fmaf(vc0[cc], dyv[cc][r], dC0[r]);
              dC1[r] = fmaf(vc1[cc], dyv[cc][r], dC1[r]);
            }
            const float ga = g0[cc] + gy0, gb = g1[cc] + gy1;  // g_t
            const float G0 = fmaf(bhat, up0, vp0[cc]), G1 = fmaf(bhat, up1, vp1[cc]);
            const float r0 = ck_ * G0 - sk_ * G1, r1 = sk_ * G0 + ck_ * G1;
            s_alpha += ga * r0 + gb * r1;
            dphi += alpha * (gb * r0 - ga * r1);
            s_gamma += ga * ut0 + gb * ut1;
            const float q0 = alpha * (ck_ * ga + sk_ * gb), q1 = alpha * (ck_ * gb - sk_ * ga);
            s_bhat += q0 * up0 + q1 * up1;
            const float du0 = fmaf(gamma, ga, w0[cc]), du1 = fmaf(gamma, gb, w1[cc]);
#pragma unroll
            for (int r = 0; r < R; ++r) {
              dB0[r] = fmaf(du0, xr[cc][r], dB0[r]);
              dB1[r] = fmaf(du1, xr[cc][r], dB1[r]);
              dxp[cc][r] = fmaf(du0, t_bb[n0 * R + r], fmaf(du1, t_bb[n1 * R + r], dxp[cc][r]));
            }
            w0[cc] = bhat * q0;  // beta_hat_t q_t, the dU term of token t-1
            w1[cc] = bhat * q1;
            g0[cc] = q0;         // dL/dh_{t-1}
            g1[cc] = q1;
          }
        }
        // the row pair's sums over its PQ column quads (lanes that differ in q)
        for (int o = 1; o < PQ; o <<= 1) {
          dphi += __shfl_xor_sync(0xffffffffu, dphi, o);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            dC0[r] += __shfl_xor_sync(0xffffffffu, dC0[r], o);
            dC1[r] += __shfl_xor_sync(0xffffffffu, dC1[r], o);
            dB0[r] += __shfl_xor_sync(0xffffffffu, dB0[r], o);
            dB1[r] += __shfl_xor_sync(0xffffffffu, dB1[r], o);
          }
        }
        if (live && q == 0) {
          const int64_t bc = ((b * L + t) * G + g) * NR;
          const int kq2 = n0 / 2;
          const float th = a.theta[((b * L + t) * G + g) * K2 + kq2];
          atomicAdd(a.dtheta + ((b * L + t) * G + g) * K2 + kq2, d * dphi);
          atomicAdd(&scal[3], th * dphi);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            atomicAdd(a.dC + bc + n0 * R + r, dC0[r]);
            atomicAdd(a.dC + bc + n1 * R + r, dC1[r]);
            atomicAdd(a.dB + bc + n0 * R + r, dB0[r]);
            atomicAdd(a.dB + bc + n1 * R + r, dB1[r]);
            if (a.dC_bias) {
              atomicAdd(a.dC_bias + h * NR + n0 * R + r, dC0[r]);
              atomicAdd(a.dC_bias + h * NR + n1 * R + r, dC1[r]);
            }
            if (a.dB_bias) {
              atomicAdd(a.dB_bias + h * NR + n0 * R + r, dB0[r]);
              atomicAdd(a.dB_bias + h * NR + n1 * R + r, dB1[r]);
            }
          }
        }
      }
      // dx: this thread's column quad, summed over its row pairs here and
      // over the CTA's other row pairs through shared memory
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int r = 0; r < R; ++r) atomicAdd(&dxs[(4 * q + cc) * R + r], dxp[cc][r]);
      // the scalars: warp sums, then shared memory
      for (int o = 16; o > 0; o >>= 1) {
        s_alpha += __shfl_xor_sync(0xffffffffu, s_alpha, o);
        s_gamma += __shfl_xor_sync(0xffffffffu, s_gamma, o);
        s_bhat += __shfl_xor_sync(0xffffffffu, s_bhat, o);
      }
      if (lane == 0) {
        atomicAdd(&scal[0], s_alpha);
        atomicAdd(&scal[1], s_gamma);
        atomicAdd(&scal[2], s_bhat);
      }
      __syncthreads();
      const int64_t o_t = (b * L + t) * H + h;
      for (int i = tid; i < PR; i += kBThreads) {
        a.dx[o_t * PR + i] = dxs[i];
        dxs[i] = 0.f;
      }
      if (tid == 0) {
        const float lm = a.lam[o_t];
        const float dalpha = scal[0], dgamma = scal[1], dbhat = scal[2], tdphi = scal[3];
        a.ddt[o_t] = A_h * alpha * dalpha + lm * dgamma + (1.f - lm) * dbhat + tdphi;
        a.dlam[o_t] = d * (dgamma - dbhat);
        dA_acc = fmaf(d * alpha, dalpha, dA_acc);
        scal[0] = scal[1] = scal[2] = scal[3] = 0.f;
      }
      __syncthreads();
    }
  }
  if (tid == 0) atomicAdd(a.dA + h, dA_acc);
}

template <typename T>
cudaError_t launch_t(const BwdArgs& a, float* ckpt, float* scr, cudaStream_t s) {
  const size_t smem = sizeof(float) * (5 * (size_t)a.N * a.R + a.N + (size_t)a.P * a.R + 8);
  const dim3 grid((unsigned)(a.batch * a.H));
  switch (a.R) {
    case 1: scan_bwd_kernel<T, 1><<<grid, kBThreads, smem, s>>>(a, ckpt, scr); break;
    case 2: scan_bwd_kernel<T, 2><<<grid, kBThreads, smem, s>>>(a, ckpt, scr); break;
    case 4: scan_bwd_kernel<T, 4><<<grid, kBThreads, smem, s>>>(a, ckpt, scr); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

bool scan_bwd_supported(int64_t N, int64_t P, int R) {
  if (!(R == 1 || R == 2 || R == 4)) return false;
  if (P < 4 || P % 4 != 0 || 32 % (P / 4) != 0) return false;
  if (N < 2 || N % 2 != 0 || (N / 2) * (P / 4) > (int64_t)kBThreads * kBItems) return false;
  return sizeof(float) * (5 * N * R + N + P * R + 8) <= 48 * 1024;
}

// The larger of the two paths' scratch where the shape allows both (which
// one runs depends on the pointers' alignment too), so that one size serves.
size_t scan_bwd_workspace_bytes(const BwdArgs& a, bool bf16) {
  if (a.batch * a.H == 0 || a.L == 0) return 0;
  const int64_t nC = (a.L + kBChunk - 1) / kBChunk;
  const size_t simt = sizeof(float) * (size_t)(nC + kBChunk) * a.N * a.P * (size_t)(a.batch * a.H);
  BwdArgs shape = a;
  shape.x = shape.dy = nullptr;
  shape.dB = shape.dC = nullptr;
  shape.B = shape.C = nullptr;
  if (!scan_bwd_tc_ok(shape, bf16)) return simt;
  const size_t tc = scan_bwd_tc_workspace(a);
  return tc > simt ? tc : simt;
}

cudaError_t launch_scan_bwd(const BwdArgs& a, bool bf16, void* ws, cudaStream_t s) {
  const int64_t nseq = a.batch * a.H;
  const int64_t nC = (a.L + kBChunk - 1) / kBChunk;
  // the accumulated gradients start from zero
  cudaError_t e = cudaMemsetAsync(a.dA, 0, sizeof(float) * a.H, s);
  const size_t nbc = (size_t)a.batch * a.L * a.G * a.N * a.R;
  if (e == cudaSuccess) e = cudaMemsetAsync(a.dB, 0, sizeof(float) * nbc, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.dC, 0, sizeof(float) * nbc, s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(a.dtheta, 0, sizeof(float) * a.batch * a.L * a.G * (a.N / 2), s);
  if (e == cudaSuccess && a.dB_bias)
    e = cudaMemsetAsync(a.dB_bias, 0, sizeof(float) * a.H * a.N * a.R, s);
  if (e == cudaSuccess && a.dC_bias)
    e = cudaMemsetAsync(a.dC_bias, 0, sizeof(float) * a.H * a.N * a.R, s);
  if (e != cudaSuccess || nseq == 0 || a.L == 0) return e;
  const bool tc = scan_bwd_tc_ok(a, bf16);
  if (tc) {
    // the tensor-core path accumulates ddt and dlambda too (a chunk adds the
    // trapezoid term of the token after it)
    const size_t nt = (size_t)a.batch * a.L * a.H;
    e = cudaMemsetAsync(a.ddt, 0, sizeof(float) * nt, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dlam, 0, sizeof(float) * nt, s);
    if (e != cudaSuccess) return e;
  }
  float* w = static_cast<float*>(ws);
  if (w == nullptr) {
    e = cudaMallocAsync(reinterpret_cast<void**>(&w), scan_bwd_workspace_bytes(a, bf16), s);
    if (e != cudaSuccess) return e;
  }
  if (tc) {
    e = launch_scan_bwd_tc(a, w, s);
  } else {
    float* ckpt = w;
    float* scr = w + (size_t)nC * a.N * a.P * nseq;
    e = bf16 ? launch_t<__nv_bfloat16>(a, ckpt, scr, s) : launch_t<float>(a, ckpt, scr, s);
  }
  if (ws == nullptr) {
    const cudaError_t f = cudaFreeAsync(w, s);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

}  // namespace m3
